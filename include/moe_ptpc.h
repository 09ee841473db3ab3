/*
 * moe_ptpc.h - C ABI of the GB300 (sm_103a) PTPC-FP8 Mixture-of-Experts layer.
 *
 * The layer ("Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", the MoE
 * paragraph of the model description, and its SparseCore / GMM V2 paragraphs;
 * "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series",
 * sections 2.1.1, 2.1.4 and 2.1.5):
 *
 *   logits -> softmax top-k routing -> histogram + prefix sum + permutation
 *   into expert-contiguous rows -> per-token FP8 e4m3 quantisation ->
 *   grouped gate/up GEMM with fused SwiGLU -> per-token requantisation ->
 *   grouped down GEMM -> top-k-weighted unpermute-combine to bf16.
 *
 * PTPC ("per-token activation, per-channel weight", section 2.1.1 and Figure 3
 * of the MI300X page): every activation row carries one fp32 scale, every
 * weight output channel one fp32 scale, and a GEMM output element is
 *   out[r, n] = s_a[r] * s_w[n] * sum_k qa[r, k] * qw[n, k].
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers owned by the caller unless a parameter says
 *    otherwise; nothing here allocates device memory, and every call is
 *    asynchronous on `stream` (NULL = the legacy default stream).
 *  - Matrices are row-major with the reduction dimension contiguous.
 *  - bf16 values are passed as uint16_t bit patterns; FP8 values as uint8_t
 *    e4m3 codes (OCP "E4M3": bias 7, max 448, no infinities).
 *  - The return value is a status (moe_status) for argument and launch
 *    errors, known before the kernels run. Errors found by a running kernel
 *    (a bounded wait that expired) are reported by moe_workspace_status() for
 *    moe_forward and its variants (each workspace has its own error word),
 *    and by moe_device_status() for the standalone steps.
 *  - Device pointers must be 16-byte aligned. D and I must be multiples of
 *    128; 1 <= k <= min(E, 32); E <= 1024.
 *  - NaN or infinite inputs are outside the contract.
 */
#ifndef MOE_PTPC_H
#define MOE_PTPC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* A CUDA stream (cudaStream_t). */
typedef struct CUstream_st* moe_stream_t;

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* null pointer, bad size, misaligned pointer  */
  MOE_ERR_UNSUPPORTED = -2, /* valid but outside the supported shapes      */
  MOE_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed        */
  MOE_ERR_WORKSPACE = -4,   /* workspace missing or too small              */
  MOE_ERR_TIMEOUT = -5      /* a kernel's bounded wait expired             */
} moe_status;

typedef enum moe_dtype { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 } moe_dtype;

typedef enum moe_gemm_kind {
  MOE_GEMM_GATEUP_SWIGLU = 0, /* h = silu(x Wg^T) * (x Wu^T), fp32 out      */
  MOE_GEMM_DOWN = 1           /* y = h Wd^T, fp32 out                        */
} moe_gemm_kind;

/* Dimensions of one layer call. */
typedef struct moe_dims {
  int32_t T;           /* tokens                                             */
  int32_t D;           /* hidden size                                        */
  int32_t E;           /* routed experts                                     */
  int32_t k;           /* experts per token                                  */
  int32_t I;           /* expert intermediate size                           */
  int32_t shared;      /* 1: one always-on shared expert of size I, else 0   */
  int32_t renormalize; /* 1: top-k weights renormalised to sum to 1          */
} moe_dims;

/* Human-readable name of a status code (static string). */
MOE_API const char* moe_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
MOE_API int moe_version(void);

/*
 * moe_router_logits - router gate projection ("Optimizing Qwen 3.5 397B MoE
 * on Ironwood TPU7x", MoE paragraph: the router gate projects each token).
 *   logits[t, e] = sum_d x[t, d] * w_r[e, d], accumulated in fp64 and rounded
 *   once to fp32, so the fp32 logits are the exactly rounded dot products.
 *   x      [T, D] bf16;  w_r [E, D] bf16;  logits [T, E] fp32 (written).
 * Errors: MOE_ERR_INVALID_ARG for null pointers or non-positive sizes.
 */
MOE_API int moe_router_logits(const uint16_t* x, const uint16_t* w_r, int T,
                              int E, int D, float* logits, moe_stream_t stream);

/*
 * moe_route - softmax top-k routing (same paragraph; the [tokens, k] id and
 * weight arrays of the TPU page's expert-parallel routing paragraph).
 *   Per token: the k largest fp32 logits, ties to the lower expert index, in
 *   descending order; topk_w[t, j] = softmax probability of the chosen expert,
 *   renormalised over the k chosen when `renormalize` (a softmax over the k
 *   chosen logits), else the plain softmax over all E. fp32 arithmetic.
 *   logits [T, E] fp32;  topk_ids [T, k] int32 and topk_w [T, k] fp32 (written).
 * Errors: MOE_ERR_INVALID_ARG (null, T < 0, k outside 1..min(E, 32)),
 *         MOE_ERR_UNSUPPORTED (E > 1024).  T == 0 is a no-op.
 */
MOE_API int moe_route(const float* logits, int T, int E, int k, int renormalize,
                      int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/*
 * moe_permute - expert histogram, prefix sum and stable permutation (TPU
 * page, SparseCore permute paragraph: rows gathered into expert-contiguous
 * order with no padding).
 *   With flat index f = t * k + j and R = T * k:
 *   expert_counts[e]  = #{f : topk_ids[f] == e}                 [E]
 *   expert_offsets    = exclusive prefix sum of counts          [E + 1]
 *   sorted_to_flat[s] = flat index stored at sorted row s        [R]
 *   flat_to_sorted[f] = sorted row of flat index f               [R]
 *   Rows of one expert keep ascending f (a stable counting sort), so every
 *   output is unique and deterministic.
 *   ws: device scratch of at least moe_permute_workspace_size(T, E, k) bytes.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED (E > 1024),
 *         MOE_ERR_WORKSPACE.  Ids outside [0, E) are outside the contract.
 */
MOE_API size_t moe_permute_workspace_size(int T, int E, int k);
MOE_API int moe_permute(const int32_t* topk_ids, int T, int E, int k,
                        int32_t* expert_counts, int32_t* expert_offsets,
                        int32_t* sorted_to_flat, int32_t* flat_to_sorted,
                        void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_permute_noalloc - the same permutation as moe_permute, for callers that
 * cannot allocate device memory. The pages have no counterpart of this entry
 * point; it exists for hosts that embed the layer in a framework which has
 * already reserved the device memory in its own arena, or serving loops that
 * may not call cudaMalloc/cudaFree (both synchronise the device).
 *   Inputs, outputs, results and errors are those of moe_permute; there is no
 *   workspace argument. Scratch: a fixed 1 MiB device array inside the
 *   library (held on every GPU that loads the library until the process
 *   exits), enough for T * k <= 2048 * floor(262144 / E) flat entries (for
 *   E = 128: 4,194,304; for E = 1024: 524,288). Larger calls return
 *   MOE_ERR_UNSUPPORTED before launching anything.
 *   The first call on each device (with that device current) looks up the
 *   array's device address and caches it for the life of the process; make
 *   it before any stream capture on the device. cudaDeviceReset (or anything
 *   else that tears down the device's context and reloads the library's
 *   module) invalidates that cached address: do not call this entry point on
 *   a device after resetting it.
 *   All calls share the array and it keeps the last call's contents (nothing
 *   in it needs to start at zero): calls whose kernels overlap on the GPU race
 *   on it, so the caller must serialise them. Allocates nothing.
 */
MOE_API int moe_permute_noalloc(const int32_t* topk_ids, int T, int E, int k,
                                int32_t* expert_counts, int32_t* expert_offsets,
                                int32_t* sorted_to_flat,
                                int32_t* flat_to_sorted, moe_stream_t stream);

/*
 * moe_quant_ptpc - per-row FP8 e4m3 quantisation with optional scatter
 * (MI300X page, section 2.1.1: per-token activation and per-channel weight
 * scales; section 2.1.5: per-token quantisation fused into the producer).
 *   For each row r < rows of `in` [rows, cols] (bf16 or fp32):
 *     s_r = fp32(max(amax_r, 1e-12) / 448),  q = e4m3_rne_sat(fp32(v / s_r)),
 *   both divisions IEEE fp32. A weight matrix W[N, K] quantised with this
 *   call gets one scale per output channel.
 *   Destinations: if dst_rows is NULL, row r goes to output row r (copies must
 *   be 1); else to rows dst_rows[r * copies + c] for c < copies. If
 *   extra_row_base >= 0 it is also written to row extra_row_base + r.
 *   out_q [*, cols] uint8 and out_scale [*] fp32 are indexed by output row.
 * Errors: MOE_ERR_INVALID_ARG (null, cols not a positive multiple of 16,
 *         bad dtype, copies < 1), MOE_ERR_UNSUPPORTED (cols > 32768 or
 *         copies > 32).
 */
MOE_API int moe_quant_ptpc(const void* in, int in_dtype, int64_t rows, int cols,
                           const int32_t* dst_rows, int copies,
                           int64_t extra_row_base, uint8_t* out_q,
                           float* out_scale, moe_stream_t stream);

/*
 * moe_router_topk - router projection and top-k selection in one kernel (TPU
 * page, closing roadmap paragraph: the top-k fused with the router matmul).
 *   logits[t, e] = sum_d x[t, d] * w_r[e, d] on the tensor cores (bf16
 *   operands, fp32 accumulation; the accumulation order is the hardware's,
 *   so the logits are the fp32 GEMM result, not moe_router_logits' exactly
 *   rounded ones); then, per token, the selection and weights of moe_route
 *   on those logits: the k largest in decreasing order, equal values to the
 *   lower expert index; softmax over the chosen k (renormalize) or over all E.
 *   x [T, D] bf16, w_r [E, D] bf16; topk_ids [T, k] int32 and topk_w [T, k]
 *   fp32 written; logits_out [T, E] fp32 written when not NULL (testing).
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned pointers, k > E),
 *         MOE_ERR_UNSUPPORTED (E > 512, k > 16 or D not a multiple of 64;
 *         moe_router_logits + moe_route cover those).
 */
MOE_API int moe_router_topk(const uint16_t* x, const uint16_t* w_r, int T, int D,
                            int E, int k, int renormalize, int32_t* topk_ids,
                            float* topk_w, float* logits_out, moe_stream_t stream);

/*
 * moe_add_rmsnorm_quant - the MoE block's FP8 input straight from the
 * residual stream: add + RMSNorm + per-token quantisation in one pass (MI300X
 * page, section 2.1.5, the fusion table; the AllReduce of that operator needs
 * tensor parallelism and is not part of it here). For each row t < rows:
 *   r = bf16_rne(fp32(x[t]) + fp32(residual[t]))       -> residual_out[t]
 *   ms = fp32(sum_d r[d]^2 / cols)                      (squares summed in fp64)
 *   inv = fp32_rn(1 / sqrt(fp32(ms + eps)))             (correctly rounded)
 *   v = fp32(fp32(r * inv) * gamma)
 *   s_t = fp32(max(amax(v), 1e-12) / 448), q = e4m3_rne_sat(fp32(v / s_t))
 * and, when gate_w is set, gate_out[t] = sigmoid(v . gate_w).
 *   x, residual, residual_out [rows, cols] bf16; gamma, gate_w [cols] bf16;
 *   destinations of q / s_t as for moe_quant_ptpc (dst_rows, copies,
 *   extra_row_base). residual_out may alias residual (each row is read
 *   before it is written, by the same block).
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned pointers, cols not a
 *         positive multiple of 16, eps < 0 or NaN, copies < 1, gate_w and
 *         gate_out not both set or both NULL), MOE_ERR_UNSUPPORTED (cols >
 *         32768 or copies > 32).
 */
MOE_API int moe_add_rmsnorm_quant(const uint16_t* x, const uint16_t* residual,
                                  const uint16_t* gamma, float eps, int64_t rows,
                                  int cols, uint16_t* residual_out,
                                  const int32_t* dst_rows, int copies,
                                  int64_t extra_row_base, uint8_t* out_q,
                                  float* out_scale, const uint16_t* gate_w,
                                  float* gate_out, moe_stream_t stream);

/*
 * moe_shared_gate - shared-expert gate sigmoid(x[t] . w_g), fp32 (the TPU
 * page's shared expert runs on every token; its gate is a sigmoid).
 *   x [T, D] bf16 (D a multiple of 16);  w_g [D] bf16;  gate [T] fp32.
 */
MOE_API int moe_shared_gate(const uint16_t* x, const uint16_t* w_g, int T,
                            int D, float* gate, moe_stream_t stream);

/*
 * moe_grouped_gemm - PTPC FP8 grouped GEMM on the tcgen05 tensor cores (TPU
 * page, GMM V2 paragraph: gate and up packed in one tile with SwiGLU fused,
 * ragged per-expert row slices with no padding).
 *   Group g owns activation rows [group_offsets[g], group_offsets[g + 1]) of
 *   A [a_rows, K] (e4m3, row scales a_scale [a_rows]); group_offsets is a
 *   DEVICE array of groups + 1 non-decreasing entries <= a_rows.
 *   MOE_GEMM_GATEUP_SWIGLU: W [groups, 2N, K] (rows 0..N-1 gate, N..2N-1 up),
 *     w_scale [groups, 2N]; out [a_rows, N] fp32:
 *       g = s_a s_wg (qa . qwg),  u = s_a s_wu (qa . qwu),  h = g sigmoid(g) u.
 *   MOE_GEMM_DOWN: W [groups, N, K], w_scale [groups, N]; out [a_rows, N] fp32:
 *       y = s_a s_w (qa . qw).
 *   Rows outside every group are not written. Zero-row groups read nothing.
 *   rows_hint: expected rows per non-empty group (<= 0: a_rows / groups); it
 *   only selects the token-tile width.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED (N or K not multiples of
 *         128, out_dtype not MOE_DTYPE_F32, groups > 1025), MOE_ERR_CUDA.
 */
MOE_API int moe_grouped_gemm(int kind, const uint8_t* A, const float* a_scale,
                             int64_t a_rows, const uint8_t* W,
                             const float* w_scale, const int32_t* group_offsets,
                             int groups, int N, int K, void* out, int out_dtype,
                             int rows_hint, moe_stream_t stream);

/*
 * moe_combine - unpermute and top-k-weighted reduction back to bf16 (TPU
 * page, SparseCore unpermute paragraph: indirect gather plus local reduce).
 *   out[t, :] = bf16_rne( sum_{j<k} topk_w[t, j] * y[flat_to_sorted[t k + j], :]
 *                         + shared_gate[t] * y_shared[t, :] )
 *   summed in fp32 in slot order j = 0..k-1, the shared term last.
 *   y [*, D] fp32; flat_to_sorted [T * k]; topk_w [T, k] fp32;
 *   y_shared [T, D] fp32 and shared_gate [T] fp32, both NULL when there is no
 *   shared expert; out [T, D] bf16 (written).
 */
MOE_API int moe_combine(const float* y, const int32_t* flat_to_sorted,
                        const float* topk_w, int T, int k, int D,
                        const float* y_shared, const float* shared_gate,
                        uint16_t* out, moe_stream_t stream);

/*
 * The down projection's output y in fp16 (an encoding between the down GEMM
 * and the combine; the pages leave y's precision open). Rounding y to bf16
 * (8 significant bits) would breach the layer's accuracy bound on the
 * largest outputs; fp16 keeps 11 bits and halves y's HBM traffic against
 * fp32. Its range is guaranteed by construction:
 *   y16[r, n] = fp16_rne( acc[r, n] * w_scale[g, n] * rho_g ),
 *   rho_g = 60000 / (448^2 * K * w_bound[g])   (in fp32: ((60000 / 448^2) / K)
 *                                               / w_bound[g], IEEE divisions),
 *   row_scale[r] = a_scale[r] / rho_g           (IEEE fp32 division),
 * so that y[r, n] = row_scale[r] * y16[r, n] up to fp16 rounding, where acc
 * is the fp32 dot product of the codes. Every product of two e4m3 codes is
 * at most 448^2 in magnitude, so |y16| <= 60000 < 65504 whenever
 * w_bound[g] >= w_scale[g, n] for every n. Values below fp16's normal range
 * (6.1e-5, about 1e-9 of that bound) keep an absolute error of at most
 * 2^-25 * row_scale.
 */

/*
 * moe_scale_max - bound[g] = max_n scale[g, n] over a [groups, N] fp32
 * array (w_bound for the down weights' scales s_d). Returns MOE_OK,
 * MOE_ERR_INVALID_ARG or MOE_ERR_CUDA.
 */
MOE_API int moe_scale_max(const float* scale, int groups, int N, float* bound,
                          moe_stream_t stream);

/*
 * moe_grouped_gemm_down_f16 - moe_grouped_gemm(MOE_GEMM_DOWN) with y written
 * in the fp16 encoding above. Arguments as for moe_grouped_gemm, plus
 * w_bound [groups] fp32 (from moe_scale_max of w_scale), y16 [a_rows, N]
 * fp16 (written, 16-byte aligned) and row_scale [a_rows] fp32 (written for
 * the rows of the groups). Returns as moe_grouped_gemm.
 */
MOE_API int moe_grouped_gemm_down_f16(const uint8_t* A, const float* a_scale,
                                      int64_t a_rows, const uint8_t* W,
                                      const float* w_scale, const float* w_bound,
                                      const int32_t* group_offsets, int groups,
                                      int N, int K, uint16_t* y16, float* row_scale,
                                      int rows_hint, moe_stream_t stream);

/*
 * moe_combine_f16 - moe_combine over the fp16 encoding:
 *   out[t, :] = bf16_rne( sum_{j<k} (topk_w[t, j] * row_scale[r_j]) * y16[r_j, :]
 *                + (shared_gate[t] * row_scale_shared[t]) * y16_shared[t, :] ),
 *   r_j = flat_to_sorted[t k + j], in fp32, slot order, the shared term last.
 *   y16_shared, row_scale_shared and shared_gate are all NULL or all set.
 */
MOE_API int moe_combine_f16(const uint16_t* y16, const float* row_scale,
                            const int32_t* flat_to_sorted, const float* topk_w,
                            int T, int k, int D, const uint16_t* y16_shared,
                            const float* row_scale_shared, const float* shared_gate,
                            uint16_t* out, moe_stream_t stream);

/*
 * moe_forward - the whole layer, every step above chained on `stream`.
 *   x [T, D] bf16. Router input: exactly one of router_logits [T, E] fp32 and
 *   router_w [E, D] bf16. With router_w the routing is moe_router_topk's
 *   (tensor-core logits, top-k fused) where that op applies (E <= 512,
 *   k <= 16, D a multiple of 64) and T * E * D >= 2^20; otherwise
 *   moe_router_logits + moe_route (exactly rounded logits).
 *   Weights, pre-quantised per output channel with moe_quant_ptpc:
 *     w_gu [G, 2I, D] e4m3, s_gu [G, 2I];  w_d [G, D, I] e4m3, s_d [G, D],
 *   where G = E + dims->shared and group E is the shared expert.
 *   shared_gate_w [D] bf16 when dims->shared, else NULL.
 *   out [T, D] bf16 (written). topk_ids_out [T, k] / topk_w_out [T, k]:
 *   optional, receive the routing when non-NULL.
 *   ws: device workspace of moe_forward_workspace_size(dims) bytes; it holds
 *   the routing, permutation, quantised activations and GEMM intermediates,
 *   and in its first 256 bytes the forward's error word: each call clears it
 *   (in stream order) before its first kernel, and its kernels record there
 *   the bounded waits that expire; moe_workspace_status() reads it. Two
 *   forwards in flight at once need two workspaces.
 *   A batch of at most 4 tokens on router_logits (no router_w), with y in
 *   fp32, a supported shape (moe_forward_single_launch) and 16-byte aligned
 *   s_gu and s_d, runs as one
 *   cooperative launch of one CTA per SM ("Ultimate Latency Optimization of
 *   Qwen3 and Qwen3-VL on AMD MI300X Series", sections 2.1.4-2.1.5: the
 *   small-batch MoE is bound by streaming the chosen experts' weights, and
 *   the per-token steps are fused into their neighbours): the same steps and
 *   roundings, products summed in another fp32 order, every intermediate
 *   left in the workspace as the chained kernels leave it; a grid-wide
 *   barrier whose wait expires sets error bit 5 (1 << 5). It runs only when
 *   the environment variable MOE_SMALL_FORWARD=1 is set (off by default:
 *   slower than the chained kernels on GB300).
 * Errors: those of the steps; MOE_ERR_WORKSPACE if ws_bytes is too small.
 */
MOE_API size_t moe_forward_workspace_size(const moe_dims* dims);

/*
 * moe_forward_single_launch - 1 when moe_forward (router_weights = 0: given
 *   logits, 1: router_w) or moe_forward_prenorm (prenorm = 1) with these dims
 *   runs as the single cooperative launch described at moe_forward, 0 when
 *   it chains its kernels, a negative status for invalid dims. Host only.
 */
MOE_API int moe_forward_single_launch(const moe_dims* dims, int router_weights,
                                      int prenorm);
MOE_API int moe_forward(const moe_dims* dims, const uint16_t* x,
                        const float* router_logits, const uint16_t* router_w,
                        const uint8_t* w_gu, const float* s_gu,
                        const uint8_t* w_d, const float* s_d,
                        const uint16_t* shared_gate_w, uint16_t* out,
                        int32_t* topk_ids_out, float* topk_w_out, void* ws,
                        size_t ws_bytes, moe_stream_t stream);

/*
 * moe_forward_intermediates - where a forward keeps its intermediates inside
 * workspace `ws` (for inspection and tests; no kernel runs, nothing is
 * copied). After a moe_forward (or variant) with the same dims and ws has
 * completed on its stream, the fields below point into ws and hold that
 * forward's values; R = T k routed rows, rows = R + T (shared) or R, sorted
 * rows in expert order (the layout of moe_permute), G = E + shared:
 *   topk_ids, topk_w [T, k]: the routing (valid only when the forward was not
 *     given topk_ids_out / topk_w_out, which then received it);
 *   expert_offsets [G + 1], sorted_to_flat [R], flat_to_sorted [R];
 *   xq [rows, D] e4m3 and sx [rows] fp32: the token's codes and scale at each
 *     of its sorted rows; gate [T] fp32: the shared expert's gate;
 *   h [rows, I] fp32: SwiGLU output of the gate/up GEMM; hq [rows, I] e4m3 and
 *     sh [rows] fp32: its per-row requantisation;
 *   y: the down GEMM's output, fp32 [rows, D] when y_fp16 == 0, else fp16 codes
 *     [rows, D] with y = y_row_scale[r] * code.
 * Returns MOE_OK, MOE_ERR_INVALID_ARG (bad dims or NULL out) or
 * MOE_ERR_WORKSPACE (ws NULL, misaligned or smaller than the forward needs).
 * No counterpart in the pages (inspection support).
 */
typedef struct moe_intermediates {
  int32_t* topk_ids;
  float* topk_w;
  int32_t* expert_offsets;
  int32_t* sorted_to_flat;
  int32_t* flat_to_sorted;
  uint8_t* xq;
  float* sx;
  float* gate;
  float* h;
  uint8_t* hq;
  float* sh;
  void* y;
  float* y_row_scale;
  int32_t y_fp16;
} moe_intermediates;

MOE_API int moe_forward_intermediates(const moe_dims* dims, void* ws, size_t ws_bytes,
                                      moe_intermediates* out);

/*
 * moe_forward_workspace_layout - the sub-buffers of the forward workspace for
 * `dims`: writes the byte offset and size of each (up to max_entries; host
 * arrays, both non-NULL, or both NULL to only count) and returns their
 * number (a negative status for bad dims). Every sub-buffer is followed by
 * at least 256 bytes that no kernel writes (a guard band: a test fills the
 * workspace with a pattern and checks the bands after a forward).
 * No counterpart in the pages (inspection support).
 */
MOE_API int moe_forward_workspace_layout(const moe_dims* dims, size_t* offsets,
                                         size_t* sizes, int max_entries);

/*
 * moe_forward_profiled - moe_forward with timing marks: identical work and
 *   arguments, plus `events`, an array of MOE_FORWARD_EVENTS cudaEvent_t
 *   created by the caller, recorded on `stream` at the step boundaries:
 *   [0] start, [1] after the router projection (no-op without router_w),
 *   [2] after routing, [3] after the permutation, [4] after the x
 *   quantisation, [5] after the gate/up GEMM, [6] after the requantisation,
 *   [7] after the down GEMM, [8] after the combine.
 * Errors: those of moe_forward; MOE_ERR_INVALID_ARG if n_events differs.
 */
#define MOE_FORWARD_EVENTS 9
MOE_API int moe_forward_profiled(const moe_dims* dims, const uint16_t* x,
                                 const float* router_logits,
                                 const uint16_t* router_w, const uint8_t* w_gu,
                                 const float* s_gu, const uint8_t* w_d,
                                 const float* s_d,
                                 const uint16_t* shared_gate_w, uint16_t* out,
                                 int32_t* topk_ids_out, float* topk_w_out,
                                 void* ws, size_t ws_bytes, void* const* events,
                                 int n_events, moe_stream_t stream);

/*
 * moe_device_status - synchronise `stream`, then read and clear the device
 * error word that kernels set when a bounded wait expires or a grouped GEMM
 * finds group offsets that describe more rows than `a_rows`. Returns MOE_OK;
 * MOE_ERR_INVALID_ARG when only bad-data bits (16, 128) are set; MOE_ERR_TIMEOUT when
 * a wait expired; MOE_ERR_CUDA if the stream reported a CUDA error.
 * `detail` (nullable) receives the raw error bits:
 *   1 TMA producer wait, 2 MMA issuer wait, 4 epilogue wait, 8 drain wait,
 *   16 tile map larger than the launch (offsets past a_rows; those tiles are
 *   not computed), 32 tile scheduler wait, 64 moe_debug_expire_wait,
 *   128 (checked build libmoe_ptpc_check.so only) an expert id, row map entry
 *   or destination row out of range: the access was skipped. MOE_ERR_INVALID_ARG
 *   is returned when only bits 16 and 128 are set.
 */
MOE_API int moe_device_status(moe_stream_t stream, unsigned* detail);

/*
 * moe_workspace_status - the same for the kernels of the forwards that ran
 * on workspace `ws` (moe_forward, moe_forward_profiled, moe_forward_prenorm,
 * or moe_debug_expire_wait given that workspace): enqueue on `stream` a
 * one-thread kernel that takes the workspace's error word and clears it in
 * one atomic exchange, copy the bits back and synchronise `stream`. Call it
 * on the stream the forward ran on (or after synchronising with it). A
 * forward clears the word when it starts, so the bits are those of the most
 * recent forward on `ws` (and of debug waits queued after it); a second call
 * without a new forward returns MOE_OK. Status values and `detail` bits as
 * for moe_device_status. Errors: MOE_ERR_INVALID_ARG (ws NULL, misaligned or
 * ws_bytes < 256), MOE_ERR_CUDA.
 */
MOE_API int moe_workspace_status(void* ws, size_t ws_bytes, moe_stream_t stream,
                                 unsigned* detail);

/*
 * moe_forward_prenorm - moe_forward fed from the residual stream: the
 * quantisation step becomes moe_add_rmsnorm_quant(x, pre->residual,
 * pre->gamma, pre->eps), which also writes pre->residual_out, and the shared
 * gate takes the normalised activations. The routing comes from
 * router_logits (required; there is no router_w form, the router would read
 * the normalised activations). Other arguments as for moe_forward. `events`
 * is NULL, or MOE_FORWARD_EVENTS events as for moe_forward_profiled (then
 * the steps are serialised and marked).
 */
typedef struct moe_prenorm {
  const uint16_t* residual;   /* [T, D] bf16 */
  const uint16_t* gamma;      /* [D] bf16 */
  float eps;                  /* >= 0 */
  uint16_t* residual_out;     /* [T, D] bf16, may alias residual */
} moe_prenorm;

MOE_API int moe_forward_prenorm(const moe_dims* dims, const moe_prenorm* pre,
                                const uint16_t* x, const float* router_logits,
                                const uint8_t* w_gu, const float* s_gu,
                                const uint8_t* w_d, const float* s_d,
                                const uint16_t* shared_gate_w, uint16_t* out,
                                int32_t* topk_ids_out, float* topk_w_out, void* ws,
                                size_t ws_bytes, void* const* events, int n_events,
                                moe_stream_t stream);

/*
 * moe_debug_expire_wait - failure-detection check without a GPU fault: one
 * thread waits on an mbarrier that nothing arrives on, bounded exactly like
 * the waits of the layer's kernels but with a limit of `limit_us`
 * microseconds (1 .. 1,000,000), and records the expiry in an error word:
 * that of the forward workspace `ws` (ws_bytes >= 256) when ws is non-NULL,
 * else the device error word of the standalone steps. The kernel then ends
 * normally and the context stays usable: the next moe_workspace_status(ws)
 * (or moe_device_status()) returns MOE_ERR_TIMEOUT with `detail` bit 64 and
 * clears it. No counterpart in the pages (test support). Returns MOE_OK,
 * MOE_ERR_INVALID_ARG (limit out of range, bad workspace; nothing launched)
 * or MOE_ERR_CUDA.
 */
MOE_API int moe_debug_expire_wait(int limit_us, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/*
 * FP8 with per-K-block scales: the alternatives to PTPC that the pages
 * compare it with ("Ultimate Latency Optimization of Qwen3 and Qwen3-VL on
 * AMD MI300X Series", section 2.1.1: BlockScale's fixed K block against
 * PTPC's none, PTPC 15-30% faster on ROCm; the MI355X DeepSeek-R1 page,
 * "MoRI Quantized All-to-All": one fp32 scale per 128 elements; "Optimizing
 * Qwen 3.5 397B MoE on Ironwood TPU7x", GMM V2 paragraph: activations
 * quantised per 512-wide subchannel). Every block uses the PTPC quantiser:
 * s = fp32(max(amax_block, 1e-12) / 448), q = e4m3_rne_sat(fp32(v / s)).
 */
typedef enum moe_scale_kind {
  MOE_SCALE_PTPC = 0,      /* a_scale [a_rows], w_scale [groups, N]            */
  MOE_SCALE_SUB512 = 1,    /* a_scale [a_rows, K/512], w_scale [groups, N]     */
  MOE_SCALE_BLOCK128 = 2   /* a_scale [a_rows, K/128],
                              w_scale [groups, N/128, K/128]                   */
} moe_scale_kind;

/*
 * moe_quant_blocks - per-row FP8 quantisation of in [rows, K] bf16 in
 * 1 x block pieces along K (block 128 or 512): q [rows, K] e4m3 (written),
 * scales [rows, K/block] fp32 (written), scales[r, b] for
 * in[r, b*block .. (b+1)*block). Device pointers; in 8-byte aligned (block
 * 128) or 16-byte aligned (512), q 4- or 16-byte aligned.
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned pointers, rows < 0, block
 *         not 128 or 512, K not a positive multiple of block).
 */
MOE_API int moe_quant_blocks(const uint16_t* in_bf16, int64_t rows, int K, int block,
                             uint8_t* q, float* scales, moe_stream_t stream);

/*
 * moe_quant_weight_blocks - BlockScale-128 weight quantisation of
 * w [rows, K] fp32 (rows = groups * N, both multiples of 128) in 128 x 128
 * blocks: q [rows, K] e4m3 (written), scales [rows/128, K/128] fp32
 * (written). Device pointers, 16-byte aligned.
 * Errors: MOE_ERR_INVALID_ARG (null or misaligned pointers, sizes not
 *         positive multiples of 128), MOE_ERR_UNSUPPORTED (rows > 128 * 65535).
 */
MOE_API int moe_quant_weight_blocks(const float* w, int64_t rows, int K, uint8_t* q,
                                    float* scales, moe_stream_t stream);

/*
 * moe_grouped_gemm_scaled - FP8 grouped GEMM with the scale granularity
 * `scale_kind` (moe_scale_kind), all three on one tcgen05 engine: the tensor
 * cores accumulate each scale group of K (all of K for PTPC, 512 for
 * SUB512, 128 for BLOCK128) in TMEM, and the epilogue scales and sums the
 * groups in fp32:
 *   PTPC:     y[r, n] = w_scale[g, n] * fp32(P[r, n] * a_scale[r])
 *   SUB512:   y[r, n] = w_scale[g, n] * sum_j fp32(P_j[r, n] * a_scale[r, j])
 *   BLOCK128: y[r, n] = sum_b fp32(P_b[r, n] * fp32(a_scale[r, b] *
 *                                                   w_scale[g, n/128, b]))
 * (P_j: the FP8 dot product over scale group j, fp32 tensor-core
 * accumulation.) Group g owns rows [group_offsets[g], group_offsets[g+1]) of
 * A [a_rows, K] e4m3; W [groups, N, K] e4m3; out [a_rows, N] fp32 (rows
 * outside every group not written). group_offsets is a DEVICE array of
 * groups + 1 non-decreasing entries <= a_rows. A, W, out 16-byte aligned.
 * Errors: MOE_ERR_INVALID_ARG (unknown kind, null or misaligned pointers,
 *         negative sizes), MOE_ERR_UNSUPPORTED (N or K not multiples of 128,
 *         K not a multiple of 512 for SUB512, K > 39168 for BLOCK128 (a
 *         tile's scales are staged in shared memory), groups > 1025),
 *         MOE_ERR_CUDA.
 */
MOE_API int moe_grouped_gemm_scaled(int scale_kind, const uint8_t* A, const float* a_scale,
                                    int64_t a_rows, const uint8_t* W, const float* w_scale,
                                    const int32_t* group_offsets, int groups, int N, int K,
                                    float* out, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PTPC_H */
