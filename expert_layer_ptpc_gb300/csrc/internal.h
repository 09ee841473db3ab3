// Internal launchers behind the C ABI. Each validates nothing (api.cu does)
// and enqueues its kernels on `stream`.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Launch `kernel`; with `pdl` the launch may overlap the tail of the previous
// kernel in the stream (programmatic dependent launch), and the kernel
// orders itself with pdl_wait().
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, void (*kernel)(KArgs...),
                          Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxGroups = kMaxExperts + 1;

// Address of the device error word of the current device.
unsigned* device_error_word();

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_r, int T,
                                 int E, int D, float* logits,
                                 cudaStream_t stream, bool pdl);

cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int renormalize, int32_t* ids, float* w,
                         cudaStream_t stream, bool pdl);

// Scratch bytes of the permutation for R = T * k flat entries.
size_t permute_ws_bytes(int64_t R, int E);

// Histogram, scan and stable scatter. `extra_group_rows` >= 0 appends one more
// group (index E) of that many rows after the routed ones: counts[E] and
// offsets[E + 1] are written too (the shared expert's rows R .. R + T - 1).
cudaError_t launch_permute(const int32_t* ids, int64_t R, int E,
                           int32_t* counts, int32_t* offsets, int32_t* s2f,
                           int32_t* f2s, int extra_group_rows, void* ws,
                           cudaStream_t stream, bool pdl);

// Per-row e4m3 quantisation with scatter; `gate_w` non-null also computes
// gate_out[r] = sigmoid(in[r] . gate_w) (bf16 input only). `release_early`
// lets the next kernel launch before this one's dependency wait (see
// quant.cu for when that is safe). `out_rows`: rows of out_q / out_scale,
// which the checked build holds destinations to (-1: unknown).
cudaError_t launch_quant(const void* in, int in_dtype, int64_t rows, int cols,
                         const int32_t* dst_rows, int copies,
                         int64_t extra_row_base, uint8_t* out_q,
                         float* out_scale, const uint16_t* gate_w,
                         float* gate_out, cudaStream_t stream, bool pdl,
                         bool release_early, int64_t out_rows = -1);

// Add + RMSNorm + per-token quantisation (see quant.cu); same destinations
// and limits as launch_quant.
cudaError_t launch_add_rmsnorm_quant(const uint16_t* x, const uint16_t* res,
                                     const uint16_t* gamma, float eps, int64_t rows,
                                     int cols, uint16_t* res_out,
                                     const int32_t* dst_rows, int copies,
                                     int64_t extra_row_base, uint8_t* out_q,
                                     float* out_scale, const uint16_t* gate_w,
                                     float* gate_out, cudaStream_t stream, bool pdl,
                                     int64_t out_rows = -1);

// Router projection (tcgen05, bf16) with the top-k selection and softmax in
// its epilogue (router_gemm.cu). Returns a moe_status.
bool router_topk_supported(int E, int k, int D);
int launch_router_topk(const uint16_t* x, const uint16_t* w_r, int T, int D, int E,
                       int k, int renormalize, int32_t* ids, float* weights,
                       float* logits_out, cudaStream_t stream, bool pdl);

// FP8 grouped GEMM with PTPC (0), 512-subchannel (1) or BlockScale-128 (2)
// scales, and the block quantisers (gemm_scaled.cu). Return a moe_status.
int launch_grouped_gemm_scaled(int mode, const uint8_t* A, const float* a_scale,
                               int64_t a_rows, const uint8_t* W, const float* w_scale,
                               const int32_t* offsets, int groups, int N, int K,
                               float* out, cudaStream_t stream);
int launch_quant_blocks(const uint16_t* in, int64_t rows, int K, int block, uint8_t* q,
                        float* scales, cudaStream_t stream);
int launch_quant_weight_blocks(const float* w, int64_t rows, int K, uint8_t* q,
                               float* scales, cudaStream_t stream);

// Largest row length launch_quant handles.
constexpr int kMaxQuantCols = 32768;

cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* w_g, int T,
                               int D, float* gate, cudaStream_t stream);

// Returns a moe_status.
int launch_grouped_gemm(int kind, const uint8_t* A, const float* a_scale,
                        int64_t a_rows, const uint8_t* W, const float* w_scale,
                        const int32_t* offsets, int groups, int N, int K,
                        float* out, int rows_hint, cudaStream_t stream,
                        bool pdl);

// The CTA-pair (cta_group::2) grouped GEMM for wide token tiles (bn 128 or
// 256; gate/up also 192 and 512); needs N divisible by 128 (gate/up) or 256
// (down). Returns a status.
bool grouped_gemm_pair_supported(int kind, int N);
int launch_grouped_gemm_pair(int kind, const uint8_t* A, const float* a_scale,
                             int64_t a_rows, const uint8_t* W,
                             const float* w_scale, const int32_t* offsets,
                             int groups, int N, int K, float* out, int bn,
                             cudaStream_t stream, bool pdl);

cudaError_t launch_combine(const float* y, const int32_t* f2s,
                           const float* topk_w, int T, int k, int D,
                           const float* y_shared, const float* shared_gate,
                           uint16_t* out, cudaStream_t stream, bool pdl);

// The down projection with y written as fp16 codes plus one fp32 factor per
// row (single-CTA kernel). Returns a moe_status.
int launch_grouped_gemm_down_f16(const uint8_t* A, const float* a_scale,
                                 int64_t a_rows, const uint8_t* W,
                                 const float* w_scale, const float* w_bound,
                                 const int32_t* offsets, int groups, int N, int K,
                                 uint16_t* y16, float* row_scale, int rows_hint,
                                 cudaStream_t stream, bool pdl);

// The same on the CTA pair (N a multiple of 256, bn 128 or 256).
int launch_grouped_gemm_pair_down_f16(const uint8_t* A, const float* a_scale,
                                      int64_t a_rows, const uint8_t* W,
                                      const float* w_scale, const float* w_bound,
                                      const int32_t* offsets, int groups, int N,
                                      int K, uint16_t* y16, float* row_scale, int bn,
                                      cudaStream_t stream, bool pdl);

// bound[g] = max_n scale[g, n] over a [groups, N] fp32 array.
cudaError_t launch_scale_max(const float* scale, int groups, int N, float* bound,
                             cudaStream_t stream, bool pdl);

// combine over fp16 codes: y[r] = row_scale[r] * y16[r].
cudaError_t launch_combine_f16(const uint16_t* y16, const float* row_scale,
                               const int32_t* f2s, const float* topk_w, int T,
                               int k, int D, const uint16_t* y16_shared,
                               const float* row_scale_shared,
                               const float* shared_gate, uint16_t* out,
                               cudaStream_t stream, bool pdl);

// The whole layer in one cooperative launch for batches of at most
// kSfMaxTokens tokens on given router logits (small_forward.cu): routing,
// permutation, x codes, gate/up + SwiGLU, one grid barrier, h codes, down +
// combine, with every intermediate left where the multi-kernel path leaves
// it. `grid_counter` must be zero. Returns a moe_status-like code (0 ok,
// -1 unsupported shape, -3 launch failure).
constexpr int kSfMaxTokens = 4;
bool small_forward_supported(int T, int D, int E, int k, int I, int shared);
int launch_small_forward(int T, int D, int E, int k, int I, int shared, int renormalize,
                         const uint16_t* x, const float* logits, const uint8_t* w_gu,
                         const float* s_gu, const uint8_t* w_d, const float* s_d,
                         const uint16_t* gate_w, uint16_t* out, int32_t* ids, float* tw,
                         int32_t* counts, int32_t* offsets, int32_t* s2f, int32_t* f2s,
                         uint8_t* xq, float* sx, float* gate, float* h, uint8_t* hq,
                         float* sh, float* y, unsigned* grid_counter,
                         cudaStream_t stream);

}  // namespace moe
