// C ABI of the PTPC-FP8 MoE layer: argument checks, workspace layout and the
// chaining of the kernels on the caller's stream. Declared in moe_ptpc.h.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "../../include/moe_ptpc.h"
#include "common.cuh"
#include "internal.h"

namespace moe {

// Set by kernels of the standalone entry points whose bounded wait ran out;
// read and cleared by moe_device_status(). moe_forward's kernels report into
// a word inside the forward's own workspace instead (moe_workspace_status).
__device__ unsigned g_error_word;
// Where moe_device_status's read-and-clear leaves the old value.
__device__ unsigned g_error_taken;

namespace {

// The error word of the launches the calling thread is making, when a
// forward has set one (ErrorWordScope).
thread_local unsigned* t_error_word = nullptr;

unsigned* symbol_address(const void* symbol) {
  void* p = nullptr;
  return cudaGetSymbolAddress(&p, symbol) == cudaSuccess ? static_cast<unsigned*>(p)
                                                         : nullptr;
}

// Per-device addresses of g_error_word (slot 0) and g_error_taken (slot 1).
unsigned* global_word(int which) {
  static std::mutex mu;
  static unsigned* addr[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev][which] == nullptr)
    addr[dev][which] = symbol_address(which == 0 ? static_cast<const void*>(&g_error_word)
                                                 : static_cast<const void*>(&g_error_taken));
  return addr[dev][which];
}

}  // namespace

unsigned* device_error_word() {
  return t_error_word != nullptr ? t_error_word : global_word(0);
}

// While alive, the kernels the calling thread launches report into `word`.
struct ErrorWordScope {
  unsigned* prev;
  explicit ErrorWordScope(unsigned* word) : prev(t_error_word) { t_error_word = word; }
  ~ErrorWordScope() { t_error_word = prev; }
  ErrorWordScope(const ErrorWordScope&) = delete;
  ErrorWordScope& operator=(const ErrorWordScope&) = delete;
};

// taken = the word's bits; the word = 0, in one atomic step, so that a bit a
// kernel sets concurrently is either taken now or left for the next read.
__global__ void take_error_word_kernel(unsigned* word, unsigned* taken) {
  *taken = atomicExch(word, 0u);
}

// One thread waits, with a bounded wait like every wait of the layer's
// kernels, on an mbarrier that nothing arrives on; the wait expires after
// `limit_ns` and records the expiry in the error word.
__global__ void expire_wait_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_barrier_init();
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(smem_u32(&bar), 0)) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, kErrDebugWait);
      return;
    }
  }
}

namespace {

inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

inline int cuda_status(cudaError_t e) {
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Byte offsets of the intermediates inside the moe_forward workspace. The
// first kForwardStatusBytes hold the forward's error word and the slot its
// read-and-clear copies from (moe_workspace_status).
constexpr size_t kForwardStatusBytes = 256;
// the single-launch forward's grid barrier counter, inside the status bytes
constexpr size_t kGridCounterOffset = 64;

// MOE_SMALL_FORWARD=1 turns on the single-launch forward for a few tokens.
// It is off by default: on GB300 at T=1 (D=4096, 512 experts, top-10 +
// shared) it took 69-79 us against 53-56 us for the chained kernels, its
// CUDA-core dot products and its 4-slot weight ring being slower than the
// tensor-core GEMMs' streaming.
int small_forward_mode() {
  static const int mode = [] {
    const char* v = std::getenv("MOE_SMALL_FORWARD");
    return (v != nullptr && v[0] == '1') ? 1 : 0;
  }();
  return mode;
}
constexpr size_t kGuardBytes = 256;

struct ForwardLayout {
  size_t status, ids, w, logits, counts, offsets, s2f, f2s, perm, xq, sx, gate, h,
      hq, sh, y, row_scale, w_bound, total;
};

// The expert output y goes through HBM in fp32 while it is small, and in the
// fp16 encoding (half the bytes, one factor per row) once its fp32 size
// reaches 32 MiB; below that the extra bound kernel costs more than it saves.
inline bool y_in_fp16(const moe_dims& d) {
  const int64_t rows = (int64_t)d.T * d.k + (d.shared ? d.T : 0);
  return rows * d.D * 4 >= (int64_t(32) << 20);
}

ForwardLayout forward_layout(const moe_dims& d) {
  const int64_t R = (int64_t)d.T * d.k;
  const int64_t rows = R + (d.shared ? d.T : 0);
  const int64_t G = (int64_t)d.E + (d.shared ? 1 : 0);
  ForwardLayout L{};
  size_t off = 0;
  // every sub-buffer is followed by at least kGuardBytes that no kernel
  // writes: a guard band, so that a test can fill the workspace with a
  // pattern and find any write past a buffer's end (compute-sanitizer is not
  // available to catch it)
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes + kGuardBytes);
    return o;
  };
  L.status = take(kForwardStatusBytes);
  L.ids = take(R * 4);
  L.w = take(R * 4);
  L.logits = take((size_t)d.T * d.E * 4);
  L.counts = take(G * 4);
  L.offsets = take((G + 1) * 4);
  L.s2f = take(R * 4);
  L.f2s = take(R * 4);
  L.perm = take(permute_ws_bytes(R, d.E));
  L.xq = take(rows * d.D);
  L.sx = take(rows * 4);
  L.gate = take((size_t)d.T * 4);
  L.h = take(rows * d.I * 4);
  L.hq = take(rows * d.I);
  L.sh = take(rows * 4);
  L.y = take(rows * d.D * 4);   // fp32, or fp16 codes in the first half
  L.row_scale = take(rows * 4);
  L.w_bound = take(G * 4);
  L.total = off;
  return L;
}

// Whether moe_forward runs the layer as one launch: at most kSfMaxTokens
// tokens, given router logits, no pre-norm, y in fp32 and a supported shape.
bool small_forward_applies(const moe_dims& d, bool router_weights, bool prenorm) {
  return small_forward_mode() != 0 && !router_weights && !prenorm && !y_in_fp16(d) &&
         small_forward_supported(d.T, d.D, d.E, d.k, d.I, d.shared);
}

int check_dims(const moe_dims* d) {
  if (d == nullptr) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->D <= 0 || d->E <= 0 || d->I <= 0 || d->k <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d->shared != 0 && d->shared != 1) return MOE_ERR_INVALID_ARG;
  if (d->k > d->E || d->k > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (d->E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (d->D % 128 != 0 || d->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)d->T * (d->k + 1) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int moe_version(void) { return 100; }

int moe_router_logits(const uint16_t* x, const uint16_t* w_r, int T, int E,
                      int D, float* logits, moe_stream_t stream) {
  if (T < 0 || E <= 0 || D <= 0 || D % 2 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_r || !logits || !aligned16(x) || !aligned16(w_r))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_router_logits(x, w_r, T, E, D, logits, stream, false));
}

int moe_route(const float* logits, int T, int E, int k, int renormalize,
              int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
  if (T < 0 || E <= 0 || k < 1 || k > E || k > kMaxTopK)
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
  return cuda_status(
      launch_route(logits, T, E, k, renormalize ? 1 : 0, topk_ids, topk_w, stream,
                   false));
}

size_t moe_permute_workspace_size(int T, int E, int k) {
  if (T < 0 || E <= 0 || k <= 0) return 0;
  return permute_ws_bytes((int64_t)T * k, E);
}

int moe_permute(const int32_t* topk_ids, int T, int E, int k,
                int32_t* expert_counts, int32_t* expert_offsets,
                int32_t* sorted_to_flat, int32_t* flat_to_sorted, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || E <= 0 || k < 1 || k > E || k > kMaxTopK)
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)T * k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (!expert_counts || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!topk_ids || !sorted_to_flat || !flat_to_sorted))
    return MOE_ERR_INVALID_ARG;
  const size_t need = permute_ws_bytes((int64_t)T * k, E);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return MOE_ERR_WORKSPACE;
  return cuda_status(launch_permute(topk_ids, (int64_t)T * k, E, expert_counts,
                                    expert_offsets, sorted_to_flat,
                                    flat_to_sorted, -1, ws, stream, false));
}

int moe_quant_ptpc(const void* in, int in_dtype, int64_t rows, int cols,
                   const int32_t* dst_rows, int copies, int64_t extra_row_base,
                   uint8_t* out_q, float* out_scale, moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || copies < 1)
    return MOE_ERR_INVALID_ARG;
  if (cols > kMaxQuantCols || copies > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (in_dtype != MOE_DTYPE_BF16 && in_dtype != MOE_DTYPE_F32)
    return MOE_ERR_INVALID_ARG;
  if (dst_rows == nullptr && copies != 1) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!in || !out_q || !out_scale || !aligned16(in) || !aligned16(out_q))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_quant(in, in_dtype, rows, cols, dst_rows, copies,
                                  extra_row_base, out_q, out_scale, nullptr,
                                  nullptr, stream, false, false));
}

int moe_shared_gate(const uint16_t* x, const uint16_t* w_g, int T, int D,
                    float* gate, moe_stream_t stream) {
  if (T < 0 || D <= 0 || D % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !w_g || !gate || !aligned16(x) || !aligned16(w_g))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_shared_gate(x, w_g, T, D, gate, stream));
}

int moe_grouped_gemm(int kind, const uint8_t* A, const float* a_scale,
                     int64_t a_rows, const uint8_t* W, const float* w_scale,
                     const int32_t* group_offsets, int groups, int N, int K,
                     void* out, int out_dtype, int rows_hint,
                     moe_stream_t stream) {
  if (kind != MOE_GEMM_GATEUP_SWIGLU && kind != MOE_GEMM_DOWN)
    return MOE_ERR_INVALID_ARG;
  if (a_rows < 0 || groups < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (out_dtype != MOE_DTYPE_F32) return MOE_ERR_UNSUPPORTED;
  if (groups > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  if (a_rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (a_rows == 0 || groups == 0) return MOE_OK;
  if (!A || !a_scale || !W || !w_scale || !group_offsets || !out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return launch_grouped_gemm(kind, A, a_scale, a_rows, W, w_scale, group_offsets,
                             groups, N, K, static_cast<float*>(out), rows_hint,
                             stream, false);
}

int moe_quant_blocks(const uint16_t* in_bf16, int64_t rows, int K, int block, uint8_t* q,
                     float* scales, moe_stream_t stream) {
  if (rows < 0 || (block != 128 && block != 512) || K <= 0 || K % block != 0)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!in_bf16 || !q || !scales) return MOE_ERR_INVALID_ARG;
  const uintptr_t ain = reinterpret_cast<uintptr_t>(in_bf16);
  const uintptr_t aq = reinterpret_cast<uintptr_t>(q);
  if (block == 128 ? (ain % 8 != 0 || aq % 4 != 0) : (ain % 16 != 0 || aq % 16 != 0))
    return MOE_ERR_INVALID_ARG;
  return launch_quant_blocks(in_bf16, rows, K, block, q, scales, stream);
}

int moe_quant_weight_blocks(const float* w, int64_t rows, int K, uint8_t* q, float* scales,
                            moe_stream_t stream) {
  if (rows < 0 || rows % 128 != 0 || K <= 0 || K % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (rows / 128 > 65535) return MOE_ERR_UNSUPPORTED;
  if (!w || !q || !scales) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(q)) return MOE_ERR_INVALID_ARG;
  return launch_quant_weight_blocks(w, rows, K, q, scales, stream);
}

int moe_grouped_gemm_scaled(int scale_kind, const uint8_t* A, const float* a_scale,
                            int64_t a_rows, const uint8_t* W, const float* w_scale,
                            const int32_t* group_offsets, int groups, int N, int K,
                            float* out, moe_stream_t stream) {
  if (scale_kind != MOE_SCALE_PTPC && scale_kind != MOE_SCALE_SUB512 &&
      scale_kind != MOE_SCALE_BLOCK128)
    return MOE_ERR_INVALID_ARG;
  if (a_rows < 0 || groups < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (scale_kind == MOE_SCALE_SUB512 && K % 512 != 0) return MOE_ERR_UNSUPPORTED;
  if (groups > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  if (a_rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (a_rows == 0 || groups == 0) return MOE_OK;
  if (!A || !a_scale || !W || !w_scale || !group_offsets || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return launch_grouped_gemm_scaled(scale_kind, A, a_scale, a_rows, W, w_scale,
                                    group_offsets, groups, N, K, out, stream);
}

int moe_scale_max(const float* scale, int groups, int N, float* bound,
                  moe_stream_t stream) {
  if (groups < 0 || N <= 0) return MOE_ERR_INVALID_ARG;
  if (groups == 0) return MOE_OK;
  if (!scale || !bound) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_scale_max(scale, groups, N, bound, stream, false));
}

int moe_grouped_gemm_down_f16(const uint8_t* A, const float* a_scale,
                              int64_t a_rows, const uint8_t* W, const float* w_scale,
                              const float* w_bound, const int32_t* group_offsets,
                              int groups, int N, int K, uint16_t* y16,
                              float* row_scale, int rows_hint, moe_stream_t stream) {
  if (a_rows < 0 || groups < 0 || N <= 0 || K <= 0) return MOE_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (groups > kMaxGroups) return MOE_ERR_UNSUPPORTED;
  if (a_rows >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (a_rows == 0 || groups == 0) return MOE_OK;
  if (!A || !a_scale || !W || !w_scale || !w_bound || !group_offsets || !y16 ||
      !row_scale)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(y16)) return MOE_ERR_INVALID_ARG;
  return launch_grouped_gemm_down_f16(A, a_scale, a_rows, W, w_scale, w_bound,
                                      group_offsets, groups, N, K, y16, row_scale,
                                      rows_hint, stream, false);
}

int moe_combine_f16(const uint16_t* y16, const float* row_scale,
                    const int32_t* flat_to_sorted, const float* topk_w, int T, int k,
                    int D, const uint16_t* y16_shared, const float* row_scale_shared,
                    const float* shared_gate, uint16_t* out, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > kMaxTopK || D <= 0 || D % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  const bool s1 = y16_shared != nullptr, s2 = row_scale_shared != nullptr,
             s3 = shared_gate != nullptr;
  if (s1 != s2 || s1 != s3) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y16 || !row_scale || !flat_to_sorted || !topk_w || !out || !aligned16(y16) ||
      !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (s1 && !aligned16(y16_shared)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_f16(y16, row_scale, flat_to_sorted, topk_w, T, k,
                                        D, y16_shared, row_scale_shared, shared_gate,
                                        out, stream, false));
}

int moe_combine(const float* y, const int32_t* flat_to_sorted,
                const float* topk_w, int T, int k, int D, const float* y_shared,
                const float* shared_gate, uint16_t* out, moe_stream_t stream) {
  if (T < 0 || k < 1 || k > kMaxTopK || D <= 0 || D % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  if ((y_shared == nullptr) != (shared_gate == nullptr)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!y || !flat_to_sorted || !topk_w || !out || !aligned16(y) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (y_shared != nullptr && !aligned16(y_shared)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(y, flat_to_sorted, topk_w, T, k, D, y_shared,
                                    shared_gate, out, stream, false));
}

size_t moe_forward_workspace_size(const moe_dims* dims) {
  if (check_dims(dims) != MOE_OK) return 0;
  return forward_layout(*dims).total;
}

int moe_forward_workspace_layout(const moe_dims* dims, size_t* offsets, size_t* sizes,
                                 int max_entries) {
  if (check_dims(dims) != MOE_OK) return MOE_ERR_INVALID_ARG;
  const ForwardLayout L = forward_layout(*dims);
  const moe_dims& d = *dims;
  const int64_t R = (int64_t)d.T * d.k;
  const int64_t rows = R + (d.shared ? d.T : 0);
  const int64_t G = (int64_t)d.E + (d.shared ? 1 : 0);
  const size_t off[] = {L.status, L.ids, L.w, L.logits, L.counts, L.offsets, L.s2f,
                        L.f2s, L.perm, L.xq, L.sx, L.gate, L.h, L.hq, L.sh, L.y,
                        L.row_scale, L.w_bound};
  const size_t size[] = {kForwardStatusBytes, (size_t)R * 4, (size_t)R * 4,
                         (size_t)d.T * d.E * 4, (size_t)G * 4, (size_t)(G + 1) * 4,
                         (size_t)R * 4, (size_t)R * 4, permute_ws_bytes(R, d.E),
                         (size_t)rows * d.D, (size_t)rows * 4, (size_t)d.T * 4,
                         (size_t)rows * d.I * 4, (size_t)rows * d.I, (size_t)rows * 4,
                         (size_t)rows * d.D * 4, (size_t)rows * 4, (size_t)G * 4};
  const int n = (int)(sizeof(off) / sizeof(off[0]));
  if (offsets != nullptr && sizes != nullptr)
    for (int i = 0; i < n && i < max_entries; ++i) {
      offsets[i] = off[i];
      sizes[i] = size[i];
    }
  return n;
}

int moe_forward_intermediates(const moe_dims* dims, void* ws, size_t ws_bytes,
                              moe_intermediates* out) {
  if (check_dims(dims) != MOE_OK || out == nullptr) return MOE_ERR_INVALID_ARG;
  const ForwardLayout L = forward_layout(*dims);
  if (ws == nullptr || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  uint8_t* b = static_cast<uint8_t*>(ws);
  out->topk_ids = reinterpret_cast<int32_t*>(b + L.ids);
  out->topk_w = reinterpret_cast<float*>(b + L.w);
  out->expert_offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  out->sorted_to_flat = reinterpret_cast<int32_t*>(b + L.s2f);
  out->flat_to_sorted = reinterpret_cast<int32_t*>(b + L.f2s);
  out->xq = b + L.xq;
  out->sx = reinterpret_cast<float*>(b + L.sx);
  out->gate = reinterpret_cast<float*>(b + L.gate);
  out->h = reinterpret_cast<float*>(b + L.h);
  out->hq = b + L.hq;
  out->sh = reinterpret_cast<float*>(b + L.sh);
  out->y = b + L.y;
  out->y_row_scale = reinterpret_cast<float*>(b + L.row_scale);
  out->y_fp16 = y_in_fp16(*dims) ? 1 : 0;
  return MOE_OK;
}

}  // extern "C"

namespace {

int forward_impl(const moe_dims* dims, const moe_prenorm* pre, const uint16_t* x,
                 const float* router_logits, const uint16_t* router_w,
                 const uint8_t* w_gu, const float* s_gu, const uint8_t* w_d,
                 const float* s_d, const uint16_t* shared_gate_w, uint16_t* out,
                 int32_t* topk_ids_out, float* topk_w_out, void* ws,
                 size_t ws_bytes, cudaEvent_t const* ev, cudaStream_t stream) {
  auto mark = [&](int i) {
    if (ev != nullptr) cudaEventRecord(ev[i], stream);
  };
  int st = check_dims(dims);
  if (st != MOE_OK) return st;
  const moe_dims d = *dims;
  if (d.T == 0) {   // empty batch: nothing to read or write but the error word
    if (ws != nullptr && ws_bytes >= kForwardStatusBytes && aligned16(ws))
      return cuda_status(cudaMemsetAsync(ws, 0, sizeof(unsigned), stream));
    return MOE_OK;
  }
  if ((router_logits == nullptr) == (router_w == nullptr)) return MOE_ERR_INVALID_ARG;
  if (d.shared && shared_gate_w == nullptr) return MOE_ERR_INVALID_ARG;
  if (!d.shared && shared_gate_w != nullptr) return MOE_ERR_INVALID_ARG;
  if (!x || !w_gu || !s_gu || !w_d || !s_d || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_gu) || !aligned16(w_d) || !aligned16(out))
    return MOE_ERR_INVALID_ARG;
  if (router_w != nullptr && !aligned16(router_w)) return MOE_ERR_INVALID_ARG;
  if (shared_gate_w != nullptr && !aligned16(shared_gate_w)) return MOE_ERR_INVALID_ARG;
  if (pre != nullptr) {   // the layer input comes from the residual stream
    if (router_w != nullptr) return MOE_ERR_UNSUPPORTED;
    if (!pre->residual || !pre->gamma || !pre->residual_out ||
        !aligned16(pre->residual) || !aligned16(pre->gamma) ||
        !aligned16(pre->residual_out) || !(pre->eps >= 0.0f))
      return MOE_ERR_INVALID_ARG;
  }
  const ForwardLayout L = forward_layout(d);
  if (ws == nullptr || ws_bytes < L.total || !aligned16(ws)) return MOE_ERR_WORKSPACE;

  uint8_t* base = static_cast<uint8_t*>(ws);
  auto at = [&](size_t off) { return static_cast<void*>(base + off); };
  // This forward's kernels report expired waits into the workspace's own
  // error word, cleared first (in stream order), so that forwards on other
  // streams and workspaces never see each other's errors.
  auto* err_word = static_cast<unsigned*>(at(L.status));
  if (cudaMemsetAsync(err_word, 0, sizeof(unsigned), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  ErrorWordScope err_scope(err_word);
  const int64_t R = (int64_t)d.T * d.k;
  const int64_t rows = R + (d.shared ? d.T : 0);
  const int G = d.E + (d.shared ? 1 : 0);
  int32_t* ids = topk_ids_out ? topk_ids_out : static_cast<int32_t*>(at(L.ids));
  float* tw = topk_w_out ? topk_w_out : static_cast<float*>(at(L.w));
  auto* counts = static_cast<int32_t*>(at(L.counts));
  auto* offsets = static_cast<int32_t*>(at(L.offsets));
  auto* s2f = static_cast<int32_t*>(at(L.s2f));
  auto* f2s = static_cast<int32_t*>(at(L.f2s));
  auto* xq = static_cast<uint8_t*>(at(L.xq));
  auto* sx = static_cast<float*>(at(L.sx));
  auto* gate = static_cast<float*>(at(L.gate));
  auto* h = static_cast<float*>(at(L.h));
  auto* hq = static_cast<uint8_t*>(at(L.hq));
  auto* sh = static_cast<float*>(at(L.sh));
  auto* y = static_cast<float*>(at(L.y));
  auto* y16 = static_cast<uint16_t*>(at(L.y));
  auto* row_scale = static_cast<float*>(at(L.row_scale));
  auto* w_bound = static_cast<float*>(at(L.w_bound));
  const bool f16 = y_in_fp16(d);

  // A batch of a few tokens on given logits: the whole layer in one
  // cooperative launch (small_forward.cu), the same intermediates left in
  // the workspace. Its grid barrier counts in the status region.
  if (small_forward_applies(d, router_w != nullptr, pre != nullptr) && aligned16(s_gu) &&
      aligned16(s_d)) {
    auto* grid_counter = static_cast<unsigned*>(at(L.status + kGridCounterOffset));
    if (cudaMemsetAsync(grid_counter, 0, sizeof(unsigned), stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    for (int i = 0; i <= 4; ++i) mark(i);
    const int r = launch_small_forward(
        d.T, d.D, d.E, d.k, d.I, d.shared, d.renormalize ? 1 : 0, x, router_logits, w_gu,
        s_gu, w_d, s_d, shared_gate_w, out, ids, tw, counts, offsets, s2f, f2s, xq, sx,
        gate, h, hq, sh, y, grid_counter, stream);
    if (r != 0) return MOE_ERR_CUDA;
    for (int i = 5; i <= 8; ++i) mark(i);
    return MOE_OK;
  }

  // Kernels after the first overlap their launch with the previous kernel's
  // tail (programmatic dependent launch); each orders itself with pdl_wait().
  // Event marks between the steps serialise them instead.
  const bool pdl = ev == nullptr;
  mark(0);
  bool first = true;
  if (f16) {   // the down weights' scale bound of every group (weights only)
    st = cuda_status(launch_scale_max(s_d, G, d.D, w_bound, stream, false));
    if (st != MOE_OK) return st;
    first = false;
  }
  const float* logits = router_logits;
  // router weights: the tensor-core router with the top-k in its epilogue
  // where it applies and the projection has at least 2^20 multiply-adds;
  // below that (launch latency dominates) and for unsupported shapes, the
  // exactly rounded router GEMM and the route kernel
  const bool fused_router =
      router_w != nullptr && router_topk_supported(d.E, d.k, d.D) &&
      (int64_t)d.T * d.E * d.D >= (int64_t(1) << 20);
  if (fused_router) {
    st = launch_router_topk(x, router_w, d.T, d.D, d.E, d.k, d.renormalize ? 1 : 0,
                            ids, tw, nullptr, stream, pdl && !first);
    if (st != MOE_OK) return st;
    first = false;
  } else if (router_w != nullptr) {
    auto* lg = static_cast<float*>(at(L.logits));
    st = cuda_status(
        launch_router_logits(x, router_w, d.T, d.E, d.D, lg, stream, pdl && !first));
    if (st != MOE_OK) return st;
    logits = lg;
    first = false;
  }
  mark(1);
  if (!fused_router) {
    st = cuda_status(launch_route(logits, d.T, d.E, d.k, d.renormalize ? 1 : 0, ids,
                                  tw, stream, pdl && !first));
    if (st != MOE_OK) return st;
  }
  mark(2);
  st = cuda_status(launch_permute(ids, R, d.E, counts, offsets, s2f, f2s,
                                  d.shared ? d.T : -1, at(L.perm), stream, pdl));
  if (st != MOE_OK) return st;
  mark(3);
  // x -> FP8 codes written straight into each token's k expert rows (and its
  // shared-expert row R + t), plus the shared-expert gate. (Writing each
  // token's codes once and gathering them in the gate/up GEMM's producers
  // with TMA tile::gather4 was measured 2.4x slower in that GEMM: four rows
  // per copy instruction instead of 32 or 64.)
  if (pre != nullptr)   // r = x + residual, RMSNorm, then the same quantiser
    st = cuda_status(launch_add_rmsnorm_quant(
        x, pre->residual, pre->gamma, pre->eps, d.T, d.D, pre->residual_out, f2s,
        d.k, d.shared ? R : -1, xq, sx, d.shared ? shared_gate_w : nullptr,
        d.shared ? gate : nullptr, stream, pdl, rows));
  else
    st = cuda_status(launch_quant(x, MOE_DTYPE_BF16, d.T, d.D, f2s, d.k,
                                  d.shared ? R : -1, xq, sx,
                                  d.shared ? shared_gate_w : nullptr,
                                  d.shared ? gate : nullptr, stream, pdl, false, rows));
  if (st != MOE_OK) return st;
  mark(4);
  const int hint = (int)std::max<int64_t>(1, R / d.E);
  st = launch_grouped_gemm(MOE_GEMM_GATEUP_SWIGLU, xq, sx, rows, w_gu, s_gu,
                           offsets, G, d.I, d.D, h, hint, stream, pdl);
  if (st != MOE_OK) return st;
  mark(5);
  st = cuda_status(launch_quant(h, MOE_DTYPE_F32, rows, d.I, nullptr, 1, -1, hq,
                                sh, nullptr, nullptr, stream, pdl,
                                /*release_early=*/true, rows));
  if (st != MOE_OK) return st;
  mark(6);
  if (f16)
    st = launch_grouped_gemm_down_f16(hq, sh, rows, w_d, s_d, w_bound, offsets, G,
                                      d.D, d.I, y16, row_scale, hint, stream, pdl);
  else
    st = launch_grouped_gemm(MOE_GEMM_DOWN, hq, sh, rows, w_d, s_d, offsets, G,
                             d.D, d.I, y, hint, stream, pdl);
  if (st != MOE_OK) return st;
  mark(7);
  if (f16)
    st = cuda_status(launch_combine_f16(
        y16, row_scale, f2s, tw, d.T, d.k, d.D, d.shared ? y16 + R * d.D : nullptr,
        d.shared ? row_scale + R : nullptr, d.shared ? gate : nullptr, out, stream,
        pdl));
  else
    st = cuda_status(launch_combine(y, f2s, tw, d.T, d.k, d.D,
                                    d.shared ? y + R * d.D : nullptr,
                                    d.shared ? gate : nullptr, out, stream, pdl));
  if (st != MOE_OK) return st;
  mark(8);
  return MOE_OK;
}

}  // namespace

namespace {

// Read and clear an error word on `stream` (after everything queued before),
// then map its bits to a status.
int take_status(unsigned* word, unsigned* taken, moe_stream_t stream, unsigned* detail) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  take_error_word_kernel<<<1, 1, 0, s>>>(word, taken);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  unsigned bits = 0;
  if (cudaMemcpyAsync(&bits, taken, sizeof(bits), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (detail) *detail = bits;
  if (bits == 0) return MOE_OK;
  // only bad data (group offsets past a_rows; in the checked build, an index
  // out of range) and no expired wait
  return (bits & ~(moe::kErrBadIndex | moe::kErrCheck)) == 0 ? MOE_ERR_INVALID_ARG
                                                              : MOE_ERR_TIMEOUT;
}

bool forward_status_ok(const void* ws, size_t ws_bytes) {
  return ws != nullptr && ws_bytes >= kForwardStatusBytes && aligned16(ws);
}

}  // namespace

extern "C" {

int moe_forward(const moe_dims* dims, const uint16_t* x,
                const float* router_logits, const uint16_t* router_w,
                const uint8_t* w_gu, const float* s_gu, const uint8_t* w_d,
                const float* s_d, const uint16_t* shared_gate_w, uint16_t* out,
                int32_t* topk_ids_out, float* topk_w_out, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
  return forward_impl(dims, nullptr, x, router_logits, router_w, w_gu, s_gu, w_d,
                      s_d, shared_gate_w, out, topk_ids_out, topk_w_out, ws, ws_bytes,
                      nullptr, stream);
}

int moe_forward_prenorm(const moe_dims* dims, const moe_prenorm* pre,
                        const uint16_t* x, const float* router_logits,
                        const uint8_t* w_gu, const float* s_gu, const uint8_t* w_d,
                        const float* s_d, const uint16_t* shared_gate_w,
                        uint16_t* out, int32_t* topk_ids_out, float* topk_w_out,
                        void* ws, size_t ws_bytes, void* const* events, int n_events,
                        moe_stream_t stream) {
  if (pre == nullptr || router_logits == nullptr) return MOE_ERR_INVALID_ARG;
  if (events != nullptr) {
    if (n_events != MOE_FORWARD_EVENTS) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i)
      if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
  }
  return forward_impl(dims, pre, x, router_logits, nullptr, w_gu, s_gu, w_d, s_d,
                      shared_gate_w, out, topk_ids_out, topk_w_out, ws, ws_bytes,
                      reinterpret_cast<cudaEvent_t const*>(events), stream);
}

int moe_router_topk(const uint16_t* x, const uint16_t* w_r, int T, int D, int E,
                    int k, int renormalize, int32_t* topk_ids, float* topk_w,
                    float* logits_out, moe_stream_t stream) {
  if (T < 0 || D <= 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (!router_topk_supported(E, k, D)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!x || !w_r || !topk_ids || !topk_w || !aligned16(x) || !aligned16(w_r))
    return MOE_ERR_INVALID_ARG;
  return launch_router_topk(x, w_r, T, D, E, k, renormalize ? 1 : 0, topk_ids, topk_w,
                            logits_out, stream, false);
}

int moe_add_rmsnorm_quant(const uint16_t* x, const uint16_t* residual,
                          const uint16_t* gamma, float eps, int64_t rows, int cols,
                          uint16_t* residual_out, const int32_t* dst_rows, int copies,
                          int64_t extra_row_base, uint8_t* out_q, float* out_scale,
                          const uint16_t* gate_w, float* gate_out,
                          moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || copies < 1 || !(eps >= 0.0f))
    return MOE_ERR_INVALID_ARG;
  if (cols > kMaxQuantCols || copies > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (dst_rows == nullptr && copies != 1) return MOE_ERR_INVALID_ARG;
  if ((gate_w == nullptr) != (gate_out == nullptr)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!x || !residual || !gamma || !residual_out || !out_q || !out_scale)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(gamma) ||
      !aligned16(residual_out) || !aligned16(out_q) ||
      (gate_w != nullptr && !aligned16(gate_w)))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_add_rmsnorm_quant(
      x, residual, gamma, eps, rows, cols, residual_out, dst_rows, copies,
      extra_row_base, out_q, out_scale, gate_w, gate_out, stream, false));
}

int moe_forward_profiled(const moe_dims* dims, const uint16_t* x,
                         const float* router_logits, const uint16_t* router_w,
                         const uint8_t* w_gu, const float* s_gu,
                         const uint8_t* w_d, const float* s_d,
                         const uint16_t* shared_gate_w, uint16_t* out,
                         int32_t* topk_ids_out, float* topk_w_out, void* ws,
                         size_t ws_bytes, void* const* events, int n_events,
                         moe_stream_t stream) {
  if (events == nullptr || n_events != MOE_FORWARD_EVENTS) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i)
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
  return forward_impl(dims, nullptr, x, router_logits, router_w, w_gu, s_gu, w_d,
                      s_d, shared_gate_w, out, topk_ids_out, topk_w_out, ws, ws_bytes,
                      reinterpret_cast<cudaEvent_t const*>(events), stream);
}


int moe_debug_expire_wait(int limit_us, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
  if (ws != nullptr && !forward_status_ok(ws, ws_bytes)) return MOE_ERR_INVALID_ARG;
  unsigned* err = ws != nullptr ? static_cast<unsigned*>(ws) : moe::device_error_word();
  if (err == nullptr) return MOE_ERR_CUDA;
  moe::expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      1000ull * (unsigned long long)limit_us, err);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_device_status(moe_stream_t stream, unsigned* detail) {
  if (detail) *detail = 0;
  unsigned* word = global_word(0);
  unsigned* taken = global_word(1);
  if (word == nullptr || taken == nullptr) return MOE_ERR_CUDA;
  return take_status(word, taken, stream, detail);
}

int moe_forward_single_launch(const moe_dims* dims, int router_weights, int prenorm) {
  const int st = check_dims(dims);
  if (st != MOE_OK) return st;
  return dims->T > 0 && small_forward_applies(*dims, router_weights != 0, prenorm != 0)
             ? 1
             : 0;
}

int moe_workspace_status(void* ws, size_t ws_bytes, moe_stream_t stream,
                         unsigned* detail) {
  if (detail) *detail = 0;
  if (!forward_status_ok(ws, ws_bytes)) return MOE_ERR_INVALID_ARG;
  auto* w = static_cast<unsigned*>(ws);
  return take_status(w, w + 1, stream, detail);
}

}  // extern "C"
