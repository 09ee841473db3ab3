// Unpermute and top-k-weighted combine back to bf16.
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", SparseCore unpermute
// paragraph: the expert outputs are gathered back per token by the routing
// map and reduced locally, without materialising padded intermediates.
//
//   out[t] = bf16_rne( sum_{j<k} w[t, j] * y[flat_to_sorted[t k + j]]
//                      + gate[t] * y_shared[t] )
// summed in fp32, slot order j = 0..k-1, shared term last.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kVec = 8;        // elements per thread (2 x float4 in, 16 B out)
constexpr int kThreads = 128;  // a block covers 1024 columns of one token

__global__ void __launch_bounds__(kThreads) combine_kernel(
    const float* __restrict__ y, const int32_t* __restrict__ f2s,
    const float* __restrict__ topk_w, int k, int D,
    const float* __restrict__ y_shared, const float* __restrict__ gate,
    __nv_bfloat16* __restrict__ out, int64_t nrows, unsigned* __restrict__ err) {
  const int t = blockIdx.x;
  __shared__ int32_t rows[kMaxTopK];
  __shared__ float wts[kMaxTopK];
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x < k) {
    const int32_t r = f2s[(int64_t)t * k + threadIdx.x];
    const bool ok = MOE_CHECKED(r >= 0 && r < nrows, err);
    rows[threadIdx.x] = ok ? r : 0;
    wts[threadIdx.x] = ok ? topk_w[(int64_t)t * k + threadIdx.x] : 0.f;
  }
  __syncthreads();
  const float g = y_shared != nullptr ? gate[t] : 0.f;
  const int c = (blockIdx.y * kThreads + threadIdx.x) * kVec;
  if (c < D) {
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const float* src = y + (int64_t)rows[j] * D + c;
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 b = *reinterpret_cast<const float4*>(src + 4);
      const float w = wts[j];
      acc[0] = fmaf(w, a.x, acc[0]); acc[1] = fmaf(w, a.y, acc[1]);
      acc[2] = fmaf(w, a.z, acc[2]); acc[3] = fmaf(w, a.w, acc[3]);
      acc[4] = fmaf(w, b.x, acc[4]); acc[5] = fmaf(w, b.y, acc[5]);
      acc[6] = fmaf(w, b.z, acc[6]); acc[7] = fmaf(w, b.w, acc[7]);
    }
    if (y_shared != nullptr) {
      const float* src = y_shared + (int64_t)t * D + c;
      const float4 a = *reinterpret_cast<const float4*>(src);
      const float4 b = *reinterpret_cast<const float4*>(src + 4);
      acc[0] = fmaf(g, a.x, acc[0]); acc[1] = fmaf(g, a.y, acc[1]);
      acc[2] = fmaf(g, a.z, acc[2]); acc[3] = fmaf(g, a.w, acc[3]);
      acc[4] = fmaf(g, b.x, acc[4]); acc[5] = fmaf(g, b.y, acc[5]);
      acc[6] = fmaf(g, b.z, acc[6]); acc[7] = fmaf(g, b.w, acc[7]);
    }
    uint4 packed;
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4*>(out + (int64_t)t * D + c) = packed;
  }
}

// The same reduction over the down projection's fp16 encoding: the row
// factor folds into the slot weight, c_j = w[t, j] * row_scale[r_j], and
// out = bf16_rne( sum_j c_j * y16[r_j] + (gate[t] * row_scale_shared[t]) *
// y16_shared[t] ), in fp32 and slot order like combine_kernel. A thread
// covers VEC columns (VEC / 8 16-byte loads per slot): 16 where D allows, so
// that each block's dependent prologue (routing map, then row factors) is
// paid once per 32 bytes of every slot row instead of once per 16.
template <int VEC>
__global__ void __launch_bounds__(kThreads) combine_f16_kernel(
    const __half* __restrict__ y16, const float* __restrict__ row_scale,
    const int32_t* __restrict__ f2s, const float* __restrict__ topk_w, int k, int D,
    const __half* __restrict__ y16_shared, const float* __restrict__ row_scale_shared,
    const float* __restrict__ gate, __nv_bfloat16* __restrict__ out, int64_t nrows,
    unsigned* __restrict__ err) {
  const int t = blockIdx.x;
  __shared__ int32_t rows[kMaxTopK];
  __shared__ float coef[kMaxTopK];
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x < k) {
    const int32_t r = f2s[(int64_t)t * k + threadIdx.x];
    const bool ok = MOE_CHECKED(r >= 0 && r < nrows, err);
    rows[threadIdx.x] = ok ? r : 0;
    coef[threadIdx.x] = ok ? topk_w[(int64_t)t * k + threadIdx.x] * row_scale[r] : 0.f;
  }
  __syncthreads();
  const int c = (blockIdx.y * kThreads + threadIdx.x) * VEC;
  if (c >= D) return;
  constexpr int kLd = VEC / 8;
  float acc[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) acc[i] = 0.f;
  auto add = [&](const __half* src, float w) {
    uint4 raw[kLd];
#pragma unroll
    for (int l = 0; l < kLd; ++l) raw[l] = reinterpret_cast<const uint4*>(src)[l];
#pragma unroll
    for (int l = 0; l < kLd; ++l) {
      const __half2* h = reinterpret_cast<const __half2*>(&raw[l]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        acc[8 * l + 2 * i] = fmaf(w, f.x, acc[8 * l + 2 * i]);
        acc[8 * l + 2 * i + 1] = fmaf(w, f.y, acc[8 * l + 2 * i + 1]);
      }
    }
  };
  for (int j = 0; j < k; ++j) add(y16 + (int64_t)rows[j] * D + c, coef[j]);
  if (y16_shared != nullptr)
    add(y16_shared + (int64_t)t * D + c, gate[t] * row_scale_shared[t]);
#pragma unroll
  for (int l = 0; l < kLd; ++l) {
    uint4 packed;
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&packed);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      p[i] = __floats2bfloat162_rn(acc[8 * l + 2 * i], acc[8 * l + 2 * i + 1]);
    *reinterpret_cast<uint4*>(out + (int64_t)t * D + c + 8 * l) = packed;
  }
}

}  // namespace

cudaError_t launch_combine_f16(const uint16_t* y16, const float* row_scale,
                               const int32_t* f2s, const float* topk_w, int T,
                               int k, int D, const uint16_t* y16_shared,
                               const float* row_scale_shared,
                               const float* shared_gate, uint16_t* out,
                               cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  auto go = [&](auto kern, int vec) {
    const dim3 grid((unsigned)T, (unsigned)((D / vec + kThreads - 1) / kThreads));
    return launch_kernel(pdl, grid, dim3(kThreads), 0, stream, kern,
                         reinterpret_cast<const __half*>(y16), row_scale, f2s, topk_w,
                         k, D, reinterpret_cast<const __half*>(y16_shared),
                         row_scale_shared, shared_gate,
                         reinterpret_cast<__nv_bfloat16*>(out), (int64_t)T * k,
                         device_error_word());
  };
  if (D % 16 == 0) return go(combine_f16_kernel<16>, 16);
  return go(combine_f16_kernel<8>, 8);
}

cudaError_t launch_combine(const float* y, const int32_t* f2s,
                           const float* topk_w, int T, int k, int D,
                           const float* y_shared, const float* shared_gate,
                           uint16_t* out, cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((unsigned)T, (unsigned)((D / kVec + kThreads - 1) / kThreads));
  return launch_kernel(pdl, grid, dim3(kThreads), 0, stream, combine_kernel, y,
                       f2s, topk_w, k, D, y_shared, shared_gate,
                       reinterpret_cast<__nv_bfloat16*>(out), (int64_t)T * k,
                       device_error_word());
}

}  // namespace moe
