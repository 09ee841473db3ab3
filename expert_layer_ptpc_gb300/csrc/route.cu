// Router projection and softmax top-k routing.
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", MoE paragraph: a router
// gate projects each token and the top-k routed experts are chosen through a
// softmax distribution; its Numerical Verification Layer paragraph: gating is
// held to an fp32 reference, so the selection here is an exact comparison of
// fp32 logits (ties to the lower expert index).
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// logits[t, e] = x[t] . w_r[e]: one warp per (t, e), fp64 accumulation of the
// exact bf16 x bf16 products, one rounding to fp32.
// ---------------------------------------------------------------------------
__global__ void router_logits_kernel(const __nv_bfloat16* __restrict__ x,
                                     const __nv_bfloat16* __restrict__ w, int T,
                                     int E, int D, float* __restrict__ logits) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t pair = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (pair >= (int64_t)T * E) return;
  const int t = (int)(pair / E), e = (int)(pair % E);
  const __nv_bfloat16* xr = x + (int64_t)t * D;
  const __nv_bfloat16* wr = w + (int64_t)e * D;
  double acc = 0.0;
  for (int d = lane_id() * 2; d < D; d += 64) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(xr + d);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(wr + d);
    acc += (double)__low2float(a) * (double)__low2float(b);
    acc += (double)__high2float(a) * (double)__high2float(b);
  }
  acc = warp_sum_f64(acc);
  if (lane_id() == 0) logits[pair] = (float)acc;
}

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* w_r, int T,
                                 int E, int D, float* logits,
                                 cudaStream_t stream, bool pdl) {
  const int64_t pairs = (int64_t)T * E;
  if (pairs == 0) return cudaSuccess;
  const int warps = 8;
  const int64_t blocks = (pairs + warps - 1) / warps;
  return launch_kernel(pdl, dim3((unsigned)blocks), dim3(warps * 32), 0, stream,
                       router_logits_kernel,
                       reinterpret_cast<const __nv_bfloat16*>(x),
                       reinterpret_cast<const __nv_bfloat16*>(w_r), T, E, D,
                       logits);
}

// ---------------------------------------------------------------------------
// Top-k: one warp per token, the warp selection of topk.cuh on the token's
// row of logits (held as order keys in registers: k rounds of a max and a
// min reduction over the warp; the chosen values and the softmax sum read
// the row again, from L1).
// ---------------------------------------------------------------------------
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renormalize,
    int32_t* __restrict__ ids, float* __restrict__ weights) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;   // whole warps
  select_warp<NPL>(logits + (int64_t)t * E, E, k, renormalize, t, ids, weights,
                   nullptr);
}

cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int renormalize, int32_t* ids, float* w,
                         cudaStream_t stream, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int warps = 8;
  const dim3 grid((unsigned)((T + warps - 1) / warps)), block(warps * 32);
  const int npl = (E + 31) / 32;
  auto go = [&](auto kern) {
    return launch_kernel(pdl, grid, block, 0, stream, kern, logits, T, E, k,
                         renormalize, ids, w);
  };
  if (npl <= 1) return go(route_kernel<1>);
  if (npl <= 2) return go(route_kernel<2>);
  if (npl <= 4) return go(route_kernel<4>);
  if (npl <= 8) return go(route_kernel<8>);
  if (npl <= 16) return go(route_kernel<16>);
  return go(route_kernel<32>);
}

}  // namespace moe
