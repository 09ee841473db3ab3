// Router projection and softmax top-k routing.
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", MoE paragraph: a router
// gate projects each token and the top-k routed experts are chosen through a
// softmax distribution; its Numerical Verification Layer paragraph: gating is
// held to an fp32 reference, so the selection here is an exact comparison of
// fp32 logits (ties to the lower expert index).
#include "common.cuh"
#include "internal.h"

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
// Top-k: one warp per token. Lane l holds logits l, l+32, ... (NPL of them) in
// registers. Each of k rounds takes every lane's best untaken entry and
// reduces (value, index) over the warp: larger value wins, equal values go to
// the lower index. Lane j keeps the j-th winner, then the warp forms the
// softmax weights.
// ---------------------------------------------------------------------------
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(
    const float* __restrict__ logits, int T, int E, int k, int renormalize,
    int32_t* __restrict__ ids, float* __restrict__ weights) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const int lane = (int)lane_id();
  const float* row = logits + (int64_t)t * E;
  float v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? row[e] : -INFINITY;
  }
  uint32_t taken = 0;
  float my_val = -INFINITY;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    // this lane's best untaken entry (scan in increasing index order, strict
    // comparison keeps the lowest index among equal values)
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      const bool ok = e < E && !((taken >> i) & 1u);
      if (ok && (v[i] > bv || bi == 0x7fffffff)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == lane) {
      my_val = bv;
      my_idx = bi;
    }
  }
  // weights
  const float top = __shfl_sync(0xffffffffu, my_val, 0);
  float denom;
  if (renormalize) {
    const float p = lane < k ? expf(my_val - top) : 0.f;
    denom = warp_sum(p);
  } else {
    // softmax over all E: the maximum of all logits is the top-1 logit
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) s += expf(v[i] - top);
    }
    denom = warp_sum(s);
  }
  if (lane < k) {
    ids[(int64_t)t * k + lane] = my_idx;
    weights[(int64_t)t * k + lane] = expf(my_val - top) / denom;
  }
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
