// Warp top-k selection shared by the routing kernels (route.cu on given
// logits, router_gemm.cu on the fused router GEMM's logits).
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", MoE paragraph: the top-k
// routed experts of a token are chosen through a softmax distribution over
// its router logits. Selection rule: larger fp32 value first, equal values
// to the lower expert index; weights are the softmax over the chosen k
// (renormalize) or over all E, evaluated at the chosen k.
#pragma once

#include "common.cuh"

namespace moe {

// An unsigned key with the order of the fp32 values (-0 and +0 equal).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One token's top k over row[0..E) by one warp: lane holds the keys of the
// experts lane + 32 i (i < NI) in registers; k rounds of a warp argmax (a
// max of the keys, then the lowest expert index holding it: larger value
// first, equal values to the lower index, the selection rule above),
// then the softmax weights.
template <int NI>
__device__ __forceinline__ void select_warp(const float* row, int E, int k,
                                            int renormalize, int64_t tok,
                                            int32_t* __restrict__ ids,
                                            float* __restrict__ weights,
                                            float* __restrict__ logits_out) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    const float v = e < E ? row[e] : 0.f;
    key[i] = e < E ? order_key(v) : 0u;   // 0: below every value, never chosen
    if (logits_out != nullptr && e < E) logits_out[tok * E + e] = v;
  }
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      if (key[i] > bk) {
        bk = key[i];
        bi = lane + 32 * i;
      }
    }
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t wi = __reduce_min_sync(0xffffffffu, bk == mk ? (uint32_t)bi : 0xffffffffu);
    if ((int)(wi & 31u) == lane) {
#pragma unroll
      for (int i = 0; i < NI; ++i)
        if (i == (int)(wi >> 5)) key[i] = 0u;
    }
    if (j == lane) my_idx = (int)wi;
  }
  const float my_val = lane < k ? row[my_idx] : 0.f;
  const float top = __shfl_sync(0xffffffffu, my_val, 0);
  float den;
  if (renormalize) {
    den = warp_sum(lane < k ? expf(my_val - top) : 0.f);
  } else {
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += expf(row[e] - top);
    den = warp_sum(s);
  }
  if (lane < k) {
    ids[tok * k + lane] = my_idx;
    weights[tok * k + lane] = expf(my_val - top) / den;
  }
}

}  // namespace moe
