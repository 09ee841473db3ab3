// The whole layer in one launch for batches of a few tokens.
//
// "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series",
// section 2.1.4 (the decode MoE is bound by how fast the chosen experts'
// weights stream in) and section 2.1.5 (fusing the small per-token steps into
// their neighbours): with a handful of tokens the layer is about 140 MB of
// weight reads, and a chain of seven launches (route, permutation, quantiser,
// gate/up GEMM, requantiser, down GEMM, combine) loses most of its time to
// launch gaps and to each GEMM's ramp and drain. Here one CTA per SM
// (a cooperative launch, so all are resident) runs:
//
//   0. routing (softmax top-k, as route.cu) and the stable permutation of the
//      T*k rows, every CTA for itself (a few hundred operations);
//   1. the per-token quantisation of x (s = fp32(max(amax, 1e-12) / 448),
//      codes e4m3 RNE saturating, IEEE divisions, as quant.cu), every CTA;
//   2. gate/up: the touched experts' (expert, channel) pairs are split evenly
//      over the CTAs; each streams its weight rows into a shared-memory ring
//      (1D bulk copies, up to 32 KB) and takes the dot products with the
//      decoded x codes on CUDA cores (fp32 products of e4m3 values are exact;
//      fp32 sums), then SwiGLU, writing h in fp32;
//   -- one grid-wide barrier (a counter in the workspace, bounded spin);
//   3. the per-row requantisation of h, every CTA for itself;
//   4. down + combine: each CTA owns D / #CTAs output channels, streams those
//      rows of every touched expert's W_d (prefetched during steps 2-3: they
//      do not depend on h), forms y for its channels of every row and
//      combines each token's k rows (fp32 in slot order, the shared expert
//      last, one bf16 rounding, as combine.cu).
//
// The arithmetic of every step is that of the multi-kernel path (same
// roundings; only the order of the fp32 sums differs), and every intermediate
// the multi-kernel path leaves in the workspace (routing, permutation, x
// codes, h, h codes, y in fp32) is written to the same place.
//
// Roles: warps 0-7 compute, warp 8 (lane 0) issues the copies. Every wait is
// bounded (1 s) and reports through the error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kSfCompute = 8;                 // compute warps
constexpr int kSfThreads = 32 * (kSfCompute + 1);
constexpr int kSfSlotBytes = 32768;          // weight rows of one slot (at most)
constexpr int kSfScaleBytes = 256;           // their channel scales, behind them
constexpr int kSfSlotStride = kSfSlotBytes + kSfScaleBytes;
constexpr int kSfSlots = 4;
constexpr int kSfActBytes = 65536;            // x decoded (f32), then h codes decoded
constexpr int kSfMaxRows = kSfMaxTokens * (kMaxTopK + 1);
constexpr int kSfYBlk = 32;                   // output channels per down chunk (max)
constexpr int kSfSmem = kSfSlots * kSfSlotStride + kSfActBytes +
                        kSfMaxRows * kSfYBlk * 4 + 128;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// This CTA's arrival at the grid barrier, ordered after every write the
// CTA's compute warps made before meeting (release at GPU scope).
__device__ __forceinline__ void grid_arrive(unsigned* counter) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
}

// Four e4m3 codes (one 32-bit word) to fp32, exactly (e4m3 -> f16 -> f32).
__device__ __forceinline__ float4 decode4(uint32_t w) {
  uint32_t lo, hi;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((uint16_t)(w & 0xffffu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((uint16_t)(w >> 16)));
  const __half2 l = *reinterpret_cast<const __half2*>(&lo);
  const __half2 h = *reinterpret_cast<const __half2*>(&hi);
  return make_float4(__low2float(l), __high2float(l), __low2float(h), __high2float(h));
}

__device__ __forceinline__ float decode1(uint8_t c) {
  uint32_t hh;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"((uint16_t)c));
  return __low2float(*reinterpret_cast<const __half2*>(&hh));
}

// Dot product of a row of n e4m3 codes (shared memory) with n fp32 values
// (shared memory), by one warp: lane l takes the 4-code words l, l + 32, ...
// (consecutive lanes read consecutive words and float4s, so neither read has
// bank conflicts); fp32 fused multiply-adds of exact products, then a warp
// sum.
__device__ __forceinline__ float warp_dot(const uint8_t* codes, const float* vals, int n,
                                          int lane) {
  const uint32_t* c32 = reinterpret_cast<const uint32_t*>(codes);
  const float4* v4 = reinterpret_cast<const float4*>(vals);
  float acc0 = 0.f, acc1 = 0.f;
  const int nw = n / 4;
  int w = lane;
#pragma unroll 4
  for (; w + 32 < nw; w += 64) {
    const float4 f0 = decode4(c32[w]), f1 = decode4(c32[w + 32]);
    const float4 x0 = v4[w], x1 = v4[w + 32];
    acc0 = fmaf(f0.x, x0.x, acc0); acc0 = fmaf(f0.y, x0.y, acc0);
    acc0 = fmaf(f0.z, x0.z, acc0); acc0 = fmaf(f0.w, x0.w, acc0);
    acc1 = fmaf(f1.x, x1.x, acc1); acc1 = fmaf(f1.y, x1.y, acc1);
    acc1 = fmaf(f1.z, x1.z, acc1); acc1 = fmaf(f1.w, x1.w, acc1);
  }
  if (w < nw) {
    const float4 f0 = decode4(c32[w]);
    const float4 x0 = v4[w];
    acc0 = fmaf(f0.x, x0.x, acc0); acc0 = fmaf(f0.y, x0.y, acc0);
    acc0 = fmaf(f0.z, x0.z, acc0); acc0 = fmaf(f0.w, x0.w, acc0);
  }
  return warp_sum(acc0 + acc1);
}

struct SfArgs {
  int T, D, E, k, I, shared, renormalize;
  const __nv_bfloat16* x;
  const float* logits;
  const uint8_t* w_gu;
  const float* s_gu;
  const uint8_t* w_d;
  const float* s_d;
  const __nv_bfloat16* gate_w;
  __nv_bfloat16* out;
  int32_t* ids;
  float* tw;
  int32_t* counts;
  int32_t* offsets;
  int32_t* s2f;
  int32_t* f2s;
  uint8_t* xq;
  float* sx;
  float* gate;
  float* h;
  uint8_t* hq;
  float* sh;
  float* y;
  unsigned* grid_counter;
  unsigned* err;
};

// One group of the layer: an expert (or the shared one, index E) with its
// rows first_row .. first_row + nrows - 1 in the sorted layout.
struct SfGroup {
  int g, first_row, nrows;
};

__global__ void __launch_bounds__(kSfThreads, 1) small_forward_kernel(const SfArgs a) {
  extern __shared__ __align__(128) uint8_t sf_smem[];
  uint8_t* ring = sf_smem;
  float* act = reinterpret_cast<float*>(sf_smem + kSfSlots * kSfSlotStride);
  float* yblk = reinterpret_cast<float*>(sf_smem + kSfSlots * kSfSlotStride + kSfActBytes);
  __shared__ int32_t ids_s[kSfMaxTokens * kMaxTopK];
  __shared__ float w_s[kSfMaxTokens * kMaxTopK];
  __shared__ int32_t f2s_s[kSfMaxTokens * kMaxTopK];
  __shared__ int32_t s2f_s[kSfMaxTokens * kMaxTopK];
  __shared__ int32_t row_tok[kSfMaxRows];        // token of each sorted row
  __shared__ SfGroup grp[kSfMaxRows + 1];
  __shared__ float sx_s[kSfMaxTokens], gate_s[kSfMaxTokens], sh_s[kSfMaxRows];
  __shared__ float red[kSfThreads / 32][2];
  __shared__ int ngroups;
  __shared__ __align__(8) uint64_t bars[2 * kSfSlots + 3];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, D = a.D, E = a.E, k = a.k, I = a.I;
  const int R = T * k;
  const int rows = R + (a.shared ? T : 0);
  const bool lead = blockIdx.x == 0;   // writes the shared intermediates
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[kSfSlots + s]); };
  const uint32_t cbar = smem_u32(&bars[2 * kSfSlots]);       // compute warps met
  const uint32_t gbar = smem_u32(&bars[2 * kSfSlots + 1]);   // grid barrier passed
  const uint32_t hbar = smem_u32(&bars[2 * kSfSlots + 2]);   // h copied in

  if (tid == 0) {
    for (int s = 0; s < kSfSlots; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kSfCompute);
    }
    mbar_init(cbar, kSfCompute);
    mbar_init(gbar, 1);
    mbar_init(hbar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }

  // ---------------- 0. routing and permutation (every CTA) ----------------
  if (warp < T) {
    const float* row = a.logits + (int64_t)warp * E;
    const int npl = (E + 31) / 32;
    if (npl <= 1) select_warp<1>(row, E, k, a.renormalize, warp, ids_s, w_s, nullptr);
    else if (npl <= 2) select_warp<2>(row, E, k, a.renormalize, warp, ids_s, w_s, nullptr);
    else if (npl <= 4) select_warp<4>(row, E, k, a.renormalize, warp, ids_s, w_s, nullptr);
    else if (npl <= 8) select_warp<8>(row, E, k, a.renormalize, warp, ids_s, w_s, nullptr);
    else if (npl <= 16) select_warp<16>(row, E, k, a.renormalize, warp, ids_s, w_s, nullptr);
    else select_warp<32>(row, E, k, a.renormalize, warp, ids_s, w_s, nullptr);
  }
  __syncthreads();
  // stable counting order: flat entry i goes to the rank of (expert, i)
  for (int i = tid; i < R; i += kSfThreads) {
    const int e = ids_s[i];
    int rank = 0;
    for (int j = 0; j < R; ++j) {
      const int ej = ids_s[j];
      rank += (ej < e || (ej == e && j < i)) ? 1 : 0;
    }
    f2s_s[i] = rank;
    s2f_s[rank] = i;
    row_tok[rank] = i / k;
    if (lead) {
      a.f2s[i] = rank;
      a.s2f[rank] = i;
      a.ids[i] = e;
      a.tw[i] = w_s[i];
    }
  }
  for (int t = tid; t < (a.shared ? T : 0); t += kSfThreads) row_tok[R + t] = t;
  if (lead) {   // counts and offsets of every group (the shared one: index E)
    const int G = E + (a.shared ? 1 : 0);
    for (int e = tid; e <= G; e += kSfThreads) {
      int below = 0;
      if (e <= E) {
        for (int i = 0; i < R; ++i) below += ids_s[i] < e ? 1 : 0;
      } else {
        below = R + T;   // offsets[E + 1], shared rows included
      }
      a.offsets[e] = below;
    }
  }
  __syncthreads();
  if (lead) {
    const int G = E + (a.shared ? 1 : 0);
    for (int e = tid; e < G; e += kSfThreads) a.counts[e] = a.offsets[e + 1] - a.offsets[e];
  }
  if (tid == 0) {   // the touched groups in order, with their sorted rows
    int n = 0;
    for (int r = 0; r < R;) {
      const int e = ids_s[s2f_s[r]];
      int r1 = r + 1;
      while (r1 < R && ids_s[s2f_s[r1]] == e) ++r1;
      grp[n++] = SfGroup{e, r, r1 - r};
      r = r1;
    }
    if (a.shared) grp[n++] = SfGroup{E, R, T};
    ngroups = n;
  }

  // ---------------- 1. x -> e4m3 codes, per token (every CTA) ----------------
  for (int t = 0; t < T; ++t) {
    const __nv_bfloat16* xr = a.x + (int64_t)t * D;
    float amax = 0.f, dot = 0.f;
    for (int c = 8 * tid; c < D; c += 8 * kSfThreads) {
      const uint4 raw = *reinterpret_cast<const uint4*>(xr + c);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v0 = __low2float(b[i]), v1 = __high2float(b[i]);
        amax = fmaxf(amax, fmaxf(fabsf(v0), fabsf(v1)));
        if (a.shared) {
          dot = fmaf(v0, __bfloat162float(a.gate_w[c + 2 * i]), dot);
          dot = fmaf(v1, __bfloat162float(a.gate_w[c + 2 * i + 1]), dot);
        }
      }
    }
    amax = warp_max(amax);
    dot = warp_sum(dot);
    if (lane == 0) {
      red[warp][0] = amax;
      red[warp][1] = dot;
    }
    __syncthreads();
    if (tid == 0) {
      float m = 0.f, d = 0.f;
      for (int w = 0; w < kSfThreads / 32; ++w) {
        m = fmaxf(m, red[w][0]);
        d += red[w][1];
      }
      sx_s[t] = __fdiv_rn(fmaxf(m, 1e-12f), 448.0f);
      gate_s[t] = 1.0f / (1.0f + expf(-d));
    }
    __syncthreads();
    const float s = sx_s[t];
    float* xf = act + (int64_t)t * D;
    for (int c = 8 * tid; c < D; c += 8 * kSfThreads) {
      const uint4 raw = *reinterpret_cast<const uint4*>(xr + c);
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
      uint16_t q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        q[i] = f32x2_to_e4m3x2(__fdiv_rn(__low2float(b[i]), s),
                               __fdiv_rn(__high2float(b[i]), s));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xf[c + 2 * i] = decode1((uint8_t)(q[i] & 0xff));
        xf[c + 2 * i + 1] = decode1((uint8_t)(q[i] >> 8));
      }
      if (lead) {   // the codes of every row of token t
        const uint2 packed = make_uint2((uint32_t)q[0] | ((uint32_t)q[1] << 16),
                                        (uint32_t)q[2] | ((uint32_t)q[3] << 16));
        for (int j = 0; j < k; ++j)
          *reinterpret_cast<uint2*>(a.xq + (int64_t)f2s_s[t * k + j] * D + c) = packed;
        if (a.shared) *reinterpret_cast<uint2*>(a.xq + (int64_t)(R + t) * D + c) = packed;
      }
    }
    if (lead && tid == 0) {
      for (int j = 0; j < k; ++j) a.sx[f2s_s[t * k + j]] = s;
      if (a.shared) {
        a.sx[R + t] = s;
        a.gate[t] = gate_s[t];
      }
    }
  }
  __syncthreads();

  // ---------------- the streamed weight slots ----------------
  // gate/up: this CTA's share [p0, p1) of the (group, channel) pairs, in
  // units of up to 8 channels of one group, each as two slots (its gate
  // rows, then its up rows); down: this CTA's output channels [d0, d1) in
  // chunks of up to dmax rows, each chunk one slot per group.
  const int ng = ngroups;
  const int64_t P = (int64_t)ng * I;
  const int64_t p0 = P * blockIdx.x / gridDim.x, p1 = P * (blockIdx.x + 1) / gridDim.x;
  const int dlo = (int)((int64_t)D * blockIdx.x / gridDim.x);
  const int dhi = (int)((int64_t)D * (blockIdx.x + 1) / gridDim.x);
  const int dmax = min(kSfYBlk, kSfSlotBytes / I);
  // a slot's channel scales: the 16-byte aligned run of floats that holds
  // scale[idx .. idx + n) (it never reaches past the array, whose rows are
  // multiples of 16 bytes); returns the first float's offset in the run
  auto scale_run = [](int64_t idx, int n, int64_t& start, uint32_t& bytes) {
    start = idx & ~int64_t(3);
    const int64_t end = (idx + n + 3) & ~int64_t(3);
    bytes = (uint32_t)((end - start) * 4);
    return (int)(idx - start);
  };
  // visit(f): f(kind, group index, first row or channel, count) for every slot
  // in order; kind 0: gate rows, 1: up rows, 2: down rows
  auto visit = [&](auto&& f) {
    for (int gi = 0; gi < ng; ++gi) {
      const int64_t gb = (int64_t)gi * I;
      const int64_t lo = max(p0, gb), hi = min(p1, gb + I);
      for (int64_t c0 = lo; c0 < hi; c0 += 8) {
        const int nc = hi - c0 < 8 ? (int)(hi - c0) : 8;
        if (!f(0, gi, (int)(c0 - gb), nc)) return;
        if (!f(1, gi, (int)(c0 - gb), nc)) return;
      }
    }
    for (int d0 = dlo; d0 < dhi; d0 += dmax) {
      const int nd = min(dmax, dhi - d0);
      for (int gi = 0; gi < ng; ++gi)
        if (!f(2, gi, d0, nd)) return;
    }
  };

  if (warp == kSfCompute) {
    // ---------------- producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int last_phase[kSfSlots];
#pragma unroll
      for (int i = 0; i < kSfSlots; ++i) last_phase[i] = -1;
      uint32_t q = 0;
      visit([&](int kind, int gi, int first, int n) -> bool {
        const int s = (int)(q % kSfSlots);
        const uint32_t ph = (q / kSfSlots) & 1u;
        ++q;
        if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, &abort_flag, a.err,
                               kErrTimeoutProducer))
          return false;
        const int g = grp[gi].g;
        const uint8_t* src;
        const float* ssrc;
        uint32_t bytes, sbytes;
        int64_t sstart;
        if (kind < 2) {
          const int64_t row = (int64_t)g * 2 * I + (kind == 1 ? I : 0) + first;
          src = a.w_gu + row * D;
          bytes = (uint32_t)(n * D);
          scale_run(row, n, sstart, sbytes);
          ssrc = a.s_gu + sstart;
        } else {
          const int64_t row = (int64_t)g * D + first;
          src = a.w_d + row * I;
          bytes = (uint32_t)(n * I);
          scale_run(row, n, sstart, sbytes);
          ssrc = a.s_d + sstart;
        }
        mbar_arrive_expect_tx(full_bar(s), bytes + sbytes);
        bulk_load(smem_u32(ring + s * kSfSlotStride), src, bytes, full_bar(s), pol);
        bulk_load(smem_u32(ring + s * kSfSlotStride + kSfSlotBytes), ssrc, sbytes,
                  full_bar(s), pol);
#pragma unroll
        for (int i = 0; i < kSfSlots; ++i)
          if (i == s) last_phase[i] = (int)ph;
        return true;
      });
      // every copy has landed before the shared memory is released
#pragma unroll
      for (int i = 0; i < kSfSlots; ++i) {
        if (last_phase[i] >= 0) {
          volatile int no_abort = 0;
          mbar_wait_bounded(full_bar(i), (uint32_t)last_phase[i], &no_abort, a.err,
                            kErrTimeoutDrain);
        }
      }
    }
  } else {
    // ---------------- compute warps ----------------
    uint32_t q = 0, cph = 0;
    bool ok = true;
    float gacc[kSfMaxTokens + 1];   // gate dot products of this warp's channel
    float swg = 0.f, swu = 0.f;     // and its weight scales
    // all compute warps have reached this point (bounded)
    auto compute_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(cbar);
      const bool r = warp_wait(cbar, cph, &abort_flag, a.err, kErrTimeoutEpilogue);
      cph ^= 1u;
      return r;
    };
    bool down_started = false;
    int cur_d0 = -1, cur_nd = 0, groups_done = 0;
    // every h this CTA writes is out: meet the other CTAs (bounded), then
    // requantise every row of h (codes decoded into `act`; the lead CTA also
    // writes the codes and scales out)
    auto barrier_and_requant = [&]() -> bool {
      __threadfence();
      if (!compute_sync()) return false;
      if (warp == 0 && lane == 0) {
        grid_arrive(a.grid_counter);
        const unsigned long long t0 = global_timer_ns();
        unsigned seen = 0;
        for (uint32_t spin = 0;; ++spin) {
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                       : "=r"(seen)
                       : "l"(a.grid_counter)
                       : "memory");
          if (seen >= gridDim.x) break;
          if ((spin & 63u) == 63u && global_timer_ns() - t0 > kWaitLimitNs) {
            abort_flag = 1;
            atomicOr(a.err, kErrTimeoutSched);
            break;
          }
        }
        if (!abort_flag) {
          // every row of h into `act` with one bulk copy (written through the
          // generic proxy by every CTA, read here through the async one)
          asm volatile("fence.proxy.async.global;" ::: "memory");
          const uint32_t hbytes = (uint32_t)(rows * I * 4);
          mbar_arrive_expect_tx(hbar, hbytes);
          bulk_load(smem_u32(act), a.h, hbytes, hbar, l2_policy_evict_first());
        }
        mbar_arrive(gbar);
      }
      if (!warp_wait(gbar, 0, &abort_flag, a.err, kErrTimeoutEpilogue)) return false;
      if (abort_flag) return false;
      if (!warp_wait(hbar, 0, &abort_flag, a.err, kErrTimeoutEpilogue)) return false;
      for (int r = warp; r < rows; r += kSfCompute) {
        float* hf = act + (int64_t)r * I;
        float m = 0.f;
        for (int c = lane; c < I; c += 32) m = fmaxf(m, fabsf(hf[c]));
        m = warp_max(m);
        const float s = __fdiv_rn(fmaxf(m, 1e-12f), 448.0f);
        if (lane == 0) {
          sh_s[r] = s;
          if (lead) a.sh[r] = s;
        }
        for (int c = 2 * lane; c < I; c += 64) {
          const uint16_t q2 = f32x2_to_e4m3x2(__fdiv_rn(hf[c], s), __fdiv_rn(hf[c + 1], s));
          hf[c] = decode1((uint8_t)(q2 & 0xff));
          hf[c + 1] = decode1((uint8_t)(q2 >> 8));
          if (lead) *reinterpret_cast<uint16_t*>(a.hq + (int64_t)r * I + c) = q2;
        }
      }
      return compute_sync();
    };
    visit([&](int kind, int gi, int first, int n) -> bool {
      if (kind == 2 && !down_started) {
        down_started = true;
        if (!barrier_and_requant()) return ok = false;
      }
      const int s = (int)(q % kSfSlots);
      const uint32_t ph = (q / kSfSlots) & 1u;
      ++q;
      if (!warp_wait(full_bar(s), ph, &abort_flag, a.err, kErrTimeoutEpilogue))
        return ok = false;
      const uint8_t* slot = ring + s * kSfSlotStride;
      const float* sscale = reinterpret_cast<const float*>(slot + kSfSlotBytes);
      const SfGroup G = grp[gi];
      if (kind < 2) {
        // gate (kind 0) or up (kind 1) rows of channels first .. first + n - 1;
        // warp w takes channel first + w
        if (warp < n) {
          const uint8_t* wrow = slot + (int64_t)warp * D;
          const int c = first + warp;
          // the channel's weight scale, copied in with the slot
          {
            int64_t st;
            uint32_t sb;
            const int o = scale_run((int64_t)G.g * 2 * I + (kind == 1 ? I : 0) + first, n,
                                    st, sb);
            if (kind == 0) swg = sscale[o + warp];
            else swu = sscale[o + warp];
          }
          for (int j = 0; j < G.nrows; ++j) {
            const int r = G.first_row + j;
            const float v = warp_dot(wrow, act + (int64_t)row_tok[r] * D, D, lane);
            if (kind == 0) {
              gacc[j] = v;
            } else if (lane == 0) {
              const float sxr = sx_s[row_tok[r]];
              const float gg = gacc[j] * sxr * swg;
              const float uu = v * sxr * swu;
              a.h[(int64_t)r * I + c] = __fdividef(gg * uu, 1.0f + __expf(-gg));
            }
          }
        }
      } else {
        // down rows first .. first + n - 1 of group G; warp w takes rows w,
        // w + 8, ...; y of every row of the group for those channels
        if (first != cur_d0) {
          cur_d0 = first;
          cur_nd = n;
          groups_done = 0;
        }
        // the rows' channel scales came in with the slot
        int64_t st;
        uint32_t sb;
        const int so = scale_run((int64_t)G.g * D + first, n, st, sb);
        for (int dd = warp; dd < n; dd += kSfCompute) {
          const uint8_t* wrow = slot + (int64_t)dd * I;
          const float sd = sscale[so + dd];
          for (int j = 0; j < G.nrows; ++j) {
            const int r = G.first_row + j;
            const float v = warp_dot(wrow, act + (int64_t)r * I, I, lane);
            if (lane == 0) {
              const float yv = v * sh_s[r] * sd;
              yblk[r * kSfYBlk + dd] = yv;
              a.y[(int64_t)r * D + first + dd] = yv;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      if (kind == 2 && ++groups_done == ng) {
        // every row's y for channels cur_d0 .. + cur_nd: combine
        if (!compute_sync()) return ok = false;
        for (int e = warp * 32 + lane; e < T * cur_nd; e += kSfCompute * 32) {
          const int t = e / cur_nd, dd = e % cur_nd;
          float acc = 0.f;
          for (int j = 0; j < k; ++j)
            acc = fmaf(w_s[t * k + j], yblk[f2s_s[t * k + j] * kSfYBlk + dd], acc);
          if (a.shared) acc = fmaf(gate_s[t], yblk[(R + t) * kSfYBlk + dd], acc);
          a.out[(int64_t)t * D + cur_d0 + dd] = __float2bfloat16_rn(acc);
        }
        if (!compute_sync()) return ok = false;
      }
      return true;
    });
    (void)ok;
    if (!down_started) {
      // no output channel of this CTA needs h: count it in; the lead CTA
      // still waits and writes the h codes out
      if (lead) {
        barrier_and_requant();
      } else {
        __threadfence();
        if (compute_sync() && warp == 0 && lane == 0) grid_arrive(a.grid_counter);
      }
    }
  }
  __syncthreads();
}

}  // namespace

bool small_forward_supported(int T, int D, int E, int k, int I, int shared) {
  const int rows = T * k + (shared ? T : 0);
  return T >= 1 && T <= kSfMaxTokens && E <= 1024 && k <= kMaxTopK && D % 16 == 0 &&
         I % 16 == 0 && (int64_t)T * D * 4 <= kSfActBytes &&
         (int64_t)rows * I * 4 <= kSfActBytes && 8 * D <= kSfSlotBytes &&
         I <= kSfSlotBytes && rows <= kSfMaxRows;
}

int launch_small_forward(int T, int D, int E, int k, int I, int shared, int renormalize,
                         const uint16_t* x, const float* logits, const uint8_t* w_gu,
                         const float* s_gu, const uint8_t* w_d, const float* s_d,
                         const uint16_t* gate_w, uint16_t* out, int32_t* ids, float* tw,
                         int32_t* counts, int32_t* offsets, int32_t* s2f, int32_t* f2s,
                         uint8_t* xq, float* sx, float* gate, float* h, uint8_t* hq,
                         float* sh, float* y, unsigned* grid_counter,
                         cudaStream_t stream) {
  if (!small_forward_supported(T, D, E, k, I, shared)) return -1;
  if (cudaFuncSetAttribute(small_forward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSfSmem) != cudaSuccess)
    return -3;
  SfArgs a;
  a.T = T; a.D = D; a.E = E; a.k = k; a.I = I; a.shared = shared;
  a.renormalize = renormalize;
  a.x = reinterpret_cast<const __nv_bfloat16*>(x);
  a.logits = logits;
  a.w_gu = w_gu; a.s_gu = s_gu; a.w_d = w_d; a.s_d = s_d;
  a.gate_w = reinterpret_cast<const __nv_bfloat16*>(gate_w);
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  a.ids = ids; a.tw = tw; a.counts = counts; a.offsets = offsets;
  a.s2f = s2f; a.f2s = f2s; a.xq = xq; a.sx = sx; a.gate = gate;
  a.h = h; a.hq = hq; a.sh = sh; a.y = y;
  a.grid_counter = grid_counter;
  a.err = device_error_word();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sm_count());
  cfg.blockDim = dim3(kSfThreads);
  cfg.dynamicSmemBytes = kSfSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, small_forward_kernel, a);
  return e == cudaSuccess ? 0 : -3;
}

}  // namespace moe
