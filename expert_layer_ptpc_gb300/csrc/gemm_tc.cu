// PTPC FP8 grouped GEMMs on the fifth-generation tensor cores (tcgen05).
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", GMM V2 paragraph: one
// grouped GEMM over all experts, each expert a dynamically bounded slice of
// rows with no padding, gate and up projections packed in one tile through two
// operand reads with SwiGLU fused into the epilogue. "Ultimate Latency
// Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series", section 2.1.1:
// with per-token and per-channel scales the dequantisation is a rank-1 scaling
// of the FP8 dot products, applied once in the epilogue (no K blocks); section
// 2.1.4: fine-grained scheduling of work tiles over the compute units.
//
// Orientation ("weights as the MMA's M side"): a work tile is 128 output
// channels of one expert times BN of its token rows. A = 128 weight rows
// (K-major), B = BN activation rows (K-major); the accumulator in TMEM is
// [128 lanes = channels] x [BN columns = tokens]. The same engine serves
// decode (BN = 16: the weights stream from HBM once, the MMA is cheap) and
// prefill (BN up to 256: each weight tile is reused across many tokens).
// For gate/up, two accumulators (gate, up) share one B tile, so a thread
// holds gate and up of the same channel and token and applies SwiGLU alone.
//
// CTA = 6 warps, persistent over a static tile sequence:
//   warp 0      TMA producer (one lane): weight and activation tiles into a
//               STAGES-deep ring of shared-memory stages (128-byte swizzle)
//   warp 1      TMEM allocator and MMA issuer (one lane): tcgen05.mma
//               kind::f8f6f4, M=128, N=BN, K=32 per instruction, into one of
//               two accumulator buffers
//   warps 2-5   epilogue: tcgen05.ld of its 32 TMEM lanes, PTPC dequant,
//               SwiGLU, fp32 stores (coalesced: a warp writes 32 channels)
// Every wait is bounded (common.cuh): a wait that runs out raises the device
// error word, the CTA's roles stop, in-flight copies and MMAs are drained and
// the TMEM is freed before the kernel returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;   // output channels per tile (MMA M)
constexpr int kBK = 128;   // K bytes per stage = one 128-byte swizzle row
constexpr int kStageBudget = 200 * 1024;

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int BN, bool GATEUP>
struct Cfg {
  static constexpr int kNumA = GATEUP ? 2 : 1;
  static constexpr int kATile = kBM * kBK;
  static constexpr int kBTile = BN * kBK;
  static constexpr int kStage = kNumA * kATile + kBTile;
  static constexpr int kStages = (kStageBudget / kStage) > 10 ? 10 : (kStageBudget / kStage);
  static constexpr int kAccCols = kNumA * BN;               // one buffer
  static constexpr int kTmemCols = pow2_at_least(2 * kAccCols);
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kSmemBytes =
      1024 + kStages * kStage + kNumBars * 8 + 16 + 4 * (kMaxGroups + 1) + 64;
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kStages >= 2, "pipeline depth");
};

struct TileInfo {
  int group, ctile, row0, row_end;
};

__device__ __forceinline__ TileInfo decode_tile(int tile, const int* prefix,
                                                int groups, const int32_t* offsets,
                                                int bn) {
  int lo = 0, hi = groups - 1;   // largest g with prefix[g] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  // skip empty groups that share the same prefix value
  const int g = lo;
  const int start = offsets[g], end = offsets[g + 1];
  const int tt = (end - start + bn - 1) / bn;
  const int local = tile - prefix[g];
  TileInfo t;
  t.group = g;
  t.ctile = local / tt;
  t.row0 = start + (local % tt) * bn;
  t.row_end = end;
  return t;
}

// Warp-uniform bounded wait (all lanes return the same answer).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          unsigned* err, unsigned code) {
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t spin = 0;; ++spin) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((spin & 63u) == 63u) {
      int bail = 0;
      if (lane_id() == 0) {
        if (*abort_flag) {
          bail = 1;
        } else if (global_timer_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1;
          atomicOr(err, code);
          bail = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, bail, 0)) return false;
    }
  }
}

template <int BN, bool GATEUP>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap tm_w,
    const __grid_constant__ CUtensorMap tm_a, const float* __restrict__ a_scale,
    const float* __restrict__ w_scale, const int32_t* __restrict__ offsets,
    int groups, int N, int K, float* __restrict__ out,
    unsigned* __restrict__ err) {
  using C = Cfg<BN, GATEUP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* prefix = reinterpret_cast<int*>(tmem_holder + 4);   // groups + 1
  __shared__ int warp_tot[kThreads / 32 + 1];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_ctiles = N / kBM;
  const int kblocks = K / kBK;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::kStages + s); };
  auto accf_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + b); };
  auto acce_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * C::kStages + 4);
  auto stage_a = [&](int s, int which) {
    return smem_u32(smem + s * C::kStage + which * C::kATile);
  };
  auto stage_b = [&](int s) {
    return smem_u32(smem + s * C::kStage + C::kNumA * C::kATile);
  };

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_a);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);

  // tile prefix: prefix[g] = sum_{g' < g} ceil(rows_g' / BN) * n_ctiles
  {
    const int per = (groups + kThreads - 1) / kThreads;
    const int g0 = threadIdx.x * per;
    int local = 0;
    for (int g = g0; g < g0 + per && g < groups; ++g)
      local += ((offsets[g + 1] - offsets[g] + BN - 1) / BN) * n_ctiles;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int g = g0; g < g0 + per && g < groups; ++g) {
      prefix[g] = run;
      run += ((offsets[g + 1] - offsets[g] + BN - 1) / BN) * n_ctiles;
    }
    if (threadIdx.x == kThreads - 1) prefix[groups] = base + incl;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const int total_tiles = prefix[groups];

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_a = l2_policy_evict_last();
      int last_phase[C::kStages];
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) last_phase[s] = -1;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      // The weights and the tile map (offsets come from the permutation, two
      // launches back) do not depend on the previous kernel: stream the first
      // stages' weight tiles before waiting for it, then add the activations.
      const int first = blockIdx.x;
      int npre = 0;
      TileInfo t0{};
      int w0 = 0;
      if (first < total_tiles) {
        t0 = decode_tile(first, prefix, groups, offsets, BN);
        w0 = GATEUP ? t0.group * 2 * N + t0.ctile * kBM : t0.group * N + t0.ctile * kBM;
        npre = kblocks < C::kStages ? kblocks : C::kStages;
        for (int kb = 0; kb < npre; ++kb) {   // fresh ring: stage kb, phase 0
          mbar_arrive_expect_tx(full_bar(kb), C::kStage);
          tma_load_2d(stage_a(kb, 0), &tm_w, kb * kBK, w0, full_bar(kb), pol_w);
          if (GATEUP)
            tma_load_2d(stage_a(kb, 1), &tm_w, kb * kBK, w0 + N, full_bar(kb), pol_w);
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      for (int kb = 0; kb < npre; ++kb) {
        tma_load_2d(stage_b(kb), &tm_a, kb * kBK, t0.row0, full_bar(kb), pol_a);
#pragma unroll
        for (int i = 0; i < C::kStages; ++i)
          if (i == kb) last_phase[i] = 0;
      }
      s = npre % C::kStages;
      ph = npre == C::kStages ? 1u : 0u;
      for (int tile = first; ok && tile < total_tiles; tile += gridDim.x) {
        const TileInfo ti = tile == first ? t0 : decode_tile(tile, prefix, groups, offsets, BN);
        const int wrow0 = GATEUP ? ti.group * 2 * N + ti.ctile * kBM
                                 : ti.group * N + ti.ctile * kBM;
        const int wrow1 = wrow0 + N;   // up projection rows (gate/up only)
        for (int kb = tile == first ? npre : 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1, abort_flag, err,
                                 kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), C::kStage);
          tma_load_2d(stage_a(s, 0), &tm_w, kb * kBK, wrow0, full_bar(s), pol_w);
          if (GATEUP)
            tma_load_2d(stage_a(s, 1), &tm_w, kb * kBK, wrow1, full_bar(s), pol_w);
          tma_load_2d(stage_b(s), &tm_a, kb * kBK, ti.row0, full_bar(s), pol_a);
#pragma unroll
          for (int i = 0; i < C::kStages; ++i)
            if (i == s) last_phase[i] = (int)ph;
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
      }
      // drain: every issued copy has landed before shared memory is released
#pragma unroll
      for (int i = 0; i < C::kStages; ++i) {
        if (last_phase[i] >= 0) {
          volatile int no_abort = 0;
          mbar_wait_bounded(full_bar(i), (uint32_t)last_phase[i], &no_abort, err,
                            kErrTimeoutDrain);
        }
      }
    } else {
      pdl_wait();
      pdl_launch_dependents();
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kBM, BN);
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total_tiles;
           tile += gridDim.x, ++it) {
        const int ab = it & 1;
        const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(acce_bar(ab), acc_ph ^ 1, abort_flag, err,
                               kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(ab * C::kAccCols);
        const uint32_t d1 = d0 + BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(full_bar(s), ph, abort_flag, err,
                                 kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a0 = stage_a(s, 0), b = stage_b(s);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk) {
            const uint32_t acc = (kb | kk) != 0;
            const uint64_t bdesc = smem_desc_k_sw128(b + kk * 32);
            mma_f8f6f4(d0, smem_desc_k_sw128(a0 + kk * 32), bdesc, idesc, acc);
            if (GATEUP) {
              const uint32_t a1 = stage_a(s, 1);
              mma_f8f6f4(d1, smem_desc_k_sw128(a1 + kk * 32), bdesc, idesc, acc);
            }
          }
          mma_commit(empty_bar(s));   // stage free once these MMAs complete
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) mma_commit(accf_bar(ab));   // accumulator ready
      }
      // drain: all MMAs complete before TMEM is released
      mma_commit(drain_bar);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain_bar, 0, &no_abort, err, kErrTimeoutDrain);
    }
  } else {
    // ---------------- epilogue ----------------
    pdl_wait();
    pdl_launch_dependents();
    const int q = warp & 3;               // TMEM lane quarter of this warp
    const int m = q * 32 + lane;          // channel within the tile
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      const int ab = it & 1;
      const uint32_t acc_ph = (uint32_t)(it >> 1) & 1u;
      if (!warp_wait(accf_bar(ab), acc_ph, abort_flag, err, kErrTimeoutEpilogue))
        break;
      tc_fence_after_sync();
      const TileInfo ti = decode_tile(tile, prefix, groups, offsets, BN);
      const int ch = ti.ctile * kBM + m;
      const int nvalid = min(BN, ti.row_end - ti.row0);
      const uint32_t taddr =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * C::kAccCols);
      if (GATEUP) {
        const float swg = w_scale[(int64_t)ti.group * 2 * N + ch];
        const float swu = w_scale[(int64_t)ti.group * 2 * N + N + ch];
        for (int n0 = 0; n0 < nvalid; n0 += 16) {
          float ag[16], au[16];
          tmem_ld_x16(taddr + n0, ag);
          tmem_ld_x16(taddr + BN + n0, au);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (n0 + j < nvalid) {
              const int row = ti.row0 + n0 + j;
              const float sx = a_scale[row];
              const float g = ag[j] * sx * swg;
              const float u = au[j] * sx * swu;
              const float h = g / (1.0f + expf(-g)) * u;
              out[(int64_t)row * N + ch] = h;
            }
          }
        }
      } else {
        const float sw = w_scale[(int64_t)ti.group * N + ch];
        for (int n0 = 0; n0 < nvalid; n0 += 16) {
          float acc[16];
          tmem_ld_x16(taddr + n0, acc);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (n0 + j < nvalid) {
              const int row = ti.row0 + n0 + j;
              out[(int64_t)row * N + ch] = acc[j] * a_scale[row] * sw;
            }
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(acce_bar(ab));
    }
  }

  // ---------------- tear-down ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows, K] uint8 matrix, box = 128 bytes of K x box_rows rows,
// 128-byte swizzle; rows past the end read as zero.
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int K,
               int box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

template <int BN, bool GATEUP>
int run(const uint8_t* A, const float* a_scale, int64_t a_rows, const uint8_t* W,
        const float* w_scale, const int32_t* offsets, int groups, int N, int K,
        float* out, cudaStream_t stream, bool pdl) {
  using C = Cfg<BN, GATEUP>;
  CUtensorMap tm_w, tm_a;
  const int64_t w_rows = (int64_t)groups * (GATEUP ? 2 : 1) * N;
  if (!make_tmap(&tm_w, W, w_rows, K, kBM)) return -3;
  if (!make_tmap(&tm_a, A, a_rows, K, BN)) return -3;
  auto kern = grouped_gemm_kernel<BN, GATEUP>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return -3;
  const int64_t upper = ((a_rows + BN - 1) / BN + groups) * (int64_t)(N / kBM);
  const int grid = (int)std::min<int64_t>(upper, sm_count());
  if (grid <= 0) return 0;
  const cudaError_t e = launch_kernel(
      pdl, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, kern, tm_w, tm_a,
      a_scale, w_scale, offsets, groups, N, K, out, device_error_word());
  return e == cudaSuccess ? 0 : -3;
}

}  // namespace

int launch_grouped_gemm(int kind, const uint8_t* A, const float* a_scale,
                        int64_t a_rows, const uint8_t* W, const float* w_scale,
                        const int32_t* offsets, int groups, int N, int K,
                        float* out, int rows_hint, cudaStream_t stream,
                        bool pdl) {
  if (a_rows == 0 || groups == 0) return 0;
  const int64_t avg = rows_hint > 0 ? rows_hint : std::max<int64_t>(1, a_rows / groups);
  if (kind == 0) {
    if (avg <= 16) return run<16, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
    if (avg <= 32) return run<32, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
    if (avg <= 64) return run<64, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
    return run<128, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  }
  if (avg <= 16) return run<16, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  if (avg <= 32) return run<32, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  if (avg <= 64) return run<64, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  if (avg <= 128) return run<128, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  return run<256, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
}

}  // namespace moe
