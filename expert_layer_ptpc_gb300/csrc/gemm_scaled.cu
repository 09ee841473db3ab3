// FP8 grouped GEMM with a choice of scale granularity, and the block
// quantisers that feed it: PTPC (one scale per token and per output
// channel), 512-subchannel (activation scales per 512-wide K group) and
// BlockScale-128 (per-128 fp32 scales on both operands).
//
// "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series",
// section 2.1.1: BlockScale ties the scales to a fixed K block that the GEMM
// tile must respect, and PTPC, which has none, ran 15-30% faster on ROCm. The
// MI355X DeepSeek-R1 page (SGLang / AMD), "MoRI Quantized All-to-All": FP8
// blockwise means one fp32 scale per 128 elements. "Optimizing Qwen 3.5 397B
// MoE on Ironwood TPU7x", GMM V2 paragraph: FP8 activations quantised per
// 512-wide subchannel.
//
// One engine runs all three, so that the comparison isolates the scale
// granularity. The tensor cores accumulate a group of K blocks (all of K for
// PTPC, 4 blocks of 128 for 512-subchannel, 1 for BlockScale-128) into one of
// four TMEM buffers; the epilogue warps read each finished group, multiply it
// by its scales (staged in shared memory once per tile) and add it into fp32
// registers while the MMAs fill the next buffers:
//   PTPC:      y[t, n] = sw[n] * fp32(P[t, n] * sa[t])
//   sub-512:   y[t, n] = sw[n] * sum_g fp32(P_g[t, n] * sa[t, g])
//   block-128: y[t, n] = sum_b fp32(P_b[t, n] * fp32(sa[t, b] * sw[n/128, b]))
// (each sum an fp32 fma chain in group order; P the tensor cores' fp32
// accumulation of the exact e4m3 products of its blocks).
//
// Tile: 128 output channels (MMA M) x 128 tokens (MMA N) of one expert, K
// blocks of 128 bytes; one CTA per tile.
//   warp 0      TMEM allocation and MMA issue (one lane)
//   warps 1-3   TMA producers: two 64-row weight boxes and two 64-row token
//               boxes per stage, shared out between them
//   warps 4-19  epilogue: warp w reads TMEM lanes 32 (w % 4).. (channels) and
//               one quarter of the 128 token columns (four warps per
//               scheduler hide the TMEM load latency of the promotion)
// Every wait is bounded; a wait that runs out raises the device error word
// and the roles stop after draining their copies and MMAs.
#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kSBM = 128;                 // channels per tile (MMA M)
constexpr int kSBN = 128;                 // tokens per tile (MMA N)
constexpr int kSProd0 = 1, kSProds = 3;   // producer warps
constexpr int kSEpi0 = 4, kSEpis = 16;    // epilogue warps
constexpr int kSThreads = 32 * (kSEpi0 + kSEpis);
constexpr int kSCols = kSBN / 4;          // token columns per epilogue thread
constexpr int kSATile = kSBM * kBK;       // 16 KB
constexpr int kSStage = kSATile + kSBN * kBK;
constexpr int kSMaxStages = 6;
constexpr int kSBoxRows = 32;
constexpr int kSBoxes = 8;                // per stage: 4 weight + 4 token boxes of 32 rows
constexpr int kSAccBufs = 4;              // TMEM accumulators: 4 x 128 columns
constexpr int kSNumBars = 2 * kSMaxStages + 2 * kSAccBufs + 1;
constexpr int kSScaleLd = kSBN + 4;       // staged scales: [group][token], rows 16-byte aligned
constexpr int kSSmemLimit = 232448;

// Shared memory of a launch with `stages` stages and `ng` scale groups.
constexpr int scaled_smem_bytes(int stages, int ng) {
  return 1024 + stages * kSStage + ng * kSScaleLd * 4 + kSNumBars * 8 + 16 +
         4 * (kMaxGroups + 1) + 64;
}

enum : int { kModePtpc = 0, kModeSub512 = 1, kModeBlock128 = 2 };

template <int MODE>
__global__ void __launch_bounds__(kSThreads, 1) grouped_gemm_scaled_kernel(
    const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
    const float* __restrict__ a_scale, const float* __restrict__ w_scale,
    const int32_t* __restrict__ offsets, int groups, int64_t a_rows, int N, int K,
    int stages, float* __restrict__ out, unsigned* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int kblocks = K / kBK;
  // K blocks per scale group, and the groups
  const int gk = MODE == kModeBlock128 ? 1 : MODE == kModeSub512 ? 4 : kblocks;
  const int ngroups = kblocks / gk;
  float* sscale = reinterpret_cast<float*>(smem + stages * kSStage);   // [ngroups][132]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sscale + ngroups * kSScaleLd);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kSNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* prefix = reinterpret_cast<int*>(tmem_holder + 4);   // groups + 1
  __shared__ int warp_tot[kSThreads / 32];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_ctiles = N / kSBM;
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kSMaxStages + s); };
  auto accf_bar = [&](int b) { return smem_u32(bars + 2 * kSMaxStages + b); };
  auto acce_bar = [&](int b) { return smem_u32(bars + 2 * kSMaxStages + kSAccBufs + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * kSMaxStages + 2 * kSAccBufs);

  pdl_wait();
  // tile prefix: prefix[g] = sum_{g' < g} ceil(rows_g' / 128) * n_ctiles
  {
    const int per = (groups + kSThreads - 1) / kSThreads;
    const int g0 = threadIdx.x * per;
    int local = 0;
    for (int g = g0; g < g0 + per && g < groups; ++g)
      local += ((offsets[g + 1] - offsets[g] + kSBN - 1) / kSBN) * n_ctiles;
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
      run += ((offsets[g + 1] - offsets[g] + kSBN - 1) / kSBN) * n_ctiles;
    }
    if (threadIdx.x == kSThreads - 1) prefix[groups] = base + incl;
  }
  __syncthreads();
  const int tile = blockIdx.x;
  if (tile >= prefix[groups]) {   // the grid is an upper bound on the tiles
    pdl_launch_dependents();
    return;
  }
  const TileInfo ti = decode_tile(tile, prefix, groups, offsets, kSBN);
  const int wrow0 = ti.group * N + ti.ctile * kSBM;   // first weight row

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), kSBoxes);   // one arrival per box
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < kSAccBufs; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), kSEpis);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_a);
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_holder), kSAccBufs * kSBN);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  pdl_launch_dependents();

  if (warp >= kSProd0 && warp < kSProd0 + kSProds) {
    // ---------------- TMA producers: box lane * 3 + p, one per lane ----------------
    const int p = warp - kSProd0;
    const int b = lane * kSProds + p;
    if (b < kSBoxes) {
      const uint32_t bytes = kSBoxRows * kBK;
      const uint64_t pol_w = l2_policy_evict_normal();   // shared by the token tiles
      const uint64_t pol_a = l2_policy_evict_last();     // shared by the channel tiles
      int s = 0;
      uint32_t ph = 0;
      int issued = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kErrTimeoutProducer))
          break;
        mbar_arrive_expect_tx(full_bar(s), bytes);
        const uint32_t st = smem_u32(smem + s * kSStage);
        if (b < kSBoxes / 2)
          tma_load_2d(st + b * kSBoxRows * kBK, &tm_w, kb * kBK, wrow0 + b * kSBoxRows,
                      full_bar(s), pol_w);
        else
          tma_load_2d(st + kSATile + (b - kSBoxes / 2) * kSBoxRows * kBK, &tm_a, kb * kBK,
                      ti.row0 + (b - kSBoxes / 2) * kSBoxRows, full_bar(s), pol_a);
        ++issued;
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
      for (int i = 0; i < stages && i < issued; ++i) {   // every copy landed
        const int last = i + (issued - 1 - i) / stages * stages;
        volatile int no_abort = 0;
        mbar_wait_bounded(full_bar(i), (uint32_t)((last / stages) & 1), &no_abort, err,
                          kErrTimeoutDrain);
      }
    }
  } else if (warp == 0) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_e4m3_f32(kSBM, kSBN);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int g = 0; g < ngroups && ok; ++g) {
        const int b = g % kSAccBufs;
        if (!mbar_wait_bounded(acce_bar(b), (uint32_t)((g / kSAccBufs) & 1) ^ 1u, abort_flag,
                               err, kErrTimeoutMma))
          break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)(b * kSBN);
        for (int j = 0; j < gk; ++j) {
          if (!mbar_wait_bounded(full_bar(s), ph, abort_flag, err, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a = smem_u32(smem + s * kSStage), bt = a + kSATile;
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk)
            mma_f8f6f4(d, smem_desc_k_sw128(a + kk * 32), smem_desc_k_sw128(bt + kk * 32),
                       idesc, (j | kk) != 0);
          mma_commit(empty_bar(s));
          if (++s == stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) mma_commit(accf_bar(b));
      }
      mma_commit(drain_bar);   // every MMA complete before TMEM is released
      volatile int no_abort = 0;
      mbar_wait_bounded(drain_bar, 0, &no_abort, err, kErrTimeoutDrain);
    }
  } else {
    // ---------------- epilogue: promote each group into registers ----------------
    const int e = warp - kSEpi0;
    const int q = warp & 3;            // TMEM lane quarter: channels 32q..32q+31
    const int quarter = e >> 2;        // token columns quarter*32 .. quarter*32+31
    const int col0 = quarter * kSCols;
    // every group's multiplier of each of the tile's 128 token columns,
    // [group][token]: the activation scale, times the weight block's scale
    // for BlockScale-128 (read once, coalesced)
    {
      const float* swb = MODE == kModeBlock128
                             ? w_scale + ((int64_t)ti.group * n_ctiles + ti.ctile) * kblocks
                             : nullptr;
      const int64_t base = (int64_t)ti.row0 * ngroups;
      const int64_t lim = a_rows * ngroups;
      for (int i = threadIdx.x - kSEpi0 * 32; i < kSBN * ngroups; i += kSEpis * 32) {
        const int r = i / ngroups, g = i - r * ngroups;
        float v = base + i < lim ? a_scale[base + i] : 0.f;
        if (MODE == kModeBlock128) v = __fmul_rn(v, swb[g]);
        sscale[g * kSScaleLd + r] = v;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kSEpis * 32) : "memory");
    }
    float acc[kSCols];
#pragma unroll
    for (int c = 0; c < kSCols; ++c) acc[c] = 0.f;
    bool ok = true;
    for (int g = 0; g < ngroups; ++g) {
      const int b = g % kSAccBufs;
      if (!warp_wait(accf_bar(b), (uint32_t)((g / kSAccBufs) & 1), abort_flag, err,
                     kErrTimeoutEpilogue)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float* m = sscale + g * kSScaleLd + col0;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                             (uint32_t)(b * kSBN + col0);
#pragma unroll
      for (int h = 0; h < kSCols; h += 32) {   // 32 columns at a time (registers)
        float p[32];
        tmem_ld_x16(taddr + (uint32_t)h, *reinterpret_cast<float(*)[16]>(p));
        tmem_ld_x16(taddr + (uint32_t)(h + 16), *reinterpret_cast<float(*)[16]>(p + 16));
        tmem_ld_wait();
        if (h + 32 == kSCols) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(b));   // buffer free for group g + 4
        }
#pragma unroll
        for (int c4 = 0; c4 < 32; c4 += 4) {
          const float4 mm = *reinterpret_cast<const float4*>(m + h + c4);
          acc[h + c4] = fmaf(p[c4], mm.x, acc[h + c4]);
          acc[h + c4 + 1] = fmaf(p[c4 + 1], mm.y, acc[h + c4 + 1]);
          acc[h + c4 + 2] = fmaf(p[c4 + 2], mm.z, acc[h + c4 + 2]);
          acc[h + c4 + 3] = fmaf(p[c4 + 3], mm.w, acc[h + c4 + 3]);
        }
      }
    }
    if (ok) {
      const int n = ti.ctile * kSBM + q * 32 + lane;   // this thread's channel
      const float wch = MODE == kModeBlock128 ? 1.0f : w_scale[(int64_t)ti.group * N + n];
      const int nvalid = min(kSBN, ti.row_end - ti.row0) - col0;
#pragma unroll
      for (int c = 0; c < kSCols; ++c) {
        if (c < nvalid) {
          const float y = MODE == kModeBlock128 ? acc[c] : __fmul_rn(acc[c], wch);
          out[((int64_t)ti.row0 + col0 + c) * N + n] = y;   // a warp: 32 channels
        }
      }
    }
  }

  // ---------------- tear-down ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kSAccBufs * kSBN);
  }
}

// Per-row quantisation in 1 x BLOCK pieces along K, one warp per piece
// (lane = BLOCK / 32 consecutive elements); the quantiser of quant.cu:
// s = fp32(max(amax, 1e-12) / 448), q = e4m3_rne_sat(fp32(v / s)).
template <int BLOCK>
__global__ void __launch_bounds__(256) quant_blocks_kernel(
    const __nv_bfloat16* __restrict__ in, int64_t rows, int K, uint8_t* __restrict__ q,
    float* __restrict__ scales) {
  constexpr int kPer = BLOCK / 32;   // 4 or 16 elements per lane
  pdl_wait();
  pdl_launch_dependents();
  const int nb = K / BLOCK;
  const int64_t piece = (int64_t)blockIdx.x * 8 + threadIdx.x / 32;
  if (piece >= rows * nb) return;
  const int lane = threadIdx.x & 31;
  const int64_t r = piece / nb;
  const int b = (int)(piece % nb);
  const __nv_bfloat16* src = in + r * K + (int64_t)b * BLOCK + lane * kPer;
  float v[kPer];
  if constexpr (kPer == 4) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
    v[0] = __low2float(h[0]); v[1] = __high2float(h[0]);
    v[2] = __low2float(h[1]); v[3] = __high2float(h[1]);
  } else {
#pragma unroll
    for (int u = 0; u < kPer / 8; ++u) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + 8 * u);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * u + 2 * i] = __low2float(h[i]);
        v[8 * u + 2 * i + 1] = __high2float(h[i]);
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = warp_max(amax);
  const float s = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
  uint32_t w[kPer / 4];
#pragma unroll
  for (int j = 0; j < kPer / 4; ++j) {
    const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[4 * j], s), __fdiv_rn(v[4 * j + 1], s));
    const uint16_t hi =
        f32x2_to_e4m3x2(__fdiv_rn(v[4 * j + 2], s), __fdiv_rn(v[4 * j + 3], s));
    w[j] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  uint8_t* dst = q + r * K + (int64_t)b * BLOCK + lane * kPer;
  if constexpr (kPer == 4) {
    *reinterpret_cast<uint32_t*>(dst) = w[0];
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (lane == 0) scales[r * nb + b] = s;
}

// 128 x 128 block quantisation of an fp32 matrix: one CTA per block, thread
// t holds row t / 2, columns 64 (t % 2) .. +63.
__global__ void __launch_bounds__(256) quant_weight_blocks_kernel(
    const float* __restrict__ w, int K, uint8_t* __restrict__ q,
    float* __restrict__ scales) {
  __shared__ float red[8];
  pdl_wait();
  pdl_launch_dependents();
  const int kb = blockIdx.x, rb = blockIdx.y;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t row = (int64_t)rb * 128 + (t >> 1);
  const int col = kb * 128 + (t & 1) * 64;
  const float* src = w + row * K + col;
  float v[64];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float4 a = *reinterpret_cast<const float4*>(src + 4 * i);
    v[4 * i] = a.x; v[4 * i + 1] = a.y; v[4 * i + 2] = a.z; v[4 * i + 3] = a.w;
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = warp_max(amax);
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  float a = lane < 8 ? red[lane] : 0.f;
  a = warp_max(a);
  const float s = __fdiv_rn(fmaxf(a, 1e-12f), 448.0f);
  uint8_t* dst = q + row * K + col;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint32_t wd[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float* x = v + 16 * u + 4 * j;
      const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
      const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
      wd[j] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    *reinterpret_cast<uint4*>(dst + 16 * u) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
  if (t == 0) scales[(int64_t)rb * (K / 128) + kb] = s;
}

}  // namespace

int launch_grouped_gemm_scaled(int mode, const uint8_t* A, const float* a_scale,
                               int64_t a_rows, const uint8_t* W, const float* w_scale,
                               const int32_t* offsets, int groups, int N, int K,
                               float* out, cudaStream_t stream) {
  if (a_rows == 0 || groups == 0) return 0;
  CUtensorMap tm_w, tm_a;
  if (!make_tmap(&tm_w, W, (int64_t)groups * N, K, kSBoxRows)) return -3;
  if (!make_tmap(&tm_a, A, a_rows, K, kSBoxRows)) return -3;
  auto kern = mode == kModeBlock128 ? grouped_gemm_scaled_kernel<kModeBlock128>
              : mode == kModeSub512 ? grouped_gemm_scaled_kernel<kModeSub512>
                                    : grouped_gemm_scaled_kernel<kModePtpc>;
  const int kblocks = K / kBK;
  const int ng = mode == kModeBlock128 ? kblocks : mode == kModeSub512 ? kblocks / 4 : 1;
  int stages = kSMaxStages;
  while (stages > 2 && scaled_smem_bytes(stages, ng) > kSSmemLimit) --stages;
  const int smem = scaled_smem_bytes(stages, ng);
  if (smem > kSSmemLimit) return -2;   // K too long for the staged scales
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  const int64_t tiles = token_tiles_upper(a_rows, groups, kSBN) * (N / kSBM);
  if (tiles >= (int64_t(1) << 31)) return -2;
  kern<<<(unsigned)tiles, kSThreads, smem, stream>>>(tm_w, tm_a, a_scale, w_scale, offsets,
                                                     groups, a_rows, N, K, stages, out,
                                                     device_error_word());
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_quant_blocks(const uint16_t* in, int64_t rows, int K, int block, uint8_t* q,
                        float* scales, cudaStream_t stream) {
  if (rows == 0) return 0;
  const int64_t pieces = rows * (K / block);
  const int64_t grid = (pieces + 7) / 8;
  if (grid >= (int64_t(1) << 31)) return -2;
  const auto* x = reinterpret_cast<const __nv_bfloat16*>(in);
  if (block == 128)
    quant_blocks_kernel<128><<<(unsigned)grid, 256, 0, stream>>>(x, rows, K, q, scales);
  else
    quant_blocks_kernel<512><<<(unsigned)grid, 256, 0, stream>>>(x, rows, K, q, scales);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_quant_weight_blocks(const float* w, int64_t rows, int K, uint8_t* q,
                               float* scales, cudaStream_t stream) {
  if (rows == 0) return 0;
  if (rows / 128 > 65535) return -2;
  quant_weight_blocks_kernel<<<dim3((unsigned)(K / 128), (unsigned)(rows / 128)), 256, 0,
                               stream>>>(w, K, q, scales);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace moe
