// PTPC FP8 grouped GEMMs on a pair of SMs (tcgen05 cta_group::2).
//
// Same computation as gemm_tc.cu ("Optimizing Qwen 3.5 397B MoE on Ironwood
// TPU7x", GMM V2 paragraph; "Ultimate Latency Optimization of Qwen3 and
// Qwen3-VL on AMD MI300X Series", section 2.1.1), for wide token tiles where
// the tensor cores, not HBM, set the pace. Two CTAs of a cluster run one MMA
// of M = 256 rows: each CTA holds 128 weight rows and half of the BN token
// rows in its shared memory, and receives its 128 accumulator rows (x BN
// token columns) in its own TMEM. Each SM therefore loads half of the token
// tile that a single-CTA 128-row MMA of the same width would need, which
// halves the shared-memory traffic per multiply-add on the B side.
//
// Tile = 256 MMA rows x BN tokens of one expert:
//   gate/up: 128 channels; each CTA holds the gate and the up rows of its 64
//            channels ctile*128 + rank*64 + [0, 64), interleaved in blocks
//            of 16 (16 gate rows, the same channels' 16 up rows, ...) by one
//            5D TMA box, so that SwiGLU partners land in one warp's TMEM
//            lane quarter, 16 lanes apart;
//   down:    256 output channels, 128 per CTA.
//
// Roles per CTA (12 warps, 16 with the second epilogue set), both CTAs of
// the pair:
//   warp 0      TMEM allocation (both CTAs); the MMA issuer (leader)
//   warps 1-4   epilogue on this CTA's TMEM rows (12-15: a second set taking
//               every other 32-token chunk, for the down projection's fp16
//               output and the wide tiles)
//   warps 5-10  TMA producers: up to three per box (this CTA's weight box,
//               its token boxes), taking turns by stage, into its own ring
//               of stages of one or two 128-byte K atoms; both CTAs' copies
//               complete on the leader's stage barrier, which expects both
//               halves
//   warp 11     tile scheduler (cluster launch control)
// The leader's commits are multicast to both CTAs (stage free, accumulator
// ready); both CTAs' epilogues release an accumulator buffer by arriving on
// the leader's barrier (the peer with a relaxed arrive: the signal publishes
// no memory). All waits are bounded (common.cuh).
#include <cuda_fp16.h>

#include <algorithm>

#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace gemm;

__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
      "r"(ncols)
      : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
// D (+)= A * B^T over the CTA pair (M = 256), issued by one leader thread.
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc,
                                         uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at this offset in every CTA of `mask` when the
// leader's MMAs issued so far complete.
__device__ __forceinline__ void mma_commit_pair_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
      "multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar)
      : "memory");
}

// 2D tiled load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const void* tmap,
                                                 int32_t x, int32_t y, uint32_t bar,
                                                 uint64_t cache_policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::"
      "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(cache_policy)
      : "memory");
}

// 5D tiled load (the interleaved gate/up weights) into this CTA's shared
// memory; `pair` counts its completion on the leader's barrier (a
// shared::cluster address), else on this CTA's own.
__device__ __forceinline__ void tma_load_5d(uint32_t smem_dst, const void* tmap, int32_t x0,
                                            int32_t x3, int32_t x4, uint32_t bar,
                                            uint64_t cache_policy, bool pair) {
  if (pair)
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::"
        "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, %3, %4, %5}], [%6], %7;" ::"r"(
            smem_dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x0), "r"(0), "r"(x3), "r"(x4), "r"(bar),
        "l"(cache_policy)
        : "memory");
  else
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes."
        "L2::cache_hint [%0], [%1, {%2, %3, %3, %4, %5}], [%6], %7;" ::"r"(smem_dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x0), "r"(0), "r"(x3), "r"(x4), "r"(bar),
        "l"(cache_policy)
        : "memory");
}

__device__ __forceinline__ bool warp_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag,
                                                  unsigned* err, unsigned code) {
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t spin = 0;; ++spin) {
    const bool ok = mbar_try_wait_cluster(bar, parity);
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

template <int BN, bool GATEUP, bool OUT16 = false, bool WIDE = false, int KS = 1>
struct PairCfg {
  static constexpr int kHalfB = BN / 2;                  // token rows per CTA
  // TMA boxes of one stage (per CTA): the weights in one 128-row box
  // (gate/up: the 5D interleaving box), then 64-row token boxes.
  static constexpr int kWBoxes = 1;
  static constexpr int kWBoxRows = 128;
  static constexpr int kTBoxRows = kHalfB % 64 == 0 ? 64 : kHalfB;   // BN 192: one 96-row box
  static constexpr int kTBoxes = kHalfB / kTBoxRows;
  static constexpr int kBoxes = kWBoxes + kTBoxes;
  // A stage holds KS atoms of K (128 bytes each): the K blocks x, x + 128,
  // ... of the weights (A), then of the tokens (B), atom after atom. The
  // MMA issuer pays a fixed cost per stage (one full-barrier wait, one
  // commit) besides one per MMA, so two atoms (eight MMAs) per stage halve
  // the first where the tiles are narrower than 256 tokens.
  static constexpr int kAAtom = 128 * kBK;               // this CTA's 128 MMA rows
  static constexpr int kBAtom = kHalfB * kBK;
  static constexpr int kATile = KS * kAAtom;
  static constexpr int kBTile = KS * kBAtom;
  static constexpr int kStage = kATile + kBTile;
  static constexpr int kStages = (kStageBudget / kStage) > 10 ? 10 : (kStageBudget / kStage);
  // Producer warps per box: one thread issues a TMA copy about every 0.35 us
  // on GB300, so where the warps allow, kPar warps share each box and take
  // turns by stage (warp kPar*b + p: the stages q with q % kPar == p).
  // One-atom stages keep two warps per box with an even stage count; the
  // twice larger two-atom stages take up to three.
  static constexpr int kPar =
      KS == 1 ? ((2 * kBoxes <= kMaxBoxes && kStages % 2 == 0) ? 2 : 1)
              : (kMaxBoxes / kBoxes >= 3 ? 3 : kMaxBoxes / kBoxes >= 2 ? 2 : 1);
  static_assert(kBoxes * kPar <= kMaxBoxes, "producer warps");
  // a warp's next stage in a slot waits for the slot's previous stage, at
  // most one phase back (no parity aliasing) when kPar <= kStages
  static_assert(kPar <= kStages, "producer turns");
  static_assert(KS == 1 || !WIDE, "two-atom stages: narrow tiles");
  static constexpr int kAccBufs = 2 * BN <= 512 ? 2 : 1;
  static constexpr int kTmemCols = pow2_at_least(kAccBufs * BN);
  static constexpr int kChunk = 32;                      // epilogue columns per pass
  static constexpr int kTileCh = GATEUP ? 128 : 256;     // channels per tile
  static constexpr int kNumBars = 2 * kStages + 5;
  // output staging for TMA stores, per epilogue warp a box of 32 tokens x
  // 32 channels (down) or 16 channels (gate/up)
  static constexpr int kOutRows = 32;
  static constexpr int kOutCols = GATEUP ? 16 : 32;
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= (WIDE ? 512 : 256), "token tile");
  static_assert(!WIDE || (GATEUP && BN == 512), "wide tiles: gate/up, 512 tokens");
  static_assert(kStages >= 3, "pipeline depth");
  // fp16 down output: four more epilogue warps (12-15, the same TMEM lane
  // quarters) take every other 32-token chunk. A down tile's K is short
  // (K = I), and four warps drained 128 channels x 256 tokens slower than
  // the MMAs filled them. Their fp16 boxes fit the same staging bytes.
  // Wide gate/up tiles (one accumulator buffer, so the epilogue does not
  // overlap the next tile's MMAs) use the second set too.
  static constexpr bool kWideEpi = (!GATEUP && OUT16) || WIDE;
  static constexpr int kEpiSets = kWideEpi ? 2 : 1;
  static constexpr int kThreadsT = kThreads + (kWideEpi ? 4 * 32 : 0);
  // fp16 boxes of the down projection's second set fit the first set's bytes
  static constexpr int kOutBytes =
      4 * (GATEUP ? kEpiSets : 1) * kOutRows * kOutCols * 4;
  static constexpr int kSmemBytes = 1024 + kStages * kStage + kOutBytes +
                                    kNumBars * 8 + 16 + 8 * (kMaxGroups + 1) + 64;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Token rows a tile holds, and its MMA width: those rows rounded up to a
// multiple of 32, at least 64 so that each CTA's share is at least one
// 32-row token box. A partial tile then neither loads nor multiplies more
// than 31 rows past its end. A wide tile (up to 512 tokens) runs as two MMAs
// per K step, N1 = 256 columns and N2 = the rest, at least 64; the width is
// N1 + N2.
__device__ __forceinline__ int tile_rows(const TileInfo& ti) {
  return min(ti.width, ti.row_end - ti.row0);
}
__device__ __forceinline__ int pair_width(const TileInfo& ti) {
  const int n = max(64, (tile_rows(ti) + 31) & ~31);
  return n <= 256 ? n : 256 + max(64, n - 256);
}

// Token box t (ROWS rows) of a CTA (rank) in a tile of MMA width n: whether
// it is loaded, the row of the stage's token tile it fills and the first
// token row it copies. Narrow tiles: the CTA's n/2 tokens. Wide tiles
// (64-row boxes): boxes 0-1 fill rows 0-127 with the CTA's half of the
// first N1 tokens, boxes 2-3 rows 128-255 with its half of the next N2.
template <bool WIDE, int ROWS>
__device__ __forceinline__ bool token_box(int t, int n, int row0, int rank, int& smem_row,
                                          int& token_row) {
  if constexpr (!WIDE) {
    const int half = n / 2;
    smem_row = t * ROWS;
    token_row = row0 + rank * half + t * ROWS;
    return t * ROWS < half;
  } else {
    const int n1 = min(n, 256), n2 = n - n1;
    if (t < 2) {
      smem_row = t * 64;
      token_row = row0 + rank * (n1 / 2) + t * 64;
      return t * 64 < n1 / 2;
    }
    smem_row = 128 + (t - 2) * 64;
    token_row = row0 + n1 + rank * (n2 / 2) + (t - 2) * 64;
    return (t - 2) * 64 < n2 / 2;
  }
}

// OUT16 (down projection only): y as fp16 codes plus one factor per row, the
// encoding of the single-CTA kernel (gemm_tc.cu, fp16_rho).
template <int BN, bool GATEUP, bool OUT16, bool WIDE, int KS>
__global__ void __launch_bounds__(PairCfg<BN, GATEUP, OUT16, WIDE, KS>::kThreadsT, 1)
    grouped_gemm_pair_kernel(
    const __grid_constant__ CUtensorMap tm_w,
    const __grid_constant__ CUtensorMap tm_a,
    const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ a_scale,
    const float* __restrict__ w_scale, const int32_t* __restrict__ offsets,
    int groups, int N, int K, float* __restrict__ out,
    __half* __restrict__ out16, float* __restrict__ row_scale,
    const float* __restrict__ w_bound, int balanced, unsigned* __restrict__ err) {
  static_assert(!(OUT16 && GATEUP), "fp16 output is for the down projection");
  using C = PairCfg<BN, GATEUP, OUT16, WIDE, KS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* outstage = reinterpret_cast<float*>(smem + C::kStages * C::kStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage +
                                               C::kOutBytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* prefix = reinterpret_cast<int*>(tmem_holder + 4);   // groups + 1
  // the group offsets, copied: tile decoding reads only shared memory
  int* soff = prefix + (kMaxGroups + 1);
  __shared__ int warp_tot[C::kThreadsT / 32 + 1];
  __shared__ Sched sched;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_rank();        // 0: the leader issues the MMAs
  const int first_tile = (int)cluster_index();  // handed out first
  const int n_ctiles = N / C::kTileCh;
  const int kblocks = K / (kBK * KS);   // stages of a tile

  // full (leader's is the one used): both halves of a stage landed;
  // empty: stage free in this CTA (the leader's multicast commit)
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::kStages + s); };
  auto accf_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + b); };
  auto acce_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * C::kStages + 4);
  auto stage_a = [&](int s) { return smem_u32(smem + s * C::kStage); };
  auto stage_b = [&](int s) { return smem_u32(smem + s * C::kStage + C::kATile); };

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), C::kBoxes);   // the leader's producer warps
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 8 * C::kEpiSets);   // each epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    // ring consumers: each producer, each epilogue warp, the leader's MMA issuer
    sched_init(sched, C::kBoxes * C::kPar + 4 * C::kEpiSets + (rank == 0 ? 1 : 0));
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_a);
  }
  if (warp == kMmaWarp) tmem_alloc_pair(smem_u32(tmem_holder), C::kTmemCols);

  {   // tile prefix: prefix[g] = sum_{g' < g} ceil(rows_g' / BN) * n_ctiles
    const int per = (groups + C::kThreadsT - 1) / C::kThreadsT;
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
      soff[g] = offsets[g];
      run += ((offsets[g + 1] - offsets[g] + BN - 1) / BN) * n_ctiles;
    }
    if (threadIdx.x == C::kThreadsT - 1) {
      prefix[groups] = base + incl;
      soff[groups] = offsets[groups];
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const int total_tiles = prefix[groups];
  // an expert's rows in ceil(rows / BN) tiles of BN rows (the last partial),
  // or, balanced, of equal widths (multiples of 32)
  auto decode = [&](int tile) {
    return balanced ? decode_tile_balanced(tile, prefix, groups, soff, BN)
                    : decode_tile(tile, prefix, groups, soff, BN);
  };

  // down: this CTA's first weight row of a tile
  auto weight_row = [&](const TileInfo& ti) {
    return ti.group * N + ti.ctile * 256 + (int)rank * 128;
  };
  // Both CTAs' copies of stage s complete on the leader's full[s]: the
  // leader's own with a plain TMA, the peer's with the pair form.
  auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y, int s,
                  uint64_t pol) {
    if (rank == 0) tma_load_2d(dst, tm, x, y, full_bar(s), pol);
    else tma_load_2d_pair(dst, tm, x, y, map_to_rank(full_bar(s), 0), pol);
  };

  const int pwarp = producer_box(warp);             // producer warp index, or -1
  const int box = pwarp >= 0 ? pwarp / C::kPar : -1;
  const int par = pwarp >= 0 ? pwarp % C::kPar : 0;  // the stages it takes
  if (warp == kSchedWarp) {
    // ---------------- tile scheduler (both CTAs; the leader requests) ----------------
    if (lane == 0)
      sched_run(sched, first_tile, total_tiles, 2, rank, abort_flag, err, decode);
  } else if (box >= 0) {
    // ---------------- TMA producers (both CTAs): box `box` of every stage ----------------
    // (of every kPar-th stage, from stage `par` on)
    const bool weight_box = box < C::kWBoxes;
    if (lane == 0 && box < C::kBoxes) {
      const uint64_t pol = weight_box ? l2_policy_evict_normal() : l2_policy_evict_last();
      // bytes of this box in one CTA (all atoms of the stage); the leader
      // expects both CTAs' bytes
      const uint32_t bytes =
          (uint32_t)(KS * (weight_box ? C::kWBoxRows : C::kTBoxRows) * kBK);
      auto issue = [&](int s, int kb, const TileInfo& ti) {
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          const int x = (kb * KS + j) * kBK;
          const uint32_t sa = stage_a(s) + j * C::kAAtom, sb = stage_b(s) + j * C::kBAtom;
          if (GATEUP && box == 0) {   // gate and up rows of this CTA's 64 channels
            tma_load_5d(sa, &tm_w, x, (ti.ctile * 128 + (int)rank * 64) / 16, ti.group,
                        rank == 0 ? full_bar(s) : map_to_rank(full_bar(s), 0), pol,
                        rank != 0);
          } else if (weight_box) {    // down: this CTA's 128 rows
            load(sa, &tm_w, x, weight_row(ti), s, pol);
          } else {                    // rows of this CTA's half of the token tile
            int srow, trow;
            if (token_box<WIDE, C::kTBoxRows>(box - C::kWBoxes, pair_width(ti), ti.row0,
                                              (int)rank, srow, trow))
              load(sb + srow * kBK, &tm_a, x, trow, s, pol);
          }
        }
      };
      // a token box past the tile's MMA width is not loaded by either CTA
      auto expect = [&](int s, const TileInfo& ti) {
        if (rank != 0) return;
        int srow, trow;
        const bool used = weight_box || token_box<WIDE, C::kTBoxRows>(box - C::kWBoxes, pair_width(ti),
                                                        ti.row0, 0, srow, trow);
        mbar_arrive_expect_tx(full_bar(s), used ? 2 * bytes : 0u);
      };
      int qlast = -1;   // the last stage this warp issued
      // q numbers this CTA's stages in order (tile by tile, K block by K
      // block); stage q fills slot q % kStages in phase (q / kStages) & 1,
      // and this warp issues the stages with q % kPar == par
      uint32_t q = 0;
      bool ok = true;
      // weights and the tile map do not depend on the previous kernel
      int npre = 0;
      TileInfo t0{};
      if (weight_box && first_tile < total_tiles) {
        t0 = decode(first_tile);
        npre = kblocks < C::kStages ? kblocks : C::kStages;
        for (int kb = par; kb < npre; kb += C::kPar) {   // fresh ring: phase 0
          expect(kb, t0);
          issue(kb, kb, t0);
          qlast = kb;
        }
        q = (uint32_t)npre;
      }
      pdl_wait();
      pdl_launch_dependents();
      TileCursor cur;
      for (bool first = true; ok; first = false) {
        TileInfo ti;
        const int tile = next_tile_thread(sched, cur, box == 0 && par == 0 && rank == 0,
                                          abort_flag, err, kErrTimeoutProducer, ti);
        if (tile < 0) break;
        const bool pre = first && npre > 0 && tile == first_tile;
        for (int kb = pre ? npre : 0; kb < kblocks; ++kb, ++q) {
          if ((int)(q % C::kPar) != par) continue;
          const int s = (int)(q % C::kStages);
          const uint32_t ph = (q / C::kStages) & 1u;
          if (!wait_cluster_bounded(empty_bar(s), ph ^ 1, abort_flag, err,
                                    kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          expect(s, ti);
          issue(s, kb, ti);
          qlast = (int)q;
        }
      }
      // drain: this warp's copies have landed before the CTA's memory is
      // released. The MMA issuer consumes the stages in order, so once its
      // commit has freed this warp's last stage (in both CTAs), every copy
      // of the warp has landed. No later stage uses that slot (a warp's
      // turns are kPar <= kStages stages apart), so the phase parity of the
      // wait is unambiguous.
      if (qlast >= 0) {
        volatile int no_abort = 0;
        wait_cluster_bounded(empty_bar(qlast % C::kStages),
                             (uint32_t)(qlast / C::kStages) & 1u, &no_abort, err,
                             kErrTimeoutDrain);
      }
    } else {
      pdl_wait();
      pdl_launch_dependents();
    }
  } else if (warp == kMmaWarp) {
    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader) ----------------
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      TileCursor cur;
      for (; ok; ++it) {
        TileInfo ti;
        const int tile =
            next_tile_thread(sched, cur, false, abort_flag, err, kErrTimeoutMma, ti);
        if (tile < 0) break;
        const int ab = it % C::kAccBufs;
        const uint32_t acc_ph = (uint32_t)(it / C::kAccBufs) & 1u;
        if (!wait_cluster_bounded(acce_bar(ab), acc_ph ^ 1, abort_flag, err,
                                  kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d = tmem_base + (uint32_t)(ab * BN);
        const int n = pair_width(ti);
        const int n1 = min(n, 256), n2 = n - n1;   // n2 > 0: wide tiles only
        const uint32_t idesc = idesc_e4m3_f32(256, n1);
        const uint32_t idesc2 = idesc_e4m3_f32(256, n2 > 0 ? n2 : 64);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_cluster_bounded(full_bar(s), ph, abort_flag, err, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < KS * kBK / 32; ++kk) {   // 32 K bytes per MMA
            const int j = kk / (kBK / 32), k32 = (kk % (kBK / 32)) * 32;
            const uint32_t a = stage_a(s) + j * C::kAAtom + k32;
            const uint32_t b = stage_b(s) + j * C::kBAtom + k32;
            const uint64_t adesc = smem_desc_k_sw128(a);
            mma_pair(d, adesc, smem_desc_k_sw128(b), idesc, (kb | kk) != 0);
            if (WIDE && n2 > 0)   // columns 256.. from token rows 128.. of the stage
              mma_pair(d + 256, adesc, smem_desc_k_sw128(b + 128 * kBK), idesc2,
                       (kb | kk) != 0);
          }
          mma_commit_pair_mc(empty_bar(s), 0x3);   // stage free in both CTAs
          if (++s == C::kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) mma_commit_pair_mc(accf_bar(ab), 0x3);   // accumulators ready
      }
      mma_commit_pair(drain_bar);
      volatile int no_abort = 0;
      mbar_wait_bounded(drain_bar, 0, &no_abort, err, kErrTimeoutDrain);
    }
  } else {
    // ---------------- epilogue (both CTAs) ----------------
    pdl_wait();
    pdl_launch_dependents();
    const int q = warp & 3;               // TMEM lane quarter of this warp
    const int m = q * 32 + lane;          // accumulator row of this thread
    int it = 0;
    bool ok = true;
    // Output of C::kOutRows tokens from token r0 on, for this warp's 32
    // channels ch0 + lane (v[j] = token r0 + j). A box inside the expert goes
    // through shared memory and one TMA store; a box crossing the expert's end
    // is stored directly, so rows of the next expert are never written.
    // epilogue warp index e = 0..3 (warps 1-4), 4..7 (12-15)
    const int e_idx = warp < kSchedWarp ? warp - kEpiWarp0 : warp - kSchedWarp + 3;
    const int eset = warp < kSchedWarp ? 0 : 1;
    float* obuf = OUT16 ? reinterpret_cast<float*>(reinterpret_cast<__half*>(outstage) +
                                                   e_idx * C::kOutRows * 32)
                        : outstage + e_idx * C::kOutRows * C::kOutCols;
    auto emit = [&](int r0, int row_end, int ch0, const float* v) {
      if (r0 + C::kOutRows <= row_end) {
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        if constexpr (OUT16) {
          __half* o16 = reinterpret_cast<__half*>(obuf);
#pragma unroll
          for (int j = 0; j < C::kOutRows; ++j) o16[j * 32 + lane] = __float2half_rn(v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < C::kOutRows; ++j) obuf[j * 32 + lane] = v[j];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_out, ch0, r0, smem_u32(obuf));
          bulk_commit();
        }
      } else {
#pragma unroll
        for (int j = 0; j < C::kOutRows; ++j) {
          if (r0 + j < row_end) {
            const int64_t o = (int64_t)(r0 + j) * N + ch0 + lane;
            if constexpr (OUT16) out16[o] = __float2half_rn(v[j]);
            else out[o] = v[j];
          }
        }
      }
    };
    TileCursor cur;
    for (; ok; ++it) {
      TileInfo ti;
      const int tile =
          next_tile_warp(sched, cur, abort_flag, err, kErrTimeoutEpilogue, ti);
      if (tile < 0) break;
      const int ab = it % C::kAccBufs;
      const uint32_t acc_ph = (uint32_t)(it / C::kAccBufs) & 1u;
      const int nvalid = tile_rows(ti);
      // gate/up: this thread's channel, its two weight scales and the first
      // chunk's token scales, loaded while the MMAs finish
      const bool is_gate = lane < 16;
      const int ch_gu = ti.ctile * 128 + (int)rank * 64 + q * 16 + (lane & 15);
      float swg = 0.f, swu = 0.f, sx_next = 0.f;
      if constexpr (GATEUP) {
        swg = w_scale[(int64_t)ti.group * 2 * N + ch_gu];
        swu = w_scale[(int64_t)ti.group * 2 * N + N + ch_gu];
        const int nfirst = C::kChunk * eset;
        sx_next = nfirst + lane < nvalid ? a_scale[ti.row0 + nfirst + lane] : 0.f;
      }
      // down: this thread's channel scale and, for fp16 output, the rows'
      // factors a_scale / rho (written by the tile of the first channels)
      const int ch_d = ti.ctile * 256 + (int)rank * 128 + m;
      float sw_d = 0.f, swr_d = 0.f;
      if constexpr (!GATEUP) {
        sw_d = w_scale[(int64_t)ti.group * N + ch_d];
        swr_d = sw_d;
        if constexpr (OUT16) {
          const float rho = fp16_rho(w_bound[ti.group], K);
          swr_d = sw_d * rho;
          if (ti.ctile == 0 && rank == 0) {   // one factor per row
            for (int r = e_idx * 32 + lane; r < nvalid; r += 128 * C::kEpiSets)
              row_scale[ti.row0 + r] = __fdiv_rn(a_scale[ti.row0 + r], rho);
          }
        }
      }
      if (!warp_wait_cluster(accf_bar(ab), acc_ph, abort_flag, err,
                             kErrTimeoutEpilogue))
        break;
      tc_fence_after_sync();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * BN);
      if (GATEUP) {
        // TMEM lanes 32q .. 32q+15 hold the gate rows of channels ch0 + [0,
        // 16), ch0 = ctile*128 + rank*64 + 16q, and lanes 32q+16 .. 32q+31
        // the up rows of the same channels. Per 32-column chunk a gate
        // thread trades its columns 16-31 for its up partner's (lane + 16)
        // columns 0-15, one shuffle each, so every thread finishes 16
        // outputs of its channel.
        const int ch = ch_gu;
        const int c0 = is_gate ? 0 : 16;           // this thread's columns
        // token scales of a chunk (lane = column), loaded one chunk ahead;
        // with two epilogue sets, set e takes chunks e, e + 2, ...
        constexpr int kStep = C::kChunk * C::kEpiSets;
        for (int n0 = C::kChunk * eset; n0 < nvalid; n0 += kStep) {
          const float sx_l = sx_next;
          if (n0 + kStep < nvalid)
            sx_next = n0 + kStep + lane < nvalid ? a_scale[ti.row0 + n0 + kStep + lane] : 0.f;
          float a[C::kChunk];
          tmem_ld_x16(taddr + n0, *reinterpret_cast<float(*)[16]>(&a[0]));
          tmem_ld_x16(taddr + n0 + 16, *reinterpret_cast<float(*)[16]>(&a[16]));
          tmem_ld_wait();
          float hv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float got =
                __shfl_xor_sync(0xffffffffu, is_gate ? a[16 + j] : a[j], 16);
            const float g = is_gate ? a[j] : got;
            const float u = is_gate ? got : a[16 + j];
            const float sx = __shfl_sync(0xffffffffu, sx_l, c0 + j);
            const float gg = g * sx * swg;
            const float uu = u * sx * swu;
            hv[j] = __fdividef(gg * uu, 1.0f + __expf(-gg));
          }
          // 32 tokens x this warp's 16 channels: one TMA store through shared
          // memory ([token][channel]); a chunk crossing the tile's end is
          // stored directly, so rows past it are never written
          if (n0 + C::kChunk <= nvalid) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 16; ++j) obuf[(c0 + j) * 16 + (lane & 15)] = hv[j];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tm_out, ch - (lane & 15), ti.row0 + n0, smem_u32(obuf));
              bulk_commit();
            }
          } else {
            float* o = out + (int64_t)(ti.row0 + n0 + c0) * N + ch;
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (n0 + c0 + j < nvalid) o[(int64_t)j * N] = hv[j];
          }
        }
      } else {
        const int ch = ch_d;
        const float sw = sw_d, swr = swr_d;
        for (int n0 = 32 * eset; n0 < nvalid; n0 += 32 * C::kEpiSets) {
          float acc[32];
          tmem_ld_x16(taddr + n0, *reinterpret_cast<float(*)[16]>(&acc[0]));
          tmem_ld_x16(taddr + n0 + 16, *reinterpret_cast<float(*)[16]>(&acc[16]));
          tmem_ld_wait();
          float v[32];
          if constexpr (OUT16) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = acc[j] * swr;
          } else {
            const float sx_l = n0 + lane < nvalid ? a_scale[ti.row0 + n0 + lane] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = acc[j] * __shfl_sync(0xffffffffu, sx_l, j) * sw;
          }
          emit(ti.row0 + n0, ti.row0 + nvalid, ch - lane, v);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(acce_bar(ab));
        else mbar_arrive_cluster_relaxed(map_to_rank(acce_bar(ab), 0));
      }
    }
    if (lane == 0) bulk_wait_all();   // this warp's TMA stores are complete
  }

  // ---------------- tear-down ----------------
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();   // the leader's MMAs (which use both CTAs) are complete
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <int BN, bool GATEUP, bool OUT16 = false, bool WIDE = false, int KS = 1>
int run_pair(const uint8_t* A, const float* a_scale, int64_t a_rows,
             const uint8_t* W, const float* w_scale, const int32_t* offsets,
             int groups, int N, int K, float* out, cudaStream_t stream, bool pdl,
             int balanced, __half* out16 = nullptr, float* row_scale = nullptr,
             const float* w_bound = nullptr) {
  using C = PairCfg<BN, GATEUP, OUT16, WIDE, KS>;
  if (K % (kBK * KS) != 0) return -1;
  CUtensorMap tm_w, tm_a;
  if (GATEUP) {   // one box: 64 channels' gate and up rows, interleaved by 16
    if (!make_tmap_gateup_interleaved(&tm_w, W, groups, N, K)) return -3;
  } else if (!make_tmap(&tm_w, W, (int64_t)groups * N, K, C::kWBoxRows)) {
    return -3;
  }
  if (!make_tmap(&tm_a, A, a_rows, K, C::kTBoxRows)) return -3;
  CUtensorMap tm_out;
  const bool made = OUT16
                        ? make_tmap_out(&tm_out, out16, a_rows, N, C::kOutRows, 32, 2)
                        : make_tmap_out(&tm_out, out, a_rows, N, C::kOutRows, C::kOutCols, 4);
  if (!made) return -3;
  auto kern = grouped_gemm_pair_kernel<BN, GATEUP, OUT16, WIDE, KS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return -3;
  const int64_t upper = token_tiles_upper(a_rows, groups, BN) * (int64_t)(N / C::kTileCh);
  // one cluster per possible tile; the ones that run first take the rest
  // over (cluster launch control, see the scheduler)
  if (upper <= 0) return 0;
  if (2 * upper > INT32_MAX) return -2;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * upper));
  cfg.blockDim = dim3(C::kThreadsT);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, tm_w, tm_a, tm_out, a_scale, w_scale, offsets,
                         groups, N, K, out, out16, row_scale, w_bound, balanced,
                         device_error_word());
  return e == cudaSuccess ? 0 : -3;
}

}  // namespace

bool grouped_gemm_pair_supported(int kind, int N) {
  return N % (kind == 0 ? 128 : 256) == 0;
}

int launch_grouped_gemm_pair(int kind, const uint8_t* A, const float* a_scale,
                             int64_t a_rows, const uint8_t* W,
                             const float* w_scale, const int32_t* offsets,
                             int groups, int N, int K, float* out, int bn,
                             cudaStream_t stream, bool pdl) {
  const int bal = balanced_tiles();
  if (kind == 0) {
    if (bn > 256)   // wide tiles are always balanced
      return run_pair<512, true, false, true>(A, a_scale, a_rows, W, w_scale, offsets,
                                              groups, N, K, out, stream, pdl, 1);
    // two K atoms per stage where K allows
    const bool ks2 = pair_k_atoms() == 2 && K % (2 * kBK) == 0;
    if (bn == 192)
      return ks2 ? run_pair<192, true, false, false, 2>(A, a_scale, a_rows, W, w_scale,
                                                        offsets, groups, N, K, out, stream,
                                                        pdl, bal)
                 : run_pair<192, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N,
                                       K, out, stream, pdl, bal);
    if (bn <= 128)
      return ks2 ? run_pair<128, true, false, false, 2>(A, a_scale, a_rows, W, w_scale,
                                                        offsets, groups, N, K, out, stream,
                                                        pdl, bal)
                 : run_pair<128, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N,
                                       K, out, stream, pdl, bal);
    return ks2 ? run_pair<256, true, false, false, 2>(A, a_scale, a_rows, W, w_scale,
                                                      offsets, groups, N, K, out, stream,
                                                      pdl, bal)
               : run_pair<256, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K,
                                     out, stream, pdl, bal);
  }
  const bool ks2 = pair_k_atoms() == 2 && K % (2 * kBK) == 0;
  if (bn <= 128)
    return ks2 ? run_pair<128, false, false, false, 2>(A, a_scale, a_rows, W, w_scale,
                                                       offsets, groups, N, K, out, stream,
                                                       pdl, bal)
               : run_pair<128, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N,
                                      K, out, stream, pdl, bal);
  return ks2 ? run_pair<256, false, false, false, 2>(A, a_scale, a_rows, W, w_scale,
                                                     offsets, groups, N, K, out, stream, pdl,
                                                     bal)
             : run_pair<256, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K,
                                    out, stream, pdl, bal);
}

int launch_grouped_gemm_pair_down_f16(const uint8_t* A, const float* a_scale,
                                      int64_t a_rows, const uint8_t* W,
                                      const float* w_scale, const float* w_bound,
                                      const int32_t* offsets, int groups, int N,
                                      int K, uint16_t* y16, float* row_scale, int bn,
                                      cudaStream_t stream, bool pdl) {
  __half* o = reinterpret_cast<__half*>(y16);
  const int bal = balanced_tiles();
  const bool ks2 = pair_k_atoms() == 2 && K % (2 * kBK) == 0;
  if (bn <= 128)
    return ks2 ? run_pair<128, false, true, false, 2>(A, a_scale, a_rows, W, w_scale,
                                                      offsets, groups, N, K, nullptr,
                                                      stream, pdl, bal, o, row_scale,
                                                      w_bound)
               : run_pair<128, false, true>(A, a_scale, a_rows, W, w_scale, offsets,
                                            groups, N, K, nullptr, stream, pdl, bal, o,
                                            row_scale, w_bound);
  return ks2 ? run_pair<256, false, true, false, 2>(A, a_scale, a_rows, W, w_scale, offsets,
                                                    groups, N, K, nullptr, stream, pdl, bal,
                                                    o, row_scale, w_bound)
             : run_pair<256, false, true>(A, a_scale, a_rows, W, w_scale, offsets, groups,
                                          N, K, nullptr, stream, pdl, bal, o, row_scale,
                                          w_bound);
}

}  // namespace moe
