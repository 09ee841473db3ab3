// Pieces shared by the grouped-GEMM kernels (single-CTA and CTA-pair).
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace gemm {

// Warp roles of a GEMM CTA. TMA issue is serialised per warp, and the
// shared-memory operand feed of one SM grows with the number of warps that
// issue copies (about 43 GB/s per SM with one, 129 GB/s with six on GB300),
// so each TMA box of a stage has a producer warp of its own.
constexpr int kMmaWarp = 0;        // TMEM allocation and MMA issue
constexpr int kEpiWarp0 = 1;       // warps 1-4: epilogue (one TMEM lane quarter each)
constexpr int kProdWarp0 = 5;      // warps 5-10: producers, one box of a stage each
constexpr int kMaxBoxes = 6;
constexpr int kSchedWarp = kProdWarp0 + kMaxBoxes;   // warp 11: tile scheduler
constexpr int kThreads = 32 * (kSchedWarp + 1);

// Index of the box a warp loads (-1 for warps that are not producers).
__device__ __forceinline__ int producer_box(int warp) {
  return warp >= kProdWarp0 && warp < kSchedWarp ? warp - kProdWarp0 : -1;
}
constexpr int kBK = 128;        // K bytes per stage = one 128-byte swizzle row
constexpr int kStageBudget = 200 * 1024;

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

// Factor that maps the down projection's scaled accumulator into fp16 range
// for an expert whose largest weight scale is `bound`: every product of two
// e4m3 codes is at most 448^2 in magnitude, so |acc| <= 448^2 K and
// |acc * s_d * rho| <= 60000 < 65504 (the largest finite fp16) for every
// s_d <= bound. Computed in fp32 as ((60000 / 448^2) / K) / bound with IEEE
// divisions, once per tile, so every CTA gets the same value; its three
// roundings leave |acc * s_d * rho| below 60000.02, which fp16 rounds to at
// most 60000. (The fp64 form cost each epilogue warp 700-900 cycles per
// tile on GB300's narrow fp64 pipe.)
__device__ __forceinline__ float fp16_rho(float bound, int K) {
  float r = __fdiv_rn(__fdiv_rn(60000.0f / 200704.0f, (float)K), bound);
  if (!(r <= 3.0e38f)) r = 3.0e38f;   // a zero bound: any finite factor works
  return r;
}

struct TileInfo {
  int group, ctile, row0, row_end;
  int width;   // token rows of the tile (the last tile of a group may hold fewer)
};

__device__ __forceinline__ TileInfo decode_tile(int tile, const int* prefix,
                                                int groups, const int32_t* offsets,
                                                int bn) {
  // the largest g with prefix[g] <= tile; empty groups share their
  // successor's prefix value, so this is the non-empty group owning the tile
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int start = offsets[g], end = offsets[g + 1];
  const int tt = (end - start + bn - 1) / bn;
  const int local = tile - prefix[g];
  TileInfo t;
  t.group = g;
  t.ctile = local / tt;
  t.row0 = start + (local % tt) * bn;
  t.row_end = end;
  t.width = bn;
  return t;
}

// Balanced tiles of at most bn_max rows: a group of r rows is cut into
// tt = ceil(r / bn_max) tiles of w = 32 * ceil(ceil(r / tt) / 32) rows, the
// last one holding the rest (w <= bn_max, and every tile holds rows). The
// prefix counts ceil(r / bn_max) tiles per channel tile, as for decode_tile.
__device__ __forceinline__ TileInfo decode_tile_balanced(int tile, const int* prefix,
                                                         int groups,
                                                         const int32_t* offsets,
                                                         int bn_max) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int start = offsets[g], end = offsets[g + 1];
  const int rows = end - start;
  const int tt = (rows + bn_max - 1) / bn_max;
  const int w = ((rows + tt - 1) / tt + 31) / 32 * 32;
  const int local = tile - prefix[g];
  TileInfo t;
  t.group = g;
  t.ctile = local / tt;
  t.row0 = start + (local % tt) * w;
  t.row_end = end;
  t.width = w;
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


// ---------------------------------------------------------------------------
// Cluster helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_addr)
               : "memory");
}
// Relaxed arrive on another CTA's barrier, for a signal that publishes no
// memory: an epilogue warp telling the MMA issuer that its tcgen05.ld of an
// accumulator have completed (tcgen05.wait::ld, then
// tcgen05.fence::before_thread_sync). The release form made the peer CTA's
// epilogue warps wait 2,000-3,200 cycles per tile on GB300.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a barrier that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool wait_cluster_bounded(uint32_t bar, uint32_t parity,
                                                     volatile int* abort_flag,
                                                     unsigned* err, unsigned code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t spin = 0;; ++spin) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((spin & 63u) == 63u) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(err, code);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dynamic tile scheduler (cluster launch control)
// ---------------------------------------------------------------------------
// The grid has one CTA (or CTA pair) per possible tile, more than can be
// resident. A CTA that runs takes its own tile, then cancels the launch of a
// CTA that has not started yet and takes that CTA's tile instead
// (clusterlaunchcontrol.try_cancel), until no launch is left to cancel. Tiles
// are thus handed out one at a time, in launch order (neighbouring tiles,
// which share weight and token tiles in L2, still run side by side), to
// whichever SM frees up first: ragged experts, narrowed tail tiles and
// unequal tile costs no longer leave some SMs with more work than others.
//
// One scheduler thread per CTA publishes the sequence to the CTA's roles
// through a small ring in shared memory, each tile with its decoded
// coordinates (expert, channel tile, rows), so that no role decodes a tile
// on its own critical path; -1 ends it. The next tile is
// requested only when the first producer has taken the last one, so a CTA
// holds at most one tile in reserve beyond those in its pipeline. In a CTA
// pair the leader requests, the response is multicast to both CTAs, and both
// schedulers publish the same sequence.
constexpr int kRing = 4;

struct Sched {
  alignas(16) uint4 resp[2];   // cancel responses (double-buffered)
  uint64_t full[kRing];        // tile[i] written
  uint64_t empty[kRing];       // every consumer has read tile[i]
  uint64_t taken;              // the first producer took a tile
  uint64_t resp_bar[2];        // a response landed (16 bytes expected)
  uint64_t resp_free[2];       // pair: the peer has read a response
  int tile[kRing];
  TileInfo info[kRing];        // tile[i] decoded
};

// `consumers`: arrivals that free a ring slot (one per consuming thread or
// warp of this CTA). Called by one thread before the CTA's first barrier.
__device__ __forceinline__ void sched_init(Sched& sc, int consumers) {
  for (int i = 0; i < kRing; ++i) {
    mbar_init(smem_u32(&sc.full[i]), 1);
    mbar_init(smem_u32(&sc.empty[i]), consumers);
  }
  mbar_init(smem_u32(&sc.taken), 1);
  for (int b = 0; b < 2; ++b) {
    mbar_init(smem_u32(&sc.resp_bar[b]), 1);
    mbar_init(smem_u32(&sc.resp_free[b]), 1);
  }
}

__device__ __forceinline__ void clc_try_cancel(uint32_t resp, uint32_t bar, bool multicast) {
  if (multicast)
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes."
        "multicast::cluster::all.b128 [%0], [%1];" ::"r"(resp),
        "r"(bar)
        : "memory");
  else
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes."
        "b128 [%0], [%1];" ::"r"(resp),
        "r"(bar)
        : "memory");
}

// Whether the request cancelled a launch, and the x index of the first CTA of
// the cancelled cluster.
__device__ __forceinline__ bool clc_query(uint32_t resp, uint32_t& x) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b128 v;\n\t"
      "ld.shared.b128 v, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, v;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, v;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(resp)
      : "memory");
  return ok != 0;
}

// The scheduler thread. `first`: this CTA's (pair's) own tile; `cta_per_tile`:
// 1, or 2 for CTA pairs; `rank`: rank in the pair (0 requests); `decode`
// maps a tile index to its TileInfo.
template <typename Decode>
__device__ inline void sched_run(Sched& sc, int first, int total, int cta_per_tile,
                                 uint32_t rank, volatile int* abort_flag,
                                 unsigned* err, Decode decode) {
  int slot = 0;
  uint32_t ph = 0;
  uint32_t resp_ph[2] = {0u, 0u}, free_ph[2] = {0u, 0u};
  int uses[2] = {0, 0};
  uint32_t taken_ph = 0;
  auto publish = [&](int t) -> bool {
    if (!mbar_wait_bounded(smem_u32(&sc.empty[slot]), ph ^ 1u, abort_flag, err,
                           kErrTimeoutSched))
      return false;
    if (t >= 0) sc.info[slot] = decode(t);
    *reinterpret_cast<volatile int*>(&sc.tile[slot]) = t;
    mbar_arrive(smem_u32(&sc.full[slot]));
    if (++slot == kRing) {
      slot = 0;
      ph ^= 1u;
    }
    return true;
  };
  // offsets that need more tiles than the grid has CTAs (rows past a_rows)
  if ((int64_t)total * cta_per_tile > (int64_t)gridDim.x) atomicOr(err, kErrBadIndex);
  bool ok = true, pending_take = false;
  if (first < total) {
    ok = publish(first);
    pending_take = true;
  }
  int b = 0;
  while (ok) {
    if (rank == 0 && pending_take) {   // request just in time
      if (!mbar_wait_bounded(smem_u32(&sc.taken), taken_ph, abort_flag, err,
                             kErrTimeoutSched))
        break;
      taken_ph ^= 1u;
    }
    pending_take = false;
    mbar_arrive_expect_tx(smem_u32(&sc.resp_bar[b]), 16);
    if (rank == 0) {
      if (cta_per_tile > 1 && uses[b] > 0) {   // the peer read this buffer
        if (!wait_cluster_bounded(smem_u32(&sc.resp_free[b]), free_ph[b], abort_flag,
                                  err, kErrTimeoutSched))
          break;
        free_ph[b] ^= 1u;
      }
      fence_proxy_async_smem();
      clc_try_cancel(smem_u32(&sc.resp[b]), smem_u32(&sc.resp_bar[b]), cta_per_tile > 1);
    }
    ++uses[b];
    if (!mbar_wait_bounded(smem_u32(&sc.resp_bar[b]), resp_ph[b], abort_flag, err,
                           kErrTimeoutSched))
      break;
    resp_ph[b] ^= 1u;
    uint32_t x = 0;
    const bool got = clc_query(smem_u32(&sc.resp[b]), x);
    if (cta_per_tile > 1 && rank != 0)
      mbar_arrive_cluster(map_to_rank(smem_u32(&sc.resp_free[b]), 0));
    b ^= 1;
    if (!got) break;   // nothing left to cancel: never request again
    const int t = (int)(x / (uint32_t)cta_per_tile);
    if (t < total) {
      ok = publish(t);
      pending_take = true;
    }
  }
  publish(-1);
}

// A consumer's position in the ring.
struct TileCursor {
  int slot = 0;
  uint32_t phase = 0;
};

// Next tile for a role run by one thread (-1: no more, or a wait ran out),
// its coordinates in `ti`. `take` marks the first producer, whose taking
// releases the next request.
__device__ __forceinline__ int next_tile_thread(Sched& sc, TileCursor& c, bool take,
                                                volatile int* abort_flag, unsigned* err,
                                                unsigned code, TileInfo& ti) {
  if (!mbar_wait_bounded(smem_u32(&sc.full[c.slot]), c.phase, abort_flag, err, code))
    return -1;
  const int t = *reinterpret_cast<volatile int*>(&sc.tile[c.slot]);
  if (t >= 0) ti = sc.info[c.slot];
  mbar_arrive(smem_u32(&sc.empty[c.slot]));
  if (take && t >= 0) mbar_arrive(smem_u32(&sc.taken));
  if (++c.slot == kRing) {
    c.slot = 0;
    c.phase ^= 1u;
  }
  return t;
}

// Next tile for a role run by a whole warp (the same answer in every lane).
__device__ __forceinline__ int next_tile_warp(Sched& sc, TileCursor& c,
                                              volatile int* abort_flag, unsigned* err,
                                              unsigned code, TileInfo& ti) {
  if (!warp_wait(smem_u32(&sc.full[c.slot]), c.phase, abort_flag, err, code)) return -1;
  const int t = *reinterpret_cast<volatile int*>(&sc.tile[c.slot]);
  if (t >= 0) ti = sc.info[c.slot];
  __syncwarp();
  if (lane_id() == 0) mbar_arrive(smem_u32(&sc.empty[c.slot]));
  if (++c.slot == kRing) {
    c.slot = 0;
    c.phase ^= 1u;
  }
  return t;
}

// Upper bound on the token tiles of `groups` expert slices that hold
// `a_rows` rows in all, BN rows per tile. A non-empty slice of r rows has
// floor((r - 1) / BN) + 1 tiles, and at most min(groups, a_rows) slices are
// non-empty, so the total is at most floor((a_rows - ne) / BN) + ne with
// ne = min(groups, a_rows). The grid has one CTA (pair) per possible tile,
// and every surplus one costs a cancellation round trip, so the bound is
// kept tight (exact when every slice holds at most BN rows).
inline int64_t token_tiles_upper(int64_t a_rows, int groups, int bn) {
  const int64_t ne = a_rows < groups ? a_rows : (int64_t)groups;
  return (a_rows - ne) / bn + ne;
}

// Row-major [rows, K] uint8 matrix as a 2D TMA tensor map: box = 128 bytes
// of K x box_rows rows, 128-byte swizzle; rows past the end read as zero.
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int K,
               int box_rows);

// The gate/up weights [groups][2N][K] (gate rows, then up rows) as a 5D TMA
// tensor map whose 16 KB box holds 4 blocks of 16 channels, each as its 16
// gate rows followed by the same channels' 16 up rows (128-byte swizzle).
// Coordinates: (k, 0, 0, first channel / 16, expert). Needs N % 64 == 0.
bool make_tmap_gateup_interleaved(CUtensorMap* map, const void* W, int groups, int N,
                                  int K);

// Row-major [rows, cols] fp32 (elem_bytes 4) or fp16 (2) matrix as a 2D TMA
// tensor map for stores of box_rows x box_cols boxes (no swizzle).
bool make_tmap_out(CUtensorMap* map, void* base, int64_t rows, int cols,
                   int box_rows, int box_cols, int elem_bytes);

// Streaming multiprocessors of the current device (cached).
int sm_count();

// MOE_GEMM_CTA_PAIR: 1 forces the CTA-pair kernel for wide token tiles, 0
// disables it, unset (-1) leaves the choice to the dispatch rule.
int cta_pair_mode();

// MOE_GEMM_DOWN_PAIR: the same switch for the down projection alone (its
// fp16-output form); unset (-1) follows MOE_GEMM_CTA_PAIR, then the rule.
int down_pair_mode();

// Token tiles of the CTA-pair kernels: 1 (default) cuts an expert's rows into
// equal tiles (widths rounded up to 32 rows), MOE_GEMM_BALANCED=0 into
// full tiles and one partial tail.
int balanced_tiles();

// MOE_GEMM_WIDE: 1 runs gate/up CTA-pair tiles of up to 512 tokens (two MMAs
// per K step) above 256 rows per expert, 0 never; unset (-1): the rule.
int wide_tiles_mode();

// MOE_GEMM_PAIR_BN=128 / 256: token tile of the CTA-pair kernels when they
// run; unset (0): from the rows per expert.
int pair_bn_mode();

// K atoms (128 bytes of K each) per stage of the gate/up CTA-pair kernel:
// 2 (default) where K is a multiple of 256, MOE_GEMM_KATOMS=1 one.
int pair_k_atoms();

}  // namespace gemm
}  // namespace moe
