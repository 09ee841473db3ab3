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
constexpr int kThreads = 32 * (kProdWarp0 + kMaxBoxes);

// Index of the box a warp loads (-1 for warps that are not producers).
__device__ __forceinline__ int producer_box(int warp) {
  return warp >= kProdWarp0 ? warp - kProdWarp0 : -1;
}
constexpr int kBK = 128;        // K bytes per stage = one 128-byte swizzle row
constexpr int kStageBudget = 200 * 1024;

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

struct TileInfo {
  int group, ctile, row0, row_end;
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


// Row-major [rows, K] uint8 matrix as a 2D TMA tensor map: box = 128 bytes
// of K x box_rows rows, 128-byte swizzle; rows past the end read as zero.
bool make_tmap(CUtensorMap* map, const void* base, int64_t rows, int K,
               int box_rows);

// Row-major [rows, cols] fp32 matrix as a 2D TMA tensor map for stores of
// box_rows x box_cols boxes (no swizzle).
bool make_tmap_f32(CUtensorMap* map, void* base, int64_t rows, int cols,
                   int box_rows, int box_cols);

// Streaming multiprocessors of the current device (cached).
int sm_count();

// Whether wide token tiles use the CTA-pair kernel (MOE_GEMM_CTA_PAIR=1).
bool cta_pair_enabled();

}  // namespace gemm
}  // namespace moe
