// Expert histogram, prefix sum and stable permutation of the flat
// (token, slot) pairs into expert-contiguous rows.
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x", SparseCore permute
// paragraph: token rows are gathered by routing index into one contiguous
// buffer without padded intermediates. Here the gather itself is fused into
// the quantiser (quant.cu); this file produces the row map.
//
// Order: a stable counting sort. The flat indices are cut into chunks of
// kChunk entries and each chunk into one sub-chunk per warp. Within a warp,
// 32 consecutive entries are ranked with __match_any_sync (lanes that share
// an expert, lower lanes first); warps and chunks are ordered by prefix sums
// of their per-expert counts. The result does not depend on scheduling.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
// Flat entries per block: up to kSmallChunk entries are sorted by one block
// (one launch); larger inputs take three launches over kChunk-entry chunks,
// small enough that every chunk's serial work is short and the chunks
// spread over many SMs.
constexpr int kSmallChunk = 8192;
constexpr int kChunk = 2048;

// Exclusive prefix sum of vals[0..n) in shared memory (n <= 2 * kThreads),
// in place; returns the total. All threads of the block must call it.
__device__ int block_exclusive_scan(int* vals, int n, int* warp_tot) {
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  // each thread owns two consecutive entries
  const int i0 = 2 * tid, i1 = 2 * tid + 1;
  const int a = i0 < n ? vals[i0] : 0;
  const int b = i1 < n ? vals[i1] : 0;
  int s = a + b;
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kWarps) warp_tot[lane] = wi - w;   // exclusive warp offsets
    if (lane == kWarps - 1) warp_tot[kWarps] = wi;  // block total
  }
  __syncthreads();
  const int excl = warp_tot[warp] + incl - s;
  if (i0 < n) vals[i0] = excl;
  if (i1 < n) vals[i1] = excl + a;
  const int total = warp_tot[kWarps];
  __syncthreads();
  return total;
}

// A chunk of PL * kThreads entries: warp w owns the sub-chunk of PL * 32
// entries starting at PL * 32 w, lane l holds its entries 32 i + l.

// Load this warp's sub-chunk: lane holds entries begin + 32 i + lane
// (i < PL); -1 past the end. All loads are issued before any is used.
template <int PL>
__device__ __forceinline__ void load_warp_ids(const int32_t* __restrict__ ids,
                                              int64_t f0, int64_t R, int E, int (&e)[PL],
                                              unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t begin = f0 + (int64_t)warp * (PL * 32);
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int64_t f = begin + 32 * i + lane;
    e[i] = f < R ? ids[f] : -1;
#ifdef MOE_CHECK
    if (f < R && !MOE_CHECKED(e[i] >= 0 && e[i] < E, err)) e[i] = -1;
#endif
  }
}

// Per-warp expert histograms of one chunk: whist[w * E + e].
template <int PL>
__device__ void chunk_warp_histograms(const int (&e)[PL], int E, int* whist) {
  for (int i = threadIdx.x; i < kWarps * E; i += kThreads) whist[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < PL; ++i)
    if (e[i] >= 0) atomicAdd(&whist[warp * E + e[i]], 1);
  __syncthreads();
}

// Turn per-warp counts into per-warp starting rows: for every expert e,
// whist[w][e] <- base[e] + sum_{w' < w} count_{w'}[e].
__device__ void warp_bases(const int* base, int E, int* whist) {
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int run = base[e];
    for (int w = 0; w < kWarps; ++w) {
      const int c = whist[w * E + e];
      whist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
}

// Stable scatter of one chunk given per-warp starting rows. 32 consecutive
// entries at a time: lanes with the same expert are ranked by lane order.
template <int PL>
__device__ void chunk_scatter(const int (&e)[PL], int64_t f0, int64_t R, int E,
                              int* whist, int32_t* __restrict__ s2f,
                              int32_t* __restrict__ f2s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* base = whist + warp * E;
  const int64_t begin = f0 + (int64_t)warp * (PL * 32);
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    if (begin + 32 * i >= R) break;               // warp-uniform
    const int64_t f = begin + 32 * i + lane;
    const bool valid = e[i] >= 0;
    const int key = valid ? e[i] : -1 - lane;     // distinct sentinels
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    int pos = 0;
    if (valid) pos = base[key] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (valid) {
      s2f[pos] = (int32_t)f;
      f2s[f] = pos;
      if (lane == __ffs(peers) - 1) base[key] += __popc(peers);
    }
    __syncwarp();
  }
}

__device__ void write_extra_group(int E, int total, int extra,
                                  int32_t* counts, int32_t* offsets) {
  if (extra >= 0 && threadIdx.x == 0) {
    counts[E] = extra;
    offsets[E + 1] = total + extra;
  }
}

// R <= kSmallChunk: everything in one block.
__global__ void __launch_bounds__(kThreads) permute_small_kernel(
    const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ s2f,
    int32_t* __restrict__ f2s, int extra, unsigned* __restrict__ err) {
  extern __shared__ int smem[];
  int* whist = smem;                       // kWarps * E
  int* scan = whist + kWarps * E;          // E + 1
  int* warp_tot = scan + E + 1;            // kWarps + 1
  pdl_wait();
  pdl_launch_dependents();
  constexpr int PL = kSmallChunk / kThreads;
  int mine[PL];
  load_warp_ids<PL>(ids, 0, R, E, mine, err);
  chunk_warp_histograms<PL>(mine, E, whist);
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int c = 0;
    for (int w = 0; w < kWarps; ++w) c += whist[w * E + e];
    scan[e] = c;
    counts[e] = c;
  }
  __syncthreads();
  const int total = block_exclusive_scan(scan, E, warp_tot);
  for (int e = threadIdx.x; e < E; e += kThreads) offsets[e] = scan[e];
  if (threadIdx.x == 0) offsets[E] = total;
  write_extra_group(E, total, extra, counts, offsets);
  warp_bases(scan, E, whist);
  chunk_scatter<PL>(mine, 0, R, E, whist, s2f, f2s);
}

// R > kSmallChunk, pass 1: per-chunk expert counts -> hist[c * E + e].
__global__ void __launch_bounds__(kThreads) permute_hist_kernel(
    const int32_t* __restrict__ ids, int64_t R, int E, int* __restrict__ hist,
    unsigned* __restrict__ err) {
  extern __shared__ int smem[];
  pdl_wait();
  pdl_launch_dependents();
  const int64_t f0 = (int64_t)blockIdx.x * kChunk;
  for (int i = threadIdx.x; i < E; i += kThreads) smem[i] = 0;
  // every load in flight before the first atomic
  constexpr int PL = kChunk / kThreads;
  int e[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int64_t f = f0 + threadIdx.x + (int64_t)i * kThreads;
    e[i] = f < R ? ids[f] : -1;
#ifdef MOE_CHECK
    if (f < R && !MOE_CHECKED(e[i] >= 0 && e[i] < E, err)) e[i] = -1;
#endif
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < PL; ++i)
    if (e[i] >= 0) atomicAdd(&smem[e[i]], 1);
  __syncthreads();
  for (int i = threadIdx.x; i < E; i += kThreads)
    hist[(int64_t)blockIdx.x * E + i] = smem[i];
}

// Pass 2 (one block): counts, offsets, and every chunk's starting row per
// expert, written over hist.
__global__ void __launch_bounds__(kThreads) permute_scan_kernel(
    int nchunks, int E, int* __restrict__ hist, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int extra) {
  extern __shared__ int smem[];
  int* scan = smem;              // E + 1
  int* warp_tot = scan + E + 1;  // kWarps + 1
  pdl_wait();
  pdl_launch_dependents();
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int c = 0;
    for (int ch = 0; ch < nchunks; ++ch) c += hist[(int64_t)ch * E + e];
    scan[e] = c;
    counts[e] = c;
  }
  __syncthreads();
  const int total = block_exclusive_scan(scan, E, warp_tot);
  for (int e = threadIdx.x; e < E; e += kThreads) {
    offsets[e] = scan[e];
    int run = scan[e];
    for (int ch = 0; ch < nchunks; ++ch) {
      const int c = hist[(int64_t)ch * E + e];
      hist[(int64_t)ch * E + e] = run;
      run += c;
    }
  }
  if (threadIdx.x == 0) offsets[E] = total;
  write_extra_group(E, total, extra, counts, offsets);
}

// Pass 3: stable scatter of each chunk from its starting rows.
__global__ void __launch_bounds__(kThreads) permute_scatter_kernel(
    const int32_t* __restrict__ ids, int64_t R, int E,
    const int* __restrict__ hist, int32_t* __restrict__ s2f,
    int32_t* __restrict__ f2s, unsigned* __restrict__ err) {
  extern __shared__ int smem[];
  int* whist = smem;                  // kWarps * E
  int* base = whist + kWarps * E;     // E
  pdl_wait();
  pdl_launch_dependents();
  const int64_t f0 = (int64_t)blockIdx.x * kChunk;
  for (int e = threadIdx.x; e < E; e += kThreads)
    base[e] = hist[(int64_t)blockIdx.x * E + e];
  constexpr int PL = kChunk / kThreads;
  int mine[PL];
  load_warp_ids<PL>(ids, f0, R, E, mine, err);
  chunk_warp_histograms<PL>(mine, E, whist);
  warp_bases(base, E, whist);
  chunk_scatter<PL>(mine, f0, R, E, whist, s2f, f2s);
}

}  // namespace

size_t permute_ws_bytes(int64_t R, int E) {
  if (R <= kSmallChunk) return 0;
  const int64_t nchunks = (R + kChunk - 1) / kChunk;
  return (size_t)(nchunks * E * sizeof(int));
}

cudaError_t launch_permute(const int32_t* ids, int64_t R, int E,
                           int32_t* counts, int32_t* offsets, int32_t* s2f,
                           int32_t* f2s, int extra_group_rows, void* ws,
                           cudaStream_t stream, bool pdl) {
  if (R <= kSmallChunk) {
    const size_t smem = (size_t)(kWarps * E + E + 1 + kWarps + 1) * sizeof(int);
    cudaError_t err = cudaFuncSetAttribute(
        permute_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(pdl, dim3(1), dim3(kThreads), smem, stream,
                         permute_small_kernel, ids, (int)R, E, counts, offsets,
                         s2f, f2s, extra_group_rows, device_error_word());
  }
  const int nchunks = (int)((R + kChunk - 1) / kChunk);
  int* hist = static_cast<int*>(ws);
  cudaError_t err = launch_kernel(pdl, dim3(nchunks), dim3(kThreads),
                                  E * sizeof(int), stream, permute_hist_kernel,
                                  ids, R, E, hist, device_error_word());
  if (err != cudaSuccess) return err;
  const size_t smem_scan = (size_t)(E + 1 + kWarps + 1) * sizeof(int);
  err = launch_kernel(pdl, dim3(1), dim3(kThreads), smem_scan, stream,
                      permute_scan_kernel, nchunks, E, hist, counts, offsets,
                      extra_group_rows);
  if (err != cudaSuccess) return err;
  const size_t smem_sc = (size_t)(kWarps * E + E) * sizeof(int);
  err = cudaFuncSetAttribute(permute_scatter_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_sc);
  if (err != cudaSuccess) return err;
  return launch_kernel(pdl, dim3(nchunks), dim3(kThreads), smem_sc, stream,
                       permute_scatter_kernel, ids, R, E, (const int*)hist, s2f,
                       f2s, device_error_word());
}

}  // namespace moe
