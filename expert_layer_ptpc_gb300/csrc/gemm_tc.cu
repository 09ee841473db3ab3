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
// CTA = 11 warps, persistent over a static tile sequence:
//   warp 0      TMEM allocator and MMA issuer (one lane): tcgen05.mma
//               kind::f8f6f4, M=128, N=BN, K=32 per instruction, into one of
//               two accumulator buffers
//   warps 1-4   epilogue: tcgen05.ld of its 32 TMEM lanes, PTPC dequant,
//               SwiGLU, fp32 stores (coalesced: a warp writes 32 channels)
//   warps 5-10  TMA producers, one lane each: the 64-row weight boxes and the
//               token boxes of a stage (one box per warp), into a STAGES-
//               deep ring of shared-memory stages (128-byte swizzle)
// Every wait is bounded (common.cuh): a wait that runs out raises the device
// error word, the CTA's roles stop, in-flight copies and MMAs are drained and
// the TMEM is freed before the kernel returns.
#include <cuda_fp16.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gemm_common.cuh"

namespace moe {

namespace {

using namespace gemm;

constexpr int kBM = 128;   // output channels per tile (MMA M)

template <int BN, int BMW, bool GATEUP, bool OUT16 = false, int MINB = 1>
struct Cfg {
  // BMW = output channels per tile. 128: the MMA's 128 rows are 128 channels
  // (gate/up: a second MMA for the up rows). 64: for small token tiles, a
  // tile is 64 channels so twice as many tiles spread over the SMs; gate/up
  // packs 64 gate and the matching 64 up rows into one 128-row operand.
  static constexpr bool kPacked = BMW == 64;
  // MMAs per K step: gate and up tiles, or (down, BMW = 256) two 128-channel
  // halves that share one token tile (its rows are read once per 256
  // channels instead of once per 128)
  static constexpr int kNumA = ((GATEUP && !kPacked) || BMW == 256) ? 2 : 1;
  static constexpr int kATile = kBM * kBK;                     // one 128-row operand
  static constexpr int kBTile = BN * kBK;
  static constexpr int kStage = kNumA * kATile + kBTile;
  // TMA boxes of one stage: 64-row weight boxes (gate/up: two per 128-row
  // tile, or one gate + one up when packed; down: two), then token boxes of
  // up to 64 rows. One producer warp per box.
  static constexpr int kWBoxes = GATEUP ? (kPacked ? 2 : 4) : BMW / 64;
  static constexpr int kTBoxRows = BN < 64 ? BN : 64;
  static constexpr int kTBoxes = BN / kTBoxRows;
  static constexpr int kBoxes = kWBoxes + kTBoxes;
  static_assert(kBoxes <= kMaxBoxes, "one producer warp per box");
  // MINB = 2: two CTAs share an SM, each with half the stage budget. For
  // tiles of at most 16 tokens, which stream their weights once with almost
  // no tensor work: one CTA's per-tile overhead (epilogue, tile hand-over)
  // then overlaps the other's streaming, and an SM given a second tile of a
  // launch with fewer tiles than two per SM streams both at once.
  static constexpr int kBudget = MINB == 2 ? 96 * 1024 : kStageBudget;
  static constexpr int kStages = (kBudget / kStage) > 10 ? 10 : (kBudget / kStage);
  static constexpr int kAccCols = kNumA * BN;                  // one buffer
  // two accumulator buffers (epilogue of one tile overlaps the next tile's
  // MMAs) when they fit in the 512 TMEM columns, else one
  static constexpr int kAccBufs = 2 * kAccCols <= 512 ? 2 : 1;
  static constexpr int kTmemCols = pow2_at_least(kAccBufs * kAccCols);
  static constexpr int kNumBars = 2 * kStages + 7;
  static constexpr int kXBytes = (GATEUP && kPacked) ? 64 * 16 * 4 : 0;
  // wide tiles stage each epilogue warp's 32 channels x 32 tokens of fp32
  // output in shared memory and write it with one TMA store
  static constexpr bool kStagedOut = !kPacked && BN >= 64;
  static constexpr int kOutBytes = kStagedOut ? 4 * 32 * 32 * 4 : 0;
  static constexpr int kSmemBytes = 1024 + kStages * kStage + kXBytes + kOutBytes +
                                    kNumBars * 8 + 16 + 8 * (kMaxGroups + 1) + 64;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(MINB == 1 || (MINB == 2 && 2 * (kSmemBytes + 1024) <= 233472 &&
                              2 * kTmemCols <= 512),
                "two CTAs per SM");
  static_assert(BMW == 64 || BMW == 128 || (BMW == 256 && !GATEUP && BN == 128),
                "tile width");
  static_assert(kTmemCols <= 512, "TMEM budget");
  static_assert(kStages >= 2, "pipeline depth");
  // fp16 down output with staged stores: four more epilogue warps (12-15,
  // the same TMEM lane quarters) take every other 32-token chunk; their
  // fp16 boxes fit the same staging bytes
  static constexpr bool kWideEpi = kStagedOut && OUT16;
  static constexpr int kEpiSets = kWideEpi ? 2 : 1;
  static constexpr int kThreadsT = kThreads + (kWideEpi ? 4 * 32 : 0);
};

// OUT16 (down projection only): y is written as fp16 codes with one fp32
// factor per row instead of fp32 values (see the down epilogue).
template <int BN, int BMW, bool GATEUP, bool OUT16, int MINB>
__global__ void __launch_bounds__(Cfg<BN, BMW, GATEUP, OUT16, MINB>::kThreadsT, MINB)
    grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap tm_w,
    const __grid_constant__ CUtensorMap tm_a,
    const __grid_constant__ CUtensorMap tm_out, const float* __restrict__ a_scale,
    const float* __restrict__ w_scale, const int32_t* __restrict__ offsets,
    int groups, int N, int K, float* __restrict__ out,
    __half* __restrict__ out16, float* __restrict__ row_scale,
    const float* __restrict__ w_bound, unsigned* __restrict__ err) {
  static_assert(!(OUT16 && GATEUP), "fp16 output is for the down projection");
  using C = Cfg<BN, BMW, GATEUP, OUT16, MINB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* xbuf = reinterpret_cast<float*>(smem + C::kStages * C::kStage);
  float* outstage = reinterpret_cast<float*>(smem + C::kStages * C::kStage + C::kXBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage +
                                               C::kXBytes + C::kOutBytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* prefix = reinterpret_cast<int*>(tmem_holder + 4);   // groups + 1
  // the group offsets, copied: tile decoding reads only shared memory
  int* soff = prefix + (kMaxGroups + 1);
  __shared__ int warp_tot[C::kThreadsT / 32 + 1];
  __shared__ Sched sched;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_ctiles = N / BMW;
  const int kblocks = K / kBK;

  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + C::kStages + s); };
  auto accf_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + b); };
  auto acce_bar = [&](int b) { return smem_u32(bars + 2 * C::kStages + 2 + b); };
  const uint32_t drain_bar = smem_u32(bars + 2 * C::kStages + 4);
  const uint32_t xfull_bar = smem_u32(bars + 2 * C::kStages + 5);
  const uint32_t xempty_bar = smem_u32(bars + 2 * C::kStages + 6);
  auto stage_a = [&](int s, int which) {
    return smem_u32(smem + s * C::kStage + which * C::kATile);
  };
  auto stage_b = [&](int s) {
    return smem_u32(smem + s * C::kStage + C::kNumA * C::kATile);
  };

  // ---------------- set-up ----------------
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), C::kBoxes);   // one arrival per box
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 4 * C::kEpiSets);   // one per epilogue warp
    }
    mbar_init(drain_bar, 1);
    mbar_init(xfull_bar, 64);
    mbar_init(xempty_bar, 64);
    // ring consumers: each producer, the MMA issuer, each epilogue warp
    sched_init(sched, C::kBoxes + 1 + 4 * C::kEpiSets);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_a);
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);

  // tile prefix: prefix[g] = sum_{g' < g} ceil(rows_g' / BN) * n_ctiles
  {
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
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  const int total_tiles = prefix[groups];

  // first weight row of a tile (gate rows for gate/up)
  auto weight_row = [&](const TileInfo& ti) {
    return GATEUP ? ti.group * 2 * N + ti.ctile * BMW : ti.group * N + ti.ctile * BMW;
  };

  const int box = producer_box(warp);
  if (warp == kSchedWarp) {
    // ---------------- tile scheduler ----------------
    // (touches nothing the previous kernel writes)
    if (lane == 0)
      sched_run(sched, blockIdx.x, total_tiles, 1, 0, abort_flag, err, [&](int t) {
        return decode_tile(t, prefix, groups, soff, BN);
      });
  } else if (box >= 0) {
    // ---------------- TMA producers: box `box` of every stage ----------------
    const bool weight_box = box < C::kWBoxes;
    if (lane == 0 && box < C::kBoxes) {
      // small token tiles read each weight tile once: stream it past L2;
      // wider tiles share a weight tile between neighbouring token tiles
      const uint64_t pol = !weight_box ? l2_policy_evict_last()
                           : BN <= 32  ? l2_policy_evict_first()
                                       : l2_policy_evict_normal();
      const uint32_t bytes =
          weight_box ? 64u * kBK : (uint32_t)(C::kTBoxRows * kBK);
      // weight row of this producer's box in tile ti, and its stage offset
      auto box_row = [&](const TileInfo& ti, int& off) {
        const int wrow = weight_row(ti);
        if (GATEUP && !C::kPacked) {   // boxes 0,1: gate halves; 2,3: up halves
          off = (box >= 2 ? C::kATile : 0) + (box & 1) * 64 * kBK;
          return wrow + (box >= 2 ? N : 0) + (box & 1) * 64;
        } else if (GATEUP) {           // packed: 64 gate rows, 64 up rows
          off = box * 64 * kBK;
          return wrow + (box == 1 ? N : 0);
        }
        // down: 64-row quarters (halves) of the tile
        off = (box >> 1) * C::kATile + (box & 1) * 64 * kBK;
        return wrow + box * 64;
      };
      auto issue = [&](int s, int kb, const TileInfo& ti) {
        const int x = kb * kBK;
        if (weight_box) {
          int off;
          const int row = box_row(ti, off);
          tma_load_2d(stage_a(s, 0) + off, &tm_w, x, row, full_bar(s), pol);
        } else {
          const int t = box - C::kWBoxes;
          tma_load_2d(stage_b(s) + t * C::kTBoxRows * kBK, &tm_a, x,
                      ti.row0 + t * C::kTBoxRows, full_bar(s), pol);
        }
      };
      int last_phase[C::kStages];
#pragma unroll
      for (int i = 0; i < C::kStages; ++i) last_phase[i] = -1;
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      // The weights and the tile map (offsets come from the permutation, two
      // launches back) do not depend on the previous kernel: the weight
      // producers fill the first stages before waiting for it.
      const int first = blockIdx.x;   // the scheduler hands this tile out first
      int npre = 0;
      TileInfo t0{};
      if (weight_box && first < total_tiles) {
        t0 = decode_tile(first, prefix, groups, soff, BN);
        npre = kblocks < C::kStages ? kblocks : C::kStages;
        for (int kb = 0; kb < npre; ++kb) {   // fresh ring: stage kb, phase 0
          mbar_arrive_expect_tx(full_bar(kb), bytes);
          issue(kb, kb, t0);
#pragma unroll
          for (int i = 0; i < C::kStages; ++i)
            if (i == kb) last_phase[i] = 0;
        }
        s = npre % C::kStages;
        ph = npre == C::kStages ? 1u : 0u;
      }
      pdl_wait();
      pdl_launch_dependents();
      TileCursor cur;
      for (bool first_tile = true; ok; first_tile = false) {
        TileInfo ti;
        const int tile = next_tile_thread(sched, cur, box == 0, abort_flag, err,
                                          kErrTimeoutProducer, ti);
        if (tile < 0) break;
        const bool pre = first_tile && npre > 0 && tile == first;
        for (int kb = pre ? npre : 0; kb < kblocks; ++kb) {
          if (!mbar_wait_bounded(empty_bar(s), ph ^ 1, abort_flag, err,
                                 kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(s), bytes);
          issue(s, kb, ti);
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
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    pdl_launch_dependents();
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      TileCursor cur;
      for (; ok; ++it) {
        TileInfo ti;
        const int tile = next_tile_thread(sched, cur, false, abort_flag, err,
                                          kErrTimeoutMma, ti);
        if (tile < 0) break;
        const int ab = it % C::kAccBufs;
        const uint32_t acc_ph = (uint32_t)(it / C::kAccBufs) & 1u;
        if (!mbar_wait_bounded(acce_bar(ab), acc_ph ^ 1, abort_flag, err,
                               kErrTimeoutMma)) break;
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + (uint32_t)(ab * C::kAccCols);
        const uint32_t d1 = d0 + BN;
        // An expert's last token tile is usually partial: narrow the MMA to
        // the smallest width (halving BN, not below 32) that covers its rows.
        int n_mma = BN;
        {
          const int nvalid = ti.row_end - ti.row0;
          while (n_mma >= 64 && n_mma / 2 >= nvalid) n_mma /= 2;
        }
        const uint32_t idesc = idesc_e4m3_f32(kBM, n_mma);
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
            if (C::kNumA == 2) {
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
    const int m = q * 32 + lane;          // accumulator row (lane) of this thread
    int it = 0;
    uint32_t xc = 0;                      // gate/up exchanges so far (packed)
    // Output of 32 tokens (v[j] = token n0 + j) for this warp's 32 channels
    // ch0 + lane. A full 32-token box inside the expert goes through shared
    // memory and one TMA store; a partial box at the expert's end is stored
    // directly, so rows of the next expert are never written.
    // [token][channel]; epilogue warp index e = 0..3 (warps 1-4), 4..7 (12-15)
    const int e_idx = warp < kSchedWarp ? warp - kEpiWarp0 : warp - kSchedWarp + 3;
    const int eset = warp < kSchedWarp ? 0 : 1;
    float* obuf = OUT16 ? reinterpret_cast<float*>(reinterpret_cast<__half*>(outstage) +
                                                   e_idx * 32 * 32)
                        : outstage + e_idx * 32 * 32;
    auto emit = [&](const TileInfo& ti, int n0, int nvalid, int ch0,
                    const float (&v)[32]) {
      if (n0 + 32 <= nvalid) {
        if (lane == 0) bulk_wait_read_all();   // the previous box has left obuf
        __syncwarp();
        if constexpr (OUT16) {
          __half* o16 = reinterpret_cast<__half*>(obuf);
#pragma unroll
          for (int j = 0; j < 32; ++j) o16[j * 32 + lane] = __float2half_rn(v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) obuf[j * 32 + lane] = v[j];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tm_out, ch0, ti.row0 + n0, smem_u32(obuf));
          bulk_commit();
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (n0 + j < nvalid) {
            const int64_t o = (int64_t)(ti.row0 + n0 + j) * N + ch0 + lane;
            if constexpr (OUT16) out16[o] = __float2half_rn(v[j]);
            else out[o] = v[j];
          }
        }
      }
    };
    bool ok = true;
    TileCursor cur;
    for (; ok; ++it) {
      TileInfo ti;
      const int tile =
          next_tile_warp(sched, cur, abort_flag, err, kErrTimeoutEpilogue, ti);
      if (tile < 0) break;
      const int ab = it % C::kAccBufs;
      const uint32_t acc_ph = (uint32_t)(it / C::kAccBufs) & 1u;
      const int nvalid = min(BN, ti.row_end - ti.row0);
      // What does not depend on the accumulators is read (and the rows'
      // factors written) while the MMAs finish, off the epilogue's path.
      // fp16 output: y16 = acc * s_d * rho with rho from the expert's scale
      // bound, so |y16| <= 60000 whatever the data; the row's factor
      // a_scale / rho (written once, by the tile of the first channels)
      // turns the codes back into y.
      float rho = 1.0f;
      if constexpr (OUT16) {
        rho = fp16_rho(w_bound[ti.group], K);
        if (ti.ctile == 0) {
          for (int r = (warp - kEpiWarp0) * 32 + lane; r < nvalid; r += 128)
            row_scale[ti.row0 + r] = __fdiv_rn(a_scale[ti.row0 + r], rho);
        }
      }
      // down projection, staged output: each 128-channel half's channel scale
      float sw_half[C::kNumA];
#pragma unroll
      for (int which = 0; which < C::kNumA; ++which)
        sw_half[which] = !GATEUP && C::kStagedOut
                             ? w_scale[(int64_t)ti.group * N + ti.ctile * BMW +
                                       which * 128 + q * 32 + lane]
                             : 0.f;
      if (!warp_wait(accf_bar(ab), acc_ph, abort_flag, err, kErrTimeoutEpilogue))
        break;
      tc_fence_after_sync();
      const uint32_t taddr =
          tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * C::kAccCols);
      if (GATEUP && C::kPacked) {
        // lanes 0-63: gate of channels ctile*64 + m; lanes 64-127: up of the
        // same channels. Up values pass to the gate threads through xbuf.
        const bool is_gate = q < 2;
        const int ch = ti.ctile * 64 + (is_gate ? m : m - 64);
        const float swg = w_scale[(int64_t)ti.group * 2 * N + ch];
        const float swu = w_scale[(int64_t)ti.group * 2 * N + N + ch];
        for (int n0 = 0; ok && n0 < nvalid; n0 += 16, ++xc) {
          float a[16];
          tmem_ld_x16(taddr + n0, a);
          tmem_ld_wait();
          if (!is_gate) {
            if (!warp_wait(xempty_bar, (xc & 1u) ^ 1u, abort_flag, err,
                           kErrTimeoutEpilogue)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) xbuf[j * 64 + (m - 64)] = a[j];
            mbar_arrive(xfull_bar);
          } else {
            if (!warp_wait(xfull_bar, xc & 1u, abort_flag, err,
                           kErrTimeoutEpilogue)) {
              ok = false;
              break;
            }
            float u[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) u[j] = xbuf[j * 64 + m];
            mbar_arrive(xempty_bar);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (n0 + j < nvalid) {
                const int row = ti.row0 + n0 + j;
                const float sx = a_scale[row];
                const float g = a[j] * sx * swg;
                const float uu = u[j] * sx * swu;
                out[(int64_t)row * N + ch] = __fdividef(g * uu, 1.0f + __expf(-g));
              }
            }
          }
        }
      } else if (GATEUP && C::kStagedOut) {
        const int ch0 = ti.ctile * kBM + q * 32;
        const float swg = w_scale[(int64_t)ti.group * 2 * N + ch0 + lane];
        const float swu = w_scale[(int64_t)ti.group * 2 * N + N + ch0 + lane];
        for (int n0 = 0; n0 < nvalid; n0 += 32) {
          float ag[32], au[32], v[32];
          tmem_ld_x16(taddr + n0, *reinterpret_cast<float(*)[16]>(&ag[0]));
          tmem_ld_x16(taddr + n0 + 16, *reinterpret_cast<float(*)[16]>(&ag[16]));
          tmem_ld_x16(taddr + BN + n0, *reinterpret_cast<float(*)[16]>(&au[0]));
          tmem_ld_x16(taddr + BN + n0 + 16, *reinterpret_cast<float(*)[16]>(&au[16]));
          tmem_ld_wait();
          // one coalesced load of the 32 token scales, broadcast by shuffle
          const float sx_l = n0 + lane < nvalid ? a_scale[ti.row0 + n0 + lane] : 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float sx = __shfl_sync(0xffffffffu, sx_l, j);
            const float g = ag[j] * sx * swg;
            const float u = au[j] * sx * swu;
            v[j] = __fdividef(g * u, 1.0f + __expf(-g));
          }
          emit(ti, n0, nvalid, ch0, v);
        }
      } else if (C::kStagedOut) {   // down projection, wide tiles
       for (int which = 0; which < C::kNumA; ++which) {   // 128-channel halves
        const int ch0 = ti.ctile * BMW + which * 128 + q * 32;
        const uint32_t ta = taddr + (uint32_t)(which * BN);
        const float sw = sw_half[which];
        const float swr = sw * rho;
        for (int n0 = 32 * eset; n0 < nvalid; n0 += 32 * C::kEpiSets) {
          float acc[32], v[32];
          tmem_ld_x16(ta + n0, *reinterpret_cast<float(*)[16]>(&acc[0]));
          tmem_ld_x16(ta + n0 + 16, *reinterpret_cast<float(*)[16]>(&acc[16]));
          tmem_ld_wait();
          if constexpr (OUT16) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = acc[j] * swr;
          } else {
            const float sx_l = n0 + lane < nvalid ? a_scale[ti.row0 + n0 + lane] : 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = acc[j] * __shfl_sync(0xffffffffu, sx_l, j) * sw;
          }
          emit(ti, n0, nvalid, ch0, v);
        }
       }
      } else if (GATEUP) {
        const int ch = ti.ctile * kBM + m;
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
              out[(int64_t)row * N + ch] = __fdividef(g * u, 1.0f + __expf(-g));
            }
          }
        }
      } else if (m < BMW) {   // down projection (packed: lanes 0-63 only)
        const int ch = ti.ctile * BMW + m;
        const float sw = w_scale[(int64_t)ti.group * N + ch];
        const float swr = sw * rho;
        for (int n0 = 0; n0 < nvalid; n0 += 16) {
          float acc[16];
          tmem_ld_x16(taddr + n0, acc);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (n0 + j < nvalid) {
              const int row = ti.row0 + n0 + j;
              if constexpr (OUT16)
                out16[(int64_t)row * N + ch] = __float2half_rn(acc[j] * swr);
              else
                out[(int64_t)row * N + ch] = acc[j] * a_scale[row] * sw;
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce_bar(ab));
    }
    // this warp's output stores are complete before the kernel ends
    if (C::kStagedOut && lane == 0) bulk_wait_all();
  }

  // ---------------- tear-down ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// out (fp32) or, with OUT16, out16 + row_scale given w_bound (down only).
template <int BN, int BMW, bool GATEUP, bool OUT16 = false, int MINB = 1>
int run(const uint8_t* A, const float* a_scale, int64_t a_rows, const uint8_t* W,
        const float* w_scale, const int32_t* offsets, int groups, int N, int K,
        float* out, cudaStream_t stream, bool pdl, __half* out16 = nullptr,
        float* row_scale = nullptr, const float* w_bound = nullptr) {
  using C = Cfg<BN, BMW, GATEUP, OUT16, MINB>;
  CUtensorMap tm_w, tm_a;
  const int64_t w_rows = (int64_t)groups * (GATEUP ? 2 : 1) * N;
  if (!make_tmap(&tm_w, W, w_rows, K, 64)) return -3;
  if (!make_tmap(&tm_a, A, a_rows, K, C::kTBoxRows)) return -3;
  CUtensorMap tm_out{};
  if (C::kStagedOut) {
    const bool made = OUT16 ? make_tmap_out(&tm_out, out16, a_rows, N, 32, 32, 2)
                            : make_tmap_out(&tm_out, out, a_rows, N, 32, 32, 4);
    if (!made) return -3;
  }
  auto kern = grouped_gemm_kernel<BN, BMW, GATEUP, OUT16, MINB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return -3;
  // one CTA per possible tile; the ones that run first take the rest over
  // (cluster launch control, see the scheduler)
  const int64_t upper = token_tiles_upper(a_rows, groups, BN) * (int64_t)(N / BMW);
  if (upper <= 0) return 0;
  if (upper > INT32_MAX) return -2;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)upper);
  cfg.blockDim = dim3(C::kThreadsT);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, tm_w, tm_a, tm_out, a_scale, w_scale, offsets,
                         groups, N, K, out, out16, row_scale, w_bound,
                         device_error_word());
  return e == cudaSuccess ? 0 : -3;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

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

}  // namespace

namespace gemm {

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

bool make_tmap_gateup_interleaved(CUtensorMap* map, const void* W, int groups, int N,
                                  int K) {
  auto fn = encode_fn();
  if (fn == nullptr || N % 64 != 0) return false;
  // dims (innermost first): K bytes, 16 rows of a channel block, gate / up,
  // channel blocks, experts; a box walks them in that order, so its 128
  // rows arrive as [block][gate, up][16 rows]
  const cuuint64_t dims[5] = {(cuuint64_t)K, 16, 2, (cuuint64_t)(N / 16),
                              (cuuint64_t)groups};
  const cuuint64_t strides[4] = {(cuuint64_t)K, (cuuint64_t)N * K, (cuuint64_t)16 * K,
                                 (cuuint64_t)2 * N * K};
  const cuuint32_t box[5] = {(cuuint32_t)kBK, 16, 2, 4, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(W), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_out(CUtensorMap* map, void* base, int64_t rows, int cols,
                   int box_rows, int box_cols, int elem_bytes) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType type =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  return fn(map, type, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static std::atomic<int> cached[64];   // 0: not asked yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int cta_pair_mode() {
  static const int mode = [] {
    const char* v = std::getenv("MOE_GEMM_CTA_PAIR");
    if (v == nullptr || v[0] == '\0') return -1;
    return v[0] == '1' ? 1 : v[0] == '0' ? 0 : -1;
  }();
  return mode;
}

int wide_tiles_mode() {
  static const int mode = [] {
    const char* v = std::getenv("MOE_GEMM_WIDE");
    if (v == nullptr || v[0] == '\0') return -1;
    return v[0] == '1' ? 1 : v[0] == '0' ? 0 : -1;
  }();
  return mode;
}

int pair_bn_mode() {
  static const int bn = [] {
    const char* v = std::getenv("MOE_GEMM_PAIR_BN");
    const int b = v != nullptr ? std::atoi(v) : 0;
    return b == 128 || b == 192 || b == 256 ? b : 0;
  }();
  return bn;
}

int pair_k_atoms() {
  static const int ks = [] {
    const char* v = std::getenv("MOE_GEMM_KATOMS");
    return (v != nullptr && v[0] == '1') ? 1 : 2;
  }();
  return ks;
}

int balanced_tiles() {
  static const int mode = [] {
    const char* v = std::getenv("MOE_GEMM_BALANCED");
    return (v != nullptr && v[0] == '0') ? 0 : 1;
  }();
  return mode;
}

int down_pair_mode() {
  static const int mode = [] {
    const char* v = std::getenv("MOE_GEMM_DOWN_PAIR");
    if (v == nullptr || v[0] == '\0') return -1;
    return v[0] == '1' ? 1 : v[0] == '0' ? 0 : -1;
  }();
  return mode;
}

}  // namespace gemm

int launch_grouped_gemm(int kind, const uint8_t* A, const float* a_scale,
                        int64_t a_rows, const uint8_t* W, const float* w_scale,
                        const int32_t* offsets, int groups, int N, int K,
                        float* out, int rows_hint, cudaStream_t stream,
                        bool pdl) {
  if (a_rows == 0 || groups == 0) return 0;
  const int64_t avg = rows_hint > 0 ? rows_hint : std::max<int64_t>(1, a_rows / groups);
  // Wide token tiles of the gate/up projection run one M = 256 MMA over a
  // pair of SMs (each loads half of the token tile, one N = 256 instruction
  // per K step instead of two N = 128 ones). On GB300 that wins from about
  // 256 rows per expert on; the down projection, bound by its fp32 output
  // writes, stays on the single-CTA kernel. MOE_GEMM_CTA_PAIR=1 / =0 forces
  // the pair kernel on (every shape with more than 64 rows per expert) / off.
  const int pair_mode = cta_pair_mode();
  const bool pair = pair_mode == 1   ? avg > 64
                    : pair_mode == 0 ? false
                                     : kind == 0 && avg >= 256;
  // From 256 to 384 rows per expert an expert takes two balanced tiles of at
  // most 192 tokens. With one-atom stages their 28 KB stage left room for
  // seven in the ring instead of six 32 KB ones (uniform 320 rows per expert
  // 1.156 -> 1.105 ms, T=16384 gate/up 1.289 -> 1.257 ms); with two-atom
  // stages (K a multiple of 256) the ring holds three of 56 KB.
  // Tiles of up to 512 tokens (two MMAs per K step, one accumulator buffer)
  // move 25-30% fewer operand bytes per FLOP, but their epilogue cannot
  // overlap the next tile's MMAs: on GB300 they tie at 320 rows per expert
  // (T=16384 gate/up 1.384 ms either way) and lose at 512 (prefill 0.634 ->
  // 0.721 ms). MOE_GEMM_WIDE=1 turns them on above 256 rows per expert.
  const bool wide = kind == 0 && avg > 256 && wide_tiles_mode() == 1;
  if (pair && grouped_gemm_pair_supported(kind, N))
    return launch_grouped_gemm_pair(kind, A, a_scale, a_rows, W, w_scale, offsets,
                                    groups, N, K, out,
                                    wide              ? 512
                                    : pair_bn_mode()  ? pair_bn_mode()
                                    : avg <= 128      ? 128
                                    : avg <= 256      ? 256
                                    : avg <= 384      ? 192
                                                      : 256,
                                    stream, pdl);
  if (kind == 0) {
    if (avg <= 16) {
      // fewer tiles than two per SM: two CTAs an SM, so no SM streams a
      // second tile alone after the others are done
      if (token_tiles_upper(a_rows, groups, 16) * (N / 64) <= 2 * (int64_t)sm_count())
        return run<16, 64, true, false, 2>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
      return run<16, 64, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
    }
    if (avg <= 32) return run<32, 64, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
    if (avg <= 64) return run<64, 128, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
    return run<128, 128, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  }
  // 16-token down tiles (short K, per-tile overhead) always run two CTAs an SM
  if (avg <= 16) return run<16, 128, false, false, 2>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  if (avg <= 32) return run<32, 128, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  if (avg <= 64) return run<64, 128, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  // 128-token tiles of 256 channels read each token tile once per 256
  // channels: the SMs' operand feed, not HBM, bounded the 128-channel tiles
  if (avg <= 128 && N % 256 == 0) return run<128, 256, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  if (avg <= 128) return run<128, 128, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
  return run<256, 128, false>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K, out, stream, pdl);
}

int launch_grouped_gemm_down_f16(const uint8_t* A, const float* a_scale,
                                 int64_t a_rows, const uint8_t* W,
                                 const float* w_scale, const float* w_bound,
                                 const int32_t* offsets, int groups, int N, int K,
                                 uint16_t* y16, float* row_scale, int rows_hint,
                                 cudaStream_t stream, bool pdl) {
  if (a_rows == 0 || groups == 0) return 0;
  const int64_t avg = rows_hint > 0 ? rows_hint : std::max<int64_t>(1, a_rows / groups);
  // From 256 rows per expert on, token tiles of up to 256 rows (balanced
  // widths) run on a CTA pair: one M = 256 MMA of 256 channels per K step,
  // each SM loading 128 weight rows and half of the token tile, so a weight
  // tile is read once per 256 tokens instead of once per 128 (T=16384, 320
  // rows per expert: 0.860 -> 0.773 ms; prefill 0.399 -> 0.334 ms). At 80
  // rows per expert (T=4096) the single CTA's 128-token tiles stay ahead
  // (0.386 vs 0.413 ms). MOE_GEMM_DOWN_PAIR=1 / =0 (or MOE_GEMM_CTA_PAIR=1 /
  // =0) forces the pair (above 64 rows per expert) or the single CTA.
  const int dm = down_pair_mode() >= 0 ? down_pair_mode() : cta_pair_mode();
  const bool pair = dm == 1 ? avg > 64 : dm == 0 ? false : avg >= 256;
  if (pair && grouped_gemm_pair_supported(1, N))
    return launch_grouped_gemm_pair_down_f16(
        A, a_scale, a_rows, W, w_scale, w_bound, offsets, groups, N, K, y16, row_scale,
        pair_bn_mode() ? pair_bn_mode() : avg <= 128 ? 128 : 256, stream, pdl);
  __half* o = reinterpret_cast<__half*>(y16);
#define MOE_DOWN16(bn, minb)                                                             \
  return run<bn, 128, false, true, minb>(A, a_scale, a_rows, W, w_scale, offsets, groups, \
                                         N, K, nullptr, stream, pdl, o, row_scale, w_bound)
  if (avg <= 16) MOE_DOWN16(16, 2);
  if (avg <= 32) MOE_DOWN16(32, 1);
  if (avg <= 64) MOE_DOWN16(64, 1);
  // 128 tokens x 256 channels up to 384 rows per expert: at 320 (T=16384,
  // 512 experts, top-10) they beat 256 x 128 tiles, 0.970 -> 0.934 ms
  if (avg <= 384 && N % 256 == 0)
    return run<128, 256, false, true>(A, a_scale, a_rows, W, w_scale, offsets, groups, N, K,
                                      nullptr, stream, pdl, o, row_scale, w_bound);
  if (avg <= 128) MOE_DOWN16(128, 1);
  MOE_DOWN16(256, 1);
#undef MOE_DOWN16
}

}  // namespace moe
