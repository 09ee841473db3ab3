// Router projection on the tensor cores with the top-k selection and the
// softmax fused into its epilogue.
//
// "Optimizing Qwen 3.5 397B MoE on Ironwood TPU7x" (Google Developers Blog),
// closing roadmap paragraph: the routing logits are computed on the matrix
// unit and handed to the vector unit for top_k, a serialisation the authors
// plan to remove by fusing the two. Here one kernel does both: a CTA takes
// 128 tokens, multiplies them by every expert's router row with
// tcgen05.mma.kind::f16 (bf16 operands, fp32 accumulators in TMEM: lane =
// token, column = expert), and then each epilogue thread scans its token's
// logits straight out of TMEM. It keeps a running top-k (larger value first,
// equal values to the lower expert index, the selection rule of route.cu) and
// the softmax sums, and writes only the k ids and weights.
//
//   logits[t, e] = sum_d x[t, d] * W_r[e, d]     (fp32 accumulation)
//   ids[t, :]    = the k largest logits of row t, in decreasing order
//   w[t, j]      = exp(l_j - l_0) / sum_{i<k} exp(l_i - l_0)    (renormalize)
//                  exp(l_j - l_0) / sum_{e<E} exp(l_e - l_0)     (otherwise)
//
// The accumulation order of the tensor cores is not an exact fp64 sum, so
// the logits here are the fp32 GEMM result, not moe_router_logits' exactly
// rounded ones. The selection on them is exact.
//
// Roles: warp 0 allocates TMEM and issues the MMAs (one thread); warps 4-7
// are TMA producers, which split the boxes of every stage between them (the
// token rows and the router matrix, in boxes of at most kRBoxRows rows: a
// single issuing thread caps an SM's feed far below the MMA rate); warps 0-3
// read the accumulators (warp w reads TMEM lanes 32w..32w+31). Every wait is
// bounded.
//
// The projection streams T x D activations and E x D router weights through
// few tiles, so a grid of one CTA per 128 tokens leaves most SMs idle. A
// cluster of C CTAs therefore splits K: each CTA accumulates its D/C slice,
// parks its partial logits in shared memory, and each rank sums the C
// partials of its own share of the tile's rows in rank order (a fixed
// summation order, over distributed shared memory) and selects on them, one
// warp per token.
#include <math.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "gemm_common.cuh"
#include "topk.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kRProd0 = 4;               // first producer warp
constexpr int kRProds = 4;               // producer warps
constexpr int kRThreads = 32 * (kRProd0 + kRProds);
constexpr int kRWarps = kRThreads / 32;
constexpr int kRBoxRows = 64;            // rows per TMA box (tokens and router matrix)
constexpr int kRBK = 64;                 // bf16 elements of K per stage (128 bytes),
                                         // 32 (64 bytes) for the widest expert tiles
constexpr int kRTile = 128;              // tokens per tile (MMA M)
constexpr int kRMaxN = 512;              // expert columns (two N = 256 MMAs)
constexpr int kRMaxK = 16;               // top-k kept in registers (KT <= 16)
constexpr int kRMaxCluster = 16;

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32
// accumulator, both K-major: bits 4-5 D format (1 = f32), 7-9 A format and
// 10-12 B format (1 = bf16), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void cluster_barrier() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Shared-memory descriptor of a K-major operand whose rows are `rowb` bytes:
// 128 (128-byte swizzle) or 64 (64-byte swizzle); 8-row groups 8 * rowb
// bytes apart. Bits as for smem_desc_k_sw128, swizzle mode 2 or 4.
__device__ __forceinline__ uint64_t smem_desc_k_sw(uint32_t saddr, int rowb) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>((8 * rowb) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(rowb == 128 ? 2 : 4) << 61;
  return d;
}

// (not volatile: independent loads may overlap; the cluster barriers order
// them against the stores)
__device__ __forceinline__ float4 ld_cluster_v4(uint32_t addr) {
  float4 v;
  asm("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "r"(addr));
  return v;
}

// Launch geometry, fixed on the host.
struct RouterGeom {
  int n_pad;      // expert columns: E rounded up to 16 up to 256, else 512
  int stages;
  int csplit;     // CTAs of a cluster splitting K (1: no split)
  int chunk;      // expert columns exchanged per round of the split reduction
  int xbox, nxb;  // token box rows and token boxes per stage
  int wbox, nwb;  // router-matrix box rows and boxes per stage
  int kb;         // bf16 elements of K per stage: 64, or 32 for 512 expert rows
                  // (40 KB stages instead of 80 KB: five in flight, not two)
};

// A stage: 128 token rows (the MMA's A; rows past those loaded are never
// read back) + n_pad expert rows, 128 bytes each (rows past E read as zero
// and are never selected).
template <int KT>   // capacity of the running top-k, >= k
__global__ void __launch_bounds__(kRThreads, 1) router_topk_kernel(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
    int T, int D, int E, int k, int renormalize, const RouterGeom g,
    int32_t* __restrict__ ids, float* __restrict__ weights,
    float* __restrict__ logits_out, unsigned* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int n_pad = g.n_pad, stages = g.stages, csplit = g.csplit;
  const int rowb = 2 * g.kb;                     // bytes of a row's K step
  const int a_bytes = kRTile * rowb;
  const int stage_bytes = a_bytes + n_pad * rowb;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + stages * stage_bytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * stages + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + stages + s); };
  const uint32_t acc_bar = smem_u32(bars + 2 * stages);
  const uint32_t xchg_bar = smem_u32(bars + 2 * stages + 1);   // upper-half lists ready
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = csplit > 1 ? cluster_rank() : 0;
  const int tile0 = (int)(blockIdx.x / csplit) * kRTile;
  const int kpc = D / g.kb / csplit;            // K blocks of this CTA's slice
  const int kb0 = (int)rank * kpc;
  const int nbox = g.nxb + g.nwb;
  const int nprod = nbox < kRProds ? nbox : kRProds;
  const uint32_t tmem_cols = n_pad <= 32 ? 32 : n_pad <= 64 ? 64 : n_pad <= 128 ? 128
                             : n_pad <= 256 ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), (uint32_t)nprod);   // one arrival per producer
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_bar, 1);
    mbar_init(xchg_bar, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_holder), tmem_cols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_holder;
  pdl_wait();
  pdl_launch_dependents();

  const int prod = warp - kRProd0;
  if (prod >= 0 && prod < nprod && lane == 0) {
    // ---------------- TMA producers: boxes prod, prod + nprod, ... ----------------
    // W_r is read by every CTA; x again by the quantiser that follows
    const uint64_t pol = l2_policy_evict_last();
    uint32_t bytes = 0;
    for (int b = prod; b < nbox; b += nprod)
      bytes += (uint32_t)((b < g.nxb ? g.xbox : g.wbox) * rowb);
    int s = 0;
    uint32_t ph = 0;
    int issued = 0;
    for (int kb = kb0; kb < kb0 + kpc; ++kb) {
      if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kErrTimeoutProducer))
        break;
      mbar_arrive_expect_tx(full_bar(s), bytes);
      const uint32_t st = smem_u32(smem + s * stage_bytes);
      for (int b = prod; b < nbox; b += nprod) {
        if (b < g.nxb) {
          const int r = b * g.xbox;
          tma_load_2d(st + r * rowb, &tm_x, kb * g.kb, tile0 + r, full_bar(s), pol);
        } else {
          const int r = (b - g.nxb) * g.wbox;
          tma_load_2d(st + a_bytes + r * rowb, &tm_w, kb * g.kb, r, full_bar(s), pol);
        }
      }
      ++issued;
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    for (int i = 0; i < stages && i < issued; ++i) {   // every copy landed before exit
      const int last = i + (issued - 1 - i) / stages * stages;   // last use of stage i
      volatile int no_abort = 0;
      mbar_wait_bounded(full_bar(i), (uint32_t)((last / stages) & 1), &no_abort, err,
                        kErrTimeoutDrain);
    }
  } else if (warp == 0 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const int n0 = n_pad < 256 ? n_pad : 256;
    const uint32_t idesc = idesc_bf16_f32(kRTile, n0);
    int s = 0;
    uint32_t ph = 0;
    for (int kb = kb0; kb < kb0 + kpc; ++kb) {
      if (!mbar_wait_bounded(full_bar(s), ph, abort_flag, err, kErrTimeoutMma)) break;
      tc_fence_after_sync();
      const uint32_t a = smem_u32(smem + s * stage_bytes), b = a + a_bytes;
      // descriptors of the stage; a K step of 32 bytes adds 2 to the
      // address field (bytes >> 4), 256 expert rows add 16 * rowb
      const uint64_t da = smem_desc_k_sw(a, rowb), db = smem_desc_k_sw(b, rowb);
      // K = 16 per instruction (32 bytes): 4 or 2 per stage, fully unrolled
      // (the issuing thread's instruction count is on the critical path)
      auto issue = [&](auto ksteps) {
#pragma unroll
        for (int kk = 0; kk < decltype(ksteps)::value; ++kk) {
          const uint32_t acc = (kb != kb0) || (kk != 0);
          mma_bf16(tmem_base, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), idesc, acc);
          if (n_pad > 256)
            mma_bf16(tmem_base + 256u, da + (uint64_t)(2 * kk),
                     db + (uint64_t)((256 * rowb) >> 4) + (uint64_t)(2 * kk), idesc, acc);
        }
      };
      if (g.kb == 64) issue(std::integral_constant<int, 4>{});
      else issue(std::integral_constant<int, 2>{});
      mma_commit(empty_bar(s));
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    mma_commit(acc_bar);   // also completes (with no result) after an abort
  }

  // ---------------- epilogue ----------------
  __syncwarp();
  const bool epi = warp < 4;
  // (every warp waits: without a K split, warps 4-7 scan half the columns)
  const bool have = warp_wait(acc_bar, 0, abort_flag, err, kErrTimeoutEpilogue);
  tc_fence_after_sync();
  const int lrow = warp * 32 + lane;
  const int rows_t = min(T - tile0, kRTile);   // token rows of this tile
  const uint32_t trow = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
  if (csplit > 1) {
    // The stages are free (every copy and MMA has completed). part: this
    // CTA's partial logits of `chunk` columns, [rows_t][chunk + 4] fp32;
    // fin: the summed logits of this rank's rows, [own][n_pad + 4] (rows of
    // 16-byte multiples: vector accesses; the +4 keeps the row-per-lane
    // stores free of bank conflicts).
    const int cc = g.chunk;
    const int per = (rows_t + csplit - 1) / csplit;
    const int own0 = (int)rank * per;
    const int own = max(0, min(per, rows_t - own0));
    const int ldp = cc + 4, ldf = n_pad + 4;
    float* part = reinterpret_cast<float*>(smem);
    float* fin = part + rows_t * ldp;
    const int c4n = cc / 4;
    const int items = own * c4n;   // (row, 4 columns) of this rank's rows
    constexpr int kU = 4;          // items in flight per thread
    for (int h = 0; h < n_pad; h += cc) {
      if (epi) {
        for (int c0 = 0; c0 < cc; c0 += 16) {
          float l[16];
          tmem_ld_x16(trow + (uint32_t)(h + c0), l);
          tmem_ld_wait();
          if (lrow < rows_t) {
            float4* dst = reinterpret_cast<float4*>(part + lrow * ldp + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = have ? make_float4(l[4 * q], l[4 * q + 1], l[4 * q + 2], l[4 * q + 3])
                            : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      cluster_barrier();   // every CTA's partials of this chunk are in place
      for (int p0 = threadIdx.x; p0 < items; p0 += kU * kRThreads) {
        float4 acc[kU];
        uint32_t src[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int p = min(p0 + u * kRThreads, items - 1);
          src[u] = smem_u32(part + (own0 + p / c4n) * ldp + 4 * (p % c4n));
          acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll 4
        for (int r = 0; r < csplit; ++r) {   // rank order: a fixed summation order
          float4 v[kU];
#pragma unroll
          for (int u = 0; u < kU; ++u) v[u] = ld_cluster_v4(map_to_rank(src[u], (uint32_t)r));
#pragma unroll
          for (int u = 0; u < kU; ++u) {
            acc[u].x += v[u].x;
            acc[u].y += v[u].y;
            acc[u].z += v[u].z;
            acc[u].w += v[u].w;
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int p = p0 + u * kRThreads;
          if (p < items)
            *reinterpret_cast<float4*>(fin + (p / c4n) * ldf + h + 4 * (p % c4n)) = acc[u];
        }
      }
      cluster_barrier();   // peers' partials no longer read
    }
    __syncthreads();
    for (int q = warp; q < own; q += kRWarps) {
      const float* row = fin + q * ldf;
      const int64_t tok = (int64_t)tile0 + own0 + q;
      if (E <= 128)
        select_warp<4>(row, E, k, renormalize, tok, ids, weights, logits_out);
      else if (E <= 256)
        select_warp<8>(row, E, k, renormalize, tok, ids, weights, logits_out);
      else
        select_warp<16>(row, E, k, renormalize, tok, ids, weights, logits_out);
    }
  } else if (have) {
    // thread = token: scan the logits straight out of TMEM with a running
    // top-k and the softmax sums. Warps w and w + 4 read the same TMEM lanes:
    // w scans the lower expert columns, w + 4 the upper ones, and hands its
    // list and sums over through shared memory (the stages are free) for w
    // to merge.
    const int row = (warp & 3) * 32 + lane;
    const int upper = warp >> 2;
    const int c_split = (n_pad / 2 + 15) / 16 * 16;
    const int c_begin = upper ? c_split : 0, c_end = upper ? n_pad : c_split;
    const int t = tile0 + row;
    const bool row_ok = row < rows_t;
    float vals[KT];
    int idx[KT];
#pragma unroll
    for (int i = 0; i < KT; ++i) {
      vals[i] = -INFINITY;
      idx[i] = 0x7fffffff;
    }
    float m = -INFINITY, ssum = 0.f;   // online softmax over the scanned experts
    for (int c0 = c_begin; c0 < c_end; c0 += 16) {
      float l[16];
      tmem_ld_x16(trow + (uint32_t)c0, l);
      tmem_ld_wait();
      if (row_ok && logits_out != nullptr) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < E) logits_out[(int64_t)t * E + c0 + j] = l[j];
      }
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j >= E) continue;
        cm = fmaxf(cm, l[j]);
        float cv = l[j];
        int ci = c0 + j;
#pragma unroll
        for (int i = 0; i < KT; ++i) {   // insert: strict >, ties keep the lower index
          if (i < k && cv > vals[i]) {
            const float tv = vals[i];
            const int ti = idx[i];
            vals[i] = cv;
            idx[i] = ci;
            cv = tv;
            ci = ti;
          }
        }
      }
      if (!renormalize && cm > -INFINITY) {
        if (cm > m) {
          ssum = m == -INFINITY ? 0.f : ssum * expf(m - cm);
          m = cm;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < E) ssum += expf(l[j] - m);
      }
    }
    // the upper half's list and sums -> shared memory -> merged by the lower
    float* xf = reinterpret_cast<float*>(smem) + row * (2 * KT + 2);
    int* xi = reinterpret_cast<int*>(xf) + KT;
    bool ok = true;
    if (upper) {
#pragma unroll
      for (int i = 0; i < KT; ++i) {
        xf[i] = vals[i];
        xi[i] = idx[i];
      }
      xf[2 * KT] = m;
      xf[2 * KT + 1] = ssum;
      __syncwarp();
      if (lane == 0) mbar_arrive(xchg_bar);
      ok = false;   // the lower warp writes this token
    } else {
      ok = warp_wait(xchg_bar, 0, abort_flag, err, kErrTimeoutEpilogue);
      if (ok) {
#pragma unroll
        for (int i2 = 0; i2 < KT; ++i2) {   // every upper index is larger: ties stay
          if (i2 < k) {
            float cv = xf[i2];
            int ci = xi[i2];
#pragma unroll
            for (int i = 0; i < KT; ++i) {
              if (i < k && cv > vals[i]) {
                const float tv = vals[i];
                const int ti = idx[i];
                vals[i] = cv;
                idx[i] = ci;
                cv = tv;
                ci = ti;
              }
            }
          }
        }
        const float m2 = xf[2 * KT], s2 = xf[2 * KT + 1];
        if (!renormalize && m2 > -INFINITY) {
          if (m2 > m) {
            ssum = (m == -INFINITY ? 0.f : ssum * expf(m - m2)) + s2;
            m = m2;
          } else {
            ssum += s2 * expf(m2 - m);
          }
        }
      }
    }
    if (ok && row_ok) {
      float denom;
      if (renormalize) {
        denom = 0.f;
#pragma unroll
        for (int i = 0; i < KT; ++i)
          if (i < k) denom += expf(vals[i] - vals[0]);
      } else {
        denom = ssum * expf(m - vals[0]);   // m == vals[0]: the factor is 1
      }
#pragma unroll
      for (int i = 0; i < KT; ++i) {
        if (i < k) {
          ids[(int64_t)t * k + i] = idx[i];
          weights[(int64_t)t * k + i] = expf(vals[i] - vals[0]) / denom;
        }
      }
    }
  }

  // ---------------- tear-down ----------------
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn_bf16() {
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

// [rows, D] bf16 as a 2D TMA map: boxes of 64 elements (128 bytes) of K x
// box_rows rows, 128-byte swizzle; rows past the end read as zero.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int D,
                    int box_rows, int kb) {
  auto fn = encode_fn_bf16();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kb, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            kb == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool router_topk_supported(int E, int k, int D) {
  return E >= 1 && E <= kRMaxN && k >= 1 && k <= kRMaxK && k <= E && D % kRBK == 0;
}

namespace {

// Largest K split (a cluster of that many CTAs) that keeps the grid within
// one CTA per SM, divides the K blocks, fits the exchange buffers in the
// stages and can be co-scheduled; sets g.chunk for it.
template <typename Kern>
int pick_split(Kern kern, RouterGeom& g, int T, int D, size_t smem, cudaLaunchConfig_t cfg,
               cudaLaunchAttribute* attr) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = (T + kRTile - 1) / kRTile;
  const int kblocks = D / g.kb;
  const size_t avail = (size_t)g.stages * (kRTile + g.n_pad) * 2 * g.kb;
  const int rows = T < kRTile ? T : kRTile;
  for (int c = kRMaxCluster; c >= 2; c /= 2) {
    if (kblocks % c != 0 || tiles * c > sms) continue;
    const int per = (rows + c - 1) / c;
    int cc = 0;
    for (int cand : {g.n_pad, 256, 128}) {
      if (cand > g.n_pad || g.n_pad % cand != 0) continue;
      if ((size_t)rows * (cand + 4) * 4 + (size_t)per * (g.n_pad + 4) * 4 <= avail) {
        cc = cand;
        break;
      }
    }
    if (cc == 0) continue;
    // how many clusters of c CTAs with this shared memory can be resident at
    // once (all tiles in one wave, or a smaller split)
    // per device (up to 64) and shared-memory class: 1 + the count, 0 when
    // not asked yet (racing first askers store the same answer)
    static std::atomic<int> known[64][2][kRMaxCluster + 1];
    const int slot = g.n_pad > 256 ? 1 : 0;
    std::atomic<int>& ans = known[dev >= 0 && dev < 64 ? dev : 0][slot][c];
    if (ans.load(std::memory_order_relaxed) == 0) {
      if (c > 8) cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      attr[0].val.clusterDim.x = (unsigned)c;
      cfg.gridDim = dim3((unsigned)(tiles * c));
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
      cudaGetLastError();   // a refused size is not an error of this call
      ans.store(1 + n, std::memory_order_relaxed);
    }
    if (ans.load(std::memory_order_relaxed) - 1 < tiles) continue;
    g.chunk = cc;
    return c;
  }
  g.chunk = g.n_pad;
  return 1;
}

}  // namespace

int launch_router_topk(const uint16_t* x, const uint16_t* w_r, int T, int D, int E,
                       int k, int renormalize, int32_t* ids, float* weights,
                       float* logits_out, cudaStream_t stream, bool pdl) {
  if (T == 0) return 0;
  if (!router_topk_supported(E, k, D)) return -2;
  RouterGeom g{};
  g.n_pad = E <= 256 ? (E + 15) / 16 * 16 : 512;
  // (a single tile's K slices are short: there the larger step wins)
  g.kb = g.n_pad > 256 && T > kRTile ? 32 : kRBK;
  const int stage_bytes = (kRTile + g.n_pad) * 2 * g.kb;
  g.stages = (200 * 1024) / stage_bytes;
  if (g.stages > 8) g.stages = 8;
  if (g.stages < 2) g.stages = 2;
  // token boxes cover only the rows a batch of fewer than 128 tokens has
  const int a_rows = T < kRTile ? (T + 7) / 8 * 8 : kRTile;
  g.xbox = a_rows < kRBoxRows ? a_rows : kRBoxRows;
  g.nxb = (a_rows + g.xbox - 1) / g.xbox;
  g.wbox = g.n_pad < kRBoxRows ? g.n_pad : kRBoxRows;
  while (g.n_pad % g.wbox != 0) g.wbox /= 2;
  g.nwb = g.n_pad / g.wbox;
  CUtensorMap tm_x, tm_w;
  if (!make_tmap_bf16(&tm_x, x, T, D, g.xbox, g.kb)) return -3;
  if (!make_tmap_bf16(&tm_w, w_r, E, D, g.wbox, g.kb)) return -3;
  const int smem = 1024 + g.stages * stage_bytes + (2 * g.stages + 2) * 8 + 16;
  auto kern = k <= 2 ? router_topk_kernel<2>
              : k <= 4 ? router_topk_kernel<4>
              : k <= 8 ? router_topk_kernel<8> : router_topk_kernel<16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kRThreads);
  cfg.stream = stream;
  g.csplit = pick_split(kern, g, T, D, (size_t)smem, cfg, attr);
  // (the answers above are shared by the KT instances; the opt-in is per kernel)
  if (g.csplit > 8 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess)
    return -3;
  const int tiles = (T + kRTile - 1) / kRTile;
  attr[0].val.clusterDim.x = (unsigned)g.csplit;
  cfg.gridDim = dim3((unsigned)(tiles * g.csplit));
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, T, D, E, k, renormalize,
                                           g, ids, weights, logits_out, device_error_word());
  return e == cudaSuccess ? 0 : -3;
}

}  // namespace moe
