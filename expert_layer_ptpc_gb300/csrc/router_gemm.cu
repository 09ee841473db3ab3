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
// Roles: warp 0 allocates TMEM and issues the MMAs (one thread); warps 4..
// are TMA producers, one per box of a stage (the token box and the router
// matrix in boxes of up to 128 rows: a single issuing thread caps an SM's
// feed far below the MMA rate); warps 0-3 run the epilogue (warp w reads TMEM
// lanes 32w..32w+31). Every wait is bounded.
//
// A batch of at most 64 tokens is one tile, which one SM would stream the
// whole router matrix for. There, a cluster of C CTAs splits K: each CTA
// accumulates its D/C slice, parks its partial logits in shared memory, and
// the cluster's first CTA sums the C partials in rank order (distributed
// shared memory) before the selection.
#include <math.h>

#include "gemm_common.cuh"

namespace moe {
namespace {

using namespace gemm;

constexpr int kRProd0 = 4;               // first producer warp
constexpr int kRBBoxRows = 128;          // router-matrix rows per TMA box
constexpr int kRMaxBoxes = 1 + 512 / kRBBoxRows;
constexpr int kRThreads = 32 * (kRProd0 + kRMaxBoxes);
constexpr int kRBK = 64;                 // bf16 elements of K per stage (128 bytes)
constexpr int kRTile = 128;              // tokens per CTA (MMA M)
constexpr int kRMaxN = 512;              // expert columns (two N = 256 MMAs)
constexpr int kRMaxK = 16;               // top-k kept in registers (KT <= 16)

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A and B, fp32
// accumulator, both K-major: bits 4-5 D format (1 = f32), 7-9 A format and
// 10-12 B format (1 = bf16), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// (not volatile: independent loads may overlap; the cluster barriers order
// them against the stores)
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
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

// n_pad: expert columns, E rounded up to a multiple of 16 up to 256, else
// 512 (two full N = 256 MMAs); stages of 128 token rows + n_pad expert rows
// of 128 bytes each (rows past E read as zero and are never selected).
template <int KT>   // capacity of the running top-k, >= k
__global__ void __launch_bounds__(kRThreads, 1) router_topk_kernel(
    const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
    int T, int D, int E, int n_pad, int k, int renormalize, int stages, int csplit,
    int32_t* __restrict__ ids, float* __restrict__ weights,
    float* __restrict__ logits_out, unsigned* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int a_bytes = kRTile * 128;
  const int b_bytes = n_pad * 128;
  const int stage_bytes = a_bytes + b_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + stages * stage_bytes);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * stages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + stages + s); };
  const uint32_t acc_bar = smem_u32(bars + 2 * stages);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = csplit > 1 ? cluster_rank() : 0;
  const int tile0 = (int)(blockIdx.x / csplit) * kRTile;
  const int kpc = D / kRBK / csplit;            // K blocks of this CTA's slice
  const int kb0 = (int)rank * kpc;
  const uint32_t tmem_cols = n_pad <= 32 ? 32 : n_pad <= 64 ? 64 : n_pad <= 128 ? 128
                             : n_pad <= 256 ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full_bar(s), 1 + (n_pad + kRBBoxRows - 1) / kRBBoxRows);   // boxes
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_bar, 1);
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

  const int box = warp - kRProd0;        // 0: tokens; 1..: router-matrix rows
  const int nboxes = 1 + (n_pad + kRBBoxRows - 1) / kRBBoxRows;
  if (box >= 0 && box < nboxes && lane == 0) {
    // ---------------- TMA producers: box `box` of every stage ----------------
    const uint64_t pol = l2_policy_evict_last();   // W_r is read by every CTA
    const int brow = (box - 1) * kRBBoxRows;
    const uint32_t bytes =
        box == 0 ? (uint32_t)a_bytes
                 : (uint32_t)(min(kRBBoxRows, n_pad - brow) * 128);
    int s = 0;
    uint32_t ph = 0;
    int last_phase[8];
    for (int i = 0; i < 8; ++i) last_phase[i] = -1;
    for (int kb = kb0; kb < kb0 + kpc; ++kb) {
      if (!mbar_wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, err, kErrTimeoutProducer))
        break;
      mbar_arrive_expect_tx(full_bar(s), bytes);
      const uint32_t st = smem_u32(smem + s * stage_bytes);
      if (box == 0)
        tma_load_2d(st, &tm_x, kb * kRBK, tile0, full_bar(s), pol);
      else
        tma_load_2d(st + a_bytes + brow * 128, &tm_w, kb * kRBK, brow, full_bar(s), pol);
      last_phase[s] = (int)ph;
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    for (int i = 0; i < stages; ++i) {   // every copy landed before exit
      if (last_phase[i] >= 0) {
        volatile int no_abort = 0;
        mbar_wait_bounded(full_bar(i), (uint32_t)last_phase[i], &no_abort, err,
                          kErrTimeoutDrain);
      }
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
#pragma unroll
      for (int kk = 0; kk < kRBK / 16; ++kk) {   // K = 16 per instruction (32 bytes)
        const uint32_t acc = (kb != kb0) || (kk != 0);
        for (int h = 0; h < n_pad; h += 256)
          mma_bf16(tmem_base + (uint32_t)h, smem_desc_k_sw128(a + kk * 32),
                   smem_desc_k_sw128(b + h * 128 + kk * 32), idesc, acc);
      }
      mma_commit(empty_bar(s));
      if (++s == stages) {
        s = 0;
        ph ^= 1u;
      }
    }
    mma_commit(acc_bar);   // also completes (with no result) after an abort
  }

  // ---------------- epilogue (warps 0-3): thread = token ----------------
  __syncwarp();
  const bool epi = warp < 4;
  const bool have = epi && warp_wait(acc_bar, 0, abort_flag, err, kErrTimeoutEpilogue);
  tc_fence_after_sync();
  const int lrow = warp * 32 + lane;
  const int t = tile0 + lrow;
  const uint32_t trow = tmem_base + ((uint32_t)(warp * 32) << 16);
  float vals[KT];
  int idx[KT];
#pragma unroll
  for (int i = 0; i < KT; ++i) {
    vals[i] = -INFINITY;
    idx[i] = 0x7fffffff;
  }
  float m = -INFINITY, ssum = 0.f;   // online softmax over all experts
  bool scanned = false;
  const int ldp = n_pad + 1;
  float* part = reinterpret_cast<float*>(smem);
  const bool row_ok = t < T;
  if (csplit > 1) {
    // partial logits of this K slice -> shared memory (the stages are free:
    // every copy and MMA has completed), [row][n_pad + 1] fp32
    if (epi) {
      for (int c0 = 0; c0 < n_pad; c0 += 16) {
        float l[16];
        tmem_ld_x16(trow + (uint32_t)c0, l);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j) part[lrow * ldp + c0 + j] = have ? l[j] : 0.f;
        }
      }
    }
    cluster_barrier();   // every CTA's partials are in place
    // CTA r sums its slice of the columns over the ranks (in rank order, a
    // fixed summation order) into the first CTA's buffer
    if (epi) {   // (row, column) pairs of this CTA's slice over the 128 threads
      const int cs = n_pad / csplit;
      const int rows = min(T - tile0, kRTile);
      for (int p = lrow; p < rows * cs; p += 128) {
        const int r0 = p / cs, c = (int)rank * cs + p % cs;
        const uint32_t src = smem_u32(part + r0 * ldp + c);
        float acc = 0.f;
        for (int r = 0; r < csplit; ++r) acc += ld_cluster_f32(map_to_rank(src, (uint32_t)r));
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(map_to_rank(src, 0)), "f"(acc)
                     : "memory");
      }
    }
    cluster_barrier();   // the sums are in place; peers' memory no longer read
    if (epi && rank == 0) {
      // a warp per token (few tokens here): lanes hold strided experts; k
      // rounds of a warp argmax, larger value first, equal values to the
      // lower index (route.cu's rule)
      const int rows = min(T - tile0, kRTile);
      for (int r0 = warp; r0 < rows; r0 += 4) {
        const float* row = part + r0 * ldp;
        const int tok = tile0 + r0;
        if (logits_out != nullptr)
          for (int e = lane; e < E; e += 32) logits_out[(int64_t)tok * E + e] = row[e];
        uint32_t taken = 0;   // bit i: expert lane + 32 i chosen
        float my_val = -INFINITY;
        int my_idx = 0;
        for (int j = 0; j < k; ++j) {
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          for (int i = 0; lane + 32 * i < E; ++i) {
            const float v = row[lane + 32 * i];
            if (!((taken >> i) & 1u) && (v > bv || bi == 0x7fffffff)) {
              bv = v;
              bi = lane + 32 * i;
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
              bv = ov;
              bi = oi;
            }
          }
          if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
          if (j == lane) {
            my_val = bv;
            my_idx = bi;
          }
        }
        const float top = __shfl_sync(0xffffffffu, my_val, 0);
        float den = 0.f;
        if (renormalize) {
          den = warp_sum(lane < k ? expf(my_val - top) : 0.f);
        } else {
          float s = 0.f;
          for (int e = lane; e < E; e += 32) s += expf(row[e] - top);
          den = warp_sum(s);
        }
        if (lane < k) {
          ids[(int64_t)tok * k + lane] = my_idx;
          weights[(int64_t)tok * k + lane] = expf(my_val - top) / den;
        }
      }
    }
  }
  // the scan: from TMEM (one CTA per tile) or from the summed partials (the
  // cluster's first CTA); a running top-k and the softmax sums
  const bool from_tmem = csplit == 1;
  if (from_tmem && have) {
    for (int c0 = 0; c0 < n_pad; c0 += 16) {
      float l[16];
      if (from_tmem) {
        tmem_ld_x16(trow + (uint32_t)c0, l);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) l[j] = part[lrow * ldp + c0 + j];
      }
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
    scanned = true;
  }
  if (epi && scanned && t < T) {
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
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [rows, D] bf16 as a 2D TMA map: boxes of 64 elements (128 bytes) of K x
// box_rows rows, 128-byte swizzle; rows past the end read as zero.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t rows, int D,
                    int box_rows) {
  auto fn = encode_fn_bf16();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kRBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool router_topk_supported(int E, int k, int D) {
  return E >= 1 && E <= kRMaxN && k >= 1 && k <= kRMaxK && k <= E && D % kRBK == 0;
}

int launch_router_topk(const uint16_t* x, const uint16_t* w_r, int T, int D, int E,
                       int k, int renormalize, int32_t* ids, float* weights,
                       float* logits_out, cudaStream_t stream, bool pdl) {
  if (T == 0) return 0;
  if (!router_topk_supported(E, k, D)) return -2;
  const int n_pad = E <= 256 ? (E + 15) / 16 * 16 : 512;
  CUtensorMap tm_x, tm_w;
  if (!make_tmap_bf16(&tm_x, x, T, D, kRTile)) return -3;
  if (!make_tmap_bf16(&tm_w, w_r, E, D, n_pad < kRBBoxRows ? n_pad : kRBBoxRows))
    return -3;
  const int stage_bytes = kRTile * 128 + n_pad * 128;
  int stages = (200 * 1024) / stage_bytes;
  if (stages > 8) stages = 8;
  if (stages < 2) stages = 2;
  const int smem = 1024 + stages * stage_bytes + (2 * stages + 1) * 8 + 16;
  auto kern = k <= 2 ? router_topk_kernel<2>
              : k <= 4 ? router_topk_kernel<4>
              : k <= 8 ? router_topk_kernel<8> : router_topk_kernel<16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return -3;
  // split K over a cluster for a single tile of at most 64 tokens (its
  // partials, 64 x (n_pad + 1) fp32, fit in the stages)
  const int kblocks = D / kRBK;
  int csplit = 1;
  if (T <= 64)
    for (int c : {8, 4, 2})
      if (kblocks % c == 0 && (size_t)T * (n_pad + 1) * 4 <= (size_t)stages * stage_bytes) {
        csplit = c;
        break;
      }
  const int tiles = (T + kRTile - 1) / kRTile;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)csplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(tiles * csplit));
  cfg.blockDim = dim3(kRThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, kern, tm_x, tm_w, T, D, E, n_pad, k,
                         renormalize, stages, csplit, ids, weights, logits_out,
                         device_error_word());
  return e == cudaSuccess ? 0 : -3;
}

}  // namespace moe
