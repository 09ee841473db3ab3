// Per-row FP8 e4m3 quantisation (PTPC) with fused scatter into permuted rows.
//
// "Ultimate Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series",
// section 2.1.1 and Figure 3: activations get one scale per token, weights
// one per output channel; section 2.1.5: per-token quantisation is fused into
// the kernel that produces or moves the rows. Here the quantiser also does
// the permute gather of the TPU page's SparseCore paragraph: each token row is
// read once and its FP8 codes are written straight to its k expert rows.
//
//   s = fp32(max(amax, 1e-12) / 448),  q = e4m3_rne_sat(fp32(v / s))
//
// Both divisions are IEEE round-to-nearest (__fdiv_rn), so codes and scales
// are the exactly rounded values of that definition.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kVec = 16;        // elements per thread per unit (16 bytes of codes)
constexpr int kMaxThreads = 512;
constexpr int kWarpsPerBlock = 8;   // rows per block of the warp-per-row kernels

__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&v)[kVec]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 raw = *reinterpret_cast<const uint4*>(p + 8 * h);
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * h + 2 * i] = __low2float(b[i]);
      v[8 * h + 2 * i + 1] = __high2float(b[i]);
    }
  }
}

__device__ __forceinline__ void load_vec(const float* p, float (&v)[kVec]) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float4 a = *reinterpret_cast<const float4*>(p + 4 * h);
    v[4 * h] = a.x; v[4 * h + 1] = a.y; v[4 * h + 2] = a.z; v[4 * h + 3] = a.w;
  }
}

// One block per row; each thread holds UNITS vectors of kVec elements, so the
// row is read from memory once. The row maximum (and the gate's dot product)
// is reduced over the block, the scale is formed once, and every thread
// writes its 16-byte code vectors to each destination row.
template <typename InT, int UNITS>
__global__ void __launch_bounds__(kMaxThreads) quant_rows_kernel(
    const InT* __restrict__ in, int64_t rows, int cols,
    const int32_t* __restrict__ dst_rows, int copies, int64_t extra_row_base,
    uint8_t* __restrict__ out_q, float* __restrict__ out_scale,
    const __nv_bfloat16* __restrict__ gate_w, float* __restrict__ gate_out,
    int release_early, int64_t out_rows, unsigned* __restrict__ err) {
  __shared__ float red_max[kMaxThreads / 32];
  __shared__ float red_dot[kMaxThreads / 32];
  __shared__ int64_t dst[kMaxTopK + 1];
  // release_early: the next kernel may start before this one waits. Only
  // for a successor whose pre-wait part reads nothing this kernel's
  // predecessor produces (the down GEMM reads the tile map and weights).
  if (release_early) pdl_launch_dependents();
  pdl_wait();
  if (!release_early) pdl_launch_dependents();
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int nunits = cols / kVec;
  const InT* row = in + r * cols;

  float v[UNITS][kVec];
  float amax = 0.f, dot = 0.f;
#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = tid + i * blockDim.x;
    if (u < nunits) {
      load_vec(row + u * kVec, v[i]);
#pragma unroll
      for (int j = 0; j < kVec; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
      if (gate_w != nullptr) {
        float g[kVec];
        load_vec(gate_w + u * kVec, g);
#pragma unroll
        for (int j = 0; j < kVec; ++j) dot = fmaf(v[i][j], g[j], dot);
      }
    }
  }
  amax = warp_max(amax);
  dot = warp_sum(dot);
  if (lane == 0) {
    red_max[warp] = amax;
    red_dot[warp] = dot;
  }
  // destination rows of this row
  const int nmain = dst_rows != nullptr ? copies : 1;
  const int ndst = nmain + (extra_row_base >= 0 ? 1 : 0);
  // strided: a block narrower than ndst (32 threads, 32 copies + the shared
  // row) still fills every entry
  for (int i = tid; i < ndst; i += blockDim.x) {
    int64_t d = i < nmain ? (dst_rows != nullptr ? (int64_t)dst_rows[r * copies + i] : r)
                          : extra_row_base + r;
    // checked build: a destination outside [0, out_rows) is skipped
    if (!MOE_CHECKED(d >= 0 && (out_rows < 0 || d < out_rows), err)) d = -1;
    dst[i] = d;
  }
  __syncthreads();
  if (warp == 0) {
    float a = lane < nwarps ? red_max[lane] : 0.f;
    float d = lane < nwarps ? red_dot[lane] : 0.f;
    a = warp_max(a);
    d = warp_sum(d);
    if (lane == 0) {
      red_max[0] = a;
      red_dot[0] = d;
    }
  }
  __syncthreads();
  const float s = __fdiv_rn(fmaxf(red_max[0], 1e-12f), 448.0f);
  for (int i = tid; i < ndst; i += blockDim.x)
    if (dst[i] >= 0) out_scale[dst[i]] = s;
  if (gate_w != nullptr && tid == 0) gate_out[r] = 1.0f / (1.0f + expf(-red_dot[0]));

#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = tid + i * blockDim.x;
    if (u < nunits) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[i][4 * q], s),
                                            __fdiv_rn(v[i][4 * q + 1], s));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[i][4 * q + 2], s),
                                            __fdiv_rn(v[i][4 * q + 3], s));
        w[q] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      const uint4 packed = make_uint4(w[0], w[1], w[2], w[3]);
      for (int d = 0; d < ndst; ++d)
        if (dst[d] >= 0) *reinterpret_cast<uint4*>(out_q + dst[d] * cols + u * kVec) = packed;
    }
  }
}

// The same quantiser for rows of at most 64 vectors (1024 elements): one warp
// per row and kWarpsPerBlock rows per block, so that narrow rows (h of a
// 512-wide expert) are not one single-warp block each, and the reductions
// stay in the warp. The row maximum is order-independent, so scales and
// codes equal quant_rows_kernel's bit for bit; only the gate's dot product is
// summed in another order (lane's units first, then across the warp).
template <typename InT, int UNITS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) quant_rows_warp_kernel(
    const InT* __restrict__ in, int64_t rows, int cols,
    const int32_t* __restrict__ dst_rows, int copies, int64_t extra_row_base,
    uint8_t* __restrict__ out_q, float* __restrict__ out_scale,
    const __nv_bfloat16* __restrict__ gate_w, float* __restrict__ gate_out,
    int release_early, int64_t out_rows, unsigned* __restrict__ err) {
  if (release_early) pdl_launch_dependents();
  pdl_wait();
  if (!release_early) pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (r >= rows) return;   // whole warps: r is uniform within a warp
  const int nunits = cols / kVec;
  const InT* row = in + r * cols;

  float v[UNITS][kVec];
  float amax = 0.f, dot = 0.f;
#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = lane + 32 * i;
    if (u < nunits) {
      load_vec(row + u * kVec, v[i]);
#pragma unroll
      for (int j = 0; j < kVec; ++j) amax = fmaxf(amax, fabsf(v[i][j]));
      if (gate_w != nullptr) {
        float g[kVec];
        load_vec(gate_w + u * kVec, g);
#pragma unroll
        for (int j = 0; j < kVec; ++j) dot = fmaf(v[i][j], g[j], dot);
      }
    }
  }
  // destination rows: lane d holds the d-th (the launcher sends rows with at
  // most 32 destinations here)
  const int nmain = dst_rows != nullptr ? copies : 1;
  const int ndst = nmain + (extra_row_base >= 0 ? 1 : 0);
  int64_t my_dst = 0;
  if (lane < ndst) {
    my_dst = lane < nmain ? (dst_rows != nullptr ? (int64_t)dst_rows[r * copies + lane] : r)
                          : extra_row_base + r;
    // checked build: a destination outside [0, out_rows) is skipped
    if (!MOE_CHECKED(my_dst >= 0 && (out_rows < 0 || my_dst < out_rows), err)) my_dst = -1;
  }
  amax = warp_max(amax);
  const float s = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
  if (lane < ndst && my_dst >= 0) out_scale[my_dst] = s;
  if (gate_w != nullptr) {
    dot = warp_sum(dot);
    if (lane == 0) gate_out[r] = 1.0f / (1.0f + expf(-dot));
  }

#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = lane + 32 * i;
    uint4 packed = make_uint4(0u, 0u, 0u, 0u);
    if (u < nunits) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[i][4 * q], s),
                                            __fdiv_rn(v[i][4 * q + 1], s));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[i][4 * q + 2], s),
                                            __fdiv_rn(v[i][4 * q + 3], s));
        w[q] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      packed = make_uint4(w[0], w[1], w[2], w[3]);
    }
    // every lane takes part in the shuffles; only lanes with a unit store
    for (int d = 0; d < ndst; ++d) {
      const int64_t dd = __shfl_sync(0xffffffffu, my_dst, d);
      if (u < nunits && dd >= 0) *reinterpret_cast<uint4*>(out_q + dd * cols + u * kVec) = packed;
    }
  }
}

// Add + RMSNorm + PTPC quantisation of one token row per block ("Ultimate
// Latency Optimization of Qwen3 and Qwen3-VL on AMD MI300X Series", section
// 2.1.5: AddRMSNorm and per-token quant fused into one operator):
//   r = bf16_rne(x + res)                  (written back: the new residual)
//   ms = fp32(S / D), S = sum r^2          (S exact, see below)
//   inv = fp32_rn(1 / sqrt(fp32(ms + eps)))  (__frsqrt_rn, correctly rounded)
//   v = fp32(fp32(r * inv) * gamma)
// then the quantiser of quant_rows_kernel on v, and optionally the shared
// expert's gate sigmoid(v . w_g). The row stays in registers throughout: x,
// res and gamma are read once, r and the codes written once per destination.
//
// S in integers: a bf16 value is r = s * 2^(e - 134) with an 8-bit integer
// significand s (e the fp32 exponent field), so r^2 = s^2 * 2^(2e - 268) with
// s^2 < 2^16. Every square is placed on the grid 2^(2 emax - 268 - sbits) of
// the row's largest exponent emax and the row is summed in a 64-bit integer,
// which is exact and independent of the summation order (sbits leaves room
// for cols squares of up to 2^16). A square more than 2^sbits below the
// largest (|r| under 2^-17 of the row's largest for cols = 4096) keeps only
// its bits on the grid. The one rounding to double of the integer sum then
// equals the exactly rounded sum the reference takes. (A plain fp64 sum
// would also be exact, but GB300's fp64 rate made it the kernel's
// bottleneck.)
template <int UNITS>
__global__ void __launch_bounds__(kMaxThreads) add_rmsnorm_quant_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* res,   // res_out may
    const __nv_bfloat16* __restrict__ gamma, float eps, int cols,     // alias res
    __nv_bfloat16* res_out, const int32_t* __restrict__ dst_rows,
    int copies, int64_t extra_row_base, uint8_t* __restrict__ out_q,
    float* __restrict__ out_scale, const __nv_bfloat16* __restrict__ gate_w,
    float* __restrict__ gate_out, int sbits, int64_t out_rows, unsigned* __restrict__ err) {
  __shared__ unsigned long long red_sq[kMaxThreads / 32];
  __shared__ int red_e[kMaxThreads / 32];
  __shared__ float red_max[kMaxThreads / 32];
  __shared__ float red_dot[kMaxThreads / 32];
  __shared__ int64_t dst[kMaxTopK + 1];
  __shared__ float s_inv;
  pdl_wait();
  pdl_launch_dependents();
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int nunits = cols / kVec;

  float v[UNITS][kVec];
  int emax = 0;
#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = tid + i * blockDim.x;
    if (u < nunits) {
      float a[kVec], b[kVec];
      load_vec(x + r * cols + u * kVec, a);
      load_vec(res + r * cols + u * kVec, b);
      uint32_t packed[kVec / 2];
#pragma unroll
      for (int j = 0; j < kVec; j += 2) {
        const __nv_bfloat162 p =
            __floats2bfloat162_rn(__fadd_rn(a[j], b[j]), __fadd_rn(a[j + 1], b[j + 1]));
        v[i][j] = __low2float(p);
        v[i][j + 1] = __high2float(p);
        packed[j / 2] = *reinterpret_cast<const uint32_t*>(&p);
        emax = max(emax, max((int)((__float_as_uint(v[i][j]) >> 23) & 0xFFu),
                             (int)((__float_as_uint(v[i][j + 1]) >> 23) & 0xFFu)));
      }
      uint4* o = reinterpret_cast<uint4*>(res_out + r * cols + u * kVec);
      o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    }
  }
  // the row's largest exponent field
  emax = __reduce_max_sync(0xffffffffu, emax);
  if (lane == 0) red_e[warp] = emax;
  __syncthreads();
  emax = 1;   // zeros and subnormals sit at exponent 1
  for (int w = 0; w < nwarps; ++w) emax = max(emax, red_e[w]);
  unsigned long long sq = 0;
#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = tid + i * blockDim.x;
    if (u < nunits) {
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        const uint32_t b = __float_as_uint(v[i][j]);
        int e = (int)((b >> 23) & 0xFFu);
        uint32_t sig = (b >> 16) & 0x7Fu;
        if (e != 0) sig |= 0x80u; else e = 1;
        const unsigned long long s2 = (unsigned long long)(sig * sig);
        const int sh = sbits - 2 * (emax - e);
        sq += sh >= 0 ? (s2 << sh) : (sh > -32 ? (s2 >> -sh) : 0ull);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if (lane == 0) red_sq[warp] = sq;
  __syncthreads();
  if (tid == 0) {
    unsigned long long t = 0;
    for (int w = 0; w < nwarps; ++w) t += red_sq[w];
    // S = t * 2^(2 emax - 268 - sbits): one rounding (of t), then exact
    const double S = ldexp(__ull2double_rn(t), 2 * emax - 268 - sbits);
    const float ms = (float)(S / (double)cols);
    s_inv = __frsqrt_rn(__fadd_rn(ms, eps));
  }
  __syncthreads();
  const float inv = s_inv;

  float amax = 0.f, dot = 0.f;
#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = tid + i * blockDim.x;
    if (u < nunits) {
      float g[kVec];
      load_vec(gamma + u * kVec, g);
#pragma unroll
      for (int j = 0; j < kVec; ++j) {
        v[i][j] = __fmul_rn(__fmul_rn(v[i][j], inv), g[j]);
        amax = fmaxf(amax, fabsf(v[i][j]));
      }
      if (gate_w != nullptr) {
        float w[kVec];
        load_vec(gate_w + u * kVec, w);
#pragma unroll
        for (int j = 0; j < kVec; ++j) dot = fmaf(v[i][j], w[j], dot);
      }
    }
  }
  amax = warp_max(amax);
  dot = warp_sum(dot);
  if (lane == 0) {
    red_max[warp] = amax;
    red_dot[warp] = dot;
  }
  const int nmain = dst_rows != nullptr ? copies : 1;
  const int ndst = nmain + (extra_row_base >= 0 ? 1 : 0);
  // strided: a block narrower than ndst (32 threads, 32 copies + the shared
  // row) still fills every entry
  for (int i = tid; i < ndst; i += blockDim.x) {
    int64_t d = i < nmain ? (dst_rows != nullptr ? (int64_t)dst_rows[r * copies + i] : r)
                          : extra_row_base + r;
    // checked build: a destination outside [0, out_rows) is skipped
    if (!MOE_CHECKED(d >= 0 && (out_rows < 0 || d < out_rows), err)) d = -1;
    dst[i] = d;
  }
  __syncthreads();
  if (warp == 0) {
    float a = lane < nwarps ? red_max[lane] : 0.f;
    float d = lane < nwarps ? red_dot[lane] : 0.f;
    a = warp_max(a);
    d = warp_sum(d);
    if (lane == 0) {
      red_max[0] = a;
      red_dot[0] = d;
    }
  }
  __syncthreads();
  const float s = __fdiv_rn(fmaxf(red_max[0], 1e-12f), 448.0f);
  for (int i = tid; i < ndst; i += blockDim.x)
    if (dst[i] >= 0) out_scale[dst[i]] = s;
  if (gate_w != nullptr && tid == 0) gate_out[r] = 1.0f / (1.0f + expf(-red_dot[0]));
#pragma unroll
  for (int i = 0; i < UNITS; ++i) {
    const int u = tid + i * blockDim.x;
    if (u < nunits) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[i][4 * q], s),
                                            __fdiv_rn(v[i][4 * q + 1], s));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[i][4 * q + 2], s),
                                            __fdiv_rn(v[i][4 * q + 3], s));
        w[q] = (uint32_t)lo | ((uint32_t)hi << 16);
      }
      const uint4 packed = make_uint4(w[0], w[1], w[2], w[3]);
      for (int d = 0; d < ndst; ++d)
        if (dst[d] >= 0) *reinterpret_cast<uint4*>(out_q + dst[d] * cols + u * kVec) = packed;
    }
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) shared_gate_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
    int T, int D, float* __restrict__ gate) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (t >= T) return;
  float dot = 0.f;
  for (int c = (int)lane_id() * kVec; c < D; c += 32 * kVec) {
    float v[kVec], g[kVec];
    load_vec(x + (int64_t)t * D + c, v);
    load_vec(w + c, g);
#pragma unroll
    for (int i = 0; i < kVec; ++i) dot = fmaf(v[i], g[i], dot);
  }
  dot = warp_sum(dot);
  if (lane_id() == 0) gate[t] = 1.0f / (1.0f + expf(-dot));
}

template <typename InT>
cudaError_t launch_rows(const InT* in, int64_t rows, int cols,
                        const int32_t* dst_rows, int copies,
                        int64_t extra_row_base, uint8_t* out_q,
                        float* out_scale, const __nv_bfloat16* gate_w,
                        float* gate_out, cudaStream_t stream, bool pdl,
                        bool release_early, int64_t out_rows) {
  const int nunits = cols / kVec;
  const int ndst = (dst_rows != nullptr ? copies : 1) + (extra_row_base >= 0 ? 1 : 0);
  if (nunits <= 64 && ndst <= 32) {
    const dim3 grid((unsigned)((rows + kWarpsPerBlock - 1) / kWarpsPerBlock));
    auto go = [&](auto kern) {
      return launch_kernel(pdl, grid, dim3(kWarpsPerBlock * 32), 0, stream, kern, in,
                           rows, cols, dst_rows, copies, extra_row_base, out_q,
                           out_scale, gate_w, gate_out, release_early ? 1 : 0, out_rows,
                           device_error_word());
    };
    if (nunits <= 32) return go(quant_rows_warp_kernel<InT, 1>);
    return go(quant_rows_warp_kernel<InT, 2>);
  }
  int threads = std::min(kMaxThreads, ((nunits + 31) / 32) * 32);
  const int units = (nunits + threads - 1) / threads;
  const dim3 grid((unsigned)rows), block(threads);
  auto go = [&](auto kern) {
    return launch_kernel(pdl, grid, block, 0, stream, kern, in, rows, cols,
                         dst_rows, copies, extra_row_base, out_q, out_scale,
                         gate_w, gate_out, release_early ? 1 : 0, out_rows,
                         device_error_word());
  };
  if (units <= 1) return go(quant_rows_kernel<InT, 1>);
  if (units <= 2) return go(quant_rows_kernel<InT, 2>);
  return go(quant_rows_kernel<InT, 4>);
}

}  // namespace

cudaError_t launch_quant(const void* in, int in_dtype, int64_t rows, int cols,
                         const int32_t* dst_rows, int copies,
                         int64_t extra_row_base, uint8_t* out_q,
                         float* out_scale, const uint16_t* gate_w,
                         float* gate_out, cudaStream_t stream, bool pdl,
                         bool release_early, int64_t out_rows) {
  if (rows == 0) return cudaSuccess;
  if (in_dtype == 0)
    return launch_rows(static_cast<const __nv_bfloat16*>(in), rows, cols,
                       dst_rows, copies, extra_row_base, out_q, out_scale,
                       reinterpret_cast<const __nv_bfloat16*>(gate_w), gate_out,
                       stream, pdl, release_early, out_rows);
  return launch_rows(static_cast<const float*>(in), rows, cols, dst_rows, copies,
                     extra_row_base, out_q, out_scale,
                     (const __nv_bfloat16*)nullptr, (float*)nullptr, stream, pdl,
                     release_early, out_rows);
}

cudaError_t launch_add_rmsnorm_quant(const uint16_t* x, const uint16_t* res,
                                     const uint16_t* gamma, float eps, int64_t rows,
                                     int cols, uint16_t* res_out,
                                     const int32_t* dst_rows, int copies,
                                     int64_t extra_row_base, uint8_t* out_q,
                                     float* out_scale, const uint16_t* gate_w,
                                     float* gate_out, cudaStream_t stream, bool pdl,
                                     int64_t out_rows) {
  if (rows == 0) return cudaSuccess;
  const int nunits = cols / kVec;
  const int threads = std::min(kMaxThreads, ((nunits + 31) / 32) * 32);
  const int units = (nunits + threads - 1) / threads;
  const dim3 grid((unsigned)rows), block(threads);
  auto bf = [](const uint16_t* p) { return reinterpret_cast<const __nv_bfloat16*>(p); };
  // grid of the integer sum of squares: cols squares below 2^16 each must
  // stay under 2^64
  int lg = 0;
  while ((1 << lg) < cols) ++lg;
  const int sbits = 63 - 16 - lg;
  auto go = [&](auto kern) {
    return launch_kernel(pdl, grid, block, 0, stream, kern, bf(x), bf(res), bf(gamma),
                         eps, cols, reinterpret_cast<__nv_bfloat16*>(res_out),
                         dst_rows, copies, extra_row_base, out_q, out_scale,
                         bf(gate_w), gate_out, sbits, out_rows, device_error_word());
  };
  if (units <= 1) return go(add_rmsnorm_quant_kernel<1>);
  if (units <= 2) return go(add_rmsnorm_quant_kernel<2>);
  return go(add_rmsnorm_quant_kernel<4>);
}

// bound[g] = max over n of scale[g, n]: one block per group. The scales are
// positive (max(amax, 1e-12) / 448), and fmaxf is exact, so the result is
// independent of the reduction order.
__global__ void __launch_bounds__(256) scale_max_kernel(const float* __restrict__ scale,
                                                        int N, float* __restrict__ bound) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float part[8];
  const float* row = scale + (int64_t)blockIdx.x * N;
  float m = 0.f;
  for (int n = threadIdx.x; n < N; n += 256) m = fmaxf(m, row[n]);
  m = warp_max(m);
  if (lane_id() == 0) part[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = part[0];
    for (int w = 1; w < 8; ++w) r = fmaxf(r, part[w]);
    bound[blockIdx.x] = r;
  }
}

cudaError_t launch_scale_max(const float* scale, int groups, int N, float* bound,
                             cudaStream_t stream, bool pdl) {
  if (groups == 0) return cudaSuccess;
  return launch_kernel(pdl, dim3(groups), dim3(256), 0, stream, scale_max_kernel,
                       scale, N, bound);
}

cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* w_g, int T,
                               int D, float* gate, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return launch_kernel(false, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, stream,
                       shared_gate_kernel,
                       reinterpret_cast<const __nv_bfloat16*>(x),
                       reinterpret_cast<const __nv_bfloat16*>(w_g), T, D, gate);
}

}  // namespace moe
