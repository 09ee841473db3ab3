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
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kUnit = 8;   // elements per lane per step

__device__ __forceinline__ void load_unit(const __nv_bfloat16* p, float (&v)[kUnit]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __low2float(h[i]);
    v[2 * i + 1] = __high2float(h[i]);
  }
}

__device__ __forceinline__ void load_unit(const float* p, float (&v)[kUnit]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename InT>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) quant_rows_kernel(
    const InT* __restrict__ in, int64_t rows, int cols,
    const int32_t* __restrict__ dst_rows, int copies, int64_t extra_row_base,
    uint8_t* __restrict__ out_q, float* __restrict__ out_scale,
    const __nv_bfloat16* __restrict__ gate_w, float* __restrict__ gate_out) {
  const int64_t r = (int64_t)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (r >= rows) return;
  const int lane = (int)lane_id();
  const InT* row = in + r * cols;

  // pass 1: row amax (and the shared-expert gate's dot product)
  float amax = 0.f, dot = 0.f;
  for (int c = lane * kUnit; c < cols; c += 32 * kUnit) {
    float v[kUnit];
    load_unit(row + c, v);
#pragma unroll
    for (int i = 0; i < kUnit; ++i) amax = fmaxf(amax, fabsf(v[i]));
    if (gate_w != nullptr) {
      float w[kUnit];
      load_unit(gate_w + c, w);
#pragma unroll
      for (int i = 0; i < kUnit; ++i) dot = fmaf(v[i], w[i], dot);
    }
  }
  amax = warp_max(amax);
  const float s = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);

  // destinations of this row
  const int ndst = (dst_rows != nullptr ? copies : 1) + (extra_row_base >= 0 ? 1 : 0);
  if (lane == 0) {
    for (int d = 0; d < ndst; ++d) {
      const int64_t o = d < (dst_rows != nullptr ? copies : 1)
                            ? (dst_rows != nullptr ? (int64_t)dst_rows[r * copies + d] : r)
                            : extra_row_base + r;
      out_scale[o] = s;
    }
    if (gate_w != nullptr) gate_out[r] = 0.f;  // placeholder, set below
  }
  if (gate_w != nullptr) {
    dot = warp_sum(dot);
    if (lane == 0) gate_out[r] = 1.0f / (1.0f + expf(-dot));
  }

  // pass 2: quantise and store to every destination
  for (int c = lane * kUnit; c < cols; c += 32 * kUnit) {
    float v[kUnit];
    load_unit(row + c, v);
    uint32_t packed[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(v[4 * i], s), __fdiv_rn(v[4 * i + 1], s));
      const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(v[4 * i + 2], s), __fdiv_rn(v[4 * i + 3], s));
      packed[i] = (uint32_t)lo | ((uint32_t)hi << 16);
    }
    const uint2 q = make_uint2(packed[0], packed[1]);
    for (int d = 0; d < ndst; ++d) {
      const int64_t o = d < (dst_rows != nullptr ? copies : 1)
                            ? (dst_rows != nullptr ? (int64_t)dst_rows[r * copies + d] : r)
                            : extra_row_base + r;
      *reinterpret_cast<uint2*>(out_q + o * cols + c) = q;
    }
  }
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) shared_gate_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
    int T, int D, float* __restrict__ gate) {
  const int t = blockIdx.x * kWarpsPerBlock + threadIdx.x / 32;
  if (t >= T) return;
  float dot = 0.f;
  for (int c = (int)lane_id() * kUnit; c < D; c += 32 * kUnit) {
    float v[kUnit], g[kUnit];
    load_unit(x + (int64_t)t * D + c, v);
    load_unit(w + c, g);
#pragma unroll
    for (int i = 0; i < kUnit; ++i) dot = fmaf(v[i], g[i], dot);
  }
  dot = warp_sum(dot);
  if (lane_id() == 0) gate[t] = 1.0f / (1.0f + expf(-dot));
}

}  // namespace

cudaError_t launch_quant(const void* in, int in_dtype, int64_t rows, int cols,
                         const int32_t* dst_rows, int copies,
                         int64_t extra_row_base, uint8_t* out_q,
                         float* out_scale, const uint16_t* gate_w,
                         float* gate_out, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const auto* gw = reinterpret_cast<const __nv_bfloat16*>(gate_w);
  if (in_dtype == 0) {
    quant_rows_kernel<__nv_bfloat16><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(in), rows, cols, dst_rows, copies,
        extra_row_base, out_q, out_scale, gw, gate_out);
  } else {
    quant_rows_kernel<float><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
        static_cast<const float*>(in), rows, cols, dst_rows, copies,
        extra_row_base, out_q, out_scale, nullptr, nullptr);
  }
  return cudaGetLastError();
}

cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* w_g, int T,
                               int D, float* gate, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  shared_gate_kernel<<<blocks, kWarpsPerBlock * 32, 0, stream>>>(
      reinterpret_cast<const __nv_bfloat16*>(x),
      reinterpret_cast<const __nv_bfloat16*>(w_g), T, D, gate);
  return cudaGetLastError();
}

}  // namespace moe
