// simt_fwd.cuh -- general prefill kernel on the CUDA cores (fp32 FMA).
//
// Serves the fp32 path (whose accuracy bar rules out reduced-precision tensor
// cores) and any shape the tensor-core kernels do not cover.  One warp per
// output row (b, i, h); the 32 lanes split the head dimension, the warp walks
// the row's window [max(0, i-W+1), i] key by key with an online max/sum whose
// denominator starts with the sink term exp(s_h - m) ("MiMo-V2-Flash Technical
// Report" summary, 前置知识: sink bias in the softmax denominator).
#pragma once

#include "device_common.cuh"

namespace swa {

template <typename Tin>
__device__ __forceinline__ float to_f32(Tin x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename Tin, int D>
__global__ void __launch_bounds__(256) simt_fwd_kernel(const Tin* __restrict__ q,
                                                       const Tin* __restrict__ k,
                                                       const Tin* __restrict__ v,
                                                       const float* __restrict__ sink,
                                                       float* __restrict__ out,
                                                       float* __restrict__ lse, int B, int T,
                                                       int Hq, int Hkv, int W, float scale) {
  constexpr int DPL = D / 32;  // head-dim elements per lane
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t nrows = (int64_t)B * T * Hq;
  if (row >= nrows) return;
  // Row order (b, i, h), h fastest: neighbouring warps share key/value rows.
  const int h = (int)(row % Hq);
  const int64_t bi = row / Hq;
  const int i = (int)(bi % T);
  const int b = (int)(bi / T);
  const int kvh = h / (Hq / Hkv);

  float qr[DPL];
  const Tin* qp = q + (((int64_t)b * T + i) * Hq + h) * D + lane * DPL;
#pragma unroll
  for (int t = 0; t < DPL; ++t) qr[t] = to_f32(qp[t]);

  const float s_h = sink[h];
  float m = s_h;
  float l = (s_h == -INFINITY) ? 0.f : 1.f;  // exp(s_h - m) with m = s_h
  float acc[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) acc[t] = 0.f;

  const int j0 = max(0, i - W + 1);
  const int64_t kv_stride = (int64_t)Hkv * D;
  const Tin* kp = k + (((int64_t)b * T + j0) * Hkv + kvh) * D + lane * DPL;
  const Tin* vp = v + (((int64_t)b * T + j0) * Hkv + kvh) * D + lane * DPL;
  for (int j = j0; j <= i; ++j, kp += kv_stride, vp += kv_stride) {
    float part = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) part = fmaf(qr[t], to_f32(kp[t]), part);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    const float x = part * scale;
    if (x > m) {
      const float c = expf(m - x);
      l *= c;
#pragma unroll
      for (int t = 0; t < DPL; ++t) acc[t] *= c;
      m = x;
    }
    const float p = expf(x - m);
    l += p;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[t] = fmaf(p, to_f32(vp[t]), acc[t]);
  }
  const float inv_l = 1.f / l;
  float* op = out + (((int64_t)b * T + i) * Hq + h) * D + lane * DPL;
#pragma unroll
  for (int t = 0; t < DPL; ++t) op[t] = acc[t] * inv_l;
  if (lse != nullptr && lane == 0) lse[((int64_t)b * Hq + h) * T + i] = m + logf(l);
}

}  // namespace swa
