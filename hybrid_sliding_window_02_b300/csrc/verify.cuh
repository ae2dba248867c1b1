// verify.cuh -- multi-token verify against the ring cache, general kernel.
//
// Speculative decoding with multi-token prediction ("MiMo-V2-Flash Technical
// Report" summary, section 核心方法: MTP drafts checked by the main model)
// runs the attention of L drafted tokens at positions pos .. pos+L-1 in one
// pass.  Their keys and values arrive with the call (k_new, v_new); the
// W-slot ring holds the tokens before them, slot s at position
// p(s) = (pos-1) - ((pos-1-s) mod W), empty when p(s) < 0 (the fixed O(W)
// cache of the "pwwt.cn" essay, section 1.1).  New token j attends to the
// keys at positions [pos+j-W+1, pos+j], as every prefill row does: the ring
// slots whose positions fall there, then new tokens 0..j.  Rejected drafts
// never enter the ring; the accepted ones are appended afterwards.
//
// One warp per output row (b, j, h), lanes over the head dimension, online
// softmax whose denominator starts with the sink term.  Serves every shape the
// tensor-core verify kernel does not take.
#pragma once

#include "device_common.cuh"
#include "simt_fwd.cuh"

namespace swa {

template <typename Tin, int D>
__global__ void __launch_bounds__(256) verify_simt_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k_new, const Tin* __restrict__ v_new,
    const Tin* __restrict__ k_ring, const Tin* __restrict__ v_ring,
    const int64_t* __restrict__ pos, const float* __restrict__ sink, float* __restrict__ out,
    float* __restrict__ lse, int B, int L, int Hq, int Hkv, int W, float scale) {
  constexpr int DPL = D / 32;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (int64_t)B * L * Hq) return;
  const int h = (int)(row % Hq);
  const int64_t bj = row / Hq;
  const int j = (int)(bj % L);
  const int b = (int)(bj / L);
  const int kvh = h / (Hq / Hkv);
  const int64_t p0 = pos[b];
  const int64_t lo = p0 + j - W + 1;  // first position in this token's window

  float qr[DPL];
  const Tin* qp = q + (((int64_t)b * L + j) * Hq + h) * D + lane * DPL;
#pragma unroll
  for (int t = 0; t < DPL; ++t) qr[t] = to_f32(qp[t]);
  const float s_h = sink[h];
  float m = s_h;
  float l = (s_h == -INFINITY) ? 0.f : 1.f;
  float acc[DPL];
#pragma unroll
  for (int t = 0; t < DPL; ++t) acc[t] = 0.f;

  auto visit = [&](const Tin* kp, const Tin* vp) {
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
    const float pr = expf(x - m);
    l += pr;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[t] = fmaf(pr, to_f32(vp[t]), acc[t]);
  };

  if (p0 >= 0) {
    const int64_t ring0 = ((int64_t)b * Hkv + kvh) * W * D + lane * DPL;
    for (int s = 0; s < W; ++s) {
      const int64_t a = p0 - 1 - s;
      const int64_t ps = p0 - 1 - (((a % W) + W) % W);
      if (ps < 0 || ps < lo) continue;
      visit(k_ring + ring0 + (int64_t)s * D, v_ring + ring0 + (int64_t)s * D);
    }
    for (int i = 0; i <= j; ++i) {
      if (p0 + i < lo) continue;
      const int64_t off = (((int64_t)b * L + i) * Hkv + kvh) * D + lane * DPL;
      visit(k_new + off, v_new + off);
    }
  }
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  float* op = out + (((int64_t)b * L + j) * Hq + h) * D + lane * DPL;
#pragma unroll
  for (int t = 0; t < DPL; ++t) op[t] = acc[t] * inv_l;
  if (lse != nullptr && lane == 0) lse[((int64_t)b * Hq + h) * L + j] = m + logf(l);
}

}  // namespace swa
