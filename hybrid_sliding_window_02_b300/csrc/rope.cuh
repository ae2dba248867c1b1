// rope.cuh -- rotary position embedding at absolute positions, and the fused
// step that precedes a decode: rotate the new token's q and k, write k and v
// into ring slot pos mod W.
//
// RoPE's theta is fixed at inference and the position index keeps counting up
// while the window slides (ICML 2026 talk write-up, Q&A K), so a token is
// rotated at its absolute position p, which reaches 2^18 and beyond.  The
// pages give no variant; this is the rotate-half form over the first rot_dim
// dimensions, angle a_i = p * theta^(-2 i / rot_dim) for pair (i, i + rot_dim/2).
// At p = 262143 an fp32 product p * f has an absolute error near 0.016 rad, too
// coarse for bf16 outputs, so each token's angles are formed and reduced
// modulo 2 pi in fp64 (once per token, shared by all heads through shared
// memory) and only the rotation runs in fp32.
#pragma once

#include "device_common.cuh"
#include "simt_fwd.cuh"

namespace swa {

constexpr int kRopeThreads = 256;
constexpr int kRopeMaxHalf = 64;   // rot_dim <= 128

template <typename Tin>
__device__ __forceinline__ Tin from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// cos / sin of a_i = p * theta^(-2 i / rot_dim) for i < half, into shared memory.
__device__ __forceinline__ void rope_angles(int64_t p, int half, double log2_theta,
                                            float* cs, float* sn) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double f = exp2(-(2.0 * i / (2 * half)) * log2_theta);
    const double a = (double)p * f;
    const double r = a - two_pi * rint(a / two_pi);  // in [-pi, pi]
    float s, c;
    sincosf((float)r, &s, &c);
    cs[i] = c;
    sn[i] = s;
  }
}

// Rotate one D-vector (src -> dst; they may alias) with the angles in cs / sn.
template <typename Tin>
__device__ __forceinline__ void rope_rotate_vec(const Tin* src, Tin* dst, int D, int half,
                                                const float* cs, const float* sn, int lane0,
                                                int stride) {
  for (int i = lane0; i < half; i += stride) {
    const float x0 = to_f32(src[i]), x1 = to_f32(src[i + half]);
    const float y0 = x0 * cs[i] - x1 * sn[i];
    const float y1 = x1 * cs[i] + x0 * sn[i];
    dst[i] = from_f32<Tin>(y0);
    dst[i + half] = from_f32<Tin>(y1);
  }
  if (src != dst)
    for (int d = 2 * half + lane0; d < D; d += stride) dst[d] = src[d];
}

// In place on x [B, T, H, D]: token (b, t) at position pos0[b] + t.  One block
// per token (grid-stride over tokens).
template <typename Tin>
__global__ void __launch_bounds__(kRopeThreads) rope_inplace_kernel(
    Tin* __restrict__ x, const int64_t* __restrict__ pos0, int B, int T, int H, int D, int half,
    double log2_theta) {
  __shared__ float cs[kRopeMaxHalf], sn[kRopeMaxHalf];
  const int64_t ntok = (int64_t)B * T;
  for (int64_t tok = blockIdx.x; tok < ntok; tok += gridDim.x) {
    const int b = (int)(tok / T);
    const int t = (int)(tok - (int64_t)b * T);
    __syncthreads();  // previous token's angles are no longer read
    rope_angles(pos0[b] + t, half, log2_theta, cs, sn);
    __syncthreads();
    Tin* base = x + tok * H * D;
    // thread -> (head, pair): pairs of consecutive threads share a head
    for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
      const int h = idx / half, i = idx - h * half;
      Tin* v = base + (int64_t)h * D;
      const float x0 = to_f32(v[i]), x1 = to_f32(v[i + half]);
      v[i] = from_f32<Tin>(x0 * cs[i] - x1 * sn[i]);
      v[i + half] = from_f32<Tin>(x1 * cs[i] + x0 * sn[i]);
    }
  }
}

// The new token of sequence b at position pos[b]: q_out[b] = rope(q_in[b]),
// k_ring[b, g, pos mod W] = rope(k_in[b, g]), v_ring[b, g, pos mod W] =
// v_in[b, g].  A negative pos leaves q_out[b] and the rings untouched.
template <typename Tin>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(
    const Tin* __restrict__ q_in, const Tin* __restrict__ k_in, const Tin* __restrict__ v_in,
    Tin* __restrict__ q_out, Tin* __restrict__ k_ring, Tin* __restrict__ v_ring,
    const int64_t* __restrict__ pos, int Hq, int Hkv, int D, int W, int half,
    double log2_theta) {
  __shared__ float cs[kRopeMaxHalf], sn[kRopeMaxHalf];
  const int b = blockIdx.x;
  const int64_t p = pos[b];
  if (p < 0) return;
  rope_angles(p, half, log2_theta, cs, sn);
  __syncthreads();
  const int64_t slot = p % W;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int h = warp; h < Hq + 2 * Hkv; h += nw) {
    if (h < Hq) {
      const int64_t off = ((int64_t)b * Hq + h) * D;
      rope_rotate_vec<Tin>(q_in + off, q_out + off, D, half, cs, sn, lane, 32);
    } else if (h < Hq + Hkv) {
      const int g = h - Hq;
      rope_rotate_vec<Tin>(k_in + ((int64_t)b * Hkv + g) * D,
                           k_ring + (((int64_t)b * Hkv + g) * W + slot) * D, D, half, cs, sn,
                           lane, 32);
    } else {
      const int g = h - Hq - Hkv;
      const Tin* src = v_in + ((int64_t)b * Hkv + g) * D;
      Tin* dst = v_ring + (((int64_t)b * Hkv + g) * W + slot) * D;
      for (int d = lane; d < D; d += 32) dst[d] = src[d];
    }
  }
}

}  // namespace swa
