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
// memory) and only the rotation runs in fp32.  The frequencies f_i come from
// the host as an fp64 table: this GPU's fp64 rate is low, and an fp64 exp2 per
// angle cost more than the whole memory traffic of a decode step's rotation.
#pragma once

#include "device_common.cuh"
#include "griddep.cuh"
#include "simt_fwd.cuh"

namespace swa {

constexpr int kRopeThreads = 256;
constexpr int kRopeMaxHalf = 64;   // rot_dim <= 128

constexpr int kRopeMaxTok = 8;   // tokens per block of rope_inplace_kernel

// f[i] = theta^(-2 i / rot_dim), i < rot_dim / 2, computed on the host in fp64.
struct RopeFreq {
  double f[kRopeMaxHalf];
};

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

// cos and sin of a = p * f: the product and its reduction to [-pi, pi] in
// fp64 (a multiply, a rint and an fma), the sine and cosine in fp32.
__device__ __forceinline__ void rope_angle(int64_t p, double f, float& c, float& s) {
  const double two_pi = 6.283185307179586476925286766559;
  const double inv_two_pi = 0.15915494309189533576888376337251;
  const double a = (double)p * f;
  const double r = fma(-rint(a * inv_two_pi), two_pi, a);
  sincosf((float)r, &s, &c);
}

// cos / sin of a_i = p * f_i for i < half, into shared memory.
__device__ __forceinline__ void rope_angles(int64_t p, int half, const RopeFreq& fr, float* cs,
                                            float* sn) {
  for (int i = threadIdx.x; i < half; i += blockDim.x) rope_angle(p, fr.f[i], cs[i], sn[i]);
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

// One 16-byte chunk pair of a row, elements [i0, i0 + V) (ra) and their
// partners [i0 + half, i0 + half + V) (rb), rotated and stored to dst.  i0
// and half are multiples of V and the row is 16-byte aligned.
template <typename Tin>
__device__ __forceinline__ void rope_pair_chunk(uint4 ra, uint4 rb, Tin* dst, int i0, int half,
                                                const float* cs, const float* sn) {
  const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
  uint32_t ya[4], yb[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    if constexpr (sizeof(Tin) == 2) {
      // two bf16 per word, the lower element in the low half
      const int i = i0 + 2 * w;
      const float a0 = __uint_as_float(wa[w] << 16), a1 = __uint_as_float(wa[w] & 0xffff0000u);
      const float b0 = __uint_as_float(wb[w] << 16), b1 = __uint_as_float(wb[w] & 0xffff0000u);
      ya[w] = pack_bf16x2(a0 * cs[i] - b0 * sn[i], a1 * cs[i + 1] - b1 * sn[i + 1]);
      yb[w] = pack_bf16x2(b0 * cs[i] + a0 * sn[i], b1 * cs[i + 1] + a1 * sn[i + 1]);
    } else {
      const int i = i0 + w;
      const float a = __uint_as_float(wa[w]), b = __uint_as_float(wb[w]);
      ya[w] = __float_as_uint(a * cs[i] - b * sn[i]);
      yb[w] = __float_as_uint(b * cs[i] + a * sn[i]);
    }
  }
  *reinterpret_cast<uint4*>(dst + i0) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
  *reinterpret_cast<uint4*>(dst + i0 + half) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
}

// In place on x [B, T, H, D]: token (b, t) at position pos0[b] + t.  Each
// block takes tpb consecutive tokens at a time (grid-stride), so that a
// tensor with few heads still gives every thread work; the tokens' angles
// are formed once per block.  With vec (half a multiple of V, rows 16-byte
// aligned) a task is one 16-byte chunk pair of one head, two per thread per
// round, and the first round's chunks are loaded before the angles are
// formed; otherwise (tpb = 1) element by element.
template <typename Tin>
__global__ void __launch_bounds__(kRopeThreads) rope_inplace_kernel(
    Tin* __restrict__ x, const int64_t* __restrict__ pos0, int B, int T, int H, int D, int half,
    int vec, int tpb, const __grid_constant__ RopeFreq fr) {
  __shared__ float cs[kRopeMaxTok][kRopeMaxHalf], sn[kRopeMaxTok][kRopeMaxHalf];
  constexpr int V = 16 / (int)sizeof(Tin);
  const int nr = half / V;   // chunk pairs per head
  const int n = H * nr;      // tasks per token
  const int64_t ntok = (int64_t)B * T;
  for (int64_t tok0 = (int64_t)blockIdx.x * tpb; tok0 < ntok; tok0 += (int64_t)gridDim.x * tpb) {
    const int nt = (int)min((int64_t)tpb, ntok - tok0);
    auto angles = [&]() {
      for (int idx = threadIdx.x; idx < nt * half; idx += blockDim.x) {
        const int tt = idx / half, i = idx - tt * half;
        const int64_t tok = tok0 + tt;
        const int b = (int)(tok / T);
        const int64_t p = pos0[b] + (tok - (int64_t)b * T);
        rope_angle(p, fr.f[i], cs[tt][i], sn[tt][i]);
      }
    };
    __syncthreads();  // the previous tokens' angles are no longer read
    if (vec) {
      const int ntask = nt * n;
      uint4 ra[2], rb[2];
      auto row_of = [&](int j, int& i0) -> Tin* {
        const int tt = j / n, jj = j - tt * n;
        const int h = jj / nr;
        i0 = (jj - h * nr) * V;
        return x + ((tok0 + tt) * H + h) * D;
      };
      auto load = [&](int j0) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = j0 + k * (int)blockDim.x;
          if (j < ntask) {
            int i0;
            const Tin* row = row_of(j, i0);
            ra[k] = *reinterpret_cast<const uint4*>(row + i0);
            rb[k] = *reinterpret_cast<const uint4*>(row + i0 + half);
          }
        }
      };
      load(threadIdx.x);
      angles();
      __syncthreads();
      for (int j0 = threadIdx.x; j0 < ntask; j0 += 2 * (int)blockDim.x) {
        if (j0 != (int)threadIdx.x) load(j0);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = j0 + k * (int)blockDim.x;
          if (j < ntask) {
            int i0;
            Tin* row = row_of(j, i0);
            const int tt = j / n;
            rope_pair_chunk<Tin>(ra[k], rb[k], row, i0, half, cs[tt], sn[tt]);
          }
        }
      }
      continue;
    }
    angles();
    __syncthreads();
    // thread -> (head, pair): pairs of consecutive threads share a head
    Tin* base = x + tok0 * H * D;
    for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
      const int h = idx / half, i = idx - h * half;
      Tin* v = base + (int64_t)h * D;
      const float x0 = to_f32(v[i]), x1 = to_f32(v[i + half]);
      v[i] = from_f32<Tin>(x0 * cs[0][i] - x1 * sn[0][i]);
      v[i + half] = from_f32<Tin>(x1 * cs[0][i] + x0 * sn[0][i]);
    }
  }
}

// Work of one token's fused step in 16-byte chunks of V elements, in this
// order: q rows rotated (Hq x half/V chunk pairs), q's dimensions past rot_dim
// copied when q_out is not q_in (Hq x (D - rot_dim)/V), k rows rotated into
// the ring slot (Hkv x half/V) and their dimensions past rot_dim copied (Hkv x
// (D - rot_dim)/V), v rows copied (Hkv x D/V).
struct RopeAppendTasks {
  int nr, np, nd;      // chunks per row: rotated pairs, past rot_dim, whole row
  int qr, qp, kr, kp, v;
  __host__ __device__ int total() const { return qr + qp + kr + kp + v; }
};

__host__ __device__ inline RopeAppendTasks rope_append_tasks(int Hq, int Hkv, int D, int half,
                                                             int V, bool q_copy) {
  RopeAppendTasks t;
  t.nr = half / V;
  t.np = (D - 2 * half) / V;
  t.nd = D / V;
  t.qr = Hq * t.nr;
  t.qp = q_copy ? Hq * t.np : 0;
  t.kr = Hkv * t.nr;
  t.kp = Hkv * t.np;
  t.v = Hkv * t.nd;
  return t;
}

// The new token of sequence b at position pos[b]: q_out[b] = rope(q_in[b]),
// k_ring[b, g, pos mod W] = rope(k_in[b, g]), v_ring[b, g, pos mod W] =
// v_in[b, g].  A negative pos leaves q_out[b] and the rings untouched.
// Grid (B, S): with vec (half a multiple of V, every row 16-byte aligned) the
// S blocks of a token share its chunk tasks, so that every task's loads are in
// flight at once; otherwise block (b, 0) does the token element by element.
template <typename Tin>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(
    const Tin* q_in, const Tin* __restrict__ k_in, const Tin* __restrict__ v_in, Tin* q_out,
    Tin* __restrict__ k_ring, Tin* __restrict__ v_ring, const int64_t* __restrict__ pos, int Hq,
    int Hkv, int D, int W, int half, int vec, const __grid_constant__ RopeFreq fr) {
  __shared__ float cs[kRopeMaxHalf], sn[kRopeMaxHalf];
  // a decode launched after this step may start its set-up now; it waits for
  // this grid to complete before it touches memory
  if (threadIdx.x == 0) grid_dep_launch();
  const int b = blockIdx.x;
  const int64_t p = pos[b];
  if (p < 0) return;
  if (!vec && blockIdx.y != 0) return;
  const int64_t slot = p % W;
  const Tin* qi = q_in + (int64_t)b * Hq * D;
  Tin* qo = q_out + (int64_t)b * Hq * D;
  const Tin* ki = k_in + (int64_t)b * Hkv * D;
  const Tin* vi = v_in + (int64_t)b * Hkv * D;
  Tin* kr = k_ring + ((int64_t)b * Hkv * W + slot) * D;   // row g at kr + g W D
  Tin* vr = v_ring + ((int64_t)b * Hkv * W + slot) * D;
  const int64_t ring_row = (int64_t)W * D;
  if (vec) {
    constexpr int V = 16 / (int)sizeof(Tin);
    const RopeAppendTasks tk = rope_append_tasks(Hq, Hkv, D, half, V, q_in != q_out);
    const int n = tk.total();
    // task t: source row, destination row, first element, rotated or copied
    auto locate = [&](int t, const Tin*& src, Tin*& dst, int& i0, bool& rot) {
      int u = t;
      if (u < tk.qr) {
        const int h = u / tk.nr;
        src = qi + (int64_t)h * D, dst = qo + (int64_t)h * D, i0 = (u - h * tk.nr) * V, rot = true;
        return;
      }
      u -= tk.qr;
      if (u < tk.qp) {
        const int h = u / tk.np;
        src = qi + (int64_t)h * D, dst = qo + (int64_t)h * D;
        i0 = 2 * half + (u - h * tk.np) * V, rot = false;
        return;
      }
      u -= tk.qp;
      if (u < tk.kr) {
        const int g = u / tk.nr;
        src = ki + (int64_t)g * D, dst = kr + g * ring_row, i0 = (u - g * tk.nr) * V, rot = true;
        return;
      }
      u -= tk.kr;
      if (u < tk.kp) {
        const int g = u / tk.np;
        src = ki + (int64_t)g * D, dst = kr + g * ring_row;
        i0 = 2 * half + (u - g * tk.np) * V, rot = false;
        return;
      }
      u -= tk.kp;
      const int g = u / tk.nd;
      src = vi + (int64_t)g * D, dst = vr + g * ring_row, i0 = (u - g * tk.nd) * V, rot = false;
    };
    // the first task's chunks are loaded before the angles are formed, so
    // that their latency overlaps the angle arithmetic
    const int stride = gridDim.y * blockDim.x;
    int t = blockIdx.y * blockDim.x + threadIdx.x;
    const Tin* src = nullptr;
    Tin* dst = nullptr;
    int i0 = 0;
    bool rot = false;
    uint4 ra = make_uint4(0u, 0u, 0u, 0u), rb = ra;
    if (t < n) {
      locate(t, src, dst, i0, rot);
      ra = *reinterpret_cast<const uint4*>(src + i0);
      if (rot) rb = *reinterpret_cast<const uint4*>(src + i0 + half);
    }
    rope_angles(p, half, fr, cs, sn);
    __syncthreads();
    for (bool first = true; t < n; t += stride, first = false) {
      if (!first) {
        locate(t, src, dst, i0, rot);
        ra = *reinterpret_cast<const uint4*>(src + i0);
        if (rot) rb = *reinterpret_cast<const uint4*>(src + i0 + half);
      }
      if (rot)
        rope_pair_chunk<Tin>(ra, rb, dst, i0, half, cs, sn);
      else
        *reinterpret_cast<uint4*>(dst + i0) = ra;
    }
    return;
  }
  rope_angles(p, half, fr, cs, sn);
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int h = warp; h < Hq + 2 * Hkv; h += nw) {
    if (h < Hq) {
      rope_rotate_vec<Tin>(qi + (int64_t)h * D, qo + (int64_t)h * D, D, half, cs, sn, lane, 32);
    } else if (h < Hq + Hkv) {
      const int g = h - Hq;
      rope_rotate_vec<Tin>(ki + (int64_t)g * D, kr + g * ring_row, D, half, cs, sn, lane, 32);
    } else {
      const int g = h - Hq - Hkv;
      for (int d = lane; d < D; d += 32) vr[g * ring_row + d] = vi[(int64_t)g * D + d];
    }
  }
}

}  // namespace swa
