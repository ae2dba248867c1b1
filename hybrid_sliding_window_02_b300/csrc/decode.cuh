// decode.cuh -- one-token decode against the W-slot ring cache, and the ring
// append that precedes it.
//
// The ring ("pwwt.cn" MiMo-V2-Flash essay, section 1.1: the sliding-window KV
// cache has a fixed size, O(W) memory, independent of sequence length) holds,
// in slot s, position p(s) = pos - ((pos - s) mod W); slots with p(s) < 0 are
// empty.  Positions only grow as the window slides (ICML 2026 talk write-up,
// Q&A K), so the token at pos overwrote slot pos mod W.
//
// Decode is bound by HBM traffic: each (sequence, kv head) reads its W x D keys
// and values once.  One CTA per (b, kv head): a single thread issues three
// bulk copies (TMA, cp.async.bulk) of the contiguous key ring, value ring and
// the G query rows of the group into shared memory, so the whole 64 KB per CTA
// is in flight at once; scores start as soon as keys and queries land, while
// values are still arriving.  Eight warps then compute the G x W scores,
// the sink-seeded softmax and the G x D outputs from shared memory.  G is
// 1, 2, 4, 8 or 16 per CTA; a kv head with another number of query heads runs
// as sibling CTAs of the largest of those that divides it, each reading the
// rings.
#pragma once

#include "device_common.cuh"
#include "griddep.cuh"

namespace swa {

constexpr int kDecodeThreads = 256;
constexpr int kDecodeWarps = kDecodeThreads / 32;
constexpr int kDecodeMaxRingBytes = 163840;  // 2 * W * D * sizeof(Tin) limit

// Shared-memory carve-up (bytes) for one decode CTA.
struct DecodeSmem {
  int k_off, v_off, q_off, p_off, linv_off, bar_off, total;
};

template <typename Tin, int D, int G>
__host__ __device__ inline DecodeSmem decode_smem_layout(int W) {
  DecodeSmem s;
  const int ring = W * D * (int)sizeof(Tin);
  const int red = kDecodeWarps * G * D * 4;  // cross-warp partial sums alias the key ring
  const int kreg = ring > red ? ring : red;
  s.k_off = 0;
  s.v_off = (kreg + 127) & ~127;
  s.q_off = s.v_off + ((ring + 127) & ~127);
  s.p_off = s.q_off + ((G * D * (int)sizeof(Tin) + 127) & ~127);
  s.linv_off = s.p_off + ((W * G * 4 + 127) & ~127);
  s.bar_off = s.linv_off + ((G * 4 + 127) & ~127);
  s.total = s.bar_off + 64;
  return s;
}

__host__ __device__ constexpr int log2i(int x) { return x <= 1 ? 0 : 1 + log2i(x / 2); }

template <typename Tin>
struct Vec16;  // 16 bytes of input elements, widened to fp32
template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const void* p, float (&f)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      f[2 * t] = __uint_as_float(w[t] << 16);
      f[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
    }
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const void* p, float (&f)[4]) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    f[0] = u.x; f[1] = u.y; f[2] = u.z; f[3] = u.w;
  }
};

template <typename Tin, int D, int G>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k_ring, const Tin* __restrict__ v_ring,
    const int64_t* __restrict__ pos, const float* __restrict__ sink, float* __restrict__ out,
    float* __restrict__ lse, int Hq, int Hkv, int W, int rep, float scale_log2) {
  constexpr int EPL = Vec16<Tin>::N;       // elements per 16-byte lane chunk
  constexpr int LPK = D / EPL;             // lanes per key row
  constexpr int KPW = 32 / LPK;            // keys per warp instruction
  extern __shared__ __align__(128) uint8_t smem[];
  const DecodeSmem L = decode_smem_layout<Tin, D, G>(W);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // CTA = (sequence b, kv head, sibling): a kv head's G R query heads run as
  // R sibling CTAs of G heads each (rep = R), every one reading the rings
  const int bk = blockIdx.x / rep;         // ring unit b * Hkv + kv head
  const int b = bk / Hkv;
  const int qg = (bk % Hkv) * rep + (int)(blockIdx.x % rep);   // query group: heads qg G ..
  const uint32_t bar_kq = smem_u32(smem + L.bar_off);
  const uint32_t bar_v = bar_kq + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.bar_off + 16);

  const int64_t ring_elems = (int64_t)W * D;
  const uint32_t ring_bytes = (uint32_t)(ring_elems * sizeof(Tin));
  const uint32_t q_bytes = (uint32_t)(G * D * sizeof(Tin));
  if (tid == 0) {
    *abort_flag = 0;
    mbar_init(bar_kq, 1);
    mbar_init(bar_v, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_kq, ring_bytes + q_bytes);
    tma_load_1d(smem_u32(smem + L.k_off), k_ring + (int64_t)bk * ring_elems, ring_bytes, bar_kq);
    tma_load_1d(smem_u32(smem + L.q_off), q + ((int64_t)b * Hq + qg * G) * D, q_bytes, bar_kq);
    mbar_arrive_expect_tx(bar_v, ring_bytes);
    tma_load_1d(smem_u32(smem + L.v_off), v_ring + (int64_t)bk * ring_elems, ring_bytes, bar_v);
  }
  const int64_t p_now = pos[b];
  // slot s holds position pos - ((pos - s) mod W): with pos >= W-1 every slot
  // is filled; otherwise exactly the slots s <= pos are (position s).
  const bool ring_full = p_now >= (int64_t)W - 1;
  auto slot_valid = [&](int s) { return ring_full || (int64_t)s <= p_now; };

  // ---- scores: warp w takes keys w*KPW + kg, stepping by 8*KPW ----------------
  const int kg = lane / LPK;             // key within the warp instruction
  const int dc = (lane % LPK) * EPL;     // first head-dim element of this lane
  const bool kq_ok = mbar_wait(bar_kq, 0, kErrWaitDecode, abort_flag);
  float* P = reinterpret_cast<float*>(smem + L.p_off);  // P[s * G + g]
  if (kq_ok) {
    float qf[G][EPL];
    const Tin* qs = reinterpret_cast<const Tin*>(smem + L.q_off);
#pragma unroll
    for (int g = 0; g < G; ++g) Vec16<Tin>::load(qs + g * D + dc, qf[g]);
    const Tin* ks = reinterpret_cast<const Tin*>(smem + L.k_off);
    for (int s0 = warp * KPW; s0 < W; s0 += kDecodeWarps * KPW) {
      const int s = s0 + kg;
      float kf[EPL];
      float part[G];
      if (s < W) {
        Vec16<Tin>::load(ks + (int64_t)s * D + dc, kf);
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) kf[e] = 0.f;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) a = fmaf(qf[g][e], kf[e], a);
        part[g] = a;
      }
      // Sum the G partial dots over the LPK lanes of this key.  Each step
      // halves the values a lane keeps (it sends the other half to its
      // partner), so a lane ends with NV complete sums for heads hoff.. .
      int hoff = 0;
      constexpr int NV = (G >> log2i(LPK)) > 0 ? (G >> log2i(LPK)) : 1;
      const int l = lane % LPK;
#pragma unroll
      for (int off = LPK / 2, c = G; off > 0; off >>= 1) {
        if (c > 1) {
          const int half = c / 2;
          const bool upper = (l & off) != 0;
#pragma unroll
          for (int j = 0; j < half; ++j) {
            const float send = upper ? part[j] : part[j + half];
            const float keep = upper ? part[j + half] : part[j];
            part[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
          }
          if (upper) hoff += half;
          c = half;
        } else {
          part[0] += __shfl_xor_sync(0xffffffffu, part[0], off);
        }
      }
      // lanes that share hoff hold identical sums: the lowest of them writes
      const int dup = LPK / (G / NV);  // lanes per distinct hoff
      if (s < W && (l % dup) == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) P[s * G + hoff + j] = part[j] * scale_log2;
      }
    }
  }
  __syncthreads();

  // ---- sink-seeded softmax over the valid slots, one head per warp ----------
  float* linv = reinterpret_cast<float*>(smem + L.linv_off);
  if (kq_ok) {
    for (int g = warp; g < G; g += kDecodeWarps) {
      const int h = qg * G + g;
      const float sk = sink[h] * 1.4426950408889634f;  // log2(e)
      float m = sk;
      for (int s = lane; s < W; s += 32) {
        if (slot_valid(s)) m = fmaxf(m, P[s * G + g]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float l = 0.f;
      for (int s = lane; s < W; s += 32) {
        const float e = slot_valid(s) ? ex2_approx(P[s * G + g] - m) : 0.f;
        P[s * G + g] = e;
        l += e;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      // sink term; a -inf sink contributes nothing (and m then comes from a key)
      if (sk != -INFINITY) l += ex2_approx(sk - m);
      if (lane == 0) {
        linv[g] = l > 0.f ? 1.f / l : 0.f;  // no valid slot and a -inf sink: out = 0
        if (lse != nullptr) lse[(int64_t)b * Hq + h] = (m + __log2f(l)) * 0.6931471805599453f;
      }
    }
  }
  const bool v_ok = kq_ok && mbar_wait(bar_v, 0, kErrWaitDecode, abort_flag);
  __syncthreads();

  // ---- values: same key split as the scores, then a cross-warp sum ----------
  float* red = reinterpret_cast<float*>(smem + L.k_off);  // keys are dead now
  if (v_ok) {
    float acc[G][EPL];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
    const Tin* vs = reinterpret_cast<const Tin*>(smem + L.v_off);
    for (int s0 = warp * KPW; s0 < W; s0 += kDecodeWarps * KPW) {
      const int s = s0 + kg;
      // empty slots (position < 0) may hold anything, NaN included: skip them
      const bool valid = s < W && slot_valid(s);
      if (valid) {
        float vf[EPL];
        Vec16<Tin>::load(vs + (int64_t)s * D + dc, vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float p = P[s * G + g];
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
        }
      }
    }
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], off);
    }
    if (kg == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < EPL; ++e) red[(warp * G + g) * D + dc + e] = acc[g][e];
    }
  }
  __syncthreads();
  if (v_ok) {
    float* ob = out + ((int64_t)b * Hq + qg * G) * D;
    for (int o = tid; o < G * D; o += kDecodeThreads) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) a += red[w * G * D + o];
      ob[o] = a * linv[o / D];
    }
  }
}

// ring append: k_ring[b, g, pos mod W, :] = k_new[b, g, :] (and the same for v)
template <typename Tin>
__global__ void ring_append_kernel(const Tin* __restrict__ k_new, const Tin* __restrict__ v_new,
                                   Tin* __restrict__ k_ring, Tin* __restrict__ v_ring,
                                   const int64_t* __restrict__ pos, int B, int Hkv, int D, int W) {
  // a decode launched after the append may start its set-up now; it waits for
  // this grid to complete before it touches memory
  if (threadIdx.x == 0) grid_dep_launch();
  constexpr int EPV = 16 / sizeof(Tin);
  const int vecs_per_row = D / EPV;
  const int64_t total = (int64_t)B * Hkv * vecs_per_row;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bg = t / vecs_per_row;
    const int c = (int)(t % vecs_per_row);
    const int b = (int)(bg / Hkv);
    const int64_t p = pos[b];
    if (p < 0) continue;
    const int64_t slot = p % W;
    const int64_t src = bg * D + (int64_t)c * EPV;
    const int64_t dst = (bg * W + slot) * D + (int64_t)c * EPV;
    *reinterpret_cast<uint4*>(k_ring + dst) = *reinterpret_cast<const uint4*>(k_new + src);
    *reinterpret_cast<uint4*>(v_ring + dst) = *reinterpret_cast<const uint4*>(v_new + src);
  }
}

}  // namespace swa
