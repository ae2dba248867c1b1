// verify_tc.cuh -- multi-token verify against the 128-slot ring with the ring
// contractions on the 5th-generation tensor cores.
//
// Operation: as in verify.cuh (drafted tokens at positions pos .. pos+L-1
// checked in one pass; "MiMo-V2-Flash Technical Report" summary, section
// 核心方法), for bf16 inputs, D = 128, W = 128, groups of 8 query heads and
// L <= 4 drafted tokens.  Per group (sequence b, kv head g) the 8L query rows
// r = 8 j + h (token j, head h; padded to 32) meet the 128 ring slots and the
// L new keys:
//   S^T = K_ring Q^T       tcgen05, M = 128 slots, N = 32 rows, K = 128 dims
//   new-key scores         CUDA cores: thread t takes row t / 4, new key t % 4
//   O^T = V_ring^T P^T     tcgen05, M = 128 dims (V MN-major), N = 32, K = 128
//   + P_new V_new          CUDA cores, thread = dim
// Like the decode kernel: persistent CTAs, a producer thread keeping two
// groups' K, V, Q and new K / V in flight (TMA; the new rows by bulk copies),
// one MMA thread, two softmax warpgroups on alternate groups.  A softmax
// thread holds one slot's 32 row scores; the max and the sum over slots are
// transposing warp-shuffle reductions (31 shuffles leave lane l with row l)
// finished across the four warps in shared memory.
#pragma once

#include "device_common.cuh"

namespace swa {
namespace vertc {

constexpr int kThreads = 320;
constexpr int kWarpProducer = 8, kWarpMma = 9;
constexpr int kG = 8;
constexpr int kLmax = 4;
constexpr int kN = 32;              // MMA N: rows 8 j + h, padded
constexpr int kW = 128;
constexpr int kD = 128;
constexpr uint32_t kStages = 2;

constexpr int kHalf = kW * 128;                 // 128 rows x 64 bf16
constexpr int kQHalf = kN * 128;                // 32 rows x 64 bf16
constexpr int kStageK = 0, kStageV = 2 * kHalf, kStageQ = 4 * kHalf;
constexpr int kStageKn = kStageQ + 2 * kQHalf;  // new keys [4][128] bf16, plain rows
constexpr int kStageVn = kStageKn + kLmax * kD * 2;
constexpr int kStageBytes = kStageVn + kLmax * kD * 2;  // 74 KB
constexpr int kPBytes = 2 * kQHalf;             // P^T: 32 rows x 128 slots bf16
constexpr int kOffStage = 0;
constexpr int kOffP = kOffStage + (int)kStages * kStageBytes;
// per warpgroup: red_max[4][32], red_sum[4][32], new_max[32], new_sum[32], pnew[32][4]
constexpr int kRedFloats = 4 * 32 + 4 * 32 + 32 + 32 + 32 * 4;
constexpr int kOffRed = kOffP + 2 * kPBytes;
constexpr int kOffBar = kOffRed + 2 * kRedFloats * 4;
constexpr int kBarFull = 0, kBarEmpty = kStages, kBarSFull = 2 * kStages,
              kBarPFull = kBarSFull + 2, kBarOFull = kBarPFull + 2, kBarRed = kBarOFull + 2,
              kBarDrain = kBarRed + 4, kNumBars = kBarDrain + 1;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;

constexpr uint32_t kTmemCols = 128;
__host__ __device__ constexpr uint32_t col_s(int w) { return 64u * (uint32_t)w; }
__host__ __device__ constexpr uint32_t col_o(int w) { return 64u * (uint32_t)w + 32u; }

struct Params {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int64_t* pos;
  const float* sink;
  float* out;
  float* lse;
  int B, L, Hq, Hkv;
  int units;          // B * Hkv
  float scale_log2;
};

// Lane l ends with the max (kMax) or sum over the warp's 32 lanes of v[l].
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16, n = 32; off >= 1; off >>= 1, n >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_q, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  const int nk = p.units > (int)blockIdx.x
                     ? (p.units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                     : 0;
  const int L = p.L;

  if (tid == 0) {
    *abort_flag = 0;
    for (uint32_t s = 0; s < kStages; ++s) {
      mbar_init(bar(kBarFull + s), 1);
      mbar_init(bar(kBarEmpty + s), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(kBarSFull + w), 1);
      mbar_init(bar(kBarPFull + w), 128);
      mbar_init(bar(kBarOFull + w), 1);
      mbar_init(bar(kBarRed + 2 * w), 128);
      mbar_init(bar(kBarRed + 2 * w + 1), 128);
    }
    mbar_init(bar(kBarDrain), 1);
    fence_mbar_init();
  }
  // New-key rows L..3 of both stages are never written by a copy: zero them
  // once (their weights are 0, and 0 * NaN would not be).
  for (int i = tid; i < (int)kStages * 2 * kLmax * kD * 2 / 16; i += kThreads) {
    const int st = i / (2 * kLmax * kD * 2 / 16), r = i % (2 * kLmax * kD * 2 / 16);
    st_shared_v4(sbase + kOffStage + st * kStageBytes + kStageKn + 16 * r, 0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (warp == kWarpMma) {
    tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    prefetch_tmap(&map_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (warp == kWarpProducer) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      const uint32_t bytes = 4 * kHalf + 2 * (8 * L * 128) + 2 * (L * kD * 2);
      int k = 0;
      for (; k < nk; ++k) {
        const int u = (int)blockIdx.x + k * (int)gridDim.x;
        const int b = u / p.Hkv, g = u - b * p.Hkv;
        const uint32_t s = (uint32_t)k % kStages;
        if (!mbar_wait(bar(kBarEmpty + s), (((uint32_t)k / kStages) & 1) ^ 1, kErrWaitKvEmpty,
                       abort_flag))
          break;
        const uint32_t st = sbase + kOffStage + s * kStageBytes;
        const uint32_t fb = bar(kBarFull + s);
        mbar_arrive_expect_tx(fb, bytes);
        tma_load_4d(st + kStageK, &map_k, 0, u * kW, 0, 0, fb);
        tma_load_4d(st + kStageK + kHalf, &map_k, 64, u * kW, 0, 0, fb);
        tma_load_4d(st + kStageV, &map_v, 0, u * kW, 0, 0, fb);
        tma_load_4d(st + kStageV + kHalf, &map_v, 64, u * kW, 0, 0, fb);
        tma_load_4d(st + kStageQ, &map_q, 0, g * kG, 0, b, fb);
        tma_load_4d(st + kStageQ + kQHalf, &map_q, 64, g * kG, 0, b, fb);
        for (int i = 0; i < L; ++i) {
          const int64_t row = ((int64_t)b * L + i) * p.Hkv + g;
          tma_load_1d(st + kStageKn + i * kD * 2, p.k_new + row * kD, kD * 2, fb);
          tma_load_1d(st + kStageVn + i * kD * 2, p.v_new + row * kD, kD * 2, fb);
        }
      }
      if (k < nk) {
        for (int j = (k > (int)kStages ? k - (int)kStages : 0); j < k; ++j)
          mbar_wait_drain(bar(kBarFull + (uint32_t)j % kStages), ((uint32_t)j / kStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_bf16(kN, false, false);
      const uint32_t idesc_o = umma_idesc_bf16(kN, true, false);
      auto issue_s = [&](int k) -> bool {
        const uint32_t s = (uint32_t)k % kStages;
        if (!mbar_wait(bar(kBarFull + s), ((uint32_t)k / kStages) & 1, kErrWaitKvFull,
                       abort_flag))
          return false;
        tc_fence_after();
        const uint32_t st = sbase + kOffStage + s * kStageBytes;
        const uint64_t kdesc = umma_sdesc(st + kStageK, 16, 1024, 2);
        const uint64_t qdesc = umma_sdesc(st + kStageQ, 16, 1024, 2);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t a_off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
          const uint32_t b_off = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
          umma_bf16_ss(tmem + col_s(k & 1), kdesc + a_off, qdesc + b_off, idesc_s, kk > 0);
        }
        umma_commit(bar(kBarSFull + (k & 1)));
        return true;
      };
      bool ok = nk > 0 && issue_s(0);
      for (int k = 0; ok && k < nk; ++k) {
        if (k + 1 < nk && !issue_s(k + 1)) break;
        const uint32_t s = (uint32_t)k % kStages;
        const int w = k & 1;
        if (!mbar_wait(bar(kBarPFull + w), ((uint32_t)k >> 1) & 1, kErrWaitPFull, abort_flag))
          break;
        tc_fence_after();
        const uint32_t st = sbase + kOffStage + s * kStageBytes;
        const uint64_t vdesc = umma_sdesc(st + kStageV, kHalf, 1024, 2);
        const uint64_t pdesc = umma_sdesc(sbase + kOffP + w * kPBytes, 16, 1024, 2);
#pragma unroll
        for (int kb = 0; kb < kW / 16; ++kb) {
          const uint32_t a_off = (kb * 16 * 128) >> 4;
          const uint32_t b_off = ((kb >> 2) * kQHalf + (kb & 3) * 32) >> 4;
          umma_bf16_ss(tmem + col_o(w), vdesc + a_off, pdesc + b_off, idesc_o, kb > 0);
        }
        umma_commit(bar(kBarOFull + w));
        umma_commit(bar(kBarEmpty + s));
      }
      umma_commit(bar(kBarDrain));
      mbar_wait_drain(bar(kBarDrain), 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax + output (warps 0..7) =======================
    const int w = warp >> 2;
    const int quad = warp & 3;
    const int t = quad * 32 + lane;            // slot (softmax) / dim (output)
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed) + w * kRedFloats;
    float* red_max = red;                      // [4][32]
    float* red_sum = red + 128;                // [4][32]
    float* new_max = red + 256;                // [32]
    float* new_sum = red + 288;                // [32]
    float* pnew = red + 320;                   // [32][4]
    const uint32_t pbuf = sbase + kOffP + w * kPBytes;
    const uint32_t bar_max = bar(kBarRed + 2 * w), bar_sum = bar(kBarRed + 2 * w + 1);
    const int nrow = kG * L;                   // live rows of N
    const int nr = t >> 2, ni = t & 3;         // new-key score pair of this thread
    for (int k = w; k < nk; k += 2) {
      const int u = (int)blockIdx.x + k * (int)gridDim.x;
      const int b = u / p.Hkv, g = u - b * p.Hkv;
      const uint32_t s = (uint32_t)k % kStages;
      const uint32_t st = sbase + kOffStage + s * kStageBytes;
      const int64_t p0 = p.pos[b];
      // position held by slot t (ring of the tokens before p0); window of row c
      // starts at p0 + c / 8 - (W - 1)
      const int64_t a = p0 - 1 - t;
      const int64_t pt = p0 - 1 - (((a % kW) + kW) % kW);
      const bool live = p0 >= 0 && pt >= 0;
      float sk8[kG];
#pragma unroll
      for (int h = 0; h < kG; ++h) sk8[h] = p.sink[g * kG + h] * 1.4426950408889634f;
      if (!mbar_wait(bar(kBarSFull + w), ((uint32_t)k >> 1) & 1, kErrWaitSFull, abort_flag))
        break;
      // the stage's Q and new rows were written by copies this thread reads
      if (!mbar_wait(bar(kBarFull + s), ((uint32_t)k / kStages) & 1, kErrWaitKvFull, abort_flag))
        break;
      tc_fence_after();
      float x[kN];
      {
        uint32_t v[kN];
        tmem_ld32(tmem + lane_addr + col_s(w), v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          const bool ok = live && c < nrow && pt >= p0 + (c >> 3) - (kW - 1);
          x[c] = ok ? __uint_as_float(v[c]) * p.scale_log2 : -INFINITY;
        }
      }
      // score of new key ni for row nr (drafts attend causally among themselves)
      float sn = -INFINITY;
      if (p0 >= 0 && nr < nrow && ni < L && ni <= (nr >> 3)) {
        const uint32_t qrow = st + kStageQ + nr * 128;
        const uint32_t krow = st + kStageKn + ni * kD * 2;
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {   // 16 chunks of 8 dims
          const uint32_t qa = qrow + (c >> 3) * kQHalf + ((((c & 7) ^ (nr & 7))) << 4);
          uint32_t qv[4], kv[4];
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(qv[0]), "=r"(qv[1]), "=r"(qv[2]), "=r"(qv[3]) : "r"(qa));
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(kv[0]), "=r"(kv[1]), "=r"(kv[2]), "=r"(kv[3]) : "r"(krow + 16 * c));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(qv[e] << 16), __uint_as_float(kv[e] << 16), acc);
            acc = fmaf(__uint_as_float(qv[e] & 0xffff0000u), __uint_as_float(kv[e] & 0xffff0000u),
                       acc);
          }
        }
        sn = acc * p.scale_log2;
      }
      // ---- max over slots and new keys, per row ----
      {
        float mv[kN];
#pragma unroll
        for (int c = 0; c < kN; ++c) mv[c] = x[c];
        red_max[quad * 32 + lane] = warp_transpose_reduce32<true>(mv, lane);
        float nm = fmaxf(sn, __shfl_xor_sync(0xffffffffu, sn, 1));
        nm = fmaxf(nm, __shfl_xor_sync(0xffffffffu, nm, 2));
        if (ni == 0) new_max[nr] = nm;
      }
      mbar_arrive(bar_max);
      if (!mbar_wait(bar_max, ((uint32_t)k >> 1) & 1, kErrWaitDecode, abort_flag)) break;
      float m[kN];
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        const float mr = fmaxf(fmaxf(red_max[c], red_max[32 + c]),
                               fmaxf(red_max[64 + c], red_max[96 + c]));
        m[c] = fmaxf(fmaxf(mr, new_max[c]), sk8[c & 7]);
        if (m[c] == -INFINITY) m[c] = 0.f;  // nothing to attend to: all weights 0
      }
      // ---- weights: ring part to shared memory (bf16 P^T), new part kept ----
#pragma unroll
      for (int c = 0; c < kN; ++c) x[c] = ex2_approx(x[c] - m[c]);
      float pn = 0.f;
      {
        float mn = m[0];
#pragma unroll
        for (int c = 1; c < kN; ++c) mn = (nr == c) ? m[c] : mn;
        pn = ex2_approx(sn - mn);
        pnew[nr * 4 + ni] = pn;
      }
      const uint32_t p_off = (t >> 6) * kQHalf + 2 * (t & 7);
      const int p_chunk = (t & 63) >> 3;
#pragma unroll
      for (int c = 0; c < kN; ++c)
        st_shared_u16(pbuf + p_off + c * 128 + (((p_chunk ^ c) & 7) << 4),
                      __bfloat16_as_ushort(__float2bfloat16_rn(x[c])));
      if (!live) {  // empty slot: zero its values so that 0 * V stays 0
        const uint32_t vrow = st + kStageV + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          st_shared_v4(vrow + 16 * c, 0u, 0u, 0u, 0u);
          st_shared_v4(vrow + kHalf + 16 * c, 0u, 0u, 0u, 0u);
        }
      }
      // this group's new values, read now: the stage is handed back to the
      // producer as soon as the PV product completes
      float vn[kLmax];
      {
        const uint16_t* vs = reinterpret_cast<const uint16_t*>(smem + s * kStageBytes + kStageVn);
#pragma unroll
        for (int i = 0; i < kLmax; ++i)
          vn[i] = __uint_as_float((uint32_t)vs[i * kD + t] << 16);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + w));
      // ---- sums ----
      red_sum[quad * 32 + lane] = warp_transpose_reduce32<false>(x, lane);
      {
        float ns = pn + __shfl_xor_sync(0xffffffffu, pn, 1);
        ns += __shfl_xor_sync(0xffffffffu, ns, 2);
        if (ni == 0) new_sum[nr] = ns;
      }
      mbar_arrive(bar_sum);
      if (!mbar_wait(bar_sum, ((uint32_t)k >> 1) & 1, kErrWaitDecode, abort_flag)) break;
      float inv_l[kN];
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        float lt = (red_sum[c] + red_sum[32 + c]) + (red_sum[64 + c] + red_sum[96 + c]) +
                   new_sum[c];
        if (sk8[c & 7] != -INFINITY) lt += ex2_approx(sk8[c & 7] - m[c]);
        inv_l[c] = lt > 0.f ? 1.f / lt : 0.f;
        if (t == c && c < nrow && p.lse != nullptr)
          p.lse[((int64_t)b * p.Hq + g * kG + (c & 7)) * L + (c >> 3)] =
              (m[c] + __log2f(lt)) * 0.6931471805599453f;
      }
      // ---- output: O^T[dim t][row c] + sum_i pnew[c][i] v_new[i][t] ----
      if (!mbar_wait(bar(kBarOFull + w), ((uint32_t)k >> 1) & 1, kErrWaitOFull, abort_flag))
        break;
      tc_fence_after();
      uint32_t o[kN];
      tmem_ld32(tmem + lane_addr + col_o(w), o);
      tmem_ld_wait();
      tc_fence_before();
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        if (c < nrow) {
          const float4 pw = *reinterpret_cast<const float4*>(pnew + 4 * c);
          float acc = __uint_as_float(o[c]);
          acc = fmaf(pw.x, vn[0], acc);
          acc = fmaf(pw.y, vn[1], acc);
          acc = fmaf(pw.z, vn[2], acc);
          acc = fmaf(pw.w, vn[3], acc);
          p.out[(((int64_t)b * L + (c >> 3)) * p.Hq + g * kG + (c & 7)) * kD + t] =
              acc * inv_l[c];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace vertc
}  // namespace swa
