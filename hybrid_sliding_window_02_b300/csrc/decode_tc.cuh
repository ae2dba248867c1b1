// decode_tc.cuh -- one-token decode against the 128-slot ring cache with the
// per-group contractions on the 5th-generation tensor cores.
//
// Operation: for each sequence b and kv head g, the G query heads of the
// group (G = 1, 2, 4, 8 or 16; larger multiples of 8 as groups of 8) attend
// to the W = 128 ring slots of (b, g) with the sink-biased softmax
// ("MiMo-V2-Flash Technical Report" summary, section 前置知识; the fixed-size
// O(W) sliding-window cache of the "pwwt.cn" essay, section 1.1).
// Slot s holds position pos - ((pos - s) mod W); while pos < W - 1 the slots
// s > pos are empty and are ignored whatever they hold.
//
// The call moves about 147 MB (two 32 KB rings per group) and is bound by HBM
// bandwidth, but each group's work is a dense contraction of G heads x 128
// slots x 128 dims twice over: on the CUDA cores the FMAs alone take about
// two thirds of the transfer time (G = 8), so they run on the tensor cores
// instead and the CUDA cores only do the softmax:
//   S^T = K q^T      M = 128 slots, N = 16 (G heads + 16 - G unused), K = 128 dims
//   O^T = V^T P^T    M = 128 dims (V read MN-major), N = 16, K = 128 slots
// Persistent CTAs (one per SM) take groups u = blockIdx.x, + gridDim.x, ...;
// a producer thread keeps groups' K and q (two slots, free once S^T is done)
// and V (four slots, free once the PV is done) in flight through two rings of
// shared memory (TMA, 128-byte swizzle), so HBM never waits on the math.  Two
// threads issue the MMAs, one the S^T products and one the O^T products, so
// that waiting for a group's K slot to land never delays the PV of the group
// before it (and with it the release of that group's V slot).  Two softmax
// warpgroups (three for G = 16 or D = 64) take the groups in turn: thread =
// slot reads its G head scores from TMEM, the max and the sum over slots are
// warp-shuffle reductions (one transposed butterfly for all heads) finished
// across the four warps in shared memory, the bf16 P^T goes to shared memory
// for the second MMA, and after it thread = dim reads O^T from TMEM and writes
// out[b, h, dim] (each warp 128 contiguous bytes).
#pragma once

#include "device_common.cuh"
#include "griddep.cuh"

namespace swa {
namespace dectc {

// Softmax warpgroups: two, taking alternate groups; three for 16 heads per kv
// head, whose longer per-group chain (the softmax of 16 heads between the two
// products) left HBM idle with two, and for D = 64, whose groups carry half
// the bytes for the same chain.  Then three special warps.
__host__ __device__ constexpr int num_wg(int G, int D) { return (G > 8 || D == 64) ? 3 : 2; }
__host__ __device__ constexpr int threads_for(int G, int D) { return 32 * (4 * num_wg(G, D) + 3); }
constexpr int kMaxWG = 3;
constexpr int kN = 16;             // MMA N: the G heads of a group padded to 16
constexpr int kW = 128;            // ring slots
constexpr int kD = 128;            // largest head dimension (64 is the other)

// Two rings in shared memory (128-byte swizzle): K slots (2) hold K and q and
// are free once S^T completes; V slots (4) hold V and are free once the PV
// completes.  Whole-group stages (68 KB) fitted three times.
constexpr uint32_t kKSlots = 2, kVSlots = 4;
constexpr int kHalf = kW * 128;                 // 128 rows x 64 bf16 = 16 KB
constexpr int kQHalf = kN * 128;                // 16 rows x 64 bf16 = 2 KB
constexpr int kKK = 0, kKQ = 2 * kHalf;
constexpr int kKSlotBytes = kKQ + 2 * kQHalf;       // 36 KB
constexpr int kVSlotBytes = 2 * kHalf;              // 32 KB
constexpr int kPBytes = 2 * kQHalf;                 // P^T: 16 heads x 128 slots bf16
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + (int)kKSlots * kKSlotBytes;
constexpr int kOffP = kOffV + (int)kVSlots * kVSlotBytes;       // one buffer per warpgroup
constexpr int kOffRed = kOffP + kMaxWG * kPBytes;               // [wg][warp][head] floats
constexpr int kRedBytes = 2 * 4 * kN * 4;                       // room for G <= 16
constexpr int kOffBar = kOffRed + kMaxWG * kRedBytes;
constexpr int kBarKFull = 0, kBarKEmpty = kBarKFull + kKSlots, kBarVFull = kBarKEmpty + kKSlots,
              kBarVEmpty = kBarVFull + kVSlots, kBarSFull = kBarVEmpty + kVSlots,
              kBarPFull = kBarSFull + kMaxWG, kBarOFull = kBarPFull + kMaxWG,
              kBarRed = kBarOFull + kMaxWG, kBarDrain = kBarRed + 2 * kMaxWG,
              kNumBars = kBarDrain + 2;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;

static_assert(kSmemBytes <= 227 * 1024, "decode stages fit shared memory");
// TMEM columns of S^T and O^T for warpgroup w (16 columns each)
__host__ __device__ constexpr uint32_t col_s(int w) { return 32u * (uint32_t)w; }
__host__ __device__ constexpr uint32_t col_o(int w) { return 32u * (uint32_t)w + 16u; }

struct Params {
  const int64_t* pos;
  const float* sink;
  float* out;
  float* lse;
  int B, Hq, Hkv;
  int rep;            // query groups of kG heads per kv head (G / 8 for G = 24, 32, ...; else 1)
  int units;          // B * Hkv * rep
  float scale_log2;   // log2(e) / sqrt(D)
};

// Group u of the call: ring unit ur = (sequence b, kv head g), and the query
// heads [gq kG, gq kG + kG) it serves.  With G = 8 R (R > 2) the 8-head
// instance runs R sibling groups per kv head, each reading the kv head's
// rings; the siblings are consecutive, so neighbouring CTAs take them in the
// same round and the later reads come from L2.
struct GroupCoords {
  int ur, b, g, gq;
  __device__ __forceinline__ GroupCoords(int u, const Params& p) {
    ur = u;
    int sib = 0;
    if (p.rep != 1) {
      ur = u / p.rep;
      sib = u - ur * p.rep;
    }
    b = ur / p.Hkv;
    g = ur - b * p.Hkv;
    gq = g * p.rep + sib;
  }
};

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}

__device__ __forceinline__ void reg_fence8(uint32_t (&r)[8]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
               "+r"(r[6]), "+r"(r[7]));
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Reduces v[h] over the 32 lanes of a warp for every head h < G (1, 2, 4, 8
// or 16) with a transposed butterfly: at each of the first log2 G steps a lane
// hands the half of its values it does not keep to its partner and combines
// the half it keeps with the partner's, then the last 5 - log2 G steps
// combine one value.  That is G - 1 + 5 - log2 G shuffles in all, against 5 G
// for one butterfly per head (16 against 80 at G = 16).  Lane l ends with the
// result for head l >> (5 - log2 G); v is used up.
template <int kG, bool kMax>
__device__ __forceinline__ float warp_reduce_heads(float (&v)[kG], int lane) {
  constexpr int kLg = kG == 1 ? 0 : kG == 2 ? 1 : kG == 4 ? 2 : kG == 8 ? 3 : 4;
  static_assert((1 << kLg) == kG, "G is a power of two up to 16");
#pragma unroll
  for (int st = 0; st < kLg; ++st) {
    const int off = 16 >> st;
    const int half = kG >> (st + 1);
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float give = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, give, off);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
#pragma unroll
  for (int off = 16 >> kLg; off > 0; off >>= 1) {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
    v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
  }
  return v[0];
}

// G query heads per kv head (1, 2, 4, 8 or 16), head dimension kHd (64 or
// 128).  With kHd = 64 only the first 64-dimension half of each staging
// buffer is loaded; S^T is 4 K-steps deep, and O^T keeps M = 128 with the
// second half of V^T pointed at the first, so TMEM lanes 64..127 hold a copy
// that no thread reads.
template <int kG, int kHd>
__global__ void __launch_bounds__(threads_for(kG, kHd), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_q, const Params p) {
  static_assert(kG >= 1 && kG <= kN, "a group's heads fill at most the 16 MMA columns");
  constexpr int kNWG = num_wg(kG, kHd);
  constexpr int kThreads = threads_for(kG, kHd);
  constexpr int kWarpProducer = 4 * kNWG, kWarpMma = kWarpProducer + 1, kWarpPv = kWarpProducer + 2;
  constexpr uint32_t kTmemCols = kNWG > 2 ? 128 : 64;   // 32 columns per warpgroup
  static_assert(kHd == 64 || kHd == 128, "head dimension 64 or 128");
  constexpr int kHalves = kHd / 64;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
  const int nk = p.units > (int)blockIdx.x
                     ? (p.units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                     : 0;  // groups of this CTA

  if (tid == 0) {
    *abort_flag = 0;
    for (uint32_t s = 0; s < kKSlots; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarKEmpty + s), 1);
    }
    for (uint32_t s = 0; s < kVSlots; ++s) {
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarVEmpty + s), 1);
    }
    for (int w = 0; w < kNWG; ++w) {
      mbar_init(bar(kBarSFull + w), 1);
      mbar_init(bar(kBarPFull + w), 128);
      mbar_init(bar(kBarOFull + w), 1);
      mbar_init(bar(kBarRed + 2 * w), 128);
      mbar_init(bar(kBarRed + 2 * w + 1), 128);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrain + 1), 1);
    fence_mbar_init();
  }
  // P^T rows G..15 (the padding heads) stay zero for the whole kernel
  for (int i = tid; i < kNWG * kPBytes / 16; i += kThreads)
    st_shared_v4(sbase + kOffP + 16 * i, 0u, 0u, 0u, 0u);
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
  // Launched as a programmatic dependent: the set-up above and an L2
  // prefetch of this CTA's first K/V ring (a hint that reads nothing into
  // the CTA) may overlap the previous kernel on the stream; every load and
  // store below waits for that kernel to complete.
  if (warp == kWarpProducer && lane == 0 && nk > 0) {
    const int u0 = GroupCoords((int)blockIdx.x, p).ur;   // ring of this CTA's first group
    for (int hv = 0; hv < kHalves; ++hv) {
      tma_prefetch_l2_4d(&map_k, 64 * hv, u0 * kW, 0, 0);
      tma_prefetch_l2_4d(&map_v, 64 * hv, u0 * kW, 0, 0);
    }
  }
  if (tid == 0) grid_dep_launch();
  grid_dep_wait();

  if (warp == kWarpProducer) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      int nkld = 0, nvld = 0;  // K / V slot loads issued
      for (int k = 0; k < nk; ++k) {
        const GroupCoords gc((int)blockIdx.x + k * (int)gridDim.x, p);
        const uint32_t ks = (uint32_t)k % kKSlots;
        if (!mbar_wait(bar(kBarKEmpty + ks), (((uint32_t)k / kKSlots) & 1) ^ 1, kErrWaitKvEmpty,
                       abort_flag))
          break;
        const uint32_t kst = sbase + kOffK + ks * kKSlotBytes;
        const uint32_t kb = bar(kBarKFull + ks);
        mbar_arrive_expect_tx(kb, kHalves * (kHalf + kQHalf));
        tma_load_4d(kst + kKK, &map_k, 0, gc.ur * kW, 0, 0, kb);
        tma_load_4d(kst + kKQ, &map_q, 0, gc.b * p.Hq + gc.gq * kG, 0, 0, kb);
        if constexpr (kHalves == 2) {
          tma_load_4d(kst + kKK + kHalf, &map_k, 64, gc.ur * kW, 0, 0, kb);
          tma_load_4d(kst + kKQ + kQHalf, &map_q, 64, gc.b * p.Hq + gc.gq * kG, 0, 0, kb);
        }
        ++nkld;
        const uint32_t vs = (uint32_t)k % kVSlots;
        if (!mbar_wait(bar(kBarVEmpty + vs), (((uint32_t)k / kVSlots) & 1) ^ 1, kErrWaitKvEmpty,
                       abort_flag))
          break;
        const uint32_t vst = sbase + kOffV + vs * kVSlotBytes;
        const uint32_t vb = bar(kBarVFull + vs);
        mbar_arrive_expect_tx(vb, kHalves * kHalf);
        tma_load_4d(vst, &map_v, 0, gc.ur * kW, 0, 0, vb);
        if constexpr (kHalves == 2) tma_load_4d(vst + kHalf, &map_v, 64, gc.ur * kW, 0, 0, vb);
        ++nvld;
      }
      if (nvld < nk) {  // stopped early: let the copies already issued land
        for (int j = (nkld > (int)kKSlots ? nkld - (int)kKSlots : 0); j < nkld; ++j)
          mbar_wait_drain(bar(kBarKFull + (uint32_t)j % kKSlots), ((uint32_t)j / kKSlots) & 1);
        for (int j = (nvld > (int)kVSlots ? nvld - (int)kVSlots : 0); j < nvld; ++j)
          mbar_wait_drain(bar(kBarVFull + (uint32_t)j % kVSlots), ((uint32_t)j / kVSlots) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ====== MMA issuers: S^T of every group (warp 9), O^T of every group (warp 10) ======
    // Two threads, so that the wait for a group's K slot to land (S side)
    // never holds back the PV of the group before it and the release of its
    // V slot.
    if (lane == 0) {
      const bool s_side = (warp == kWarpMma);
      const uint32_t idesc_s = umma_idesc_bf16(kN, false, false);
      const uint32_t idesc_o = umma_idesc_bf16(kN, true, false);
      bool ok = true;
      for (int k = 0; ok && k < nk; ++k) {
        const int w = k % kNWG;
        const uint32_t use = (uint32_t)(k / kNWG);   // uses of buffer w before this one
        if (s_side) {
          // S^T of group k into TMEM buffer k % kNWG once its K slot has landed
          // and the softmax of group k - kNWG has read that buffer (P full)
          const uint32_t ks = (uint32_t)k % kKSlots;
          const uint32_t kst = sbase + kOffK + ks * kKSlotBytes;
          if (!mbar_wait(bar(kBarKFull + ks), ((uint32_t)k / kKSlots) & 1, kErrWaitKvFull,
                         abort_flag)) {
            ok = false;
            break;
          }
          if (k >= kNWG && !mbar_wait(bar(kBarPFull + w), (use - 1) & 1,
                                      kErrWaitPFull, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kdesc = umma_sdesc(kst + kKK, 16, 1024, 2);
          const uint64_t qdesc = umma_sdesc(kst + kKQ, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk) {
            const uint32_t a_off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            const uint32_t b_off = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + col_s(w), kdesc + a_off, qdesc + b_off, idesc_s, kk > 0);
          }
          umma_commit(bar(kBarSFull + w));
          umma_commit(bar(kBarKEmpty + ks));   // K and q are no longer read
        } else {
          // O^T = V^T P^T once the V slot has landed and the softmax of this
          // group has written P^T
          const uint32_t vs = (uint32_t)k % kVSlots;
          const uint32_t vst = sbase + kOffV + vs * kVSlotBytes;
          if (!mbar_wait(bar(kBarVFull + vs), ((uint32_t)k / kVSlots) & 1, kErrWaitKvFull,
                         abort_flag) ||
              !mbar_wait(bar(kBarPFull + w), use & 1, kErrWaitPFull, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // V^T as the M = 128 operand: its second 64-dimension atom is the
          // slot's second half, or, at kHd = 64, the first again
          const uint64_t vdesc = umma_sdesc(vst, kHalves == 2 ? kHalf : 0, 1024, 2);
          const uint64_t pdesc = umma_sdesc(sbase + kOffP + w * kPBytes, 16, 1024, 2);
#pragma unroll
          for (int kb = 0; kb < kW / 16; ++kb) {
            const uint32_t a_off = (kb * 16 * 128) >> 4;
            const uint32_t b_off = ((kb >> 2) * kQHalf + (kb & 3) * 32) >> 4;
            umma_bf16_ss(tmem + col_o(w), vdesc + a_off, pdesc + b_off, idesc_o, kb > 0);
          }
          umma_commit(bar(kBarOFull + w));
          umma_commit(bar(kBarVEmpty + vs));
        }
      }
      // every MMA this thread issued completes before TMEM is released
      const uint32_t db = bar(kBarDrain + (s_side ? 0 : 1));
      umma_commit(db);
      mbar_wait_drain(db, 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax + output (warps 0..7) =======================
    const int w = warp >> 2;                   // warpgroup: takes groups k with k % kNWG == w
    const int quad = warp & 3;
    const int t = quad * 32 + lane;            // slot (softmax) / dim (output)
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed) + w * (4 * kG * 2);
    const uint32_t pbuf = sbase + kOffP + w * kPBytes;
    // P^T[h][t] lives at half (t / 64), row h, 16-byte chunk ((t % 64) / 8) ^ h,
    // element t % 8 (128-byte swizzle, rows of 64 slots)
    const uint32_t p_off = (t >> 6) * kQHalf + 2 * (t & 7);
    const int p_chunk = (t & 63) >> 3;
    // The cross-warp exchanges of a warpgroup go through two mbarriers (one
    // per reduction) rather than bar.sync, so that a timed-out wait elsewhere
    // can never leave the other warps blocked.
    const uint32_t bar_max = bar(kBarRed + 2 * w), bar_sum = bar(kBarRed + 2 * w + 1);
    for (int k = w; k < nk; k += kNWG) {
      const uint32_t ph = (uint32_t)(k / kNWG) & 1;   // phase of this warpgroup's barriers
      const GroupCoords gc((int)blockIdx.x + k * (int)gridDim.x, p);
      const int b = gc.b, g = gc.gq;   // g: the query group (heads g kG ..)
      const uint32_t vs = (uint32_t)k % kVSlots;
      const int64_t pnow = p.pos[b];
      const bool full_ring = pnow >= kW - 1;
      const bool valid = full_ring || (int64_t)t <= pnow;
      if (!mbar_wait(bar(kBarSFull + w), ph, kErrWaitSFull, abort_flag))
        break;
      tc_fence_after();
      uint32_t sr[kG > 8 ? 16 : 8];
      tmem_ld8(tmem + lane_addr + col_s(w), *reinterpret_cast<uint32_t(*)[8]>(&sr[0]));
      if constexpr (kG > 8)
        tmem_ld8(tmem + lane_addr + col_s(w) + 8, *reinterpret_cast<uint32_t(*)[8]>(&sr[8]));
      tmem_ld_wait();
      reg_fence8(*reinterpret_cast<uint32_t(*)[8]>(&sr[0]));
      if constexpr (kG > 8) reg_fence8(*reinterpret_cast<uint32_t(*)[8]>(&sr[8]));
      float x[kG], m[kG];
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        x[h] = valid ? __uint_as_float(sr[h]) * p.scale_log2 : -INFINITY;
        m[h] = x[h];
      }
      {
        // the warp's max for head lane >> (5 - log2 G); the first lane of each
        // head publishes it
        const float mine = warp_reduce_heads<kG, true>(m, lane);
        if ((lane & (32 / kG - 1)) == 0) red[quad * kG + lane / (32 / kG)] = mine;
      }
      mbar_arrive(bar_max);
      if (!mbar_wait(bar_max, ph, kErrWaitDecode, abort_flag)) break;
      float sk[kG], l[kG];
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        sk[h] = p.sink[g * kG + h] * 1.4426950408889634f;
        m[h] = fmaxf(fmaxf(fmaxf(red[h], red[kG + h]), fmaxf(red[2 * kG + h], red[3 * kG + h])),
                     sk[h]);
        // with no valid slot and no sink (not reachable for pos >= 0) keep m finite
        const float mb = m[h] == -INFINITY ? 0.f : m[h];
        x[h] = ex2_approx(x[h] - mb);
        l[h] = x[h];
      }
      // bf16 P^T to shared memory for the second MMA
#pragma unroll
      for (int h = 0; h < kG; ++h)
        st_shared_u16(pbuf + p_off + h * 128 + (((p_chunk ^ h) & 7) << 4),
                      __bfloat16_as_ushort(__float2bfloat16_rn(x[h])));
      // empty slots may hold anything (NaN included): zero their values so
      // that 0 * V stays 0 in the MMA
      // (the V slot is waited for here: S^T needed only the K slot)
      if (!full_ring &&
          !mbar_wait(bar(kBarVFull + vs), ((uint32_t)k / kVSlots) & 1, kErrWaitKvFull, abort_flag))
        break;
      if (!full_ring && !valid) {
        const uint32_t vrow = sbase + kOffV + vs * kVSlotBytes + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          st_shared_v4(vrow + 16 * c, 0u, 0u, 0u, 0u);
          if constexpr (kHalves == 2) st_shared_v4(vrow + kHalf + 16 * c, 0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + w));
      {
        const float mine = warp_reduce_heads<kG, false>(l, lane);
        if ((lane & (32 / kG - 1)) == 0) red[4 * kG + quad * kG + lane / (32 / kG)] = mine;
      }
      mbar_arrive(bar_sum);
      if (!mbar_wait(bar_sum, ph, kErrWaitDecode, abort_flag)) break;
      float inv_l[kG];
#pragma unroll
      for (int h = 0; h < kG; ++h) {
        float lt = (red[4 * kG + h] + red[5 * kG + h]) + (red[6 * kG + h] + red[7 * kG + h]);
        if (sk[h] != -INFINITY) lt += ex2_approx(sk[h] - m[h]);
        inv_l[h] = lt > 0.f ? 1.f / lt : 0.f;
        if (t == h && p.lse != nullptr)
          p.lse[(int64_t)b * p.Hq + g * kG + h] = (m[h] + __log2f(lt)) * 0.6931471805599453f;
      }
      // O^T[dim t][h] -> out[b, g*G + h, t]
      if (!mbar_wait(bar(kBarOFull + w), ph, kErrWaitOFull, abort_flag))
        break;
      tc_fence_after();
      uint32_t o[kG > 8 ? 16 : 8];
      tmem_ld8(tmem + lane_addr + col_o(w), *reinterpret_cast<uint32_t(*)[8]>(&o[0]));
      if constexpr (kG > 8)
        tmem_ld8(tmem + lane_addr + col_o(w) + 8, *reinterpret_cast<uint32_t(*)[8]>(&o[8]));
      tmem_ld_wait();
      reg_fence8(*reinterpret_cast<uint32_t(*)[8]>(&o[0]));
      if constexpr (kG > 8) reg_fence8(*reinterpret_cast<uint32_t(*)[8]>(&o[8]));
      tc_fence_before();
      float* ob = p.out + ((int64_t)b * p.Hq + g * kG) * kHd + t;
      if (t < kHd) {
#pragma unroll
        for (int h = 0; h < kG; ++h) ob[h * kHd] = __uint_as_float(o[h]) * inv_l[h];
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

}  // namespace dectc
}  // namespace swa
