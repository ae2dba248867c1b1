// verify_tc.cuh -- multi-token verify against the 128-slot ring with the
// contractions on the 5th-generation tensor cores.
//
// Operation: as in verify.cuh (drafted tokens at positions pos .. pos+L-1
// checked in one pass; "MiMo-V2-Flash Technical Report" summary, section
// 核心方法), for bf16 inputs, D = 64 or 128, W = 128, 1, 2, 4 or 8 query
// heads per kv head (or a multiple of 8, as sibling groups of 8) and L <= 8
// drafted tokens.  Per group (sequence b, kv head g) the 8L query rows (GL
// for G < 8)
// r = 8 j + h (token j, head h) sit in the first lanes of a 128-row tile:
//   S = Q K_ring^T             tcgen05 SS, M = 128 rows, N = 128 slots, K = 128
//   S_new = Q K_new^T          tcgen05 SS, N = 16 (the L <= 8 drafted keys;
//                              columns L..15 are masked), into the first 16 columns of
//                              the warpgroup's O buffer, which are free from
//                              the output of group k - 2 to the PV of group k
//   O = P_ring V_ring + P_new V_new
//                              tcgen05 TS: P (bf16) written over S in TMEM,
//                              V MN-major; the new values as one K = 16 step
// Thread = row: lane r of the warpgroup's first warp (rows 32..63, for L > 4,
// of its second) reads its 128 slot scores and its new-key scores and runs
// the sink-seeded softmax alone (as the global-attention kernel does per key
// block), so no reduction crosses lanes.  The rows past 8L are padding that no
// one reads.  The kernel comes in two sizes: up to 32 rows (L <= 4: one
// softmax warp and three that zero empty slots per warpgroup) and up to 64
// (L <= 8: two and two, and a Q staging area twice as large).  (Scoring the new keys on
// the CUDA cores instead, as 128-long FMA chains on three warps, put ~1700
// cycles per group on the softmax's critical path.)
//
// Masks.  Slot s holds position p(s) = (pos-1) - ((pos-1-s) mod W).  Once
// pos >= W the ring is full and row j's window [pos+j-W+1, pos+j] leaves out
// exactly the j+1 oldest slots, (pos + i) mod W for i <= j: only the 32-column
// chunks that arc touches are tested column by column.  While pos < W the
// slots s >= pos are empty (their values are zeroed in shared memory so that
// 0 * V stays 0) and every column is tested.
//
// Persistent CTAs.  The loads go into two rings (TMA): K slots (Q, K ring,
// K_new), released as soon as S and S_new complete, and V slots (V ring,
// V_new), released when the PV completes; with whole-group stages only two
// fitted in shared memory, and the producer spent most of each group waiting
// for one to be released after its PV.  Two MMA-issuing threads (one for the
// S products, one for the PV products, so that waiting for a K slot to land
// never delays the PV of the group before it and the release of its V slot),
// two warpgroups on alternate groups, each with its own S / O pair in TMEM:
// S_w [256 w, 256 w + 128), O_w [256 w + 128, 256 w + 256).  S of group k
// overwrites P of group k - 2, and S_new overwrites O of group k - 2, so both
// are issued once the output of group k - 2 has been read out of TMEM (which
// follows that group's PV).
#pragma once

#include "device_common.cuh"
#include "griddep.cuh"

namespace swa {
namespace vertc {

constexpr int kThreads = 352;
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpPv = 10;
constexpr int kG = 8;
constexpr int kLmax = 8;            // drafted tokens of the larger kernel size
constexpr int kW = 128;
constexpr int kD = 128;            // largest head dimension (64 is the other)
constexpr int kNewRows = 16;        // new keys padded to one K = 16 MMA step

// Two rings in shared memory (128-byte swizzle everywhere):
//   K slots (2): Q [2 halves x kRows rows: 4 or 8 KB each], K ring [2 x 16 KB],
//                K_new [2 x 1 KB: 8 rows].  Free once S and S_new complete.
//   V slots (3): V ring [2 x 16 KB], V_new [2 x 2 KB: 16 rows, rows L..15
//                zero].  Free once the PV completes.
// An M = 128 MMA reads 128 rows (16 KB) from each Q half base, and the N = 16
// S_new MMA reads 16 rows (2 KB) from each K_new half base: the rows past
// those that hold data fall on later data in shared memory and only feed TMEM
// lanes or columns that no one reads.
// kRows = 32 (L <= 4) or 64 (L <= 8) query rows per group.
template <int kRows>
struct Layout {
  static constexpr int kHalf = 128 * 128;                // 128 rows x 64 bf16 = 16 KB
  static constexpr int kQHalf = kRows * 128;             // kRows rows x 64 bf16
  static constexpr int kKnHalf = 8 * 128;                // 8 rows x 64 bf16 = 1 KB
  static constexpr int kNewHalf = kNewRows * 128;        // 16 rows x 64 bf16 = 2 KB
  static constexpr uint32_t kKSlots = 2, kVSlots = 3;
  static constexpr int kKQ = 0, kKK = 2 * kQHalf, kKKn = kKK + 2 * kHalf;
  static constexpr int kKSlotBytes = kKKn + 2 * kKnHalf;        // 42 or 50 KB
  static constexpr int kVV = 0, kVVn = 2 * kHalf;
  static constexpr int kVSlotBytes = kVVn + 2 * kNewHalf;       // 36 KB
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + (int)kKSlots * kKSlotBytes;
  static constexpr int kOffBar = kOffV + (int)kVSlots * kVSlotBytes;
  static constexpr int kBarKFull = 0, kBarKEmpty = kBarKFull + kKSlots,
                       kBarVFull = kBarKEmpty + kKSlots, kBarVEmpty = kBarVFull + kVSlots,
                       kBarSFull = kBarVEmpty + kVSlots, kBarPFull = kBarSFull + 2,
                       kBarOFull = kBarPFull + 2, kBarODone = kBarOFull + 2,
                       kBarDrain = kBarODone + 2, kNumBars = kBarDrain + 2;
  static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
  static constexpr int kOffAbort = kOffTmemSlot + 8;
  static constexpr int kSmemBytes = kOffAbort + 8 + 1024;
};
static_assert(Layout<64>::kSmemBytes <= 227 * 1024, "verify stages fit shared memory");

constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int w) { return 256u * (uint32_t)w; }
__host__ __device__ constexpr uint32_t col_o(int w) { return 256u * (uint32_t)w + 128u; }

struct Params {
  const int64_t* pos;
  const float* sink;
  float* out;
  float* lse;
  int B, L, Hq, Hkv;
  int rep;            // groups of 8 query heads per kv head (G / 8)
  int units;          // B * Hkv * rep
  float scale_log2;
};

// Group u of the call: ring unit ur = (sequence b, kv head g), and the query
// heads [gq kGv, gq kGv + kGv) it serves.  With G = 8 R the R sibling groups of
// a kv head each read its rings and drafted keys and values; the siblings
// are consecutive, so neighbouring CTAs take them in the same round and the
// later reads come from L2.
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

// kRows query rows per group (32 or 64), head dimension kHd (64 or 128: with
// 64 only the first 64-dimension half of each staging buffer is loaded, the
// score products are 4 K-steps deep and PV has N = 64), kGv query heads per
// group (8, or G = 1, 2, 4 with kRows = 32): row r = kGv j + h.
template <int kRows, int kHd, int kGv>
__global__ void __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v,
                     const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_kn,
                     const __grid_constant__ CUtensorMap map_vn, const Params p) {
  using Lay = Layout<kRows>;
  constexpr int kHalf = Lay::kHalf, kQHalf = Lay::kQHalf, kKnHalf = Lay::kKnHalf,
                kNewHalf = Lay::kNewHalf, kKQ = Lay::kKQ, kKK = Lay::kKK, kKKn = Lay::kKKn,
                kKSlotBytes = Lay::kKSlotBytes, kVV = Lay::kVV, kVVn = Lay::kVVn,
                kVSlotBytes = Lay::kVSlotBytes, kOffK = Lay::kOffK, kOffV = Lay::kOffV,
                kOffBar = Lay::kOffBar, kOffTmemSlot = Lay::kOffTmemSlot,
                kOffAbort = Lay::kOffAbort;
  constexpr uint32_t kKSlots = Lay::kKSlots, kVSlots = Lay::kVSlots;
  constexpr int kBarKFull = Lay::kBarKFull, kBarKEmpty = Lay::kBarKEmpty,
                kBarVFull = Lay::kBarVFull, kBarVEmpty = Lay::kBarVEmpty,
                kBarSFull = Lay::kBarSFull, kBarPFull = Lay::kBarPFull,
                kBarOFull = Lay::kBarOFull, kBarODone = Lay::kBarODone,
                kBarDrain = Lay::kBarDrain;
  constexpr int kSoftWarps = kRows / 32;        // softmax warps per warpgroup
  static_assert(kGv == 8 || ((kGv == 1 || kGv == 2 || kGv == 4) && kRows == 32),
                "8 query heads per group, or 1, 2 or 4 in 32 rows");
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
                     : 0;
  const int L = p.L;

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
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(kBarSFull + w), 1);
      mbar_init(bar(kBarPFull + w), 128);
      mbar_init(bar(kBarOFull + w), 1);
      mbar_init(bar(kBarODone + w), 32 * kSoftWarps);
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrain + 1), 1);
    fence_mbar_init();
  }
  // new value rows L..15 of every V slot are never written by a copy: zero
  // them once (their weights are 0, and 0 * NaN would not be)
  for (int i = tid; i < (int)kVSlots * 2 * kNewHalf / 16; i += kThreads) {
    const int sl = i / (2 * kNewHalf / 16), r = i % (2 * kNewHalf / 16);
    st_shared_v4(sbase + kOffV + sl * kVSlotBytes + kVVn + 16 * r, 0u, 0u, 0u, 0u);
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
    prefetch_tmap(&map_kn);
    prefetch_tmap(&map_vn);
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
      const uint32_t kbytes = kHalves * (kHalf + kGv * L * 128 + L * 128);
      const uint32_t vbytes = kHalves * (kHalf + L * 128);
      int nkld = 0, nvld = 0;  // K / V slot loads issued
      for (int k = 0; k < nk; ++k) {
        const GroupCoords gc((int)blockIdx.x + k * (int)gridDim.x, p);
        const int b = gc.b, g = gc.g;
        // K slot: Q, K ring, K_new
        const uint32_t ks = (uint32_t)k % kKSlots;
        if (!mbar_wait(bar(kBarKEmpty + ks), (((uint32_t)k / kKSlots) & 1) ^ 1, kErrWaitKvEmpty,
                       abort_flag))
          break;
        const uint32_t kst = sbase + kOffK + ks * kKSlotBytes;
        const uint32_t kb = bar(kBarKFull + ks);
        mbar_arrive_expect_tx(kb, kbytes);
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) {
          tma_load_4d(kst + kKQ + hf * kQHalf, &map_q, 64 * hf, gc.gq * kGv, 0, b, kb);
          tma_load_4d(kst + kKK + hf * kHalf, &map_k, 64 * hf, gc.ur * kW, 0, 0, kb);
          tma_load_4d(kst + kKKn + hf * kKnHalf, &map_kn, 64 * hf, g, 0, b, kb);
        }
        ++nkld;
        // V slot: V ring, V_new
        const uint32_t vs = (uint32_t)k % kVSlots;
        if (!mbar_wait(bar(kBarVEmpty + vs), (((uint32_t)k / kVSlots) & 1) ^ 1, kErrWaitKvEmpty,
                       abort_flag))
          break;
        const uint32_t vst = sbase + kOffV + vs * kVSlotBytes;
        const uint32_t vb = bar(kBarVFull + vs);
        mbar_arrive_expect_tx(vb, vbytes);
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) {
          tma_load_4d(vst + kVV + hf * kHalf, &map_v, 64 * hf, gc.ur * kW, 0, 0, vb);
          tma_load_4d(vst + kVVn + hf * kNewHalf, &map_vn, 64 * hf, g, 0, b, vb);
        }
        ++nvld;
      }
      if (nvld < nk) {
        // copies still in flight land before the CTA exits
        for (int j = (nkld > (int)kKSlots ? nkld - (int)kKSlots : 0); j < nkld; ++j)
          mbar_wait_drain(bar(kBarKFull + (uint32_t)j % kKSlots), ((uint32_t)j / kKSlots) & 1);
        for (int j = (nvld > (int)kVSlots ? nvld - (int)kVSlots : 0); j < nvld; ++j)
          mbar_wait_drain(bar(kBarVFull + (uint32_t)j % kVSlots), ((uint32_t)j / kVSlots) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ====== MMA issuers: S of every group (warp 9), O of every group (warp 10) ======
    // Two threads, so that the wait for a group's K slot to land (S side)
    // never holds back the PV of the group before it and the release of its
    // V slot.
    if (lane == 0) {
      const bool s_side = (warp == kWarpMma);
      const uint32_t idesc_s = umma_idesc_bf16(kW, false, false);
      const uint32_t idesc_n = umma_idesc_bf16(kNewRows, false, false);
      const uint32_t idesc_o = umma_idesc_bf16(kHd, false, true);
      bool ok = true;
      for (int k = 0; ok && k < nk; ++k) {
        const int w = k & 1;
        if (s_side) {
          const uint32_t ks = (uint32_t)k % kKSlots;
          const uint32_t kst = sbase + kOffK + ks * kKSlotBytes;
          if (!mbar_wait(bar(kBarKFull + ks), ((uint32_t)k / kKSlots) & 1, kErrWaitKvFull,
                         abort_flag)) {
            ok = false;
            break;
          }
          // S_w holds P of group k - 2 until that group's PV has completed, and
          // O_w its output until the warpgroup has read it (which follows)
          if (k >= 2 && !mbar_wait(bar(kBarODone + w), (((uint32_t)k >> 1) - 1) & 1,
                                   kErrWaitOFull, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qdesc = umma_sdesc(kst + kKQ, 16, 1024, 2);
          const uint64_t kdesc = umma_sdesc(kst + kKK, 16, 1024, 2);
          const uint64_t kndesc = umma_sdesc(kst + kKKn, 16, 1024, 2);
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk) {
            const uint32_t qoff = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
            const uint32_t koff = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + col_s(w), qdesc + qoff, kdesc + koff, idesc_s, kk > 0);
          }
          // S_new = Q K_new^T into O_w columns [0, 16)
#pragma unroll
          for (int kk = 0; kk < kHd / 16; ++kk) {
            const uint32_t qoff = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
            const uint32_t noff = ((kk >> 2) * kKnHalf + (kk & 3) * 32) >> 4;
            umma_bf16_ss(tmem + col_o(w), qdesc + qoff, kndesc + noff, idesc_n, kk > 0);
          }
          umma_commit(bar(kBarSFull + w));
          umma_commit(bar(kBarKEmpty + ks));   // Q, K and K_new are no longer read
        } else {
          // O = P V once the V slot has landed and the softmax of this group
          // has written P
          const uint32_t vs = (uint32_t)k % kVSlots;
          const uint32_t vst = sbase + kOffV + vs * kVSlotBytes;
          if (!mbar_wait(bar(kBarVFull + vs), ((uint32_t)k / kVSlots) & 1, kErrWaitKvFull,
                         abort_flag) ||
              !mbar_wait(bar(kBarPFull + w), ((uint32_t)k >> 1) & 1, kErrWaitPFull, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t vdesc = umma_sdesc(vst + kVV, kHalf, 1024, 2);
          const uint64_t vndesc = umma_sdesc(vst + kVVn, kNewHalf, 1024, 2);
#pragma unroll
          for (int kb = 0; kb < kW / 16; ++kb)
            umma_bf16_ts(tmem + col_o(w), tmem + col_s(w) + kb * 8,
                         vdesc + (uint32_t)(kb * 16 * 128 >> 4), idesc_o, kb > 0);
          umma_bf16_ts(tmem + col_o(w), tmem + col_s(w) + 64, vndesc, idesc_o, 1u);
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
    const int w = warp >> 2;                       // warpgroup: groups k with k % 2 == w
    const int wq = warp & 3;                       // warp within the warpgroup
    const int nrow = kGv * L;
    if (wq < kSoftWarps) {
      // ============ softmax + output: thread = row r (TMEM lane r) ============
      const int r = 32 * wq + lane;
      const uint32_t lane_addr = (uint32_t)(32 * wq) << 16;
      const int j = r / kGv, h = r % kGv;
      const uint32_t s_addr = tmem + lane_addr + col_s(w), o_addr = tmem + lane_addr + col_o(w);
      for (int k = w; k < nk; k += 2) {
        const GroupCoords gc((int)blockIdx.x + k * (int)gridDim.x, p);
        const int b = gc.b, g = gc.gq;   // g: the query group (heads g kGv ..)
        const int64_t p0 = p.pos[b];
        const float sk = p.sink[g * kGv + h] * 1.4426950408889634f;
        if (!mbar_wait(bar(kBarSFull + w), ((uint32_t)k >> 1) & 1, kErrWaitSFull, abort_flag))
          break;
        tc_fence_after();
        uint32_t sr[kW], snr[8];
#pragma unroll
        for (int c = 0; c < kW / 32; ++c) tmem_ld32(s_addr + c * 32, sr + c * 32);
        tmem_ld8(o_addr, snr);                      // S_new: new keys 0..7 of row r
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kW / 32; ++c) reg_fence32(sr + c * 32);
        reg_fence8(snr);
        // ---- mask the ring slots outside row j's window ----
        if (p0 >= kW) {
          const int a0 = (int)(p0 & (kW - 1));     // slot of the oldest position
#pragma unroll
          for (int q = 0; q < kW / 32; ++q) {
            // does the arc a0 .. a0 + L - 1 (mod W) touch columns [32 q, 32 q + 32)?
            const bool touch = (((32 * q - a0) & (kW - 1)) < L) ||
                               (((a0 - 32 * q) & (kW - 1)) < 32);
            if (touch) {
#pragma unroll
              for (int c = 32 * q; c < 32 * q + 32; ++c)
                if (((c - a0) & (kW - 1)) <= j) sr[c] = __float_as_uint(-INFINITY);
            }
          }
        } else {
          // partial ring: slot s holds position s when s < pos, else nothing
          const int lo = (int)p0 + j - (kW - 1);   // first position of the window
#pragma unroll
          for (int c = 0; c < kW; ++c)
            if (c >= p0 || c < lo) sr[c] = __float_as_uint(-INFINITY);
        }
        // ---- max over the window and the new keys, seeded with the sink ----
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          m8[e] = fmaxf(__uint_as_float(sr[e]), __uint_as_float(sr[e + 8]));
#pragma unroll
        for (int c = 16; c < kW; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            m8[e] = max3f(m8[e], __uint_as_float(sr[c + e]), __uint_as_float(sr[c + 8 + e]));
        const float mring = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                                  fmaxf(m8[6], m8[7])) * p.scale_log2;
        // new key i of row j counts when it exists (i < L), is causal (i <= j)
        // and the sequence is live (pos >= 0)
        // new keys a row may see: 4 or 8 (at most the 8 drafted tokens)
        constexpr int kNew = kRows / kGv < kLmax ? kRows / kGv : kLmax;
        float sv[kNew];
#pragma unroll
        for (int i = 0; i < kNew; ++i)
          sv[i] = (p0 >= 0 && i < L && i <= j) ? __uint_as_float(snr[i]) * p.scale_log2
                                               : -INFINITY;
        float m = fmaxf(mring, sk);
#pragma unroll
        for (int i = 0; i < kNew; ++i) m = fmaxf(m, sv[i]);
        if (m == -INFINITY) m = 0.f;                // nothing to attend to
        // ---- weights: bf16 P over S columns [0, 64), new keys at [64, 72) ----
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m, -m);
        float2 l2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) l2[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kW / 16; ++c) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 xx = ffma2(make_float2(__uint_as_float(sr[16 * c + 2 * e]),
                                                __uint_as_float(sr[16 * c + 2 * e + 1])),
                                    sc2, nm2);
            const float2 pp = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
            l2[e & 3] = fadd2(l2[e & 3], pp);
            pk[e] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st8(s_addr + c * 8, pk);
        }
        float pn[kNew], ln = 0.f;
#pragma unroll
        for (int i = 0; i < kNew; ++i) {
          pn[i] = ex2_approx(sv[i] - m);
          ln += pn[i];
        }
        {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) pk[e] = 0u;
#pragma unroll
          for (int e = 0; e < kNew / 2; ++e) pk[e] = pack_bf16x2(pn[2 * e], pn[2 * e + 1]);
          tmem_st8(s_addr + 64, pk);
        }
        float l;
        {
          const float2 a = fadd2(fadd2(l2[0], l2[1]), fadd2(l2[2], l2[3]));
          l = (a.x + a.y) + ln;
          if (sk != -INFINITY) l += ex2_approx(sk - m);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + w));
        if (r < nrow && p.lse != nullptr)
          p.lse[((int64_t)b * p.Hq + g * kGv + h) * L + j] = (m + __log2f(l)) * 0.6931471805599453f;
        // ---- output row: O / l ----
        if (!mbar_wait(bar(kBarOFull + w), ((uint32_t)k >> 1) & 1, kErrWaitOFull, abort_flag))
          break;
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        float* orow = p.out + (((int64_t)b * L + j) * p.Hq + g * kGv + h) * kHd;
#pragma unroll
        for (int c = 0; c < kHd / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
          tmem_ld_wait();
          reg_fence32(o);
          if (c == kHd / 32 - 1) {
            // O_w has been read: S_new of group k + 2 may overwrite it
            tc_fence_before();
            mbar_arrive(bar(kBarODone + w));
          }
          if (r < nrow) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              st_global_v4(orow + c * 32 + 4 * e,
                           __float_as_uint(__uint_as_float(o[4 * e]) * inv_l),
                           __float_as_uint(__uint_as_float(o[4 * e + 1]) * inv_l),
                           __float_as_uint(__uint_as_float(o[4 * e + 2]) * inv_l),
                           __float_as_uint(__uint_as_float(o[4 * e + 3]) * inv_l));
          }
        }
        tc_fence_before();
      }
    } else {
      // ============ empty-slot values (the other warps of the warpgroup) ============
      constexpr int kHelpers = 32 * (4 - kSoftWarps);   // 96 or 64 threads
      const int t = (wq - kSoftWarps) * 32 + lane;
      for (int k = w; k < nk; k += 2) {
        const int b = GroupCoords((int)blockIdx.x + k * (int)gridDim.x, p).b;
        const uint32_t vs = (uint32_t)k % kVSlots;
        const uint32_t vst = sbase + kOffV + vs * kVSlotBytes;
        const int64_t p0 = p.pos[b];
        if (!mbar_wait(bar(kBarVFull + vs), ((uint32_t)k / kVSlots) & 1, kErrWaitKvFull,
                       abort_flag))
          break;
        // P full counts this group's arrivals only once group k - 2's phase
        // has completed: arriving earlier would complete that phase without
        // the softmax warp
        if (k >= 2 && !mbar_wait(bar(kBarPFull + w), (((uint32_t)k >> 1) - 1) & 1, kErrWaitPFull,
                                 abort_flag))
          break;
        // empty slots (pos < W): zero their values in the V slot before the PV
        if (p0 < kW) {
          for (int sl = t; sl < kW; sl += kHelpers) {
            if (sl >= p0) {
              const uint32_t vrow = vst + kVV + sl * 128;
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                st_shared_v4(vrow + 16 * c, 0u, 0u, 0u, 0u);
                if constexpr (kHalves == 2) st_shared_v4(vrow + kHalf + 16 * c, 0u, 0u, 0u, 0u);
              }
            }
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(bar(kBarPFull + w));
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
