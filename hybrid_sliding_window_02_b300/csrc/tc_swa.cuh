// tc_swa.cuh -- sliding-window prefill on the 5th-generation tensor cores.
//
// Operation: causal sliding-window attention with GQA and a per-head sink bias
// in the softmax denominator ("MiMo-V2-Flash Technical Report" summary, section
// 前置知识; 128-token window in section 核心方法).  This kernel covers W <= 129,
// bf16 inputs, D = 128 or 64, and G = 4 or any multiple of 8 query heads per
// kv head.  With D = 64 the score products are 4 K-steps deep instead of 8, PV
// has N = 64, O takes 64 TMEM columns, and only the first 64-dimension half
// of each staging buffer is used (the layout is the same).
//
// Tiling.  One tile = kNpos consecutive positions x kG query heads = 128 MMA
// rows (row r = position (r / kG), head (r % kG)): 16 positions x 8 heads, or
// 32 positions x 4 heads when G = 4.  With G = 8 R the kv head's query heads
// form R groups of 8 ("tile groups") that share its keys and values; each
// group is walked on its own.  The keys that tile n needs span positions
// [n kNpos - W + 1, n kNpos + kNpos - 1], i.e. the key blocks of 16 from
// n kNew - 8 to n kNew + kNew - 1 (kNew = kNpos / 16 new blocks per tile):
// a 128 x 144 score tile for 8 heads (89% in the window) or 128 x 160 for 4
// heads (80%), where a 128-position single-head tile would need 256 keys (50%
// useful).  The whole window fits in tensor memory, so the softmax is an
// exact single pass seeded with the sink (no rescaling).
//
// Persistent CTAs (one per SM) walk a contiguous range of tiles (order in
// TileWalk).  Consecutive tiles of one (b, tile group) share 8 of their key
// blocks, so keys and values live in a ring of 16-key blocks in shared memory
// and each key/value row is loaded once per run.
//
// Roles (480 threads), all connected by mbarriers:
//   warp 12     TMA producer: Q tiles (4 stages, to cover the HBM latency seen
//               under full load) and new K/V blocks (12-slot ring)
//   warp 13     TMEM owner + issuer of S = Q K^T (SS: M=128, N=144 or 160
//               split at the ring wrap, K=128)
//   warp 14     issuer of O = P V (TS: P from TMEM, V MN-major, N=128,
//               K=16 per block); releases the ring blocks
//               One issuing thread for both paced the kernel: its barrier
//               waits and bookkeeping, slowed by sharing a sub-partition with
//               three busy warps, came to ~5000 cycles per tile.
//   warps 0..7  softmax, two threads per row: warp w reads TMEM lanes
//               [32 (w % 4), +32); warps 0..3 take the first half of the
//               score columns, warps 4..7 the second.  Each half forms
//               2^(x - m_half) and the half's log-sum-exp; the two halves
//               swap that one value through four TMEM columns (one per half
//               and tile parity), combine it with the sink into the row's
//               log-sum-exp L, and write bf16 P = 2^(x - L) to TMEM; lse ->
//               global.  Two softmax warps per SM sub-partition hide each
//               other's latencies; the exponentials stay exact single-pass.
//   warps 8..11 epilogue: O (TMEM) -> global (fp32, or bf16
//               rounded from the same fp32 values).  The 16x256b
//               TMEM read gives each group of 4 threads 32 contiguous bytes of
//               a row, so every warp store fills whole 32-byte sectors (8
//               heads: one position's 4 KB contiguous; 4 heads: two
//               positions' 2 KB each); this measured clearly faster than one
//               32-byte store per thread per row.
// TMEM (kN = 144 or 160 score columns): S [0, kN), P0 [kN, 1.5 kN), P1
// [1.5 kN, 2 kN) (bf16 pairs), exchange [2 kN, 2 kN + 4), O [384, 512).
// QK^T of tile t+1 runs while softmax works on tile t (S is read out at once).
// P is double-buffered, so the softmax of tile t writes its P while tile
// t-1's PV may still be running; O is single-buffered, as the epilogue
// empties it into registers long before the next PV is issued (that PV waits
// for the softmax of the next tile).  TMEM holds no more: S, two P, O and
// the exchange take 420 (8 heads) or 452 (4 heads) of 512 columns, two O
// buffers would need 548.
// 15 warps put 4 on three of the SM's sub-partitions, which caps registers at
// 128 per thread: a softmax thread holds 72 or 80 scores, an epilogue thread
// 64 output values at a time.
#pragma once

#include "device_common.cuh"

namespace swa {
namespace tcswa {

constexpr int kThreads = 480;
constexpr int kWarpProducer = 12, kWarpMma = 13, kWarpPv = 14;
constexpr int kWarpEpi0 = 8;
constexpr int kD = 128;          // largest head dimension (64 is the other)
constexpr int kBlk = 16;         // keys per ring block
constexpr uint32_t kRing = 12;   // ring slots
constexpr uint32_t kQStages = 4;
constexpr int kMaxW = 8 * kBlk + 1;  // 129: 8 blocks before a tile's first key block
constexpr int kGroup = 8;        // heads of a tile group when G is a multiple of 8

// Tile shape for kG query heads per tile (8, or 4 when G = 4).
template <int kG>
struct Shape {
  static constexpr int kNpos = 128 / kG;        // positions per tile
  static constexpr int kNew = kNpos / kBlk;     // key blocks a tile adds to its run
  static constexpr int kNB = 8 + kNew;          // key blocks per tile window
  static constexpr int kN = kNB * kBlk;         // score columns: 144 or 160
  static constexpr int kNh = kN / 2;            // columns per softmax half
  static constexpr uint32_t kColP = kN;         // P buffers [kN, kN + kNh), [kN + kNh, 2 kN)
  static constexpr uint32_t kColX = 2 * kN;     // half-row exchange, 4 columns
};

// shared-memory map (bytes); swizzled regions 1024-aligned
constexpr int kQHalf = 128 * 128;                     // 128 rows x 64 bf16
constexpr int kQStage = 2 * kQHalf;                   // 32 KB
constexpr int kBlkHalf = kBlk * 128;                  // 16 keys x 64 bf16 = 2 KB
constexpr int kRingHalf = kRing * kBlkHalf;           // 24 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQStages * kQStage;     // 128 KB
constexpr int kOffV = kOffK + 2 * kRingHalf;          // +48 KB
constexpr int kOffBar = kOffV + 2 * kRingHalf;        // +48 KB
// barriers
constexpr int kBarQFull = 0, kBarQEmpty = kQStages, kBarKvFull = 2 * kQStages,
              kBarKvEmpty = kBarKvFull + kRing, kBarSFull = kBarKvEmpty + kRing,
              kBarSFree = kBarSFull + 1, kBarPFull = kBarSFree + 1, kBarPFree = kBarPFull + 2,
              kBarOFull = kBarPFree + 2, kBarOFree = kBarOFull + 1, kBarXchg = kBarOFree + 1,
              kBarDrain = kBarXchg + 4, kNumBars = kBarDrain + 2;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;      // + slack for 1024 alignment

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 384;
static_assert(2 * Shape<4>::kN + 4 <= (int)kColO && 2 * Shape<8>::kN + 4 <= (int)kColO,
              "S, two P buffers and the exchange end before O");

struct Params {
  const float* sink;
  void* out;            // float, or bf16 with kBf16Out
  float* lse;
  int B, T, Hq, Hkv, W;
  int Hg;               // tile groups per sequence: Hq / (heads per tile)
  int rep;              // tile groups per kv head (1 unless G = 16, 24, ...)
  int n_first;          // first tile of each sequence computed
  int ntiles_seq;       // tiles computed per (sequence, tile group): n_first .. n_first + ntiles_seq - 1
  int total_tiles;      // B * Hg * ntiles_seq (< 2^31, checked on the host)
  float scale_log2;     // log2(e) / sqrt(D)
  int out_align32;      // out is 32-byte aligned (bf16 output stores whole sectors)
  int withhold_cta;     // testing aid: this CTA's producer issues no load (-1: none), so
                        // its waits run out and it takes the error path
};

// Tile order: (sibling r, sequence b, kv head, n), where the tile group is
// grp = kv head x rep + r.  With rep > 1 the CTAs split into rep equal sets
// that walk the same (b, kv head, n) tiles of sibling groups at the same
// pace, so the second set reads each key/value row shortly after the first
// one brought it into L2; walking a kv head's groups one after the other put
// ~110 us of other traffic between the two reads and each row came from HBM
// twice.
struct TileWalk {
  int b, kvh, r, n;
  int grp;   // kvh * rep + r: query heads [grp kG, grp kG + kG)
  __device__ __forceinline__ void start(uint32_t u, const Params& p) {
    const uint32_t bk = u / (uint32_t)p.ntiles_seq;
    n = p.n_first + (int)(u - bk * (uint32_t)p.ntiles_seq);
    const uint32_t nbk = (uint32_t)(p.B * p.Hkv);
    r = (int)(bk / nbk);
    const uint32_t bk2 = bk - (uint32_t)r * nbk;
    b = (int)(bk2 / (uint32_t)p.Hkv);
    kvh = (int)(bk2 - (uint32_t)b * (uint32_t)p.Hkv);
    grp = kvh * p.rep + r;
  }
  __device__ __forceinline__ void next(const Params& p) {
    if (++n == p.n_first + p.ntiles_seq) {
      n = p.n_first;
      if (++kvh == p.Hkv) {
        kvh = 0;
        if (++b == p.B) {
          b = 0;
          ++r;
        }
      }
      grp = kvh * p.rep + r;
    }
  }
};

template <bool kBf16Out, int kG, int kHd>
__global__ void __launch_bounds__(kThreads, 1)
    swa_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v, const Params p) {
  using S = Shape<kG>;
  constexpr int kNpos = S::kNpos, kNew = S::kNew, kNB = S::kNB, kNh = S::kNh;
  static_assert(kHd == 64 || kHd == 128, "head dimension 64 or 128");
  constexpr int kHalves = kHd / 64;   // 64-dimension halves of q, k, v rows
  auto col_p = [](int b) { return S::kColP + (uint32_t)(kNh * b); };
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

  // contiguous tile range of this CTA: the grid (a multiple of rep) splits
  // into rep sets of CTAs, set r dividing the tiles of sibling r evenly, so
  // that CTA c of every set walks the same (b, kv head, n) tiles in step
  const uint32_t cps = gridDim.x / (uint32_t)p.rep;          // CTAs per set
  const uint32_t set = blockIdx.x / cps, cc = blockIdx.x - set * cps;
  const uint32_t tiles_set = (uint32_t)p.total_tiles / (uint32_t)p.rep;
  const uint32_t per = tiles_set / cps;
  const uint32_t rem = tiles_set % cps;
  const uint32_t t_begin = set * tiles_set + cc * per + (cc < rem ? cc : rem);
  const int ntile = (int)(per + (cc < rem ? 1 : 0));

  if (tid == 0) {
    *abort_flag = 0;
    for (uint32_t s = 0; s < kQStages; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
    }
    for (uint32_t s = 0; s < kRing; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarPFull + s), 256);
      mbar_init(bar(kBarPFree + s), 1);
    }
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), 128);
    for (int s = 0; s < 4; ++s) mbar_init(bar(kBarXchg + s), 64);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSFree), 256);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrain + 1), 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (warp == kWarpProducer) {
    // ======================= TMA producer =======================
    if (lane == 0 && (int)blockIdx.x != p.withhold_cta) {
      uint32_t seq = 0;  // key blocks loaded so far
      int prev_bk = -1;
      int q_issued = 0;  // Q tiles loaded so far
      bool ok = true;
      TileWalk w;
      w.start(t_begin, p);
      for (int it = 0; it < ntile && ok; ++it, w.next(p)) {
        const int b = w.b, grp = w.grp, n = w.n;
        const int kvh = grp / p.rep;
        const uint32_t qs = (uint32_t)it % kQStages;
        const uint32_t qph = ((uint32_t)it / kQStages) & 1;
        if (!mbar_wait(bar(kBarQEmpty + qs), qph ^ 1, kErrWaitQEmpty, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t qdst = sbase + kOffQ + qs * kQStage;
        mbar_arrive_expect_tx(bar(kBarQFull + qs), kHalves * kQHalf);
        tma_load_4d(qdst, &map_q, 0, grp * kG, n * kNpos, b, bar(kBarQFull + qs));
        if constexpr (kHalves == 2)
          tma_load_4d(qdst + kQHalf, &map_q, 64, grp * kG, n * kNpos, b, bar(kBarQFull + qs));
        ++q_issued;
        const int bk = b * p.Hg + grp;
        const int last_blk = n * kNew + kNew - 1;
        const int first_blk = last_blk - ((bk != prev_bk) ? kNB : kNew) + 1;
        prev_bk = bk;
        for (int m = first_blk; m <= last_blk; ++m, ++seq) {
          const uint32_t slot = seq % kRing;
          if (!mbar_wait(bar(kBarKvEmpty + slot), ((seq / kRing) & 1) ^ 1, kErrWaitKvEmpty,
                         abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t kb = bar(kBarKvFull + slot);
          mbar_arrive_expect_tx(kb, 2 * kHalves * kBlkHalf);
          const uint32_t kdst = sbase + kOffK + slot * kBlkHalf;
          const uint32_t vdst = sbase + kOffV + slot * kBlkHalf;
          tma_load_4d(kdst, &map_k, 0, kvh, m * kBlk, b, kb);
          tma_load_4d(vdst, &map_v, 0, kvh, m * kBlk, b, kb);
          if constexpr (kHalves == 2) {
            tma_load_4d(kdst + kRingHalf, &map_k, 64, kvh, m * kBlk, b, kb);
            tma_load_4d(vdst + kRingHalf, &map_v, 64, kvh, m * kBlk, b, kb);
          }
        }
      }
      // Copies still in flight must land before the CTA exits: wait (bounded)
      // for the last phase armed on every barrier a copy signals.
      if (!ok) {
        for (int j = (q_issued > (int)kQStages ? q_issued - (int)kQStages : 0); j < q_issued; ++j)
          mbar_wait_drain(bar(kBarQFull + (uint32_t)j % kQStages), ((uint32_t)j / kQStages) & 1);
        for (uint32_t s2 = (seq > kRing ? seq - kRing : 0); s2 < seq; ++s2)
          mbar_wait_drain(bar(kBarKvFull + s2 % kRing), (s2 / kRing) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ============ MMA issuers: S = Q K^T (warp 13), O = P V (warp 14) ============
    // Each issuing thread waits only on its own barriers, so one thread's
    // waits and bookkeeping no longer hold back the other's MMAs.
    if (lane == 0) {
      const bool s_side = (warp == kWarpMma);
      const uint32_t idesc_o = umma_idesc_bf16(kHd, false, true);
      // Descriptors are built once; per operand they differ only in the
      // start-address field (address >> 4, bits 0..13), advanced by adding
      // the byte offset >> 4 (shared addresses stay below 2^18: no carry).
      const uint64_t qdesc0 = umma_sdesc(sbase + kOffQ, 16, 1024, 2);
      const uint64_t kdesc0 = umma_sdesc(sbase + kOffK, 16, 1024, 2);
      const uint64_t vdesc0 = umma_sdesc(sbase + kOffV, kRingHalf, 1024, 2);
      uint32_t seq = 0;      // blocks loaded (mirrors the producer)
      int prev_bk = -1;
      bool ok = true;
      TileWalk w;
      w.start(t_begin, p);
      for (int it = 0; it < ntile && ok; ++it) {
        const int bk = w.b * p.Hg + w.grp;
        const bool new_run = (bk != prev_bk);
        prev_bk = bk;
        const int nnew = new_run ? kNB : kNew;
        const uint32_t ws = seq + nnew - kNB;  // first block of this tile's window
        w.next(p);
        if (s_side) {
          // wait for this tile's Q and new key/value blocks
          const uint32_t qs = (uint32_t)it % kQStages;
          if (!mbar_wait(bar(kBarQFull + qs), ((uint32_t)it / kQStages) & 1, kErrWaitQFull,
                         abort_flag)) {
            ok = false;
            break;
          }
          for (int r = 0; r < nnew; ++r) {
            const uint32_t s2 = seq + r;
            if (!mbar_wait(bar(kBarKvFull + s2 % kRing), (s2 / kRing) & 1, kErrWaitKvFull,
                           abort_flag)) {
              ok = false;
              break;
            }
          }
          if (!ok) break;
          seq += nnew;
          if (!mbar_wait(bar(kBarSFree), (it & 1) ^ 1, kErrWaitSFree, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // S = Q K^T; the window's blocks may wrap around the ring end
          const uint32_t slot0 = ws % kRing;
          const uint32_t seg1 = (slot0 + kNB <= kRing) ? kNB : kRing - slot0;
          const uint32_t d_s = tmem + kColS;
          const uint32_t idesc1 = umma_idesc_bf16(seg1 * kBlk, false, false);
          const uint32_t idesc2 = umma_idesc_bf16((kNB - seg1) * kBlk, false, false);
          const uint64_t qd = qdesc0 + qs * (kQStage >> 4);
          const uint64_t kd1 = kdesc0 + slot0 * (kBlkHalf >> 4);
          if (seg1 == (uint32_t)kNB) {
#pragma unroll
            for (int kk = 0; kk < kHd / 16; ++kk) {
              const uint32_t a_off = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
              const uint32_t k_off = ((kk >> 2) * kRingHalf + (kk & 3) * 32) >> 4;
              umma_bf16_ss(d_s, qd + a_off, kd1 + k_off, idesc1, kk > 0);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < kHd / 16; ++kk) {
              const uint32_t a_off = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
              const uint32_t k_off = ((kk >> 2) * kRingHalf + (kk & 3) * 32) >> 4;
              umma_bf16_ss(d_s, qd + a_off, kd1 + k_off, idesc1, kk > 0);
              umma_bf16_ss(d_s + seg1 * kBlk, qd + a_off, kdesc0 + k_off, idesc2, kk > 0);
            }
          }
          umma_commit(bar(kBarSFull));
          umma_commit(bar(kBarQEmpty + qs));
        } else {
          seq += nnew;
          // the last tile of a run releases every block of its window, the
          // others only the oldest kNew (their S reads completed before the
          // softmax that produced this P)
          const bool run_end = (it + 1 >= ntile) || (w.b * p.Hg + w.grp != bk);
          const int pb = it & 1;
          if (!mbar_wait(bar(kBarPFull + pb), (it >> 1) & 1, kErrWaitPFull, abort_flag)) {
            ok = false;
            break;
          }
          // O is single-buffered: the epilogue has read tile it - 1's O out of it
          if (!mbar_wait(bar(kBarOFree), (it & 1) ^ 1, kErrWaitOFree, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_o = tmem + kColO;
          uint32_t slot = ws % kRing;
#pragma unroll
          for (int kb = 0; kb < kNB; ++kb) {
            umma_bf16_ts(d_o, tmem + col_p(pb) + kb * (kBlk / 2),
                         vdesc0 + slot * (kBlkHalf >> 4), idesc_o, kb > 0 ? 1u : 0u);
            slot = (slot + 1 == kRing) ? 0 : slot + 1;
          }
          umma_commit(bar(kBarOFull));
          umma_commit(bar(kBarPFree + pb));
          const int nrel = run_end ? kNB : kNew;
          slot = ws % kRing;
          for (int r = 0; r < nrel; ++r) {
            umma_commit(bar(kBarKvEmpty + slot));
            slot = (slot + 1 == kRing) ? 0 : slot + 1;
          }
        }
      }
      // every MMA this thread issued completes before TMEM is released
      const uint32_t db = bar(kBarDrain + (s_side ? 0 : 1));
      umma_commit(db);
      mbar_wait_drain(db, 0);
    }
    __syncwarp();
  } else if (warp < kWarpEpi0) {
    // ======================= softmax (warps 0..7) =======================
    const int quad = warp & 3, half = warp >> 2;
    const int r = quad * 32 + lane;           // tile row = TMEM lane
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const int c0 = half * kNh;                // first score column of this half
    const int pos_in_tile = r / kG, g = r % kG;
    const uint32_t xbar = bar(kBarXchg + quad);
    TileWalk w;
    w.start(t_begin, p);
    for (int it = 0; it < ntile; ++it, w.next(p)) {
      const int b = w.b, grp = w.grp, n = w.n;
      const int h = grp * kG + g;
      const float sk = p.sink[h] * 1.4426950408889634f;
      const int i = n * kNpos + pos_in_tile;            // query position
      const int key0 = (n * kNew - 8) * kBlk;           // key of column 0
      // valid columns [lo, hi] of this half, in half-local indices
      const int lo = max(0, i - p.W + 1) - key0 - c0;
      const int hi = i - key0 - c0;
      if (!mbar_wait(bar(kBarSFull), it & 1, kErrWaitSFull, abort_flag)) break;
      tc_fence_after();
      uint32_t sr[kNh];
      {
        const uint32_t a = tmem + lane_addr + kColS + c0;
        if constexpr (kNh % 16 == 0) {
          // 80 columns per half, 16 at a time
#pragma unroll
          for (int c = 0; c < kNh / 16; ++c)
            tmem_ld16(a + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&sr[16 * c]));
        } else if (half == 0) {
          // half 0: columns 0..71 as 16,16,16,16,8; half 1: 72..143 as 8,16,16,16,16
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld16(a + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&sr[16 * c]));
          tmem_ld8(a + 64, &sr[64]);
        } else {
          tmem_ld8(a, &sr[0]);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld16(a + 8 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&sr[8 + 16 * c]));
        }
      }
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < kNh / 8; ++c) reg_fence8(&sr[8 * c]);
      tc_fence_before();
      mbar_arrive(bar(kBarSFree));

      // Mask in place.  Columns [kNpos, 128) are inside every row's window
      // whenever the warp's rows all have their first valid column <= kNpos and
      // their last >= 127 (W = 128, n past the first tiles): then only the
      // first kNew key blocks (half 0) or the last kNew (half 1) need the
      // per-column test.
      const bool mid_ok = __all_sync(0xffffffffu, lo + c0 <= kNpos && hi + c0 >= 127);
      if (mid_ok && half == 0) {
#pragma unroll
        for (int c = 0; c < kNpos; ++c)
          if (c < lo || c > hi) sr[c] = __float_as_uint(-INFINITY);
      } else if (mid_ok) {
#pragma unroll
        for (int c = 128 - kNh; c < kNh; ++c)
          if (c < lo || c > hi) sr[c] = __float_as_uint(-INFINITY);
      } else {
#pragma unroll
        for (int c = 0; c < kNh; ++c)
          if (c < lo || c > hi) sr[c] = __float_as_uint(-INFINITY);
      }
      // max over the half row: 8 independent chains of 3-input max, then a tree
      float m8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[k + 8]));
#pragma unroll
      for (int c = 16; c + 16 <= kNh; c += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          m8[k] = max3f(m8[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
#pragma unroll
      for (int k = 0; k < 8; ++k) m8[k] = fmaxf(m8[k], __uint_as_float(sr[kNh - 8 + k]));
      const float mraw = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                               fmaxf(m8[6], m8[7]));
      // exponent offset of this half: its max (scale > 0 commutes with max),
      // or 0 when every column of the half is outside the window
      const float mh = (mraw == -INFINITY) ? 0.f : mraw * p.scale_log2;
      // p = 2^(x scale - mh) in place: scale-and-subtract and the sum two
      // columns per instruction (f32x2)
      const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
      const float2 nm2 = make_float2(-mh, -mh);
      float l8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) l8[k] = 0.f;
#pragma unroll
      for (int c = 0; c < kNh; c += 2) {
        const float2 xx = ffma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                sc2, nm2);
        const float a = ex2_approx(xx.x), bb = ex2_approx(xx.y);
        sr[c] = __float_as_uint(a);
        sr[c + 1] = __float_as_uint(bb);
        l8[c & 7] += a;
        l8[(c + 1) & 7] += bb;
      }
      const float lh = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      // log2-sum-exp of this half (-inf when empty), swapped with the other
      // half of the row through TMEM column kColX + 2 (tile parity) + half
      const float lse_h = (lh > 0.f) ? mh + __log2f(lh) : -INFINITY;
      const uint32_t xcol = tmem + lane_addr + S::kColX + 2 * (it & 1);
      {
        const uint32_t v = __float_as_uint(lse_h);
        tmem_st1(xcol + half, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(xbar);
      if (!mbar_wait(xbar, it & 1, kErrWaitXchg, abort_flag)) break;
      tc_fence_after();
      const float lse_o = __uint_as_float(tmem_ld1(xcol + (half ^ 1)));
      // row log2-sum-exp with the sink: L = log2(2^lse_h + 2^lse_o + 2^sk)
      const float mm = fmaxf(fmaxf(lse_h, lse_o), sk);
      const float L = mm + __log2f(ex2_approx(lse_h - mm) + ex2_approx(lse_o - mm) +
                                   ex2_approx(sk - mm));
      // P = 2^(x scale - L) = p 2^(mh - L); an empty half has p = 0
      const float f = (lh > 0.f) ? ex2_approx(mh - L) : 0.f;
      // bf16 P -> TMEM buffer it % 2 once tile it - 2's PV has consumed it
      const int pb = it & 1;
      if (!mbar_wait(bar(kBarPFree + pb), ((it >> 1) & 1) ^ 1, kErrWaitPFree, abort_flag)) break;
      tc_fence_after();
      {
        // packed columns [kNh/2 half, kNh/2 (half + 1)): 8 heads: half 0 as
        // 8,8,8,8,4 and half 1 as 4,8,8,8,8 (each store aligned to its width);
        // 4 heads: 8 at a time
        const uint32_t pa = tmem + lane_addr + col_p(pb) + half * (kNh / 2);
        if constexpr ((kNh / 2) % 8 == 0) {
          // packed and stored 8 at a time, so that the scores already packed
          // free their registers (80 scores plus 40 packed words overflowed
          // the 128-register cap)
#pragma unroll
          for (int c = 0; c < kNh / 16; ++c) {
            uint32_t pk8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              pk8[e] = pack_bf16x2(__uint_as_float(sr[16 * c + 2 * e]) * f,
                                   __uint_as_float(sr[16 * c + 2 * e + 1]) * f);
            tmem_st8(pa + 8 * c, pk8);
          }
        } else {
        uint32_t pk[kNh / 2];
#pragma unroll
        for (int e = 0; e < kNh / 2; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(sr[2 * e]) * f, __uint_as_float(sr[2 * e + 1]) * f);
        if (half == 0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_st8(pa + 8 * c, *reinterpret_cast<const uint32_t(*)[8]>(&pk[8 * c]));
          tmem_st4(pa + 32, &pk[32]);
        } else {
          tmem_st4(pa, &pk[0]);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_st8(pa + 4 + 8 * c, *reinterpret_cast<const uint32_t(*)[8]>(&pk[4 + 8 * c]));
        }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull + pb));
      if (half == 0 && p.lse != nullptr && i < p.T)
        p.lse[((long long)b * p.Hq + h) * p.T + i] = L * 0.6931471805599453f;
    }
  } else {
    // ======================= epilogue (warps 8..11) =======================
    const int sub = warp & 3;                 // TMEM lanes [32 sub, 32 sub + 32)
    const int quad = lane & 3, rr = lane >> 2;
    TileWalk w;
    w.start(t_begin, p);
    for (int it = 0; it < ntile; ++it, w.next(p)) {
      const int b = w.b, grp = w.grp, n = w.n;
      if (!mbar_wait(bar(kBarOFull), it & 1, kErrWaitOFull, abort_flag)) break;
      tc_fence_after();
      const uint32_t col = tmem + kColO + ((uint32_t)(sub * 32) << 16);
      if constexpr (kBf16Out) {
        // thread = tile row (TMEM lane 32 sub + lane): position (32 sub +
        // lane) / kG, head lane % kG; 64 consecutive columns per round,
        // rounded to bf16 and written as whole 32-byte sectors
        const int pos = n * kNpos + (32 * sub + lane) / kG;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                              (((long long)b * p.T + pos) * p.Hq + grp * kG + lane % kG) * kHd;
#pragma unroll
        for (int rd = 0; rd < kHalves; ++rd) {
          uint32_t o[64];
          tmem_ld32(col + 64 * rd, o);
          tmem_ld32(col + 64 * rd + 32, o + 32);
          tmem_ld_wait();
          reg_fence32(o);
          reg_fence32(o + 32);
          if (rd == kHalves - 1) {
            tc_fence_before();
            mbar_arrive(bar(kBarOFree));
          }
          if (pos < p.T) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e)
                pk[e] = pack_bf16x2(__uint_as_float(o[32 * c + 2 * e]),
                                    __uint_as_float(o[32 * c + 2 * e + 1]));
              float* dst = reinterpret_cast<float*>(orow + 64 * rd + 32 * c);
              if (p.out_align32) {
                st_global_v8(dst, pk);
                st_global_v8(dst + 8, pk + 8);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  st_global_v4(dst + 4 * e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
              }
            }
          }
        }
      } else {
      // rows of this thread: 32 sub + 16 hf + 8 k + rr (k = 0, 1), i.e.
      // position (row / kG), head (row % kG); columns 8j + 2 quad + {0, 1}
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t o[kHd / 2];
        if constexpr (kHd == 128)
          tmem_ld_16x256b_x16(col + ((uint32_t)(16 * hf) << 16), o);
        else
          tmem_ld_16x256b_x8(col + ((uint32_t)(16 * hf) << 16), o);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kHd / 32; ++c) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(&o[c * 16]));
        if (hf == 1) {
          tc_fence_before();
          mbar_arrive(bar(kBarOFree));
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int row = 32 * sub + 16 * hf + 8 * k + rr;
          const int pos = n * kNpos + row / kG;
          if (pos < p.T) {
            const long long e0 =
                (((long long)b * p.T + pos) * p.Hq + grp * kG + row % kG) * kHd + 2 * quad;
            float* orow = static_cast<float*>(p.out) + e0;
#pragma unroll
            for (int j = 0; j < kHd / 8; ++j)
              st_global_v2(orow + 8 * j, o[4 * j + 2 * k], o[4 * j + 2 * k + 1]);
          }
        }
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

}  // namespace tcswa
}  // namespace swa
