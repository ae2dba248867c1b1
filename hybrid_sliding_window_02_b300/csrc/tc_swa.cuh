// tc_swa.cuh -- sliding-window prefill on the 5th-generation tensor cores.
//
// Operation: causal sliding-window attention with GQA and a per-head sink bias
// in the softmax denominator ("MiMo-V2-Flash Technical Report" summary, section
// 前置知识; 128-token window in section 核心方法).  This kernel covers W <= 129
// (the window plus one 16-position tile spans at most 9 key blocks), bf16
// inputs, D = 128 and groups of 8 query heads per kv head.
//
// Tiling.  One tile = 16 consecutive positions x the 8 query heads of one kv
// head = 128 MMA rows (row r = position (r / 8), head (r % 8)).  The keys that
// tile n needs span positions [16n - W + 1, 16n + 15], i.e. key blocks
// n-8 .. n of 16 keys: a 128 x 144 score tile of which 89% is in the window
// (a 128-position single-head tile would need 256 keys, 50% useful).  The
// whole window fits in tensor memory, so the softmax is an exact single pass
// seeded with the sink (no rescaling).
//
// Persistent CTAs (one per SM) walk a contiguous range of tiles in
// (b, kv head, n) order.  Consecutive tiles of one (b, kv head) share 8 of
// their 9 key blocks, so keys and values live in a 10-slot ring of 16-key
// blocks in shared memory and each key/value row is loaded from HBM once per
// run.  Roles (192 threads):
//   warp 0      TMA producer: Q tile (2 stages) and new K/V blocks (ring)
//   warp 1      TMEM owner + single-thread tcgen05.mma issuer:
//                 S = Q K^T   (M=128, N=144 split at the ring wrap, K=128)
//                 O = P V     (M=128, N=128, K=16 per block, V MN-major)
//   warps 2..5  softmax (TMEM -> registers -> bf16 P in shared memory) and
//               epilogue (TMEM O -> 1/l scaling -> swizzled staging -> TMA store)
// S is double-buffered in TMEM so QK^T of tile t+1 overlaps softmax of tile t;
// output stores are asynchronous bulk tensor copies.
#pragma once

#include "device_common.cuh"

namespace swa {
namespace tcswa {

constexpr int kThreads = 192;
constexpr int kG = 8;            // query heads per tile (one kv group)
constexpr int kNpos = 16;        // positions per tile
constexpr int kD = 128;
constexpr int kBlk = 16;         // keys per ring block
constexpr int kNB = 9;           // blocks per tile window
constexpr int kN = kNB * kBlk;   // 144 score columns
constexpr int kRing = 10;        // ring slots
constexpr int kQStages = 2;
constexpr int kMaxW = (kNB - 1) * kBlk + 1;  // 129

// shared-memory map (bytes); swizzled regions 1024-aligned
constexpr int kQHalf = 128 * 128;                     // 128 rows x 64 bf16
constexpr int kQStage = 2 * kQHalf;                   // 32 KB
constexpr int kBlkHalf = kBlk * 128;                  // 16 keys x 64 bf16 = 2 KB
constexpr int kRingHalf = kRing * kBlkHalf;           // 20 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQStages * kQStage;     // 64 KB
constexpr int kOffV = kOffK + 2 * kRingHalf;          // +40 KB
constexpr int kOffP = kOffV + 2 * kRingHalf;          // +40 KB
constexpr int kPChunk = 128 * 128;                    // 128 rows x 64 keys bf16
constexpr int kOffStage = kOffP + 3 * kPChunk;        // +48 KB
constexpr int kStageBytes = 128 * 128;                // 128 rows x 32 fp32
constexpr int kOffBar = kOffStage + 2 * kStageBytes;  // +32 KB
// barriers
constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarKvFull = 4, kBarKvEmpty = 4 + kRing,
              kBarSFull = 4 + 2 * kRing, kBarSFree = kBarSFull + 2, kBarPFull = kBarSFree + 2,
              kBarPFree = kBarPFull + 1, kBarOFull = kBarPFree + 1, kBarOFree = kBarOFull + 1,
              kNumBars = kBarOFree + 1;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;      // + slack for 1024 alignment

// TMEM columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = kN, kColO = 2 * kN;  // 0, 144, 288 (+128 = 416)

struct Params {
  const float* sink;
  float* lse;
  int B, T, Hq, Hkv, W;
  int ntiles_seq;       // ceil(T / 16)
  long long total_tiles;
  float scale_log2;     // log2(e) / sqrt(D)
};

__device__ __forceinline__ void tile_coords(long long u, const Params& p, int& b, int& kvh,
                                            int& n) {
  const long long bk = u / p.ntiles_seq;
  n = (int)(u - bk * p.ntiles_seq);
  b = (int)(bk / p.Hkv);
  kvh = (int)(bk - (long long)b * p.Hkv);
}

__global__ void __launch_bounds__(kThreads, 1)
    swa_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                      const __grid_constant__ CUtensorMap map_k,
                      const __grid_constant__ CUtensorMap map_v,
                      const __grid_constant__ CUtensorMap map_o, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

  // contiguous tile range of this CTA
  const long long per = p.total_tiles / gridDim.x, rem = p.total_tiles % gridDim.x;
  const long long t_begin = blockIdx.x * per + (blockIdx.x < rem ? blockIdx.x : rem);
  const long long t_end = t_begin + per + (blockIdx.x < rem ? 1 : 0);
  const int ntile = (int)(t_end - t_begin);

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarQFull + s), 1);
      mbar_init(bar(kBarQEmpty + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarSFree + s), 128);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
    mbar_init(bar(kBarPFull), 128);
    mbar_init(bar(kBarPFree), 1);
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), 128);
    fence_mbar_init();
    prefetch_tmap(&map_q);
    prefetch_tmap(&map_k);
    prefetch_tmap(&map_v);
    prefetch_tmap(&map_o);
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      long long seq = 0;  // key blocks loaded so far
      int prev_bk = -1;
      for (int it = 0; it < ntile; ++it) {
        int b, kvh, n;
        tile_coords(t_begin + it, p, b, kvh, n);
        const int qs = it & 1;
        if (!mbar_wait(bar(kBarQEmpty + qs), ((it >> 1) & 1) ^ 1, kErrWaitQEmpty, abort_flag))
          break;
        const uint32_t qdst = sbase + kOffQ + qs * kQStage;
        mbar_arrive_expect_tx(bar(kBarQFull + qs), kQStage);
        tma_load_4d(qdst, &map_q, 0, kvh * kG, n * kNpos, b, bar(kBarQFull + qs));
        tma_load_4d(qdst + kQHalf, &map_q, 64, kvh * kG, n * kNpos, b, bar(kBarQFull + qs));
        const int bk = b * p.Hkv + kvh;
        const int first_blk = (bk != prev_bk) ? n - (kNB - 1) : n;
        prev_bk = bk;
        bool ok = true;
        for (int m = first_blk; m <= n; ++m, ++seq) {
          const int slot = (int)(seq % kRing);
          if (!mbar_wait(bar(kBarKvEmpty + slot), (int)((seq / kRing) & 1) ^ 1, kErrWaitKvEmpty,
                         abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t kb = bar(kBarKvFull + slot);
          mbar_arrive_expect_tx(kb, 4 * kBlkHalf);
          const uint32_t kdst = sbase + kOffK + slot * kBlkHalf;
          const uint32_t vdst = sbase + kOffV + slot * kBlkHalf;
          tma_load_4d(kdst, &map_k, 0, kvh, m * kBlk, b, kb);
          tma_load_4d(kdst + kRingHalf, &map_k, 64, kvh, m * kBlk, b, kb);
          tma_load_4d(vdst, &map_v, 0, kvh, m * kBlk, b, kb);
          tma_load_4d(vdst + kRingHalf, &map_v, 64, kvh, m * kBlk, b, kb);
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc_s_unit = umma_idesc_bf16(kBlk, false, false);
      (void)idesc_s_unit;
      const uint32_t idesc_o = umma_idesc_bf16(kD, false, true);
      long long seq = 0;     // blocks loaded (mirrors the producer)
      int prev_bk = -1;
      int pending = -1;      // tile whose PV is still to be issued
      long long pending_ws = 0;
      bool pending_run_end = false;
      bool ok = true;

      auto issue_pv = [&](int j, long long ws, bool run_end) -> bool {
        if (!mbar_wait(bar(kBarPFull), j & 1, kErrWaitPFull, abort_flag)) return false;
        if (!mbar_wait(bar(kBarOFree), (j & 1) ^ 1, kErrWaitOFree, abort_flag)) return false;
        tc_fence_after();
        for (int kb = 0; kb < kNB; ++kb) {
          const int slot = (int)((ws + kb) % kRing);
          const uint64_t adesc =
              umma_sdesc(sbase + kOffP + (kb >> 2) * kPChunk + (kb & 3) * 32, 16, 1024, 2);
          const uint64_t bdesc =
              umma_sdesc(sbase + kOffV + slot * kBlkHalf, kRingHalf, 1024, 2);
          umma_bf16_ss(tmem + kColO, adesc, bdesc, idesc_o, kb > 0 ? 1u : 0u);
        }
        umma_commit(bar(kBarOFull));
        umma_commit(bar(kBarPFree));
        // release key blocks no later tile of this run needs
        const int nrel = run_end ? kNB : 1;
        for (int r = 0; r < nrel; ++r) umma_commit(bar(kBarKvEmpty + (int)((ws + r) % kRing)));
        return true;
      };

      for (int it = 0; it < ntile && ok; ++it) {
        int b, kvh, n;
        tile_coords(t_begin + it, p, b, kvh, n);
        const int bk = b * p.Hkv + kvh;
        const bool new_run = (bk != prev_bk);
        prev_bk = bk;
        const int nnew = new_run ? kNB : 1;
        // a new run needs the whole ring: finish the previous tile first
        if (new_run && pending >= 0) {
          if (!issue_pv(pending, pending_ws, true)) { ok = false; break; }
          pending = -1;
        }
        // wait for this tile's Q and new key/value blocks
        const int qs = it & 1;
        if (!mbar_wait(bar(kBarQFull + qs), (it >> 1) & 1, kErrWaitQFull, abort_flag)) {
          ok = false;
          break;
        }
        for (int r = 0; r < nnew; ++r) {
          const long long s = seq + r;
          if (!mbar_wait(bar(kBarKvFull + (int)(s % kRing)), (int)((s / kRing) & 1),
                         kErrWaitKvFull, abort_flag)) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
        seq += nnew;
        const long long ws = seq - kNB;  // first block of this tile's window
        const int sb = it & 1;
        if (!mbar_wait(bar(kBarSFree + sb), ((it >> 1) & 1) ^ 1, kErrWaitSFree, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // S = Q K^T; the window's blocks may wrap around the ring end
        const int slot0 = (int)(ws % kRing);
        const int seg1 = (slot0 + kNB <= kRing) ? kNB : kRing - slot0;
        const uint32_t d_s = tmem + (sb ? kColS1 : kColS0);
        const uint32_t qbase = sbase + kOffQ + qs * kQStage;
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * kRingHalf + (kk & 3) * 32;
          const uint64_t adesc = umma_sdesc(qbase + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024, 2);
          const uint64_t b1 = umma_sdesc(sbase + kOffK + slot0 * kBlkHalf + koff, 16, 1024, 2);
          umma_bf16_ss(d_s, adesc, b1, umma_idesc_bf16(seg1 * kBlk, false, false), kk > 0);
          if (seg1 < kNB) {
            const uint64_t b2 = umma_sdesc(sbase + kOffK + koff, 16, 1024, 2);
            umma_bf16_ss(d_s + seg1 * kBlk, adesc, b2,
                         umma_idesc_bf16((kNB - seg1) * kBlk, false, false), kk > 0);
          }
        }
        umma_commit(bar(kBarSFull + sb));
        umma_commit(bar(kBarQEmpty + qs));
        if (pending >= 0) {
          if (!issue_pv(pending, pending_ws, pending_run_end)) { ok = false; break; }
        }
        pending = it;
        pending_ws = ws;
        // is the next tile in the same run?
        bool run_end = true;
        if (it + 1 < ntile) {
          int b2, kvh2, n2;
          tile_coords(t_begin + it + 1, p, b2, kvh2, n2);
          run_end = (b2 * p.Hkv + kvh2) != bk;
        }
        pending_run_end = run_end;
      }
      if (ok && pending >= 0) issue_pv(pending, pending_ws, true);
    }
  } else {
    // ======================= softmax + epilogue (warps 2..5) =======================
    const int sub = warp & 3;                 // TMEM sub-partition of this warp
    const int r = sub * 32 + lane;            // tile row = TMEM lane
    const int ct = tid - 64;                  // 0..127 within the compute group
    const uint32_t lane_addr = (uint32_t)(sub * 32) << 16;
    const int pos_in_tile = r >> 3, g = r & 7;
    for (int it = 0; it < ntile; ++it) {
      int b, kvh, n;
      tile_coords(t_begin + it, p, b, kvh, n);
      const int sb = it & 1;
      if (!mbar_wait(bar(kBarSFull + sb), (it >> 1) & 1, kErrWaitSFull, abort_flag)) break;
      tc_fence_after();
      float s[kN];
      {
        const uint32_t base = tmem + lane_addr + (sb ? kColS1 : kColS0);
#pragma unroll
        for (int c = 0; c < kNB; ++c) {
          uint32_t v[16];
          tmem_ld16(base + c * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) s[c * 16 + e] = __uint_as_float(v[e]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarSFree + sb));

      // mask + sink-seeded softmax (exact: the whole window is in this row)
      const int i = n * kNpos + pos_in_tile;            // query position
      const int key0 = (n - (kNB - 1)) * kBlk;          // key of column 0
      const int jlo = max(0, i - p.W + 1);
      const int c_lo = jlo - key0, c_hi = i - key0;     // valid columns [c_lo, c_hi]
      const int h = kvh * kG + g;
      const float sk = p.sink[h] * 1.4426950408889634f;
      float mx = sk;
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        s[c] = (c >= c_lo && c <= c_hi) ? s[c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      float l = (sk == -INFINITY) ? 0.f : ex2_approx(sk - mx);
#pragma unroll
      for (int c = 0; c < kN; ++c) {
        s[c] = ex2_approx(s[c] - mx);
        l += s[c];
      }
      // P (bf16, unnormalised) -> shared memory, K-major 128-byte swizzle
      if (!mbar_wait(bar(kBarPFree), (it & 1) ^ 1, kErrWaitPFree, abort_flag)) break;
      {
        const uint32_t prow = sbase + kOffP + r * 128;
#pragma unroll
        for (int u = 0; u < kN / 8; ++u) {
          const int chunk = u >> 3, unit = u & 7;
          const uint32_t addr = prow + chunk * kPChunk + ((unit ^ (r & 7)) << 4);
          st_shared_v4(addr, pack_bf16x2(s[8 * u + 0], s[8 * u + 1]),
                       pack_bf16x2(s[8 * u + 2], s[8 * u + 3]),
                       pack_bf16x2(s[8 * u + 4], s[8 * u + 5]),
                       pack_bf16x2(s[8 * u + 6], s[8 * u + 7]));
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(kBarPFull));

      // epilogue: O (TMEM) -> registers -> scaled, swizzled staging -> TMA store
      if (!mbar_wait(bar(kBarOFull), it & 1, kErrWaitOFull, abort_flag)) break;
      tc_fence_after();
      float o[kD];
#pragma unroll
      for (int c = 0; c < kD / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + kColO + c * 16, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) o[c * 16 + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(bar(kBarOFree));
      const float inv_l = 1.f / l;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int buf = q4 & 1;
        if (ct == 0) bulk_wait_read<1>();
        named_bar_sync(1, 128);
        const uint32_t srow = sbase + kOffStage + buf * kStageBytes + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float* x = &o[q4 * 32 + u * 4];
          st_shared_v4(srow + ((u ^ (r & 7)) << 4), __float_as_uint(x[0] * inv_l),
                       __float_as_uint(x[1] * inv_l), __float_as_uint(x[2] * inv_l),
                       __float_as_uint(x[3] * inv_l));
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (ct == 0) {
          tma_store_4d(&map_o, sbase + kOffStage + buf * kStageBytes, q4 * 32, kvh * kG,
                       n * kNpos, b);
          bulk_commit();
        }
      }
      if (p.lse != nullptr && i < p.T)
        p.lse[((long long)b * p.Hq + h) * p.T + i] = (mx + __log2f(l)) * 0.6931471805599453f;
    }
    if (ct == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tcswa
}  // namespace swa
