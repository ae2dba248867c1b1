// tc_global.cuh -- global (full causal) attention, and any window wider than
// the sliding-window kernel covers, on the 5th-generation tensor cores.
//
// Operation: the same sink-biased softmax attention as the sliding-window
// kernel ("MiMo-V2-Flash Technical Report" summary, section 前置知识: the
// global layers of the hybrid stack attend to the whole causal prefix; every
// head adds a learnable bias to its softmax denominator), for bf16 inputs,
// D = 64 or 128 and 1, 2, 4 or any multiple of 8 query heads per kv head,
// any window W (W >= T is the global layer).  Keys are visited in blocks of
// 128 with an online softmax: the running max starts at the sink logit and
// the running denominator at exp(sink - max), so the sink is counted exactly
// once whatever the order.
//
// Work item = one group of 8 query heads of one sequence x 32 consecutive
// positions, split into two Q tiles of 16 positions x 8 heads (128 MMA rows
// each, row r = position r / 8, head r % 8); with G = 1, 2 or 4 query heads
// per kv head, 256 / G positions in two tiles of 128 / G positions x G heads
// (row r = position r / G, head r % G).  Both tiles share every K/V block
// the CTA loads, which halves the K/V traffic out of L2 against one tile per
// block.
// Items go to persistent CTAs (one per SM), dealt round by round in
// alternating direction, in an order whose item lengths change smoothly
// (item_coords), which keeps the per-CTA totals within about one item of
// each other without any shared counter.
//
// Roles (352 threads):
//   warp 8      TMA producer: the two Q tiles of an item, then K_j and V_j for
//               every key block j into a ring of 32 KB slots
//   warp 9      TMEM owner + issuer of S   = Q_i K_j^T  (SS, M = N = K = 128)
//   warp 10     issuer of                O_i += P_i V_j   (TS, P_i from TMEM,
//               V MN-major, N = D)
//   warps 0..3  softmax of tile 0, warps 4..7 softmax of tile 1: thread =
//               row; S -> mask -> running max / sum -> bf16 P_i in TMEM;
//               after the last block O / l -> out and the lse.
// The tensor pipe accepts only a few MMAs ahead of the one executing, so a
// single issuing thread that stops at a barrier between two groups of MMAs
// leaves the pipe idle for that wait (about 100-200 cycles each, as the
// issuing warp shares its sub-partition with two softmax warps).  With the S
// and PV products issued from two threads, one thread's waits are covered by
// the other's MMAs; each accumulator still receives its MMAs in order, so the
// results are unchanged.
// TMEM (D = 128): S [0,128) shared by the two tiles, P0 [128,192), P1
// [192,256) (bf16 pairs), O0 [256,384), O1 [384,512).  S goes to one buffer
// that each softmax empties into registers at once, so an S waits only for
// the other tile's read of the previous one, and P never shares columns
// with S.  A softmax
// rewrites P_i (and rescales O_i) only after the tile's previous PV has
// completed, which it learns from a commit barrier.
//
// Rescaling: the running max m only moves when a block's max exceeds it by
// more than 8 (log2 units).  Otherwise p = 2^(x - m) <= 256 and the stale m
// is kept; the final O / l is the same quotient.  When a row's max does move
// after the item's first block, its warp rescales O_i in TMEM (read,
// multiply, write) before releasing P_i.
//
// D = 64: a q, k or v row is one 128-byte swizzle atom instead of two, so
// every load copies one half, S takes 4 K-steps instead of 8 and PV has
// N = 64.  The shared-memory layout stays that of D = 128 (the second half of
// each buffer is unused).  With O at 64 columns per tile, TMEM has room for
// one S buffer per tile: S0 [0,128), S1 [128,256), P0 [256,320), P1
// [320,384), O0 [384,448), O1 [448,512).  An S then waits only for its own
// tile's softmax to read the previous one; with half the MMA work per block
// for the same softmax, the chain through the shared buffer (S0, read, S1,
// read, ...) would set the pace.
#pragma once

#include "device_common.cuh"

namespace swa {
namespace tcglobal {

constexpr int kThreads = 352;
constexpr int kWarpProducer = 8, kWarpMma = 9, kWarpPv = 10;
constexpr int kG = 8;                   // query heads per tile (one kv group), or G = 1, 2, 4
constexpr int kTiles = 2;               // Q tiles per work item
// positions per Q tile and per work item for kGt heads per tile (128 rows)
__host__ __device__ constexpr int npos_for(int kGt) { return 128 / kGt; }
__host__ __device__ constexpr int item_pos_for(int kGt) { return kTiles * npos_for(kGt); }
constexpr int kBlk = 128;               // keys per block
constexpr uint32_t kSlots = 5;          // K/V ring slots (one K or V block each)
constexpr float kRescaleLog2 = 8.0f;    // move the running max only past this

// shared memory (bytes), laid out for D = 128; swizzled operands 1024-aligned
constexpr int kQHalf = 128 * 128;           // 128 rows x 64 bf16
constexpr int kQTile = 2 * kQHalf;          // 32 KB
constexpr int kSlotHalf = kBlk * 128;       // 128 keys x 64 bf16
constexpr int kSlotBytes = 2 * kSlotHalf;   // 32 KB
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kTiles * kQTile;
constexpr int kOffBar = kOffKV + (int)kSlots * kSlotBytes;
constexpr int kBarQFull = 0, kBarQEmpty = kBarQFull + kTiles, kBarKvFull = kBarQEmpty + kTiles,
              kBarKvEmpty = kBarKvFull + kSlots, kBarSFull = kBarKvEmpty + kSlots,
              kBarSFree = kBarSFull + kTiles, kBarPFull = kBarSFree + kTiles,
              kBarPvDone = kBarPFull + kTiles, kBarOFull = kBarPvDone + kTiles,
              kBarDrain = kBarOFull + kTiles, kNumBars = kBarDrain + 2;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 8;
constexpr int kSmemBytes = kOffAbort + 8 + 1024;  // + slack for 1024 alignment

constexpr uint32_t kTmemCols = 512;
// TMEM columns of S_i, P_i and O_i: at D = 128 one S buffer shared by the two
// tiles, at D = 64 one per tile (kSplitS)
template <int kHd>
struct Cols {
  static constexpr bool kSplitS = kHd == 64;
  __host__ __device__ static constexpr uint32_t s(int i) { return kSplitS ? 128u * (uint32_t)i : 0u; }
  __host__ __device__ static constexpr uint32_t p(int i) {
    return (kSplitS ? 256u : 128u) + 64u * (uint32_t)i;
  }
  __host__ __device__ static constexpr uint32_t o(int i) {
    return kSplitS ? 384u + 64u * (uint32_t)i : 256u + 128u * (uint32_t)i;
  }
};
static_assert(Cols<64>::o(1) + 64 <= kTmemCols && Cols<128>::o(1) + 128 <= kTmemCols,
              "TMEM layout fits the allocation");

struct Params {
  const float* sink;
  void* out;          // float, or bf16 with kBf16Out
  float* lse;
  int B, T, Hq, Hkv, W;
  int Hg;             // head groups of a tile per sequence: Hq / (heads per tile)
  int rep;            // groups per kv head: G / 8 for G = 8 R, else 1 (1 with scores or sparse mode)
  int item_pos;       // positions per work item: 32 (8 heads per tile) or 64 (4)
  int nitem_seq;      // ceil(T / item_pos)
  int total_items;    // B * Hg * nitem_seq (< 2^31, checked on the host)
  float scale_log2;   // log2(e) / sqrt(D)
  // block scores (optional): blockmax[b][kvh][ceil(T/4)][ceil(T/128)], the max
  // scaled logit of each (4-position group, 128-key block) over the group's
  // 8 heads; written for the blocks an item visits
  float* blockmax;
  int nqg, nkb;
  // sparse mode (optional): the item visits the key blocks listed in
  // blk_idx[b][kvh][p0 / qb_size][0 .. topk) (increasing, -1 padded) instead
  // of every block of its window
  const int* blk_idx;
  int qb_size, topk, nqb;
};

struct Item {
  int b, grp, kvh, p0;  // query heads [8 grp, 8 grp + 8), kv head grp / rep; first position of tile 0
  int jlo, nb;        // key blocks jlo .. jlo + nb - 1, or blocks[0 .. nb)
  const int* blocks;  // sparse mode: the item's block list
};

// The u-th item: the (sequence, head group) pairs one after another, the
// items of each in order of decreasing causal length for the last pair and
// every second one before it, increasing for the others (a snake: lengths
// change smoothly from one pair to the next and the run ends on the shortest
// items).  The CTAs then share one or two kv heads at any moment, whose keys
// and values (16.8 MB per kv head at T = 32768) stay in L2.  Dealt over all
// kv heads at once, the live keys and values of all 8 heads (134 MB)
// overflowed it and were re-read from HBM: 2.8x the inputs in the dense
// layer, 3.5x in the sparse one (its items are of nearly equal length, so
// the order only decides which keys are live together).
__device__ __forceinline__ Item item_coords(uint32_t u, const Params& p) {
  Item it;
  const uint32_t bkn = (uint32_t)(p.B * p.Hg);
  const uint32_t bk = u / (uint32_t)p.nitem_seq;
  uint32_t r = u - bk * (uint32_t)p.nitem_seq;
  if ((bkn - 1 - bk) & 1u) r = (uint32_t)p.nitem_seq - 1 - r;
  const int n2 = p.nitem_seq - 1 - (int)r;
  it.b = (int)(bk / (uint32_t)p.Hg);
  it.grp = (int)(bk - (uint32_t)it.b * (uint32_t)p.Hg);
  it.kvh = it.grp / p.rep;
  it.p0 = n2 * p.item_pos;
  if (p.blk_idx != nullptr) {
    it.blocks = p.blk_idx + (((int64_t)it.b * p.Hkv + it.kvh) * p.nqb + it.p0 / p.qb_size) * p.topk;
    // the item's blocks are the entries before the first negative one; the
    // entries are read with independent loads (a loop that stops at the
    // first -1 chains one global-load latency per entry, ~10k cycles per
    // item start)
    int nb = p.topk;
#pragma unroll 8
    for (int i = p.topk - 1; i >= 0; --i)
      if (__ldg(it.blocks + i) < 0) nb = i;
    it.jlo = 0;
    it.nb = nb;
    return it;
  }
  it.blocks = nullptr;
  const int last = min(it.p0 + p.item_pos - 1, p.T - 1);
  const int first_key = max(0, it.p0 - p.W + 1);
  it.jlo = first_key / kBlk;
  it.nb = last / kBlk - it.jlo + 1;
  return it;
}

// key block of step t of an item
__device__ __forceinline__ int item_block(const Item& it, int t) {
  return it.blocks != nullptr ? __ldg(it.blocks + t) : it.jlo + t;
}

// The k-th item of CTA c: rounds of gridDim.x items, dealt in alternating
// direction.  Returns false past the end.
__device__ __forceinline__ bool cta_item(int k, const Params& p, Item& it) {
  const uint32_t g = gridDim.x;
  const uint32_t idx = (k & 1) ? (g - 1 - blockIdx.x) : blockIdx.x;
  const uint64_t u = (uint64_t)k * g + idx;
  if (u >= (uint64_t)p.total_items) return false;
  it = item_coords((uint32_t)u, p);
  return true;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

template <bool kBf16Out, bool kScores, int kHd, int kGt>
__global__ void __launch_bounds__(kThreads, 1)
    swa_fwd_tc_global_kernel(const __grid_constant__ CUtensorMap map_q,
                             const __grid_constant__ CUtensorMap map_k,
                             const __grid_constant__ CUtensorMap map_v, const Params p) {
  static_assert(kHd == 64 || kHd == 128, "head dimension 64 or 128");
  static_assert(kGt == 8 || ((kGt == 1 || kGt == 2 || kGt == 4) && !kScores),
                "8 heads per tile, or 1, 2 or 4 without block scores");
  constexpr int kNpos = npos_for(kGt);   // positions per Q tile: row r = position r / kGt, head r % kGt
  constexpr int kHalves = kHd / 64;   // 64-dimension halves of q, k, v rows
  using C = Cols<kHd>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return sbase + kOffBar + 8u * i; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

  if (tid == 0) {
    *abort_flag = 0;
    for (int i = 0; i < kTiles; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQEmpty + i), 1);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarPFull + i), 128);
      mbar_init(bar(kBarPvDone + i), 1);
      mbar_init(bar(kBarOFull + i), 1);
    }
    for (int i = 0; i < kTiles; ++i) mbar_init(bar(kBarSFree + i), 128);
    for (uint32_t s = 0; s < kSlots; ++s) {
      mbar_init(bar(kBarKvFull + s), 1);
      mbar_init(bar(kBarKvEmpty + s), 1);
    }
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
    if (lane == 0) {
      uint32_t seq = 0;  // K/V blocks loaded so far (K and V count separately)
      uint32_t q_armed[kTiles] = {};  // Q loads issued per tile
      Item it;
      bool ok = true;
      uint32_t kn = 0;   // items with at least one key block so far
      for (int k = 0; ok && cta_item(k, p, it); ++k) {
        // an empty block list (sparse mode) has no loads and no MMAs; the
        // softmax warps write its rows from the sink alone
        if (it.nb == 0) continue;
        for (int i = 0; i < kTiles; ++i) {
          if (!mbar_wait(bar(kBarQEmpty + i), (kn & 1) ^ 1, kErrWaitQEmpty, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t qdst = sbase + kOffQ + i * kQTile;
          const int pos = it.p0 + i * kNpos;
          mbar_arrive_expect_tx(bar(kBarQFull + i), kHalves * kQHalf);
          tma_load_4d(qdst, &map_q, 0, it.grp * kGt, pos, it.b, bar(kBarQFull + i));
          if constexpr (kHalves == 2)
            tma_load_4d(qdst + kQHalf, &map_q, 64, it.grp * kGt, pos, it.b, bar(kBarQFull + i));
          ++q_armed[i];
        }
        // The next item's Q tiles and first key blocks go to L2 now, so that
        // its loads (issued only once this item has released the Q buffers)
        // do not start from HBM: with short items (sparse mode) that wait
        // measured ~6 us per item.
        {
          Item nx;
          if (ok && cta_item(k + 1, p, nx)) {
            for (int i = 0; i < kTiles; ++i)
              for (int hv = 0; hv < kHalves; ++hv)
                tma_prefetch_l2_4d(&map_q, 64 * hv, nx.grp * kGt, nx.p0 + i * kNpos, nx.b);
            for (int t = 0; t < 2 && t < nx.nb; ++t) {
              const int key = item_block(nx, t) * kBlk;
              for (int hv = 0; hv < kHalves; ++hv) {
                tma_prefetch_l2_4d(&map_k, 64 * hv, nx.kvh, key, nx.b);
                tma_prefetch_l2_4d(&map_v, 64 * hv, nx.kvh, key, nx.b);
              }
            }
          }
        }
        for (int t = 0; ok && t < 2 * it.nb; ++t, ++seq) {
          const uint32_t slot = seq % kSlots;
          if (!mbar_wait(bar(kBarKvEmpty + slot), ((seq / kSlots) & 1) ^ 1, kErrWaitKvEmpty,
                         abort_flag)) {
            ok = false;
            break;
          }
          const CUtensorMap* map = (t & 1) ? &map_v : &map_k;
          const int key = item_block(it, t >> 1) * kBlk;
          const uint32_t dst = sbase + kOffKV + slot * kSlotBytes;
          const uint32_t fb = bar(kBarKvFull + slot);
          mbar_arrive_expect_tx(fb, kHalves * kSlotHalf);
          tma_load_4d(dst, map, 0, it.kvh, key, it.b, fb);
          if constexpr (kHalves == 2) tma_load_4d(dst + kSlotHalf, map, 64, it.kvh, key, it.b, fb);
        }
        ++kn;
      }
      // Copies still in flight must land before the CTA exits: wait (bounded)
      // for the last phase armed on every barrier a copy signals.
      if (!ok) {
        for (int i = 0; i < kTiles; ++i)
          if (q_armed[i] > 0) mbar_wait_drain(bar(kBarQFull + i), (q_armed[i] - 1) & 1);
        for (uint32_t s = (seq > kSlots ? seq - kSlots : 0); s < seq; ++s)
          mbar_wait_drain(bar(kBarKvFull + s % kSlots), (s / kSlots) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ============ MMA issuers: S products (warp 9), PV products (warp 10) ============
    // Two issuing threads keep the tensor pipe fed while either one waits on
    // a barrier; each accumulator still receives its MMAs in program order.
    if (lane == 0) {
      const bool s_side = (warp == kWarpMma);
      const uint32_t idesc_s = umma_idesc_bf16(kBlk, false, false);
      const uint32_t idesc_o = umma_idesc_bf16(kHd, false, true);
      const uint64_t qdesc0 = umma_sdesc(sbase + kOffQ, 16, 1024, 2);
      const uint64_t kdesc0 = umma_sdesc(sbase + kOffKV, 16, 1024, 2);
      const uint64_t vdesc0 = umma_sdesc(sbase + kOffKV, kSlotHalf, 1024, 2);
      uint32_t gblk = 0;      // key blocks consumed so far (all items)
      uint32_t ns = 0;        // S products issued (S0 and S1 alternate)
      uint32_t ns_t[kTiles] = {};   // per tile
      bool ok = true;
      // K of block g is ring load 2g, V of block g is load 2g + 1
      auto wait_load = [&](uint32_t seq, uint32_t& slot) -> bool {
        slot = seq % kSlots;
        return mbar_wait(bar(kBarKvFull + slot), (seq / kSlots) & 1, kErrWaitKvFull, abort_flag);
      };
      // S = Q_i K^T once the softmax that read the buffer's previous S (the
      // other tile's with one shared buffer, this tile's with one per tile)
      // has emptied it
      auto issue_s = [&](int i, uint32_t ks) -> bool {
        const uint32_t used = C::kSplitS ? ns_t[i] : ns;
        if (used > 0 && !mbar_wait(bar(kBarSFree + (C::kSplitS ? i : 0)), (used - 1) & 1,
                                   kErrWaitSFree, abort_flag))
          return false;
        tc_fence_after();
        const uint64_t qd = qdesc0 + (uint32_t)(i * kQTile >> 4);
        const uint64_t kd = kdesc0 + (ks * kSlotBytes >> 4);
#pragma unroll
        for (int kk = 0; kk < kHd / 16; ++kk) {
          const uint32_t a_off = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
          const uint32_t b_off = ((kk >> 2) * kSlotHalf + (kk & 3) * 32) >> 4;
          umma_bf16_ss(tmem + C::s(i), qd + a_off, kd + b_off, idesc_s, kk > 0);
        }
        umma_commit(bar(kBarSFull + i));
        ++ns;
        ++ns_t[i];
        return true;
      };
      // O_i += P_i V for block number blk
      auto issue_pv = [&](int i, uint32_t vs, uint32_t blk, bool first, bool last) -> bool {
        if (!mbar_wait(bar(kBarPFull + i), blk & 1, kErrWaitPFull, abort_flag)) return false;
        tc_fence_after();
        const uint64_t vd = vdesc0 + (vs * kSlotBytes >> 4);
#pragma unroll
        for (int kb = 0; kb < kBlk / 16; ++kb)
          umma_bf16_ts(tmem + C::o(i), tmem + C::p(i) + kb * 8,
                       vd + (uint32_t)(kb * 16 * 128 >> 4), idesc_o, (!first || kb > 0));
        umma_commit(bar(kBarPvDone + i));
        if (last) umma_commit(bar(kBarOFull + i));
        return true;
      };

      Item it;
      uint32_t kn = 0;   // items with at least one key block so far
      for (int k = 0; ok && cta_item(k, p, it); ++k) {
        if (it.nb == 0) continue;   // no loads, no MMAs
        for (int t = 0; t < it.nb; ++t, ++gblk) {
          uint32_t slot;
          if (s_side) {
            if (!wait_load(2 * gblk, slot)) { ok = false; break; }
            if (t == 0 && !mbar_wait(bar(kBarQFull + 0), kn & 1, kErrWaitQFull, abort_flag)) {
              ok = false;
              break;
            }
            if (!issue_s(0, slot)) { ok = false; break; }
            if (t == 0 && !mbar_wait(bar(kBarQFull + 1), kn & 1, kErrWaitQFull, abort_flag)) {
              ok = false;
              break;
            }
            if (!issue_s(1, slot)) { ok = false; break; }
            umma_commit(bar(kBarKvEmpty + slot));
            if (t == it.nb - 1)
              for (int i = 0; i < kTiles; ++i) umma_commit(bar(kBarQEmpty + i));
          } else {
            if (!wait_load(2 * gblk + 1, slot)) { ok = false; break; }
            const bool first = t == 0, last = t == it.nb - 1;
            if (!issue_pv(0, slot, gblk, first, last)) { ok = false; break; }
            if (!issue_pv(1, slot, gblk, first, last)) { ok = false; break; }
            umma_commit(bar(kBarKvEmpty + slot));
          }
        }
        ++kn;
      }
      // every MMA this thread issued completes before TMEM is released
      const uint32_t db = bar(kBarDrain + (s_side ? 0 : 1));
      umma_commit(db);
      mbar_wait_drain(db, 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue (warps 0..7) =======================
    const int ti = warp >> 2;                       // Q tile of this warpgroup
    const int quad = warp & 3;                      // TMEM lanes [32 quad, 32 quad + 32)
    const int r = quad * 32 + lane;                 // tile row
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + C::s(ti);
    const uint32_t p_addr = tmem + lane_addr + C::p(ti);
    const uint32_t o_addr = tmem + lane_addr + C::o(ti);
    const int g = r % kGt;
    uint32_t npv = 0;
    uint32_t kn = 0;   // items with at least one key block so far
    Item it;
    for (int k = 0; cta_item(k, p, it); ++k) {
      const int h = it.grp * kGt + g;
      const int pos = it.p0 + ti * kNpos + r / kGt;
      if (it.nb == 0) {
        // no key block selected: the sink alone, out = 0 and lse = sink
        if (pos < p.T) {
          const long long e0 = (((long long)it.b * p.T + pos) * p.Hq + h) * kHd;
          if constexpr (kBf16Out) {
            uint32_t* orow = reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.out) + e0);
            for (int e = 0; e < kHd / 8; ++e) st_global_v4(reinterpret_cast<float*>(orow + 4 * e), 0u, 0u, 0u, 0u);
          } else {
            float* orow = static_cast<float*>(p.out) + e0;
            for (int e = 0; e < kHd / 4; ++e) st_global_v4(orow + 4 * e, 0u, 0u, 0u, 0u);
          }
          if (p.lse != nullptr) p.lse[((long long)it.b * p.Hq + h) * p.T + pos] = p.sink[h];
        }
        continue;
      }
      const float sk = p.sink[h] * 1.4426950408889634f;  // log2 units
      float m_run = sk;                                   // -inf for no sink
      float l = (sk == -INFINITY) ? 0.f : 1.f;            // exp2(sk - m_run)
      // valid keys of this row: [key_lo, pos]
      const int key_lo = max(0, pos - p.W + 1);
      bool ok = true;
      for (int t = 0; t < it.nb; ++t, ++npv) {
        const int kblk = item_block(it, t);
        const int key0 = kblk * kBlk;
        const int c_lo = key_lo - key0, c_hi = pos - key0;
        if (!mbar_wait(bar(kBarSFull + ti), npv & 1, kErrWaitSFull, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kBlk];
#pragma unroll
        for (int c = 0; c < kBlk / 32; ++c) tmem_ld32(s_addr + c * 32, sr + c * 32);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kBlk / 32; ++c) reg_fence32(sr + c * 32);
        // S is in registers: the next S may overwrite the buffer
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + (C::kSplitS ? ti : 0)));
        // P_i and O_i are free once the tile's previous PV has completed (in
        // this order it ran before the S just read, so the wait is short)
        if (npv > 0 &&
            !mbar_wait(bar(kBarPvDone + ti), (npv - 1) & 1, kErrWaitPvDone, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // mask in place: scores outside [c_lo, c_hi] become -inf
        const bool full = __all_sync(0xffffffffu, c_lo <= 0 && c_hi >= kBlk - 1);
        if (!full) {
#pragma unroll
          for (int c = 0; c < kBlk; ++c)
            if (c < c_lo || c > c_hi) sr[c] = __float_as_uint(-INFINITY);
        }
        // block max: 8 independent chains of 3-input max, then a tree
        float m8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = fmaxf(__uint_as_float(sr[e]), __uint_as_float(sr[e + 8]));
#pragma unroll
        for (int c = 16; c < kBlk; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e)
            m8[e] = max3f(m8[e], __uint_as_float(sr[c + e]), __uint_as_float(sr[c + 8 + e]));
        const float mraw = max3f(max3f(m8[0], m8[1], m8[2]), max3f(m8[3], m8[4], m8[5]),
                                 fmaxf(m8[6], m8[7]));
        const float m_cand = mraw * p.scale_log2;  // scale > 0 commutes with max
        if constexpr (kScores) {
          // block score of this warp's 4 positions x 8 heads (rows past T excluded)
          float bm = pos < p.T ? mraw : -INFINITY;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
          const int qg = (it.p0 + ti * kNpos + quad * 4) >> 2;
          if (lane == 0 && qg < p.nqg)
            p.blockmax[(((int64_t)it.b * p.Hkv + it.kvh) * p.nqg + qg) * p.nkb + kblk] =
                bm * (p.scale_log2 * 0.6931471805599453f);
        }
        const bool grow = m_cand > m_run + kRescaleLog2;  // false for -inf
        float f = 1.f;                                    // factor for O and l
        if (grow) {
          f = ex2_approx(m_run - m_cand);
          l *= f;
          m_run = m_cand;
        }
        const float mb = (m_run == -INFINITY) ? 0.f : m_run;
        // p = 2^(x - m) -> bf16 pairs in P_i, 16 columns at a time; the
        // scale-and-subtract and the running sum go two columns per
        // instruction (f32x2)
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nmb2 = make_float2(-mb, -mb);
        float2 l2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) l2[e] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kBlk / 16; ++c) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 xx = ffma2(make_float2(__uint_as_float(sr[16 * c + 2 * e]),
                                                __uint_as_float(sr[16 * c + 2 * e + 1])),
                                    sc2, nmb2);
            const float2 pp = make_float2(ex2_approx(xx.x), ex2_approx(xx.y));
            l2[e & 3] = fadd2(l2[e & 3], pp);
            pk[e] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st8(p_addr + c * 8, pk);
        }
        {
          const float2 a = fadd2(fadd2(l2[0], l2[1]), fadd2(l2[2], l2[3]));
          l += a.x + a.y;
        }
        // A moved max also rescales O, which holds the earlier blocks of the
        // item complete; the item's first block has no O yet.
        if (t > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int c = 0; c < kHd / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_addr + c * 32, o);
            tmem_ld_wait();
            reg_fence32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(o_addr + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + ti));
      }
      if (!ok) break;
      // ---- epilogue: out = O / l, lse ----
      if (!mbar_wait(bar(kBarOFull + ti), kn & 1, kErrWaitOFull, abort_flag)) break;
      ++kn;
      tc_fence_after();
      const float inv_l = 1.f / l;
      if constexpr (kBf16Out) {
        const long long e0 = (((long long)it.b * p.T + pos) * p.Hq + h) * kHd;
#pragma unroll
        for (int c = 0; c < kHd / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(o_addr + c * 32, o);
          tmem_ld_wait();
          reg_fence32(o);
          if (pos < p.T) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                  __uint_as_float(o[2 * e + 1]) * inv_l);
            float* orow = reinterpret_cast<float*>(static_cast<__nv_bfloat16*>(p.out) + e0 + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              st_global_v4(orow + 4 * e, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
      } else {
        // O read in the 16x256b shape: thread (rr, qd) = (lane / 4, lane % 4)
        // holds rows 16 hf + 8 kk + rr of this warp's lanes (tile row
        // 32 quad + 16 hf + 8 kk + rr: position row / kGt, head row % kGt),
        // columns 8 j + 2 qd + {0, 1}.  A quad then writes whole 32-byte
        // sectors, and one store covers 8 consecutive rows (8 D floats, the
        // heads of one or two positions); each row's 1 / l comes from the
        // thread that owns the row (lane 16 hf + 8 kk + rr).
        const int rr = lane >> 2, qd = lane & 3;
        const uint32_t o_warp = tmem + ((uint32_t)(quad * 32) << 16) + C::o(ti);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t o[kHd / 2];
          if constexpr (kHd == 128)
            tmem_ld_16x256b_x16(o_warp + ((uint32_t)(16 * hf) << 16), o);
          else
            tmem_ld_16x256b_x8(o_warp + ((uint32_t)(16 * hf) << 16), o);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kHd / 32; ++c) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(&o[c * 16]));
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const float il = __shfl_sync(0xffffffffu, inv_l, 16 * hf + 8 * kk + rr);
            const int row = 32 * quad + 16 * hf + 8 * kk + rr;   // tile row of these values
            const int pos_k = it.p0 + ti * kNpos + row / kGt;
            if (pos_k < p.T) {
              float* orow = static_cast<float*>(p.out) +
                            (((long long)it.b * p.T + pos_k) * p.Hq + it.grp * kGt + row % kGt) * kHd +
                            2 * qd;
#pragma unroll
              for (int j = 0; j < kHd / 8; ++j)
                st_global_v2(orow + 8 * j,
                             __float_as_uint(__uint_as_float(o[4 * j + 2 * kk]) * il),
                             __float_as_uint(__uint_as_float(o[4 * j + 2 * kk + 1]) * il));
            }
          }
        }
      }
      tc_fence_before();
      if (p.lse != nullptr && pos < p.T)
        p.lse[((long long)it.b * p.Hq + h) * p.T + pos] =
            (m_run + __log2f(l)) * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tcglobal
}  // namespace swa
