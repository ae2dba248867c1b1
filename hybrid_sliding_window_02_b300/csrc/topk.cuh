// topk.cuh -- block selection for the sparse layers of High Sparse ("MiMo-V2.5"
// ICML 2026 talk write-up, section 02: the full-attention layers' block-level
// scores choose the tokens the sparse layers attend to; block-level selection
// with a configurable capacity).
//
// Input: block scores [B, Hkv, ceil(T/4), ceil(T/128)] (the max scaled logit of
// each 4-position query group and 128-key block, as the global-attention
// kernel emits them).  For each query block of QB positions (QB a multiple of
// 4 dividing 128) and kv head, the key block holding the query block's last
// position (the causal diagonal) is always kept, then the topk - 1 earlier
// blocks with the highest score (the max over the query block's groups; ties
// go to the smaller index).  Output: idx [B, Hkv, ceil(T/QB), topk] int32,
// increasing, padded with -1.
//
// One warp per (b, kv head, query block): the aggregated scores of the
// candidate blocks go to shared memory, topk - 1 rounds of a warp-wide
// (score, -index) maximum pick the blocks, and a ballot compacts them in order.
#pragma once

#include "device_common.cuh"

namespace swa {

constexpr int kTopkWarps = 4;
constexpr int kTopkMaxBlocks = 4096;   // T <= 524288
constexpr int kTopkMax = 64;

__global__ void __launch_bounds__(kTopkWarps * 32) topk_blocks_kernel(
    const float* __restrict__ scores, int* __restrict__ idx, int B, int T, int Hkv, int QB,
    int topk) {
  extern __shared__ __align__(16) uint8_t topk_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqg = (T + 3) / 4, nkb = (T + 127) / 128, nqb = (T + QB - 1) / QB;
  float* agg = reinterpret_cast<float*>(topk_smem) + warp * nkb;
  uint32_t* taken = reinterpret_cast<uint32_t*>(topk_smem + kTopkWarps * nkb * 4) +
                    warp * ((nkb + 31) / 32);
  const int64_t unit = (int64_t)blockIdx.x * kTopkWarps + warp;
  if (unit >= (int64_t)B * Hkv * nqb) return;
  const int qb = (int)(unit % nqb);
  const int64_t bg = unit / nqb;               // b * Hkv + g
  const int last = min(qb * QB + QB, T) - 1;
  const int diag = last / 128;
  const int qg0 = qb * QB / 4, qg1 = min((qb + 1) * QB / 4, nqg);
  const float* sc = scores + bg * nqg * (int64_t)nkb;
  for (int kb = lane; kb < diag; kb += 32) {
    float m = -INFINITY;
    for (int qg = qg0; qg < qg1; ++qg) m = fmaxf(m, __ldg(sc + (int64_t)qg * nkb + kb));
    agg[kb] = m;
  }
  for (int w = lane; w < (nkb + 31) / 32; w += 32) taken[w] = 0u;
  __syncwarp();
  if (lane == 0) taken[diag >> 5] |= 1u << (diag & 31);
  __syncwarp();
  // topk - 1 rounds: the untaken earlier block with the highest score, the
  // smallest index among equal scores
  for (int t = 1; t < topk; ++t) {
    float best = -INFINITY;
    int bi = -1;
    for (int kb = lane; kb < diag; kb += 32) {
      if ((taken[kb >> 5] >> (kb & 31)) & 1u) continue;
      const float v = agg[kb];
      if (bi < 0 || v > best) {  // ascending scan: equal scores keep the smaller index
        best = v;
        bi = kb;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      const bool better = oi >= 0 && (bi < 0 || ob > best || (ob == best && oi < bi));
      if (better) {
        best = ob;
        bi = oi;
      }
    }
    if (bi < 0) break;                          // every earlier block is taken
    if (lane == 0) taken[bi >> 5] |= 1u << (bi & 31);
    __syncwarp();
  }
  // write the taken blocks in increasing order, then -1
  int* out = idx + unit * topk;
  int n = 0;
  for (int base = 0; base <= diag; base += 32) {
    const int kb = base + lane;
    const bool sel = kb <= diag && ((taken[kb >> 5] >> (kb & 31)) & 1u);
    const uint32_t mask = __ballot_sync(0xffffffffu, sel);
    if (sel) out[n + __popc(mask & ((1u << lane) - 1u))] = kb;
    n += __popc(mask);
  }
  for (int i = n + lane; i < topk; i += 32) out[i] = -1;
}

}  // namespace swa
