/*
 * swa_oracle.c -- CPU fp64 oracle for sliding-window attention with a
 * per-head attention-sink bias.  TEST INFRASTRUCTURE ONLY: it is called by the
 * tests, by the package's smoke check and by the benchmark's CPU-baseline leg,
 * never by the library path.  It shares no code with the CUDA kernels.
 *
 * What it computes (plain definition, written out):
 *
 *   Hybrid attention, "MiMo-V2-Flash Technical Report" summary page, section
 *   "前置知识" (prerequisites), items "混合注意力机制" and "注意力sink偏置":
 *   a sliding-window layer lets token i attend only to a local window of W
 *   tokens, a global layer to the whole (causal) sequence; every head adds a
 *   learnable bias s_h to its softmax denominator, which acts as a virtual
 *   "sink" token that takes weight but contributes no value.  The window is
 *   128 tokens ("wiki-for-amaranth" MiMo-V2 engineering notes, section
 *   "关键架构决策", item 1).  GQA is used in every attention layer ("MiMo-V2.5"
 *   ICML 2026 talk write-up, section 02).
 *
 *   For batch b, query head h, position i, with G = Hq/Hkv and kv = h / G:
 *     keys j in [max(0, i-W+1), i]                      (exactly W when i >= W-1)
 *     x_j  = (sum_d q[b,i,h,d] * k[b,j,kv,d]) / sqrt(D)
 *     m    = max(s_h, max_j x_j)                        (first pass)
 *     l    = exp(s_h - m) + sum_j exp(x_j - m)          (second pass)
 *     o    = sum_j exp(x_j - m) * v[b,j,kv,:] / l
 *     lse  = m + log(l)                                 (natural log, sink included)
 *   W >= T is the global (full causal) layer.
 *
 *   Decode ("pwwt.cn" MiMo-V2-Flash essay, section 1.1: the sliding-window KV
 *   cache has fixed size, O(W) memory; ICML talk write-up, Q&A K: position
 *   indices keep increasing while the window slides): one query at position
 *   pos against a W-slot ring whose slot s holds position
 *   p(s) = pos - ((pos - s) mod W); slots with p(s) < 0 are empty and skipped.
 *   Then the same formula as above over the valid slots.
 *
 *   Multi-token verify: L drafted tokens at positions pos..pos+L-1 are checked
 *   in one pass (the multi-token prediction drafts of the MiMo-V2-Flash
 *   technical report summary, section 核心方法); their keys and values come
 *   separately and the ring holds the tokens before pos.  Each new token takes
 *   the keys of its own window, as in the prefill (see oracle_swa_sink_verify).
 *
 * Inputs arrive in their storage type (dtype code 0 = fp32, 1 = bf16 bit
 * patterns, 2 = fp64) and are widened to fp64 exactly; all arithmetic is fp64
 * with libm exp/log.  Layouts: q [B,T,Hq,D], k/v [B,T,Hkv,D], out [B,T,Hq,D],
 * lse [B,Hq,T]; decode q [B,Hq,D], rings [B,Hkv,W,D], out [B,Hq,D], lse [B,Hq].
 * Rows are independent; OpenMP spreads them over host threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <omp.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

/* Widen element idx of a typed array to double (bf16 -> upper half of fp32). */
static double widen(const void* base, int dtype, int64_t idx) {
  if (dtype == ORC_F64) return ((const double*)base)[idx];
  if (dtype == ORC_F32) return (double)((const float*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* One attention row over an explicit list of key rows (indices into k/v).
 * qoff: element offset of the query vector; koff[n]: element offset of key /
 * value vector n.  Writes D outputs to o and returns the lse. */
static double attend_row(const void* q, int64_t qoff, const void* k, const void* v,
                         const int64_t* koff, int nkeys, double s_h, int D, int dtype,
                         double* x /* scratch, nkeys */, double* o) {
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  double m = s_h;
  for (int n = 0; n < nkeys; ++n) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += widen(q, dtype, qoff + d) * widen(k, dtype, koff[n] + d);
    x[n] = dot * inv_sqrt_d;
    if (x[n] > m) m = x[n];
  }
  double l = exp(s_h - m);
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (int n = 0; n < nkeys; ++n) {
    double e = exp(x[n] - m);
    l += e;
    for (int d = 0; d < D; ++d) o[d] += e * widen(v, dtype, koff[n] + d);
  }
  for (int d = 0; d < D; ++d) o[d] /= l;
  return m + log(l);
}

/* One prefill row (b, h, i). */
static void prefill_row(const void* q, const void* k, const void* v, const double* sink,
                        int64_t b, int64_t h, int64_t i, int64_t T, int Hq, int Hkv, int D,
                        int64_t W, int dtype, int64_t* koff, double* x, double* o,
                        double* lse_out) {
  const int64_t G = Hq / Hkv;
  const int64_t kv = h / G;
  int64_t j0 = i - W + 1;
  if (j0 < 0) j0 = 0;
  int n = 0;
  for (int64_t j = j0; j <= i; ++j) koff[n++] = ((b * T + j) * Hkv + kv) * D;
  const int64_t qoff = ((b * T + i) * Hq + h) * D;
  *lse_out = attend_row(q, qoff, k, v, koff, n, sink[h], D, dtype, x, o);
}

/* Full prefill: every (b, h, i).  out/lse are fp64. */
int oracle_swa_sink_fwd(const void* q, const void* k, const void* v, const double* sink,
                        double* out, double* lse, int64_t B, int64_t T, int Hq, int Hkv,
                        int D, int64_t W, int dtype, int nthreads) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || W <= 0) return -1;
  const int64_t maxk = W < T ? W : T;
  const int64_t nrows = B * Hq * T;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  {
    int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (maxk > 0 ? maxk : 1));
    double* x = (double*)malloc(sizeof(double) * (maxk > 0 ? maxk : 1));
    double* o = (double*)malloc(sizeof(double) * D);
    if (!koff || !x || !o) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 64)
      for (int64_t r = 0; r < nrows; ++r) {
        const int64_t b = r / (Hq * T), h = (r / T) % Hq, i = r % T;
        double l;
        prefill_row(q, k, v, sink, b, h, i, T, Hq, Hkv, D, W, dtype, koff, x, o, &l);
        memcpy(out + ((b * T + i) * Hq + h) * D, o, sizeof(double) * D);
        lse[(b * Hq + h) * T + i] = l;
      }
    }
    free(koff); free(x); free(o);
  }
  return bad ? -2 : 0;
}

/* Selected prefill rows: sel holds nsel (b, h, i) triples; out_rows is
 * [nsel, D], lse_rows [nsel].  Used for sampled checks at full size. */
int oracle_swa_sink_fwd_rows(const void* q, const void* k, const void* v, const double* sink,
                             const int64_t* sel, int64_t nsel, double* out_rows,
                             double* lse_rows, int64_t B, int64_t T, int Hq, int Hkv, int D,
                             int64_t W, int dtype, int nthreads) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || W <= 0) return -1;
  for (int64_t s = 0; s < nsel; ++s) {
    const int64_t b = sel[3 * s], h = sel[3 * s + 1], i = sel[3 * s + 2];
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= T) return -1;
  }
  const int64_t maxk = W < T ? W : T;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  {
    int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (maxk > 0 ? maxk : 1));
    double* x = (double*)malloc(sizeof(double) * (maxk > 0 ? maxk : 1));
    if (!koff || !x) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t s = 0; s < nsel; ++s) {
        prefill_row(q, k, v, sink, sel[3 * s], sel[3 * s + 1], sel[3 * s + 2], T, Hq, Hkv, D,
                    W, dtype, koff, x, out_rows + s * D, &lse_rows[s]);
      }
    }
    free(koff); free(x);
  }
  return bad ? -2 : 0;
}

/* Decode: one query per sequence against a W-slot ring (slot = position mod W). */
int oracle_swa_sink_decode(const void* q, const void* k_ring, const void* v_ring,
                           const int64_t* pos, const double* sink, double* out, double* lse,
                           int64_t B, int Hq, int Hkv, int D, int64_t W, int dtype,
                           int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || W <= 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    if (pos[b] < 0) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t nrows = B * Hq;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  {
    int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * W);
    double* x = (double*)malloc(sizeof(double) * W);
    if (!koff || !x) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t r = 0; r < nrows; ++r) {
        const int64_t b = r / Hq, h = r % Hq, kv = h / G;
        int n = 0;
        for (int64_t s = 0; s < W; ++s) {
          const int64_t p = pos[b] - (((pos[b] - s) % W + W) % W); /* mod in [0, W) */
          if (p < 0) continue;
          koff[n++] = ((b * Hkv + kv) * W + s) * D;
        }
        lse[b * Hq + h] = attend_row(q, (b * Hq + h) * D, k_ring, v_ring, koff, n, sink[h], D,
                                     dtype, x, out + (b * Hq + h) * D);
      }
    }
    free(koff); free(x);
  }
  return bad ? -2 : 0;
}

/* Multi-token verify (speculative decoding with multi-token prediction: the
 * drafted tokens are checked in one pass).  L new tokens sit at positions
 * pos, ..., pos+L-1; their keys and values arrive in k_new / v_new, and the
 * W-slot ring holds the tokens before them: slot s holds position
 * p(s) = (pos-1) - ((pos-1-s) mod W), empty when p(s) < 0.  New token j
 * attends to the positions [pos+j-W+1, pos+j] of the same definition as the
 * prefill: the ring slots whose positions fall there, then new tokens 0..j.
 * Layouts: q [B,L,Hq,D], k_new/v_new [B,L,Hkv,D], rings [B,Hkv,W,D],
 * out [B,L,Hq,D], lse [B,Hq,L]. */
int oracle_swa_sink_verify(const void* q, const void* k_new, const void* v_new,
                           const void* k_ring, const void* v_ring, const int64_t* pos,
                           const double* sink, double* out, double* lse, int64_t B, int64_t L,
                           int Hq, int Hkv, int D, int64_t W, int dtype, int nthreads) {
  if (B < 0 || L <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || W <= 0) return -1;
  for (int64_t b = 0; b < B; ++b)
    if (pos[b] < 0) return -1;
  const int64_t G = Hq / Hkv;
  const int64_t nrows = B * L * Hq;
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  {
    /* key n: source (0 = ring, 1 = new) and element offset of its vector */
    int* src = (int*)malloc(sizeof(int) * (W + L));
    int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (W + L));
    double* x = (double*)malloc(sizeof(double) * (W + L));
    if (!src || !koff || !x) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t r = 0; r < nrows; ++r) {
        const int64_t b = r / (L * Hq), j = (r / Hq) % L, h = r % Hq, kv = h / G;
        const int64_t p_now = pos[b] + j;          /* position of this query */
        const int64_t lo = p_now - W + 1;          /* first position in its window */
        int n = 0;
        for (int64_t s = 0; s < W; ++s) {
          const int64_t p = (pos[b] - 1) - (((pos[b] - 1 - s) % W + W) % W);
          if (p < 0 || p < lo) continue;
          src[n] = 0;
          koff[n++] = ((b * Hkv + kv) * W + s) * D;
        }
        for (int64_t i = 0; i <= j; ++i) {
          if (pos[b] + i < lo) continue;           /* only when W <= j */
          src[n] = 1;
          koff[n++] = ((b * L + i) * Hkv + kv) * D;
        }
        const int64_t qoff = ((b * L + j) * Hq + h) * D;
        double m = sink[h];
        for (int k = 0; k < n; ++k) {
          const void* kb = src[k] ? k_new : k_ring;
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += widen(q, dtype, qoff + d) * widen(kb, dtype, koff[k] + d);
          x[k] = dot * inv_sqrt_d;
          if (x[k] > m) m = x[k];
        }
        double l = exp(sink[h] - m);
        double* o = out + qoff;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int k = 0; k < n; ++k) {
          const void* vb = src[k] ? v_new : v_ring;
          const double e = exp(x[k] - m);
          l += e;
          for (int d = 0; d < D; ++d) o[d] += e * widen(vb, dtype, koff[k] + d);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
        lse[(b * Hq + h) * L + j] = m + log(l);
      }
    }
    free(src); free(koff); free(x);
  }
  return bad ? -2 : 0;
}

/* Rotary position embedding, applied to q and k before attention (ICML 2026
 * talk write-up, Q&A K: RoPE's theta is fixed at inference and the position
 * index keeps counting up while the window slides, so each token is rotated
 * at its absolute position).  The pages give no variant; this is the
 * rotate-half form over the first rot_dim dimensions: for i < rot_dim / 2,
 *   a_i = p * theta^(-2 i / rot_dim)
 *   y[i]             = x[i] cos a_i - x[i + rot_dim/2] sin a_i
 *   y[i + rot_dim/2] = x[i + rot_dim/2] cos a_i + x[i] sin a_i
 * and y[d] = x[d] for d >= rot_dim.  x is [B, T, H, D] in its storage type,
 * token (b, t) at position pos0[b] + t; y is written in fp64. */
int oracle_rope(const void* x, const int64_t* pos0, double* y, int64_t B, int64_t T, int H,
                int D, int rot_dim, double theta, int dtype) {
  if (B < 0 || T < 0 || H <= 0 || D <= 0 || rot_dim < 0 || rot_dim > D || rot_dim % 2 ||
      !(theta > 0.0))
    return -1;
  const int half = rot_dim / 2;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < T; ++t) {
      const double p = (double)(pos0[b] + t);
      for (int h = 0; h < H; ++h) {
        const int64_t base = ((b * T + t) * H + h) * D;
        for (int i = 0; i < half; ++i) {
          const double a = p * pow(theta, -2.0 * i / rot_dim);
          const double x0 = widen(x, dtype, base + i), x1 = widen(x, dtype, base + i + half);
          y[base + i] = x0 * cos(a) - x1 * sin(a);
          y[base + i + half] = x1 * cos(a) + x0 * sin(a);
        }
        for (int d = rot_dim; d < D; ++d) y[base + d] = widen(x, dtype, base + d);
      }
    }
  return 0;
}

/* ---- High Sparse: block scores from a global layer, block selection, and
 * attention over the selected blocks ("MiMo-V2.5" ICML 2026 talk write-up,
 * section 02: the full-attention layers' FlashAttention block-level scores are
 * reused, at no extra cost, to choose the tokens the sparse layers attend to;
 * sparse layers share the full layer's KV cache; selection is by block with a
 * configurable capacity).  The page gives no formula; the readings are:
 *   block score  max over the scaled logits x_ij = q_i.k_j / sqrt(D) of the
 *                valid (window / causal) pairs with query position i in a
 *                group of 4 consecutive positions, query head h in kv group g,
 *                key j in a block of 128; -inf when the block has none
 *   selection    per query block of QB positions: the key block holding the
 *                block's last position (the causal diagonal), then the
 *                topk - 1 highest-scoring earlier blocks (score of a block =
 *                max over the query block's groups; ties: smaller index
 *                first); listed in increasing order, padded with -1
 *   sparse layer causal attention of query i over the keys j <= i of the
 *                blocks selected for its query block, sink in the denominator */

/* blockmax [B, Hkv, ceil(T/4), ceil(T/128)] (fp64) */
int oracle_block_max(const void* q, const void* k, double* blockmax, int64_t B, int64_t T,
                     int Hq, int Hkv, int D, int64_t W, int dtype, int nthreads) {
  if (B < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || W <= 0) return -1;
  const int64_t G = Hq / Hkv, nqg = (T + 3) / 4, nkb = (T + 127) / 128;
  const double inv_sqrt_d = 1.0 / sqrt((double)D);
  const int64_t n = B * Hkv * nqg;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  for (int64_t r = 0; r < n; ++r) {
    const int64_t b = r / (Hkv * nqg), g = (r / nqg) % Hkv, qg = r % nqg;
    double* row = blockmax + r * nkb;
    for (int64_t kb = 0; kb < nkb; ++kb) row[kb] = -INFINITY;
    for (int64_t i = 4 * qg; i < 4 * qg + 4 && i < T; ++i) {
      int64_t j0 = i - W + 1;
      if (j0 < 0) j0 = 0;
      for (int64_t hh = 0; hh < G; ++hh) {
        const int64_t h = g * G + hh;
        const int64_t qoff = ((b * T + i) * Hq + h) * D;
        for (int64_t j = j0; j <= i; ++j) {
          const int64_t koff = ((b * T + j) * Hkv + g) * D;
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += widen(q, dtype, qoff + d) * widen(k, dtype, koff + d);
          const double x = dot * inv_sqrt_d;
          if (x > row[j / 128]) row[j / 128] = x;
        }
      }
    }
  }
  return 0;
}

/* scores [B, Hkv, nqg, nkb] fp32 (block maxima as produced above, in any
 * precision the caller chose); idx [B, Hkv, nqb, topk] int32 with
 * nqb = ceil(T / QB).  QB must be a multiple of 4 and divide 128. */
int oracle_topk_blocks(const float* scores, int32_t* idx, int64_t B, int64_t T, int Hkv, int QB,
                       int topk) {
  if (B < 0 || T <= 0 || Hkv <= 0 || QB <= 0 || QB % 4 || 128 % QB || topk <= 0) return -1;
  const int64_t nqg = (T + 3) / 4, nkb = (T + 127) / 128, nqb = (T + QB - 1) / QB;
  double* agg = (double*)malloc(sizeof(double) * (nkb > 0 ? nkb : 1));
  unsigned char* taken = (unsigned char*)malloc(nkb > 0 ? nkb : 1);
  if (!agg || !taken) { free(agg); free(taken); return -2; }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t g = 0; g < Hkv; ++g)
      for (int64_t qb = 0; qb < nqb; ++qb) {
        int32_t* out = idx + ((b * Hkv + g) * nqb + qb) * topk;
        int64_t last = qb * QB + QB - 1;
        if (last > T - 1) last = T - 1;
        const int64_t diag = last / 128;          /* the causal diagonal block */
        for (int64_t kb = 0; kb < nkb; ++kb) {
          agg[kb] = -INFINITY;
          taken[kb] = 0;
        }
        for (int64_t qg = qb * QB / 4; qg < (qb + 1) * QB / 4 && qg < nqg; ++qg)
          for (int64_t kb = 0; kb <= diag; ++kb) {
            const double v = scores[((b * Hkv + g) * nqg + qg) * nkb + kb];
            if (v > agg[kb]) agg[kb] = v;
          }
        taken[diag] = 1;
        /* topk - 1 rounds of "highest score, smallest index" among earlier blocks */
        for (int t = 1; t < topk; ++t) {
          int64_t best = -1;
          for (int64_t kb = 0; kb < diag; ++kb) {
            if (taken[kb]) continue;
            if (best < 0 || agg[kb] > agg[best]) best = kb;
          }
          if (best < 0) break;
          taken[best] = 1;
        }
        int n = 0;
        for (int64_t kb = 0; kb <= diag; ++kb)
          if (taken[kb]) out[n++] = (int32_t)kb;
        while (n < topk) out[n++] = -1;
      }
  free(agg);
  free(taken);
  return 0;
}

/* Attention of the sparse layer over the selected blocks (see above).
 * idx [B, Hkv, nqb, topk] int32 (-1 = unused); out [B,T,Hq,D], lse [B,Hq,T]. */
int oracle_sparse_fwd(const void* q, const void* k, const void* v, const double* sink,
                      const int32_t* idx, double* out, double* lse, int64_t B, int64_t T, int Hq,
                      int Hkv, int D, int QB, int topk, int dtype, int nthreads) {
  if (B < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || QB <= 0 || topk <= 0)
    return -1;
  const int64_t G = Hq / Hkv, nqb = (T + QB - 1) / QB;
  const int64_t nrows = B * Hq * T;
  int bad = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
  {
    int64_t* koff = (int64_t*)malloc(sizeof(int64_t) * (int64_t)topk * 128);
    double* x = (double*)malloc(sizeof(double) * (int64_t)topk * 128);
    double* o = (double*)malloc(sizeof(double) * D);
    if (!koff || !x || !o) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 64)
      for (int64_t r = 0; r < nrows; ++r) {
        const int64_t b = r / (Hq * T), h = (r / T) % Hq, i = r % T, g = h / G;
        const int32_t* sel = idx + ((b * Hkv + g) * nqb + i / QB) * topk;
        int n = 0;
        for (int t = 0; t < topk; ++t) {
          if (sel[t] < 0) continue;
          for (int64_t j = (int64_t)sel[t] * 128; j < (int64_t)sel[t] * 128 + 128 && j <= i; ++j)
            koff[n++] = ((b * T + j) * Hkv + g) * D;
        }
        const double l = attend_row(q, ((b * T + i) * Hq + h) * D, k, v, koff, n, sink[h], D,
                                    dtype, x, o);
        memcpy(out + ((b * T + i) * Hq + h) * D, o, sizeof(double) * D);
        lse[(b * Hq + h) * T + i] = l;
      }
    }
    free(koff); free(x); free(o);
  }
  return bad ? -2 : 0;
}

int oracle_num_threads(void) { return omp_get_max_threads(); }
