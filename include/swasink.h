/*
 * swasink.h -- C ABI of libswasink.so: sliding-window attention with a
 * per-head attention-sink bias, for one B300 GPU (sm_103a).
 *
 * The operation ("MiMo-V2-Flash Technical Report" summary page, section
 * 前置知识, items 混合注意力机制 and 注意力sink偏置; window of 128 tokens and
 * 5:1 window:global layers in section 核心方法; GQA in every attention layer:
 * "MiMo-V2.5" ICML 2026 talk write-up, section 02):
 *
 *   for batch b, query head h, position i, kv head g = h / (Hq / Hkv):
 *     x_j  = q[b,i,h,:] . k[b,j,g,:] / sqrt(D)     for j in [max(0, i-W+1), i]
 *     m    = max(sink[h], max_j x_j)
 *     l    = exp(sink[h] - m) + sum_j exp(x_j - m)
 *     out[b,i,h,:] = sum_j exp(x_j - m) v[b,j,g,:] / l
 *     lse[b,h,i]   = m + ln(l)
 *
 * The sink adds to the softmax denominator only (a virtual token with value
 * 0).  W >= T gives the global (full causal) layer of the hybrid stack.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *     and contiguous in the layouts stated per call, 16-byte aligned (the
 *     host-memory prefill, swa_sink_fwd_host, also takes HOST pointers).  The
 *     library allocates no memory and keeps no state between calls beyond
 *     per-device settings and, for swa_sink_fwd_host, two streams and a set of
 *     events per device.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Results are valid once the stream reaches them.
 *     The tensor-core decode and verify kernels are launched as programmatic
 *     dependents: they may start their set-up, and an L2 prefetch of their
 *     first K/V ring, while the kernel before them on the stream finishes,
 *     but they read and write no buffer before that kernel has completed, so
 *     stream order holds as for any launch.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error and touches no memory.  A failed launch
 *     returns SWA_ECUDA (text in swa_last_error()).  Nothing traps on the
 *     device: a device-side wait that runs past its time limit records a code
 *     readable with swa_device_error() and the kernel returns early.
 *   - The current CUDA device (cudaSetDevice) must be the one that holds the
 *     device buffers and owns `stream`: the library launches on the current
 *     device and sets its kernels' attributes there.
 *   - Sizes are int; element offsets are computed in 64 bits.
 */
#ifndef SWASINK_H
#define SWASINK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SWA_OK = 0,
  SWA_EINVAL = -1,       /* bad argument: null pointer, size <= 0, Hq % Hkv, alignment */
  SWA_EUNSUPPORTED = -2, /* valid but not implemented: D not in {64,128}, window too large for decode */
  SWA_ECUDA = -3         /* a CUDA launch or API call failed */
} swa_status;

typedef enum { SWA_F32 = 0, SWA_BF16 = 1 } swa_dtype;

/*
 * swa_sink_fwd -- prefill (every position of every sequence).
 *   q    [B, T, Hq,  D]  in_dtype     (queries, RoPE already applied)
 *   k    [B, T, Hkv, D]  in_dtype
 *   v    [B, T, Hkv, D]  in_dtype
 *   sink [Hq]            float32      (per query head, on the scaled-logit scale;
 *                                      finite, or -inf for no sink)
 *   out  [B, T, Hq,  D]  float32      (written)
 *   lse  [B, Hq, T]      float32      (written; may be NULL to skip)
 *   W >= 1 window length; W >= T means global causal attention.
 *   Requirements: B,T,Hq,Hkv,D,W >= 1; Hq % Hkv == 0; D in {64, 128};
 *   q, k, v, out, lse 16-byte aligned.  out must not overlap the inputs.
 * Returns SWA_OK, SWA_EINVAL, SWA_EUNSUPPORTED or SWA_ECUDA.
 */
swa_status swa_sink_fwd(const void* q, const void* k, const void* v, const float* sink,
                        float* out, float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                        swa_dtype in_dtype, void* stream);

/*
 * swa_sink_fwd_ex -- swa_sink_fwd with a choice of output type: out_dtype
 * SWA_F32 is swa_sink_fwd; SWA_BF16 writes out [B, T, Hq, D] as bf16, each
 * value the round-to-nearest-even of the fp32 value swa_sink_fwd would write
 * (lse stays fp32).  The bf16 output is available where swa_sink_fwd_path
 * names a tensor-core kernel ("tc_swa", "tc_global"); elsewhere the call
 * returns SWA_EUNSUPPORTED.  It halves the output bytes, which dominate the
 * sliding-window layer's memory traffic.
 */
swa_status swa_sink_fwd_ex(const void* q, const void* k, const void* v, const float* sink,
                           void* out, float* lse, int B, int T, int Hq, int Hkv, int D, int W,
                           swa_dtype in_dtype, swa_dtype out_dtype, void* stream);

/*
 * swa_sink_fwd_host -- swa_sink_fwd_ex with q, k, v taken from HOST memory and
 * out, lse written to HOST memory, in chunks: the chunk's inputs are copied to
 * the device, its prefill runs, and its outputs are copied back, while the
 * copies of the neighbouring chunks run at the same time (host-to-device on
 * one stream, the prefill on `stream`, device-to-host on another; each
 * chunk's steps are chained by events).  On the sliding-window tensor-core
 * path (swa_sink_fwd_path "tc_swa") a chunk is one sequence x a range of
 * positions (about 16 chunks in all, at least 512 positions each, and a piece
 * of 512 positions split off the first and the last, whose copies overlap
 * nothing), staged at its own place in the device buffers, so that every copy
 * is one contiguous range; the prefill of a chunk computes its positions
 * only, reading the window's earlier keys copied with the chunks before it.  On the other paths a chunk is one sequence x a share of the kv
 * heads (half of them when Hkv is even; the whole batch as one chunk when a
 * share would break the 16-byte alignment of the staging).  The results are
 * those of swa_sink_fwd_ex on the whole batch, bit for bit.
 *   q_h, k_h, v_h       host, layouts as swa_sink_fwd; pinned (page-locked)
 *                       memory lets the copies overlap, pageable memory works
 *                       but the copies then serialise with the host
 *   sink                DEVICE [Hq] float32 (a layer parameter, resident)
 *   out_h, lse_h        host outputs (lse_h may be NULL, then lse_d too)
 *   q_d, k_d, v_d, out_d, lse_d
 *                       device buffers of the full sizes of q, k, v, out and
 *                       lse, owned by the caller (the library allocates no
 *                       memory); they hold the data in transit, in a layout
 *                       of the library's choosing
 * The call is asynchronous with respect to the host, like the others: it is
 * ordered after earlier work on `stream`, later work on `stream` sees the
 * copies to the host completed, and out_h / lse_h may be read once `stream`
 * has been synchronised.  The library keeps two CUDA streams and a set of
 * events per device for these calls (created on first use); calls from
 * several host threads are serialised while they enqueue.  Argument rules and
 * return values are those of swa_sink_fwd_ex; on SWA_ECUDA part of the work
 * may have been enqueued, and later work on `stream` still follows it.
 */
swa_status swa_sink_fwd_host(const void* q_h, const void* k_h, const void* v_h,
                             const float* sink, void* out_h, float* lse_h, void* q_d,
                             void* k_d, void* v_d, void* out_d, float* lse_d, int B, int T,
                             int Hq, int Hkv, int D, int W, swa_dtype in_dtype,
                             swa_dtype out_dtype, void* stream);

/* Size in bytes of the staging array swa_sink_fwd_host_static uses (64 MiB). */
#define SWA_HOST_STATIC_BYTES (64u * 1024u * 1024u)

/*
 * swa_sink_fwd_host_static -- swa_sink_fwd_host without device buffers from
 * the caller: the data in transit is staged in one array of
 * SWA_HOST_STATIC_BYTES that the library reserves on each GPU that loads it,
 * held until the process exits.  The pages have no counterpart to this call;
 * it serves callers that cannot call cudaMalloc: code whose device memory is
 * owned by another allocator (a framework's caching allocator, a budget fixed
 * at start-up) and loops that must not call cudaMalloc or cudaFree, which can
 * synchronise the whole device.  The call allocates no device memory itself.
 *   q_h, k_h, v_h, sink, out_h, lse_h, sizes, dtypes and stream: as
 *   swa_sink_fwd_host (lse_h may be NULL).
 *   The staging needs q, k, v, out and (if lse_h is given) lse in full, each
 *   rounded up to 256 bytes: with bf16 inputs, fp32 output and lse, D = 128,
 *   Hq = 64 and Hkv = 8 that is 53,504 bytes per position, about 1250
 *   positions in all.  Larger sizes return SWA_EUNSUPPORTED, with the bytes
 *   needed in swa_last_error(), before anything is enqueued.
 *   The first call on a device looks up the array's device address (with
 *   that device current) and keeps it; make that first call before any
 *   stream capture.  The library keeps the streams and events of
 *   swa_sink_fwd_host as well.
 *   Every call on a device shares the one array, which keeps the last call's
 *   contents; each call writes every staged byte before reading it, so
 *   nothing needs clearing between calls.  Calls whose GPU work overlaps
 *   (on different streams, or from several host threads) race on the array
 *   and corrupt each other's results: order them on one stream, or
 *   synchronise between them.
 * Returns SWA_OK, SWA_EINVAL, SWA_EUNSUPPORTED or SWA_ECUDA as
 * swa_sink_fwd_host does.
 */
swa_status swa_sink_fwd_host_static(const void* q_h, const void* k_h, const void* v_h,
                                    const float* sink, void* out_h, float* lse_h, int B, int T,
                                    int Hq, int Hkv, int D, int W, swa_dtype in_dtype,
                                    swa_dtype out_dtype, void* stream);

/*
 * swa_sink_decode -- one query token per sequence against a W-slot ring cache
 * ("pwwt.cn" MiMo-V2-Flash essay, section 1.1: the sliding-window KV cache has
 * a fixed size, O(W) memory; ICML 2026 talk write-up, Q&A K: positions keep
 * increasing while the window slides).
 *   q      [B, Hq, D]       in_dtype   (the token at position pos[b])
 *   k_ring [B, Hkv, W, D]   in_dtype   slot s holds position pos - ((pos - s) mod W)
 *   v_ring [B, Hkv, W, D]   in_dtype
 *   pos    [B]              int64      >= 0; the token at pos must already be in the ring
 *   sink   [Hq]             float32
 *   out    [B, Hq, D]       float32    (written)
 *   lse    [B, Hq]          float32    (written; may be NULL)
 *   Slots whose position would be negative (pos < W-1) are ignored, whatever
 *   they hold.  Requires 2*W*D*sizeof(in_dtype) <= 163840 (W <= 320 at bf16,
 *   D = 128), else SWA_EUNSUPPORTED.  pos values are read on the device; a
 *   negative pos leaves every slot empty: out = 0 and lse = sink[h].
 *   sink values must be finite or -inf (-inf = no sink).
 */
swa_status swa_sink_decode(const void* q, const void* k_ring, const void* v_ring,
                           const int64_t* pos, const float* sink, float* out, float* lse,
                           int B, int Hq, int Hkv, int D, int W, swa_dtype in_dtype,
                           void* stream);

/*
 * swa_ring_append -- write one new token per sequence into its ring slot
 * (slot = pos[b] mod W), the cache update that precedes swa_sink_decode: the
 * sliding-window KV cache of fixed size, O(W) memory whatever the sequence
 * length ("pwwt.cn" MiMo-V2-Flash essay, section 1.1).
 *   k_new, v_new [B, Hkv, D] dtype;  k_ring, v_ring [B, Hkv, W, D] dtype (updated)
 *   pos [B] int64 >= 0 (device); a negative pos leaves that sequence's ring unchanged.
 */
swa_status swa_ring_append(const void* k_new, const void* v_new, void* k_ring, void* v_ring,
                           const int64_t* pos, int B, int Hkv, int D, int W, swa_dtype dtype,
                           void* stream);

/*
 * swa_sink_verify -- multi-token verify: the attention of L drafted tokens at
 * positions pos .. pos+L-1 in one pass, for speculative decoding with
 * multi-token prediction ("MiMo-V2-Flash Technical Report" summary, section
 * 核心方法: MTP drafts checked by the main model).  The drafts' keys and values
 * come with the call; the ring holds the tokens BEFORE them and is not
 * changed (append the accepted prefix afterwards with swa_ring_append).
 *   q      [B, L, Hq, D]    in_dtype   (the drafted tokens, RoPE applied)
 *   k_new  [B, L, Hkv, D]   in_dtype
 *   v_new  [B, L, Hkv, D]   in_dtype
 *   k_ring [B, Hkv, W, D]   in_dtype   slot s holds position (pos-1) - ((pos-1-s) mod W)
 *   v_ring [B, Hkv, W, D]   in_dtype
 *   pos    [B]              int64      position of drafted token 0 (device)
 *   sink   [Hq]             float32
 *   out    [B, L, Hq, D]    float32    (written)
 *   lse    [B, Hq, L]       float32    (written; may be NULL)
 *   Token j attends to positions [pos+j-W+1, pos+j]: the ring slots whose
 *   positions fall there (slots of negative positions are empty and ignored,
 *   whatever they hold) and drafted tokens 0..j; the result equals the
 *   prefill rows pos .. pos+L-1 of the whole sequence.  A negative pos leaves
 *   nothing to attend to: out = 0, lse = sink[h].  Requires 1 <= L <= 64, the
 *   shape rules of swa_sink_decode, and k_new / v_new 16-byte aligned.
 */
swa_status swa_sink_verify(const void* q, const void* k_new, const void* v_new,
                           const void* k_ring, const void* v_ring, const int64_t* pos,
                           const float* sink, float* out, float* lse, int B, int L, int Hq,
                           int Hkv, int D, int W, swa_dtype in_dtype, void* stream);

/*
 * swa_rope -- rotary position embedding in place, at absolute positions (ICML
 * 2026 talk write-up, Q&A K: RoPE's theta is fixed at inference and position
 * indices keep counting up while the window slides).  The pages give no
 * variant; this is the rotate-half form over the first rot_dim dimensions:
 * for i < rot_dim/2, a_i = p * theta^(-2 i / rot_dim) and the pair
 * (x[i], x[i + rot_dim/2]) is rotated by a_i; dimensions >= rot_dim pass.
 *   x    [B, T, H, D]  dtype   (updated; q or k of a prefill)
 *   pos0 [B]           int64   token (b, t) is at position pos0[b] + t (device)
 *   Requires D in {64, 128}, rot_dim even with 2 <= rot_dim <= D, theta > 0.
 *   Angles are formed in fp64 and reduced modulo 2 pi before the fp32 rotation.
 */
swa_status swa_rope(void* x, const int64_t* pos0, int B, int T, int H, int D, int rot_dim,
                    double theta, swa_dtype dtype, void* stream);

/*
 * swa_rope_append -- the step before a decode, fused: rotate the new token's
 * query and key at position pos[b] (as swa_rope) and write key and value into
 * ring slot pos[b] mod W (the fixed O(W) cache of the "pwwt.cn" essay,
 * section 1.1).
 *   q_in  [B, Hq, D]  dtype      q_out [B, Hq, D] dtype (written; may equal q_in)
 *   k_in, v_in [B, Hkv, D] dtype (k before rotation)
 *   k_ring, v_ring [B, Hkv, W, D] dtype (one slot per sequence updated)
 *   pos   [B] int64 (device); a negative pos leaves q_out[b] and the rings untouched.
 *   Requires what swa_rope requires, 16-byte aligned buffers and Hq + 2 Hkv <=
 *   2^20 (SWA_EUNSUPPORTED beyond); q_out overlaps no input other than q_in.
 */
swa_status swa_rope_append(const void* q_in, const void* k_in, const void* v_in, void* q_out,
                           void* k_ring, void* v_ring, const int64_t* pos, int B, int Hq,
                           int Hkv, int D, int W, int rot_dim, double theta, swa_dtype dtype,
                           void* stream);

/*
 * High Sparse ("MiMo-V2.5" ICML 2026 talk write-up, section 02): the
 * full-attention layers' block-level scores are reused to choose the tokens
 * the sparse layers attend to, the sparse layers share the full layer's KV
 * cache, and selection is by block with a configurable capacity.  The page
 * gives no formula; the three calls below follow the readings stated with
 * each.
 *
 * swa_sink_fwd_scores -- swa_sink_fwd_ex on the tensor-core global kernel
 * (bf16 inputs, D = 64 or 128, Hq = 8 Hkv, any W; W >= T is the
 * full-attention layer) that also writes the block scores:
 *   blockmax [B, Hkv, ceil(T/4), ceil(T/128)] float32:
 *     blockmax[b,g,c,n] = max of q_i.k_j / sqrt(D) over query positions
 *     i in [4c, 4c+4), the 8 query heads of kv head g, keys j in
 *     [128n, 128n+128) with j in row i's window.
 *   Entries of blocks with no such pair are not written: initialise the
 *   buffer to -inf.  Other shapes return SWA_EUNSUPPORTED.
 */
swa_status swa_sink_fwd_scores(const void* q, const void* k, const void* v, const float* sink,
                               void* out, float* lse, float* blockmax, int B, int T, int Hq,
                               int Hkv, int D, int W, swa_dtype in_dtype, swa_dtype out_dtype,
                               void* stream);

/*
 * swa_topk_blocks -- block selection from those scores.  For each kv head and
 * query block of QB positions (QB a multiple of 4 dividing 128): the key block
 * holding the query block's last position (the causal diagonal), then the
 * topk - 1 earlier key blocks with the highest score (a block's score is the
 * max over the query block's 4-position groups; ties go to the smaller index).
 *   scores [B, Hkv, ceil(T/4), ceil(T/128)] float32
 *   idx    [B, Hkv, ceil(T/QB), topk] int32 (written): increasing, -1 padded
 *   Requires 1 <= topk <= 64 and ceil(T/128) <= 4096.
 */
swa_status swa_topk_blocks(const float* scores, int* idx, int B, int T, int Hkv, int QB,
                           int topk, void* stream);

/*
 * swa_sink_sparse_fwd -- a sparse layer: causal attention of query i over
 * the keys j <= i of the key blocks selected for its query block, sink bias in
 * the denominator as in swa_sink_fwd.  k and v are the full-attention layer's
 * (the shared KV cache).
 *   idx [B, Hkv, ceil(T/QB), topk] int32: increasing block indices, -1 padded
 *   (as swa_topk_blocks writes them); QB in {32, 64, 128}.  A list is read up
 *   to its first negative entry: entries after it are ignored, and a list
 *   whose first entry is negative selects no key (its rows get out = 0 and
 *   lse = sink[h], the sink alone).  The entries
 *   before it must be distinct block indices in [0, ceil(T/128)); their
 *   order does not change the result beyond rounding (each key is masked
 *   causally on its own).  A repeated index counts its keys twice; an index
 *   past the end gives unspecified values, but every access stays inside
 *   q, k, v, out and lse (the loads are bounded by the tensor maps).
 *   Other arguments as swa_sink_fwd_ex; bf16 inputs, D = 64 or 128, Hq = 8 Hkv
 *   only (else SWA_EUNSUPPORTED).
 */
swa_status swa_sink_sparse_fwd(const void* q, const void* k, const void* v, const float* sink,
                               const int* idx, void* out, float* lse, int B, int T, int Hq,
                               int Hkv, int D, int QB, int topk, swa_dtype in_dtype,
                               swa_dtype out_dtype, void* stream);

/* Name of the prefill kernel swa_sink_fwd would launch for these sizes, or
 * "invalid": bf16 inputs take "tc_swa" (the sliding-window tensor-core kernel)
 * when W <= 129 and Hq / Hkv is 4 or a multiple of 8 up to 512 (D = 64 or
 * 128), and "tc_global" (the online-softmax tensor-core kernel, any window)
 * for the other bf16 cases with Hq / Hkv 1, 2, 4 or a multiple of 8 (D = 64
 * or 128); everything else takes "simt" (CUDA cores, fp32 or bf16 inputs). */
const char* swa_sink_fwd_path(int B, int T, int Hq, int Hkv, int D, int W, swa_dtype in_dtype);

/* Name of the decode kernel swa_sink_decode would launch for these sizes
 * ("tc_decode" for bf16, D = 64 or 128, W = 128 and Hq / Hkv in {1, 2, 4, 8, 16}
 * or a larger multiple of 8, run as groups of 8 heads; "simt_decode"
 * otherwise), or "invalid". */
const char* swa_sink_decode_path(int B, int Hq, int Hkv, int D, int W, swa_dtype in_dtype);

/* Name of the verify kernel swa_sink_verify would launch ("tc_verify" for
 * bf16, D = 64 or 128, W = 128, Hq / Hkv 1, 2, 4 or a multiple of 8 (groups
 * of 8 heads) and L <= 8; "simt_verify" otherwise), or "invalid". */
const char* swa_sink_verify_path(int B, int L, int Hq, int Hkv, int D, int W, swa_dtype in_dtype);

/* Static text for a status code. */
const char* swa_status_str(swa_status s);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* swa_last_error(void);

/* Reads and clears the device-side error word of the current device
 * (synchronises the device).  0 = none; otherwise a code naming the wait
 * that ran past its limit.  Returns SWA_ECUDA in *code's place on failure. */
int swa_device_error(void);

/*
 * swa_test_withhold_loads -- testing aid for the failure path: in the next
 * launch of the sliding-window tensor-core prefill kernel (swa_sink_fwd_path
 * "tc_swa") made from the calling host thread, CTA number `cta` issues none
 * of its loads.  Its waits then run past their 2 s limit: the first records
 * a wait code (0x101..0x10c) in the device error word, the CTA's other roles
 * see it and stop waiting, the CTA frees its tensor memory and returns,
 * leaving its tiles' out and lse rows unwritten.  The other CTAs finish
 * normally and the device stays usable.  Applies to one launch; -1 cancels.
 * Returns SWA_EINVAL for cta < -1.  Not for production use.
 */
swa_status swa_test_withhold_loads(int cta);

/* Library version, major*10000 + minor*100 + patch. */
int swa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWASINK_H */
