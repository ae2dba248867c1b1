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
 *     and contiguous in the layouts stated per call, 16-byte aligned.  The
 *     library allocates no memory and keeps no state between calls.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Results are valid once the stream reaches them.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns an error and touches no memory.  A failed launch
 *     returns SWA_ECUDA (text in swa_last_error()).  Nothing traps on the
 *     device: a device-side wait that runs past its time limit records a code
 *     readable with swa_device_error() and the kernel returns early.
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
 * (slot = pos[b] mod W), the cache update that precedes swa_sink_decode.
 *   k_new, v_new [B, Hkv, D] dtype;  k_ring, v_ring [B, Hkv, W, D] dtype (updated)
 *   pos [B] int64 >= 0 (device); a negative pos leaves that sequence's ring unchanged.
 */
swa_status swa_ring_append(const void* k_new, const void* v_new, void* k_ring, void* v_ring,
                           const int64_t* pos, int B, int Hkv, int D, int W, swa_dtype dtype,
                           void* stream);

/* Name of the prefill kernel swa_sink_fwd would launch for these sizes
 * ("tc_swa", "tc_global", "simt"), or "invalid". */
const char* swa_sink_fwd_path(int B, int T, int Hq, int Hkv, int D, int W, swa_dtype in_dtype);

/* Name of the decode kernel swa_sink_decode would launch for these sizes
 * ("tc_decode" for bf16, D = 128, W = 128, Hq = 8 Hkv; "simt_decode"
 * otherwise), or "invalid". */
const char* swa_sink_decode_path(int B, int Hq, int Hkv, int D, int W, swa_dtype in_dtype);

/* Static text for a status code. */
const char* swa_status_str(swa_status s);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* swa_last_error(void);

/* Reads and clears the device-side error word of the current device
 * (synchronises the device).  0 = none; otherwise a code naming the wait
 * that ran past its limit.  Returns SWA_ECUDA in *code's place on failure. */
int swa_device_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int swa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWASINK_H */
