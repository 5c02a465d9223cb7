/*
 * attn.h -- C ABI of libattn.so, a GB300 (sm_103a) attention-forward library.
 *
 * The operation is multi-head scaled-dot-product attention computed in one
 * fused pass ("A Thread-Register Decoupled GPU Execution Model for Efficient
 * Tensor Computation", Background, Equ. 1 -- referenced there, not printed;
 * its standard content is used):
 *
 *   S = Q K^T * scale (+ causal mask),  P = softmax(S) row-wise,  O = P V,
 *   LSE = ln sum_j exp(S_ij)   (natural log, over visible keys, scale included)
 *
 * with grouped-query sharing (same page, Methodology: GQA "eight heads per
 * group" and MQA): query head h reads KV head h / (Hq / Hkv).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE memory owned by the caller.  The library
 *    never allocates, frees or synchronises on these paths; each call enqueues
 *    its kernels on `stream` and returns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - Layout is row-major, contiguous: Q [B,Hq,Sq,D], K and V [B,Hkv,Sk,D]
 *    (bf16), O [B,Hq,Sq,D] and LSE [B,Hq,Sq] (fp32).
 *  - The return value is an attn_status.  Arguments are validated before any
 *    launch; a rejected call launches nothing.  ATTN_ERR_CUDA reports a launch
 *    failure (cudaGetLastError).  Errors raised asynchronously by a kernel
 *    surface on the caller's next synchronisation, as in CUDA itself; a kernel
 *    whose internal wait gave up records ATTN_ERR_TIMEOUT, readable with
 *    attn_debug_status().
 *  - Thread safety: calls may be made concurrently from several host threads.
 */
#ifndef TENSOR_ATTN_FWD_GB300_ATTN_H
#define TENSOR_ATTN_FWD_GB300_ATTN_H

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, Hq % Hkv != 0, ... */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. an unsupported D) */
    ATTN_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    ATTN_ERR_CUDA = 4,         /* the CUDA runtime reported an error */
    ATTN_ERR_TIMEOUT = 5,      /* a kernel's bounded wait expired (device status) */
    ATTN_ERR_BOUNDS = 6        /* debug builds (-DATTN_DEBUG_BOUNDS): a kernel skipped a
                                  store outside its output buffer (device status) */
} attn_status;

/*
 * Prefill / general attention forward.
 * Source: "A Thread-Register Decoupled GPU Execution Model for Efficient
 * Tensor Computation", Background (Equ. 1; fused FlashAttention-style
 * computation; softmax phase interleaved with the two GEMMs, Fig. 2) and
 * Methodology (GQA/MQA).  Causal masking is bottom-right aligned: query row i
 * sees key j iff j <= i + Sk - Sq.  A row that sees no key gets O = 0 and
 * LSE = -inf.
 *
 *   q  [B,Hq,Sq,D] bf16     k, v [B,Hkv,Sk,D] bf16
 *   o  [B,Hq,Sq,D] fp32     lse  [B,Hq,Sq]    fp32
 *   B >= 1, Hq >= 1, Hkv >= 1, Hq % Hkv == 0, Sq >= 1, Sk >= 1,
 *   D in {64, 128, 256} (D = 256 runs a one-query-tile-per-CTA kernel)
 *   causal in {0, 1}; scale is applied to QK^T (callers usually pass 1/sqrt(D)).
 * All pointers must be 16-byte aligned.
 */
ATTN_API int attn_fwd(const void *q, const void *k, const void *v, float *o, float *lse,
             int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
             void *stream);

/*
 * attn_fwd with a bf16 output: identical computation and arguments, except
 * that o is [B,Hq,Sq,D] bf16 (each fp32 result rounded to nearest even),
 * halving the output traffic.  LSE stays fp32.
 * Source: as attn_fwd (the FlashAttention-style kernels the page compares
 * against write their output in the input precision).
 */
ATTN_API int attn_fwd_bf16o(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                            float scale, void *stream);

/*
 * Prefill forward over KV splits, for shapes with too few (batch, head, 256
 * query rows) work items to fill the GPU -- chunked prefill, a short query
 * chunk against a long cache (Sq << Sk).  The same computation as attn_fwd,
 * cut along the keys as split-KV decode cuts it ([FIBER] Evaluation: decode
 * and its split-KV combine); the partials are merged by attn_combine.
 *   Split s covers KV tiles [s*t, (s+1)*t) of 128 keys, t = ceil(ceil(Sk/128) /
 *   num_splits), with the causal mask of attn_fwd (bottom-right).
 *   o_part    float [num_splits, B, Hq, Sq, D]: split s's output normalised by
 *             its own row sum; rows the split leaves without keys get 0.
 *   lse_part  float [num_splits, B, Hq, Sq]: split s's log-sum-exp, -inf for
 *             rows without keys.
 *   Merge with attn_combine(o_part, lse_part, o, lse, B * Sq, Hq, D, num_splits):
 *   that call reads the partials as num_splits x (B*Hq*Sq rows) x D, which is
 *   their layout, and writes O [B,Hq,Sq,D] and LSE [B,Hq,Sq].
 *   1 <= num_splits <= ceil(Sk / 128), else ATTN_ERR_INVALID_ARG; D 64 or 128,
 *   else ATTN_ERR_UNSUPPORTED.  Other arguments and errors as attn_fwd.
 */
ATTN_API int attn_fwd_splitkv(const void *q, const void *k, const void *v, float *o_part,
                              float *lse_part, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                              int causal, int num_splits, float scale, void *stream);

/*
 * A split count for attn_fwd_splitkv on the current device (a measured rule of
 * this library, not part of the method).  The prefill's work items are pairs
 * of 128-row query tiles: B * Hq * ceil(Sq / 256) of them, or B * Hq / 2 when
 * Sq <= 128 and Hq / Hkv is even (two query heads of one KV group share an
 * item).  With the items already filling at least 80 % of the SMs, or with
 * Sk <= 2 * Sq and fewer than 16 128-key tiles (the combine would cost more
 * than the split saves), 1 (use attn_fwd); otherwise the largest count that
 * still runs every item in one round on the SMs (floor(SMs / items)), with at
 * least four 128-key tiles per split.  Always 1 for D = 256.  Host-only:
 * launches nothing.
 *   Returns ATTN_ERR_INVALID_ARG for non-positive sizes or Hq % Hkv != 0,
 *   ATTN_ERR_CUDA if the device cannot be queried.
 */
ATTN_API int attn_fwd_num_splits(int B, int Hq, int Hkv, int Sq, int Sk, int D, int *num_splits);

/*
 * Split-KV decode, first stage: per-split partial results for one query row
 * per head.  Source: same page, Methodology and Evaluation (FlashDecoding:
 * decode is GEMV plus softmax, memory bound, no tensor cores).
 *
 * The key axis is cut into num_splits chunks of ceil(Sk / num_splits) keys;
 * split s covers keys [s*chunk, min(Sk, (s+1)*chunk)).  For each split,
 * o_part holds the split's own normalised output and lse_part its own
 * log-sum-exp; an empty split writes O = 0 and LSE = -inf.
 *
 *   q [B,Hq,1,D] bf16;  k, v [B,Hkv,Sk,D] bf16 (contiguous KV per sequence)
 *   o_part [num_splits,B,Hq,D] fp32;  lse_part [num_splits,B,Hq] fp32
 *     (caller-owned workspace, fully overwritten)
 *   1 <= num_splits <= Sk; D in {64, 128, 256}; no mask.
 */
ATTN_API int attn_decode_splitkv(const void *q, const void *k, const void *v, float *o_part,
                        float *lse_part, int B, int Hq, int Hkv, int Sk, int D,
                        int num_splits, float scale, void *stream);

/*
 * Split-KV decode over sequences of different lengths (first stage).
 * Source: "VDCores: Resource Decoupled Programming and Execution for
 * Asynchronous GPUs", Evaluation (the dynamic-attention-length case study:
 * decode requests whose KV lengths differ) applied to the FlashDecoding split
 * of "A Thread-Register Decoupled GPU Execution Model for Efficient Tensor
 * Computation", Methodology.
 *
 * Same as attn_decode_splitkv, except that sequence b attends only to its
 * first seqlens[b] keys: k and v are [B,Hkv,Sk,D] buffers of capacity Sk per
 * sequence, and keys at or past seqlens[b] are never read into the result
 * (their contents may be anything, including NaN).  Each sequence is split on
 * its own: chunk_b = ceil(seqlens[b] / num_splits).  A sequence of length 0
 * yields O = 0 and LSE = -inf after attn_combine.
 *
 *   seqlens: device int32 [B], 4-byte aligned; values are clamped to [0, Sk].
 *   Other arguments, layouts and errors as for attn_decode_splitkv.
 */
ATTN_API int attn_decode_splitkv_varlen(const void *q, const void *k, const void *v,
                                        const int *seqlens, float *o_part, float *lse_part,
                                        int B, int Hq, int Hkv, int Sk, int D, int num_splits,
                                        float scale, void *stream);

/*
 * Split-KV decode over a paged KV cache (first stage; combine with
 * attn_combine).  Source: "VDCores: Resource Decoupled Programming and
 * Execution for Asynchronous GPUs", Evaluation (decode attention whose
 * per-request length changes step by step); the cache is held in fixed-size
 * pages so that a sequence can grow without moving its keys.  The pages print
 * no layout; this one keeps each (page, KV head) block contiguous.
 *
 * Key t (0 <= t < seqlens[b]) of sequence b, KV head g, is
 *   k_cache[block_table[b * max_pages + t / page_size], g, t % page_size, :]
 * (same for v_cache); sequence b attends to exactly its seqlens[b] keys.
 *
 *   q           [B,Hq,1,D] bf16 (as attn_decode_splitkv)
 *   k_cache, v_cache  [num_pages, Hkv, page_size, D] bf16, 16-byte aligned
 *   block_table device int32 [B, max_pages]; entries in [0, num_pages).  An
 *               entry outside that range that a sequence reaches sets
 *               ATTN_ERR_INVALID_ARG in the device status word
 *               (attn_debug_status) and that block reads page 0 instead.
 *   seqlens     device int32 [B], clamped to [0, max_pages * page_size]
 *   page_size   a multiple of 32 (else ATTN_ERR_UNSUPPORTED)
 *   o_part, lse_part, num_splits, scale, stream: as attn_decode_splitkv,
 *   except the split rule: chunk = 32 * ceil(ceil(len / num_splits) / 32)
 *   (whole 32-key blocks), split s covers [s*chunk, min(len, (s+1)*chunk)).
 *   1 <= num_splits <= max_pages * page_size.
 */
ATTN_API int attn_decode_splitkv_paged(const void *q, const void *k_cache, const void *v_cache,
                                       const int *block_table, const int *seqlens,
                                       float *o_part, float *lse_part, int B, int Hq, int Hkv,
                                       int num_pages, int page_size, int max_pages, int D,
                                       int num_splits, float scale, void *stream);

/*
 * Rotary-embedding table for attn_qkv_rope.
 * Source: "A Thread-Register Decoupled GPU Execution Model for Efficient
 * Tensor Computation", Background (RoPE around the projections); the standard
 * rotary frequencies theta_i = base^(-2i/D).
 *   table [max_pos, D/2, 2] fp32 device, 16-byte aligned:
 *     table[p][i] = (cos(p * theta_i), sin(p * theta_i)), computed in double
 *     precision and rounded to fp32.
 *   D even, base > 1 (10000 in the usual models).
 */
ATTN_API int attn_rope_table(float *table, int max_pos, int D, float base, void *stream);

/*
 * QKV projection with the rotary embedding applied in its epilogue, writing
 * the attention inputs.  Source: same page, Background (the hidden states are
 * projected to Q, K and V by GEMMs with the weight matrices) and "VDCores:
 * Resource Decoupled Programming and Execution for Asynchronous GPUs",
 * Evaluation (QKV-Projection + RoPE as one fused pattern).
 *
 *   x  [B*S, hidden] bf16 (token t = b*S + s), hidden % 8 == 0
 *   w  [(Hq + 2*Hkv)*D, hidden] bf16: the rows of Wq, then Wk, then Wv
 *      (the usual [out_features, in_features] weight layout)
 *   y = x w^T; head n of y (columns [n*D, (n+1)*D)) is query head n for
 *   n < Hq, then Hkv key heads, then Hkv value heads.
 *   rope_table from attn_rope_table, at least max_pos rows
 *   positions device int32 [B*S] (position of each token), or NULL for
 *      position = s; a position outside [0, max_pos) sets
 *      ATTN_ERR_INVALID_ARG in the device status word and is clamped.
 *   style 0 rotates dims (2i, 2i+1) of each Q and K head, style 1 rotates
 *      dims (i, i + D/2):  (a, b) -> (a cos - b sin, a sin + b cos).
 *   q [B,Hq,S,D], k, v [B,Hkv,S,D] bf16 outputs (the attn_fwd inputs),
 *      rounded to nearest even from the fp32 accumulator.
 *   D in {64, 128, 256}; Hq % Hkv == 0.  All pointers 16-byte aligned
 *   (positions 4-byte).
 */
ATTN_API int attn_qkv_rope(const void *x, const void *w, const float *rope_table,
                           const int *positions, void *q, void *k, void *v, int B, int S,
                           int hidden, int Hq, int Hkv, int D, int max_pos, int style,
                           void *stream);

/*
 * A split count for attn_decode_splitkv (and its varlen / paged forms) on the
 * current device.  The pages leave the split count to the caller; this is a
 * measured rule for this library's decode kernel, not part of the method.
 * With B * Hkv * ceil((Hq/Hkv) / 16) CTAs per split already filling at least
 * 80 % of the SMs, one split streams K/V fastest.  Otherwise, at D = 256
 * (where a CTA takes a whole SM) floor(SMs / CTAs per split), so that they run
 * in one wave; at D = 64 and 128 ceil(SMs / CTAs per split), twice that at
 * D = 64, rounded to the nearest power of two.  At most 32 splits (the
 * combine's one pass over a warp of partials), each keeping at least 128 KB of
 * K and V per KV head (32768 / D keys).  Host-only: launches nothing.
 *
 *   *num_splits receives the count (>= 1, <= max(1, min(32, Sk / (32768 / D)))).
 *   Returns ATTN_ERR_INVALID_ARG for non-positive sizes or Hq % Hkv != 0,
 *   ATTN_ERR_CUDA if the device cannot be queried.
 */
ATTN_API int attn_decode_num_splits(int B, int Hq, int Hkv, int Sk, int D, int *num_splits);

/*
 * Split-KV decode, second stage: log-sum-exp combine of the partials.
 * Source: same page (FlashDecoding's reduction across key splits).
 *   lse = ln sum_s exp(lse_s);  o = sum_s exp(lse_s - lse) * o_s
 * Rows whose splits are all empty get o = 0, lse = -inf.
 *
 *   o_part [num_splits,B,Hq,D], lse_part [num_splits,B,Hq] (fp32, as written
 *   by attn_decode_splitkv);  o [B,Hq,D] fp32;  lse [B,Hq] fp32.
 *   D in {64, 128, 256}.
 */
ATTN_API int attn_combine(const float *o_part, const float *lse_part, float *o, float *lse, int B,
                 int Hq, int D, int num_splits, void *stream);

/*
 * Decode in one launch: the split-KV partials of attn_decode_splitkv (or, with
 * seqlens, of attn_decode_splitkv_varlen), and their log-sum-exp combine
 * (attn_combine's formula).  Source: "A Thread-Register Decoupled GPU
 * Execution Model for Efficient Tensor Computation", Methodology and
 * Evaluation (FlashDecoding: per-split partials, then the reduction across
 * splits); with seqlens, "VDCores: Resource Decoupled Programming and
 * Execution for Asynchronous GPUs", Evaluation (dynamic attention length).  The combine of each (batch, KV
 * head, 16-query-head slice) group runs in the CTA that completes the group's
 * last split, found with one int32 counter per group, so it overlaps the
 * streaming of other groups and needs no second kernel.
 *
 *   q, k, v, B, Hq, Hkv, Sk, D, num_splits, scale, stream: as attn_decode_splitkv
 *   seqlens   optional device int32 [B] (NULL: every sequence has Sk keys), as
 *             attn_decode_splitkv_varlen
 *   o [B,Hq,D], lse [B,Hq]: fp32 results, 16-byte aligned
 *   o_part [num_splits,B,Hq,D], lse_part [num_splits,B,Hq]: fp32 workspace,
 *             16-byte aligned; holds the partials after the call
 *   counters  device int32 [attn_decode_fused_counters(B, Hq, Hkv)], all zero
 *             on entry.  A call that completes without a device-side error
 *             leaves them zero, so one zeroed array serves every later call on
 *             the same stream.  Calls whose kernels may overlap (other streams)
 *             need arrays of their own.  After a call that reported
 *             ATTN_ERR_TIMEOUT (attn_debug_status), zero the array again.
 *   Returns the argument errors of attn_decode_splitkv, and ATTN_ERR_INVALID_ARG
 *   for NULL o, lse or counters; ATTN_ERR_MISALIGNED for an unaligned output or
 *   counter array.
 */
ATTN_API int attn_decode_fused(const void *q, const void *k, const void *v, const int *seqlens,
                               float *o, float *lse, float *o_part, float *lse_part,
                               int *counters, int B, int Hq, int Hkv, int Sk, int D,
                               int num_splits, float scale, void *stream);

/*
 * attn_decode_fused over a paged cache: the partials of
 * attn_decode_splitkv_paged (its cache layout, block table, sequence lengths
 * and split rule) and their combine in one launch, with o, lse and counters
 * as attn_decode_fused.  Source: as attn_decode_splitkv_paged ("VDCores:
 * Resource Decoupled Programming and Execution for Asynchronous GPUs",
 * Evaluation) and attn_combine.  Returns the argument errors of both.
 */
ATTN_API int attn_decode_fused_paged(const void *q, const void *k_cache, const void *v_cache,
                                     const int *block_table, const int *seqlens, float *o,
                                     float *lse, float *o_part, float *lse_part, int *counters,
                                     int B, int Hq, int Hkv, int num_pages, int page_size,
                                     int max_pages, int D, int num_splits, float scale,
                                     void *stream);

/*
 * Number of int32 counters attn_decode_fused needs: B * Hkv * ceil((Hq/Hkv)/16).
 * Host-only.  ATTN_ERR_INVALID_ARG for non-positive sizes or Hq % Hkv != 0.
 */
ATTN_API int attn_decode_fused_counters(int B, int Hq, int Hkv, int *count);

/*
 * Attention backward: gradients of sum(dO * O) for the attn_fwd computation.
 * Source: "A Thread-Register Decoupled GPU Execution Model for Efficient
 * Tensor Computation", Methodology and Evaluation (the FlashAttention backward
 * pass: recompute the scores, then dV = P^T dO, dS = P * (dO V^T - Delta),
 * dQ = scale * dS K, dK = scale * dS^T Q, with Delta = rowsum(dO * O)).
 * dK and dV sum over the query heads that share a KV head.
 *
 *   q [B,Hq,Sq,D], k, v [B,Hkv,Sk,D], dout [B,Hq,Sq,D]   bf16
 *   o [B,Hq,Sq,D] fp32 and lse [B,Hq,Sq] fp32            as written by attn_fwd
 *   dq [B,Hq,Sq,D], dk, dv [B,Hkv,Sk,D]                  fp32 outputs
 *   delta_ws [B,Hq,Sq] fp32                              caller-owned workspace
 *   Same causal / scale / size rules as attn_fwd; D in {64, 128}.
 * Enqueues three kernels (Delta, dK/dV, dQ) on `stream`.
 */
ATTN_API int attn_bwd(const void *q, const void *k, const void *v, const float *o,
                      const float *lse, const void *dout, float *dq, float *dk, float *dv,
                      float *delta_ws, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                      float scale, void *stream);

/* Human-readable name of a status code (static string, never NULL). */
ATTN_API const char *attn_status_string(int status);

/*
 * Debug: synchronise `stream`, then read and clear this device's kernel
 * status word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT (a kernel's bounded wait
 * expired since the last read) or ATTN_ERR_CUDA (the synchronisation itself
 * failed).  Not for the hot path: it blocks the calling thread.
 */
ATTN_API int attn_debug_status(void *stream);

/*
 * Self-test of the kernels' bounded waits (failure detection without a fault).
 * Launches one thread that waits on an mbarrier nothing ever arrives on, with
 * the loop every kernel's waits use, until `limit_ns` nanoseconds have passed;
 * it then records ATTN_ERR_TIMEOUT in the device status word -- as a kernel
 * whose producer stalled would -- and returns.  The context stays usable.
 *   limit_ns   1,000 .. 1,000,000,000 (else ATTN_ERR_INVALID_ARG)
 *   waited_ns  device pointer (8-byte aligned) that receives the time the wait
 *              took, or NULL
 * Returns ATTN_OK once the kernel is enqueued on `stream`; read the outcome
 * with attn_debug_status().  Not for the hot path.
 */
ATTN_API int attn_wait_selftest(unsigned long long limit_ns, unsigned long long *waited_ns,
                                void *stream);

/* Library ABI version, (major << 16) | minor. */
ATTN_API int attn_version(void);

/*
 * Split-KV decode and LSE combine in one call that allocates nothing.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory when they call in -- for example a
 * plug-in run by a host framework that owns all device memory and gives the
 * plug-in no allocator, or a latency-critical serving loop that may not call
 * cudaMalloc/cudaFree (which can synchronise the whole device).  Such callers
 * cannot supply the o_part/lse_part workspace that attn_decode_splitkv needs.
 *
 * Computes exactly what attn_decode_splitkv followed by attn_combine compute
 * (same arguments, same layouts, same results), but keeps the per-split
 * partials in a fixed scratch array that is part of the library's own device
 * image: ATTN_NOALLOC_SCRATCH_FLOATS floats (16 MiB), reserved on every GPU
 * that loads the library until the process exits.
 *
 *   q [B,Hq,1,D] bf16; k, v [B,Hkv,Sk,D] bf16; o [B,Hq,D] fp32; lse [B,Hq] fp32
 *   (caller-owned device memory, 16-byte aligned).
 *   Requires num_splits * B * Hq * (D + 1) <= ATTN_NOALLOC_SCRATCH_FLOATS;
 *   larger requests return ATTN_ERR_UNSUPPORTED and launch nothing.
 *   Other argument errors are reported as for attn_decode_splitkv.
 *
 * Set-up: the first call on a device looks up that device's address of the
 * scratch array (cudaGetSymbolAddress, no allocation) with the device current;
 * make that first call before any stream capture.  No call ever allocates or
 * frees device memory.
 * Sharing: every call on a device uses the same scratch array, and the array
 * keeps the last call's partials.  Nothing needs to start at zero -- each call
 * overwrites every partial it reads -- but calls whose kernels overlap on the
 * GPU (different streams, or different host threads) race on the array and
 * must be serialised by the caller, e.g. by issuing them on one stream.
 */
#define ATTN_NOALLOC_SCRATCH_FLOATS (4u * 1024u * 1024u)
ATTN_API int attn_decode_noalloc(const void *q, const void *k, const void *v, float *o,
                                 float *lse, int B, int Hq, int Hkv, int Sk, int D,
                                 int num_splits, float scale, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* TENSOR_ATTN_FWD_GB300_ATTN_H */
