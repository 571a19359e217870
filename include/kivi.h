/*
 * kivi.h -- C ABI of libkivi: a KIVI-style quantized KV cache and its
 * decode-attention step, on one GB300 (sm_103a).
 *
 * Method (source: "Literature audit -- Group 2 (KV-cache compression primary
 * sources)", section 1 "KIVI -- kivi2024", list "Core algorithm
 * (implementation-grade)"):
 *   item 1  asymmetric round-to-nearest group quantizer, z = min,
 *           s = (max - min) / (2^B - 1), code = round((x - z) / s),
 *           B = 2 or 4 chosen separately for keys and values;
 *   item 2  keys quantized per channel in groups of G consecutive tokens;
 *   item 3  values quantized per token in groups of G channels;
 *   item 4  fp16 residual window of R tokens: prefill keeps the last t mod R
 *           keys and the last R values in fp16; during decode the fp16 key
 *           block is quantized whole when it holds R keys (R % G == 0) and
 *           the fp16 value queue pops and quantizes its oldest token when it
 *           holds R + 1;
 *   item 5  decode attention = softmax((q K_quant^T || q K_full^T) / sqrt(d))
 *           (V_quant || V_full).
 *
 * Conventions for every call:
 *   - tensor pointers are DEVICE pointers owned by the caller, read or
 *     written in stream order on `stream` (a cudaStream_t; 0 = legacy
 *     default stream).  Host-side arrays are named as such.
 *   - fp16 means IEEE binary16; tensors are dense, row-major, no padding.
 *   - every call validates all arguments before it changes anything; on an
 *     error nothing is launched and the cache is unchanged.
 *   - a CUDA error inside a call poisons the handle: later calls return
 *     KIVI_ERR_STATE (destroy still works).
 *   - calls on one handle are not thread-safe; different handles are
 *     independent.
 *   - no call allocates device memory except kivi_cache_create.
 * Supported shapes: k_bits, v_bits in {2, 4}; G in {16, 32, 64, 128};
 * d in {64, 128, 256} with d % G == 0; R % G == 0 (item 4's assertion);
 * 1 <= b <= 1024; h_q a multiple of h_kv with h_q / h_kv <= 8.
 * Anything else returns KIVI_ERR_UNSUPPORTED.
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KIVI_ABI_VERSION 6

typedef struct kivi_cache *kivi_cache_t;   /* opaque, library-owned */
typedef struct CUstream_st *kivi_stream_t; /* the same type as cudaStream_t */

typedef enum {
    KIVI_OK = 0,
    KIVI_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad handle */
    KIVI_ERR_UNSUPPORTED = 2,  /* shape or bit width outside the list above */
    KIVI_ERR_CAPACITY = 3,     /* a sequence would exceed max_tokens */
    KIVI_ERR_STATE = 4,        /* handle poisoned by an earlier CUDA error */
    KIVI_ERR_CUDA = 5,         /* a CUDA call failed (see kivi_last_error) */
    KIVI_ERR_OOM = 6           /* device or host allocation failed */
} kivi_status;

/* Create an empty cache for b sequences of h_kv KV heads of dimension d,
 * holding up to max_tokens tokens per sequence; k_bits / v_bits per item 1,
 * group size G per items 2-3, residual length R per item 4.  All device
 * memory of the cache is allocated here (packed codes, fp16 scale/zero,
 * fp16 residual windows, counters, decode partials).  *out receives the
 * handle; release it with kivi_cache_destroy. */
kivi_status kivi_cache_create(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R,
                              int max_tokens, kivi_cache_t *out);

/* Free every resource of the cache.  The handle is invalid afterwards;
 * passing it to any call returns KIVI_ERR_INVALID_ARG. */
kivi_status kivi_cache_destroy(kivi_cache_t c);

/* Prefill (item 4): reset every sequence and fill it from K and V, fp16
 * [b][h_kv][t_stride][d] (device).  Sequence i takes its first t[i] tokens
 * (t: HOST array of b int32, 0 <= t[i] <= t_stride, t[i] <= max_tokens).
 * Keys [0, t - t mod R) and values [0, max(t - R, 0)) are quantized; the
 * rest stays fp16.  Reads K and V in stream order; they may be freed or
 * reused once the stream has passed this call. */
kivi_status kivi_prefill(kivi_cache_t c, const void *K, const void *V, const int32_t *t,
                         int t_stride, kivi_stream_t stream);

/* Prefill with its attention: kivi_prefill(K, V, t, t_stride) and, from
 * the same pass over K and V, the prompt's causal attention in full
 * precision ("Literature audit -- Group 2", section 1 KIVI: its backends
 * list runs the prefill's attention on the unquantized K/V and quantizes
 * the cache after it; its limitations paragraph lists that unfused
 * quantization as open).  For sequence i, query head h (kv head
 * h / (h_q / h_kv)) and token tau < t[i]:
 *   out[i][h][tau] = sum_{s <= tau} softmax_s(q[i][h][tau] . K[i][j][s] / sqrt(d)) V[i][j][s]
 * q and out: fp16 [b][h_q][t_stride][d] (device, 16-byte aligned); rows
 * tau >= t[i] of out are not written.  The cache afterwards is bitwise the
 * one kivi_prefill leaves.  Scores accumulate in fp32; the softmax weights
 * enter the weighted sum of values rounded to fp16.  One launch.  Supports
 * d 64 or 128 and G <= 64 (KIVI_ERR_UNSUPPORTED otherwise); h_q a multiple
 * of h_kv, at most 8 times it. */
kivi_status kivi_prefill_attn(kivi_cache_t c, const void *q, const void *K, const void *V, const int32_t *t,
                              int t_stride, int h_q, void *out, kivi_stream_t stream);

/* Append one token to every sequence: k and v fp16 [b][h_kv][d] (device).
 * First, per sequence, the maintenance of item 4 left over from the previous
 * step: the fp16 key block is quantized if it holds R keys, and the oldest
 * fp16 value is popped and quantized if the queue holds R + 1.  Then k and
 * v join the fp16 windows.  Returns KIVI_ERR_CAPACITY (and changes nothing)
 * if any sequence is full. */
kivi_status kivi_append(kivi_cache_t c, const void *k, const void *v, kivi_stream_t stream);

/* Decode attention (item 5) for every sequence and query head.  q fp16
 * [b][h_q][d] (device), out fp16 [b][h_q][d] (device, caller-owned);
 * query head i reads KV head i / (h_q / h_kv).  Scores are q.k / sqrt(d)
 * over the quantized keys followed by the fp16 keys, one softmax over both,
 * weights applied to the quantized then fp16 values; fp32 accumulation.
 * A sequence with no tokens gets an all-zero output.  Read-only on the
 * cache (the call can be repeated, with bitwise identical results).  Preconditions: inputs finite and
 * |q_c| * s < 65504 for every key scale s (the scaled query is staged in
 * fp16 for the tensor-core contraction).  The kernel is launched as a
 * programmatic dependent of the previous kernel on the stream: its blocks
 * may be placed and set up while that kernel finishes, but nothing in
 * global memory is read before it has completed, so stream order holds. */
kivi_status kivi_decode_attn(kivi_cache_t c, const void *q, int h_q, void *out,
                             kivi_stream_t stream);

/* Decode attention with each token's attention weight: out as
 * kivi_decode_attn computes it (bitwise the same), and, for sequence i,
 * query head h and token t < T_i, probs[(i h_q + h) ld + t] = the softmax
 * weight of token t in that head's attention (fp32, device; tokens in
 * sequence order, quantized and fp16 alike; a row's weights sum to 1).
 * Entries t >= T_i are left as they were.  mass (device, same layout, may
 * be NULL) accumulates the weights: mass[...] += probs[...] for t < T_i, so
 * that repeated steps sum each token's attention over decode steps.  That
 * sum is H2O's eviction score ("Literature audit -- Group 2 (KV-cache
 * compression primary sources)", section 4 "H2O (Heavy-Hitter Oracle)":
 * per head, each key's softmax weights added over the query rows seen so
 * far), and section 1 "KIVI" counts KIVI as orthogonal to, and combinable
 * with, such eviction.  Token positions are stable across appends, so mass
 * rows stay aligned.
 * ld >= 1 and ld >= every T_i; probs and mass 4-byte aligned and distinct
 * (KIVI_ERR_INVALID_ARG otherwise).  Two launches: the decode kernel writes
 * raw scores into probs, a second kernel turns them into weights. */
kivi_status kivi_decode_attn_probs(kivi_cache_t c, const void *q, int h_q, void *out, float *probs,
                                   float *mass, int64_t ld, kivi_stream_t stream);

/* One decode step in one call: kivi_append(k, v) then kivi_decode_attn(q,
 * h_q, out), once both sets of arguments have been validated (a failed call
 * changes nothing; KIVI_ERR_CAPACITY if a sequence is full).  The cache
 * afterwards is bitwise the one the two calls leave; out agrees with theirs
 * within the decode tolerance (the work may be split differently).
 *
 * With h_q / h_kv <= 4 and no more (sequence, kv head) pairs than twice
 * the GPU's SM count, the step is one kernel launch: the decode kernel
 * appends the token itself (item 4's one-token maintenance: the new key
 * and value, and the value token leaving the queue, quantized per token as
 * in kivi_append) for every sequence whose key window is not full.  On a
 * step where some sequence's key window is full (every R steps per
 * sequence) the append kernel first handles just those sequences (two
 * launches).  Otherwise the call launches the append kernel and then the
 * decode kernel (with many pairs the append kernel's parallel appends are
 * faster than appends spread over the persistent decode CTAs).  The
 * environment variable KIVI_FUSED_STEP=0 forces two launches, =1 the fused
 * kernel wherever h_q / h_kv <= 4.  kivi_decode_plan reports the call's
 * launches.  k and v must stay unchanged until the call's work on `stream`
 * completes (the fused kernel reads them). */
kivi_status kivi_append_decode(kivi_cache_t c, const void *k, const void *v, const void *q, int h_q,
                               void *out, kivi_stream_t stream);

/* Per-sequence token counts (HOST arrays of b int32; any may be NULL):
 * T total, Tqk quantized keys, Tqv quantized values.  The fp16 windows hold
 * T - Tqk keys and T - Tqv values.  Reads the host mirror; no sync. */
kivi_status kivi_cache_lengths(kivi_cache_t c, int32_t *T, int32_t *Tqk, int32_t *Tqv);

/* Byte sizes of the six arrays kivi_cache_export writes, in its order. */
kivi_status kivi_cache_export_sizes(kivi_cache_t c, size_t sizes[6]);

/* Copy the cache's contents into HOST buffers (sizes from
 * kivi_cache_export_sizes), in the packed format below, then synchronize
 * `stream`.  Any pointer may be NULL to skip that array.  (On the device
 * the first four arrays are stored interleaved as block records, see
 * kivi_cache_export_records; this call splits them apart on the host.)
 *   Kc  uint32 [b][h_kv][fcap/64][2 d k_bits]  key codes, 64-token blocks
 *   Ksz fp16   [b][h_kv][fcap/G][2][d]          key scale (row 0), zero (row 1)
 *   Vc  uint32 [b][h_kv][fcap/16][d v_bits / 2] value codes, 16-token blocks
 *   Vsz fp16   [b][h_kv][fcap/16][2][d/G][16]   value scale / zero per token
 *   Kf  fp16   [b][h_kv][R][d]                  fp16 keys, token tau at tau % R
 *   Vf  fp16   [b][h_kv][R+1][d]                fp16 values, tau at tau % (R+1)
 * fcap = max_tokens rounded up to a multiple of max(64, G).
 * Inside a key block kb, the word of lane L = 4g + t (g < 8, t < 4) and lane
 * word u = (2 j + hh) (k_bits/2) + wi (j < d/16, hh < 2, wi < k_bits/2) is
 * word (u/4) 128 + 4 L + u%4.  Its low 16 bits hold channel 16j + 8hh + 2t,
 * its high 16 bits that channel + 1, each packing along tokens: the field at
 * bits [r k_bits, (r+1) k_bits) of a half is token 64 kb + 8 (wi 16/k_bits
 * + r) + g (item 2's packing along the token axis, interleaved by 8).
 * Inside a value block vb, the word of lane L and lane word u = p nwv + w
 * (p < 2, w < nwv = d v_bits / 128) is word (u/cs) 32 cs + L cs + u%cs with
 * cs = min(4, d v_bits / 64).  Its low half holds token 16 vb + 2t + 8p,
 * its high half that token + 1, each packing along channels: the field at
 * bits [r v_bits, (r+1) v_bits) is channel 8 (w 16/v_bits + r) + g.
 * Fields of tokens not yet quantized are zero. */
kivi_status kivi_cache_export(kivi_cache_t c, void *Kc, void *Ksz, void *Vc, void *Vsz, void *Kf,
                              void *Vf, kivi_stream_t stream);

/* The packed arrays as the device stores them: one record per 64-token
 * block kb of each (sequence i, kv head j), records ordered [b][h_kv][fcap/64],
 * each record holding, back to back, in the element formats above:
 *   Kc block kb                      2 d k_bits words
 *   Ksz rows of the block's groups   [max(1, 64/G)][2][d] fp16 (G = 128: the
 *                                    rows of group kb/2, in both its records)
 *   Vc value blocks 4kb .. 4kb+3     4 (d v_bits / 2) words
 *   Vsz value blocks 4kb .. 4kb+3    4 [2][d/G][16] fp16
 * except that inside a record every scale or zero row is stored lane-major:
 * in a key row (d halves) channel c = 16 jj + 8 hh + 2 t + lo (t < 4,
 * lo < 2) sits at position t d/4 + 4 jj + 2 hh + lo, and in a value row (16
 * halves) token tau = 2 t + 8 p + lo sits at 4 t + 2 p + lo.
 * With records == NULL, writes the byte size of all records to *bytes.
 * Otherwise copies them into `records` (host or device memory, *bytes at
 * least that size; cudaMemcpyDefault), synchronizes `stream` and sets *bytes
 * to the size copied.  Errors: KIVI_ERR_INVALID_ARG (bytes NULL, buffer too
 * small). */
kivi_status kivi_cache_export_records(kivi_cache_t c, void *records, size_t *bytes,
                                      kivi_stream_t stream);

/* Synchronize `stream` and read the device status word into *flags (HOST).
 * 0 means no kernel recorded an anomaly; bit 0: a counter out of range,
 * bit 1: a bounded wait for a shared-memory copy ran out.  Clears it. */
kivi_status kivi_cache_check(kivi_cache_t c, uint32_t *flags, kivi_stream_t stream);

/* Kernel timing for measurement: when on, kivi_decode_attn records a pair
 * of CUDA events around its attention kernel(s) (up to 4096 pairs, then it
 * stops recording).  kivi_profile_read synchronizes them, returns the summed
 * milliseconds and the number of launches timed, and clears the record. */
kivi_status kivi_profile_enable(kivi_cache_t c, int on);
kivi_status kivi_profile_read(kivi_cache_t c, double *total_ms, int *launches);

/* How the last decode call (kivi_decode_attn, kivi_decode_attn_probs or
 * kivi_append_decode) was launched (HOST outputs, any may be NULL):
 * persistent CTAs of the decode kernel, and the call's launches of the
 * decode kernel (1) plus kivi_append_decode's append kernel when it
 * launched one (the weights' finalizing kernel is not counted). */
kivi_status kivi_decode_plan(kivi_cache_t c, int *splits, int *launches);

/* A packed cache held in caller-owned device memory: the block records
 * that kivi_cache_export_records documents, the fp16 windows Kf and Vf as
 * kivi_cache_export documents them (fcap as there), and the per-sequence
 * counters as DEVICE int32 arrays of b entries. */
typedef struct {
    int b, h_kv, d, k_bits, v_bits, G, R, max_tokens;
    const void *blocks, *Kf, *Vf;   /* device, 16-byte aligned */
    const int32_t *T, *Tqk, *Tqv;   /* device counters */
} kivi_packed_cache;

/* Decode attention that allocates nothing.  (The pages have no counterpart:
 * this is a library service for callers that cannot call cudaMalloc, e.g.
 * code running while a framework's memory pool owns the device memory, in
 * an allocator callback, or under a real-time budget that forbids device
 * allocation after start-up.)  Computes exactly what kivi_decode_attn
 * computes, over the cache described by *cache; q and out as there; the
 * shape rules are kivi_cache_create's.
 * Its scratch (split partials, merge tickets, status word) lives in one
 * fixed 16 MiB __device__ array inside the library; shapes whose scratch
 * b * h_q * P * (d + 4) * 4 bytes plus tickets exceed it (P: the most
 * persistent CTAs sharing one (sequence, kv head, head group)) are
 * rejected with KIVI_ERR_UNSUPPORTED and a kivi_last_error() message.  The
 * call launches on `stream` and clears the tickets itself; all calls share
 * the array, so calls whose kernels overlap on the GPU race and must not be
 * issued.  CUDA loads device code and __device__ arrays lazily: the first
 * call on a device loads the array (16 MiB of device memory, held until the
 * process exits) and looks up its device address (cudaGetSymbolAddress)
 * with that device current, and the first call of each shape (d, k_bits,
 * v_bits, G) loads that kernel's code.  So make one warm-up call per device
 * and shape before a memory pool takes the device memory, and before any
 * stream capture; later calls take no device memory.  After a
 * cudaDeviceReset the entry point must not be used (the looked-up address
 * is stale).  The kernel's status word is cleared by each call and not
 * reported: this path has no counterpart of kivi_cache_check.  No
 * cudaMalloc, cudaFree or other allocating routine is called. */
kivi_status kivi_decode_attn_noalloc(const kivi_packed_cache *cache, const void *q, int h_q,
                                     void *out, kivi_stream_t stream);

/* The launch plan kivi_decode_attn would use for a cache of this shape
 * (kivi_cache_create's rules; max_tokens sets the capacity) holding these
 * per-sequence counters (HOST arrays of b int32, 0 <= Tqk, Tqv <= T <=
 * max_tokens) for h_q query heads, on a GPU with num_sms SMs.  Host-only:
 * no CUDA call is made, so it runs without a GPU.  out (HOST, 6 int64):
 * persistent CTAs, warps per CTA, ring stages per warp, the most split
 * partials any (sequence, kv head, group of up to 4 query heads) receives,
 * the partial slots a cache of this shape holds for each, and the total
 * work units (a fully quantized 64-token block is one unit, any other
 * block a fixed larger weight).  The kernel requires partials <= slots. */
kivi_status kivi_plan_preview(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R, int max_tokens,
                              int h_q, const int32_t *T, const int32_t *Tqk, const int32_t *Tqv, int num_sms,
                              int64_t out[6]);

const char *kivi_status_str(kivi_status s);
/* Text of the last error on the calling thread ("" if none). */
const char *kivi_last_error(void);
int kivi_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KIVI_H */
