// kivi_internal.cuh -- geometry, device-array bundle and layout index math
// shared by the kernels and the host manager of libkivi.
//
// The packed format is the one the C header documents (kivi_cache_export):
// keys in 64-token blocks, each uint32 word carrying two channels, each
// 16-bit half packing one channel along tokens (tokens interleaved by 8, so
// one lane's word feeds the A operand of an m16n8k16 MMA directly); values
// in 16-token blocks, each word carrying two tokens, each half packing one
// token along channels (channels interleaved by 8).  Scale and zero are fp16.
//
// In device memory the four packed arrays are interleaved by 64-token block:
// the record of block kb of (sequence i, kv head j) holds, back to back,
//   key codes of block kb          kc_blk words
//   key scale/zero rows            [groups of block kb][2][d] fp16
//   value codes of blocks 4kb..+3  4 vc_blk words
//   value scale/zero of the same   4 vsz_blk fp16
// so the decode kernel fetches a block with one bulk copy.  With G = 128 a
// key group spans two blocks and both records carry its rows.
//
// Inside a record the scale and zero rows are stored lane-major, so that
// the decode kernel's lane t (t < 4) reads its values with one vector load:
//   key row (d halves): channel c = 16 jj + 8 hh + 2 t + lo sits at
//     position t (d / 4) + 4 jj + 2 hh + lo;
//   value row (16 halves, one per token of a 16-token block): token
//     tau = 2 t + 8 p + lo sits at position 4 t + 2 p + lo.
// kivi_cache_export undoes the permutation (its arrays are in natural order).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define KIVI_MAX_BATCH 1024
#define KIVI_MAX_QPERKV 8
#define KIVI_KBLK 64   // tokens per key block
#define KIVI_VBLK 16   // tokens per value block

// status-word bits (also documented in kivi.h)
#define KIVI_FLAG_COUNTER 1u
#define KIVI_FLAG_WAIT 2u

struct KiviGeom {
    int b, h, d, kbits, vbits, G, R;
    int fcap;     // capacity rounded up to a multiple of max(64, G)
    int nkb;      // key blocks per (sequence, head)   = fcap / 64
    int nkg;      // key groups per (sequence, head)   = fcap / G
    int nvb;      // value blocks per (sequence, head) = fcap / 16
    int kc_blk;   // words per key block   = 2 d kbits
    int vc_blk;   // words per value block = d vbits / 2
    int vsz_blk;  // halves per value block of scale/zero = 2 (d/G) 16
    int kgr;      // key groups whose rows a record holds = max(1, 64 / G)
    int off_ksz, off_vc, off_vsz, rec_bytes;   // record layout (bytes)
    int smax;     // decode partials the buffer holds per (sequence, query head)
};

// Fills the derived fields of g from b, h, d, kbits, vbits, G, R and the
// token capacity.
inline void kivi_geom_init(KiviGeom &g, int max_tokens) {
    const int q = g.G > 64 ? g.G : 64;
    g.fcap = (max_tokens + q - 1) / q * q;
    g.nkb = g.fcap / 64;
    g.nkg = g.fcap / g.G;
    g.nvb = g.fcap / 16;
    g.kc_blk = 2 * g.d * g.kbits;
    g.vc_blk = g.d * g.vbits / 2;
    g.vsz_blk = 2 * (g.d / g.G) * 16;
    g.kgr = g.G >= 64 ? 1 : 64 / g.G;
    g.off_ksz = g.kc_blk * 4;
    g.off_vc = g.off_ksz + g.kgr * 2 * g.d * 2;
    g.off_vsz = g.off_vc + 4 * g.vc_blk * 4;
    g.rec_bytes = g.off_vsz + 4 * g.vsz_blk * 2;
    g.smax = 0;
}

struct KiviDev {
    unsigned char *blk;     // block records [b][h][nkb][rec_bytes]
    __half *Kf;
    __half *Vf;
    int *T, *Tqk, *Tqv;     // device counters [b] (the current one of the cache's two sets)
    unsigned *status;       // anomaly flags
    float *part;            // decode partials [b][h_q][smax][d + 4]: m, l, 2 unused, acc[d]
    unsigned *merge_ticket; // [b][h][4] arrivals of decode CTAs (split-K merge)
    float *ml;              // [b][h_q][2] softmax max and 1 / sum (weights output)
};

// Optional per-token attention-weight output of a decode call: p[i][h][t]
// (row stride ld) receives the raw scores during the decode kernel and the
// softmax weights after the finalizing kernel; mass (may be null, same
// layout) accumulates the weights.
struct ProbsOut {
    float *p;
    float *mass;
    long long ld;
};

// A decode launch that also appends this step's token (kivi_append_decode
// on one-token steps): k, v are the new rows (fp16 [b][h][d]); the kernel
// appends every sequence whose key window is not full (the others were
// appended by a preceding append launch restricted to them) and writes
// those sequences' counters after the append into nxt ([3][b], the other
// counter set).  The decode kernel reads the counters before the append.
struct FusedStep {
    const __half *k, *v;
    int *nxt;
};

struct SeqLens {
    int t[KIVI_MAX_BATCH];
};

// Key-window flush staging: a round covers this many aligned tokens (a
// multiple of max(64, G), so it holds whole groups and whole 64-token
// blocks), as many as keep the fp16 rows within 48 KB of shared memory and
// no more than a window can touch; and the round's shared-memory bytes
// (rows, then scale, zero and reciprocal per group and channel, fp32).
__host__ __device__ __forceinline__ int flush_round_tokens(const KiviGeom &g) {
    const int ch = g.G > 64 ? g.G : 64;
    int n = 48 * 1024 / (g.d * 2) / ch;
    if (n < 1) n = 1;
    const int need = (g.R + ch - 1) / ch + 1;
    return ch * (n < need ? n : need);
}
__host__ __device__ __forceinline__ size_t flush_smem_bytes(const KiviGeom &g) {
    const int r = flush_round_tokens(g);
    return (size_t)r * g.d * 2 + 3 * (size_t)(r / g.G) * g.d * 4;
}

// Every sequence's counters before an append, from the host mirror (kernel
// parameters: the append needs no device read before its row loads).
struct AppendCounters {
    int T[KIVI_MAX_BATCH], Tqk[KIVI_MAX_BATCH], Tqv[KIVI_MAX_BATCH];
    // the sequence of each grid row: sequences that flush their key window
    // first, so that their long CTAs start in the launch's first wave
    int order[KIVI_MAX_BATCH];
};
// Fills ac.order (b sequences, residual length R) from ac's counters.
inline void append_order(AppendCounters &ac, int b, int R) {
    int n = 0;
    for (int i = 0; i < b; ++i)
        if (ac.T[i] - ac.Tqk[i] == R) ac.order[n++] = i;
    for (int i = 0; i < b; ++i)
        if (ac.T[i] - ac.Tqk[i] != R) ac.order[n++] = i;
}

// Counters of one sequence before an append are in range.
__device__ __forceinline__ bool append_counters_ok(const KiviGeom &g, int T, int Tqk, int Tqv) {
    const int R = g.R;
    return T >= 0 && T < g.fcap && Tqk >= 0 && Tqk % R == 0 && T - Tqk >= 0 && T - Tqk <= R && Tqv >= 0 &&
           T - Tqv >= 0 && T - Tqv <= R + 1;
}

// ---- records and slice bases ----------------------------------------------------
__host__ __device__ __forceinline__ size_t rec_off(const KiviGeom &g, int i, int j, int kb) {
    return (((size_t)i * g.h + j) * g.nkb + kb) * (size_t)g.rec_bytes;
}
// key code words of block kb
__host__ __device__ __forceinline__ uint32_t *kc_words(const KiviGeom &g, unsigned char *blk, int i, int j,
                                                       int kb) {
    return reinterpret_cast<uint32_t *>(blk + rec_off(g, i, j, kb));
}
// key scale/zero rows held by record kb: [kgr][2][d]
__host__ __device__ __forceinline__ __half *ksz_rows(const KiviGeom &g, unsigned char *blk, int i, int j,
                                                     int kb) {
    return reinterpret_cast<__half *>(blk + rec_off(g, i, j, kb) + g.off_ksz);
}
// value code words of value block vb
__host__ __device__ __forceinline__ uint32_t *vc_words(const KiviGeom &g, unsigned char *blk, int i, int j,
                                                       int vb) {
    return reinterpret_cast<uint32_t *>(blk + rec_off(g, i, j, vb >> 2) + g.off_vc) + (size_t)(vb & 3) * g.vc_blk;
}
// value scale/zero halves of value block vb: [2][d/G][16]
__host__ __device__ __forceinline__ __half *vsz_halves(const KiviGeom &g, unsigned char *blk, int i, int j,
                                                       int vb) {
    return reinterpret_cast<__half *>(blk + rec_off(g, i, j, vb >> 2) + g.off_vsz) + (size_t)(vb & 3) * g.vsz_blk;
}
// position of channel c inside a key scale / zero row (lane-major, above)
__host__ __device__ __forceinline__ int ksz_pos(int d, int c) {
    return ((c >> 1) & 3) * (d >> 2) + ((c >> 4) << 2) + (((c >> 3) & 1) << 1) + (c & 1);
}
// position of token tau (mod 16) inside a value scale / zero row
__host__ __device__ __forceinline__ int vsz_pos(int tau) {
    return (((tau >> 1) & 3) << 2) + (((tau >> 3) & 1) << 1) + (tau & 1);
}
// scale (sz = 0) or zero (sz = 1) of key group grp, channel c: written to
// every record that holds the group, read from the first
__device__ __forceinline__ void ksz_store(const KiviGeom &g, unsigned char *blk, int i, int j, int grp, int c,
                                          __half s16, __half z16) {
    const int pc = ksz_pos(g.d, c);
    if (g.G <= 64) {
        __half *r = ksz_rows(g, blk, i, j, grp / g.kgr) + (size_t)(grp % g.kgr) * 2 * g.d;
        r[pc] = s16;
        r[g.d + pc] = z16;
    } else {
        for (int k = 0; k < g.G / 64; ++k) {
            __half *r = ksz_rows(g, blk, i, j, grp * (g.G / 64) + k);
            r[pc] = s16;
            r[g.d + pc] = z16;
        }
    }
}
__device__ __forceinline__ __half ksz_load(const KiviGeom &g, unsigned char *blk, int i, int j, int grp, int c,
                                           int sz) {
    const int pc = ksz_pos(g.d, c);
    if (g.G <= 64) return ksz_rows(g, blk, i, j, grp / g.kgr)[((size_t)(grp % g.kgr) * 2 + sz) * g.d + pc];
    return ksz_rows(g, blk, i, j, grp * (g.G / 64))[(size_t)sz * g.d + pc];
}
__host__ __device__ __forceinline__ size_t kf_slice(const KiviGeom &g, int i, int j) {
    return ((size_t)i * g.h + j) * (size_t)g.R * g.d;
}
__host__ __device__ __forceinline__ size_t vf_slice(const KiviGeom &g, int i, int j) {
    return ((size_t)i * g.h + j) * (size_t)(g.R + 1) * g.d;
}

// ---- key word geometry -------------------------------------------------------
// Word wb (0 <= wb < kc_blk) of a key block: lane L = (wb % 128) / 4, lane
// word u = (wb / 128) * 4 + wb % 4, (j, hh, wi) from u; channels c0, c0 + 1;
// slot r of each half is token 8 (wi * cph + r) + (L / 4) of the block.
struct KWord {
    int c0;    // channel of the low half (high half: c0 + 1)
    int g;     // token class: tokens g + 8 * pos
    int pos0;  // position of slot 0 (slot r is position pos0 + r)
};
__device__ __forceinline__ KWord kword_decode(int wb, int kbits) {
    int L = (wb & 127) >> 2;
    int u = (wb >> 7) * 4 + (wb & 3);
    int nwk = kbits >> 1;
    int jh = u / nwk, wi = u - jh * nwk;
    int j = jh >> 1, hh = jh & 1;
    KWord w;
    w.g = L >> 2;
    w.c0 = 16 * j + 8 * hh + 2 * (L & 3);
    w.pos0 = wi * (16 / kbits);
    return w;
}

// ---- value word geometry -------------------------------------------------------
__device__ __forceinline__ int v_cs(const KiviGeom &g) {
    int wl = g.d * g.vbits / 64;   // words per lane per value block
    return wl < 4 ? wl : 4;
}
struct VWord {
    int tt0;   // token (within the 16-token block) of the low half; high half tt0 + 1
    int g;     // channel class: channels g + 8 * ci
    int ci0;   // ci of slot 0 (slot r is ci0 + r)
};
__device__ __forceinline__ VWord vword_decode(int wb, int d, int vbits, int cs) {
    int chunk = wb / (32 * cs);
    int rem = wb - chunk * 32 * cs;
    int L = rem / cs, e = rem - L * cs;
    int u = chunk * cs + e;
    int nwv = d * vbits / 128;
    int p = u / nwv, w = u - p * nwv;
    VWord v;
    v.g = L >> 2;
    v.tt0 = 2 * (L & 3) + 8 * p;
    v.ci0 = w * (16 / vbits);
    return v;
}
// fp16 scale (sz = 0) or zero (sz = 1) of value token tau, channel group gi,
// within its value block's scale/zero halves
__device__ __forceinline__ int vsz_in_block(const KiviGeom &g, int tau, int gi, int sz) {
    return (sz * (g.d / g.G) + gi) * 16 + vsz_pos(tau & 15);
}

// ---- the quantizer (item 1), bit-exact with IEEE fp32 ---------------------------
// Scale: fp32 (max - min) / (2^B - 1) with IEEE division, rounded to fp16
// (nearest, ties to even); zero: min (exact in fp16).  A code is
// round-half-even((x - z) / s) from the stored fp16 s and z, clamped to
// [0, 2^B - 1]; a stored scale of 0 gives code 0.
struct QParams {
    float sf, zf;
    __half s16, z16;
};
__device__ __forceinline__ QParams qparams(float mn, float mx, int bits) {
    QParams p;
    float s32 = __fdiv_rn(__fsub_rn(mx, mn), (float)((1 << bits) - 1));
    p.s16 = __float2half_rn(s32);
    p.z16 = __float2half_rn(mn);
    p.sf = __half2float(p.s16);
    p.zf = __half2float(p.z16);
    return p;
}
__device__ __forceinline__ uint32_t qcode(float x, float sf, float zf, int bits) {
    if (sf == 0.0f) return 0u;
    int q = __float2int_rn(__fdiv_rn(__fsub_rn(x, zf), sf));
    int qmax = (1 << bits) - 1;
    q = q < 0 ? 0 : (q > qmax ? qmax : q);
    return (uint32_t)q;
}

// The same code from a precomputed rs = RN(1 / sf).  (x - z) * rs lies
// within a few ulps of the correctly rounded quotient, so both round to the
// same integer unless they sit next to a rounding tie (k + 1/2); there the
// IEEE division decides.  Bit-identical to qcode, without a division per
// code.
__device__ __forceinline__ uint32_t qcode_rcp(float x, float sf, float zf, float rs, int bits) {
    if (sf == 0.0f) return 0u;
    const float dlt = __fsub_rn(x, zf);
    float q = __fmul_rn(dlt, rs);
    float k = rintf(q);
    // |q - k| close to 1/2: q lies next to a tie
    if (fabsf(q - k) > 0.5f - 1.0e-5f * fmaxf(1.0f, fabsf(q))) k = rintf(__fdiv_rn(dlt, sf));
    const float qmax = (float)((1 << bits) - 1);
    k = fminf(fmaxf(k, 0.0f), qmax);
    return (uint32_t)k;
}

// ---- host-side launchers (kivi_pack.cu, kivi_decode.cu) ----------------------------
struct DecodePlan {
    int ctas;        // persistent CTAs (grid size)
    int qgroups;     // head groups of <= 4 query heads per kv head
    int warps;       // warps per CTA
    int stages;      // shared-memory stages per warp
    int max_parts;   // most partials any (sequence, kv head, head group) receives
    int launches;    // kernel launches per decode call
};

// Work units of one decode call: per sequence i, each of its (kv head, head
// group) pairs counts full[i] fully quantized blocks (one unit each) and its
// remaining blocks (mixed_weight units each); start[] is the prefix over
// sequences of the units of one pair.
struct DecodeUnits {
    long long total;
    int mixed_weight;
    int lead;   // units of a pair ahead of its blocks (no work: they stand for a segment's fixed cost)
    int start[KIVI_MAX_BATCH + 1];
    int full[KIVI_MAX_BATCH];
};

// Sets the calling thread's text for kivi_last_error() (kivi_api.cu).
void kivi_set_last_error(const char *msg);
// Validates a cache shape by kivi_cache_create's rules: returns a
// kivi_status value (0 = supported) and sets the error text (kivi_api.cu).
int kivi_check_shape(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R, int max_tokens);

cudaError_t kivi_launch_prefill(const KiviGeom &g, const KiviDev &dv, const __half *K,
                                const __half *V, const SeqLens &lens, int t_stride,
                                cudaStream_t st);
// The prefill with its causal attention (kivi_prefill_attn.cu): O = the
// attention of Q over K, V (fp16 [b][hq][t_stride][d] and [b][h][t_stride][d])
// and the cache filled as kivi_launch_prefill fills it.  d in {64, 128},
// G <= 64 (cudaErrorInvalidValue otherwise).
cudaError_t kivi_launch_prefill_attn(const KiviGeom &g, const KiviDev &dv, const __half *Q, const __half *K,
                                     const __half *V, __half *O, const SeqLens &lens, int t_stride, int hq,
                                     cudaStream_t st);
// nxt: the other counter set ([3][b]: T, Tqk, Tqv), which receives the
// counters after the append (dv's set is left as it was).
// only_flush: append only the sequences whose key window is full now (the
// others' CTAs return at once; a fused decode launch appends them).
cudaError_t kivi_launch_append(const KiviGeom &g, const KiviDev &dv, const __half *k,
                               const __half *v, const AppendCounters &ac, int *nxt, cudaStream_t st,
                               bool only_flush = false);
// The decode plan and its work units (kivi_decode.cu); fused: the launch
// also appends the step's token (its plan charges the owners' appends).
DecodePlan kivi_plan_decode(const KiviGeom &g, int hq, const int *T, const int *Tqk, const int *Tqv,
                            int num_sms, DecodeUnits *units, bool fused = false);
// partial slots per (sequence, query head) a cache of this shape allocates
int kivi_partial_slots(int b, int h, int num_sms);
// Scores left in po.p by the decode kernel's weights variant -> weights
// (and mass += weights), for rows of up to maxT tokens (kivi_probs.cu).
cudaError_t kivi_launch_probs_finalize(const KiviGeom &g, const KiviDev &dv, int hq, const ProbsOut &po,
                                       int maxT, cudaStream_t st);
// po (may be null): also write the per-token weights (launches the
// finalizing kernel after the decode kernel; maxT = max_i T_i).
// fs (may be null; not with po): the launch also appends the step's token
// (FusedStep).  Its units come from the counters after the append, except
// that a sequence the launch appends counts its value queue before the pop
// (the popped token's block is staged as a window block).
cudaError_t kivi_launch_decode(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                               __half *out, const DecodePlan &plan, const DecodeUnits &units,
                               cudaStream_t st, cudaEvent_t ev0, cudaEvent_t ev1,
                               const ProbsOut *po = nullptr, int maxT = 0, const FusedStep *fs = nullptr);
