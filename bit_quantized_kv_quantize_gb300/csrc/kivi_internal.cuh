// kivi_internal.cuh -- geometry, device-array bundle and layout index math
// shared by the kernels and the host manager of libkivi.
//
// The packed format is the one the C header documents (kivi_cache_export):
// keys in 64-token blocks, each uint32 word carrying two channels, each
// 16-bit half packing one channel along tokens (tokens interleaved by 8, so
// one lane's word feeds the A operand of an m16n8k16 MMA directly); values
// in 16-token blocks, each word carrying two tokens, each half packing one
// token along channels (channels interleaved by 8).  Scale and zero are fp16.
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
    int smax;     // decode partials the buffer holds per (sequence, query head)
};

struct KiviDev {
    uint32_t *Kc;
    __half *Ksz;
    uint32_t *Vc;
    __half *Vsz;
    __half *Kf;
    __half *Vf;
    int *T, *Tqk, *Tqv;     // device counters [b]
    unsigned *ticket;       // [b] arrivals of the append kernel's CTAs
    unsigned *status;       // anomaly flags
    float *part;            // decode partials [b][h * KIVI_MAX_QPERKV][smax][d + 2]
    unsigned *merge_ticket; // [b][h] arrivals of decode CTAs (split-K merge)
};

struct SeqLens {
    int t[KIVI_MAX_BATCH];
};

// ---- slice bases -----------------------------------------------------------
__host__ __device__ __forceinline__ size_t kc_slice(const KiviGeom &g, int i, int j) {
    return ((size_t)i * g.h + j) * (size_t)g.nkb * g.kc_blk;
}
__host__ __device__ __forceinline__ size_t ksz_slice(const KiviGeom &g, int i, int j) {
    return ((size_t)i * g.h + j) * (size_t)g.nkg * 2 * g.d;
}
__host__ __device__ __forceinline__ size_t vc_slice(const KiviGeom &g, int i, int j) {
    return ((size_t)i * g.h + j) * (size_t)g.nvb * g.vc_blk;
}
__host__ __device__ __forceinline__ size_t vsz_slice(const KiviGeom &g, int i, int j) {
    return ((size_t)i * g.h + j) * (size_t)g.nvb * g.vsz_blk;
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
// word index inside the slice and bit shift of (channel c, token tau)
__device__ __forceinline__ size_t kc_locate(const KiviGeom &g, int c, int tau, int *shift) {
    int kb = tau >> 6, pos = (tau & 63) >> 3, gg = tau & 7;
    int cph = 16 / g.kbits, nwk = g.kbits >> 1;
    int wi = pos / cph, r = pos - wi * cph;
    int j = c >> 4, hh = (c >> 3) & 1, t = (c & 7) >> 1, hi = c & 1;
    int L = 4 * gg + t;
    int u = (2 * j + hh) * nwk + wi;
    *shift = 16 * hi + r * g.kbits;
    return (size_t)kb * g.kc_blk + (size_t)(u >> 2) * 128 + 4 * L + (u & 3);
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
__device__ __forceinline__ size_t vc_locate(const KiviGeom &g, int c, int tau, int *shift) {
    int vb = tau >> 4, tt = tau & 15;
    int p = tt >> 3, t = (tt & 7) >> 1, hi = tt & 1;
    int gg = c & 7, ci = c >> 3;
    int cph = 16 / g.vbits;
    int w = ci / cph, r = ci - w * cph;
    int nwv = g.d * g.vbits / 128, cs = v_cs(g);
    int L = 4 * gg + t;
    int u = p * nwv + w;
    *shift = 16 * hi + r * g.vbits;
    return (size_t)vb * g.vc_blk + (size_t)(u / cs) * 32 * cs + (size_t)L * cs + (u % cs);
}
// fp16 scale (sz = 0) or zero (sz = 1) of value token tau, channel group gi
__device__ __forceinline__ size_t vsz_locate(const KiviGeom &g, int tau, int gi, int sz) {
    return (size_t)(tau >> 4) * g.vsz_blk + ((size_t)sz * (g.d / g.G) + gi) * 16 + (tau & 15);
}
__device__ __forceinline__ size_t ksz_locate(const KiviGeom &g, int grp, int c, int sz) {
    return ((size_t)grp * 2 + sz) * g.d + c;
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
    int start[KIVI_MAX_BATCH + 1];
    int full[KIVI_MAX_BATCH];
};

// Sets the calling thread's text for kivi_last_error() (kivi_api.cu).
void kivi_set_last_error(const char *msg);

cudaError_t kivi_launch_prefill(const KiviGeom &g, const KiviDev &dv, const __half *K,
                                const __half *V, const SeqLens &lens, int t_stride,
                                cudaStream_t st);
cudaError_t kivi_launch_append(const KiviGeom &g, const KiviDev &dv, const __half *k,
                               const __half *v, cudaStream_t st);
DecodePlan kivi_plan_decode(const KiviGeom &g, int hq, const int *T, const int *Tqk, const int *Tqv,
                            int num_sms, DecodeUnits *units);
// partial slots per (sequence, query head) a cache of this shape allocates
int kivi_partial_slots(int b, int h, int num_sms);
cudaError_t kivi_launch_decode(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                               __half *out, const DecodePlan &plan, const DecodeUnits &units,
                               cudaStream_t st, cudaEvent_t ev0, cudaEvent_t ev1);
