/*
 * kivi_oracle.c -- plain, slow CPU oracle for the KIVI quantized KV cache
 * and its decode-attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA
 * library; the only common ground is the written layout specification that
 * both follow (the export format in ko_export below).
 *
 * Source: "Literature audit -- Group 2 (KV-cache compression primary
 * sources)", section 1 "KIVI -- kivi2024", list "Core algorithm
 * (implementation-grade)", items 1-5:
 *   item 1  asymmetric round-to-nearest group quantizer: z = min(X),
 *           s = (max(X) - min(X)) / (2^B - 1), Q = round((X - z) / s),
 *           dequant Q*s + z; B in {2, 4}, separately for keys and values.
 *   item 2  keys per channel, grouped along tokens (one (s, z) per channel
 *           per G consecutive tokens).
 *   item 3  values per token, grouped along channels (d/G groups a token).
 *   item 4  fp16 residual window: prefill keeps the last t mod R keys and
 *           the last R values in fp16; decode quantizes the fp16 key block
 *           whole when it holds R keys; the value queue pops and quantizes
 *           its oldest token when it holds R + 1.
 *   item 5  decode attention = softmax((q K_quant^T || q K_full^T)/sqrt(d))
 *           (V_quant || V_full).
 *
 * Arithmetic: fp32 with IEEE division, rintf (round half to even), no FMA
 * contraction (build with -ffp-contract=off, never -ffast-math).
 *
 * Readings where the pages are silent:
 *   - "round" is round-half-to-even (rintf).
 *   - the scale is stored as fp16 (round-to-nearest-even of the fp32
 *     scale); the zero is min(X), which is exact in fp16.  Codes are
 *     computed from the STORED scale and zero, so dequantisation uses
 *     exactly what is stored.
 *   - codes are clamped to [0, 2^B - 1] (the fp16 scale may round below the
 *     fp32 one); a group whose stored scale is 0 gets all codes 0.
 *   - prefill with t mod R == 0 quantizes all t keys (no fp16 keys).
 *   - maintenance (key flush at R, value pop at R + 1) runs lazily at the
 *     start of the next append, so each step's attention sees the newest
 *     token in fp16; this is the reference order (attend, then quantize).
 *   - GQA: query head i reads kv head i / (h_q / h_kv).
 *   - a sequence with no tokens attends to nothing: its output is 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kivi_oracle.h"

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------- */
/* IEEE 754 binary16 <-> binary32, written from the format's definition.   */
/* ---------------------------------------------------------------------- */

float ko_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    float v;
    if (e == 0) {
        v = ldexpf((float)m, -24);               /* subnormal: m * 2^-24 */
    } else if (e == 31) {
        v = m ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(1024 + m), e - 25);   /* (1 + m/1024) 2^(e-15) */
    }
    return sign ? -v : v;
}

/* shift right by s >= 1 with round-half-to-even */
static uint32_t shr_rne(uint32_t v, int s)
{
    if (s >= 32) return 0;
    uint32_t q = v >> s;
    uint32_t r = v & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (r > half || (r == half && (q & 1u))) q += 1;
    return q;
}

uint16_t ko_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u)                          /* inf or nan */
        return (uint16_t)(sign | (ax > 0x7f800000u ? 0x7e00u : 0x7c00u));
    if (ax == 0) return sign;
    int E = (int)(ax >> 23) - 127;                   /* unbiased exponent */
    uint32_t M = ax & 0x7fffffu;                     /* 24-bit significand */
    if (ax >> 23) M |= 0x800000u; else E = -126;     /* fp32 subnormal */
    if (E >= -14) {
        /* normal fp16 range: keep 11 significant bits */
        uint32_t q = shr_rne(M, 13);
        if (q == 2048u) { q = 1024u; E += 1; }
        if (E > 15) return (uint16_t)(sign | 0x7c00u);   /* overflow */
        return (uint16_t)(sign | ((uint32_t)(E + 15) << 10) | (q - 1024u));
    }
    /* fp16 subnormal: count units of 2^-24; value = M * 2^(E-23) */
    int s = -E - 1;                                  /* >= 14 */
    uint32_t q = shr_rne(M, s);                      /* q <= 1024 */
    return (uint16_t)(sign | q);                     /* 1024 -> 0x0400 */
}

/* ---------------------------------------------------------------------- */
/* Item 1: the asymmetric round-to-nearest group quantizer.                */
/* ---------------------------------------------------------------------- */

void ko_quantize_group(const float *x, int n, int stride, int bits,
                       uint16_t *s_out, uint16_t *z_out,
                       uint8_t *codes, int code_stride)
{
    float mn = x[0], mx = x[0];
    for (int i = 1; i < n; ++i) {
        float v = x[(size_t)i * stride];
        if (v < mn) mn = v;
        if (v > mx) mx = v;
    }
    int qmax = (1 << bits) - 1;
    float s32 = (mx - mn) / (float)qmax;
    uint16_t s16 = ko_f32_to_f16(s32);
    uint16_t z16 = ko_f32_to_f16(mn);
    float sf = ko_f16_to_f32(s16);
    float zf = ko_f16_to_f32(z16);
    for (int i = 0; i < n; ++i) {
        int q = 0;
        if (sf != 0.0f) {
            float v = x[(size_t)i * stride];
            float r = rintf((v - zf) / sf);
            q = r < 0.0f ? 0 : (r > (float)qmax ? qmax : (int)r);
        }
        codes[(size_t)i * code_stride] = (uint8_t)q;
    }
    *s_out = s16;
    *z_out = z16;
}

float ko_dequant(uint8_t code, uint16_t s16, uint16_t z16)
{
    return (float)code * ko_f16_to_f32(s16) + ko_f16_to_f32(z16);
}

/* ---------------------------------------------------------------------- */
/* The cache: plain natural-order arrays.                                  */
/* ---------------------------------------------------------------------- */

struct ko_cache {
    int b, h, d, kbits, vbits, G, R;
    int cap;                     /* capacity in tokens per sequence */
    int capg;                    /* cap rounded up to whole key groups: array stride */
    int *T, *Tqk, *Tqv;          /* per sequence */
    uint8_t *kcode;              /* [b][h][d][capg]   channel-major (item 2) */
    uint16_t *ks, *kz;           /* [b][h][capg/G][d] one pair per channel per G tokens */
    uint8_t *vcode;              /* [b][h][capg][d]   token-major (item 3) */
    uint16_t *vs, *vz;           /* [b][h][capg][d/G] one pair per token per G channels */
    uint16_t *kf;                /* [b][h][R][d]     kf[i] is token Tqk + i */
    uint16_t *vf;                /* [b][h][R+1][d]   vf[i] is token Tqv + i */
};

#define IDX_KCODE(o, i, j, c, t) ((((size_t)(i) * (o)->h + (j)) * (o)->d + (c)) * (o)->capg + (t))
#define IDX_KSZ(o, i, j, g, c)   ((((size_t)(i) * (o)->h + (j)) * ((o)->capg / (o)->G) + (g)) * (o)->d + (c))
#define IDX_VCODE(o, i, j, t, c) ((((size_t)(i) * (o)->h + (j)) * (o)->capg + (t)) * (o)->d + (c))
#define IDX_VSZ(o, i, j, t, g)   ((((size_t)(i) * (o)->h + (j)) * (o)->capg + (t)) * ((o)->d / (o)->G) + (g))
#define IDX_KF(o, i, j, r, c)    ((((size_t)(i) * (o)->h + (j)) * (o)->R + (r)) * (o)->d + (c))
#define IDX_VF(o, i, j, r, c)    ((((size_t)(i) * (o)->h + (j)) * ((o)->R + 1) + (r)) * (o)->d + (c))

int ko_create(int b, int h, int d, int kbits, int vbits, int G, int R, int cap,
              ko_cache **out)
{
    if (b < 1 || h < 1 || d < 1 || G < 1 || R < 1 || cap < 1) return 1;
    if ((kbits != 2 && kbits != 4) || (vbits != 2 && vbits != 4)) return 1;
    if (R % G != 0 || d % G != 0) return 1;        /* item 4 asserts R % G == 0 */
    int capr = ((cap + G - 1) / G) * G;            /* whole key groups */
    ko_cache *o = (ko_cache *)calloc(1, sizeof *o);
    if (!o) return 2;
    o->b = b; o->h = h; o->d = d; o->kbits = kbits; o->vbits = vbits;
    o->G = G; o->R = R; o->cap = cap; o->capg = capr;
    size_t bh = (size_t)b * h;
    o->T = (int *)calloc((size_t)b, sizeof(int));
    o->Tqk = (int *)calloc((size_t)b, sizeof(int));
    o->Tqv = (int *)calloc((size_t)b, sizeof(int));
    o->kcode = (uint8_t *)calloc(bh * d * capr, 1);
    o->ks = (uint16_t *)calloc(bh * (capr / G) * d, 2);
    o->kz = (uint16_t *)calloc(bh * (capr / G) * d, 2);
    o->vcode = (uint8_t *)calloc(bh * capr * d, 1);
    o->vs = (uint16_t *)calloc(bh * capr * (d / G), 2);
    o->vz = (uint16_t *)calloc(bh * capr * (d / G), 2);
    o->kf = (uint16_t *)calloc(bh * R * d, 2);
    o->vf = (uint16_t *)calloc(bh * (R + 1) * d, 2);
    if (!o->T || !o->Tqk || !o->Tqv || !o->kcode || !o->ks || !o->kz ||
        !o->vcode || !o->vs || !o->vz || !o->kf || !o->vf) {
        ko_destroy(o);
        return 2;
    }
    *out = o;
    return 0;
}

void ko_destroy(ko_cache *o)
{
    if (!o) return;
    free(o->T); free(o->Tqk); free(o->Tqv);
    free(o->kcode); free(o->ks); free(o->kz);
    free(o->vcode); free(o->vs); free(o->vz);
    free(o->kf); free(o->vf);
    free(o);
}

void ko_lengths(const ko_cache *o, int *T, int *Tqk, int *Tqv)
{
    for (int i = 0; i < o->b; ++i) {
        T[i] = o->T[i];
        Tqk[i] = o->Tqk[i];
        Tqv[i] = o->Tqv[i];
    }
}

/* Item 2: quantize keys [t0, t0 + n) of one (sequence, kv head), taken from
 * src[(token - t0) * d + c], per channel in groups of G tokens.  t0 and n
 * are multiples of G. */
static void quantize_keys(ko_cache *o, int i, int j, const float *src, int t0, int n)
{
    int d = o->d, G = o->G;
    for (int c = 0; c < d; ++c) {
        for (int g0 = 0; g0 < n; g0 += G) {
            int g = (t0 + g0) / G;
            ko_quantize_group(src + (size_t)g0 * d + c, G, d, o->kbits,
                              &o->ks[IDX_KSZ(o, i, j, g, c)],
                              &o->kz[IDX_KSZ(o, i, j, g, c)],
                              &o->kcode[IDX_KCODE(o, i, j, c, t0 + g0)], 1);
        }
    }
}

/* Item 3: quantize one value token (d floats) per channel group of G. */
static void quantize_value(ko_cache *o, int i, int j, const float *v, int t)
{
    int d = o->d, G = o->G;
    for (int g = 0; g < d / G; ++g) {
        ko_quantize_group(v + (size_t)g * G, G, 1, o->vbits,
                          &o->vs[IDX_VSZ(o, i, j, t, g)],
                          &o->vz[IDX_VSZ(o, i, j, t, g)],
                          &o->vcode[IDX_VCODE(o, i, j, t, (size_t)g * G)], 1);
    }
}

int ko_prefill(ko_cache *o, const uint16_t *K, const uint16_t *V,
               const int *t, int t_stride)
{
    int d = o->d, R = o->R;
    for (int i = 0; i < o->b; ++i)
        if (t[i] < 0 || t[i] > t_stride || t[i] > o->cap) return 1;
    float *buf = (float *)malloc((size_t)(t_stride > 0 ? t_stride : 1) * d * sizeof(float));
    if (!buf) return 2;
    for (int i = 0; i < o->b; ++i) {
        int ti = t[i];
        int nqk = ti - ti % R;                 /* item 4: last t mod R keys stay fp16 */
        int nqv = ti > R ? ti - R : 0;         /* item 4: last R values stay fp16 */
        for (int j = 0; j < o->h; ++j) {
            const uint16_t *Kij = K + ((size_t)i * o->h + j) * t_stride * d;
            const uint16_t *Vij = V + ((size_t)i * o->h + j) * t_stride * d;
            for (size_t e = 0; e < (size_t)nqk * d; ++e) buf[e] = ko_f16_to_f32(Kij[e]);
            quantize_keys(o, i, j, buf, 0, nqk);
            for (int r = 0; r < ti - nqk; ++r)
                memcpy(&o->kf[IDX_KF(o, i, j, r, 0)], Kij + (size_t)(nqk + r) * d, (size_t)d * 2);
            for (int tok = 0; tok < nqv; ++tok) {
                for (int c = 0; c < d; ++c) buf[c] = ko_f16_to_f32(Vij[(size_t)tok * d + c]);
                quantize_value(o, i, j, buf, tok);
            }
            for (int r = 0; r < ti - nqv; ++r)
                memcpy(&o->vf[IDX_VF(o, i, j, r, 0)], Vij + (size_t)(nqv + r) * d, (size_t)d * 2);
        }
        o->T[i] = ti;
        o->Tqk[i] = nqk;
        o->Tqv[i] = nqv;
    }
    free(buf);
    return 0;
}

int ko_append(ko_cache *o, const uint16_t *k, const uint16_t *v)
{
    int d = o->d, R = o->R;
    for (int i = 0; i < o->b; ++i)
        if (o->T[i] + 1 > o->cap) return 3;
    float *buf = (float *)malloc((size_t)R * d * sizeof(float));
    if (!buf) return 2;
    for (int i = 0; i < o->b; ++i) {
        int flush = (o->T[i] - o->Tqk[i]) == R;       /* key buffer reached R */
        int pop = (o->T[i] - o->Tqv[i]) == R + 1;     /* value queue reached R + 1 */
        for (int j = 0; j < o->h; ++j) {
            if (flush) {
                for (size_t e = 0; e < (size_t)R * d; ++e)
                    buf[e] = ko_f16_to_f32(o->kf[IDX_KF(o, i, j, 0, 0) + e]);
                quantize_keys(o, i, j, buf, o->Tqk[i], R);
            }
            if (pop) {
                for (int c = 0; c < d; ++c) buf[c] = ko_f16_to_f32(o->vf[IDX_VF(o, i, j, 0, c)]);
                quantize_value(o, i, j, buf, o->Tqv[i]);
                memmove(&o->vf[IDX_VF(o, i, j, 0, 0)], &o->vf[IDX_VF(o, i, j, 1, 0)],
                        (size_t)R * d * 2);
            }
            int nk = o->T[i] - (o->Tqk[i] + (flush ? R : 0));
            int nv = o->T[i] - (o->Tqv[i] + (pop ? 1 : 0));
            memcpy(&o->kf[IDX_KF(o, i, j, nk, 0)], k + ((size_t)i * o->h + j) * d, (size_t)d * 2);
            memcpy(&o->vf[IDX_VF(o, i, j, nv, 0)], v + ((size_t)i * o->h + j) * d, (size_t)d * 2);
        }
        if (flush) o->Tqk[i] += R;
        if (pop) o->Tqv[i] += 1;
        o->T[i] += 1;
    }
    free(buf);
    return 0;
}

/* Dequantized keys and values of one (sequence, kv head) in token order:
 * quantized tokens first, then the fp16 residual (item 5's concatenation). */
void ko_dequant_kv(const ko_cache *o, int i, int j, float *Khat, float *Vhat)
{
    int d = o->d, G = o->G;
    for (int tok = 0; tok < o->T[i]; ++tok) {
        for (int c = 0; c < d; ++c) {
            float kv, vv;
            if (tok < o->Tqk[i])
                kv = ko_dequant(o->kcode[IDX_KCODE(o, i, j, c, tok)],
                                o->ks[IDX_KSZ(o, i, j, tok / G, c)],
                                o->kz[IDX_KSZ(o, i, j, tok / G, c)]);
            else
                kv = ko_f16_to_f32(o->kf[IDX_KF(o, i, j, tok - o->Tqk[i], c)]);
            if (tok < o->Tqv[i])
                vv = ko_dequant(o->vcode[IDX_VCODE(o, i, j, tok, c)],
                                o->vs[IDX_VSZ(o, i, j, tok, c / G)],
                                o->vz[IDX_VSZ(o, i, j, tok, c / G)]);
            else
                vv = ko_f16_to_f32(o->vf[IDX_VF(o, i, j, tok - o->Tqv[i], c)]);
            Khat[(size_t)tok * d + c] = kv;
            Vhat[(size_t)tok * d + c] = vv;
        }
    }
}

/* Item 5: decode attention for every (sequence, query head).
 * q is fp16 [b][hq][d]; out is fp32 [b][hq][d].  When prow is not NULL it
 * receives the softmax weights themselves, prow[tok] = p[tok] / l for the T
 * tokens (the per-token attention that an accumulated-attention eviction
 * score, H2O's in the same survey's section on token eviction, sums over
 * decode steps). */
static void decode_one(const ko_cache *o, int i, int j, const uint16_t *q,
                       float *outp, float *Khat, float *Vhat, float *p, float *prow)
{
    int d = o->d, T = o->T[i];
    if (T == 0) {
        for (int c = 0; c < d; ++c) outp[c] = 0.0f;
        return;
    }
    ko_dequant_kv(o, i, j, Khat, Vhat);
    float rs = sqrtf((float)d);
    float m = -INFINITY;
    for (int tok = 0; tok < T; ++tok) {
        float dot = 0.0f;
        for (int c = 0; c < d; ++c) dot += ko_f16_to_f32(q[c]) * Khat[(size_t)tok * d + c];
        p[tok] = dot / rs;
        if (p[tok] > m) m = p[tok];
    }
    float l = 0.0f;
    for (int tok = 0; tok < T; ++tok) {
        p[tok] = expf(p[tok] - m);
        l += p[tok];
    }
    for (int c = 0; c < d; ++c) {
        float acc = 0.0f;
        for (int tok = 0; tok < T; ++tok) acc += p[tok] * Vhat[(size_t)tok * d + c];
        outp[c] = acc / l;
    }
    if (prow)
        for (int tok = 0; tok < T; ++tok) prow[tok] = p[tok] / l;
}

int ko_decode(const ko_cache *o, const uint16_t *q, int hq, float *out)
{
    return ko_decode_subset(o, q, hq, out, NULL, 0);
}

static int g_threads = 1;

/* Number of host threads ko_decode_subset spreads its (sequence, query head)
 * pairs over (each pair is computed exactly as in the serial loop). */
int ko_set_threads(int n)
{
#ifdef _OPENMP
    g_threads = n < 1 ? 1 : n;
#else
    (void)n;
    g_threads = 1;
#endif
    return g_threads;
}

/* Decode only the listed (sequence, query head) pairs (pairs[2k], pairs[2k+1]);
 * pairs == NULL means all.  Rows of out that are not listed are untouched. */
int ko_decode_subset(const ko_cache *o, const uint16_t *q, int hq, float *out,
                     const int *pairs, int npairs)
{
    return ko_decode_probs(o, q, hq, out, NULL, 0, pairs, npairs);
}

/* As ko_decode_subset; probs (may be NULL) is fp32 [b][hq][ld] and row
 * (i, qh) of a listed pair receives its T_i softmax weights in [0, T_i);
 * the rest of the row is untouched.  ld >= max T_i. */
int ko_decode_probs(const ko_cache *o, const uint16_t *q, int hq, float *out,
                    float *probs, long long ld, const int *pairs, int npairs)
{
    int d = o->d;
    if (hq < o->h || hq % o->h != 0) return 1;
    if (probs)
        for (int i = 0; i < o->b; ++i) if (o->T[i] > ld) return 1;
    int maxT = 1;
    for (int i = 0; i < o->b; ++i) if (o->T[i] > maxT) maxT = o->T[i];
    int nt = g_threads;
    float **bufs = (float **)calloc((size_t)nt * 3, sizeof(float *));
    if (!bufs) return 2;
    int bad = 0;
    for (int w = 0; w < nt; ++w) {
        bufs[3 * w] = (float *)malloc((size_t)maxT * d * sizeof(float));
        bufs[3 * w + 1] = (float *)malloc((size_t)maxT * d * sizeof(float));
        bufs[3 * w + 2] = (float *)malloc((size_t)maxT * sizeof(float));
        if (!bufs[3 * w] || !bufs[3 * w + 1] || !bufs[3 * w + 2]) bad = 1;
    }
    if (!bad) {
        int grp = hq / o->h;
        int n = pairs ? npairs : o->b * hq;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
#endif
        for (int k = 0; k < n; ++k) {
            int w = 0;
#ifdef _OPENMP
            w = omp_get_thread_num();
#endif
            int i = pairs ? pairs[2 * k] : k / hq;
            int qh = pairs ? pairs[2 * k + 1] : k % hq;
            if (i < 0 || i >= o->b || qh < 0 || qh >= hq) continue;
            decode_one(o, i, qh / grp, q + ((size_t)i * hq + qh) * d,
                       out + ((size_t)i * hq + qh) * d,
                       bufs[3 * w], bufs[3 * w + 1], bufs[3 * w + 2],
                       probs ? probs + ((size_t)i * hq + qh) * (size_t)ld : NULL);
        }
    }
    for (int w = 0; w < nt; ++w) {
        free(bufs[3 * w]); free(bufs[3 * w + 1]); free(bufs[3 * w + 2]);
    }
    free(bufs);
    return bad ? 2 : 0;
}

/* Causal attention of a prompt's queries over its own raw fp16 keys and
 * values: the full-precision prefill attention of "Literature audit --
 * Group 2", section 1 KIVI (its backends list runs the prefill's attention
 * on the unquantized K/V), i.e. core-algorithm item 5's softmax(q K^T /
 * sqrt(d)) V with keys s <= tau only.  In double.  Q: fp16 [b][hq][ts][d];
 * K, V: fp16 [b][h][ts][d] (query head qh reads kv head qh / (hq / h)).
 * With rows == NULL, out is double [b][hq][ts][d] and receives every row
 * tau < t[i] (the others untouched); else out is double [nrows][d] and row
 * k receives (i, qh, tau) = rows[3k..3k+2]. */
static void prefill_row(const uint16_t *q, const uint16_t *K, const uint16_t *V, int tau, int d,
                        double *p, double *outp)
{
    double rs = sqrt((double)d), m = -INFINITY;
    for (int s = 0; s <= tau; ++s) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += (double)ko_f16_to_f32(q[c]) * (double)ko_f16_to_f32(K[(size_t)s * d + c]);
        p[s] = dot / rs;
        if (p[s] > m) m = p[s];
    }
    double l = 0.0;
    for (int s = 0; s <= tau; ++s) {
        p[s] = exp(p[s] - m);
        l += p[s];
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int s = 0; s <= tau; ++s) acc += p[s] * (double)ko_f16_to_f32(V[(size_t)s * d + c]);
        outp[c] = acc / l;
    }
}

int ko_prefill_attn(const uint16_t *Q, const uint16_t *K, const uint16_t *V, const int *t, int b, int hq,
                    int h, int ts, int d, const int *rows, int nrows, double *out)
{
    if (h < 1 || hq < h || hq % h != 0) return 1;
    int maxt = 1;
    for (int i = 0; i < b; ++i) {
        if (t[i] < 0 || t[i] > ts) return 1;
        if (t[i] > maxt) maxt = t[i];
    }
    /* the work: (i, qh, tau) triples */
    long long n = 0;
    int *all = NULL;
    const int compact = rows != NULL;
    if (!rows) {
        for (int i = 0; i < b; ++i) n += (long long)hq * t[i];
        all = (int *)malloc((size_t)(n > 0 ? n : 1) * 3 * sizeof(int));
        if (!all) return 2;
        long long k = 0;
        for (int i = 0; i < b; ++i)
            for (int qh = 0; qh < hq; ++qh)
                for (int tau = 0; tau < t[i]; ++tau) {
                    all[3 * k] = i;
                    all[3 * k + 1] = qh;
                    all[3 * k + 2] = tau;
                    ++k;
                }
        rows = all;
    } else {
        n = nrows;
    }
    int nt = g_threads, bad = 0;
    double **bufs = (double **)calloc((size_t)nt, sizeof(double *));
    if (!bufs) {
        free(all);
        return 2;
    }
    for (int w = 0; w < nt; ++w) {
        bufs[w] = (double *)malloc((size_t)maxt * sizeof(double));
        if (!bufs[w]) bad = 1;
    }
    if (!bad) {
        int grp = hq / h;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nt) schedule(dynamic, 16)
#endif
        for (long long k = 0; k < n; ++k) {
            int w = 0;
#ifdef _OPENMP
            w = omp_get_thread_num();
#endif
            int i = rows[3 * k], qh = rows[3 * k + 1], tau = rows[3 * k + 2];
            if (i < 0 || i >= b || qh < 0 || qh >= hq || tau < 0 || tau >= t[i]) continue;
            size_t kv = ((size_t)i * h + qh / grp) * ts * d;
            size_t qo = (((size_t)i * hq + qh) * ts + tau) * d;
            prefill_row(Q + qo, K + kv, V + kv, tau, d, bufs[w], out + (compact ? (size_t)k * d : qo));
        }
    }
    for (int w = 0; w < nt; ++w) free(bufs[w]);
    free(bufs);
    free(all);
    return bad ? 2 : 0;
}

/* Bulk conversions, for tests and input preparation. */
void ko_f32_to_f16_n(const float *x, uint16_t *y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = ko_f32_to_f16(x[i]);
}

void ko_f16_to_f32_n(const uint16_t *x, float *y, size_t n)
{
    for (size_t i = 0; i < n; ++i) y[i] = ko_f16_to_f32(x[i]);
}

/* Raw natural-order state, for tests. */
void ko_state(const ko_cache *o, uint8_t *kcode, uint16_t *ks, uint16_t *kz,
              uint8_t *vcode, uint16_t *vs, uint16_t *vz, uint16_t *kf, uint16_t *vf)
{
    size_t bh = (size_t)o->b * o->h;
    if (kcode) memcpy(kcode, o->kcode, bh * o->d * o->capg);
    if (ks) memcpy(ks, o->ks, bh * (o->capg / o->G) * o->d * 2);
    if (kz) memcpy(kz, o->kz, bh * (o->capg / o->G) * o->d * 2);
    if (vcode) memcpy(vcode, o->vcode, bh * o->capg * o->d);
    if (vs) memcpy(vs, o->vs, bh * o->capg * (o->d / o->G) * 2);
    if (vz) memcpy(vz, o->vz, bh * o->capg * (o->d / o->G) * 2);
    if (kf) memcpy(kf, o->kf, bh * o->R * o->d * 2);
    if (vf) memcpy(vf, o->vf, bh * (o->R + 1) * o->d * 2);
}

int ko_capacity(const ko_cache *o) { return o->cap; }
int ko_capacity_stride(const ko_cache *o) { return o->capg; }

/* ---------------------------------------------------------------------- */
/* Export to the packed device format (the written layout specification).  */
/* ---------------------------------------------------------------------- */
/*
 * Word and field positions, restated here from the specification:
 *   keys, 64-token blocks: in block kb, lane L = 4g + t and lane word
 *     u = (16-channel step j * 2 + half-step hh) * (Bk/2) + wi, stored at
 *     word (u / 4) * 128 + L * 4 + u % 4 of the block.  Its low 16 bits
 *     hold channel c0 = 16j + 8hh + 2t, its high 16 bits channel c0 + 1;
 *     in each half, slot r (0 <= r < 16/Bk) at bits [r*Bk, r*Bk + Bk) is
 *     token 64 kb + 8 (wi * 16/Bk + r) + g.
 *   key scale/zero: [group][0][channel] = scale, [group][1][channel] = zero.
 *   values, 16-token sub-blocks: in sub-block vb, lane word u = p * nwv + w
 *     (nwv = d*Bv/128), stored at word (u / cs) * 32 * cs + L * cs + u % cs
 *     with cs = min(4, d*Bv/64).  Low half: token 16 vb + 2t + 8p, high
 *     half: that token + 1; slot r at bits [r*Bv, r*Bv + Bv) is channel
 *     8 (w * 16/Bv + r) + g.
 *   value scale/zero: [sub-block][0][channel group][token % 16] = scale,
 *     [.][1][.][.] = zero.
 *   fp16 residual: key token tau at slot tau % R, value token at tau % (R+1).
 * Bits, words and entries for tokens not yet quantized are zero.
 */
static int div_up(int a, int b) { return (a + b - 1) / b; }

/* The packed format needs G a power of two in [16, 128], d a multiple of 64
 * dividing into whole groups, and sizes its arrays for the capacity rounded
 * up to a multiple of max(64, G) tokens. */
int ko_export_supported(const ko_cache *o)
{
    int G = o->G, d = o->d;
    if (G != 16 && G != 32 && G != 64 && G != 128) return 0;
    if (d % 64 != 0 || d > 256 || d % G != 0) return 0;
    return 1;
}

static int format_cap(const ko_cache *o)
{
    int q = o->G > 64 ? o->G : 64;
    return div_up(o->cap, q) * q;
}

void ko_export_sizes(const ko_cache *o, size_t *n_kc, size_t *n_ksz, size_t *n_vc,
                     size_t *n_vsz, size_t *n_kf, size_t *n_vf)
{
    size_t bh = (size_t)o->b * o->h;
    int d = o->d, fc = format_cap(o);
    *n_kc = bh * (size_t)(fc / 64) * (size_t)(2 * d * o->kbits);       /* uint32 words */
    *n_ksz = bh * (size_t)(fc / o->G) * (size_t)(2 * d);               /* fp16 */
    *n_vc = bh * (size_t)(fc / 16) * (size_t)(d * o->vbits / 2);       /* uint32 words */
    *n_vsz = bh * (size_t)(fc / 16) * (size_t)(2 * (d / o->G) * 16);   /* fp16 */
    *n_kf = bh * (size_t)o->R * d;
    *n_vf = bh * (size_t)(o->R + 1) * d;
}

int ko_export(const ko_cache *o, uint32_t *Kc, uint16_t *Ksz, uint32_t *Vc,
              uint16_t *Vsz, uint16_t *Kf, uint16_t *Vf)
{
    if (!ko_export_supported(o)) return 1;
    int d = o->d, G = o->G, R = o->R, Bk = o->kbits, Bv = o->vbits;
    int fc = format_cap(o);
    int nkb = fc / 64, nkg = fc / G, nvb = fc / 16;
    size_t kc_blk = (size_t)2 * d * Bk, vc_blk = (size_t)d * Bv / 2;
    int cph_k = 16 / Bk, cph_v = 16 / Bv;
    int nwv = d * Bv / 128, cs = d * Bv / 64 < 4 ? d * Bv / 64 : 4;
    size_t nkc, nksz, nvc, nvsz, nkf, nvf;
    ko_export_sizes(o, &nkc, &nksz, &nvc, &nvsz, &nkf, &nvf);
    memset(Kc, 0, nkc * 4); memset(Ksz, 0, nksz * 2);
    memset(Vc, 0, nvc * 4); memset(Vsz, 0, nvsz * 2);
    memset(Kf, 0, nkf * 2); memset(Vf, 0, nvf * 2);
    for (int i = 0; i < o->b; ++i) {
        for (int j = 0; j < o->h; ++j) {
            size_t bhi = (size_t)i * o->h + j;
            /* key codes: visit every (channel, token) and place its bits */
            for (int tok = 0; tok < o->Tqk[i]; ++tok) {
                int kb = tok / 64, pos = (tok % 64) / 8, g = tok % 8;
                int wi = pos / cph_k, r = pos % cph_k;
                for (int c = 0; c < d; ++c) {
                    int jj = c / 16, hh = (c % 16) / 8, t = (c % 8) / 2, hi = c % 2;
                    int L = 4 * g + t;
                    int u = (jj * 2 + hh) * (Bk / 2) + wi;
                    size_t w = bhi * nkb * kc_blk + (size_t)kb * kc_blk +
                               (size_t)(u / 4) * 128 + (size_t)L * 4 + u % 4;
                    uint32_t code = o->kcode[IDX_KCODE(o, i, j, c, tok)];
                    Kc[w] |= code << (16 * hi + r * Bk);
                }
            }
            for (int g = 0; g < o->Tqk[i] / G; ++g) {
                for (int c = 0; c < d; ++c) {
                    size_t base = (bhi * nkg + g) * 2 * d;
                    Ksz[base + c] = o->ks[IDX_KSZ(o, i, j, g, c)];
                    Ksz[base + d + c] = o->kz[IDX_KSZ(o, i, j, g, c)];
                }
            }
            /* value codes */
            for (int tok = 0; tok < o->Tqv[i]; ++tok) {
                int vb = tok / 16, tt = tok % 16;
                int p = tt / 8, t = (tt % 8) / 2, hi = tt % 2;
                for (int c = 0; c < d; ++c) {
                    int g = c % 8, ci = c / 8;
                    int w = ci / cph_v, r = ci % cph_v;
                    int L = 4 * g + t;
                    int u = p * nwv + w;
                    size_t wd = bhi * nvb * vc_blk + (size_t)vb * vc_blk +
                                (size_t)(u / cs) * 32 * cs + (size_t)L * cs + u % cs;
                    uint32_t code = o->vcode[IDX_VCODE(o, i, j, tok, c)];
                    Vc[wd] |= code << (16 * hi + r * Bv);
                }
                for (int gi = 0; gi < d / G; ++gi) {
                    size_t base = (bhi * nvb + vb) * 2 * (d / G) * 16;
                    Vsz[base + (size_t)gi * 16 + tt] = o->vs[IDX_VSZ(o, i, j, tok, gi)];
                    Vsz[base + (size_t)(d / G + gi) * 16 + tt] = o->vz[IDX_VSZ(o, i, j, tok, gi)];
                }
            }
            /* fp16 residual windows at their ring slots */
            for (int tok = o->Tqk[i]; tok < o->T[i]; ++tok)
                memcpy(&Kf[(bhi * R + tok % R) * d], &o->kf[IDX_KF(o, i, j, tok - o->Tqk[i], 0)],
                       (size_t)d * 2);
            for (int tok = o->Tqv[i]; tok < o->T[i]; ++tok)
                memcpy(&Vf[(bhi * (R + 1) + tok % (R + 1)) * d],
                       &o->vf[IDX_VF(o, i, j, tok - o->Tqv[i], 0)], (size_t)d * 2);
        }
    }
    return 0;
}
