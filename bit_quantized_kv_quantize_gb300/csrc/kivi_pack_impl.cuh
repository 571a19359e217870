// kivi_pack_impl.cuh -- the quantize-and-pack arithmetic of one staged tile
// of keys or values, shared by the prefill pack kernels (kivi_pack.cu) and
// the prefill attention kernel's epilogue (kivi_prefill_attn.cu).
//
// Method: "Literature audit -- Group 2", section 1 KIVI, core algorithm
// items 1-3 (the quantizer; per-channel key groups of G tokens; per-token
// value groups of G channels).
#pragma once
#include "kivi_internal.cuh"

namespace {


// Row stride of a staged key tile: D + 32 halves (a multiple of 32 words
// plus 16), so that the two halves of a warp, which read rows one apart in
// pack_key_tile's scans and word reads, fall in different banks.
__host__ __device__ constexpr int key_xsd(int D) { return D + 32; }

// ---------------------------------------------------------------------------
// Codes two at a time.  The quantizer (item 1) is round-half-even((x - z)
// / s) clamped to [0, 2^B - 1] with IEEE fp32 division, s and z the group's
// stored fp16 scale and zero.  The fast path computes, for the two values
// of a word slot at once (packed fp32x2 instructions):
//   d = x - z (fp32, one rounding: a mixed fp16 + fp32 add), q = d * rs
//   with rs = RN(1 / s) (0 when s is 0), and round(q) by adding 1.5 * 2^23
//   (round to nearest, ties to even: the integer lands in the low mantissa
//   bits, which a multiply-add then places in its field).
// q >= 0 since z is the group's min, and with a normal fp16 scale a
// member's q stays below (2^B - 1)(1 + 2^-11), so no clamp is needed (a
// tile holding a subnormal scale takes the exact path throughout).  q lies
// within a few ulps of the correctly rounded quotient d / s, so both round
// alike unless q sits next to a tie (k + 1/2): a word with any such value
// is redone with the IEEE division.  Bit-exact with the definition.
// ---------------------------------------------------------------------------
typedef unsigned long long u64;

__device__ __forceinline__ u64 f2p(float a, float b) {
    return (u64)__float_as_uint(a) | ((u64)__float_as_uint(b) << 32);
}
__device__ __forceinline__ float f2lo(u64 v) { return __uint_as_float((unsigned)v); }
__device__ __forceinline__ float f2hi(u64 v) { return __uint_as_float((unsigned)(v >> 32)); }
__device__ __forceinline__ u64 f2sub(u64 a, u64 b) {
    u64 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 f2add(u64 a, u64 b) {
    u64 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 f2mul(u64 a, u64 b) {
    u64 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// the code from the IEEE quotient d / s itself (the quantizer's own
// definition), for the rare word next to a rounding tie
template <int BITS>
__device__ __forceinline__ uint32_t exact_code(float d, float sf) {
    if (sf == 0.0f) return 0u;
    float k = rintf(__fdiv_rn(d, sf));
    k = fminf(fmaxf(k, 0.0f), (float)((1 << BITS) - 1));
    return (uint32_t)k;
}
// distance from 1/2 below which a product quotient may round unlike the
// IEEE quotient: a member's quotient is below 2 * 2^B, so 1e-5 * 2^B covers
// the few ulps between them
template <int BITS>
__host__ __device__ constexpr float kTie() { return 0.5f - 1.0e-5f * (float)(1 << BITS); }
// a nonzero scale below fp16's normal range (its rounding may push a
// member's quotient past 2^B - 1 / 2)
__device__ __forceinline__ int subnormal_scale(float sf) { return sf != 0.0f && sf < 6.103515625e-05f; }

// d = x - z of two fp16 values x (the halves of xh) against their groups'
// fp32 zeros nz = -z: one mixed-precision add each (fp16 operand, fp32
// result, one rounding), so x needs no separate conversion
__device__ __forceinline__ u64 sub_zero2(uint32_t xh, float nz0, float nz1) {
    float d0, d1;
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "r"(xh), "f"(nz0), "f"(nz1));
    return f2p(d0, d1);
}

constexpr float kMagic = 12582912.0f;     // 1.5 * 2^23: adding it rounds to an integer
constexpr uint32_t kMagicBits = 0x4B400000u;   // its bit pattern (the integer sits in the low bits)

// A word is built as sum_s (bits of round(q_s) + 1.5 * 2^23) << s plus this
// constant, which cancels the magic's bits: each code lands in its field
// with one multiply-add (no mask, shift and or).  s runs over the fields
// 16 h + r BITS (h < 2, r < 16 / BITS).
template <int BITS>
__host__ __device__ constexpr uint32_t word_bias() {
    uint32_t w = 0;
    for (int h = 0; h < 2; ++h)
        for (int r = 0; r < 16 / BITS; ++r) w -= kMagicBits << (16 * h + r * BITS);
    return w;
}
__device__ __forceinline__ uint32_t mad_u32(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// Fast path for the two values of a slot (differences d from their zeros,
// their groups' rs): adds their rounded quotients into the word at fields
// s0, s1 and returns the larger distance |q - round(q)|; the caller redoes
// the word exactly when that distance is next to 1/2.  No clamp: with a
// normal fp16 scale a member's quotient stays below (2^B - 1)(1 + 2^-11),
// so the rounded code is at most 2^B - 1 (a tile with a subnormal scale
// takes the exact path throughout).
__device__ __forceinline__ float add_codes2(u64 d, u64 rs, int s0, int s1, uint32_t &word) {
    const u64 q = f2mul(d, rs);
    const u64 M2 = f2p(kMagic, kMagic);
    const u64 t = f2add(q, M2);
    const u64 r = f2sub(q, f2sub(t, M2));   // q - round(q)
    word = mad_u32((uint32_t)t, 1u << s0, word);
    word = mad_u32((uint32_t)(t >> 32), 1u << s1, word);
    return fmaxf(fabsf(f2lo(r)), fabsf(f2hi(r)));
}

__device__ __forceinline__ __half2 u2h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// 16-byte asynchronous global -> shared copy; zero-filled when !valid (src
// must still be a valid address)
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// scale, zero and RN(1 / scale) of a group from its fp16 min and max
__device__ __forceinline__ void group_params(__half mn, __half mx, int bits, __half &s16, __half &z16, float &sf,
                                             float &zf, float &rs) {
    const QParams p = qparams(__half2float(mn), __half2float(mx), bits);
    s16 = p.s16;
    z16 = p.z16;
    sf = p.sf;
    zf = p.zf;
    rs = p.sf == 0.0f ? 0.0f : __frcp_rn(p.sf);
}

// The exact word, out of line (taken rarely; kept out of the fast loop).
// Key word: slot r of both halves is token (xw's row) + 8 r, channels c0,
// c0 + 1; fw points at the word's first group's (s, -z, rs) rows at c0.
template <int KBITS, int G, int D>
__device__ __noinline__ uint32_t exact_key_word(const __half *xw, const float *fw) {
    constexpr int cph = 16 / KBITS;
    constexpr int RPG = G / 8 < cph ? G / 8 : cph;
    uint32_t word = 0;
#pragma unroll
    for (int r = 0; r < cph; ++r) {
        const float *f = fw + (size_t)(r / RPG) * 3 * D;
        const float2 s2 = *reinterpret_cast<const float2 *>(f);
        const float2 nz = *reinterpret_cast<const float2 *>(f + D);
        const uint32_t xh = *reinterpret_cast<const uint32_t *>(xw + (size_t)8 * r * key_xsd(D));
        const u64 dd = sub_zero2(xh, nz.x, nz.y);
        word |= (exact_code<KBITS>(f2lo(dd), s2.x) << (r * KBITS)) |
                (exact_code<KBITS>(f2hi(dd), s2.y) << (16 + r * KBITS));
    }
    return word;
}
// Value word: slot r holds channel 8 (ci0 + r) + g of the pair row xr; fp
// points at the pair's (s, -z, rs) of the word's first group.
template <int VBITS, int G, int D>
__device__ __noinline__ uint32_t exact_value_word(const uint32_t *xr, const float2 *fp, int ci0, int g) {
    constexpr int cph = 16 / VBITS, ngi = D / G;
    uint32_t word = 0;
#pragma unroll
    for (int r = 0; r < cph; ++r) {
        const int c = 8 * (ci0 + r) + g;
        const float2 s2 = fp[(8 * r) / G], nz = fp[ngi + (8 * r) / G];
        const u64 dd = sub_zero2(xr[c], nz.x, nz.y);
        word |= (exact_code<VBITS>(f2lo(dd), s2.x) << (r * VBITS)) |
                (exact_code<VBITS>(f2hi(dd), s2.y) << (16 + r * VBITS));
    }
    return word;
}

// ---------------------------------------------------------------------------
// Keys of one tile of TB = max(64, G) tokens (item 2: per-channel groups of
// G tokens along the tokens), staged in shared memory as rows
// xs[TB][key_xsd(D)] fp16, rows past ntok (a multiple of G) zero.  rec: the
// cache record of the tile's first 64-token block (records rec_bytes
// apart); sfz: shared scratch [TB / G][3][D] fp32.  Writes the groups'
// scale and zero rows and the blocks' code words.  Called by every thread
// of the CTA (any multiple of 32 threads).
// ---------------------------------------------------------------------------

template <int KBITS, int G, int D>
__device__ __forceinline__ void pack_key_tile(const __half *xs, float *sfz, int ntok, unsigned char *rec,
                                              int rec_bytes, int off_ksz) {
    constexpr int TB = G > KIVI_KBLK ? G : KIVI_KBLK;
    constexpr int NG = TB / G, xsd = key_xsd(D), KGR = G >= KIVI_KBLK ? 1 : KIVI_KBLK / G;
    const int ngr = ntok / G;

    // Scale and zero per (group, channel): item e is (group gr, channel
    // pair c, c + 1, token parity th); lanes l and l ^ 16 scan the even and
    // odd tokens of one group and channel pair (the min / max of fp16
    // values is exact in fp16), then lane th takes channel c + th.
    int slow = 0;
#pragma unroll 2
    for (int e = threadIdx.x; e < NG * D; e += blockDim.x) {
        const int th = (e >> 4) & 1;
        const int cp = (e & 15) | ((e >> 5) << 4);
        const int gr = cp / (D / 2), c = 2 * (cp % (D / 2));
        const __half2 *col = reinterpret_cast<const __half2 *>(xs + (size_t)(gr * G + th) * xsd + c);
        __half2 mn = col[0], mx = mn;
#pragma unroll 8
        for (int k = 1; k < G / 2; ++k) {
            const __half2 x = col[(size_t)k * xsd];   // row gr G + 2 k + th
            mn = __hmin2(mn, x);
            mx = __hmax2(mx, x);
        }
        mn = __hmin2(mn, __shfl_xor_sync(0xffffffffu, mn, 16));
        mx = __hmax2(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const int ch = c + th;
        float sf = 0.f, zf = 0.f, rs = 0.f;
        if (gr < ngr) {
            __half s16, z16;
            group_params(th ? __high2half(mn) : __low2half(mn), th ? __high2half(mx) : __low2half(mx), KBITS, s16,
                         z16, sf, zf, rs);
            // the group's scale / zero rows: row gr % KGR of the record of
            // its block (G > 64: in every record the group spans)
            const int pc = ksz_pos(D, ch);
#pragma unroll
            for (int k = 0; k < (G > KIVI_KBLK ? G / KIVI_KBLK : 1); ++k) {
                __half *r = reinterpret_cast<__half *>(rec + (size_t)(gr / KGR + k) * rec_bytes + off_ksz) +
                            (size_t)(gr % KGR) * 2 * D;
                r[pc] = s16;
                r[D + pc] = z16;
            }
        }
        sfz[(gr * 3 + 0) * D + ch] = sf;
        sfz[(gr * 3 + 1) * D + ch] = -zf;
        sfz[(gr * 3 + 2) * D + ch] = rs;
        slow |= subnormal_scale(sf);
    }
    // a subnormal scale anywhere: the exact path for the whole tile
    slow = __syncthreads_or(slow);

    // packed words of every 64-token block that starts inside the tile
    constexpr int cph = 16 / KBITS;
    // a word's slots span 8 cph tokens: this many groups (slot r is in
    // group r / RPG of the word's first)
    constexpr int RPG = G / 8 < cph ? G / 8 : cph;
    constexpr int GW = cph / RPG;
    constexpr int kc_blk = 2 * D * KBITS;
    const int nblk = (ntok + KIVI_KBLK - 1) / KIVI_KBLK;
    // words are independent: unrolled so that a thread keeps several in flight
#pragma unroll 4
    for (int e = threadIdx.x; e < nblk * kc_blk; e += blockDim.x) {
        const int kbl = e / kc_blk, wb = e - kbl * kc_blk;
        const KWord kw = kword_decode(wb, KBITS);
        // Slot r holds token trow + 8 r + g (g < 8).  trow is a multiple of
        // 32, and of G whenever G <= 32; for G >= 64 the word's tokens lie
        // in one group.  So slot r's group is trow / G + r / RPG.
        const int trow = kbl * KIVI_KBLK + 8 * kw.pos0;
        const float *fw = sfz + (size_t)(trow / G) * 3 * D + kw.c0;
        float2 nz[GW];
        u64 rr[GW];
#pragma unroll
        for (int k = 0; k < GW; ++k) {
            const float *f = fw + (size_t)k * 3 * D;
            const float2 r2 = *reinterpret_cast<const float2 *>(f + 2 * D);
            nz[k] = *reinterpret_cast<const float2 *>(f + D);
            rr[k] = f2p(r2.x, r2.y);
        }
        // slot r of both halves: token trow + 8 r + g, channels c0 and c0 + 1
        const __half *xw = xs + (size_t)(trow + kw.g) * xsd + kw.c0;
        uint32_t word = word_bias<KBITS>();
        float rmax = 0.f;
        if (!slow) {
#pragma unroll
            for (int r = 0; r < cph; ++r) {
                const uint32_t xh = *reinterpret_cast<const uint32_t *>(xw + (size_t)8 * r * xsd);
                rmax = fmaxf(rmax, add_codes2(sub_zero2(xh, nz[r / RPG].x, nz[r / RPG].y), rr[r / RPG],
                                              r * KBITS, 16 + r * KBITS, word));
            }
        }
        if (slow || rmax > kTie<KBITS>())   // next to a tie: the IEEE quotients decide
            word = exact_key_word<KBITS, G, D>(xw, fw);
        reinterpret_cast<uint32_t *>(rec + (size_t)kbl * rec_bytes)[wb] = word;
    }
}

// ---------------------------------------------------------------------------
// Values of one 64-token tile (item 3: per-token groups of G channels),
// staged in shared memory with token pairs interleaved: xs2[32][D + 4]
// 32-bit words, element (pair k, channel c) the half2 of tokens 2k and
// 2k + 1 at channel c, tokens past ntok zero.  tok0: the tile's first
// token (a multiple of 64) in sequence i, kv head j.  sfz: shared scratch
// [32][3][D / G] float2.  Writes the tokens' scale and zero halves and the
// value blocks' code words; tokens past ntok get zero scale, zero and
// codes.  Called by every thread of the CTA (any multiple of 32 threads).
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int value_ps(int D) { return D + 4; }

template <int VBITS, int G, int D>
__device__ __forceinline__ void pack_value_tile(const uint32_t *xs2, float2 *sfz, int ntok, int tok0,
                                                const KiviGeom &g, const KiviDev &dv, int i, int j) {
    constexpr int ngi = D / G, ps = value_ps(D);
    // scale and zero per (token, channel group), both tokens of a pair at once
    const int nvblk = (ntok + KIVI_VBLK - 1) / KIVI_VBLK;   // value blocks touched
    int slow = 0;
#pragma unroll 2
    for (int e = threadIdx.x; e < nvblk * 8 * ngi; e += blockDim.x) {
        const int k = e / ngi, gi = e - k * ngi;
        const int tau = tok0 + 2 * k;   // even: the pair's halves are adjacent in a scale row
        __half2 s16 = __floats2half2_rn(0.f, 0.f), z16 = s16;
        float2 sf = make_float2(0.f, 0.f), zf = sf, rs = sf;
        if (2 * k < ntok) {
            // fp16 min / max (exact); the scan starts at a pair-dependent
            // offset so that the warp's threads read different banks
            const uint32_t *x = xs2 + (size_t)k * ps + gi * G;
            const int rot = (k + 8 * gi) & (G - 1);
            __half2 mn = u2h2(x[rot]), mx = mn;
#pragma unroll 8
            for (int c = 1; c < G; ++c) {
                const __half2 v = u2h2(x[(c + rot) & (G - 1)]);
                mn = __hmin2(mn, v);
                mx = __hmax2(mx, v);
            }
            __half s0, z0, s1, z1;
            group_params(__low2half(mn), __low2half(mx), VBITS, s0, z0, sf.x, zf.x, rs.x);
            if (2 * k + 1 < ntok) group_params(__high2half(mn), __high2half(mx), VBITS, s1, z1, sf.y, zf.y, rs.y);
            else s1 = z1 = __float2half_rn(0.f);
            s16 = __halves2half2(s0, s1);
            z16 = __halves2half2(z0, z1);
        }
        __half *vsz = vsz_halves(g, dv.blk, i, j, tau >> 4);
        *reinterpret_cast<__half2 *>(vsz + vsz_in_block(g, tau, gi, 0)) = s16;   // tokens past ntok: zero
        *reinterpret_cast<__half2 *>(vsz + vsz_in_block(g, tau, gi, 1)) = z16;
        sfz[(k * 3 + 0) * ngi + gi] = sf;
        sfz[(k * 3 + 1) * ngi + gi] = make_float2(-zf.x, -zf.y);   // -z
        sfz[(k * 3 + 2) * ngi + gi] = rs;
        slow |= subnormal_scale(sf.x) | subnormal_scale(sf.y);
    }
    slow = __syncthreads_or(slow);

    constexpr int cs = D * VBITS / 64 < 4 ? D * VBITS / 64 : 4;
    constexpr int cph = 16 / VBITS;
    constexpr int vc_blk = D * VBITS / 2;
    // words are independent: unrolled so that a thread keeps several in flight
#pragma unroll 4
    for (int e = threadIdx.x; e < nvblk * vc_blk; e += blockDim.x) {
        const int vbl = e / vc_blk, wb = e - vbl * vc_blk;
        const VWord vw = vword_decode(wb, D, VBITS, cs);
        // Slot r holds channel 8 (ci0 + r) + g (g < 8) of tokens tt0, tt0 + 1
        // (one pair); 8 ci0 is a multiple of 32, and of G whenever G <= 32;
        // for G >= 64 the word's channels lie in one group.  So slot r's
        // group is 8 ci0 / G + (8 r) / G.
        const int k = (vbl * KIVI_VBLK + vw.tt0) >> 1;
        const int gi0 = 8 * vw.ci0 / G;
        const uint32_t *xr = xs2 + (size_t)k * ps;
        const float2 *fp = sfz + (size_t)k * 3 * ngi + gi0;
        uint32_t word = word_bias<VBITS>();
        float rmax = 0.f;
        if (!slow) {
#pragma unroll
            for (int r = 0; r < cph; ++r) {
                const int c = 8 * (vw.ci0 + r) + vw.g;
                const float2 nz = fp[ngi + (8 * r) / G], r2 = fp[2 * ngi + (8 * r) / G];
                rmax = fmaxf(rmax, add_codes2(sub_zero2(xr[c], nz.x, nz.y), f2p(r2.x, r2.y), r * VBITS,
                                              16 + r * VBITS, word));
            }
        }
        if (slow || rmax > kTie<VBITS>())   // next to a tie: the IEEE quotients decide
            word = exact_value_word<VBITS, G, D>(xr, fp, vw.ci0, vw.g);
        vc_words(g, dv.blk, i, j, tok0 / KIVI_VBLK + vbl)[wb] = word;
    }
}

}  // namespace
