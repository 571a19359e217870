// kivi_pack.cu -- quantize-and-pack kernels: prefill (keys, values, fp16
// residual fill) and the per-token append with its lazy maintenance.
//
// Method: "Literature audit -- Group 2", section 1 KIVI, core algorithm
// items 1-4 (quantizer, per-channel key groups along tokens, per-token value
// groups along channels, fp16 residual window with the key-block flush at R
// and the value-queue pop at R + 1).
//
// All kernels stream HBM once: a CTA stages its token tile in shared memory,
// computes per-group min/max, then writes whole packed words (coalesced:
// consecutive threads write consecutive words).
#include "kivi_append_impl.cuh"

namespace {

__device__ __forceinline__ void flag(unsigned *status, unsigned f) { atomicOr(status, f); }

// Shared-memory tiles keep each token row padded by 16 bytes, so reads of
// one channel across tokens fall in different banks.
__host__ __device__ __forceinline__ int xs_stride(int d) { return d + 8; }

// ---------------------------------------------------------------------------
// Two codes at a time.  x, z, s, rs (= RN(1 / s), 0 when s is 0) hold two
// independent (value, group) pairs; the arithmetic is the quantizer's
// (item 1), bit-exact with round-half-even((x - z) / s) clamped to
// [0, 2^B - 1] with IEEE fp32 division:
//   d = x - z (fp32, RN), q = d * rs; q >= 0 since z is the group's min;
//   q is clamped above at 2^B - 1, then rounded to the nearest integer by
//   adding 1.5 * 2^23 (RN, ties to even: the integer lands in the low
//   mantissa bits, which are the code);
//   q lies within a few ulps of the correctly rounded quotient d / s, so
//   both round alike unless q sits next to a tie (k + 1/2): there the IEEE
//   division decides.  For a group member the quotient is below
//   2 * 2^B (below 2^B unless a subnormal fp16 scale rounded down), so the
//   margin 1e-5 * 2^B covers those few ulps.
// Packed fp32x2 instructions (two lanes of arithmetic per instruction)
// carry the subtraction, product and rounding.
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

// the quotient's own code, for the rare value next to a tie
template <int BITS>
__device__ __noinline__ unsigned tie_code(float d, float sf) {
    if (sf == 0.0f) return 0u;
    float k = rintf(__fdiv_rn(d, sf));
    k = fminf(fmaxf(k, 0.0f), (float)((1 << BITS) - 1));
    return (unsigned)k;
}

// codes of (x.lo, x.hi) against (z, s, rs) of their groups
template <int BITS>
__device__ __forceinline__ uint2 qcode2(u64 x, u64 z, u64 s, u64 rs) {
    constexpr float kMagic = 12582912.0f;   // 1.5 * 2^23
    constexpr float kQmax = (float)((1 << BITS) - 1);
    const u64 d = f2sub(x, z);
    const u64 q0 = f2mul(d, rs);
    const u64 q = f2p(fminf(f2lo(q0), kQmax), fminf(f2hi(q0), kQmax));
    const u64 M2 = f2p(kMagic, kMagic);
    const u64 t = f2add(q, M2);
    const u64 r = f2sub(q, f2sub(t, M2));   // q - round(q)
    uint2 c = make_uint2((unsigned)t & ((1u << BITS) - 1u), (unsigned)(t >> 32) & ((1u << BITS) - 1u));
    constexpr float kTie = 0.5f - 1.0e-5f * (float)(1 << BITS);
    if (fmaxf(fabsf(f2lo(r)), fabsf(f2hi(r))) > kTie) {
        c.x = tie_code<BITS>(f2lo(d), f2lo(s));
        c.y = tie_code<BITS>(f2hi(d), f2hi(s));
    }
    return c;
}

__device__ __forceinline__ __half2 u2h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ u64 h2_to_f2(uint32_t h) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return f2p(f.x, f.y);
}

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

// ---------------------------------------------------------------------------
// Prefill keys: one CTA per (super block of TB = max(64, G) tokens, kv head,
// sequence).  Quantizes tokens [0, nqk), nqk = t - t mod R.  The tile is
// staged in shared memory (rows padded against bank conflicts; rows past
// the quantized range are zero, and so are their groups' parameters, so
// every field there comes out 0).
// ---------------------------------------------------------------------------
template <int KBITS, int G>
__global__ void __launch_bounds__(256) prefill_keys_kernel(KiviGeom g, KiviDev dv,
                                                           const __half *__restrict__ K,
                                                           SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int TB = G > KIVI_KBLK ? G : KIVI_KBLK;
    constexpr int NG = TB / G;   // groups of the tile
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqk = t - t % g.R;
    const int tok0 = sb * TB;
    if (tok0 >= nqk) return;
    const int d = g.d, xsd = xs_stride(d);
    const int ntok = min(TB, nqk - tok0);   // a multiple of G
    const int ngr = ntok / G;

    __half *xs = reinterpret_cast<__half *>(smem);                        // [TB][xsd]
    float *sfz = reinterpret_cast<float *>(smem + (size_t)TB * xsd * 2);  // [NG][3][d]: s, z, 1/s

    const __half *src = K + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    const int vpr = d / 8;   // 16-byte vectors per row
    for (int e = threadIdx.x; e < TB * vpr; e += blockDim.x) {
        const int r = e / vpr, c = e - r * vpr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < ntok) v = reinterpret_cast<const uint4 *>(src)[e];
        reinterpret_cast<uint4 *>(xs + (size_t)r * xsd)[c] = v;
    }
    __syncthreads();

    // scale and zero per (group, channel): the min / max of fp16 values is
    // exact in fp16, taken two channels at a time
    const int dp = d / 2;
    for (int e = threadIdx.x; e < NG * dp; e += blockDim.x) {
        const int gr = e / dp, c = 2 * (e - gr * dp);
        float2 sf2 = make_float2(0.f, 0.f), zf2 = sf2, rs2 = sf2;
        if (gr < ngr) {
            const __half2 *col = reinterpret_cast<const __half2 *>(xs + (size_t)gr * G * xsd + c);
            __half2 mn = col[0], mx = mn;
#pragma unroll 8
            for (int k = 1; k < G; ++k) {
                const __half2 x = col[(size_t)k * (xsd / 2)];
                mn = __hmin2(mn, x);
                mx = __hmax2(mx, x);
            }
            __half s16, z16;
            group_params(__low2half(mn), __low2half(mx), KBITS, s16, z16, sf2.x, zf2.x, rs2.x);
            ksz_store(g, dv.blk, i, j, tok0 / G + gr, c, s16, z16);
            group_params(__high2half(mn), __high2half(mx), KBITS, s16, z16, sf2.y, zf2.y, rs2.y);
            ksz_store(g, dv.blk, i, j, tok0 / G + gr, c + 1, s16, z16);
        }
        *reinterpret_cast<float2 *>(sfz + (gr * 3 + 0) * d + c) = sf2;
        *reinterpret_cast<float2 *>(sfz + (gr * 3 + 1) * d + c) = zf2;
        *reinterpret_cast<float2 *>(sfz + (gr * 3 + 2) * d + c) = rs2;
    }
    __syncthreads();

    // packed words of every 64-token block that starts inside [tok0, nqk)
    constexpr int cph = 16 / KBITS;
    // a word's slots span 8 cph tokens: this many groups (slot r is in
    // group r / RPG of the word's first)
    constexpr int RPG = G / 8 < cph ? G / 8 : cph;
    constexpr int GW = cph / RPG;
    const int kc_blk = g.kc_blk;
    const int nblk = (ntok + KIVI_KBLK - 1) / KIVI_KBLK;
    for (int e = threadIdx.x; e < nblk * kc_blk; e += blockDim.x) {
        const int kbl = e / kc_blk, wb = e - kbl * kc_blk;
        const KWord kw = kword_decode(wb, KBITS);
        // Slot r holds token trow + 8 r + g (g < 8).  trow is a multiple of
        // 32, and of G whenever G <= 32; for G >= 64 the word's tokens lie
        // in one group.  So slot r's group is trow / G + r / RPG.
        const int trow = kbl * KIVI_KBLK + 8 * kw.pos0;
        const float *fw = sfz + (size_t)(trow / G) * 3 * d + kw.c0;
        u64 zz[GW], ss[GW], rr[GW];
#pragma unroll
        for (int k = 0; k < GW; ++k) {
            const float *f = fw + (size_t)k * 3 * d;
            const float2 s2 = *reinterpret_cast<const float2 *>(f);
            const float2 z2 = *reinterpret_cast<const float2 *>(f + d);
            const float2 r2 = *reinterpret_cast<const float2 *>(f + 2 * d);
            ss[k] = f2p(s2.x, s2.y);
            zz[k] = f2p(z2.x, z2.y);
            rr[k] = f2p(r2.x, r2.y);
        }
        uint32_t word = 0;
#pragma unroll
        for (int r = 0; r < cph; ++r) {
            // slot r of both halves: token tl, channels c0 and c0 + 1
            const int tl = trow + 8 * r + kw.g;
            const u64 x = h2_to_f2(*reinterpret_cast<const uint32_t *>(xs + (size_t)tl * xsd + kw.c0));
            const uint2 cd = qcode2<KBITS>(x, zz[r / RPG], ss[r / RPG], rr[r / RPG]);
            word |= (cd.x << (r * KBITS)) | (cd.y << (16 + r * KBITS));
        }
        kc_words(g, dv.blk, i, j, tok0 / KIVI_KBLK + kbl)[wb] = word;
    }
}

// ---------------------------------------------------------------------------
// Prefill values: one CTA per (64 tokens = 4 value blocks, kv head,
// sequence).  Quantizes tokens [0, nqv), nqv = max(t - R, 0).  A value word
// holds two consecutive tokens (its halves) at the same channels, so the
// tile is staged with token pairs interleaved: element (pair k, channel c)
// is a half2 of tokens 2k and 2k + 1 at channel c, and one 32-bit load
// gives both halves of a slot.  Tokens past nqv are zero, with zero scale
// and zero: their fields come out 0.
// ---------------------------------------------------------------------------
template <int VBITS, int G>
__global__ void __launch_bounds__(256) prefill_values_kernel(KiviGeom g, KiviDev dv,
                                                             const __half *__restrict__ V,
                                                             SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqv = t > g.R ? t - g.R : 0;
    const int tok0 = sb * 64;
    if (tok0 >= nqv) return;
    const int d = g.d, ngi = d / G;
    const int ps = d + 4;   // pair row stride in 32-bit words (padded)
    const int ntok = min(64, nqv - tok0);
    uint32_t *xs2 = reinterpret_cast<uint32_t *>(smem);                    // [32][ps] half2 pairs
    float2 *sfz = reinterpret_cast<float2 *>(smem + (size_t)32 * ps * 4);  // [32][3][ngi]: s, z, 1/s pairs

    // stage: rows 2k and 2k + 1, 8 channels at a time, interleaved by halves
    const __half *src = V + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    const int vpr = d / 8;
    for (int e = threadIdx.x; e < 32 * vpr; e += blockDim.x) {
        const int k = e / vpr, c8 = e - k * vpr;
        uint4 a = make_uint4(0u, 0u, 0u, 0u), b = a;
        if (2 * k < ntok) a = reinterpret_cast<const uint4 *>(src + (size_t)(2 * k) * d)[c8];
        if (2 * k + 1 < ntok) b = reinterpret_cast<const uint4 *>(src + (size_t)(2 * k + 1) * d)[c8];
        uint4 lo, hi;
        lo.x = __byte_perm(a.x, b.x, 0x5410);
        lo.y = __byte_perm(a.x, b.x, 0x7632);
        lo.z = __byte_perm(a.y, b.y, 0x5410);
        lo.w = __byte_perm(a.y, b.y, 0x7632);
        hi.x = __byte_perm(a.z, b.z, 0x5410);
        hi.y = __byte_perm(a.z, b.z, 0x7632);
        hi.z = __byte_perm(a.w, b.w, 0x5410);
        hi.w = __byte_perm(a.w, b.w, 0x7632);
        uint4 *dst = reinterpret_cast<uint4 *>(xs2 + (size_t)k * ps + 8 * c8);
        dst[0] = lo;
        dst[1] = hi;
    }
    __syncthreads();

    // scale and zero per (token, channel group), both tokens of a pair at once
    const int nvblk = (ntok + KIVI_VBLK - 1) / KIVI_VBLK;   // value blocks touched
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
        *reinterpret_cast<__half2 *>(vsz + vsz_in_block(g, tau, gi, 0)) = s16;   // tokens past nqv: zero
        *reinterpret_cast<__half2 *>(vsz + vsz_in_block(g, tau, gi, 1)) = z16;
        sfz[(k * 3 + 0) * ngi + gi] = sf;
        sfz[(k * 3 + 1) * ngi + gi] = zf;
        sfz[(k * 3 + 2) * ngi + gi] = rs;
    }
    __syncthreads();

    const int cs = v_cs(g);
    constexpr int cph = 16 / VBITS;
    const int vc_blk = g.vc_blk;
    for (int e = threadIdx.x; e < nvblk * vc_blk; e += blockDim.x) {
        const int vbl = e / vc_blk, wb = e - vbl * vc_blk;
        const VWord vw = vword_decode(wb, d, VBITS, cs);
        // Slot r holds channel 8 (ci0 + r) + g (g < 8) of tokens tt0, tt0 + 1
        // (one pair); 8 ci0 is a multiple of 32, and of G whenever G <= 32;
        // for G >= 64 the word's channels lie in one group.  So slot r's
        // group is 8 ci0 / G + (8 r) / G.
        const int k = (vbl * KIVI_VBLK + vw.tt0) >> 1;
        const int gi0 = 8 * vw.ci0 / G;
        const uint32_t *xr = xs2 + (size_t)k * ps;
        const float2 *fp = sfz + (size_t)k * 3 * ngi + gi0;
        uint32_t word = 0;
#pragma unroll
        for (int r = 0; r < cph; ++r) {
            const int c = 8 * (vw.ci0 + r) + vw.g;
            const float2 s2 = fp[(8 * r) / G], z2 = fp[ngi + (8 * r) / G], r2 = fp[2 * ngi + (8 * r) / G];
            const uint2 cd = qcode2<VBITS>(h2_to_f2(xr[c]), f2p(z2.x, z2.y), f2p(s2.x, s2.y), f2p(r2.x, r2.y));
            word |= (cd.x << (r * VBITS)) | (cd.y << (16 + r * VBITS));
        }
        vc_words(g, dv.blk, i, j, tok0 / KIVI_VBLK + vbl)[wb] = word;
    }
}

template <int BITS, int G>
cudaError_t launch_prefill_kv(const KiviGeom &g, const KiviDev &dv, const __half *K, const __half *V,
                              const SeqLens &lens, int t_stride, int maxt, cudaStream_t st) {
    constexpr int TB = G > KIVI_KBLK ? G : KIVI_KBLK;
    const int xsd = xs_stride(g.d);
    cudaError_t e = cudaSuccess;
    if (g.kbits == BITS) {
        const size_t smk = (size_t)TB * xsd * 2 + (size_t)(TB / G) * 3 * g.d * 4;
        e = cudaFuncSetAttribute(prefill_keys_kernel<BITS, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smk);
        if (e != cudaSuccess) return e;
        prefill_keys_kernel<BITS, G><<<dim3((maxt + TB - 1) / TB, g.h, g.b), 256, smk, st>>>(g, dv, K, lens,
                                                                                           t_stride);
    }
    if (g.vbits == BITS) {
        const size_t smv = (size_t)32 * (g.d + 4) * 4 + (size_t)32 * 3 * (g.d / G) * 8;
        e = cudaFuncSetAttribute(prefill_values_kernel<BITS, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smv);
        if (e != cudaSuccess) return e;
        prefill_values_kernel<BITS, G><<<dim3((maxt + 63) / 64, g.h, g.b), 256, smv, st>>>(g, dv, V, lens,
                                                                                         t_stride);
    }
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_prefill_g(const KiviGeom &g, const KiviDev &dv, const __half *K, const __half *V,
                             const SeqLens &lens, int t_stride, int maxt, cudaStream_t st) {
    cudaError_t e = launch_prefill_kv<2, G>(g, dv, K, V, lens, t_stride, maxt, st);
    if (e != cudaSuccess) return e;
    return launch_prefill_kv<4, G>(g, dv, K, V, lens, t_stride, maxt, st);
}

// ---------------------------------------------------------------------------
// Prefill fp16 windows and counters: one CTA per (kv head, sequence).
// Key token tau in [nqk, t) goes to slot tau % R; value token tau in
// [nqv, t) to slot tau % (R + 1).
// ---------------------------------------------------------------------------
__global__ void prefill_residual_kernel(KiviGeom g, KiviDev dv, const __half *__restrict__ K,
                                        const __half *__restrict__ V, SeqLens lens, int t_stride) {
    const int j = blockIdx.x, i = blockIdx.y;
    const int t = lens.t[i];
    const int nqk = t - t % g.R, nqv = t > g.R ? t - g.R : 0;
    const int vpt = g.d / 8;   // uint4 per token
    const uint4 *ks = reinterpret_cast<const uint4 *>(K + ((size_t)i * g.h + j) * t_stride * g.d);
    const uint4 *vs = reinterpret_cast<const uint4 *>(V + ((size_t)i * g.h + j) * t_stride * g.d);
    uint4 *kf = reinterpret_cast<uint4 *>(dv.Kf + kf_slice(g, i, j));
    uint4 *vf = reinterpret_cast<uint4 *>(dv.Vf + vf_slice(g, i, j));
    for (int e = threadIdx.x; e < (t - nqk) * vpt; e += blockDim.x) {
        int tau = nqk + e / vpt, c = e % vpt;
        kf[(size_t)(tau % g.R) * vpt + c] = ks[(size_t)tau * vpt + c];
    }
    for (int e = threadIdx.x; e < (t - nqv) * vpt; e += blockDim.x) {
        int tau = nqv + e / vpt, c = e % vpt;
        vf[(size_t)(tau % (g.R + 1)) * vpt + c] = vs[(size_t)tau * vpt + c];
    }
    if (j == 0 && threadIdx.x == 0) {
        dv.T[i] = t;
        dv.Tqk[i] = nqk;
        dv.Tqv[i] = nqv;
    }
}

// ---------------------------------------------------------------------------
// Append: one CTA per (kv head, sequence): append_pair (kivi_append_impl.cuh),
// then the last CTA of a sequence to finish advances that sequence's
// counters (all CTAs read them first).
// ---------------------------------------------------------------------------
// One CTA per (kv head j, sequence i).  The counters before the append come
// from the host mirror (ac); the device's current set is read only to check
// that the two agree.  CTA j = 0 of each sequence writes the counters after
// the append into the other set (nxt), so no CTA waits for another.
__global__ void __launch_bounds__(1024) append_kernel(KiviGeom g, KiviDev dv,
                                                     const __half *__restrict__ knew,
                                                     const __half *__restrict__ vnew, AppendCounters ac,
                                                     int *__restrict__ nxt) {
    // the decode launch that usually follows may start its set-up now: it
    // waits for this whole grid before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int j = blockIdx.x, i = blockIdx.y;
    const int R = g.R;
    const int T = ac.T[i], Tqk = ac.Tqk[i], Tqv = ac.Tqv[i];
    int dT = T, dTqk = Tqk, dTqv = Tqv;
    if (threadIdx.x == 0) {
        dT = dv.T[i];
        dTqk = dv.Tqk[i];
        dTqv = dv.Tqv[i];
    }
    if (!append_counters_ok(g, T, Tqk, Tqv)) {
        if (threadIdx.x == 0) flag(dv.status, KIVI_FLAG_COUNTER);
        return;
    }
    append_pair(g, dv, knew, vnew, i, j, T, Tqk, Tqv);
    if (threadIdx.x == 0) {
        if (dT != T || dTqk != Tqk || dTqv != Tqv) flag(dv.status, KIVI_FLAG_COUNTER);
        if (j == 0) {
            nxt[i] = T + 1;
            nxt[g.b + i] = Tqk + ((T - Tqk) == R ? R : 0);
            nxt[2 * g.b + i] = Tqv + ((T - Tqv) == R + 1 ? 1 : 0);
        }
    }
}

}  // namespace

cudaError_t kivi_launch_prefill(const KiviGeom &g, const KiviDev &dv, const __half *K,
                                const __half *V, const SeqLens &lens, int t_stride,
                                cudaStream_t st) {
    int maxt = 0;
    for (int i = 0; i < g.b; ++i) maxt = lens.t[i] > maxt ? lens.t[i] : maxt;
    if (maxt > 0) {
        cudaError_t e;
        switch (g.G) {
        case 16: e = launch_prefill_g<16>(g, dv, K, V, lens, t_stride, maxt, st); break;
        case 32: e = launch_prefill_g<32>(g, dv, K, V, lens, t_stride, maxt, st); break;
        case 64: e = launch_prefill_g<64>(g, dv, K, V, lens, t_stride, maxt, st); break;
        default: e = launch_prefill_g<128>(g, dv, K, V, lens, t_stride, maxt, st); break;
        }
        if (e != cudaSuccess) return e;
    }
    prefill_residual_kernel<<<dim3(g.h, g.b), 256, 0, st>>>(g, dv, K, V, lens, t_stride);
    return cudaGetLastError();
}

cudaError_t kivi_launch_append(const KiviGeom &g, const KiviDev &dv, const __half *k,
                               const __half *v, const AppendCounters &ac, int *nxt, cudaStream_t st) {
    // When some sequence flushes its key window now: shared memory for the
    // staged window rows and their groups' scale, zero and reciprocal, and
    // four times the threads (the flush is latency-bound arithmetic over
    // R x d keys; the other steps move one token).
    bool flush = false;
    for (int i = 0; i < g.b; ++i) flush |= ac.T[i] - ac.Tqk[i] == g.R;
    const size_t smem = flush ? flush_smem_bytes(g) : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    append_kernel<<<dim3(g.h, g.b), flush ? 1024 : 256, smem, st>>>(g, dv, k, v, ac, nxt);
    return cudaGetLastError();
}
