// kivi_decode_impl.cuh -- split-K decode attention over the quantized cache.
//
// Method: "Literature audit -- Group 2", section 1 KIVI, core algorithm
// item 5: scores q.k / sqrt(d) over the quantized keys followed by the fp16
// keys, one softmax over both, weights applied to the quantized values
// followed by the fp16 values.  Query head i reads kv head i / (h_q / h_kv)
// (GQA, README note of 2025-01-18 in the same section).
//
// Work split.  A CTA owns one (sequence, kv head, group of <= 4 query heads)
// and a token range, so each packed word is read from HBM once.  Full 64-token
// blocks whose keys AND values are quantized go through the tensor-core path:
// each warp streams its blocks through a private ring of shared-memory stages
// filled by bulk TMA copies (cp.async.bulk + mbarrier) and runs
//   scores   S[tok, col] = sum_c (4 + code) * B[c, col]      (m16n8k16, f16 in, f32 acc)
//   values   O[ch, col]  = sum_t (4 + code) * P[t, col]
// with the unpacked code in the A operand (one shift + one lop3 per half2:
// the 2-bit field lands in the top mantissa bits of fp16 4.0, the 4-bit field
// in those of 16.0) and the per-group scale folded into B.  Column pairs
// (2e, 2e+1) carry an exact two-term fp16 split of B for query head e:
//   keys:   q_c s = hi + lo with hi = RN(q s), lo = fma(q, s, -hi)  (exact)
//   values: p s  = hi + lo from p = ph + pl (fp16 hi/lo of the fp32 weight)
// so the tensor-core sums carry fp32-level precision.  The zero points and
// the +4 / +16 offset enter through small MMAs over the scale/zero rows:
//   keys:   corr[g, e] = sum_c q_c z_c - off sum_c q_c s_c
//   values: corr[gi, e] = sum_t p_t z_t - off sum_t p_t s_t
// Blocks holding fp16 keys or values (the residual window) form a short tail
// handled on CUDA cores by extra CTAs.  Every CTA writes (m, l, acc[d]) in
// base 2 (scores pre-multiplied by log2(e) / sqrt(d)); the last CTA of each
// (sequence, kv head, head group) merges the partials with log-sum-exp
// weights and writes the fp16 output.
#pragma once
#include "kivi_internal.cuh"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWaitIters = 1 << 24;   // bounded mbarrier waits

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned smem_u32(const void *p) {
    return (unsigned)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned phase) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0;
}

// bounded wait: false if the barrier did not complete within the limit
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned phase) {
    for (int it = 0; it < kMaxWaitIters; ++it)
        if (mbar_try_wait(bar, phase)) return true;
    return false;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) { return h2u(__hmul2(u2h(a), u2h(b))); }
__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
    return h2u(__hfma2(u2h(a), u2h(b), u2h(c)));
}

// Unpack field r of both 16-bit halves of w as fp16 (off + code).  The field
// is moved (by a shift shared between fields, or none) to a mantissa
// position p of an fp16 constant whose exponent makes bit p weigh 1, and
// or-ed into it: the value is 2^(10 - p) + code.
//   keys:   p in {4, 6, 8} (offsets 64, 16, 4); the accumulator carries
//           off * sum(q s), removed with the zero-point MMA's sum(q s) row;
//           against score-sized sums this costs < 1e-4 relative.
//   values: any p <= 8; the offset is subtracted in fp16 before the MMA
//           (exact), because the weighted value sums can be far smaller
//           than off * sum(p s).
struct View {
    int shl, shr;          // shift left / right applied to the word
    uint32_t mask, magic;  // field mask at its target position, fp16 pattern of the offset
    float off;
};
__host__ __device__ constexpr View at_pos(int p, int width, int shl, int shr) {
    // field of `width` bits at mantissa bit p; fp16 2^(10 - p) = exponent field 25 - p
    return View{shl, shr, (((1u << width) - 1u) << p) * 0x10001u, (uint32_t)(25 - p) * 0x04000400u,
                (float)(1 << (10 - p))};
}
template <int BITS, bool KEY>
__host__ __device__ constexpr View view_of(int r) {
    if (BITS == 4) {
        if (KEY)   // field bits [4r, 4r + 4) -> bits 6..9, offset 16
            return r <= 1 ? at_pos(6, 4, 6 - 4 * r, 0) : at_pos(6, 4, 0, 4 * r - 6);
        // values: slots 0, 1 in place (p = 0, 4); slots 2, 3 shifted to p = 4
        return r == 0 ? at_pos(0, 4, 0, 0) : (r == 1 ? at_pos(4, 4, 0, 0) : at_pos(4, 4, 0, 4 * r - 4));
    }
    // 2-bit field bits [2r, 2r + 2)
    if (KEY) {
        switch (r) {
        case 0: return at_pos(4, 2, 4, 0);
        case 1: return at_pos(6, 2, 4, 0);
        case 2: return at_pos(4, 2, 0, 0);
        case 3: return at_pos(6, 2, 0, 0);
        case 4: return at_pos(8, 2, 0, 0);
        case 5: return at_pos(4, 2, 0, 6);
        case 6: return at_pos(6, 2, 0, 6);
        default: return at_pos(8, 2, 0, 6);
        }
    }
    // values: slots 0..4 in place (p = 0, 2, 4, 6, 8); slots 5..7 via one shift
    return r <= 4 ? at_pos(2 * r, 2, 0, 0) : at_pos(2 * r - 6, 2, 0, 6);
}
// (x & mask) | magic as one lop3 with both constants as immediates; the
// plain C++ form compiles to two ALU instructions on this target.
template <uint32_t MASK, uint32_t MAGIC>
__device__ __forceinline__ uint32_t and_or(uint32_t x) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "n"(MASK), "n"(MAGIC));
    return r;
}
template <int BITS, bool KEY, int R>
__device__ __forceinline__ uint32_t unpack_t(uint32_t w) {
    constexpr View v = view_of<BITS, KEY>(R);
    const uint32_t x = v.shl ? (w << v.shl) : (v.shr ? (w >> v.shr) : w);
    return and_or<v.mask, v.magic>(x);
}
// runtime-looking slot index r (a constant once the caller's loops unroll)
template <int BITS, bool KEY>
__device__ __forceinline__ uint32_t unpack(uint32_t w, int r) {
    switch (r) {
    case 0: return unpack_t<BITS, KEY, 0>(w);
    case 1: return unpack_t<BITS, KEY, 1>(w);
    case 2: return unpack_t<BITS, KEY, 2>(w);
    case 3: return unpack_t<BITS, KEY, 3>(w);
    case 4: return unpack_t<BITS, KEY, (BITS == 2 ? 4 : 3)>(w);
    case 5: return unpack_t<BITS, KEY, (BITS == 2 ? 5 : 3)>(w);
    case 6: return unpack_t<BITS, KEY, (BITS == 2 ? 6 : 3)>(w);
    default: return unpack_t<BITS, KEY, (BITS == 2 ? 7 : 3)>(w);
    }
}
// value fields: the exact code as fp16 (offset subtracted, exact)
template <int BITS>
__device__ __forceinline__ uint32_t unpack_exact(uint32_t w, int r) {
    const View v = view_of<BITS, false>(r);
    return h2u(__hsub2(u2h(unpack<BITS, false>(w, r)), u2h(v.magic)));
}
template <int BITS, bool KEY>
__host__ __device__ constexpr float slot_offset(int r) { return view_of<BITS, KEY>(r).off; }

// ---------------------------------------------------------------------------
// CUDA-core path for the tail (the last blocks, holding fp16 keys or values):
// one warp per token, lane owns channels lane + 32 k.  Geometry is
// compile-time except R (one modulo per token).
// ---------------------------------------------------------------------------
template <int D, int KB, int VB, int SH>
__device__ __forceinline__ void tail_load(const KiviGeom &g, const uint32_t *kc, const __half *ksz,
                                          const __half *kf, const uint32_t *vc, const __half *vsz,
                                          const __half *vf, int Tqk, int Tqv, int tau, int lane,
                                          float (&kv)[D / 32], float (&vv)[D / 32]) {
    constexpr int CPL = D / 32;
    constexpr int G = 16 << SH;
    constexpr int CPHK = 16 / KB, NWK = KB / 2, CPHV = 16 / VB, NWV = D * VB / 128;
    constexpr int WLV = D * VB / 64, CSV = WLV < 4 ? WLV : 4;
    constexpr int KC_BLK = 2 * D * KB, VC_BLK = D * VB / 2, VSZ_BLK = 2 * (D / G) * 16;
    if (tau < Tqk) {
        const int kb = tau >> 6, pos = (tau & 63) >> 3, gg = tau & 7;
        const int wi = pos / CPHK, r = pos % CPHK;
        const __half *sz = ksz + (size_t)(tau / G) * 2 * D;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int c = lane + 32 * k;
            const int u = (2 * (c >> 4) + ((c >> 3) & 1)) * NWK + wi;
            const int L = 4 * gg + ((c & 7) >> 1);
            const uint32_t w = __ldg(kc + (size_t)kb * KC_BLK + (u >> 2) * 128 + 4 * L + (u & 3));
            const uint32_t code = (w >> (16 * (c & 1) + r * KB)) & ((1u << KB) - 1u);
            kv[k] = (float)code * __half2float(sz[c]) + __half2float(sz[D + c]);
        }
    } else {
        const __half *src = kf + (size_t)(tau % g.R) * D;
#pragma unroll
        for (int k = 0; k < CPL; ++k) kv[k] = __half2float(src[lane + 32 * k]);
    }
    if (tau < Tqv) {
        const int vb = tau >> 4, tt = tau & 15;
        const int p = tt >> 3, t = (tt & 7) >> 1, hi = tt & 1;
        const __half *sz = vsz + (size_t)vb * VSZ_BLK;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            const int c = lane + 32 * k;
            const int ci = c >> 3, w = ci / CPHV, r = ci % CPHV;
            const int L = 4 * (c & 7) + t, u = p * NWV + w;
            const uint32_t word = __ldg(vc + (size_t)vb * VC_BLK + (u / CSV) * 32 * CSV + L * CSV + (u % CSV));
            const uint32_t code = (word >> (16 * hi + r * VB)) & ((1u << VB) - 1u);
            const int gi = c / G;
            vv[k] = (float)code * __half2float(sz[gi * 16 + tt]) + __half2float(sz[(D / G + gi) * 16 + tt]);
        }
    } else {
        const __half *src = vf + (size_t)(tau % (g.R + 1)) * D;
#pragma unroll
        for (int k = 0; k < CPL; ++k) vv[k] = __half2float(src[lane + 32 * k]);
    }
}

// Tail CTA: tokens [t0, t1) (at most KIVI_TAILBLK), one warp per token, lane
// owns channels lane + 32 k; each warp loads all of its tokens before
// computing so that their memory latencies overlap.
template <int D, int KB, int VB, int SH>
__device__ void tail_tokens(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, int i,
                            int j, int e0, int nh, int t0, int t1, float *wm, float *wl, float *wo) {
    constexpr int CPL = D / 32;
    constexpr int TPW = 4;   // tokens per warp: KIVI_TAILBLK / 8 warps
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int hg = hq / g.h;
    const int Tqk = dv.Tqk[i], Tqv = dv.Tqv[i];
    const float qscale = kLog2e * rsqrtf((float)D);
    float qr[4][CPL], m[4], l[4], acc[4][CPL];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        m[e] = -INFINITY;
        l[e] = 0.f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            acc[e][k] = 0.f;
            qr[e][k] = e < nh ? __half2float(q[((size_t)i * hq + j * hg + e0 + e) * D + lane + 32 * k]) * qscale
                              : 0.f;
        }
    }
    const uint32_t *kc = dv.Kc + kc_slice(g, i, j);
    const __half *ksz = dv.Ksz + ksz_slice(g, i, j);
    const __half *kf = dv.Kf + kf_slice(g, i, j);
    const uint32_t *vc = dv.Vc + vc_slice(g, i, j);
    const __half *vsz = dv.Vsz + vsz_slice(g, i, j);
    const __half *vf = dv.Vf + vf_slice(g, i, j);
    for (int base = t0 + warp; base < t1; base += nw * TPW) {
        float kv[TPW][CPL], vv[TPW][CPL];
#pragma unroll
        for (int x = 0; x < TPW; ++x) {
            const int tau = base + x * nw;
            if (tau < t1)
                tail_load<D, KB, VB, SH>(g, kc, ksz, kf, vc, vsz, vf, Tqk, Tqv, tau, lane, kv[x], vv[x]);
        }
#pragma unroll
        for (int x = 0; x < TPW; ++x) {
            if (base + x * nw >= t1) break;
            float dot[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                dot[e] = 0.f;
#pragma unroll
                for (int k = 0; k < CPL; ++k) dot[e] = fmaf(qr[e][k], kv[x][k], dot[e]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int e = 0; e < 4; ++e) dot[e] += __shfl_xor_sync(0xffffffffu, dot[e], o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mn = fmaxf(m[e], dot[e]);
                const float corr = ex2(m[e] - mn);
                const float p = ex2(dot[e] - mn);
                l[e] = l[e] * corr + p;
#pragma unroll
                for (int k = 0; k < CPL; ++k) acc[e][k] = fmaf(p, vv[x][k], acc[e][k] * corr);
                m[e] = mn;
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (lane == 0) {
            wm[e] = m[e];
            wl[e] = l[e];
        }
#pragma unroll
        for (int k = 0; k < CPL; ++k) wo[e * D + lane + 32 * k] = acc[e][k];
    }
}

// ---------------------------------------------------------------------------
// Tensor-core path over full blocks.
// ---------------------------------------------------------------------------
struct StageGeom {
    int kc_bytes, ksz_bytes, vc_bytes, vsz_bytes, bytes;
};
__host__ __device__ __forceinline__ StageGeom stage_geom(const KiviGeom &g) {
    StageGeom s;
    s.kc_bytes = g.kc_blk * 4;
    s.ksz_bytes = (g.G >= KIVI_KBLK ? 1 : KIVI_KBLK / g.G) * 2 * g.d * 2;
    s.vc_bytes = 4 * g.vc_blk * 4;
    s.vsz_bytes = 4 * g.vsz_blk * 2;
    s.bytes = s.kc_bytes + s.ksz_bytes + s.vc_bytes + s.vsz_bytes;
    return s;
}

// Bytes of one warp's region of the dynamic shared memory: its ring of
// stages, which after the main loop also holds the warp's result
// (m[4], l[4], o[4][d] in fp32).
__host__ __device__ __forceinline__ size_t warp_region(const KiviGeom &g, int stages) {
    size_t ring = (size_t)stages * stage_geom(g).bytes;
    size_t res = ((size_t)(8 + 4 * g.d) * 4 + 127) / 128 * 128;
    return ring > res ? ring : res;
}
__host__ __device__ __forceinline__ size_t bar_region(int warps, int stages) {
    return ((size_t)warps * stages * 8 + 127) / 128 * 128;
}

__device__ __forceinline__ void issue_block(const KiviGeom &g, const StageGeom &sg, unsigned char *st,
                                            uint64_t *bar, const uint32_t *kc, const __half *ksz,
                                            const uint32_t *vc, const __half *vsz, int kb) {
    mbar_expect_tx(bar, (unsigned)sg.bytes);
    const int grp0 = g.G >= KIVI_KBLK ? (kb * KIVI_KBLK) / g.G : kb * (KIVI_KBLK / g.G);
    bulk_g2s(st, kc + (size_t)kb * g.kc_blk, sg.kc_bytes, bar);
    bulk_g2s(st + sg.kc_bytes, ksz + (size_t)grp0 * 2 * g.d, sg.ksz_bytes, bar);
    bulk_g2s(st + sg.kc_bytes + sg.ksz_bytes, vc + (size_t)kb * 4 * g.vc_blk, sg.vc_bytes, bar);
    bulk_g2s(st + sg.kc_bytes + sg.ksz_bytes + sg.vc_bytes, vsz + (size_t)kb * 4 * g.vsz_blk,
             sg.vsz_bytes, bar);
}

template <int D, int KB, int VB, int SH>
__device__ void mma_blocks(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, int i, int j,
                           int e0, int nh, int kb_begin, int kb_end, int stages, size_t wstride,
                           unsigned char *ring, uint64_t *bars, float *wm, float *wl, float *wo) {
    constexpr int NJ = D / 16;              // k-steps over channels / M-tiles of channels
    constexpr int NWK = KB / 2;             // key words per (j, hh) per lane
    constexpr int CPHK = 16 / KB;           // key fields per 16-bit half
    constexpr int CPHV = 16 / VB;           // value fields per 16-bit half
    constexpr int NWV = D * VB / 128;       // value words per token pair per lane
    constexpr int WLV = D * VB / 64;        // value words per lane per 16-token block
    constexpr int CSV = WLV < 4 ? WLV : 4;  // value chunk size
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const bool odd = gq & 1;
    const int eB = gq >> 1;                 // query head of this thread's B column
    const int hg = hq / g.h;
    const StageGeom sg = stage_geom(g);
    constexpr int sh = SH;                  // log2(G / 16): M-tile m -> group m >> sh
    constexpr int ngi = (D / 16) >> SH;     // value channel groups (d / G)
    constexpr int nkrows = 2 * (SH >= 2 ? 1 : (4 >> SH));   // key scale/zero rows per block
    const float alpha = kLog2e * rsqrtf((float)D);

    // ---- query fragments (B operand of the score MMA) ----
    uint32_t qB[NJ][2];
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t v = 0;
            if (eB < nh)
                v = *reinterpret_cast<const uint32_t *>(
                    q + ((size_t)i * hq + j * hg + e0 + eB) * D + 16 * jj + 8 * hh + 2 * tq);
            qB[jj][hh] = v;
        }
    const uint32_t nm = odd ? 0xBC00BC00u : 0u;     // -1 for lo columns, 0 for hi
    const uint32_t m1 = odd ? 0x3C003C00u : 0u;     // 1 for lo columns, 0 for hi

    float oacc[NJ][4];
#pragma unroll
    for (int mm = 0; mm < NJ; ++mm) oacc[mm][0] = oacc[mm][1] = oacc[mm][2] = oacc[mm][3] = 0.f;
    float zacc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    float mrun = -INFINITY, lrun = 0.f;

    const uint32_t *kc = dv.Kc + kc_slice(g, i, j);
    const __half *ksz = dv.Ksz + ksz_slice(g, i, j);
    const uint32_t *vc = dv.Vc + vc_slice(g, i, j);
    const __half *vsz = dv.Vsz + vsz_slice(g, i, j);
    unsigned char *myring = ring + (size_t)warp * wstride;
    uint64_t *mybars = bars + warp * stages;

    const int nb = kb_begin + warp < kb_end ? (kb_end - kb_begin - warp + nw - 1) / nw : 0;
    int issued = nb < stages ? nb : stages;
    if (lane == 0)
        for (int it = 0; it < issued; ++it)
            issue_block(g, sg, myring + (size_t)it * sg.bytes, mybars + it, kc, ksz, vc, vsz,
                        kb_begin + warp + it * nw);
    __syncwarp();

    bool timed_out = false;
    for (int it = 0; it < nb; ++it) {
        const int st = it % stages;
        const unsigned phase = (unsigned)(it / stages) & 1u;
        if (!mbar_wait(mybars + st, phase)) {
            timed_out = true;
            break;
        }
        const unsigned char *sb = myring + (size_t)st * sg.bytes;
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(sb);
        const __half *sKsz = reinterpret_cast<const __half *>(sb + sg.kc_bytes);
        const uint32_t *sV = reinterpret_cast<const uint32_t *>(sb + sg.kc_bytes + sg.ksz_bytes);
        const __half *sVsz =
            reinterpret_cast<const __half *>(sb + sg.kc_bytes + sg.ksz_bytes + sg.vc_bytes);

        // ---- key zero-point correction: rows = (group, s|z) of this block ----
        float dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
            uint32_t a0 = 0, a2 = 0;
            if (gq < nkrows) {
                a0 = *reinterpret_cast<const uint32_t *>(sKsz + gq * D + 16 * jj + 2 * tq);
                a2 = *reinterpret_cast<const uint32_t *>(sKsz + gq * D + 16 * jj + 8 + 2 * tq);
            }
            mma16816(dc, a0, 0u, a2, 0u, qB[jj][0], qB[jj][1]);
        }
        // sum_c q_c z_c (row 2rp + 1) and sum_c q_c s_c (row 2rp) of group rp for
        // head tq; rows are held by lanes 4 row + tq (column 2 tq)
        float kz[4], ks[4];
#pragma unroll
        for (int rp = 0; rp < 4; ++rp) {
            if (rp > (3 >> sh)) { kz[rp] = ks[rp] = 0.f; continue; }
            kz[rp] = __shfl_sync(0xffffffffu, dc[0], ((2 * rp + 1) & 7) * 4 + tq);
            ks[rp] = __shfl_sync(0xffffffffu, dc[0], ((2 * rp) & 7) * 4 + tq);
        }

        // ---- scores ----
        float sc[4][4];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) sc[mm][0] = sc[mm][1] = sc[mm][2] = sc[mm][3] = 0.f;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
            uint32_t W[2][NWK];   // [hh][wi]
            if (KB == 2) {
                const uint4 w4 = *reinterpret_cast<const uint4 *>(sK + (jj >> 1) * 128 + lane * 4);
                W[0][0] = (jj & 1) ? w4.z : w4.x;
                W[1][0] = (jj & 1) ? w4.w : w4.y;
            } else {
                const uint4 w4 = *reinterpret_cast<const uint4 *>(sK + jj * 128 + lane * 4);
                W[0][0] = w4.x;
                W[0][NWK - 1] = w4.y;
                W[1][0] = w4.z;
                W[1][NWK - 1] = w4.w;
            }
            uint32_t b0[4], b1[4];
#pragma unroll
            for (int rp = 0; rp < 4; ++rp) {
                if (rp > (3 >> sh)) continue;   // groups present in this block
                b0[rp] = b1[rp] = 0u;
                const uint32_t s0 = *reinterpret_cast<const uint32_t *>(sKsz + 2 * rp * D + 16 * jj + 2 * tq);
                const uint32_t s1 = *reinterpret_cast<const uint32_t *>(sKsz + 2 * rp * D + 16 * jj + 8 + 2 * tq);
                const uint32_t h0 = hmul2u(qB[jj][0], s0), h1 = hmul2u(qB[jj][1], s1);
                b0[rp] = hfma2u(qB[jj][0], s0, hmul2u(h0, nm));
                b1[rp] = hfma2u(qB[jj][1], s1, hmul2u(h1, nm));
            }
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const int rp = mm >> sh;
                const int wi = (2 * mm) / CPHK, r0 = (2 * mm) % CPHK;
                const uint32_t a0 = unpack<KB, true>(W[0][wi], r0), a1 = unpack<KB, true>(W[0][wi], r0 + 1);
                const uint32_t a2 = unpack<KB, true>(W[1][wi], r0), a3 = unpack<KB, true>(W[1][wi], r0 + 1);
                mma16816(sc[mm], a0, a1, a2, a3, b0[rp], b1[rp]);
            }
        }

        // ---- online softmax (head tq; rows 16 mm + gq and + 8) ----
        float p[4][2];
        float mx = -INFINITY;
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            // row g of tile mm reads field slot r0, row g + 8 slot r0 + 1
            const int rp = mm >> sh, r0 = (2 * mm) % CPHK;
            const float o0 = slot_offset<KB, true>(r0), o1 = slot_offset<KB, true>(r0 + 1);
            p[mm][0] = (sc[mm][0] + sc[mm][1] + fmaf(-o0, ks[rp], kz[rp])) * alpha;
            p[mm][1] = (sc[mm][2] + sc[mm][3] + fmaf(-o1, ks[rp], kz[rp])) * alpha;
            mx = fmaxf(mx, fmaxf(p[mm][0], p[mm][1]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(mrun, mx);
        const float scl = ex2(mrun - mnew);
        mrun = mnew;
        float ps = 0.f;
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            p[mm][0] = ex2(p[mm][0] - mnew);
            p[mm][1] = ex2(p[mm][1] - mnew);
            ps += p[mm][0] + p[mm][1];
        }
        lrun = lrun * scl + ps;
        if (__any_sync(0xffffffffu, scl != 1.f)) {   // the running max moved for some head
#pragma unroll
            for (int mm = 0; mm < NJ; ++mm) {
                oacc[mm][0] *= scl;
                oacc[mm][1] *= scl;
                oacc[mm][2] *= scl;
                oacc[mm][3] *= scl;
            }
            zacc[0][0] *= scl;
            zacc[0][1] *= scl;
            zacc[0][2] *= scl;
            zacc[0][3] *= scl;
        }

        // ---- weights times values, 16 tokens at a time ----
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const __half2 ph = __floats2half2_rn(p[kk][0], p[kk][1]);
            const float2 phf = __half22float2(ph);
            const __half2 pl = __floats2half2_rn(p[kk][0] - phf.x, p[kk][1] - phf.y);
            const int src1 = 8 * tq + eB, src2 = 8 * tq + 4 + eB;
            const uint32_t h1 = __shfl_sync(0xffffffffu, h2u(ph), src1);
            const uint32_t h2 = __shfl_sync(0xffffffffu, h2u(ph), src2);
            const uint32_t l1 = __shfl_sync(0xffffffffu, h2u(pl), src1);
            const uint32_t l2 = __shfl_sync(0xffffffffu, h2u(pl), src2);
            const uint32_t PH0 = prmt(h1, h2, 0x5410u), PH1 = prmt(h1, h2, 0x7632u);
            const uint32_t PL0 = prmt(l1, l2, 0x5410u), PL1 = prmt(l1, l2, 0x7632u);
            const uint32_t PL0m = hmul2u(PL0, m1), PL1m = hmul2u(PL1, m1);
            const __half *vszk = sVsz + kk * g.vsz_blk;
            uint32_t b0[16], b1[16];
#pragma unroll
            for (int gi = 0; gi < 16; ++gi) {
                if (gi >= ngi) continue;
                const uint32_t v0 = *reinterpret_cast<const uint32_t *>(vszk + gi * 16 + 2 * tq);
                const uint32_t v1 = *reinterpret_cast<const uint32_t *>(vszk + gi * 16 + 2 * tq + 8);
                const uint32_t h0 = hmul2u(PH0, v0), hh1 = hmul2u(PH1, v1);
                b0[gi] = hfma2u(PL0m, v0, hfma2u(PH0, v0, hmul2u(h0, nm)));
                b1[gi] = hfma2u(PL1m, v1, hfma2u(PH1, v1, hmul2u(hh1, nm)));
            }
            // value codes of this 16-token block: WLV words per lane
            uint32_t Wv[WLV];
            const uint32_t *sVk = sV + kk * g.vc_blk;
#pragma unroll
            for (int ch = 0; ch < WLV / CSV; ++ch) {
                if (CSV == 4) {
                    const uint4 w4 = *reinterpret_cast<const uint4 *>(sVk + ch * 128 + lane * 4);
                    Wv[ch * 4 + 0] = w4.x;
                    Wv[ch * 4 + 1] = w4.y;
                    Wv[ch * 4 + 2] = w4.z;
                    Wv[ch * 4 + 3] = w4.w;
                } else {
                    const uint2 w2 = *reinterpret_cast<const uint2 *>(sVk + ch * 64 + lane * 2);
                    Wv[ch * 2 + 0] = w2.x;
                    Wv[ch * 2 + 1] = w2.y;
                }
            }
#pragma unroll
            for (int mm = 0; mm < NJ; ++mm) {
                const int ci0 = 2 * mm;
                const int w = ci0 / CPHV, r0 = ci0 % CPHV;
                const uint32_t Wp0 = Wv[0 * NWV + w], Wp1 = Wv[1 * NWV + w];
                const uint32_t a0 = unpack_exact<VB>(Wp0, r0), a1 = unpack_exact<VB>(Wp0, r0 + 1);
                const uint32_t a2 = unpack_exact<VB>(Wp1, r0), a3 = unpack_exact<VB>(Wp1, r0 + 1);
                const int gi = mm >> sh;
                mma16816(oacc[mm], a0, a1, a2, a3, b0[gi], b1[gi]);
            }
            // value zero points: rows [z][gi][16 tokens] (the codes entered exactly)
            const uint32_t bz0 = odd ? PL0 : PH0, bz1 = odd ? PL1 : PH1;
            {
                const __half *zrow = vszk + ngi * 16;
                uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
                if (gq < ngi) {
                    a0 = *reinterpret_cast<const uint32_t *>(zrow + gq * 16 + 2 * tq);
                    a2 = *reinterpret_cast<const uint32_t *>(zrow + gq * 16 + 2 * tq + 8);
                }
                if (gq + 8 < ngi) {
                    a1 = *reinterpret_cast<const uint32_t *>(zrow + (gq + 8) * 16 + 2 * tq);
                    a3 = *reinterpret_cast<const uint32_t *>(zrow + (gq + 8) * 16 + 2 * tq + 8);
                }
                mma16816(zacc[0], a0, a1, a2, a3, bz0, bz1);
            }
        }

        // ---- refill this stage ----
        __syncwarp();
        if (it + stages < nb) {
            if (lane == 0) {
                fence_proxy_async();
                issue_block(g, sg, myring + (size_t)st * sg.bytes, mybars + st, kc, ksz, vc, vsz,
                            kb_begin + warp + (it + stages) * nw);
            }
            ++issued;
        }
    }
    if (timed_out) {
        if (lane == 0) atomicOr(dv.status, KIVI_FLAG_WAIT);
        // wait (bounded) for this warp's copies still in flight before leaving;
        // the consumed count is where the loop stopped
        for (int it = 0; it < issued; ++it) {
            if (mbar_try_wait(mybars + (it % stages), (unsigned)(it / stages) & 1u)) continue;
            mbar_wait(mybars + (it % stages), (unsigned)(it / stages) & 1u);
        }
        mrun = -INFINITY;
        lrun = 0.f;
#pragma unroll
        for (int mm = 0; mm < NJ; ++mm) oacc[mm][0] = oacc[mm][1] = oacc[mm][2] = oacc[mm][3] = 0.f;
    }

    // ---- per-warp result ----
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 4);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 8);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 16);
    // value zero-point sums per channel group gi: row gi of zacc (column pair 2 tq)
    const float zr0 = zacc[0][0] + zacc[0][1], zr1 = zacc[0][2] + zacc[0][3];
    float vz[16];
#pragma unroll
    for (int gi = 0; gi < 16; ++gi)
        vz[gi] = gi < ngi ? __shfl_sync(0xffffffffu, gi < 8 ? zr0 : zr1, (gi & 7) * 4 + tq) : 0.f;
    if (gq == 0) {
        wm[tq] = mrun;
        wl[tq] = lrun;
    }
#pragma unroll
    for (int mm = 0; mm < NJ; ++mm) {
        const int gi = mm >> sh;
        wo[tq * D + 16 * mm + gq] = oacc[mm][0] + oacc[mm][1] + vz[gi];
        wo[tq * D + 16 * mm + gq + 8] = oacc[mm][2] + oacc[mm][3] + vz[gi];
    }
}

// ---------------------------------------------------------------------------
// The kernel: MMA CTAs (x < splits) and tail CTAs (x >= splits), then the
// CTA-level merge of warps and the last-CTA merge of splits.
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// The kernel: MMA CTAs (x < splits) and tail CTAs (x >= splits), then the
// CTA-level merge of warps and the last-CTA merge of splits.
// ---------------------------------------------------------------------------
template <int D, int KB, int VB, int SH>
__global__ void __launch_bounds__(256, 2)
    decode_kernel(KiviGeom g, KiviDev dv, const __half *__restrict__ q, int hq,
                  __half *__restrict__ out, DecodePlan plan) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int i = blockIdx.z, j = blockIdx.y / plan.qgroups, qg = blockIdx.y % plan.qgroups;
    const int hg = hq / g.h;
    const int e0 = qg * 4, nh = min(4, hg - e0);
    const int T = dv.T[i], Tqk = dv.Tqk[i], Tqv = dv.Tqv[i];
    const int nfull = min(Tqk, Tqv) / KIVI_KBLK;
    const int nsplit_total = plan.splits + plan.tails;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + bar_region(nw, plan.stages);
    const size_t wstride = warp_region(g, plan.stages);
    float *wres = reinterpret_cast<float *>(ring + warp * wstride);
    float *wm = wres, *wl = wres + 4, *wo = wres + 8;

    // CTAs x < tails take the tail (dispatched first: short, latency-bound,
    // they overlap the streaming CTAs); the rest stream whole blocks.
    const int s = blockIdx.x;
    if (s >= plan.tails) {
        if (threadIdx.x < nw * plan.stages) mbar_init(bars + threadIdx.x, 1);
        fence_mbar_init();
        __syncthreads();
        const int kb0 = (s - plan.tails) * plan.blocks_per, kb1 = min(nfull, kb0 + plan.blocks_per);
        mma_blocks<D, KB, VB, SH>(g, dv, q, hq, i, j, e0, nh, kb0, kb1, plan.stages, wstride, ring,
                                  bars, wm, wl, wo);
    } else {
        const int t0 = nfull * KIVI_KBLK + s * KIVI_TAILBLK;
        const int t1 = min(T, t0 + KIVI_TAILBLK);
        tail_tokens<D, KB, VB, SH>(g, dv, q, hq, i, j, e0, nh, t0, t1, wm, wl, wo);
    }
    __syncthreads();

    // ---- merge the warps of this CTA into one partial per query head ----
    float *part = dv.part;
    for (int x = threadIdx.x; x < nh * (D + 2); x += blockDim.x) {
        const int e = x / (D + 2), c = x % (D + 2);
        float M = -INFINITY;
        for (int w = 0; w < nw; ++w) M = fmaxf(M, reinterpret_cast<const float *>(ring + w * wstride)[e]);
        float val = 0.f;
        if (c == 0) {
            val = M;
        } else if (M != -INFINITY) {
            for (int w = 0; w < nw; ++w) {
                const float *r = reinterpret_cast<const float *>(ring + w * wstride);
                const float f = ex2(r[e] - M);
                val += f * (c == 1 ? r[4 + e] : r[8 + e * D + (c - 2)]);
            }
        }
        part[(((size_t)i * hq + j * hg + e0 + e) * g.smax + s) * (D + 2) + c] = val;
    }

    // ---- the last CTA of this (sequence, kv head, head group) merges ----
    __shared__ int s_last;
    __shared__ float sML[8];
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned *tk = dv.merge_ticket + ((size_t)i * g.h + j) * 4 + qg;
        const unsigned prev = atomicAdd(tk, 1u);
        s_last = prev == (unsigned)nsplit_total - 1u;
        if (s_last) *tk = 0u;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < nh) {
        const int e = threadIdx.x;
        const float *pp = part + ((size_t)i * hq + j * hg + e0 + e) * g.smax * (D + 2);
        float M = -INFINITY;
        for (int x = 0; x < nsplit_total; ++x) M = fmaxf(M, __ldcg(pp + (size_t)x * (D + 2)));
        float L = 0.f;
        if (M != -INFINITY)
            for (int x = 0; x < nsplit_total; ++x)
                L += ex2(__ldcg(pp + (size_t)x * (D + 2)) - M) * __ldcg(pp + (size_t)x * (D + 2) + 1);
        sML[e] = M;
        sML[4 + e] = L;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < nh * D; x += blockDim.x) {
        const int e = x / D, c = x % D;
        const float M = sML[e], L = sML[4 + e];
        const float *pp = part + ((size_t)i * hq + j * hg + e0 + e) * g.smax * (D + 2);
        float a = 0.f;
        if (M != -INFINITY) {
            for (int y = 0; y < nsplit_total; ++y)
                a += ex2(__ldcg(pp + (size_t)y * (D + 2)) - M) * __ldcg(pp + (size_t)y * (D + 2) + 2 + c);
            a = a / L;
        }
        out[((size_t)i * hq + j * hg + e0 + e) * D + c] = __float2half_rn(a);
    }
}

template <int D, int KB, int VB, int SH>
cudaError_t launch_t(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, __half *out,
                     const DecodePlan &plan, cudaStream_t st) {
    const size_t smem = bar_region(plan.warps, plan.stages) + (size_t)plan.warps * warp_region(g, plan.stages);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, KB, VB, SH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.splits + plan.tails, g.h * plan.qgroups, g.b);
    decode_kernel<D, KB, VB, SH><<<grid, plan.warps * 32, smem, st>>>(g, dv, q, hq, out, plan);
    return cudaGetLastError();
}

template <int D, int KB, int VB>
cudaError_t launch_g(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, __half *out,
                     const DecodePlan &plan, cudaStream_t st) {
    switch (g.G) {
    case 16: return launch_t<D, KB, VB, 0>(g, dv, q, hq, out, plan, st);
    case 32: return launch_t<D, KB, VB, 1>(g, dv, q, hq, out, plan, st);
    case 64: return launch_t<D, KB, VB, 2>(g, dv, q, hq, out, plan, st);
    default:
        if constexpr (D >= 128) return launch_t<D, KB, VB, 3>(g, dv, q, hq, out, plan, st);
        return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_d(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, __half *out,
                     const DecodePlan &plan, cudaStream_t st) {
    if (g.kbits == 2 && g.vbits == 2) return launch_g<D, 2, 2>(g, dv, q, hq, out, plan, st);
    if (g.kbits == 2 && g.vbits == 4) return launch_g<D, 2, 4>(g, dv, q, hq, out, plan, st);
    if (g.kbits == 4 && g.vbits == 2) return launch_g<D, 4, 2>(g, dv, q, hq, out, plan, st);
    return launch_g<D, 4, 4>(g, dv, q, hq, out, plan, st);
}

}  // namespace
