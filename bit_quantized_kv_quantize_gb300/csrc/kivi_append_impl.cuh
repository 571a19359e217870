// kivi_append_impl.cuh -- the append step of one (sequence, kv head) slice:
// the lazy maintenance of the residual windows, then the new token.
//
// Method: "Literature audit -- Group 2", section 1 KIVI, core algorithm
// item 4: when the key window holds R tokens it is quantized as R / G
// per-channel groups (item 2) and emptied; when the value queue holds R + 1
// tokens its oldest token is quantized per token (item 3); then the new key
// and value join the windows.  The maintenance runs at the start of the
// append that finds the window full, so each step's attention sees its
// newest token in fp16.
#pragma once
#include "kivi_internal.cuh"

// Counters of one sequence before an append are in range.
__device__ __forceinline__ bool append_counters_ok(const KiviGeom &g, int T, int Tqk, int Tqv) {
    const int R = g.R;
    return T >= 0 && T < g.fcap && Tqk >= 0 && Tqk % R == 0 && T - Tqk >= 0 && T - Tqk <= R && Tqv >= 0 &&
           T - Tqv >= 0 && T - Tqv <= R + 1;
}

// Append the token (knew, vnew: fp16 [b][h][d]) to slice (i, j) whose
// counters are T, Tqk, Tqv (in range).  Called by every thread of a CTA (any
// block size); the counters themselves are left to the caller.
__device__ __forceinline__ void append_pair(const KiviGeom &g, const KiviDev &dv, const __half *__restrict__ knew,
                                            const __half *__restrict__ vnew, int i, int j, int T, int Tqk,
                                            int Tqv) {
    const int d = g.d, R = g.R;
    const bool flush = (T - Tqk) == R;
    const bool pop = (T - Tqv) == R + 1;
    // One round trip for the rows this step needs: the new key and value
    // (kept in registers, written last) and the value leaving the queue.
    const int nv8 = d / 8;   // 16-byte chunks per row
    __shared__ __align__(16) __half s_row[256];   // d <= 256
    uint4 kn_c = make_uint4(0u, 0u, 0u, 0u), vn_c = kn_c;
    if ((int)threadIdx.x < nv8) {
        kn_c = reinterpret_cast<const uint4 *>(knew + ((size_t)i * g.h + j) * d)[threadIdx.x];
        vn_c = reinterpret_cast<const uint4 *>(vnew + ((size_t)i * g.h + j) * d)[threadIdx.x];
        if (pop)
            reinterpret_cast<uint4 *>(s_row)[threadIdx.x] = reinterpret_cast<const uint4 *>(
                dv.Vf + vf_slice(g, i, j) + (size_t)(Tqv % (R + 1)) * d)[threadIdx.x];
    }
    const __half *kf = dv.Kf + kf_slice(g, i, j);
    __half *kfw = dv.Kf + kf_slice(g, i, j);
    __half *vfw = dv.Vf + vf_slice(g, i, j);

    // the flushed groups' scale and zero (fp32), when they fit
    constexpr int kSzCap = 2048;
    __shared__ float s_ks[kSzCap], s_kz[kSzCap];
    if (flush) {
        // keys [Tqk, Tqk + R): token tau lives in slot tau - Tqk (Tqk % R == 0)
        const int ngr = R / g.G;
        const bool sz_smem = ngr * d <= kSzCap;
        for (int e = threadIdx.x; e < ngr * d; e += blockDim.x) {
            int gr = e / d, c = e - gr * d;
            const __half *col = kf + (size_t)gr * g.G * d + c;
            float mn = __half2float(col[0]), mx = mn;
#pragma unroll 8
            for (int k = 1; k < g.G; ++k) {   // independent loads: several in flight
                float x = __half2float(col[(size_t)k * d]);
                mn = fminf(mn, x);
                mx = fmaxf(mx, x);
            }
            QParams p = qparams(mn, mx, g.kbits);
            ksz_store(g, dv.blk, i, j, Tqk / g.G + gr, c, p.s16, p.z16);
            if (sz_smem) {
                s_ks[e] = p.sf;
                s_kz[e] = p.zf;
            }
        }
        __syncthreads();
        const int kb0 = Tqk / KIVI_KBLK, kb1 = (Tqk + R - 1) / KIVI_KBLK;
        const int cph = 16 / g.kbits;
        for (int e = threadIdx.x; e < (kb1 - kb0 + 1) * g.kc_blk; e += blockDim.x) {
            int kb = kb0 + e / g.kc_blk, wb = e % g.kc_blk;
            KWord kw = kword_decode(wb, g.kbits);
            uint32_t *kc = kc_words(g, dv.blk, i, j, kb);
            uint32_t old = kc[wb];
            uint32_t word = 0;
            for (int half = 0; half < 2; ++half) {
                int c = kw.c0 + half;
#pragma unroll 8
                for (int r = 0; r < cph; ++r) {
                    int tau = kb * KIVI_KBLK + 8 * (kw.pos0 + r) + kw.g;
                    int sh = 16 * half + r * g.kbits;
                    uint32_t mask = ((1u << g.kbits) - 1u) << sh;
                    if (tau < Tqk) {
                        word |= old & mask;                     // earlier tokens stay
                    } else if (tau < Tqk + R) {
                        int grp = tau / g.G;
                        float sf, zf;
                        if (sz_smem) {   // the value ksz_store just wrote, as fp32
                            sf = s_ks[(grp - Tqk / g.G) * d + c];
                            zf = s_kz[(grp - Tqk / g.G) * d + c];
                        } else {
                            sf = __half2float(ksz_load(g, dv.blk, i, j, grp, c, 0));
                            zf = __half2float(ksz_load(g, dv.blk, i, j, grp, c, 1));
                        }
                        float x = __half2float(kf[(size_t)(tau - Tqk) * d + c]);
                        word |= qcode(x, sf, zf, g.kbits) << sh;
                    }                                           // later tokens: zero
                }
            }
            kc[wb] = word;
        }
    }

    if (pop) {
        // value token Tqv (slot Tqv % (R + 1)), staged in s_row
        const __half *x = s_row;
        const int ngi = d / g.G;
        const int vb = Tqv / KIVI_VBLK, tt = Tqv % KIVI_VBLK;
        __half *vsz = vsz_halves(g, dv.blk, i, j, vb);
        uint32_t *vc = vc_words(g, dv.blk, i, j, vb);
        if (tt == 0) {   // a fresh value block: clear it so untouched fields read zero
            for (int e = threadIdx.x; e < g.vc_blk; e += blockDim.x) vc[e] = 0u;
            for (int e = threadIdx.x; e < g.vsz_blk; e += blockDim.x) vsz[e] = __float2half_rn(0.f);
        }
        __shared__ float s_sf[16], s_zf[16];   // d / G <= 16
        __syncthreads();
        for (int gi = threadIdx.x; gi < ngi; gi += blockDim.x) {
            float mn = __half2float(x[gi * g.G]), mx = mn;
            for (int k = 1; k < g.G; ++k) {
                float v = __half2float(x[gi * g.G + k]);
                mn = fminf(mn, v);
                mx = fmaxf(mx, v);
            }
            QParams p = qparams(mn, mx, g.vbits);
            vsz[vsz_in_block(g, Tqv, gi, 0)] = p.s16;
            vsz[vsz_in_block(g, Tqv, gi, 1)] = p.z16;
            s_sf[gi] = p.sf;
            s_zf[gi] = p.zf;
        }
        __syncthreads();
        // the token's halves: lane class g (8) x channel words w (d vbits / 128)
        const int nwv = d * g.vbits / 128, cph = 16 / g.vbits, cs = v_cs(g);
        const int p = tt >> 3, tq = (tt & 7) >> 1, half = tt & 1;
        for (int e = threadIdx.x; e < 8 * nwv; e += blockDim.x) {
            int gg = e / nwv, w = e - gg * nwv;
            uint32_t bits = 0;
            for (int r = 0; r < cph; ++r) {
                int c = 8 * (w * cph + r) + gg;
                int gi = c / g.G;
                bits |= qcode(__half2float(x[c]), s_sf[gi], s_zf[gi], g.vbits) << (r * g.vbits);
            }
            int L = 4 * gg + tq, u = p * nwv + w;
            size_t wd = (size_t)(u / cs) * 32 * cs + (size_t)L * cs + (u % cs);
            reinterpret_cast<uint16_t *>(vc + wd)[half] = (uint16_t)bits;
        }
    }
    __syncthreads();   // maintenance has read the slots the new token overwrites

    if ((int)threadIdx.x < nv8) {
        reinterpret_cast<uint4 *>(kfw + (size_t)(T % R) * d)[threadIdx.x] = kn_c;
        reinterpret_cast<uint4 *>(vfw + (size_t)(T % (R + 1)) * d)[threadIdx.x] = vn_c;
    }
}
