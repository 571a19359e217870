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

    if (flush) {
        // Keys [Tqk, Tqk + R) (token tau in window slot tau - Tqk, as
        // Tqk % R == 0), one round of CH aligned tokens at a time
        // (flush_round_tokens: whole groups and 64-token blocks): the
        // round's window rows come into shared memory with one round trip,
        // then its groups get their scale and zero and its blocks their
        // code words.  Shared memory (dynamic, flush_smem_bytes): rows
        // [CH][d] fp16, then s, z and RN(1 / s) [CH/G][d] fp32.  G, d and
        // the block's word count are powers of two: indices are shifts and
        // masks.
        extern __shared__ __align__(16) unsigned char flush_smem[];
        const int G = g.G, CH = flush_round_tokens(g);
        const int CA = G > KIVI_KBLK ? G : KIVI_KBLK;   // alignment of a round's start
        const int lgG = __ffs(G) - 1, lgd = __ffs(d) - 1, lgw = __ffs(g.kc_blk) - 1;
        __half *xs = reinterpret_cast<__half *>(flush_smem);
        float *s_ks = reinterpret_cast<float *>(flush_smem + (size_t)CH * d * 2);
        float *s_kz = s_ks + (CH / G) * d;
        float *s_kr = s_kz + (CH / G) * d;
        const int nv = d / 8;   // 16-byte pieces per row
        const int cph = 16 / g.kbits;
        for (int cs = Tqk / CA * CA; cs < Tqk + R; cs += CH) {
            const int ta = max(cs, Tqk), tb = min(cs + CH, Tqk + R);   // multiples of G
            for (int e = threadIdx.x; e < (tb - ta) * nv; e += blockDim.x) {
                const int tau = ta + e / nv, c8 = e % nv;
                reinterpret_cast<uint4 *>(xs + (size_t)(tau - cs) * d)[c8] =
                    reinterpret_cast<const uint4 *>(kf + (size_t)(tau - Tqk) * d)[c8];
            }
            __syncthreads();
            const int gr0 = ta >> lgG, ngr = (tb - ta) >> lgG;
            for (int e = threadIdx.x; e < ngr * d; e += blockDim.x) {
                const int gr = e >> lgd, c = e & (d - 1);
                const __half *col = xs + (size_t)((gr0 + gr) * G - cs) * d + c;
                float mn = __half2float(col[0]), mx = mn;
                for (int k = 1; k < G; ++k) {
                    const float x = __half2float(col[(size_t)k * d]);
                    mn = fminf(mn, x);
                    mx = fmaxf(mx, x);
                }
                const QParams p = qparams(mn, mx, g.kbits);
                ksz_store(g, dv.blk, i, j, gr0 + gr, c, p.s16, p.z16);
                s_ks[e] = p.sf;
                s_kz[e] = p.zf;
                s_kr[e] = p.sf == 0.0f ? 0.0f : __frcp_rn(p.sf);
            }
            __syncthreads();
            const int kb0 = cs / KIVI_KBLK, nkb = CH / KIVI_KBLK;
            for (int e = threadIdx.x; e < nkb * g.kc_blk; e += blockDim.x) {
                const int kb = kb0 + (e >> lgw), wb = e & (g.kc_blk - 1);
                const int t0 = kb * KIVI_KBLK;
                if (t0 >= tb || t0 + KIVI_KBLK <= ta) continue;   // no window token in this block
                const KWord kw = kword_decode(wb, g.kbits);
                uint32_t *kc = kc_words(g, dv.blk, i, j, kb);
                const uint32_t old = t0 < Tqk ? kc[wb] : 0u;   // earlier tokens' codes stay
                uint32_t word = 0;
                for (int half = 0; half < 2; ++half) {
                    const int c = kw.c0 + half;
                    for (int r = 0; r < cph; ++r) {
                        const int tau = t0 + 8 * (kw.pos0 + r) + kw.g;
                        const int sh = 16 * half + r * g.kbits;
                        if (tau < Tqk) {
                            word |= old & (((1u << g.kbits) - 1u) << sh);
                        } else if (tau < tb) {   // later tokens: zero
                            const int sz = (((tau >> lgG) - gr0) << lgd) + c;
                            word |= qcode_rcp(__half2float(xs[((tau - cs) << lgd) + c]), s_ks[sz], s_kz[sz],
                                              s_kr[sz], g.kbits) << sh;
                        }
                    }
                }
                kc[wb] = word;
            }
            __syncthreads();   // the next chunk reuses the rows
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
