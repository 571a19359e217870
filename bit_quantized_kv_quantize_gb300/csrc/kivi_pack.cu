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

// ---------------------------------------------------------------------------
// Prefill keys: one CTA per (super block of TB = max(64, G) tokens, kv head,
// sequence).  Quantizes tokens [0, nqk), nqk = t - t mod R.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prefill_keys_kernel(KiviGeom g, KiviDev dv,
                                                           const __half *__restrict__ K,
                                                           SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int TB = g.G > KIVI_KBLK ? g.G : KIVI_KBLK;
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqk = t - t % g.R;
    const int tok0 = sb * TB;
    if (tok0 >= nqk) return;
    const int d = g.d;
    const int ntok = min(TB, nqk - tok0);   // a multiple of G
    const int ngr = ntok / g.G;

    __half *xs = reinterpret_cast<__half *>(smem);                     // [TB][d]
    float *sfz = reinterpret_cast<float *>(smem + (size_t)TB * d * 2); // [TB/G][2][d]

    // stage the tile (16-byte vectors)
    const __half *src = K + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    const int nvec = ntok * d / 8;
    for (int e = threadIdx.x; e < nvec; e += blockDim.x)
        reinterpret_cast<uint4 *>(xs)[e] = reinterpret_cast<const uint4 *>(src)[e];
    __syncthreads();

    // scale and zero per (group, channel)
    for (int e = threadIdx.x; e < ngr * d; e += blockDim.x) {
        int gr = e / d, c = e - gr * d;
        float mn = __half2float(xs[(size_t)gr * g.G * d + c]), mx = mn;
        for (int k = 1; k < g.G; ++k) {
            float x = __half2float(xs[((size_t)gr * g.G + k) * d + c]);
            mn = fminf(mn, x);
            mx = fmaxf(mx, x);
        }
        QParams p = qparams(mn, mx, g.kbits);
        ksz_store(g, dv.blk, i, j, tok0 / g.G + gr, c, p.s16, p.z16);
        sfz[(gr * 2 + 0) * d + c] = p.sf;
        sfz[(gr * 2 + 1) * d + c] = p.zf;
    }
    __syncthreads();

    // packed words of every 64-token block that starts inside [tok0, nqk)
    const int nblk = (ntok + KIVI_KBLK - 1) / KIVI_KBLK;
    const int cph = 16 / g.kbits;
    for (int e = threadIdx.x; e < nblk * g.kc_blk; e += blockDim.x) {
        int kbl = e / g.kc_blk, wb = e - kbl * g.kc_blk;
        KWord kw = kword_decode(wb, g.kbits);
        uint32_t word = 0;
#pragma unroll 2
        for (int half = 0; half < 2; ++half) {
            int c = kw.c0 + half;
            for (int r = 0; r < cph; ++r) {
                int tl = kbl * KIVI_KBLK + 8 * (kw.pos0 + r) + kw.g;   // token within the tile
                if (tl < ntok) {
                    int gr = tl / g.G;
                    float x = __half2float(xs[(size_t)tl * d + c]);
                    uint32_t q = qcode(x, sfz[(gr * 2) * d + c], sfz[(gr * 2 + 1) * d + c], g.kbits);
                    word |= q << (16 * half + r * g.kbits);
                }
            }
        }
        kc_words(g, dv.blk, i, j, tok0 / KIVI_KBLK + kbl)[wb] = word;
    }
}

// ---------------------------------------------------------------------------
// Prefill values: one CTA per (64 tokens = 4 value blocks, kv head,
// sequence).  Quantizes tokens [0, nqv), nqv = max(t - R, 0).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) prefill_values_kernel(KiviGeom g, KiviDev dv,
                                                             const __half *__restrict__ V,
                                                             SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqv = t > g.R ? t - g.R : 0;
    const int tok0 = sb * 64;
    if (tok0 >= nqv) return;
    const int d = g.d, ngi = d / g.G;
    const int ntok = min(64, nqv - tok0);
    __half *xs = reinterpret_cast<__half *>(smem);                          // [64][d]
    float *sfz = reinterpret_cast<float *>(smem + (size_t)64 * d * 2);     // [64][2][ngi]

    const __half *src = V + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    for (int e = threadIdx.x; e < ntok * d / 8; e += blockDim.x)
        reinterpret_cast<uint4 *>(xs)[e] = reinterpret_cast<const uint4 *>(src)[e];
    __syncthreads();

    const int nvblk = (ntok + KIVI_VBLK - 1) / KIVI_VBLK;   // value blocks touched
    for (int e = threadIdx.x; e < nvblk * KIVI_VBLK * ngi; e += blockDim.x) {
        int tl = e / ngi, gi = e - tl * ngi;
        int tau = tok0 + tl;
        __half s16 = __float2half_rn(0.f), z16 = s16;
        if (tl < ntok) {
            const __half *x = xs + (size_t)tl * d + gi * g.G;
            float mn = __half2float(x[0]), mx = mn;
            for (int k = 1; k < g.G; ++k) {
                float v = __half2float(x[k]);
                mn = fminf(mn, v);
                mx = fmaxf(mx, v);
            }
            QParams p = qparams(mn, mx, g.vbits);
            s16 = p.s16;
            z16 = p.z16;
            sfz[(tl * 2 + 0) * ngi + gi] = p.sf;
            sfz[(tl * 2 + 1) * ngi + gi] = p.zf;
        }
        __half *vsz = vsz_halves(g, dv.blk, i, j, tau >> 4);
        vsz[vsz_in_block(g, tau, gi, 0)] = s16;   // tokens past nqv: zero
        vsz[vsz_in_block(g, tau, gi, 1)] = z16;
    }
    __syncthreads();

    const int cs = v_cs(g), cph = 16 / g.vbits;
    for (int e = threadIdx.x; e < nvblk * g.vc_blk; e += blockDim.x) {
        int vbl = e / g.vc_blk, wb = e - vbl * g.vc_blk;
        VWord vw = vword_decode(wb, d, g.vbits, cs);
        uint32_t word = 0;
        for (int half = 0; half < 2; ++half) {
            int tl = vbl * KIVI_VBLK + vw.tt0 + half;
            if (tl >= ntok) continue;
            for (int r = 0; r < cph; ++r) {
                int c = 8 * (vw.ci0 + r) + vw.g;
                int gi = c / g.G;
                float x = __half2float(xs[(size_t)tl * d + c]);
                uint32_t q = qcode(x, sfz[(tl * 2) * ngi + gi], sfz[(tl * 2 + 1) * ngi + gi], g.vbits);
                word |= q << (16 * half + r * g.vbits);
            }
        }
        vc_words(g, dv.blk, i, j, tok0 / KIVI_VBLK + vbl)[wb] = word;
    }
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
        dv.ticket[i] = 0u;
    }
}

// ---------------------------------------------------------------------------
// Append: one CTA per (kv head, sequence): append_pair (kivi_append_impl.cuh),
// then the last CTA of a sequence to finish advances that sequence's
// counters (all CTAs read them first).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) append_kernel(KiviGeom g, KiviDev dv,
                                                     const __half *__restrict__ knew,
                                                     const __half *__restrict__ vnew) {
    const int j = blockIdx.x, i = blockIdx.y;
    const int R = g.R;
    const int T = dv.T[i], Tqk = dv.Tqk[i], Tqv = dv.Tqv[i];
    if (!append_counters_ok(g, T, Tqk, Tqv)) {
        if (threadIdx.x == 0) flag(dv.status, KIVI_FLAG_COUNTER);
        return;
    }
    append_pair(g, dv, knew, vnew, i, j, T, Tqk, Tqv);

    // last CTA of this sequence advances the counters
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned prev = atomicAdd(&dv.ticket[i], 1u);
        if (prev == (unsigned)g.h - 1u) {
            dv.T[i] = T + 1;
            dv.Tqk[i] = Tqk + ((T - Tqk) == R ? R : 0);
            dv.Tqv[i] = Tqv + ((T - Tqv) == R + 1 ? 1 : 0);
            dv.ticket[i] = 0u;
            __threadfence();
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
        const int TB = g.G > KIVI_KBLK ? g.G : KIVI_KBLK;
        size_t smk = (size_t)TB * g.d * 2 + (size_t)(TB / g.G) * 2 * g.d * 4;
        cudaError_t e = cudaFuncSetAttribute(prefill_keys_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
        if (e != cudaSuccess) return e;
        dim3 gk((maxt + TB - 1) / TB, g.h, g.b);
        prefill_keys_kernel<<<gk, 256, smk, st>>>(g, dv, K, lens, t_stride);
        size_t smv = (size_t)64 * g.d * 2 + (size_t)64 * 2 * (g.d / g.G) * 4;
        e = cudaFuncSetAttribute(prefill_values_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smv);
        if (e != cudaSuccess) return e;
        dim3 gv((maxt + 63) / 64, g.h, g.b);
        prefill_values_kernel<<<gv, 256, smv, st>>>(g, dv, V, lens, t_stride);
    }
    prefill_residual_kernel<<<dim3(g.h, g.b), 256, 0, st>>>(g, dv, K, V, lens, t_stride);
    return cudaGetLastError();
}

cudaError_t kivi_launch_append(const KiviGeom &g, const KiviDev &dv, const __half *k,
                               const __half *v, cudaStream_t st) {
    append_kernel<<<dim3(g.h, g.b), 256, 0, st>>>(g, dv, k, v);
    return cudaGetLastError();
}
