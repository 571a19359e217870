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

// qcode_rcp for a bit width known at compile time, where rs is 0 whenever
// sf is 0 (then (x - z) * rs = 0 gives code 0, as qcode does).  For a
// group member the quotient lies in [0, 2 * 2^BITS) (below 2^BITS unless a
// subnormal fp16 scale rounded down), so the single margin 1e-5 * 2^BITS
// is at least the few ulps of |q| by which the product can miss the
// quotient: the IEEE division still decides every code next to a tie.
template <int BITS>
__device__ __forceinline__ uint32_t qcode_rcp_t(float x, float sf, float zf, float rs) {
    const float dlt = __fsub_rn(x, zf);
    const float q = __fmul_rn(dlt, rs);
    float k = rintf(q);
    if (fabsf(q - k) > 0.5f - 1.0e-5f * (float)(1 << BITS)) k = rintf(__fdiv_rn(dlt, sf));
    k = fminf(fmaxf(k, 0.0f), (float)((1 << BITS) - 1));
    return (uint32_t)k;
}

// ---------------------------------------------------------------------------
// Prefill keys: one CTA per (super block of TB = max(64, G) tokens, kv head,
// sequence).  Quantizes tokens [0, nqk), nqk = t - t mod R.
// ---------------------------------------------------------------------------
template <int KBITS, int G>
__global__ void __launch_bounds__(256) prefill_keys_kernel(KiviGeom g, KiviDev dv,
                                                           const __half *__restrict__ K,
                                                           SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int TB = G > KIVI_KBLK ? G : KIVI_KBLK;
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqk = t - t % g.R;
    const int tok0 = sb * TB;
    if (tok0 >= nqk) return;
    const int d = g.d, xsd = xs_stride(d);
    const int ntok = min(TB, nqk - tok0);   // a multiple of G
    const int ngr = ntok / G;

    __half *xs = reinterpret_cast<__half *>(smem);                        // [TB][xsd]
    float *sfz = reinterpret_cast<float *>(smem + (size_t)TB * xsd * 2);  // [TB/G][3][d]: s, z, 1/s

    // stage the tile (16-byte vectors)
    const __half *src = K + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    const int vpr = d / 8;   // vectors per row
    for (int e = threadIdx.x; e < ntok * vpr; e += blockDim.x) {
        const int r = e / vpr, c = e - r * vpr;
        reinterpret_cast<uint4 *>(xs + (size_t)r * xsd)[c] = reinterpret_cast<const uint4 *>(src)[e];
    }
    __syncthreads();

    // scale and zero per (group, channel): the min / max of fp16 values is
    // exact in fp16, taken two channels at a time
    const int dp = d / 2;
    for (int e = threadIdx.x; e < ngr * dp; e += blockDim.x) {
        const int gr = e / dp, c = 2 * (e - gr * dp);
        const __half2 *col = reinterpret_cast<const __half2 *>(xs + (size_t)gr * G * xsd + c);
        __half2 mn = col[0], mx = mn;
#pragma unroll 8
        for (int k = 1; k < G; ++k) {
            const __half2 x = col[(size_t)k * (xsd / 2)];
            mn = __hmin2(mn, x);
            mx = __hmax2(mx, x);
        }
        const float2 mnf = __half22float2(mn), mxf = __half22float2(mx);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const QParams p = qparams(h ? mnf.y : mnf.x, h ? mxf.y : mxf.x, KBITS);
            ksz_store(g, dv.blk, i, j, tok0 / G + gr, c + h, p.s16, p.z16);
            sfz[(gr * 3 + 0) * d + c + h] = p.sf;
            sfz[(gr * 3 + 1) * d + c + h] = p.zf;
            sfz[(gr * 3 + 2) * d + c + h] = p.sf == 0.0f ? 0.0f : __frcp_rn(p.sf);
        }
    }
    __syncthreads();

    // packed words of every 64-token block that starts inside [tok0, nqk)
    constexpr int cph = 16 / KBITS;
    const int kc_blk = g.kc_blk;
    const int nblk = (ntok + KIVI_KBLK - 1) / KIVI_KBLK;
    for (int e = threadIdx.x; e < nblk * kc_blk; e += blockDim.x) {
        const int kbl = e / kc_blk, wb = e - kbl * kc_blk;
        const KWord kw = kword_decode(wb, KBITS);
        // Slot r holds token trow + 8 r + g (g < 8).  trow is a multiple of
        // 32, and of G whenever G <= 32; for G >= 64 the word's tokens lie
        // in one group.  So slot r's group is trow / G + (8 r) / G: a
        // compile-time step, and slots of one group share their loads.
        const int trow = kbl * KIVI_KBLK + 8 * kw.pos0;
        const float *fw = sfz + (size_t)(trow / G) * 3 * d + kw.c0;
        uint32_t word = 0;
#pragma unroll
        for (int r = 0; r < cph; ++r) {
            // slot r of both halves: token tl, channels c0 and c0 + 1
            const int tl = trow + 8 * r + kw.g;   // token within the tile
            if (tl < ntok) {
                const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(xs + (size_t)tl * xsd + kw.c0));
                const float *f = fw + (size_t)((8 * r) / G) * 3 * d;
                word |= qcode_rcp_t<KBITS>(x.x, f[0], f[d], f[2 * d]) << (r * KBITS);
                word |= qcode_rcp_t<KBITS>(x.y, f[1], f[d + 1], f[2 * d + 1]) << (16 + r * KBITS);
            }
        }
        kc_words(g, dv.blk, i, j, tok0 / KIVI_KBLK + kbl)[wb] = word;
    }
}

// ---------------------------------------------------------------------------
// Prefill values: one CTA per (64 tokens = 4 value blocks, kv head,
// sequence).  Quantizes tokens [0, nqv), nqv = max(t - R, 0).
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
    const int d = g.d, ngi = d / G, xsd = xs_stride(d);
    const int ntok = min(64, nqv - tok0);
    __half *xs = reinterpret_cast<__half *>(smem);                         // [64][xsd]
    float *sfz = reinterpret_cast<float *>(smem + (size_t)64 * xsd * 2);   // [64][3][ngi]: s, z, 1/s

    const __half *src = V + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    const int vpr = d / 8;
    for (int e = threadIdx.x; e < ntok * vpr; e += blockDim.x) {
        const int r = e / vpr, c = e - r * vpr;
        reinterpret_cast<uint4 *>(xs + (size_t)r * xsd)[c] = reinterpret_cast<const uint4 *>(src)[e];
    }
    __syncthreads();

    const int nvblk = (ntok + KIVI_VBLK - 1) / KIVI_VBLK;   // value blocks touched
    for (int e = threadIdx.x; e < nvblk * KIVI_VBLK * ngi; e += blockDim.x) {
        const int tl = e / ngi, gi = e - tl * ngi;
        const int tau = tok0 + tl;
        __half s16 = __float2half_rn(0.f), z16 = s16;
        if (tl < ntok) {
            // fp16 min / max (exact), two channels at a time; the scan
            // starts at a token-dependent offset so that the warp's threads
            // read different banks
            const __half2 *x = reinterpret_cast<const __half2 *>(xs + (size_t)tl * xsd + gi * G);
            constexpr int GP = G / 2;
            const int rot = tl & (GP - 1);
            __half2 mn2 = x[rot], mx2 = mn2;
#pragma unroll 8
            for (int k = 1; k < GP; ++k) {
                const __half2 v = x[(k + rot) & (GP - 1)];
                mn2 = __hmin2(mn2, v);
                mx2 = __hmax2(mx2, v);
            }
            const float mn = fminf(__low2float(mn2), __high2float(mn2));
            const float mx = fmaxf(__low2float(mx2), __high2float(mx2));
            const QParams p = qparams(mn, mx, VBITS);
            s16 = p.s16;
            z16 = p.z16;
            sfz[(tl * 3 + 0) * ngi + gi] = p.sf;
            sfz[(tl * 3 + 1) * ngi + gi] = p.zf;
            sfz[(tl * 3 + 2) * ngi + gi] = p.sf == 0.0f ? 0.0f : __frcp_rn(p.sf);
        }
        __half *vsz = vsz_halves(g, dv.blk, i, j, tau >> 4);
        vsz[vsz_in_block(g, tau, gi, 0)] = s16;   // tokens past nqv: zero
        vsz[vsz_in_block(g, tau, gi, 1)] = z16;
    }
    __syncthreads();

    const int cs = v_cs(g);
    constexpr int cph = 16 / VBITS;
    const int vc_blk = g.vc_blk;
    for (int e = threadIdx.x; e < nvblk * vc_blk; e += blockDim.x) {
        const int vbl = e / vc_blk, wb = e - vbl * vc_blk;
        const VWord vw = vword_decode(wb, d, VBITS, cs);
        // Slot r holds channel 8 (ci0 + r) + g (g < 8); 8 ci0 is a multiple
        // of 32, and of G whenever G <= 32; for G >= 64 the word's channels
        // lie in one group.  So slot r's group is 8 ci0 / G + (8 r) / G.
        const int gi0 = 8 * vw.ci0 / G;
        uint32_t word = 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int tl = vbl * KIVI_VBLK + vw.tt0 + half;
            if (tl >= ntok) continue;
            const float *ft = sfz + (size_t)tl * 3 * ngi + gi0;
#pragma unroll
            for (int r = 0; r < cph; ++r) {
                const int c = 8 * (vw.ci0 + r) + vw.g;
                const float x = __half2float(xs[(size_t)tl * xsd + c]);
                const float *f = ft + (8 * r) / G;
                word |= qcode_rcp_t<VBITS>(x, f[0], f[ngi], f[2 * ngi]) << (16 * half + r * VBITS);
            }
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
        const size_t smv = (size_t)64 * xsd * 2 + (size_t)64 * 3 * (g.d / G) * 4;
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
