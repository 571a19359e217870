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
#include "kivi_pack_impl.cuh"

namespace {

__device__ __forceinline__ void flag(unsigned *status, unsigned f) { atomicOr(status, f); }

// ---------------------------------------------------------------------------
// Prefill keys: one CTA per (tile of TB = max(64, G) tokens, kv head,
// sequence).  Quantizes tokens [0, nqk), nqk = t - t mod R: the tile is
// staged with asynchronous 16-byte copies (rows past the quantized range
// zero-filled), then pack_key_tile.
// ---------------------------------------------------------------------------
template <int KBITS, int G, int D>
__global__ void __launch_bounds__(256) prefill_keys_kernel(KiviGeom g, KiviDev dv,
                                                           const __half *__restrict__ K,
                                                           SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int TB = G > KIVI_KBLK ? G : KIVI_KBLK;
    constexpr int xsd = key_xsd(D);
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqk = t - t % g.R;
    const int tok0 = sb * TB;
    if (tok0 >= nqk) return;
    const int ntok = min(TB, nqk - tok0);   // a multiple of G
    __half *xs = reinterpret_cast<__half *>(smem);                        // [TB][xsd]
    float *sfz = reinterpret_cast<float *>(smem + (size_t)TB * xsd * 2);  // [TB / G][3][D]
    const __half *src = K + (((size_t)i * g.h + j) * t_stride + tok0) * D;
    constexpr int vpr = D / 8;   // 16-byte pieces per row
    for (int e = threadIdx.x; e < TB * vpr; e += blockDim.x) {
        const int r = e / vpr, c = e - r * vpr;
        cp_async16(xs + (size_t)r * xsd + 8 * c, src + (size_t)min(r, ntok - 1) * D + 8 * c, r < ntok);
    }
    cp_async_wait_all();
    __syncthreads();
    pack_key_tile<KBITS, G, D>(xs, sfz, ntok, dv.blk + rec_off(g, i, j, tok0 / KIVI_KBLK), g.rec_bytes, g.off_ksz);
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
template <int VBITS, int G, int D>
__global__ void __launch_bounds__(256) prefill_values_kernel(KiviGeom g, KiviDev dv,
                                                             const __half *__restrict__ V,
                                                             SeqLens lens, int t_stride) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int sb = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int t = lens.t[i];
    const int nqv = t > g.R ? t - g.R : 0;
    const int tok0 = sb * 64;
    if (tok0 >= nqv) return;
    constexpr int d = D;
    constexpr int ps = value_ps(D);   // pair row stride in 32-bit words (padded)
    const int ntok = min(64, nqv - tok0);
    uint32_t *xs2 = reinterpret_cast<uint32_t *>(smem);                    // [32][ps] half2 pairs
    float2 *sfz = reinterpret_cast<float2 *>(smem + (size_t)32 * ps * 4);  // [32][3][D / G]: s, z, 1/s pairs

    // stage: rows 2k and 2k + 1, 8 channels at a time, interleaved by halves
    const __half *src = V + (((size_t)i * g.h + j) * t_stride + tok0) * d;
    constexpr int vpr = d / 8;
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

    pack_value_tile<VBITS, G, D>(xs2, sfz, ntok, tok0, g, dv, i, j);
}

template <int BITS, int G, int D>
cudaError_t launch_prefill_kvd(const KiviGeom &g, const KiviDev &dv, const __half *K, const __half *V,
                               const SeqLens &lens, int t_stride, int maxt, cudaStream_t st) {
    constexpr int TB = G > KIVI_KBLK ? G : KIVI_KBLK;
    cudaError_t e = cudaSuccess;
    if (g.kbits == BITS) {
        const size_t smk = (size_t)TB * key_xsd(D) * 2 + (size_t)(TB / G) * 3 * D * 4;
        e = cudaFuncSetAttribute(prefill_keys_kernel<BITS, G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smk);
        if (e != cudaSuccess) return e;
        prefill_keys_kernel<BITS, G, D><<<dim3((maxt + TB - 1) / TB, g.h, g.b), 256, smk, st>>>(g, dv, K, lens,
                                                                                              t_stride);
    }
    if (g.vbits == BITS) {
        const size_t smv = (size_t)32 * (D + 4) * 4 + (size_t)32 * 3 * (D / G) * 8;
        e = cudaFuncSetAttribute(prefill_values_kernel<BITS, G, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smv);
        if (e != cudaSuccess) return e;
        prefill_values_kernel<BITS, G, D><<<dim3((maxt + 63) / 64, g.h, g.b), 256, smv, st>>>(g, dv, V, lens,
                                                                                            t_stride);
    }
    return cudaGetLastError();
}

template <int G, int D>
cudaError_t launch_prefill_gd(const KiviGeom &g, const KiviDev &dv, const __half *K, const __half *V,
                              const SeqLens &lens, int t_stride, int maxt, cudaStream_t st) {
    cudaError_t e = launch_prefill_kvd<2, G, D>(g, dv, K, V, lens, t_stride, maxt, st);
    if (e != cudaSuccess) return e;
    return launch_prefill_kvd<4, G, D>(g, dv, K, V, lens, t_stride, maxt, st);
}

template <int G>
cudaError_t launch_prefill_g(const KiviGeom &g, const KiviDev &dv, const __half *K, const __half *V,
                             const SeqLens &lens, int t_stride, int maxt, cudaStream_t st) {
    switch (g.d) {
    case 64:
        if constexpr (G <= 64) return launch_prefill_gd<G, 64>(g, dv, K, V, lens, t_stride, maxt, st);
        return cudaErrorInvalidValue;
    case 128: return launch_prefill_gd<G, 128>(g, dv, K, V, lens, t_stride, maxt, st);
    default: return launch_prefill_gd<G, 256>(g, dv, K, V, lens, t_stride, maxt, st);
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
    }
}

// ---------------------------------------------------------------------------
// Append: one CTA per (kv head, sequence; grid row y is sequence
// ac.order[y], the flushing ones first): append_pair (kivi_append_impl.cuh),
// then the last CTA of a sequence to finish advances that sequence's
// counters (all CTAs read them first).
// ---------------------------------------------------------------------------
// One CTA per (kv head j, sequence i).  The counters before the append come
// from the host mirror (ac); the device's current set is read only to check
// that the two agree.  CTA j = 0 of each sequence writes the counters after
// the append into the other set (nxt), so no CTA waits for another.
// only_flush: sequences whose key window is not full are left to the fused
// decode launch that follows (their CTAs return at once).
__global__ void __launch_bounds__(1024) append_kernel(KiviGeom g, KiviDev dv,
                                                     const __half *__restrict__ knew,
                                                     const __half *__restrict__ vnew, AppendCounters ac,
                                                     int *__restrict__ nxt, int only_flush) {
    // the decode launch that usually follows may start its set-up now: it
    // waits for this whole grid before it reads anything
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int j = blockIdx.x, i = ac.order[blockIdx.y];
    const int R = g.R;
    const int T = ac.T[i], Tqk = ac.Tqk[i], Tqv = ac.Tqv[i];
    if (only_flush && T - Tqk != R) return;
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
                               const __half *v, const AppendCounters &ac, int *nxt, cudaStream_t st,
                               bool only_flush) {
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
    append_kernel<<<dim3(g.h, g.b), flush ? 1024 : 256, smem, st>>>(g, dv, k, v, ac, nxt, only_flush ? 1 : 0);
    return cudaGetLastError();
}
