// kivi_prefill_attn.cu -- causal prefill attention over the prompt's fp16
// keys and values, with the cache's quantize-and-pack in its epilogue.
//
// Method: "Literature audit -- Group 2", section 1 KIVI.  Its list of
// supported backends runs the prefill's attention in full precision (flash
// attention on the unquantized K/V) and fills the quantized cache
// afterwards; its limitations paragraph lists that unfused quantization as
// open.  This kernel does both in one pass over K and V: the attention of
// core-algorithm item 5's formula with a causal mask over the raw fp16 keys
// and values, and, in the epilogue of the CTA that holds a 64-token tile of
// K and V for its own query rows (its diagonal tile), the prefill split and
// packing of items 2-4 for that tile.
//
// Layout.  A CTA computes 64 query rows of one query head (4 warps, 16 rows
// each) and walks the key tiles 0..(its own) with an online softmax
// (flash-attention style): scores and P V on m16n8k16 fp16 MMAs with fp32
// accumulation, P rounded to fp16 for the second product.  K and V tiles
// are double-buffered in shared memory by asynchronous 16-byte copies, in a
// swizzled layout (16-byte chunk c of row r at chunk c ^ (r mod 8)) that
// keeps the ldmatrix reads free of bank conflicts.  Grid: (query tiles,
// query heads, sequences), the longest tiles first.
#include "kivi_mma.cuh"
#include "kivi_pack_impl.cuh"

namespace {

constexpr int kTileRows = 64;   // query rows and keys per tile

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// halves offset of 16-byte chunk c of row r in a swizzled [64][D] tile
template <int D>
__device__ __forceinline__ int swz(int r, int c) {
    return r * D + ((c ^ (r & 7)) << 3);
}

// rows [0, valid) of a [64][D] tile from src (rows D apart), the rest zero
template <int D>
__device__ __forceinline__ void load_tile(__half *dst, const __half *src, int valid) {
    constexpr int CPR = D / 8;
    const int last = valid > 0 ? valid - 1 : 0;
    for (int e = threadIdx.x; e < kTileRows * CPR; e += blockDim.x) {
        const int r = e / CPR, c = e - r * CPR;
        cp_async16(dst + swz<D>(r, c), src + (size_t)min(r, last) * D + 8 * c, r < valid);
    }
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The cache's share of the diagonal tile [tb, tb + 64) of (sequence i, kv
// head j): keys [tb, nqk) and values [tb, nqv) packed by the prefill pack
// kernels' tile routines, window tokens copied to their fp16 slots.  kt, vt:
// the swizzled K and V tiles; work: free shared memory for the staging.
template <int D, int KB, int VB, int G>
__device__ void pack_diagonal(const KiviGeom &g, const KiviDev &dv, const __half *kt, const __half *vt,
                              unsigned char *work, int i, int j, int tb, int t) {
    constexpr int CPR = D / 8;
    const int nqk = t - t % g.R, nqv = t > g.R ? t - g.R : 0;
    // the tile routines see the tokens past the quantized range as zeros,
    // as the prefill pack kernels stage them
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    if (tb < nqk) {
        const int ntk = min(kTileRows, nqk - tb);
        __half *xs = reinterpret_cast<__half *>(work);   // [64][key_xsd(D)]
        float *sfz = reinterpret_cast<float *>(work + (size_t)kTileRows * key_xsd(D) * 2);
        for (int e = threadIdx.x; e < kTileRows * CPR; e += blockDim.x) {
            const int r = e / CPR, c = e - r * CPR;
            *reinterpret_cast<uint4 *>(xs + (size_t)r * key_xsd(D) + 8 * c) =
                r < ntk ? *reinterpret_cast<const uint4 *>(kt + swz<D>(r, c)) : zero;
        }
        __syncthreads();
        pack_key_tile<KB, G, D>(xs, sfz, ntk, dv.blk + rec_off(g, i, j, tb / KIVI_KBLK), g.rec_bytes, g.off_ksz);
        __syncthreads();   // the staging is reused below
    }
    if (tb < nqv) {
        const int ntv = min(kTileRows, nqv - tb);
        uint32_t *xs2 = reinterpret_cast<uint32_t *>(work);   // [32][value_ps(D)] token pairs
        float2 *sfz = reinterpret_cast<float2 *>(work + (size_t)32 * value_ps(D) * 4);
        for (int e = threadIdx.x; e < 32 * CPR; e += blockDim.x) {
            const int k = e / CPR, c = e - k * CPR;
            const uint4 a = 2 * k < ntv ? *reinterpret_cast<const uint4 *>(vt + swz<D>(2 * k, c)) : zero;
            const uint4 b = 2 * k + 1 < ntv ? *reinterpret_cast<const uint4 *>(vt + swz<D>(2 * k + 1, c)) : zero;
            uint4 lo, hi;
            lo.x = __byte_perm(a.x, b.x, 0x5410);
            lo.y = __byte_perm(a.x, b.x, 0x7632);
            lo.z = __byte_perm(a.y, b.y, 0x5410);
            lo.w = __byte_perm(a.y, b.y, 0x7632);
            hi.x = __byte_perm(a.z, b.z, 0x5410);
            hi.y = __byte_perm(a.z, b.z, 0x7632);
            hi.z = __byte_perm(a.w, b.w, 0x5410);
            hi.w = __byte_perm(a.w, b.w, 0x7632);
            uint4 *dst = reinterpret_cast<uint4 *>(xs2 + (size_t)k * value_ps(D) + 8 * c);
            dst[0] = lo;
            dst[1] = hi;
        }
        __syncthreads();
        pack_value_tile<VB, G, D>(xs2, sfz, ntv, tb, g, dv, i, j);
    }
    // window tokens of the tile: keys [nqk, t) to slot tau mod R, values
    // [nqv, t) to slot tau mod (R + 1)
    const int te = min(tb + kTileRows, t);
    uint4 *kf = reinterpret_cast<uint4 *>(dv.Kf + kf_slice(g, i, j));
    uint4 *vf = reinterpret_cast<uint4 *>(dv.Vf + vf_slice(g, i, j));
    for (int e = threadIdx.x; e < (te - tb) * CPR; e += blockDim.x) {
        const int tau = tb + e / CPR, c = e % CPR;
        if (tau >= nqk)
            kf[(size_t)(tau % g.R) * CPR + c] = *reinterpret_cast<const uint4 *>(kt + swz<D>(tau - tb, c));
        if (tau >= nqv)
            vf[(size_t)(tau % (g.R + 1)) * CPR + c] = *reinterpret_cast<const uint4 *>(vt + swz<D>(tau - tb, c));
    }
}

template <int D, int KB, int VB>
__device__ void pack_diagonal_g(const KiviGeom &g, const KiviDev &dv, const __half *kt, const __half *vt,
                                unsigned char *work, int i, int j, int tb, int t) {
    switch (g.G) {
    case 16: pack_diagonal<D, KB, VB, 16>(g, dv, kt, vt, work, i, j, tb, t); break;
    case 32: pack_diagonal<D, KB, VB, 32>(g, dv, kt, vt, work, i, j, tb, t); break;
    default: pack_diagonal<D, KB, VB, 64>(g, dv, kt, vt, work, i, j, tb, t); break;
    }
}

// Q, O: fp16 [b][hq][t_stride][D]; K, V: fp16 [b][h_kv][t_stride][D].
template <int D>
__global__ void __launch_bounds__(128, 2)
    prefill_attn_kernel(KiviGeom g, KiviDev dv, const __half *__restrict__ Q, const __half *__restrict__ K,
                        const __half *__restrict__ V, __half *__restrict__ O, SeqLens lens, int t_stride,
                        int hq) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int TILE = kTileRows * D;   // halves
    constexpr int NK = D / 16, NO = D / 8;
    // [stage 0: K, V][Q][stage 1: K, V]: once the loop is over, the stage
    // not holding the diagonal tile and Q's are one free stretch of 3 tiles
    __half *st0 = reinterpret_cast<__half *>(smem);
    __half *sq = st0 + 2 * TILE;
    __half *st1 = sq + TILE;
    const int qt = gridDim.x - 1 - blockIdx.x;   // the longest tiles first
    const int h = blockIdx.y, i = blockIdx.z;
    const int hg = hq / g.h, j = h / hg;
    const int t = lens.t[i];
    const int tb = qt * kTileRows;
    if (tb >= t) {
        if (tb == 0 && h == 0 && threadIdx.x == 0) {   // an empty sequence
            dv.T[i] = 0;
            dv.Tqk[i] = 0;
            dv.Tqv[i] = 0;
        }
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
    const __half *kbase = K + ((size_t)i * g.h + j) * t_stride * D;
    const __half *vbase = V + ((size_t)i * g.h + j) * t_stride * D;
    load_tile<D>(sq, Q + (((size_t)i * hq + h) * t_stride + tb) * D, min(kTileRows, t - tb));
    load_tile<D>(st0, kbase, min(kTileRows, t));
    load_tile<D>(st0 + TILE, vbase, min(kTileRows, t));
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // the warp's 16 query rows as A fragments
    uint32_t qa[NK][4];
#pragma unroll
    for (int kk = 0; kk < NK; ++kk)
        ldsm_x4(qa[kk], sq + swz<D>(warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * kk + (lane >> 4)));

    const float sl2 = 1.4426950408889634f / sqrtf((float)D);   // log2(e) / sqrt(d)
    float o[NO][4];
#pragma unroll
    for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    const int row0 = tb + warp * 16 + gq;   // rows row0 and row0 + 8

    for (int kt = 0; kt <= qt; ++kt) {
        const __half *ks = (kt & 1) ? st1 : st0;
        const __half *vs = ks + TILE;
        if (kt < qt) {   // the next tile streams in while this one is used
            __half *kn = (kt & 1) ? st0 : st1;
            const int nb = (kt + 1) * kTileRows;
            load_tile<D>(kn, kbase + (size_t)nb * D, min(kTileRows, t - nb));
            load_tile<D>(kn + TILE, vbase + (size_t)nb * D, min(kTileRows, t - nb));
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // scores of the warp's 16 rows against the tile's 64 keys
        float sc[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < NK; ++kk)
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                uint32_t b[4];
                ldsm_x4(b, ks + swz<D>(16 * p + (lane & 7) + 8 * (lane >> 4), 2 * kk + ((lane >> 3) & 1)));
                mma16816(sc[2 * p], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b[0], b[1]);
                mma16816(sc[2 * p + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b[2], b[3]);
            }
        if (kt == qt) {   // causal mask: key > row
#pragma unroll
            for (int n = 0; n < 8; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (tb + 8 * n + 2 * tq + (e & 1) > row0 + 8 * (e >> 1)) sc[n][e] = -INFINITY;
        }
        // online softmax (base 2): new row maxima over the quad's 16 keys each
        float mx0 = mrow[0], mx1 = mrow[1];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
            mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float al0 = ex2((mrow[0] - mx0) * sl2), al1 = ex2((mrow[1] - mx1) * sl2);
        mrow[0] = mx0;
        mrow[1] = mx1;
        const float ms0 = mx0 * sl2, ms1 = mx1 * sl2;
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            sc[n][0] = ex2(fmaf(sc[n][0], sl2, -ms0));
            sc[n][1] = ex2(fmaf(sc[n][1], sl2, -ms0));
            sc[n][2] = ex2(fmaf(sc[n][2], sl2, -ms1));
            sc[n][3] = ex2(fmaf(sc[n][3], sl2, -ms1));
            ls0 += sc[n][0] + sc[n][1];
            ls1 += sc[n][2] + sc[n][3];
        }
        lrow[0] = fmaf(lrow[0], al0, ls0);
        lrow[1] = fmaf(lrow[1], al1, ls1);
#pragma unroll
        for (int n = 0; n < NO; ++n) {
            o[n][0] *= al0;
            o[n][1] *= al0;
            o[n][2] *= al1;
            o[n][3] *= al1;
        }
        // P V: P (fp16) as the A operand, 16 keys per step
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a0 = pack_h2(sc[2 * kk][0], sc[2 * kk][1]);
            const uint32_t a1 = pack_h2(sc[2 * kk][2], sc[2 * kk][3]);
            const uint32_t a2 = pack_h2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            const uint32_t a3 = pack_h2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
            for (int nn = 0; nn < NO / 2; ++nn) {
                uint32_t b[4];
                ldsm_x4_t(b, vs + swz<D>(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * nn + (lane >> 4)));
                mma16816(o[2 * nn], a0, a1, a2, a3, b[0], b[1]);
                mma16816(o[2 * nn + 1], a0, a1, a2, a3, b[2], b[3]);
            }
        }
        __syncthreads();   // the stage is refilled two tiles on
    }

    // rows' sums over the quad, then the output rows inside the sequence
    float l0 = lrow[0], l1 = lrow[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float r0 = 1.f / l0, r1 = 1.f / l1;
    __half *orow = O + (((size_t)i * hq + h) * t_stride + row0) * D + 2 * tq;
#pragma unroll
    for (int n = 0; n < NO; ++n) {
        if (row0 < t) *reinterpret_cast<uint32_t *>(orow + 8 * n) = pack_h2(o[n][0] * r0, o[n][1] * r0);
        if (row0 + 8 < t)
            *reinterpret_cast<uint32_t *>(orow + (size_t)8 * D + 8 * n) = pack_h2(o[n][2] * r1, o[n][3] * r1);
    }

    // epilogue: the first query head of each kv head packs its diagonal tile
    if (h % hg == 0) {
        const __half *kd = (qt & 1) ? st1 : st0;
        unsigned char *work = reinterpret_cast<unsigned char *>((qt & 1) ? st0 : sq);
        if (g.kbits == 2 && g.vbits == 2) pack_diagonal_g<D, 2, 2>(g, dv, kd, kd + TILE, work, i, j, tb, t);
        else if (g.kbits == 2) pack_diagonal_g<D, 2, 4>(g, dv, kd, kd + TILE, work, i, j, tb, t);
        else if (g.vbits == 2) pack_diagonal_g<D, 4, 2>(g, dv, kd, kd + TILE, work, i, j, tb, t);
        else pack_diagonal_g<D, 4, 4>(g, dv, kd, kd + TILE, work, i, j, tb, t);
        if (tb == 0 && j == 0 && threadIdx.x == 0) {
            dv.T[i] = t;
            dv.Tqk[i] = t - t % g.R;
            dv.Tqv[i] = t > g.R ? t - g.R : 0;
        }
    }
}

template <int D>
cudaError_t launch_d(const KiviGeom &g, const KiviDev &dv, const __half *Q, const __half *K, const __half *V,
                     __half *O, const SeqLens &lens, int t_stride, int hq, int maxt, cudaStream_t st) {
    const size_t smem = (size_t)5 * kTileRows * D * 2;
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int nqt = maxt > 0 ? (maxt + kTileRows - 1) / kTileRows : 1;
    prefill_attn_kernel<D><<<dim3(nqt, hq, g.b), 128, smem, st>>>(g, dv, Q, K, V, O, lens, t_stride, hq);
    return cudaGetLastError();
}

}  // namespace

cudaError_t kivi_launch_prefill_attn(const KiviGeom &g, const KiviDev &dv, const __half *Q, const __half *K,
                                     const __half *V, __half *O, const SeqLens &lens, int t_stride, int hq,
                                     cudaStream_t st) {
    if (g.G > 64 || (g.d != 64 && g.d != 128)) return cudaErrorInvalidValue;
    int maxt = 0;
    for (int i = 0; i < g.b; ++i) maxt = lens.t[i] > maxt ? lens.t[i] : maxt;
    return g.d == 64 ? launch_d<64>(g, dv, Q, K, V, O, lens, t_stride, hq, maxt, st)
                     : launch_d<128>(g, dv, Q, K, V, O, lens, t_stride, hq, maxt, st);
}
