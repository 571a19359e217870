// kivi_prefill_attn.cu -- causal prefill attention over the prompt's fp16
// keys and values on the 5th-generation tensor cores, with the cache's
// quantize-and-pack in its epilogue.
//
// Method: "Literature audit -- Group 2", section 1 KIVI.  Its list of
// supported backends runs the prefill's attention in full precision (flash
// attention on the unquantized K/V) and fills the quantized cache
// afterwards; its limitations paragraph lists that unfused quantization as
// open.  This kernel does both in one pass over K and V: the attention of
// core-algorithm item 5's formula with a causal mask over the raw fp16 keys
// and values, and, in the epilogue of the CTA that holds the 64-token K and
// V tiles of its own query rows (its diagonal tiles), the prefill split and
// packing of items 2-4 for those tiles.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kivi_mma.cuh"
#include "kivi_pack_impl.cuh"
#include "kivi_tcgen05.cuh"

namespace {

constexpr int kTileRows = 64;   // tokens of a packed tile

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// byte offset of 16-byte chunk c of row r in a 64-row fp16 tile in the
// tensor cores' no-swizzle core-matrix layout, chunk-major (the attention
// kernel's layout below)
template <int D>
__device__ __forceinline__ int chunk_at(int r, int c) {
    return c * kTileRows * 16 + r * 16;
}

// The cache's share of the diagonal tile [tb, tb + 64) of (sequence i, kv
// head j): keys [tb, nqk) and values [tb, nqv) packed by the prefill pack
// kernels' tile routines, window tokens copied to their fp16 slots.  kt, vt:
// the K and V tiles (core-matrix layout); work: free shared memory for the
// staging.
template <int D, int KB, int VB, int G>
__device__ void pack_diagonal(const KiviGeom &g, const KiviDev &dv, const unsigned char *kt, const unsigned char *vt,
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
                r < ntk ? *reinterpret_cast<const uint4 *>(kt + chunk_at<D>(r, c)) : zero;
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
            const uint4 a = 2 * k < ntv ? *reinterpret_cast<const uint4 *>(vt + chunk_at<D>(2 * k, c)) : zero;
            const uint4 b =
                2 * k + 1 < ntv ? *reinterpret_cast<const uint4 *>(vt + chunk_at<D>(2 * k + 1, c)) : zero;
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
            kf[(size_t)(tau % g.R) * CPR + c] = *reinterpret_cast<const uint4 *>(kt + chunk_at<D>(tau - tb, c));
        if (tau >= nqv)
            vf[(size_t)(tau % (g.R + 1)) * CPR + c] =
                *reinterpret_cast<const uint4 *>(vt + chunk_at<D>(tau - tb, c));
    }
}

template <int D, int KB, int VB>
__device__ void pack_diagonal_g(const KiviGeom &g, const KiviDev &dv, const unsigned char *kt,
                                const unsigned char *vt, unsigned char *work, int i, int j, int tb, int t) {
    switch (g.G) {
    case 16: pack_diagonal<D, KB, VB, 16>(g, dv, kt, vt, work, i, j, tb, t); break;
    case 32: pack_diagonal<D, KB, VB, 32>(g, dv, kt, vt, work, i, j, tb, t); break;
    default: pack_diagonal<D, KB, VB, 64>(g, dv, kt, vt, work, i, j, tb, t); break;
    }
}
template <int D>
__device__ void pack_diagonal_bits(const KiviGeom &g, const KiviDev &dv, const unsigned char *kt,
                                   const unsigned char *vt, unsigned char *work, int i, int j, int tb, int t) {
    if (g.kbits == 2 && g.vbits == 2) pack_diagonal_g<D, 2, 2>(g, dv, kt, vt, work, i, j, tb, t);
    else if (g.kbits == 2) pack_diagonal_g<D, 2, 4>(g, dv, kt, vt, work, i, j, tb, t);
    else if (g.vbits == 2) pack_diagonal_g<D, 4, 2>(g, dv, kt, vt, work, i, j, tb, t);
    else pack_diagonal_g<D, 4, 4>(g, dv, kt, vt, work, i, j, tb, t);
}

// ---------------------------------------------------------------------------
// The attention on the 5th-generation tensor cores (tcgen05): a CTA is 128
// query rows of one query head, 4 warps, and thread r owns row r (tensor-
// memory lane r).  Per 64-key tile kt: S = Q K^T (M 128, N 64, K d) into one
// of two S buffers in tensor memory; each thread reads its row of S, applies
// the causal mask and the online softmax (base 2, its whole row in
// registers) and writes its fp16 weights P back over the first 32 columns
// of the same S buffer (fp16 pairs, its own lane), from which O += P V
// (M 128, N d, K 64) takes them as its A operand: P never passes through
// shared memory, whose bandwidth the S MMAs' operands already fill (an
// M 128 x N 64 x K 16 MMA reads 6 KB of them in its 48 cycles).  O
// accumulates in tensor memory.  Completions arrive on mbarriers (bounded
// waits).
//
// Pipeline: S of tile kt + 1 is issued as tile kt starts (its buffer held
// S and P of tile kt - 1: free once P V of tile kt - 1 is done), so it runs
// under the softmax of tile kt; P V of tile kt - 1 runs under that softmax
// too, which waits for it only before a rescale of O.  Q, K and V tiles
// come by TMA, one tensor copy each, a few stages deep.  The running
// maximum is raised lazily: O and the row sum are rescaled only when a
// row's maximum grows by more than 8 (log2 units), so P stays below 2^8.
//
// Tiles in shared memory use the no-swizzle core-matrix layout, chunk-major:
// row r, 16-byte chunk c of a tile of ROWS rows at byte c ROWS 16 + r 16
// (core matrices of 8 rows x 16 bytes contiguous).  A tensor map over the
// fp16 [rows][D] array with dimensions (8 elements, rows, D / 8 chunks) and
// strides (2 D bytes, 16 bytes) writes exactly this with one copy per tile
// (rows past the array read as zero); value rows past the sequence are
// zeroed after the copy, as the weights they meet are zero.
// Per 128-row slot: Q [128][D] and its tensor-memory columns, S / P buffers
// in 0-63 and 64-127, O in 128-(128 + D): 256 columns; K and V stages
// [64][D] each, shared by the slots.
// ---------------------------------------------------------------------------
constexpr int kTcRows = 128, kTcKeys = 64;

// byte offset of 16-byte chunk c of row r in a chunk-major tile of ROWS rows
template <int ROWS>
__device__ __forceinline__ int cm_at(int r, int c) {
    return c * ROWS * 16 + r * 16;
}

__device__ __forceinline__ bool tc_wait_bar(uint64_t *bar, unsigned phase) {
    for (int it = 0; it < (1 << 24); ++it) {
        unsigned ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(tc_smem_u32(bar)), "r"(phase)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// one TMA tile copy (rows row0.. of the tensor map's array, all D columns)
// into dst, completing `bytes` on bar (one thread)
__device__ __forceinline__ void tma_tile(void *dst, const CUtensorMap *tm, int row0, uint64_t *bar,
                                         unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc_smem_u32(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(tc_smem_u32(dst)),
        "l"(tm), "r"(0), "r"(row0), "r"(0), "r"(tc_smem_u32(bar))
        : "memory");
}


// K and V stages of the attention CTA: three with two heads (160 KB at
// d = 128; the CTA holds all 512 tensor-memory columns, one CTA per SM),
// four with two query tiles of one head (192 KB: the CTA's four diagonal
// tiles are still in their stages for the pack epilogue), two with one head
// (two CTAs per SM).
__host__ __device__ constexpr int kv_stages(int NH, bool QT) { return QT ? 4 : NH == 2 ? 3 : 2; }
// Producer warps: two with two slots; one with one (a sixth warp would
// leave one CTA per SM at 168 registers: a one-slot 4k MHA call went 410 ->
// 444 us).
__host__ __device__ constexpr int producer_warps(int NH) { return NH == 2 ? 2 : 1; }

// A wait that also gives up when another warp of the CTA has given up
// (*abort set): false then, or after the iteration limit.
__device__ __forceinline__ bool tc_wait_bar_ab(uint64_t *bar, unsigned phase, const volatile int *abort) {
    for (int it = 0; it < (1 << 24); ++it) {
        unsigned ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(tc_smem_u32(bar)), "r"(phase)
            : "memory");
        if (ok) return true;
        if ((it & 255) == 255 && *abort) return false;
    }
    return false;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc_smem_u32(bar)) : "memory");
}

// NH slots of 128 query rows per CTA: NH query heads of one kv head (QT
// false: 1, or 2 when a kv head serves an even number of query heads), or
// (QT) NH consecutive query tiles of one head; each K and V tile then feeds
// every slot's MMAs.  Warps 0 .. 4 NH - 1 run the softmax: thread tid owns
// row tid mod 128 of slot tid / 128 (slot e has its own Q tile and
// tensor-memory columns [256 e, 256 e + 256)).  With two heads, two producer
// warps, each issuing from its lane 0, so that one's waits do not hold the
// other's MMAs back (a tcgen05.mma issue waits while the tensor pipe is
// busy): warp 8 the Q and K copies and S = Q K^T, warp 9 the V copies and
// O += P V (a commit tracks its own thread's MMAs); with one head, warp 4
// issues everything.  The warps meet on mbarriers only, one per S / P
// buffer: S done (MMA commit), P written (every softmax warp), P V done
// (MMA commit: the buffer is free again); and the copies' landings.
// At most 168 registers a thread: a scheduler partition's 16 K registers
// then hold three warps, so two one-head CTAs (five warps each) share an SM.
template <int D, int NH, bool QT>
__global__ void __maxnreg__(168)
    prefill_attn_tc_kernel(KiviGeom g, KiviDev dv, const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           __half *__restrict__ O, SeqLens lens, int t_stride, int hq) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int QB = kTcRows * D * 2, KVB = kTcKeys * D * 2;
    constexpr unsigned QLBO = kTcRows * 16, KLBO = kTcKeys * 16;   // chunk strides
    constexpr int NSW = 4 * NH;   // softmax warps
    constexpr int NPROD = producer_warps(NH);
    constexpr int KS = kv_stages(NH, QT);   // K and V stages: tile m in stage m mod KS
    constexpr int CR = QT ? NH * kTcRows : kTcRows;   // the CTA's query rows
    unsigned char *sQ = smem;                // head slot e at sQ + e QB
    unsigned char *sK = smem + NH * QB;      // stage s at sK + s KVB
    unsigned char *sV = sK + KS * KVB;       // stage s at sV + s KVB
    // S buffer 0 / 1 done, P V of buffer 0 / 1's tile done (the buffer is
    // free), Q landed, K stages landed, V stages landed, P of buffer 0 / 1
    // written
    constexpr int NB = 7 + 2 * KS;
    __shared__ __align__(8) uint64_t bars[NB];
    uint64_t *const bS = bars, *const bF = bars + 2, *const bQ = bars + 4, *const bK = bars + 5,
                    *const bV = bK + KS, *const bP = bV + KS;
    // K / V tile m: its stage and the phase its landing completes
    auto stg = [](int m) { return m % KS; };
    auto sph = [](int m) { return (unsigned)(m / KS) & 1u; };
    __shared__ uint32_t s_taddr;
    __shared__ int s_abort;   // a wait ran out: every warp stops
    const int qt = gridDim.x - 1 - blockIdx.x;   // the longest tiles first
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, hs = min(tid >> 7, NH - 1), rr = tid & 127;
    // the CTA's first head, this thread's (QT: one head, slot e = query tile e)
    const int h0 = QT ? blockIdx.y : blockIdx.y * NH, h = QT ? h0 : h0 + hs, i = blockIdx.z;
    const int hg = hq / g.h, j = h0 / hg;
    const int t = lens.t[i];
    const int tb = qt * CR;                                 // the CTA's first query row
    const int tbs = tb + (QT ? hs * kTcRows : 0);           // this thread's slot's first row
    if (tb >= t) {
        if (tb == 0 && h0 == 0 && threadIdx.x == 0) {   // an empty sequence
            dv.T[i] = 0;
            dv.Tqk[i] = 0;
            dv.Tqv[i] = 0;
        }
        return;
    }
    const int krow0 = (i * g.h + j) * t_stride;   // this kv head's first row in K and V
    const int nt = min((t + kTcKeys - 1) / kTcKeys, (tb + CR) / kTcKeys);   // key tiles
    if (tid == 0) {
        for (int k = 0; k < NB; ++k)   // Q's: one arrival per head slot's copy; P written: per softmax warp
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(tc_smem_u32(&bars[k])),
                         "r"(k == 4 ? NH : k >= 5 + 2 * KS ? NSW : 1)
                         : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    __syncthreads();
    if (warp == 0) tc_alloc(&s_taddr, 256 * NH);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = s_taddr;
    const volatile int *abort = &s_abort;
    bool ok = true;
    float lsum = 0.f;
    constexpr uint32_t ID_S = tc_idesc_f16(kTcRows, kTcKeys, 0), ID_O = tc_idesc_f16(kTcRows, D, 1);
    // O += P V of tile kt for every head slot: P (fp16 pairs) in the first 32
    // columns of the slot's S buffer kt mod 2, V from its stage; the commit
    // frees the S buffer and V's stage
    auto issue_pv = [&](int kt) {
        const int b = kt & 1;
        const unsigned char *v = sV + stg(kt) * KVB;
#pragma unroll
        for (int e = 0; e < NH; ++e)
#pragma unroll
            for (int c = 0; c < kTcKeys / 16; ++c)
                tc_mma_f16_ta(taddr + 256 * e + 128, taddr + 256 * e + 64 * b + 8 * c,
                              tc_desc(v + 256 * c, 128, KLBO), ID_O, kt > 0 || c > 0);
        tc_commit(&bF[b]);
    };
    if (NPROD == 1 && warp == NSW) {
        // ---- one producer (lane 0): every copy and MMA ----
        if (lane == 0) {
            auto issue_s = [&](int kt) {   // S of tile kt into buffer kt mod 2 of every head slot
                const unsigned char *k = sK + stg(kt) * KVB;
#pragma unroll
                for (int e = 0; e < NH; ++e) {
                    const uint32_t tS = taddr + 256 * e + 64 * (kt & 1);
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        tc_mma_f16(tS, tc_desc(sQ + e * QB + 2 * c * QLBO, QLBO, 128),
                                   tc_desc(k + 2 * c * KLBO, KLBO, 128), ID_S, c > 0);
                }
                tc_commit(&bS[kt & 1]);
            };
            // completions issued per barrier (for the drain after a time-out)
            int nK[KS], nV[KS], nS[2] = {0, 0}, nF[2] = {0, 0};
#pragma unroll
            for (int e = 0; e < NH; ++e)
                tma_tile(sQ + e * QB, &tmQ, (i * hq + h0 + (QT ? 0 : e)) * t_stride + tb + (QT ? e * kTcRows : 0), bQ,
                         QB);
            // K of the first KS tiles, V of the first KS - 1 (their stages are free)
#pragma unroll
            for (int m = 0; m < KS; ++m) {
                nK[m] = m < nt ? 1 : 0;
                nV[m] = m < nt && m < KS - 1 ? 1 : 0;
                if (nK[m]) tma_tile(sK + m * KVB, &tmK, krow0 + m * kTcKeys, &bK[m], KVB);
                if (nV[m]) tma_tile(sV + m * KVB, &tmV, krow0 + m * kTcKeys, &bV[m], KVB);
            }
            ok = tc_wait_bar_ab(bQ, 0, abort) && tc_wait_bar_ab(&bK[0], 0, abort);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                nS[0] = 1;
            }
            for (int kt = 0; kt < nt && ok; ++kt) {
                const int b = kt & 1;
                if (kt + 1 < nt) {
                    // S of the next tile: its K landed, its buffer free (P V
                    // of tile kt - 1 read its weights there)
                    ok = tc_wait_bar_ab(&bK[stg(kt + 1)], sph(kt + 1), abort) &&
                         (kt == 0 || tc_wait_bar_ab(&bF[b ^ 1], (unsigned)((kt - 1) >> 1) & 1u, abort));
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(kt + 1);
                    ++nS[b ^ 1];
                }
                if (kt + KS < nt) {   // K KS tiles on, into the stage S of this tile read
                    ok = tc_wait_bar_ab(&bS[b], (unsigned)(kt >> 1) & 1u, abort);
                    if (!ok) break;
                    tma_tile(sK + stg(kt) * KVB, &tmK, krow0 + (kt + KS) * kTcKeys, &bK[stg(kt)], KVB);
                    ++nK[stg(kt)];
                }
                if (kt + KS - 1 < nt) {   // V KS - 1 tiles on, into the stage P V of tile kt - 1 read
                    ok = kt == 0 || tc_wait_bar_ab(&bF[b ^ 1], (unsigned)((kt - 1) >> 1) & 1u, abort);
                    if (!ok) break;
                    const int vs = stg(kt + KS - 1);   // tile kt - 1's stage (at kt = 0: the last, unused)
                    tma_tile(sV + vs * KVB, &tmV, krow0 + (kt + KS - 1) * kTcKeys, &bV[vs], KVB);
                    ++nV[vs];
                }
                // P V of this tile: its weights written and, on the tile the
                // sequence cuts, V's rows past it zeroed (every softmax warp)
                ok = tc_wait_bar_ab(&bP[b], (unsigned)(kt >> 1) & 1u, abort) &&
                     tc_wait_bar_ab(&bV[stg(kt)], sph(kt), abort);
                if (!ok) break;
                tc_fence_after();
                issue_pv(kt);
                ++nF[b];
            }
            if (!ok) {
                // flag it, and let every issued copy and MMA finish (bounded:
                // each barrier's last completion is phase (count - 1) mod 2)
                // before shared and tensor memory are released
                s_abort = 1;
                atomicOr(dv.status, KIVI_FLAG_WAIT);
                tc_wait_bar(bQ, 0u);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    if (nS[k] > 0) tc_wait_bar(&bS[k], (unsigned)(nS[k] - 1) & 1u);
                    if (nF[k] > 0) tc_wait_bar(&bF[k], (unsigned)(nF[k] - 1) & 1u);
                }
#pragma unroll
                for (int m = 0; m < KS; ++m) {
                    if (nK[m] > 0) tc_wait_bar(&bK[m], (unsigned)(nK[m] - 1) & 1u);
                    if (nV[m] > 0) tc_wait_bar(&bV[m], (unsigned)(nV[m] - 1) & 1u);
                }
            }
        }
        __syncwarp();
    } else if (NPROD == 2 && warp == NSW) {
        // ---- the S producer (lane 0): Q and K copies, S = Q K^T ----
        if (lane == 0) {
            auto issue_s = [&](int kt) {   // S of tile kt into buffer kt mod 2 of every head slot
                const unsigned char *k = sK + stg(kt) * KVB;
#pragma unroll
                for (int e = 0; e < NH; ++e) {
                    const uint32_t tS = taddr + 256 * e + 64 * (kt & 1);
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        tc_mma_f16(tS, tc_desc(sQ + e * QB + 2 * c * QLBO, QLBO, 128),
                                   tc_desc(k + 2 * c * KLBO, KLBO, 128), ID_S, c > 0);
                }
                tc_commit(&bS[kt & 1]);
            };
            // completions issued per barrier (for the drain after a time-out)
            int nK[KS], nS[2] = {0, 0};
#pragma unroll
            for (int e = 0; e < NH; ++e)
                tma_tile(sQ + e * QB, &tmQ, (i * hq + h0 + (QT ? 0 : e)) * t_stride + tb + (QT ? e * kTcRows : 0), bQ,
                         QB);
#pragma unroll
            for (int m = 0; m < KS; ++m) {   // K of the first KS tiles
                nK[m] = m < nt ? 1 : 0;
                if (nK[m]) tma_tile(sK + m * KVB, &tmK, krow0 + m * kTcKeys, &bK[m], KVB);
            }
            ok = tc_wait_bar_ab(bQ, 0, abort) && tc_wait_bar_ab(&bK[0], 0, abort);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                nS[0] = 1;
            }
            for (int kt = 0; kt < nt && ok; ++kt) {
                const int b = kt & 1;
                if (kt + 1 < nt) {
                    // S of the next tile: its K landed, its buffer free (P V
                    // of tile kt - 1 read its weights there)
                    ok = tc_wait_bar_ab(&bK[stg(kt + 1)], sph(kt + 1), abort) &&
                         (kt == 0 || tc_wait_bar_ab(&bF[b ^ 1], (unsigned)((kt - 1) >> 1) & 1u, abort));
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(kt + 1);
                    ++nS[b ^ 1];
                }
                if (kt + KS < nt) {   // K KS tiles on, into the stage S of this tile read
                    ok = tc_wait_bar_ab(&bS[b], (unsigned)(kt >> 1) & 1u, abort);
                    if (!ok) break;
                    tma_tile(sK + stg(kt) * KVB, &tmK, krow0 + (kt + KS) * kTcKeys, &bK[stg(kt)], KVB);
                    ++nK[stg(kt)];
                }
            }
            if (!ok) {
                // flag it, and let every copy and MMA this thread issued finish
                // (bounded: each barrier's last completion is phase
                // (count - 1) mod 2) before shared and tensor memory are released
                s_abort = 1;
                atomicOr(dv.status, KIVI_FLAG_WAIT);
                tc_wait_bar(bQ, 0u);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (nS[k] > 0) tc_wait_bar(&bS[k], (unsigned)(nS[k] - 1) & 1u);
#pragma unroll
                for (int m = 0; m < KS; ++m)
                    if (nK[m] > 0) tc_wait_bar(&bK[m], (unsigned)(nK[m] - 1) & 1u);
            }
        }
        __syncwarp();
    } else if (NPROD == 2 && warp == NSW + 1) {
        // ---- the P V producer (lane 0): V copies, O += P V ----
        if (lane == 0) {
            int nV[KS], nF[2] = {0, 0};
#pragma unroll
            for (int m = 0; m < KS; ++m) {   // V of the first KS - 1 tiles
                nV[m] = m < nt && m < KS - 1 ? 1 : 0;
                if (nV[m]) tma_tile(sV + m * KVB, &tmV, krow0 + m * kTcKeys, &bV[m], KVB);
            }
            for (int kt = 0; kt < nt && ok; ++kt) {
                const int b = kt & 1;
                if (kt + KS - 1 < nt) {   // V KS - 1 tiles on, into the stage P V of tile kt - 1 read
                    ok = kt == 0 || tc_wait_bar_ab(&bF[b ^ 1], (unsigned)((kt - 1) >> 1) & 1u, abort);
                    if (!ok) break;
                    const int vs = stg(kt + KS - 1);   // tile kt - 1's stage (at kt = 0: the last, unused)
                    tma_tile(sV + vs * KVB, &tmV, krow0 + (kt + KS - 1) * kTcKeys, &bV[vs], KVB);
                    ++nV[vs];
                }
                // P V of this tile: its weights written and, on the tile the
                // sequence cuts, V's rows past it zeroed (every softmax warp)
                ok = tc_wait_bar_ab(&bP[b], (unsigned)(kt >> 1) & 1u, abort) &&
                     tc_wait_bar_ab(&bV[stg(kt)], sph(kt), abort);
                if (!ok) break;
                tc_fence_after();
                issue_pv(kt);
                ++nF[b];
            }
            if (!ok) {   // as above
                s_abort = 1;
                atomicOr(dv.status, KIVI_FLAG_WAIT);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (nF[k] > 0) tc_wait_bar(&bF[k], (unsigned)(nF[k] - 1) & 1u);
#pragma unroll
                for (int m = 0; m < KS; ++m)
                    if (nV[m] > 0) tc_wait_bar(&bV[m], (unsigned)(nV[m] - 1) & 1u);
            }
        }
        __syncwarp();
    } else {
        // ---- the softmax warps ----
        const uint32_t tH = taddr + 256 * hs, tO = tH + 128;          // this head slot's columns
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;   // this warp's tensor-memory lanes
        const float sl2 = 1.4426950408889634f / sqrtf((float)D);      // log2(e) / sqrt(d)
        const int row = tbs + rr;
        float mref = -INFINITY;   // the row's reference maximum (raw score units)
        for (int kt = 0; kt < nt; ++kt) {
            const int b = kt & 1;
            ok = __all_sync(0xffffffffu, tc_wait_bar_ab(&bS[b], (unsigned)(kt >> 1) & 1u, abort));
            if (!ok) break;
            tc_fence_after();
            // this row's 64 scores (P takes their place)
            const uint32_t tS = tH + 64 * b;
            uint32_t sr[2][32];
            tc_ld32(tS + lane_off, sr[0]);
            tc_ld32(tS + lane_off + 32, sr[1]);
            tc_wait_ld();
            float sc[64];
            if (kt * kTcKeys + kTcKeys - 1 > tbs) {   // a tile the causal mask cuts (the slot's last two)
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const int key = kt * kTcKeys + c;
                    sc[c] = key > row ? -INFINITY : __uint_as_float(sr[c >> 5][c & 31]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) sc[c] = __uint_as_float(sr[c >> 5][c & 31]);
            }
            // the row maximum over eight independent chains
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = sc[k];
#pragma unroll
            for (int c = 8; c < 64; ++c) m8[c & 7] = fmaxf(m8[c & 7], sc[c]);
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            // lazy rescale: only when the maximum grew by more than 2^8 in weight
            const bool grow = mx != -INFINITY && (mref == -INFINITY || (mx - mref) * sl2 > 8.f);
            const float alpha = grow && mref != -INFINITY ? ex2((mref - mx) * sl2) : 1.f;
            if (grow) mref = mx;
            const float ms = mref * sl2;
            uint32_t pw[32];
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const float p0 = ex2(fmaf(sc[2 * c], sl2, -ms)), p1 = ex2(fmaf(sc[2 * c + 1], sl2, -ms));
                l4[c & 3] += p0 + p1;
                pw[c] = pack_h2(p0, p1);
            }
            lsum = lsum * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
            // a rescale of O, once P V of the previous tile added to it
            if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = __all_sync(0xffffffffu,
                                tc_wait_bar_ab(&bF[b ^ 1], (unsigned)((kt - 1) >> 1) & 1u, abort));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tc_ld32(tO + lane_off + c0, o);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tc_st32(tO + lane_off + c0, o);
                }
            }
            // P: this row's 64 weights as fp16 pairs over the first 32
            // columns of the S buffer (the A operand of P V)
            tc_st32(tS + lane_off, pw);
            // V's rows past the sequence on the tile it cuts: zeroed once
            // the tile landed (they meet zero weights, and the array there
            // holds whatever it holds), a share per softmax warp
            if (kt * kTcKeys + kTcKeys > t) {
                ok = __all_sync(0xffffffffu, tc_wait_bar_ab(&bV[stg(kt)], sph(kt), abort));
                if (!ok) break;
                const int r0 = t - kt * kTcKeys;
                unsigned char *v = sV + stg(kt) * KVB;
                for (int e = tid; e < (kTcKeys - r0) * (D / 8); e += 32 * NSW) {
                    const int r = r0 + e / (D / 8), c = e % (D / 8);
                    *reinterpret_cast<uint4 *>(v + cm_at<kTcKeys>(r, c)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // P, O's rescale and the zeroed rows before P V
            tc_wait_st();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bP[b]);
        }
        // the last P V done
        if (ok)
            ok = __all_sync(0xffffffffu,
                            tc_wait_bar_ab(&bF[(nt - 1) & 1], (unsigned)((nt - 1) >> 1) & 1u, abort));
        if (!ok) {   // stop the others' waits too
            if (lane == 0) {
                s_abort = 1;
                atomicOr(dv.status, KIVI_FLAG_WAIT);
            }
        } else {
            tc_fence_after();
            // the output rows (tcgen05.ld is warp-wide: every lane loads, the
            // rows inside the sequence are stored)
            const float r = 1.f / lsum;
            __half *orow = O + (((size_t)i * hq + h) * t_stride + min(row, t - 1)) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tc_ld32(tO + lane_off + c0, o);
                tc_wait_ld();
                if (row < t)
#pragma unroll
                    for (int c = 0; c < 32; c += 8)
                        *reinterpret_cast<uint4 *>(orow + c0 + c) =
                            make_uint4(pack_h2(__uint_as_float(o[c]) * r, __uint_as_float(o[c + 1]) * r),
                                       pack_h2(__uint_as_float(o[c + 2]) * r, __uint_as_float(o[c + 3]) * r),
                                       pack_h2(__uint_as_float(o[c + 4]) * r, __uint_as_float(o[c + 5]) * r),
                                       pack_h2(__uint_as_float(o[c + 6]) * r, __uint_as_float(o[c + 7]) * r));
            }
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok) && !s_abort;
    if (warp == 0) tc_dealloc(taddr, 256 * NH);
    if (!ok) return;

    // epilogue: the first query head of each kv head packs the tile's two
    // 64-token key / value tiles, still in their stages; Q's region holds
    // the staging (generic stores after the copies' and MMAs' accesses)
    if (h0 % hg == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int k = 0; k < CR / kTcKeys; ++k) {
            const int kb = tb + k * kTcKeys, kt = kb / kTcKeys;
            if (kb >= t) break;
            pack_diagonal_bits<D>(g, dv, sK + stg(kt) * KVB, sV + stg(kt) * KVB, sQ, i, j, kb, t);
            __syncthreads();   // the staging is reused
        }
        if (tb == 0 && j == 0 && threadIdx.x == 0) {
            dv.T[i] = t;
            dv.Tqk[i] = t - t % g.R;
            dv.Tqv[i] = t > g.R ? t - g.R : 0;
        }
    }
}

// The encoder of TMA tensor maps, from the driver (through the runtime, no
// link to the driver library); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Tensor map over an fp16 [rows][D] array giving chunk-major core-matrix
// tiles of box_rows rows (see above): dimensions (8, rows, D / 8), strides
// (2 D bytes, 16 bytes), box (8, box_rows, D / 8).
cudaError_t make_tile_map(CUtensorMap *tm, const __half *base, long long rows, int D, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dim[3] = {8, (cuuint64_t)rows, (cuuint64_t)(D / 8)};
    const cuuint64_t str[2] = {(cuuint64_t)D * 2, 16};
    const cuuint32_t box[3] = {8, (cuuint32_t)box_rows, (cuuint32_t)(D / 8)};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half *>(base), dim, str, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int NH, bool QT>
cudaError_t launch_tc(const KiviGeom &g, const KiviDev &dv, const __half *Q, const __half *K, const __half *V,
                      __half *O, const SeqLens &lens, int t_stride, int hq, int maxt, cudaStream_t st) {
    const size_t smem = (size_t)NH * kTcRows * D * 2 + (size_t)2 * kv_stages(NH, QT) * kTcKeys * D * 2;
    const long long ts = t_stride > 0 ? t_stride : 1;
    CUtensorMap tq, tk, tv;   // unused when every sequence is empty (the CTAs only write counters)
    memset(&tq, 0, sizeof tq);
    memset(&tk, 0, sizeof tk);
    memset(&tv, 0, sizeof tv);
    cudaError_t e = cudaSuccess;
    if (maxt > 0) {
        e = make_tile_map(&tq, Q, (long long)g.b * hq * ts, D, kTcRows);
        if (e == cudaSuccess) e = make_tile_map(&tk, K, (long long)g.b * g.h * ts, D, kTcKeys);
        if (e == cudaSuccess) e = make_tile_map(&tv, V, (long long)g.b * g.h * ts, D, kTcKeys);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(prefill_attn_tc_kernel<D, NH, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    constexpr int CR = QT ? NH * kTcRows : kTcRows;
    const int nqt = maxt > 0 ? (maxt + CR - 1) / CR : 1;
    prefill_attn_tc_kernel<D, NH, QT>
        <<<dim3(nqt, QT ? hq : hq / NH, g.b), 128 * NH + 32 * producer_warps(NH), smem, st>>>(g, dv, tq, tk, tv, O,
                                                                                            lens, t_stride, hq);
    return cudaGetLastError();
}

}  // namespace

cudaError_t kivi_launch_prefill_attn(const KiviGeom &g, const KiviDev &dv, const __half *Q, const __half *K,
                                     const __half *V, __half *O, const SeqLens &lens, int t_stride, int hq,
                                     cudaStream_t st) {
    if (g.G > 64 || (g.d != 64 && g.d != 128)) return cudaErrorInvalidValue;
    int maxt = 0;
    for (int i = 0; i < g.b; ++i) maxt = lens.t[i] > maxt ? lens.t[i] : maxt;
    if (maxt > 0 && ((long long)g.b * hq * t_stride >= (1LL << 31))) return cudaErrorInvalidValue;   // TMA row coordinates
    // two query heads a CTA when a kv head serves an even number of them
    // (d = 128: the 160 KB of shared memory keep one CTA, which holds all
    // 512 tensor-memory columns, per SM)
    if (g.d == 64) return launch_tc<64, 1, false>(g, dv, Q, K, V, O, lens, t_stride, hq, maxt, st);
    // d = 128: two query heads of a kv head a CTA when a kv head serves an
    // even number of them, else two query tiles of one head
    return (hq / g.h) % 2 == 0 ? launch_tc<128, 2, false>(g, dv, Q, K, V, O, lens, t_stride, hq, maxt, st)
                               : launch_tc<128, 2, true>(g, dv, Q, K, V, O, lens, t_stride, hq, maxt, st);
}
