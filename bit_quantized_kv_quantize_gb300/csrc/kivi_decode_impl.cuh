// kivi_decode_impl.cuh -- persistent split-K decode attention over the
// quantized cache.
//
// Method: "Literature audit -- Group 2", section 1 KIVI, core algorithm
// item 5: scores q.k / sqrt(d) over the quantized keys followed by the fp16
// keys, one softmax over both, weights applied to the quantized values
// followed by the fp16 values.  Query head i reads kv head i / (h_q / h_kv)
// (GQA, README note of 2025-01-18 in the same section).
//
// Work split.  The grid is persistent (two CTAs per SM).  The 64-token blocks
// of every (sequence, kv head, group of <= 4 query heads) are laid end to end
// as work units and each CTA takes an equal contiguous share, so all CTAs
// stream about the same number of bytes.  Inside a CTA, each warp streams its
// blocks through a private ring of shared-memory stages filled by bulk TMA
// copies (cp.async.bulk + mbarrier) and runs
//   scores   S[tok, col] = sum_c (off + code) * B[c, col]   (m16n8k16, f16 in, f32 acc)
//   values   O[ch, col]  = sum_t code * P[t, col]
// with the unpacked code in the A operand (one lop3, sometimes after a shift:
// the field becomes mantissa bits of an fp16 constant) and the per-group
// scale folded into B.  Column pairs (2e, 2e+1) carry an exact two-term fp16
// split of B for query head e:
//   keys:   q_c s = hi + lo with hi = RN(q s), lo = fma(q, s, -hi)  (exact)
//   values: p s  = hi + lo from p = ph + pl (fp16 hi/lo of the fp32 weight)
// so the tensor-core sums carry fp32-level precision.  The zero points (and
// the key offset) enter through small MMAs over the scale/zero rows.  Blocks
// that also hold tokens of the fp16 windows add, for those tokens, MMAs over
// fp16 rows copied into shared memory.  Each CTA merges its warps per pair
// and writes (m, l, acc[d]) in base 2 (scores pre-multiplied by
// log2(e) / sqrt(d)); the last CTA to finish a pair merges its partials
// with log-sum-exp weights and writes the fp16 output.
#pragma once
#include "kivi_internal.cuh"
#include "kivi_mma.cuh"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWaitIters = 1 << 24;   // bounded mbarrier waits
constexpr int kFastMerge = 16;   // partials a pair's final merge reads in one round trip ...
constexpr int kFastMergeV = 4;   // ... with at most this many accumulators a thread

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
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
// L2 eviction-priority policies: the streamed records are read once
// (evict first); the tail data prefetched long before its use is kept
// (evict last)
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, unsigned bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}


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
template <int BITS, bool KEY>
__host__ __device__ constexpr float slot_offset(int r) { return view_of<BITS, KEY>(r).off; }

// Value fields for the P.V contraction: off + code as fp16 (2-bit fields
// at mantissa positions 6 and 8, offsets 16 and 4; 4-bit at position 4,
// offset 64), no subtraction per code.  The accumulator is kept centred
// instead: at the end of each block every row loses (off + c0) times the
// block's sum_t p_t s_t of its group (c0 = (2^B - 1) / 2; a small MMA over
// the scale rows gives those sums), and the group midpoints z + c0 s go
// into the zero-point accumulator.  So the accumulators hold the centred
// sums sum p s (code - c0) and sum p (z + c0 s), both near the size of the
// output (N(0, 1) values put the group midpoints near 0), rather than
// c0 s sum(p): that is what bounds the fp32 accumulation error at long
// contexts.  The offset lives in the accumulator for one block only; small
// offsets keep that transient small.
__host__ __device__ constexpr View view_val(int bits, int r) {
    if (bits == 4) return r == 0 ? at_pos(4, 4, 4, 0) : (r == 1 ? at_pos(4, 4, 0, 0) : at_pos(4, 4, 0, 4 * r - 4));
    switch (r) {   // 2-bit field bits [2r, 2r + 2) -> mantissa bits 6 or 8
    case 0: return at_pos(6, 2, 6, 0);
    case 1: return at_pos(8, 2, 6, 0);
    case 2: return at_pos(6, 2, 2, 0);
    case 3: return at_pos(6, 2, 0, 0);
    case 4: return at_pos(8, 2, 0, 0);
    case 5: return at_pos(6, 2, 0, 4);
    case 6: return at_pos(8, 2, 0, 4);
    default: return at_pos(8, 2, 0, 6);
    }
}
template <int BITS, int R>
__device__ __forceinline__ uint32_t unpack_val_t(uint32_t w) {
    constexpr View v = view_val(BITS, R);
    const uint32_t x = v.shl ? (w << v.shl) : (v.shr ? (w >> v.shr) : w);
    return and_or<v.mask, v.magic>(x);
}
template <int BITS>
__device__ __forceinline__ uint32_t unpack_val_raw(uint32_t w, int r) {
    switch (r) {
    case 0: return unpack_val_t<BITS, 0>(w);
    case 1: return unpack_val_t<BITS, 1>(w);
    case 2: return unpack_val_t<BITS, 2>(w);
    case 3: return unpack_val_t<BITS, 3>(w);
    case 4: return unpack_val_t<BITS, (BITS == 2 ? 4 : 3)>(w);
    case 5: return unpack_val_t<BITS, (BITS == 2 ? 5 : 3)>(w);
    case 6: return unpack_val_t<BITS, (BITS == 2 ? 6 : 3)>(w);
    default: return unpack_val_t<BITS, (BITS == 2 ? 7 : 3)>(w);
    }
}


// ---------------------------------------------------------------------------
// Shared-memory geometry
// ---------------------------------------------------------------------------
// The block record's layout for a kernel variant, at compile time (the same
// numbers kivi_geom_init derives at run time; the launcher checks they agree).
template <int D, int KB, int VB, int SH>
struct Rec {
    static constexpr int G = 16 << SH;
    static constexpr int KGR = G >= 64 ? 1 : 64 / G;
    static constexpr int KC = 2 * D * KB * 4;           // key code bytes
    static constexpr int KSZ = KGR * 2 * D * 2;         // key scale/zero bytes
    static constexpr int VC_BLK = D * VB / 2;           // words per value block
    static constexpr int VSZ_BLK = 2 * (D / G) * 16;    // halves per value block
    static constexpr int VC = 4 * VC_BLK * 4;
    static constexpr int VSZ = 4 * VSZ_BLK * 2;
    static constexpr int OFF_KSZ = KC, OFF_VC = KC + KSZ, OFF_VSZ = KC + KSZ + VC;
    static constexpr int BYTES = KC + KSZ + VC + VSZ;
};
// One warp's region of dynamic shared memory: its ring of stages; at the end
// of a segment it also holds the warp's result (m[4], l[4], o[4][d] in
// fp32).  Between the two, the CTA stages its mixed blocks across the
// regions.
__host__ __device__ __forceinline__ size_t warp_region(const KiviGeom &g, int stages) {
    const size_t sb = (size_t)g.rec_bytes;   // a stage holds one block record
    size_t ring = (size_t)(stages >= 2 ? stages : 2) * sb;
    size_t res = (size_t)(8 + 4 * g.d) * 4;
    size_t m = ring > res ? ring : res;
    return (m + 127) / 128 * 128;
}
// the warps' ring barriers, the CTA's mixed-block barrier and the fused
// append's
__host__ __device__ __forceinline__ size_t bar_region(int warps, int stages) {
    return ((size_t)(warps * stages + 2) * 8 + 127) / 128 * 128;
}
// bytes a mixed block stages in the ring: its record, up to 64 key and 64
// value rows of 2 d bytes, and a zero row
__host__ __device__ __forceinline__ size_t mixed_region(const KiviGeom &g) {
    return (size_t)g.rec_bytes + (size_t)(2 * KIVI_KBLK + 1) * (2 * g.d);
}
// Rows of tokens [a, b) a block stages from a window ring of `ring` rows (a
// well-formed cache never holds more than the ring; the clamp keeps reads
// inside it whatever the counters say).
__device__ __forceinline__ int rows_to_stage(int a, int b, int ring) { return max(0, min(b - a, ring)); }
// Copy those rows into consecutive rows at dst: at most two bulk copies (the
// ring may wrap once); the bytes land on `bar`.
template <int D>
__device__ __forceinline__ void copy_rows(unsigned char *dst, const __half *win, int ring, int a, int b,
                                          uint64_t *bar) {
    const int n = rows_to_stage(a, b, ring);
    if (n == 0) return;
    const int r0 = a % ring;
    const int n1 = min(n, ring - r0);
    bulk_g2s(dst, win + (size_t)r0 * D, (unsigned)n1 * D * 2, bar);
    if (n > n1) bulk_g2s(dst + (size_t)n1 * D * 2, win, (unsigned)(n - n1) * D * 2, bar);
}

// ---------------------------------------------------------------------------
// The append of one (sequence, kv head) pair inside a decode launch (item
// 4's one-token maintenance), by one warp of the CTA that owns the pair's
// append.  rows: [3][D] fp16 in shared memory, filled by bulk copies the
// warp issued at the start of the segment on fbar: the value token leaving
// the queue (row 0, when pop), the new key and the new value.  When the
// value queue is full its oldest token Tqv0 is quantized per token (item 3:
// groups of G channels) into the record of its block with the append
// kernel's arithmetic (qparams, qcode), a token opening a 16-token value
// block first clearing that block; the new rows go to their window slots
// (T0 mod R, T0 mod (R + 1): the latter the popped token's slot), and the
// sequence's counters after the append to nxt (kv head 0).  Out of line:
// it runs once per pair and stays off the streaming loop's registers.
// The global writes are ordered before the launch's later bulk copies of
// the record by a proxy fence here and the barrier before those copies.
// ---------------------------------------------------------------------------
template <int D, int KB, int VB, int SH>
__device__ __noinline__ void fused_append_pair(const KiviGeom &g, const KiviDev &dv, const FusedStep &fs, int i,
                                               int j, int T0, int Tqk, int Tqv0, bool pop, __half *rows,
                                               uint64_t *fbar, unsigned phase) {
    using RG = Rec<D, KB, VB, SH>;
    constexpr int G = 16 << SH, NGI = D / G, M = D / 32;
    constexpr int CPH = 16 / VB, NWV = D * VB / 128, WL = D * VB / 64, CS = WL < 4 ? WL : 4;
    const int lane = threadIdx.x & 31;
    if (!__all_sync(0xffffffffu, mbar_wait(fbar, phase))) {
        if (lane == 0) atomicOr(dv.status, KIVI_FLAG_WAIT);
        mbar_wait(fbar, phase);   // bounded: let the copies land before the rows are reused
        return;
    }
    __half *vwin = dv.Vf + vf_slice(g, i, j);
    if (pop) {
        const __half *x = rows;
        unsigned char *sc = reinterpret_cast<unsigned char *>(rows);   // the popped row, once read
        const int tt = Tqv0 % KIVI_KBLK, vbl = tt >> 4, t16 = tt & 15;
        unsigned char *grec = dv.blk + rec_off(g, i, j, Tqv0 / KIVI_KBLK);
        uint32_t *vc = reinterpret_cast<uint32_t *>(grec + RG::OFF_VC) + (size_t)vbl * RG::VC_BLK;
        __half *vsz = reinterpret_cast<__half *>(grec + RG::OFF_VSZ) + (size_t)vbl * RG::VSZ_BLK;
        float v[M], mn[M], mx[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            v[m] = __half2float(x[lane + 32 * m]);
            mn[m] = mx[m] = v[m];
        }
        // group minima and maxima (exact in any order): over the lanes of
        // a group, then over the 32-channel chunks a group spans
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int o = 1; o < (G < 32 ? G : 32); o <<= 1) {
                mn[m] = fminf(mn[m], __shfl_xor_sync(0xffffffffu, mn[m], o));
                mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xffffffffu, mx[m], o));
            }
        if (t16 == 0) {   // a fresh value block
            for (int e = lane; e < RG::VC_BLK; e += 32) vc[e] = 0u;
            for (int e = lane; e < RG::VSZ_BLK / 2; e += 32) reinterpret_cast<uint32_t *>(vsz)[e] = 0u;
        }
        __syncwarp();   // the block is cleared and every lane has read its channels
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float gmn = mn[m], gmx = mx[m];
#pragma unroll
            for (int m2 = 0; m2 < M; ++m2)
                if (G > 32 && m2 != m && (32 * m2) / G == (32 * m) / G) {
                    gmn = fminf(gmn, mn[m2]);
                    gmx = fmaxf(gmx, mx[m2]);
                }
            const QParams p = qparams(gmn, gmx, VB);
            sc[lane + 32 * m] = (unsigned char)qcode(v[m], p.sf, p.zf, VB);
            const int c = lane + 32 * m;
            if (c % G == 0) {   // the group's first channel writes its scale and zero
                const int gi = c / G, ps = vsz_pos(t16);
                vsz[gi * 16 + ps] = p.s16;
                vsz[(NGI + gi) * 16 + ps] = p.z16;
            }
        }
        __syncwarp();
        // the token's 16-bit halves: channel class gg (8) x channel word w
        const int p8 = t16 >> 3, tq = (t16 & 7) >> 1, half = t16 & 1;
        for (int e = lane; e < 8 * NWV; e += 32) {
            const int gg = e / NWV, w = e - gg * NWV;
            uint32_t bits = 0;
#pragma unroll
            for (int r = 0; r < CPH; ++r) bits |= (uint32_t)sc[8 * (w * CPH + r) + gg] << (r * VB);
            const int L = 4 * gg + tq, u = p8 * NWV + w;
            reinterpret_cast<uint16_t *>(vc + (size_t)(u / CS) * 32 * CS + (size_t)L * CS + (u % CS))[half] =
                (uint16_t)bits;
        }
    }
    for (int e = lane; e < D / 4; e += 32) {
        const bool isv = e >= D / 8;
        const int c8 = isv ? e - D / 8 : e;
        __half *dst = isv ? vwin + (size_t)(T0 % (g.R + 1)) * D : dv.Kf + kf_slice(g, i, j) + (size_t)(T0 % g.R) * D;
        reinterpret_cast<uint4 *>(dst)[c8] = reinterpret_cast<const uint4 *>(rows + (isv ? 2 : 1) * D)[c8];
    }
    if (j == 0 && lane == 0) {
        fs.nxt[i] = T0 + 1;
        fs.nxt[g.b + i] = Tqk;
        fs.nxt[2 * g.b + i] = Tqv0 + (pop ? 1 : 0);
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
}

// Stage block kb: one bulk copy of its record (packed keys, key scale/zero
// rows, packed values, value scale/zero rows, back to back).  Lane 0 issues.
template <int BYTES>
__device__ __forceinline__ void issue_block(unsigned char *st, uint64_t *bar, const unsigned char *recs, int kb,
                                            uint64_t policy) {
    if ((threadIdx.x & 31) == 0) {
        mbar_expect_tx(bar, (unsigned)BYTES);
        bulk_g2s_hint(st, recs + (size_t)kb * BYTES, (unsigned)BYTES, bar, policy);
    }
}

// L2 prefetches for a block that will be read late: its packed data, and the
// fp16 window rows [a, b) of a ring of `ring` rows (at most `ring` rows, so
// at most one wrap).
__device__ __forceinline__ void prefetch_l2(const void *p, unsigned bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(policy)
                 : "memory");
}

template <int D>
__device__ __forceinline__ void prefetch_rows(const __half *win, int ring, int a, int b, uint64_t policy) {
    if (a >= b) return;
    const int r0 = a % ring, n = min(b - a, ring);
    const int n1 = min(n, ring - r0);
    prefetch_l2(win + (size_t)r0 * D, (unsigned)n1 * D * 2, policy);
    if (n > n1) prefetch_l2(win, (unsigned)(n - n1) * D * 2, policy);
}


// ---------------------------------------------------------------------------
// Per-warp running state of one (sequence, kv head, head group) segment.
// Thread (gq, tq) owns query head tq's running max / sum and the output
// accumulators of channel rows 16 mm + gq and + 8 (columns: tq hi, tq lo).
// ---------------------------------------------------------------------------
template <int D>
struct WarpAcc {
    float oacc[D / 16][4];
    float zacc[4];
    float mrun, lrun;
};

template <int D>
__device__ __forceinline__ void acc_reset(WarpAcc<D> &A) {
#pragma unroll
    for (int mm = 0; mm < D / 16; ++mm) A.oacc[mm][0] = A.oacc[mm][1] = A.oacc[mm][2] = A.oacc[mm][3] = 0.f;
    A.zacc[0] = A.zacc[1] = A.zacc[2] = A.zacc[3] = 0.f;
    A.mrun = -INFINITY;
    A.lrun = 0.f;
}

// Online softmax over the block: p[t][0..1] holds the scores (log2 units) of
// rows gq and gq + 8 of tile t for head tq; on return it holds the weights
// exp2(score - m).  At least one score of the block is finite.
template <int D>
__device__ __forceinline__ void softmax_update(WarpAcc<D> &A, float (&p)[4][2]) {
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < 4; ++t) mx = fmaxf(mx, fmaxf(p[t][0], p[t][1]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mnew = fmaxf(A.mrun, mx);
    const float scl = ex2(A.mrun - mnew);
    A.mrun = mnew;
    float ps = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        p[t][0] = ex2(p[t][0] - mnew);
        p[t][1] = ex2(p[t][1] - mnew);
        ps += p[t][0] + p[t][1];
    }
    A.lrun = A.lrun * scl + ps;
    if (__any_sync(0xffffffffu, scl != 1.f)) {   // the running max moved for some head
#pragma unroll
        for (int mm = 0; mm < D / 16; ++mm) {
            A.oacc[mm][0] *= scl;
            A.oacc[mm][1] *= scl;
            A.oacc[mm][2] *= scl;
            A.oacc[mm][3] *= scl;
        }
        A.zacc[0] *= scl;
        A.zacc[1] *= scl;
        A.zacc[2] *= scl;
        A.zacc[3] *= scl;
    }
}

// Weights of tile rows (gq, gq + 8) for head tq -> B fragments of the P.V
// MMA (k = tokens 2tq, 2tq+1 and 2tq+8, 2tq+9; column gq = head gq/2,
// hi or lo), as fp16 hi and lo parts.
struct PFrag {
    uint32_t PH0, PH1, PL0, PL1;
};
__device__ __forceinline__ PFrag p_fragments(float p0, float p1, int tq, int eB) {
    const __half2 ph = __floats2half2_rn(p0, p1);
    const float2 phf = __half22float2(ph);
    const __half2 pl = __floats2half2_rn(p0 - phf.x, p1 - phf.y);
    const int src1 = 8 * tq + eB, src2 = 8 * tq + 4 + eB;
    const uint32_t h1 = __shfl_sync(0xffffffffu, h2u(ph), src1);
    const uint32_t h2 = __shfl_sync(0xffffffffu, h2u(ph), src2);
    const uint32_t l1 = __shfl_sync(0xffffffffu, h2u(pl), src1);
    const uint32_t l2 = __shfl_sync(0xffffffffu, h2u(pl), src2);
    PFrag f;
    f.PH0 = prmt(h1, h2, 0x5410u);
    f.PH1 = prmt(h1, h2, 0x7632u);
    f.PL0 = prmt(l1, l2, 0x5410u);
    f.PL1 = prmt(l1, l2, 0x7632u);
    return f;
}

// ---------------------------------------------------------------------------
// One 64-token block, read from a shared-memory stage that a bulk TMA copy
// filled with the block's record (packed codes and scale/zero rows).
//
// MIXED blocks also hold tokens of the fp16 windows (keys >= Tqk, values >=
// Tqv) or run past the end T; they are taken one 16-token tile at a time
// (tmask).  Their quantized tokens still go through the packed path (value
// weights masked to the quantized tokens); their window tokens are
// multiplied from fp16 rows in shared memory with ldmatrix fragments (a row
// of zeros stands in for tokens outside the window); scores past T are
// masked.
// ---------------------------------------------------------------------------
struct MixCtx {
    int tb;                              // first token of the block
    int tmask;                           // its 16-token tiles to take (bit t: tile t)
    int T, Tqk, Tqv;
    const unsigned char *krows, *vrows;  // window rows of tokens ka.., va.. (stride RS bytes)
    int ka, va, RS;
    const unsigned char *zrow;           // 2 d zero bytes
};
__device__ __forceinline__ const __half *key_row(const MixCtx &m, int tau) {
    return reinterpret_cast<const __half *>(tau >= m.Tqk && tau < m.T ? m.krows + (size_t)(tau - m.ka) * m.RS
                                                                        : m.zrow);
}
__device__ __forceinline__ const __half *value_row(const MixCtx &m, int tau) {
    return reinterpret_cast<const __half *>(tau >= m.Tqv && tau < m.T ? m.vrows + (size_t)(tau - m.va) * m.RS
                                                                        : m.zrow);
}
__device__ __forceinline__ uint32_t keep_halves(uint32_t x, bool lo, bool hi) {
    return x & ((lo ? 0x0000FFFFu : 0u) | (hi ? 0xFFFF0000u : 0u));
}

// PROBS: the block's scores (log2 units) of head tq also go to srow[0..63]
// (tokens tb.. of that head's weights row; null for absent heads).
template <int D, int KB, int VB, int SH, bool MIXED, bool PROBS>
__device__ __forceinline__ void do_block(WarpAcc<D> &A, const uint32_t (&qB)[D / 16][2],
                                         const unsigned char *sb, float alpha, const MixCtx &mx, float *srow) {
    using RG = Rec<D, KB, VB, SH>;
    constexpr int NJ = D / 16;
    constexpr int CPHK = 16 / KB, NWK = KB / 2;
    constexpr int CPHV = 16 / VB, NWV = D * VB / 128;
    constexpr int WLV = D * VB / 64, CSV = WLV < 4 ? WLV : 4;
    constexpr int sh = SH;
    constexpr int ngi = (D / 16) >> SH;
    constexpr int nkrows = 2 * (SH >= 2 ? 1 : (4 >> SH));
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const bool odd = gq & 1;
    const int eB = gq >> 1;
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t nm = odd ? 0xBC00BC00u : 0u;   // -1 for lo columns, 0 for hi
    const uint32_t m1 = odd ? 0x3C003C00u : 0u;   // 1 for lo columns, 0 for hi
    const uint32_t *sK = reinterpret_cast<const uint32_t *>(sb);
    const __half *sKsz = reinterpret_cast<const __half *>(sb + RG::OFF_KSZ);
    const uint32_t *sV = reinterpret_cast<const uint32_t *>(sb + RG::OFF_VC);
    const __half *sVsz = reinterpret_cast<const __half *>(sb + RG::OFF_VSZ);

    // ---- key zero points: sum_c q_c z_c and sum_c q_c s_c per group ----
    // (rows gq >= nkrows repeat a present row: their results are not used)
    float dc[4] = {0.f, 0.f, 0.f, 0.f};
    const int zkrow = gq & (nkrows - 1);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        // rows are lane-major: lane t's channels 16 jj + 2 t (+1) and
        // 16 jj + 8 + 2 t (+1) are the four halves at t d/4 + 4 jj
        const uint2 za = *reinterpret_cast<const uint2 *>(sKsz + zkrow * D + tq * (D / 4) + 4 * jj);
        const uint32_t a0 = za.x, a2 = za.y;
        mma16816(dc, a0, 0u, a2, 0u, qB[jj][0], qB[jj][1]);
    }
    float kz[4], ks[4];
#pragma unroll
    for (int rp = 0; rp < 4; ++rp) {
        if (rp > (3 >> sh)) { kz[rp] = ks[rp] = 0.f; continue; }
        kz[rp] = __shfl_sync(0xffffffffu, dc[0], ((2 * rp + 1) & 7) * 4 + tq);
        ks[rp] = __shfl_sync(0xffffffffu, dc[0], ((2 * rp) & 7) * 4 + tq);
    }

    // ---- scores from the packed keys ----
    float sc[4][4];
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) sc[mm][0] = sc[mm][1] = sc[mm][2] = sc[mm][3] = 0.f;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
        uint32_t W[2][NWK];
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
        // B = q s split exactly: hi columns RN(q s), lo columns q s - RN(q s)
        // (fma(q, s, RN(-q s)) with -q on lo lanes, 0 on hi lanes)
        const uint32_t qn0 = hmul2u(qB[jj][0], nm), qn1 = hmul2u(qB[jj][1], nm);
        uint32_t b0[4], b1[4];
#pragma unroll
        for (int rp = 0; rp < 4; ++rp) {
            b0[rp] = b1[rp] = 0u;
            if (rp > (3 >> sh)) continue;   // groups present in this block
            const uint2 sv = *reinterpret_cast<const uint2 *>(sKsz + 2 * rp * D + tq * (D / 4) + 4 * jj);
            const uint32_t s0 = sv.x, s1 = sv.y;
            b0[rp] = hfma2u(qB[jj][0], s0, hmul2u(qn0, s0));
            b1[rp] = hfma2u(qB[jj][1], s1, hmul2u(qn1, s1));
        }
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            if (MIXED && !((mx.tmask >> mm) & 1)) continue;
            const int rp = mm >> sh;
            const int wi = (2 * mm) / CPHK, r0 = (2 * mm) % CPHK;
            const uint32_t a0 = unpack<KB, true>(W[0][wi], r0), a1 = unpack<KB, true>(W[0][wi], r0 + 1);
            const uint32_t a2 = unpack<KB, true>(W[1][wi], r0), a3 = unpack<KB, true>(W[1][wi], r0 + 1);
            mma16816(sc[mm], a0, a1, a2, a3, b0[rp], b1[rp]);
        }
    }
    float p[4][2];
#pragma unroll
    for (int mm = 0; mm < 4; ++mm) {
        // row gq of tile mm reads field slot r0, row gq + 8 slot r0 + 1
        const int rp = mm >> sh, r0 = (2 * mm) % CPHK;
        const float o0 = slot_offset<KB, true>(r0), o1 = slot_offset<KB, true>(r0 + 1);
        p[mm][0] = (sc[mm][0] + sc[mm][1] + fmaf(-o0, ks[rp], kz[rp])) * alpha;
        p[mm][1] = (sc[mm][2] + sc[mm][3] + fmaf(-o1, ks[rp], kz[rp])) * alpha;
    }
    if (MIXED) {
        // tiles of window keys (Tqk is a multiple of G >= 16: tiles are whole)
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
            const int tau0 = mx.tb + 16 * mm;
            if (!((mx.tmask >> mm) & 1)) {   // not taken now
                p[mm][0] = p[mm][1] = -INFINITY;
                continue;
            }
            if (tau0 >= mx.Tqk && tau0 < mx.T) {
                const __half *krow = key_row(mx, tau0 + rr + 8 * (mi & 1));
                float f[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int jj = 0; jj < NJ; ++jj) {
                    uint32_t a[4];
                    ldsm_x4(a, krow + 8 * (2 * jj + (mi >> 1)));
                    mma16816(f, a[0], a[1], a[2], a[3], odd ? 0u : qB[jj][0], odd ? 0u : qB[jj][1]);
                }
                p[mm][0] = f[0] * alpha;
                p[mm][1] = f[2] * alpha;
            }
            if (tau0 + gq >= mx.T) p[mm][0] = -INFINITY;
            if (tau0 + gq + 8 >= mx.T) p[mm][1] = -INFINITY;
        }
    }
    if constexpr (PROBS) {
        if (srow) {
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                if (MIXED && !((mx.tmask >> mm) & 1)) continue;
                const int t0 = 16 * mm + gq;
                if (!MIXED || mx.tb + t0 < mx.T) srow[t0] = p[mm][0];
                if (!MIXED || mx.tb + t0 + 8 < mx.T) srow[t0 + 8] = p[mm][1];
            }
        }
    }
    softmax_update<D>(A, p);

    // ---- weights times values, 16 tokens at a time ----
    // sacc: the block's sum_t p_t s_t per (value group, column), for the
    // centring at the end (rows = groups, like zacc)
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        if (MIXED && !((mx.tmask >> kk) & 1)) continue;
        const PFrag f = p_fragments(p[kk][0], p[kk][1], tq, eB);
        // weights of quantized value tokens (tokens 2tq, 2tq+1 | 2tq+8, 2tq+9)
        uint32_t PH0 = f.PH0, PH1 = f.PH1, PL0 = f.PL0, PL1 = f.PL1;
        if (MIXED) {
            const int tk = mx.tb + 16 * kk + 2 * tq;
            const bool q0 = tk < mx.Tqv, q1 = tk + 1 < mx.Tqv, q8 = tk + 8 < mx.Tqv, q9 = tk + 9 < mx.Tqv;
            PH0 = keep_halves(PH0, q0, q1);
            PL0 = keep_halves(PL0, q0, q1);
            PH1 = keep_halves(PH1, q8, q9);
            PL1 = keep_halves(PL1, q8, q9);
        }
        // B = p s split: hi columns RN(ph s), lo columns (ph s - RN(ph s)) + pl s
        const uint32_t PL0m = hmul2u(PL0, m1), PL1m = hmul2u(PL1, m1);
        const uint32_t PH0n = hmul2u(PH0, nm), PH1n = hmul2u(PH1, nm);
        const __half *vszk = sVsz + kk * RG::VSZ_BLK;
        uint32_t b0[16], b1[16];
#pragma unroll
        for (int gi = 0; gi < 16; ++gi) {
            b0[gi] = b1[gi] = 0u;
            if (gi >= ngi) continue;
            // rows are lane-major: tokens 2 t, 2 t + 1, 2 t + 8, 2 t + 9 at 4 t
            const uint2 vv = *reinterpret_cast<const uint2 *>(vszk + gi * 16 + 4 * tq);
            const uint32_t v0 = vv.x, v1 = vv.y;
            b0[gi] = hfma2u(PL0m, v0, hfma2u(PH0, v0, hmul2u(PH0n, v0)));
            b1[gi] = hfma2u(PL1m, v1, hfma2u(PH1, v1, hmul2u(PH1n, v1)));
        }
        uint32_t Wv[WLV];
        const uint32_t *sVk = sV + kk * RG::VC_BLK;
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
            const uint32_t a0 = unpack_val_raw<VB>(Wp0, r0), a1 = unpack_val_raw<VB>(Wp0, r0 + 1);
            const uint32_t a2 = unpack_val_raw<VB>(Wp1, r0), a3 = unpack_val_raw<VB>(Wp1, r0 + 1);
            mma16816(A.oacc[mm], a0, a1, a2, a3, b0[mm >> sh], b1[mm >> sh]);
        }
        // value zero points and scales: rows [z or s][gi][16 tokens] (rows
        // gq >= ngi repeat a present row, rows gq + 8 only exist with 16 groups)
        const uint32_t bz0 = odd ? PL0 : PH0, bz1 = odd ? PL1 : PH1;
        const int zvrow = ngi >= 8 ? gq : (gq & (ngi - 1));
        {
            const __half *zrow = vszk + ngi * 16;
            const uint2 za = *reinterpret_cast<const uint2 *>(zrow + zvrow * 16 + 4 * tq);
            const uint32_t a0 = za.x, a2 = za.y;
            uint32_t a1 = 0, a3 = 0;
            if (ngi > 8) {
                const uint2 zb = *reinterpret_cast<const uint2 *>(zrow + (gq + 8) * 16 + 4 * tq);
                a1 = zb.x;
                a3 = zb.y;
            }
            mma16816(A.zacc, a0, a1, a2, a3, bz0, bz1);
        }
        {
            const __half *srw = vszk;
            const uint2 sa = *reinterpret_cast<const uint2 *>(srw + zvrow * 16 + 4 * tq);
            const uint32_t a0 = sa.x, a2 = sa.y;
            uint32_t a1 = 0, a3 = 0;
            if (ngi > 8) {
                const uint2 sb2 = *reinterpret_cast<const uint2 *>(srw + (gq + 8) * 16 + 4 * tq);
                a1 = sb2.x;
                a3 = sb2.y;
            }
            mma16816(sacc, a0, a1, a2, a3, bz0, bz1);
        }
        if (MIXED) {
            // window value tokens of this tile: fp16 rows, A = rows transposed
            const int tau0 = mx.tb + 16 * kk;
            if (tau0 + 15 >= mx.Tqv && tau0 < mx.T) {
                const __half *vrow = value_row(mx, tau0 + rr + 8 * (mi >> 1));
                const uint32_t c0 = odd ? f.PL0 : f.PH0, c1 = odd ? f.PL1 : f.PH1;
#pragma unroll
                for (int mm = 0; mm < NJ; ++mm) {
                    uint32_t a[4];
                    ldsm_x4_t(a, vrow + 8 * (2 * mm + (mi & 1)));
                    mma16816(A.oacc[mm], a[0], a[1], a[2], a[3], c0, c1);
                }
            }
        }
    }
    // centre the accumulators: rows of m-tile mm are value fields r0 (row
    // gq) and r0 + 1 (row gq + 8) of group mm >> sh; sacc row g holds that
    // group's sum over the block (lane 4 g' + tq holds rows g' and g' + 8)
    constexpr float c0 = 0.5f * (float)((1 << VB) - 1);
#pragma unroll
    for (int gi = 0; gi < ngi; ++gi) {
        const int src = (gi & 7) * 4 + tq;
        const float s0 = __shfl_sync(0xffffffffu, gi < 8 ? sacc[0] : sacc[2], src);
        const float s1 = __shfl_sync(0xffffffffu, gi < 8 ? sacc[1] : sacc[3], src);
#pragma unroll
        for (int mm = 0; mm < NJ; ++mm) {
            if ((mm >> sh) != gi) continue;
            const int r0 = (2 * mm) % CPHV;
            const float f0 = view_val(VB, r0).off + c0, f1 = view_val(VB, r0 + 1).off + c0;
            A.oacc[mm][0] = fmaf(-f0, s0, A.oacc[mm][0]);
            A.oacc[mm][1] = fmaf(-f0, s1, A.oacc[mm][1]);
            A.oacc[mm][2] = fmaf(-f1, s0, A.oacc[mm][2]);
            A.oacc[mm][3] = fmaf(-f1, s1, A.oacc[mm][3]);
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) A.zacc[k] = fmaf(c0, sacc[k], A.zacc[k]);
}

// Per-warp result: m, l per head and o[head][d] = sum p v (value zero points
// included), written at the start of the warp's region.
template <int D, int SH>
__device__ __forceinline__ void warp_result(WarpAcc<D> &A, float *wres) {
    constexpr int NJ = D / 16;
    constexpr int ngi = (D / 16) >> SH;
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    float lrun = A.lrun;
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 4);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 8);
    lrun += __shfl_xor_sync(0xffffffffu, lrun, 16);
    const float zr0 = A.zacc[0] + A.zacc[1], zr1 = A.zacc[2] + A.zacc[3];
    float vz[16];
#pragma unroll
    for (int gi = 0; gi < 16; ++gi)
        vz[gi] = gi < ngi ? __shfl_sync(0xffffffffu, gi < 8 ? zr0 : zr1, (gi & 7) * 4 + tq) : 0.f;
    __syncwarp();
    if (gq == 0) {
        wres[tq] = A.mrun;
        wres[4 + tq] = lrun;
    }
    float *wo = wres + 8;
#pragma unroll
    for (int mm = 0; mm < NJ; ++mm) {
        const int gi = mm >> SH;
        wo[tq * D + 16 * mm + gq] = A.oacc[mm][0] + A.oacc[mm][1] + vz[gi];
        wo[tq * D + 16 * mm + gq + 8] = A.oacc[mm][2] + A.oacc[mm][3] + vz[gi];
    }
}

// ---------------------------------------------------------------------------
// The persistent kernel.  Work units: for each (sequence i, kv head j, head
// group qg), its blocks whose keys and values are all quantized (one unit
// each) and its remaining blocks (MW units each), laid end to end; CTA c
// takes units [c U / C, (c+1) U / C).  Each stretch of one (i, j, qg) inside
// a CTA is a segment.  Its fully quantized blocks stream through the warps'
// rings; its other blocks (those holding fp16 window tokens, at the end of
// the sequence) are then staged one at a time by the whole CTA, record and
// window rows with one round trip, and split into 16-token tiles over the
// warps.  The warps merge in shared memory and write one partial per
// segment; the last CTA to finish a segment of that (i, j, qg) merges all
// of its partials.
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int cta_of_unit(long long u, long long U, int C) {
    if ((unsigned long long)U * (unsigned)C < (1ull << 32))   // 32-bit arithmetic suffices (u < U)
        return (int)(((unsigned)(u + 1) * (unsigned)C - 1u) / (unsigned)U);
    return (int)(((u + 1) * C - 1) / U);
}

template <int D, int KB, int VB, int SH, bool PROBS, bool FUSED>
__global__ void __launch_bounds__(256, 2)
    decode_kernel(KiviGeom g, KiviDev dv, const __half *__restrict__ q, int hq,
                  __half *__restrict__ out, DecodePlan plan, DecodeUnits units, ProbsOut po, FusedStep fs) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int NJ = D / 16;
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int eB = gq >> 1;
    const int hg = hq / g.h, QG = plan.qgroups, HQG = g.h * QG;
    using RG = Rec<D, KB, VB, SH>;
    const size_t wstride = warp_region(g, plan.stages);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    unsigned char *ring = smem + bar_region(nw, plan.stages);
    unsigned char *myregion = ring + warp * wstride;
    uint64_t *mybars = bars + warp * plan.stages;
    const float alpha = kLog2e * rsqrtf((float)D);
    const long long U = units.total;
    const int C = gridDim.x, c = blockIdx.x;
    long long u = (long long)c * U / C;
    const long long u_end = (long long)(c + 1) * U / C;
    __shared__ int s_seg[11];   // i, jq, o0, o1, Wi; T, Tqk, Tqv (after the append); fused flags;
                                // the pair's first CTA and its number of CTAs (partials)
    __shared__ int s_last;
    __shared__ float sML[8];    // per head: max over the warps (or partials), then the weighted sum of l
    __shared__ float sWt[32];   // [warp][head]: the warp's weight
    __shared__ __align__(16) __half s_frows[FUSED ? 3 * D : 8];   // the fused append's rows
    __shared__ unsigned s_fphase;                                 // ... and the phase of their barrier
    // The barriers live for the whole kernel: a warp's n-th block (counted
    // across all its segments) goes to slot n % stages and completes phase
    // n / stages of that slot's barrier.
    if (threadIdx.x <= nw * plan.stages + 1) mbar_init(bars + threadIdx.x, 1);
    if (threadIdx.x == 0) s_fphase = 0u;
    fence_mbar_init();
    __syncthreads();
    // The kernel is launched as a programmatic dependent of the one before
    // it on the stream (usually the append): the set-up above touched only
    // shared memory and parameters; nothing in global memory is read before
    // that kernel has finished.  A dependent launched after this one (the
    // weights' finalizing kernel) may in turn start its own set-up.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int rslot = 0;         // this warp's next ring slot to consume ...
    unsigned rphase = 0;   // ... and the phase its barrier completes next
    bool dead = false;     // a wait of this warp timed out: it streams no more blocks
    bool cdead = false;   // a wait of the CTA's mixed-block barrier timed out
    uint64_t *cbar = bars + nw * plan.stages;   // the CTA's mixed-block barrier
    uint64_t *fbar = cbar + 1;                   // the fused append's rows
    unsigned cphase = 0;
    const uint64_t pol_stream = policy_evict_first();
    // mixed blocks staged per round: as many regions as the ring holds (<= 2)
    const size_t mreg = mixed_region(g);
    const int mper = max(1, min(2, (int)(max((size_t)nw * wstride, mreg) / mreg)));

    while (u < u_end) {
        if (threadIdx.x == 0) {
            int lo = 0, hi = g.b;   // largest i with HQG * start[i] <= u
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if ((long long)HQG * units.start[mid] <= u) lo = mid; else hi = mid;
            }
            // Counters (read first: their loads are in flight during the
            // arithmetic below).  FUSED: the device holds them before this
            // step's append; a sequence whose key window is not full is
            // appended by this launch (flag 1; flag 2: its value queue's
            // oldest token pops), the others were appended by the launch
            // before (the counters after the append follow from item 4's
            // schedule either way).
            int T = dv.T[lo], Tqk = dv.Tqk[lo], Tqv = dv.Tqv[lo], fl = 0;
            const int Wi = units.start[lo + 1] - units.start[lo];
            const long long rem = u - (long long)HQG * units.start[lo];
            const int o0 = (int)(rem % Wi);
            s_seg[0] = lo;
            s_seg[1] = (int)(rem / Wi);
            s_seg[2] = o0;
            s_seg[3] = (int)min((long long)Wi, o0 + (u_end - u));
            s_seg[4] = Wi;
            // the CTAs that share this pair
            const long long Pp = u - o0;
            const int cf = cta_of_unit(Pp, U, C);
            s_seg[9] = cf;
            s_seg[10] = cta_of_unit(Pp + Wi - 1, U, C) - cf + 1;
            if constexpr (FUSED) {
                if (append_counters_ok(g, T, Tqk, Tqv)) {
                    const bool pop = T - Tqv == g.R + 1, app = T - Tqk != g.R;
                    fl = (app ? 1 : 0) | (pop ? 2 : 0);
                    if (!app) Tqk += g.R;
                    Tqv += pop ? 1 : 0;
                    T += 1;
                } else {
                    atomicOr(dv.status, KIVI_FLAG_COUNTER);
                }
            }
            s_seg[5] = T;
            s_seg[6] = Tqk;
            s_seg[7] = Tqv;
            s_seg[8] = fl;
        }
        // the rings were last written and read by generic stores and loads
        // (the previous segment's merge): order them before the async copies
        fence_proxy_async();
        __syncthreads();
        const int i = s_seg[0], jq = s_seg[1], o0 = s_seg[2], o1 = s_seg[3], Wi = s_seg[4];
        const int j = jq / QG, qg = jq % QG;
        const int e0 = qg * 4, nh = min(4, hg - e0);
        const int T = s_seg[5], Tqk = s_seg[6], Tqv = s_seg[7];
        const bool app = FUSED && (s_seg[8] & 1), pop = FUSED && (s_seg[8] & 2);
        const int Tqv0 = pop ? Tqv - 1 : Tqv;   // the value queue before this launch's pop
        // an appending sequence stages the popped token's block as a window
        // block: it counts its value queue before the pop
        const int nfull = min(Tqk, app ? Tqv0 : Tqv) / KIVI_KBLK;
        const int nblk = (T + KIVI_KBLK - 1) / KIVI_KBLK;
        const int nfh = units.full[i];
        const int MW = units.mixed_weight;

        // query fragments of this (sequence, kv head, head group)
        uint32_t qB[NJ][2];
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                qB[jj][hh] = eB < nh ? *reinterpret_cast<const uint32_t *>(
                                           q + ((size_t)i * hq + j * hg + e0 + eB) * D + 16 * jj + 8 * hh + 2 * tq)
                                     : 0u;
        WarpAcc<D> A;
        acc_reset<D>(A);
        // PROBS: this lane's head's row of scores (null for absent heads)
        float *prow = nullptr;
        if constexpr (PROBS)
            if (tq < nh) prow = po.p + ((size_t)i * hq + j * hg + e0 + tq) * (size_t)po.ld;

        // Blocks of the segment: past the pair's lead of units.lead units
        // (no blocks), with b0, b1 the segment's range counted from the
        // lead's end, units [b0, min(b1, nfh)) are blocks of the same index,
        // units nfh + MW m in [b0, b1) are block nfh + m; blocks past the
        // data (>= nblk) are skipped.
        const unsigned char *recs = dv.blk + rec_off(g, i, j, 0);
        const int b0 = max(o0 - units.lead, 0), b1 = max(o1 - units.lead, 0);
        const int nA = max(0, min(b1, nfh) - b0);
        const int m0 = b0 > nfh ? (b0 - nfh + MW - 1) / MW : 0;
        const int m1 = b1 > nfh ? (b1 - nfh + MW - 1) / MW : 0;
        const int nL = nA + max(0, m1 - m0);
        auto blk = [&](int x) { return x < nA ? b0 + x : nfh + m0 + (x - nA); };
        auto first_at_least = [&](int kb) {   // first x with blk(x) >= kb (blk increases)
            int lo = 0, hi = nL;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (blk(mid) >= kb) hi = mid; else lo = mid + 1;
            }
            return lo;
        };
        const int nD = first_at_least(nblk);            // blocks with data
        const int xm = min(first_at_least(nfull), nD);  // mixed blocks: [xm, nD)
        // Packed blocks [0, xm) stream through the warps' rings, interleaved
        // (warp w takes blocks w, w + nw, ...: the CTA's warps read adjacent
        // records together); mixed blocks [xm, nD) follow, one at a time,
        // with the whole CTA (below).
        int taken = 0;   // blocks this warp has taken
        auto grab = [&]() { return warp + nw * taken++; };
        const __half *kwin = dv.Kf + kf_slice(g, i, j), *vwin = dv.Vf + vf_slice(g, i, j);
        if (threadIdx.x == 0) {
            // the mixed blocks are read last: bring their records and window
            // rows into L2 now
            const uint64_t keep = policy_evict_last();
            for (int x = xm; x < nD; ++x) {
                const int kb = blk(x), tb = kb * KIVI_KBLK, te = min(tb + KIVI_KBLK, T);
                prefetch_l2(recs + (size_t)kb * RG::BYTES, (unsigned)RG::BYTES, keep);
                prefetch_rows<D>(kwin, g.R, max(tb, Tqk), te, keep);
                prefetch_rows<D>(vwin, g.R + 1, max(tb, Tqv), te, keep);
            }
        }
        // Slots and phases advance incrementally: the ring position (rslot,
        // rphase) of the next block to consume and the slot of the next
        // block to issue carry over from segment to segment.
        int issued = 0, consumed = 0;
        bool more = !dead;   // blocks may be left to take
        int islot = rslot;
        auto next_slot = [&](int sl) { return sl + 1 == plan.stages ? 0 : sl + 1; };
        auto take_and_issue = [&]() {
            const int x = grab();
            if (x >= xm) {
                more = false;
                return;
            }
            issue_block<RG::BYTES>(myregion + (size_t)islot * RG::BYTES, mybars + islot, recs, blk(x), pol_stream);
            islot = next_slot(islot);
            ++issued;
        };
        while (more && issued < plan.stages) take_and_issue();
        // FUSED: the pair's append is done by the CTA holding, in this
        // segment, the block its maintenance touches (the popped value
        // token's, else the new token's), with its last warp, while that
        // warp's first ring copies are in flight: the rows it needs are
        // bulk-copied, then fused_append_pair.  No other CTA of the launch
        // reads what it writes (the popped token's record fields, which this
        // CTA stages afterwards; the window slots the new token takes, which
        // every CTA skips).
        if constexpr (FUSED) {
            if (app && qg == 0 && warp == nw - 1) {
                const int ob = (pop ? Tqv0 : T - 1) / KIVI_KBLK;
                const int xo = first_at_least(ob);
                if (xo >= xm && xo < nD && blk(xo) == ob) {
                    if (lane == 0) {
                        const size_t kv_off = ((size_t)i * g.h + j) * D;
                        mbar_expect_tx(fbar, (pop ? 3u : 2u) * 2 * D);
                        if (pop) bulk_g2s(s_frows, vwin + (size_t)(Tqv0 % (g.R + 1)) * D, 2 * D, fbar);
                        bulk_g2s(s_frows + D, fs.k + kv_off, 2 * D, fbar);
                        bulk_g2s(s_frows + 2 * D, fs.v + kv_off, 2 * D, fbar);
                    }
                    fused_append_pair<D, KB, VB, SH>(g, dv, fs, i, j, T - 1, Tqk, Tqv0, pop, s_frows, fbar, s_fphase);
                    if (lane == 0) s_fphase ^= 1u;
                    __syncwarp();
                }
            }
        }
        __syncwarp();
        MixCtx mc;   // unused by the packed path
        bool timed_out = false;
        while (consumed < issued) {
            if (!__all_sync(0xffffffffu, mbar_wait(mybars + rslot, rphase))) {
                timed_out = true;
                break;
            }
            float *srow = nullptr;
            if constexpr (PROBS)   // the warp's consumed-th block is its grab of that index
                if (prow) srow = prow + (size_t)blk(warp + nw * consumed) * KIVI_KBLK;
            do_block<D, KB, VB, SH, false, PROBS>(A, qB, myregion + (size_t)rslot * RG::BYTES, alpha, mc, srow);
            __syncwarp();
            // Refill the slot just read.  Its packed data was only read (by
            // loads whose values the block has consumed): no proxy fence.
            if (more) take_and_issue();
            rslot = next_slot(rslot);
            rphase ^= rslot == 0 ? 1u : 0u;
            ++consumed;
        }
        if (timed_out) {
            if (lane == 0) atomicOr(dv.status, KIVI_FLAG_WAIT);
            // wait (bounded) for this warp's copies still in flight before
            // its region is reused; the warp then streams nothing more
            for (; consumed < issued; ++consumed) {
                mbar_wait(mybars + rslot, rphase);
                rslot = next_slot(rslot);
                rphase ^= rslot == 0 ? 1u : 0u;
            }
            acc_reset<D>(A);
            dead = true;
        }

        // ---- mixed blocks: per round the CTA stages up to mper of them,
        // each block's record and fp16 window rows (a few bulk copies: the
        // rows are consecutive in their rings) in a region of the ring, with
        // one round trip; then the warps take their 16-token tiles (tile t
        // of the round's block k goes to warp (4 k + t) mod nw).  The rows
        // are not padded: the tiles' ldmatrix reads conflict on banks, a
        // small cost next to more copies.
        // Row r of a block's key (value) rows is token tb + r.  An appending
        // sequence's new token T0 is not read from the windows (its slots
        // are being written by the pair's owner): its key and value rows
        // are copied from the step's inputs with the round's other copies.
        const int RS = 2 * D;
        // the new token T0 = T - 1 if appended here (else none: T)
        const int tnew = (FUSED && (s_seg[8] & 1)) ? T - 1 : T;
        for (int x0 = xm; x0 < nD && !cdead; x0 += mper) {
            const int nrb = min(mper, nD - x0);
            fence_proxy_async();   // earlier generic reads and writes of the ring
            __syncthreads();
            if (warp == 0) {
                unsigned bytes = 0;
                for (int k = 0; k < nrb; ++k) {
                    const int kb = blk(x0 + k), tb = kb * KIVI_KBLK, te = min(tb + KIVI_KBLK, tnew);
                    bytes += RG::BYTES + (rows_to_stage(max(tb, Tqk), te, g.R) +
                                         rows_to_stage(max(tb, Tqv), te, g.R + 1)) * 2 * D;
                    if (tnew < T && tnew >= tb && tnew < tb + KIVI_KBLK) bytes += 4 * D;
                }
                if (lane == 0) mbar_expect_tx(cbar, bytes);
                for (int k = 0; k < nrb && lane == 0; ++k) {
                    const int kb = blk(x0 + k), tb = kb * KIVI_KBLK, te = min(tb + KIVI_KBLK, tnew);
                    unsigned char *reg = ring + (size_t)k * mreg;
                    const int ka = max(tb, Tqk), va = max(tb, Tqv);
                    bulk_g2s(reg, recs + (size_t)kb * RG::BYTES, (unsigned)RG::BYTES, cbar);
                    copy_rows<D>(reg + RG::BYTES + (size_t)(ka - tb) * RS, kwin, g.R, ka, te, cbar);
                    copy_rows<D>(reg + RG::BYTES + (size_t)(KIVI_KBLK + va - tb) * RS, vwin, g.R + 1, va, te,
                                 cbar);
                    if (tnew < T && tnew >= tb && tnew < tb + KIVI_KBLK) {
                        const size_t kv_off = ((size_t)i * g.h + j) * D;
                        bulk_g2s(reg + RG::BYTES + (size_t)(tnew - tb) * RS, fs.k + kv_off, 2 * D, cbar);
                        bulk_g2s(reg + RG::BYTES + (size_t)(KIVI_KBLK + tnew - tb) * RS, fs.v + kv_off, 2 * D,
                                 cbar);
                    }
                }
            }
            for (int k = 0; k < nrb; ++k) {
                unsigned char *zrow = ring + (size_t)k * mreg + RG::BYTES + (size_t)2 * KIVI_KBLK * RS;
                for (int e = threadIdx.x; e < 2 * D / 16; e += blockDim.x)
                    reinterpret_cast<uint4 *>(zrow)[e] = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
            const bool ok = mbar_wait(cbar, cphase);
            cphase ^= 1u;
            if (!__syncthreads_and(ok)) {
                if (threadIdx.x == 0) atomicOr(dv.status, KIVI_FLAG_WAIT);
                mbar_wait(cbar, cphase ^ 1u);   // bounded: let the copies land before the ring is reused
                cdead = true;
                break;
            }
            for (int w4 = warp; w4 < 4 * nrb; w4 += nw) {
                const int k = w4 >> 2, t = w4 & 3;
                const int kb = blk(x0 + k), tb = kb * KIVI_KBLK;
                if (tb + 16 * t >= T || dead) continue;
                unsigned char *reg = ring + (size_t)k * mreg;
                mc.tb = tb;
                mc.tmask = 1 << t;
                mc.T = T;
                mc.Tqk = Tqk;
                mc.Tqv = Tqv;
                mc.krows = reg + RG::BYTES;
                mc.vrows = reg + RG::BYTES + (size_t)KIVI_KBLK * RS;
                mc.ka = tb;
                mc.va = tb;
                mc.zrow = reg + RG::BYTES + (size_t)2 * KIVI_KBLK * RS;
                mc.RS = RS;
                do_block<D, KB, VB, SH, true, PROBS>(A, qB, reg, alpha, mc, PROBS && prow ? prow + tb : nullptr);
            }
        }
        __syncthreads();   // the ring holds mixed data no longer needed

        // ---- merge the warps into this CTA's partial of (i, j, qg) ----
        // A partial is PS = D + 4 floats: m, l, two unused, acc[D] (rows
        // 16-byte aligned for the vector loads of the final merge).
        constexpr int PS = D + 4, NC4 = D / 4;
        __syncwarp();
        warp_result<D, SH>(A, reinterpret_cast<float *>(myregion));
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane 4 w + e: warp w's weight for head e, relative to the max
            // over the warps; lanes 0-3 also hold the sum of the weighted l
            const int w = lane >> 2, e = lane & 3;
            const float *r = reinterpret_cast<const float *>(ring + (size_t)w * wstride);
            const float m = w < nw ? r[e] : -INFINITY;
            float M = m;
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 4));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
            M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
            const float wt = M == -INFINITY ? 0.f : ex2(m - M);
            float L = w < nw ? wt * r[4 + e] : 0.f;
            L += __shfl_xor_sync(0xffffffffu, L, 4);
            L += __shfl_xor_sync(0xffffffffu, L, 8);
            L += __shfl_xor_sync(0xffffffffu, L, 16);
            sWt[lane] = wt;
            if (lane < 4) {
                sML[lane] = M;
                sML[4 + lane] = L;
            }
        }
        __syncthreads();
        const int cfirst = s_seg[9], np = s_seg[10];
        const int slot = c - cfirst;
        float *const prow0 = dv.part + ((size_t)i * hq + j * hg + e0) * g.smax * PS;   // head e: + e smax PS
        for (int x = threadIdx.x; x < nh * (NC4 + 1); x += blockDim.x) {
            const int e = x / (NC4 + 1), c4 = x % (NC4 + 1);
            float *dst = prow0 + ((size_t)e * g.smax + slot) * PS;
            if (c4 == NC4) {
                *reinterpret_cast<float2 *>(dst) = make_float2(sML[e], sML[4 + e]);
            } else {
                float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int w = 0; w < nw; ++w) {
                    const float wt = sWt[4 * w + e];
                    const float4 o4 = *reinterpret_cast<const float4 *>(
                        reinterpret_cast<const float *>(ring + (size_t)w * wstride) + 8 + e * D + 4 * c4);
                    a4.x = fmaf(wt, o4.x, a4.x);
                    a4.y = fmaf(wt, o4.y, a4.y);
                    a4.z = fmaf(wt, o4.z, a4.z);
                    a4.w = fmaf(wt, o4.w, a4.w);
                }
                *reinterpret_cast<float4 *>(dst + 4 + 4 * c4) = a4;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            // one acquire-release add: it releases the partial the CTA's
            // threads wrote before the barrier above (a release is cumulative)
            // and, in the last CTA, acquires every earlier CTA's partial (the
            // adds on the ticket form one release sequence); the barrier below
            // passes the acquire on to the merging threads
            unsigned *tk = dv.merge_ticket + ((size_t)i * g.h + j) * 4 + qg;
            unsigned prev;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(tk) : "memory");
            s_last = prev == (unsigned)np - 1u;
            if (s_last) *tk = 0u;
        }
        __syncthreads();
        if (s_last && np <= kFastMerge &&
            np <= kFastMergeV * max(1, min(8, (int)blockDim.x / (nh * NC4)))) {
            // Merge the pair's partials (up to kFastMerge of them) with one
            // round trip: each thread loads every partial's (m, l) of its
            // head, and m and the column's accumulator of its own partials
            // sub, sub + S, ... (at most kFastMergeV), all together, forms
            // the weights itself, and the S subsets of a column are summed
            // in shared memory (the ring is free: the warps' results were
            // merged above).
            const int ncol = nh * NC4;
            const int S = max(1, min(8, (int)blockDim.x / ncol));
            float4 *sm_a = reinterpret_cast<float4 *>(ring);   // [S][ncol]
            for (int it = threadIdx.x; it < ncol * S; it += blockDim.x) {
                const int col = it % ncol, sub = it / ncol;
                const int e = col / NC4, c4 = col % NC4;
                const float *hp = prow0 + (size_t)e * g.smax * PS;
                float2 ml[kFastMerge];
                float mv[kFastMergeV];
                float4 v[kFastMergeV];
#pragma unroll
                for (int y = 0; y < kFastMerge; ++y)
                    ml[y] = y < np ? __ldcg(reinterpret_cast<const float2 *>(hp + (size_t)y * PS))
                                   : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int y = 0; y < kFastMergeV; ++y) {
                    const int ys = sub + y * S;
                    mv[y] = ys < np ? __ldcg(hp + (size_t)ys * PS) : -INFINITY;
                    v[y] = ys < np ? __ldcg(reinterpret_cast<const float4 *>(hp + (size_t)ys * PS + 4 + 4 * c4))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                float M = -INFINITY;
#pragma unroll
                for (int y = 0; y < kFastMerge; ++y) M = fmaxf(M, ml[y].x);
                float L = 0.f;
                if (M != -INFINITY)
#pragma unroll
                    for (int y = 0; y < kFastMerge; ++y)
                        if (y < np) L = fmaf(ex2(ml[y].x - M), ml[y].y, L);
                const float inv = L > 0.f ? 1.f / L : 0.f;
                float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if (M != -INFINITY)
#pragma unroll
                    for (int y = 0; y < kFastMergeV; ++y) {
                        if (sub + y * S >= np) continue;
                        const float w = ex2(mv[y] - M) * inv;
                        a4.x = fmaf(w, v[y].x, a4.x);
                        a4.y = fmaf(w, v[y].y, a4.y);
                        a4.z = fmaf(w, v[y].z, a4.z);
                        a4.w = fmaf(w, v[y].w, a4.w);
                    }
                sm_a[it] = a4;
                if constexpr (PROBS) {
                    if (c4 == 0 && sub == 0) {
                        float *mlo = dv.ml + ((size_t)i * hq + j * hg + e0 + e) * 2;
                        mlo[0] = M;
                        mlo[1] = inv;
                    }
                }
            }
            __syncthreads();
            for (int col = threadIdx.x; col < ncol; col += blockDim.x) {
                const int e = col / NC4, c4 = col % NC4;
                float4 a4 = sm_a[col];
                for (int k = 1; k < S; ++k) {
                    const float4 b4 = sm_a[k * ncol + col];
                    a4.x += b4.x;
                    a4.y += b4.y;
                    a4.z += b4.z;
                    a4.w += b4.w;
                }
                const __half2 lo = __floats2half2_rn(a4.x, a4.y), hi = __floats2half2_rn(a4.z, a4.w);
                uint2 o2;
                o2.x = h2u(lo);
                o2.y = h2u(hi);
                *reinterpret_cast<uint2 *>(out + ((size_t)i * hq + j * hg + e0 + e) * D + 4 * c4) = o2;
            }
        } else if (s_last) {
            // Merge the pair's partials.  When they fit in the ring (free:
            // the warps' results were merged above) beside the scratch
            // below, they are bulk-copied there, one copy per head, with one
            // round trip; otherwise they are read from global memory.  Their
            // (m, l) go to shared memory, each head's weights are formed
            // there by one warp, then the accumulators are read as float4
            // columns, S partials per column in flight (S threads a column,
            // summed in shared memory).
            const int ncol = nh * NC4;
            const int S = max(1, min(8, (int)blockDim.x / ncol));
            const size_t hbytes = (size_t)np * PS * 4;   // one head's partials
            const bool staged = !cdead && (size_t)nh * hbytes + (size_t)8 * np * 4 + (size_t)S * ncol * 16 <=
                                              max((size_t)nw * wstride, mreg);
            float *stage = reinterpret_cast<float *>(ring);   // [nh][np][PS] when staged
            float *sm_m = reinterpret_cast<float *>(ring + (staged ? (size_t)nh * hbytes : 0));   // [nh][np]
            float *sm_w = sm_m + 4 * np;                      // [nh][np]: l, then the weights
            float4 *sm_a = reinterpret_cast<float4 *>(sm_w + 4 * np);   // [S][nh NC4] (16-byte aligned)
            // head e's partial y: stage + (e np + y) PS, else prow0 + (e smax + y) PS
            const size_t hst = staged ? (size_t)np * PS : (size_t)g.smax * PS;
            bool mok = true;
            if (staged) {
                fence_proxy_async();   // the ring's earlier generic reads and writes
                __syncthreads();
                if (threadIdx.x == 0) {
                    // the partials were written by generic stores (of this and
                    // the other CTAs, ordered by the ticket): order them
                    // before the asynchronous copies that read them
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    mbar_expect_tx(cbar, (unsigned)(nh * hbytes));
                    for (int e = 0; e < nh; ++e)
                        bulk_g2s(stage + (size_t)e * np * PS, prow0 + (size_t)e * g.smax * PS, (unsigned)hbytes,
                                 cbar);
                }
                const bool ok = mbar_wait(cbar, cphase);
                cphase ^= 1u;
                if (!__syncthreads_and(ok)) {
                    if (threadIdx.x == 0) atomicOr(dv.status, KIVI_FLAG_WAIT);
                    mbar_wait(cbar, cphase ^ 1u);   // bounded: let the copies land before the ring is reused
                    cdead = true;
                    mok = false;
                }
            }
            const float *pbase = staged ? stage : prow0;
            auto ld2 = [&](const float *p) {
                return staged ? *reinterpret_cast<const float2 *>(p) : __ldcg(reinterpret_cast<const float2 *>(p));
            };
            auto ld4 = [&](const float *p) {
                return staged ? *reinterpret_cast<const float4 *>(p) : __ldcg(reinterpret_cast<const float4 *>(p));
            };
            for (int x = threadIdx.x; mok && x < nh * np; x += blockDim.x) {
                const int e = x / np, y = x % np;
                const float2 ml = ld2(pbase + (size_t)e * hst + (size_t)y * PS);
                sm_m[x] = ml.x;
                sm_w[x] = ml.y;
            }
            __syncthreads();
            if (mok && warp < nh) {
                const int e = warp;
                float M = -INFINITY;
                for (int y = lane; y < np; y += 32) M = fmaxf(M, sm_m[e * np + y]);
                for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                float L = 0.f;
                if (M != -INFINITY)
                    for (int y = lane; y < np; y += 32) L = fmaf(ex2(sm_m[e * np + y] - M), sm_w[e * np + y], L);
                for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
                const float inv = L > 0.f ? 1.f / L : 0.f;
                __syncwarp();
                for (int y = lane; y < np; y += 32)
                    sm_w[e * np + y] = M == -INFINITY ? 0.f : ex2(sm_m[e * np + y] - M) * inv;
                if constexpr (PROBS) {
                    if (lane == 0) {
                        float *ml = dv.ml + ((size_t)i * hq + j * hg + e0 + e) * 2;
                        ml[0] = M;
                        ml[1] = inv;
                    }
                }
            }
            __syncthreads();
            // (column, subset) items: S subsets of the partials per float4
            // column when the CTA has threads for them, else one; each
            // thread takes items in turn
            for (int it = threadIdx.x; mok && it < ncol * S; it += blockDim.x) {
                const int col = it % ncol, sub = it / ncol;
                const int e = col / NC4, c4 = col % NC4;
                const float *src = pbase + (size_t)e * hst + 4 + 4 * c4;
                const float *wr = sm_w + e * np;
                float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
                int y = sub;
                for (; y + 3 * S < np; y += 4 * S) {   // four partials in flight
                    const float4 v0 = ld4(src + (size_t)y * PS);
                    const float4 v1 = ld4(src + (size_t)(y + S) * PS);
                    const float4 v2 = ld4(src + (size_t)(y + 2 * S) * PS);
                    const float4 v3 = ld4(src + (size_t)(y + 3 * S) * PS);
                    const float w0 = wr[y], w1 = wr[y + S], w2 = wr[y + 2 * S], w3 = wr[y + 3 * S];
                    a4.x = fmaf(w0, v0.x, fmaf(w1, v1.x, fmaf(w2, v2.x, fmaf(w3, v3.x, a4.x))));
                    a4.y = fmaf(w0, v0.y, fmaf(w1, v1.y, fmaf(w2, v2.y, fmaf(w3, v3.y, a4.y))));
                    a4.z = fmaf(w0, v0.z, fmaf(w1, v1.z, fmaf(w2, v2.z, fmaf(w3, v3.z, a4.z))));
                    a4.w = fmaf(w0, v0.w, fmaf(w1, v1.w, fmaf(w2, v2.w, fmaf(w3, v3.w, a4.w))));
                }
                for (; y < np; y += S) {
                    const float4 v = ld4(src + (size_t)y * PS);
                    const float w0 = wr[y];
                    a4.x = fmaf(w0, v.x, a4.x);
                    a4.y = fmaf(w0, v.y, a4.y);
                    a4.z = fmaf(w0, v.z, a4.z);
                    a4.w = fmaf(w0, v.w, a4.w);
                }
                sm_a[it] = a4;
            }
            __syncthreads();
            for (int col = threadIdx.x; col < ncol; col += blockDim.x) {
                const int e = col / NC4, c4 = col % NC4;
                float4 a4 = sm_a[col];
                for (int k = 1; k < S; ++k) {
                    const float4 b4 = sm_a[k * ncol + col];
                    a4.x += b4.x;
                    a4.y += b4.y;
                    a4.z += b4.z;
                    a4.w += b4.w;
                }
                const __half2 lo = __floats2half2_rn(a4.x, a4.y), hi = __floats2half2_rn(a4.z, a4.w);
                uint2 o2;
                o2.x = h2u(lo);
                o2.y = h2u(hi);
                *reinterpret_cast<uint2 *>(out + ((size_t)i * hq + j * hg + e0 + e) * D + 4 * c4) = o2;
            }
        }
        __syncthreads();
        u += o1 - o0;
    }
}

template <int D, int KB, int VB, int SH, bool PROBS, bool FUSED>
cudaError_t launch_t(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, __half *out,
                     const DecodePlan &plan, const DecodeUnits &units, const ProbsOut &po, const FusedStep &fs,
                     cudaStream_t st) {
    using RG = Rec<D, KB, VB, SH>;
    if (g.rec_bytes != RG::BYTES || g.off_ksz != RG::OFF_KSZ || g.off_vc != RG::OFF_VC ||
        g.off_vsz != RG::OFF_VSZ || g.vc_blk != RG::VC_BLK || g.vsz_blk != RG::VSZ_BLK)
        return cudaErrorInvalidValue;   // the record layout the kernel was compiled for
    size_t rings = (size_t)plan.warps * warp_region(g, plan.stages);
    if (rings < mixed_region(g)) rings = mixed_region(g);
    const size_t smem = bar_region(plan.warps, plan.stages) + rings;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, KB, VB, SH, PROBS, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: the CTAs may be placed while the
    // previous kernel (the append) finishes; the kernel waits for it
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.ctas);
    cfg.blockDim = dim3(plan.warps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<D, KB, VB, SH, PROBS, FUSED>, g, dv, q, hq, out, plan, units, po,
                              fs);
}

template <int D, int KB, int VB, bool PROBS, bool FUSED>
cudaError_t launch_g(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, __half *out,
                     const DecodePlan &plan, const DecodeUnits &units, const ProbsOut &po, const FusedStep &fs,
                     cudaStream_t st) {
    switch (g.G) {
    case 16: return launch_t<D, KB, VB, 0, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
    case 32: return launch_t<D, KB, VB, 1, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
    case 64: return launch_t<D, KB, VB, 2, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
    default:
        if constexpr (D >= 128) return launch_t<D, KB, VB, 3, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
        return cudaErrorInvalidValue;
    }
}

// PROBS: the weights variant; FUSED: the variant that appends (fs).
template <int D, bool PROBS, bool FUSED = false>
cudaError_t launch_d(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq, __half *out,
                     const DecodePlan &plan, const DecodeUnits &units, const ProbsOut &po, cudaStream_t st,
                     const FusedStep &fs = FusedStep{nullptr, nullptr, nullptr}) {
    static_assert(!(PROBS && FUSED), "the weights variant does not append");
    if (g.kbits == 2 && g.vbits == 2) return launch_g<D, 2, 2, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
    if (g.kbits == 2 && g.vbits == 4) return launch_g<D, 2, 4, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
    if (g.kbits == 4 && g.vbits == 2) return launch_g<D, 4, 2, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
    return launch_g<D, 4, 4, PROBS, FUSED>(g, dv, q, hq, out, plan, units, po, fs, st);
}

}  // namespace
