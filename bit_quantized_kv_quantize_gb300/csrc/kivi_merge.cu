// kivi_merge.cu -- the split-K merge of the decode step.
//
// The persistent decode kernel (kivi_decode_impl.cuh) leaves, for every
// (sequence i, kv head j, group of <= 4 query heads) and every CTA that took
// part of it, a partial (m, l, acc[d]) per query head in base 2: m the
// largest score, l the sum of 2^(s - m), acc the weighted value sum.  Here
// the partials of each (sequence, query head) row are combined with
// log-sum-exp weights,
//   M = max_y m_y,  L = sum_y 2^(m_y - M) l_y,
//   out[c] = sum_y 2^(m_y - M) acc_y[c] / L,
// which is item 5's softmax over all tokens split into the CTAs' token
// ranges (the flash-decoding combination; not on the pages).
//
// A row's partials sit in slots 0 .. np-1 of its partial buffer, np being
// the number of persistent CTAs whose unit ranges overlap the row's pair:
// the same arithmetic as the decode kernel's, from the same plan.
#include "kivi_internal.cuh"

namespace {

constexpr int kMaxSlots = 640;   // partial slots a row may have (the host checks)

__host__ __device__ __forceinline__ long long cta_of(long long u, long long U, int C) {
    return ((u + 1) * C - 1) / U;
}

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// CTA = (row, chunk of CP channels); thread (s, c): channel chunk*CP + c,
// partials s, s + S, ...; the S partial sums of a channel meet in shared
// memory.  PROBS: chunk 0 also stores the row's M and 1 / L for the
// attention-weight finalizing kernel.
template <int D, bool PROBS>
__global__ void __launch_bounds__(256) merge_kernel(KiviGeom g, KiviDev dv, int hq, __half *__restrict__ out,
                                                    DecodePlan plan, DecodeUnits units, int S, int CP) {
    // a programmatic dependent of the decode kernel: its partials are read
    // only once that grid has finished; the next kernel (the weights'
    // finalizing kernel) may start its own set-up
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float s_m[kMaxSlots], s_l[kMaxSlots];
    __shared__ float s_acc[256];
    __shared__ float s_ML[2];
    const int chunks = (D + CP - 1) / CP;
    const int row = blockIdx.x / chunks, chunk = blockIdx.x % chunks;
    const int i = row / hq, h = row % hq;
    const int hg = hq / g.h, j = h / hg, e = h % hg;
    const int QG = plan.qgroups, qg = e / 4;
    const long long HQG = (long long)g.h * QG;
    const long long U = units.total;
    const int C = plan.ctas;
    const int Wi = units.start[i + 1] - units.start[i];
    const long long Pp = HQG * units.start[i] + (long long)(j * QG + qg) * Wi;
    const int np = (int)(cta_of(Pp + Wi - 1, U, C) - cta_of(Pp, U, C)) + 1;
    const float *pp = dv.part + (size_t)row * g.smax * (D + 2);
    for (int y = threadIdx.x; y < np; y += blockDim.x) {
        s_m[y] = __ldcg(pp + (size_t)y * (D + 2));
        s_l[y] = __ldcg(pp + (size_t)y * (D + 2) + 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        float M = -INFINITY;
        for (int y = threadIdx.x; y < np; y += 32) M = fmaxf(M, s_m[y]);
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        if (M != -INFINITY)
            for (int y = threadIdx.x; y < np; y += 32) L = fmaf(ex2f(s_m[y] - M), s_l[y], L);
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (threadIdx.x == 0) {
            s_ML[0] = M;
            s_ML[1] = L > 0.f ? 1.f / L : 0.f;
            if (PROBS && chunk == 0) {
                dv.ml[2 * row] = M;
                dv.ml[2 * row + 1] = s_ML[1];
            }
        }
    }
    __syncthreads();
    const float M = s_ML[0], invL = s_ML[1];
    const int s = threadIdx.x / CP, cl = threadIdx.x % CP;
    const int cc = chunk * CP + cl;
    float a = 0.f;
    if (cc < D && M != -INFINITY) {
        const float *col = pp + 2 + cc;
        int y = s;
        // four partials in flight per step
        for (; y + 3 * S < np; y += 4 * S) {
            const float v0 = __ldcg(col + (size_t)y * (D + 2));
            const float v1 = __ldcg(col + (size_t)(y + S) * (D + 2));
            const float v2 = __ldcg(col + (size_t)(y + 2 * S) * (D + 2));
            const float v3 = __ldcg(col + (size_t)(y + 3 * S) * (D + 2));
            a = fmaf(ex2f(s_m[y] - M), v0, a);
            a = fmaf(ex2f(s_m[y + S] - M), v1, a);
            a = fmaf(ex2f(s_m[y + 2 * S] - M), v2, a);
            a = fmaf(ex2f(s_m[y + 3 * S] - M), v3, a);
        }
        for (; y < np; y += S) a = fmaf(ex2f(s_m[y] - M), __ldcg(col + (size_t)y * (D + 2)), a);
    }
    s_acc[threadIdx.x] = a;
    __syncthreads();
    if (s == 0 && cc < D) {
        for (int k = 1; k < S; ++k) a += s_acc[k * CP + cl];
        out[(size_t)row * D + cc] = __float2half_rn(a * invL);
    }
}

template <int D, bool PROBS>
cudaError_t launch_merge_t(const KiviGeom &g, const KiviDev &dv, int hq, __half *out, const DecodePlan &plan,
                           const DecodeUnits &units, cudaStream_t st) {
    // S partial sums per channel: enough threads that each sums a few
    // partials, at most 256 threads a CTA
    int S = 1;
    while (S < 8 && plan.max_parts > 4 * S) S *= 2;
    const int CP = D * S <= 256 ? D : 256 / S;
    const int chunks = (D + CP - 1) / CP;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(g.b * hq * chunks));
    cfg.blockDim = dim3((unsigned)(CP * S));
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel<D, PROBS>, g, dv, hq, out, plan, units, S, CP);
}

}  // namespace

cudaError_t kivi_launch_merge(const KiviGeom &g, const KiviDev &dv, int hq, __half *out, const DecodePlan &plan,
                              const DecodeUnits &units, bool probs, cudaStream_t st) {
    if (plan.max_parts > kMaxSlots) return cudaErrorInvalidValue;
    switch (g.d) {
    case 64: return probs ? launch_merge_t<64, true>(g, dv, hq, out, plan, units, st)
                          : launch_merge_t<64, false>(g, dv, hq, out, plan, units, st);
    case 128: return probs ? launch_merge_t<128, true>(g, dv, hq, out, plan, units, st)
                           : launch_merge_t<128, false>(g, dv, hq, out, plan, units, st);
    default: return probs ? launch_merge_t<256, true>(g, dv, hq, out, plan, units, st)
                          : launch_merge_t<256, false>(g, dv, hq, out, plan, units, st);
    }
}
