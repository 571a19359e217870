// kivi_probs.cu -- the second half of the attention-weight output: the
// decode kernel's weights variant leaves, for every (sequence i, query head)
// row, the T_i raw scores s (log2 units) in the weights buffer and the row's
// softmax max M and 1 / sum in the cache's scratch; here each score becomes
// its weight 2^(s - M) / sum, and the optional mass buffer accumulates it.
#include <cstdint>

#include "kivi_internal.cuh"

namespace {

// Tokens of one row a CTA covers.
constexpr int kChunk = 4096;

__device__ __forceinline__ float weight_of(float s, float M, float inv) { return exp2f(s - M) * inv; }

__device__ __forceinline__ void finalize_one(float *p, float *mass, int t, float M, float inv) {
    const float w = weight_of(p[t], M, inv);
    p[t] = w;
    if (mass) mass[t] += w;
}

// CTA x covers chunk x % chunks of row x / chunks.  VEC (both buffers
// 16-byte aligned): the tokens before the row's first 16-byte boundary go
// one at a time, the rest four at a time.
template <bool VEC>
__global__ void __launch_bounds__(256) probs_finalize_kernel(const int *__restrict__ T,
                                                             const float *__restrict__ ml, int hq,
                                                             int chunks, ProbsOut po) {
    // a programmatic dependent of the decode kernel: wait for it to finish
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x / chunks, ch = blockIdx.x % chunks;
    const int t0 = ch * kChunk, t1 = min(T[row / hq], t0 + kChunk);
    if (t0 >= t1) return;
    const float M = ml[2 * row], inv = ml[2 * row + 1];
    const size_t base = (size_t)row * po.ld;
    float *p = po.p + base;
    float *mass = po.mass ? po.mass + base : nullptr;
    if constexpr (VEC) {
        // first token at or after t0 whose address is 16-byte aligned
        const int ta = min(t1, t0 + (int)((4 - (base + t0) % 4) % 4));
        if ((int)threadIdx.x < ta - t0) finalize_one(p, mass, t0 + threadIdx.x, M, inv);
        const int n4 = (t1 - ta) >> 2;
        float4 *p4 = reinterpret_cast<float4 *>(p + ta);
        float4 *m4 = mass ? reinterpret_cast<float4 *>(mass + ta) : nullptr;
        for (int k = threadIdx.x; k < n4; k += blockDim.x) {
            float4 w = p4[k];
            w.x = weight_of(w.x, M, inv);
            w.y = weight_of(w.y, M, inv);
            w.z = weight_of(w.z, M, inv);
            w.w = weight_of(w.w, M, inv);
            p4[k] = w;
            if (m4) {
                float4 a = m4[k];
                a.x += w.x;
                a.y += w.y;
                a.z += w.z;
                a.w += w.w;
                m4[k] = a;
            }
        }
        const int tt = ta + 4 * n4 + threadIdx.x;
        if (tt < t1) finalize_one(p, mass, tt, M, inv);   // < 4 tokens remain
    } else {
        for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) finalize_one(p, mass, t, M, inv);
    }
}

}  // namespace

cudaError_t kivi_launch_probs_finalize(const KiviGeom &g, const KiviDev &dv, int hq, const ProbsOut &po,
                                       int maxT, cudaStream_t st) {
    const int chunks = (maxT + kChunk - 1) / kChunk;
    const unsigned grid = (unsigned)(g.b * hq) * chunks;
    const bool vec = ((uintptr_t)po.p & 15u) == 0 && ((uintptr_t)po.mass & 15u) == 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec) return cudaLaunchKernelEx(&cfg, probs_finalize_kernel<true>, (const int *)dv.T, (const float *)dv.ml, hq,
                                       chunks, po);
    return cudaLaunchKernelEx(&cfg, probs_finalize_kernel<false>, (const int *)dv.T, (const float *)dv.ml, hq, chunks,
                              po);
}
