// kivi_decode.cu -- split-K decode attention over the quantized cache.
//
// Method: "Literature audit -- Group 2", section 1 KIVI, core algorithm
// item 5: scores q.k / sqrt(d) over the quantized keys followed by the fp16
// keys, one softmax over both, weights applied to the quantized values
// followed by the fp16 values.  Query head i reads kv head i / (h_q / h_kv).
//
// Each CTA owns one (sequence, kv head, token range) and all query heads of
// that kv head, so every packed K/V word is read from HBM once.  It keeps an
// online softmax (running max m, running sum l, unnormalized accumulator)
// per query head in base 2 (scores pre-multiplied by log2(e) / sqrt(d)),
// and writes (m, l, acc[d]) as a partial; a second kernel merges the
// partials of each (sequence, query head) with log-sum-exp weights.
#include "kivi_internal.cuh"

namespace {

constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Dequantized key channel c of token tau (quantized or fp16 residual).
__device__ __forceinline__ float key_at(const KiviGeom &g, const uint32_t *kc, const __half *ksz,
                                        const __half *kf, int Tqk, int c, int tau) {
    if (tau < Tqk) {
        int sh;
        size_t w = kc_locate(g, c, tau, &sh);
        uint32_t code = (kc[w] >> sh) & ((1u << g.kbits) - 1u);
        int grp = tau / g.G;
        return (float)code * __half2float(ksz[ksz_locate(g, grp, c, 0)]) +
               __half2float(ksz[ksz_locate(g, grp, c, 1)]);
    }
    return __half2float(kf[(size_t)(tau % g.R) * g.d + c]);
}

__device__ __forceinline__ float value_at(const KiviGeom &g, const uint32_t *vc, const __half *vsz,
                                          const __half *vf, int Tqv, int c, int tau) {
    if (tau < Tqv) {
        int sh;
        size_t w = vc_locate(g, c, tau, &sh);
        uint32_t code = (vc[w] >> sh) & ((1u << g.vbits) - 1u);
        int gi = c / g.G;
        return (float)code * __half2float(vsz[vsz_locate(g, tau, gi, 0)]) +
               __half2float(vsz[vsz_locate(g, tau, gi, 1)]);
    }
    return __half2float(vf[(size_t)(tau % (g.R + 1)) * g.d + c]);
}

// Generic CUDA-core path: one warp per token, lane owns channels lane + 32k.
template <int CPL>   // channels per lane = d / 32
__global__ void __launch_bounds__(kWarps * 32) decode_generic_kernel(KiviGeom g, KiviDev dv,
                                                                    const __half *__restrict__ q,
                                                                    int hq, DecodePlan plan) {
    const int s = blockIdx.x, j = blockIdx.y, i = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hg = hq / g.h;
    const int d = g.d;
    const int T = dv.T[i], Tqk = dv.Tqk[i], Tqv = dv.Tqv[i];
    const int span = plan.blocks_per * KIVI_KBLK;
    const int t0 = s * span, t1 = min(T, t0 + span);
    const float qscale = kLog2e * rsqrtf((float)d);

    float qr[KIVI_MAX_QPERKV][CPL];
    for (int e = 0; e < KIVI_MAX_QPERKV; ++e)
#pragma unroll
        for (int k = 0; k < CPL; ++k)
            qr[e][k] = e < hg ? __half2float(q[((size_t)i * hq + j * hg + e) * d + lane + 32 * k]) * qscale
                              : 0.f;
    float m[KIVI_MAX_QPERKV], l[KIVI_MAX_QPERKV], acc[KIVI_MAX_QPERKV][CPL];
    for (int e = 0; e < KIVI_MAX_QPERKV; ++e) {
        m[e] = -INFINITY;
        l[e] = 0.f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) acc[e][k] = 0.f;
    }

    const uint32_t *kc = dv.Kc + kc_slice(g, i, j);
    const __half *ksz = dv.Ksz + ksz_slice(g, i, j);
    const __half *kf = dv.Kf + kf_slice(g, i, j);
    const uint32_t *vc = dv.Vc + vc_slice(g, i, j);
    const __half *vsz = dv.Vsz + vsz_slice(g, i, j);
    const __half *vf = dv.Vf + vf_slice(g, i, j);

    for (int tau = t0 + warp; tau < t1; tau += kWarps) {
        float kv[CPL], vv[CPL];
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
            kv[k] = key_at(g, kc, ksz, kf, Tqk, lane + 32 * k, tau);
            vv[k] = value_at(g, vc, vsz, vf, Tqv, lane + 32 * k, tau);
        }
        for (int e = 0; e < hg; ++e) {
            float dot = 0.f;
#pragma unroll
            for (int k = 0; k < CPL; ++k) dot = fmaf(qr[e][k], kv[k], dot);
            float sc = warp_sum(dot);
            float mn = fmaxf(m[e], sc);
            float corr = exp2f(m[e] - mn);
            float p = exp2f(sc - mn);
            l[e] = l[e] * corr + p;
#pragma unroll
            for (int k = 0; k < CPL; ++k) acc[e][k] = fmaf(p, vv[k], acc[e][k] * corr);
            m[e] = mn;
        }
    }

    // combine the warps of this CTA
    __shared__ float sm[kWarps][KIVI_MAX_QPERKV], sl[kWarps][KIVI_MAX_QPERKV];
    extern __shared__ float sacc[];   // [kWarps][hg][d]
    if (lane == 0)
        for (int e = 0; e < hg; ++e) {
            sm[warp][e] = m[e];
            sl[warp][e] = l[e];
        }
    for (int e = 0; e < hg; ++e)
#pragma unroll
        for (int k = 0; k < CPL; ++k) sacc[((size_t)warp * hg + e) * d + lane + 32 * k] = acc[e][k];
    __syncthreads();
    for (int x = threadIdx.x; x < hg * (d + 2); x += blockDim.x) {
        int e = x / (d + 2), c = x % (d + 2);
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm[w][e]);
        float val = 0.f;
        if (c == 0) {
            val = M;
        } else if (M != -INFINITY) {
            for (int w = 0; w < kWarps; ++w) {
                float f = exp2f(sm[w][e] - M);
                val += f * (c == 1 ? sl[w][e] : sacc[((size_t)w * hg + e) * d + (c - 2)]);
            }
        }
        dv.part[(((size_t)i * hq + j * hg + e) * g.smax + s) * (d + 2) + c] = val;
    }
}

// Merge the splits of one (sequence, query head): log-sum-exp weights.
__global__ void merge_kernel(KiviGeom g, KiviDev dv, int hq, int splits, __half *__restrict__ out) {
    const int qh = blockIdx.x, i = blockIdx.y;
    const int d = g.d;
    const float *pp = dv.part + ((size_t)i * hq + qh) * g.smax * (d + 2);
    __shared__ float sM, sL;
    if (threadIdx.x == 0) {
        float M = -INFINITY;
        for (int s = 0; s < splits; ++s) M = fmaxf(M, pp[(size_t)s * (d + 2)]);
        float L = 0.f;
        if (M != -INFINITY)
            for (int s = 0; s < splits; ++s) L += exp2f(pp[(size_t)s * (d + 2)] - M) * pp[(size_t)s * (d + 2) + 1];
        sM = M;
        sL = L;
    }
    __syncthreads();
    const float M = sM, L = sL;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
        float a = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < splits; ++s) {
                const float *p = pp + (size_t)s * (d + 2);
                a += exp2f(p[0] - M) * p[2 + c];
            }
            a = a / L;
        }
        out[((size_t)i * hq + qh) * d + c] = __float2half_rn(a);
    }
}

}  // namespace

DecodePlan kivi_plan_decode(const KiviGeom &g, int hq, int maxT, int num_sms) {
    (void)hq;
    (void)num_sms;
    DecodePlan p;
    int nblk = (maxT + KIVI_KBLK - 1) / KIVI_KBLK;
    if (nblk < 1) nblk = 1;
    p.blocks_per = 16;
    p.splits = (nblk + p.blocks_per - 1) / p.blocks_per;
    if (p.splits > g.smax) {
        p.blocks_per = (nblk + g.smax - 1) / g.smax;
        p.splits = (nblk + p.blocks_per - 1) / p.blocks_per;
    }
    p.qgroups = 1;
    p.launches = 2;
    return p;
}

cudaError_t kivi_launch_decode(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                               __half *out, const DecodePlan &plan, cudaStream_t st,
                               cudaEvent_t ev0, cudaEvent_t ev1) {
    const int hg = hq / g.h;
    dim3 grid(plan.splits, g.h, g.b);
    size_t sm = (size_t)kWarps * hg * g.d * sizeof(float);
    if (ev0) cudaEventRecord(ev0, st);
    switch (g.d) {
    case 64:
        decode_generic_kernel<2><<<grid, kWarps * 32, sm, st>>>(g, dv, q, hq, plan);
        break;
    case 128:
        decode_generic_kernel<4><<<grid, kWarps * 32, sm, st>>>(g, dv, q, hq, plan);
        break;
    default:
        cudaFuncSetAttribute(decode_generic_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm);
        decode_generic_kernel<8><<<grid, kWarps * 32, sm, st>>>(g, dv, q, hq, plan);
        break;
    }
    merge_kernel<<<dim3(hq, g.b), 128, 0, st>>>(g, dv, hq, plan.splits, out);
    if (ev1) cudaEventRecord(ev1, st);
    return cudaGetLastError();
}
