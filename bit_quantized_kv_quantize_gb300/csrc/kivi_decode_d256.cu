// kivi_decode_d256.cu -- decode-attention kernels for head dimension 256
// (one translation unit per head dimension so the variants build in parallel).
#include "kivi_decode_impl.cuh"

cudaError_t kivi_launch_decode_d256(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                                   __half *out, const DecodePlan &plan, const DecodeUnits &units,
                                   cudaStream_t st) {
    return launch_d<256, false>(g, dv, q, hq, out, plan, units, ProbsOut{nullptr, nullptr, 0}, st);
}
