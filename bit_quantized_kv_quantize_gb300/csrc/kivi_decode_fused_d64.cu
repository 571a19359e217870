// kivi_decode_fused_d64.cu -- decode-attention kernels for head dimension 64
// that also append the step's token (kivi_append_decode on steps whose
// appends need no key-window flush).
#include "kivi_decode_impl.cuh"

cudaError_t kivi_launch_decode_fused_d64(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                                   __half *out, const DecodePlan &plan, const DecodeUnits &units,
                                   const FusedStep &fs, cudaStream_t st) {
    return launch_d<64, false, true>(g, dv, q, hq, out, plan, units, ProbsOut{nullptr, nullptr, 0}, st, fs);
}
