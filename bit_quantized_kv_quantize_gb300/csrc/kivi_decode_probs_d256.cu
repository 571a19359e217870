// kivi_decode_probs_d256.cu -- decode-attention kernels for head dimension 256
// that also write each token's score for the attention-weight output.
#include "kivi_decode_impl.cuh"

cudaError_t kivi_launch_decode_probs_d256(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                                         __half *out, const DecodePlan &plan, const DecodeUnits &units,
                                         const ProbsOut &po, cudaStream_t st) {
    return launch_d<256, true>(g, dv, q, hq, out, plan, units, po, st);
}
