// kivi_decode.cu -- launch planning and dispatch of the decode-attention
// kernels (kivi_decode_impl.cuh, instantiated per head dimension in
// kivi_decode_d{64,128,256}.cu).
//
// The plan splits each (sequence, kv head) token axis into chunks of whole
// 64-token blocks (split-K, one CTA each) so that the grid covers the GPU's
// SMs several times over, and adds the tail CTAs that cover the last blocks
// holding fp16 keys or values (at most R + 64 tokens).
#include <cstdlib>

#include "kivi_internal.cuh"

cudaError_t kivi_launch_decode_d64(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                   const DecodePlan &, cudaStream_t);
cudaError_t kivi_launch_decode_d128(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                    const DecodePlan &, cudaStream_t);
cudaError_t kivi_launch_decode_d256(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                    const DecodePlan &, cudaStream_t);

namespace {
int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    int x = atoi(v);
    return x > 0 ? x : dflt;
}

int stage_bytes(const KiviGeom &g) {
    int ksz = (g.G >= KIVI_KBLK ? 1 : KIVI_KBLK / g.G) * 2 * g.d * 2;
    return g.kc_blk * 4 + ksz + 4 * g.vc_blk * 4 + 4 * g.vsz_blk * 2;
}
}  // namespace

int kivi_min_blocks_per_split() { return 8; }

DecodePlan kivi_plan_decode(const KiviGeom &g, int hq, const int *Tqk, const int *Tqv, int num_sms) {
    DecodePlan p;
    const int hg = hq / g.h;
    p.qgroups = (hg + 3) / 4;
    // the tail spans at most R + 1 fp16 tokens plus 63 of a partly fp16 block
    p.tails = (g.R + KIVI_KBLK + KIVI_TAILBLK - 1) / KIVI_TAILBLK;
    // Two CTAs per SM (the kernel is compiled for <= 128 registers a thread):
    // each CTA gets ~110 KB of shared memory for its warps' rings of stages.
    const int sb = stage_bytes(g);
    const int budget = env_int("KIVI_DECODE_SMEM_KB", 110) * 1024;
    p.warps = env_int("KIVI_DECODE_WARPS", 8);
    if (p.warps > 8) p.warps = 8;
    while (p.warps > 1 && budget / (p.warps * sb) < 2) p.warps /= 2;
    int stages = budget / (p.warps * sb);
    stages = stages > 4 ? 4 : (stages < 1 ? 1 : stages);
    p.stages = env_int("KIVI_DECODE_STAGES", stages);
    while (p.stages > 1 && (size_t)p.warps * p.stages * sb > 220 * 1024) --p.stages;
    const size_t cta_smem = (size_t)p.warps * p.stages * sb + 1024;
    int per_sm = (int)((227 * 1024) / cta_smem);
    per_sm = per_sm > 2 ? 2 : (per_sm < 1 ? 1 : per_sm);
    int nfull = 0;
    for (int i = 0; i < g.b; ++i) {
        int n = (Tqk[i] < Tqv[i] ? Tqk[i] : Tqv[i]) / KIVI_KBLK;
        nfull = n > nfull ? n : nfull;
    }
    const long pairs = (long)g.b * g.h * p.qgroups;
    const int waves = env_int("KIVI_DECODE_WAVES", 2);
    const long slots = (long)num_sms * per_sm * waves;
    int splits = (int)((slots + pairs - 1) / pairs);
    if (splits < 1) splits = 1;
    // blocks per split: a multiple of the warp count (warps get equal shares)
    const int min_bp = env_int("KIVI_DECODE_MIN_BLOCKS", kivi_min_blocks_per_split());
    int bp = nfull > 0 ? (nfull + splits - 1) / splits : 1;
    if (bp < min_bp) bp = min_bp;
    bp = (bp + p.warps - 1) / p.warps * p.warps;
    splits = nfull > 0 ? (nfull + bp - 1) / bp : 0;
    if (splits + p.tails > g.smax) {
        bp = (nfull + (g.smax - p.tails) - 1) / (g.smax - p.tails);
        splits = (nfull + bp - 1) / bp;
    }
    p.splits = splits;
    p.blocks_per = bp;
    p.launches = 1;
    return p;
}

cudaError_t kivi_launch_decode(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                               __half *out, const DecodePlan &plan, cudaStream_t st,
                               cudaEvent_t ev0, cudaEvent_t ev1) {
    if (ev0) cudaEventRecord(ev0, st);
    cudaError_t e;
    switch (g.d) {
    case 64: e = kivi_launch_decode_d64(g, dv, q, hq, out, plan, st); break;
    case 128: e = kivi_launch_decode_d128(g, dv, q, hq, out, plan, st); break;
    default: e = kivi_launch_decode_d256(g, dv, q, hq, out, plan, st); break;
    }
    if (ev1) cudaEventRecord(ev1, st);
    return e;
}
