// kivi_decode.cu -- launch planning and dispatch of the decode-attention
// kernel (kivi_decode_impl.cuh, instantiated per head dimension in
// kivi_decode_d{64,128,256}.cu, and with the score output for the
// attention weights in kivi_decode_probs_d{64,128,256}.cu; kivi_probs.cu
// turns those scores into weights).
//
// The kernel is persistent: a fixed grid of CTAs (two per SM) splits the
// work units of all (sequence, kv head, head group) pairs evenly, so every
// CTA streams about the same number of bytes whatever the batch and context
// lengths (no partial last wave).  A unit is one 64-token block; blocks that
// hold fp16 window tokens (the last few of each sequence) are staged by the
// whole CTA with one round trip each and count MW units.
#include <cstdlib>

#include "kivi_internal.cuh"

cudaError_t kivi_launch_decode_d64(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                   const DecodePlan &, const DecodeUnits &, cudaStream_t);
cudaError_t kivi_launch_decode_d128(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                    const DecodePlan &, const DecodeUnits &, cudaStream_t);
cudaError_t kivi_launch_decode_d256(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                    const DecodePlan &, const DecodeUnits &, cudaStream_t);
cudaError_t kivi_launch_decode_fused_d64(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                         const DecodePlan &, const DecodeUnits &, const FusedStep &, cudaStream_t);
cudaError_t kivi_launch_decode_fused_d128(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                          const DecodePlan &, const DecodeUnits &, const FusedStep &, cudaStream_t);
cudaError_t kivi_launch_decode_fused_d256(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                          const DecodePlan &, const DecodeUnits &, const FusedStep &, cudaStream_t);
cudaError_t kivi_launch_decode_probs_d64(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                         const DecodePlan &, const DecodeUnits &, const ProbsOut &,
                                         cudaStream_t);
cudaError_t kivi_launch_decode_probs_d128(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                          const DecodePlan &, const DecodeUnits &, const ProbsOut &,
                                          cudaStream_t);
cudaError_t kivi_launch_decode_probs_d256(const KiviGeom &, const KiviDev &, const __half *, int, __half *,
                                          const DecodePlan &, const DecodeUnits &, const ProbsOut &,
                                          cudaStream_t);

namespace {
int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    int x = atoi(v);
    return x > 0 ? x : dflt;
}


long long cta_of(long long u, long long U, int C) { return ((u + 1) * C - 1) / U; }

constexpr int kCtasPerSm = 2;   // the kernel is compiled for <= 128 registers a thread

}  // namespace

int kivi_partial_slots(int b, int h, int num_sms) {
    const int cmax = num_sms * kCtasPerSm;
    return (2 * cmax + b * h - 1) / (b * h) + 4;
}

DecodePlan kivi_plan_decode(const KiviGeom &g, int hq, const int *T, const int *Tqk, const int *Tqv,
                            int num_sms, DecodeUnits *units, bool fused) {
    DecodePlan p;
    const int hg = hq / g.h;
    p.qgroups = (hg + 3) / 4;
    p.launches = 1;
    // shared memory: two CTAs per SM, ~110 KB each for the warps' rings of at
    // least two stages
    const int sb = g.rec_bytes;   // a stage holds one block record
    const int budget = env_int("KIVI_DECODE_SMEM_KB", 110) * 1024;
    p.warps = env_int("KIVI_DECODE_WARPS", 8);
    if (p.warps > 8) p.warps = 8;
    while (p.warps > 1 && budget / (p.warps * sb) < 2) --p.warps;
    int stages = budget / (p.warps * sb);
    stages = stages > 4 ? 4 : (stages < 2 ? 2 : stages);
    p.stages = env_int("KIVI_DECODE_STAGES", stages);
    while (p.stages > 2 && (size_t)p.warps * p.stages * sb > 220 * 1024) --p.stages;

    // units per pair of each sequence: a lead of units standing for the
    // fixed cost of a segment (its set-up and its merge: a CTA whose range
    // takes in a pair's start gets that many fewer blocks), one per fully
    // quantized block, MW per block holding window tokens
    const int MW = env_int("KIVI_DECODE_MIXED_WEIGHT", 12);
    const char *le = getenv("KIVI_DECODE_LEAD");
    units->mixed_weight = MW;
    units->lead = le && *le ? (atoi(le) > 0 ? atoi(le) : 0) : 3;
    // A launch that also appends: the pair's append falls to the CTA
    // holding the pair's last blocks, which the partition charges with a
    // tail of units after them (no blocks), scaled to the blocks a CTA
    // takes (about 1 unit per 25, at most 4: ~2 us of a 32k CTA's ~60).
    int tail = 0;
    if (fused) {
        long long base = 0;
        for (int i = 0; i < g.b; ++i) {
            const int nf = (Tqk[i] < Tqv[i] ? Tqk[i] : Tqv[i]) / KIVI_KBLK;
            const int nb = (T[i] + KIVI_KBLK - 1) / KIVI_KBLK;
            base += (long long)g.h * p.qgroups * (units->lead + nf + MW * (nb - nf));
        }
        const long long per_cta = base / ((long long)num_sms * kCtasPerSm);
        tail = (int)(per_cta / 25 > 4 ? 4 : per_cta / 25);
        const char *ta = getenv("KIVI_DECODE_FUSED_TAIL");
        if (ta && *ta) tail = atoi(ta) > 0 ? atoi(ta) : 0;
    }
    units->start[0] = 0;
    for (int i = 0; i < g.b; ++i) {
        const int nf = (Tqk[i] < Tqv[i] ? Tqk[i] : Tqv[i]) / KIVI_KBLK;
        const int nb = (T[i] + KIVI_KBLK - 1) / KIVI_KBLK;
        int w = units->lead + nf + MW * (nb - nf) + tail;
        if (w < 1) w = 1;   // an empty sequence still gets its (zero) output written
        units->full[i] = nf;
        units->start[i + 1] = units->start[i] + w;
    }
    const long long HQG = (long long)g.h * p.qgroups;
    units->total = HQG * units->start[g.b];
    const long long U = units->total;
    int C = env_int("KIVI_DECODE_CTAS", num_sms * kCtasPerSm);
    if ((long long)C > U) C = (int)U;
    // every pair's partials must fit the cache's slots
    for (;;) {
        int worst = 1;
        for (int i = 0; i < g.b; ++i) {
            const int w = units->start[i + 1] - units->start[i];
            for (long long jq = 0; jq < HQG; ++jq) {
                const long long P = HQG * units->start[i] + jq * w;
                const int np = (int)(cta_of(P + w - 1, U, C) - cta_of(P, U, C) + 1);
                worst = np > worst ? np : worst;
            }
        }
        if (worst <= g.smax || C == 1) {
            p.max_parts = worst;
            break;
        }
        C = (int)((long long)C * g.smax / (worst + 1));
        if (C < 1) C = 1;
    }
    p.ctas = C;
    return p;
}

cudaError_t kivi_launch_decode(const KiviGeom &g, const KiviDev &dv, const __half *q, int hq,
                               __half *out, const DecodePlan &plan, const DecodeUnits &units,
                               cudaStream_t st, cudaEvent_t ev0, cudaEvent_t ev1, const ProbsOut *po,
                               int maxT, const FusedStep *fs) {
    if (po && fs) return cudaErrorInvalidValue;
    if (ev0) cudaEventRecord(ev0, st);
    cudaError_t e;
    if (fs) {
        switch (g.d) {
        case 64: e = kivi_launch_decode_fused_d64(g, dv, q, hq, out, plan, units, *fs, st); break;
        case 128: e = kivi_launch_decode_fused_d128(g, dv, q, hq, out, plan, units, *fs, st); break;
        default: e = kivi_launch_decode_fused_d256(g, dv, q, hq, out, plan, units, *fs, st); break;
        }
    } else if (po) {
        switch (g.d) {
        case 64: e = kivi_launch_decode_probs_d64(g, dv, q, hq, out, plan, units, *po, st); break;
        case 128: e = kivi_launch_decode_probs_d128(g, dv, q, hq, out, plan, units, *po, st); break;
        default: e = kivi_launch_decode_probs_d256(g, dv, q, hq, out, plan, units, *po, st); break;
        }
    } else {
        switch (g.d) {
        case 64: e = kivi_launch_decode_d64(g, dv, q, hq, out, plan, units, st); break;
        case 128: e = kivi_launch_decode_d128(g, dv, q, hq, out, plan, units, st); break;
        default: e = kivi_launch_decode_d256(g, dv, q, hq, out, plan, units, st); break;
        }
    }
    if (ev1) cudaEventRecord(ev1, st);
    if (e == cudaSuccess && po && maxT > 0) e = kivi_launch_probs_finalize(g, dv, hq, *po, maxT, st);
    return e;
}
