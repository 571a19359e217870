// kivi_api.cu -- host side of libkivi: the C ABI declared in include/kivi.h.
//
// Owns the cache's device memory, keeps a host mirror of the per-sequence
// counters (T, Tqk, Tqv) that evolves by the same rule as the device copy
// (KIVI core algorithm item 4), validates every argument before touching
// anything, and launches the kernels of kivi_pack.cu / kivi_decode.cu on the
// caller's stream.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <set>
#include <vector>

#include "../../include/kivi.h"
#include "kivi_internal.cuh"

namespace {

constexpr uint32_t kMagic = 0x4b495649u;   // "KIVI"
constexpr int kMaxProfile = 4096;

thread_local char g_err[512] = "";

void set_err(const char *fmt, const char *a = "", long v = 0) {
    snprintf(g_err, sizeof g_err, fmt, a, v);
}

std::mutex g_live_mu;
std::set<void *> g_live;

}  // namespace

void kivi_set_last_error(const char *msg) { snprintf(g_err, sizeof g_err, "%s", msg ? msg : ""); }

struct kivi_cache {
    uint32_t magic;
    bool poisoned;
    int max_tokens;
    int device;
    int num_sms;
    KiviGeom g;
    KiviDev dv;
    // Two device counter sets [2][3][b] (T, Tqk, Tqv): dv points at set
    // `parity`; an append reads the host mirror and writes the other set,
    // which then becomes current (no CTA of the append waits for another).
    int *cnt;
    int parity;
    std::vector<int> T, Tqk, Tqv;   // host mirror
    DecodePlan last_plan;
    bool profiling;
    std::vector<cudaEvent_t> ev;   // pairs
    int nprof;
};

namespace {

kivi_status fail_cuda(kivi_cache *c, cudaError_t e, const char *where) {
    if (c) c->poisoned = true;
    snprintf(g_err, sizeof g_err, "%s: %s", where, cudaGetErrorString(e));
    return KIVI_ERR_CUDA;
}

kivi_status check_handle(kivi_cache_t c) {
    if (!c) {
        set_err("null cache handle");
        return KIVI_ERR_INVALID_ARG;
    }
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        if (!g_live.count((void *)c)) {
            set_err("unknown or destroyed cache handle");
            return KIVI_ERR_INVALID_ARG;
        }
    }
    if (c->magic != kMagic) {
        set_err("corrupt cache handle");
        return KIVI_ERR_INVALID_ARG;
    }
    if (c->poisoned) {
        set_err("cache poisoned by an earlier CUDA error");
        return KIVI_ERR_STATE;
    }
    return KIVI_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

// The cache shapes the library supports (kivi_cache_create's rules); also
// used by the allocation-free decode (kivi_noalloc.cu).
int kivi_check_shape(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R, int max_tokens) {
    if (b < 1 || h_kv < 1 || d < 1 || G < 1 || R < 1 || max_tokens < 1) {
        set_err("sizes must be positive");
        return KIVI_ERR_INVALID_ARG;
    }
    if (b > KIVI_MAX_BATCH) {
        set_err("b above %s%ld", "", KIVI_MAX_BATCH);
        return KIVI_ERR_UNSUPPORTED;
    }
    if ((k_bits != 2 && k_bits != 4) || (v_bits != 2 && v_bits != 4)) {
        set_err("bits must be 2 or 4");
        return KIVI_ERR_UNSUPPORTED;
    }
    if (G != 16 && G != 32 && G != 64 && G != 128) {
        set_err("G must be 16, 32, 64 or 128");
        return KIVI_ERR_UNSUPPORTED;
    }
    if (d != 64 && d != 128 && d != 256) {
        set_err("d must be 64, 128 or 256");
        return KIVI_ERR_UNSUPPORTED;
    }
    if (d % G != 0 || R % G != 0 || R > 4096) {
        set_err("need d %% G == 0, R %% G == 0 and R <= 4096");
        return KIVI_ERR_UNSUPPORTED;
    }
    const int q = G > KIVI_KBLK ? G : KIVI_KBLK;
    if ((long)max_tokens + q > (1L << 30)) {
        set_err("max_tokens too large");
        return KIVI_ERR_UNSUPPORTED;
    }
    return KIVI_OK;
}

namespace {

kivi_status check_shape(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R, int max_tokens) {
    return (kivi_status)kivi_check_shape(b, h_kv, d, k_bits, v_bits, G, R, max_tokens);
}

void free_dev(kivi_cache *c) {
    KiviDev &d = c->dv;
    void *ps[] = {d.blk, d.Kf, d.Vf, c->cnt, d.status, d.part, d.merge_ticket, d.ml};
    for (void *p : ps)
        if (p) cudaFree(p);
    memset(&d, 0, sizeof d);
    c->cnt = nullptr;
}

void point_counters(kivi_cache *c) {
    const int b = c->g.b;
    int *set = c->cnt + (size_t)c->parity * 3 * b;
    c->dv.T = set;
    c->dv.Tqk = set + b;
    c->dv.Tqv = set + 2 * b;
}

kivi_status check_decode_args(kivi_cache *c, const void *q, int h_q, const void *out) {
    if (!q || !out) {
        set_err("q or out is null");
        return KIVI_ERR_INVALID_ARG;
    }
    if (h_q < 1 || h_q % c->g.h != 0) {
        set_err("h_q must be a positive multiple of h_kv");
        return KIVI_ERR_INVALID_ARG;
    }
    if (h_q / c->g.h > KIVI_MAX_QPERKV) {
        set_err("h_q / h_kv above 8");
        return KIVI_ERR_UNSUPPORTED;
    }
    if (!aligned16(q) || !aligned16(out)) {
        set_err("q and out must be 16-byte aligned");
        return KIVI_ERR_INVALID_ARG;
    }
    return KIVI_OK;
}

kivi_status check_append_args(kivi_cache *c, const void *k, const void *v) {
    if (!k || !v) {
        set_err("k or v is null");
        return KIVI_ERR_INVALID_ARG;
    }
    if (!aligned16(k) || !aligned16(v)) {
        set_err("k and v must be 16-byte aligned");
        return KIVI_ERR_INVALID_ARG;
    }
    for (int i = 0; i < c->g.b; ++i)
        if (c->T[i] + 1 > c->max_tokens) {
            set_err("sequence %s%ld is full", "", i);
            return KIVI_ERR_CAPACITY;
        }
    return KIVI_OK;
}

// host mirror of one append (item 4's lazy maintenance, then the token)
void advance_mirror(kivi_cache *c) {
    const int R = c->g.R;
    for (int i = 0; i < c->g.b; ++i) {
        if (c->T[i] - c->Tqk[i] == R) c->Tqk[i] += R;
        if (c->T[i] - c->Tqv[i] == R + 1) c->Tqv[i] += 1;
        c->T[i] += 1;
    }
}

// Launch the append kernel from the host mirror, then make the counter set
// it writes current and advance the mirror.
kivi_status launch_append(kivi_cache *c, const void *k, const void *v, kivi_stream_t stream,
                          const char *what) {
    const int b = c->g.b;
    AppendCounters ac;   // entries past b are never read
    memcpy(ac.T, c->T.data(), (size_t)b * sizeof(int));
    memcpy(ac.Tqk, c->Tqk.data(), (size_t)b * sizeof(int));
    memcpy(ac.Tqv, c->Tqv.data(), (size_t)b * sizeof(int));
    append_order(ac, b, c->g.R);
    int *nxt = c->cnt + (size_t)(1 - c->parity) * 3 * b;
    cudaError_t e = kivi_launch_append(c->g, c->dv, (const __half *)k, (const __half *)v, ac, nxt,
                                       (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(c, e, what);
    c->parity ^= 1;
    point_counters(c);
    advance_mirror(c);
    return KIVI_OK;
}

// Plan and launch the decode kernel; units come from (T, Tqk, Tqv).
kivi_status launch_decode(kivi_cache *c, const void *q, int h_q, void *out, kivi_stream_t stream,
                          const int *T, const int *Tqk, const int *Tqv, const char *what,
                          const ProbsOut *po = nullptr, const FusedStep *fs = nullptr) {
    DecodeUnits units;
    DecodePlan plan = kivi_plan_decode(c->g, h_q, T, Tqk, Tqv, c->num_sms, &units, fs != nullptr);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (c->profiling && c->nprof < kMaxProfile) {
        if ((int)c->ev.size() < 2 * (c->nprof + 1)) {
            cudaEvent_t a, b;
            if (cudaEventCreate(&a) == cudaSuccess && cudaEventCreate(&b) == cudaSuccess) {
                c->ev.push_back(a);
                c->ev.push_back(b);
            }
        }
        if ((int)c->ev.size() >= 2 * (c->nprof + 1)) {
            e0 = c->ev[2 * c->nprof];
            e1 = c->ev[2 * c->nprof + 1];
            c->nprof++;
        }
    }
    int maxT = 0;
    for (int i = 0; i < c->g.b; ++i) maxT = T[i] > maxT ? T[i] : maxT;
    cudaError_t e = kivi_launch_decode(c->g, c->dv, (const __half *)q, h_q, (__half *)out, plan, units,
                                       (cudaStream_t)stream, e0, e1, po, maxT, fs);
    if (e != cudaSuccess) return fail_cuda(c, e, what);
    c->last_plan = plan;
    return KIVI_OK;
}

// Whether kivi_append_decode appends inside the decode launch.  The fused
// kernel relies on one head group per kv head (h_q / h_kv <= 4: every
// window block has a single reader CTA), and it pays only while the
// (sequence, kv head) pairs do not outnumber the persistent CTAs: each
// pair's append is a short serial task on one CTA, where the append kernel
// runs them all at once (measured on GB300: one launch saves 2-5 us per
// step with 8-64 pairs, and costs 5-10 us with 512).  KIVI_FUSED_STEP=0
// keeps the two launches, =1 forces the fused one where it is possible.
bool fused_step(const kivi_cache *c, int h_q) {
    if (h_q / c->g.h > 4) return false;
    const char *e = getenv("KIVI_FUSED_STEP");
    if (e && e[0] == '0' && e[1] == 0) return false;
    if (e && e[0] == '1' && e[1] == 0) return true;
    return (long)c->g.b * c->g.h <= 2L * c->num_sms;
}

// One step as one launch: the decode kernel appends every sequence whose
// key window is not full (item 4: the new token and at most one popped
// value token); sequences that flush their key window now are appended
// first by the append kernel, restricted to them (a second launch on those
// steps only).  The units count an appended sequence's value queue before
// its pop.  Both kernels write the counters after the append into the
// other set, which then becomes current.
kivi_status launch_fused_step(kivi_cache *c, const void *k, const void *v, const void *q, int h_q, void *out,
                              kivi_stream_t stream) {
    const int b = c->g.b, R = c->g.R;
    std::vector<int> Tp(b), Tqkp(b), Tqvp(b);
    bool any_flush = false;
    for (int i = 0; i < b; ++i) {
        const bool flush = c->T[i] - c->Tqk[i] == R, pop = c->T[i] - c->Tqv[i] == R + 1;
        Tp[i] = c->T[i] + 1;
        Tqkp[i] = c->Tqk[i] + (flush ? R : 0);
        Tqvp[i] = c->Tqv[i] + (flush && pop ? 1 : 0);
        any_flush |= flush;
    }
    int *nxt = c->cnt + (size_t)(1 - c->parity) * 3 * b;
    if (any_flush) {
        AppendCounters ac;   // entries past b are never read
        memcpy(ac.T, c->T.data(), (size_t)b * sizeof(int));
        memcpy(ac.Tqk, c->Tqk.data(), (size_t)b * sizeof(int));
        memcpy(ac.Tqv, c->Tqv.data(), (size_t)b * sizeof(int));
        append_order(ac, b, c->g.R);
        cudaError_t e = kivi_launch_append(c->g, c->dv, (const __half *)k, (const __half *)v, ac, nxt,
                                           (cudaStream_t)stream, true);
        if (e != cudaSuccess) return fail_cuda(c, e, "append_decode");
    }
    const FusedStep fs{(const __half *)k, (const __half *)v, nxt};
    kivi_status s = launch_decode(c, q, h_q, out, stream, Tp.data(), Tqkp.data(), Tqvp.data(), "append_decode",
                                  nullptr, &fs);
    if (s != KIVI_OK) return s;
    c->last_plan.launches += any_flush ? 1 : 0;
    c->parity ^= 1;
    point_counters(c);
    advance_mirror(c);
    return KIVI_OK;
}


}  // namespace

extern "C" {

int kivi_abi_version(void) { return KIVI_ABI_VERSION; }

const char *kivi_last_error(void) { return g_err; }

const char *kivi_status_str(kivi_status s) {
    switch (s) {
    case KIVI_OK: return "ok";
    case KIVI_ERR_INVALID_ARG: return "invalid argument";
    case KIVI_ERR_UNSUPPORTED: return "unsupported shape or bit width";
    case KIVI_ERR_CAPACITY: return "capacity exceeded";
    case KIVI_ERR_STATE: return "cache poisoned by an earlier CUDA error";
    case KIVI_ERR_CUDA: return "CUDA error";
    case KIVI_ERR_OOM: return "out of memory";
    }
    return "unknown status";
}

kivi_status kivi_cache_create(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R,
                              int max_tokens, kivi_cache_t *out) {
    g_err[0] = 0;
    if (!out) {
        set_err("out is null");
        return KIVI_ERR_INVALID_ARG;
    }
    *out = nullptr;
    kivi_status sc = check_shape(b, h_kv, d, k_bits, v_bits, G, R, max_tokens);
    if (sc != KIVI_OK) return sc;
    kivi_cache *c = new (std::nothrow) kivi_cache();
    if (!c) {
        set_err("host allocation failed");
        return KIVI_ERR_OOM;
    }
    c->magic = kMagic;
    c->poisoned = false;
    c->max_tokens = max_tokens;
    c->profiling = false;
    c->nprof = 0;
    memset(&c->last_plan, 0, sizeof c->last_plan);
    KiviGeom &g = c->g;
    g.b = b; g.h = h_kv; g.d = d; g.kbits = k_bits; g.vbits = v_bits; g.G = G; g.R = R;
    kivi_geom_init(g, max_tokens);
    c->T.assign(b, 0);
    c->Tqk.assign(b, 0);
    c->Tqv.assign(b, 0);

    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        snprintf(g_err, sizeof g_err, "no CUDA device: %s", cudaGetErrorString(e));
        return KIVI_ERR_CUDA;
    }
    // decode partials per (sequence, query head): one per persistent CTA that
    // touches the pair (the plan keeps the count within this bound)
    g.smax = kivi_partial_slots(b, h_kv, c->num_sms);
    KiviDev &dv = c->dv;
    memset(&dv, 0, sizeof dv);
    const size_t bh = (size_t)b * h_kv;
    struct Req { void **p; size_t bytes; } reqs[] = {
        {(void **)&dv.blk, bh * g.nkb * g.rec_bytes},
        {(void **)&dv.Kf, bh * R * d * 2},
        {(void **)&dv.Vf, bh * (R + 1) * d * 2},
        {(void **)&c->cnt, (size_t)2 * 3 * b * 4},
        {(void **)&dv.status, 4},
        {(void **)&dv.part, bh * KIVI_MAX_QPERKV * g.smax * (d + 4) * 4},
        {(void **)&dv.merge_ticket, bh * 4 * 4},
        {(void **)&dv.ml, bh * KIVI_MAX_QPERKV * 2 * 4},
    };
    for (auto &r : reqs) {
        e = cudaMalloc(r.p, r.bytes);
        if (e == cudaSuccess) e = cudaMemset(*r.p, 0, r.bytes);
        if (e != cudaSuccess) {
            free_dev(c);
            delete c;
            cudaGetLastError();
            snprintf(g_err, sizeof g_err, "device allocation failed: %s", cudaGetErrorString(e));
            return e == cudaErrorMemoryAllocation ? KIVI_ERR_OOM : KIVI_ERR_CUDA;
        }
    }
    c->parity = 0;
    point_counters(c);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_dev(c);
        delete c;
        snprintf(g_err, sizeof g_err, "create: %s", cudaGetErrorString(e));
        return KIVI_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        g_live.insert(c);
    }
    *out = c;
    return KIVI_OK;
}

kivi_status kivi_cache_destroy(kivi_cache_t c) {
    g_err[0] = 0;
    if (!c) {
        set_err("null cache handle");
        return KIVI_ERR_INVALID_ARG;
    }
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        if (!g_live.erase((void *)c)) {
            set_err("unknown or destroyed cache handle");
            return KIVI_ERR_INVALID_ARG;
        }
    }
    cudaDeviceSynchronize();
    cudaGetLastError();
    free_dev(c);
    for (cudaEvent_t e : c->ev) cudaEventDestroy(e);
    c->magic = 0;
    delete c;
    return KIVI_OK;
}

kivi_status kivi_prefill(kivi_cache_t c, const void *K, const void *V, const int32_t *t,
                         int t_stride, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    if (!t || t_stride < 0) {
        set_err("t is null or t_stride negative");
        return KIVI_ERR_INVALID_ARG;
    }
    SeqLens lens;
    int maxt = 0;
    for (int i = 0; i < c->g.b; ++i) {
        if (t[i] < 0 || t[i] > t_stride) {
            set_err("t[i] outside [0, t_stride] for i = %s%ld", "", i);
            return KIVI_ERR_INVALID_ARG;
        }
        if (t[i] > c->max_tokens) {
            set_err("t[i] above max_tokens for i = %s%ld", "", i);
            return KIVI_ERR_CAPACITY;
        }
        lens.t[i] = t[i];
        maxt = t[i] > maxt ? t[i] : maxt;
    }
    if (maxt > 0 && (!K || !V)) {
        set_err("K or V is null");
        return KIVI_ERR_INVALID_ARG;
    }
    if (maxt > 0 && (!aligned16(K) || !aligned16(V))) {
        set_err("K and V must be 16-byte aligned");
        return KIVI_ERR_INVALID_ARG;
    }
    cudaError_t e = kivi_launch_prefill(c->g, c->dv, (const __half *)K, (const __half *)V, lens,
                                        t_stride, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(c, e, "prefill");
    for (int i = 0; i < c->g.b; ++i) {
        c->T[i] = t[i];
        c->Tqk[i] = t[i] - t[i] % c->g.R;
        c->Tqv[i] = t[i] > c->g.R ? t[i] - c->g.R : 0;
    }
    return KIVI_OK;
}

kivi_status kivi_prefill_attn(kivi_cache_t c, const void *q, const void *K, const void *V, const int32_t *t,
                              int t_stride, int h_q, void *out, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    if (c->g.G > 64 || (c->g.d != 64 && c->g.d != 128)) {
        set_err("prefill attention supports d 64 or 128 and G <= 64");
        return KIVI_ERR_UNSUPPORTED;
    }
    if (h_q < c->g.h || h_q % c->g.h != 0 || h_q / c->g.h > KIVI_MAX_QPERKV) {
        set_err("h_q must be a multiple of h_kv, at most %s%ld times it", "", KIVI_MAX_QPERKV);
        return KIVI_ERR_INVALID_ARG;
    }
    if (!t || t_stride < 0) {
        set_err("t is null or t_stride negative");
        return KIVI_ERR_INVALID_ARG;
    }
    SeqLens lens;
    int maxt = 0;
    for (int i = 0; i < c->g.b; ++i) {
        if (t[i] < 0 || t[i] > t_stride) {
            set_err("t[i] outside [0, t_stride] for i = %s%ld", "", i);
            return KIVI_ERR_INVALID_ARG;
        }
        if (t[i] > c->max_tokens) {
            set_err("t[i] above max_tokens for i = %s%ld", "", i);
            return KIVI_ERR_CAPACITY;
        }
        lens.t[i] = t[i];
        maxt = t[i] > maxt ? t[i] : maxt;
    }
    if (maxt > 0 && (!q || !K || !V || !out)) {
        set_err("q, K, V or out is null");
        return KIVI_ERR_INVALID_ARG;
    }
    if (maxt > 0 && (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out))) {
        set_err("q, K, V and out must be 16-byte aligned");
        return KIVI_ERR_INVALID_ARG;
    }
    cudaError_t e = kivi_launch_prefill_attn(c->g, c->dv, (const __half *)q, (const __half *)K, (const __half *)V,
                                             (__half *)out, lens, t_stride, h_q, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail_cuda(c, e, "prefill_attn");
    for (int i = 0; i < c->g.b; ++i) {
        c->T[i] = t[i];
        c->Tqk[i] = t[i] - t[i] % c->g.R;
        c->Tqv[i] = t[i] > c->g.R ? t[i] - c->g.R : 0;
    }
    return KIVI_OK;
}

kivi_status kivi_append(kivi_cache_t c, const void *k, const void *v, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    s = check_append_args(c, k, v);
    if (s != KIVI_OK) return s;
    return launch_append(c, k, v, stream, "append");
}

kivi_status kivi_decode_attn(kivi_cache_t c, const void *q, int h_q, void *out,
                             kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    s = check_decode_args(c, q, h_q, out);
    if (s != KIVI_OK) return s;
    return launch_decode(c, q, h_q, out, stream, c->T.data(), c->Tqk.data(), c->Tqv.data(), "decode_attn");
}

kivi_status kivi_decode_attn_probs(kivi_cache_t c, const void *q, int h_q, void *out, float *probs,
                                   float *mass, int64_t ld, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    s = check_decode_args(c, q, h_q, out);
    if (s != KIVI_OK) return s;
    if (!probs || probs == mass) {
        set_err("probs is null or the same buffer as mass");
        return KIVI_ERR_INVALID_ARG;
    }
    if (((uintptr_t)probs & 3u) || ((uintptr_t)mass & 3u)) {
        set_err("probs and mass must be 4-byte aligned");
        return KIVI_ERR_INVALID_ARG;
    }
    int maxT = 0;
    for (int i = 0; i < c->g.b; ++i) maxT = c->T[i] > maxT ? c->T[i] : maxT;
    if (ld < 1 || ld < maxT) {
        set_err("ld must be at least 1 and at least every sequence's token count");
        return KIVI_ERR_INVALID_ARG;
    }
    const ProbsOut po{probs, mass, (long long)ld};
    return launch_decode(c, q, h_q, out, stream, c->T.data(), c->Tqk.data(), c->Tqv.data(), "decode_attn_probs",
                         &po);
}

kivi_status kivi_append_decode(kivi_cache_t c, const void *k, const void *v, const void *q, int h_q,
                               void *out, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    s = check_append_args(c, k, v);
    if (s != KIVI_OK) return s;
    s = check_decode_args(c, q, h_q, out);
    if (s != KIVI_OK) return s;
    if (fused_step(c, h_q)) return launch_fused_step(c, k, v, q, h_q, out, stream);
    s = launch_append(c, k, v, stream, "append_decode");
    if (s != KIVI_OK) return s;
    s = launch_decode(c, q, h_q, out, stream, c->T.data(), c->Tqk.data(), c->Tqv.data(), "append_decode");
    if (s == KIVI_OK) c->last_plan.launches += 1;
    return s;
}

kivi_status kivi_cache_lengths(kivi_cache_t c, int32_t *T, int32_t *Tqk, int32_t *Tqv) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK && s != KIVI_ERR_STATE) return s;
    for (int i = 0; i < c->g.b; ++i) {
        if (T) T[i] = c->T[i];
        if (Tqk) Tqk[i] = c->Tqk[i];
        if (Tqv) Tqv[i] = c->Tqv[i];
    }
    return KIVI_OK;
}

kivi_status kivi_cache_export_sizes(kivi_cache_t c, size_t sizes[6]) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK && s != KIVI_ERR_STATE) return s;
    if (!sizes) {
        set_err("sizes is null");
        return KIVI_ERR_INVALID_ARG;
    }
    const KiviGeom &g = c->g;
    const size_t bh = (size_t)g.b * g.h;
    sizes[0] = bh * g.nkb * g.kc_blk * 4;
    sizes[1] = bh * g.nkg * 2 * g.d * 2;
    sizes[2] = bh * g.nvb * g.vc_blk * 4;
    sizes[3] = bh * g.nvb * g.vsz_blk * 2;
    sizes[4] = bh * g.R * g.d * 2;
    sizes[5] = bh * (g.R + 1) * g.d * 2;
    return KIVI_OK;
}

kivi_status kivi_cache_export(kivi_cache_t c, void *Kc, void *Ksz, void *Vc, void *Vsz, void *Kf,
                              void *Vf, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    const KiviGeom &g = c->g;
    size_t sz[6];
    kivi_cache_export_sizes(c, sz);
    cudaStream_t st = (cudaStream_t)stream;
    const void *src[2] = {c->dv.Kf, c->dv.Vf};
    void *dst[2] = {Kf, Vf};
    for (int k = 0; k < 2; ++k) {
        if (!dst[k]) continue;
        cudaError_t e = cudaMemcpyAsync(dst[k], src[k], sz[4 + k], cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return fail_cuda(c, e, "export");
    }
    std::vector<unsigned char> rec;
    if (Kc || Ksz || Vc || Vsz) {
        rec.resize((size_t)g.b * g.h * g.nkb * g.rec_bytes);
        cudaError_t e = cudaMemcpyAsync(rec.data(), c->dv.blk, rec.size(), cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return fail_cuda(c, e, "export");
    }
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail_cuda(c, e, "export");
    if (rec.empty()) return KIVI_OK;
    // split the block records into the four documented arrays
    const size_t kcb = (size_t)g.kc_blk * 4, vcb = (size_t)4 * g.vc_blk * 4, vszb = (size_t)4 * g.vsz_blk * 2;
    const size_t rowsb = (size_t)2 * g.d * 2;   // one key group's scale and zero rows
    for (int i = 0; i < g.b; ++i)
        for (int j = 0; j < g.h; ++j)
            for (int kb = 0; kb < g.nkb; ++kb) {
                const unsigned char *r = rec.data() + rec_off(g, i, j, kb);
                const size_t slice = (size_t)i * g.h + j;
                if (Kc) memcpy((unsigned char *)Kc + (slice * g.nkb + kb) * kcb, r, kcb);
                if (Vc) memcpy((unsigned char *)Vc + (slice * g.nkb + kb) * vcb, r + g.off_vc, vcb);
                // scale / zero rows: undo the record's lane-major order
                if (Vsz) {
                    const uint16_t *src = reinterpret_cast<const uint16_t *>(r + g.off_vsz);
                    uint16_t *dst = reinterpret_cast<uint16_t *>((unsigned char *)Vsz + (slice * g.nkb + kb) * vszb);
                    for (int row = 0; row < 4 * g.vsz_blk / 16; ++row)
                        for (int tau = 0; tau < 16; ++tau) dst[row * 16 + tau] = src[row * 16 + vsz_pos(tau)];
                }
                if (Ksz && (g.G <= KIVI_KBLK || kb % (g.G / KIVI_KBLK) == 0)) {
                    // G > 64: the rows of group kb / (G / 64), from the first of its records
                    const int nrow = g.G <= KIVI_KBLK ? 2 * g.kgr : 2;
                    const size_t grp0 = g.G <= KIVI_KBLK ? (size_t)kb * g.kgr : (size_t)kb / (g.G / KIVI_KBLK);
                    const uint16_t *src = reinterpret_cast<const uint16_t *>(r + g.off_ksz);
                    uint16_t *dst = reinterpret_cast<uint16_t *>((unsigned char *)Ksz + (slice * g.nkg + grp0) * rowsb);
                    for (int row = 0; row < nrow; ++row)
                        for (int ch = 0; ch < g.d; ++ch) dst[(size_t)row * g.d + ch] = src[(size_t)row * g.d + ksz_pos(g.d, ch)];
                }
            }
    return KIVI_OK;
}

kivi_status kivi_cache_export_records(kivi_cache_t c, void *records, size_t *bytes, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    if (!bytes) {
        set_err("bytes is null");
        return KIVI_ERR_INVALID_ARG;
    }
    const KiviGeom &g = c->g;
    const size_t need = (size_t)g.b * g.h * g.nkb * g.rec_bytes;
    if (!records) {
        *bytes = need;
        return KIVI_OK;
    }
    if (*bytes < need) {
        snprintf(g_err, sizeof g_err, "records buffer holds %zu bytes, %zu needed", *bytes, need);
        return KIVI_ERR_INVALID_ARG;
    }
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(records, c->dv.blk, need, cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail_cuda(c, e, "export_records");
    *bytes = need;
    return KIVI_OK;
}

kivi_status kivi_cache_check(kivi_cache_t c, uint32_t *flags, kivi_stream_t stream) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    if (!flags) {
        set_err("flags is null");
        return KIVI_ERR_INVALID_ARG;
    }
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(flags, c->dv.status, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->dv.status, 0, 4, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return fail_cuda(c, e, "check");
    return KIVI_OK;
}

kivi_status kivi_profile_enable(kivi_cache_t c, int on) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    c->profiling = on != 0;
    return KIVI_OK;
}

kivi_status kivi_profile_read(kivi_cache_t c, double *total_ms, int *launches) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK) return s;
    double tot = 0.0;
    for (int k = 0; k < c->nprof; ++k) {
        cudaError_t e = cudaEventSynchronize(c->ev[2 * k + 1]);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, c->ev[2 * k], c->ev[2 * k + 1]);
        if (e != cudaSuccess) return fail_cuda(c, e, "profile_read");
        tot += ms;
    }
    if (total_ms) *total_ms = tot;
    if (launches) *launches = c->nprof;
    c->nprof = 0;
    return KIVI_OK;
}

kivi_status kivi_plan_preview(int b, int h_kv, int d, int k_bits, int v_bits, int G, int R, int max_tokens,
                              int h_q, const int32_t *T, const int32_t *Tqk, const int32_t *Tqv, int num_sms,
                              int64_t out[6]) {
    g_err[0] = 0;
    kivi_status s = check_shape(b, h_kv, d, k_bits, v_bits, G, R, max_tokens);
    if (s != KIVI_OK) return s;
    if (!T || !Tqk || !Tqv || !out) {
        set_err("a pointer argument is null");
        return KIVI_ERR_INVALID_ARG;
    }
    if (h_q < 1 || h_q % h_kv != 0 || num_sms < 1) {
        set_err("need h_q a positive multiple of h_kv and num_sms >= 1");
        return KIVI_ERR_INVALID_ARG;
    }
    if (h_q / h_kv > KIVI_MAX_QPERKV) {
        set_err("h_q / h_kv above 8");
        return KIVI_ERR_UNSUPPORTED;
    }
    for (int i = 0; i < b; ++i)
        if (T[i] < 0 || T[i] > max_tokens || Tqk[i] < 0 || Tqk[i] > T[i] || Tqv[i] < 0 || Tqv[i] > T[i]) {
            set_err("need 0 <= Tqk, Tqv <= T <= max_tokens (i = %s%ld)", "", i);
            return KIVI_ERR_INVALID_ARG;
        }
    KiviGeom g;
    g.b = b;
    g.h = h_kv;
    g.d = d;
    g.kbits = k_bits;
    g.vbits = v_bits;
    g.G = G;
    g.R = R;
    kivi_geom_init(g, max_tokens);
    g.smax = kivi_partial_slots(b, h_kv, num_sms);
    DecodeUnits units;
    const DecodePlan plan = kivi_plan_decode(g, h_q, T, Tqk, Tqv, num_sms, &units);
    out[0] = plan.ctas;
    out[1] = plan.warps;
    out[2] = plan.stages;
    out[3] = plan.max_parts;
    out[4] = g.smax;
    out[5] = units.total;
    return KIVI_OK;
}

kivi_status kivi_decode_plan(kivi_cache_t c, int *splits, int *launches) {
    g_err[0] = 0;
    kivi_status s = check_handle(c);
    if (s != KIVI_OK && s != KIVI_ERR_STATE) return s;
    if (splits) *splits = c->last_plan.ctas;
    if (launches) *launches = c->last_plan.launches;
    return KIVI_OK;
}

}  // extern "C"
