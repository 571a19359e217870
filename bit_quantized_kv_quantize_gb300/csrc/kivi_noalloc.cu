// kivi_noalloc.cu -- decode attention that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs while its framework's
// memory pool owns all device memory, inside an allocator callback, or under
// a real-time budget that forbids allocation after start-up.  For them,
// kivi_decode_attn_noalloc reads a packed cache that lives in memory the
// caller already owns and keeps its own scratch (the split-K partials, the
// merge tickets and the status word) in one file-scope __device__ array of
// fixed size, instead of the per-cache buffers kivi_cache_create allocates.
//
// CUDA loads a library's device code and __device__ arrays lazily, on first
// use: the array (KIVI_NOALLOC_SCRATCH_BYTES) takes device memory on a device
// from the first call there (the address look-up loads it), and the decode
// kernel's code when a call first launches that kernel variant (head
// dimension, bit widths, G); both stay until the process exits.  Later calls
// of an already-used shape take no device memory.  All calls share the
// array, so calls whose kernels overlap on the GPU (different streams, or
// different host threads) race on it; the tickets that must start at zero
// and the status word are cleared by each call, the partials are fully
// rewritten before they are read.
// The status word in the array is cleared by each call and never read back:
// this path reports no device-side anomaly (a bounded wait that ran out).
#include <cstring>
#include <mutex>

#include "../../include/kivi.h"
#include "kivi_internal.cuh"

#define KIVI_NOALLOC_SCRATCH_BYTES (16u << 20)   // 16 MiB
#define KIVI_NOALLOC_MAX_DEVICES 64

static __device__ __align__(256) unsigned char g_noalloc_scratch[KIVI_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_mu;
unsigned char *g_addr[KIVI_NOALLOC_MAX_DEVICES];   // device address of the array, per device

kivi_status fail(kivi_status s, const char *msg) {
    kivi_set_last_error(msg);   // readable through kivi_last_error()
    return s;
}

// The array's name is only a host-side stand-in in host code; the kernel
// needs its device address, looked up once per device with that device
// current.  A cudaDeviceReset unloads the module and makes the cached
// address stale: the entry point is not to be used after a reset.
kivi_status scratch_address(unsigned char **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= KIVI_NOALLOC_MAX_DEVICES)
        return fail(KIVI_ERR_CUDA, "no usable CUDA device");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return fail(KIVI_ERR_CUDA, cudaGetErrorString(e));
        g_addr[dev] = static_cast<unsigned char *>(p);
    }
    *out = g_addr[dev];
    return KIVI_OK;
}

}  // namespace

extern "C" kivi_status kivi_decode_attn_noalloc(const kivi_packed_cache *pc, const void *q, int h_q,
                                                void *out, kivi_stream_t stream) {
    kivi_set_last_error("");
    if (!pc || !q || !out) return fail(KIVI_ERR_INVALID_ARG, "cache, q or out is null");
    const int b = pc->b, h = pc->h_kv, d = pc->d, G = pc->G, R = pc->R;
    // the same shape rules as kivi_cache_create (they also bound max_tokens,
    // so the capacity arithmetic below stays in range)
    const int sc = kivi_check_shape(b, h, d, pc->k_bits, pc->v_bits, G, R, pc->max_tokens);
    if (sc != KIVI_OK) return (kivi_status)sc;   // the error text is set
    if (h_q < 1 || h_q % h != 0) return fail(KIVI_ERR_INVALID_ARG, "h_q must be a positive multiple of h_kv");
    if (h_q / h > KIVI_MAX_QPERKV) return fail(KIVI_ERR_UNSUPPORTED, "h_q / h_kv above 8");
    const void *ptrs[] = {pc->blocks, pc->Kf, pc->Vf, q, out};
    for (const void *p : ptrs)
        if (!p || ((uintptr_t)p & 15u)) return fail(KIVI_ERR_INVALID_ARG, "array pointers must be non-null and 16-byte aligned");
    if (!pc->T || !pc->Tqk || !pc->Tqv) return fail(KIVI_ERR_INVALID_ARG, "counter pointers are null");

    KiviGeom g;
    g.b = b; g.h = h; g.d = d; g.kbits = pc->k_bits; g.vbits = pc->v_bits; g.G = G; g.R = R;
    kivi_geom_init(g, pc->max_tokens);
    // Plan for the capacity (the counters stay on the device): every
    // sequence is taken as full; blocks past a sequence's data are skipped.
    int full[KIVI_MAX_BATCH];
    for (int i = 0; i < b; ++i) full[i] = g.fcap;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(KIVI_ERR_CUDA, "no usable CUDA device");
    g.smax = kivi_partial_slots(b, h, sms);
    DecodeUnits units;   // on the stack: no allocation
    const DecodePlan plan = kivi_plan_decode(g, h_q, full, full, full, sms, &units);
    g.smax = plan.max_parts;   // partial stride: exactly what this plan writes

    const size_t part_bytes = (size_t)b * h_q * g.smax * (d + 4) * sizeof(float);
    const size_t ticket_off = (part_bytes + 255) / 256 * 256;
    const size_t ticket_bytes = (size_t)b * h * 4 * sizeof(unsigned);
    const size_t status_off = ticket_off + (ticket_bytes + 255) / 256 * 256;
    if (status_off + 256 > KIVI_NOALLOC_SCRATCH_BYTES)
        return fail(KIVI_ERR_UNSUPPORTED,
                    "decode scratch for this shape exceeds the fixed 16 MiB no-alloc array");

    unsigned char *scratch = nullptr;
    kivi_status s = scratch_address(&scratch);
    if (s != KIVI_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    // the merge tickets and the status word must start at zero
    cudaError_t e = cudaMemsetAsync(scratch + ticket_off, 0, status_off + 256 - ticket_off, st);
    if (e != cudaSuccess) return fail(KIVI_ERR_CUDA, cudaGetErrorString(e));

    KiviDev dv;
    memset(&dv, 0, sizeof dv);
    dv.blk = (unsigned char *)pc->blocks;
    dv.Kf = (__half *)pc->Kf;
    dv.Vf = (__half *)pc->Vf;
    dv.T = (int *)pc->T;
    dv.Tqk = (int *)pc->Tqk;
    dv.Tqv = (int *)pc->Tqv;
    dv.part = reinterpret_cast<float *>(scratch);
    dv.merge_ticket = reinterpret_cast<unsigned *>(scratch + ticket_off);
    dv.status = reinterpret_cast<unsigned *>(scratch + status_off);
    e = kivi_launch_decode(g, dv, (const __half *)q, h_q, (__half *)out, plan, units, st, nullptr,
                           nullptr);
    if (e != cudaSuccess) return fail(KIVI_ERR_CUDA, cudaGetErrorString(e));
    return KIVI_OK;
}
