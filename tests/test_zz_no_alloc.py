"""The allocation-free decode entry point, called through the C ABI.

kivi_decode_attn_noalloc serves callers that cannot call cudaMalloc (a
framework's memory pool owns the device memory, an allocator callback, a
real-time budget): it reads a packed cache held in the caller's memory and
keeps its scratch in a fixed array inside the library.  Its output must
match kivi_decode_attn on the same cache, within the attention tolerance,
on two calls in a row (the second reuses the scratch the first left behind).
This file runs last so that a failure here leaves every other test run.
"""
import ctypes

import numpy as np
import pytest

from bit_quantized_kv_quantize_gb300 import workloads as W
from tests import kivi_testutil as U

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


class PackedCache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("b", "h_kv", "d", "k_bits", "v_bits", "G", "R",
                                            "max_tokens")] + \
               [(n, ctypes.c_void_p) for n in ("blocks", "Kf", "Vf", "T", "Tqk", "Tqv")]


CASES = [
    # workload, b, prefill (0: ragged 300-900), steps, field overrides
    ("llama3_8b_gqa_32k", 2, 3000, 3, {}),
    ("kivi4_serving", 6, 0, 2, {}),
    ("tiny_kivi2", 3, 0, 5, dict(h_q=8, h_kv=2, kbits=4, vbits=2, G=16, R=32)),
]


@pytest.mark.parametrize("name,b,prefill,steps,over", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_decode_attn(name, b, prefill, steps, over):
    from bit_quantized_kv_quantize_gb300 import kivi as K
    w = W.small(W.WORKLOADS[name], b=b, prefill=prefill or 900, ragged=(300, 900) if prefill == 0 else (),
                **over)
    cap = int(w.lengths().max()) + steps + 4
    cache = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    Kh, Vh, lens = W.prefill_kv(w)
    cache.prefill(torch.from_numpy(Kh).cuda(), torch.from_numpy(Vh).cuda(), lens)
    for s in range(steps):
        k, v = W.step_kv(w, s)
        cache.append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda())

    # the same cache in caller-owned device memory (the documented block
    # records and fp16 windows)
    ex = cache.export()
    dev = {key: torch.from_numpy(ex[key].view(np.uint8).copy()).cuda() for key in ("Kf", "Vf")}
    dev["blocks"] = torch.from_numpy(cache.export_records()).cuda()
    T, Tqk, Tqv = cache.lengths()
    cnt = {n: torch.from_numpy(x.astype(np.int32)).cuda() for n, x in (("T", T), ("Tqk", Tqk), ("Tqv", Tqv))}
    pc = PackedCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap,
                     *[dev[key].data_ptr() for key in ("blocks", "Kf", "Vf")],
                     *[cnt[n].data_ptr() for n in ("T", "Tqk", "Tqv")])
    fn = K.lib.kivi_decode_attn_noalloc
    fn.argtypes = [ctypes.POINTER(PackedCache), ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stream = torch.cuda.current_stream()
    for call in range(2):
        q = torch.from_numpy(W.step_q(w, 10 + call)).cuda()
        ref = cache.decode(q).float().cpu().numpy()
        out = torch.full_like(q, float("nan"))
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = fn(ctypes.byref(pc), q.data_ptr(), w.h_q, out.data_ptr(), stream.cuda_stream)
        assert rc == 0, K.lib.kivi_last_error().decode()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        # the first call of a shape may load the array and the kernel's code
        # (lazy module loading); a later call takes no device memory
        if call == 1:
            assert free1 == free0, f"second no-alloc call took {free0 - free1} bytes of device memory"
        U.compare_output(out.float().cpu().numpy(), ref, f"{name} no-alloc call {call}")
    cache.close()


def test_noalloc_rejects_oversized_scratch():
    from bit_quantized_kv_quantize_gb300 import kivi as K
    buf = torch.zeros(1 << 12, dtype=torch.uint8, device="cuda")
    p = buf.data_ptr()
    # 1024 sequences x 64 query heads x 128k tokens needs far more than 16 MiB of partials
    pc = PackedCache(1024, 8, 128, 2, 2, 32, 128, 131072, p, p, p, p, p, p)
    fn = K.lib.kivi_decode_attn_noalloc
    fn.argtypes = [ctypes.POINTER(PackedCache), ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                   ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(ctypes.byref(pc), p, 64, p, None) == 2
    assert b"16 MiB" in K.lib.kivi_last_error()
