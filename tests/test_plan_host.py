"""The decode planner through kivi_plan_preview (host-only, no GPU): the
persistent grid, the ring, and the bound every plan must keep — no
(sequence, kv head, head group) receives more split partials than the
cache holds slots for (the kernel's merge relies on it)."""
import ctypes
import os

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_quantized_kv_quantize_gb300 import build as B
    L = ctypes.CDLL(B.build())
    i32, vp = ctypes.c_int, ctypes.c_void_p
    L.kivi_plan_preview.argtypes = [i32] * 9 + [vp, vp, vp, i32, vp]
    L.kivi_plan_preview.restype = i32
    return L


def preview(lib, shape, hq, T, Tqk, Tqv, sms):
    b = shape[0]
    arrs = [np.ascontiguousarray(np.asarray(x, np.int32).reshape(b)) for x in (T, Tqk, Tqv)]
    out = np.zeros(6, np.int64)
    rc = lib.kivi_plan_preview(*shape, hq, *(a.ctypes.data for a in arrs), sms, out.ctypes.data)
    return rc, dict(zip(("ctas", "warps", "stages", "max_parts", "slots", "units"), out.tolist()))


def state_after(t, steps, R):
    """Counters after prefill of t tokens and `steps` appends (lazy
    maintenance: flush when the key window holds R, pop at R + 1)."""
    T, Tqk, Tqv = t, t - t % R, max(t - R, 0)
    for _ in range(steps):
        if T - Tqk == R:
            Tqk += R
        if T - Tqv == R + 1:
            Tqv += 1
        T += 1
    return T, Tqk, Tqv


def test_default_workload_plan(lib):
    """b = 8, 32 query / 8 kv heads, d = 128, 2-bit, G = 32, R = 128, 32767
    tokens + 1 appended, 152 SMs: two CTAs per SM, eight warps, each pair's
    units = a lead of 3 (a segment's fixed cost) + full blocks + 12 per
    block holding fp16 tokens."""
    T, Tqk, Tqv = state_after(32767, 1, 128)
    rc, p = preview(lib, (8, 8, 128, 2, 2, 32, 128, 40000), 32, [T] * 8, [Tqk] * 8, [Tqv] * 8, 152)
    assert rc == 0
    assert p["ctas"] == 304 and p["warps"] == 8 and p["stages"] >= 2
    nf, nb = min(Tqk, Tqv) // 64, -(-T // 64)
    assert p["units"] == 8 * 8 * (3 + nf + 12 * (nb - nf))
    assert p["max_parts"] <= p["slots"]


@pytest.mark.parametrize("seed", range(40))
def test_random_shapes_keep_the_partial_bound(lib, seed):
    rng = np.random.default_rng(seed)
    d = int(rng.choice([64, 128, 256]))
    G = int(rng.choice([g for g in (16, 32, 64, 128) if d % g == 0]))
    R = G * int(rng.integers(1, 9))
    kb, vb = (int(x) for x in rng.choice([2, 4], 2))
    b = int(rng.integers(1, 65))
    h = int(rng.integers(1, 9))
    hq = h * int(rng.integers(1, 9))
    cap = int(rng.integers(1, 70000))
    sms = int(rng.choice([1, 2, 16, 100, 152]))
    T, Tqk, Tqv = [], [], []
    for _ in range(b):
        t = int(rng.integers(0, cap + 1))
        steps = int(rng.integers(0, min(300, cap - t) + 1))
        s = state_after(t, steps, R)
        T.append(s[0]), Tqk.append(s[1]), Tqv.append(s[2])
    rc, p = preview(lib, (b, h, d, kb, vb, G, R, cap), hq, T, Tqk, Tqv, sms)
    assert rc == 0
    assert 1 <= p["ctas"] <= 2 * sms
    assert 1 <= p["warps"] <= 8 and 2 <= p["stages"] <= 4
    assert p["max_parts"] <= p["slots"], p
    groups = -(-(hq // h) // 4)
    assert p["units"] >= b * h * groups   # every pair, even an empty one, has a unit


def test_rejected_arguments(lib):
    ok = (2, 2, 128, 2, 2, 32, 128, 1000)
    assert preview(lib, ok, 4, [10, 0], [0, 0], [0, 0], 152)[0] == 0
    assert preview(lib, ok, 3, [10, 0], [0, 0], [0, 0], 152)[0] == 1            # h_q % h_kv
    assert preview(lib, ok, 18, [10, 0], [0, 0], [0, 0], 152)[0] == 2           # > 8 query heads a kv head
    assert preview(lib, ok, 4, [1001, 0], [0, 0], [0, 0], 152)[0] == 1          # T above capacity
    assert preview(lib, ok, 4, [10, 0], [11, 0], [0, 0], 152)[0] == 1           # Tqk above T
    assert preview(lib, ok, 4, [10, 0], [0, 0], [0, 0], 0)[0] == 1              # no SMs
    assert preview(lib, (2, 2, 128, 3, 2, 32, 128, 1000), 4, [1, 1], [0, 0], [0, 0], 152)[0] == 2
