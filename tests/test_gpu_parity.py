"""GPU parity: libkivi (CUDA, called through the C ABI) against the CPU oracle
on the same seeded inputs.  Packed codes, scale/zero words and fp16 windows
must be bit-exact; attention outputs within 2e-3 max-abs and 1e-3 relative L2.
"""
import os
import zlib

import numpy as np
import pytest

import oracle
from bit_quantized_kv_quantize_gb300 import workloads as W
from tests import kivi_testutil as U

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from bit_quantized_kv_quantize_gb300 import kivi as K

oracle.set_threads(os.cpu_count() or 1)


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class Pair:
    """A GPU cache and an oracle cache fed identical inputs."""

    def __init__(self, b, h, d, kb, vb, G, R, cap):
        self.dims = (b, h, d, kb, vb, G, R)
        self.cap = cap
        self.gpu = K.KiviCache(b, h, d, kb, vb, G, R, cap)
        self.ora = oracle.Cache(b, h, d, kb, vb, G, R, cap)
        self.g = U.geometry(b, h, d, kb, vb, G, R, cap)

    def prefill(self, Kh, Vh, lens):
        self.gpu.prefill(_dev(Kh), _dev(Vh), lens)
        self.ora.prefill(Kh, Vh, lens)

    def append(self, k, v):
        self.gpu.append(_dev(k), _dev(v))
        self.ora.append(k, v)

    def check_state(self, what="", seqs=None):
        T, Tqk, Tqv = self.ora.lengths()
        gT, gTqk, gTqv = self.gpu.lengths()
        assert np.array_equal(T, gT) and np.array_equal(Tqk, gTqk) and np.array_equal(Tqv, gTqv)
        gex = self.gpu.export()
        oex = self.ora.export()
        b, h = self.dims[:2]
        for i in (range(b) if seqs is None else seqs):
            for j in range(h):
                U.compare_slice(gex, self.g, i, j, oex, self.g, i, j, int(T[i]), int(Tqk[i]),
                                int(Tqv[i]), what=f"{what} seq {i} head {j}")
        assert self.gpu.check() == 0

    def step_fused(self, k, v, q, what=""):
        """One fused append + decode on the GPU against append then decode in the oracle."""
        out = self.gpu.append_decode(_dev(k), _dev(v), _dev(q)).float().cpu().numpy()
        self.ora.append(k, v)
        return U.compare_output(out, self.ora.decode(q), what)

    def check_decode(self, q, what="", pairs=None):
        out = self.gpu.decode(_dev(q)).float().cpu().numpy()
        ref = self.ora.decode(q, pairs=pairs)
        if pairs is not None:
            idx = tuple(np.asarray(pairs).T)
            return U.compare_output(out[idx], ref[idx], what)
        return U.compare_output(out, ref, what)


def _rand_kv(rng, b, h, t, d, kscale=1.0):
    Kh = (rng.standard_normal((b, h, max(t, 1), d)) * kscale).astype(np.float16)
    Vh = rng.standard_normal((b, h, max(t, 1), d)).astype(np.float16)
    return Kh, Vh


# ---------------------------------------------------------------------------
# The tiny reference workload: every step checked.
# ---------------------------------------------------------------------------

def test_tiny_kivi2_every_step():
    w = W.WORKLOADS["tiny_kivi2"]
    p = Pair(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, w.capacity())
    Kh, Vh, lens = W.prefill_kv(w)
    p.prefill(Kh, Vh, lens)
    p.check_state("prefill")
    p.check_decode(W.step_q(w, 0), "prefill decode")
    for s in range(w.steps):
        k, v = W.step_kv(w, s)
        p.append(k, v)
        p.check_state(f"step {s}")
        p.check_decode(W.step_q(w, s), f"step {s}")


# ---------------------------------------------------------------------------
# The one-call step (kivi_append_decode): the append kernel, then the
# decode kernel launched as its programmatic dependent.
# ---------------------------------------------------------------------------

def test_fused_step_tiny_every_step():
    w = W.WORKLOADS["tiny_kivi2"]
    p = Pair(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, w.capacity())
    Kh, Vh, lens = W.prefill_kv(w)
    p.prefill(Kh, Vh, lens)
    for s in range(w.steps):
        k, v = W.step_kv(w, s)
        p.step_fused(k, v, W.step_q(w, s), f"fused step {s}")
        p.check_state(f"fused step {s}")


FUSED = [
    # b, h, hq, d, kb, vb, G, R, lens, steps
    (8, 2, 8, 128, 4, 4, 32, 128, [300, 317, 512, 640, 700, 767, 800, 899], 200),
    (3, 2, 2, 64, 2, 2, 32, 32, [0, 1, 31], 70),
    (2, 1, 3, 256, 2, 2, 64, 128, [300, 64], 135),
    (2, 2, 4, 128, 2, 2, 128, 128, [511, 128], 130),
    # G = 16 and 4-bit keys at d = 64 (pops open fresh value blocks)
    (4, 2, 2, 64, 4, 2, 16, 64, [0, 63, 64, 130], 140),
    # two head groups per kv head: the two-launch path
    (2, 1, 8, 128, 2, 4, 16, 64, [100, 0], 80),
]


@pytest.mark.parametrize("case", FUSED, ids=[f"fused{i}" for i in range(len(FUSED))])
def test_fused_step_ragged(case):
    """Ragged batches over enough fused steps to cross key flushes and value
    pops in every sequence; outputs every step, the cache every 9th."""
    b, h, hq, d, kb, vb, G, R, lens, steps = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))
    p = Pair(b, h, d, kb, vb, G, R, max(lens) + steps + 3)
    Kh, Vh = _rand_kv(rng, b, h, max(lens), d, kscale=3.0)
    p.prefill(Kh, Vh, np.array(lens, np.int32))
    for s in range(steps):
        k = (rng.standard_normal((b, h, d)) * 3).astype(np.float16)
        v = rng.standard_normal((b, h, d)).astype(np.float16)
        q = rng.standard_normal((b, hq, d)).astype(np.float16)
        p.step_fused(k, v, q, f"fused step {s}")
        if s % 9 == 0 or s == steps - 1:
            p.check_state(f"fused step {s}")


@pytest.mark.parametrize("tail,case", [(3, 0), (9, 1)])
def test_fused_step_with_tail_units(monkeypatch, tail, case):
    """The one-launch plan's trailing units (they hold no blocks) and the
    pairs' lead units forced larger than these small shapes get: the same
    results, step by step."""
    monkeypatch.setenv("KIVI_DECODE_FUSED_TAIL", str(tail))
    monkeypatch.setenv("KIVI_DECODE_LEAD", str(tail + 2))
    test_fused_step_ragged(FUSED[case])


def test_fused_step_launch_count(monkeypatch):
    """kivi_append_decode is one launch on steps without a key-window
    flush, two on flush steps, and two with KIVI_FUSED_STEP=0, with more
    than one head group per kv head, or with more (sequence, kv head) pairs
    than twice the SM count (unless KIVI_FUSED_STEP=1)."""
    h, d, R = 2, 64, 32
    rng = np.random.default_rng(5)
    many = torch.cuda.get_device_properties(0).multi_processor_count + 1   # b h > 2 SMs
    for b, hq, env in ((2, 4, None), (2, 4, "0"), (2, 16, None), (many, 2, None), (many, 2, "1")):
        if env is None:
            monkeypatch.delenv("KIVI_FUSED_STEP", raising=False)
        else:
            monkeypatch.setenv("KIVI_FUSED_STEP", env)
        Kh, Vh = _rand_kv(rng, b, h, 40, d)
        c = K.KiviCache(b, h, d, 2, 2, 32, R, 128)
        c.prefill(_dev(Kh), _dev(Vh), np.array([40, 9] * (b // 2) + [40] * (b % 2), np.int32))
        one = env != "0" and hq // h <= 4 and (env == "1" or b * h <= 2 * (many - 1))
        nflush = 0
        for s in range(30):
            T, Tqk, _ = c.lengths()
            flush = bool(np.any(T - Tqk == R))
            k = _dev(rng.standard_normal((b, h, d)).astype(np.float16))
            v = _dev(rng.standard_normal((b, h, d)).astype(np.float16))
            q = _dev(rng.standard_normal((b, hq, d)).astype(np.float16))
            c.append_decode(k, v, q)
            launches = c.plan()[1]
            assert launches == (1 + flush if one else 2), (hq, env, s, launches)
            nflush += flush
        assert 0 < nflush < 30
        assert c.check() == 0
        c.close()


def test_fused_step_matches_two_calls():
    """Same inputs through kivi_append_decode and through kivi_append +
    kivi_decode_attn: identical caches, outputs within the tolerance."""
    w = W.small(W.WORKLOADS["llama3_8b_gqa_32k"], b=2, prefill=3000)
    caches = [K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, 3200) for _ in range(2)]
    Kh, Vh, lens = W.prefill_kv(w)
    for c in caches:
        c.prefill(_dev(Kh), _dev(Vh), lens)
    for s in range(140):
        k, v = W.step_kv(w, s)
        q = _dev(W.step_q(w, s))
        a = caches[0].append_decode(_dev(k), _dev(v), q).float().cpu().numpy()
        caches[1].append(_dev(k), _dev(v))
        b_ = caches[1].decode(q).float().cpu().numpy()
        U.compare_output(a, b_, f"step {s}")
    ea, eb = caches[0].export(), caches[1].export()
    for key in ea:
        assert np.array_equal(ea[key], eb[key]), key
    assert all(np.array_equal(x, y) for x, y in zip(caches[0].lengths(), caches[1].lengths()))
    assert caches[0].check() == 0 and caches[1].check() == 0
    for c in caches:
        c.close()


# ---------------------------------------------------------------------------
# Edge cases: lengths around G and R, ragged batches with an empty sequence,
# bit widths, group sizes, head dims, MHA.
# ---------------------------------------------------------------------------

EDGE = [
    # b, h, hq, d, kb, vb, G, R, lens, appends
    (3, 2, 2, 64, 2, 2, 32, 32, [0, 1, 31], 70),
    (3, 2, 4, 64, 2, 2, 32, 32, [32, 33, 63], 40),
    (4, 1, 8, 128, 4, 4, 32, 128, [127, 128, 129, 256], 140),
    (2, 2, 2, 128, 2, 4, 32, 64, [0, 200], 70),
    (2, 2, 6, 128, 4, 2, 16, 48, [47, 96], 60),
    (2, 1, 3, 256, 2, 2, 64, 128, [300, 64], 135),
    (2, 2, 4, 128, 2, 2, 128, 128, [511, 128], 130),
    (1, 1, 1, 64, 4, 4, 16, 16, [5], 50),
]


@pytest.mark.parametrize("case", EDGE, ids=[f"edge{i}" for i in range(len(EDGE))])
def test_edge_cases(case):
    b, h, hq, d, kb, vb, G, R, lens, appends = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))
    cap = max(lens) + appends + 3
    p = Pair(b, h, d, kb, vb, G, R, cap)
    Kh, Vh = _rand_kv(rng, b, h, max(lens), d, kscale=3.0)
    p.prefill(Kh, Vh, np.array(lens, np.int32))
    p.check_state("prefill")
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    p.check_decode(q, "prefill decode")
    for s in range(appends):
        k = (rng.standard_normal((b, h, d)) * 3).astype(np.float16)
        v = rng.standard_normal((b, h, d)).astype(np.float16)
        p.append(k, v)
        if s % 7 == 0 or s == appends - 1:
            p.check_state(f"step {s}")
            q = rng.standard_normal((b, hq, d)).astype(np.float16)
            p.check_decode(q, f"step {s}")


def test_constant_tiny_and_outlier_groups():
    """Constant groups (scale 0), spreads that give subnormal fp16 scales,
    huge outlier channels, and exact ties."""
    b, h, d, G, R, t = 2, 2, 128, 32, 32, 200
    rng = np.random.default_rng(99)
    Kh = rng.standard_normal((b, h, t, d)).astype(np.float32)
    Vh = rng.standard_normal((b, h, t, d)).astype(np.float32)
    Kh[0, 0, :64, :] = 0.5                          # constant key groups
    Kh[0, 1, :, 5] = 1.0 + rng.integers(0, 2, t) * 2.0 ** -10   # one-ulp spreads
    Kh[1, 0, :, :] *= 1e-6                          # subnormal scales
    Kh[1, 1, :, 7] *= 300                           # outlier channel
    Vh[0, 0, :, :32] = -2.0                         # constant value groups
    Vh[1, 0, :, :] *= 1e-6
    Vh[1, 1, ::3, :] = np.round(Vh[1, 1, ::3, :] * 2) / 2   # exact ties on coarse grids
    Kh, Vh = Kh.astype(np.float16), Vh.astype(np.float16)
    for kb in (2, 4):
        p = Pair(b, h, d, kb, kb, G, R, t + 40)
        p.prefill(Kh, Vh, np.array([t, t - 17], np.int32))
        p.check_state(f"prefill {kb}-bit")
        q = rng.standard_normal((b, 2 * h, d)).astype(np.float16)
        p.check_decode(q, f"decode {kb}-bit")
        for s in range(35):
            p.append(Kh[:, :, s].copy(), Vh[:, :, s].copy())
        p.check_state(f"appends {kb}-bit")
        p.check_decode(q, f"decode after appends {kb}-bit")


def test_decode_is_read_only_and_repeatable():
    w = W.small(W.WORKLOADS["llama3_8b_gqa_32k"], b=2, prefill=1000)
    gpu = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, 2000)
    Kh, Vh, lens = W.prefill_kv(w)
    gpu.prefill(_dev(Kh), _dev(Vh), lens)
    q = _dev(W.step_q(w, 0))
    before = gpu.export()
    o1 = gpu.decode(q).clone()
    o2 = gpu.decode(q).clone()
    after = gpu.export()
    assert torch.equal(o1, o2)
    for k in before:
        assert np.array_equal(before[k], after[k])


@pytest.mark.parametrize("G,kb,vb,d", [(32, 2, 2, 128), (16, 4, 2, 64), (64, 2, 4, 128), (128, 4, 4, 256)])
def test_block_records_match_the_packed_arrays(G, kb, vb, d):
    """The device's block records, split by the documented record layout
    (scale and zero rows lane-major), equal the four packed arrays of
    kivi_cache_export."""
    b, h, R, cap = 2, 2, max(G, 128), 800
    gpu = K.KiviCache(b, h, d, kb, vb, G, R, cap)
    rng = np.random.default_rng(G * 31 + kb)
    Kh, Vh = _rand_kv(rng, b, h, 600, d)
    gpu.prefill(_dev(Kh), _dev(Vh), [600, 437])
    for s in range(R + 3):   # crosses a key flush and value pops
        k, v = _rand_kv(rng, b, h, 1, d)
        gpu.append(_dev(k[:, :, 0]), _dev(v[:, :, 0]))
    ex = gpu.export()
    rec = gpu.export_records()
    g = U.geometry(b, h, d, kb, vb, G, R, cap)
    kgr = max(1, 64 // G)
    sizes = [g["kc_blk"] * 4, kgr * 2 * d * 2, 4 * g["vc_blk"] * 4, 4 * g["vsz_blk"] * 2]
    rb = sum(sizes)
    assert rec.size == b * h * g["nkb"] * rb
    rec = rec.reshape(b, h, g["nkb"], rb)
    o = np.cumsum([0] + sizes)
    Kc = rec[..., o[0]:o[1]].copy().view(np.uint32).reshape(-1)
    Vc = rec[..., o[2]:o[3]].copy().view(np.uint32).reshape(-1)
    # scale / zero rows are lane-major inside a record: value token
    # tau = 2t + 8p + lo at 4t + 2p + lo, key channel c = 16jj + 8hh + 2t + lo
    # at t d/4 + 4jj + 2hh + lo
    tau = np.arange(16)
    vpos = 4 * ((tau >> 1) & 3) + 2 * ((tau >> 3) & 1) + (tau & 1)
    Vsz = rec[..., o[3]:o[4]].copy().view(np.uint16).reshape(-1, 16)[:, vpos].reshape(-1)
    ch = np.arange(d)
    kpos = ((ch >> 1) & 3) * (d // 4) + 4 * (ch >> 4) + 2 * ((ch >> 3) & 1) + (ch & 1)
    rows = rec[..., o[1]:o[2]].copy().view(np.uint16).reshape(b, h, g["nkb"], kgr, 2, d)[..., kpos]
    if G <= 64:
        Ksz = rows.reshape(-1)
    else:   # both records of a group carry its rows
        assert np.array_equal(rows[:, :, 0::2], rows[:, :, 1::2])
        Ksz = rows[:, :, 0::2].reshape(-1)
    assert np.array_equal(Kc, ex["Kc"])
    assert np.array_equal(Ksz, ex["Ksz"])
    assert np.array_equal(Vc, ex["Vc"])
    assert np.array_equal(Vsz, ex["Vsz"])


def test_non_default_stream():
    w = W.small(W.WORKLOADS["tiny_kivi2"], prefill=100)
    p = Pair(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, 200)
    Kh, Vh, lens = W.prefill_kv(w)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p.prefill(Kh, Vh, lens)
        for st in range(5):
            k, v = W.step_kv(w, st)
            p.append(k, v)
        q = W.step_q(w, 0)
        out = p.gpu.decode(_dev(q))
    s.synchronize()
    U.compare_output(out.float().cpu().numpy(), p.ora.decode(q), "side stream")
    p.check_state("side stream")


def test_errors_leave_state_unchanged():
    d = 64
    gpu = K.KiviCache(1, 1, d, 2, 2, 32, 32, 40)
    Kh = _dev(np.ones((1, 1, 40, d), np.float16))
    gpu.prefill(Kh, Kh, [40])
    before = gpu.export()
    k = _dev(np.ones((1, 1, d), np.float16))
    with pytest.raises(K.CapacityError):
        gpu.append(k, k)
    with pytest.raises(K.KiviError):
        gpu.decode(_dev(np.ones((1, 9, d), np.float16)))   # more than 8 query heads a kv head
    after = gpu.export()
    for key in before:
        assert np.array_equal(before[key], after[key])
    assert tuple(int(x[0]) for x in gpu.lengths()) == (40, 32, 8)
    with pytest.raises(K.KiviError):
        gpu.prefill(Kh, Kh, [41])
    h = gpu.handle
    gpu.close()
    assert K.lib.kivi_append(h, k.data_ptr(), k.data_ptr(), None) == 1   # destroyed handle


# ---------------------------------------------------------------------------
# Full-size workloads, sampled: the launch configuration the benchmark times.
# ---------------------------------------------------------------------------

def _full_size(name):
    """The workload at full size, as the benchmark runs it: prefill, one
    append, one decode.  Every (sequence, kv head) slice of the cache is
    compared bit-exact with an oracle of that slice, and the whole output
    (every sequence and query head) with the oracle's, within the tolerance
    over the whole output."""
    from concurrent.futures import ThreadPoolExecutor
    w = W.WORKLOADS[name]
    cap = w.capacity()
    gpu = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    Kh, Vh, lens = W.prefill_kv(w)
    gpu.prefill(_dev(Kh), _dev(Vh), lens)
    del Kh, Vh
    k, v = W.step_kv(w, 0)
    gpu.append(_dev(k), _dev(v))
    q = W.step_q(w, 0)
    out = gpu.decode(_dev(q)).float().cpu().numpy()
    gex = gpu.export()
    assert gpu.check() == 0
    gg = U.geometry(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    og = U.geometry(1, 1, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    T, Tqk, Tqv = gpu.lengths()
    hg = w.group
    ref = np.zeros_like(out)

    def one(ij):
        i, j = ij
        n = int(lens[i])
        ora = oracle.Cache(1, 1, w.d, w.kbits, w.vbits, w.G, w.R, cap)
        ora.prefill(W.prefill_slice(w, "K", i, j, n)[None, None], W.prefill_slice(w, "V", i, j, n)[None, None],
                    [n])
        ora.append(np.ascontiguousarray(k[i:i + 1, j:j + 1]), np.ascontiguousarray(v[i:i + 1, j:j + 1]))
        U.compare_slice(gex, gg, i, j, ora.export(), og, 0, 0, int(T[i]), int(Tqk[i]), int(Tqv[i]),
                        what=f"{name} seq {i} head {j}")
        ref[i, j * hg:(j + 1) * hg] = ora.decode(np.ascontiguousarray(q[i:i + 1, j * hg:(j + 1) * hg]))[0]
        ora.close()

    slices = [(i, j) for i in range(w.b) for j in range(w.h_kv)]
    with ThreadPoolExecutor(max(1, min(len(slices), (os.cpu_count() or 1) // 2))) as ex:
        list(ex.map(one, slices))
    U.compare_output(out, ref, what=f"{name} whole output")
    gpu.close()


def test_full_llama2_7b_4k():
    _full_size("llama2_7b_4k")


def test_full_llama3_8b_gqa_32k():
    _full_size("llama3_8b_gqa_32k")


def test_full_long_128k():
    _full_size("long_128k")


def test_kivi4_serving_ragged_256_steps():
    """Ragged 4-bit serving batch: the cache is compared bit-exact at sampled
    steps (every flush and pop path is crossed), attention for sequences 0-3
    at every step and for all sequences at steps 0, 1, 63, 127, 128, 255."""
    w = W.WORKLOADS["kivi4_serving"]
    cap = w.capacity()
    p = Pair(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    Kh, Vh, lens = W.prefill_kv(w)
    p.prefill(Kh, Vh, lens)
    del Kh, Vh
    p.check_state("prefill", seqs=range(0, w.b, 9))
    first = [(i, qh) for i in range(4) for qh in range(w.h_q)]
    for s in range(w.steps):
        k, v = W.step_kv(w, s)
        p.append(k, v)
        q = W.step_q(w, s)
        if s in (0, 1, 63, 127, 128, 255):
            p.check_decode(q, f"step {s} all")
            p.check_state(f"step {s}", seqs=range(w.b))
        else:
            p.check_decode(q, f"step {s} seqs 0-3", pairs=first)
            if s % 16 == 5:
                p.check_state(f"step {s}", seqs=range(s % 7, w.b, 5))
