"""GPU parity of the attention-weight output (kivi_decode_attn_probs) against
the oracle's softmax weights: every token's weight of every (sequence, query
head) row, entries past a sequence's length untouched, the accumulated mass
over decode steps, and the attention output bitwise equal to the plain
decode call's.

Tolerance: a weight is 2^(s - M) / L with s an fp32 score whose error is a
few fp32 ulps of the dot product's terms; the relative error of a weight is
then about 1e-5 at the score ranges used here.  The bar is 1e-3 relative
(plus 1e-30 absolute for weights that underflow to subnormals), and each
row's weights sum to 1 within 1e-4.
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

RTOL_P = 1e-3
ATOL_P = 1e-30
SENTINEL = -7.25


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def compare_probs(gpu, ref, T, what=""):
    """gpu, ref: [b, hq, ld]; rows compared over [0, T_i)."""
    for i in range(gpu.shape[0]):
        n = int(T[i])
        g, r = gpu[i, :, :n].astype(np.float64), ref[i, :, :n].astype(np.float64)
        assert np.all(np.isfinite(g)), f"{what}: non-finite weights in sequence {i}"
        bad = np.abs(g - r) > RTOL_P * np.abs(r) + ATOL_P
        if bad.any():
            h, t = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: seq {i} head {h} token {t}: gpu {g[h, t]!r} oracle {r[h, t]!r}")
        if n:
            assert np.all(np.abs(g.sum(1) - 1.0) < 1e-4), f"{what}: seq {i} rows do not sum to 1"


def _probs_step(gpu, ora, q, ld, what, mass=None):
    """decode_probs on both sides; the GPU weights buffer starts as a
    sentinel that must survive past each sequence's length."""
    b, hq = q.shape[:2]
    probs = torch.full((b, hq, ld), SENTINEL, dtype=torch.float32, device="cuda")
    out = gpu.decode_probs(_dev(q), probs, mass=mass)
    plain = gpu.decode(_dev(q))
    assert torch.equal(out, plain), f"{what}: output differs from kivi_decode_attn"
    ref_out, ref_p = ora.decode_probs(q, ld=ld)
    U.compare_output(out.float().cpu().numpy(), ref_out, what)
    T = ora.lengths()[0]
    gp = probs.cpu().numpy()
    compare_probs(gp, ref_p, T, what)
    for i in range(b):
        assert np.all(gp[i, :, int(T[i]):] == SENTINEL), f"{what}: seq {i} written past its length"
    return ref_p


CASES = [
    # b, h, hq, d, kb, vb, G, R, lens, appends
    (3, 2, 2, 64, 2, 2, 32, 32, [0, 1, 31], 70),
    (4, 1, 8, 128, 4, 4, 32, 128, [127, 128, 129, 256], 140),
    (2, 2, 6, 128, 4, 2, 16, 48, [47, 96], 60),
    (2, 1, 3, 256, 2, 2, 64, 128, [300, 64], 135),
    (2, 2, 4, 128, 2, 2, 128, 128, [511, 128], 130),
    (1, 1, 1, 64, 4, 4, 16, 16, [5], 50),
]


@pytest.mark.parametrize("case", CASES, ids=[f"probs{i}" for i in range(len(CASES))])
def test_probs_ragged(case):
    """Ragged batches, MHA and GQA, every bit width, G and head dimension;
    weights after prefill and at sampled steps across key flushes and value
    pops (tokens quantized and fp16, blocks whole and partial)."""
    b, h, hq, d, kb, vb, G, R, lens, appends = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))
    cap = max(lens) + appends + 3
    gpu = K.KiviCache(b, h, d, kb, vb, G, R, cap)
    ora = oracle.Cache(b, h, d, kb, vb, G, R, cap)
    Kh = (rng.standard_normal((b, h, max(lens + [1]), d)) * 3).astype(np.float16)
    Vh = rng.standard_normal((b, h, max(lens + [1]), d)).astype(np.float16)
    gpu.prefill(_dev(Kh), _dev(Vh), np.array(lens, np.int32))
    ora.prefill(Kh, Vh, np.array(lens, np.int32))
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    _probs_step(gpu, ora, q, cap + 5, "prefill")
    for s in range(appends):
        k = (rng.standard_normal((b, h, d)) * 3).astype(np.float16)
        v = rng.standard_normal((b, h, d)).astype(np.float16)
        gpu.append(_dev(k), _dev(v))
        ora.append(k, v)
        if s % 11 == 0 or s == appends - 1:
            q = rng.standard_normal((b, hq, d)).astype(np.float16)
            _probs_step(gpu, ora, q, cap, f"step {s}")
    gpu.close()


@pytest.mark.parametrize("pad", [0, 3])
def test_mass_accumulates_over_steps(pad):
    """mass += weights at every step (the accumulated-attention score):
    after 150 steps of a ragged GQA batch it equals the sum of the oracle's
    per-step weights, token by token, with zeros past each length.  Rows of
    a multiple of 4 floats take the vector path, the odd width the scalar
    one."""
    b, h, hq, d, kb, vb, G, R = 3, 2, 8, 128, 2, 2, 32, 64
    lens = [200, 0, 333]
    steps = 150
    rng = np.random.default_rng(4242)
    cap = max(lens) + steps + 1 + pad
    gpu = K.KiviCache(b, h, d, kb, vb, G, R, cap)
    ora = oracle.Cache(b, h, d, kb, vb, G, R, cap)
    Kh = (rng.standard_normal((b, h, max(lens), d)) * 2).astype(np.float16)
    Vh = rng.standard_normal((b, h, max(lens), d)).astype(np.float16)
    gpu.prefill(_dev(Kh), _dev(Vh), np.array(lens, np.int32))
    ora.prefill(Kh, Vh, np.array(lens, np.int32))
    mass = torch.zeros((b, hq, cap), dtype=torch.float32, device="cuda")
    probs = torch.empty_like(mass)
    ref = np.zeros((b, hq, cap), np.float64)
    for s in range(steps):
        k = (rng.standard_normal((b, h, d)) * 2).astype(np.float16)
        v = rng.standard_normal((b, h, d)).astype(np.float16)
        q = rng.standard_normal((b, hq, d)).astype(np.float16)
        gpu.append(_dev(k), _dev(v))
        ora.append(k, v)
        gpu.decode_probs(_dev(q), probs, mass=mass)
        ref += ora.decode_probs(q, ld=cap)[1]
    got = mass.cpu().numpy().astype(np.float64)
    T = ora.lengths()[0]
    for i in range(b):
        n = int(T[i])
        err = np.abs(got[i, :, :n] - ref[i, :, :n])
        assert np.all(err <= RTOL_P * ref[i, :, :n] + 1e-6), f"seq {i}: max error {err.max():.3e}"
        assert not got[i, :, n:].any()
        # every step adds one unit of attention to each head's row
        np.testing.assert_allclose(got[i].sum(1), steps, rtol=1e-4)
    gpu.close()


def test_probs_full_llama3_8b_gqa_32k_sampled():
    """The 32k GQA workload at full size: sampled (sequence, kv head) slices
    against the oracle token by token; every row sums to 1."""
    w = W.WORKLOADS["llama3_8b_gqa_32k"]
    cap = w.capacity()
    gpu = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    Kh, Vh, lens = W.prefill_kv(w)
    gpu.prefill(_dev(Kh), _dev(Vh), lens)
    del Kh, Vh
    k, v = W.step_kv(w, 0)
    gpu.append(_dev(k), _dev(v))
    q = W.step_q(w, 0)
    T = gpu.lengths()[0]
    ld = int(T.max())
    probs = torch.full((w.b, w.h_q, ld), SENTINEL, dtype=torch.float32, device="cuda")
    out = gpu.decode_probs(_dev(q), probs)
    assert torch.equal(out, gpu.decode(_dev(q)))
    gp = probs.cpu().numpy()
    for i in range(w.b):
        n = int(T[i])
        assert np.all(np.abs(gp[i, :, :n].astype(np.float64).sum(1) - 1.0) < 1e-4)
    hg = w.group
    for (i, j) in [(0, 0), (3, 5), (7, 7)]:
        n = int(lens[i])
        ora = oracle.Cache(1, 1, w.d, w.kbits, w.vbits, w.G, w.R, cap)
        ora.prefill(W.prefill_slice(w, "K", i, j, n)[None, None], W.prefill_slice(w, "V", i, j, n)[None, None],
                    [n])
        ora.append(k[i:i + 1, j:j + 1], v[i:i + 1, j:j + 1])
        qs = np.ascontiguousarray(q[i:i + 1, j * hg:(j + 1) * hg])
        _, ref = ora.decode_probs(qs, ld=ld)
        compare_probs(gp[i:i + 1, j * hg:(j + 1) * hg], ref, [int(T[i])], f"seq {i} head {j}")
    gpu.close()


def test_probs_argument_errors():
    d = 64
    gpu = K.KiviCache(2, 1, d, 2, 2, 32, 32, 100)
    x = _dev(np.ones((2, 1, 90, d), np.float16))
    gpu.prefill(x, x, [90, 40])
    q = _dev(np.ones((2, 2, d), np.float16))
    with pytest.raises(K.KiviError):   # a row shorter than a sequence
        gpu.decode_probs(q, torch.zeros((2, 2, 89), dtype=torch.float32, device="cuda"))
    p = torch.zeros((2, 2, 90), dtype=torch.float32, device="cuda")
    with pytest.raises(K.KiviError):   # the same buffer twice
        gpu.decode_probs(q, p, mass=p)
    with pytest.raises(TypeError):
        gpu.decode_probs(q, p.half())
    with pytest.raises(ValueError):
        gpu.decode_probs(q, torch.zeros((2, 3, 90), dtype=torch.float32, device="cuda"))
    gpu.decode_probs(q, p)
    np.testing.assert_allclose(p.sum(2).cpu().numpy(), 1.0, rtol=1e-5)
    gpu.close()


def test_probs_unaligned_buffers():
    """Buffers that start off a 16-byte boundary (a view one float in) take
    the one-token-at-a-time path and give the same weights and mass."""
    b, h, hq, d = 2, 2, 4, 128
    rng = np.random.default_rng(77)
    gpu = K.KiviCache(b, h, d, 2, 2, 32, 128, 5000)
    Kh = rng.standard_normal((b, h, 4500, d)).astype(np.float16)
    Vh = rng.standard_normal((b, h, 4500, d)).astype(np.float16)
    gpu.prefill(_dev(Kh), _dev(Vh), [4500, 4099])
    q = _dev(rng.standard_normal((b, hq, d)).astype(np.float16))
    ld = 4502
    n = b * hq * ld
    pa = torch.zeros((b, hq, ld), dtype=torch.float32, device="cuda")
    ma = torch.ones_like(pa)
    pu = torch.zeros(n + 1, dtype=torch.float32, device="cuda")[1:].view(b, hq, ld)
    mu = torch.ones(n + 1, dtype=torch.float32, device="cuda")[1:].view(b, hq, ld)
    assert pu.data_ptr() % 16 and mu.data_ptr() % 16
    gpu.decode_probs(q, pa, mass=ma)
    gpu.decode_probs(q, pu, mass=mu)
    assert torch.equal(pa, pu) and torch.equal(ma, mu)
    np.testing.assert_allclose(pa.sum(2).cpu().numpy(), 1.0, rtol=1e-5)
    gpu.close()
