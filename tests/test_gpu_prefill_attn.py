"""GPU parity of kivi_prefill_attn: the prompt's causal attention (fp16
inputs, fp32 scores, fp16 softmax weights in the value product) against the
oracle's double-precision causal attention, within 2e-3 max-abs and 1e-3
relative L2 over the valid rows; and the cache it leaves, bitwise against
kivi_prefill's and the oracle's."""
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
    import os
    oracle.set_threads(os.cpu_count() or 1)


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _compare_rows(got, ref, lens, what):
    """got, ref: [b, hq, ts, d]; compare the rows tau < lens[i] as one output."""
    g = np.concatenate([got[i, :, :n].reshape(-1, got.shape[-1]) for i, n in enumerate(lens) if n])
    r = np.concatenate([ref[i, :, :n].reshape(-1, ref.shape[-1]) for i, n in enumerate(lens) if n])
    return U.compare_output(g, r, what)


CASES = [
    # b, h_kv, h_q, d, k_bits, v_bits, G, R, lens
    (2, 2, 4, 64, 2, 2, 32, 32, [100, 1]),
    (1, 2, 2, 128, 4, 4, 16, 64, [257]),
    (3, 1, 8, 128, 2, 4, 64, 128, [0, 64, 600]),
    (2, 4, 8, 128, 2, 2, 32, 128, [1000, 777]),
    (2, 2, 6, 64, 4, 2, 16, 32, [63, 65]),
    (1, 1, 6, 128, 2, 2, 32, 128, [300]),      # d 128, even group: two query heads a CTA
    (2, 2, 6, 128, 4, 2, 32, 64, [200, 129]),  # d 128, odd group: two query tiles of one head a CTA
    (2, 2, 2, 128, 2, 4, 32, 64, [1000, 517]),  # MHA, longer: two query tiles a CTA, its four diagonal tiles packed
]


@pytest.mark.parametrize("case", CASES, ids=[f"pa{i}" for i in range(len(CASES))])
def test_prefill_attn_parity(case):
    b, h, hq, d, kb, vb, G, R, lens = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))
    ts = max(max(lens), 1) + 5
    Q = (rng.standard_normal((b, hq, ts, d)) * 1.5).astype(np.float16)
    Kh = (rng.standard_normal((b, h, ts, d)) * 1.5).astype(np.float16)
    Vh = rng.standard_normal((b, h, ts, d)).astype(np.float16)
    Kh[:, :, :, 3] *= 8   # an outlier channel
    t = np.array(lens, np.int32)
    cap = max(max(lens), 1) + 8
    a = K.KiviCache(b, h, d, kb, vb, G, R, cap)
    out = torch.full((b, hq, ts, d), 7.0, dtype=torch.float16, device="cuda")   # sentinel past each length
    a.prefill_attn(_dev(Q), _dev(Kh), _dev(Vh), t, out=out)
    got = out.float().cpu().numpy()
    ref = oracle.prefill_attention(Q, Kh, Vh, t)
    _compare_rows(got, ref, lens, f"prefill attention {case}")
    for i, n in enumerate(lens):
        assert np.all(got[i, :, n:] == 7.0), "rows past the length were written"
    # the cache: bitwise kivi_prefill's, and the oracle's
    p = K.KiviCache(b, h, d, kb, vb, G, R, cap)
    p.prefill(_dev(Kh), _dev(Vh), t)
    ea, ep = a.export(), p.export()
    for key in ea:
        assert np.array_equal(ea[key], ep[key]), key
    assert all(np.array_equal(x, y) for x, y in zip(a.lengths(), p.lengths()))
    o = oracle.Cache(b, h, d, kb, vb, G, R, cap)
    o.prefill(Kh, Vh, t)
    g = U.geometry(b, h, d, kb, vb, G, R, cap)
    oex = o.export()
    T, Tqk, Tqv = o.lengths()
    for i in range(b):
        for j in range(h):
            U.compare_slice(ea, g, i, j, oex, g, i, j, int(T[i]), int(Tqk[i]), int(Tqv[i]), what=f"{case} {i} {j}")
    # the cache decodes as the oracle does
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    U.compare_output(a.decode(_dev(q)).float().cpu().numpy(), o.decode(q), f"decode after {case}")
    assert a.check() == 0
    for c in (a, p):
        c.close()
    o.close()


def test_prefill_attn_unsupported_shapes():
    for d, G in ((256, 32), (128, 128)):
        c = K.KiviCache(1, 1, d, 2, 2, G, 128, 256)
        x = torch.zeros((1, 1, 64, d), dtype=torch.float16, device="cuda")
        with pytest.raises(K.KiviError):
            c.prefill_attn(x, x, x, [64])
        c.close()


def test_prefill_attn_full_llama3_8b_gqa_32k():
    """The 32k GQA workload at full size: sampled rows (the first, the tile
    edges, the last, random ones) of every (sequence, query head) against
    the oracle; the cache bitwise against kivi_prefill's."""
    w = W.WORKLOADS["llama3_8b_gqa_32k"]
    Kh, Vh, lens = W.prefill_kv(w)
    Q = W.prefill_q(w)
    cap = int(lens.max()) + 8
    a = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    out = a.prefill_attn(_dev(Q), _dev(Kh), _dev(Vh), lens)
    rng = np.random.default_rng(7)
    rows = []
    for i in range(w.b):
        n = int(lens[i])
        for qh in range(w.h_q):
            taus = {0, 63, 64, 65, n // 2, n - 65, n - 1} | set(rng.integers(0, n, 3).tolist())
            rows += [(i, qh, tau) for tau in sorted(taus)]
    rows = np.array(rows, np.int32)
    ref = oracle.prefill_attention(Q, Kh, Vh, lens, rows=rows)
    ix = torch.from_numpy(rows.astype(np.int64)).cuda()
    g = out[ix[:, 0], ix[:, 1], ix[:, 2]].float().cpu().numpy()
    del out
    U.compare_output(g, ref, "prefill attention 32k sampled rows")
    p = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    p.prefill(_dev(Kh), _dev(Vh), lens)
    ea, ep = a.export(), p.export()
    for key in ea:
        assert np.array_equal(ea[key], ep[key]), key
    assert a.check() == 0
    a.close()
    p.close()


def test_prefill_attn_all_empty():
    """Every sequence empty: nothing attended, the counters reset, and a
    decode afterwards writes zero outputs (as after kivi_prefill)."""
    c = K.KiviCache(2, 2, 64, 2, 2, 32, 32, 128)
    x = torch.zeros((2, 2, 4, 64), dtype=torch.float16, device="cuda")
    c.prefill_attn(x, x, x, [0, 0])
    assert all(not np.any(a) for a in c.lengths())
    out = c.decode(torch.ones((2, 2, 64), dtype=torch.float16, device="cuda"))
    assert not out.float().abs().sum().item()
    assert c.check() == 0
    c.close()


RISING = [
    # b, h_kv, h_q, d, lens: one variant of the kernel each
    (1, 1, 2, 64, [700]),    # d 64: one slot a CTA
    (1, 1, 2, 128, [700]),   # two query heads a CTA
    (1, 1, 3, 128, [700]),   # two query tiles of one head a CTA
]


@pytest.mark.parametrize("case", RISING, ids=[f"rise{i}" for i in range(len(RISING))])
def test_prefill_attn_rising_scores(case):
    """Keys of the first 64-token tile are zero, so a row's maximum score
    starts at 0 and jumps on a later tile: the kernel then rescales O and
    the row sum (it does so only when the maximum grows by more than 8 in
    log2 units), after the previous tile's P V and before the next.  The
    case is checked to reach that branch on many rows before the GPU runs
    it.  (Keys whose scale keeps rising along the prompt make late rows so
    peaked that the fp16 weights' rounding alone comes to the tolerance: an
    emulation of the kernel's arithmetic gives 2.2e-3 there.)"""
    b, h, hq, d, lens = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))
    ts = max(lens) + 5
    Q = (rng.standard_normal((b, hq, ts, d)) * 1.5).astype(np.float16)
    scale = np.where(np.arange(ts) < 64, 0.0, 1.0)[None, None, :, None]
    Kh = (rng.standard_normal((b, h, ts, d)) * 1.5 * scale).astype(np.float16)
    Vh = rng.standard_normal((b, h, ts, d)).astype(np.float16)
    t = np.array(lens, np.int32)
    # precondition: the running maximum of raw scores, taken over whole
    # 64-key tiles, grows by more than 8 / (log2(e) / sqrt(d)) on many rows
    lim = 8.0 * np.sqrt(d) / np.log2(np.e)
    n, grows, rows = lens[0], 0, 0
    for qh in range(hq):
        s = Q[0, qh, :n].astype(np.float64) @ Kh[0, qh * h // hq, :n].astype(np.float64).T
        for tau in range(128, n, 7):
            m = s[tau, :64].max()
            rows += 1
            for k0 in range(64, tau + 1, 64):
                mt = s[tau, k0:min(k0 + 64, tau + 1)].max()
                if mt - m > lim:
                    grows += 1
                    break
                m = max(m, mt)
    assert grows > rows // 5, (grows, rows)
    cap = max(lens) + 8
    a = K.KiviCache(b, h, d, 2, 2, 32, 64, cap)
    out = a.prefill_attn(_dev(Q), _dev(Kh), _dev(Vh), t)
    got = out.float().cpu().numpy()
    ref = oracle.prefill_attention(Q, Kh, Vh, t)
    _compare_rows(got, ref, lens, f"prefill attention, rising scores {case}")
    assert a.check() == 0
    a.close()
