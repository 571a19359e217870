"""Pins for the CPU oracle: checks against facts the pages and mathematics fix,
never against a retyped copy of the oracle's own formulas.

Source of every fact: "Literature audit -- Group 2", section 1 KIVI, list
"Core algorithm (implementation-grade)", items 1-5.
"""
import os

import numpy as np
import pytest

import oracle
from bit_quantized_kv_quantize_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# fp16 conversion: numpy's converter is an independent implementation.
# --------------------------------------------------------------------------

def test_f16_to_f32_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f32_to_f16_matches_numpy_rne():
    rng = np.random.default_rng(1)
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
    fin = allh[np.isfinite(allh)].astype(np.float32)
    # exact fp16 values, their fp32 neighbours, and midpoints (ties)
    up = np.nextafter(fin, np.float32(np.inf))
    dn = np.nextafter(fin, np.float32(-np.inf))
    srt = np.unique(fin.astype(np.float64))
    mids = ((srt[1:] + srt[:-1]) / 2).astype(np.float32)
    rand = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(100000) * 1e-5).astype(np.float32),
        (rng.standard_normal(100000) * 3e4).astype(np.float32),
        np.array([65504, 65519.99, 65520, 70000, 2.0**-25, 2.0**-25 * 1.0001, 2.0**-26,
                  1e-40, -1e-40, 3.0e38], np.float32),
    ])
    x = np.concatenate([fin, up, dn, mids, np.nextafter(mids, np.float32(0)),
                        np.nextafter(mids, np.float32(np.inf)), rand])
    ours = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------
# Item 1: the quantizer.
# --------------------------------------------------------------------------

def _read_quant_golden():
    rows = []
    with open(os.path.join(GOLDEN, "quantizer_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, xs, s16, z16, codes, _ = [p.strip() for p in line.split("|")]
            rows.append((int(bits), np.array([float(v) for v in xs.split()], np.float32),
                         int(s16, 16), int(z16, 16), [int(c) for c in codes.split()]))
    return rows


@pytest.mark.parametrize("row", _read_quant_golden())
def test_quantizer_hand_worked_examples(row):
    bits, x, s16, z16, codes = row
    assert np.array_equal(x.astype(np.float16).astype(np.float32), x)
    s, z, c = oracle.quantize_group(x, bits)
    assert (s, z) == (s16, z16)
    assert c.tolist() == codes


def _groups(rng, n, G):
    """Many groups with varied ranges, offsets, outliers, tiny and zero spreads."""
    out = []
    for k in range(n):
        kind = k % 6
        if kind == 0:
            x = rng.standard_normal(G)
        elif kind == 1:
            x = rng.standard_normal(G) * 10.0 ** rng.integers(-4, 4) + rng.standard_normal() * 100
        elif kind == 2:
            x = rng.standard_normal(G)
            x[rng.integers(G)] *= 40
        elif kind == 3:
            x = np.full(G, rng.standard_normal())
        elif kind == 4:
            x = rng.standard_normal(G) * 1e-6
        else:
            x = rng.uniform(-3e4, 3e4, G)
        out.append(x.astype(np.float16).astype(np.float32))
    return out


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_invariants(bits):
    """Item 1 fixes: min gets code 0 and dequantizes to min exactly; max gets
    the top code; every element is within half a step of its dequantized
    value; the stored scale is the fp16 nearest (max - min)/(2^B - 1)."""
    rng = np.random.default_rng(bits)
    qmax = 2 ** bits - 1
    for x in _groups(rng, 3000, 32):
        s16, z16, codes = oracle.quantize_group(x, bits)
        sf = float(np.uint16(s16).view(np.float16))
        zf = float(np.uint16(z16).view(np.float16))
        mn, mx = float(x.min()), float(x.max())
        assert zf == mn
        exact = (mx - mn) / qmax
        if sf == 0.0:
            assert np.all(codes == 0)
            assert exact <= 2.0 ** -25   # only a spread below half an fp16 unit rounds to 0
            continue
        # fp16 nearest: relative 2^-11 in the normal range, 2^-25 absolute below it
        assert abs(sf - exact) <= max(2.0 ** -11 * exact, 2.0 ** -25) * (1 + 1e-12)
        assert np.all(codes[x == mn] == 0)
        xhat = codes.astype(np.float64) * sf + zf
        if sf >= 2.0 ** -14:   # normal scale: the bound of item 1
            assert np.all(codes[x == mx] == qmax)
            assert np.all(np.abs(x - xhat) <= sf / 2 * (1 + 1e-6) + 1e-7 * np.abs(x))
        else:                  # subnormal scale: clamped top, error <= 3 exact steps
            assert np.all(np.abs(x - xhat) <= 3 * exact + 2.0 ** -24)


@pytest.mark.parametrize("bits", [2, 4])
def test_quantizer_brute_force_nearest(bits):
    """Brute force over all pairs of a small fp16 grid: each code is the
    nearest point of the grid {z + c s} (ties: the even code)."""
    qmax = 2 ** bits - 1
    vals = np.unique(np.array([-2, -1.5, -1, -0.75, -0.5, -0.3, 0, 0.1, 0.25, 0.3, 0.5, 0.7, 1,
                               1.25, 2, 3, 5.5], np.float16).astype(np.float32))
    for a in vals:
        for b in vals:
            for c in vals:
                x = np.array([a, b, c], np.float32)
                s16, z16, codes = oracle.quantize_group(x, bits)
                sf = float(np.uint16(s16).view(np.float16))
                zf = float(np.uint16(z16).view(np.float16))
                if sf == 0:
                    assert np.all(codes == 0)
                    continue
                grid = zf + np.arange(qmax + 1) * sf
                for xi, ci in zip(x.astype(np.float64), codes):
                    dist = np.abs(grid - xi)
                    best = dist.min()
                    cands = np.nonzero(np.abs(dist - best) <= 1e-9 * max(1, abs(xi)))[0]
                    want = cands[0] if len(cands) == 1 else [k for k in cands if k % 2 == 0][0]
                    assert ci == want, (x, ci, want)


def test_quantizer_on_grid_roundtrip():
    """Values already on a power-of-two grid (min and max present) reproduce exactly."""
    rng = np.random.default_rng(7)
    for bits in (2, 4):
        qmax = 2 ** bits - 1
        for _ in range(500):
            s = 2.0 ** rng.integers(-8, 4)
            z = float(np.float16(rng.integers(-64, 64) * s))
            k = rng.integers(0, qmax + 1, 32)
            k[0], k[1] = 0, qmax
            x = (z + k * s).astype(np.float32)
            if not np.array_equal(x.astype(np.float16).astype(np.float32), x):
                continue
            s16, z16, codes = oracle.quantize_group(x, bits)
            assert np.array_equal(codes, k)
            xhat = np.array([oracle.dequant(int(ci), s16, z16) for ci in codes], np.float32)
            assert np.array_equal(xhat, x)


# --------------------------------------------------------------------------
# Items 2-4: cache state, grouping and the residual schedule.
# --------------------------------------------------------------------------

def _cache_with(b, h, d, kb, vb, G, R, cap, lens, seed=0, key_scale=None):
    rng = np.random.default_rng(seed)
    ts = max(1, int(max(lens)))
    K = rng.standard_normal((b, h, ts, d)).astype(np.float32)
    V = rng.standard_normal((b, h, ts, d)).astype(np.float32)
    if key_scale is not None:
        K *= key_scale
    K, V = K.astype(np.float16), V.astype(np.float16)
    c = oracle.Cache(b, h, d, kb, vb, G, R, cap)
    c.prefill(K, V, np.asarray(lens, np.int32))
    return c, K, V


@pytest.mark.parametrize("t,R", [(0, 32), (1, 32), (31, 32), (32, 32), (33, 32), (64, 32),
                                 (100, 32), (256, 32), (300, 128), (4096, 128), (127, 128)])
def test_prefill_split(t, R):
    """Item 4: prefill quantizes keys [0, t - t mod R) and values [0, max(t - R, 0))."""
    c, K, V = _cache_with(1, 2, 64, 2, 2, 32, R, max(t, 1) + 8, [t])
    T, Tqk, Tqv = c.lengths()
    assert (T[0], Tqk[0], Tqv[0]) == (t, t - t % R, max(t - R, 0))
    st = c.state()
    # the fp16 windows hold the raw tails, in token order
    nk, nv = t - Tqk[0], t - Tqv[0]
    assert np.array_equal(st["kf"][0, :, :nk], K[0, :, Tqk[0]:t].view(np.uint16))
    assert np.array_equal(st["vf"][0, :, :nv], V[0, :, Tqv[0]:t].view(np.uint16))


def test_grouping_axes():
    """Item 2: one (s, z) per channel per G tokens; item 3: one per token per G
    channels.  Scaling every key token group and every value channel group by
    a different power of ten makes any other grouping violate the error bound."""
    b, h, d, G, R, t = 1, 1, 64, 32, 32, 256
    tok_scale = 10.0 ** np.repeat(np.arange(t // G) % 5 - 2, G)            # per token group
    ch_scale = 10.0 ** (np.arange(d) // G * 2 - 1.0)                        # per channel group
    rng = np.random.default_rng(3)
    K = (rng.standard_normal((b, h, t, d)) * tok_scale[None, None, :, None]).astype(np.float16)
    V = (rng.standard_normal((b, h, t, d)) * ch_scale[None, None, None, :]).astype(np.float16)
    c = oracle.Cache(b, h, d, 2, 2, G, R, t + 8)
    c.prefill(K, V, [t])
    Kh, Vh = c.dequant_kv(0, 0)
    Kr, Vr = K[0, 0].astype(np.float64), V[0, 0].astype(np.float64)
    # per-group half-step bound with the group's own range
    for g in range(t // G):
        blk = Kr[g * G:(g + 1) * G]
        step = (blk.max(0) - blk.min(0)) / 3
        err = np.abs(Kh[g * G:(g + 1) * G] - blk)
        assert np.all(err <= step / 2 * 1.002 + 1e-7), g
    nqv = t - R
    for gi in range(d // G):
        blk = Vr[:nqv, gi * G:(gi + 1) * G]
        step = (blk.max(1) - blk.min(1)) / 3
        err = np.abs(Vh[:nqv, gi * G:(gi + 1) * G] - blk)
        assert np.all(err <= step[:, None] / 2 * 1.002 + 1e-7), gi
    # fp16 tail reproduced exactly
    assert np.array_equal(Vh[nqv:], Vr[nqv:].astype(np.float32))


def _flush_closed_form(t, R, n):
    """Append n (1-based) starts with a key flush iff the key buffer then holds
    R keys: n >= 2 and (t + n - 1) % R == 0 (item 4)."""
    return n >= 2 and (t + n - 1) % R == 0


def _pop_closed_form(t, R, n):
    """Append n starts with a value pop iff the queue then holds R + 1 tokens:
    min(t, R) + n - 1 >= R + 1 (item 4)."""
    return min(t, R) + n - 1 >= R + 1


@pytest.mark.parametrize("t,R", [(0, 32), (5, 4), (31, 32), (32, 32), (100, 32), (256, 64),
                                 (129, 128)])
def test_residual_schedule_closed_form(t, R):
    G = 32 if R % 32 == 0 else R
    c, _, _ = _cache_with(1, 1, 64, 2, 2, G, R, t + 3 * R + 8, [t])
    rng = np.random.default_rng(11)
    prev = [int(x[0]) for x in c.lengths()]
    for n in range(1, 3 * R + 3):
        k = rng.standard_normal((1, 1, 64)).astype(np.float16)
        v = rng.standard_normal((1, 1, 64)).astype(np.float16)
        c.append(k, v)
        T, Tqk, Tqv = [int(x[0]) for x in c.lengths()]
        assert T == prev[0] + 1
        assert (Tqk - prev[1] == R) == _flush_closed_form(t, R, n)
        assert Tqk - prev[1] in (0, R)
        assert (Tqv - prev[2] == 1) == _pop_closed_form(t, R, n)
        # invariants of item 4 after every append: Tqk a multiple of R,
        # 1 <= |Kf| <= R, 1 <= |Vf| <= R + 1
        assert Tqk % R == 0 and 1 <= T - Tqk <= R and 1 <= T - Tqv <= R + 1
        prev = [T, Tqk, Tqv]


def _reference_order_counts(t, R, steps):
    """Restates item 4 in the reference order: push the new token, attend,
    then flush the key block if it holds R keys and pop one value if the queue
    holds R + 1.  Returns the counts after each step's maintenance."""
    T, nk, nv = t, t % R, min(t, R)
    qk, qv = t - t % R, max(t - R, 0)
    out = []
    for _ in range(steps):
        T += 1
        nk += 1
        nv += 1
        if nk == R:
            qk += R
            nk = 0
        if nv == R + 1:
            qv += 1
            nv -= 1
        out.append((T, qk, qv))
    return out


@pytest.mark.parametrize("t,R", [(0, 32), (7, 32), (32, 32), (95, 32), (300, 64)])
def test_lazy_maintenance_matches_reference_order(t, R):
    """Maintenance deferred to the next append leaves the same quantized set
    as maintenance right after each step's attention."""
    ref = _reference_order_counts(t, R, 4 * R)
    c, _, _ = _cache_with(1, 1, 64, 2, 2, 32, R, t + 4 * R + 8, [t])
    rng = np.random.default_rng(5)
    for n in range(4 * R):
        c.append(rng.standard_normal((1, 1, 64)).astype(np.float16),
                 rng.standard_normal((1, 1, 64)).astype(np.float16))
        if n >= 1:
            T, Tqk, Tqv = [int(x[0]) for x in c.lengths()]
            # the lazy state after append n+1 has applied step n's maintenance
            assert (Tqk, Tqv) == ref[n - 1][1:]


def test_flush_and_pop_quantize_the_right_tokens():
    """Keys flushed at R and values popped at R + 1 carry the codes of
    quantizing exactly those raw tokens (item 4 with items 1-3)."""
    b, h, d, G, R, t = 1, 1, 64, 32, 64, 100
    c, K, V = _cache_with(b, h, d, 2, 2, G, R, t + 300, [t], seed=9)
    rawk = [K[0, 0, i] for i in range(t)]
    rawv = [V[0, 0, i] for i in range(t)]
    rng = np.random.default_rng(10)
    for _ in range(250):
        k = (rng.standard_normal((1, 1, d)) * 3).astype(np.float16)
        v = rng.standard_normal((1, 1, d)).astype(np.float16)
        c.append(k, v)
        rawk.append(k[0, 0])
        rawv.append(v[0, 0])
    T, Tqk, Tqv = [int(x[0]) for x in c.lengths()]
    st = c.state()
    rk = np.stack(rawk).astype(np.float32)
    rv = np.stack(rawv).astype(np.float32)
    for g in range(Tqk // G):
        for ch in range(0, d, 7):
            s, z, codes = oracle.quantize_group(rk[g * G:(g + 1) * G, ch], 2)
            assert st["ks"][0, 0, g, ch] == s and st["kz"][0, 0, g, ch] == z
            assert np.array_equal(st["kcode"][0, 0, ch, g * G:(g + 1) * G], codes)
    for tok in range(0, Tqv, 13):
        for gi in range(d // G):
            s, z, codes = oracle.quantize_group(rv[tok, gi * G:(gi + 1) * G], 2)
            assert st["vs"][0, 0, tok, gi] == s and st["vz"][0, 0, tok, gi] == z
            assert np.array_equal(st["vcode"][0, 0, tok, gi * G:(gi + 1) * G], codes)
    # residual windows hold the raw newest tokens
    assert np.array_equal(st["kf"][0, 0, :T - Tqk].view(np.float16), np.stack(rawk[Tqk:T]))
    assert np.array_equal(st["vf"][0, 0, :T - Tqv].view(np.float16), np.stack(rawv[Tqv:T]))


def test_capacity_and_arguments():
    with pytest.raises(ValueError):
        oracle.Cache(1, 1, 64, 3, 2, 32, 32, 64)      # bits not in {2, 4}
    with pytest.raises(ValueError):
        oracle.Cache(1, 1, 64, 2, 2, 32, 48, 64)      # R % G != 0 (item 4's assertion)
    c = oracle.Cache(1, 1, 64, 2, 2, 32, 32, 10)
    z = np.zeros((1, 1, 10, 64), np.float16)
    c.prefill(z, z, [10])
    with pytest.raises(OverflowError):
        c.append(np.zeros((1, 1, 64), np.float16), np.zeros((1, 1, 64), np.float16))


# --------------------------------------------------------------------------
# Item 5: decode attention.
# --------------------------------------------------------------------------

def _dense_attention(q, K, V):
    """Textbook softmax(q K^T / sqrt(d)) V in fp64."""
    q, K, V = (np.asarray(a, np.float64) for a in (q, K, V))
    s = K @ q / np.sqrt(K.shape[1])
    p = np.exp(s - s.max())
    return p @ V / p.sum()


def test_attention_unquantized_equals_dense():
    """With R >= T nothing is quantized (item 4), so the result is plain
    softmax attention over the raw keys and values."""
    b, h, hq, d, G, R, t = 2, 2, 4, 64, 32, 256, 200
    c, K, V = _cache_with(b, h, d, 2, 2, G, R, t + 8, [t, 57])
    q = np.random.default_rng(2).standard_normal((b, hq, d)).astype(np.float16)
    out = c.decode(q)
    lens = [t, 57]
    for i in range(b):
        for qh in range(hq):
            j = qh // (hq // h)
            ref = _dense_attention(q[i, qh], K[i, j, :lens[i]], V[i, j, :lens[i]])
            np.testing.assert_allclose(out[i, qh], ref, rtol=2e-5, atol=2e-6)


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 4), (2, 4), (4, 2)])
def test_attention_equals_dense_over_dequantized(kb, vb):
    b, h, hq, d, G, R = 2, 2, 4, 64, 32, 32
    lens = [300, 77]
    c, K, V = _cache_with(b, h, d, kb, vb, G, R, 400, lens, seed=4)
    rng = np.random.default_rng(8)
    for _ in range(40):
        c.append(rng.standard_normal((b, h, d)).astype(np.float16),
                 rng.standard_normal((b, h, d)).astype(np.float16))
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    out = c.decode(q)
    for i in range(b):
        for qh in range(hq):
            Kh, Vh = c.dequant_kv(i, qh // (hq // h))
            ref = _dense_attention(q[i, qh], Kh, Vh)
            np.testing.assert_allclose(out[i, qh], ref, rtol=3e-5, atol=3e-6)


def test_attention_on_grid_inputs_equals_dense_over_raw():
    """Keys and values on a power-of-two grid, with every group spanning the
    full code range, quantize exactly; quantized attention then equals dense
    attention over the raw cache."""
    b, h, d, G, R, t = 1, 1, 64, 32, 32, 192
    rng = np.random.default_rng(12)
    K = rng.integers(0, 4, (t, d)).astype(np.float64)
    K[0::G, :] = 0
    K[1::G, :] = 3                      # each key group (G tokens of a channel) spans 0..3
    V = rng.integers(0, 4, (t, d)).astype(np.float64)
    V[:, 0::G] = 0
    V[:, 1::G] = 3                      # each value group (G channels of a token) spans 0..3
    K = (K * 0.25 - 0.5).astype(np.float16)[None, None]
    V = (V * 0.5 + 1.0).astype(np.float16)[None, None]
    c = oracle.Cache(b, h, d, 2, 2, G, R, t + 4)
    c.prefill(K, V, [t])
    assert c.lengths()[1][0] == t and c.lengths()[2][0] == t - R
    Kh, Vh = c.dequant_kv(0, 0)
    assert np.array_equal(Kh, K[0, 0].astype(np.float32))
    assert np.array_equal(Vh, V[0, 0].astype(np.float32))
    q = rng.standard_normal((1, 1, d)).astype(np.float16)
    out = c.decode(q)
    np.testing.assert_allclose(out[0, 0], _dense_attention(q[0, 0], K[0, 0], V[0, 0]),
                               rtol=2e-5, atol=2e-6)


def test_gqa_equals_mha_with_repeated_kv():
    """Query head i reads kv head i / (h_q / h_kv): identical to MHA over kv
    heads repeated h_q / h_kv times."""
    b, h, hq, d, G, R, t = 1, 2, 8, 64, 32, 32, 160
    rng = np.random.default_rng(13)
    K = rng.standard_normal((b, h, t, d)).astype(np.float16)
    V = rng.standard_normal((b, h, t, d)).astype(np.float16)
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    g = oracle.Cache(b, h, d, 2, 2, G, R, t + 4)
    g.prefill(K, V, [t])
    m = oracle.Cache(b, hq, d, 2, 2, G, R, t + 4)
    m.prefill(np.repeat(K, hq // h, axis=1), np.repeat(V, hq // h, axis=1), [t])
    assert np.array_equal(g.decode(q), m.decode(q))


def test_attention_special_cases():
    d = 64
    # one token: the output is that token's value
    c = oracle.Cache(1, 1, d, 2, 2, 32, 32, 8)
    V = np.random.default_rng(1).standard_normal((1, 1, 1, d)).astype(np.float16)
    c.prefill(np.zeros_like(V), V, [1])
    q = np.ones((1, 1, d), np.float16)
    assert np.array_equal(c.decode(q)[0, 0], V[0, 0, 0].astype(np.float32))
    # no tokens: defined as zero output
    e = oracle.Cache(1, 1, d, 2, 2, 32, 32, 8)
    e.prefill(np.zeros((1, 1, 1, d), np.float16), np.zeros((1, 1, 1, d), np.float16), [0])
    assert np.array_equal(e.decode(q), np.zeros((1, 1, d), np.float32))
    # equal keys: the output is the mean of the values
    c2 = oracle.Cache(1, 1, d, 2, 2, 32, 32, 8)
    V2 = np.random.default_rng(2).standard_normal((1, 1, 4, d)).astype(np.float16)
    c2.prefill(np.ones((1, 1, 4, d), np.float16), V2, [4])
    np.testing.assert_allclose(c2.decode(q)[0, 0], V2[0, 0].astype(np.float64).mean(0), rtol=1e-6,
                               atol=1e-7)


def _dense_weights(q, K):
    """Textbook softmax(q K^T / sqrt(d)) weights in fp64."""
    s = np.asarray(K, np.float64) @ np.asarray(q, np.float64) / np.sqrt(K.shape[1])
    p = np.exp(s - s.max())
    return p / p.sum()


def test_probs_unquantized_equal_dense_weights():
    """With R >= T nothing is quantized: each row of weights is the plain
    softmax over the raw keys, summing to 1, zeros after T_i."""
    b, h, hq, d, G, R, t = 2, 2, 4, 64, 32, 256, 200
    lens = [t, 57]
    c, K, V = _cache_with(b, h, d, 2, 2, G, R, t + 8, lens)
    q = np.random.default_rng(2).standard_normal((b, hq, d)).astype(np.float16)
    out, probs = c.decode_probs(q, ld=t + 5)
    assert np.array_equal(out, c.decode(q))
    for i in range(b):
        for qh in range(hq):
            j = qh // (hq // h)
            ref = _dense_weights(q[i, qh], K[i, j, :lens[i]])
            np.testing.assert_allclose(probs[i, qh, :lens[i]], ref, rtol=2e-5, atol=1e-9)
            assert abs(float(probs[i, qh, :lens[i]].astype(np.float64).sum()) - 1.0) < 1e-5
            assert not probs[i, qh, lens[i]:].any()


@pytest.mark.parametrize("kb,vb", [(2, 2), (4, 2)])
def test_probs_over_dequantized_and_consistent_with_output(kb, vb):
    """After prefill and appends (quantized and fp16 tokens mixed): the
    weights are the dense softmax over the dequantized keys, and weights
    times dequantized values give the attention output (token by token, so
    a shifted or swapped token index fails)."""
    b, h, hq, d, G, R = 2, 2, 8, 64, 32, 32
    lens = [300, 77]
    c, K, V = _cache_with(b, h, d, kb, vb, G, R, 400, lens, seed=5)
    rng = np.random.default_rng(9)
    for _ in range(37):
        c.append(rng.standard_normal((b, h, d)).astype(np.float16),
                 rng.standard_normal((b, h, d)).astype(np.float16))
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    out, probs = c.decode_probs(q)
    T = c.lengths()[0]
    for i in range(b):
        for qh in range(hq):
            Kh, Vh = c.dequant_kv(i, qh // (hq // h))
            ref = _dense_weights(q[i, qh], Kh)
            np.testing.assert_allclose(probs[i, qh, :T[i]], ref, rtol=3e-5, atol=1e-9)
            np.testing.assert_allclose(probs[i, qh, :T[i]].astype(np.float64) @ Vh, out[i, qh],
                                       rtol=1e-4, atol=1e-5)


def test_probs_special_cases():
    d = 64
    q = np.ones((1, 1, d), np.float16)
    # one token: weight 1
    c = oracle.Cache(1, 1, d, 2, 2, 32, 32, 8)
    c.prefill(np.zeros((1, 1, 1, d), np.float16), np.ones((1, 1, 1, d), np.float16), [1])
    assert c.decode_probs(q)[1].tolist() == [[[1.0]]]
    # equal keys: uniform weights 1 / T
    c2 = oracle.Cache(1, 1, d, 2, 2, 32, 32, 80)
    c2.prefill(np.ones((1, 1, 70, d), np.float16), np.ones((1, 1, 70, d), np.float16), [70])
    np.testing.assert_allclose(c2.decode_probs(q)[1][0, 0], np.full(70, 1 / 70), rtol=1e-6)
    # no tokens: the row is left as it was (zeros)
    e = oracle.Cache(1, 1, d, 2, 2, 32, 32, 8)
    e.prefill(np.zeros((1, 1, 1, d), np.float16), np.zeros((1, 1, 1, d), np.float16), [0])
    assert not e.decode_probs(q, ld=4)[1].any()
    # a row narrower than a sequence is refused
    with pytest.raises(ValueError):
        c2.decode_probs(q, ld=69)


# --------------------------------------------------------------------------
# Packed device format.
# --------------------------------------------------------------------------

def _read_layout_golden():
    rows = []
    with open(os.path.join(GOLDEN, "layout_placements.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, ch, tok, word, bit = line.split()
                rows.append((a, int(ch), int(tok), int(word), int(bit)))
    return rows


@pytest.mark.parametrize("row", _read_layout_golden())
def test_layout_single_code_placement(row):
    """A single nonzero entry quantizes to code 3 (its group is {0, 1}: s = 1/3)
    and every other group is constant (code 0); the export must then hold
    exactly one field 0b11 at the hand-derived word and bit."""
    arr, ch, tok, word, bit = row
    d, G, R, t = 64, 32, 32, 256
    K = np.zeros((1, 1, t, d), np.float16)
    V = np.zeros((1, 1, t, d), np.float16)
    (K if arr == "K" else V)[0, 0, tok, ch] = 1.0
    c = oracle.Cache(1, 1, d, 2, 2, G, R, t)
    c.prefill(K, V, [t])
    ex = c.export()
    words = ex["Kc"] if arr == "K" else ex["Vc"]
    nz = np.nonzero(words)[0]
    assert nz.tolist() == [word]
    assert int(words[word]) == 3 << bit


def _read_layout_golden_d128():
    rows = []
    with open(os.path.join(GOLDEN, "layout_placements_d128.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                a, bits, ch, tok, word, bit = line.split()
                rows.append((a, int(bits), int(ch), int(tok), int(word), int(bit)))
    return rows


@pytest.mark.parametrize("row", _read_layout_golden_d128())
def test_layout_single_code_placement_d128(row):
    """d = 128 (value words four to a lane group, cs = 4) at 2 and 4 bits: a
    single entry 1.0 in an all-zero cache is the top code 2^B - 1 of its
    group {0, 1}; the export holds exactly that field at the hand-derived
    word and bit."""
    arr, bits, ch, tok, word, bit = row
    d, G, R, t = 128, 32, 32, 256
    K = np.zeros((1, 1, t, d), np.float16)
    V = np.zeros((1, 1, t, d), np.float16)
    (K if arr == "K" else V)[0, 0, tok, ch] = 1.0
    c = oracle.Cache(1, 1, d, bits, bits, G, R, t)
    c.prefill(K, V, [t])
    ex = c.export()
    words = ex["Kc"] if arr == "K" else ex["Vc"]
    nz = np.nonzero(words)[0]
    assert nz.tolist() == [word]
    assert int(words[word]) == ((1 << bits) - 1) << bit


@pytest.mark.parametrize("kb,vb,d", [(2, 2, 64), (4, 4, 128), (2, 4, 128), (4, 2, 256)])
def test_layout_is_a_packing(kb, vb, d):
    """All-maximal codes fill every bit of every full word exactly once (the
    fields tile the words); keys pack along tokens (a 16-bit half holds one
    channel, item 2) and values along channels (a half holds one token, item 3)."""
    G, R, t = 32, 32, 256
    K = np.zeros((1, 1, t, d), np.float16)
    V = np.zeros((1, 1, t, d), np.float16)
    K[0, 0, ::G] = 1.0       # every key group spans {0, 1}: code 0 at its first token
    V[0, 0, :, ::G] = 1.0    # every value group spans {0, 1}
    K = (1.0 - K.astype(np.float32)).astype(np.float16)   # now code 3 everywhere but one token a group
    c = oracle.Cache(1, 1, d, kb, vb, G, R, t)
    c.prefill(K, V, [t])
    st = c.state()
    nfields_k = int(np.count_nonzero(st["kcode"][0, 0, :, :t]))
    ex = c.export()
    bits_k = sum(bin(int(w)).count("1") for w in ex["Kc"])
    assert bits_k == nfields_k * kb
    # channel-pure key halves: build codes that depend on the channel only
    K2 = np.zeros((1, 1, t, d), np.float32)
    chval = np.arange(d) % 3 + 1                  # code wanted for channel c
    K2[0, 0, :, :] = 0
    K2[0, 0, 0::G, :] = 0
    K2[0, 0, 1::G, :] = 3                          # group range [0, 3] -> s = 1 (2-bit)
    for g0 in range(0, t, G):
        K2[0, 0, g0 + 2:g0 + G, :] = chval[None, :]
    c2 = oracle.Cache(1, 1, d, 2, 2, G, R, t)
    c2.prefill(K2.astype(np.float16), V, [t])
    kc = c2.export()["Kc"]
    halves = np.concatenate([kc & 0xFFFF, kc >> 16]).astype(np.uint32)
    for hw in halves:
        fields = {(int(hw) >> (2 * r)) & 3 for r in range(8)}
        assert len(fields - {0, 3}) <= 1   # one channel's code besides the two range tokens
    # token-pure value halves
    V2 = np.zeros((1, 1, t, d), np.float32)
    tokval = np.arange(t) % 3 + 1
    V2[0, 0, :, 0::G] = 0
    V2[0, 0, :, 1::G] = 3
    for gi in range(d // G):
        V2[0, 0, :, gi * G + 2:(gi + 1) * G] = tokval[:, None]
    c3 = oracle.Cache(1, 1, d, 2, 2, G, R, t)
    c3.prefill(K2.astype(np.float16), V2.astype(np.float16), [t])
    vc = c3.export()["Vc"]
    halves = np.concatenate([vc & 0xFFFF, vc >> 16]).astype(np.uint32)
    for hw in halves:
        fields = {(int(hw) >> (2 * r)) & 3 for r in range(8)}
        assert len(fields - {0, 3}) <= 1


def test_export_zero_padding_and_ring_slots():
    """Fields of tokens not yet quantized are zero; fp16 residual token tau sits
    at slot tau % R (keys) and tau % (R + 1) (values)."""
    d, G, R, t = 64, 32, 32, 100
    c, K, V = _cache_with(1, 1, d, 2, 2, G, R, 200, [t], seed=21)
    T, Tqk, Tqv = [int(x[0]) for x in c.lengths()]
    ex = c.export()
    kblk = 2 * d * 2
    # key block containing Tqk = 96: tokens 96..127 of block 1 must be zero fields
    # -> only positions (token % 64) / 8 < 4 may be nonzero in block 1
    blk1 = ex["Kc"][kblk:2 * kblk]
    assert np.all((blk1 & 0xFF00FF00) == 0)
    kf = ex["Kf"].reshape(R, d)
    for tok in range(Tqk, T):
        assert np.array_equal(kf[tok % R], K[0, 0, tok].view(np.uint16))
    vf = ex["Vf"].reshape(R + 1, d)
    for tok in range(Tqv, T):
        assert np.array_equal(vf[tok % (R + 1)], V[0, 0, tok].view(np.uint16))


# --------------------------------------------------------------------------
# Workload generator sanity (shapes and determinism only).
# --------------------------------------------------------------------------

def test_workload_slices_are_reproducible():
    w = W.small(W.WORKLOADS["llama3_8b_gqa_32k"], b=2, prefill=300)
    K, V, lens = W.prefill_kv(w)
    assert K.shape == (2, 8, 300, 128) and np.all(lens == 300)
    assert np.array_equal(W.prefill_slice(w, "K", 1, 5, 300), K[1, 5])
    ch = W.outlier_channels(w, 1, 5)
    assert ch.size == 3
    assert np.abs(K[1, 5][:, ch].astype(np.float32)).std() > 4 * np.abs(
        np.delete(K[1, 5], ch, axis=1).astype(np.float32)).std()
    w4 = W.WORKLOADS["kivi4_serving"]
    L = w4.lengths()
    assert L.min() >= 1024 and L.max() <= 4096 and L.shape == (64,)


def test_threaded_decode_equals_serial():
    """The GPU tests run the oracle's decode with one (sequence, query head)
    row per host thread; each row is computed exactly as in the serial loop,
    so outputs and weights must agree bit for bit with one thread, for all
    rows and for a listed subset."""
    rng = np.random.default_rng(11)
    b, h, hq, d, G, R = 3, 2, 8, 64, 16, 32
    lens = np.array([0, 77, 150], np.int32)
    K = (rng.standard_normal((b, h, 150, d)) * 2).astype(np.float16)
    V = rng.standard_normal((b, h, 150, d)).astype(np.float16)
    c = oracle.Cache(b, h, d, 4, 2, G, R, 200)
    c.prefill(K, V, lens)
    for s in range(5):
        c.append(rng.standard_normal((b, h, d)).astype(np.float16),
                 rng.standard_normal((b, h, d)).astype(np.float16))
    q = rng.standard_normal((b, hq, d)).astype(np.float16)
    pairs = [(2, 7), (1, 0), (2, 3), (0, 5)]
    try:
        assert oracle.set_threads(1) == 1
        o1, p1 = c.decode_probs(q)
        s1 = c.decode(q, pairs=pairs)
        nt = oracle.set_threads(max(4, os.cpu_count() or 1))
        on, pn = c.decode_probs(q)
        sn = c.decode(q, pairs=pairs)
    finally:
        oracle.set_threads(os.cpu_count() or 1)
    if nt == 1:
        pytest.skip("the oracle was built without OpenMP")
    assert np.array_equal(o1.view(np.uint32), on.view(np.uint32))
    assert np.array_equal(p1.view(np.uint32), pn.view(np.uint32))
    assert np.array_equal(s1.view(np.uint32), sn.view(np.uint32))
    assert np.all(np.isfinite(o1)) and np.count_nonzero(o1) == o1.size


# ---------------------------------------------------------------------------
# Prefill attention (the full-precision causal attention of the prompt,
# "Literature audit -- Group 2", section 1 KIVI, backends list; item 5's
# formula with keys s <= tau).
# ---------------------------------------------------------------------------

def _prompt(rng, b, hq, h, ts, d, scale=1.0):
    Q = (rng.standard_normal((b, hq, ts, d)) * scale).astype(np.float16)
    K = (rng.standard_normal((b, h, ts, d)) * scale).astype(np.float16)
    V = rng.standard_normal((b, h, ts, d)).astype(np.float16)
    return Q, K, V


def test_prefill_attention_first_row_and_equal_keys():
    """Row 0 sees one key: it is v_0.  With every key equal the weights are
    uniform: row tau is the mean of v_0 .. v_tau."""
    rng = np.random.default_rng(21)
    Q, K, V = _prompt(rng, 2, 4, 2, 40, 64)
    t = [40, 17]
    out = oracle.prefill_attention(Q, K, V, t)
    for i in range(2):
        for qh in range(4):
            assert np.array_equal(out[i, qh, 0], V[i, qh // 2, 0].astype(np.float64))
    Ke = np.broadcast_to(K[:, :, :1], K.shape).copy()
    out = oracle.prefill_attention(Q, Ke, V, t)
    for i in range(2):
        for qh in range(4):
            v = V[i, qh // 2].astype(np.float64)
            mean = np.cumsum(v, axis=0) / np.arange(1, 41)[:, None]
            np.testing.assert_allclose(out[i, qh, :t[i]], mean[:t[i]], rtol=1e-12, atol=1e-12)
            assert not out[i, qh, t[i]:].any()   # rows past t untouched


def test_prefill_attention_is_causal():
    """Row tau depends on keys and values s <= tau only."""
    rng = np.random.default_rng(22)
    Q, K, V = _prompt(rng, 1, 2, 1, 50, 64)
    a = oracle.prefill_attention(Q, K, V, [50])
    K2, V2 = K.copy(), V.copy()
    K2[:, :, 30:] = rng.standard_normal(K2[:, :, 30:].shape).astype(np.float16)
    V2[:, :, 30:] = rng.standard_normal(V2[:, :, 30:].shape).astype(np.float16)
    b = oracle.prefill_attention(Q, K2, V2, [50])
    assert np.array_equal(a[:, :, :30], b[:, :, :30])
    assert np.abs(a[:, :, 30:] - b[:, :, 30:]).max() > 1e-2


def test_prefill_attention_last_row_equals_decode():
    """The last prompt row attends to every key: it is the decode attention
    of that query over an unquantized cache holding the prompt (the decode
    routine, fp32, with its own scores and softmax)."""
    rng = np.random.default_rng(23)
    b, hq, h, t, d = 2, 8, 2, 100, 128
    Q, K, V = _prompt(rng, b, hq, h, t, d, scale=2.0)
    out = oracle.prefill_attention(Q, K, V, [t, t])
    c = oracle.Cache(b, h, d, 2, 2, 32, 128, 256)   # t < R: nothing quantized
    c.prefill(K, V, np.array([t, t], np.int32))
    dec = c.decode(np.ascontiguousarray(Q[:, :, t - 1]))
    np.testing.assert_allclose(dec, out[:, :, t - 1], rtol=2e-5, atol=2e-5)
    c.close()


def test_prefill_attention_gqa_and_rows():
    """Query heads of one kv head equal an MHA problem with the kv head
    repeated; a listed subset of rows equals the same rows of the full
    computation."""
    rng = np.random.default_rng(24)
    Q, K, V = _prompt(rng, 2, 6, 2, 33, 64)
    t = [33, 20]
    g = oracle.prefill_attention(Q, K, V, t)
    m = oracle.prefill_attention(Q, np.repeat(K, 3, axis=1), np.repeat(V, 3, axis=1), t)
    assert np.array_equal(g, m)
    rows = np.array([[0, 0, 0], [0, 5, 32], [1, 3, 19], [1, 2, 7]], np.int32)
    s = oracle.prefill_attention(Q, K, V, t, rows=rows)
    for k, (i, qh, tau) in enumerate(rows):
        assert np.array_equal(s[k], g[i, qh, tau])
