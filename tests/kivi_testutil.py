"""Shared helpers for the GPU parity tests: run the same seeded inputs through
libkivi (via the thin binding) and through the CPU oracle, and compare.

The comparison rules follow the packed format's definition: whole words of
every quantized block (zero fields included), scale/zero of every quantized
group or token, and the fp16 window slots of the live tokens.
"""
from __future__ import annotations

import numpy as np

import oracle

ATOL = 2e-3    # max-abs tolerance of the attention output
RTOL_L2 = 1e-3  # relative L2 tolerance over the whole output


def geometry(b, h, d, kb, vb, G, R, cap):
    q = max(64, G)
    fcap = -(-cap // q) * q
    return dict(b=b, h=h, d=d, kb=kb, vb=vb, G=G, R=R, fcap=fcap,
                kc_blk=2 * d * kb, nkb=fcap // 64, nkg=fcap // G, vc_blk=d * vb // 2,
                nvb=fcap // 16, vsz_blk=2 * (d // G) * 16)


def slice_views(ex, g, i, j):
    """Views of the (sequence i, head j) slice of an export dict."""
    b, h, d, R = g["b"], g["h"], g["d"], g["R"]
    Kc = ex["Kc"].reshape(b, h, g["nkb"], g["kc_blk"])[i, j]
    Ksz = ex["Ksz"].reshape(b, h, g["nkg"], 2, d)[i, j]
    Vc = ex["Vc"].reshape(b, h, g["nvb"], g["vc_blk"])[i, j]
    Vsz = ex["Vsz"].reshape(b, h, g["nvb"], 2, d // g["G"], 16)[i, j]
    Kf = ex["Kf"].reshape(b, h, R, d)[i, j]
    Vf = ex["Vf"].reshape(b, h, R + 1, d)[i, j]
    return Kc, Ksz, Vc, Vsz, Kf, Vf


def compare_slice(gex, gg, gi, gj, oex, og, oi, oj, T, Tqk, Tqv, what=""):
    """Bit-exact comparison of one slice; raises AssertionError naming the first mismatch."""
    a = slice_views(gex, gg, gi, gj)
    b = slice_views(oex, og, oi, oj)
    R = gg["R"]
    nkb = -(-Tqk // 64)
    nvb = -(-Tqv // 16)
    checks = [
        ("Kc", a[0][:nkb], b[0][:nkb]),
        ("Ksz", a[1][:Tqk // gg["G"]], b[1][:Tqk // gg["G"]]),
        ("Vc", a[2][:nvb], b[2][:nvb]),
        ("Vsz", a[3][:nvb], b[3][:nvb]),
    ]
    ks = [tau % R for tau in range(Tqk, T)]
    vs = [tau % (R + 1) for tau in range(Tqv, T)]
    checks += [("Kf", a[4][ks], b[4][ks]), ("Vf", a[5][vs], b[5][vs])]
    for name, x, y in checks:
        if not np.array_equal(x, y):
            idx = np.argwhere(x != y)[0]
            raise AssertionError(f"{what} {name} differs at {tuple(idx)}: gpu {x[tuple(idx)]!r} "
                                 f"oracle {y[tuple(idx)]!r} (T={T}, Tqk={Tqk}, Tqv={Tqv})")


def compare_output(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    err = np.abs(gpu - ref)
    maxabs = float(err.max()) if err.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(gpu - ref)) / den if den > 0 else float(np.linalg.norm(gpu - ref))
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    assert maxabs <= ATOL, f"{what}: max-abs error {maxabs:.3e} > {ATOL}"
    assert rel <= RTOL_L2, f"{what}: relative L2 error {rel:.3e} > {RTOL_L2}"
    return maxabs, rel


def oracle_for(w_or_dims, cap):
    b, h, d, kb, vb, G, R = w_or_dims
    return oracle.Cache(b, h, d, kb, vb, G, R, cap)
