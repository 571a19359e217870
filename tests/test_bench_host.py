"""Host-side pieces of bench.py that need no GPU: the algorithmic byte count
behind the roofline, the step modes, the workload variants and the
argument checks."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from bit_quantized_kv_quantize_gb300 import workloads as W  # noqa: E402


def test_bytes_per_quantized_token_head():
    """A fully quantized 2-bit token of one kv head at d = 128, G = 32 is
    32 B of key codes + 32 B of value codes + 16 B of key scale/zero (two
    fp16 per channel per 32 tokens) + 16 B of value scale/zero (two fp16
    per 32-channel group): 96 B; q and out add 2 x 2 B per query channel."""
    w = W.WORKLOADS["llama3_8b_gqa_32k"]
    n = 4096
    T = np.full(w.b, n)
    got = bench.algorithmic_bytes(w, T, T, T)
    assert got == w.b * w.h_kv * n * 96 + 2 * w.b * w.h_q * w.d * 2


def test_bytes_of_fp16_window_tokens_and_scores():
    """An fp16 key or value token costs 2 d bytes; the weights output adds
    one fp32 score per (query head, token)."""
    w = W.small(W.WORKLOADS["llama3_8b_gqa_32k"], b=2)
    T = np.array([1000, 700])
    Tqk = np.array([896, 640])
    Tqv = np.array([872, 572])
    base = bench.algorithmic_bytes(w, T, T, T)
    got = bench.algorithmic_bytes(w, T, Tqk, Tqv)
    per_k, per_v = w.d * w.kbits // 8 + 4 * w.d // w.G, w.d * w.vbits // 8 + 4 * w.d // w.G
    extra = w.h_kv * sum((t - a) * (2 * w.d - per_k) + (t - c) * (2 * w.d - per_v)
                         for t, a, c in zip(T, Tqk, Tqv))
    assert got == base + extra
    assert bench.algorithmic_bytes(w, T, Tqk, Tqv, scores=True) == got + 4 * w.h_q * int(T.sum())


def test_four_bit_costs_the_codes_twice():
    w2 = W.WORKLOADS["llama3_8b_gqa_32k"]
    w4 = W.small(w2, kbits=4, vbits=4)
    T = np.full(w2.b, 2048)
    codes2 = w2.b * w2.h_kv * 2048 * (2 * w2.d * 2 // 8)
    assert bench.algorithmic_bytes(w4, T, T, T) - bench.algorithmic_bytes(w2, T, T, T) == codes2


def test_step_modes_and_config():
    class A:
        pass
    a = A()
    assert bench.step_mode(a) == "fused"   # the default: one kivi_append_decode call
    a.two = True
    assert bench.step_mode(a) == "two"
    a.probs = True
    assert bench.step_mode(a) == "probs"
    assert bench.prefill_attn_flops(W.WORKLOADS["tiny_kivi2"], [3]) == 4.0 * 2 * 64 * 6
    w = W.WORKLOADS["llama3_8b_gqa_32k"]
    for mode, name in bench.STEP_NAMES.items():
        cfg = bench.workload_config(w, mode)
        assert cfg["workload"] == w.name and cfg["step"] == name
        assert cfg["context"] == int(w.lengths().max()) + 1
        assert "flushed" in cfg["l2"]
    json.dumps(bench.workload_config(w))


def _run(*args):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=120)


def test_arguments_rejected():
    r = _run("--warmup", "2")
    assert r.returncode != 0 and "warmup" in r.stderr
    r = _run("--group", "64", "--residual", "96")
    assert r.returncode != 0 and "R % G" in r.stderr


def test_variant_keeps_the_shape():
    w = W.WORKLOADS["llama3_8b_gqa_32k"]
    v = W.small(w, kbits=4, vbits=2, G=64, R=128)
    assert (v.b, v.h_q, v.h_kv, v.d, v.prefill) == (w.b, w.h_q, w.h_kv, w.d, w.prefill)
    assert (v.kbits, v.vbits, v.G, v.R) == (4, 2, 64, 128)


def test_traffic_quoted_only_for_its_source():
    """roofline.traffic comes from an ncu capture keyed by the decode
    kernel's source hash: quoted only for that source (null otherwise), and
    every recorded capture read the cache once (no re-reads)."""
    h = bench.source_hash()
    assert len(h) == 16 and h == bench.source_hash()
    assert bench.NCU_TRAFFIC.get("0" * 16) is None
    # the captured call: prefill t tokens, append one (the maintenance it
    # leaves waits for the next append), then decode
    w = W.WORKLOADS[bench.DEFAULT_WORKLOAD]
    t = w.lengths()
    alg = bench.algorithmic_bytes(w, t + 1, t - t % w.R, np.maximum(t - w.R, 0))
    for per_mode in bench.NCU_TRAFFIC.values():
        assert set(per_mode) <= set(bench.STEP_NAMES)
        for traffic in per_mode.values():
            assert 1.0 <= traffic / alg < 1.05   # read once, no re-reads
