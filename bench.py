#!/usr/bin/env python3
"""Benchmark: KIVI quantized-KV decode step on one GB300.

A step is one decode step of the whole cache: one kivi_append_decode call --
the append (the lazy key-block flush / value-queue pop of the KIVI residual
window, then the new token) and the split-K attention over the quantized and
fp16 segments with its merge.  Where it pays (see kivi.h) that is one launch
of the decode kernel, which appends the token itself; otherwise the append
kernel and the decode kernel.  --two times kivi_append + kivi_decode_attn,
--probs the step with per-token attention weights.  Prefill packing runs
once before timing and is reported separately; --prefill-attn times the
prefill with its causal attention (kivi_prefill_attn) instead.

Prints ONE JSON line.  Default workload: Llama-3-8B GQA layer shape at 32k
context (batch 8, 32 query / 8 kv heads, d 128, 2-bit K/V, G 32, R 128).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline]

--impl reference times the CPU oracle (plain C, fp32) on the host cores over
the same workload (--warmup untimed and --steps timed steps).  Under torchrun (N > 1) every rank
runs an independent replica of the workload on its own GPU (the path has no
exchange step); rank 0 prints the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_kv_quantize_gb300 import workloads as W  # noqa: E402

METRIC = "quantized-KV decode attention µs/step and cache GB/s vs HBM peak (1×GB300)"
DEFAULT_WORKLOAD = "llama3_8b_gqa_32k"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) of one decode-attention launch, from an ncu
# capture of the kernel whose source hash is recorded beside it, per step
# mode (the one-launch step's kernel, and the plain one); reported only
# while the kernel source is unchanged (llama3_8b_gqa_32k, the default
# workload).
NCU_TRAFFIC = {"3b1e4c20734282ed": {"fused": 204195072 + 6233600, "two": 205795584 + 2664448}}


def algorithmic_bytes(w: W.Workload, T, Tqk, Tqv, scores: bool = False) -> int:
    """Cache bytes one decode-attention call must read, plus q and out:
    packed codes and fp16 scale/zero of the quantized tokens and the fp16
    residual tokens, per (sequence, kv head); with scores, also the fp32
    score of every (sequence, query head, token) the kernel writes for the
    attention-weight output."""
    d, G = w.d, w.G
    per_qk = d * w.kbits // 8 + 4 * d // G
    per_qv = d * w.vbits // 8 + 4 * d // G
    T, Tqk, Tqv = (np.asarray(x, np.int64) for x in (T, Tqk, Tqv))
    cache = w.h_kv * int(np.sum(Tqk * per_qk + Tqv * per_qv + ((T - Tqk) + (T - Tqv)) * 2 * d))
    extra = 4 * w.h_q * int(np.sum(T)) if scores else 0
    return cache + 2 * w.b * w.h_q * d * 2 + extra


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if j.get("hbm_gbs"):
            return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("kivi_decode.cu", "kivi_decode_impl.cuh", "kivi_internal.cuh", "kivi_mma.cuh"):
        with open(os.path.join(ROOT, "bit_quantized_kv_quantize_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx = float(p[2])
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    backend = "nccl" if os.environ.get("KIVI_BENCH_BACKEND", "") != "gloo" else "gloo"
    dist.init_process_group(backend)
    return rank, ws, dist


def reduce_max(x: float, dist, device=None) -> float:
    """Max over ranks (replicas run independently; the slowest sets the time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        import torch
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline object)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name (or the architecture when none is listed)."""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def _oracle_sample(w: W.Workload, bs: int, hs: int, cap: int):
    """An oracle cache of the first bs sequences x hs kv heads of the
    workload, and (K, V, lengths) to prefill it with."""
    import oracle
    lens = w.lengths()[:bs]
    ts = int(max(1, lens.max()))
    Kh = np.zeros((bs, hs, ts, w.d), np.float16)
    Vh = np.zeros_like(Kh)
    for i in range(bs):
        for j in range(hs):
            n = int(lens[i])
            Kh[i, j, :n] = W.prefill_slice(w, "K", i, j, n)
            Vh[i, j, :n] = W.prefill_slice(w, "V", i, j, n)
    return oracle.Cache(bs, hs, w.d, w.kbits, w.vbits, w.G, w.R, cap), Kh, Vh, lens


def _oracle_step(c, w, s, bs, hs):
    k, v = W.step_kv(w, s)
    q = W.step_q(w, s)
    k = np.ascontiguousarray(k[:bs, :hs])
    v = np.ascontiguousarray(v[:bs, :hs])
    q = np.ascontiguousarray(q[:bs, :hs * w.group])
    t0 = time.perf_counter()
    c.append(k, v)
    c.decode(q)
    return time.perf_counter() - t0


def oracle_time(w: W.Workload, budget_s: float = 15.0, max_pairs: int = 8):
    """The oracle (as it stands) on a bounded sample of the workload: the
    first b' sequences x h' kv heads (b' h' <= max_pairs) with all their
    query heads, timed per decode step (append + attention) on all host
    threads and on one, and its prefill (quantize + pack) once; each scaled
    to all b x h_kv (sequence, kv head) pairs by token count.  Returns the
    cpu_baseline fields."""
    import oracle
    cores = os.cpu_count() or 1
    lens = w.lengths()
    bs = min(w.b, max_pairs)
    hs = min(w.h_kv, max(1, max_pairs // bs))
    max_steps = 400
    # room for both timed loops (all threads, then one)
    c, Kh, Vh, lp = _oracle_sample(w, bs, hs, int(lens.max()) + 2 * max_steps + 8)
    t0 = time.perf_counter()
    c.prefill(Kh, Vh, lp)
    prefill_s = time.perf_counter() - t0
    del Kh, Vh
    scale = float(lens.sum() * w.h_kv) / float(max(1, lp.sum()) * hs)
    oracle.set_threads(cores)
    steps, elapsed = 0, 0.0
    while steps < max_steps and elapsed < budget_s:
        elapsed += _oracle_step(c, w, steps, bs, hs)
        steps += 1
    oracle.set_threads(1)
    steps1, elapsed1 = 0, 0.0
    while steps1 < max_steps and elapsed1 < budget_s / 3:
        elapsed1 += _oracle_step(c, w, steps + steps1, bs, hs)
        steps1 += 1
    oracle.set_threads(cores)
    c.close()
    us = elapsed / steps * scale * 1e6
    sample = (f"{bs} sequence(s) x {hs} kv head(s) of {w.b} x {w.h_kv}, {steps} step(s) of "
              f"append + attention over {w.group} query heads per kv head on {cores} threads "
              f"({elapsed:.1f} s) and {steps1} on one ({elapsed1:.1f} s), prefill once; "
              f"scaled by token count to the whole batch")
    return {"value": round(us, 3), "unit": "us/step", "cores": cores, "kind": "oracle",
            "sample": sample, "cpu_model": cpu_model(),
            "single_thread_us_per_step": round(elapsed1 / max(1, steps1) * scale * 1e6, 3),
            "prefill_us": round(prefill_s * scale * 1e6, 1)}


def run_reference(args, w):
    """The reference arm: the oracle, as it stands, on the host cores, over
    the whole workload (every sequence and kv head): prefill once, --warmup
    untimed steps, then --steps timed steps of append + attention."""
    import oracle
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and int(os.environ.get("RANK", "0")) != 0:
        return 0
    t0 = time.time()
    cores = os.cpu_count() or 1
    lens = w.lengths()
    n = args.warmup + args.steps
    c, Kh, Vh, lp = _oracle_sample(w, w.b, w.h_kv, int(lens.max()) + n + 8)
    tp = time.perf_counter()
    c.prefill(Kh, Vh, lp)
    prefill_s = time.perf_counter() - tp
    del Kh, Vh
    oracle.set_threads(cores)
    for s in range(args.warmup):
        _oracle_step(c, w, s, w.b, w.h_kv)
    times = [_oracle_step(c, w, args.warmup + s, w.b, w.h_kv) for s in range(args.steps)]
    c.close()
    us = sum(times) / len(times) * 1e6
    sample = (f"the whole workload ({w.b} x {w.h_kv} (sequence, kv head) pairs), {args.steps} timed "
              f"step(s) of append + attention after {args.warmup} untimed, on {cores} threads")
    line = {
        "metric": METRIC, "value": round(us, 3), "unit": "us/step", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "impl": "reference",
        "config": workload_config(w, step_mode(args)),
        "cpu_baseline": {"value": round(us, 3), "unit": "us/step", "cores": cores,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model(),
                         "prefill_us": round(prefill_s * 1e6, 1)},
        "e2e": {"value": round(us, 3), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(time.time() - t0, 1),
    }
    print(json.dumps(line), flush=True)
    return 0


EXTRA_LAUNCHES = {"two": 1, "fused": 0, "probs": 2}
STEP_NAMES = {"two": "kivi_append + kivi_decode_attn", "fused": "kivi_append_decode",
              "probs": "kivi_append + kivi_decode_attn_probs (weights, accumulated mass)"}


def step_mode(args) -> str:
    return "probs" if getattr(args, "probs", False) else ("two" if getattr(args, "two", False) else "fused")


def workload_config(w, mode="fused"):
    T = int(w.lengths().max()) + 1
    return {"workload": w.name,
            "step": STEP_NAMES[mode], "b": w.b, "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d,
            "k_bits": w.kbits, "v_bits": w.vbits, "G": w.G, "R": w.R,
            "context": T if not w.ragged else f"ragged {w.ragged[0]}-{w.ragged[1]}",
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)",
            "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, w):
    import torch
    rank, ws, dist = dist_setup()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bit_quantized_kv_quantize_gb300 import kivi as K

    t_start = time.time()
    cap = int(w.lengths().max()) + args.warmup + 3 * args.steps + 8
    cache = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    Kh, Vh, lens = W.prefill_kv(w)
    Kd = torch.from_numpy(Kh).to(dev)
    Vd = torch.from_numpy(Vh).to(dev)
    del Kh, Vh
    stream = torch.cuda.current_stream(dev)
    # prefill pack: median of five timed runs after one untimed run (K and V
    # are each larger than L2 at the long workloads)
    cache.prefill(Kd, Vd, lens)
    torch.cuda.synchronize(dev)
    pre = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cache.prefill(Kd, Vd, lens)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        pre.append(e0.elapsed_time(e1))
    prefill_ms = statistics.median(pre)
    del Kd, Vd
    torch.cuda.empty_cache()

    nsteps = args.warmup + 2 * args.steps + 1
    host_k, host_v, host_q = [], [], []
    for s in range(nsteps):
        k, v = W.step_kv(w, s)
        host_k.append(k)
        host_v.append(v)
        host_q.append(W.step_q(w, s))
    kd = [torch.from_numpy(x).to(dev) for x in host_k]
    vd = [torch.from_numpy(x).to(dev) for x in host_v]
    qd = [torch.from_numpy(x).to(dev) for x in host_q]
    out = torch.empty((w.b, w.h_q, w.d), dtype=torch.float16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    mode = step_mode(args)
    if mode == "probs":   # per-token weights and their running sum, one row per query head
        probs = torch.zeros((w.b, w.h_q, cap), dtype=torch.float32, device=dev)
        mass = torch.zeros_like(probs)

    def run_step(k, v, q):
        if mode == "two":
            cache.append(k, v)
            cache.decode(q, out)
        elif mode == "fused":
            cache.append_decode(k, v, q, out)
        else:
            cache.append(k, v)
            cache.decode_probs(q, probs, mass=mass, out=out)

    def step(s):
        run_step(kd[s], vd[s], qd[s])

    for s in range(args.warmup):
        flush.fill_(s)
        step(s)
    torch.cuda.synchronize(dev)

    # ---- device-timed regions: inputs resident in HBM --------------------
    # Region 1 gives the step time: nothing but the step runs between its
    # events.  Region 2 (as many steps, continuing) has the library record an
    # event pair around every decode-kernel launch, for that kernel's own
    # duration (the roofline); those events sit between the append and the
    # decode launch, so region 2's steps are slower and only its kernel
    # times are used.
    def timed(n0, profile):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        nbytes, nlaunch = [], []
        cache.profile(profile)
        cache.profile_read()
        barrier(dist, dev)
        torch.cuda.synchronize(dev)
        for n in range(args.steps):
            flush.fill_(n)
            starts[n].record(stream)
            step(n0 + n)
            ends[n].record(stream)
            T, Tqk, Tqv = cache.lengths()
            nbytes.append(algorithmic_bytes(w, T, Tqk, Tqv, scores=mode == "probs"))
            # the library's launches of the step's last call, plus the
            # separate append call and the weights' finalizing kernel
            nlaunch.append(cache.plan()[1] + EXTRA_LAUNCHES[mode])
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        prof = cache.profile_read()
        cache.profile(False)
        return [a.elapsed_time(b) for a, b in zip(starts, ends)], nbytes, prof, nlaunch

    with ClockSampler(local) as clk:
        step_ms, _, _, step_launches = timed(args.warmup, False)
        inst_ms, bytes_steps, (attn_ms_total, attn_launches), _ = timed(args.warmup + args.steps, True)
    ms_per_step = reduce_max(sum(step_ms) / args.steps, dist, dev)
    ms_instrumented = reduce_max(sum(inst_ms) / args.steps, dist, dev)
    attn_ms = reduce_max(attn_ms_total / max(1, attn_launches), dist, dev)
    assert cache.check() == 0, "device status word set during the benchmark"
    splits = cache.plan()[0]

    # ---- end to end through the C ABI with host buffers ------------------
    pin_k = [torch.from_numpy(x).pin_memory() for x in host_k]
    pin_v = [torch.from_numpy(x).pin_memory() for x in host_v]
    pin_q = [torch.from_numpy(x).pin_memory() for x in host_q]
    out_h = torch.empty((w.b, w.h_q, w.d), dtype=torch.float16).pin_memory()
    kbuf = torch.empty_like(kd[0])
    vbuf = torch.empty_like(vd[0])
    qbuf = torch.empty_like(qd[0])
    # the same cache continues (the sequences keep growing); inputs cycle
    e2e_ms = []
    for n in range(args.steps):
        s = n % nsteps
        flush.fill_(n)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kbuf.copy_(pin_k[s], non_blocking=True)
        vbuf.copy_(pin_v[s], non_blocking=True)
        qbuf.copy_(pin_q[s], non_blocking=True)
        run_step(kbuf, vbuf, qbuf)
        out_h.copy_(out, non_blocking=True)
        b.record(stream)
        e2e_ms.append((a, b))
    torch.cuda.synchronize(dev)
    e2e_per = reduce_max(sum(a.elapsed_time(b) for a, b in e2e_ms) / len(e2e_ms), dist, dev)
    h2d = int(kbuf.numel() * 2 + vbuf.numel() * 2 + qbuf.numel() * 2)
    d2h = int(out.numel() * 2)

    peak, peak_kind = load_peaks()
    bytes_per = float(np.mean(bytes_steps))
    achieved = bytes_per / (attn_ms * 1e-3) / 1e9
    us_step = ms_per_step * 1e3
    line = {
        "metric": METRIC,
        "value": round(us_step, 3),
        "unit": "us/step",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u2/u4 codes, f16 in, f32 accumulate",
        "data": "synthetic",
        "config": workload_config(w, mode),
        "attn_us": round(attn_ms * 1e3, 3),
        "us_per_step_with_kernel_events": round(ms_instrumented * 1e3, 3),
        "cache_gbs": round(bytes_per / (attn_ms * 1e-3) / 1e9, 1),
        "bytes_per_step": int(bytes_per),
        "prefill_us": round(prefill_ms * 1e3, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": "decode_kernel (persistent stream-K over TMA-staged block records, mma.sync, last-CTA merge)",
                     "traffic": (NCU_TRAFFIC.get(source_hash(), {}).get(mode)
                                 if w == W.WORKLOADS[DEFAULT_WORKLOAD] else None)},
        "e2e": {"value": round(e2e_per * 1e3, 3), "unit": "us/step",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(sum(step_launches)),
        "splits": splits,
        "clocks": clk.summary(),
        "source_hash": source_hash(),
    }
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = oracle_time(w, budget_s=float(os.environ.get("KIVI_ORACLE_BUDGET_S", "15")))
    line["wall_s"] = round(time.time() - t_start, 1)
    cache.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_ncu_case(args, w):
    """Minimal launch sequence for profiler captures: prefill the workload,
    append one token, then --steps decode calls (no flush buffer, no oracle);
    with --fused, --steps kivi_append_decode calls instead."""
    import torch
    from bit_quantized_kv_quantize_gb300 import kivi as K
    dev = torch.device("cuda", 0)
    cap = int(w.lengths().max()) + args.steps + 8
    cache = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, cap)
    Kh, Vh, lens = W.prefill_kv(w)
    Kd, Vd = torch.from_numpy(Kh).to(dev), torch.from_numpy(Vh).to(dev)
    del Kh, Vh
    cache.prefill(Kd, Vd, lens)
    del Kd, Vd
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    k, v = W.step_kv(w, 0)
    cache.append(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev))
    q = torch.from_numpy(W.step_q(w, 0)).to(dev)
    out = torch.empty_like(q)
    for s in range(args.steps):
        if args.fused:
            k, v = W.step_kv(w, s + 1)
            cache.append_decode(torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev), q, out)
        else:
            cache.decode(q, out)
    torch.cuda.synchronize(dev)
    assert cache.check() == 0
    T, Tqk, Tqv = cache.lengths()
    print(json.dumps({"ncu_case": w.name, "decode_calls": args.steps, "plan": cache.plan(),
                      "bytes_per_decode": algorithmic_bytes(w, T, Tqk, Tqv)}), flush=True)
    cache.close()
    return 0


def prefill_attn_flops(w, lens) -> float:
    """2 x the multiply-adds of the prompt's causal attention: q.k and p v,
    d each, per query head and (row tau, key s <= tau) pair."""
    pairs = sum(int(n) * (int(n) + 1) // 2 for n in lens)
    return 4.0 * w.h_q * w.d * pairs


def run_prefill_attn(args, w):
    """kivi_prefill_attn (causal attention + the cache's quantize / pack in
    its epilogue, one launch) on the workload's prompt, against kivi_prefill
    (the pack kernels alone).  Inputs (K, V, Q: about 4 GB at 32k) exceed L2;
    median of the timed calls."""
    import torch
    from bit_quantized_kv_quantize_gb300 import kivi as K
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    Kh, Vh, lens = W.prefill_kv(w)
    Qh = W.prefill_q(w)
    Kd, Vd, Qd = (torch.from_numpy(x).to(dev) for x in (Kh, Vh, Qh))
    del Kh, Vh, Qh
    out = torch.empty_like(Qd)
    cache = K.KiviCache(w.b, w.h_kv, w.d, w.kbits, w.vbits, w.G, w.R, int(lens.max()) + 8)
    stream = torch.cuda.current_stream(dev)
    n = max(1, min(args.steps, 10))

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)

    with ClockSampler(dev.index) as clk:
        us = timed(lambda: cache.prefill_attn(Qd, Kd, Vd, lens, out=out))
        pack_us = timed(lambda: cache.prefill(Kd, Vd, lens))
    assert cache.check() == 0
    flops = prefill_attn_flops(w, lens)
    tf = flops / (us * 1e-6) / 1e12
    peak = None
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            peak = json.load(f).get("bf16_tflops")
    line = {
        "metric": "causal prefill attention with the KIVI quantize/pack epilogue, us per call (1xGB300)",
        "value": round(us, 1), "unit": "us/call", "n_gpus": 1, "steps": n, "warmup": args.warmup,
        "higher_is_better": False, "vs_baseline": None, "dtype": "f16 in, f32 accumulate",
        "data": "synthetic", "impl": "ours",
        "config": {"workload": w.name, "call": "kivi_prefill_attn", "b": w.b, "h_q": w.h_q, "h_kv": w.h_kv,
                   "d": w.d, "k_bits": w.kbits, "v_bits": w.vbits, "G": w.G, "R": w.R,
                   "tokens": int(lens.max()), "l2": "inputs larger than L2"},
        "pack_only_us": round(pack_us, 1),
        "roofline": {"bound": "tensor", "achieved": round(tf, 1),
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tf / peak, 3) if peak else None,
                     "peak_source": "measured bf16_tflops (the fp16 MMA rate is the same)" if peak else None,
                     "flops_per_call": flops},
        "gpu_launches": n,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    cache.close()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--k-bits", type=int, choices=(2, 4), help="override the workload's key bits")
    ap.add_argument("--v-bits", type=int, choices=(2, 4), help="override the workload's value bits")
    ap.add_argument("--group", type=int, choices=(16, 32, 64, 128), help="override the group size G")
    ap.add_argument("--residual", type=int, help="override the residual length R (a multiple of G)")
    ap.add_argument("--tokens", type=int,
                    help="override the prompt length (a smaller case of the workload, for profiler captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--two", action="store_true",
                    help="time a step as kivi_append + kivi_decode_attn instead of one "
                         "kivi_append_decode call")
    ap.add_argument("--fused", action="store_true", help="the default step (one kivi_append_decode call)")
    ap.add_argument("--probs", action="store_true",
                    help="time a step as kivi_append + kivi_decode_attn_probs (per-token weights "
                         "and their accumulated mass)")
    ap.add_argument("--ncu", action="store_true",
                    help="run only prefill, one append and --steps decode calls (profiler captures)")
    ap.add_argument("--prefill-attn", action="store_true",
                    help="time kivi_prefill_attn (causal attention + pack epilogue) against kivi_prefill")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = W.WORKLOADS[args.workload]
    over = {k: v for k, v in (("kbits", args.k_bits), ("vbits", args.v_bits), ("G", args.group),
                              ("R", args.residual), ("prefill", args.tokens)) if v is not None}
    if over:   # a variant of the workload (bits / group / residual sweep, a shorter prompt)
        if args.tokens is not None and (args.tokens < 1 or w.ragged):
            ap.error("--tokens needs a positive count and a workload of equal lengths")
        w = W.small(w, **over)
        if w.R % w.G or w.d % w.G:
            ap.error("need R % G == 0 and d % G == 0")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.ncu:
        return run_ncu_case(args, w)
    if args.prefill_attn:
        return run_prefill_attn(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
