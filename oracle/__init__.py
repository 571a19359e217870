"""CPU oracle for the KIVI quantized KV cache and decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never
does.  The arithmetic lives in ``kivi_oracle.c`` (plain C, fp32, rintf, no FMA
contraction); this module only builds it and marshals numpy arrays.

fp16 data crosses this boundary as numpy ``float16`` arrays (their bit
patterns are what the C code reads).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kivi_oracle.c into liboracle.so next to it (gcc, -ffp-contract=off)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "kivi_oracle.h"))
    ):
        return _LIB
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-o", _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _u16p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _f32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _i32p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            vp = ctypes.c_void_p
            L.ko_f16_to_f32.restype = ctypes.c_float
            L.ko_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.ko_f32_to_f16.restype = ctypes.c_uint16
            L.ko_f32_to_f16.argtypes = [ctypes.c_float]
            L.ko_f32_to_f16_n.argtypes = [vp, vp, ctypes.c_size_t]
            L.ko_f16_to_f32_n.argtypes = [vp, vp, ctypes.c_size_t]
            L.ko_quantize_group.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            vp, vp, vp, ctypes.c_int]
            L.ko_dequant.restype = ctypes.c_float
            L.ko_dequant.argtypes = [ctypes.c_uint8, ctypes.c_uint16, ctypes.c_uint16]
            L.ko_create.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(vp)]
            L.ko_destroy.argtypes = [vp]
            L.ko_prefill.argtypes = [vp, vp, vp, vp, ctypes.c_int]
            L.ko_append.argtypes = [vp, vp, vp]
            L.ko_decode.argtypes = [vp, vp, ctypes.c_int, vp]
            L.ko_decode_subset.argtypes = [vp, vp, ctypes.c_int, vp, vp, ctypes.c_int]
            L.ko_decode_probs.argtypes = [vp, vp, ctypes.c_int, vp, vp, ctypes.c_longlong, vp, ctypes.c_int]
            L.ko_set_threads.argtypes = [ctypes.c_int]
            L.ko_prefill_attn.argtypes = [vp, vp, vp, vp] + [ctypes.c_int] * 5 + [vp, ctypes.c_int, vp]
            L.ko_lengths.argtypes = [vp, vp, vp, vp]
            L.ko_dequant_kv.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp]
            L.ko_state.argtypes = [vp] * 9
            L.ko_capacity.argtypes = [vp]
            L.ko_capacity_stride.argtypes = [vp]
            L.ko_export_supported.argtypes = [vp]
            L.ko_export_sizes.argtypes = [vp] + [ctypes.POINTER(ctypes.c_size_t)] * 6
            L.ko_export.argtypes = [vp] * 7
            _lib = L
    return _lib


def f32_to_f16_bits(x) -> np.ndarray:
    """Round fp32 values to fp16 (round-half-to-even) with the oracle's converter."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().ko_f32_to_f16_n(x.ctypes.data, y.ctypes.data, x.size)
    return y


def f16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    y = np.empty(h.shape, dtype=np.float32)
    lib().ko_f16_to_f32_n(h.ctypes.data, y.ctypes.data, h.size)
    return y


def quantize_group(x, bits: int):
    """Quantize one group (item 1).  Returns (scale fp16 bits, zero fp16 bits, codes uint8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    codes = np.zeros(x.size, np.uint8)
    lib().ko_quantize_group(x.ctypes.data, x.size, 1, bits, s.ctypes.data, z.ctypes.data,
                            codes.ctypes.data, 1)
    return int(s[0]), int(z[0]), codes


def dequant(code: int, s16: int, z16: int) -> float:
    return float(lib().ko_dequant(code, s16, z16))


def set_threads(n: int) -> int:
    return int(lib().ko_set_threads(int(n)))


def prefill_attention(Q, K, V, t, rows=None) -> np.ndarray:
    """Causal attention of the prompt's queries over its raw fp16 keys and
    values, in double (ko_prefill_attn).  Q: fp16 [b, hq, ts, d]; K, V: fp16
    [b, h, ts, d]; t: tokens per sequence.  Returns float64 [b, hq, ts, d]
    with every row tau < t[i] (zeros elsewhere), or, given ``rows`` (an
    [n, 3] array of (i, qh, tau)), float64 [n, d]: those rows."""
    Q, K, V = _f16(Q), _f16(K), _f16(V)
    b, hq, ts, d = Q.shape
    h = K.shape[1]
    assert K.shape == (b, h, ts, d) and V.shape == K.shape
    t = np.ascontiguousarray(np.broadcast_to(np.asarray(t, np.int32), (b,)))
    if rows is None:
        rp, n = None, 0
        out = np.zeros((b, hq, ts, d), np.float64)
    else:
        rows = np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 3))
        rp, n = rows.ctypes.data, rows.shape[0]
        out = np.zeros((n, d), np.float64)
    rc = lib().ko_prefill_attn(Q.ctypes.data, K.ctypes.data, V.ctypes.data, t.ctypes.data, b, hq, h, ts, d,
                               rp, n, out.ctypes.data)
    if rc != 0:
        raise ValueError(f"ko_prefill_attn failed ({rc})")
    return out


def _f16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float16:
        raise TypeError("fp16 array expected")
    return np.ascontiguousarray(a)


class Cache:
    """The oracle cache: b sequences x h kv heads, natural-order arrays."""

    def __init__(self, b, h, d, kbits, vbits, G, R, cap):
        self.b, self.h, self.d = b, h, d
        self.kbits, self.vbits, self.G, self.R, self.cap = kbits, vbits, G, R, cap
        self._h = ctypes.c_void_p()
        rc = lib().ko_create(b, h, d, kbits, vbits, G, R, cap, ctypes.byref(self._h))
        if rc != 0:
            raise ValueError(f"oracle create failed ({rc})")

    def close(self):
        if self._h:
            lib().ko_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, K, V, t):
        K, V = _f16(K), _f16(V)
        t = np.ascontiguousarray(t, dtype=np.int32)
        if K.shape != V.shape or K.ndim != 4 or K.shape[:2] != (self.b, self.h) or K.shape[3] != self.d:
            raise ValueError("K, V must be [b, h, t_stride, d]")
        rc = lib().ko_prefill(self._h, K.ctypes.data, V.ctypes.data, t.ctypes.data, K.shape[2])
        if rc != 0:
            raise ValueError(f"oracle prefill failed ({rc})")

    def append(self, k, v):
        k, v = _f16(k), _f16(v)
        if k.shape != (self.b, self.h, self.d) or v.shape != k.shape:
            raise ValueError("k, v must be [b, h, d]")
        rc = lib().ko_append(self._h, k.ctypes.data, v.ctypes.data)
        if rc == 3:
            raise OverflowError("oracle capacity exceeded")
        if rc != 0:
            raise ValueError(f"oracle append failed ({rc})")

    def decode(self, q, pairs=None) -> np.ndarray:
        """Attention output fp32 [b, hq, d]; with pairs, only those (seq, qhead) rows are filled."""
        q = _f16(q)
        hq = q.shape[1]
        out = np.zeros((self.b, hq, self.d), np.float32)
        if pairs is None:
            rc = lib().ko_decode(self._h, q.ctypes.data, hq, out.ctypes.data)
        else:
            pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
            rc = lib().ko_decode_subset(self._h, q.ctypes.data, hq, out.ctypes.data,
                                        pr.ctypes.data, pr.shape[0])
        if rc != 0:
            raise ValueError(f"oracle decode failed ({rc})")
        return out

    def decode_probs(self, q, ld=None, pairs=None):
        """(out fp32 [b, hq, d], probs fp32 [b, hq, ld]): the attention output and
        each token's softmax weight (row (i, h) holds T_i weights, zeros after)."""
        q = _f16(q)
        hq = q.shape[1]
        T = self.lengths()[0]
        ld = int(max(1, T.max())) if ld is None else int(ld)
        out = np.zeros((self.b, hq, self.d), np.float32)
        probs = np.zeros((self.b, hq, ld), np.float32)
        pr, npr = None, 0
        if pairs is not None:
            pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
            npr = pr.shape[0]
        rc = lib().ko_decode_probs(self._h, q.ctypes.data, hq, out.ctypes.data, probs.ctypes.data, ld,
                                   None if pr is None else pr.ctypes.data, npr)
        if rc != 0:
            raise ValueError(f"oracle decode failed ({rc})")
        return out, probs

    def lengths(self):
        T = np.zeros(self.b, np.int32)
        Tqk = np.zeros(self.b, np.int32)
        Tqv = np.zeros(self.b, np.int32)
        lib().ko_lengths(self._h, T.ctypes.data, Tqk.ctypes.data, Tqv.ctypes.data)
        return T, Tqk, Tqv

    def dequant_kv(self, i, j):
        T = int(self.lengths()[0][i])
        Kh = np.zeros((max(T, 1), self.d), np.float32)
        Vh = np.zeros((max(T, 1), self.d), np.float32)
        lib().ko_dequant_kv(self._h, i, j, Kh.ctypes.data, Vh.ctypes.data)
        return Kh[:T], Vh[:T]

    def state(self):
        b, h, d, G, R = self.b, self.h, self.d, self.G, self.R
        cg = lib().ko_capacity_stride(self._h)
        st = dict(
            kcode=np.zeros((b, h, d, cg), np.uint8),
            ks=np.zeros((b, h, cg // G, d), np.uint16),
            kz=np.zeros((b, h, cg // G, d), np.uint16),
            vcode=np.zeros((b, h, cg, d), np.uint8),
            vs=np.zeros((b, h, cg, d // G), np.uint16),
            vz=np.zeros((b, h, cg, d // G), np.uint16),
            kf=np.zeros((b, h, R, d), np.uint16),
            vf=np.zeros((b, h, R + 1, d), np.uint16),
        )
        lib().ko_state(self._h, *[st[k].ctypes.data for k in
                                  ("kcode", "ks", "kz", "vcode", "vs", "vz", "kf", "vf")])
        return st

    def export_sizes(self):
        n = [ctypes.c_size_t() for _ in range(6)]
        lib().ko_export_sizes(self._h, *[ctypes.byref(x) for x in n])
        return tuple(int(x.value) for x in n)

    def export(self):
        """The cache in the packed device format (flat arrays; see kivi_oracle.c)."""
        if not lib().ko_export_supported(self._h):
            raise ValueError("shape not representable in the packed format")
        nkc, nksz, nvc, nvsz, nkf, nvf = self.export_sizes()
        ex = dict(Kc=np.zeros(nkc, np.uint32), Ksz=np.zeros(nksz, np.uint16),
                  Vc=np.zeros(nvc, np.uint32), Vsz=np.zeros(nvsz, np.uint16),
                  Kf=np.zeros(nkf, np.uint16), Vf=np.zeros(nvf, np.uint16))
        lib().ko_export(self._h, *[ex[k].ctypes.data for k in ("Kc", "Ksz", "Vc", "Vsz", "Kf", "Vf")])
        return ex
