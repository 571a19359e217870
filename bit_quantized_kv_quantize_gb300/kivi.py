"""Thin Python binding of libkivi's C ABI (include/kivi.h).

Argument marshalling only: every step of the cache and of decode attention
runs in the library's CUDA kernels.  torch supplies device memory and the
current CUDA stream.  There is no fallback: if libkivi.so is missing or
fails to load, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkivi.so")

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "capacity exceeded",
          4: "poisoned", 5: "CUDA error", 6: "out of memory"}

EXPORTS = ["kivi_cache_create", "kivi_cache_destroy", "kivi_prefill", "kivi_append",
           "kivi_decode_attn", "kivi_cache_lengths", "kivi_cache_export_sizes",
           "kivi_cache_export", "kivi_cache_check", "kivi_profile_enable", "kivi_profile_read",
           "kivi_decode_plan", "kivi_status_str", "kivi_last_error", "kivi_abi_version",
           "kivi_decode_attn_noalloc", "kivi_cache_export_records", "kivi_append_decode",
           "kivi_decode_attn_probs", "kivi_plan_preview", "kivi_prefill_attn"]


class KiviError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class CapacityError(KiviError):
    pass


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, st = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
    L.kivi_cache_create.argtypes = [i32] * 8 + [ctypes.POINTER(vp)]
    L.kivi_cache_destroy.argtypes = [vp]
    L.kivi_prefill.argtypes = [vp, vp, vp, vp, i32, vp]
    L.kivi_prefill_attn.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, vp]
    L.kivi_append.argtypes = [vp, vp, vp, vp]
    L.kivi_decode_attn.argtypes = [vp, vp, i32, vp, vp]
    L.kivi_decode_attn_probs.argtypes = [vp, vp, i32, vp, vp, vp, ctypes.c_int64, vp]
    L.kivi_plan_preview.argtypes = [i32] * 9 + [vp, vp, vp, i32, vp]
    L.kivi_cache_lengths.argtypes = [vp, vp, vp, vp]
    L.kivi_cache_export_sizes.argtypes = [vp, ctypes.POINTER(ctypes.c_size_t)]
    L.kivi_cache_export.argtypes = [vp] * 8
    L.kivi_cache_check.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    L.kivi_profile_enable.argtypes = [vp, i32]
    L.kivi_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32)]
    L.kivi_decode_plan.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.kivi_status_str.restype = ctypes.c_char_p
    L.kivi_status_str.argtypes = [st]
    L.kivi_last_error.restype = ctypes.c_char_p
    for name in EXPORTS:
        f = getattr(L, name)
        if name not in ("kivi_status_str", "kivi_last_error"):
            f.restype = ctypes.c_int
    return L


lib = _load()


def _check(rc: int):
    if rc != 0:
        msg = lib.kivi_last_error().decode()
        raise (CapacityError if rc == 3 else KiviError)(rc, msg)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev_f32_rows(x, lead, name):
    """Pointer of a contiguous CUDA fp32 tensor [*lead, ld]."""
    import torch
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.float32):
        raise TypeError(f"{name} must be a CUDA float32 tensor")
    if x.dim() != len(lead) + 1 or tuple(x.shape[:-1]) != tuple(lead) or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [{', '.join(map(str, lead))}, ld] tensor")
    return x.data_ptr()


def _dev_fp16(x, shape, name):
    import torch
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float16:
        raise TypeError(f"{name} must be a CUDA float16 tensor")
    if tuple(x.shape) != tuple(shape) or not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous with shape {tuple(shape)}, got {tuple(x.shape)}")
    return ctypes.c_void_p(x.data_ptr())


class KiviCache:
    """A KIVI quantized KV cache of b sequences x h_kv heads on the current GPU."""

    def __init__(self, b, h_kv, d, k_bits=2, v_bits=2, G=32, R=128, max_tokens=4096):
        self.b, self.h_kv, self.d = b, h_kv, d
        self.k_bits, self.v_bits, self.G, self.R = k_bits, v_bits, G, R
        self.max_tokens = max_tokens
        self._h = ctypes.c_void_p()
        _check(lib.kivi_cache_create(b, h_kv, d, k_bits, v_bits, G, R, max_tokens,
                                     ctypes.byref(self._h)))

    # -- lifecycle ---------------------------------------------------------
    def close(self):
        if self._h:
            h, self._h = self._h, ctypes.c_void_p()
            _check(lib.kivi_cache_destroy(h))

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    # -- hot path ----------------------------------------------------------
    def prefill(self, K, V, t, stream=None):
        """K, V: CUDA fp16 [b, h_kv, t_stride, d]; t: per-sequence token counts."""
        t = np.ascontiguousarray(np.broadcast_to(np.asarray(t, np.int32), (self.b,)))
        ts = K.shape[2]
        kp = _dev_fp16(K, (self.b, self.h_kv, ts, self.d), "K")
        vp = _dev_fp16(V, (self.b, self.h_kv, ts, self.d), "V")
        _check(lib.kivi_prefill(self._h, kp, vp, t.ctypes.data, ts, _stream(stream)))

    def prefill_attn(self, Q, K, V, t, out=None, stream=None):
        """prefill(K, V, t) and the prompt's causal attention: Q CUDA fp16
        [b, h_q, t_stride, d] -> out (same shape; rows past each sequence's
        length untouched).  One launch."""
        import torch
        t = np.ascontiguousarray(np.broadcast_to(np.asarray(t, np.int32), (self.b,)))
        ts, hq = K.shape[2], Q.shape[1]
        qp = _dev_fp16(Q, (self.b, hq, ts, self.d), "Q")
        kp = _dev_fp16(K, (self.b, self.h_kv, ts, self.d), "K")
        vp = _dev_fp16(V, (self.b, self.h_kv, ts, self.d), "V")
        if out is None:
            out = torch.zeros_like(Q)
        op = _dev_fp16(out, (self.b, hq, ts, self.d), "out")
        _check(lib.kivi_prefill_attn(self._h, qp, kp, vp, t.ctypes.data, ts, hq, op, _stream(stream)))
        return out

    def append(self, k, v, stream=None):
        """k, v: CUDA fp16 [b, h_kv, d]."""
        kp = _dev_fp16(k, (self.b, self.h_kv, self.d), "k")
        vp = _dev_fp16(v, (self.b, self.h_kv, self.d), "v")
        _check(lib.kivi_append(self._h, kp, vp, _stream(stream)))

    def decode(self, q, out=None, stream=None):
        """q: CUDA fp16 [b, h_q, d] -> out CUDA fp16 [b, h_q, d]."""
        import torch
        hq = q.shape[1]
        qp = _dev_fp16(q, (self.b, hq, self.d), "q")
        if out is None:
            out = torch.empty_like(q)
        op = _dev_fp16(out, (self.b, hq, self.d), "out")
        _check(lib.kivi_decode_attn(self._h, qp, hq, op, _stream(stream)))
        return out

    def decode_probs(self, q, probs, mass=None, out=None, stream=None):
        """decode(q), and each token's softmax weight into probs (CUDA fp32
        [b, h_q, ld], ld >= every sequence's length; entries past a
        sequence's length untouched); mass (same shape, optional) += probs.
        Returns out."""
        import torch
        hq = q.shape[1]
        qp = _dev_fp16(q, (self.b, hq, self.d), "q")
        if out is None:
            out = torch.empty_like(q)
        op = _dev_fp16(out, (self.b, hq, self.d), "out")
        pp = _dev_f32_rows(probs, (self.b, hq), "probs")
        mp = 0
        if mass is not None:
            if tuple(mass.shape) != tuple(probs.shape):
                raise ValueError("mass must have the shape of probs")
            mp = _dev_f32_rows(mass, (self.b, hq), "mass")
        _check(lib.kivi_decode_attn_probs(self._h, qp, hq, op, pp, mp or None, probs.shape[2],
                                          _stream(stream)))
        return out

    def append_decode(self, k, v, q, out=None, stream=None):
        """append(k, v) then decode(q) in one call; returns out.

        One launch where the decode kernel appends the token itself (see
        kivi_append_decode in kivi.h for when), else the append kernel and
        the decode kernel as its programmatic dependent."""
        import torch
        hq = q.shape[1]
        kp = _dev_fp16(k, (self.b, self.h_kv, self.d), "k")
        vp = _dev_fp16(v, (self.b, self.h_kv, self.d), "v")
        qp = _dev_fp16(q, (self.b, hq, self.d), "q")
        if out is None:
            out = torch.empty_like(q)
        op = _dev_fp16(out, (self.b, hq, self.d), "out")
        _check(lib.kivi_append_decode(self._h, kp, vp, qp, hq, op, _stream(stream)))
        return out

    # -- inspection ----------------------------------------------------------
    def lengths(self):
        T = np.zeros(self.b, np.int32)
        Tqk = np.zeros(self.b, np.int32)
        Tqv = np.zeros(self.b, np.int32)
        _check(lib.kivi_cache_lengths(self._h, T.ctypes.data, Tqk.ctypes.data, Tqv.ctypes.data))
        return T, Tqk, Tqv

    def export(self, stream=None):
        """The whole device state in the packed format (host numpy arrays)."""
        sz = (ctypes.c_size_t * 6)()
        _check(lib.kivi_cache_export_sizes(self._h, sz))
        dt = [np.uint32, np.uint16, np.uint32, np.uint16, np.uint16, np.uint16]
        arrs = [np.zeros(int(n) // np.dtype(t).itemsize, t) for n, t in zip(sz, dt)]
        _check(lib.kivi_cache_export(self._h, *[a.ctypes.data for a in arrs], _stream(stream)))
        return dict(zip(["Kc", "Ksz", "Vc", "Vsz", "Kf", "Vf"], arrs))

    def export_records(self, stream=None) -> np.ndarray:
        """The packed arrays as the device stores them (block records, uint8)."""
        n = ctypes.c_size_t(0)
        _check(lib.kivi_cache_export_records(self._h, None, ctypes.byref(n), _stream(stream)))
        buf = np.zeros(int(n.value), np.uint8)
        _check(lib.kivi_cache_export_records(self._h, buf.ctypes.data, ctypes.byref(n), _stream(stream)))
        return buf

    def check(self, stream=None) -> int:
        f = ctypes.c_uint32(0)
        _check(lib.kivi_cache_check(self._h, ctypes.byref(f), _stream(stream)))
        return int(f.value)

    def profile(self, on: bool):
        _check(lib.kivi_profile_enable(self._h, 1 if on else 0))

    def profile_read(self):
        ms = ctypes.c_double(0)
        n = ctypes.c_int(0)
        _check(lib.kivi_profile_read(self._h, ctypes.byref(ms), ctypes.byref(n)))
        return float(ms.value), int(n.value)

    def plan(self):
        s = ctypes.c_int(0)
        n = ctypes.c_int(0)
        _check(lib.kivi_decode_plan(self._h, ctypes.byref(s), ctypes.byref(n)))
        return int(s.value), int(n.value)
