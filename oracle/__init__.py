"""fp64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package. It shares no code with the CUDA library and imports
nothing from it; it is built from ``oracle.c`` with the host C compiler.

Functions (semantics in ``oracle.c``; source of the method: "[TIL] Optimizing paged
attention", sections "Data Layout", "Baseline" and "V4 (Context-axis parallelism)"):

* ``decode``  -- softmax(scale * q K^T) V per (sequence, query head), two-pass, fp64
* ``partial`` -- the (max, sum, unnormalised accumulator) state of one token range
* ``combine`` -- log-sum-exp merge of such states
* ``append_kv`` -- the cache write of one new token per sequence
* ``prefill`` -- causal attention of several new tokens per sequence
* ``half_to_double`` -- the exact binary16 widening the oracle uses
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", _SRC, "-o", tmp,
            "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i32 = ctypes.c_int
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_decode.restype = i32
    lib.oracle_decode.argtypes = [i32] * 8 + [p] * 5 + [ctypes.c_double, p, ctypes.c_int64, p,
                                                      i32]
    lib.oracle_partial.restype = i32
    lib.oracle_partial.argtypes = [i32] * 8 + [p] * 5 + [ctypes.c_double, ctypes.c_int64, i32,
                                                       i32, p, p, p]
    lib.oracle_combine.restype = None
    lib.oracle_combine.argtypes = [i32, i32, p, p, p, p]
    lib.oracle_prefill.restype = i32
    lib.oracle_prefill.argtypes = [i32] * 8 + [p] * 6 + [ctypes.c_double, p, ctypes.c_int64, p, i32]
    lib.oracle_append_kv.restype = i32
    lib.oracle_append_kv.argtypes = [i32] * 8 + [p] * 6
    lib.oracle_max_threads.restype = i32
    lib.oracle_max_threads.argtypes = []
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _inputs(w):
    q = np.ascontiguousarray(w.query, dtype=np.float16).view(np.uint16)
    k = np.ascontiguousarray(w.key_cache, dtype=np.float16).view(np.uint16)
    v = np.ascontiguousarray(w.value_cache, dtype=np.float16).view(np.uint16)
    bt = np.ascontiguousarray(w.block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(w.context_lengths, dtype=np.int32)
    dims = [int(w.batch), int(w.query_heads), int(w.kv_heads), int(w.head_dim),
            int(w.page_size), int(w.max_pages_per_sequence), int(w.num_physical_pages),
            int(getattr(w, "cache_layout", 0))]
    return dims, q, k, v, bt, ctx


class Oracle:
    """The oracle functions bound to one compiled copy of ``oracle.c``."""

    def __init__(self, path: str = None):
        self._lib = _bind(path) if path else _load()

    def max_threads(self) -> int:
        return int(self._lib.oracle_max_threads())

    def half_to_double(self, bits: int) -> float:
        return float(self._lib.oracle_half_to_double(int(bits) & 0xFFFF))

    def decode(self, w, rows=None, scale=None, threads: int = 0) -> np.ndarray:
        """fp64 output. ``rows=None``: shape [batch, query_heads, head_dim]; otherwise the
        listed flat rows ``b * query_heads + h``, shape [len(rows), head_dim]."""
        lib = self._lib
        dims, q, k, v, bt, ctx = _inputs(w)
        s = float(w.scale if scale is None else scale)
        if rows is None:
            out = np.zeros((w.batch, w.query_heads, w.head_dim), dtype=np.float64)
            rc = lib.oracle_decode(*dims, _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(ctx), s, None,
                                   0, _ptr(out), int(threads))
        else:
            r = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
            out = np.zeros((r.size, w.head_dim), dtype=np.float64)
            rc = lib.oracle_decode(*dims, _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(ctx), s,
                                   _ptr(r), int(r.size), _ptr(out), int(threads))
        if rc:
            raise ValueError(f"oracle_decode rejected the inputs (code {rc})")
        return out

    def partial(self, w, row: int, t0: int, t1: int, scale=None):
        """(m, l, acc[head_dim]) of flat row ``b * query_heads + h`` over tokens [t0, t1)."""
        lib = self._lib
        dims, q, k, v, bt, ctx = _inputs(w)
        s = float(w.scale if scale is None else scale)
        m = np.zeros(1)
        l = np.zeros(1)
        acc = np.zeros(w.head_dim)
        rc = lib.oracle_partial(*dims, _ptr(q), _ptr(k), _ptr(v), _ptr(bt), _ptr(ctx), s,
                                int(row), int(t0), int(t1), _ptr(m), _ptr(l), _ptr(acc))
        if rc:
            raise ValueError(f"oracle_partial rejected the inputs (code {rc})")
        return float(m[0]), float(l[0]), acc

    def prefill(self, w, query, query_start, rows=None, scale=None, threads: int = 0):
        """Causal multi-token attention: query [total][qh][hd] fp16 holds each sequence's
        last n_b tokens (n_b = query_start[b+1] - query_start[b]). fp64 output [total][qh][hd]
        (or the listed flat rows i * qh + h)."""
        lib = self._lib
        dims, _, k, v, bt, ctx = _inputs(w)
        qq = np.ascontiguousarray(query, dtype=np.float16).view(np.uint16)
        qs = np.ascontiguousarray(query_start, dtype=np.int32)
        s = float(w.scale if scale is None else scale)
        total = int(qs[-1])
        if rows is None:
            out = np.zeros((total, w.query_heads, w.head_dim))
            rc = lib.oracle_prefill(*dims, _ptr(qq), _ptr(qs), _ptr(k), _ptr(v), _ptr(bt), _ptr(ctx),
                                    s, None, 0, _ptr(out), int(threads))
        else:
            r = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
            out = np.zeros((r.size, w.head_dim))
            rc = lib.oracle_prefill(*dims, _ptr(qq), _ptr(qs), _ptr(k), _ptr(v), _ptr(bt), _ptr(ctx),
                                    s, _ptr(r), int(r.size), _ptr(out), int(threads))
        if rc:
            raise ValueError(f"oracle_prefill rejected the inputs (code {rc})")
        return out

    def append_kv(self, w, new_key, new_value):
        """Caches after appending new_key/new_value ([batch][kv_heads][head_dim] fp16) at
        token index context_lengths[b]; returns (key_cache, value_cache, flags)."""
        lib = self._lib
        dims, q, k, v, bt, ctx = _inputs(w)
        k = k.copy()
        v = v.copy()
        nk = np.ascontiguousarray(new_key, dtype=np.float16).view(np.uint16)
        nv = np.ascontiguousarray(new_value, dtype=np.float16).view(np.uint16)
        rc = lib.oracle_append_kv(*dims, _ptr(nk), _ptr(nv), _ptr(bt), _ptr(ctx), _ptr(k), _ptr(v))
        if rc < 0:
            raise ValueError("oracle_append_kv rejected the dimensions")
        return k.view(np.float16), v.view(np.float16), int(rc)

    def combine(self, m, l, acc) -> np.ndarray:
        """Log-sum-exp merge of states m[n], l[n], acc[n, head_dim] -> normalised row."""
        lib = self._lib
        m = np.ascontiguousarray(m, dtype=np.float64).reshape(-1)
        l = np.ascontiguousarray(l, dtype=np.float64).reshape(-1)
        acc = np.ascontiguousarray(acc, dtype=np.float64)
        n = m.size
        hd = acc.shape[-1]
        acc = acc.reshape(n, hd)
        out = np.zeros(hd)
        lib.oracle_combine(int(n), int(hd), _ptr(m), _ptr(l), _ptr(acc), _ptr(out))
        return out


_default = None


def _oracle() -> "Oracle":
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def max_threads() -> int:
    return _oracle().max_threads()


def half_to_double(bits: int) -> float:
    return _oracle().half_to_double(bits)


def decode(w, rows=None, scale=None, threads: int = 0) -> np.ndarray:
    return _oracle().decode(w, rows=rows, scale=scale, threads=threads)


def partial(w, row: int, t0: int, t1: int, scale=None):
    return _oracle().partial(w, row, t0, t1, scale=scale)


def combine(m, l, acc) -> np.ndarray:
    return _oracle().combine(m, l, acc)


def append_kv(w, new_key, new_value):
    return _oracle().append_kv(w, new_key, new_value)


def prefill(w, query, query_start, rows=None, scale=None, threads: int = 0):
    return _oracle().prefill(w, query, query_start, rows=rows, scale=scale, threads=threads)
