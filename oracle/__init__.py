"""CPU oracle for fused attention + Ulysses post-attention All-to-All layout.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package. The
product path (``all_layout_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, POSIX threads); this module
builds it with gcc and marshals numpy arrays through ctypes. See ``oracle.c``
for the definitions and the passages of the X-Stage pages they follow:

* ``attention``       - exact softmax(q k^T / sqrt(d)) v per (batch, head)
                        (pith.science review, glossary "FlashAttention"; Fig. 5 (d)).
* ``attention_rows``  - the same, only for a list of query rows (row sample).
* ``shard_layout``    - o[B][H][N][d] -> recv[P][B][N/P][H][d] (Fig. 5 (d)-(e):
                        the post-attention All-to-All restores the sequence partition).
* ``shard_layout_inverse`` - recv back to o.

Pins (tests that tie this oracle to something other than itself) are in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no -march)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_attention.argtypes = [u16p, u16p, u16p, f64p] + [ctypes.c_int] * 5
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = ([u16p, u16p, u16p, i64p, ctypes.c_int, f64p]
                                              + [ctypes.c_int] * 5)
        lib.oracle_attention_rows.restype = ctypes.c_int
        for name in ("oracle_shard_layout", "oracle_shard_layout_inverse"):
            fn = getattr(lib, name)
            fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 6
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _bits(a) -> np.ndarray:
    """Accept a numpy uint16 array of bf16 bits or a torch bf16 CPU tensor."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        a = a.contiguous().view(dtype=__import__("torch").int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {a.dtype}")
    return a


def attention(q, k, v, threads: int | None = None) -> np.ndarray:
    """Exact attention in fp64. q, k, v: [B, H, N, d] bf16 -> float64 [B, H, N, d]."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    if not (q.shape == k.shape == v.shape and q.ndim == 4):
        raise ValueError("q, k, v must all be [B, H, N, d]")
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d), dtype=np.float64)
    lib = _load()
    rc = lib.oracle_attention(
        q.ctypes.data_as(lib.oracle_attention.argtypes[0]),
        k.ctypes.data_as(lib.oracle_attention.argtypes[1]),
        v.ctypes.data_as(lib.oracle_attention.argtypes[2]),
        o.ctypes.data_as(lib.oracle_attention.argtypes[3]),
        B, N, H, d, threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attention failed ({rc})")
    return o


def attention_rows(q, k, v, rows, threads: int | None = None) -> np.ndarray:
    """Exact attention for the query rows ``rows`` of every (b, h).

    Returns float64 [B, H, len(rows), d]; row t is query row ``rows[t]``.
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.zeros((B, H, rows.size, d), dtype=np.float64)
    lib = _load()
    fn = lib.oracle_attention_rows
    rc = fn(q.ctypes.data_as(fn.argtypes[0]), k.ctypes.data_as(fn.argtypes[1]),
            v.ctypes.data_as(fn.argtypes[2]), rows.ctypes.data_as(fn.argtypes[3]),
            int(rows.size), o.ctypes.data_as(fn.argtypes[5]),
            B, N, H, d, threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed ({rc})")
    return o


def shard_layout(o: np.ndarray, P: int) -> np.ndarray:
    """o [B, H, N, d] (any dtype) -> recv [P, B, N/P, H, d], bit for bit."""
    o = np.ascontiguousarray(o)
    B, H, N, d = o.shape
    if N % P:
        raise ValueError("N must be divisible by P")
    out = np.empty((P, B, N // P, H, d), dtype=o.dtype)
    rc = _load().oracle_shard_layout(o.ctypes.data, out.ctypes.data, B, N, H, d, P,
                                     o.dtype.itemsize)
    if rc != 0:
        raise RuntimeError(f"oracle_shard_layout failed ({rc})")
    return out


def shard_layout_inverse(recv: np.ndarray) -> np.ndarray:
    """recv [P, B, N/P, H, d] -> o [B, H, N, d], bit for bit."""
    recv = np.ascontiguousarray(recv)
    P, B, R, H, d = recv.shape
    N = P * R
    out = np.empty((B, H, N, d), dtype=recv.dtype)
    rc = _load().oracle_shard_layout_inverse(recv.ctypes.data, out.ctypes.data,
                                             B, N, H, d, P, recv.dtype.itemsize)
    if rc != 0:
        raise RuntimeError(f"oracle_shard_layout_inverse failed ({rc})")
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (bits << 16 as fp32)."""
    b = _bits(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
