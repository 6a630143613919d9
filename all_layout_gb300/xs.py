"""ctypes binding of libxs (include/xs.h): argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; this module
turns torch CUDA tensors into device pointers and a stream handle and raises
``XsError`` on a non-OK status. Importing it loads ``libxs.so`` and fails
loudly if the library has not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libxs.so")
_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "include", "xs.h")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_ALIGN, ERR_CUDA, ERR_TIMEOUT = range(6)
FLAG_COMPLETION_COUPLED = 1
MAX_SHARDS = 8


class XsError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"libxs.so is not built ({_LIB_PATH}); run __graft_entry__.build()")
_lib = ctypes.CDLL(_LIB_PATH)

_vp, _i = ctypes.c_void_p, ctypes.c_int
_PP = ctypes.POINTER(ctypes.c_void_p)
_lib.xs_attn_fused.argtypes = [_vp, _vp, _vp, _PP, _i, _i, _i, _i, _i, _i, _vp]
_lib.xs_attn_fused_ex.argtypes = [_vp, _vp, _vp, _PP, _i, _i, _i, _i, _i, _i, _i, _vp, _vp]
_lib.xs_attn.argtypes = [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]
_lib.xs_scatter.argtypes = [_vp, _PP, _i, _i, _i, _i, _i, _vp]
_lib.xs_attn_serial.argtypes = [_vp, _vp, _vp, _vp, _PP, _i, _i, _i, _i, _i, _vp]
_lib.xs_attn_ulysses.argtypes = [_PP, _PP, _PP, _PP] + [_i] * 8 + [_vp]
_lib.xs_store_burst_probe.argtypes = [_vp, ctypes.c_ulonglong, _i, ctypes.c_ulonglong, _i,
                                      ctypes.c_ulonglong, _i, _vp, _vp]
_lib.xs_attn_serial_noalloc.argtypes = [_vp, _vp, _vp, _PP, _i, _i, _i, _i, _i, _vp]
for _f in ("xs_attn_fused", "xs_attn_fused_ex", "xs_attn", "xs_scatter", "xs_attn_serial", "xs_attn_serial_noalloc",
           "xs_attn_ulysses", "xs_store_burst_probe",
           "xs_last_device_status", "xs_selftest_bounded_wait"):
    getattr(_lib, _f).restype = _i
_lib.xs_status_string.argtypes = [_i]
_lib.xs_status_string.restype = ctypes.c_char_p
_lib.xs_last_device_status.argtypes = [_vp]
_lib.xs_selftest_bounded_wait.argtypes = [_vp]
_lib.xs_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
_lib.xs_set_wait_limit_ns.restype = ctypes.c_ulonglong
_lib.xs_abi_version.restype = _i
_lib.xs_selftest_exp2.argtypes = [_vp, _vp, _vp, _i, _vp]
_lib.xs_selftest_exp2.restype = _i
_lib.xs_set_workspace.argtypes = [_vp, ctypes.c_ulonglong, _vp]
_lib.xs_set_workspace.restype = _i
_lib.xs_workspace_bytes.argtypes = [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_ulonglong),
                                    ctypes.POINTER(ctypes.c_int)]
_lib.xs_workspace_bytes.restype = _i


def library():
    """The loaded ctypes library (for direct C-ABI calls)."""
    return _lib


def library_path() -> str:
    return _LIB_PATH


def declared_symbols():
    """Function names declared in include/xs.h."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"\b(xs_[a-z_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return _lib.xs_status_string(int(status)).decode()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def _shard_array(shards):
    arr = (ctypes.c_void_p * max(1, len(shards)))()
    for i, s in enumerate(shards):
        arr[i] = s if isinstance(s, int) else (s.data_ptr() if s is not None else None)
    return ctypes.cast(arr, _PP), arr


def _check(status, what):
    if status != OK:
        raise XsError(status, what)


def _dims(q):
    B, H, N, d = q.shape
    return int(B), int(N), int(H), int(d)


def attn_fused(q, k, v, shards, store_tile: int = 8, stream=None):
    """Fused attention + shard layout. q, k, v: [B, H, N, d] bf16 CUDA tensors;
    shards: P tensors [B, N/P, H, d] bf16."""
    B, N, H, d = _dims(q)
    pp, keep = _shard_array(shards)
    _check(_lib.xs_attn_fused(_ptr(q), _ptr(k), _ptr(v), pp, B, N, H, d, len(shards),
                              int(store_tile), _stream(stream)), "xs_attn_fused")


def attn_fused_ex(q, k, v, shards, store_tile: int = 8, flags: int = 0, spans=None,
                  stream=None):
    """xs_attn_fused_ex: optional completion-coupled stores and per-tile store
    spans (spans: an int64 CUDA tensor of 2*B*H*(N/128) entries, or None)."""
    B, N, H, d = _dims(q)
    pp, keep = _shard_array(shards)
    _check(_lib.xs_attn_fused_ex(_ptr(q), _ptr(k), _ptr(v), pp, B, N, H, d, len(shards),
                                 int(store_tile), int(flags), _ptr(spans), _stream(stream)),
           "xs_attn_fused_ex")


def attn(q, k, v, o, stream=None):
    """Attention alone into o [B, H, N, d] bf16."""
    B, N, H, d = _dims(q)
    _check(_lib.xs_attn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, N, H, d, _stream(stream)),
           "xs_attn")


def scatter(o, shards, stream=None):
    """Layout alone: o [B, H, N, d] -> shards."""
    B, N, H, d = _dims(o)
    pp, keep = _shard_array(shards)
    _check(_lib.xs_scatter(_ptr(o), pp, B, N, H, d, len(shards), _stream(stream)), "xs_scatter")


def attn_serial(q, k, v, o_scratch, shards, stream=None):
    """Serial execution: attention into o_scratch, then the layout kernel."""
    B, N, H, d = _dims(q)
    pp, keep = _shard_array(shards)
    _check(_lib.xs_attn_serial(_ptr(q), _ptr(k), _ptr(v), _ptr(o_scratch), pp, B, N, H, d,
                               len(shards), _stream(stream)), "xs_attn_serial")


def attn_ulysses(q_shards, k_shards, v_shards, out_shards, h0, H, store_tile: int = 8,
                 stream=None):
    """Both Ulysses All-to-Alls fused: q/k/v_shards are P sequence shards
    [B, N/P, H_total, d]; computes heads [h0, h0 + H) and stores them into
    out_shards [B, N/P, H_total, d]."""
    B, R, H_total, d = (int(x) for x in q_shards[0].shape)
    P = len(q_shards)
    qp, kq = _shard_array(q_shards)
    kp, kk = _shard_array(k_shards)
    vp, kv = _shard_array(v_shards)
    op, ko = _shard_array(out_shards)
    _check(_lib.xs_attn_ulysses(qp, kp, vp, op, B, R * P, H_total, int(h0), int(H), d, P,
                                int(store_tile), _stream(stream)), "xs_attn_ulysses")


def attn_serial_noalloc(q, k, v, shards, stream=None):
    """Serial execution with the intermediate o kept in the library's fixed
    scratch array (no device allocation; see xs_attn_serial_noalloc in xs.h)."""
    B, N, H, d = _dims(q)
    pp, keep = _shard_array(shards)
    _check(_lib.xs_attn_serial_noalloc(_ptr(q), _ptr(k), _ptr(v), pp, B, N, H, d, len(shards),
                                       _stream(stream)), "xs_attn_serial_noalloc")


def store_burst_probe(dst, K, burst_bytes, n_bursts, gap_ns, mode, times, stream=None):
    """Store-burst probe (see xs_store_burst_probe): dst a uint8 CUDA tensor,
    times an int64 CUDA tensor of 2*K*n_bursts entries."""
    _check(_lib.xs_store_burst_probe(_ptr(dst), dst.numel() * dst.element_size(), int(K),
                                     int(burst_bytes), int(n_bursts), int(gap_ns), int(mode),
                                     _ptr(times), _stream(stream)), "xs_store_burst_probe")


def last_device_status(stream=None) -> int:
    return int(_lib.xs_last_device_status(_stream(stream)))


def set_wait_limit_ns(limit_ns: int) -> int:
    return int(_lib.xs_set_wait_limit_ns(int(limit_ns)))


def selftest_bounded_wait(stream=None):
    _check(_lib.xs_selftest_bounded_wait(_stream(stream)), "xs_selftest_bounded_wait")


def selftest_exp2(x, stream=None):
    """(polynomial 2^x, MUFU 2^x) for a float32 CUDA tensor x (see xs_selftest_exp2)."""
    x = x.contiguous()
    poly, mufu = torch.empty_like(x), torch.empty_like(x)
    _check(_lib.xs_selftest_exp2(_ptr(x), _ptr(poly), _ptr(mufu), x.numel(), _stream(stream)),
           "xs_selftest_exp2")
    return poly, mufu


def alloc_shards(B, N, H, d, P, device="cuda"):
    """P separate destination buffers [B, N/P, H, d] bf16 (one allocation each)."""
    return [torch.empty((B, N // P, H, d), dtype=torch.bfloat16, device=device)
            for _ in range(P)]


def set_workspace(ws=None, stream=None):
    """Registers a caller-owned uint8 CUDA tensor as the workspace of the
    balanced (stream-K) schedule on its device (None removes it). Keep the
    tensor alive while registered."""
    if ws is None:
        _check(_lib.xs_set_workspace(None, 0, _stream(stream)), "xs_set_workspace")
        return
    if not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    _check(_lib.xs_set_workspace(ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "xs_set_workspace")


def workspace_bytes(B: int, N: int, H: int, d: int):
    """(bytes, cut): the workspace a launch of this shape would use with ample
    workspace, and 1 if it would take the balanced schedule (else 0)."""
    b, sp = ctypes.c_ulonglong(0), ctypes.c_int(0)
    _check(_lib.xs_workspace_bytes(B, N, H, d, ctypes.byref(b), ctypes.byref(sp)),
           "xs_workspace_bytes")
    return int(b.value), int(sp.value)


def alloc_workspace(B: int, N: int, H: int, d: int, device="cuda"):
    """Allocates (through torch) and registers the workspace a shape needs;
    returns the tensor (None when that shape keeps whole units)."""
    n, _ = workspace_bytes(B, N, H, d)
    if n == 0:
        return None
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    set_workspace(ws)
    return ws
