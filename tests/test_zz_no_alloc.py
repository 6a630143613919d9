"""xs_attn_serial_noalloc: serial attention-then-layout for callers that cannot
allocate device memory (a host framework that owns all device memory through
its own allocator or a fixed memory plan, or a loop where cudaMalloc would
synchronise the device). The intermediate o lives in a fixed array inside the
library instead of a caller-supplied buffer.

Both entry points run the same two deterministic kernels on the same inputs;
only where the intermediate o lives differs. So the output of
xs_attn_serial_noalloc must equal the output of xs_attn_serial byte for byte, on
two calls in a row, and also after a larger call has left its o in the array
(a smaller call must read only what it wrote); one shape is also checked
against the fp64 oracle within the tolerance every parity test uses. This file
is collected last so that a stop-at-first-failure run has already run every
other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from all_layout_gb300 import inputs
from gpu_util import assert_close, shards_f64


@pytest.fixture(scope="module")
def xs():
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs as _xs
    return _xs


def _call_noalloc(xs, q, k, v, shards, B, N, H, d, stream):
    """Direct C-ABI call; returns the status code."""
    lib = xs.library()
    arr = (ctypes.c_void_p * len(shards))(*[s.data_ptr() for s in shards])
    pp = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    return lib.xs_attn_serial_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), pp, B, N, H, d,
                                      len(shards), ctypes.c_void_p(stream.cuda_stream))


def _bits(shards):
    return np.stack([s.cpu().view(torch.int16).numpy() for s in shards])


@pytest.mark.gpu
def test_noalloc_matches_serial_on_two_calls(xs):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    # The larger case (24 MiB of o) comes first, so the smaller calls after it run
    # on an array that still holds the larger call's o.
    cases = [(1, 6, 1024, 128, 8, 42), (2, 12, 4096, 128, 8, 43), (1, 4, 256, 64, 2, 41),
             (1, 6, 1024, 128, 8, 42)]
    for (B, H, N, d, P, seed) in cases:
        q, k, v = (t.cuda() for t in inputs.qkv(B, N, H, d, seed=seed))
        ref_shards = xs.alloc_shards(B, N, H, d, P)
        scratch = torch.empty_like(q)
        xs.attn_serial(q, k, v, scratch, ref_shards, stream=stream)
        ref = _bits(ref_shards)
        for call in range(2):
            got_shards = xs.alloc_shards(B, N, H, d, P)
            for s in got_shards:
                s.fill_(float("nan"))
            assert _call_noalloc(xs, q, k, v, got_shards, B, N, H, d, stream) == xs.OK
            torch.cuda.synchronize()
            assert xs.last_device_status() == xs.OK
            assert np.array_equal(_bits(got_shards), ref), \
                f"noalloc B{B} H{H} N{N} d{d} call {call}: bytes differ from xs_attn_serial"


@pytest.mark.gpu
def test_noalloc_against_oracle(xs):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    B, H, N, d, P = 1, 3, 640, 128, 5
    qh, kh, vh = inputs.qkv(B, N, H, d, seed=44)
    q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
    shards = xs.alloc_shards(B, N, H, d, P)
    for s in shards:
        s.fill_(float("nan"))
    assert _call_noalloc(xs, q, k, v, shards, B, N, H, d, stream) == xs.OK
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    assert_close(shards_f64(shards), oracle.shard_layout(oracle.attention(qh, kh, vh), P),
                 "noalloc vs oracle")


def test_noalloc_rejects_oversize(xs):
    """A problem whose intermediate o exceeds the fixed array is refused before
    any device work (no pointer is dereferenced)."""
    lib = xs.library()
    A = 0x10000
    arr = (ctypes.c_void_p * 8)(*([A] * 8))
    pp = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    # 1 x 24 x 8192 x 128 x 2 bytes = 48 MiB > 32 MiB
    assert lib.xs_attn_serial_noalloc(A, A, A, pp, 1, 8192, 24, 128, 8, None) == xs.ERR_INVALID
    assert lib.xs_attn_serial_noalloc(A, A, A, pp, -1, 256, 4, 64, 2, None) == xs.ERR_INVALID
    # B*H*N*d = 2^120 wraps to 0 in 64 bits: still refused
    big = 1 << 30
    assert lib.xs_attn_serial_noalloc(A, A, A, pp, big, big, big, big, 8, None) == xs.ERR_INVALID
