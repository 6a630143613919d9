"""C-ABI library checks that need no GPU: it builds, loads, exports every
symbol include/xs.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import re
import subprocess

import pytest

ROOT_HEADER = "include/xs.h"


@pytest.fixture(scope="module")
def xs():
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs as _xs
    return _xs


def test_exports_every_declared_symbol(xs):
    declared = xs.declared_symbols()
    assert {"xs_attn_fused", "xs_attn", "xs_scatter", "xs_attn_serial"} <= set(declared)
    out = subprocess.run(["nm", "-D", "--defined-only", xs.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (xs_\w+)", out))
    missing = [s for s in declared if s not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for s in declared:
        assert hasattr(xs.library(), s)


def test_status_strings(xs):
    for code in range(6):
        assert xs.status_string(code)
    assert "unknown" in xs.status_string(99)
    assert xs.library().xs_abi_version() == 1


A = 0x10000   # a 16-byte aligned fake device address; never dereferenced


def _fused(xs, q=A, k=A, v=A, shards=(A, A), B=1, N=256, H=4, d=64, P=None, st=8):
    lib = xs.library()
    arr = (ctypes.c_void_p * max(1, len(shards)))(*shards)
    pp = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)) if shards is not None else None
    return lib.xs_attn_fused(q, k, v, pp, B, N, H, d, len(shards) if P is None else P, st, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1),
    (dict(shards=(A, None)), 1), (dict(B=-1), 1), (dict(N=-128), 1), (dict(H=-2), 1),
    (dict(P=0), 1), (dict(shards=(A,) * 9), 1), (dict(N=384, shards=(A,) * 5), 1),
    (dict(st=3), 1), (dict(st=0), 1), (dict(st=16), 1),
    (dict(d=96), 2), (dict(d=512), 2), (dict(d=256, st=2), 2), (dict(d=256, st=1), 2),
    (dict(N=200, shards=(A, A)), 2),
    (dict(B=1 << 10, H=1 << 14, N=1 << 7, shards=(A, A)), 2),    # B*H*N = 2^31 rows
    (dict(q=A + 8), 3), (dict(v=A + 2), 3), (dict(shards=(A, A + 4)), 3),
    (dict(B=0), 0), (dict(H=0), 0), (dict(N=0), 0),
])
def test_fused_validation(xs, kw, code):
    assert _fused(xs, **kw) == code


def test_null_shard_array(xs):
    lib = xs.library()
    assert lib.xs_attn_fused(A, A, A, None, 1, 256, 4, 64, 2, 8, None) == xs.ERR_INVALID
    assert lib.xs_scatter(A, None, 1, 256, 4, 64, 2, None) == xs.ERR_INVALID
    assert lib.xs_attn_serial(A, A, A, A, None, 1, 256, 4, 64, 2, None) == xs.ERR_INVALID


def test_other_entry_points_validate(xs):
    lib = xs.library()
    arr = (ctypes.c_void_p * 2)(A, A)
    pp = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    assert lib.xs_attn(A, A, A, None, 1, 256, 4, 64, None) == xs.ERR_INVALID
    assert lib.xs_attn(A, A, A, A + 2, 1, 256, 4, 64, None) == xs.ERR_ALIGN
    assert lib.xs_attn(A, A, A, A, 1, 256, 4, 48, None) == xs.ERR_UNSUPPORTED
    assert lib.xs_scatter(A, pp, 1, 256, 4, 64, 3, None) == xs.ERR_INVALID    # P > len or N%P
    assert lib.xs_scatter(A, pp, 1, 256, 4, 96, 2, None) == xs.ERR_UNSUPPORTED
    assert lib.xs_attn_serial(A, A, A, None, pp, 1, 256, 4, 64, 2, None) == xs.ERR_INVALID
    assert lib.xs_attn_serial(A, A, A, A, pp, 1, 0, 4, 64, 2, None) == xs.OK   # empty


def test_wait_limit_setter(xs):
    old = xs.set_wait_limit_ns(12345)
    assert xs.set_wait_limit_ns(0) == 12345
    assert xs.set_wait_limit_ns(old) == 2_000_000_000


def test_product_path_does_not_import_oracle():
    import pathlib
    pkg = pathlib.Path(__file__).resolve().parent.parent / "all_layout_gb300"
    for f in list(pkg.rglob("*.py")) + list(pkg.rglob("*.cu")) + list(pkg.rglob("*.cuh")):
        text = f.read_text()
        assert "import oracle" not in text and "from oracle" not in text, f
        assert "liboracle" not in text, f


def _ulysses(xs, q=(A, A), k=(A, A), v=(A, A), out=(A, A), B=1, N=256, Ht=4, h0=0, H=4, d=64,
             P=None, st=8):
    lib = xs.library()

    def arr(t):
        if t is None:
            return None
        a = (ctypes.c_void_p * max(1, len(t)))(*t)
        return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p))
    return lib.xs_attn_ulysses(arr(q), arr(k), arr(v), arr(out), B, N, Ht, h0, H, d,
                               len(out) if P is None else P, st, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(v=(A, None)), 1), (dict(out=(A, None)), 1),
    (dict(Ht=0, H=0), 1), (dict(h0=-1), 1), (dict(h0=2, H=3), 1), (dict(H=-1), 1),
    (dict(st=5), 1), (dict(N=384), 2),   # 192-row input shards straddle tiles
    (dict(d=32), 2), (dict(N=128), 2),
    (dict(k=(A, A + 8)), 3), (dict(out=(A + 2, A)), 3),
    (dict(H=0), 0), (dict(B=0), 0),
])
def test_ulysses_validation(xs, kw, code):
    assert _ulysses(xs, **kw) == code
