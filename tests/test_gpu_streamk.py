"""Parity of the balanced (stream-K) schedule (xs_set_workspace) with the fp64
CPU oracle.

With a workspace registered, a launch may give every CTA an equal contiguous
range of (unit, key tile) iterations; units cut by a range boundary are
computed in pieces whose partial results are merged on the GPU. The outputs
must meet the same gates as the whole-unit schedule (|err| <= 1e-2 +
1e-2*|ref|, relative RMS <= 1e-2), exact placement stays bit-exact, and
repeated launches give identical bytes (the per-unit counters return to zero)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from all_layout_gb300 import inputs
from gpu_util import (all_finite_dev, assert_close, gather_rows, gather_rows_dev, sample_rows,
                      shards_bits, shards_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs as _xs
    torch.cuda.set_device(0)
    return _xs


@pytest.fixture
def ws(xs):
    """A 96 MiB workspace registered for the test, removed afterwards."""
    buf = torch.empty(96 << 20, dtype=torch.uint8, device="cuda")
    xs.set_workspace(buf)
    yield buf
    xs.set_workspace(None)


def _dev(*ts):
    return tuple(t.cuda() for t in ts)


def _fused(xs, q, k, v, P, st=8):
    B, H, N, d = q.shape
    shards = xs.alloc_shards(B, N, H, d, P)
    for s in shards:
        s.fill_(float("nan"))
    xs.attn_fused(*_dev(q, k, v), shards, store_tile=st)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    return shards


def _cut(xs, B, N, H, d):
    return xs.workspace_bytes(B, N, H, d)[1]


# (B, H, N, d, P, q_scale), each taking the balanced schedule on 144..160 SMs:
# units cut into up to 7 pieces, an odd tile count (the last unit's second
# tile is empty), one item per CTA, several batches, d = 64, peaked rows.
SK_SHAPES = [
    (1, 2, 2944, 128, 2, 1.0),
    (1, 1, 2816, 64, 4, 1.0),
    (1, 1, 2048, 128, 2, 4.0),
    (2, 1, 1664, 128, 4, 2.0),
    (3, 1, 1792, 64, 7, 1.0),
    (2, 1, 2944, 64, 1, 1.0),
]


@pytest.mark.parametrize("B,H,N,d,P,qs", SK_SHAPES)
def test_streamk_shapes_vs_oracle(xs, ws, B, H, N, d, P, qs):
    assert _cut(xs, B, N, H, d) == 1, "shape chosen to take the balanced schedule"
    q, k, v = inputs.qkv(B, N, H, d, seed=71 + N + H, q_scale=qs)
    ref = oracle.shard_layout(oracle.attention(q, k, v), P)
    for st in (2, 8):
        assert_close(shards_f64(_fused(xs, q, k, v, P, st)), ref, f"stream-K st={st}")


def test_streamk_image_dit_full(xs, ws):
    w = inputs.WORKLOADS["image_dit"]
    assert _cut(xs, w.B, w.N, w.H, w.d) == 1
    q, k, v = inputs.workload_qkv(w)
    ref = oracle.shard_layout(oracle.attention(q, k, v), w.P)
    assert_close(shards_f64(_fused(xs, q, k, v, w.P, w.store_tile)), ref, w.name + " stream-K")


@pytest.mark.parametrize("key", ["peaked_16k", "d64"])
def test_streamk_sampled(xs, ws, key):
    w = inputs.WORKLOADS["peaked_16k"] if key == "peaked_16k" else \
        inputs.Workload("d64 B1 N4096 H48", 1, 4096, 48, 64, 8, seed=97)
    assert _cut(xs, w.B, w.N, w.H, w.d) == 1
    q, k, v = inputs.workload_qkv(w)
    got = shards_f64(_fused(xs, q, k, v, w.P, w.store_tile))
    assert np.all(np.isfinite(got))
    rows = sample_rows(w.N, w.P, np.random.default_rng(w.seed), extra=8)
    assert_close(gather_rows(got, rows, w.N, w.P), oracle.attention_rows(q, k, v, rows),
                 w.name + " stream-K")


@pytest.mark.parametrize("B,H,N,d,P", [(1, 2, 2944, 128, 4), (2, 1, 2816, 64, 8)])
def test_streamk_one_hot_exact(xs, ws, B, H, N, d, P):
    assert _cut(xs, B, N, H, d) == 1
    q, k, v, perm = inputs.one_hot_case(B, N, H, d, seed=19)
    got = shards_bits(_fused(xs, q, k, v, P, 8))
    o_exp = np.take_along_axis(inputs.bits(v), perm[..., None].repeat(d, axis=3), axis=2)
    exp = oracle.shard_layout(o_exp, P)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        raise AssertionError(f"{len(bad)} mismatching elements, first at {tuple(bad[0])}")


def test_streamk_repeatable_and_fallback(xs):
    """Two balanced launches in a row give the same bytes; a workspace too small
    for the schedule (header only) gives the whole-unit bytes; so does none."""
    B, H, N, d, P = 1, 2, 2944, 128, 2
    q, k, v = inputs.qkv(B, N, H, d, seed=83)
    plain = shards_bits(_fused(xs, q, k, v, P))
    big = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    small = torch.empty(16384, dtype=torch.uint8, device="cuda")
    try:
        xs.set_workspace(big)
        a = shards_bits(_fused(xs, q, k, v, P))
        b = shards_bits(_fused(xs, q, k, v, P))
        assert np.array_equal(a, b)
        assert np.all(big[:16384].cpu().numpy() == 0)       # counters back at zero
        xs.set_workspace(small)
        assert np.array_equal(shards_bits(_fused(xs, q, k, v, P)), plain)
    finally:
        xs.set_workspace(None)
    assert np.array_equal(shards_bits(_fused(xs, q, k, v, P)), plain)


def test_streamk_attention_alone_serial_and_spans(xs, ws):
    B, H, N, d, P = 1, 2, 2944, 128, 2
    q, k, v = inputs.qkv(B, N, H, d, seed=89)
    qd, kd, vd = _dev(q, k, v)
    o = torch.empty_like(qd)
    xs.attn(qd, kd, vd, o)
    torch.cuda.synchronize()
    o_ref = oracle.attention(q, k, v)
    assert_close(o.float().cpu().numpy(), o_ref, "attn stream-K")
    scratch = torch.empty_like(qd)
    shards = xs.alloc_shards(B, N, H, d, P)
    xs.attn_serial(qd, kd, vd, scratch, shards)
    torch.cuda.synchronize()
    fused = _fused(xs, q, k, v, P)
    assert np.array_equal(shards_bits(shards), shards_bits(fused))
    n_tiles = B * H * (N // 128)
    for flags in (0, xs.FLAG_COMPLETION_COUPLED):
        spans = torch.zeros(2 * n_tiles, dtype=torch.int64, device="cuda")
        out = xs.alloc_shards(B, N, H, d, P)
        xs.attn_fused_ex(qd, kd, vd, out, store_tile=8, flags=flags, spans=spans)
        torch.cuda.synchronize()
        assert xs.last_device_status() == xs.OK
        assert np.array_equal(shards_bits(out), shards_bits(fused))
        t = spans.view(n_tiles, 2).cpu().numpy()
        assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])


def test_set_workspace_validation(xs):
    lib = xs.library()
    assert lib.xs_set_workspace(ctypes.c_void_p(0x10080), 1 << 20, None) == xs.ERR_ALIGN
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    assert lib.xs_set_workspace(ctypes.c_void_p(buf.data_ptr()), 4096, None) == xs.ERR_INVALID
    assert lib.xs_set_workspace(None, 0, None) == xs.OK
    n = ctypes.c_ulonglong(7)
    assert lib.xs_workspace_bytes(1, 1000, 2, 128, ctypes.byref(n), None) == xs.ERR_UNSUPPORTED
    assert lib.xs_workspace_bytes(1, 1024, 2, 96, ctypes.byref(n), None) == xs.ERR_UNSUPPORTED
    assert lib.xs_workspace_bytes(1, 1024, 2, 128, None, None) == xs.ERR_INVALID
    assert lib.xs_workspace_bytes(0, 1024, 2, 128, ctypes.byref(n), None) == xs.OK and n.value == 0


def _seq_shards(t, P):
    """[B, H, N, d] -> P device tensors [B, N/P, H, d] (the sequence partition)."""
    sh = oracle.shard_layout(inputs.bits(t), P)
    return [torch.from_numpy(sh[p].view(np.int16)).view(torch.bfloat16).cuda() for p in range(P)]


def test_streamk_ulysses_both_all_to_alls(xs, ws):
    """Both All-to-Alls fused (inputs read from sequence shards, one call per
    rank's head share) under the balanced schedule."""
    B, Ht, N, d, P, ranks = 1, 4, 2816, 128, 2, 2
    per = Ht // ranks
    assert _cut(xs, B, N, per, d) == 1
    q, k, v = inputs.qkv(B, N, Ht, d, seed=101)
    qs, ks, vs = _seq_shards(q, P), _seq_shards(k, P), _seq_shards(v, P)
    out = xs.alloc_shards(B, N, Ht, d, P)
    for o in out:
        o.fill_(float("nan"))
    for r in range(ranks):
        xs.attn_ulysses(qs, ks, vs, out, h0=r * per, H=per, store_tile=8)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    ref = oracle.shard_layout(oracle.attention(q, k, v), P)
    assert_close(shards_f64(out), ref, "ulysses stream-K")


# ------------------------------------------------------------------ the benchmark's launch

def test_streamk_video_dit_sampled(xs):
    """The video-DiT workload (B1 N65536 H24 d128 P8) in the launch configuration the
    benchmark times: the workspace it registers (xs.alloc_workspace), store_tile 8.
    Sampled rows (every destination's first and last row, every slab position,
    random rows) against the oracle, and every destination element written."""
    w = inputs.WORKLOADS["video_dit"]
    assert _cut(xs, w.B, w.N, w.H, w.d) == 1, "the benchmark's launch takes the balanced schedule"
    q, k, v = inputs.workload_qkv(w)
    ws = xs.alloc_workspace(w.B, w.N, w.H, w.d)
    try:
        shards = _fused(xs, q, k, v, w.P, w.store_tile)
    finally:
        xs.set_workspace(None)
    del ws
    assert all_finite_dev(shards)
    rows = sample_rows(w.N, w.P, np.random.default_rng(w.seed), extra=16)
    assert_close(gather_rows_dev(shards, rows, w.N, w.P), oracle.attention_rows(q, k, v, rows),
                 w.name + " stream-K")


@pytest.mark.parametrize("st", [8, 2])
def test_streamk_one_hot_exact_64k(xs, ws, st):
    """Exact placement at N = 65536 under the balanced schedule: the matching key
    out-scores the 16 keys one bit away by 2*128/sqrt(128) (the rest by more), so the
    other weights sum to < 2^-28 and every output row is V's row perm[n] bit for bit,
    whichever CTA finishes its pieces."""
    B, H, N, d, P = 1, 2, 65536, 128, 8
    assert _cut(xs, B, N, H, d) == 1
    q, k, v, perm = inputs.one_hot_case(B, N, H, d, seed=23)
    got = shards_bits(_fused(xs, q, k, v, P, st))
    o_exp = np.take_along_axis(inputs.bits(v), perm[..., None].repeat(d, axis=3), axis=2)
    exp = oracle.shard_layout(o_exp, P)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        raise AssertionError(f"{len(bad)} mismatching elements, first at {tuple(bad[0])}")


@pytest.mark.parametrize("idx", [5, 30, 55, 89])
def test_sweep_points_sampled_with_workspace(xs, ws, idx):
    """The sweep points of the whole-unit parity test, in the schedule the sweep
    times (a workspace registered)."""
    w = inputs.sweep_points()[idx]
    q, k, v = inputs.workload_qkv(w)
    shards = _fused(xs, q, k, v, w.P, w.store_tile)
    assert all_finite_dev(shards)
    rows = sample_rows(w.N, w.P, np.random.default_rng(w.seed), extra=8)
    assert_close(gather_rows_dev(shards, rows, w.N, w.P), oracle.attention_rows(q, k, v, rows),
                 w.name + (" stream-K" if _cut(xs, w.B, w.N, w.H, w.d) else " whole units"))


@pytest.mark.parametrize("st,flags", [(8, 0), (8, 1), (2, 0)])
def test_streamk_fused_ex_vs_oracle(xs, ws, st, flags):
    """xs_attn_fused_ex (completion-coupled flag, per-tile spans) against the oracle
    under the balanced schedule."""
    B, H, N, d, P = 1, 2, 2944, 128, 4
    assert _cut(xs, B, N, H, d) == 1
    q, k, v = inputs.qkv(B, N, H, d, seed=67)
    out = xs.alloc_shards(B, N, H, d, P)
    for s in out:
        s.fill_(float("nan"))
    n_tiles = B * H * (N // 128)
    spans = torch.zeros(2 * n_tiles, dtype=torch.int64, device="cuda")
    xs.attn_fused_ex(*_dev(q, k, v), out, store_tile=st, flags=flags, spans=spans)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    assert_close(shards_f64(out), oracle.shard_layout(oracle.attention(q, k, v), P),
                 f"fused_ex st={st} flags={flags}")
    t = spans.view(n_tiles, 2).cpu().numpy()
    assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])


# (B, H, N, d, P): shapes that take the balanced schedule, one per kernel.
@pytest.mark.parametrize("B,H,N,d,P", [(1, 2, 2944, 128, 4), (1, 1, 2816, 64, 4),
                                       (1, 2, 2944, 256, 4)])
def test_workspace_writes_stay_within_reported_bytes(xs, B, H, N, d, P):
    """A workspace of exactly the bytes xs_workspace_bytes reports: the balanced
    schedule's partial results and merge counters stay inside it (a canary
    after it is untouched), and the output still matches the oracle."""
    n, cut = xs.workspace_bytes(B, N, H, d)
    assert cut == 1 and n > 0
    canary = 1 << 20
    buf = torch.full((n + canary,), 0xA5, dtype=torch.uint8, device="cuda")
    q, k, v = inputs.qkv(B, N, H, d, seed=331 + N + d)
    ref = oracle.shard_layout(oracle.attention(q, k, v), P)
    xs.set_workspace(buf[:n])
    try:
        for st in ((8,) if d == 256 else (8, 2)):
            assert_close(shards_f64(_fused(xs, q, k, v, P, st)), ref, f"d{d} st={st} exact workspace")
    finally:
        xs.set_workspace(None)
    assert bool((buf[n:] == 0xA5).all()), "the balanced schedule wrote past its workspace"


@pytest.mark.parametrize("H,d", [(4, 64), (2, 128), (2, 256)])
def test_streamk_odd_tile_count_long_sampled(xs, H, d):
    """N = 65408 (511 query tiles: the last unit of every head has a tile the second
    group sits out) under the balanced schedule with the workspace the library
    reports: sampled rows, the last rows of the sequence among them, against the
    oracle, and every destination element written."""
    B, N, P = 1, 65408, 8
    assert _cut(xs, B, N, H, d) == 1
    q, k, v = inputs.qkv(B, N, H, d, seed=347 + d)
    buf = xs.alloc_workspace(B, N, H, d)
    try:
        shards = _fused(xs, q, k, v, P, 8)
    finally:
        xs.set_workspace(None)
    del buf
    assert all_finite_dev(shards)
    rows = sample_rows(N, P, np.random.default_rng(347 + d), extra=12)
    assert N - 1 in rows
    assert_close(gather_rows_dev(shards, rows, N, P), oracle.attention_rows(q, k, v, rows),
                 f"N65408 H{H} d{d} stream-K")
