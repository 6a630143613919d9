"""Head dimension 256 (the d = 256 kernel: one query tile per CTA, scores
double-buffered in Tensor Memory) against the fp64 CPU oracle, through the C ABI.

Same gates as every parity test: |err| <= 1e-2 + 1e-2*|ref| elementwise and a
relative RMS <= 1e-2; placement bit-exact on the one-hot case; the layout kernel
bit-exact on raw 16-bit tags."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from all_layout_gb300 import inputs
from gpu_util import (all_finite_dev, assert_close, gather_rows_dev, sample_rows, shards_bits,
                      shards_f64)

pytestmark = pytest.mark.gpu
D = 256


@pytest.fixture(scope="module")
def xs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs as _xs
    torch.cuda.set_device(0)
    return _xs


def _dev(*ts):
    return tuple(t.cuda() for t in ts)


def _fused(xs, q, k, v, P):
    B, H, N, d = q.shape
    shards = xs.alloc_shards(B, N, H, d, P)
    for s in shards:
        s.fill_(float("nan"))
    xs.attn_fused(*_dev(q, k, v), shards, store_tile=8)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    return shards


@pytest.mark.parametrize("B,H,N,P,qs", [
    (1, 2, 512, 4, 1.0),       # several KV steps, both S buffers in turn
    (2, 1, 384, 3, 1.0),       # odd tile count, several batches
    (1, 3, 256, 2, 4.0),       # peaked rows: the running max jumps, O is rescaled
    (1, 1, 128, 1, 1.0),       # one tile, one KV step
    (1, 5, 1024, 8, 2.0),      # more units than fit one step of the schedule per CTA
])
def test_wide_vs_oracle(xs, B, H, N, P, qs):
    q, k, v = inputs.qkv(B, N, H, D, seed=211 + N + H, q_scale=qs)
    ref = oracle.shard_layout(oracle.attention(q, k, v), P)
    assert_close(shards_f64(_fused(xs, q, k, v, P)), ref, f"d256 B{B} H{H} N{N} P{P}")


@pytest.mark.parametrize("B,H,N,P", [(1, 2, 1024, 8), (2, 1, 384, 3), (1, 3, 2048, 4)])
def test_wide_one_hot_exact(xs, B, H, N, P):
    q, k, v, perm = inputs.one_hot_case(B, N, H, D, seed=27)
    got = shards_bits(_fused(xs, q, k, v, P))
    o_exp = np.take_along_axis(inputs.bits(v), perm[..., None].repeat(D, axis=3), axis=2)
    exp = oracle.shard_layout(o_exp, P)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)
        raise AssertionError(f"{len(bad)} mismatching elements, first at {tuple(bad[0])}")


def test_wide_attention_alone_serial_and_layout(xs):
    B, H, N, P = 1, 3, 640, 5
    q, k, v = inputs.qkv(B, N, H, D, seed=223)
    qd, kd, vd = _dev(q, k, v)
    o = torch.empty_like(qd)
    xs.attn(qd, kd, vd, o)
    torch.cuda.synchronize()
    o_ref = oracle.attention(q, k, v)
    assert_close(o.float().cpu().numpy(), o_ref, "d256 attention alone")
    scratch = torch.empty_like(qd)
    shards = xs.alloc_shards(B, N, H, D, P)
    xs.attn_serial(qd, kd, vd, scratch, shards)
    torch.cuda.synchronize()
    fused = _fused(xs, q, k, v, P)
    assert np.array_equal(shards_bits(shards), shards_bits(fused))     # same arithmetic
    assert np.array_equal(scratch.cpu().view(torch.int16).numpy(), o.cpu().view(torch.int16).numpy())
    # the layout kernel alone, on raw 16-bit tags
    tags = inputs.tags(B, N, H, D, seed=7)
    out = xs.alloc_shards(B, N, H, D, P)
    xs.scatter(tags.cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(shards_bits(out), oracle.shard_layout(inputs.bits(tags), P))


def test_wide_sampled_16k(xs):
    w = inputs.WORKLOADS["wide_16k"]
    q, k, v = inputs.workload_qkv(w)
    shards = _fused(xs, q, k, v, w.P)
    assert all_finite_dev(shards)
    rows = sample_rows(w.N, w.P, np.random.default_rng(w.seed), extra=16)
    assert_close(gather_rows_dev(shards, rows, w.N, w.P), oracle.attention_rows(q, k, v, rows), w.name)


@pytest.fixture
def ws(xs):
    buf = torch.empty(96 << 20, dtype=torch.uint8, device="cuda")
    xs.set_workspace(buf)
    yield buf
    xs.set_workspace(None)


@pytest.mark.parametrize("B,H,N,P,qs", [(1, 2, 2944, 4, 1.0), (2, 1, 1664, 2, 4.0), (1, 1, 3456, 8, 1.0)])
def test_wide_streamk_vs_oracle(xs, ws, B, H, N, P, qs):
    """With a workspace the d = 256 kernel cuts the last waves into equal ranges of
    (tile, key tile) iterations; pieces of a cut tile merge on the GPU."""
    assert xs.workspace_bytes(B, N, H, D)[1] == 1, "shape chosen to take the balanced schedule"
    q, k, v = inputs.qkv(B, N, H, D, seed=241 + N, q_scale=qs)
    ref = oracle.shard_layout(oracle.attention(q, k, v), P)
    assert_close(shards_f64(_fused(xs, q, k, v, P)), ref, f"d256 stream-K B{B} H{H} N{N}")


def test_wide_streamk_one_hot_exact_and_repeatable(xs, ws):
    B, H, N, P = 1, 2, 2944, 4
    assert xs.workspace_bytes(B, N, H, D)[1] == 1
    q, k, v, perm = inputs.one_hot_case(B, N, H, D, seed=31)
    a = shards_bits(_fused(xs, q, k, v, P))
    b = shards_bits(_fused(xs, q, k, v, P))
    assert np.array_equal(a, b)                           # same bytes launch to launch
    assert np.all(ws[:16384].cpu().numpy() == 0)          # merge counters back at zero
    o_exp = np.take_along_axis(inputs.bits(v), perm[..., None].repeat(D, axis=3), axis=2)
    assert np.array_equal(a, oracle.shard_layout(o_exp, P))


def test_wide_streamk_sampled_16k(xs):
    """The wide 16K workload in the launch the benchmark times (its workspace)."""
    w = inputs.WORKLOADS["wide_16k"]
    assert xs.workspace_bytes(w.B, w.N, w.H, w.d)[1] == 1
    q, k, v = inputs.workload_qkv(w)
    buf = xs.alloc_workspace(w.B, w.N, w.H, w.d)
    try:
        shards = _fused(xs, q, k, v, w.P)
    finally:
        xs.set_workspace(None)
    del buf
    assert all_finite_dev(shards)
    rows = sample_rows(w.N, w.P, np.random.default_rng(w.seed + 1), extra=16)
    assert_close(gather_rows_dev(shards, rows, w.N, w.P), oracle.attention_rows(q, k, v, rows),
                 w.name + " stream-K")


def _seq_shards(t, P):
    sh = oracle.shard_layout(inputs.bits(t), P)
    return [torch.from_numpy(sh[p].view(np.int16)).view(torch.bfloat16).cuda() for p in range(P)]


def test_wide_ulysses_both_all_to_alls(xs):
    B, Ht, N, P, ranks = 1, 4, 512, 4, 2
    q, k, v = inputs.qkv(B, N, Ht, D, seed=233)
    qs, ks, vs = _seq_shards(q, P), _seq_shards(k, P), _seq_shards(v, P)
    out = xs.alloc_shards(B, N, Ht, D, P)
    for o in out:
        o.fill_(float("nan"))
    per = Ht // ranks
    for r in range(ranks):
        xs.attn_ulysses(qs, ks, vs, out, h0=r * per, H=per, store_tile=8)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    assert_close(shards_f64(out), oracle.shard_layout(oracle.attention(q, k, v), P), "d256 ulysses")


@pytest.mark.parametrize("flags", [0, 1])
def test_wide_fused_ex(xs, flags):
    B, H, N, P = 1, 2, 768, 4
    q, k, v = inputs.qkv(B, N, H, D, seed=239)
    out = xs.alloc_shards(B, N, H, D, P)
    n_tiles = B * H * (N // 128)
    spans = torch.zeros(2 * n_tiles, dtype=torch.int64, device="cuda")
    xs.attn_fused_ex(*_dev(q, k, v), out, store_tile=8, flags=flags, spans=spans)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    assert_close(shards_f64(out), oracle.shard_layout(oracle.attention(q, k, v), P), "d256 fused_ex")
    t = spans.view(n_tiles, 2).cpu().numpy()
    assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])


def test_wide_validation(xs):
    lib = xs.library()
    A = 0x10000
    arr = (ctypes.c_void_p * 2)(A, A)
    pp = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))
    for st in (1, 2, 4):
        assert lib.xs_attn_fused(A, A, A, pp, 1, 256, 4, D, 2, st, None) == xs.ERR_UNSUPPORTED


def test_wide_streamk_ulysses_and_spans(xs, ws):
    """d = 256 under the balanced schedule: both All-to-Alls fused (two ranks' head
    shares read from sequence shards) and fused_ex spans over tiles cut into pieces
    that merge on another CTA."""
    B, Ht, N, P, ranks = 1, 4, 2816, 2, 2
    per = Ht // ranks
    assert xs.workspace_bytes(B, N, per, D)[1] == 1
    q, k, v = inputs.qkv(B, N, Ht, D, seed=251)
    qs, ks, vs = _seq_shards(q, P), _seq_shards(k, P), _seq_shards(v, P)
    out = xs.alloc_shards(B, N, Ht, D, P)
    for o in out:
        o.fill_(float("nan"))
    for r in range(ranks):
        xs.attn_ulysses(qs, ks, vs, out, h0=r * per, H=per, store_tile=8)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    ref = oracle.shard_layout(oracle.attention(q, k, v), P)
    assert_close(shards_f64(out), ref, "d256 ulysses stream-K")
    # fused_ex on the same problem as one call: spans recorded for every tile
    out2 = xs.alloc_shards(B, N, Ht, D, P)
    n_tiles = B * Ht * (N // 128)
    spans = torch.zeros(2 * n_tiles, dtype=torch.int64, device="cuda")
    xs.attn_fused_ex(*_dev(q, k, v), out2, store_tile=8, flags=xs.FLAG_COMPLETION_COUPLED, spans=spans)
    torch.cuda.synchronize()
    assert xs.last_device_status() == xs.OK
    assert_close(shards_f64(out2), ref, "d256 fused_ex stream-K")
    t = spans.view(n_tiles, 2).cpu().numpy()
    assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])
