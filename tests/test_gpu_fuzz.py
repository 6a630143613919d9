"""Seeded random shapes against the fp64 oracle, through the C ABI.

The shapes are drawn once from a fixed seed: B, H, N (a multiple of 128, odd
tile counts included), d in {64, 128, 256}, P dividing N into 16-row-aligned
shards, store_tile (8 only at d = 256), with or without a workspace (so some
launches take the balanced schedule with units cut into pieces on several
CTAs). Sizes stay small enough for the full oracle to finish in seconds.
XS_FUZZ_SHAPES and XS_FUZZ_SEED draw a longer or different list (default 28
shapes from seed 2024)."""
import os

import numpy as np
import pytest
import torch

import oracle
from all_layout_gb300 import inputs
from gpu_util import assert_close, shards_bits, shards_f64

pytestmark = pytest.mark.gpu


def _shapes(n=int(os.environ.get("XS_FUZZ_SHAPES", "28")),
            seed=int(os.environ.get("XS_FUZZ_SEED", "2024"))):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128, 256]))
        tiles = int(rng.integers(1, 19))
        N = 128 * tiles
        B = int(rng.integers(1, 4))
        H = int(rng.integers(1, 5))
        if B * H * N * d > 3 * 4 * 1536 * 128:      # keep the oracle to seconds
            continue
        Ps = [p for p in range(1, 9) if N % p == 0 and (N // p) % 16 == 0]
        P = int(rng.choice(Ps))
        st = 8 if d == 256 else int(rng.choice([1, 2, 4, 8]))
        ws = bool(rng.integers(0, 2))
        qs = float(rng.choice([1.0, 1.0, 2.0, 4.0]))
        out.append((B, H, N, d, P, st, ws, qs, 400 + len(out)))
    return out


@pytest.fixture(scope="module")
def xs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs as _xs
    torch.cuda.set_device(0)
    return _xs


@pytest.mark.parametrize("B,H,N,d,P,st,use_ws,qs,seed", _shapes())
def test_random_shape(xs, B, H, N, d, P, st, use_ws, qs, seed):
    q, k, v = inputs.qkv(B, N, H, d, seed=seed, q_scale=qs)
    buf = torch.empty(128 << 20, dtype=torch.uint8, device="cuda") if use_ws else None
    if use_ws:
        xs.set_workspace(buf)
    try:
        shards = xs.alloc_shards(B, N, H, d, P)
        for s in shards:
            s.fill_(float("nan"))
        xs.attn_fused(*(t.cuda() for t in (q, k, v)), shards, store_tile=st)
        torch.cuda.synchronize()
        assert xs.last_device_status() == xs.OK
        got = shards_f64(shards)
        again = xs.alloc_shards(B, N, H, d, P)
        xs.attn_fused(*(t.cuda() for t in (q, k, v)), again, store_tile=st)
        torch.cuda.synchronize()
    finally:
        if use_ws:
            xs.set_workspace(None)
    what = f"B{B} H{H} N{N} d{d} P{P} st{st} ws{int(use_ws)} q*{qs}"
    assert_close(got, oracle.shard_layout(oracle.attention(q, k, v), P), what)
    assert np.array_equal(shards_bits(again), shards_bits(shards)), what + ": not repeatable"
