"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module only draws numbers and arranges them; it holds none of the
attention or layout arithmetic and imports nothing else from this package.
All tensors are CPU torch tensors in the [B, H, N, d] head-partition layout
(the layout each head partition has after the pre-attention All-to-All,
X-Stage Figure 5 (c)).

Recipe for ``qkv``: ``torch.Generator().manual_seed(seed)``, then
``torch.randn`` in fp32 for q, k, v in that order, each rounded to bf16
(round to nearest even). ``q_scale`` multiplies q after rounding; a power of
two keeps that exact.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One attention + layout problem: batch B, sequence N, heads H, head dim d,
    P destination shards, the store-burst chunk and the input seed."""
    name: str
    B: int
    N: int
    H: int
    d: int
    P: int
    seed: int
    q_scale: float = 1.0
    store_tile: int = 8

    @property
    def flops(self) -> int:
        """Algorithmic attention flops: 2*N*N*d for Q K^T plus 2*N*N*d for P V,
        per (batch, head)."""
        return 4 * self.B * self.N * self.N * self.H * self.d


# The pages' DiT workloads (sequence lengths 8K-64K on an eight-GPU node, X-Stage
# Table 3 / Figure 11) stand in as these synthetic shapes.
WORKLOADS = {
    "small": Workload("small B1 N256 H4 d64 P2", 1, 256, 4, 64, 2, seed=1),
    "image_dit": Workload("image-DiT B1 N4096 H24 d128 P8", 1, 4096, 24, 128, 8, seed=2),
    "peaked_16k": Workload("peaked B1 N16384 H24 d128 P8 q*4", 1, 16384, 24, 128, 8,
                           seed=3, q_scale=4.0),
    "video_dit": Workload("video-DiT B1 N65536 H24 d128 P8", 1, 65536, 24, 128, 8, seed=4),
    # Head dimension 64 at twice the heads (48 x 64 = 24 x 128), a sweep shape.
    "d64_16k": Workload("d64 B1 N16384 H48 d64 P8", 1, 16384, 48, 64, 8, seed=7),
    # Head dimension 256 at the same model width (12 heads x 256 = 24 x 128).
    "wide_4k": Workload("wide B1 N4096 H12 d256 P8", 1, 4096, 12, 256, 8, seed=5),
    "wide_16k": Workload("wide B1 N16384 H12 d256 P8", 1, 16384, 12, 256, 8, seed=6),
}


def sweep_points():
    """The 96-point sweep: N x P x (H, d) x store_tile, seeds 100 + index."""
    pts = []
    i = 0
    for N in (1024, 4096, 16384, 32768):
        for P in (2, 4, 8):
            for H, d in ((24, 128), (48, 64)):
                for st in (1, 2, 4, 8):
                    pts.append(Workload(f"sweep N{N} P{P} H{H} d{d} st{st}", 1, N, H, d,
                                        P, seed=100 + i, store_tile=st))
                    i += 1
    return pts


def qkv(B: int, N: int, H: int, d: int, seed: int, q_scale: float = 1.0):
    """q, k, v ~ N(0, 1) as bf16 CPU tensors [B, H, N, d] (see module docstring)."""
    g = torch.Generator().manual_seed(int(seed))
    out = []
    for _ in range(3):
        out.append(torch.randn((B, H, N, d), generator=g, dtype=torch.float32)
                   .to(torch.bfloat16))
    if q_scale != 1.0:
        out[0] = out[0] * q_scale
    return tuple(out)


def workload_qkv(w: Workload):
    return qkv(w.B, w.N, w.H, w.d, w.seed, w.q_scale)


def tags(B: int, N: int, H: int, d: int, seed: int) -> torch.Tensor:
    """Raw 16-bit patterns (every value, NaN and Inf patterns included) viewed as
    bf16 [B, H, N, d], for bit-exact layout tests."""
    rng = np.random.default_rng(int(seed))
    bits = rng.integers(0, 1 << 16, size=(B, H, N, d), dtype=np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (a view of the same bytes)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def one_hot_case(B: int, N: int, H: int, d: int, seed: int, amplitude: float = 128.0):
    """Inputs whose attention output, rounded to bf16, is exactly a permutation
    of V's rows.

    Key j carries the sign pattern of its 16 low bits in channels 0..15
    (+1 where the bit is set, -1 where it is clear; 0 in every other channel).
    Query n carries ``amplitude`` times the sign pattern of perm[b, h, n]. The
    matching key then out-scores every other key by at least
    2 * amplitude / sqrt(d) (22.6 at amplitude 128, d 128), so the other
    softmax weights sum to below 2^-28 and the output row is V's row perm[n]
    plus less than 2^-20 relative, which bf16 rounding removes because every
    V entry is an integer in [1, 255] (exact in bf16, never 0).
    V: channels 0..3 = 1 + the four 4-bit digits of j, channel 4 = 1 + h,
    channel 5 = 1 + b, the rest hashed into [1, 250].

    Returns (q, k, v, perm) with perm an int64 numpy array [B, H, N].
    Requires N <= 65536, H <= 254, B <= 254 and d >= 16.
    """
    if N > (1 << 16) or d < 16 or H > 254 or B > 254:
        raise ValueError("one_hot_case needs N <= 65536, d >= 16, B and H <= 254")
    rng = np.random.default_rng(int(seed))
    j = np.arange(N, dtype=np.int64)
    signs = np.where((j[:, None] >> np.arange(16)[None, :]) & 1, 1.0, -1.0)  # [N, 16]
    k = np.zeros((B, H, N, d), dtype=np.float32)
    k[..., :16] = signs[None, None]
    perm = np.stack([np.stack([rng.permutation(N) for _ in range(H)]) for _ in range(B)])
    q = np.zeros((B, H, N, d), dtype=np.float32)
    q[..., :16] = amplitude * signs[perm]
    bb = np.arange(B, dtype=np.int64)[:, None, None, None]
    hh = np.arange(H, dtype=np.int64)[None, :, None, None]
    jj = j[None, None, :, None]
    cc = np.arange(d, dtype=np.int64)[None, None, None, :]
    hashed = 1 + (jj * 2654435761 + cc * 40503 + hh * 9973 + bb * 7919 + int(seed)) % 250
    v = hashed.astype(np.float32)
    for c in range(4):
        v[..., c] = (1 + ((j >> (4 * c)) & 15))[None, None]
    v[..., 4] = 1 + np.arange(H)[None, :, None]
    v[..., 5] = 1 + np.arange(B)[:, None, None]
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)
    return to(q), to(k), to(v), perm
