"""Checks that tie an attention / layout implementation to facts fixed by the
mathematics, independently of the implementation itself.

Each ``check_*`` takes an implementation and raises AssertionError when it
disagrees. ``tests/test_oracle.py`` runs them on the CPU oracle (must pass) and
on deliberately broken numpy variants (each must fail at least one), which
shows the checks are strong enough to catch a dropped term, a wrong scale, a
wrong sign, a transposed operand or a shifted index.

An attention implementation is ``f(q_bits, k_bits, v_bits) -> float64 o`` with
bf16 bit patterns [B, H, N, d] in. A layout implementation is
``g(o, P) -> recv [P, B, N/P, H, d]``.
"""
from __future__ import annotations

import math

import mpmath
import numpy as np

TOL = 1e-12


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 bits (via fp32; used only to build exact inputs)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def random_bits(rng, shape, mean=0.0, std=1.0):
    return f64_to_bf16_bits(rng.normal(mean, std, size=shape))


# ---------------------------------------------------------------- attention pins

def check_brute_force(attn, rng):
    """Direct sum_j exp(s_j) v_j / sum_j exp(s_j) in 40-digit arithmetic, with no
    max subtraction, on tiny random problems."""
    mpmath.mp.dps = 40
    for (B, H, N, d) in ((1, 1, 1, 4), (1, 2, 5, 8), (2, 2, 16, 8), (1, 1, 16, 2)):
        q, k, v = (random_bits(rng, (B, H, N, d)) for _ in range(3))
        got = attn(q, k, v)
        Q, K, V = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
        for b in range(B):
            for h in range(H):
                for n in range(N):
                    ws = []
                    for j in range(N):
                        dot = mpmath.fsum(mpmath.mpf(Q[b, h, n, c]) * mpmath.mpf(K[b, h, j, c])
                                          for c in range(d))
                        ws.append(mpmath.exp(dot / mpmath.sqrt(d)))
                    den = mpmath.fsum(ws)
                    for c in range(d):
                        num = mpmath.fsum(ws[j] * mpmath.mpf(V[b, h, j, c]) for j in range(N))
                        ref = float(num / den)
                        assert abs(got[b, h, n, c] - ref) <= TOL * (1 + abs(ref)), \
                            (b, h, n, c, got[b, h, n, c], ref)


def check_identical_v_rows(attn, rng):
    """If every key's value row is the same row r, every output row is r."""
    B, H, N, d = 1, 3, 37, 8
    q, k = random_bits(rng, (B, H, N, d), std=3.0), random_bits(rng, (B, H, N, d))
    row = random_bits(rng, (B, H, 1, d))
    v = np.repeat(row, N, axis=2)
    got = attn(q, k, v)
    exp = np.broadcast_to(bits_to_f64(row), got.shape)
    assert np.max(np.abs(got - exp)) <= TOL * (1 + np.max(np.abs(exp)))


def check_zero_query_mean(attn, rng):
    """q = 0 makes every score 0, so the output is the column mean of V."""
    B, H, N, d = 2, 2, 29, 8
    q = np.zeros((B, H, N, d), dtype=np.uint16)
    k = random_bits(rng, (B, H, N, d))
    v = random_bits(rng, (B, H, N, d), mean=1.0)
    got = attn(q, k, v)
    mean = bits_to_f64(v).mean(axis=2, keepdims=True)
    assert np.max(np.abs(got - mean)) <= TOL * (1 + np.max(np.abs(mean)))


def check_key_permutation(attn, rng):
    """Permuting keys together with their value rows leaves the output unchanged."""
    B, H, N, d = 1, 2, 41, 8
    q, k, v = (random_bits(rng, (B, H, N, d), std=2.0) for _ in range(3))
    perm = rng.permutation(N)
    a = attn(q, k, v)
    b = attn(q, k[:, :, perm], v[:, :, perm])
    assert np.max(np.abs(a - b)) <= TOL * (1 + np.max(np.abs(a)))


def check_query_permutation(attn, rng):
    """Permuting query rows permutes the output rows the same way."""
    B, H, N, d = 1, 2, 23, 8
    q, k, v = (random_bits(rng, (B, H, N, d)) for _ in range(3))
    perm = rng.permutation(N)
    a = attn(q, k, v)
    b = attn(q[:, :, perm], k, v)
    assert np.max(np.abs(a[:, :, perm] - b)) <= TOL * (1 + np.max(np.abs(a)))


def check_two_key_logistic(attn, rng):
    """With two keys, the weight of key 0 is the logistic function of the score
    gap: o = sigma(g) v0 + (1 - sigma(g)) v1 with g = q.(k0 - k1) / sqrt(d).
    Uses d = 4 so that a 1/d or missing scale changes the answer."""
    B, H, N, d = 1, 1, 2, 4
    for trial in range(8):
        q = random_bits(rng, (B, H, N, d), std=2.0)
        k = random_bits(rng, (B, H, N, d), std=2.0)
        v = random_bits(rng, (B, H, N, d))
        got = attn(q, k, v)
        Q, K, V = bits_to_f64(q)[0, 0], bits_to_f64(k)[0, 0], bits_to_f64(v)[0, 0]
        for n in range(N):
            g = float(np.dot(Q[n], K[0] - K[1])) / 2.0  # sqrt(4) = 2
            sig = 1.0 / (1.0 + math.exp(-g))
            exp = sig * V[0] + (1.0 - sig) * V[1]
            assert np.max(np.abs(got[0, 0, n] - exp)) <= 1e-12 * (1 + np.max(np.abs(exp))), \
                (trial, n, got[0, 0, n], exp)


def check_one_hot(attn, one_hot_inputs):
    """Query n matches only key perm[n]: the output row is V's row perm[n]."""
    q, k, v, perm = one_hot_inputs
    got = attn(q, k, v)
    V = bits_to_f64(v)
    B, H, N, d = V.shape
    exp = np.take_along_axis(V, perm[..., None].repeat(d, axis=3), axis=2)
    assert np.max(np.abs(got - exp)) <= 1e-6, np.max(np.abs(got - exp))


ATTENTION_PINS = (check_brute_force, check_identical_v_rows, check_zero_query_mean,
                  check_key_permutation, check_query_permutation, check_two_key_logistic)


# ---------------------------------------------------------------- layout pins

def check_layout_sequence_partition(layout, rng):
    """Figure 5 (d)-(e): after the post-attention All-to-All, destination p holds
    the contiguous sequence block p of every head. Concatenating the shards along
    the sequence axis must give o with heads moved behind tokens, [B, N, H, d]."""
    for (B, H, N, d, P) in ((1, 3, 12, 4, 3), (2, 2, 16, 8, 4), (1, 1, 8, 2, 1), (2, 3, 10, 2, 5)):
        o = rng.integers(0, 1 << 16, size=(B, H, N, d), dtype=np.uint16)
        recv = layout(o, P)
        assert recv.shape == (P, B, N // P, H, d)
        whole = np.concatenate([recv[p] for p in range(P)], axis=1)   # [B, N, H, d]
        assert np.array_equal(whole, np.transpose(o, (0, 2, 1, 3)))


def check_layout_tags(layout, rng):
    """Each destination element names where it came from: tag (b, h, n, c) must
    land at shard n // (N/P), row n % (N/P)."""
    B, H, N, d, P = 2, 3, 24, 4, 4
    b, h, n, c = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), np.arange(d),
                             indexing="ij")
    tag = (((b * H + h) * N + n) * d + c).astype(np.int64)
    recv = layout(tag, P)
    R = N // P
    for p in range(P):
        for bb in range(B):
            for i in range(R):
                for hh in range(H):
                    t = recv[p, bb, i, hh]
                    exp = ((bb * H + hh) * N + (p * R + i)) * d + np.arange(d)
                    assert np.array_equal(t, exp), (p, bb, i, hh)


LAYOUT_PINS = (check_layout_sequence_partition, check_layout_tags)
