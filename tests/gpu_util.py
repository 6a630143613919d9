"""Helpers for the GPU parity tests: tolerance gates, shard gathering, row samples."""
from __future__ import annotations

import numpy as np
import torch

# Floating-point gate (elementwise) and the added relative-RMS gate.
ATOL, RTOL, REL_RMS = 1e-2, 1e-2, 1e-2


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """|got - ref| <= ATOL + RTOL*|ref| everywhere, relative RMS <= REL_RMS, no NaN/Inf."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    if bad.any():
        idx = tuple(int(i) for i in np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of tolerance; first at {idx}: "
                             f"got {got[idx]!r} ref {ref[idx]!r}; max abs err {err.max():.3e}")
    den = np.sqrt(np.sum(ref ** 2))
    rel = np.sqrt(np.sum((got - ref) ** 2)) / den if den > 0 else np.sqrt(np.sum(got ** 2))
    assert rel <= REL_RMS, f"{what}: relative RMS {rel:.3e} > {REL_RMS}"
    return float(err.max()), float(rel)


def shards_f64(shards) -> np.ndarray:
    """P device tensors [B, N/P, H, d] bf16 -> float64 numpy [P, B, N/P, H, d]."""
    return np.stack([s.float().cpu().numpy() for s in shards]).astype(np.float64)


def shards_bits(shards) -> np.ndarray:
    return np.stack([s.cpu().view(torch.int16).numpy().view(np.uint16) for s in shards])


def sample_rows(N: int, P: int, rng, extra: int = 24) -> np.ndarray:
    """Rows covering every shard's first and last row, every 16-row slab position
    of a 128-row tile, and random rows."""
    R = N // P
    rows = set()
    for p in range(P):
        rows.add(p * R)
        rows.add(p * R + R - 1)
    for s in range(8):
        rows.add((s * 16 + 5 + 128 * s) % N)
    rows.update(int(r) for r in rng.integers(0, N, size=extra))
    return np.array(sorted(rows), dtype=np.int64)


def gather_rows(got_shards: np.ndarray, rows: np.ndarray, N: int, P: int) -> np.ndarray:
    """From [P, B, N/P, H, d] pick query rows -> [B, H, len(rows), d]."""
    R = N // P
    p, i = rows // R, rows % R
    sel = got_shards[p, :, i]              # [len(rows), B, H, d]
    return np.transpose(sel, (1, 2, 0, 3))


def gather_rows_dev(shards, rows: np.ndarray, N: int, P: int) -> np.ndarray:
    """Pick query rows from P device shards [B, N/P, H, d] on the GPU and return
    them as float64 [B, H, len(rows), d] (only the sampled rows leave the device)."""
    R = N // P
    out = []
    for r in rows:
        p, i = int(r) // R, int(r) % R
        out.append(shards[p][:, i])                        # [B, H, d]
    sel = torch.stack(out, dim=2)                         # [B, H, rows, d]
    return sel.float().cpu().numpy().astype(np.float64)


def all_finite_dev(shards) -> bool:
    """Every element of every device shard is finite (no NaN fill left)."""
    return all(bool(torch.isfinite(s).all()) for s in shards)
