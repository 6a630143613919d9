"""Residual-slope test of the fused store path (Figure 11 analog).

Pith review of X-Stage, "If this is right": under the completion-coupled model
(the issuer blocked until its stores are visible) the sender-visible residual
over FlashAttention alone grows linearly with sequence length, while the
X-Stage model predicts a flat, near-zero residual because the Q-loop between
two stores of a producer exceeds the recovery gap. Figure 11 plots
E_res(M) / T_FA against M.

For each sequence length N this measures, on one GPU and with the same kernel:
  T_attn      attention alone (xs_attn),
  T_fused     fused stores into the P destinations (xs_attn_fused, store_tile 8),
  T_coupled   the same with XS_FLAG_COMPLETION_COUPLED,
and reports E_res / T_attn for both, a least-squares slope of E_res against N,
and the distribution of per-tile store-issue spans (xs_attn_fused_ex spans).

Run as ``python -m all_layout_gb300.residual`` for a JSON report.
"""
from __future__ import annotations

import json

import numpy as np
import torch

from . import xs


def _time_ms(fns, reps: int, flush: torch.Tensor) -> list:
    """Median time of each function, the calls interleaved (one of each per
    round) so that a clock that drifts during the run (the power cap engaging
    at long N) biases none of them."""
    ts = [[] for _ in fns]
    for fn in fns:
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    for _ in range(reps):
        for i, fn in enumerate(fns):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts[i].append(a.elapsed_time(b))
    return [float(np.median(t)) for t in ts]


def measure(N: int, H: int = 24, d: int = 128, P: int = 8, B: int = 1, reps: int = 10,
            seed: int = 7) -> dict:
    g = torch.Generator(device="cuda").manual_seed(seed)
    q, k, v = (torch.randn((B, H, N, d), device="cuda", generator=g).to(torch.bfloat16)
               for _ in range(3))
    shards = xs.alloc_shards(B, N, H, d, P)
    o = torch.empty_like(q)
    flush = torch.empty(128 << 20, dtype=torch.float32, device="cuda")
    t_attn, t_fused, t_coupled = _time_ms(
        [lambda: xs.attn(q, k, v, o), lambda: xs.attn_fused(q, k, v, shards, 8),
         lambda: xs.attn_fused_ex(q, k, v, shards, 8, xs.FLAG_COMPLETION_COUPLED)], reps, flush)
    n_tiles = B * H * (N // 128)
    spans = {}
    for name, flags in (("fused", 0), ("coupled", xs.FLAG_COMPLETION_COUPLED)):
        buf = torch.zeros(2 * n_tiles, dtype=torch.int64, device="cuda")
        xs.attn_fused_ex(q, k, v, shards, 8, flags, buf)
        torch.cuda.synchronize()
        t = buf.view(n_tiles, 2).cpu().numpy()
        sp = (t[:, 1] - t[:, 0]).astype(np.float64)
        spans[name] = {"p50_ns": float(np.percentile(sp, 50)), "p90_ns": float(np.percentile(sp, 90)),
                       "p99_ns": float(np.percentile(sp, 99)), "max_ns": float(sp.max()),
                       "tiles": int(n_tiles)}
    return {"N": N, "H": H, "d": d, "P": P, "t_attn_ms": t_attn, "t_fused_ms": t_fused,
            "t_coupled_ms": t_coupled, "res_fused": (t_fused - t_attn) / t_attn,
            "res_coupled": (t_coupled - t_attn) / t_attn, "spans": spans}


def sweep(Ns=(1024, 2048, 4096, 8192, 16384, 32768, 65536), **kw) -> dict:
    rows = [measure(N, reps=5 if N >= 32768 else 10, **kw) for N in Ns]
    x = np.array([r["N"] for r in rows], dtype=np.float64)
    out = {"rows": rows}
    for key in ("fused", "coupled"):
        e = np.array([(r[f"t_{key}_ms"] - r["t_attn_ms"]) for r in rows])   # E_res in ms
        slope, icpt = np.polyfit(x, e, 1)
        out[f"slope_{key}_us_per_1k_tokens"] = float(slope * 1e3 * 1e3)
    return out


if __name__ == "__main__":
    print(json.dumps(sweep(), indent=1))
