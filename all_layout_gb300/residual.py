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
the distribution of per-tile store-issue spans (xs_attn_fused_ex spans), and
the SM clocks and throttle reasons sampled while each N ran.

Run as ``python -m all_layout_gb300.residual [--whole-units] [--markdown FILE]``.
"""
from __future__ import annotations

import json
import sys
import time

import numpy as np
import torch

from . import clocks, xs
from .build import kernel_sha


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


def sweep(Ns=(1024, 2048, 4096, 8192, 16384, 32768, 65536), balanced: bool = True, **kw) -> dict:
    ws = None
    if balanced:
        need = max(xs.workspace_bytes(1, N, kw.get("H", 24), kw.get("d", 128))[0] for N in Ns)
        if need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            xs.set_workspace(ws)
    rows, spans = [], []
    with clocks.ClockSampler(clocks.physical_gpu_index(torch.cuda.current_device()),
                             period_ms=50) as clk:
        for N in Ns:
            t0 = time.time()
            r = measure(N, reps=5 if N >= 32768 else 10, **kw)
            spans.append((t0, time.time()))
            r["stream_k"] = int(ws is not None and xs.workspace_bytes(1, N, r["H"], r["d"])[1])
            rows.append(r)
    for r, (t0, t1) in zip(rows, spans):
        r["clocks"] = clocks.summary_near(clk.lines, t0, t1)
    if ws is not None:
        xs.set_workspace(None)
    x = np.array([r["N"] for r in rows], dtype=np.float64)
    out = {"rows": rows, "balanced": balanced}
    for key in ("fused", "coupled"):
        e = np.array([(r[f"t_{key}_ms"] - r["t_attn_ms"]) for r in rows])   # E_res in ms
        slope, icpt = np.polyfit(x, e, 1)
        out[f"slope_{key}_us_per_1k_tokens"] = float(slope * 1e3 * 1e3)
    return out


def markdown(rep: dict, command: str) -> str:
    rows = rep["rows"]
    out = ["# Residual-slope test: fused stores vs attention alone (Figure 11 analog, one GB300)", "",
           f"Command (repository root): `{command}` (H=24, d=128, P=8, B=1, store_tile 8; L2",
           "flushed before every timed call; median of 10 calls, 5 at N >= 32K, the three calls",
           "interleaved round by round; " + ("a workspace registered, so each N takes the schedule the "
                                             "cost model picks" if rep["balanced"] else
                                             "no workspace: whole units") + ").",
           "`coupled` = `xs_attn_fused_ex` with XS_FLAG_COMPLETION_COUPLED (each issuing warp waits for",
           "its stores to complete, the pages' counterfactual). Span = per-tile store-issue span (first",
           "slab issued -> last issuing warp released). SM clock: median of the nvidia-smi samples",
           "taken while that N ran (the nearest sample when it ran shorter than the 50 ms period).",
           f"kernel_sha: {kernel_sha()}", "",
           "| N | stream-K | T_attn ms | T_fused ms | T_coupled ms | E_res/T_attn fused | "
           "E_res/T_attn coupled | span p50 / p99 (fused) | SM MHz | throttle reasons |",
           "|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        c, s = r["clocks"], r["spans"]["fused"]
        out.append(f"| {r['N']} | {'yes' if r['stream_k'] else 'no'} | {r['t_attn_ms']:.3f} | "
                   f"{r['t_fused_ms']:.3f} | {r['t_coupled_ms']:.3f} | {100 * r['res_fused']:.2f}% | "
                   f"{100 * r['res_coupled']:.2f}% | {s['p50_ns']:.0f} / {s['p99_ns']:.0f} ns | "
                   f"{c['sm_mhz'] or '-'} | {', '.join(c['reasons']) or 'none'} |")
    out += ["", f"Least-squares slope of E_res against N: fused "
            f"{rep['slope_fused_us_per_1k_tokens']:.2f} us per 1K tokens, coupled "
            f"{rep['slope_coupled_us_per_1k_tokens']:.2f} us per 1K tokens."]
    return "\n".join(out) + "\n"


if __name__ == "__main__":
    args = sys.argv[1:]
    balanced = "--whole-units" not in args
    rep = sweep(balanced=balanced)
    if "--markdown" in args:
        with open(args[args.index("--markdown") + 1], "w") as f:
            f.write(markdown(rep, "python -m all_layout_gb300.residual"
                             + ("" if balanced else " --whole-units")))
    print(json.dumps(rep, indent=1))
