"""The 96-point sweep: N in {1024, 4096, 16384, 32768} x P in {2, 4, 8} x
(H, d) in {(24, 128), (48, 64)} x store_tile in {1, 2, 4, 8}, fused vs serial
(attention then the layout kernel) vs attention alone, one GPU.

Inputs are N(0, 1) bf16 drawn on the device per shape (timing only; the parity
of sweep points is covered by the GPU tests with the seeded CPU generator).
L2 is flushed before every timed call. By default a workspace is registered, so
each shape takes the schedule the library's cost model picks (stream-K or whole
units). SM clocks and throttle reasons are sampled during the whole run and
reported per point.

Run as ``python -m all_layout_gb300.sweep [--whole-units] [--markdown FILE]``.
"""
from __future__ import annotations

import json
import sys
import time

import numpy as np
import torch

from . import clocks, inputs, xs
from .build import kernel_sha


def _time_ms(fns, reps, flush):
    """Median time of each function, the calls interleaved (one of each per
    round) so that a clock that drifts during a point (the power cap engaging)
    biases none of the ratios."""
    for fn in fns:
        for _ in range(2):
            fn()
    torch.cuda.synchronize()
    ts = [[] for _ in fns]
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


def run(points=None, reps: int = 7, balanced: bool = True):
    """Times every point; with `balanced`, a workspace is registered so that each
    launch may take the stream-K schedule (the same for all three paths)."""
    points = points or inputs.sweep_points()
    flush = torch.empty(128 << 20, dtype=torch.float32, device="cuda")
    rows, cache, spans = [], {}, []
    ws = None
    if balanced:
        need = max(xs.workspace_bytes(w.B, w.N, w.H, w.d)[0] for w in points)
        if need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            xs.set_workspace(ws)
    with clocks.ClockSampler(clocks.physical_gpu_index(torch.cuda.current_device()),
                             period_ms=50) as clk:
        for w in points:
            key = (w.N, w.H, w.d)
            if key not in cache:
                cache.clear()
                g = torch.Generator(device="cuda").manual_seed(w.seed)
                cache[key] = tuple(torch.randn((w.B, w.H, w.N, w.d), device="cuda", generator=g)
                                   .to(torch.bfloat16) for _ in range(3))
            q, k, v = cache[key]
            shards = xs.alloc_shards(w.B, w.N, w.H, w.d, w.P)
            o = torch.empty_like(q)
            t0 = time.time()
            t_f, t_s, t_a = _time_ms([lambda: xs.attn_fused(q, k, v, shards, w.store_tile),
                                      lambda: xs.attn_serial(q, k, v, o, shards),
                                      lambda: xs.attn(q, k, v, o)], reps, flush)
            spans.append((t0, time.time()))
            rows.append({"N": w.N, "P": w.P, "H": w.H, "d": w.d, "store_tile": w.store_tile,
                         "stream_k": int(ws is not None and xs.workspace_bytes(w.B, w.N, w.H, w.d)[1]),
                         "t_fused_ms": t_f, "t_serial_ms": t_s, "t_attn_ms": t_a,
                         "tflops_fused": w.flops / (t_f * 1e-3) / 1e12,
                         "serial_over_fused": t_s / t_f, "fused_over_attn": t_f / t_a})
    for r, (t0, t1) in zip(rows, spans):
        r["clocks"] = clocks.summary_near(clk.lines, t0, t1)
    if ws is not None:
        xs.set_workspace(None)
    return rows


def markdown(rows, command: str) -> str:
    """The sweep as a markdown table with per-point clocks and a summary."""
    out = ["# Sweep: fused vs serial vs attention alone (one GB300)", "",
           f"Command (repository root): `{command}` (N(0,1) bf16 inputs drawn on the device, L2",
           "flushed before every timed call, median of 7 calls per path, the three paths interleaved",
           "round by round; a workspace is registered unless `--whole-units`, so each shape takes the",
           "schedule the cost model picks: `stream-K` column). SM clock: median of the nvidia-smi",
           "samples taken while the point ran (the nearest sample for points shorter than 50 ms).",
           f"kernel_sha: {kernel_sha()}", "",
           "| N | H | d | P | store_tile | stream-K | fused TFLOP/s | fused ms | serial / fused "
           "| fused / attention alone | SM MHz | throttle reasons |",
           "|---|---|---|---|---|---|---|---|---|---|---|---|"]
    for r in rows:
        c = r["clocks"]
        out.append(f"| {r['N']} | {r['H']} | {r['d']} | {r['P']} | {r['store_tile']} | "
                   f"{'yes' if r['stream_k'] else 'no'} | {r['tflops_fused']:.0f} | "
                   f"{r['t_fused_ms']:.3f} | {r['serial_over_fused']:.3f} | "
                   f"{r['fused_over_attn']:.3f} | {c['sm_mhz'] or '-'} | "
                   f"{', '.join(c['reasons']) or 'none'} |")
    n = len(rows)
    faster = sum(r["serial_over_fused"] > 1.0 for r in rows)
    within = sum(r["fused_over_attn"] <= 1.05 for r in rows)
    sof = [r["serial_over_fused"] for r in rows]
    foa = [r["fused_over_attn"] for r in rows]
    out += ["", f"Summary: fused faster than serial at {faster}/{n} points (serial/fused median "
            f"{np.median(sof):.3f}, min {min(sof):.3f}, max {max(sof):.3f}); fused within 5% of "
            f"attention alone at {within}/{n} (fused/attention median {np.median(foa):.3f}, "
            f"max {max(foa):.3f})."]
    for st in (1, 2, 4, 8):
        sel = [r for r in rows if r["store_tile"] == st]
        if sel:
            out.append(f"store_tile {st}: fused faster than serial at "
                       f"{sum(r['serial_over_fused'] > 1.0 for r in sel)}/{len(sel)}, within 5% "
                       f"of attention alone at {sum(r['fused_over_attn'] <= 1.05 for r in sel)}/"
                       f"{len(sel)}.")
    rejected = [r for r in rows if not clocks.accepted(r["clocks"])]
    out.append(f"Points with a rejecting throttle reason or a clock stuck low: {len(rejected)}.")
    return "\n".join(out) + "\n"


if __name__ == "__main__":
    args = sys.argv[1:]
    balanced = "--whole-units" not in args
    rows = run(balanced=balanced)
    if "--markdown" in args:
        path = args[args.index("--markdown") + 1]
        cmd = "python -m all_layout_gb300.sweep" + ("" if balanced else " --whole-units")
        with open(path, "w") as f:
            f.write(markdown(rows, cmd))
    print(json.dumps(rows, indent=1))
