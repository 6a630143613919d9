"""The 96-point sweep: N in {1024, 4096, 16384, 32768} x P in {2, 4, 8} x
(H, d) in {(24, 128), (48, 64)} x store_tile in {1, 2, 4, 8}, fused vs serial
(attention then the layout kernel) vs attention alone, one GPU.

Inputs are N(0, 1) bf16 drawn on the device per shape (timing only; the parity
of sweep points is covered by the GPU tests with the seeded CPU generator).
L2 is flushed before every timed call. By default a workspace is registered, so
each shape takes the schedule the library's cost model picks (stream-K or whole
units). Run as ``python -m all_layout_gb300.sweep`` (``--whole-units`` to
register none).
"""
from __future__ import annotations

import json

import numpy as np
import torch

from . import inputs, xs


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
    rows, cache = [], {}
    ws = None
    if balanced:
        need = max(xs.workspace_bytes(w.B, w.N, w.H, w.d)[0] for w in points)
        if need:
            ws = torch.empty(need, dtype=torch.uint8, device="cuda")
            xs.set_workspace(ws)
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
        t_f, t_s, t_a = _time_ms([lambda: xs.attn_fused(q, k, v, shards, w.store_tile),
                                  lambda: xs.attn_serial(q, k, v, o, shards),
                                  lambda: xs.attn(q, k, v, o)], reps, flush)
        rows.append({"N": w.N, "P": w.P, "H": w.H, "d": w.d, "store_tile": w.store_tile,
                     "stream_k": int(ws is not None and xs.workspace_bytes(w.B, w.N, w.H, w.d)[1]),
                     "t_fused_ms": t_f, "t_serial_ms": t_s, "t_attn_ms": t_a,
                     "tflops_fused": w.flops / (t_f * 1e-3) / 1e12,
                     "serial_over_fused": t_s / t_f, "fused_over_attn": t_f / t_a})
    if ws is not None:
        xs.set_workspace(None)
    return rows


if __name__ == "__main__":
    import sys
    print(json.dumps(run(balanced="--whole-units" not in sys.argv), indent=1))
