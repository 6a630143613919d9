"""Local calibration of the Burst-Gap parameters and the store_tile choice.

Burst-Gap model (Pith review of X-Stage, "What carries the argument"): a burst
of V bytes followed by a producer-side gap G is issued in max(T0, V/R - G),
with T0 the backpressure-free issue time, R the effective drain rate and Q the
effective outstanding capacity; a schedule is backpressure-free when
V / (T0 + G) <= R and [V - R*T0]+ <= Q ("If this is right"). The pages
calibrate on remote NVLink stores of an eight-GPU node; here the same three
measurements ("What would settle it") run on stores into this GPU's own memory
through xs_store_burst_probe:

  * T0: bursts separated by a long gap (the recovered plateau);
  * R:  back-to-back bursts with no gap, large enough to be drain-limited
        (steady-state period = V / R);
  * Q:  single bursts of growing size after idle; the knee where the issue span
        leaves the backpressure-free line gives Q = V_knee - R * span(V_knee).

`choose_store_tile` applies the two bounds to the fused kernel: every producer
CTA issues store_tile slabs of 16 output rows per KV iteration, and the
iteration's compute is the gap.

Run as ``python -m all_layout_gb300.burst_gap [--markdown FILE]`` for a JSON
report (SM clocks and throttle reasons sampled during each mode's run).
"""
from __future__ import annotations

import json
import sys
import time

import numpy as np
import torch

from . import clocks, xs

MODES = {"posted": 0, "tma": 1}


def run_probe(K: int, burst_bytes: int, n_bursts: int, gap_ns: int, mode: str = "posted",
              device="cuda"):
    """Issue spans (ns) [K, n_bursts], and start / end times (ns) of every burst."""
    dst = torch.empty(K * n_bursts * burst_bytes, dtype=torch.uint8, device=device)
    times = torch.zeros(2 * K * n_bursts, dtype=torch.int64, device=device)
    xs.store_burst_probe(dst, K, burst_bytes, n_bursts, gap_ns, MODES[mode], times)
    torch.cuda.synchronize(device)
    if xs.last_device_status() != xs.OK:
        raise RuntimeError("store burst probe reported an error")
    t = times.view(K, n_bursts, 2).cpu().numpy().astype(np.int64)
    start, end = t[..., 0], t[..., 1]
    return (end - start).astype(np.float64), start, end


def measure_T0(K: int, burst_bytes: int, mode: str = "posted", gap_ns: int = 20000,
               n_bursts: int = 8) -> float:
    """Backpressure-free issue time (s): median span of bursts after a long gap."""
    span, _, _ = run_probe(K, burst_bytes, n_bursts, gap_ns, mode)
    return float(np.median(span[:, 1:])) * 1e-9


def measure_R(K: int, burst_bytes: int, mode: str = "posted", n_bursts: int = 12) -> float:
    """Effective drain rate (bytes/s) from the steady-state period of back-to-back
    bursts (the first two bursts are warm-up)."""
    _, start, end = run_probe(K, burst_bytes, n_bursts, 0, mode)
    t0 = start[:, 2].min()
    t1 = end[:, -1].max()
    return float(K * burst_bytes * (n_bursts - 2) / ((t1 - t0) * 1e-9))


def measure_knee(K: int, R: float, mode: str = "posted", sizes=None, tol: float = 0.25):
    """Isolated-burst sweep: issue span of one burst of K*B bytes after idle, for
    growing B. Returns (Q, table) with Q = V_knee - R * span(V_knee), the knee
    being the largest V whose span stays within `tol` of the small-burst issue
    line (fitted on the smallest sizes)."""
    sizes = sizes or [2048 << i for i in range(12)]
    rows = []
    for B in sizes:
        span, _, _ = run_probe(K, B, 1, 0, mode)
        rows.append((K * B, float(np.median(span[:, 0])) * 1e-9))
    V = np.array([r[0] for r in rows], dtype=np.float64)
    S = np.array([r[1] for r in rows], dtype=np.float64)
    n_fit = 4
    slope, icpt = np.polyfit(V[:n_fit], S[:n_fit], 1)
    line = icpt + slope * V
    ok = S <= (1.0 + tol) * line
    k = int(np.max(np.nonzero(ok)[0])) if ok.any() else 0
    Q = max(0.0, V[k] - R * S[k])
    return float(Q), [{"V_bytes": float(v), "span_s": float(s), "line_s": float(l)}
                      for v, s, l in zip(V, S, line)]


def max_law_check(K: int, burst_bytes: int, R: float, gaps_ns, mode: str = "posted",
                  n_bursts: int = 10):
    """Steady-state issue span of periodic bursts against max(T0(V), V/R - G).
    T0(V) is the recovered plateau for the same burst size (the pages' ledger
    lists the backpressure-free issue time per producer count and burst size)."""
    V = K * burst_bytes
    T0v = measure_T0(K, burst_bytes, mode, gap_ns=64000)
    out = []
    for g in gaps_ns:
        span, _, _ = run_probe(K, burst_bytes, n_bursts, int(g), mode)
        meas = float(np.median(span[:, 2:])) * 1e-9
        out.append({"gap_s": g * 1e-9, "measured_s": meas, "model_s": max(T0v, V / R - g * 1e-9),
                    "T0_s": T0v})
    return out


def choose_store_tile(T0: float, R: float, Q: float, K: int, slab_bytes: int,
                      gap_s: float) -> int:
    """Largest store_tile in (8, 4, 2, 1) whose burst (K producers x store_tile
    slabs) stays backpressure-free with the KV iteration's compute as the gap:
    rate bound V/(T0+G) <= R and capacity bound [V - R*T0]+ <= Q."""
    for st in (8, 4, 2, 1):
        V = K * st * slab_bytes
        rate_ok = V / (T0 + gap_s) <= R
        cap_ok = max(0.0, V - R * T0) <= Q
        if rate_ok and cap_ok:
            return st
    return 1


def calibrate(K: int | None = None, mode: str = "posted", d: int = 128,
              kv_iteration_s: float | None = None) -> dict:
    """Full local calibration and the resulting store_tile choice."""
    if K is None:
        K = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    B = 32768                                   # one 128 x 128 bf16 output tile per producer
    T0 = measure_T0(K, B, mode)
    R = measure_R(K, 1 << 20, mode)             # 1 MiB per producer: drain-limited
    Q, knee = measure_knee(K, R, mode)
    law = [max_law_check(K, B_law, R, [0, 1000, 2000, 4000, 8000, 16000, 32000], mode)
           for B_law in (1 << 16, 1 << 18, 1 << 20)]
    slab = 16 * d * 2                           # 16 rows of d bf16
    gap = kv_iteration_s if kv_iteration_s is not None else 1.8e-6
    return {"K": K, "mode": mode, "T0_s": T0, "R_bytes_per_s": R, "Q_bytes": Q,
            "knee": knee, "max_law": law, "slab_bytes": slab, "kv_iteration_s": gap,
            "store_tile": choose_store_tile(T0, R, Q, K, slab, gap)}


def calibrate_all() -> dict:
    """Both store modes, each with the clock record of its run."""
    rep = {}
    with clocks.ClockSampler(clocks.physical_gpu_index(torch.cuda.current_device())) as clk:
        for m in MODES:
            t0 = time.time()
            rep[m] = calibrate(mode=m)
            rep[m]["clocks"] = (t0, time.time())
    for m in rep:
        rep[m]["clocks"] = clocks.summary_near(clk.lines, *rep[m]["clocks"])
    return rep


def markdown(rep: dict, command: str) -> str:
    us = lambda s: f"{s * 1e6:.2f} us"
    out = ["# Local Burst-Gap calibration (stores into this GB300's own HBM)", "",
           f"Command (repository root): `{command}` (probe: `xs_store_burst_probe`,",
           f"K = {rep['posted']['K']} producer CTAs of 128 threads; %globaltimer issue spans). The pages",
           "calibrate remote NVLink stores on an eight-GPU node (R ~717 GB/s, T_iss^0 ~0.76 us at",
           "K=148, B=32 KB, Q ~4.25 MiB); these are the single-GPU analogs.", "",
           "| mode | T_iss^0 (32 KiB per producer) | R | Q (isolated-burst knee) | store_tile chosen "
           "(gap 1.8 us) | SM MHz (median, reasons) |",
           "|---|---|---|---|---|---|"]
    for m, r in rep.items():
        c = r["clocks"]
        out.append(f"| {m} | {us(r['T0_s'])} | {r['R_bytes_per_s'] / 1e9:.0f} GB/s | "
                   f"{r['Q_bytes'] / 2**20:.2f} MiB | {r['store_tile']} | "
                   f"{c['sm_mhz'] or '-'}, {', '.join(c['reasons']) or 'none'} |")
    out += ["", "Max law, steady-state issue span of periodic bursts (per producer B, aggregate "
            "V = K B):", "", "| mode | B per producer | gap | measured | max(T0(V), V/R - G) |",
            "|---|---|---|---|---|"]
    for m, r in rep.items():
        for B, rows in zip(("64 KiB", "256 KiB", "1 MiB"), r["max_law"]):
            for row in rows:
                out.append(f"| {m} | {B} | {row['gap_s'] * 1e6:.0f} us | {us(row['measured_s'])} | "
                           f"{us(row['model_s'])} |")
    return "\n".join(out) + "\n"


if __name__ == "__main__":
    rep = calibrate_all()
    args = sys.argv[1:]
    if "--markdown" in args:
        with open(args[args.index("--markdown") + 1], "w") as f:
            f.write(markdown(rep, "python -m all_layout_gb300.burst_gap"))
    print(json.dumps(rep, indent=1))
