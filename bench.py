"""Benchmark: fused non-causal attention + Ulysses post-attention All-to-All layout.

One step = one xs_attn_fused call over one batch of synthetic input already
resident in HBM (the whole hot path: attention plus the shard stores).
Metric: attention TFLOP/s = 4*B*N^2*H*d / t, with % of the measured bf16 peak,
plus fused vs serial (attention then the layout kernel) and attention-alone
times on the same GPU.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl xs|reference]
                       [--workload video_dit|peaked_16k|image_dit|small]
The default workload is the largest single-GPU configuration, video-DiT
B=1 N=65536 H=24 d=128 P=8.
Under torchrun (N > 1) every rank runs an independent replica of the workload
(the (batch, head) problems are independent; no collective on the data path);
value = total flops of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused attn+A2A-layout TFLOP/s & % bf16 peak; fused vs serial time (1 GB300)"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# ncu summaries of the fused kernel (store_tile 8, balanced schedule): workload ->
# (summary file, the workload it captured). A workload without a capture of its own
# takes the DRAM bytes of a capture of the same kernel on a smaller workload of the
# same (H, d, P), scaled by the tokens processed: every launch reads q, k, v once
# from HBM (the K/V of the heads in flight stay in L2) and writes the output once,
# so its traffic grows in proportion to B*N*H*d.
PROFILE_FILES = {"image_dit": ("ncu_attn_fused_image_dit.md", "image_dit"),
                 "peaked_16k": ("ncu_attn_fused_peaked_16k.md", "peaked_16k"),
                 "video_dit": ("ncu_attn_fused_peaked_16k.md", "peaked_16k"),
                 "d64_16k": ("ncu_attn_fused_d64_16k.md", "d64_16k"),
                 "wide_16k": ("ncu_attn_wide_d256_16k.md", "wide_16k")}
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("xs", "reference"), default="xs")
    ap.add_argument("--workload", default="video_dit",
                    help="one of all_layout_gb300.inputs.WORKLOADS (default: video-DiT N=65536)")
    ap.add_argument("--store-tile", type=int, default=None)
    ap.add_argument("--side-steps", type=int, default=30,
                    help="rounds of the interleaved fused / attention-alone / serial / layout "
                         "side timings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--whole-units", action="store_true",
                    help="register no workspace: every CTA takes whole units")
    return ap.parse_args()


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    except OSError:
        return FALLBACK_PEAKS, "fallback"


def kernel_sha() -> str:
    from all_layout_gb300.build import kernel_sha as _sha
    return _sha()


def profiled_traffic(workload: str, store_tile: int, balanced: bool):
    """(DRAM bytes per launch, how it was obtained) of the fused kernel from the
    committed ncu summary for this workload, only if that summary was taken on the
    current kernel source and in the launch configuration being timed (store_tile
    8, balanced schedule); (None, reason) otherwise."""
    from all_layout_gb300 import inputs
    entry = PROFILE_FILES.get(workload)
    if entry is None:
        return None, "no ncu capture for this workload"
    if store_tile != 8 or not balanced:
        return None, "ncu captures cover store_tile 8 with the balanced schedule only"
    fname, captured = entry
    try:
        text = open(os.path.join(ROOT, "profiles", fname)).read()
    except OSError:
        return None, f"profiles/{fname} missing"
    sha = re.search(r"kernel_sha:\s*([0-9a-f]+)", text)
    tb = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not sha or not tb or sha.group(1) != kernel_sha():
        return None, f"profiles/{fname} was taken on another kernel source"
    w, c = inputs.WORKLOADS[workload], inputs.WORKLOADS[captured]
    scale = (w.B * w.N * w.H * w.d) / (c.B * c.N * c.H * c.d)
    how = f"ncu profiles/{fname}" + ("" if scale == 1 else
                                     f" ({c.name}), scaled x{scale:g} by tokens processed")
    return float(tb.group(1)) * scale, how


def dist_setup(n_gpus):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(w, rows_per_head: int, threads: int | None = None):
    """Time the fp64 oracle on a row sample of workload w; returns (TFLOP/s, seconds,
    threads, description)."""
    import numpy as np
    import oracle
    from all_layout_gb300 import inputs
    q, k, v = inputs.qkv(w.B, w.N, w.H, w.d, w.seed, w.q_scale)
    rows = np.linspace(0, w.N - 1, rows_per_head).astype(np.int64)
    thr = threads or oracle.default_threads()
    oracle.attention_rows(q[:, :1, :8], k[:, :1, :8], v[:, :1, :8], rows[:1] % 8)  # load/build
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, rows, threads=thr)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.B * w.H * rows.size * w.N * w.d
    desc = (f"{rows.size} query rows per head x {w.B * w.H} heads of {w.name} "
            f"({flops:.3g} flops, {rows.size / w.N:.2%} of the workload)")
    return flops / dt / 1e12, dt, thr, desc


def run_reference(args, w, rank, world):
    """Reference arm: the fp64 CPU oracle on a bounded sample per step."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from all_layout_gb300 import inputs
    q, k, v = inputs.qkv(w.B, w.N, w.H, w.d, w.seed, w.q_scale)
    thr = oracle.default_threads()
    rows_per_step = 1
    rows_all = np.arange(w.N, dtype=np.int64)
    oracle.attention_rows(q, k, v, rows_all[:1], threads=thr)
    for i in range(args.warmup):
        oracle.attention_rows(q, k, v, rows_all[i % w.N: i % w.N + rows_per_step], threads=thr)
    t0 = time.perf_counter()
    for i in range(args.steps):
        r0 = (i * 97) % (w.N - rows_per_step + 1)
        oracle.attention_rows(q, k, v, rows_all[r0:r0 + rows_per_step], threads=thr)
    dt = time.perf_counter() - t0
    flops_step = 4.0 * w.B * w.H * rows_per_step * w.N * w.d
    value = flops_step * args.steps / dt / 1e12
    sample = (f"each step: {rows_per_step} query row per head x {w.B * w.H} heads of {w.name} "
              f"({flops_step:.3g} flops, fp64, exact attention + layout definition)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "N": w.N, "H": w.H, "d": w.d, "P": w.P},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_xs(args, w, rank, world, local):
    import torch

    from all_layout_gb300 import clocks, inputs, xs

    st = args.store_tile or w.store_tile
    dev = torch.device("cuda", local)
    q_h, k_h, v_h = inputs.workload_qkv(w)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    shards = xs.alloc_shards(w.B, w.N, w.H, w.d, w.P, device=dev)
    o = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Workspace of the balanced (stream-K) schedule, allocated once before
    # anything is timed; without it every CTA takes whole units.
    ws_bytes, cut = xs.workspace_bytes(w.B, w.N, w.H, w.d)
    workspace = None
    if args.whole_units or ws_bytes == 0:
        ws_bytes, cut = 0, 0
    else:
        workspace = xs.alloc_workspace(w.B, w.N, w.H, w.d, device=dev)

    def fused():
        xs.attn_fused(q, k, v, shards, store_tile=st, stream=stream)

    def timed(fn, steps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            flush.zero_()                 # L2 flush, outside the timed events
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in ev]   # ms

    for _ in range(max(3, args.warmup)):
        fused()
    torch.cuda.synchronize(dev)

    gpu_index = clocks.physical_gpu_index(local)
    with clocks.ClockSampler(gpu_index) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.time()
        step_ms = timed(fused, args.steps)
        torch.cuda.synchronize(dev)
        barrier(world)
        t1 = time.time()
    if xs.last_device_status(stream) != xs.OK:
        raise RuntimeError("an on-chip wait timed out during the timed region")
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    flops = w.flops
    value = flops * world / (ms_per_step * 1e-3) / 1e12
    clock_rec = clk.summary(t0, t1)

    # Side timings on the same GPU: fused, attention alone, serial path and the
    # layout kernel alone, one call of each per round, so that a clock that drifts
    # over the run (the power cap engaging) biases none of the ratios.
    side = max(5, args.side_steps)
    side_fns = (fused, lambda: xs.attn(q, k, v, o, stream=stream),
                lambda: xs.attn_serial(q, k, v, o, shards, stream=stream),
                lambda: xs.scatter(o, shards, stream=stream))
    side_ms = [[] for _ in side_fns]
    for _ in range(side):
        for i, fn in enumerate(side_fns):
            side_ms[i].append(timed(fn, 1)[0])
    t_fused_side, t_attn, t_serial, t_scatter = (sorted(t) for t in side_ms)
    med = lambda a: a[len(a) // 2]
    t_fused_med = med(t_fused_side)

    # End to end through the public API with host buffers: every step copies its
    # q, k, v from pinned host memory, runs the fused call and reads every shard
    # back into pinned host memory, all inside the timed region. Steps are
    # pipelined the way a serving loop runs them: two device buffer sets, one
    # stream each for uploads, compute and downloads, so step i+1's upload and
    # step i-1's download overlap step i's kernel. The same loop run one step at a
    # time is reported as "serial_ms_per_step".
    e2e = None
    if not args.no_e2e:
        qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
        sets = [((q, k, v), shards)]
        sets.append(((torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)),
                     xs.alloc_shards(w.B, w.N, w.H, w.d, w.P, device=dev)))
        outs = [[torch.empty(sh.shape, dtype=sh.dtype).pin_memory() for sh in shards] for _ in sets]
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {name: [torch.cuda.Event() for _ in sets] for name in ("up", "cmp", "down")}
        used = [False, False]
        e2e_steps = max(5, min(args.steps, 200))

        def e2e_step(i, pipelined=True):
            b = i % 2
            (qd, kd, vd), shd = sets[b]
            with torch.cuda.stream(s_up):
                if used[b]:
                    s_up.wait_event(ev["cmp"][b])        # step i-2 has read these inputs
                for hd, dd in ((qp, qd), (kp, kd), (vp, vd)):
                    dd.copy_(hd, non_blocking=True)
                ev["up"][b].record(s_up)
            stream.wait_event(ev["up"][b])
            if used[b]:
                stream.wait_event(ev["down"][b])         # step i-2's shards are on the host
            xs.attn_fused(qd, kd, vd, shd, store_tile=st, stream=stream)
            ev["cmp"][b].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev["cmp"][b])
                for ho, sd in zip(outs[b], shd):
                    ho.copy_(sd, non_blocking=True)
                ev["down"][b].record(s_down)
            used[b] = True
            if not pipelined:
                s_down.synchronize()

        def run_e2e(n, pipelined):
            torch.cuda.synchronize(dev)
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s_up)
            for i in range(n):
                e2e_step(i, pipelined)
            s_down.wait_stream(stream)
            s_down.wait_stream(s_up)
            z.record(s_down)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(z) / n

        run_e2e(4, True)
        barrier(world)
        e_ms = max_over_ranks(run_e2e(e2e_steps, True) * e2e_steps, world) / e2e_steps
        serial_ms = run_e2e(min(e2e_steps, 20), False)
        h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
        d2h = sum(sh.numel() * sh.element_size() for sh in shards)
        e2e = {"value": flops * world / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "pipelined": True, "serial_ms_per_step": serial_ms}

    pk, pk_kind = peaks()
    peak = float(pk["bf16_tflops"])
    achieved = flops / (ms_per_step * 1e-3) / 1e12        # per launch, this rank's GPU
    traffic, traffic_how = profiled_traffic(args.workload, st, workspace is not None)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": f"{pk_kind} bf16 (burst)",
                "frac_of_sustained": achieved / float(pk.get("bf16_tflops_sustained", peak)),
                "traffic": traffic, "traffic_source": traffic_how,
                "algorithmic_bytes": 4 * w.B * w.H * w.N * w.d * 2,
                "kernel": ("attn_wide_kernel (fused, d 256)" if w.d == 256 else
                           "attn_kernel<%d> (fused)" % w.d),
                "kernel_sha": kernel_sha()}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows = w.N if w.N <= 8192 else 512     # whole workload when it takes seconds
        val, dt, thr, desc = cpu_oracle_sample(w, rows)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": thr, "kind": "oracle", "sample": desc,
               "seconds": dt, "extrapolated_full_s": dt * w.N / rows}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "N": w.N, "H": w.H, "d": w.d, "P": w.P,
                       "store_tile": st, "seed": w.seed,
                       "schedule": "stream-K" if cut else "whole units",
                       "workspace_bytes": ws_bytes,
                       "l2": "flushed between timed steps (512 MiB write, outside the events)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "pct_of_peak": 100.0 * achieved / peak,
            "t_fused_ms": t_fused_med, "t_attn_ms": med(t_attn), "t_serial_ms": med(t_serial),
            "t_scatter_ms": med(t_scatter),
            "fused_over_attn": t_fused_med / med(t_attn),
            "serial_over_fused": med(t_serial) / t_fused_med,
            "hiding_ratio": (med(t_serial) - t_fused_med) / med(t_scatter),
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clock_rec, "e2e": e2e,
            "gpu_launches": args.steps,
        }
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from all_layout_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, w, rank, world)
        else:
            run_xs(args, w, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
