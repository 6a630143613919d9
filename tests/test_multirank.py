"""bench.py's multi-process host logic on CPU with the gloo backend, world size 2:
rendezvous on 127.0.0.1, the barrier, max-over-ranks timing, and the reference
arm printing exactly one JSON line from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w) == (rank, world)
    bench.barrier(w)
    got = bench.max_over_ranks(float(10 * (rank + 1)), w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    vals = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(world)]
    assert vals == [20.0, 20.0]


@pytest.mark.timeout(600)
def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "3", "--warmup", "1", "--workload", "small"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["steps"] == 3 and rec["unit"] == "TFLOP/s"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def test_roofline_traffic_only_for_the_profiled_launch():
    """The bench reports a DRAM traffic figure only from a committed ncu summary
    taken on the current kernel source, in the launch configuration being timed
    (store_tile 8, balanced schedule); a workload without a capture of its own
    takes a capture of the same (H, d, P) scaled by the tokens processed;
    otherwise null with the reason."""
    import os
    import re
    import bench
    from all_layout_gb300 import inputs
    for key, (fname, captured) in bench.PROFILE_FILES.items():
        text = open(os.path.join(ROOT, "profiles", fname)).read()
        sha = re.search(r"kernel_sha:\s*([0-9a-f]+)", text).group(1)
        tb = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text).group(1))
        w, c = inputs.WORKLOADS[key], inputs.WORKLOADS[captured]
        assert (w.H, w.d, w.P, w.B) == (c.H, c.d, c.P, c.B)
        scale = w.N / c.N
        got, how = bench.profiled_traffic(key, 8, True)
        if sha == bench.kernel_sha():
            assert got == tb * scale and fname in how
        else:
            assert got is None and "another kernel source" in how
        assert bench.profiled_traffic(key, 4, True)[0] is None
        assert bench.profiled_traffic(key, 8, False)[0] is None
    assert bench.profiled_traffic("small", 8, True)[0] is None


def test_clock_records():
    """Clock summaries: median SM clock, reasons seen, nearest sample for short
    regions, and the acceptance rule (hw/thermal reasons reject; sw_power_cap is
    kept; a clock far below max with no reason rejects)."""
    from all_layout_gb300 import clocks
    line = lambda sm, reasons=(): ", ".join([str(sm), "2070", "900.0", "0x0"] + [
        "Active" if r in reasons else "Not Active" for r in clocks.REASONS])
    rec = clocks.summarize([line(2070), line(1900, ("sw_power_cap",)), line(1800)])
    assert rec == {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert clocks.accepted(rec)
    assert not clocks.accepted(clocks.summarize([line(2070, ("hw_slowdown",))]))
    assert not clocks.accepted(clocks.summarize([line(1200), line(1210)]))
    stamped = [(1.0, line(2000)), (2.0, line(1500)), (3.0, line(1000))]
    assert clocks.summary_near(stamped, 1.9, 2.05)["sm_mhz"] == 1500.0
    assert clocks.summary_near(stamped, 2.4, 2.45)["sm_mhz"] == 1500.0    # nearest to 2.425
    assert clocks.summary_near(stamped, 0.5, 3.5)["samples"] == 3
