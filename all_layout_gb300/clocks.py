"""SM clocks and throttle reasons sampled with nvidia-smi while a timed region runs.

Every measurement module (the benchmark, the sweep, the residual-slope test)
wraps its timed region in a ``ClockSampler`` and reports ``summary(t0, t1)``
next to its numbers: the median SM clock under load, the maximum SM clock and
the throttle reasons seen (hw_slowdown, hw_thermal_slowdown,
sw_thermal_slowdown, sw_power_cap). Reading clocks changes no GPU setting.
"""
from __future__ import annotations

import os
import subprocess
import threading
import time

REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
# A timed number seen under one of these is not accepted (sw_power_cap is kept and noted).
REJECTING = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def physical_gpu_index(local_index: int = 0) -> int:
    """nvidia-smi index of the CUDA device `local_index` of this process."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            return int(vis.split(",")[local_index])
        except (ValueError, IndexError):
            pass
    return local_index


class ClockSampler:
    """Context manager: samples clocks every `period_ms` in a background process."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 100):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        """Median SM MHz, max SM MHz and the throttle reasons active between t0 and t1
        (host wall-clock seconds)."""
        return summarize([line for ts, line in self.lines if t0 <= ts <= t1])


def summary_near(stamped, t0: float, t1: float) -> dict:
    """Clock record of the (time, line) samples taken between t0 and t1; a region
    shorter than the sampling period takes the sample nearest to its middle."""
    inside = [line for ts, line in stamped if t0 <= ts <= t1]
    if not inside and stamped:
        mid = 0.5 * (t0 + t1)
        inside = [min(stamped, key=lambda e: abs(e[0] - mid))[1]]
    return summarize(inside)


def summarize(lines) -> dict:
    """Parse nvidia-smi CSV lines (the FIELDS order) into the clocks record."""
    sm, mx, reasons = [], None, set()
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx = float(parts[1])
        except ValueError:
            continue
        for name, val in zip(REASONS, parts[4:8]):
            if val.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
    sm.sort()
    return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
            "samples": len(sm)}


def accepted(rec: dict) -> bool:
    """False when a rejecting throttle reason was active, or the median SM clock
    sat below 80% of the maximum with no reason given (a leftover clock lock)."""
    if any(r in REJECTING for r in rec.get("reasons", [])):
        return False
    sm, mx = rec.get("sm_mhz"), rec.get("sm_max_mhz")
    if sm and mx and sm < 0.8 * mx and not rec.get("reasons"):
        return False
    return True
