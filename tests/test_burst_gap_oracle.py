"""Pins for the Burst-Gap model formulas (oracle/burst_gap.py): the values the
pages print (tests/golden/burst_gap_pages.json) and the model's own stated
properties (max law, only the total gap matters, recovery gap, bounds)."""
import json
import os

import pytest

from oracle import burst_gap as bg

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "burst_gap_pages.json")))
V = {k: v["value"] for k, v in GOLD["values"].items()}
MiB = 1 << 20


def test_pages_worked_numbers():
    R, T0, Q, sigma = V["R_bytes_per_s"], V["T0_s"], V["Q_bytes"], V["sigma_s_per_kv_tile"]
    Vfa = V["K_producers"] * V["B_bytes_per_producer"]          # 148 x 32 KiB
    assert Vfa / MiB == pytest.approx(V["V_fa_bytes"] / MiB, rel=0.02)        # ~4.6 MiB
    excess = bg.capacity_excess(Vfa, T0, R)
    assert excess / MiB == pytest.approx(V["capacity_excess_bytes"] / MiB, rel=0.03)   # ~4.1 MiB
    assert (Q - excess) / MiB == pytest.approx(V["capacity_margin_bytes"] / MiB, abs=0.03)  # ~0.15
    assert bg.backpressure_free(Vfa, 10e-6, T0, R, Q)           # the FA design test passes
    gstar = bg.recovery_gap(Vfa, T0, R)
    assert gstar == pytest.approx(6.0e-6, rel=0.03)
    mstar = bg.convergence_threshold(128, Vfa, T0, R, sigma)
    assert mstar == pytest.approx(V["M_star_ub_tokens"], rel=0.10)             # ~1.0K


def test_max_law_properties():
    T0, R = 1e-6, 500e9
    for Vb in (1e3, 1e5, 1e6, 1e7):
        for G in (0.0, 1e-7, 1e-6, 1e-5, 1e-4):
            t = bg.issue_time(Vb, G, T0, R)
            assert t >= T0 and t >= Vb / R - G
            assert t == pytest.approx(max(T0, Vb / R - G))
            # only the total gap matters: splitting G changes nothing
            assert bg.issue_time(Vb, G / 3 + 2 * G / 3, T0, R) == pytest.approx(t)
            # never above the completion-coupled sum
            assert t <= bg.completion_coupled_time(Vb, G, T0, R) + 1e-18
        g = bg.recovery_gap(Vb, T0, R)
        assert bg.issue_time(Vb, g, T0, R) == pytest.approx(T0)           # recovered at G*
        if g > 0:
            assert bg.issue_time(Vb, g / 2, T0, R) > T0                    # not before


def test_zero_gap_period_is_drain_limited():
    T0, R = 0.5e-6, 800e9
    Vb = 10 * R * T0                     # drain-limited burst
    assert bg.steady_state_period(Vb, 0.0, T0, R) == pytest.approx(Vb / R)
    small = 0.1 * R * T0                 # issue-limited burst
    assert bg.steady_state_period(small, 0.0, T0, R) == pytest.approx(T0)


def test_bounds():
    T0, R, Q = 1e-6, 700e9, 4 * MiB
    assert bg.rate_bound_ok(R * 2e-6, 1e-6, T0, R)
    assert not bg.rate_bound_ok(R * 3e-6, 1e-6, T0, R)
    assert bg.capacity_excess(R * T0 * 0.5, T0, R) == 0.0
    assert not bg.backpressure_free(Q + R * T0 + 1, 1.0, T0, R, Q)


# ------------------------------------------------------------------ completion-coupled counterfactual
# Pith review of X-Stage, "Core claim": the sender-visible issue time follows a max
# law, max(T0, V/R - G), "rather than a completion-coupled sum"; "If this is right":
# in the completion-coupled model the issuer is blocked until its stores are
# remotely visible, so the residual grows linearly with sequence length, while the
# max law predicts a flat one; "Implications": under the max law a producer-side gap
# overlaps the drain instead of delaying the next burst.

def _coupled_pins_hold(fn) -> bool:
    """The properties above, for a candidate completion-coupled issue time fn(V, G, T0, R)."""
    ok = True
    for T0, R in ((0.76e-6, 717e9), (1e-6, 500e9), (0.3e-6, 6.5e12)):
        for Vb in (1e3, 1e5, 4.6 * 2**20, 64 * 2**20):
            # a sum of the issue term and the whole drain term V/R ...
            ok &= abs(fn(Vb, 0.0, T0, R) - (fn(0.0, 0.0, T0, R) + Vb / R)) <= 1e-12 * (1 + Vb / R)
            ok &= abs(fn(0.0, 0.0, T0, R) - T0) <= 1e-15
            # ... so it exceeds the max law at zero gap by min(T0, V/R) ...
            ok &= abs(fn(Vb, 0.0, T0, R) - bg.issue_time(Vb, 0.0, T0, R) - min(T0, Vb / R)) \
                <= 1e-12 * (1 + Vb / R)
            # ... and a gap after the burst neither shortens nor lengthens the blocked
            # issue: the gap only delays the next burst (period = coupled time + G).
            for G in (1e-7, 1e-6, 1e-5, 1e-3):
                ok &= abs(fn(Vb, G, T0, R) - fn(Vb, 0.0, T0, R)) <= 1e-15
    return bool(ok)


def test_completion_coupled_time_pins():
    assert _coupled_pins_hold(bg.completion_coupled_time)


@pytest.mark.parametrize("mutant", [
    lambda V, G, T0, R: T0 + V / R + G,          # gap added to the blocked issue
    lambda V, G, T0, R: max(T0, V / R),          # the max law without the gap
    lambda V, G, T0, R: max(T0, V / R - G),      # the max law itself
    lambda V, G, T0, R: V / R,                   # drain only
    lambda V, G, T0, R: T0 + V / (2 * R),        # half the drain
    lambda V, G, T0, R: T0 + V * R,              # rate inverted
])
def test_completion_coupled_pins_reject_mutants(mutant):
    assert not _coupled_pins_hold(mutant)


def test_coupled_residual_grows_with_bursts_max_law_stays_flat():
    """A producer issues one burst per output tile and then computes for a Q-loop
    gap G >= G* (long sequences). Over n bursts the max law's time beyond the
    backpressure-free floor stays zero, while the completion-coupled sum exposes the
    whole drain of every burst: n * V / R, linear in the number of bursts and hence
    in sequence length (the number of output tiles per producer grows with it)."""
    R, T0 = V["R_bytes_per_s"], V["T0_s"]
    Vb = V["K_producers"] * V["B_bytes_per_producer"]
    G = 2 * bg.recovery_gap(Vb, T0, R)
    for n in (1, 8, 64, 512):
        flat = sum(bg.issue_time(Vb, G, T0, R) - T0 for _ in range(n))
        coupled = sum(bg.completion_coupled_time(Vb, G, T0, R) - T0 for _ in range(n))
        assert flat == 0.0
        assert coupled == pytest.approx(n * Vb / R, rel=1e-12)
