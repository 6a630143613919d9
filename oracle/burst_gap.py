"""Burst-Gap model of post-issue store progress (X-Stage), as plain formulas.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): used by the tests to check
the product's calibration and store_tile choice; the product implements its
own fit and never imports this module.

Source: the Pith review of "X-Stage: An Overlooked Pipeline Stage for
Communication-Computation Overlap in DiT Inference".
  * "What carries the argument": a fluid-queue abstraction with three platform
    parameters, backpressure-free issue time T0 (T_iss^0), effective drain rate
    R and effective outstanding capacity Q. The sender-visible issue time of a
    burst of V bytes followed by a producer-side gap G is max(T0, V/R - G) (a
    max law); the recovery gap is G* = [V/R - T0]+; the single-burst capacity
    bound is [V - R*T0]+ <= Q.
  * "If this is right": backpressure-free iff the rate bound V/(T0 + G) <= R and
    the capacity bound both hold; the completion-coupled model (issuer blocked
    until remote visibility) is the counterfactual.
  * "Axiom & Free-Parameter Ledger": R ~ 717 GB/s, T0 ~ 0.76 us at K = 148
    producers and B = 32 KB per producer, Q(K = 148) ~ 4.25 MiB, sigma ~ 0.79 us
    of Q-loop gap per KV tile, used for the convergence bound M*_ub (Eq. 20).

Readings where the pages are silent:
  * completion-coupled issue time = T0 + V/R (issue, then wait for the whole
    burst to drain; the gap does not overlap the drain);
  * Eq. 20 is not printed; M*_ub = block_n * G* / sigma is the reading that
    reproduces the pages' "~1.0K" (the Q-loop gap grows by sigma per KV tile of
    block_n keys, and convergence needs that gap to exceed G*).
Units: bytes, seconds, bytes/second.
"""
from __future__ import annotations


def pos(x: float) -> float:
    """[x]+ = max(x, 0)."""
    return x if x > 0.0 else 0.0


def issue_time(V: float, G: float, T0: float, R: float) -> float:
    """Sender-visible issue time of a V-byte burst followed by a gap G: the max law."""
    return max(T0, V / R - G)


def completion_coupled_time(V: float, G: float, T0: float, R: float) -> float:
    """Counterfactual: the issuer is released only when the burst has drained."""
    return T0 + V / R


def recovery_gap(V: float, T0: float, R: float) -> float:
    """G* = [V/R - T0]+: the gap after which the next burst issues at T0."""
    return pos(V / R - T0)


def capacity_excess(V: float, T0: float, R: float) -> float:
    """[V - R*T0]+: bytes a single burst leaves outstanding beyond what drains
    while it is being issued; must not exceed Q."""
    return pos(V - R * T0)


def rate_bound_ok(V: float, G: float, T0: float, R: float) -> bool:
    """Long-term rate bound V / (T0 + G) <= R."""
    return V / (T0 + G) <= R


def backpressure_free(V: float, G: float, T0: float, R: float, Q: float) -> bool:
    """Both the rate bound and the single-burst capacity bound hold."""
    return rate_bound_ok(V, G, T0, R) and capacity_excess(V, T0, R) <= Q


def steady_state_period(V: float, G: float, T0: float, R: float) -> float:
    """Period of back-to-back bursts separated by gap G: issue time plus gap."""
    return issue_time(V, G, T0, R) + G


def convergence_threshold(block_n: int, V: float, T0: float, R: float, sigma: float) -> float:
    """M*_ub: sequence length above which the Q-loop gap (sigma per KV tile of
    block_n keys) exceeds the recovery gap G*."""
    return block_n * recovery_gap(V, T0, R) / sigma
