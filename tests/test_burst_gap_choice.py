"""The calibration's store_tile choice (all_layout_gb300/burst_gap.py) against the
Burst-Gap formulas of the oracle: the largest burst whose schedule is
backpressure-free (rate bound and single-burst capacity bound, Pith review of
X-Stage, "If this is right"). Host logic only, no GPU."""
import itertools
import json
import os

import pytest

from oracle import burst_gap as bg

bgp = pytest.importorskip("all_layout_gb300.burst_gap")

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "burst_gap_pages.json")))
V = {k: v["value"] for k, v in GOLD["values"].items()}


def _expected(T0, R, Q, K, slab, gap):
    for st in (8, 4, 2, 1):
        if bg.backpressure_free(K * st * slab, gap, T0, R, Q):
            return st
    return 1


@pytest.mark.parametrize("T0,R,Q,K,slab,gap", list(itertools.product(
    (0.3e-6, 0.76e-6, 2e-6), (200e9, 717e9, 6.5e12), (0.5 * 2**20, 4.25 * 2**20, 128 * 2**20),
    (64, 148, 152), (2048, 4096), (0.2e-6, 1.8e-6, 10e-6))))
def test_choice_matches_the_model(T0, R, Q, K, slab, gap):
    assert bgp.choose_store_tile(T0, R, Q, K, slab, gap) == _expected(T0, R, Q, K, slab, gap)


def test_choice_on_the_pages_ledger():
    """With the pages' own parameters (K = 148 producers, R ~717 GB/s, T0 ~0.76 us,
    Q ~4.25 MiB) and the Q-loop gap sigma ~0.79 us per KV tile, a 128 x 128 bf16
    output tile (8 slabs of 4 KiB) per producer passes both bounds: the pages'
    "piggyback the whole tile" design."""
    slab = 16 * 128 * 2
    st = bgp.choose_store_tile(V["T0_s"], V["R_bytes_per_s"], V["Q_bytes"], V["K_producers"], slab,
                               V["sigma_s_per_kv_tile"] * 8)
    assert st == 8
    # With no gap at all the rate bound fails for the whole tile and the choice shrinks.
    assert bgp.choose_store_tile(V["T0_s"], V["R_bytes_per_s"], V["Q_bytes"], V["K_producers"], slab,
                                 0.0) < 8
