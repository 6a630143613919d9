"""Store-burst probe and local Burst-Gap calibration on the GPU (through the C ABI)."""
import numpy as np
import pytest
import torch

from oracle import burst_gap as bg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def xs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs as _xs
    return _xs


@pytest.mark.parametrize("mode", [0, 1])
def test_probe_writes_and_times(xs, mode):
    K, B, n, gap = 6, 32768, 5, 3000
    dst = torch.zeros(K * n * B, dtype=torch.uint8, device="cuda")
    times = torch.zeros(2 * K * n, dtype=torch.int64, device="cuda")
    xs.store_burst_probe(dst, K, B, n, gap, mode, times)
    torch.cuda.synchronize()
    t = times.view(K, n, 2).cpu().numpy()
    assert np.all(t[..., 1] >= t[..., 0]) and np.all(t > 0)
    assert np.all(t[:, 1:, 0] - t[:, :-1, 1] >= gap)          # the gap has no stores in it
    w = dst.view(torch.int32).view(K, n, B // 16, 4).cpu().numpy()
    c = np.arange(B // 16)
    for k in range(K):
        if mode == 0:
            exp = np.stack([c % 128, np.full_like(c, k), np.ones_like(c), 2 * np.ones_like(c)], -1)
        else:
            exp = np.stack([c % 1024, np.full_like(c, k), np.full_like(c, 0x5a5a5a5a),
                            np.zeros_like(c)], -1)
        assert np.array_equal(w[k], np.broadcast_to(exp, w[k].shape)), k


def test_probe_validation(xs):
    lib = xs.library()
    A = 0x10000
    assert lib.xs_store_burst_probe(A, 1 << 20, 0, 2048, 1, 0, 0, A, None) == xs.ERR_INVALID
    assert lib.xs_store_burst_probe(A, 1 << 20, 1, 1000, 1, 0, 0, A, None) == xs.ERR_INVALID
    assert lib.xs_store_burst_probe(A, 4096, 4, 2048, 1, 0, 0, A, None) == xs.ERR_INVALID
    assert lib.xs_store_burst_probe(A, 1 << 20, 1, 2048, 1, 0, 2, A, None) == xs.ERR_INVALID
    assert lib.xs_store_burst_probe(A + 8, 1 << 20, 1, 2048, 1, 0, 0, A, None) == xs.ERR_ALIGN


def test_local_calibration_and_max_law(xs):
    from all_layout_gb300 import burst_gap
    rep = burst_gap.calibrate()
    T0, R, Q = rep["T0_s"], rep["R_bytes_per_s"], rep["Q_bytes"]
    assert 0 < T0 < 1e-3 and 1e10 < R < 1e14 and Q >= 0
    assert rep["store_tile"] in (1, 2, 4, 8)
    # The oracle's formulas with the fitted parameters reproduce the module's model
    # column, and the model tracks the measured steady-state issue span.
    errs = []
    for rows, B in zip(rep["max_law"], (1 << 16, 1 << 18, 1 << 20)):
        for row in rows:
            pred = bg.issue_time(rep["K"] * B, row["gap_s"], row["T0_s"], R)
            assert row["model_s"] == pytest.approx(pred)
            errs.append(abs(row["measured_s"] - pred) / pred)
    assert np.median(errs) < 0.35, errs
