"""The polynomial exponential of the softmax (exp2_poly_x2 in csrc/ptx.cuh).

CPU: the coefficients embedded in the kernel are the ones the committed fit
(csrc/exp2_poly_fit.py, Remez exchange for the minimax relative error of 2^f on
[0, 1]) produces, and the fit meets its error bound at every float32 input of a
dense grid, emulated in float32 with the kernel's operation order.
GPU: the kernel's own evaluation against exact 2^x (float64) within that bound,
and against the MUFU ex2.approx results it stands in for."""
import importlib.util
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "all_layout_gb300", "csrc")
BOUND = 7.5e-5 + 4 * 2.0 ** -24      # minimax error + fp32 rounding of the evaluation


def _fit():
    spec = importlib.util.spec_from_file_location("exp2_poly_fit", os.path.join(CSRC, "exp2_poly_fit.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _embedded():
    text = open(os.path.join(CSRC, "ptx.cuh")).read()
    body = text[text.index("exp2_poly_x2"):]
    return [float(re.search(rf"\bc{i} = ([0-9.eE+-]+)f", body).group(1)) for i in range(4)]


def test_embedded_coefficients_are_the_fit():
    fit = _fit()
    assert _embedded() == fit.coefficients_f32()
    c, E = fit.remez_relative()
    assert 7.0e-5 < E < 7.6e-5        # degree 3 levels near 2^-13.7


def _emulate(x):
    """float32 emulation of exp2_poly_x2 (same operation order)."""
    c0, c1, c2, c3 = (np.float32(v) for v in _embedded())
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    n = np.floor(x)
    f = (x - n).astype(np.float32)
    fma = lambda a, b, c: (a.astype(np.float64) * np.float64(b) + np.float64(c)).astype(np.float32)
    p = fma(f, c3, c2)          # fused multiply-add: the product is exact in float64
    p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c1)).astype(np.float32)
    p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(c0)).astype(np.float32)
    bits = p.view(np.uint32).astype(np.int64) + (n.astype(np.int64) << 23)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_emulated_error_bound():
    x = np.linspace(-125.0, 9.0, 2_000_001, dtype=np.float32)
    got = _emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got / ref - 1.0)
    assert rel.max() <= BOUND, rel.max()
    # continuity across integers: no step larger than the bound at n -> n + 1
    k = np.arange(-20, 9, dtype=np.float32)
    below = _emulate(np.nextafter(k, np.float32(-np.inf)))
    at = _emulate(k)
    assert np.all(np.abs(at / below - 1.0) <= 2 * BOUND)
    # far below the range: a tiny positive number, never NaN, Inf or negative
    tiny = _emulate(np.array([-126.0, -200.0, -1e6, -np.inf], dtype=np.float32))
    assert np.all(np.isfinite(tiny)) and np.all(tiny >= 0) and np.all(tiny <= 2.0 ** -125)


@pytest.mark.gpu
def test_kernel_polynomial_against_exact_and_mufu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from all_layout_gb300 import xs
    rng = np.random.default_rng(5)
    x = np.concatenate([np.linspace(-125.0, 9.0, 1_000_001), rng.uniform(-30, 8, 200_000),
                        np.arange(-125, 9), np.arange(-125, 9) - 2.0 ** -20]).astype(np.float32)
    poly, mufu = xs.selftest_exp2(torch.from_numpy(x).cuda())
    poly = poly.cpu().numpy().astype(np.float64)
    mufu = mufu.cpu().numpy().astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.abs(poly / ref - 1.0).max() <= BOUND
    # the emulation above is what the kernel computes (up to the double rounding of
    # a float64 stand-in for the fused multiply-add: 2 ulp at most)
    emu = _emulate(x).astype(np.float64)
    assert np.abs(poly / emu - 1.0).max() <= 2.0 ** -22
    # against the MUFU results it replaces: within the polynomial's bound plus ex2.approx's own
    assert np.abs(poly / mufu - 1.0).max() <= BOUND + 2.0 ** -21
    low = np.array([-126.0, -150.0, -1000.0], dtype=np.float32)
    p2, _ = xs.selftest_exp2(torch.from_numpy(low).cuda())
    p2 = p2.cpu().numpy()
    assert np.all(np.isfinite(p2)) and np.all(p2 >= 0) and np.all(p2 <= 2.0 ** -125)
