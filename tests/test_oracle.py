"""Pins for the CPU oracle (CPU only): brute force, invariants, closed forms,
exact cases and the layout's sequence-partition meaning; plus planted-mistake
variants showing each pin set would catch a plausible error."""
import numpy as np
import pytest

import pins
from all_layout_gb300 import inputs


@pytest.fixture()
def rng():
    return np.random.default_rng(1234)


@pytest.mark.parametrize("pin", pins.ATTENTION_PINS, ids=lambda f: f.__name__)
def test_oracle_attention_pins(oracle_lib, pin, rng):
    pin(oracle_lib.attention, rng)


@pytest.mark.parametrize("d", [16, 64, 128])
def test_oracle_one_hot(oracle_lib, d):
    case = inputs.one_hot_case(2, 96, 2, d, seed=5)
    q, k, v, perm = tuple(inputs.bits(t) for t in case[:3]) + (case[3],)
    pins.check_one_hot(oracle_lib.attention, (q, k, v, perm))


@pytest.mark.parametrize("pin", pins.LAYOUT_PINS, ids=lambda f: f.__name__)
def test_oracle_layout_pins(oracle_lib, pin, rng):
    pin(oracle_lib.shard_layout, rng)


def test_layout_inverse_roundtrip(oracle_lib, rng):
    for (B, H, N, d, P) in ((1, 4, 256, 64, 2), (2, 3, 40, 8, 5), (1, 2, 9, 4, 1)):
        o = rng.integers(0, 1 << 16, size=(B, H, N, d), dtype=np.uint16)
        back = oracle_lib.shard_layout_inverse(oracle_lib.shard_layout(o, P))
        assert back.dtype == o.dtype and np.array_equal(back, o)
        f = rng.normal(size=(B, H, N, d))
        assert np.array_equal(oracle_lib.shard_layout_inverse(oracle_lib.shard_layout(f, P)), f)


def test_rows_match_full(oracle_lib, rng):
    q, k, v = (pins.random_bits(rng, (2, 3, 50, 16)) for _ in range(3))
    full = oracle_lib.attention(q, k, v)
    rows = np.array([0, 7, 49, 7, 13])
    part = oracle_lib.attention_rows(q, k, v, rows)
    assert np.array_equal(part, full[:, :, rows])


def test_thread_count_independent(oracle_lib, rng):
    q, k, v = (pins.random_bits(rng, (1, 2, 70, 8)) for _ in range(3))
    a = oracle_lib.attention(q, k, v, threads=1)
    b = oracle_lib.attention(q, k, v, threads=7)
    assert np.array_equal(a, b)


def test_empty_problem(oracle_lib):
    z = np.zeros((0, 2, 8, 4), dtype=np.uint16)
    assert oracle_lib.attention(z, z, z).shape == (0, 2, 8, 4)
    z = np.zeros((1, 2, 0, 4), dtype=np.uint16)
    assert oracle_lib.attention(z, z, z).shape == (1, 2, 0, 4)


# ------------------------------------------------------------ planted mistakes
# Plain numpy attention variants, each with one deliberate error. The pins must
# reject every one of them.

def _np_attention(q, k, v, scale=None, sign=1.0, normalise=True, softmax_axis=-1,
                  v_shift=0, swap_kv=False):
    Q, K, V = pins.bits_to_f64(q), pins.bits_to_f64(k), pins.bits_to_f64(v)
    if swap_kv:
        K, V = V, K
    d = Q.shape[-1]
    s = sign * np.einsum("bhnc,bhjc->bhnj", Q, K) * (scale if scale is not None else d ** -0.5)
    s = s - s.max(axis=softmax_axis, keepdims=True)
    w = np.exp(s)
    if normalise:
        w = w / w.sum(axis=softmax_axis, keepdims=True)
    return np.einsum("bhnj,bhjc->bhnc", w, np.roll(V, v_shift, axis=2))


MUTANTS = {
    "scale_1_over_d": lambda q, k, v: _np_attention(q, k, v, scale=1.0 / q.shape[-1]),
    "no_scale": lambda q, k, v: _np_attention(q, k, v, scale=1.0),
    "negated_scores": lambda q, k, v: _np_attention(q, k, v, sign=-1.0),
    "unnormalised": lambda q, k, v: _np_attention(q, k, v, normalise=False),
    "softmax_over_queries": lambda q, k, v: _np_attention(q, k, v, softmax_axis=-2),
    "value_rows_shifted": lambda q, k, v: _np_attention(q, k, v, v_shift=1),
    "k_and_v_swapped": lambda q, k, v: _np_attention(q, k, v, swap_kv=True),
}


def test_reference_numpy_variant_passes(rng):
    """The unmutated numpy variant passes the same pins (so mutants fail for
    their mistake, not for being numpy)."""
    for pin in pins.ATTENTION_PINS:
        pin(lambda q, k, v: _np_attention(q, k, v), np.random.default_rng(7))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_attention_mistake(name):
    mutant = MUTANTS[name]
    caught = []
    for pin in pins.ATTENTION_PINS:
        try:
            pin(mutant, np.random.default_rng(7))
        except AssertionError:
            caught.append(pin.__name__)
    case = inputs.one_hot_case(1, 64, 2, 16, seed=3)
    try:
        pins.check_one_hot(mutant, tuple(inputs.bits(t) for t in case[:3]) + (case[3],))
    except AssertionError:
        caught.append("check_one_hot")
    assert caught, f"no pin rejects mutant {name}"


LAYOUT_MUTANTS = {
    # shard p takes every P-th token instead of a contiguous block
    "interleaved_tokens": lambda o, P: np.stack(
        [np.transpose(o[:, :, p::P], (0, 2, 1, 3)) for p in range(P)]),
    # heads left in front of tokens inside each shard
    "heads_not_moved": lambda o, P: np.stack(
        [o[:, :, p * (o.shape[2] // P):(p + 1) * (o.shape[2] // P)].reshape(
            o.shape[0], o.shape[2] // P, o.shape[1], o.shape[3]) for p in range(P)]),
    # shards in reverse order
    "reversed_shards": lambda o, P: np.stack(
        [np.transpose(o[:, :, p * (o.shape[2] // P):(p + 1) * (o.shape[2] // P)], (0, 2, 1, 3))
         for p in reversed(range(P))]),
}


@pytest.mark.parametrize("name", sorted(LAYOUT_MUTANTS))
def test_pins_catch_planted_layout_mistake(name):
    caught = []
    for pin in pins.LAYOUT_PINS:
        try:
            pin(LAYOUT_MUTANTS[name], np.random.default_rng(9))
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin rejects layout mutant {name}"
