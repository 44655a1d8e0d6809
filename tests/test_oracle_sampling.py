"""Pins of the sampling oracle (Paso 8 of "Dentro de un LLM: Inferencia en Python puro para
Qwen3-0.6B en MLX": temperature, softmax, top-p nucleus, draw) against hand-computed cases,
the exact-boundary rule of the cutoff, a brute-force nucleus and the drawn frequencies.
No GPU."""

import math

import numpy as np
import pytest

import oracle

P4 = np.array([0.5, 0.3, 0.15, 0.05])


def test_greedy_is_lowest_argmax():
    assert oracle.sample_top_p(np.array([1.0, 3.0, 3.0, 2.0]), 0.0, 0.95, 0.7) == 1


def test_hand_example_unit_temperature():
    lg = np.log(P4)
    # top_p 0.7: running sums 0.5, 0.8, ... -> one below 0.7 -> keep 2: weights 0.625, 0.375
    ids, c = oracle.kept_cdf(lg, 1.0, 0.7)
    np.testing.assert_array_equal(ids, [0, 1])
    np.testing.assert_allclose(c, [0.625, 1.0], rtol=0, atol=1e-12)
    assert oracle.sample_top_p(lg, 1.0, 0.7, 0.6) == 0
    assert oracle.sample_top_p(lg, 1.0, 0.7, 0.63) == 1
    # top_p 0.9: keep 3, weights 0.5, 0.3, 0.15 over 0.95
    ids, c = oracle.kept_cdf(lg, 1.0, 0.9)
    np.testing.assert_array_equal(ids, [0, 1, 2])
    np.testing.assert_allclose(c, [0.5 / 0.95, 0.8 / 0.95, 1.0], rtol=0, atol=1e-12)
    assert oracle.sample_top_p(lg, 1.0, 0.9, 0.84) == 1
    assert oracle.sample_top_p(lg, 1.0, 0.9, 0.85) == 2


def test_draw_enumerates_kept_tokens_by_id():
    p = np.array([0.05, 0.5, 0.15, 0.3])  # the same distribution, ids permuted
    lg = np.log(p)
    ids, c = oracle.kept_cdf(lg, 1.0, 0.7)
    np.testing.assert_array_equal(ids, [1, 3])
    np.testing.assert_allclose(c, [0.625, 1.0], rtol=0, atol=1e-12)
    assert oracle.sample_top_p(lg, 1.0, 0.7, 0.6) == 1
    assert oracle.sample_top_p(lg, 1.0, 0.7, 0.63) == 3


def test_temperature_divides_the_logits():
    lg = np.log(P4)
    # T = 0.5 squares the probabilities: 0.25, 0.09, 0.0225, 0.0025 over 0.365
    p = oracle.softmax_t(lg, 0.5)
    np.testing.assert_allclose(p, P4 ** 2 / np.sum(P4 ** 2), rtol=1e-12)
    ids, c = oracle.kept_cdf(lg, 0.5, 0.9)  # running sums 0.685, 0.932 -> keep 2
    np.testing.assert_array_equal(ids, [0, 1])
    np.testing.assert_allclose(c[0], 0.25 / 0.34, rtol=1e-12)
    assert oracle.sample_top_p(lg, 0.5, 0.9, 0.73) == 0
    assert oracle.sample_top_p(lg, 0.5, 0.9, 0.74) == 1


def test_cutoff_counts_sums_strictly_below_top_p():
    # exact binary fractions: running sums 0.5, 0.75, 1.0; 0.75 is not below 0.75 -> keep 2
    ids, kp = oracle.nucleus(np.array([0.5, 0.25, 0.25]), 0.75)
    np.testing.assert_array_equal(ids, [0, 1])
    ids, _ = oracle.nucleus(np.array([0.5, 0.25, 0.25]), 0.7500001)
    np.testing.assert_array_equal(ids, [0, 1, 2])


def test_ties_keep_lowest_ids_and_top_p_one_keeps_all():
    p = np.full(10, 0.1)
    ids, _ = oracle.nucleus(p, 0.25)
    np.testing.assert_array_equal(ids, [0, 1, 2])
    ids, _ = oracle.nucleus(P4, 1.0)
    np.testing.assert_array_equal(np.sort(ids), [0, 1, 2, 3])


def _brute_nucleus(p, top_p):
    order = sorted(range(len(p)), key=lambda i: (-p[i], i))
    s = 0.0
    for k, i in enumerate(order):
        s += p[i]
        if s >= top_p:
            return set(order[:k + 1])
    return set(order)


@pytest.mark.parametrize("T,top_p", [(1.0, 0.5), (0.7, 0.9), (2.0, 0.95), (0.3, 0.99)])
def test_nucleus_and_frequencies_brute_force(T, top_p):
    rng = np.random.default_rng(7)
    lg = rng.normal(0.0, 2.0, 40)
    p = oracle.softmax_t(lg, T)
    ids, _ = oracle.nucleus(p, top_p)
    assert set(ids.tolist()) == _brute_nucleus(p.tolist(), top_p)
    # stratified u: frequencies equal the renormalised nucleus probabilities
    N = 20000
    counts = np.zeros(40)
    for k in range(N):
        counts[oracle.sample_top_p(lg, T, top_p, (k + 0.5) / N)] += 1
    kept = sorted(ids.tolist())
    want = np.zeros(40)
    want[kept] = p[kept] / p[kept].sum()
    np.testing.assert_allclose(counts / N, want, rtol=0, atol=1.0 / N + 1e-12)


def test_shift_invariance():
    rng = np.random.default_rng(3)
    lg = rng.normal(0.0, 1.0, 200)
    us = (np.arange(97) + 0.37) / 97
    a = [oracle.sample_top_p(lg, 0.8, 0.9, u) for u in us]
    b = [oracle.sample_top_p(lg + 3.0, 0.8, 0.9, u) for u in us]
    assert a == b
    assert math.isclose(oracle.softmax_t(lg + 3.0, 0.8).sum(), 1.0)
