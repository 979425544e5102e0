"""Pins for the oracle's sampler (oracle/sampler.py) against what the FlashSampling
pages and the mathematics fix.

* Sampling law: Gumbel-max gives an exact sample of softmax(logits / T)
  (summary page, Key claims) -- chi-square of >= 10^6 draws against the closed
  form computed with scipy's softmax.
* Greedy limit: T == 0 is numpy.argmax of the logits; T -> 0 converges to it.
* Partition invariance: argmax decomposes over any partition of the vocabulary
  (abstract; summary page, Method) -- tile sizes {1, 7, 128, 256, V} and random
  partitions folded in random order give identical results.
* Chunked (grouped online) variant equals the one-shot sample (abstract).
* Total order: ties go to the smaller id; NaN / -inf never win; invalid T.
"""

import numpy as np
import pytest
from scipy import special, stats

from oracle import sampler
from lm_head_exact_gb300.synthetic import bf16_bits


def _problem(B, V, d, seed, w_std=0.3):
    rng = np.random.default_rng(seed)
    h = bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = bf16_bits((rng.standard_normal((V, d)) * w_std).astype(np.float32))
    return h, W


def _draw_counts(h1, W, T, n, seed=1234, step=0, batch=125000):
    """n draws from the row h1 (repeated n times: each row has its own counters)."""
    V = W.shape[0]
    counts = np.zeros(V, dtype=np.int64)
    hrep = np.repeat(h1, n, axis=0)
    temp = np.full(n, T, np.float32)
    for lo in range(0, n, batch):
        rows = np.arange(lo, min(n, lo + batch))
        s = sampler.sample(hrep, W, temp, seed, step, rows=rows)
        counts += np.bincount(s.ids, minlength=V)
    return counts


def _chi2_pvalue(counts, probs, min_expected=5.0):
    n = counts.sum()
    exp = probs * n
    order = np.argsort(exp)
    # merge the smallest bins until every merged bin expects >= min_expected
    c_bins, e_bins, c_acc, e_acc = [], [], 0, 0.0
    for i in order:
        c_acc += counts[i]
        e_acc += exp[i]
        if e_acc >= min_expected:
            c_bins.append(c_acc)
            e_bins.append(e_acc)
            c_acc, e_acc = 0, 0.0
    if e_acc > 0:
        c_bins[-1] += c_acc
        e_bins[-1] += e_acc
    return stats.chisquare(np.array(c_bins), np.array(e_bins)).pvalue


@pytest.mark.parametrize("V", [8, 64])
@pytest.mark.parametrize("T", [0.5, 1.0, 1.5])
def test_sampling_law_chi_square(V, T):
    h, W = _problem(1, V, 16, seed=V)
    ell = sampler.logits(h, W)[0]
    probs = special.softmax(ell / T)
    counts = _draw_counts(h, W, T, 1_000_000, step=int(T * 10))
    assert counts.sum() == 1_000_000
    assert _chi2_pvalue(counts, probs) > 0.01


def test_sampling_law_wider_vocabulary():
    V = 512
    h, W = _problem(1, V, 32, seed=99, w_std=0.4)
    ell = sampler.logits(h, W)[0]
    probs = special.softmax(ell)
    counts = _draw_counts(h, W, 1.0, 200_000)
    assert _chi2_pvalue(counts, probs) > 0.01


def test_chi_square_detects_wrong_temperature():
    # The same draws tested against softmax(logits) at the wrong T must fail:
    # the test has the power to see a dropped temperature.
    V = 8
    h, W = _problem(1, V, 16, seed=V)
    ell = sampler.logits(h, W)[0]
    counts = _draw_counts(h, W, 0.5, 1_000_000, step=5)
    assert _chi2_pvalue(counts, special.softmax(ell / 1.0)) < 1e-6


def test_infinite_temperature_is_uniform():
    V = 64
    h, W = _problem(1, V, 16, seed=2)
    counts = _draw_counts(h, W, np.inf, 400_000)
    assert _chi2_pvalue(counts, np.full(V, 1.0 / V)) > 0.01


def test_greedy_is_numpy_argmax():
    h, W = _problem(64, 3000, 64, seed=4)
    s = sampler.sample(h, W, np.zeros(64, np.float32), 1234, 0)
    ell = sampler.logits(h, W)
    np.testing.assert_array_equal(s.ids, np.argmax(ell, axis=1))
    np.testing.assert_array_equal(s.zmax, ell.max(axis=1))


def test_small_temperature_converges_to_greedy():
    h, W = _problem(256, 2000, 64, seed=6)
    ell = sampler.logits(h, W)
    greedy = np.argmax(ell, axis=1)
    T = 1e-6
    s = sampler.sample(h, W, np.full(256, T, np.float32), 1234, 3)
    top2 = np.sort(ell, axis=1)[:, -2:]
    # Gumbel noise on the u grid lies in [-2.81, 16.64]: beyond a gap of
    # 19.5 * T the noise cannot reorder the top two logits.
    clear = (top2[:, 1] - top2[:, 0]) > 40 * T
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(s.ids[clear], greedy[clear])


def _tile_parts(V, t):
    return [np.arange(i, min(V, i + t)) for i in range(0, V, t)]


@pytest.mark.parametrize("tile", [1, 7, 128, 256, None])
def test_partition_invariance_tiles(tile):
    B, V = 6, 1000
    h, W = _problem(B, V, 32, seed=8)
    temp = np.array([0.0, 0.5, 1.0, 1.5, 0.7, 2.0], np.float32)
    ref = sampler.sample(h, W, temp, 1234, 11)
    ids, zmax = sampler.sample_partitioned(h, W, temp, 1234, 11, _tile_parts(V, tile or V))
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(zmax, ref.zmax)


@pytest.mark.parametrize("trial", range(5))
def test_partition_invariance_random(trial):
    rng = np.random.default_rng(100 + trial)
    B, V = 5, 777
    h, W = _problem(B, V, 24, seed=9 + trial)
    temp = rng.uniform(0.2, 2.0, size=B).astype(np.float32)
    temp[0] = 0.0
    ref = sampler.sample(h, W, temp, 42, trial)
    perm = rng.permutation(V)
    cuts = np.sort(rng.choice(np.arange(1, V), size=rng.integers(1, 40), replace=False))
    parts = np.split(perm, cuts)
    rng.shuffle(parts)
    ids, zmax = sampler.sample_partitioned(h, W, temp, 42, trial, parts)
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(zmax, ref.zmax)


@pytest.mark.parametrize("n_chunks", [1, 8, 32])
def test_chunked_equals_one_shot(n_chunks):
    B, V = 7, 4097
    h, W = _problem(B, V, 32, seed=12)
    temp = np.array([1.0, 0.0, 0.3, 1.5, 1.0, 0.9, 1.2], np.float32)
    ref = sampler.sample(h, W, temp, 1234, 77)
    bounds = [(i * V) // n_chunks for i in range(n_chunks)] + [V]
    ids, zmax = sampler.sample_chunked(h, W, temp, 1234, 77, bounds)
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(zmax, ref.zmax)


def test_chunked_with_bias_and_ragged_bounds():
    B, V = 4, 1500
    h, W = _problem(B, V, 16, seed=13)
    rng = np.random.default_rng(13)
    bias = np.zeros((B, V), np.float32)
    bias[np.arange(B)[:, None], rng.integers(0, V, size=(B, 16))] = 8.0
    temp = np.ones(B, np.float32)
    ref = sampler.sample(h, W, temp, 5, 1, bias=bias)
    bounds = [0, 1, 130, 131, 999, V]
    ids, zmax = sampler.sample_chunked(h, W, temp, 5, 1, bounds, bias=bias)
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(zmax, ref.zmax)


def test_tie_goes_to_smaller_id():
    h, _ = _problem(3, 1, 16, seed=14)
    W = np.repeat(_problem(1, 1, 16, seed=15)[1], 300, axis=0)   # identical rows
    temp = np.zeros(3, np.float32)
    s = sampler.sample(h, W, temp, 1, 0)
    np.testing.assert_array_equal(s.ids, [0, 0, 0])
    ids, _ = sampler.sample_partitioned(h, W, temp, 1, 0, [np.arange(150, 300), np.arange(150)])
    np.testing.assert_array_equal(ids, [0, 0, 0])


def test_invalid_temperature_rows():
    h, W = _problem(4, 50, 16, seed=16)
    temp = np.array([-1.0, np.nan, 1.0, 0.0], np.float32)
    s = sampler.sample(h, W, temp, 1, 0)
    assert s.ids[0] == -1 and s.ids[1] == -1
    assert s.zmax[0] == -np.inf and s.zmax[1] == -np.inf
    assert s.ids[2] >= 0 and s.ids[3] >= 0


def test_nan_and_neg_inf_never_win():
    h, W = _problem(2, 10, 8, seed=17)
    W = W.copy()
    W[3] = 0x7FC0                                        # NaN row -> NaN logits
    bias = np.zeros((2, 10), np.float32)
    bias[:, 5] = -np.inf
    bias[1, :] = -np.inf                                 # row 1: nothing can win
    s = sampler.sample(h, W, np.ones(2, np.float32), 1, 0, bias=bias)
    assert s.ids[0] not in (3, 5)
    assert s.ids[1] == -1 and s.zmax[1] == -np.inf
    allnan = np.full_like(W, 0x7FC0)
    s2 = sampler.sample(h, allnan, np.ones(2, np.float32), 1, 0)
    np.testing.assert_array_equal(s2.ids, [-1, -1])


def test_bias_spike_wins():
    h, W = _problem(8, 300, 16, seed=18)
    bias = np.zeros(300, np.float32)
    bias[217] = 1000.0                                   # shared [V] bias
    s = sampler.sample(h, W, np.full(8, 1.5, np.float32), 9, 9, bias=bias)
    np.testing.assert_array_equal(s.ids, np.full(8, 217))
    bias2 = np.zeros(300, np.float32)
    bias2[[40, 41]] = np.inf                             # equal +inf -> smaller id
    s2 = sampler.sample(h, W, np.ones(8, np.float32), 9, 9, bias=bias2)
    np.testing.assert_array_equal(s2.ids, np.full(8, 40))


def test_combine_is_a_commutative_monoid():
    rng = np.random.default_rng(19)
    n = 5000

    def rand():
        ids = rng.integers(-1, 20, size=n)
        z = rng.integers(-3, 3, size=n).astype(np.float64)   # many ties
        z[ids == -1] = -np.inf
        return ids, z

    a, b, c = rand(), rand(), rand()
    ident = (np.full(n, -1), np.full(n, -np.inf))
    for x, y in zip(sampler.combine(a, b), sampler.combine(b, a)):
        np.testing.assert_array_equal(x, y)
    for x, y in zip(sampler.combine(sampler.combine(a, b), c), sampler.combine(a, sampler.combine(b, c))):
        np.testing.assert_array_equal(x, y)
    for x, y in zip(sampler.combine(a, ident), a):
        np.testing.assert_array_equal(x, y)


def test_top2_gap():
    z = np.array([[1.0, 3.0, 2.5, np.nan], [0.0, -np.inf, np.nan, -np.inf], [2.0, 2.0, 1.0, 0.0]])
    np.testing.assert_array_equal(sampler.top2_gap(z), [0.5, np.inf, 0.0])
