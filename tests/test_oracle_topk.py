"""Pins for the oracle's Gumbel-top-k (oracle/topk.py) against what the
mathematics fixes.

* k = 1 is the sampler itself (same ids, same winning scores).
* Law: the top k perturbed scores are k draws WITHOUT replacement, each from
  the renormalized remaining mass (the Plackett-Luce law of ordered tuples):
  P(i1, ..., ik) = prod_j p_ij / (1 - sum_{l<j} p_il) with p = softmax(logits / T)
  computed by scipy.  Chi-square over ordered tuples; a plausible wrong law
  (independent draws conditioned on being distinct) is rejected.
* Partition invariance: per-part top-k lists merged give the same result.
* Total order: equal scores -> smaller id first; -inf / NaN never selected;
  rows with fewer than k selectable ids are padded with (-1, -inf).
"""

import itertools

import numpy as np
import pytest
from scipy import special, stats

from oracle import sampler, topk
from lm_head_exact_gb300.synthetic import bf16_bits


def _problem(B, V, d, seed, w_std=0.3):
    rng = np.random.default_rng(seed)
    h = bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = bf16_bits((rng.standard_normal((V, d)) * w_std).astype(np.float32))
    return h, W


def test_k1_is_the_sampler():
    B, V = 9, 300
    h, W = _problem(B, V, 32, seed=1)
    temp = np.array([1.0, 0.0, 0.5, 1.5, -1.0, np.nan, 0.7, 2.0, 1.0], np.float32)
    t = topk.sample_topk(h, W, temp, 1234, 5, 1)
    s = sampler.sample(h, W, temp, 1234, 5)
    np.testing.assert_array_equal(t.ids[:, 0], s.ids)
    np.testing.assert_array_equal(t.z[:, 0], s.zmax)


def _tuple_counts(h1, W, T, k, n, seed=99):
    """Ordered k-tuples from n rows that repeat h1 (each row has its own noise)."""
    V = W.shape[0]
    hrep = np.repeat(h1, n, axis=0)
    temp = np.full(n, T, np.float32)
    t = topk.sample_topk(hrep, W, temp, seed, 0, k)
    codes = np.zeros(n, dtype=np.int64)
    for j in range(k):
        codes = codes * V + t.ids[:, j]
    return np.bincount(codes, minlength=V ** k)


def _plackett_luce(p, k):
    V = len(p)
    probs = np.zeros(V ** k)
    for tup in itertools.permutations(range(V), k):
        pr, used = 1.0, 0.0
        for i in tup:
            pr *= p[i] / (1.0 - used)
            used += p[i]
        code = 0
        for i in tup:
            code = code * V + i
        probs[code] = pr
    return probs


def _distinct_independent(p, k):
    """Wrong law: independent draws from p, conditioned on being distinct."""
    V = len(p)
    probs = np.zeros(V ** k)
    for tup in itertools.permutations(range(V), k):
        code = 0
        for i in tup:
            code = code * V + i
        probs[code] = np.prod(p[list(tup)])
    return probs / probs.sum()


def _chi2(counts, probs):
    keep = probs > 0
    assert counts[~keep].sum() == 0, "a tuple with a repeated id was drawn"
    exp = probs[keep] * counts.sum()
    assert exp.min() >= 5
    return stats.chisquare(counts[keep], exp).pvalue


@pytest.mark.parametrize("V,k,T", [(6, 2, 1.0), (5, 3, 0.7)])
def test_plackett_luce_law(V, k, T):
    h, W = _problem(1, V, 16, seed=20 + V, w_std=0.25)
    ell = sampler.logits(h, W)[0]
    p = special.softmax(ell / T)
    counts = _tuple_counts(h, W, T, k, 300_000)
    assert _chi2(counts, _plackett_luce(p, k)) > 1e-3
    assert _chi2(counts, _distinct_independent(p, k)) < 1e-6


@pytest.mark.parametrize("trial", range(3))
def test_partition_invariance(trial):
    rng = np.random.default_rng(40 + trial)
    B, V, k = 6, 1000, 5
    h, W = _problem(B, V, 32, seed=50 + trial)
    temp = np.array([1.0, 0.0, 0.4, 1.3, 2.0, 0.8], np.float32)
    ref = topk.sample_topk(h, W, temp, 7, trial, k)
    cuts = np.sort(rng.choice(np.arange(1, V), size=rng.integers(1, 30), replace=False))
    parts = [0] + [int(c) for c in cuts] + [V]
    ids, z = topk.sample_topk_partitioned(h, W, temp, 7, trial, k, parts)
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(z, ref.z)


def test_ties_masks_and_padding():
    B, V, d, k = 3, 12, 8, 6
    h, W = _problem(B, V, d, seed=3)
    W[7] = W[2]
    W[9] = W[2]                                         # three equal logits
    temp = np.array([0.0, 1.0, 1.0], np.float32)
    bias = np.zeros((B, V), np.float32)
    bias[0, [2, 7, 9]] = 50.0                           # the three equal logits lead row 0
    bias[1, :] = -np.inf
    bias[1, [4, 5]] = 0.0                               # row 1: only two selectable ids
    bias[2, 0] = -np.inf                                # row 2: id 0 masked
    t = topk.sample_topk(h, W, temp, 11, 0, k, bias=bias)
    np.testing.assert_array_equal(t.ids[0, :3], [2, 7, 9])
    assert np.all(t.z[0, :3] == t.z[0, 0])
    assert sorted(t.ids[1, :2]) == [4, 5] and np.all(t.ids[1, 2:] == -1) and np.all(t.z[1, 2:] == -np.inf)
    assert 0 not in t.ids[2] and len(set(t.ids[2])) == k
    assert np.all(np.diff(t.z[2]) <= 0)


def test_gap_definition():
    zz = np.array([[5.0, 4.0, 3.5, 3.4, -np.inf]])
    g = topk._gaps(zz, 4)
    np.testing.assert_allclose(g[0], [1.0, 0.5, 0.1, 0.1])
    zz = np.array([[2.0, -np.inf, -np.inf]])
    assert np.all(topk._gaps(zz, 2)[0] == np.inf)
