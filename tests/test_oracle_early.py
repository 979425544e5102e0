"""Pins for the early finalization of the grouped online variant
(oracle/sampler.py: score_upper_bound, sample_chunked_early).

* The bound really bounds: every perturbed score of random problems (with
  and without bias, greedy and sampled rows) lies below it.
* G_MAX is the Gumbel quantile of the top of the uniform grid (scipy).
* Early-finalized sampling equals the one-shot sample bit for bit, stops
  after the first chunk when that chunk holds an overwhelming spike, and
  reads every chunk on unpeaked data.
"""

import numpy as np
from scipy import stats

from oracle import sampler
from lm_head_exact_gb300.synthetic import bf16_bits


def _problem(B, V, d, seed, w_std=0.3):
    rng = np.random.default_rng(seed)
    h = bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = bf16_bits((rng.standard_normal((V, d)) * w_std).astype(np.float32))
    return h, W


def test_g_max_is_the_top_of_the_grid():
    assert abs(sampler.G_MAX - stats.gumbel_r.ppf(1 - 2.0 ** -24)) < 1e-12
    g = sampler.gumbel(99, 0, np.arange(64), np.arange(4096))
    assert g.max() <= sampler.G_MAX


def test_bound_dominates_every_score():
    rng = np.random.default_rng(3)
    for trial in range(4):
        B, V, d = 16, 2000, 48
        h, W = _problem(B, V, d, seed=trial)
        temp = rng.uniform(0.05, 2.0, size=B).astype(np.float32)
        temp[:3] = 0.0
        bias = (rng.standard_normal((B, V)) * 5).astype(np.float32) if trial % 2 else None
        ell = sampler.logits(h, W, bias)
        z = sampler.scores(ell, temp, 7, trial, np.arange(B), np.arange(V))
        bmax = np.zeros(B) if bias is None else bias.max(axis=1).astype(np.float64)
        ub = sampler.score_upper_bound(sampler.row_norms(h), sampler.row_norms(W).max(), bmax, temp)
        assert np.all(z.max(axis=1) <= ub)


def test_early_equals_one_shot_on_unpeaked_data_and_reads_everything():
    B, V, d = 6, 3000, 32
    h, W = _problem(B, V, d, seed=5)
    temp = np.array([1.0, 0.5, 0.0, 1.5, 1.0, 0.7], np.float32)
    bounds = [(i * V) // 8 for i in range(8)] + [V]
    (ids, zmax), read = sampler.sample_chunked_early(h, W, temp, 1, 2, bounds)
    ref = sampler.sample(h, W, temp, 1, 2)
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(zmax, ref.zmax)
    assert read == 8


def test_early_stops_after_a_dominant_first_chunk():
    B, V, d = 5, 4000, 32
    h, W = _problem(B, V, d, seed=6)
    temp = np.array([1.0, 0.5, 0.0, 1.5, -1.0], np.float32)     # one invalid row
    bias = np.zeros((B, V), np.float32)
    bias[np.arange(B), [3, 17, 100, 250, 9]] = 1e4               # spikes in chunk 0
    bounds = [0, 500, 1500, 2500, V]
    (ids, zmax), read = sampler.sample_chunked_early(h, W, temp, 4, 4, bounds, bias=bias)
    ref = sampler.sample(h, W, temp, 4, 4, bias=bias)
    np.testing.assert_array_equal(ids, ref.ids)
    np.testing.assert_array_equal(zmax, ref.zmax)
    assert read == 1
    assert ids[4] == -1


def test_row_norms_is_numpy_norm_of_the_decoded_rows():
    import torch
    from lm_head_exact_gb300.synthetic import bf16_bits
    rng = np.random.default_rng(12)
    X = bf16_bits((rng.standard_normal((7, 300)) * 3).astype(np.float32))
    # decode through torch's own bf16 (not the oracle's decoder), norm through numpy
    dec = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_allclose(sampler.row_norms(X), np.linalg.norm(dec, axis=1), rtol=1e-15)
