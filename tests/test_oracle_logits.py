"""Pins for the oracle's bf16 decode and fp64 logits (oracle/sampler.py).

* bf16 decode is compared with torch's own bfloat16 -> float64 conversion on
  every one of the 65536 bit patterns.
* logits are compared with exact rational sums (Python ``fractions``) on tiny,
  non-square inputs, so a transposed operand, a dropped term or a missing bias
  fails.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import sampler
from lm_head_exact_gb300.synthetic import bf16_bits


def test_bf16_decode_matches_torch_on_all_patterns():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = sampler.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def _exact_logits(h_bits, W_bits, bias=None):
    hv = [[Fraction(float(x)) for x in row] for row in sampler.bf16_to_f64(h_bits)]
    Wv = [[Fraction(float(x)) for x in row] for row in sampler.bf16_to_f64(W_bits)]
    out = []
    for b, hr in enumerate(hv):
        row = []
        for v, wr in enumerate(Wv):
            s = sum(x * y for x, y in zip(hr, wr))
            if bias is not None:
                s += Fraction(float(bias[b, v] if bias.ndim == 2 else bias[v]))
            row.append(s)
        out.append(row)
    return out


@pytest.mark.parametrize("B,V,d", [(3, 5, 16), (1, 7, 8), (4, 2, 24)])
def test_logits_exact_rational(B, V, d):
    rng = np.random.default_rng(B * 100 + V * 10 + d)
    h = bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = bf16_bits((rng.standard_normal((V, d)) * 0.05).astype(np.float32))
    ours = sampler.logits(h, W)
    exact = _exact_logits(h, W)
    scale = np.abs(sampler.bf16_to_f64(h)) @ np.abs(sampler.bf16_to_f64(W)).T
    for b in range(B):
        for v in range(V):
            assert abs(Fraction(ours[b, v]) - exact[b][v]) <= Fraction(scale[b, v]) * Fraction(d, 2**52)


def test_logits_integer_inputs_are_exact():
    rng = np.random.default_rng(5)
    h = bf16_bits(rng.integers(-8, 9, size=(3, 32)).astype(np.float32))
    W = bf16_bits(rng.integers(-8, 9, size=(6, 32)).astype(np.float32))
    ours = sampler.logits(h, W)
    exact = _exact_logits(h, W)
    for b in range(3):
        for v in range(6):
            assert Fraction(ours[b, v]) == exact[b][v]


@pytest.mark.parametrize("shared", [False, True])
def test_logits_with_bias(shared):
    rng = np.random.default_rng(11)
    h = bf16_bits(rng.standard_normal((2, 8)).astype(np.float32))
    W = bf16_bits(rng.standard_normal((5, 8)).astype(np.float32))
    bias = (rng.standard_normal(5) if shared else rng.standard_normal((2, 5))).astype(np.float32)
    ours = sampler.logits(h, W, bias)
    exact = _exact_logits(h, W, bias)
    for b in range(2):
        for v in range(5):
            assert abs(Fraction(ours[b, v]) - exact[b][v]) < Fraction(1, 2**40)
