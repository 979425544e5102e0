"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: Llama-3-8B-, Qwen3-8B- and Llama-3-70B-shaped LM heads and
the chunked (grouped online) variant.

For every workload, EVERY row of one decode step is compared with the fp64
oracle over the whole vocabulary, at every batch size of the workload (a
smaller batch is a prefix of the largest, and a row's noise counter is its
batch index, so one oracle pass over the largest batch serves all of them).
The oracle's logits do not depend on the step, so they are computed once per
workload (in vocabulary blocks, to bound host memory) and reused; the other
steps compare a seeded subset of rows.  The number of rows inside the
near-tie band is logged for the run's summary.
"""

import numpy as np
import pytest

from _helpers import compare, oracle_rows, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu

_ELL = {}


def _rows(B, k, seed, must=()):
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in rng.choice(B, size=min(k, B), replace=False))
    rows.update(int(r) for r in must if r < B)
    return np.array(sorted(rows))


def _device(wl, torch):
    return (to_device(wl.h, torch), to_device(wl.W, torch), to_device(wl.temp, torch),
            None if wl.bias is None else to_device(wl.bias, torch))


def _logits(name, wl, vblock=16384):
    """fp64 oracle logits of every row of the workload (bias included),
    computed once per workload, vocabulary block by vocabulary block."""
    if name not in _ELL:
        B, V = wl.h.shape[0], wl.W.shape[0]
        ell = np.empty((B, V), dtype=np.float64)
        for v0 in range(0, V, vblock):
            v1 = min(V, v0 + vblock)
            bias = None if wl.bias is None else wl.bias[:, v0:v1]
            ell[:, v0:v1] = sampler.logits(wl.h, wl.W[v0:v1], bias)
        _ELL.clear()                     # one workload's logits at a time
        _ELL[name] = ell
    return _ELL[name]


def test_llama3_8b_batch_sweep(fs, torch_cuda):
    torch = torch_cuda
    wl = synthetic.workload("llama3_8b", 64)
    hd, Wd, td, _ = _device(wl, torch)
    ell = _logits("llama3_8b", wl)
    for step in (0, 57, 99):
        ref = oracle_rows(ell, wl.temp, wl.seed, step)
        for B in synthetic.SHAPES["llama3_8b"]["batches"]:
            ids, mx = fs.sample(hd[:B], Wd, td[:B], wl.seed, step)
            torch.cuda.synchronize()
            sub = sampler.Sample(ref.ids[:B], ref.zmax[:B], ref.gap[:B])
            compare(ids.cpu().numpy(), mx.cpu().numpy(), sub, what=f"8B B={B} step={step}")


def test_qwen3_8b_large_batch(fs, torch_cuda):
    torch = torch_cuda
    wl = synthetic.workload("qwen3_8b", 1024)
    hd, Wd, td, _ = _device(wl, torch)
    ell = _logits("qwen3_8b", wl)
    greedy_rows = np.nonzero(wl.temp == 0)[0]
    ref0 = oracle_rows(ell, wl.temp, wl.seed, 0)       # every row, step 0
    for step in (0, 9):
        for B in synthetic.SHAPES["qwen3_8b"]["batches"]:
            ids, mx = fs.sample(hd[:B], Wd, td[:B], wl.seed, step)
            torch.cuda.synchronize()
            if step == 0:
                sub = sampler.Sample(ref0.ids[:B], ref0.zmax[:B], ref0.gap[:B])
                compare(ids.cpu().numpy(), mx.cpu().numpy(), sub, what=f"qwen B={B} step=0 all rows")
            else:
                rows = _rows(B, 24, seed=B + step, must=greedy_rows[:4])
                ref = oracle_rows(ell[rows], wl.temp[rows], wl.seed, step, rows=rows)
                compare(ids.cpu().numpy(), mx.cpu().numpy(), ref, rows=rows, what=f"qwen B={B} step={step}")


def test_llama3_70b_with_bias(fs, torch_cuda):
    torch = torch_cuda
    wl = synthetic.workload("llama3_70b", 256)
    hd, Wd, td, bd = _device(wl, torch)
    ell = _logits("llama3_70b", wl)                    # bias included
    ref0 = oracle_rows(ell, wl.temp, wl.seed, 0)
    for step in (0, 3):
        for B in synthetic.SHAPES["llama3_70b"]["batches"]:
            ids, mx = fs.sample(hd[:B], Wd, td[:B], wl.seed, step, bias=bd[:B])
            torch.cuda.synchronize()
            if step == 0:
                sub = sampler.Sample(ref0.ids[:B], ref0.zmax[:B], ref0.gap[:B])
                compare(ids.cpu().numpy(), mx.cpu().numpy(), sub, what=f"70B B={B} step=0 all rows")
            else:
                rows = _rows(B, 16, seed=B)
                ref = oracle_rows(ell[rows], wl.temp[rows], wl.seed, step, rows=rows)
                compare(ids.cpu().numpy(), mx.cpu().numpy(), ref, rows=rows, what=f"70B B={B} step={step}")
            if B == 256:
                # The 16 spikes of +8 carry about 16 e^8 / (16 e^8 + V) ~ 27% of the
                # softmax mass (the logit spread is the same on and off the spikes).
                spikes = wl.bias[:B] > 0
                hit = spikes[np.arange(B), ids.cpu().numpy()].mean()
                assert 0.15 < hit < 0.40, hit


@pytest.mark.parametrize("n_chunks", [8, 32])
def test_chunked_full_size(fs, torch_cuda, n_chunks):
    torch = torch_cuda
    wl = synthetic.workload("chunked", 256)
    hd, Wd, td, _ = _device(wl, torch)
    ell = _logits("chunked", wl)
    bounds = synthetic.chunk_bounds(wl.V, n_chunks)
    step = 4
    ref = oracle_rows(ell, wl.temp, wl.seed, step)     # every row of the largest batch
    for B in synthetic.SHAPES["chunked"]["batches"]:
        ids1, mx1 = fs.sample(hd[:B], Wd, td[:B], wl.seed, step)
        cm = torch.empty(B, device="cuda")
        ci = torch.empty(B, dtype=torch.int64, device="cuda")
        for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            res = fs.sample_chunked(hd[:B], Wd[lo:hi], lo, td[:B], wl.seed, step, cm, ci,
                                    i == 0, i == n_chunks - 1)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(res[0].cpu().numpy(), ids1.cpu().numpy())
        np.testing.assert_array_equal(res[1].cpu().numpy(), mx1.cpu().numpy())
        sub = sampler.Sample(ref.ids[:B], ref.zmax[:B], ref.gap[:B])
        compare(res[0].cpu().numpy(), res[1].cpu().numpy(), sub,
                what=f"chunked {n_chunks} B={B} all rows")
