"""GPU parity of Gumbel-top-k (fs_sample_topk) against the fp64 oracle
(oracle/topk.py) on identical seeded inputs.

Comparison rule (the sampler's, per list position): ids bit-exact except at
positions whose oracle score lies within BAND of a neighbour in the order
(such swaps are counted and must stay below 0.1% of the positions); scores
within MAX_TOL; padded positions (-1, -inf) exact.
"""

import numpy as np
import pytest

from _helpers import BAND, MAX_TOL, to_device
from oracle import topk as otopk
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _problem(B, V, d, seed, w_std=0.05):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * w_std).astype(np.float32))
    temps = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temps[::7] = 0.0
    if B > 3:
        temps[3] = -1.0
    return h, W, temps


def compare_topk(ids, z, ref, rows=None, what=""):
    ids = np.asarray(ids)
    z = np.asarray(z, dtype=np.float64)
    if rows is not None:
        ids, z = ids[rows], z[rows]
    assert ids.shape == ref.ids.shape, (ids.shape, ref.ids.shape)
    pad = ref.ids == -1
    np.testing.assert_array_equal(ids[pad], -1, err_msg=f"{what}: padded positions")
    assert np.all(z[pad] == -np.inf), what
    live = ~pad
    assert np.all(np.abs(z[live] - ref.z[live]) <= MAX_TOL), (what, np.abs(z[live] - ref.z[live]).max())
    mism = (ids != ref.ids) & live
    bad = mism & ~(ref.gap < BAND)
    assert not bad.any(), f"{what}: {bad.sum()} id mismatches outside the near-tie band"
    assert mism.sum() <= max(1, int(0.001 * live.sum())), f"{what}: {mism.sum()} near-tie swaps"
    return int(mism.sum())


def _run(fs, torch, h, W, temp, seed, step, k, bias=None):
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bd = None if bias is None else to_device(bias, torch)
    ids, z = fs.sample_topk(hd, Wd, td, seed, step, k, bias=bd)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), z.cpu().numpy()


@pytest.mark.parametrize("k", [1, 3, 8, 16])
@pytest.mark.parametrize("B,V,d", [(1, 50, 64), (5, 4097, 256), (37, 3001, 128), (100, 2500, 128), (130, 4097, 64)])
def test_topk_matches_oracle(fs, torch_cuda, B, V, d, k):
    h, W, temp = _problem(B, V, d, seed=B + V + k)
    ids, z = _run(fs, torch_cuda, h, W, temp, 21, 4, k)
    compare_topk(ids, z, otopk.sample_topk(h, W, temp, 21, 4, k), what=f"B={B} V={V} d={d} k={k}")
    if B > 3:
        assert np.all(ids[3] == -1)                       # invalid temperature


@pytest.mark.parametrize("B", [4, 200])
def test_topk_masks_padding_and_ties(fs, torch_cuda, B):
    """Rows 0-3 carry the special cases; B = 200 runs them through the CTA-pair
    kernel, B = 4 through the vocabulary-major one."""
    V, d, k = 300, 64, 8
    h, W, temp = _problem(B, V, d, seed=5)
    temp[:4] = [0.0, 1.0, 1.0, 0.7]
    W[40] = W[17]
    W[250] = W[17]                                        # equal logits at ids 17, 40, 250
    bias = np.zeros((B, V), np.float32)
    bias[0, [17, 40, 250]] = 30.0                         # greedy row: the three tie at the top
    bias[1, :] = -np.inf
    bias[1, [5, 299, 100]] = 0.0                          # only three choosable ids
    bias[2, :150] = -np.inf                               # first half masked
    ids, z = _run(fs, torch_cuda, h, W, temp, 3, 9, k, bias=bias)
    np.testing.assert_array_equal(ids[0, :3], [17, 40, 250])
    assert sorted(ids[1, :3]) == [5, 100, 299] and np.all(ids[1, 3:] == -1) and np.all(z[1, 3:] == -np.inf)
    assert np.all(ids[2] >= 150)
    compare_topk(ids, z, otopk.sample_topk(h, W, temp, 3, 9, k, bias=bias), what="masks")


@pytest.mark.parametrize("B,path", [(20, "AUTO"), (64, "AUTO"), (100, "AUTO"), (200, "AUTO"), (256, "AUTO"),
                                    (300, "AUTO"), (520, "AUTO"), (256, "TC_BATCH"), (100, "TC_PAIR"),
                                    (20, "TC_VOCAB")])
def test_top1_equals_the_sampler_on_the_same_kernel(fs, torch_cuda, B, path):
    """k = 1 through the top-k epilogue and the sample through the same kernel
    (vocabulary-major for B <= 64; above that the sampler's own choice, CTA
    pairs where 256-row pair tiles waste fewer than 128 rows, else
    batch-major, or the family forced with set_path) compute identical
    scores: identical ids and maxima."""
    torch = torch_cuda
    V, d = 20011, 256
    h, W, temp = _problem(B, V, d, seed=77)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    fs.set_path(getattr(fs, "FS_PATH_" + path))
    try:
        s_ids, s_max = fs.sample(hd, Wd, td, 8, 1)
        t_ids, t_z = fs.sample_topk(hd, Wd, td, 8, 1, 1)
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(t_ids[:, 0].cpu().numpy(), s_ids.cpu().numpy())
    np.testing.assert_array_equal(t_z[:, 0].cpu().numpy(), s_max.cpu().numpy())


def test_topk_deterministic_and_distinct(fs, torch_cuda):
    torch = torch_cuda
    B, V, d, k = 200, 5003, 128, 16
    h, W, temp = _problem(B, V, d, seed=9)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    a = fs.sample_topk(hd, Wd, td, 1, 2, k)
    b = fs.sample_topk(hd, Wd, td, 1, 2, k)
    fs.set_launch_overlap(False)
    try:
        c = fs.sample_topk(hd, Wd, td, 1, 2, k)
    finally:
        fs.set_launch_overlap(True)
    torch.cuda.synchronize()
    for other in (b, c):
        np.testing.assert_array_equal(a[0].cpu().numpy(), other[0].cpu().numpy())
        np.testing.assert_array_equal(a[1].cpu().numpy(), other[1].cpu().numpy())
    ids = a[0].cpu().numpy()
    for r in range(B):
        live = ids[r][ids[r] >= 0]
        assert len(set(live.tolist())) == len(live)
    assert np.all(np.diff(a[1].cpu().numpy(), axis=1)[ids[:, 1:] >= 0] <= 0)


def test_topk_invalid_arguments(fs, torch_cuda):
    torch = torch_cuda
    h, W, temp = _problem(4, 100, 64, seed=1)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    for bad_k in (0, 17):
        with pytest.raises(fs.FlashSampleError):
            fs.sample_topk(hd, Wd, td, 1, 0, bad_k)
    with pytest.raises(fs.FlashSampleError):
        hs, Ws, ts = _problem(2, 100, 32, seed=2)
        fs.sample_topk(to_device(hs, torch), to_device(Ws, torch), to_device(ts, torch), 1, 0, 4)


def test_topk_empty_vocabulary(fs, torch_cuda):
    torch = torch_cuda
    h, _, temp = _problem(3, 1, 64, seed=4)
    W = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    ids, z = fs.sample_topk(to_device(h, torch), W, to_device(temp, torch), 1, 0, 4)
    torch.cuda.synchronize()
    assert np.all(ids.cpu().numpy() == -1) and np.all(z.cpu().numpy() == -np.inf)


@pytest.mark.parametrize("B,k", [(16, 8), (100, 8), (256, 4)])
def test_topk_llama3_8b_head(fs, torch_cuda, B, k):
    torch = torch_cuda
    wl = synthetic.workload("llama3_8b", B)
    ids, z = _run(fs, torch, wl.h, wl.W, wl.temp, wl.seed, 7, k)
    rows = np.unique(np.r_[0, B - 1, np.random.default_rng(B).choice(B, size=min(B, 4), replace=False)])
    ref = otopk.sample_topk(wl.h, wl.W, wl.temp, wl.seed, 7, k, rows=rows)
    compare_topk(ids, z, ref, rows=rows, what=f"8B head B={B} k={k}")


@pytest.mark.parametrize("rows", [16, 100, 200])
def test_topk_law_on_gpu(fs, torch_cuda, rows):
    """3 x 10^5 ordered pairs (k = 2) drawn on the GPU from one repeated row
    (every (row, step) has its own noise): chi-square against the
    Plackett-Luce law of drawing without replacement from softmax(logits / T),
    computed from scipy's softmax of the oracle's logits.  rows = 16 runs the
    vocabulary-major kernel, 100 the batch-major one, 200 the CTA-pair one."""
    from scipy import special, stats
    from oracle import sampler
    torch = torch_cuda
    V, d, k, T = 6, 64, 2, 0.9
    rng = np.random.default_rng(8)
    h1 = synthetic.bf16_bits(rng.standard_normal((1, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.12).astype(np.float32))
    steps = 300_000 // rows
    hd = to_device(np.repeat(h1, rows, axis=0), torch)
    Wd = to_device(W, torch)
    td = torch.full((rows,), T, device="cuda")
    ids = torch.empty((steps, rows, k), dtype=torch.int64, device="cuda")
    z = torch.empty((steps, rows, k), dtype=torch.float32, device="cuda")
    for s_ in range(steps):
        fs.sample_topk(hd, Wd, td, 99, s_, k, out=(ids[s_], z[s_]))
    got = ids.cpu().numpy().reshape(-1, k)
    assert np.all(got[:, 0] != got[:, 1]) and np.all(got >= 0)
    counts = np.bincount(got[:, 0] * V + got[:, 1], minlength=V * V)
    p = special.softmax(sampler.logits(h1, W)[0] / T)
    probs = np.zeros(V * V)
    for i in range(V):
        for j in range(V):
            if i != j:
                probs[i * V + j] = p[i] * p[j] / (1.0 - p[i])
    keep = probs > 0
    assert stats.chisquare(counts[keep], probs[keep] * counts.sum()).pvalue > 0.01


@pytest.mark.parametrize("B", [24, 256])
def test_topk_captured_in_cuda_graph(fs, torch_cuda, B):
    """After one eager call of the same size, a top-k call can be captured
    into a CUDA graph; replays with a changed step buffer are not possible
    (the step is baked in), so the replay must reproduce the eager result."""
    torch = torch_cuda
    V, d, k = 5003, 128, 8
    h, W, temp = _problem(B, V, d, seed=31)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    stream = torch.cuda.Stream()
    ids = torch.empty((B, k), dtype=torch.int64, device="cuda")
    z = torch.empty((B, k), dtype=torch.float32, device="cuda")
    fs.workspace_reserve(B, V, stream=stream)
    with torch.cuda.stream(stream):
        fs.sample_topk(hd, Wd, td, 4, 4, k, out=(ids, z), stream=stream)
    torch.cuda.synchronize()
    want = (ids.cpu().numpy().copy(), z.cpu().numpy().copy())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fs.sample_topk(hd, Wd, td, 4, 4, k, out=(ids, z), stream=stream)
    ids.fill_(-5)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), want[0])
    np.testing.assert_array_equal(z.cpu().numpy(), want[1])
    compare_topk(want[0], want[1], otopk.sample_topk(h, W, temp, 4, 4, k), what="graph")
    del graph


def test_topk_llama3_70b_head_with_bias(fs, torch_cuda):
    """d 8192 and the dense spike bias (16 ids per row at +8): the top 16
    carry the spikes; sampled rows against the oracle."""
    torch = torch_cuda
    B, k = 8, 16
    wl = synthetic.workload("llama3_70b", B)
    hd, Wd, td = to_device(wl.h, torch), to_device(wl.W, torch), to_device(wl.temp, torch)
    bd = to_device(wl.bias, torch)
    ids, z = fs.sample_topk(hd, Wd, td, wl.seed, 3, k, bias=bd)
    torch.cuda.synchronize()
    rows = np.array([0, 3, 7])
    ref = otopk.sample_topk(wl.h, wl.W, wl.temp, wl.seed, 3, k, bias=wl.bias, rows=rows)
    compare_topk(ids.cpu().numpy(), z.cpu().numpy(), ref, rows=rows, what="70B head, bias")
