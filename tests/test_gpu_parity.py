"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
identical seeded inputs.

Small cases are compared element by element over every row; the full-size
workloads run in the launch configuration the benchmark times and are
compared on sampled rows (the oracle computes each row over the whole
vocabulary).  Comparison rule: tests/_helpers.py.
"""

import os

import numpy as np
import pytest

from _helpers import compare, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _run(fs, torch, h, W, temp, seed, step, bias=None):
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bd = None if bias is None else to_device(bias, torch)
    ids, mx = fs.sample(hd, Wd, td, seed, step, bias=bd)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), mx.cpu().numpy()


def _problem(B, V, d, seed, w_std=0.05, temps=None):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * w_std).astype(np.float32))
    if temps is None:
        temps = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
        temps[::7] = 0.0
    return h, W, np.asarray(temps, np.float32)


@pytest.fixture(params=["simt", "tc_vocab", "tc_batch", "tc_pair"])
def path(request, fs):
    """Run the test once per kernel family (forced through fs_set_path)."""
    code = {"simt": fs.FS_PATH_SIMT, "tc_vocab": fs.FS_PATH_TC_VOCAB,
            "tc_batch": fs.FS_PATH_TC_BATCH, "tc_pair": fs.FS_PATH_TC_PAIR}[request.param]
    fs.set_path(code)
    yield request.param
    fs.set_path(fs.FS_PATH_AUTO)


# ------------------------------------------------------------------ noise
@pytest.mark.parametrize("row0,v0,step", [(0, 0, 0), (5, 3, 99), (1000, 151900, (3 << 32) + 17)])
def test_noise_words_bit_exact(fs, torch_cuda, row0, v0, step):
    n_rows, n_vocab = 33, 37
    words, g = fs.debug_noise(1234, step, row0, n_rows, v0, n_vocab)
    torch_cuda.cuda.synchronize()
    ref = sampler.philox_words(1234, step, np.arange(row0, row0 + n_rows), np.arange(v0, v0 + n_vocab))
    np.testing.assert_array_equal(words.cpu().numpy().view(np.uint32), ref)


def test_gumbel_values_within_bound(fs, torch_cuda):
    # 64 rows x 8192 ids cover ~5e5 draws, including u close to 0 and 1.
    words, g = fs.debug_noise(77, 3, 0, 64, 0, 8192)
    torch_cuda.cuda.synchronize()
    w = words.cpu().numpy().view(np.uint32)
    ref = sampler.gumbel_from_uniform(sampler.uniform_from_word(w))
    err = np.abs(g.cpu().numpy().astype(np.float64) - ref)
    assert err.max() < 1e-5, err.max()
    assert np.isfinite(g.cpu().numpy()).all()


# ------------------------------------------------------------------ small cases
def test_tiny_workload(fs, torch_cuda):
    wl = synthetic.tiny()
    ids, mx = _run(fs, torch_cuda, wl.h, wl.W, wl.temp, wl.seed, 0)
    ref = sampler.sample(wl.h, wl.W, wl.temp, wl.seed, 0)
    compare(ids, mx, ref, what="tiny")
    assert ids[0] == np.argmax(sampler.logits(wl.h, wl.W)[0])   # T = 0 row is greedy


@pytest.mark.parametrize("B", [1, 3, 8, 17, 100, 256])
@pytest.mark.parametrize("V,d", [(1, 64), (127, 64), (4097, 256), (1000, 8), (3000, 200)])
def test_ragged_shapes(fs, torch_cuda, path, B, V, d):
    h, W, temp = _problem(B, V, d, seed=B * 7 + V)
    for step in (0, 5):
        ids, mx = _run(fs, torch_cuda, h, W, temp, 42, step)
        compare(ids, mx, sampler.sample(h, W, temp, 42, step), what=f"B{B} V{V} d{d}")


def test_many_steps_many_rows(fs, torch_cuda, path):
    h, W, temp = _problem(64, 5000, 128, seed=3)
    for step in range(0, 100, 9):
        ids, mx = _run(fs, torch_cuda, h, W, temp, 1234, step)
        compare(ids, mx, sampler.sample(h, W, temp, 1234, step), what=f"step {step}")


def test_bias_per_row_and_shared(fs, torch_cuda, path):
    B, V, d = 9, 3001, 64
    h, W, temp = _problem(B, V, d, seed=11)
    rng = np.random.default_rng(11)
    bias = np.zeros((B, V), np.float32)
    for b in range(B):
        bias[b, rng.choice(V, 16, replace=False)] = 8.0
    ids, mx = _run(fs, torch_cuda, h, W, temp, 9, 1, bias=bias)
    compare(ids, mx, sampler.sample(h, W, temp, 9, 1, bias=bias), what="row bias")
    shared = rng.standard_normal(V).astype(np.float32)
    ids, mx = _run(fs, torch_cuda, h, W, temp, 9, 2, bias=shared)
    compare(ids, mx, sampler.sample(h, W, temp, 9, 2, bias=shared), what="shared bias")


def test_degenerate_rows(fs, torch_cuda, path):
    B, V, d = 6, 300, 32
    h, W, _ = _problem(B, V, d, seed=12)
    W = W.copy()
    W[10] = 0x7FC0                                    # NaN logits never win
    temp = np.array([-1.0, np.nan, 0.0, 1.0, np.inf, 0.7], np.float32)
    bias = np.zeros((B, V), np.float32)
    bias[5, :] = -np.inf                              # nothing can win
    ids, mx = _run(fs, torch_cuda, h, W, temp, 3, 4, bias=bias)
    ref = sampler.sample(h, W, temp, 3, 4, bias=bias)
    compare(ids, mx, ref, what="degenerate")
    assert ids[0] == -1 and ids[1] == -1 and ids[5] == -1
    assert 10 not in ids


def test_masked_vocabulary(fs, torch_cuda, path):
    """Constrained decoding through the bias: -inf outside an allowed set
    (a few ids, or one), NaN entries (never chosen), and +inf at two ids (the
    smaller wins the tie at +inf, in every kernel family and across CTAs),
    one-shot and chunked, against the oracle."""
    torch = torch_cuda
    B, V, d = 8, 5003, 64
    h, W, temp = _problem(B, V, d, seed=33)
    temp[:] = 1.0
    temp[3] = 0.0                                      # a greedy row under a mask
    rng = np.random.default_rng(34)
    bias = np.full((B, V), -np.inf, np.float32)
    allowed = {}
    for b in (0, 3, 4):
        allowed[b] = np.sort(rng.choice(V, size=7, replace=False))
        bias[b, allowed[b]] = 0.0
    allowed[1] = np.array([4321])
    bias[1, 4321] = 0.0                                # a single allowed id
    bias[2, :] = 0.0
    bias[2, [4000, 77]] = np.inf                       # +inf twice: the smaller id wins
    bias[5, :] = 0.0
    nan_ids = rng.choice(V, size=500, replace=False)
    bias[5, nan_ids] = np.nan                          # NaN scores never win
    bias[6, :] = 0.0
    bias[7, :] = -np.inf                               # nothing allowed: no sample
    ids, mx = _run(fs, torch, h, W, temp, 9, 2, bias=bias)
    ref = sampler.sample(h, W, temp, 9, 2, bias=bias)
    finite = [0, 1, 3, 4, 5, 6, 7]
    compare(ids[finite], mx[finite], sampler.Sample(ref.ids[finite], ref.zmax[finite], ref.gap[finite]),
            what=f"masked {path}")
    for b, ok in allowed.items():
        assert ids[b] in ok, (b, ids[b])
    assert ids[1] == 4321
    assert ids[2] == 77 and ref.ids[2] == 77 and mx[2] == np.inf
    assert ids[5] not in set(nan_ids.tolist())
    assert ids[7] == -1 and mx[7] == -np.inf
    # the same masks through the chunked variant (chunk bounds cut the allowed sets)
    hd, Wd, td, bd = to_device(h, torch), to_device(W, torch), to_device(temp, torch), to_device(bias, torch)
    bounds = synthetic.chunk_bounds(V, 5)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, 9, 2, cm, ci, i == 0, i == 4, bias_chunk=bd[:, lo:hi])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(res[0].cpu().numpy(), ids)
    np.testing.assert_array_equal(res[1].cpu().numpy(), mx)


def test_extreme_temperatures(fs, torch_cuda, path):
    """Temperatures from 1e-6 (scores ~1e6: the sample is the greedy argmax
    up to fp32 rounding of the scaled logits) to 1e30 (1/T ~ 1e-30: the
    noise alone decides), and subnormal-free ends in between, against the
    oracle."""
    B, V, d = 9, 4099, 64
    h, W, _ = _problem(B, V, d, seed=44)
    temp = np.array([1e-6, 1e-3, 0.05, 1.0, 20.0, 1e3, 1e6, 1e30, 3e-7], np.float32)
    # the parity tolerances hold on the logits: at 1/T > 1 they scale with 1/T
    scale = np.maximum(1.0, 1.0 / temp.astype(np.float64))
    greedy = np.argmax(sampler.logits(h, W), axis=1)
    for step in (0, 3):
        ids, mx = _run(fs, torch_cuda, h, W, temp, 17, step)
        ref = sampler.sample(h, W, temp, 17, step)
        near = ref.gap < 2e-3 * scale
        assert np.all((ids == ref.ids) | near), (ids, ref.ids, ref.gap)
        same = ids == ref.ids
        assert np.all(np.abs(mx[same] - ref.zmax[same]) <= 2e-3 * scale[same]), (mx, ref.zmax)
        assert ids[0] == greedy[0] and ids[8] == greedy[8]


def test_empty_batch_and_empty_vocab(fs, torch_cuda, path):
    torch = torch_cuda
    h = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((10, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.ones(0, device="cuda")
    ids, mx = fs.sample(h, W, t, 0, 0)
    assert ids.numel() == 0
    h = torch.zeros((3, 64), dtype=torch.bfloat16, device="cuda")
    W0 = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    ids, mx = fs.sample(h, W0, torch.ones(3, device="cuda"), 0, 0)
    torch.cuda.synchronize()
    assert ids.tolist() == [-1, -1, -1]
    assert mx.tolist() == [-np.inf] * 3


def test_ties_go_to_smaller_id(fs, torch_cuda, path):
    rng = np.random.default_rng(13)
    h = synthetic.bf16_bits(rng.standard_normal((4, 64)).astype(np.float32))
    row = synthetic.bf16_bits(rng.standard_normal((1, 64)).astype(np.float32))
    W = np.repeat(row, 2000, axis=0)                  # every logit identical
    ids, _ = _run(fs, torch_cuda, h, W, np.zeros(4, np.float32), 1, 0)
    np.testing.assert_array_equal(ids, 0)


def test_invalid_arguments_are_rejected(fs, torch_cuda):
    torch = torch_cuda
    h = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((10, 64), dtype=torch.bfloat16, device="cuda")
    t = torch.ones(2, device="cuda")
    with pytest.raises(fs.FlashSampleError, match="UNSUPPORTED"):
        fs.sample(h[:, 1:63].contiguous(), W[:, 1:63].contiguous(), t, 0, 0)     # d = 62
    lib = fs.library()
    import ctypes
    ids = torch.empty(2, dtype=torch.int64, device="cuda")
    mx = torch.empty(2, dtype=torch.float32, device="cuda")
    host = np.zeros((2, 64), np.uint16)
    # a host pointer where device memory is required
    st = lib.fs_sample(ctypes.c_void_p(host.ctypes.data), ctypes.c_void_p(W.data_ptr()), 2, 64, 10,
                       ctypes.c_void_p(t.data_ptr()), 0, 0, ctypes.c_void_p(ids.data_ptr()),
                       ctypes.c_void_p(mx.data_ptr()), None)
    assert st == 1 and b"not device memory" in lib.fs_last_error()
    # misaligned W
    st = lib.fs_sample(ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(W.data_ptr() + 2), 2, 64, 9,
                       ctypes.c_void_p(t.data_ptr()), 0, 0, ctypes.c_void_p(ids.data_ptr()),
                       ctypes.c_void_p(mx.data_ptr()), None)
    assert st == 2


def test_deterministic_and_step_dependent(fs, torch_cuda, path):
    h, W, temp = _problem(32, 4096, 128, seed=14, temps=np.ones(32))
    a = _run(fs, torch_cuda, h, W, temp, 5, 0)
    b = _run(fs, torch_cuda, h, W, temp, 5, 0)
    c = _run(fs, torch_cuda, h, W, temp, 5, 1)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert (a[0] != c[0]).mean() > 0.5


def test_sampling_law_on_gpu(fs, torch_cuda, path):
    """10^6 draws from one row (250 identical rows x 4000 steps; every
    (row, step) has its own counters): chi-square against softmax(logits / T)
    from the oracle's logits."""
    from scipy import special, stats
    V, d, rows, steps = 64, 64, 250, 4000
    h1, W, _ = _problem(1, V, d, seed=15, w_std=0.15)
    torch = torch_cuda
    hd = to_device(np.repeat(h1, rows, axis=0), torch)
    Wd = to_device(W, torch)
    T = 0.8
    td = torch.full((rows,), T, device="cuda")
    ids = torch.empty((steps, rows), dtype=torch.int64, device="cuda")
    mx = torch.empty((steps, rows), dtype=torch.float32, device="cuda")
    for s_ in range(steps):
        fs.sample(hd, Wd, td, 2024, s_, out=(ids[s_], mx[s_]))
    counts = np.bincount(ids.cpu().numpy().ravel(), minlength=V)
    n = rows * steps
    probs = special.softmax(sampler.logits(h1, W)[0] / T)
    assert stats.chisquare(counts, probs * n).pvalue > 0.01


# ------------------------------------------------------------------ chunked
@pytest.mark.parametrize("bounds", [[0, 1, 130, 131, 2999, 4097], None])
def test_chunked_equals_one_shot_bitwise(fs, torch_cuda, path, bounds):
    torch = torch_cuda
    B, V, d = 33, 4097, 256
    h, W, temp = _problem(B, V, d, seed=16)
    bounds = bounds or synthetic.chunk_bounds(V, 8)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    ids1, mx1 = fs.sample(hd, Wd, td, 7, 3)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    res = None
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, 7, 3, cm, ci, i == 0, i == len(bounds) - 2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(res[0].cpu().numpy(), ids1.cpu().numpy())
    np.testing.assert_array_equal(res[1].cpu().numpy(), mx1.cpu().numpy())
    compare(res[0].cpu().numpy(), res[1].cpu().numpy(), sampler.sample(h, W, temp, 7, 3), what="chunked")


# ------------------------------------------------------------------ host entry
def test_sample_host_matches_device(fs, torch_cuda, path):
    torch = torch_cuda
    h, W, temp = _problem(16, 3000, 128, seed=17)
    Wd = to_device(W, torch)
    ids_h, mx_h = fs.sample_host(h, Wd, temp, 11, 4)
    ids_d, mx_d = _run(fs, torch, h, W, temp, 11, 4)
    np.testing.assert_array_equal(ids_h, ids_d)
    np.testing.assert_array_equal(mx_h, mx_d)


def test_paths_agree_on_llama3_8b_head(fs, torch_cuda):
    """Both kernel families on the full-size head: ids equal outside near ties,
    maxima within the tolerance (they sum the logits in different orders)."""
    torch = torch_cuda
    wl = synthetic.workload("llama3_8b", 64)
    hd, Wd, td = to_device(wl.h, torch), to_device(wl.W, torch), to_device(wl.temp, torch)
    out = {}
    for name, code in (("simt", fs.FS_PATH_SIMT), ("tc", fs.FS_PATH_TC_VOCAB), ("tcb", fs.FS_PATH_TC_BATCH),
                       ("tcp", fs.FS_PATH_TC_PAIR)):
        fs.set_path(code)
        ids, mx = fs.sample(hd, Wd, td, wl.seed, 11)
        torch.cuda.synchronize()
        out[name] = (ids.cpu().numpy(), mx.cpu().numpy())
    fs.set_path(fs.FS_PATH_AUTO)
    for other in ("tc", "tcb", "tcp"):
        diff = out["simt"][0] != out[other][0]
        assert diff.sum() <= 1
        assert np.abs(out["simt"][1] - out[other][1])[~diff].max() < 1e-3


def test_device_error_word_is_clear(fs, torch_cuda):
    assert fs.device_error() == 0


# ------------------------------------------------------------------ unfused comparison path
@pytest.mark.parametrize("B,V,d", [(4, 4096, 256), (37, 4097, 512), (300, 3001, 256)])
def test_unfused_logits_and_ids(fs, torch_cuda, B, V, d):
    """The unfused pipeline's HBM logits against the oracle's fp64 logits
    (|delta| <= 2e-3), and its ids / maxima against the oracle (same rule as
    the fused path) and the fused path."""
    torch = torch_cuda
    h, W, temp = _problem(B, V, d, seed=B + V)
    rng = np.random.default_rng(B)
    bias = np.zeros((B, V), np.float32)
    bias[np.arange(B)[:, None], rng.integers(0, V, size=(B, 4))] = 3.0
    hd, Wd, td, bd = (to_device(h, torch), to_device(W, torch), to_device(temp, torch),
                      to_device(bias, torch))
    logits = torch.empty((B, V), dtype=torch.float32, device="cuda")
    ids, mx = fs.sample_unfused(hd, Wd, td, 99, 5, bias=bd, logits_out=logits)
    fids, fmx = fs.sample(hd, Wd, td, 99, 5, bias=bd)
    torch.cuda.synchronize()
    ell = sampler.logits(h, W, bias)
    assert np.abs(logits.cpu().numpy().astype(np.float64) - ell).max() <= 2e-3
    ref = sampler.sample(h, W, temp, 99, 5, bias=bias)
    compare(ids.cpu().numpy(), mx.cpu().numpy(), ref, what="unfused")
    compare(fids.cpu().numpy(), fmx.cpu().numpy(), ref, what="fused")


def test_unfused_on_llama3_8b_head(fs, torch_cuda):
    torch = torch_cuda
    wl = synthetic.workload("llama3_8b", 16)
    hd, Wd, td = to_device(wl.h, torch), to_device(wl.W, torch), to_device(wl.temp, torch)
    logits = torch.empty((16, wl.V), dtype=torch.float32, device="cuda")
    ids, mx = fs.sample_unfused(hd, Wd, td, wl.seed, 7, logits_out=logits)
    torch.cuda.synchronize()
    rows = np.array([0, 5, 15])
    ell = sampler.logits(wl.h[rows], wl.W)
    assert np.abs(logits.cpu().numpy()[rows].astype(np.float64) - ell).max() <= 2e-3
    ref = sampler.sample(wl.h, wl.W, wl.temp, wl.seed, 7)
    compare(ids.cpu().numpy(), mx.cpu().numpy(), ref, what="unfused 8B")


def test_bounded_wait_times_out_and_reports(fs, torch_cuda):
    """A wait that nobody satisfies gives up after its limit, flags the device
    error word, and leaves the context usable."""
    torch = torch_cuda
    assert fs.device_error() == 0
    fs.debug_wait_timeout(20_000_000)                 # 20 ms
    torch.cuda.synchronize()
    assert fs.device_error() == 1
    assert fs.device_error() == 0                     # read clears it
    wl = synthetic.tiny()
    ids, mx = _run(fs, torch, wl.h, wl.W, wl.temp, wl.seed, 0)
    compare(ids, mx, sampler.sample(wl.h, wl.W, wl.temp, wl.seed, 0), what="after timeout")


def test_back_to_back_calls_of_different_batch_sizes(fs, torch_cuda, path):
    """The in-kernel finish leaves its ticket and keys at zero: calls with
    shrinking and growing batches on one stream stay exact."""
    torch = torch_cuda
    h, W, temp = _problem(300, 2000, 128, seed=31)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    for B in (300, 7, 64, 1, 300):
        ids, mx = fs.sample(hd[:B], Wd, td[:B], 3, B)
        torch.cuda.synchronize()
        compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h[:B], W, temp[:B], 3, B),
                what=f"B={B}")


@pytest.mark.parametrize("B", [1, 32, 64, 128, 256])
def test_chunked_sequence_captured_in_cuda_graph(fs, torch_cuda, B):
    """After fs_workspace_reserve, a whole chunked decode step (8 launches)
    can be captured into a CUDA graph; every replay reproduces the one-shot
    sample bit for bit.  The captured step follows an eager one, so at B = 64
    and 128 it runs on the CTA-pair kernel (25 pair tiles per chunk)."""
    torch = torch_cuda
    V, d, n = 50021, 256, 8
    h, W, temp = _problem(B, V, d, seed=40 + B)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bounds = synthetic.chunk_bounds(V, n)
    stream = torch.cuda.Stream()
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    ids = torch.empty(B, dtype=torch.int64, device="cuda")
    mx = torch.empty(B, dtype=torch.float32, device="cuda")
    fs.workspace_reserve(B, V, stream=stream)

    def step():
        for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            fs.sample_chunked(hd, Wd[lo:hi], lo, td, 5, 9, cm, ci, i == 0, i == n - 1,
                              out=(ids, mx), stream=stream)

    with torch.cuda.stream(stream):
        step()                                       # warm: kernels loaded, attributes set
    torch.cuda.synchronize()
    ref_ids, ref_mx = fs.sample(hd, Wd, td, 5, 9)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(2):
        ids.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy())
        np.testing.assert_array_equal(mx.cpu().numpy(), ref_mx.cpu().numpy())


def test_many_small_chunks_overlapping_launches(fs, torch_cuda, path):
    """97 chunks of a step launched back to back: from the second chunk on,
    each chunk kernel may start while the previous one runs (programmatic
    dependent launch) and only waits before merging the carry; the result
    must still equal the one-shot sample bit for bit, step after step."""
    torch = torch_cuda
    B, V, d, n = 40, 30011, 128, 97
    h, W, temp = _problem(B, V, d, seed=77)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bounds = synthetic.chunk_bounds(V, n)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    for step in (0, 1, 2):
        ref_ids, ref_mx = fs.sample(hd, Wd, td, 3, step)
        for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, 3, step, cm, ci, i == 0, i == n - 1)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(res[0].cpu().numpy(), ref_ids.cpu().numpy())
        np.testing.assert_array_equal(res[1].cpu().numpy(), ref_mx.cpu().numpy())


@pytest.mark.parametrize("B", [40, 64, 128])
@pytest.mark.parametrize("n", [8, 32])
def test_chunk_family_rule_keeps_one_shot_samples(fs, torch_cuda, B, n):
    """Under the automatic rule, chunk calls at 32 < B <= 128 run the batch-
    major kernel, or the CTA-pair kernel once the previous step's chunk count
    shows that the step fits one wave of pairs (here from the second 8-chunk
    step on: 25 pair tiles per chunk); the one-shot call at B <= 64 runs the
    vocabulary-major kernel.  Every step must equal its one-shot sample bit
    for bit, and the oracle within the comparison rule."""
    torch = torch_cuda
    V, d = 50000, 256
    h, W, temp = _problem(B, V, d, seed=97 + B)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bounds = synthetic.chunk_bounds(V, n)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    stream = torch.cuda.Stream()      # a stream with no chunked history
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for step in (4, 5, 6):
            ref_ids, ref_mx = fs.sample(hd, Wd, td, 13, step)
            for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
                res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, 13, step, cm, ci, i == 0, i == n - 1)
            stream.synchronize()
            np.testing.assert_array_equal(res[0].cpu().numpy(), ref_ids.cpu().numpy())
            np.testing.assert_array_equal(res[1].cpu().numpy(), ref_mx.cpu().numpy())
    compare(res[0].cpu().numpy(), res[1].cpu().numpy(), sampler.sample(h, W, temp, 13, 6), what="chunked")


@pytest.mark.parametrize("B", [1, 32, 64, 256])
def test_one_call_chunked_step(fs, torch_cuda, B):
    """fs_sample_chunked_step issues a whole step's chunk calls from C: on
    ragged bounds with an empty chunk, with a per-row bias, it equals the
    one-shot sample and the per-chunk call sequence bit for bit, over steps
    in a row (the later ones with the chunk count of the previous step)."""
    torch = torch_cuda
    V, d = 30011, 256
    h, W, temp = _problem(B, V, d, seed=131 + B)
    bias = np.zeros((B, V), np.float32)
    bias[:, ::97] = 0.5
    hd, Wd, td, bd = to_device(h, torch), to_device(W, torch), to_device(temp, torch), to_device(bias, torch)
    bounds = np.array([0, 7001, 7001, 15000, 15013, 26000, V], np.int64)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    for step in (2, 3):
        ref_ids, ref_mx = fs.sample(hd, Wd, td, 17, step, bias=bd)
        ids, mx = fs.sample_chunked_step(hd, Wd, bounds, td, 17, step, cm, ci, bias=bd)
        n = len(bounds) - 1
        for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            res = fs.sample_chunked(hd, Wd[lo:hi], int(lo), td, 17, step, cm, ci, i == 0, i == n - 1,
                                    bias_chunk=bd[:, lo:hi])
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy())
        np.testing.assert_array_equal(mx.cpu().numpy(), ref_mx.cpu().numpy())
        np.testing.assert_array_equal(res[0].cpu().numpy(), ref_ids.cpu().numpy())
        np.testing.assert_array_equal(res[1].cpu().numpy(), ref_mx.cpu().numpy())
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 17, 3, bias=bias), what="chunked step")


@pytest.mark.parametrize("B", [1, 48, 200])
def test_one_call_chunked_step_with_many_chunks(fs, torch_cuda, B):
    """A one-call step of 70 uneven chunks (more than the workspace's 32 key
    sets, so some chunk calls launch without overlap) equals the one-shot
    sample bit for bit, twice in a row on a fresh stream."""
    torch = torch_cuda
    V, d = 12007, 128
    h, W, temp = _problem(B, V, d, seed=151 + B)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    g = np.random.default_rng(B)
    bounds = np.unique(np.r_[0, np.sort(g.integers(0, V, size=69)), V]).astype(np.int64)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for step in (8, 9):
            ref_ids, ref_mx = fs.sample(hd, Wd, td, 23, step)
            ids, mx = fs.sample_chunked_step(hd, Wd, bounds, td, 23, step, cm, ci)
            stream.synchronize()
            np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy())
            np.testing.assert_array_equal(mx.cpu().numpy(), ref_mx.cpu().numpy())
    assert len(bounds) - 1 > 32


@pytest.mark.parametrize("B,d", [(0, 128), (5, 40), (70, 40), (64, 256)])
def test_one_call_chunked_step_edge_cases(fs, torch_cuda, B, d):
    """fs_sample_chunked_step on the edges: B = 0 (a no-op), a model width
    below 64 (every batch size on the CUDA-core family), bounds whose chunks
    are all empty but one, greedy rows and a shared [V] bias.  Each result
    equals the one-shot sample bit for bit (and the oracle's rule)."""
    torch = torch_cuda
    V = 3001
    h, W, temp = _problem(max(B, 1), V, d, seed=171 + B + d)
    h, temp = h[:B], temp[:B]
    if B:
        temp[1::3] = 0.0
    shared = (np.random.default_rng(d).standard_normal(V) * 0.5).astype(np.float32)
    hd, Wd, td, sd = to_device(h, torch), to_device(W, torch), to_device(temp, torch), to_device(shared, torch)
    cm = torch.empty(max(B, 1), device="cuda")[:B]
    ci = torch.empty(max(B, 1), dtype=torch.int64, device="cuda")[:B]
    for bounds in ([0, 0, 0, V, V], [0, 1000, 1000, 2999, V]):
        b = np.asarray(bounds, np.int64)
        ids, mx = fs.sample_chunked_step(hd, Wd, b, td, 31, 4, cm, ci, bias=sd)
        ref_ids, ref_mx = fs.sample(hd, Wd, td, 31, 4, bias=sd)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), ref_ids.cpu().numpy())
        np.testing.assert_array_equal(mx.cpu().numpy(), ref_mx.cpu().numpy())
    if B:
        bias = np.broadcast_to(shared, (B, V))
        compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 31, 4, bias=bias),
                what=f"chunked step edges B={B} d={d}")


def test_chunked_step_interleaved_with_one_shot_calls(fs, torch_cuda, path):
    """One-shot calls of another batch size, and a Gumbel-top-k call, enqueued
    on the same stream between the chunk calls of a step: they finish through
    the stream's first key set while earlier chunks may still be running
    (programmatic launches), and the chunked step must still equal its
    one-shot sample bit for bit, and the interleaved calls their own."""
    torch = torch_cuda
    B, V, d, n = 24, 20011, 128, 6
    h, W, temp = _problem(B, V, d, seed=91)
    h2, _, temp2 = _problem(7, V, d, seed=92)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    h2d, t2d = to_device(h2, torch), to_device(temp2, torch)
    bounds = synthetic.chunk_bounds(V, n)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    ref_ids, ref_mx = fs.sample(hd, Wd, td, 5, 2)
    ref2_ids, ref2_mx = fs.sample(h2d, Wd, t2d, 6, 9)
    ref_k = fs.sample_topk(h2d, Wd, t2d, 6, 9, 4)
    torch.cuda.synchronize()
    between = []
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, 5, 2, cm, ci, i == 0, i == n - 1)
        if i == 1:
            between.append(fs.sample(h2d, Wd, t2d, 6, 9))
        if i == 3:
            between.append(fs.sample_topk(h2d, Wd, t2d, 6, 9, 4))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(res[0].cpu().numpy(), ref_ids.cpu().numpy())
    np.testing.assert_array_equal(res[1].cpu().numpy(), ref_mx.cpu().numpy())
    np.testing.assert_array_equal(between[0][0].cpu().numpy(), ref2_ids.cpu().numpy())
    np.testing.assert_array_equal(between[0][1].cpu().numpy(), ref2_mx.cpu().numpy())
    np.testing.assert_array_equal(between[1][0].cpu().numpy(), ref_k[0].cpu().numpy())
    np.testing.assert_array_equal(between[1][1].cpu().numpy(), ref_k[1].cpu().numpy())


def test_chunked_steps_on_two_streams_at_once(fs, torch_cuda, path):
    """Two chunked steps enqueued alternately on two unordered streams: each
    stream finishes through its own workspace (key sets, tickets), so the
    kernels of the two steps may overlap freely and both results stay equal
    to their one-shot samples bit for bit."""
    torch = torch_cuda
    V, d, n = 16411, 128, 5
    ha, W, ta = _problem(33, V, d, seed=101)
    hb, _, tb = _problem(200, V, d, seed=102)
    Wd = to_device(W, torch)
    args = [(to_device(ha, torch), to_device(ta, torch), 7), (to_device(hb, torch), to_device(tb, torch), 8)]
    refs = [fs.sample(h_, Wd, t_, 4, s_) for h_, t_, s_ in args]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    carries = [(torch.empty(h_.shape[0], device="cuda"), torch.empty(h_.shape[0], dtype=torch.int64, device="cuda"))
               for h_, _, _ in args]
    for st, (h_, _, _) in zip(streams, args):
        fs.workspace_reserve(h_.shape[0], V, stream=st)
    torch.cuda.synchronize()
    bounds = synthetic.chunk_bounds(V, n)
    outs = [None, None]
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        for k, ((h_, t_, s_), st, (cm, ci)) in enumerate(zip(args, streams, carries)):
            with torch.cuda.stream(st):
                outs[k] = fs.sample_chunked(h_, Wd[lo:hi], lo, t_, 4, s_, cm, ci, i == 0, i == n - 1, stream=st)
    torch.cuda.synchronize()
    for (ids, mx), (rid, rmx) in zip(outs, refs):
        np.testing.assert_array_equal(ids.cpu().numpy(), rid.cpu().numpy())
        np.testing.assert_array_equal(mx.cpu().numpy(), rmx.cpu().numpy())


@pytest.mark.parametrize("forced", ["tc_batch", "tc_pair", "auto"])
def test_batch_larger_than_one_launch(fs, torch_cuda, forced):
    """B = 20000 exceeds what one batch-major launch covers (SMs x 128 rows),
    so the call is split into consecutive launches that share the finish
    ticket; every row must still match the oracle."""
    torch = torch_cuda
    B, V, d = 20000, 300, 64
    h, W, temp = _problem(B, V, d, seed=91)
    code = {"tc_batch": fs.FS_PATH_TC_BATCH, "tc_pair": fs.FS_PATH_TC_PAIR, "auto": fs.FS_PATH_AUTO}[forced]
    fs.set_path(code)
    try:
        ids, mx = _run(fs, torch, h, W, temp, 8, 2)
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    compare(ids, mx, sampler.sample(h, W, temp, 8, 2), what=f"B=20000 {forced}")


@pytest.mark.parametrize("forced", ["tc_batch", "tc_pair"])
def test_chunked_batch_larger_than_one_launch(fs, torch_cuda, forced):
    """A chunked step whose batch needs several launches per chunk (the
    batch-major kernel covers SMs x 128 rows per launch, the lean CTA-pair
    instantiation of chunks two pairs per SM pair x 256): the launches of one
    chunk share its ticket, consecutive chunks overlap, and the result must
    still equal the one-shot sample bit for bit and match the oracle."""
    torch = torch_cuda
    B, V, d = 40000, 1000, 64
    h, W, temp = _problem(B, V, d, seed=93)
    code = {"tc_batch": fs.FS_PATH_TC_BATCH, "tc_pair": fs.FS_PATH_TC_PAIR}[forced]
    fs.set_path(code)
    try:
        hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
        ids1, mx1 = fs.sample(hd, Wd, td, 8, 3)
        cm = torch.empty(B, device="cuda")
        ci = torch.empty(B, dtype=torch.int64, device="cuda")
        bounds = [0, 333, 700, V]
        for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, 8, 3, cm, ci, i == 0, i == len(bounds) - 2)
        torch.cuda.synchronize()
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    np.testing.assert_array_equal(res[0].cpu().numpy(), ids1.cpu().numpy())
    np.testing.assert_array_equal(res[1].cpu().numpy(), mx1.cpu().numpy())
    compare(res[0].cpu().numpy(), res[1].cpu().numpy(), sampler.sample(h, W, temp, 8, 3),
            what=f"chunked B={B} {forced}")


def test_epilogue_warp_splits_agree(fs, torch_cuda):
    """The batch-major kernel scans a tile with 16 epilogue warps when one
    batch tile covers the batch (B <= 128) and with 8 above; the CTA-pair
    kernel samples with 16 and keeps its top-k lists with 8.  How the columns
    are split between warps must not change any score or decision: the same
    rows agree bit for bit across the splits."""
    torch = torch_cuda
    V, d = 7001, 256
    h, W, temp = _problem(300, V, d, seed=93)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    fs.set_path(fs.FS_PATH_TC_BATCH)
    try:
        ids16, mx16 = fs.sample(hd[:128], Wd, td[:128], 6, 11)      # one batch tile: 16 warps
        ids8, mx8 = fs.sample(hd, Wd, td, 6, 11)                    # three batch tiles: 8 warps
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    fs.set_path(fs.FS_PATH_TC_PAIR)
    try:
        p_ids, p_mx = fs.sample(hd[:256], Wd, td[:256], 6, 11)      # pair sampler: 16 warps
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    t_ids, t_z = fs.sample_topk(hd[:256], Wd, td[:256], 6, 11, 1)   # pair top-k: 8 warps
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids16.cpu().numpy(), ids8[:128].cpu().numpy())
    np.testing.assert_array_equal(mx16.cpu().numpy(), mx8[:128].cpu().numpy())
    np.testing.assert_array_equal(t_ids[:, 0].cpu().numpy(), p_ids.cpu().numpy())
    np.testing.assert_array_equal(t_z[:, 0].cpu().numpy(), p_mx.cpu().numpy())
    compare(ids8.cpu().numpy(), mx8.cpu().numpy(), sampler.sample(h, W, temp, 6, 11), what="8-warp batch")


# ------------------------------------------------------------------ launch overlap
@pytest.mark.parametrize("B", [2, 16, 96, 128, 256, 300])
def test_launch_overlap_gives_identical_results(fs, torch_cuda, B):
    """Back-to-back one-shot calls launched as programmatic dependents (the
    default) equal the same calls launched plainly, bit for bit -- also when a
    torch kernel rewrites h and T between two calls on the same stream."""
    torch = torch_cuda
    h, W, temp = _problem(B, 5000, 256, seed=60 + B)
    h2, _, temp2 = _problem(B, 1, 256, seed=61 + B)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    h2d, t2d = to_device(h2, torch), to_device(temp2, torch)

    def run(overlap):
        fs.set_launch_overlap(overlap)
        try:
            x, t = hd.clone(), td.clone()
            outs = []
            for step in range(3):
                outs.append(fs.sample(x, Wd, t, 5, step))
            x.copy_(h2d)
            t.copy_(t2d)
            outs.append(fs.sample(x, Wd, t, 5, 3))
            outs.append(fs.sample(x, Wd, t, 5, 4))
            torch.cuda.synchronize()
            return [(i.cpu().numpy(), m.cpu().numpy()) for i, m in outs]
        finally:
            fs.set_launch_overlap(True)

    on, off = run(True), run(False)
    for (i1, m1), (i0, m0) in zip(on, off):
        np.testing.assert_array_equal(i1, i0)
        np.testing.assert_array_equal(m1, m0)
    compare(on[3][0], on[3][1], sampler.sample(h2, W, temp2, 5, 3), what=f"overlap B={B}")


def test_sample_host_pinned_and_pageable_agree(fs, torch_cuda):
    """fs_sample_host reads mapped pinned buffers directly (copy kernel +
    overlapped launch + mapped results) and copies pageable ones: both give
    the device-buffer sample, for every kernel family's batch sizes."""
    torch = torch_cuda
    for B in (1, 16, 130, 300):
        h, W, temp = _problem(B, 3001, 128, seed=70 + B)
        Wd = to_device(W, torch)
        ids_d, mx_d = _run(fs, torch, h, W, temp, 12, 5)
        h_pin = torch.from_numpy(h.view(np.int16)).pin_memory()
        t_pin = torch.from_numpy(temp).pin_memory()
        ids_p, mx_p = fs.sample_host(h_pin, Wd, t_pin, 12, 5)
        ids_q, mx_q = fs.sample_host(h, Wd, temp, 12, 5)
        np.testing.assert_array_equal(ids_p, ids_d)
        np.testing.assert_array_equal(mx_p, mx_d)
        np.testing.assert_array_equal(ids_q, ids_d)
        np.testing.assert_array_equal(mx_q, mx_d)


def test_gumbel_transform_on_the_whole_uniform_grid(fs, tmp_path):
    """The device noise transform is checked on EVERY value it can see: the
    sampler's u is one of the 2^23 grid points (m + 1/2) 2^-23, and the
    library's own gumbel_from_word, compiled into a small helper from the
    library's device header, is compared with the fp64 -log(-log u) of the
    oracle at all of them.  The largest error bounds the noise error of every
    score the kernels form (the parity tolerance assumes < 1e-5)."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    here = os.path.dirname(__file__)
    src = os.path.join(here, "gpu_helpers", "gumbel_grid.cu")
    inc = os.path.join(os.path.dirname(here), "lm_head_exact_gb300", "csrc")
    exe = str(tmp_path / "gumbel_grid")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I", inc,
                        "-o", exe, src], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = str(tmp_path / "grid.f32")
    run = subprocess.run([exe, out], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    g = np.fromfile(out, dtype=np.float32)
    assert g.size == 1 << 23
    words = np.arange(1 << 23, dtype=np.uint32) << np.uint32(9)
    ref = sampler.gumbel_from_uniform(sampler.uniform_from_word(words))
    err = np.abs(g.astype(np.float64) - ref)
    worst = int(np.argmax(err))
    print(f"device Gumbel over the whole u grid: max |error| {err.max():.3g} at u = {(worst + 0.5) * 2.0 ** -23!r}")
    assert np.isfinite(g).all()
    assert err.max() < 1e-5, (err.max(), worst)
    assert g[0] == g.min() and g[-1] == g.max()          # monotone ends: the support's extremes
    # the kernels' noise pruning and early finalization bound every device
    # Gumbel value by the grid's largest fp64 value rounded up, 16.6356
    assert g.max() <= np.float32(16.6356), g.max()
    assert ref.max() < 16.6356


def test_noise_words_match_curand_philox(fs, torch_cuda, tmp_path):
    """The library's noise words equal cuRAND's device-API Philox-4x32-10
    (curandStatePhilox4_32_10_t, curand4) run as a library, with the
    sampler's key / counter layout reached through curand_init(seed,
    subsequence = step, offset = (row << 34) + 4 (id >> 2))."""
    import shutil
    import subprocess
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    src = os.path.join(os.path.dirname(__file__), "gpu_helpers", "curand_philox_words.cu")
    exe = str(tmp_path / "curand_words")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-o", exe, src],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    seed = 0x1234ABCD5678EF01
    cases = [(row0, v0, step) for row0, v0, step in ((0, 0, 0), (5, 3, 99), (1000, 151900, (3 << 32) + 17))]
    for row0, v0, step in cases:
        n_rows, n_vocab = 7, 13
        words, _ = fs.debug_noise(seed, step, row0, n_rows, v0, n_vocab)
        torch_cuda.cuda.synchronize()
        ours = words.cpu().numpy().view(np.uint32).reshape(n_rows, n_vocab)
        triples = [(row0 + r_, v0 + j, step) for r_ in range(n_rows) for j in range(n_vocab)]
        stdin = f"{seed} {len(triples)}\n" + "\n".join(f"{a} {b} {c}" for a, b, c in triples) + "\n"
        out = subprocess.run([exe], input=stdin, capture_output=True, text=True, timeout=60)
        assert out.returncode == 0, out.stderr
        theirs = np.array([int(x) for x in out.stdout.split()], dtype=np.uint64).astype(np.uint32)
        np.testing.assert_array_equal(ours.ravel(), theirs)
