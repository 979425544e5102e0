"""GPU parity of online early finalization (chunked variant): the row norms
and rest bounds against the fp64 oracle, the done flag against the oracle's
stopping point, and the result against both the oracle and the plain chunked
path, bit for bit.
"""

import numpy as np
import pytest

from _helpers import compare, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu

PATHS = ["simt", "tc_vocab", "tc_batch", "tc_pair"]


@pytest.fixture(params=PATHS)
def path(request, fs):
    code = {"simt": fs.FS_PATH_SIMT, "tc_vocab": fs.FS_PATH_TC_VOCAB,
            "tc_batch": fs.FS_PATH_TC_BATCH, "tc_pair": fs.FS_PATH_TC_PAIR}[request.param]
    fs.set_path(code)
    yield request.param
    fs.set_path(fs.FS_PATH_AUTO)


def _problem(B, V, d, seed, w_std=0.05):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    # per-row scales so that the largest row norm moves from chunk to chunk
    scale = rng.uniform(0.5, 2.0, size=(V, 1)).astype(np.float32)
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * w_std * scale).astype(np.float32))
    temps = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temps[::7] = 0.0
    return h, W, temps


def _run_early(fs, torch, hd, Wd, td, bd, bounds, seed, step, rest, rest_bias, serial=False):
    """All chunk calls in order; returns (ids, max, done after each call)."""
    B = hd.shape[0]
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    done = torch.full((1,), 7, dtype=torch.int32, device="cuda")     # stale value: the first call overwrites it
    hn = fs.row_norms(hd)
    flags = []
    res = None
    n = len(bounds) - 1
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        bc = None if bd is None else bd[:, lo:hi]
        res = fs.sample_chunked_early(hd, Wd[lo:hi], lo, td, seed, step, cm, ci, i == 0, i == n - 1,
                                      hn, rest[i], rest_bias[i], done, bias_chunk=bc, serial=serial)
        torch.cuda.synchronize()
        flags.append(int(done.item()))
    return res[0].cpu().numpy(), res[1].cpu().numpy(), flags


def _run_chunked(fs, torch, hd, Wd, td, bd, bounds, seed, step):
    B = hd.shape[0]
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    n = len(bounds) - 1
    res = None
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        bc = None if bd is None else bd[:, lo:hi].contiguous()
        res = fs.sample_chunked(hd, Wd[lo:hi], lo, td, seed, step, cm, ci, i == 0, i == n - 1, bias_chunk=bc)
    torch.cuda.synchronize()
    return res[0].cpu().numpy(), res[1].cpu().numpy()


def _rest_bias(bias, bounds):
    if bias is None:
        return [0.0] * (len(bounds) - 1)
    return [float(bias[:, hi:].max()) if hi < bias.shape[1] else 0.0 for hi in bounds[1:]]


# ------------------------------------------------------------------ norms
def test_row_norms_match_oracle(fs, torch_cuda):
    X = synthetic.normal_rows_bf16(5, 1003, 4096, 1.0)
    out = fs.row_norms(to_device(X, torch_cuda))
    torch_cuda.cuda.synchronize()
    np.testing.assert_allclose(out.cpu().numpy(), sampler.row_norms(X), rtol=1e-5)


@pytest.mark.parametrize("bounds", [None, [0, 0, 100, 100, 9000, 20011]])
def test_chunk_rest_norms_match_oracle(fs, torch_cuda, bounds):
    V, d = 20011, 256
    _, W, _ = _problem(1, V, d, seed=3)
    bounds = bounds or synthetic.chunk_bounds(V, 8)
    rest = fs.chunk_rest_norms(to_device(W, torch_cuda), bounds)
    wn = sampler.row_norms(W)
    ref = [wn[hi:].max() if hi < V else 0.0 for hi in bounds[1:]]
    np.testing.assert_allclose(rest, ref, rtol=1e-5)
    assert rest[-1] == 0.0


# ------------------------------------------------------------------ small cases, every kernel family
@pytest.mark.parametrize("serial", [False, True])
@pytest.mark.parametrize("kind", ["spiked", "flat", "mixed"])
def test_early_small_matches_oracle(fs, torch_cuda, path, kind, serial):
    torch = torch_cuda
    B, V, d, n = 37, 4099, 256, 8
    h, W, temp = _problem(B, V, d, seed=21)
    temp[5] = -1.0                                      # invalid row: final by definition, id -1
    bounds = synthetic.chunk_bounds(V, n)
    bias = None
    if kind != "flat":
        rows = None if kind == "spiked" else range(0, B, 2)
        bias = synthetic.leading_spike_bias(B, V, bounds[1], 400.0, rows=rows)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bd = None if bias is None else to_device(bias, torch)
    rest = fs.chunk_rest_norms(Wd, bounds)
    ids, mx, flags = _run_early(fs, torch, hd, Wd, td, bd, bounds, 9, 2, rest, _rest_bias(bias, bounds), serial)
    ids_c, mx_c = _run_chunked(fs, torch, hd, Wd, td, bd, bounds, 9, 2)
    np.testing.assert_array_equal(ids, ids_c)
    np.testing.assert_array_equal(mx, mx_c)
    compare(ids, mx, sampler.sample(h, W, temp, 9, 2, bias=bias), what=f"early {kind}")
    (_, _), read = sampler.sample_chunked_early(h, W, temp, 9, 2, bounds, bias=bias)
    if kind == "spiked":
        assert read == 1 and flags == [1] * n, flags
    else:
        assert read == n and flags[:-1] == [0] * (n - 1), flags
    assert ids[5] == -1


def test_early_empty_first_chunk_clears_stale_flag(fs, torch_cuda):
    """The first call resets a stale done flag even when its chunk holds no
    vocabulary (the reduction kernel runs instead of a fused one)."""
    torch = torch_cuda
    B, V, d = 9, 3001, 128
    h, W, temp = _problem(B, V, d, seed=22)
    bounds = [0, 0, 1500, V]
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    rest = fs.chunk_rest_norms(Wd, bounds)
    ids, mx, flags = _run_early(fs, torch, hd, Wd, td, None, bounds, 4, 1, rest, [0.0] * 3)
    assert flags[0] == 0
    compare(ids, mx, sampler.sample(h, W, temp, 4, 1), what="early, empty first chunk")


# ------------------------------------------------------------------ full size (chunked workload shape)
@pytest.mark.parametrize("B", [1, 32, 64, 256])
def test_early_full_size_spiked_and_flat(fs, torch_cuda, B):
    """d 4096, V 128256 in 8 chunks.  Without spikes no row is ever final
    (the bound |h||W|/T + 16.6 is far above the winning scores) and every
    chunk runs; with a +200 spike in the first chunk of every row, the first
    call finalizes all rows.  Both equal the one-shot sample bit for bit.
    (At B = 64 the second step's chunks run on the CTA-pair kernel, the
    one-shot call on the vocabulary-major kernel.)"""
    torch = torch_cuda
    wl = synthetic.workload("chunked", B)
    V = wl.W.shape[0]
    bounds = synthetic.chunk_bounds(V, 8)
    hd, Wd, td = to_device(wl.h, torch), to_device(wl.W, torch), to_device(wl.temp, torch)
    rest = fs.chunk_rest_norms(Wd, bounds)
    rows = np.unique(np.r_[0, B - 1, np.random.default_rng(B).choice(B, size=min(B, 6), replace=False)])
    for kind in ("flat", "spiked"):
        bias = None if kind == "flat" else synthetic.leading_spike_bias(B, V, bounds[1], 200.0)
        bd = None if bias is None else to_device(bias, torch)
        ids, mx, flags = _run_early(fs, torch, hd, Wd, td, bd, bounds, wl.seed, 5, rest, _rest_bias(bias, bounds))
        one_ids, one_mx = fs.sample(hd, Wd, td, wl.seed, 5, bias=bd)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids, one_ids.cpu().numpy())
        np.testing.assert_array_equal(mx, one_mx.cpu().numpy())
        ref = sampler.sample(wl.h, wl.W, wl.temp, wl.seed, 5, bias=bias, rows=rows)
        compare(ids, mx, ref, rows=rows, what=f"early full {kind} B={B}")
        assert flags == ([1] * 8 if kind == "spiked" else [0] * 7 + flags[-1:]), flags


@pytest.mark.parametrize("serial", [False, True])
@pytest.mark.parametrize("B", [1, 32, 256])
def test_early_graph_replays_do_not_leak_the_flag(fs, torch_cuda, B, serial):
    """One captured step of 32 chunks (programmatic dependent launches),
    replayed with a +400 spike in chunk 3 of every row (the chunks after it
    skip), then with the bias zeroed (no row is final): a flag left set by
    the first replay must not make the second skip.  Each replay equals the
    one-shot sample of its own bias bit for bit."""
    torch = torch_cuda
    V, d, n = 20011, 256, 32
    h, W, temp = _problem(B, V, d, seed=30 + B)
    bounds = synthetic.chunk_bounds(V, n)
    spikes = synthetic.leading_spike_bias(B, V, bounds[4], 0.0)
    g = np.random.default_rng(B)
    spikes[np.arange(B), g.integers(bounds[3], bounds[4], size=B)] = 400.0
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bd = to_device(spikes, torch)
    rest = fs.chunk_rest_norms(Wd, bounds)
    stream = torch.cuda.Stream()
    fs.workspace_reserve(B, V, stream=stream)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    ids = torch.empty(B, dtype=torch.int64, device="cuda")
    mx = torch.empty(B, dtype=torch.float32, device="cuda")
    hn = torch.empty(B, dtype=torch.float32, device="cuda")
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    chunks = [(lo, hi) for lo, hi in zip(bounds[:-1], bounds[1:])]

    def step():
        fs.row_norms(hd, out=hn, stream=stream)
        for i, (lo, hi) in enumerate(chunks):
            fs.sample_chunked_early(hd, Wd[lo:hi], lo, td, 3, 8, cm, ci, i == 0, i == n - 1, hn, rest[i], 0.0,
                                    done, bias_chunk=bd[:, lo:hi], out=(ids, mx), stream=stream, serial=serial)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for spiked in (True, False, True, False):
        bd.copy_(to_device(spikes if spiked else np.zeros_like(spikes), torch))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        flag = int(done.item())
        one_ids, one_mx = fs.sample(hd, Wd, td, 3, 8, bias=bd)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), one_ids.cpu().numpy())
        np.testing.assert_array_equal(mx.cpu().numpy(), one_mx.cpu().numpy())
        if spiked:
            assert flag == 1
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 3, 8), what=f"early graph B={B}")
    del graph


@pytest.mark.parametrize("B", [1, 32, 256])
def test_early_overlapped_chunks_stress(fs, torch_cuda, B):
    """With overlapped (programmatic dependent) launches the CTAs of one chunk
    may start on either side of the previous chunk's flag write, so some may
    skip and others run.  Full-size head in 32 chunks, winners planted in
    chunk 3: 40 graph replays with the spikes and 10 without must each equal
    the one-shot sample bit for bit and leave no device error."""
    torch = torch_cuda
    wl = synthetic.workload("chunked", B)
    V, n = wl.W.shape[0], 32
    bounds = synthetic.chunk_bounds(V, n)
    spikes = np.zeros((B, V), np.float32)
    g = np.random.default_rng(7 + B)
    spikes[np.arange(B), g.integers(bounds[3], bounds[4], size=B)] = 200.0
    hd, Wd, td = to_device(wl.h, torch), to_device(wl.W, torch), to_device(wl.temp, torch)
    bd = to_device(spikes, torch)
    rest = fs.chunk_rest_norms(Wd, bounds)
    stream = torch.cuda.Stream()
    fs.workspace_reserve(B, V, stream=stream)
    cm = torch.empty(B, device="cuda")
    ci = torch.empty(B, dtype=torch.int64, device="cuda")
    ids = torch.empty(B, dtype=torch.int64, device="cuda")
    mx = torch.empty(B, dtype=torch.float32, device="cuda")
    hn = torch.empty(B, dtype=torch.float32, device="cuda")
    done = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        fs.row_norms(hd, out=hn, stream=stream)
        for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
            fs.sample_chunked_early(hd, Wd[lo:hi], lo, td, wl.seed, 2, cm, ci, i == 0, i == n - 1, hn, rest[i],
                                    0.0, done, bias_chunk=bd[:, lo:hi], out=(ids, mx), stream=stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for spiked, reps in ((True, 40), (False, 10)):
        if not spiked:
            bd.zero_()
        one_ids, one_mx = fs.sample(hd, Wd, td, wl.seed, 2, bias=bd)
        torch.cuda.synchronize()
        want_ids, want_mx = one_ids.cpu().numpy(), one_mx.cpu().numpy()
        for _ in range(reps):
            ids.fill_(-7)
            graph.replay()
            torch.cuda.synchronize()
            np.testing.assert_array_equal(ids.cpu().numpy(), want_ids)
            np.testing.assert_array_equal(mx.cpu().numpy(), want_mx)
        if spiked:
            assert int(done.item()) == 1
    assert fs.device_error() == 0
    del graph
