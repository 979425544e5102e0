"""GPU parity of the fused kernels' LOGITS, and the signed-zero tie rule.

The fused path never writes logits (summary page, "Method": the logit tile
lives on chip), so fs_debug_fused_logits runs the very launch fs_sample_ex
runs -- same kernel family, instantiation and grid -- with the kernel's
inspection store switched on, and the accumulator values its epilogue scans
are compared element by element with the fp64 oracle's logits at
|delta| <= 2e-3, for every kernel family, ragged vocabulary and model widths,
with and without a bias, and at the Llama-3-8B head's full size.
"""

import numpy as np
import pytest

from _helpers import MAX_TOL, compare, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-3


@pytest.fixture(params=["simt", "tc_vocab", "tc_batch", "tc_pair"])
def path(request, fs):
    code = {"simt": fs.FS_PATH_SIMT, "tc_vocab": fs.FS_PATH_TC_VOCAB,
            "tc_batch": fs.FS_PATH_TC_BATCH, "tc_pair": fs.FS_PATH_TC_PAIR}[request.param]
    fs.set_path(code)
    yield request.param
    fs.set_path(fs.FS_PATH_AUTO)


def _problem(B, V, d, seed):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.05).astype(np.float32))
    temp = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temp[::7] = 0.0
    temp[3::11] = -1.0                 # invalid rows: no sample, logits still formed
    return h, W, temp


@pytest.mark.parametrize("B", [1, 17, 130])
@pytest.mark.parametrize("V,d", [(127, 64), (4097, 200), (4097, 64), (127, 200)])
def test_fused_logits_match_oracle(fs, torch_cuda, path, B, V, d):
    torch = torch_cuda
    h, W, temp = _problem(B, V, d, seed=B * 31 + V + d)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    ids, mx, lg = fs.debug_fused_logits(hd, Wd, td, 77, 5)
    ids_s, mx_s = fs.sample(hd, Wd, td, 77, 5)
    torch.cuda.synchronize()
    got = lg.cpu().numpy().astype(np.float64)
    assert not np.isnan(got).any(), "every logit must be written"
    ref = sampler.logits(h, W)
    err = np.abs(got - ref)
    assert err.max() <= LOGIT_TOL, f"{path} B={B} V={V} d={d}: max |delta| {err.max():.3g}"
    # the inspection store does not change the sample: same launch, same result
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_s.cpu().numpy())
    np.testing.assert_array_equal(mx.cpu().numpy(), mx_s.cpu().numpy())
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 77, 5), what=f"{path} B={B}")


@pytest.mark.parametrize("shared", [False, True])
def test_fused_logits_with_bias(fs, torch_cuda, path, shared):
    torch = torch_cuda
    B, V, d = 9, 3001, 128
    h, W, temp = _problem(B, V, d, seed=5)
    rng = np.random.default_rng(6)
    bias = rng.standard_normal(V if shared else (B, V)).astype(np.float32)
    hd, Wd, td, bd = to_device(h, torch), to_device(W, torch), to_device(temp, torch), to_device(bias, torch)
    ids, mx, lg = fs.debug_fused_logits(hd, Wd, td, 3, 1, bias=bd)
    torch.cuda.synchronize()
    err = np.abs(lg.cpu().numpy().astype(np.float64) - sampler.logits(h, W, bias))
    assert err.max() <= LOGIT_TOL, err.max()
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 3, 1, bias=bias), what="bias")


@pytest.mark.parametrize("B", [1, 16, 64, 128, 256])
def test_fused_logits_on_llama3_8b_head(fs, torch_cuda, B):
    """Full-size head, the kernel family the batch size selects (the one the
    benchmark times); 6 seeded rows compared over the whole vocabulary."""
    torch = torch_cuda
    fs.set_path(fs.FS_PATH_AUTO)
    wl = synthetic.workload("llama3_8b", 256)
    hd, Wd, td = to_device(wl.h[:B], torch), to_device(wl.W, torch), to_device(wl.temp[:B], torch)
    ids, mx, lg = fs.debug_fused_logits(hd, Wd, td, wl.seed, 0)
    torch.cuda.synchronize()
    rows = np.unique(np.random.default_rng(B).choice(B, size=min(6, B), replace=False))
    got = lg[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    ref = sampler.logits(wl.h[rows], wl.W)
    err = np.abs(got - ref)
    assert err.max() <= LOGIT_TOL, f"B={B} path {fs.path_for_batch(B)}: max |delta| {err.max():.3g}"
    del lg
    ref_s = sampler.sample(wl.h, wl.W, wl.temp, wl.seed, 0, rows=rows)
    compare(ids.cpu().numpy(), mx.cpu().numpy(), ref_s, rows=rows, what=f"8B head B={B}")


def test_signed_zero_scores_tie_to_the_smaller_id(fs, torch_cuda, path):
    """Greedy rows whose best logit is exactly zero at several ids, some
    formed as -0.0 and some as +0.0 (zero rows of h, and W rows of -0.0 and
    +0.0 against a positive h).  The two zeros are equal under the total
    order, so the smallest such id must win -- also when the ids sit in tiles
    of different CTAs, whose candidates meet in the packed cross-CTA key."""
    torch = torch_cuda
    B, V, d = 8, 4097, 64
    rng = np.random.default_rng(8)
    hf = np.abs(rng.standard_normal((B, d))).astype(np.float32) + 0.01
    hf[:3] = 0.0                                         # zero rows: every logit is +-0
    Wf = -(np.abs(rng.standard_normal((V, d))).astype(np.float32) * 0.05 + 0.01)   # all logits < 0 otherwise
    h, W = synthetic.bf16_bits(hf), synthetic.bf16_bits(Wf)
    neg_zero_rows, pos_zero_rows = [3, 3000], [200, 1500, 4000]
    W[neg_zero_rows] = 0x8000                            # -0.0: products with h > 0 are -0
    W[pos_zero_rows] = 0x0000
    temp = np.zeros(B, np.float32)                       # greedy
    temp[7] = 1.0                                        # one sampled row (a zero h row would be pure noise)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    ids, mx = fs.sample(hd, Wd, td, 11, 2)
    torch.cuda.synchronize()
    ids = ids.cpu().numpy()
    ref = sampler.sample(h, W, temp, 11, 2)
    assert list(ref.ids[:3]) == [0, 0, 0] and list(ref.ids[3:7]) == [3, 3, 3, 3], ref.ids
    np.testing.assert_array_equal(ids[:7], ref.ids[:7])
    assert np.all(mx.cpu().numpy()[:7] == 0.0)
    compare(ids, mx.cpu().numpy(), ref, what=f"signed zero {path}")


@pytest.mark.parametrize("B,V,d", [(64, 4097, 4096), (128, 8192, 4096), (200, 3000, 1024), (32, 1000, 8192),
                                   (256, 16032, 4096), (48, 3001, 200), (100, 2000, 72), (160, 5000, 328)])
def test_tensor_core_families_form_identical_logits(fs, torch_cuda, B, V, d):
    """The three tensor-core kernel families -- vocabulary-major (W as the
    MMA's A operand, M = 128 vocabulary rows), batch-major (h as A, one CTA)
    and the CTA pair (cta_group::2, M = 256) -- run the same K order of
    bf16 x bf16 -> fp32 MMAs, and their logits agree BIT FOR BIT: the
    MMA's rounding does not depend on the tile shape, the operand roles or
    the CTA pairing.  So which tensor-core family samples a batch cannot
    change a sample (the scan over the logits is the same arithmetic in every
    family), the property that lets chunked and one-shot calls agree exactly."""
    torch = torch_cuda
    rng = np.random.default_rng(B + V + d)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.02).astype(np.float32))
    temp = np.ones(B, np.float32)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    bits = {}
    try:
        for name, code in [("tc_vocab", fs.FS_PATH_TC_VOCAB), ("tc_batch", fs.FS_PATH_TC_BATCH),
                           ("tc_pair", fs.FS_PATH_TC_PAIR)]:
            fs.set_path(code)
            ids, mx, lg = fs.debug_fused_logits(hd, Wd, td, 21, 4)
            torch.cuda.synchronize()
            bits[name] = (lg.cpu().numpy().view(np.uint32).copy(), ids.cpu().numpy(), mx.cpu().numpy())
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    ref = bits["tc_pair"]
    for name, (lb, ids, mx) in bits.items():
        assert np.array_equal(lb, ref[0]), f"{name}: {(lb != ref[0]).sum()} logits differ from tc_pair's"
        np.testing.assert_array_equal(ids, ref[1])
        np.testing.assert_array_equal(mx, ref[2])
