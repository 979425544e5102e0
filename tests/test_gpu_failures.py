"""Failure detection without a GPU fault: injected host-side failures of an
allocation and of a launch (the library returns the failing call's error
before touching the GPU, and later calls work), the same through the
FS_FAULT environment variable, and canary guard bands around every output
buffer (a write outside the outputs would show in the guards)."""

import os
import subprocess
import sys

import numpy as np
import pytest

from _helpers import compare, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem(B, V, d, seed):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.05).astype(np.float32))
    temp = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    return h, W, temp


def test_injected_launch_failure_reports_and_recovers(fs, torch_cuda):
    torch = torch_cuda
    h, W, temp = _problem(16, 3001, 128, seed=1)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    fs.debug_set_fault(fs.FS_FAULT_LAUNCH)
    try:
        with pytest.raises(fs.FlashSampleError) as err:
            fs.sample(hd, Wd, td, 3, 1)
        assert err.value.status == "FS_ERR_CUDA" and "injected" in str(err.value)
    finally:
        fs.debug_set_fault(fs.FS_FAULT_NONE)
    assert fs.device_error() == 0
    ids, mx = fs.sample(hd, Wd, td, 3, 1)
    torch.cuda.synchronize()
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 3, 1), what="after launch fault")


def test_injected_allocation_failure_reports_and_recovers(fs, torch_cuda):
    torch = torch_cuda
    h, W, temp = _problem(8, 2000, 64, seed=2)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    stream = torch.cuda.Stream()             # a new stream: its workspace must be allocated
    fs.debug_set_fault(fs.FS_FAULT_ALLOC)
    try:
        with pytest.raises(fs.FlashSampleError) as err:
            fs.sample(hd, Wd, td, 5, 0, stream=stream)
        assert err.value.status == "FS_ERR_WORKSPACE"
    finally:
        fs.debug_set_fault(fs.FS_FAULT_NONE)
    ids, mx = fs.sample(hd, Wd, td, 5, 0, stream=stream)
    torch.cuda.synchronize()
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 5, 0), what="after alloc fault")


_ENV_FAULT = r"""
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
from lm_head_exact_gb300 import binding as fs
h = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
W = torch.zeros((100, 64), dtype=torch.bfloat16, device="cuda")
t = torch.ones(2, device="cuda")
try:
    fs.sample(h, W, t, 1, 0)
    print("no-error")
except fs.FlashSampleError as e:
    print("error", e.status)
"""


def test_fault_injection_from_the_environment(fs, torch_cuda):
    env = dict(os.environ, FS_FAULT="launch")
    r = subprocess.run([sys.executable, "-c", _ENV_FAULT.format(root=ROOT)], capture_output=True, text=True,
                       timeout=240, env=env)
    assert r.returncode == 0 and "error FS_ERR_CUDA" in r.stdout, (r.stdout, r.stderr[-2000:])


SENTINEL_ID = -123456789
SENTINEL_F = -7.25


def _guarded(torch, shape, dtype, g=37):
    """A tensor with g guard elements (rows for 2-D) on both sides; returns
    (buffer, view of the payload)."""
    if len(shape) == 1:
        buf = torch.full((shape[0] + 2 * g,), SENTINEL_ID if dtype == torch.int64 else SENTINEL_F, dtype=dtype,
                         device="cuda")
        return buf, buf[g:g + shape[0]]
    buf = torch.full((shape[0] + 2 * g, shape[1]), SENTINEL_ID if dtype == torch.int64 else SENTINEL_F, dtype=dtype,
                     device="cuda")
    return buf, buf[g:g + shape[0]]


def _guards_intact(buf, n, g=37):
    a = buf.cpu().numpy()
    s = SENTINEL_ID if a.dtype == np.int64 else SENTINEL_F
    return np.all(a[:g] == s) and np.all(a[g + n:] == s)


@pytest.mark.parametrize("B", [1, 16, 130, 300])
def test_outputs_have_intact_guard_bands(fs, torch_cuda, B):
    torch = torch_cuda
    V, d, k = 4099, 128, 8
    h, W, temp = _problem(B, V, d, seed=B)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    ids_buf, ids = _guarded(torch, (B,), torch.int64)
    mx_buf, mx = _guarded(torch, (B,), torch.float32)
    fs.sample(hd, Wd, td, 2, 2, out=(ids, mx))
    # chunked with guarded carries
    cm_buf, cm = _guarded(torch, (B,), torch.float32)
    ci_buf, ci = _guarded(torch, (B,), torch.int64)
    bounds = synthetic.chunk_bounds(V, 3)
    cids_buf, cids = _guarded(torch, (B,), torch.int64)
    cmx_buf, cmx = _guarded(torch, (B,), torch.float32)
    for i, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        fs.sample_chunked(hd, Wd[lo:hi], lo, td, 2, 2, cm, ci, i == 0, i == 2, out=(cids, cmx))
    # top-k with guarded [B, k] outputs (guard rows)
    tk_ids_buf, tk_ids = _guarded(torch, (B, k), torch.int64)
    tk_z_buf, tk_z = _guarded(torch, (B, k), torch.float32)
    fs.sample_topk(hd, Wd, td, 2, 2, k, out=(tk_ids, tk_z))
    torch.cuda.synchronize()
    for buf, n in ((ids_buf, B), (mx_buf, B), (cm_buf, B), (ci_buf, B), (cids_buf, B), (cmx_buf, B),
                   (tk_ids_buf, B), (tk_z_buf, B)):
        assert _guards_intact(buf, n)
    np.testing.assert_array_equal(cids.cpu().numpy(), ids.cpu().numpy())
    assert fs.device_error() == 0
