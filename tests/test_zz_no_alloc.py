"""fs_sample_noalloc: the allocation-free entry point.

Some callers cannot let a library allocate device memory -- their allocator
already owns the GPU's memory budget, or they cannot afford the device-wide
synchronization that freeing a workspace implies.  fs_sample_noalloc serves
them by keeping its scratch in a fixed static device array.  This test calls it
through the C ABI twice in a row (a larger call, then a smaller one, so stale
scratch contents from the first call would show up in the second) and checks
both results against fs_sample, the allocating entry point, with the same
tolerance as the other parity tests.  It also checks the batch limit and that
a call on a brand-new stream leaves the device's free memory unchanged.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest

from _helpers import MAX_TOL, to_device
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _inputs(B, V, d, seed):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.05).astype(np.float32))
    temp = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temp[::5] = 0.0
    return h, W, temp


def _noalloc(lib, torch, hd, Wd, td, seed, step, stream):
    B, d = hd.shape
    V = Wd.shape[0]
    ids = torch.empty(B, dtype=torch.int64, device="cuda")
    mx = torch.empty(B, dtype=torch.float32, device="cuda")
    st = lib.fs_sample_noalloc(ctypes.c_void_p(hd.data_ptr()), ctypes.c_void_p(Wd.data_ptr()), B, d, V,
                               ctypes.c_void_p(td.data_ptr()), seed, step, ctypes.c_void_p(ids.data_ptr()),
                               ctypes.c_void_p(mx.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    return st, ids, mx


def test_noalloc_matches_fs_sample_on_two_calls_in_a_row(fs, torch_cuda):
    torch = torch_cuda
    lib = fs.library()
    fs.set_path(fs.FS_PATH_AUTO)
    stream = torch.cuda.current_stream()
    for B, V, d, seed, step in [(200, 5003, 256, 21, 3), (16, 4097, 512, 22, 4)]:
        h, W, temp = _inputs(B, V, d, seed)
        hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
        ids_ref, mx_ref = fs.sample(hd, Wd, td, 1234, step)
        st, ids, mx = _noalloc(lib, torch, hd, Wd, td, 1234, step, stream)
        assert st == 0, lib.fs_last_error().decode()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy())
        assert np.abs(mx.cpu().numpy() - mx_ref.cpu().numpy()).max() <= MAX_TOL


def test_noalloc_rejects_batches_beyond_its_scratch(fs, torch_cuda):
    torch = torch_cuda
    lib = fs.library()
    h, W, temp = _inputs(257, 300, 64, 23)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    st, _, _ = _noalloc(lib, torch, hd, Wd, td, 1, 0, torch.cuda.current_stream())
    assert st == 2                                          # FS_ERR_UNSUPPORTED
    assert b"256" in lib.fs_last_error()


def test_noalloc_call_on_a_new_stream_allocates_nothing(fs, torch_cuda):
    torch = torch_cuda
    lib = fs.library()
    h, W, temp = _inputs(32, 4096, 256, 24)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    warm = torch.cuda.Stream()
    st, _, _ = _noalloc(lib, torch, hd, Wd, td, 1, 0, warm)      # kernels loaded, set-up done
    assert st == 0
    torch.cuda.synchronize()
    fresh = torch.cuda.Stream()
    ids = torch.empty(32, dtype=torch.int64, device="cuda")
    mx = torch.empty(32, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    st = lib.fs_sample_noalloc(ctypes.c_void_p(hd.data_ptr()), ctypes.c_void_p(Wd.data_ptr()), 32, 256, 4096,
                               ctypes.c_void_p(td.data_ptr()), 1, 1, ctypes.c_void_p(ids.data_ptr()),
                               ctypes.c_void_p(mx.data_ptr()), ctypes.c_void_p(fresh.cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
