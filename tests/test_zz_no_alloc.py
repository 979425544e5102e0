"""fs_sample_noalloc: the allocation-free entry point.

Some callers cannot let a library allocate device memory -- their allocator
already owns the GPU's memory budget, or they cannot afford the device-wide
synchronization that freeing a workspace implies.  fs_sample_noalloc serves
them by keeping its scratch in a fixed static device array.  These tests call
it through the C ABI on calls in a row (a large batch, then smaller ones, so
stale scratch contents from one call would show up in the next) and check
every result against the fp64 oracle with the same comparison rule as the
other parity tests, and against fs_sample: bit for bit where fs_sample runs a
tensor-core kernel (all of them form the same logits), within the tolerance
at B = 1, where it runs the CUDA-core kernel.  They also
check the batch and alignment limits (rejected on the host, nothing is
launched), that the status word of its bounded waits reads 0 after normal
calls, and that a call on a brand-new stream leaves the device's free memory
unchanged.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest

from _helpers import MAX_TOL, compare, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu


def _inputs(B, V, d, seed):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.05).astype(np.float32))
    temp = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temp[::5] = 0.0
    return h, W, temp


def _noalloc(lib, torch, hd, Wd, td, seed, step, stream, ids=None, mx=None):
    B, d = hd.shape
    V = Wd.shape[0]
    ids = torch.empty(B, dtype=torch.int64, device="cuda") if ids is None else ids
    mx = torch.empty(B, dtype=torch.float32, device="cuda") if mx is None else mx
    st = lib.fs_sample_noalloc(ctypes.c_void_p(hd.data_ptr()), ctypes.c_void_p(Wd.data_ptr()), B, d, V,
                               ctypes.c_void_p(td.data_ptr()), seed, step, ctypes.c_void_p(ids.data_ptr()),
                               ctypes.c_void_p(mx.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    return st, ids, mx


def test_noalloc_matches_the_oracle_on_calls_in_a_row(fs, torch_cuda):
    torch = torch_cuda
    lib = fs.library()
    fs.set_path(fs.FS_PATH_AUTO)
    stream = torch.cuda.current_stream()
    # B = 256 is the documented limit; B = 1 is where fs_sample runs the
    # CUDA-core kernel instead; 200 where it runs a batch-major one
    cases = [(256, 5003, 256, 21, 3), (200, 4097, 512, 22, 4), (1, 3001, 128, 23, 5), (16, 4097, 512, 24, 6)]
    for B, V, d, seed, step in cases:
        h, W, temp = _inputs(B, V, d, seed)
        hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
        st, ids, mx = _noalloc(lib, torch, hd, Wd, td, 1234, step, stream)
        assert st == 0, lib.fs_last_error().decode()
        ids_ref, mx_ref = fs.sample(hd, Wd, td, 1234, step)
        torch.cuda.synchronize()
        ref = sampler.sample(h, W, temp, 1234, step)
        got_ids, got_max = ids.cpu().numpy(), mx.cpu().numpy()
        compare(got_ids, got_max, ref, what=f"noalloc B={B}")
        # fs_sample may run another kernel family at this B: the same rule
        compare(ids_ref.cpu().numpy(), mx_ref.cpu().numpy(), ref, what=f"fs_sample B={B}")
        same = got_ids == ids_ref.cpu().numpy()
        assert np.abs(got_max[same] - mx_ref.cpu().numpy()[same]).max() <= MAX_TOL
        if fs.path_for_batch(B) != fs.FS_PATH_SIMT:
            # every tensor-core family forms the same logits: equal bit for bit
            np.testing.assert_array_equal(got_ids, ids_ref.cpu().numpy())
            np.testing.assert_array_equal(got_max, mx_ref.cpu().numpy())
    code = ctypes.c_int(-1)
    assert lib.fs_device_error(ctypes.byref(code)) == 0, lib.fs_last_error().decode()
    assert code.value == 0                                  # no bounded wait ran out


def test_noalloc_rejects_batches_beyond_its_scratch(fs, torch_cuda):
    torch = torch_cuda
    lib = fs.library()
    h, W, temp = _inputs(257, 300, 64, 23)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    st, _, _ = _noalloc(lib, torch, hd, Wd, td, 1, 0, torch.cuda.current_stream())
    assert st == 2                                          # FS_ERR_UNSUPPORTED
    assert b"256" in lib.fs_last_error()


def test_noalloc_rejects_misaligned_outputs_on_the_host(fs, torch_cuda):
    torch = torch_cuda
    lib = fs.library()
    h, W, temp = _inputs(8, 300, 64, 25)
    hd, Wd, td = to_device(h, torch), to_device(W, torch), to_device(temp, torch)
    ids_buf = torch.zeros(9 * 8 + 8, dtype=torch.uint8, device="cuda")
    mx_buf = torch.zeros(8 * 4 + 8, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    B, d = hd.shape

    def call(ids_ptr, mx_ptr, t_ptr):
        return lib.fs_sample_noalloc(ctypes.c_void_p(hd.data_ptr()), ctypes.c_void_p(Wd.data_ptr()), B, d, 300,
                                     ctypes.c_void_p(t_ptr), 1, 0, ctypes.c_void_p(ids_ptr),
                                     ctypes.c_void_p(mx_ptr), ctypes.c_void_p(stream.cuda_stream))

    base_i, base_m = ids_buf.data_ptr(), mx_buf.data_ptr()
    assert call(base_i + 4, base_m, td.data_ptr()) == 2 and b"out_ids" in lib.fs_last_error()
    assert call(base_i, base_m + 2, td.data_ptr()) == 2 and b"out_max" in lib.fs_last_error()
    t_buf = torch.zeros(8 * 4 + 8, dtype=torch.uint8, device="cuda")
    assert call(base_i, base_m, t_buf.data_ptr() + 1) == 2 and b"temp" in lib.fs_last_error()
    torch.cuda.synchronize()
    assert int(ids_buf.sum()) == 0 and int(mx_buf.sum()) == 0   # nothing was written


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
    st, _, _ = _noalloc(lib, torch, hd, Wd, td, 1, 1, fresh, ids, mx)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
