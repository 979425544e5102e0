"""CPU checks of the C ABI: the library builds, loads without a GPU, exports
every entry point include/flashsample.h declares, and rejects malformed
arguments on the host before touching a device."""

import ctypes
import os
import re
import subprocess

import pytest

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "flashsample.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^FS_API\s+[\w\s\*]+?\b(fs_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_api():
    names = declared_symbols()
    for required in ("fs_sample", "fs_sample_ex", "fs_sample_chunked", "fs_sample_host",
                     "fs_status_string", "fs_debug_noise"):
        assert required in names


def test_library_exports_every_declared_symbol(built_library):
    lib = ctypes.CDLL(built_library)
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", built_library], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r" T (fs_\w+)$", out.stdout, flags=re.M))
        assert set(declared_symbols()) <= exported
        # nothing else of the fs_ namespace leaks out
        assert exported <= set(declared_symbols())


def test_binding_signatures_cover_the_header(built_library):
    from lm_head_exact_gb300 import binding
    assert set(binding.SIGNATURES) == set(declared_symbols())
    binding.library()


def test_status_strings(built_library):
    from lm_head_exact_gb300 import binding
    lib = binding.library()
    names = [lib.fs_status_string(i).decode() for i in range(6)]
    assert names == ["FS_OK", "FS_ERR_INVALID_ARG", "FS_ERR_UNSUPPORTED", "FS_ERR_CUDA",
                     "FS_ERR_WORKSPACE", "FS_ERR_DEVICE_TIMEOUT"]
    assert lib.fs_status_string(99).decode() == "FS_STATUS_UNKNOWN"


def test_host_side_argument_checks(built_library):
    from lm_head_exact_gb300 import binding
    lib = binding.library()
    z = ctypes.c_void_p(0)
    # negative / unsupported shapes are refused before any CUDA call
    assert lib.fs_sample(z, z, -1, 64, 10, z, 0, 0, z, z, z) == 1
    assert "B >= 0" in lib.fs_last_error().decode()
    assert lib.fs_sample(z, z, 4, 12, 10, z, 0, 0, z, z, z) == 2
    assert "multiple of 8" in lib.fs_last_error().decode()
    assert lib.fs_sample(z, z, 4, 64, 1 << 31, z, 0, 0, z, z, z) == 2
    assert lib.fs_sample_chunked(z, z, 4, 64, 10, 5, z, z, 0, 0, 0, z, z, 1, z, z, z) == 1
    assert lib.fs_sample_chunked(z, z, 4, 64, 0, 5, z, z, 0, 0, 0, z, z, 8, z, z, z) == 1
    assert lib.fs_set_path(7) == 1
    assert lib.fs_set_launch_overlap(2) == 1
    assert lib.fs_debug_set_fault(7) == 1
    assert lib.fs_debug_set_fault(0) == 0
    # top-k: k outside [1, 16] is refused before anything else
    assert lib.fs_sample_topk(z, z, 4, 64, 10, z, z, 0, 0, 0, 0, z, z, z) == 1
    assert lib.fs_sample_topk(z, z, 4, 64, 10, z, z, 0, 0, 0, 17, z, z, z) == 1
    assert "k must be" in lib.fs_last_error().decode()
    assert lib.fs_sample_topk(z, z, 0, 64, 10, z, z, 0, 0, 0, 4, z, z, z) == 0   # B == 0
    # early finalization: batch limit, NaN bounds, bad chunk bounds
    assert lib.fs_sample_chunked_early(z, z, 4097, 64, 0, 5, z, z, 0, 0, 0, z, z, 1, z, 0.0, 0.0, z, z, z, z) == 2
    assert "B <= 4096" in lib.fs_last_error().decode()
    nan = float("nan")
    assert lib.fs_sample_chunked_early(z, z, 4, 64, 0, 5, z, z, 0, 0, 0, z, z, 1, z, nan, 0.0, z, z, z, z) == 1
    assert lib.fs_sample_chunked_early(z, z, 4, 64, 0, 5, z, z, 0, 0, 0, z, z, 1, z, -1.0, 0.0, z, z, z, z) == 1
    assert lib.fs_sample_chunked_early(z, z, 4, 64, 0, 5, z, z, 0, 0, 0, z, z, 1, z, 1.0, nan, z, z, z, z) == 1
    bounds = (ctypes.c_int64 * 3)(0, 10, 5)
    rest = (ctypes.c_float * 2)()
    assert lib.fs_chunk_rest_norms(z, 64, bounds, 2, rest, z) == 1
    assert "non-decreasing" in lib.fs_last_error().decode()
    assert lib.fs_chunk_rest_norms(z, 64, z, 0, z, z) == 0
    assert lib.fs_row_norms(z, 0, 64, z, z) == 0
    assert lib.fs_row_norms(z, 3, 12, z, z) == 2
    assert lib.fs_debug_noise(0, 0, -1, 1, 0, 1, z, z, z) == 1
    # one-call chunked step: chunk count and bounds are checked before any chunk runs
    ok = (ctypes.c_int64 * 3)(0, 5, 10)
    assert lib.fs_sample_chunked_step(z, z, 4, 64, ok, 0, z, z, 0, 0, 0, z, z, z, z, z) == 1
    assert "n_chunks" in lib.fs_last_error().decode()
    assert lib.fs_sample_chunked_step(z, z, 4, 64, z, 2, z, z, 0, 0, 0, z, z, z, z, z) == 1
    assert lib.fs_sample_chunked_step(z, z, 4, 64, bounds, 2, z, z, 0, 0, 0, z, z, z, z, z) == 1
    assert "must not decrease" in lib.fs_last_error().decode()
    shifted = (ctypes.c_int64 * 3)(3, 5, 10)
    assert lib.fs_sample_chunked_step(z, z, 4, 64, shifted, 2, z, z, 0, 0, 0, z, z, z, z, z) == 1
    assert "bounds[0]" in lib.fs_last_error().decode()
    # B == 0 is a no-op
    assert lib.fs_sample(z, z, 0, 64, 10, z, 0, 0, z, z, z) == 0


def test_product_path_refuses_cpu_tensors(built_library):
    torch = pytest.importorskip("torch")
    from lm_head_exact_gb300 import binding
    h = torch.zeros(2, 8, dtype=torch.bfloat16)
    W = torch.zeros(4, 8, dtype=torch.bfloat16)
    t = torch.ones(2)
    with pytest.raises(binding.FlashSampleError, match="CUDA tensor"):
        binding.sample(h, W, t, 0, 0)
    cm, ci = torch.zeros(2), torch.zeros(2, dtype=torch.int64)
    with pytest.raises(binding.FlashSampleError, match="CUDA tensor"):
        binding.sample_chunked_step(h, W, [0, 2, 4], t, 0, 0, cm, ci)
    with pytest.raises(binding.FlashSampleError, match="bounds"):
        binding.sample_chunked_step(h, W, [0, 2, 3], t, 0, 0, cm, ci)     # must end at W.shape[0]


def test_binding_constants_match_the_header():
    """Every FS_* integer constant of the header (flags, paths, fault kinds,
    status codes) has the same value in the Python binding."""
    from lm_head_exact_gb300 import binding
    text = open(HEADER).read()
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define\s+(FS_\w+)\s+(\d+)", text, flags=re.M)}
    enum_body = re.search(r"typedef enum fs_status \{(.*?)\} fs_status;", text, flags=re.S).group(1)
    status = {m.group(1): int(m.group(2)) for m in re.finditer(r"(FS_\w+)\s*=\s*(\d+)", enum_body)}
    assert defines, "no #define constants found"
    for name, value in defines.items():
        assert getattr(binding, name) == value, name
    assert status["FS_OK"] == binding.FS_OK
    lib = binding.library()
    for name, value in status.items():
        assert lib.fs_status_string(value).decode() == name


def test_auto_dispatch_rule(built_library):
    """The batch-size rule (host logic, no GPU): B = 1 the CUDA-core kernel,
    B <= 64 vocabulary-major, larger B CTA pairs where padding to 256-row pair
    tiles wastes fewer than 128 rows, else batch-major; a forced family is
    honoured (vocabulary-major only up to B = 256) and AUTO restores the rule."""
    from lm_head_exact_gb300 import binding as fs
    expect = {1: fs.FS_PATH_SIMT, 2: fs.FS_PATH_TC_VOCAB, 64: fs.FS_PATH_TC_VOCAB, 65: fs.FS_PATH_TC_BATCH,
              96: fs.FS_PATH_TC_BATCH, 128: fs.FS_PATH_TC_BATCH, 129: fs.FS_PATH_TC_PAIR,
              256: fs.FS_PATH_TC_PAIR, 300: fs.FS_PATH_TC_BATCH, 384: fs.FS_PATH_TC_BATCH,
              385: fs.FS_PATH_TC_PAIR, 512: fs.FS_PATH_TC_PAIR, 600: fs.FS_PATH_TC_BATCH,
              1024: fs.FS_PATH_TC_PAIR}
    for B, path in expect.items():
        assert fs.path_for_batch(B) == path, B
    try:
        fs.set_path(fs.FS_PATH_TC_VOCAB)
        assert fs.path_for_batch(200) == fs.FS_PATH_TC_VOCAB
        assert fs.path_for_batch(300) == fs.FS_PATH_TC_BATCH
        fs.set_path(fs.FS_PATH_TC_PAIR)
        assert fs.path_for_batch(16) == fs.FS_PATH_TC_PAIR
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
    assert fs.path_for_batch(16) == fs.FS_PATH_TC_VOCAB


def test_chunk_dispatch_rule(built_library):
    """Chunk calls (host logic, no GPU): B = 1, B <= 32 and B > 128 keep the
    batch-size family; 32 < B <= 128 take the CTA-pair kernel when the step
    (the previous step's chunk count) fits one wave of pairs with at most 7
    tiles per pair and every chunk has at least 24 pair tiles, else the batch-
    major kernel; a forced family is honoured.  Chunks of the 128256-row
    vocabulary: 8 chunks of 16032 rows (63 tiles: 8 x 9 = 72 pairs at k = 7),
    10 of 12826 (51 tiles: 80 pairs), 32 of 4008 (16 tiles)."""
    from lm_head_exact_gb300 import binding as fs
    V = 128256
    for B in (1, 16, 32, 129, 256):
        for n in (0, 8, 32):
            assert fs.path_for_chunks(B, -(-V // max(n, 8)), n) == fs.path_for_batch(B), (B, n)
    for B in (33, 64, 100, 128):
        assert fs.path_for_chunks(B, 16032, 8) == fs.FS_PATH_TC_PAIR, B
        assert fs.path_for_chunks(B, 16032, 0) == fs.FS_PATH_TC_BATCH, B    # first step: no count yet
        assert fs.path_for_chunks(B, 12826, 10) == fs.FS_PATH_TC_BATCH, B
        assert fs.path_for_chunks(B, 4008, 32) == fs.FS_PATH_TC_BATCH, B
        assert fs.path_for_chunks(B, 5888, 8) == fs.FS_PATH_TC_BATCH, B     # 23 pair tiles per chunk
        # 12 chunks of 42 tiles would fit one wave of pairs, but stream-launched
        # chunk grids run at most 8 at a time
        assert fs.path_for_chunks(B, 10688, 12) == fs.FS_PATH_TC_BATCH, B
    try:
        fs.set_path(fs.FS_PATH_TC_VOCAB)
        assert fs.path_for_chunks(64, 16032, 8) == fs.FS_PATH_TC_VOCAB
    finally:
        fs.set_path(fs.FS_PATH_AUTO)
