"""ctypes binding of libflashsample (include/flashsample.h).

Argument marshalling only: every step of sampling runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  If the
library is missing, or a tensor is not on a CUDA device, the call raises --
there is no CPU fallback.
"""

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libflashsample.so")

FS_OK = 0
FS_CHUNK_FIRST = 1
FS_CHUNK_LAST = 2
FS_CHUNK_SERIAL = 4
FS_PATH_AUTO, FS_PATH_SIMT, FS_PATH_TC_VOCAB, FS_PATH_TC_BATCH, FS_PATH_TC_PAIR = 0, 1, 2, 3, 4
FS_FAULT_NONE, FS_FAULT_ALLOC, FS_FAULT_LAUNCH = 0, 1, 2

_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_int = ctypes.c_int

# name -> (restype, argtypes); mirrors include/flashsample.h
SIGNATURES = {
    "fs_sample": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _u64, _u64,
                         _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_ex": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _i64,
                            _u64, _u64, _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_chunked": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _i64, _c_void_p,
                                 _c_void_p, _i64, _u64, _u64, _c_void_p, _c_void_p, _int,
                                 _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_chunked_early": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _i64, _c_void_p,
                                       _c_void_p, _i64, _u64, _u64, _c_void_p, _c_void_p, _int,
                                       _c_void_p, ctypes.c_float, ctypes.c_float, _c_void_p,
                                       _c_void_p, _c_void_p, _c_void_p]),
    "fs_row_norms": (_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p]),
    "fs_chunk_rest_norms": (_int, [_c_void_p, _i64, _c_void_p, _i64, _c_void_p, _c_void_p]),
    "fs_combine_shards": (_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_topk": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _i64,
                              _u64, _u64, _int, _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_unfused": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _i64,
                                 _u64, _u64, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_host": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _i64,
                              _u64, _u64, _c_void_p, _c_void_p, _c_void_p]),
    "fs_sample_noalloc": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _u64, _u64,
                                 _c_void_p, _c_void_p, _c_void_p]),
    "fs_workspace_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "fs_workspace_reserve": (_int, [_i64, _i64, _c_void_p]),
    "fs_workspace_release": (_int, []),
    "fs_set_path": (_int, [_int]),
    "fs_set_launch_overlap": (_int, [_int]),
    "fs_path_for_batch": (_int, [_i64]),
    "fs_sample_chunked_step": (_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _int, _c_void_p, _c_void_p,
                                      _i64, _u64, _u64, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                      _c_void_p]),
    "fs_path_for_chunks": (_int, [_i64, _i64, _int]),
    "fs_profile_events": (_int, [_c_void_p, _c_void_p]),
    "fs_device_error": (_int, [ctypes.POINTER(_int)]),
    "fs_debug_wait_timeout": (_int, [_u64, _c_void_p]),
    "fs_debug_set_fault": (_int, [_int]),
    "fs_status_string": (ctypes.c_char_p, [_int]),
    "fs_last_error": (ctypes.c_char_p, []),
    "fs_debug_noise": (_int, [_u64, _u64, _i64, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "fs_debug_fused_logits": (_int, [_c_void_p, _c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _i64,
                                     _u64, _u64, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
}


class FlashSampleError(RuntimeError):
    """A libflashsample call returned a non-OK status (or the library is missing)."""

    def __init__(self, status, detail):
        self.status = status
        super().__init__(f"{status}: {detail}")


_lib = None


def library():
    """Load libflashsample.so (once) and declare its signatures."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FlashSampleError("NOT_BUILT", f"{LIB_PATH} is missing; build it with "
                                   "`python -m lm_head_exact_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(status):
    if status != FS_OK:
        lib = library()
        raise FlashSampleError(lib.fs_status_string(status).decode(), lib.fs_last_error().decode())


def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtype=None, ndim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise FlashSampleError("FS_ERR_INVALID_ARG", f"{name} must be a CUDA tensor (no CPU fallback)")
    if dtype is not None and t.dtype != dtype:
        raise FlashSampleError("FS_ERR_INVALID_ARG", f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise FlashSampleError("FS_ERR_INVALID_ARG", f"{name} must have {ndim} dims")
    if not t.is_contiguous():
        raise FlashSampleError("FS_ERR_INVALID_ARG", f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _bias_args(bias, B, V):
    if bias is None:
        return ctypes.c_void_p(0), 0
    torch = _torch()
    if isinstance(bias, torch.Tensor) and bias.dim() == 2 and bias.stride(1) == 1:
        # a column slice of a [B, V] bias keeps its row stride
        if not bias.is_cuda or bias.dtype != torch.float32:
            raise FlashSampleError("FS_ERR_INVALID_ARG", "bias must be a float32 CUDA tensor (no CPU fallback)")
        return ctypes.c_void_p(bias.data_ptr()), bias.stride(0)
    ptr = _dev(bias, "bias", torch.float32, 1)
    return ptr, 0


def _outs(B, device, out):
    torch = _torch()
    if out is not None:
        return out
    return (torch.empty(B, dtype=torch.int64, device=device),
            torch.empty(B, dtype=torch.float32, device=device))


def sample(h, W, temp, seed, step, bias=None, out=None, stream=None):
    """Fused LM-head exact sample of one decode step.

    h: bf16 [B, d], W: bf16 [V, d], temp: fp32 [B] (CUDA tensors); bias:
    optional fp32 [B, V] or [V].  Returns (ids int64 [B], max fp32 [B]) on
    the device, enqueued on the current stream.
    """
    torch = _torch()
    B, d = h.shape
    V = W.shape[0]
    ids, mx = _outs(B, h.device, out)
    bptr, bstride = _bias_args(bias, B, V)
    check(library().fs_sample_ex(_dev(h, "h", torch.bfloat16, 2), _dev(W, "W", torch.bfloat16, 2),
                                 B, d, V, _dev(temp, "temp", torch.float32, 1), bptr, bstride,
                                 seed, step, _dev(ids, "out_ids", torch.int64),
                                 _dev(mx, "out_max", torch.float32), _stream_ptr(stream)))
    return ids, mx


def debug_fused_logits(h, W, temp, seed, step, bias=None, stream=None):
    """``sample`` with the fused kernel's logit inspection store switched on:
    returns (ids, max, logits fp32 [B, V]), the logits being the values the
    fused kernel's epilogue read (accumulator + bias, before temperature and
    noise).  Same kernel family, instantiation and launch as ``sample``."""
    torch = _torch()
    B, d = h.shape
    V = W.shape[0]
    ids, mx = _outs(B, h.device, None)
    logits = torch.full((B, V), float("nan"), dtype=torch.float32, device=h.device)
    bptr, bstride = _bias_args(bias, B, V)
    check(library().fs_debug_fused_logits(_dev(h, "h", torch.bfloat16, 2), _dev(W, "W", torch.bfloat16, 2),
                                          B, d, V, _dev(temp, "temp", torch.float32, 1), bptr, bstride,
                                          seed, step, _dev(ids, "out_ids", torch.int64),
                                          _dev(mx, "out_max", torch.float32), _dev(logits, "logits_out"),
                                          _stream_ptr(stream)))
    return ids, mx, logits


def sample_unfused(h, W, temp, seed, step, bias=None, logits_out=None, out=None, stream=None):
    """The unfused comparison pipeline (GEMM -> fp32 logits in HBM -> softmax
    -> sample).  Same inputs / outputs as ``sample``; ``logits_out`` (fp32
    [B, V] CUDA tensor) receives the logits if given."""
    torch = _torch()
    B, d = h.shape
    V = W.shape[0]
    ids, mx = _outs(B, h.device, out)
    bptr, bstride = _bias_args(bias, B, V)
    lptr = _dev(logits_out, "logits_out", torch.float32) if logits_out is not None else ctypes.c_void_p(0)
    check(library().fs_sample_unfused(_dev(h, "h", torch.bfloat16, 2), _dev(W, "W", torch.bfloat16, 2),
                                      B, d, V, _dev(temp, "temp", torch.float32, 1), bptr, bstride,
                                      seed, step, _dev(ids, "out_ids", torch.int64),
                                      _dev(mx, "out_max", torch.float32), lptr, _stream_ptr(stream)))
    return ids, mx


def sample_ex(*args, **kwargs):
    """Alias of ``sample`` (the bias argument maps to fs_sample_ex)."""
    return sample(*args, **kwargs)


def combine_shards(shard_max, shard_ids, out=None, stream=None):
    """Tensor-parallel final step: per row, the best of the R shards' (max,
    id) pairs (shard_max fp32 [R, B], shard_ids int64 [R, B], device).
    Returns (ids int64 [B], max fp32 [B])."""
    torch = _torch()
    R, B = shard_max.shape
    ids, mx = _outs(B, shard_max.device, out)
    check(library().fs_combine_shards(
        _dev(shard_max, "shard_max", torch.float32, 2), _dev(shard_ids, "shard_ids", torch.int64, 2), R, B,
        _dev(ids, "out_ids"), _dev(mx, "out_max"), _stream_ptr(stream)))
    return ids, mx


def tp_exchange(local_max, local_ids, group=None):
    """Exchange each rank's per-row (max, id) with the other ranks of
    ``group``: 8 bytes per row per rank (the fp32 max's bits and the id as
    int32), one all_gather.  Returns (all_max fp32 [R, B], all_ids int64
    [R, B]) on the inputs' device.  Communication plumbing only (NCCL for CUDA
    tensors, gloo for host tensors); the sample itself is computed by the
    library's kernels."""
    torch = _torch()
    import torch.distributed as dist
    R = dist.get_world_size(group)
    packed = torch.stack([local_max.contiguous().view(torch.int32), local_ids.to(torch.int32)], dim=1)
    parts = [torch.empty_like(packed) for _ in range(R)]
    dist.all_gather(parts, packed, group=group)
    allp = torch.stack(parts)
    return allp[..., 0].contiguous().view(torch.float32), allp[..., 1].to(torch.int64)


def sample_tp(h, W_shard, v_begin, temp, seed, step, group=None, bias_shard=None, stream=None):
    """Tensor-parallel sample: this rank holds vocabulary rows [v_begin,
    v_begin + W_shard.shape[0]); it samples its shard with global ids, the
    ranks exchange the per-row (max, id) pairs, and the combine picks the
    winner.  Every rank returns the same (ids, max), equal to sample() over
    the whole vocabulary."""
    torch = _torch()
    B = h.shape[0]
    cm = torch.empty(B, dtype=torch.float32, device=h.device)
    ci = torch.empty(B, dtype=torch.int64, device=h.device)
    local = sample_chunked(h, W_shard, v_begin, temp, seed, step, cm, ci, True, True, bias_chunk=bias_shard,
                           stream=stream)
    all_max, all_ids = tp_exchange(local[1], local[0], group=group)
    return combine_shards(all_max, all_ids, stream=stream)


def sample_topk(h, W, temp, seed, step, k, bias=None, out=None, stream=None):
    """Gumbel-top-k: k ids per row without replacement, best first.
    Returns (ids int64 [B, k], z fp32 [B, k]); -1 / -inf where a row has
    fewer than k choosable ids.  1 <= k <= 16, B <= 4096; k = 1 gives
    sample()'s ids and maxima."""
    torch = _torch()
    B, d = h.shape
    V = W.shape[0]
    if out is None:
        out = (torch.empty((B, k), dtype=torch.int64, device=h.device),
               torch.empty((B, k), dtype=torch.float32, device=h.device))
    ids, z = out
    bptr, bstride = _bias_args(bias, B, V)
    check(library().fs_sample_topk(
        _dev(h, "h", torch.bfloat16, 2), _dev(W, "W", torch.bfloat16, 2), B, d, V,
        _dev(temp, "temp", torch.float32, 1), bptr, bstride, seed, step, int(k),
        _dev(ids, "out_ids", torch.int64, 2), _dev(z, "out_z", torch.float32, 2), _stream_ptr(stream)))
    return ids, z


def sample_chunked(h, W_chunk, v_begin, temp, seed, step, carry_max, carry_ids, first, last,
                   bias_chunk=None, out=None, stream=None, serial=False):
    """One chunk [v_begin, v_begin + W_chunk.shape[0]) of the grouped online
    variant; updates (carry_max, carry_ids) in place and, when ``last``,
    returns (ids, max)."""
    torch = _torch()
    B, d = h.shape
    v_end = v_begin + W_chunk.shape[0]
    flags = (FS_CHUNK_FIRST if first else 0) | (FS_CHUNK_LAST if last else 0) | (FS_CHUNK_SERIAL if serial else 0)
    ids = mx = None
    if last:
        ids, mx = _outs(B, h.device, out)
    bptr, bstride = _bias_args(bias_chunk, B, W_chunk.shape[0])
    check(library().fs_sample_chunked(
        _dev(h, "h", torch.bfloat16, 2), _dev(W_chunk, "W_chunk", torch.bfloat16, 2), B, d,
        v_begin, v_end, _dev(temp, "temp", torch.float32, 1), bptr, bstride, seed, step,
        _dev(carry_max, "carry_max", torch.float32), _dev(carry_ids, "carry_ids", torch.int64),
        flags, _dev(ids, "out_ids") if last else ctypes.c_void_p(0),
        _dev(mx, "out_max") if last else ctypes.c_void_p(0), _stream_ptr(stream)))
    return (ids, mx) if last else None


def sample_chunked_step(h, W, bounds, temp, seed, step, carry_max, carry_ids, bias=None, out=None,
                        stream=None):
    """One whole chunked step over chunks [bounds[i], bounds[i+1]) of W in
    one C call (the per-chunk calls of ``sample_chunked`` issued from C).
    ``bounds`` may be a list or an int64 numpy array (kept by the caller to
    reuse).  Returns (ids, max)."""
    torch = _torch()
    B, d = h.shape
    b = bounds if isinstance(bounds, np.ndarray) and bounds.dtype == np.int64 else np.asarray(bounds, np.int64)
    n = len(b) - 1
    if n < 1 or b[-1] != W.shape[0]:
        raise FlashSampleError("FS_ERR_INVALID_ARG", "bounds must have >= 2 entries ending at W.shape[0]")
    ids, mx = _outs(B, h.device, out)
    bptr, bstride = _bias_args(bias, B, W.shape[0])
    check(library().fs_sample_chunked_step(
        _dev(h, "h", torch.bfloat16, 2), _dev(W, "W", torch.bfloat16, 2), B, d, ctypes.c_void_p(b.ctypes.data), n,
        _dev(temp, "temp", torch.float32, 1), bptr, bstride, seed, step,
        _dev(carry_max, "carry_max", torch.float32), _dev(carry_ids, "carry_ids", torch.int64),
        _dev(ids, "out_ids"), _dev(mx, "out_max"), _stream_ptr(stream)))
    return ids, mx


def sample_chunked_early(h, W_chunk, v_begin, temp, seed, step, carry_max, carry_ids, first, last,
                         h_norms, rest_w_norm, rest_bias_max, done, bias_chunk=None, out=None, stream=None,
                         serial=False):
    """sample_chunked with online early finalization: ``h_norms`` fp32 [B]
    (row_norms(h)), ``rest_w_norm`` / ``rest_bias_max`` host floats bounding
    the later chunks, ``done`` a device int32 [1] flag: the first call
    resets it, a chunk sets it once every row's carried best can no longer be
    overtaken, and later calls that see it set skip their work.  ``serial``
    launches the call without overlapping the previous one."""
    torch = _torch()
    B, d = h.shape
    v_end = v_begin + W_chunk.shape[0]
    flags = (FS_CHUNK_FIRST if first else 0) | (FS_CHUNK_LAST if last else 0) | (FS_CHUNK_SERIAL if serial else 0)
    ids = mx = None
    if last:
        ids, mx = _outs(B, h.device, out)
    bptr, bstride = _bias_args(bias_chunk, B, W_chunk.shape[0])
    check(library().fs_sample_chunked_early(
        _dev(h, "h", torch.bfloat16, 2), _dev(W_chunk, "W_chunk", torch.bfloat16, 2), B, d,
        v_begin, v_end, _dev(temp, "temp", torch.float32, 1), bptr, bstride, seed, step,
        _dev(carry_max, "carry_max", torch.float32), _dev(carry_ids, "carry_ids", torch.int64),
        flags, _dev(h_norms, "h_norms", torch.float32, 1), float(rest_w_norm), float(rest_bias_max),
        _dev(done, "done", torch.int32), _dev(ids, "out_ids") if last else ctypes.c_void_p(0),
        _dev(mx, "out_max") if last else ctypes.c_void_p(0), _stream_ptr(stream)))
    return (ids, mx) if last else None


def row_norms(X, out=None, stream=None):
    """fp32 Euclidean norms of the rows of a bf16 [n, d] device matrix."""
    torch = _torch()
    n, d = X.shape
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=X.device)
    check(library().fs_row_norms(_dev(X, "X", torch.bfloat16, 2), n, d, _dev(out, "out", torch.float32, 1),
                                 _stream_ptr(stream)))
    return out


def chunk_rest_norms(W, bounds, stream=None):
    """Host list: for chunk i of ``bounds`` (n_chunks + 1 row offsets into W),
    the largest row norm of W after the chunk (0 for the last).  Synchronizes."""
    torch = _torch()
    b = np.ascontiguousarray(np.asarray(bounds, dtype=np.int64))
    n = len(b) - 1
    rest = np.zeros(max(n, 0), dtype=np.float32)
    check(library().fs_chunk_rest_norms(_dev(W, "W", torch.bfloat16, 2), W.shape[1],
                                        ctypes.c_void_p(b.ctypes.data), n,
                                        ctypes.c_void_p(rest.ctypes.data), _stream_ptr(stream)))
    return [float(x) for x in rest]


def sample_host(h_host, W, temp_host, seed, step, bias=None, out_ids=None, out_max=None,
                stream=None):
    """End-to-end call with host buffers (numpy arrays or CPU tensors; pinned
    memory recommended): h_host bf16 bits uint16 [B, d] (or a bf16 tensor),
    temp_host fp32 [B]; W (and bias) stay on the device.  Copies in, samples,
    copies out and synchronizes.  Returns host (ids int64 [B], max fp32 [B])."""
    torch = _torch()

    def host_ptr(a, name):
        if isinstance(a, np.ndarray):
            if not a.flags["C_CONTIGUOUS"]:
                raise FlashSampleError("FS_ERR_INVALID_ARG", f"{name} must be C-contiguous")
            return ctypes.c_void_p(a.ctypes.data)
        if isinstance(a, torch.Tensor) and not a.is_cuda and a.is_contiguous():
            return ctypes.c_void_p(a.data_ptr())
        raise FlashSampleError("FS_ERR_INVALID_ARG", f"{name} must be a contiguous host array")

    B, d = h_host.shape
    V = W.shape[0]
    if out_ids is None:
        out_ids = np.empty(B, dtype=np.int64)
    if out_max is None:
        out_max = np.empty(B, dtype=np.float32)
    bptr, bstride = _bias_args(bias, B, V)
    check(library().fs_sample_host(host_ptr(h_host, "h_host"), _dev(W, "W", torch.bfloat16, 2),
                                   B, d, V, host_ptr(temp_host, "temp_host"), bptr, bstride,
                                   seed, step, host_ptr(out_ids, "out_ids"),
                                   host_ptr(out_max, "out_max"), _stream_ptr(stream)))
    return out_ids, out_max


def debug_noise(seed, step, row0, n_rows, v0, n_vocab, stream=None):
    """(words uint32-as-int32 [n_rows, n_vocab], gumbel fp32 [n_rows, n_vocab])
    exactly as the sampling kernels draw them."""
    torch = _torch()
    words = torch.empty((n_rows, n_vocab), dtype=torch.int32, device="cuda")
    g = torch.empty((n_rows, n_vocab), dtype=torch.float32, device="cuda")
    check(library().fs_debug_noise(seed, step, row0, n_rows, v0, n_vocab,
                                   ctypes.c_void_p(words.data_ptr()), ctypes.c_void_p(g.data_ptr()),
                                   _stream_ptr(stream)))
    return words, g


def set_path(path):
    check(library().fs_set_path(path))


def debug_set_fault(kind):
    """Host-side fault injection (FS_FAULT_NONE / _ALLOC / _LAUNCH)."""
    check(library().fs_debug_set_fault(int(kind)))


def set_launch_overlap(enable):
    """Overlapped (programmatic dependent) launch of one-shot calls: True by
    default; False where the kernel enqueued just before a call may write W."""
    check(library().fs_set_launch_overlap(1 if enable else 0))


def path_for_batch(B):
    return library().fs_path_for_batch(B)


def path_for_chunks(B, V_chunk, step_chunks):
    return library().fs_path_for_chunks(B, V_chunk, step_chunks)


def workspace_reserve(B, V, stream=None):
    check(library().fs_workspace_reserve(B, V, _stream_ptr(stream)))


def profile_events(start, stop):
    """Record torch.cuda.Event ``start``/``stop`` around the fused kernel of
    every later call on this thread (None, None to stop)."""
    if start is None:
        check(library().fs_profile_events(None, None))
    else:
        check(library().fs_profile_events(ctypes.c_void_p(start.cuda_event),
                                          ctypes.c_void_p(stop.cuda_event)))


def debug_wait_timeout(timeout_ns, stream=None):
    check(library().fs_debug_wait_timeout(timeout_ns, _stream_ptr(stream)))


def device_error():
    code = ctypes.c_int(0)
    check(library().fs_device_error(ctypes.byref(code)))
    return code.value
