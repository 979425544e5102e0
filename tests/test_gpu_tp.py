"""GPU side of the tensor-parallel variant (summary page, Method, third
paragraph): per-shard samples with global ids, then the cross-shard combine.

Every box here has one GPU, so the R shards are sampled one after another
on it (each with FS_CHUNK_FIRST | FS_CHUNK_LAST, as a rank would); the
combine must give the whole-vocabulary sample bit for bit.  The
exchange step itself is tested over gloo on CPU (test_sharded_gloo.py) and,
with NCCL at world size 1, through sample_tp below.
"""

import os
import socket
import subprocess
import sys

import numpy as np
import pytest

from _helpers import compare, to_device
from oracle import sampler
from lm_head_exact_gb300 import synthetic

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _problem(B, V, d, seed, w_std=0.05):
    rng = np.random.default_rng(seed)
    h = synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = synthetic.bf16_bits((rng.standard_normal((V, d)) * w_std).astype(np.float32))
    temps = rng.uniform(0.3, 1.5, size=B).astype(np.float32)
    temps[::7] = 0.0
    return h, W, temps


@pytest.mark.parametrize("B", [1, 16, 200])
@pytest.mark.parametrize("bounds", [[0, 2048, 4099], [0, 1, 1500, 4099], [0, 512, 1024, 1536, 2048, 2560, 3072, 3584, 4099]])
def test_emulated_shards_combine_to_the_one_shot_sample(fs, torch_cuda, B, bounds):
    torch = torch_cuda
    V, d = bounds[-1], 256
    h, W, temp = _problem(B, V, d, seed=B + len(bounds))
    bias = synthetic.leading_spike_bias(B, V, V, 3.0)
    hd, Wd, td, bd = to_device(h, torch), to_device(W, torch), to_device(temp, torch), to_device(bias, torch)
    R = len(bounds) - 1
    shard_max = torch.empty((R, B), dtype=torch.float32, device="cuda")
    shard_ids = torch.empty((R, B), dtype=torch.int64, device="cuda")
    for r, (lo, hi) in enumerate(zip(bounds[:-1], bounds[1:])):
        cm = torch.empty(B, device="cuda")
        ci = torch.empty(B, dtype=torch.int64, device="cuda")
        fs.sample_chunked(hd, Wd[lo:hi], lo, td, 5, 6, cm, ci, True, True, bias_chunk=bd[:, lo:hi],
                          out=(shard_ids[r], shard_max[r]))
    ids, mx = fs.combine_shards(shard_max, shard_ids)
    one_ids, one_mx = fs.sample(hd, Wd, td, 5, 6, bias=bd)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), one_ids.cpu().numpy())
    np.testing.assert_array_equal(mx.cpu().numpy(), one_mx.cpu().numpy())
    compare(ids.cpu().numpy(), mx.cpu().numpy(), sampler.sample(h, W, temp, 5, 6, bias=bias), what=f"tp B={B}")


def test_combine_edge_cases(fs, torch_cuda):
    torch = torch_cuda
    B = 5
    shard_max = torch.tensor([[1.0, 2.0, -np.inf, 0.5, 7.0], [1.0, 3.0, -np.inf, 0.5, 7.0]], device="cuda")
    shard_ids = torch.tensor([[9, 4, -1, 10, 3], [2, 8, -1, -1, 3000]], dtype=torch.int64, device="cuda")
    ids, mx = fs.combine_shards(shard_max, shard_ids)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), [2, 8, -1, 10, 3])     # ties -> smaller id; -1 never wins
    np.testing.assert_array_equal(mx.cpu().numpy(), [1.0, 3.0, -np.inf, 0.5, 7.0])
    empty = torch.empty((0, B), dtype=torch.float32, device="cuda")
    ids, mx = fs.combine_shards(empty, torch.empty((0, B), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert np.all(ids.cpu().numpy() == -1) and np.all(mx.cpu().numpy() == -np.inf)


_NCCL_WORLD1 = r"""
import os, sys
import numpy as np, torch, torch.distributed as dist
sys.path.insert(0, {root!r})
from lm_head_exact_gb300 import binding as fs, synthetic
dist.init_process_group("nccl", init_method="tcp://127.0.0.1:{port}", rank=0, world_size=1)
torch.cuda.set_device(0)
rng = np.random.default_rng(3)
B, V, d = 24, 5000, 128
h = torch.from_numpy(synthetic.bf16_bits(rng.standard_normal((B, d)).astype(np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
W = torch.from_numpy(synthetic.bf16_bits((rng.standard_normal((V, d)) * 0.05).astype(np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
t = torch.ones(B, device="cuda")
ids, mx = fs.sample_tp(h, W, 0, t, 11, 2)
ref_ids, ref_mx = fs.sample(h, W, t, 11, 2)
torch.cuda.synchronize()
assert torch.equal(ids, ref_ids) and torch.equal(mx, ref_mx)
dist.destroy_process_group()
print("tp-ok")
"""


def test_sample_tp_over_nccl_world_size_one(fs, torch_cuda):
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    r = subprocess.run([sys.executable, "-c", _NCCL_WORLD1.format(root=ROOT, port=port)], capture_output=True,
                       text=True, timeout=240, env=env)
    assert r.returncode == 0 and "tp-ok" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
