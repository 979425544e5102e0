"""Multi-process host logic on CPU (gloo, world size 2).

1. The sharded (tensor-parallel) variant's combine (summary page, Method,
   third paragraph; abstract): every rank samples its own vocabulary shard
   with the oracle -- global ids in the noise counters -- and the ranks
   exchange only (max, argmax) per row; the combined result must equal the
   one-shot sample bit for bit.  (The GPU peer-to-peer version is out of
   scope: every box here has one GPU.)
2. bench.py's N > 1 bookkeeping: the slowest rank's time is reported.
"""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    from lm_head_exact_gb300.synthetic import bf16_bits
    rng = np.random.default_rng(5)
    B, V, d = 9, 3001, 32
    h = bf16_bits(rng.standard_normal((B, d)).astype(np.float32))
    W = bf16_bits((rng.standard_normal((V, d)) * 0.3).astype(np.float32))
    temp = np.array([1.0, 0.0, 0.5, 1.5, 1.0, 0.7, 2.0, 1.0, 0.3], np.float32)
    return h, W, temp


def _sharded_worker(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import sampler
    h, W, temp = _problem()
    V = W.shape[0]
    lo, hi = rank * V // world, (rank + 1) * V // world
    s = sampler.sample(h, W[lo:hi], temp, 77, 3, vocab_offset=lo)
    ids = torch.from_numpy(s.ids)
    zmax = torch.from_numpy(s.zmax)
    all_ids = [torch.empty_like(ids) for _ in range(world)]
    all_max = [torch.empty_like(zmax) for _ in range(world)]
    dist.all_gather(all_ids, ids)
    dist.all_gather(all_max, zmax)
    acc = (np.full(len(ids), -1, np.int64), np.full(len(ids), -np.inf))
    for i, m in zip(all_ids, all_max):
        acc = sampler.combine(acc, (i.numpy(), m.numpy()))
    if rank == 0:
        np.savez(out_path, ids=acc[0], zmax=acc[1])
    dist.destroy_process_group()


def test_sharded_combine_equals_one_shot(tmp_path):
    from oracle import sampler
    out = str(tmp_path / "combined.npz")
    mp.start_processes(_sharded_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    got = np.load(out)
    h, W, temp = _problem()
    ref = sampler.sample(h, W, temp, 77, 3)
    np.testing.assert_array_equal(got["ids"], ref.ids)
    np.testing.assert_array_equal(got["zmax"], ref.zmax)


def _exchange_worker(rank, world, port, out_path):
    """The library's exchange step (binding.tp_exchange, 8 bytes per row per
    rank over gloo) carrying oracle shard samples of uneven shards."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import sampler
    from lm_head_exact_gb300 import binding
    h, W, temp = _problem()
    V = W.shape[0]
    bounds = {2: [0, 5, V], 3: [0, 5, 1400, V]}[world]
    lo, hi = bounds[rank], bounds[rank + 1]
    s = sampler.sample(h, W[lo:hi], temp, 77, 3, vocab_offset=lo)
    local_max = torch.from_numpy(s.zmax.astype(np.float32))
    all_max, all_ids = binding.tp_exchange(local_max, torch.from_numpy(s.ids))
    assert all_max.shape == (world, len(s.ids)) and all_ids.dtype == torch.int64
    acc = (np.full(len(s.ids), -1, np.int64), np.full(len(s.ids), -np.inf))
    for r in range(world):
        acc = sampler.combine(acc, (all_ids[r].numpy(), all_max[r].numpy().astype(np.float64)))
    if rank == 0:
        np.savez(out_path, ids=acc[0], zmax=acc[1])
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_tp_exchange_carries_the_shard_samples(tmp_path, world):
    from oracle import sampler
    out = str(tmp_path / "exchanged.npz")
    mp.start_processes(_exchange_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    got = np.load(out)
    h, W, temp = _problem()
    ref = sampler.sample(h, W, temp, 77, 3)
    np.testing.assert_array_equal(got["ids"], ref.ids)
    np.testing.assert_array_equal(got["zmax"], ref.zmax.astype(np.float32).astype(np.float64))


def _timing_worker(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(1.0 + rank, dist, device="cpu")
    bench.barrier(dist)
    if rank == 0:
        with open(out_path, "w") as f:
            f.write(repr(t))
    dist.destroy_process_group()


def test_bench_reports_the_slowest_rank(tmp_path):
    out = str(tmp_path / "t.txt")
    mp.start_processes(_timing_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
    assert float(open(out).read()) == 2.0


def test_max_over_ranks_without_process_group():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
