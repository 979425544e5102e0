"""Seeded synthetic inputs for the fused LM-head sampler.

This module only draws inputs: it holds none of the sampler's arithmetic, and
both the CUDA path and the CPU oracle receive identical arrays from it.  No
dataset or trained weight is used anywhere: the tensors stand in for the LM
heads of Llama-3-8B, Qwen3-8B and Llama-3-70B by SHAPE only (the FlashSampling
pages evaluate on such models in vLLM but publish no weights or inputs).

Recipe (also stated in the design notes):

* normals are drawn in fp32 with numpy's SFC64 generator; W is drawn in blocks
  of ``W_BLOCK_ROWS`` rows, block i from ``SeedSequence(seed, spawn_key=(i,))``,
  so the result does not depend on how many threads draw it, and a smaller V is
  a prefix of a larger one;
* h is drawn row by row from one stream, so a smaller batch is a prefix of a
  larger one;
* values are scaled by their standard deviation in fp32 and rounded to bf16
  (round to nearest, ties to even); arrays hold the raw bf16 bits (uint16);
* seeds: h = 0, W = 1, temperatures = 2, bias = 3; Philox sampling seed 1234.
"""

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

W_BLOCK_ROWS = 1024
SEED_H, SEED_W, SEED_TEMP, SEED_BIAS = 0, 1, 2, 3
SAMPLING_SEED = 1234


def bf16_bits(x):
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits.
    Inputs here are finite normals, so no NaN handling is needed."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits):
    """Widen bf16 bits to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_rows_bf16(seed, rows, cols, std):
    """[rows, cols] bf16 bits of N(0, std^2), one stream row after row."""
    g = np.random.Generator(np.random.SFC64(seed))
    x = g.standard_normal((rows, cols), dtype=np.float32)
    x *= np.float32(std)
    return bf16_bits(x)


def normal_blocks_bf16(seed, rows, cols, std, threads=None):
    """[rows, cols] bf16 bits of N(0, std^2), drawn in fixed row blocks with
    independent child seeds (thread-count independent)."""
    out = np.empty((rows, cols), dtype=np.uint16)
    nblk = (rows + W_BLOCK_ROWS - 1) // W_BLOCK_ROWS

    def draw(i):
        lo, hi = i * W_BLOCK_ROWS, min(rows, (i + 1) * W_BLOCK_ROWS)
        g = np.random.Generator(np.random.SFC64(np.random.SeedSequence(seed, spawn_key=(i,))))
        x = g.standard_normal((W_BLOCK_ROWS, cols), dtype=np.float32)[: hi - lo]
        x *= np.float32(std)
        out[lo:hi] = bf16_bits(x)

    threads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(draw, range(nblk)))
    return out


@dataclass
class Workload:
    """One synthetic LM-head sampling problem (all arrays on the host)."""
    name: str
    h: np.ndarray                 # uint16 [B, d]  bf16 bits, row-major
    W: np.ndarray                 # uint16 [V, d]  bf16 bits, row-major
    temp: np.ndarray              # float32 [B]
    bias: np.ndarray = None       # float32 [B, V] or None
    seed: int = SAMPLING_SEED
    steps: tuple = (0,)
    chunks: tuple = ()            # vocabulary chunk counts (chunked variant)
    notes: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.h.shape[0]

    @property
    def d(self):
        return self.h.shape[1]

    @property
    def V(self):
        return self.W.shape[0]


# Shapes of the five workloads; batch sizes are the sweep points.
SHAPES = {
    "tiny": dict(d=256, V=4096, batches=(4,)),
    "llama3_8b": dict(d=4096, V=128256, batches=(1, 2, 4, 8, 16, 32, 64)),
    "qwen3_8b": dict(d=4096, V=151936, batches=(128, 256, 512, 1024)),
    "llama3_70b": dict(d=8192, V=128256, batches=(1, 8, 64, 256)),
    "chunked": dict(d=4096, V=128256, batches=(1, 32, 256)),
}


def tiny():
    """d=256, V=4096, B=4; h and W ~ N(0, 0.02^2) from one stream seeded 0
    (h first, then W); per-row T = 0, 0.5, 1.0, 1.5; step 0."""
    g = np.random.Generator(np.random.SFC64(0))
    h = bf16_bits(g.standard_normal((4, 256), dtype=np.float32) * np.float32(0.02))
    W = bf16_bits(g.standard_normal((4096, 256), dtype=np.float32) * np.float32(0.02))
    temp = np.array([0.0, 0.5, 1.0, 1.5], dtype=np.float32)
    return Workload("tiny", h, W, temp, steps=(0,))


def temperatures(kind, B):
    """Per-row temperatures of a workload."""
    if kind == "qwen3_8b":
        g = np.random.Generator(np.random.SFC64(SEED_TEMP))
        t = g.uniform(0.3, 1.5, size=B).astype(np.float32)
        n_greedy = int(round(0.05 * B))
        t[g.permutation(B)[:n_greedy]] = 0.0
        return t
    return np.ones(B, dtype=np.float32)


def spike_bias(B, V, n_spikes=16, height=8.0):
    """Dense fp32 [B, V] bias: +height at n_spikes distinct random ids per row
    (seed 3), zero elsewhere -- peaked rows that stress near ties."""
    g = np.random.Generator(np.random.SFC64(SEED_BIAS))
    bias = np.zeros((B, V), dtype=np.float32)
    for b in range(B):
        bias[b, g.choice(V, size=n_spikes, replace=False)] = np.float32(height)
    return bias


def leading_spike_bias(B, V, v_hi, height, rows=None):
    """Dense fp32 [B, V] bias for the early-finalization cases: one +height
    spike per selected row (all rows by default) at a random id below v_hi
    (seed 3), zero elsewhere -- rows whose winner sits in the first chunk."""
    g = np.random.Generator(np.random.SFC64(SEED_BIAS))
    bias = np.zeros((B, V), dtype=np.float32)
    ids = g.integers(0, v_hi, size=B)
    for b in (range(B) if rows is None else rows):
        bias[b, ids[b]] = np.float32(height)
    return bias


_W_CACHE = {}


def weights(kind, V=None, d=None):
    """The W of a workload (cached per process: the large ones take seconds)."""
    shape = SHAPES[kind]
    V = V or shape["V"]
    d = d or shape["d"]
    std = 0.015 if kind == "llama3_70b" else 0.02
    key = (V, d, std)
    if key not in _W_CACHE:
        _W_CACHE[key] = normal_blocks_bf16(SEED_W, V, d, std)
    return _W_CACHE[key]


def workload(kind, B, V=None, d=None, with_bias=None):
    """Build workload ``kind`` at batch B.  ``V``/``d`` override the shape for
    reduced-size cases (W is then a prefix of the block stream)."""
    if kind == "tiny":
        return tiny()
    shape = SHAPES[kind]
    d = d or shape["d"]
    V = V or shape["V"]
    h = normal_rows_bf16(SEED_H, B, d, 1.0)
    W = weights(kind, V, d)
    temp = temperatures(kind, B)
    if with_bias is None:
        with_bias = kind == "llama3_70b"
    bias = spike_bias(B, V) if with_bias else None
    steps = {"llama3_8b": tuple(range(100))}.get(kind, tuple(range(10)))
    chunks = (8, 32) if kind == "chunked" else ()
    return Workload(kind, h, W, temp, bias, steps=steps, chunks=chunks)


def chunk_bounds(V, n_chunks):
    """Contiguous chunk boundaries [0, V/n, 2V/n, ..., V] (integer floor)."""
    return [(i * V) // n_chunks for i in range(n_chunks)] + [V]
