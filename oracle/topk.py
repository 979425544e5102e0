"""Gumbel-top-k: k samples WITHOUT replacement per row, as the plain definition
in fp64.

Source: FlashSampling: Fast and Memory-Efficient Exact Sampling.  The summary
page lists Gumbel-top-k sampling among the related work it builds on (the
Gumbel-max trick extended to k items) without describing it.  Reading taken
(also in the design notes): with the very same perturbed scores as the
sampler, z[v] = logits[v] / T + g[v] (z = logits when T == 0), the k ids with
the largest z, in decreasing z, are an ordered sample of k distinct ids drawn
without replacement from softmax(logits / T) -- each next id drawn from the
renormalized remaining mass.  Order: a larger z first, equal z -> the smaller
id first; NaN and -inf are never selected; rows with fewer than k selectable
ids are padded with id -1 and z -inf.  k = 1 is the sampler itself.

Like the one-sample case, the top-k decomposes over any partition of the
vocabulary: the top k of the union is the top k of the per-part top-k lists.
``sample_topk_partitioned`` restates that so the tests can check it.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).
"""

from dataclasses import dataclass

import numpy as np

from .sampler import NO_ID, _row_select, logits, scores


@dataclass
class TopK:
    ids: np.ndarray      # int64 [R, k]: ids in sample order, -1 padded
    z: np.ndarray        # fp64 [R, k]: their perturbed scores, -inf padded
    gap: np.ndarray      # fp64 [R, k]: distance of z[:, j] to its nearest neighbour in the order
                         #   (the (k+1)-th score included); +inf where there is none


def topk_total_order(z, vocab_ids, k):
    """The k best entries of each row of z under the total order (larger z
    first, equal z -> smaller id; NaN and -inf excluded).

    Returns (ids int64 [R, k+1], z fp64 [R, k+1]) -- one entry more than asked,
    so that callers can see the gap below the k-th -- padded with (-1, -inf).
    ``vocab_ids`` (increasing) labels the columns of z.
    """
    z = np.asarray(z, dtype=np.float64)
    vocab_ids = np.asarray(vocab_ids, dtype=np.int64)
    R, n = z.shape
    kk = k + 1
    ids = np.full((R, kk), NO_ID, dtype=np.int64)
    zz = np.full((R, kk), -np.inf)
    if n == 0:
        return ids, zz
    valid = ~np.isnan(z) & (z > -np.inf)
    key = np.where(valid, -z, np.inf)                  # ascending key = descending z; invalid last
    order = np.argsort(key, axis=1, kind="stable")     # stable: equal z keep increasing id
    m = min(kk, n)
    top = order[:, :m]
    top_valid = np.take_along_axis(valid, top, axis=1)
    ids[:, :m] = np.where(top_valid, vocab_ids[top], NO_ID)
    zz[:, :m] = np.where(top_valid, np.take_along_axis(z, top, axis=1), -np.inf)
    return ids, zz


def _gaps(zz, k):
    """Per position j < k: min(z_{j-1} - z_j, z_j - z_{j+1}) over existing
    neighbours (the (k+1)-th included), +inf for padded positions."""
    R = zz.shape[0]
    gap = np.full((R, k), np.inf)
    with np.errstate(invalid="ignore"):
        for j in range(k):
            g = np.full(R, np.inf)
            if j > 0:
                up = zz[:, j - 1] - zz[:, j]
                g = np.minimum(g, np.where(np.isfinite(up), up, np.inf))
            down = zz[:, j] - zz[:, j + 1]
            g = np.minimum(g, np.where(np.isfinite(down), down, np.inf))
            g = np.where(zz[:, j] > -np.inf, g, np.inf)
            gap[:, j] = g
    return gap


def sample_topk(h_bits, W_bits, temp, seed, step, k, bias=None, rows=None, vocab_offset=0):
    """k ids per row without replacement over the whole vocabulary (rows of W),
    with the sampler's noise (global ids in the counters)."""
    rows, h_r, t_r, bias_r = _row_select(h_bits, temp, bias, rows)
    V = W_bits.shape[0]
    vocab_ids = np.arange(vocab_offset, vocab_offset + V, dtype=np.int64)
    z = scores(logits(h_r, W_bits, bias_r), t_r, seed, step, rows, vocab_ids)
    ids, zz = topk_total_order(z, vocab_ids, k)
    return TopK(ids[:, :k], zz[:, :k], _gaps(zz, k))


def merge_topk(a, b, k):
    """Top k of the union of two (ids, z) candidate lists [R, *] (ids unique
    per row, -1 = empty) under the same total order."""
    ids = np.concatenate([np.asarray(a[0], np.int64), np.asarray(b[0], np.int64)], axis=1)
    z = np.concatenate([np.asarray(a[1], np.float64), np.asarray(b[1], np.float64)], axis=1)
    z = np.where(ids == NO_ID, -np.inf, z)
    # order by (-z, id) with the candidates' own ids (not column positions)
    key_id = np.where(ids == NO_ID, np.iinfo(np.int64).max, ids)
    R = ids.shape[0]
    out_i = np.full((R, k), NO_ID, dtype=np.int64)
    out_z = np.full((R, k), -np.inf)
    for r in range(R):
        valid = z[r] > -np.inf
        order = np.lexsort((key_id[r], -z[r]))            # primary -z, then id
        order = [j for j in order if valid[j]][:k]
        out_i[r, :len(order)] = ids[r, order]
        out_z[r, :len(order)] = z[r, order]
    return out_i, out_z


def sample_topk_partitioned(h_bits, W_bits, temp, seed, step, k, parts, bias=None):
    """The same result through a partition of the vocabulary: per-part top-k
    lists (global ids) merged pairwise.  ``parts`` = increasing boundaries
    [0, ..., V]."""
    B = h_bits.shape[0]
    acc = (np.full((B, k), NO_ID, dtype=np.int64), np.full((B, k), -np.inf))
    for lo, hi in zip(parts[:-1], parts[1:]):
        b_part = None if bias is None else np.asarray(bias, np.float32)[..., lo:hi]
        t = sample_topk(h_bits, W_bits[lo:hi], temp, seed, step, k, bias=b_part, vocab_offset=lo)
        acc = merge_topk(acc, (t.ids, t.z), k)
    return acc
