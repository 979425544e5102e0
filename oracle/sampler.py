"""Exact Gumbel-max categorical sampling from the LM head, written as its plain
definition in fp64.

Source: FlashSampling: Fast and Memory-Efficient Exact Sampling.  The summary
page (sections TL;DR, Key claims, Method) and the arXiv abstract state what is
computed:

* the LM head forms logits = h W^T for a batch of rows h (B x d) and the
  vocabulary matrix W (V x d) (summary page, Method, op (1));
* temperature scaling and Gumbel noise turn sampling from softmax(logits / T)
  into an argmax of logits / T + g with g ~ Gumbel(0, 1) iid (summary page,
  Key claims, second item; Method, op (3));
* the argmax decomposes over any partition of the vocabulary, so per-tile
  (max, argmax) pairs followed by a small reduction give the same sample
  (abstract; summary page, Method);
* the grouped online (chunked) and sharded variants are exact by the same
  hierarchical factorization (abstract; summary page, Method, last paragraph).

The method reaches, up to rounding order, a result with a plain definition, so
this module is that definition written out over the full vocabulary: no tiling
is needed to compute it.  ``sample_partitioned``, ``sample_chunked`` and
``combine`` restate the decomposition itself so the tests can check that it
really is exact.

Readings of points the pages leave open (each also listed in the design notes):

* noise: Philox-4x32-10 with key (seed mod 2^32, seed >> 32) and counter
  (v >> 2, b, step mod 2^32, step >> 32); output word (v & 3) is the 32-bit draw
  for row b, vocabulary id v (v is always the GLOBAL vocabulary id);
* uniform: u = ((x >> 9) + 1/2) * 2^-23, i.e. the odd multiples of 2^-24 in
  (0, 1) -- exact in fp32 and fp64, never 0 or 1;
* Gumbel: g = -log(-log u);
* temperature T per row: z = logits / T + g; T == 0 means greedy (z = logits,
  no noise); T < 0 or NaN makes the row invalid (id -1);
* bias (optional, fp32) is added to the logits before the division by T;
* total order for the argmax: a larger z wins, equal z goes to the smaller v;
  NaN and -inf never win; a row with no candidate returns id -1 and max -inf.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).
"""

from dataclasses import dataclass

import numpy as np

from .philox import philox4x32_10

_MASK32 = 0xFFFFFFFF
NO_ID = -1


# --------------------------------------------------------------------------
# Inputs: bf16 decode and the logits (summary page, Method, op (1)).
# --------------------------------------------------------------------------

def bf16_to_f64(bits):
    """Decode raw bf16 bit patterns (uint16) to fp64.

    bf16 is the upper half of an IEEE binary32, so the value is exactly the
    float32 whose high 16 bits are ``bits`` and whose low 16 bits are zero;
    the widening to fp64 is exact.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):      # NaN patterns stay NaN
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def logits(h_bits, W_bits, bias=None):
    """ell[b, v] = sum_k h[b, k] * W[v, k] (+ bias[b, v]) in fp64.

    ``h_bits``: uint16 [B, d]; ``W_bits``: uint16 [V, d]; ``bias``: float32
    [B, V], [V] (one vector shared by every row) or None.  bf16 -> fp64 is
    exact and every product of two bf16 values is exact in fp64; only the
    sum rounds (fp64 matmul, relative error ~1e-16 of sum |h W|).
    """
    h = bf16_to_f64(h_bits)
    W = bf16_to_f64(W_bits)
    ell = h @ W.T
    if bias is not None:
        ell = ell + np.asarray(bias, dtype=np.float32).astype(np.float64)
    return ell


# --------------------------------------------------------------------------
# Noise: counter-based uniform and the Gumbel transform.
# --------------------------------------------------------------------------

def philox_words(seed, step, rows, vocab_ids):
    """The 32-bit draw x[r, j] for row ``rows[r]`` and vocabulary id
    ``vocab_ids[j]``: word (v & 3) of Philox-4x32-10 under key
    (seed lo, seed hi) at counter (v >> 2, b, step lo, step hi)."""
    seed = int(seed)
    step = int(step)
    b = np.asarray(rows, dtype=np.uint64).reshape(-1, 1)
    v = np.asarray(vocab_ids, dtype=np.uint64).reshape(-1)
    # One generator call serves the four ids that share v >> 2.
    quad, col = np.unique(v >> np.uint64(2), return_inverse=True)
    c0 = quad.astype(np.uint32).reshape(1, -1)
    c1 = b.astype(np.uint32)
    c2 = np.uint32(step & _MASK32)
    c3 = np.uint32((step >> 32) & _MASK32)
    words = philox4x32_10(c0, c1, c2, c3, seed & _MASK32, (seed >> 32) & _MASK32)
    stacked = np.stack(words, axis=0)                       # [4, R, n_quads]
    lane = (v & np.uint64(3)).astype(np.int64)
    return stacked[lane, :, col.reshape(-1)].T              # [R, n]


def uniform_from_word(x):
    """u = ((x >> 9) + 1/2) * 2^-23: the top 23 bits of x, centred in their
    cell.  Values are (2k + 1) * 2^-24, k in [0, 2^23), so u lies in
    [2^-24, 1 - 2^-24] and is exact in fp64 (and fp32)."""
    x = np.asarray(x, dtype=np.uint32)
    return ((x >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def gumbel_from_uniform(u):
    """Standard Gumbel quantile: g = -log(-log u)."""
    return -np.log(-np.log(u))


def gumbel(seed, step, rows, vocab_ids):
    """Gumbel(0, 1) noise g[r, j] for (rows[r], vocab_ids[j]) at this step."""
    return gumbel_from_uniform(uniform_from_word(philox_words(seed, step, rows, vocab_ids)))


# --------------------------------------------------------------------------
# Scores and the total-order argmax.
# --------------------------------------------------------------------------

def scores(ell, temp, seed, step, rows, vocab_ids):
    """Perturbed scores z = ell / T + g per row (summary page, Method: logits,
    then "Gumbel/temperature scaling").

    ``ell``: fp64 [R, n]; ``temp``: the R temperatures (fp32 inputs).
    T == 0 -> z = ell (greedy); T < 0 or NaN -> the row is all NaN (invalid).
    """
    ell = np.asarray(ell, dtype=np.float64)
    T = np.asarray(temp, dtype=np.float32).astype(np.float64).reshape(-1, 1)
    z = ell / np.where(T > 0, T, 1.0) + gumbel(seed, step, rows, vocab_ids)
    z = np.where(T == 0, ell, z)
    z = np.where((T < 0) | np.isnan(T), np.nan, z)
    return z


def argmax_total_order(z, vocab_ids):
    """Row-wise argmax of z under the total order: larger z wins, equal z goes
    to the smaller vocabulary id; NaN and -inf never win.

    Returns (ids int64 [R], zmax fp64 [R]); a row without a candidate gives
    (-1, -inf).  ``vocab_ids`` (increasing) labels the columns of z.
    """
    z = np.asarray(z, dtype=np.float64)
    vocab_ids = np.asarray(vocab_ids, dtype=np.int64)
    valid = ~np.isnan(z) & (z > -np.inf)
    masked = np.where(valid, z, -np.inf)
    if z.shape[1] == 0:
        return (np.full(z.shape[0], NO_ID, dtype=np.int64),
                np.full(z.shape[0], -np.inf))
    j = np.argmax(masked, axis=1)          # first maximum = smallest id
    any_valid = valid.any(axis=1)
    ids = np.where(any_valid, vocab_ids[j], NO_ID).astype(np.int64)
    zmax = np.where(any_valid, masked[np.arange(z.shape[0]), j], -np.inf)
    return ids, zmax


def top2_gap(z):
    """z_(1) - z_(2): the gap between the two largest valid scores of each row
    (+inf when a row has fewer than two valid scores)."""
    z = np.asarray(z, dtype=np.float64)
    valid = ~np.isnan(z) & (z > -np.inf)
    masked = np.where(valid, z, -np.inf)
    if z.shape[1] < 2:
        return np.full(z.shape[0], np.inf)
    top2 = np.partition(masked, -2, axis=1)[:, -2:]     # [second, first]
    first, second = top2[:, 1], top2[:, 0]
    with np.errstate(invalid="ignore"):
        gap = np.where(first == second, 0.0, first - second)
    return np.where(second > -np.inf, gap, np.inf)


def combine(a, b):
    """Merge two (ids, zmax) partial results under the same total order.

    Associative and commutative, with identity (-1, -inf); this is the "small
    reduction over tiles" and the cross-chunk / cross-shard merge.
    """
    ia, za = np.asarray(a[0], dtype=np.int64), np.asarray(a[1], dtype=np.float64)
    ib, zb = np.asarray(b[0], dtype=np.int64), np.asarray(b[1], dtype=np.float64)
    take_b = (ib != NO_ID) & ((ia == NO_ID) | (zb > za) | ((zb == za) & (ib < ia)))
    return np.where(take_b, ib, ia), np.where(take_b, zb, za)


# --------------------------------------------------------------------------
# Samplers.
# --------------------------------------------------------------------------

@dataclass
class Sample:
    ids: np.ndarray      # int64 [R]: sampled vocabulary id, -1 if none
    zmax: np.ndarray     # fp64 [R]: winning perturbed score (max logit when greedy)
    gap: np.ndarray      # fp64 [R]: top-two perturbed-score gap of the row


def _row_select(h_bits, temp, bias, rows):
    B = h_bits.shape[0]
    rows = np.arange(B) if rows is None else np.asarray(rows, dtype=np.int64)
    h_r = h_bits[rows]
    t_r = np.asarray(temp, dtype=np.float32)[rows]
    if bias is not None:
        bias = np.asarray(bias, dtype=np.float32)
        bias = bias[rows] if bias.ndim == 2 else bias
    return rows, h_r, t_r, bias


def sample(h_bits, W_bits, temp, seed, step, bias=None, rows=None, vocab_offset=0):
    """One-shot exact sample over the whole vocabulary (rows of W).

    ``rows`` restricts the work to a subset of the batch (row indices keep
    their own noise counters).  ``vocab_offset`` is the global id of W's first
    row (used by the chunked sampler; W then holds only the chunk).
    """
    rows, h_r, t_r, bias_r = _row_select(h_bits, temp, bias, rows)
    V = W_bits.shape[0]
    vocab_ids = np.arange(vocab_offset, vocab_offset + V, dtype=np.int64)
    return sample_from_logits(logits(h_r, W_bits, bias_r), t_r, seed, step, rows, vocab_ids)


def sample_from_logits(ell, temp, seed, step, rows, vocab_ids):
    """The sample given the fp64 logits (bias included) of ``rows``: scores,
    then the total-order argmax and the top-two gap.  ``temp`` holds the
    temperatures of ``rows``; ``vocab_ids`` labels the columns of ``ell``.
    ``sample`` is logits followed by this; a caller that already holds the
    logits of many rows (they do not depend on the step) can reuse them."""
    z = scores(ell, temp, seed, step, rows, vocab_ids)
    ids, zmax = argmax_total_order(z, vocab_ids)
    return Sample(ids, zmax, top2_gap(z))


def sample_partitioned(h_bits, W_bits, temp, seed, step, parts, bias=None, rows=None):
    """The partition-argmax decomposition (abstract; summary page, Key claims):
    one (max, argmax) per part of the vocabulary, then the small reduction.

    ``parts`` is a list of integer index arrays that partition range(V), in the
    order they are folded into the result.  Scores are the same fp64 values as
    in ``sample``; only the grouping of the argmax changes.
    """
    rows, h_r, t_r, bias_r = _row_select(h_bits, temp, bias, rows)
    ell = logits(h_r, W_bits, bias_r)
    acc = (np.full(len(rows), NO_ID, dtype=np.int64), np.full(len(rows), -np.inf))
    for part in parts:
        part = np.sort(np.asarray(part, dtype=np.int64))
        z = scores(ell[:, part], t_r, seed, step, rows, part)
        acc = combine(acc, argmax_total_order(z, part))
    return acc


def sample_chunked(h_bits, W_bits, temp, seed, step, bounds, bias=None, rows=None):
    """Grouped online variant (summary page, Method, last paragraph): the
    vocabulary is streamed as contiguous chunks [bounds[i], bounds[i+1]) and a
    per-row (max, argmax) carry is merged after each chunk.  Each chunk sees
    only its own rows of W (and bias columns) and the global vocabulary ids."""
    rows_sel, _, _, _ = _row_select(h_bits, temp, None, rows)
    carry = (np.full(len(rows_sel), NO_ID, dtype=np.int64), np.full(len(rows_sel), -np.inf))
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        b_chunk = None
        if bias is not None:
            bias = np.asarray(bias, dtype=np.float32)
            b_chunk = bias[..., lo:hi]
        s = sample(h_bits, W_bits[lo:hi], temp, seed, step, bias=b_chunk, rows=rows,
                   vocab_offset=lo)
        carry = combine(carry, (s.ids, s.zmax))
    return carry



# --------------------------------------------------------------------------
# Early finalization of the grouped online variant (summary page, Method,
# last paragraph: the streaming sampler "can finalize the sample as soon as
# later tiles can no longer overtake the running maximum").  The pages give
# no bound; the reading here is Cauchy-Schwarz on the logit plus the largest
# Gumbel value the uniform grid can produce.
# --------------------------------------------------------------------------

# Largest Gumbel draw: u = 1 - 2^-24, the top of the uniform grid.
G_MAX = float(-np.log(-np.log(1.0 - 2.0 ** -24)))


def row_norms(bits):
    """Euclidean norm of every row of a bf16 matrix, fp64."""
    x = bf16_to_f64(bits)
    return np.sqrt(np.sum(x * x, axis=1))


def score_upper_bound(h_norm, w_norm_max, bias_max, temp):
    """Upper bound of z = (logit + bias) / T + g over a set of vocabulary rows
    whose largest norm is w_norm_max and largest bias is bias_max:
    |logit| <= |h| |W_v| (Cauchy-Schwarz), g <= G_MAX.  Greedy rows (T = 0)
    have no noise; rows with an invalid T never take a sample (-inf)."""
    T = np.asarray(temp, dtype=np.float32).astype(np.float64)
    lim = np.asarray(h_norm, dtype=np.float64) * w_norm_max + bias_max
    ub = np.where(T > 0, lim / np.where(T > 0, T, 1.0) + G_MAX, lim)
    return np.where((T < 0) | np.isnan(T), -np.inf, ub)


def sample_chunked_early(h_bits, W_bits, temp, seed, step, bounds, bias=None):
    """The grouped online variant with early finalization: after each chunk,
    a row is final when its carried maximum is at least the upper bound of
    every later chunk (rows with an invalid T always are); when all rows are
    final the remaining chunks are not read.  Returns ((ids, zmax), number of
    chunks read).  The sample equals the one-shot sample."""
    B = h_bits.shape[0]
    hn = row_norms(h_bits)
    wn = row_norms(W_bits)
    T = np.asarray(temp, dtype=np.float32)
    carry = (np.full(B, NO_ID, dtype=np.int64), np.full(B, -np.inf))
    n = len(bounds) - 1
    for i in range(n):
        lo, hi = bounds[i], bounds[i + 1]
        b_chunk = None if bias is None else np.asarray(bias, np.float32)[..., lo:hi]
        s = sample(h_bits, W_bits[lo:hi], temp, seed, step, bias=b_chunk, vocab_offset=lo)
        carry = combine(carry, (s.ids, s.zmax))
        rest_lo = hi
        if rest_lo >= bounds[-1]:
            return carry, i + 1
        w_rest = wn[rest_lo:].max()
        if bias is None:
            b_rest = np.zeros(B)
        else:
            bb = np.asarray(bias, np.float32).astype(np.float64)
            b_rest = bb[..., rest_lo:].max(axis=-1) * np.ones(B)
        ub = score_upper_bound(hn, w_rest, b_rest, T)
        invalid = (T < 0) | np.isnan(T)
        final = invalid | ((carry[0] != NO_ID) & (carry[1] >= ub))
        if final.all():
            return carry, i + 1
    return carry, n
