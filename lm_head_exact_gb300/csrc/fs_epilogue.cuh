// Row-major sampling epilogue shared by the batch-major tensor-core kernels:
// one thread owns one batch row and scans 32 consecutive vocabulary columns
// of its accumulator (already in registers) in increasing id order.
//
// Per element: z = logit * (1/T) + g with g the Gumbel draw of (row, id)
// (FlashSampling: Fast and Memory-Efficient Exact Sampling -- summary page,
// "Method": noise added in-tile, only the per-row (max, argmax) kept).
#pragma once

#include "fs_internal.h"

namespace fs {

struct RowScan {
  PhiloxKey key;
  uint32_t row;          // batch row b (noise counter word 1)
  uint32_t step_lo, step_hi;
  float inv_t;
  bool greedy;
  const float* bias_row;  // bias + b * stride (nullable)
};

__device__ __forceinline__ void keep_best(Best& best, float z, int32_t id) {
  if (z > best.z) {      // ids rise along the scan: strict > keeps the smaller id on ties
    best.z = z;
    best.id = id;
  }
}

template <bool kHasBias>
__device__ __forceinline__ float perturbed(const RowScan& s, float logit, uint32_t word, int64_t v_local) {
  if constexpr (kHasBias) logit += __ldg(s.bias_row + v_local);
  return s.greedy ? logit : fmaf(logit, s.inv_t, gumbel_from_word(word));
}

// Columns [v0, v0 + 32) of the call's W (local ids), global ids v_offset + v0 ...
template <bool kHasBias>
__device__ __forceinline__ void scan32(const uint32_t (&r)[32], int64_t v0, int64_t v_local_end, int64_t v_offset,
                                       const RowScan& s, Best& best) {
  const int64_t vg0 = v_offset + v0;
  if (v0 + 32 <= v_local_end && (vg0 & 3) == 0) {
    // fast path: 8 whole counter quads, every id in range.  A quad whose
    // largest scaled logit plus the largest Gumbel value cannot beat its row's
    // best cannot change the row's result (fmaf is monotone in each of its
    // scaled and added operands, and the best is replaced only by a strictly
    // larger score); when that holds on every lane, the warp skips the quad's
    // noise.  Rows whose logits sit far above the rest (large biases, peaked
    // distributions) skip most quads; the samples are the same.
    const uint32_t q0 = static_cast<uint32_t>(vg0 >> 2);
    const int32_t id0 = static_cast<int32_t>(vg0);
    const unsigned lanes = __activemask();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = 4 * q;
      float l0 = __uint_as_float(r[j + 0]), l1 = __uint_as_float(r[j + 1]);
      float l2 = __uint_as_float(r[j + 2]), l3 = __uint_as_float(r[j + 3]);
      if constexpr (kHasBias) {
        l0 += __ldg(s.bias_row + v0 + j + 0);
        l1 += __ldg(s.bias_row + v0 + j + 1);
        l2 += __ldg(s.bias_row + v0 + j + 2);
        l3 += __ldg(s.bias_row + v0 + j + 3);
      }
      const float lmax = fmaxf(fmaxf(l0, l1), fmaxf(l2, l3));
      const float bound = s.greedy ? lmax : fmaf(lmax, s.inv_t, kGumbelMax);
      if (!__any_sync(lanes, bound > best.z)) continue;
      const uint4 w = noise_words(s.key, q0 + q, s.row, s.step_lo, s.step_hi);
      keep_best(best, perturbed<kHasBias>(s, __uint_as_float(r[j + 0]), w.x, v0 + j + 0), id0 + j + 0);
      keep_best(best, perturbed<kHasBias>(s, __uint_as_float(r[j + 1]), w.y, v0 + j + 1), id0 + j + 1);
      keep_best(best, perturbed<kHasBias>(s, __uint_as_float(r[j + 2]), w.z, v0 + j + 2), id0 + j + 2);
      keep_best(best, perturbed<kHasBias>(s, __uint_as_float(r[j + 3]), w.w, v0 + j + 3), id0 + j + 3);
    }
    return;
  }
  // ragged or unaligned chunk: per-id counter quads and bounds
  uint4 w = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (v0 + j < v_local_end) {
      const int64_t vg = vg0 + j;
      if (j == 0 || (vg & 3) == 0) w = noise_words(s.key, static_cast<uint32_t>(vg >> 2), s.row, s.step_lo, s.step_hi);
      keep_best(best, perturbed<kHasBias>(s, __uint_as_float(r[j]), word_of(w, static_cast<uint32_t>(vg & 3)), v0 + j),
                static_cast<int32_t>(vg));
    }
  }
}

}  // namespace fs

namespace fs {

// ---------------------------------------------------------------------------
// Gumbel-top-k: a running list of the K best (z, id) of one row, best first
// under the same total order as the sample (a larger z, then a smaller id);
// empty entries are (-inf, kNoId).  -inf and NaN never enter.
// ---------------------------------------------------------------------------
template <int K>
struct TopList {
  float z[K];
  int32_t id[K];
};

template <int K>
__device__ __forceinline__ void topk_init(TopList<K>& t) {
#pragma unroll
  for (int i = 0; i < K; ++i) {
    t.z[i] = -INFINITY;
    t.id[i] = kNoId;
  }
}

// Insert (z, id) if it beats the last entry: walk the list, swapping the
// carried candidate in wherever it beats the entry there.
template <int K>
__device__ __forceinline__ void topk_offer(TopList<K>& t, float z, int32_t id) {
  if (!(z > -INFINITY) || !beats(z, id, t.z[K - 1], t.id[K - 1])) return;
  float cz = z;
  int32_t ci = id;
#pragma unroll
  for (int i = 0; i < K; ++i) {
    const bool take = beats(cz, ci, t.z[i], t.id[i]);
    const float oz = t.z[i];
    const int32_t oi = t.id[i];
    t.z[i] = take ? cz : oz;
    t.id[i] = take ? ci : oi;
    cz = take ? oz : cz;
    ci = take ? oi : ci;
  }
}

// scan32 with a top-K list instead of the running best.  Pass 1 computes the
// 32 scores as scan32 does, overwriting r with them, and marks those that beat
// the list's last entry at the start of the chunk (ids rise along the scan,
// so an equal score never beats an entry already in the list); pass 2 -- rare
// once the list is full -- offers each marked score to the list.
template <bool kHasBias, int K>
__device__ __forceinline__ void scan32_topk(uint32_t (&r)[32], int64_t v0, int64_t v_local_end, int64_t v_offset,
                                            const RowScan& s, TopList<K>& list) {
  const float thr = list.z[K - 1];
  const int64_t vg0 = v_offset + v0;
  uint32_t mask = 0;
  if (v0 + 32 <= v_local_end && (vg0 & 3) == 0) {
    const uint32_t q0 = static_cast<uint32_t>(vg0 >> 2);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 w = noise_words(s.key, q0 + q, s.row, s.step_lo, s.step_hi);
      const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * q + e;
        const float z = perturbed<kHasBias>(s, __uint_as_float(r[j]), words[e], v0 + j);
        r[j] = __float_as_uint(z);
        mask |= static_cast<uint32_t>(z > thr) << j;
      }
    }
  } else {
    uint4 w = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (v0 + j < v_local_end) {
        const int64_t vg = vg0 + j;
        if (j == 0 || (vg & 3) == 0) w = noise_words(s.key, static_cast<uint32_t>(vg >> 2), s.row, s.step_lo, s.step_hi);
        const float z = perturbed<kHasBias>(s, __uint_as_float(r[j]), word_of(w, static_cast<uint32_t>(vg & 3)), v0 + j);
        r[j] = __float_as_uint(z);
        mask |= static_cast<uint32_t>(z > thr) << j;
      }
    }
  }
  while (mask != 0) {
    const int j = __ffs(mask) - 1;
    mask &= mask - 1;
    uint32_t zb = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) zb = i == j ? r[i] : zb;   // r[j] without local memory
    topk_offer(list, __uint_as_float(zb), static_cast<int32_t>(vg0 + j));
  }
}

}  // namespace fs
