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
    // fast path: 8 whole counter quads, every id in range
    const uint32_t q0 = static_cast<uint32_t>(vg0 >> 2);
    const int32_t id0 = static_cast<int32_t>(vg0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 w = noise_words(s.key, q0 + q, s.row, s.step_lo, s.step_hi);
      const int j = 4 * q;
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
