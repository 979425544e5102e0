// The "small reduction over tiles" that finishes the sample (FlashSampling:
// Fast and Memory-Efficient Exact Sampling -- arXiv abstract; summary page,
// "Method"), done inside the fused kernels:
//
//   1. every CTA pushes its best candidate per batch row into that row's
//      packed 64-bit key with atomicMax (the key order is the total order of
//      candidates, so the result does not depend on which CTA comes first);
//   2. the CTA that finishes last -- counted with an atomic ticket -- reads
//      and zeroes every key, merges the chunked variant's carry and writes the
//      outputs, then zeroes the ticket for the next call.
//
// No CTA ever waits for another: there is no spin on a flag, only the ticket.
#pragma once

#include "fs_internal.h"

namespace fs {

// Final best of row b -> carry (chunked variant) and outputs.
__device__ __forceinline__ void write_row(const Finish& f, int64_t b, Best best) {
  if (f.carry_max != nullptr) {
    if (f.carry_in) {
      const int64_t cid = f.carry_ids[b];
      if (cid >= 0) {
        Best c;
        c.z = f.carry_max[b];
        c.id = static_cast<int32_t>(cid);
        best = combine(best, c);
      }
    }
    f.carry_max[b] = best.id == kNoId ? -INFINITY : best.z;
    f.carry_ids[b] = best.id == kNoId ? -1 : static_cast<int64_t>(best.id);
  }
  if (f.write_out) {
    f.out_ids[b] = best.id == kNoId ? -1 : static_cast<int64_t>(best.id);
    f.out_max[b] = best.id == kNoId ? -INFINITY : best.z;
  }
}

__device__ __forceinline__ void push_candidate(const Finish& f, int64_t b, Best c) {
  if (c.id != kNoId) atomicMax(f.keys + b, pack_key(c.z, c.id));
}

// Called by the n participating threads (index tid) of every CTA after they
// pushed all of this CTA's candidates.  `bar()` synchronizes exactly those
// threads; `flag` is a shared-memory int.  The last CTA of the grid writes
// rows [0, B) and leaves keys and ticket at zero.
template <class Bar>
__device__ __forceinline__ void finish_grid(const Finish& f, int64_t B, int tid, int n, int* flag, Bar bar) {
  __threadfence();
  bar();
  if (tid == 0) {
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    *flag = atomicAdd(f.counter, 1u) == total - 1;
  }
  bar();
  if (*flag) {
    __threadfence();
    for (int64_t b = tid; b < B; b += n) write_row(f, b, unpack_key(atomicExch(f.keys + b, 0ull)));
    if (tid == 0) atomicExch(f.counter, 0u);
  }
}

}  // namespace fs
