// The "small reduction over tiles" that finishes the sample (FlashSampling:
// Fast and Memory-Efficient Exact Sampling -- arXiv abstract; summary page,
// "Method"), done inside the fused kernels:
//
//   1. every CTA pushes its best candidate per batch row into that row's
//      packed 64-bit key with atomicMax (the key order is the total order of
//      candidates, so the result does not depend on which CTA comes first);
//   2. the CTA that finishes last -- counted with an atomic ticket -- reads
//      and zeroes every key, merges the chunked variant's carry and writes the
//      outputs, then zeroes the ticket for the next user of these keys.
//
// No CTA ever waits for another CTA of its grid: there is no spin on a flag,
// only the ticket.  Every launch owns its keys and ticket while it runs (the
// host gives each chunk of a chunked step its own set, rotating), so the
// CTAs push without waiting for the previous launch; only the last CTA waits
// for the previous kernel of the stream to complete (griddepcontrol.wait; a
// no-op without a programmatic launch) before it reads the carry the
// previous chunk wrote.  Hence a chunk completes only after the previous one
// has, and the CTAs of consecutive chunks overlap freely.
#pragma once

#include "fs_internal.h"

namespace fs {

// Row b can no longer be overtaken by the later chunks: its best perturbed
// score is at least their upper bound (Cauchy-Schwarz on the logit, the
// largest bias, the largest Gumbel value), with a margin for fp32 rounding.
__device__ __forceinline__ bool row_final(const Finish& f, int64_t b, Best best) {
  const RowTemp rt = row_temp(f.temp[b]);
  if (rt.mode == kRowInvalid) return true;
  if (best.id == kNoId) return false;
  const float lim = f.h_norms[b] * f.rest_w_norm + f.rest_bias_max;
  const float ub = rt.mode == kRowGreedy ? lim : fmaf(lim, rt.inv_t, kGumbelMax);
  return best.z >= ub + 1e-4f * fabsf(ub) + 1e-3f;
}

// Final best of row b -> carry (chunked variant) and outputs; returns the
// merged best.
__device__ __forceinline__ Best write_row(const Finish& f, int64_t b, Best best) {
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
  return best;
}

__device__ __forceinline__ void push_candidate(const Finish& f, int64_t b, Best c) {
  if (c.id != kNoId) atomicMax(f.keys + b, pack_key(c.z, c.id));
}

// Barrier over the 128 / 256 epilogue threads (named barrier 1) that also
// ANDs a predicate over them.
template <int kCount>
__device__ __forceinline__ bool named_bar1_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "n"(kCount)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ bool cta_bar_and(bool pred) { return __syncthreads_and(pred) != 0; }

// Called by the n participating threads (index tid) of every CTA after they
// pushed all of this CTA's candidates.  `bar_and(p)` synchronizes exactly
// those threads and returns the AND of their p; `flag` is a shared-memory
// int.  The last CTA of the grid writes rows [0, B) and leaves keys and
// ticket at zero.  kEarly = false compiles out the early-finalization flag
// (callers that never set Finish::done and whose register count matters).
// The flag needs no fence of its own: a later chunk reads the carry only
// after its dependency wait (or in stream order).
template <bool kEarly = true, class BarAnd>
__device__ __forceinline__ void finish_grid(const Finish& f, int64_t B, int tid, int n, int* flag, BarAnd bar_and) {
  __threadfence();
  bar_and(true);
  if (tid == 0) {
    const unsigned total = gridDim.x * gridDim.y * gridDim.z;
    *flag = atomicAdd(f.counter, 1u) == total - 1;
  }
  bar_and(true);
  if (*flag) {
    pdl_wait();                    // the previous chunk's carry (and its completion)
    __threadfence();
    bool all_final = true;
    for (int64_t b = tid; b < B; b += n) {
      const Best best = write_row(f, b, unpack_key(atomicExch(f.keys + b, 0ull)));
      if (kEarly && f.done != nullptr) all_final = all_final && row_final(f, b, best);
    }
    if (kEarly && f.done != nullptr) {
      all_final = bar_and(all_final);
      if (tid == 0) *f.done = all_final ? 1 : 0;
    }
    if (tid == 0) atomicExch(f.counter, 0u);
  }
}

// Early finalization: the *done flag of a chunk after the first, read at
// kernel entry.  The flag was reset before the first chunk and is only ever
// set within the step, by a finished chunk after its carry writes, so a 1 is
// valid for every later chunk.  With a programmatic dependent launch the
// previous chunk may set it while this grid's CTAs start, so different CTAs
// of one grid may read different values: every CTA must stay correct alone.
// A relaxed load is enough: the decision only chooses whether to compute, and
// the carry is read after the dependency wait (or in stream order).
__device__ __forceinline__ bool early_done(const Finish& f) {
  if (f.done == nullptr || !f.carry_in) return false;
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f.done) : "memory");
  return v != 0;
}

// The same, taken once per CTA: thread 0 reads the flag and every thread of
// the CTA gets its value through `slot` (a shared-memory int).  Called by all
// threads.
__device__ __forceinline__ bool early_done_cta(const Finish& f, int* slot) {
  if (f.done == nullptr || !f.carry_in) return false;
  if (threadIdx.x == 0) *slot = early_done(f) ? 1 : 0;
  __syncthreads();
  return *slot != 0;
}

// A CTA that saw the flag set loads and computes nothing but still takes its
// ticket in the cross-CTA finish (with no candidate), so that the grid's last
// CTA -- whichever it is -- merges the carry and writes the flag and, on the
// last chunk, the outputs.  Called by all threads of the CTA before any
// warp-role split; `flag` is a shared-memory int.
__device__ __forceinline__ void early_skip_cta(const Finish& f, int64_t B, bool pdl, int* flag) {
  (void)pdl;
  pdl_launch_dependents();
  finish_grid(f, B, threadIdx.x, blockDim.x, flag, cta_bar_and);
}

}  // namespace fs
