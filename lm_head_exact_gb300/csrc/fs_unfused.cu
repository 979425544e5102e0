// The unfused comparison pipeline: what a decode step does when sampling is
// NOT fused into the LM head (FlashSampling: Fast and Memory-Efficient Exact
// Sampling -- summary page, "Method", ops (1)-(4); "Key claims", first item):
//
//   (1) logits = h W^T written to HBM as fp32 [B, V]   (tensor-core GEMM: the
//       batch-major kernel in store-logits mode),
//   (2) softmax over V                                  (softmax_rows_kernel: reads
//       the logits twice, writes fp32 probabilities [B, V]),
//   (3)+(4) temperature / Gumbel and the sample          (sample_rows_kernel: reads
//       the probabilities again).
//
// It draws the same Philox noise as the fused kernels and samples by the
// exponential race argmax_v p_v / E_v with E_v = -log u_v, which orders
// candidates exactly like argmax_v (logit_v / T + g_v) with g_v = -log E_v,
// so its ids match the fused path's up to rounding.  It exists to measure the
// HBM traffic (about 20 B x V bytes per step) that fusion removes.
#include <algorithm>

#include "fs_internal.h"

namespace fs {
namespace {

constexpr int kRowThreads = 512;
constexpr int kMaxSplits = 256;   // ranges per row at most

struct MaxSum {
  float m, s;
};

__device__ __forceinline__ MaxSum ms_combine(MaxSum a, MaxSum b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return MaxSum{-INFINITY, 0.0f};
  return MaxSum{m, a.s * __expf(a.m - m) + b.s * __expf(b.m - m)};
}

__device__ __forceinline__ MaxSum ms_warp(MaxSum acc) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    MaxSum o{__shfl_xor_sync(0xffffffffu, acc.m, off), __shfl_xor_sync(0xffffffffu, acc.s, off)};
    acc = ms_combine(acc, o);
  }
  return acc;
}

// Rows are split into S contiguous ranges (a multiple of 4 ids each, so a
// noise quad never straddles two ranges) and each (range, row) gets a block,
// so that even a handful of rows spreads over the whole GPU.
__device__ __forceinline__ void split_range(int64_t V, int S, int s, int64_t* lo, int64_t* hi) {
  const int64_t per = ((V + S - 1) / S + 3) & ~int64_t(3);
  *lo = min(V, static_cast<int64_t>(s) * per);
  *hi = min(V, *lo + per);
}

// (max, sum of exp) over the block, returned to every thread.
__device__ __forceinline__ MaxSum block_max_sum(MaxSum acc, MaxSum* red) {
  acc = ms_warp(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    acc = threadIdx.x < kRowThreads / 32 ? red[threadIdx.x] : MaxSum{-INFINITY, 0.0f};
    acc = ms_warp(acc);
    if (threadIdx.x == 0) red[0] = acc;
  }
  __syncthreads();
  return red[0];
}

// Softmax pass 1: the (max, sum of exp) of x = logit / T over one range of
// one row (x = logit for greedy rows, whose argmax is all that is used);
// NaN and -inf logits count as probability 0.
__global__ void __launch_bounds__(kRowThreads)
softmax_stats_kernel(const float* __restrict__ logits, MaxSum* __restrict__ part, int64_t V, int S,
                     const float* __restrict__ temp) {
  __shared__ MaxSum red[kRowThreads / 32];
  const int64_t b = blockIdx.y;
  const RowTemp rt = row_temp(temp[b]);
  const float scale = rt.mode == kRowSample ? rt.inv_t : 1.0f;
  const float* x = logits + b * V;
  int64_t lo, hi;
  split_range(V, S, blockIdx.x, &lo, &hi);
  MaxSum acc{-INFINITY, 0.0f};
  for (int64_t i = lo + threadIdx.x; i < hi; i += kRowThreads) {
    const float v = x[i] * scale;
    if (v > -INFINITY) acc = ms_combine(acc, MaxSum{v, 1.0f});
  }
  acc = block_max_sum(acc, red);
  if (threadIdx.x == 0) part[b * S + blockIdx.x] = acc;
}

// Softmax pass 2: every block combines its row's S partial sums, then writes
// the probabilities of its range (a second read of the logits).
__global__ void __launch_bounds__(kRowThreads)
softmax_norm_kernel(const float* __restrict__ logits, const MaxSum* __restrict__ part, float* __restrict__ probs,
                    int64_t V, int S, const float* __restrict__ temp) {
  __shared__ MaxSum tot;
  const int64_t b = blockIdx.y;
  if (threadIdx.x < 32) {
    MaxSum acc{-INFINITY, 0.0f};
    for (int i = threadIdx.x; i < S; i += 32) acc = ms_combine(acc, part[b * S + i]);
    acc = ms_warp(acc);
    if (threadIdx.x == 0) tot = acc;
  }
  __syncthreads();
  const RowTemp rt = row_temp(temp[b]);
  const float scale = rt.mode == kRowSample ? rt.inv_t : 1.0f;
  const float* x = logits + b * V;
  float* y = probs + b * V;
  const float inv_s = tot.s > 0.0f ? 1.0f / tot.s : 0.0f;
  int64_t lo, hi;
  split_range(V, S, blockIdx.x, &lo, &hi);
  for (int64_t i = lo + threadIdx.x; i < hi; i += kRowThreads) {
    const float v = x[i] * scale;
    y[i] = v > -INFINITY ? __expf(v - tot.m) * inv_s : 0.0f;
  }
}

// Sample pass 1: over one range of one row, argmax_v p_v / (-log u_v)
// (greedy rows: argmax_v p_v), ties to the smaller id.
__global__ void __launch_bounds__(kRowThreads)
sample_split_kernel(const float* __restrict__ probs, int64_t V, int64_t v_offset, const float* __restrict__ temp,
                    uint64_t seed, uint64_t step, Best* __restrict__ part, int S, int64_t row0) {
  __shared__ Best red[kRowThreads / 32];
  const int64_t b = blockIdx.y;
  const RowTemp rt = row_temp(temp[b]);
  const PhiloxKey key{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
  const uint32_t step_lo = static_cast<uint32_t>(step), step_hi = static_cast<uint32_t>(step >> 32);
  const float* p = probs + b * V;
  int64_t lo, hi;
  split_range(V, S, blockIdx.x, &lo, &hi);
  Best best = best_none();
  if (rt.mode != kRowInvalid) {
    // thread t handles four consecutive ids per iteration (one Philox call)
    for (int64_t q0 = lo + 4 * static_cast<int64_t>(threadIdx.x); q0 < hi; q0 += 4 * kRowThreads) {
      uint4 w = make_uint4(0, 0, 0, 0);
      for (int j = 0; j < 4 && q0 + j < hi; ++j) {
        const int64_t vg = v_offset + q0 + j;
        if (j == 0 || (vg & 3) == 0)
          w = noise_words(key, static_cast<uint32_t>(vg >> 2), static_cast<uint32_t>(row0 + b), step_lo, step_hi);
        const float pv = p[q0 + j];
        float score = pv;
        if (rt.mode == kRowSample)
          score = pv / (-logf(uniform_from_word(word_of(w, static_cast<uint32_t>(vg & 3)))));
        if (score > best.z) {           // a thread's ids rise: strict > keeps the smaller id
          best.z = score;
          best.id = static_cast<int32_t>(vg);
        }
      }
    }
  }
  best = warp_combine(best);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x < 32) {
    best = threadIdx.x < kRowThreads / 32 ? red[threadIdx.x] : best_none();
    best = warp_combine(best);
    if (threadIdx.x == 0) part[b * S + blockIdx.x] = best;
  }
}

// Sample pass 2 (one warp per row): the best of the row's S ranges; the
// reported maximum is the fused path's score logit * (1/T) + g at the winner
// (the max logit for greedy rows).
__global__ void __launch_bounds__(32)
sample_finish_kernel(const Best* __restrict__ part, int S, const float* __restrict__ logits, int64_t V,
                     int64_t v_offset, const float* __restrict__ temp, uint64_t seed, uint64_t step,
                     int64_t* __restrict__ out_ids, float* __restrict__ out_max, int64_t row0) {
  const int64_t b = blockIdx.x;
  Best best = best_none();
  for (int i = threadIdx.x; i < S; i += 32) best = combine(best, part[b * S + i]);
  best = warp_combine(best);
  if (threadIdx.x != 0) return;
  if (best.id == kNoId) {
    out_ids[b] = -1;
    out_max[b] = -INFINITY;
    return;
  }
  const RowTemp rt = row_temp(temp[b]);
  const int64_t vg = best.id;
  const float logit = logits[b * V + (vg - v_offset)];
  float z = logit;
  if (rt.mode == kRowSample) {
    const PhiloxKey key{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
    const uint4 w = noise_words(key, static_cast<uint32_t>(vg >> 2), static_cast<uint32_t>(row0 + b),
                                static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32));
    z = fmaf(logit, rt.inv_t, gumbel_from_word(word_of(w, static_cast<uint32_t>(vg & 3))));
  }
  out_ids[b] = vg;
  out_max[b] = z;
}

}  // namespace

size_t unfused_partial_bytes(int64_t B) {
  return 2 * static_cast<size_t>(std::max<int64_t>(B, 1)) * kMaxSplits * 8;
}

cudaError_t launch_unfused_tail(const Problem& p, float* logits, float* probs, void* partials, int64_t* out_ids,
                                float* out_max, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  const int64_t V = p.V_local;
  // ranges per row: about two blocks per SM over the batch, at least 16 ids
  // per thread in each range
  const int64_t want = (2 * static_cast<int64_t>(sms) + p.B - 1) / p.B;
  const int64_t cap = std::max<int64_t>(1, V / (kRowThreads * 16));
  const int S = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(want, cap), kMaxSplits)));
  MaxSum* part_ms = static_cast<MaxSum*>(partials);
  Best* part_best = reinterpret_cast<Best*>(part_ms + static_cast<size_t>(p.B) * S);
  constexpr int64_t kMaxRows = 65535;   // grid y
  for (int64_t b0 = 0; b0 < p.B; b0 += kMaxRows) {
    const int64_t nb = std::min<int64_t>(kMaxRows, p.B - b0);
    const dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(nb));
    const float* lg = logits + b0 * V;
    float* pr = probs + b0 * V;
    const float* t = p.temp + b0;
    MaxSum* pm = part_ms + b0 * S;
    Best* pb = part_best + b0 * S;
    softmax_stats_kernel<<<grid, kRowThreads, 0, stream>>>(lg, pm, V, S, t);
    softmax_norm_kernel<<<grid, kRowThreads, 0, stream>>>(lg, pm, pr, V, S, t);
    // the noise counters take the global row b0 + b
    sample_split_kernel<<<grid, kRowThreads, 0, stream>>>(pr, V, p.v_offset, t, p.seed, p.step, pb, S,
                                                          p.row_offset + b0);
    sample_finish_kernel<<<static_cast<unsigned>(nb), 32, 0, stream>>>(pb, S, lg, V, p.v_offset, t, p.seed,
                                                                       p.step, out_ids + b0, out_max + b0,
                                                                       p.row_offset + b0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace fs
