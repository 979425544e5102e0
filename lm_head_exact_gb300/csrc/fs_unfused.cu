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
#include "fs_internal.h"

namespace fs {
namespace {

constexpr int kRowThreads = 512;

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

// One block per row: probabilities of softmax(x) with x = logit / T
// (x = logit for greedy rows, whose argmax is all that is used).  NaN and
// -inf logits get probability 0.
__global__ void __launch_bounds__(kRowThreads)
softmax_rows_kernel(const float* __restrict__ logits, float* __restrict__ probs, int64_t V,
                    const float* __restrict__ temp) {
  __shared__ MaxSum red[kRowThreads / 32];
  const int64_t b = blockIdx.x;
  const RowTemp rt = row_temp(temp[b]);
  const float scale = rt.mode == kRowSample ? rt.inv_t : 1.0f;
  const float* x = logits + b * V;
  float* y = probs + b * V;

  MaxSum acc{-INFINITY, 0.0f};
  for (int64_t i = threadIdx.x; i < V; i += kRowThreads) {
    const float v = x[i] * scale;
    if (v > -INFINITY) acc = ms_combine(acc, MaxSum{v, 1.0f});
  }
  acc = ms_warp(acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    acc = threadIdx.x < kRowThreads / 32 ? red[threadIdx.x] : MaxSum{-INFINITY, 0.0f};
    acc = ms_warp(acc);
    if (threadIdx.x == 0) red[0] = acc;
  }
  __syncthreads();
  const MaxSum tot = red[0];
  const float inv_s = tot.s > 0.0f ? 1.0f / tot.s : 0.0f;
  for (int64_t i = threadIdx.x; i < V; i += kRowThreads) {
    const float v = x[i] * scale;
    y[i] = v > -INFINITY ? __expf(v - tot.m) * inv_s : 0.0f;
  }
}

// One block per row: argmax_v p_v / (-log u_v) (greedy rows: argmax_v p_v),
// ties to the smaller id; the reported maximum is the fused path's score
// logit * (1/T) + g at the winner (the max logit for greedy rows).
__global__ void __launch_bounds__(kRowThreads)
sample_rows_kernel(const float* __restrict__ probs, const float* __restrict__ logits, int64_t V,
                   int64_t v_offset, const float* __restrict__ temp, uint64_t seed, uint64_t step,
                   int64_t* __restrict__ out_ids, float* __restrict__ out_max) {
  __shared__ Best red[kRowThreads / 32];
  const int64_t b = blockIdx.x;
  const RowTemp rt = row_temp(temp[b]);
  const PhiloxKey key{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
  const uint32_t step_lo = static_cast<uint32_t>(step), step_hi = static_cast<uint32_t>(step >> 32);
  const float* p = probs + b * V;
  Best best = best_none();
  if (rt.mode != kRowInvalid) {
    // thread t handles four consecutive ids per iteration (one Philox call)
    for (int64_t q0 = 4 * static_cast<int64_t>(threadIdx.x); q0 < V; q0 += 4 * kRowThreads) {
      uint4 w = make_uint4(0, 0, 0, 0);
      for (int j = 0; j < 4 && q0 + j < V; ++j) {
        const int64_t vg = v_offset + q0 + j;
        if (j == 0 || (vg & 3) == 0)
          w = noise_words(key, static_cast<uint32_t>(vg >> 2), static_cast<uint32_t>(b), step_lo, step_hi);
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
    if (threadIdx.x == 0) {
      if (best.id == kNoId) {
        out_ids[b] = -1;
        out_max[b] = -INFINITY;
      } else {
        const int64_t vg = best.id;
        const float logit = logits[b * V + (vg - v_offset)];
        float z = logit;
        if (rt.mode == kRowSample) {
          const uint4 w = noise_words(key, static_cast<uint32_t>(vg >> 2), static_cast<uint32_t>(b), step_lo, step_hi);
          z = fmaf(logit, rt.inv_t, gumbel_from_word(word_of(w, static_cast<uint32_t>(vg & 3))));
        }
        out_ids[b] = vg;
        out_max[b] = z;
      }
    }
  }
}

}  // namespace

cudaError_t launch_unfused_tail(const Problem& p, float* logits, float* probs, int64_t* out_ids,
                                float* out_max, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  const unsigned rows = static_cast<unsigned>(p.B);
  softmax_rows_kernel<<<rows, kRowThreads, 0, stream>>>(logits, probs, p.V_local, p.temp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sample_rows_kernel<<<rows, kRowThreads, 0, stream>>>(probs, logits, p.V_local, p.v_offset, p.temp, p.seed,
                                                       p.step, out_ids, out_max);
  return cudaGetLastError();
}

}  // namespace fs
