// Cross-part reduction: the "small reduction over tiles" that turns the
// per-(row, part) (max, argmax) candidates into the sampled id
// (FlashSampling: Fast and Memory-Efficient Exact Sampling -- arXiv abstract;
// summary page, "Method").  For the grouped online (chunked) variant it also
// merges the carried per-row (max, argmax) and writes the updated carry.
//
// Also holds the noise-inspection kernel that exposes the exact Philox words
// and Gumbel values every sampling kernel uses, for parity tests.
#include <algorithm>

#include "fs_finish.cuh"
#include "fs_internal.h"
#include "fs_sm100.cuh"

namespace fs {
namespace {

constexpr int kReduceThreads = 256;
constexpr int kRowsPerBlock = kReduceThreads / 32;

__global__ void __launch_bounds__(kReduceThreads)
reduce_kernel(Finish f, int64_t B) {
  const int lane = threadIdx.x & 31;
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (b >= B) return;
  const Partial* row = f.partials + b * f.n_parts;
  Best best = best_none();
  for (int i = lane; i < f.n_parts; i += 32) {
    const Partial q = row[i];
    Best c;
    c.z = q.z;
    c.id = q.id;
    best = combine(best, c);
  }
  best = warp_combine(best);
  if (lane == 0) write_row(f, b, best);
}

// Host-buffer entry point: copy h (bf16x8 packets) and the temperatures from
// mapped pinned host memory into device staging.  Launched before the fused
// kernel, which starts as its programmatic dependent: the fused kernel's
// prologue and first W loads overlap this copy.
__global__ void __launch_bounds__(256)
copy_in_kernel(const uint4* __restrict__ h_src, uint4* __restrict__ h_dst, int64_t n16, const float* __restrict__ t_src,
               float* __restrict__ t_dst, int64_t B) {
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) h_dst[i] = h_src[i];
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < B; i += stride) t_dst[i] = t_src[i];
}

// Cross-shard combine of the tensor-parallel variant: row b's result is the
// best of the R shards' (max, id) pairs under the total order (id -1 = none).
__global__ void __launch_bounds__(kReduceThreads)
combine_shards_kernel(const float* __restrict__ shard_max, const int64_t* __restrict__ shard_ids, int64_t R, int64_t B,
                      int64_t* __restrict__ out_ids, float* __restrict__ out_max) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * kReduceThreads + threadIdx.x;
  if (b >= B) return;
  Best best = best_none();
  for (int64_t r = 0; r < R; ++r) {
    const int64_t id = shard_ids[r * B + b];
    if (id < 0 || id >= kNoId) continue;
    Best c;
    c.z = shard_max[r * B + b];
    c.id = static_cast<int32_t>(id);
    best = combine(best, c);
  }
  out_ids[b] = best.id == kNoId ? -1 : static_cast<int64_t>(best.id);
  out_max[b] = best.id == kNoId ? -INFINITY : best.z;
}

// Gumbel-top-k merge, one 256-thread block per row over the row's n_lists
// lists of K candidates each (one per CTA, each already sorted best first;
// ids unique across lists, empty entries kNoId).  Lane l of warp w holds list
// 32 w + l in registers.  Level 1: each warp merges its 32 lists -- k rounds
// of a warp argmax over the list heads, the owner of the winning head drops
// it -- into a sorted list of k in shared memory.  Level 2: warp 0 merges the
// 8 warps' lists the same way.  The output is the row's k best in order.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

template <int K>
__device__ __forceinline__ void drop_head(float (&lz)[K], int32_t (&li)[K]) {
#pragma unroll
  for (int i = 0; i + 1 < K; ++i) {
    lz[i] = lz[i + 1];
    li[i] = li[i + 1];
  }
  lz[K - 1] = -INFINITY;
  li[K - 1] = kNoId;
}

// k rounds of a warp-wide merge of the lanes' sorted lists; calls
// emit(j, winner) on every lane.
template <int K, class Emit>
__device__ __forceinline__ void warp_merge(float (&lz)[K], int32_t (&li)[K], int k, Emit emit) {
  for (int j = 0; j < k; ++j) {
    Best h;
    h.z = lz[0];
    h.id = li[0];
    if (h.id == kNoId) h = best_none();
    const Best w = warp_combine(h);
    emit(j, w);
    if (w.id != kNoId && li[0] == w.id) drop_head(lz, li);
  }
}

template <int K>
__global__ void __launch_bounds__(kMergeThreads)
topk_merge_kernel(const Partial* __restrict__ partials, int n_lists, int k, int64_t* __restrict__ out_ids,
                  float* __restrict__ out_z) {
  __shared__ Best level1[kMergeWarps][K];
  pdl_launch_dependents();      // the next call's kernel may start its W prefetch
  pdl_wait();                   // launched as a dependent of the kernel that wrote the partials
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t b = blockIdx.x;
  float lz[K];
  int32_t li[K];
  const bool has_list = static_cast<int>(threadIdx.x) < n_lists;
  const Partial* mine = partials + (b * n_lists + threadIdx.x) * K;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const Partial c = has_list ? mine[j] : Partial{-INFINITY, kNoId};
    lz[j] = c.z;
    li[j] = c.id;
  }
  warp_merge(lz, li, k, [&](int j, Best w) {
    if (lane == 0) level1[warp][j] = w;
  });
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const Best c = (lane < kMergeWarps && j < k) ? level1[lane][j] : best_none();
      lz[j] = c.z;
      li[j] = c.id;
    }
    warp_merge(lz, li, k, [&](int j, Best w) {
      if (lane == 0) {
        out_ids[b * k + j] = w.id == kNoId ? -1 : static_cast<int64_t>(w.id);
        out_z[b * k + j] = w.id == kNoId ? -INFINITY : w.z;
      }
    });
  }
}

__global__ void debug_noise_kernel(uint64_t seed, uint64_t step, int64_t row0, int64_t n_rows,
                                   int64_t v0, int64_t n_vocab, uint32_t* words, float* gumbel) {
  const int64_t n = n_rows * n_vocab;
  const PhiloxKey key{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / n_vocab;
    const int64_t v = v0 + (i - r * n_vocab);
    const uint4 w4 = noise_words(key, static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(row0 + r),
                                 static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32));
    const uint32_t w = word_of(w4, static_cast<uint32_t>(v & 3));
    if (words != nullptr) words[i] = w;
    if (gumbel != nullptr) gumbel[i] = gumbel_from_word(w);
  }
}

// Waits on an mbarrier that nothing ever arrives on, with a short limit: the
// bounded wait must give up, flag the device error word and return, leaving
// the context usable.  Exercises the failure path of the tensor-core kernels'
// waits without faulting or hanging the GPU.
__global__ void debug_wait_kernel(int* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    abort_flag = 0;
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) sm100::mbar_wait_ns(&bar, 0, err, &abort_flag, timeout_ns);
}

}  // namespace

cudaError_t launch_debug_wait(int* err, uint64_t timeout_ns, cudaStream_t stream) {
  debug_wait_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_reduce(const Finish& f, int64_t B, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((B + kRowsPerBlock - 1) / kRowsPerBlock);
  reduce_kernel<<<blocks, kReduceThreads, 0, stream>>>(f, B);
  return cudaGetLastError();
}

cudaError_t launch_combine_shards(const float* shard_max, const int64_t* shard_ids, int64_t R, int64_t B,
                                  int64_t* out_ids, float* out_max, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int64_t blocks = (B + kReduceThreads - 1) / kReduceThreads;
  if (blocks > 2147483647) return cudaErrorInvalidValue;
  combine_shards_kernel<<<static_cast<unsigned>(blocks), kReduceThreads, 0, stream>>>(shard_max, shard_ids, R, B,
                                                                                      out_ids, out_max);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(const Partial* partials, int n_lists, int K, int64_t B, int k, int64_t* out_ids,
                              float* out_z, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  if (k < 1 || k > K || n_lists > kMergeThreads || B > 2147483647) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(B));
  switch (K) {
    case 4: return launch_kernel(topk_merge_kernel<4>, grid, dim3(kMergeThreads), 0, stream, true, partials, n_lists, k, out_ids, out_z);
    case 8: return launch_kernel(topk_merge_kernel<8>, grid, dim3(kMergeThreads), 0, stream, true, partials, n_lists, k, out_ids, out_z);
    case 16: return launch_kernel(topk_merge_kernel<16>, grid, dim3(kMergeThreads), 0, stream, true, partials, n_lists, k, out_ids, out_z);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_copy_in(const void* h_src, void* h_dst, int64_t h_bytes, const float* t_src, float* t_dst, int64_t B,
                           cudaStream_t stream) {
  const int64_t n16 = h_bytes / 16;
  const int64_t blocks = std::min<int64_t>(128, std::max<int64_t>(1, (std::max(n16, B) + 255) / 256));
  copy_in_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint4*>(h_src),
                                                                     static_cast<uint4*>(h_dst), n16, t_src, t_dst, B);
  return cudaGetLastError();
}

cudaError_t launch_debug_noise(uint64_t seed, uint64_t step, int64_t row0, int64_t n_rows,
                               int64_t v0, int64_t n_vocab, uint32_t* words, float* gumbel,
                               cudaStream_t stream) {
  const int64_t n = n_rows * n_vocab;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n + 255) / 256;
  debug_noise_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(
      seed, step, row0, n_rows, v0, n_vocab, words, gumbel);
  return cudaGetLastError();
}

}  // namespace fs
