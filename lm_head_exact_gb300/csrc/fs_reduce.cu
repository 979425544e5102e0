// Cross-part reduction: the "small reduction over tiles" that turns the
// per-(row, part) (max, argmax) candidates into the sampled id
// (FlashSampling: Fast and Memory-Efficient Exact Sampling -- arXiv abstract;
// summary page, "Method").  For the grouped online (chunked) variant it also
// merges the carried per-row (max, argmax) and writes the updated carry.
//
// Also holds the noise-inspection kernel that exposes the exact Philox words
// and Gumbel values every sampling kernel uses, for parity tests.
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
