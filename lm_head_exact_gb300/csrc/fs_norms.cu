// Row norms for the early-finalization bound of the grouped online
// (chunked) variant (FlashSampling: Fast and Memory-Efficient Exact
// Sampling -- summary page, "Method", last paragraph: the sample is final
// once the later tiles can no longer overtake the running maximum).
//
// By Cauchy-Schwarz, every logit of row b in a later chunk is at most
// |h_b| * max_{v later} |W_v|; these kernels produce the two factors.
// One warp per row: 16-byte bf16x8 loads, fp32 sum of squares, sqrtf.
#include "fs_internal.h"

namespace fs {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormWarps = kNormThreads / 32;

__device__ __forceinline__ float sq_bf16x8(uint4 q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16);
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u);
    s = fmaf(lo, lo, s);
    s = fmaf(hi, hi, s);
  }
  return s;
}

// Rows [0, n) of X (row stride d8 packets).  out[r] = |X_r| (nullable);
// *seg_max = max over the rows of |X_r| as an fp32 bit pattern (nullable;
// non-negative floats order like their bit patterns).
__global__ void __launch_bounds__(kNormThreads)
row_norms_kernel(const uint4* __restrict__ X, int64_t n, int64_t d8, float* __restrict__ out,
                 unsigned* __restrict__ seg_max) {
  const int lane = threadIdx.x & 31;
  float warp_max = 0.0f;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kNormWarps + (threadIdx.x >> 5); r < n;
       r += static_cast<int64_t>(gridDim.x) * kNormWarps) {
    const uint4* row = X + r * d8;
    float s = 0.0f;
    for (int64_t i = lane; i < d8; i += 32) s += sq_bf16x8(__ldg(row + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    const float norm = sqrtf(s);
    if (out != nullptr && lane == 0) out[r] = norm;
    warp_max = fmaxf(warp_max, norm);
  }
  if (seg_max != nullptr && lane == 0) atomicMax(seg_max, __float_as_uint(warp_max));
}

unsigned norm_blocks(int64_t n) {
  const int64_t want = (n + kNormWarps - 1) / kNormWarps;
  return static_cast<unsigned>(want < 4096 ? (want > 0 ? want : 1) : 4096);
}

}  // namespace

cudaError_t launch_row_norms(const void* X, int64_t n, int64_t d, float* out, unsigned* seg_max,
                             cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  row_norms_kernel<<<norm_blocks(n), kNormThreads, 0, stream>>>(static_cast<const uint4*>(X), n, d / 8, out,
                                                                 seg_max);
  return cudaGetLastError();
}

}  // namespace fs
