// SIMT fused LM-head sampler: the W-streaming path for very small batches.
//
// FlashSampling: Fast and Memory-Efficient Exact Sampling -- summary page,
// "Method": logits are formed on chip, perturbed with Gumbel noise, and only a
// per-row (max, argmax) survives; the B x V logits never reach HBM.
//
// Design: every warp owns whole vocabulary rows.  A row of W (d bf16) is read
// once with 16-byte coalesced loads, dotted against the (at most BG) rows of h
// that the block keeps in shared memory, and reduced across the warp.  Lanes
// 0..BG-1 then own one batch row each: they scale by 1/T, add the row's
// Philox-Gumbel draw and keep the running (max, argmax) in registers.  Each
// block pushes one candidate per batch row into the row's packed key and the
// last block to finish writes the sample (fs_finish.cuh).
#include <algorithm>

#include "fs_finish.cuh"
#include "fs_internal.h"

namespace fs {
namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kSimtUnroll = 4;

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ float dot8(uint4 a, uint4 b, float acc) {
  float a0, a1, b0, b1;
  bf16x2_to_f32(a.x, a0, a1); bf16x2_to_f32(b.x, b0, b1);
  acc = fmaf(a0, b0, acc); acc = fmaf(a1, b1, acc);
  bf16x2_to_f32(a.y, a0, a1); bf16x2_to_f32(b.y, b0, b1);
  acc = fmaf(a0, b0, acc); acc = fmaf(a1, b1, acc);
  bf16x2_to_f32(a.z, a0, a1); bf16x2_to_f32(b.z, b0, b1);
  acc = fmaf(a0, b0, acc); acc = fmaf(a1, b1, acc);
  bf16x2_to_f32(a.w, a0, a1); bf16x2_to_f32(b.w, b0, b1);
  acc = fmaf(a0, b0, acc); acc = fmaf(a1, b1, acc);
  return acc;
}

// kEarly: the instantiation for early-finalization chunks (Finish::done set).
// The plain one leaves that code out: at B = 1 the grid is sized for 8 CTAs
// per SM, which needs <= 32 registers per thread.
template <int BG, bool kEarly>
__global__ void __launch_bounds__(kSimtThreads)
simt_fused_kernel(Problem p, Finish f) {
  extern __shared__ uint4 smem_h[];            // [BG][d/8] bf16x8 packets
  __shared__ Best warp_best[kSimtWarps][BG];
  __shared__ int last_flag;
  if constexpr (kEarly) {
    if (early_done_cta(f, &last_flag)) {
      early_skip_cta(f, p.B, p.pdl, &last_flag);
      return;
    }
  }
  const int n_parts = gridDim.x;
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t n16 = p.d / 8;                 // 16-byte packets per row
  const int64_t n_groups = (p.B + BG - 1) / BG;
  const PhiloxKey key{static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32)};
  const uint32_t step_lo = static_cast<uint32_t>(p.step);
  const uint32_t step_hi = static_cast<uint32_t>(p.step >> 32);
  const uint4* hg = reinterpret_cast<const uint4*>(p.h);
  const uint4* Wg = reinterpret_cast<const uint4*>(p.W);
  const int64_t warp_stride = static_cast<int64_t>(n_parts) * kSimtWarps;

  for (int64_t g = blockIdx.y; g < n_groups; g += gridDim.y) {
    const int64_t b0 = g * BG;
    __syncthreads();                           // previous group's readers are done
    // Stage this group's rows of h (zero rows past the batch).
    for (int64_t i = threadIdx.x; i < BG * n16; i += kSimtThreads) {
      const int64_t r = i / n16;
      smem_h[i] = (b0 + r < p.B) ? hg[(b0 + r) * n16 + (i - r * n16)] : make_uint4(0, 0, 0, 0);
    }

    // Lane l < BG owns batch row b0 + l for the epilogue.
    const int64_t my_b = b0 + lane;
    const bool owns_row = lane < BG && my_b < p.B;
    const RowTemp rt = row_temp(owns_row ? p.temp[my_b] : -1.0f);
    Best best = best_none();
    __syncthreads();

    for (int64_t v = static_cast<int64_t>(blockIdx.x) * kSimtWarps + warp; v < p.V_local;
         v += warp_stride) {
      const uint4* wrow = Wg + v * n16;
      float acc[BG];
#pragma unroll
      for (int b = 0; b < BG; ++b) acc[b] = 0.0f;

      int64_t i = lane;
      for (; i + 32 * (kSimtUnroll - 1) < n16; i += 32 * kSimtUnroll) {
        uint4 w[kSimtUnroll];
#pragma unroll
        for (int u = 0; u < kSimtUnroll; ++u) w[u] = __ldg(wrow + i + 32 * u);
#pragma unroll
        for (int u = 0; u < kSimtUnroll; ++u) {
#pragma unroll
          for (int b = 0; b < BG; ++b) acc[b] = dot8(w[u], smem_h[b * n16 + i + 32 * u], acc[b]);
        }
      }
      for (; i < n16; i += 32) {
        const uint4 w = __ldg(wrow + i);
#pragma unroll
        for (int b = 0; b < BG; ++b) acc[b] = dot8(w, smem_h[b * n16 + i], acc[b]);
      }
#pragma unroll
      for (int b = 0; b < BG; ++b) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
      }

      if (owns_row) {
        float logit = 0.0f;
#pragma unroll
        for (int b = 0; b < BG; ++b)
          if (lane == b) logit = acc[b];
        if (p.bias != nullptr) logit += p.bias[my_b * p.bias_stride + v];
        if (p.dbg_logits != nullptr) p.dbg_logits[my_b * p.V_local + v] = logit;   // parity inspection only
        if (rt.mode != kRowInvalid) {
          const int64_t vg = p.v_offset + v;
          float z = logit;
          if (rt.mode == kRowSample) {
            const uint4 words = noise_words(key, static_cast<uint32_t>(vg >> 2),
                                            static_cast<uint32_t>(my_b), step_lo, step_hi);
            z = fmaf(logit, rt.inv_t, gumbel_from_word(word_of(words, static_cast<uint32_t>(vg & 3))));
          }
          if (z > best.z) {  // ids rise within a warp, so strict > keeps the smaller id on ties
            best.z = z;
            best.id = static_cast<int32_t>(vg);
          }
        }
      }
    }

    if (lane < BG) warp_best[warp][lane] = best;
    __syncthreads();
    if (threadIdx.x < BG && b0 + threadIdx.x < p.B) {
      Best r = warp_best[0][threadIdx.x];
#pragma unroll
      for (int w = 1; w < kSimtWarps; ++w) r = combine(r, warp_best[w][threadIdx.x]);
      push_candidate(f, b0 + threadIdx.x, r);
    }
  }
  finish_grid<kEarly>(f, p.B, threadIdx.x, kSimtThreads, &last_flag, cta_bar_and);
}

int pick_group(int64_t B, int64_t d) {
  int bg = 8;
  while (bg > 1 && (bg / 2 >= B || static_cast<int64_t>(bg) * d * 2 > 128 * 1024)) bg /= 2;
  return bg;
}

// One wave of CTAs: the SMs times the CTAs of this instantiation that fit on
// one SM (registers and shared memory), never more than the 8-row vocabulary
// groups, then as few as give every warp the same number of rows (B = 1 on
// the 8B head: 160.0 -> 158.5 us).
template <int BG, bool kEarly>
cudaError_t launch_variant(const Problem& p, const Finish& f, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(BG) * p.d * 2;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaError_t e = raise_smem_limit<simt_fused_kernel<BG, kEarly>>(dev, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, simt_fused_kernel<BG, kEarly>, kSimtThreads, smem);
  if (e != cudaSuccess) return e;
  const int64_t max_parts = std::min<int64_t>(static_cast<int64_t>(std::max(sms, 1)) * std::max(per_sm, 1),
                                              std::max<int64_t>(1, (p.V_local + kSimtWarps - 1) / kSimtWarps));
  // then as few CTAs as give every warp the same number of vocabulary rows
  const int64_t rows_per_warp = (p.V_local + max_parts * kSimtWarps - 1) / (max_parts * kSimtWarps);
  const int64_t warps = (p.V_local + rows_per_warp - 1) / rows_per_warp;
  const int n_parts = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(max_parts, (warps + kSimtWarps - 1) / kSimtWarps)));
  const int64_t groups = (p.B + BG - 1) / BG;
  dim3 grid(n_parts, static_cast<unsigned>(std::min<int64_t>(groups, 65535)));
  return launch_kernel(simt_fused_kernel<BG, kEarly>, grid, dim3(kSimtThreads), smem, stream, p.pdl, p, f);
}

template <int BG>
cudaError_t launch_group(const Problem& p, const Finish& f, cudaStream_t stream) {
  return f.done != nullptr ? launch_variant<BG, true>(p, f, stream) : launch_variant<BG, false>(p, f, stream);
}

}  // namespace

cudaError_t launch_simt(const Problem& p, const Finish& f, cudaStream_t stream) {
  switch (pick_group(p.B, p.d)) {
    case 1: return launch_group<1>(p, f, stream);
    case 2: return launch_group<2>(p, f, stream);
    case 4: return launch_group<4>(p, f, stream);
    default: return launch_group<8>(p, f, stream);
  }
}

}  // namespace fs
