// Host-side internals of libflashsample: the problem description handed from
// the C ABI to the kernel launchers, and the launchers themselves.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "fs_device.cuh"

namespace fs {

// One sampling problem as the kernels see it.  All pointers are device
// pointers owned by the caller except `partials`, which is library workspace.
struct Problem {
  const void* h;          // bf16 [B, d], row-major
  const void* W;          // bf16 [V_local, d], row-major: rows of the vocabulary handled here
  int64_t B;
  int64_t d;
  int64_t V_local;        // rows of W in this call
  int64_t v_offset;       // global vocabulary id of W's first row (noise counters use global ids)
  const float* temp;      // [B]
  const float* bias;      // fp32, nullable; element (b, v_local) at bias[b * bias_stride + v_local]
  int64_t bias_stride;    // 0: one [V_local] vector shared by all rows
  uint64_t seed;
  uint64_t step;
};

// Where a launch leaves its per-(row, part) candidates, and how the final
// reduction finishes them.
struct Finish {
  Partial* partials;      // [B, n_parts]
  int n_parts;
  // chunked-variant carry (nullable): merged into the result, then updated
  float* carry_max;
  int64_t* carry_ids;
  bool carry_in;          // read the carry (not the first chunk)
  bool write_out;         // write out_ids / out_max (last chunk or one-shot)
  int64_t* out_ids;
  float* out_max;
};

// Kernel families selectable by batch size (or forced for tests).
enum Path : int { kPathAuto = 0, kPathSimt = 1, kPathTcVocab = 2, kPathTcBatch = 3 };

// Number of partial candidates per row each family produces for a problem;
// used to size the workspace before launching.
int simt_num_parts(const Problem& p, int device);

// Launchers: enqueue on `stream`; return cudaSuccess or the launch error.
cudaError_t launch_simt(const Problem& p, Partial* partials, int n_parts, cudaStream_t stream);

// Tensor-core vocabulary-major path (B <= 256, d >= 64): one candidate per
// (row, CTA); `err` is the device error word its bounded waits report to.
int tc_vocab_num_parts(const Problem& p, int device);
int tc_vocab_bn(int64_t B);
cudaError_t launch_tc_vocab(const Problem& p, Partial* partials, int n_parts, int* err,
                            cudaStream_t stream);
// Tensor-core batch-major path (any B, d >= 64; used for B > 256): one
// candidate per (row, CTA group).
int tc_batch_num_parts(const Problem& p, int device);
cudaError_t launch_tc_batch(const Problem& p, Partial* partials, int n_parts, int* err,
                            cudaStream_t stream);

cudaError_t launch_reduce(const Finish& f, int64_t B, cudaStream_t stream);

// Set the calling thread's fs_last_error() text.
void record_error(const char* msg);
cudaError_t launch_debug_noise(uint64_t seed, uint64_t step, int64_t row0, int64_t n_rows,
                               int64_t v0, int64_t n_vocab, uint32_t* words, float* gumbel,
                               cudaStream_t stream);

}  // namespace fs
