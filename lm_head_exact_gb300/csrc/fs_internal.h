// Host-side internals of libflashsample: the problem description handed from
// the C ABI to the kernel launchers, and the launchers themselves.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>
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
  // Launch as a programmatic dependent of the previous kernel of the stream
  // (set for the 2nd..last chunk of a chunked step, whose inputs were all
  // written before the first chunk was enqueued).
  bool pdl = false;
  // With pdl: the preceding kernel may still be writing h, temp or bias (a
  // one-shot call after the model's last layer), so the kernel reads them
  // only after its dependency wait; only the static W is prefetched before.
  // Clear for chunks, whose inputs are all written before the first chunk.
  // Honoured by the tensor-core kernels (the CUDA-core kernel is launched
  // without the dependency instead).
  bool defer_inputs = false;
  // Global index of row 0 of h in this launch (a batch split over several
  // launches); the noise counter always uses the global row.
  int64_t row_offset = 0;
  // Parity inspection (fs_debug_fused_logits), normally nullptr: when set,
  // the fused kernel also stores every logit it forms -- the fp32
  // accumulator plus the bias, before the temperature and the noise -- at
  // dbg_logits[b * V_local + v] for rows b < B of this launch, from the same
  // accumulator values its epilogue scans.
  float* dbg_logits = nullptr;
  // A vocabulary chunk of a chunked step (fs_sample_chunked): the CTA-pair
  // kernel then runs its lean instantiation (two CTAs per SM) for chunks of
  // few tiles, or its full one with several tiles per pair for larger chunks;
  // either overlaps consecutive chunks (same arithmetic, so the same results
  // bit for bit).
  bool chunk = false;
  // Chunks per step in the previous chunked step on this stream (0: none
  // yet); sizes the tiles per pair of the full instantiation (see
  // launch_tc_pair).  Never changes a result.
  int step_chunks = 0;
  bool in_graph = false;  // chunk call made while its stream is captured into a CUDA graph
};

// Launch `kernel` on `stream`, as a programmatic dependent launch when `pdl`.
// Raises a kernel's dynamic shared memory limit to at least `bytes` on
// device `dev`, calling the runtime only when the limit this process set
// before is lower: the attribute persists, and setting it on every launch
// costs host time in chunked steps of many launches.
template <auto kKernel>
cudaError_t raise_smem_limit(int dev, int bytes) {
  static std::atomic<int> set_bytes[64];   // zero-initialized (static storage)
  const bool cached = dev >= 0 && dev < 64;
  if (cached && set_bytes[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) {
    int cur = set_bytes[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !set_bytes[dev].compare_exchange_weak(cur, bytes, std::memory_order_release)) {
    }
  }
  return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// How a launch finishes the sample.  The fused kernels reduce across CTAs
// themselves: every CTA atomicMax-es its per-row candidates into `keys`
// (packed, see pack_key), and the CTA that finishes last -- counted in
// `counter` -- turns the keys into outputs and zeroes keys and counter for the
// next call.  The separate reduction kernel instead reads `partials`.
struct Finish {
  unsigned long long* keys;   // [B], zero between calls
  unsigned int* counter;      // zero between calls
  Partial* partials;      // [B, n_parts] (reduction-kernel path only)
  int n_parts;
  // chunked-variant carry (nullable): merged into the result, then updated
  float* carry_max;
  int64_t* carry_ids;
  bool carry_in;          // read the carry (not the first chunk)
  bool write_out;         // write out_ids / out_max (last chunk or one-shot)
  int64_t* out_ids;
  float* out_max;
  // Early finalization of the chunked variant (nullable `done`): a chunk
  // whose *done is set on entry does no work; the last CTA of a chunk that
  // ran sets *done when no row can be overtaken by the later chunks, whose
  // rows have norms <= rest_w_norm and biases <= rest_bias_max.
  int* done = nullptr;
  const float* h_norms = nullptr;   // [B] Euclidean norms of the rows of h
  const float* temp = nullptr;      // [B]
  float rest_w_norm = 0.0f;
  float rest_bias_max = 0.0f;
};

// Kernel families selectable by batch size (or forced for tests).
enum Path : int { kPathAuto = 0, kPathSimt = 1, kPathTcVocab = 2, kPathTcBatch = 3, kPathTcPair = 4 };

// Launchers: enqueue on `stream`; return cudaSuccess or the launch error.
// Each fused kernel finishes the sample itself through `f` (one launch).
cudaError_t launch_simt(const Problem& p, const Finish& f, cudaStream_t stream);

// Tensor-core vocabulary-major path (B <= 256, d >= 64); `err` is the device
// error word its bounded waits report to.
int tc_vocab_bn(int64_t B);
cudaError_t launch_tc_vocab(const Problem& p, const Finish& f, int* err, cudaStream_t stream);

// Tensor-core batch-major path (any B, d >= 64).
cudaError_t launch_tc_batch(const Problem& p, const Finish& f, int* err, cudaStream_t stream);

// Tensor-core batch-major path over CTA pairs (tcgen05 cta_group::2; any B,
// d >= 64).
cudaError_t launch_tc_pair(const Problem& p, const Finish& f, int* err, cudaStream_t stream);
// Whether a chunked step of step_chunks such chunks fits one wave of CTA
// pairs with few tiles per pair (the chunk family rule of fs_api.cu).
bool tc_pair_chunk_one_wave(int64_t V_local, int64_t B, int step_chunks, bool in_graph, int device);

// Unfused comparison pipeline: tensor-core GEMM storing fp32 logits [B, V]
// (+ bias) to HBM, then row softmax into probs [B, V], then the sample.
cudaError_t launch_tc_logits(const Problem& p, float* logits, int* err, cudaStream_t stream);
// `partials`: unfused_partial_bytes(B) bytes of scratch for the per-range
// softmax sums and candidates (each row is split over several blocks).
size_t unfused_partial_bytes(int64_t B);
cudaError_t launch_unfused_tail(const Problem& p, float* logits, float* probs, void* partials, int64_t* out_ids,
                                float* out_max, cudaStream_t stream);

// Failure-path check of the bounded waits: one wait that runs out after
// timeout_ns and flags `err`.
cudaError_t launch_debug_wait(int* err, uint64_t timeout_ns, cudaStream_t stream);

// Reduction kernel over `f.partials` (used when no fused kernel runs: V == 0).
// Row norms |X_r| of a bf16 [n, d] matrix into out (nullable) and their
// maximum as fp32 bits into *seg_max (nullable, atomicMax; zero it first).
cudaError_t launch_row_norms(const void* X, int64_t n, int64_t d, float* out, unsigned* seg_max,
                             cudaStream_t stream);

// Gumbel-top-k: the batch-major kernel in top-K mode (K in {4, 8, 16}, one
// launch, B <= one launch's rows) writes per-(row, CTA group) lists to
// partials [B, tc_topk_parts(B), K]; launch_topk_merge then merges each row's
// lists (n_lists <= 256 per row, each sorted) into its k <= K best
// (out_ids / out_z [B, k]; -1 / -inf padded).
int tc_topk_parts(int64_t B, int64_t V, int device);
cudaError_t launch_tc_topk(const Problem& p, int K, Partial* partials, int* err, cudaStream_t stream);
// The vocabulary-major kernel in top-K mode, for B <= 64: partials [B,
// tc_vocab_topk_parts(V), K] (one list per (row, CTA)).
int tc_vocab_topk_parts(int64_t V, int device);
cudaError_t launch_tc_vocab_topk(const Problem& p, int K, Partial* partials, int* err, cudaStream_t stream);
// The CTA-pair kernel in top-K mode, for the batches the sampler runs on CTA
// pairs: partials [B, tc_pair_topk_parts(B, V), K] (one list per (row, pair
// group)); B <= tc_pair_topk_max_rows (one launch).
int64_t tc_pair_topk_max_rows(int device);
int tc_pair_topk_parts(int64_t B, int64_t V, int device);
cudaError_t launch_tc_pair_topk(const Problem& p, int K, Partial* partials, int* err, cudaStream_t stream);
cudaError_t launch_topk_merge(const Partial* partials, int n_lists, int K, int64_t B, int k, int64_t* out_ids,
                              float* out_z, cudaStream_t stream);

// Host-buffer entry point: h (h_bytes, a multiple of 16) and temperatures
// [B] from mapped pinned host memory into device staging; the next kernel on
// the stream may start as its programmatic dependent.
cudaError_t launch_copy_in(const void* h_src, void* h_dst, int64_t h_bytes, const float* t_src, float* t_dst, int64_t B,
                           cudaStream_t stream);

// Tensor-parallel combine: out[b] = best over r of (shard_max[r, b], shard_ids[r, b]).
cudaError_t launch_combine_shards(const float* shard_max, const int64_t* shard_ids, int64_t R, int64_t B,
                                  int64_t* out_ids, float* out_max, cudaStream_t stream);

cudaError_t launch_reduce(const Finish& f, int64_t B, cudaStream_t stream);

// Status word of fs_sample_noalloc on the current device (the bounded-wait
// error word inside its static scratch): read into *code and cleared, with
// no allocation; 0 when that entry point has not run on the device.  The
// caller has synchronized the device.
cudaError_t noalloc_take_status(int* code);

// Set the calling thread's fs_last_error() text.
void record_error(const char* msg);
cudaError_t launch_debug_noise(uint64_t seed, uint64_t step, int64_t row0, int64_t n_rows,
                               int64_t v0, int64_t n_vocab, uint32_t* words, float* gumbel,
                               cudaStream_t stream);

}  // namespace fs
