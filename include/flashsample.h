/*
 * libflashsample -- exact categorical sampling fused into the LM-head matmul,
 * for one NVIDIA GB300 (sm_103a).
 *
 * What it computes (FlashSampling: Fast and Memory-Efficient Exact Sampling;
 * summary page, sections "Method" and "Key claims"; arXiv abstract):
 *
 *   logits[b, v] = sum_k h[b, k] * W[v, k]  (+ bias[b, v])
 *   z[b, v]      = logits[b, v] / T[b] + g[b, v],   g = -log(-log u)
 *   out_ids[b]   = argmax_v z[b, v],  out_max[b] = z[b, out_ids[b]]
 *
 * so out_ids[b] is an exact sample of softmax(logits[b, :] / T[b]).  The
 * vocabulary is processed tile by tile on chip; only a per-row (max, argmax)
 * per tile survives and a small reduction over tiles finishes the sample, so
 * the B x V logits never reach device memory.
 *
 * Conventions shared by every entry point:
 *  - h is bf16 [B, d] and W is bf16 [V, d], both row-major (d contiguous).
 *    d must be a multiple of 8 and both base pointers 16-byte aligned
 *    (FS_ERR_UNSUPPORTED otherwise).  B, V < 2^31.
 *  - temp is fp32 [B].  T > 0: sample from softmax(logits / T).  T == 0:
 *    greedy (argmax of the logits, no noise; out_max is the max logit).
 *    T < 0 or NaN: no sample (out_ids = -1, out_max = -inf).
 *  - Noise: u is drawn from Philox-4x32-10 (Salmon et al., SC'11) with key
 *    (seed mod 2^32, seed >> 32) and counter (v >> 2, b, step mod 2^32,
 *    step >> 32); word (v & 3) gives x and u = ((x >> 9) + 0.5) * 2^-23.  The
 *    draw of (b, v, step) is fixed by the counter alone, so results do not
 *    depend on tiling, chunking or the kernel chosen.
 *  - Ties: equal z goes to the smaller vocabulary id.  NaN and -inf scores
 *    never win; a row without any candidate returns id -1 and max -inf.
 *  - Unless stated otherwise, pointers are DEVICE pointers owned by the
 *    caller; the call validates arguments on the host, enqueues its kernels
 *    on `stream` (a cudaStream_t; NULL is the legacy default stream) and
 *    returns without synchronizing.  Results are valid once the stream has
 *    reached that point.
 *  - The library owns one small workspace per (device, stream): a ticket
 *    counter and one packed candidate key per batch row, through which the
 *    CTAs of the fused kernel finish the sample (the last CTA to finish writes
 *    the outputs).  It grows on demand, which is not allowed inside
 *    CUDA-graph capture: call fs_workspace_reserve() first.
 *  - Errors: argument problems return FS_ERR_INVALID_ARG / FS_ERR_UNSUPPORTED
 *    before anything is enqueued; a failed CUDA call returns FS_ERR_CUDA.
 *    fs_last_error() gives a human-readable detail of the last failure on
 *    the calling thread.
 */
#ifndef FLASHSAMPLE_H_
#define FLASHSAMPLE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported entry points (the library is built with hidden visibility). */
#if defined(__GNUC__)
#define FS_API __attribute__((visibility("default")))
#else
#define FS_API
#endif

typedef enum fs_status {
  FS_OK = 0,
  FS_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad flag combination */
  FS_ERR_UNSUPPORTED = 2,     /* valid request the kernels do not handle (alignment, d % 8) */
  FS_ERR_CUDA = 3,            /* a CUDA runtime call or kernel launch failed */
  FS_ERR_WORKSPACE = 4,       /* workspace must grow but cannot (allocation failed, or capture active) */
  FS_ERR_DEVICE_TIMEOUT = 5   /* a kernel gave up a bounded wait and flagged the device error word */
} fs_status;

/* Flags of fs_sample_chunked. */
#define FS_CHUNK_FIRST 1      /* ignore the incoming carry: this chunk starts the row */
#define FS_CHUNK_LAST 2       /* write out_ids / out_max after merging this chunk */
#define FS_CHUNK_SERIAL 4     /* start only after the previous call has finished (no overlap) */

/* Kernel families (fs_set_path). */
#define FS_PATH_AUTO 0        /* chosen from the batch size B only */
#define FS_PATH_SIMT 1        /* W-streaming CUDA-core path */
#define FS_PATH_TC_VOCAB 2    /* tcgen05 tensor-core path, vocabulary rows on the MMA M axis */
#define FS_PATH_TC_BATCH 3    /* tcgen05 tensor-core path, batch rows on the MMA M axis */
#define FS_PATH_TC_PAIR 4     /* as FS_PATH_TC_BATCH, one MMA over a pair of CTAs (cta_group::2) */

/*
 * One decode step of fused sampling (summary page, "Method"; arXiv abstract).
 *   h [B, d] bf16, W [V, d] bf16, temp [B] fp32: inputs (device).
 *   seed, step: noise stream (see conventions).
 *   out_ids [B] int64, out_max [B] fp32: outputs (device).
 *   stream: cudaStream_t to enqueue on.
 * B == 0 is a no-op; V == 0 gives id -1 on every row.
 */
FS_API fs_status fs_sample(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                    const float* temp, uint64_t seed, uint64_t step,
                    int64_t* out_ids, float* out_max, void* stream);

/*
 * fs_sample with an optional fp32 bias added to the logits before the
 * division by T.  bias (device, nullable) holds element (b, v) at
 * bias[b * bias_row_stride + v]; bias_row_stride is 0 (one [V] vector shared
 * by all rows) or >= V.
 */
FS_API fs_status fs_sample_ex(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                       const float* temp, const float* bias, int64_t bias_row_stride,
                       uint64_t seed, uint64_t step,
                       int64_t* out_ids, float* out_max, void* stream);

/*
 * Grouped online (chunked) variant (arXiv abstract; summary page, "Method",
 * last paragraph): one call per contiguous vocabulary chunk [v_begin, v_end),
 * with a per-row (max, argmax) carry between calls.  Calls after the first
 * chunk are launched as programmatic dependents: a chunk's kernel may start
 * streaming its W rows while the previous chunk's kernel still runs and waits
 * for it only before merging the carry -- so between the chunk calls of one
 * step, enqueue nothing on the stream that writes h, temp, W or bias.  The result of a full
 * sequence of calls equals fs_sample on the whole vocabulary bit for bit,
 * because the noise of (b, v) depends on the global id v only and every
 * logit is formed in the same arithmetic: at B = 1 both run the CUDA-core
 * kernel; otherwise a chunk call may run another tensor-core family than the
 * one-shot call (chosen from B, the chunk size and the chunk count of the
 * previous step on the stream), and all of them form the same fp32 logits.
 *   W_chunk: rows [v_begin, v_end) of W, i.e. W + v_begin * d (device).
 *   bias_chunk: bias columns of the chunk (element (b, j) for global id
 *     v_begin + j at bias_chunk[b * bias_row_stride + j]) or NULL.
 *   carry_max [B] fp32 and carry_ids [B] int64 (device, caller-owned):
 *     read unless FS_CHUNK_FIRST, always updated (ids -1 = none yet).
 *   flags: FS_CHUNK_FIRST and/or FS_CHUNK_LAST, optionally FS_CHUNK_SERIAL
 *     (launch without the programmatic dependency).  With FS_CHUNK_LAST,
 *     out_ids / out_max are written (they may alias the carry arrays' roles
 *     but not their memory); otherwise they may be NULL.
 */
FS_API fs_status fs_sample_chunked(const void* h, const void* W_chunk, int64_t B, int64_t d,
                            int64_t v_begin, int64_t v_end, const float* temp,
                            const float* bias_chunk, int64_t bias_row_stride,
                            uint64_t seed, uint64_t step,
                            float* carry_max, int64_t* carry_ids, int flags,
                            int64_t* out_ids, float* out_max, void* stream);

/*
 * One whole chunked step: the fs_sample_chunked calls of chunks
 * [bounds[i], bounds[i+1]) for i = 0 .. n_chunks - 1 (FS_CHUNK_FIRST on the
 * first, FS_CHUNK_LAST on the last), issued from C in one call, so that a
 * host loop's per-call overhead does not bound a step of many small chunks.
 * Same kernels, launches and results as the sequence of calls (equal to
 * fs_sample on the whole vocabulary bit for bit).
 *   W: the full [bounds[n_chunks], d] matrix (device); chunk i is rows
 *     [bounds[i], bounds[i+1]).
 *   bounds: host array of n_chunks + 1 non-decreasing row offsets, bounds[0]
 *     = 0; empty chunks are allowed.
 *   bias: NULL or the [B, V] (row stride bias_row_stride, or 0 for a shared
 *     [V]) bias of the whole vocabulary; chunk i reads columns bounds[i] ...
 *   carry_max / carry_ids / out_ids / out_max / stream: as fs_sample_chunked.
 * Returns the first failing chunk call's status (later chunks not launched).
 */
FS_API fs_status fs_sample_chunked_step(const void* h, const void* W, int64_t B, int64_t d, const int64_t* bounds,
                                        int n_chunks, const float* temp, const float* bias,
                                        int64_t bias_row_stride, uint64_t seed, uint64_t step,
                                        float* carry_max, int64_t* carry_ids,
                                        int64_t* out_ids, float* out_max, void* stream);

/*
 * Chunked variant with online early finalization (summary page, "Method",
 * last paragraph: the streaming sampler may stop once the later tiles can no
 * longer overtake the running maximum).  Same arguments and result as
 * fs_sample_chunked, plus:
 *   h_norms [B] fp32 (device): |h_b| (Euclidean), e.g. from fs_row_norms.
 *   rest_w_norm: an upper bound on |W_v| for every row v >= v_end of W
 *     (0 for the last chunk), e.g. from fs_chunk_rest_norms; >= 0.
 *   rest_bias_max: an upper bound on every bias entry at ids >= v_end
 *     (0 without bias); +inf disables the early stop.  Not NaN.
 *   done (device int, caller-owned): reset to 0 by the FS_CHUNK_FIRST call
 *     (a memset enqueued before its kernel) and written by every call that
 *     runs; a call that finds *done != 0 on entry reads no W and computes
 *     nothing (a FS_CHUNK_LAST call still writes out_ids / out_max from the
 *     carry).
 * After a call, *done = 1 iff every row is final: its temperature is invalid,
 * or its carried best perturbed score z* satisfies
 *     z* >= U + 1e-4 |U| + 1e-3,
 *     U = (|h_b| rest_w_norm + rest_bias_max) / T_b + 16.6356  (T_b > 0),
 *     U =  |h_b| rest_w_norm + rest_bias_max                   (T_b == 0),
 * where 16.6356 bounds the Gumbel value of the largest uniform the noise can
 * produce, -log(-log(1 - 2^-24)), and the margin covers fp32 rounding.  By
 * Cauchy-Schwarz no later id can then win, so the result equals that of
 * fs_sample_chunked bit for bit.  As there, calls after the first are
 * programmatic dependents of the previous call: a call may read *done before
 * the previous one has finished and then does the work; a skipping call waits
 * for the previous one before it ends.  With FS_CHUNK_SERIAL a call starts
 * only after the previous one has finished and so always sees its flag: the
 * better choice when rows are expected to be final early (peaked
 * distributions), at the cost of the overlap between chunks when they are
 * not.  B <= 4096, else FS_ERR_UNSUPPORTED.
 */
FS_API fs_status fs_sample_chunked_early(const void* h, const void* W_chunk, int64_t B, int64_t d,
                                  int64_t v_begin, int64_t v_end, const float* temp,
                                  const float* bias_chunk, int64_t bias_row_stride,
                                  uint64_t seed, uint64_t step,
                                  float* carry_max, int64_t* carry_ids, int flags,
                                  const float* h_norms, float rest_w_norm, float rest_bias_max, int* done,
                                  int64_t* out_ids, float* out_max, void* stream);

/*
 * Euclidean norms of the rows of a bf16 matrix X [n, d] (row-major, device,
 * 16-byte aligned, d % 8 == 0), accumulated in fp32: out[r] = |X_r| (device,
 * [n] fp32).  Asynchronous on `stream`.  n == 0 is a no-op.
 */
FS_API fs_status fs_row_norms(const void* X, int64_t n, int64_t d, float* out, void* stream);

/*
 * Setup for fs_sample_chunked_early: for chunks [bounds[i], bounds[i+1]) of W
 * (bounds: host, n_chunks + 1 non-decreasing entries; W: device, the whole
 * [bounds[n_chunks], d] matrix), rest_w_norm[i] (host, [n_chunks]) = the
 * largest row norm of W over rows [bounds[i+1], bounds[n_chunks]), 0 when
 * empty.  Synchronizes `stream`; allocates and frees a small device buffer.
 */
FS_API fs_status fs_chunk_rest_norms(const void* W, int64_t d, const int64_t* bounds, int64_t n_chunks,
                                     float* rest_w_norm, void* stream);

/*
 * Tensor-parallel variant, final step (summary page, Method, third
 * paragraph; abstract): each of R ranks samples its own vocabulary shard
 * [v_begin, v_end) -- fs_sample_chunked with FS_CHUNK_FIRST | FS_CHUNK_LAST,
 * so ids are global and the noise is that of the whole-vocabulary call --
 * the ranks exchange only the per-row (max, id) pairs, and this call picks,
 * per row, the best pair under the sampler's total order.  The result equals
 * fs_sample over the whole vocabulary bit for bit (same kernel family for
 * the same B).
 *   shard_max [R, B] fp32 and shard_ids [R, B] int64 (device; shard r's row b
 *   at r * B + b; id -1 = no sample from that shard).
 *   out_ids [B] int64, out_max [B] fp32 (device); -1 / -inf when no shard has
 *   a sample.  R == 0 gives -1 everywhere; B == 0 is a no-op.
 */
FS_API fs_status fs_combine_shards(const float* shard_max, const int64_t* shard_ids, int64_t R, int64_t B,
                                   int64_t* out_ids, float* out_max, void* stream);

/*
 * Gumbel-top-k: k ids per row drawn WITHOUT replacement from
 * softmax(logits / T) (each next id from the renormalized remaining mass),
 * fused into the LM-head matmul like fs_sample_ex.  The summary page cites
 * Gumbel-top-k sampling among the related work; with the sampler's own
 * perturbed scores z (same noise, same temperature and bias handling), the
 * k ids of largest z are that draw.  Row b's result, best first under the
 * sampler's total order (a larger z, then a smaller id), is out_ids[b * k + j]
 * (int64) and out_z[b * k + j] (fp32, the perturbed score; the logit for
 * T == 0 rows, i.e. the top-k logits); -inf and NaN scores are never chosen,
 * and rows with fewer than k choosable ids (or an invalid T) are padded with
 * id -1 and z -inf.  k = 1 gives fs_sample_ex's ids.
 *   1 <= k <= 16 (else FS_ERR_INVALID_ARG); B <= 4096 and d >= 64 (else
 *   FS_ERR_UNSUPPORTED).  Two launches: a tensor-core kernel with a K-list
 *   epilogue (K = 4, 8 or 16 >= k; the vocabulary-major kernel for B <= 64,
 *   above that the kernel fs_sample_ex runs at that B, fs_set_path included:
 *   CTA pairs or the batch-major one, which also stands in for the other
 *   families), writing one list per (row, CTA or CTA group) to library
 *   workspace, then a block-per-row merge.  The
 *   workspace grows on the first call of a size; capture in a CUDA graph only
 *   after an eager call of the same B.
 */
FS_API fs_status fs_sample_topk(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                                const float* temp, const float* bias, int64_t bias_row_stride,
                                uint64_t seed, uint64_t step, int k,
                                int64_t* out_ids, float* out_z, void* stream);

/*
 * The UNFUSED comparison pipeline (summary page, "Method", ops (1)-(4)):
 * a tensor-core GEMM writes fp32 logits [B, V] (+ bias) to device memory,
 * a softmax kernel reads them and writes probabilities [B, V], and a sample
 * kernel re-reads those and picks argmax_v p_v / (-log u_v) with the same
 * Philox draws.  Same arguments and outputs as fs_sample_ex; ids agree with
 * the fused path up to rounding near ties.  It exists to measure the memory
 * traffic fusion removes (about 20 * B * V bytes per step).
 *   logits_out (device fp32 [B, V], nullable): where the GEMM writes the
 *     logits; NULL uses library workspace.  Probabilities always live in
 *     library workspace.  Needs d >= 64.
 */
FS_API fs_status fs_sample_unfused(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                                   const float* temp, const float* bias, int64_t bias_row_stride,
                                   uint64_t seed, uint64_t step, int64_t* out_ids, float* out_max,
                                   float* logits_out, void* stream);

/*
 * End-to-end convenience call with HOST buffers: copies h_host [B, d] bf16 and
 * temp_host [B] fp32 to the device, samples against the device-resident
 * W [V, d] (and optional device bias), copies out_ids_host [B] int64 and
 * out_max_host [B] fp32 back, and synchronizes `stream` before returning.
 * When h_host and temp_host are mapped page-locked memory (cudaHostAlloc,
 * cudaHostRegister with mapping, torch's pin_memory), a small kernel reads
 * them directly and the fused kernel starts as its programmatic dependent
 * (see fs_set_launch_overlap), writing the results straight into a mapped
 * landing area: no copy-engine transfers.  Other host memory is copied with
 * cudaMemcpyAsync (pageable memory works but is slower).  Device staging
 * lives in the library workspace of (device, stream).
 */
FS_API fs_status fs_sample_host(const void* h_host, const void* W, int64_t B, int64_t d, int64_t V,
                         const float* temp_host, const float* bias, int64_t bias_row_stride,
                         uint64_t seed, uint64_t step,
                         int64_t* out_ids_host, float* out_max_host, void* stream);

/*
 * fs_sample without any device-memory allocation.  (An engineering variant:
 * the FlashSampling paper has no counterpart.)  Same arguments, noise and
 * sampled distribution as fs_sample, but it always runs the vocabulary-major
 * tensor-core kernel, whatever B and fs_set_path say (fs_sample picks the
 * kernel family from B: the CUDA-core kernel at B = 1, the batch-major or
 * CTA-pair kernels above B = 64).  The three tensor-core families form the
 * same fp32 logits bit for bit, so its results equal fs_sample's bit for bit
 * whenever fs_sample runs a tensor-core family (every 2 <= B <= 256 under
 * FS_PATH_AUTO); at B = 1, or with FS_PATH_SIMT forced, fs_sample runs the
 * CUDA-core kernel and the two agree within the parity tolerance (ids may
 * differ only on rows whose two best perturbed scores are within rounding of
 * each other).  The
 * cross-tile finish area (ticket counter + one candidate key per row) lives
 * in a fixed static device array inside the library (2.3 KB per GPU, held
 * until the process exits) instead of a workspace the library cudaMalloc's
 * on demand.  For callers that cannot let
 * a library allocate or free device memory: an allocator that already owns
 * the GPU's memory budget, or code that cannot afford the device-wide
 * synchronization of cudaFree.
 *   Limits: 1 <= B <= 256 (larger B returns FS_ERR_UNSUPPORTED with a
 *   message), d >= 64 and a multiple of 8; no bias.  Alignment: h and W
 *   16 bytes, out_ids 8, temp and out_max 4 (else FS_ERR_UNSUPPORTED,
 *   before anything is enqueued).
 *   Errors on the device: a bounded wait that runs out sets a status word
 *   in the same static array; fs_device_error() reports and clears it and
 *   allocates nothing.
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress) and zeroes it; make that first call
 *   before any stream capture starts.
 *   Sharing: every call on a device uses the same array and finds the last
 *   call's contents there.  Calls whose kernels overlap on the GPU (e.g. on
 *   unordered streams) race on it; keep them ordered on one stream.
 */
FS_API fs_status fs_sample_noalloc(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                                   const float* temp, uint64_t seed, uint64_t step,
                                   int64_t* out_ids, float* out_max, void* stream);

/* Workspace bytes one call with (B, V) needs on the current device. */
FS_API size_t fs_workspace_bytes(int64_t B, int64_t V);

/*
 * Grow the workspace of (current device, stream) to serve calls up to
 * (B, V) without allocating, and create the device error word; required
 * before capturing fs_sample / fs_sample_ex / fs_sample_chunked calls in a
 * CUDA graph on that stream (the seed and step are then fixed in the graph).
 */
FS_API fs_status fs_workspace_reserve(int64_t B, int64_t V, void* stream);

/* Free every workspace this library holds on the current device. */
FS_API fs_status fs_workspace_release(void);

/* Force a kernel family for later calls (FS_PATH_*); FS_PATH_AUTO restores
 * the batch-size rule.  Process-wide.  The tensor-core families
 * (FS_PATH_TC_VOCAB, FS_PATH_TC_BATCH, FS_PATH_TC_PAIR) form identical
 * logits and samples; only the CUDA-core family (FS_PATH_SIMT, fp32 FFMA
 * accumulation) differs from them, within the parity tolerance. */
FS_API fs_status fs_set_path(int path);

/*
 * Launch overlap of fs_sample / fs_sample_ex (1, the default, or 0;
 * process-wide).  With 1, the tensor-core kernels (B >= 2) are launched
 * as programmatic dependents of the preceding kernel on the stream: their
 * prologues and first rings of W loads may run while that kernel finishes
 * (for example the previous decode step's sampling kernel, or the model's
 * last layer); h, temp and bias are read only after the preceding kernel has
 * completed.  W itself is read early, so the kernel enqueued immediately
 * before the call must not write W -- set 0 where it may.
 */
FS_API fs_status fs_set_launch_overlap(int enable);

/* The kernel family a one-shot call with batch size B would use under the
 * current setting (FS_PATH_SIMT / FS_PATH_TC_VOCAB / FS_PATH_TC_BATCH /
 * FS_PATH_TC_PAIR). */
FS_API int fs_path_for_batch(int64_t B);

/* The kernel family a chunk call of B rows and V_chunk vocabulary rows would
 * use under the current setting, when the previous chunked step on its stream
 * had step_chunks chunk calls (0: none yet), launched on a stream (a call
 * made during CUDA-graph capture may choose differently). */
FS_API int fs_path_for_chunks(int64_t B, int64_t V_chunk, int step_chunks);

/*
 * Timing hook: when both are non-NULL, every later sampling call on this
 * thread records cudaEvent_t `start` on its stream just before the fused
 * sampling kernel and `stop` just after it (the cross-tile reduction is
 * outside the pair).  Pass NULL, NULL to stop.  Lets a caller time the
 * dominant kernel inside a normal run without changing the work done.
 */
FS_API fs_status fs_profile_events(void* start, void* stop);

/* Read and clear the device error words of the current device -- the
 * library's own and fs_sample_noalloc's -- after synchronizing the device.
 * *code receives 0 when no kernel reported a problem.  Allocates nothing. */
FS_API fs_status fs_device_error(int* code);

/*
 * Failure-path check: enqueue a one-warp kernel whose bounded mbarrier wait
 * (the kind every tensor-core kernel uses) waits for an arrival that never
 * comes, gives up after timeout_ns (0 < timeout_ns <= 1e9) and sets the device
 * error word to 1 -- as a real stall would -- without faulting the context.
 * fs_device_error() then reports and clears it.
 */
FS_API fs_status fs_debug_wait_timeout(uint64_t timeout_ns, void* stream);

/*
 * Host-side fault injection for failure-detection tests (process-wide):
 * FS_FAULT_ALLOC makes every workspace allocation that would happen fail with
 * FS_ERR_WORKSPACE, FS_FAULT_LAUNCH makes every fused sampling launch fail
 * with FS_ERR_CUDA -- before any CUDA call is made, so the GPU and the
 * context are untouched and later calls work once FS_FAULT_NONE is set.  The
 * initial value comes from the FS_FAULT environment variable ("alloc",
 * "launch"; anything else: none).
 */
#define FS_FAULT_NONE 0
#define FS_FAULT_ALLOC 1
#define FS_FAULT_LAUNCH 2
FS_API fs_status fs_debug_set_fault(int kind);

/* Static name of a status code. */
FS_API const char* fs_status_string(fs_status s);

/* Detail of the last failure on the calling thread ("" if none). */
FS_API const char* fs_last_error(void);

/*
 * Noise inspection: for rows [row0, row0 + n_rows) and global vocabulary ids
 * [v0, v0 + n_vocab), write the 32-bit Philox draw (words, nullable) and the
 * Gumbel value the sampling kernels add (gumbel, nullable), row-major
 * [n_rows, n_vocab], device pointers.  For parity tests of the noise stage.
 */
FS_API fs_status fs_debug_noise(uint64_t seed, uint64_t step, int64_t row0, int64_t n_rows,
                         int64_t v0, int64_t n_vocab, uint32_t* words, float* gumbel,
                         void* stream);

/*
 * Logit inspection of the FUSED kernels, for parity tests (the fused path
 * never writes logits, so this is how its accumulators are checked; summary
 * page, "Method": the logit tile is computed on chip).  Runs exactly the
 * launch fs_sample_ex would run for these arguments -- the same kernel
 * family (from B and fs_set_path), instantiation and grid, same outputs --
 * with the kernel's inspection store switched on: every logit it forms, the
 * fp32 accumulator plus the bias (before the division by T and the noise),
 * is also written to logits_out[b * V + v] (device, fp32 [B, V], 4-byte
 * aligned; every element is written, rows with an invalid T included).
 * Slow (the store is uncoalesced in the vocabulary-major kernel): for tests.
 */
FS_API fs_status fs_debug_fused_logits(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                                       const float* temp, const float* bias, int64_t bias_row_stride,
                                       uint64_t seed, uint64_t step, int64_t* out_ids, float* out_max,
                                       float* logits_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FLASHSAMPLE_H_ */
