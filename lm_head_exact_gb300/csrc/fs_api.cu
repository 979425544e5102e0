// The C ABI of libflashsample: argument validation, per-(device, stream)
// workspace, kernel-family dispatch by batch size, and the host-buffer
// end-to-end entry point.  Declarations and contracts: include/flashsample.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "flashsample.h"
#include "fs_internal.h"

namespace fs {
namespace {

thread_local char g_last_error[512] = "";
thread_local cudaEvent_t g_prof_start = nullptr;
thread_local cudaEvent_t g_prof_stop = nullptr;
std::atomic<int> g_forced_path{kPathAuto};
std::atomic<int> g_launch_overlap{1};

// Host-side fault injection (FS_FAULT_*): read from the FS_FAULT environment
// variable ("alloc" or "launch") on first use, or set by fs_debug_set_fault.
// An injected fault makes the library return the error of the failing call
// without touching the GPU.
std::atomic<int> g_fault{-1};

int injected_fault() {
  int f = g_fault.load();
  if (f < 0) {
    const char* env = getenv("FS_FAULT");
    f = env == nullptr ? FS_FAULT_NONE
                       : (strcmp(env, "alloc") == 0 ? FS_FAULT_ALLOC : strcmp(env, "launch") == 0 ? FS_FAULT_LAUNCH : FS_FAULT_NONE);
    g_fault.store(f);
  }
  return f;
}

fs_status fail(fs_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

fs_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- workspace
// Per (device, stream): the finish area of the fused kernels -- kKeySets
// ticket counters (a 256-byte header) followed by kKeySets sets of one packed
// 64-bit candidate key per batch row; all zero between uses (zeroed on
// allocation, re-zeroed by the last CTA of every launch that used them) --
// plus staging for the host entry point and the unfused pipeline's logits /
// probabilities.
//
// One-shot calls use set 0.  The chunks of a chunked step use sets 0, 1, 2,
// ... in turn (the chunk's sequence number since FS_CHUNK_FIRST, modulo
// kKeySets), so consecutive chunks, which overlap on the GPU, never share
// keys or a ticket and their CTAs need not wait for each other.  Each chunk
// completes only after the previous one (its last CTA waits for it), and a
// chunk that would reuse set 0 after the first is launched without overlap,
// so every earlier chunk has completed -- and left its set zeroed -- before
// any set is reused.
constexpr int kKeySets = 32;

struct Workspace {
  void* finish = nullptr;
  size_t finish_bytes = 0;
  int64_t finish_rows = 0;      // rows per key set
  int64_t chunk_seq = 0;        // sequence number of the last chunk call since FS_CHUNK_FIRST
  int last_step_chunks = 0;     // chunk calls of the last step completed with FS_CHUNK_LAST
  void* staging = nullptr;      // device staging of fs_sample_host
  size_t staging_bytes = 0;
  void* unfused = nullptr;      // logits + probabilities of fs_sample_unfused
  size_t unfused_bytes = 0;
  void* host_out = nullptr;     // pinned (mapped) host landing area of fs_sample_host's results
  void* host_out_dev = nullptr; // its device alias
  size_t host_out_bytes = 0;
  void* topk = nullptr;         // per-(row, CTA group) candidate lists of fs_sample_topk
  size_t topk_bytes = 0;
};

std::mutex g_ws_mutex;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;
std::map<int, int*> g_error_words;   // per device: kernels' bounded-wait error word

constexpr size_t kFinishHeader = 256;

size_t finish_bytes_for(int64_t B) {
  return kFinishHeader + static_cast<size_t>(kKeySets) * static_cast<size_t>(std::max<int64_t>(B, 1)) *
                             sizeof(unsigned long long);
}
static_assert(kKeySets * sizeof(unsigned int) <= kFinishHeader, "ticket counters fit in the header");

bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) return false;
  return st != cudaStreamCaptureStatusNone;
}

// Make `*buf` hold at least `need` bytes; growth synchronizes the stream so
// that no in-flight kernel still uses the old buffer.
fs_status grow(void** buf, size_t* have, size_t need, cudaStream_t stream) {
  if (*have >= need) return FS_OK;
  if (injected_fault() == FS_FAULT_ALLOC)
    return fail(FS_ERR_WORKSPACE, "cudaMalloc(%zu) for the workspace failed: injected (FS_FAULT=alloc)", need);
  if (capturing(stream))
    return fail(FS_ERR_WORKSPACE, "workspace must grow to %zu bytes during stream capture; "
                "call fs_workspace_reserve() before capturing", need);
  if (*buf != nullptr) {
    cudaStreamSynchronize(stream);
    cudaFree(*buf);
    *buf = nullptr;
    *have = 0;
  }
  cudaError_t e = cudaMalloc(buf, need);
  if (e != cudaSuccess) {
    *buf = nullptr;
    cudaGetLastError();
    return fail(FS_ERR_WORKSPACE, "cudaMalloc(%zu) for the workspace failed: %s", need,
                cudaGetErrorString(e));
  }
  *have = need;
  return FS_OK;
}

fs_status current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  return FS_OK;
}

// Key set of a chunk call: FS_CHUNK_FIRST starts the sequence at 0, every
// later chunk call on the stream takes the next number.  *overlap_ok is false
// when the set wraps around to 0 (the call must then launch without overlap).
//
// *step_chunks receives the chunk count of the previous step on the stream
// (0 before the first step ends); a call with FS_CHUNK_LAST records its own.
fs_status next_chunk_set(cudaStream_t stream, bool first, bool last, int* set, bool* overlap_ok,
                         int* step_chunks) {
  int dev;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  Workspace& ws = g_workspaces[{dev, stream}];
  ws.chunk_seq = first ? 0 : ws.chunk_seq + 1;
  *set = static_cast<int>(ws.chunk_seq % kKeySets);
  *overlap_ok = first || *set != 0;
  *step_chunks = ws.last_step_chunks;
  if (last) ws.last_step_chunks = static_cast<int>(std::min<int64_t>(ws.chunk_seq + 1, 1 << 20));
  return FS_OK;
}

// The finish area of (current device, stream) for batches up to B rows:
// key set `set` and its ticket counter.
fs_status get_finish(cudaStream_t stream, int64_t B, Finish* f, int set = 0) {
  int dev;
  fs_status s = current_device(&dev);
  if (s != FS_OK) return s;
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  Workspace& ws = g_workspaces[{dev, stream}];
  const size_t need = finish_bytes_for(B);
  if (ws.finish_bytes < need) {
    s = grow(&ws.finish, &ws.finish_bytes, need, stream);
    if (s != FS_OK) return s;
    // on the call's stream: the kernels that use the area follow on it (a
    // plain cudaMemset would run on the legacy default stream, which a
    // non-blocking stream is not ordered after)
    cudaError_t e = cudaMemsetAsync(ws.finish, 0, ws.finish_bytes, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(FS_ERR_WORKSPACE, "zeroing the workspace failed: %s", cudaGetErrorString(e));
    }
  }
  ws.finish_rows = static_cast<int64_t>((ws.finish_bytes - kFinishHeader) / (kKeySets * sizeof(unsigned long long)));
  f->counter = static_cast<unsigned int*>(ws.finish) + set;
  f->keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws.finish) + kFinishHeader) +
            static_cast<int64_t>(set) * ws.finish_rows;
  return FS_OK;
}

// The device error word of the current device, allocated on first use and
// zeroed on `stream` -- the stream of the kernels that will report to it, so
// they are ordered after the zeroing even on a non-blocking stream.  Not
// allowed during stream capture (fs_workspace_reserve creates it first).
fs_status error_word(int** out, cudaStream_t stream) {
  int dev;
  {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  auto it = g_error_words.find(dev);
  if (it != g_error_words.end()) {
    *out = it->second;
    return FS_OK;
  }
  if (capturing(stream))
    return fail(FS_ERR_WORKSPACE, "the device error word must be created during stream capture; "
                "call fs_workspace_reserve() before capturing");
  int* w = nullptr;
  cudaError_t e = cudaMalloc(&w, sizeof(int));
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof(int), stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (w != nullptr) cudaFree(w);
    return fail(FS_ERR_WORKSPACE, "device error word: %s", cudaGetErrorString(e));
  }
  g_error_words[dev] = w;
  *out = w;
  return FS_OK;
}

// The error word of the current device if one exists (nullptr otherwise);
// never allocates.
int* existing_error_word() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  auto it = g_error_words.find(dev);
  return it == g_error_words.end() ? nullptr : it->second;
}

// ---------------------------------------------------------------- checks
fs_status check_device_ptr(const void* p, const char* name) {
  if (p == nullptr) return fail(FS_ERR_INVALID_ARG, "%s is NULL", name);
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "cudaPointerGetAttributes");
  }
  if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
    return fail(FS_ERR_INVALID_ARG, "%s is not device memory", name);
  int dev = -1;
  cudaGetDevice(&dev);
  if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
    return fail(FS_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", name,
                attr.device, dev);
  return FS_OK;
}

// Device address of mapped, page-locked host memory, or nullptr for any other
// pointer (pageable, device, unknown).
const void* mapped_device_pointer(const void* host_ptr) {
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, host_ptr) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

fs_status check_aligned(const void* p, size_t a, const char* name) {
  if (reinterpret_cast<uintptr_t>(p) % a != 0)
    return fail(FS_ERR_UNSUPPORTED, "%s must be %zu-byte aligned", name, a);
  return FS_OK;
}

#define FS_TRY(expr)                  \
  do {                                \
    fs_status _s = (expr);            \
    if (_s != FS_OK) return _s;       \
  } while (0)

fs_status check_shapes(int64_t B, int64_t d, int64_t V) {
  if (B < 0 || d <= 0 || V < 0) return fail(FS_ERR_INVALID_ARG, "need B >= 0, d > 0, V >= 0 (got %lld, %lld, %lld)",
                                            (long long)B, (long long)d, (long long)V);
  if (B >= (int64_t(1) << 31) || V >= (int64_t(1) << 31))
    return fail(FS_ERR_UNSUPPORTED, "B and V must be < 2^31");
  if (d % 8 != 0) return fail(FS_ERR_UNSUPPORTED, "d must be a multiple of 8 (got %lld)", (long long)d);
  if (d > 65536) return fail(FS_ERR_UNSUPPORTED, "d must be <= 65536 (got %lld)", (long long)d);
  return FS_OK;
}

fs_status check_problem(const Problem& p, bool need_out, const void* out_ids, const void* out_max) {
  FS_TRY(check_shapes(p.B, p.d, p.V_local));
  if (p.B == 0) return FS_OK;
  FS_TRY(check_device_ptr(p.h, "h"));
  FS_TRY(check_aligned(p.h, 16, "h"));
  FS_TRY(check_device_ptr(p.temp, "temp"));
  FS_TRY(check_aligned(p.temp, 4, "temp"));
  if (p.V_local > 0) {
    FS_TRY(check_device_ptr(p.W, "W"));
    FS_TRY(check_aligned(p.W, 16, "W"));
  }
  if (p.bias != nullptr) {
    if (p.bias_stride != 0 && p.bias_stride < p.V_local)
      return fail(FS_ERR_INVALID_ARG, "bias_row_stride must be 0 or >= V");
    if (p.bias_stride < 0) return fail(FS_ERR_INVALID_ARG, "bias_row_stride must be >= 0");
    FS_TRY(check_device_ptr(p.bias, "bias"));
    FS_TRY(check_aligned(p.bias, 4, "bias"));
  }
  if (need_out) {
    FS_TRY(check_device_ptr(out_ids, "out_ids"));
    FS_TRY(check_aligned(out_ids, 8, "out_ids"));
    FS_TRY(check_device_ptr(out_max, "out_max"));
    FS_TRY(check_aligned(out_max, 4, "out_max"));
  }
  return FS_OK;
}

// Kernel family for a call.  Auto: chosen from the batch size (and the
// model width, identical for every chunk of a chunked run), so one-shot and
// chunked runs compute every logit in the same arithmetic and agree bit for
// bit; chunk calls may take another tensor-core family (resolve_call_path),
// since all of them form the same logits.
constexpr int64_t kVocabMajorMaxBatch = 64;

// Auto rule, measured on GB300 (Llama-3-8B head, fused kernel µs):
//   B = 1: CUDA-core kernel (161 vs 168 vocabulary-major);
//   B <= 64: vocabulary-major (W streaming; back to back at B = 64: 161.2 vs
//   167.3 for the batch-major kernel, while at every B from 72 to 96 the
//   batch-major kernel wins, 167.3 vs 170.7, in alternating runs);
//   larger B: the CTA-pair kernel when padding B to 256-row pair tiles wastes
//   fewer than 128 rows (B = 256: 205 vs 217, B = 1024: 701 vs 729), otherwise
//   the single-CTA batch-major kernel (B = 128: 185 vs 193, B = 384: 307 vs 344).
// B = 1 stays on the CUDA-core kernel: measured on GB300 (8B head), the
// vocabulary-major kernel is 1.8% faster for a one-shot B = 1 step (154.3 vs
// 157.8 us) but slower on chunks, whose few 128-row tiles leave most SMs idle
// (8 chunks 195.5 vs 188.7 us, 32 chunks 234 vs 212, early stop 121 vs 91);
// chunked and one-shot calls must use the same family to agree bit for bit.
int auto_path(int64_t B) {
  if (B == 1) return kPathSimt;
  if (B <= kVocabMajorMaxBatch) return kPathTcVocab;
  const int64_t padded = (B + 255) / 256 * 256;
  return (B > 128 && padded - B < 128) ? kPathTcPair : kPathTcBatch;
}

int resolve_path(int64_t B, int64_t d) {
  int path = g_forced_path.load();
  if (path == kPathAuto) path = auto_path(B);
  if (path == kPathTcVocab && B > 256) path = kPathTcBatch;
  if ((path == kPathTcVocab || path == kPathTcBatch || path == kPathTcPair) && d < 64) path = kPathSimt;
  return path;
}

// Chunk calls of batches that fit one 128-row batch tile but not the two-
// CTAs-per-SM vocabulary-major instantiation (32 < B <= 128) run the CTA-pair
// kernel when the chunked step fits one wave of pairs with few tiles per pair,
// else the batch-major kernel.  Every tensor-core family forms the same fp32
// logits bit for bit and runs the same scan, so the samples still equal the
// one-shot call's.  Measured on GB300 (8B head, µs per chunked step, 8 / 16 /
// 32 chunks): B = 48 vocabulary-major 272 / - / 285, batch-major 242 / - /
// 234, pair 219 / - / 266; B = 64 vocabulary-major 272 / 277 / 285, batch-
// major 242 / 237 / 234; B = 128 batch-major 242 / 237 / 234, pair 223 / 252 /
// 275.  At B <= 32 (two vocabulary-major CTAs per SM: 191-202) and B = 1
// (CUDA-core logits) chunks keep the batch-size family.
constexpr int64_t kChunkVocabMaxBatch = 32;

int resolve_call_path(const Problem& p) {
  const int path = resolve_path(p.B, p.d);
  if (!p.chunk || g_forced_path.load() != kPathAuto) return path;
  if (path != kPathTcVocab && path != kPathTcBatch) return path;
  if (p.B <= kChunkVocabMaxBatch || p.B > 128) return path;
  int dev = 0;
  cudaGetDevice(&dev);
  return tc_pair_chunk_one_wave(p.V_local, p.B, p.step_chunks, p.in_graph, dev) ? kPathTcPair : kPathTcBatch;
}

// One fused launch (kernel + in-kernel cross-CTA finish) for one problem,
// finishing through key set `key_set` of the stream's workspace.
fs_status run(Problem p, Finish f, cudaStream_t stream, int key_set = 0) {
  if (p.B == 0) return FS_OK;
  if (p.V_local == 0) {                 // no vocabulary: every row gets "no sample"
    f.partials = nullptr;
    f.n_parts = 0;
    cudaError_t e = launch_reduce(f, p.B, stream);
    if (e != cudaSuccess) return cuda_fail(e, "reduction kernel launch");
    return FS_OK;
  }
  FS_TRY(get_finish(stream, p.B, &f, key_set));
  const int path = resolve_call_path(p);
  // The tensor-core kernels defer their input reads (interleaved A/B runs on
  // GB300: the overlap saves 4-8 us per back-to-back step at every B from 2
  // to 512); the CUDA-core kernel launches plainly.
  if (p.defer_inputs && path == kPathSimt) {
    p.defer_inputs = false;
    p.pdl = false;
  }
  int* err = nullptr;
  if (path != kPathSimt) FS_TRY(error_word(&err, stream));
  cudaError_t e = cudaSuccess;
  if (g_prof_start != nullptr) {
    e = cudaEventRecord(g_prof_start, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(start)");
  }
  if (injected_fault() == FS_FAULT_LAUNCH)
    return fail(FS_ERR_CUDA, "fused sampling kernel launch failed: injected (FS_FAULT=launch)");
  switch (path) {
    case kPathTcVocab:
      e = launch_tc_vocab(p, f, err, stream);
      break;
    case kPathTcBatch:
      e = launch_tc_batch(p, f, err, stream);
      break;
    case kPathTcPair:
      e = launch_tc_pair(p, f, err, stream);
      break;
    case kPathSimt:
    default:
      e = launch_simt(p, f, stream);
      break;
  }
  if (e != cudaSuccess) return cuda_fail(e, "fused sampling kernel launch");
  if (g_prof_stop != nullptr) {
    e = cudaEventRecord(g_prof_stop, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(stop)");
  }
  return FS_OK;
}

// Early-finalization inputs of one chunk call (all unset: plain chunked call).
// Rows one early-finalization call handles: one launch of every kernel
// family, so the done flag is decided by a single last CTA.
constexpr int kEarlyMaxRows = 4096;

// Gumbel-top-k limits: list length per row, and rows (one launch).
constexpr int kTopKMax = 16;
constexpr int kTopKMaxRows = 4096;

struct EarlyArgs {
  const float* h_norms = nullptr;
  float rest_w_norm = 0.0f;
  float rest_bias_max = 0.0f;
  int* done = nullptr;
};

fs_status check_carry(int64_t B, const float* carry_max, const int64_t* carry_ids) {
  if (B > 0) {
    FS_TRY(check_device_ptr(carry_max, "carry_max"));
    FS_TRY(check_aligned(carry_max, 4, "carry_max"));
    FS_TRY(check_device_ptr(carry_ids, "carry_ids"));
    FS_TRY(check_aligned(carry_ids, 8, "carry_ids"));
  }
  return FS_OK;
}

fs_status sample_chunk(const void* h, const void* W_chunk, int64_t B, int64_t d, int64_t v_begin, int64_t v_end,
                       const float* temp, const float* bias_chunk, int64_t bias_row_stride, uint64_t seed,
                       uint64_t step, float* carry_max, int64_t* carry_ids, int flags, const EarlyArgs& early,
                       int64_t* out_ids, float* out_max, void* stream, bool checked = false) {
  if (v_begin < 0 || v_end < v_begin)
    return fail(FS_ERR_INVALID_ARG, "need 0 <= v_begin <= v_end (got %lld, %lld)",
                (long long)v_begin, (long long)v_end);
  if (v_end >= (int64_t(1) << 31)) return fail(FS_ERR_UNSUPPORTED, "v_end must be < 2^31");
  if (flags & ~(FS_CHUNK_FIRST | FS_CHUNK_LAST | FS_CHUNK_SERIAL))
    return fail(FS_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  const bool last = (flags & FS_CHUNK_LAST) != 0;
  Problem p{h, W_chunk, B, d, v_end - v_begin, v_begin, temp, bias_chunk, bias_row_stride, seed, step};
  // Chunks after the first may start streaming their W rows while the
  // previous chunk's kernel is still running (programmatic dependent launch);
  // they wait for it only before merging into the shared carry.
  p.pdl = (flags & (FS_CHUNK_FIRST | FS_CHUNK_SERIAL)) == 0;
  p.chunk = true;
  if (!checked) {   // (fs_sample_chunked_step checks its pointers once per step)
    FS_TRY(check_problem(p, last, out_ids, out_max));
    FS_TRY(check_carry(B, carry_max, carry_ids));
  }
  Finish f{};
  f.carry_max = carry_max;
  f.carry_ids = carry_ids;
  f.carry_in = (flags & FS_CHUNK_FIRST) == 0;
  f.write_out = last;
  f.out_ids = out_ids;
  f.out_max = out_max;
  f.done = early.done;
  f.h_norms = early.h_norms;
  f.temp = temp;
  f.rest_w_norm = early.rest_w_norm;
  f.rest_bias_max = early.rest_bias_max;
  if (early.done != nullptr && (flags & FS_CHUNK_FIRST) != 0) {
    // reset before the first chunk: a later chunk, launched as a programmatic
    // dependent, may read the flag before the first chunk finishes
    cudaError_t e = cudaMemsetAsync(early.done, 0, sizeof(int), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(done)");
  }
  int set = 0;
  bool overlap_ok = true;
  if (B > 0)
    FS_TRY(next_chunk_set(static_cast<cudaStream_t>(stream), (flags & FS_CHUNK_FIRST) != 0, last, &set, &overlap_ok,
                          &p.step_chunks));
  if (!overlap_ok) p.pdl = false;
  p.in_graph = capturing(static_cast<cudaStream_t>(stream));
  return run(p, f, static_cast<cudaStream_t>(stream), set);
}

}  // namespace

void record_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

}  // namespace fs

using namespace fs;

extern "C" {

fs_status fs_sample_ex(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                       const float* temp, const float* bias, int64_t bias_row_stride,
                       uint64_t seed, uint64_t step,
                       int64_t* out_ids, float* out_max, void* stream) {
  g_last_error[0] = '\0';
  Problem p{h, W, B, d, V, 0, temp, bias, bias_row_stride, seed, step};
  FS_TRY(check_problem(p, true, out_ids, out_max));
  // Programmatic dependent launch: the kernel's prologue and first W loads
  // may overlap the tail of the preceding kernel of the stream; h, temp and
  // bias are read only after its dependency wait.
  p.pdl = g_launch_overlap.load() != 0;
  p.defer_inputs = p.pdl;
  Finish f{};
  f.write_out = true;
  f.out_ids = out_ids;
  f.out_max = out_max;
  return run(p, f, static_cast<cudaStream_t>(stream));
}

fs_status fs_debug_fused_logits(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                                const float* temp, const float* bias, int64_t bias_row_stride,
                                uint64_t seed, uint64_t step, int64_t* out_ids, float* out_max,
                                float* logits_out, void* stream) {
  g_last_error[0] = '\0';
  Problem p{h, W, B, d, V, 0, temp, bias, bias_row_stride, seed, step};
  FS_TRY(check_problem(p, true, out_ids, out_max));
  if (B > 0 && V > 0) {
    FS_TRY(check_device_ptr(logits_out, "logits_out"));
    FS_TRY(check_aligned(logits_out, 4, "logits_out"));
  }
  // exactly fs_sample_ex's launch, with the kernel's logit store switched on
  p.pdl = g_launch_overlap.load() != 0;
  p.defer_inputs = p.pdl;
  p.dbg_logits = logits_out;
  Finish f{};
  f.write_out = true;
  f.out_ids = out_ids;
  f.out_max = out_max;
  return run(p, f, static_cast<cudaStream_t>(stream));
}

fs_status fs_sample(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                    const float* temp, uint64_t seed, uint64_t step,
                    int64_t* out_ids, float* out_max, void* stream) {
  return fs_sample_ex(h, W, B, d, V, temp, nullptr, 0, seed, step, out_ids, out_max, stream);
}

fs_status fs_sample_chunked(const void* h, const void* W_chunk, int64_t B, int64_t d,
                            int64_t v_begin, int64_t v_end, const float* temp,
                            const float* bias_chunk, int64_t bias_row_stride,
                            uint64_t seed, uint64_t step,
                            float* carry_max, int64_t* carry_ids, int flags,
                            int64_t* out_ids, float* out_max, void* stream) {
  g_last_error[0] = '\0';
  return sample_chunk(h, W_chunk, B, d, v_begin, v_end, temp, bias_chunk, bias_row_stride, seed, step, carry_max,
                      carry_ids, flags, EarlyArgs{}, out_ids, out_max, stream);
}

fs_status fs_sample_chunked_step(const void* h, const void* W, int64_t B, int64_t d, const int64_t* bounds,
                                 int n_chunks, const float* temp, const float* bias, int64_t bias_row_stride,
                                 uint64_t seed, uint64_t step, float* carry_max, int64_t* carry_ids,
                                 int64_t* out_ids, float* out_max, void* stream) {
  g_last_error[0] = '\0';
  if (n_chunks < 1) return fail(FS_ERR_INVALID_ARG, "need n_chunks >= 1 (got %d)", n_chunks);
  if (bounds == nullptr) return fail(FS_ERR_INVALID_ARG, "bounds is NULL");
  if (bounds[0] != 0) return fail(FS_ERR_INVALID_ARG, "bounds[0] must be 0 (got %lld)", (long long)bounds[0]);
  for (int i = 0; i < n_chunks; ++i)
    if (bounds[i + 1] < bounds[i])
      return fail(FS_ERR_INVALID_ARG, "bounds must not decrease (bounds[%d] = %lld > bounds[%d] = %lld)", i,
                  (long long)bounds[i], i + 1, (long long)bounds[i + 1]);
  if (d < 0) return fail(FS_ERR_INVALID_ARG, "need d >= 0 (got %lld)", (long long)d);
  if (bounds[n_chunks] >= (int64_t(1) << 31)) return fail(FS_ERR_UNSUPPORTED, "bounds[n_chunks] must be < 2^31");
  // the pointers and shapes of the whole step are checked once: every
  // chunk's W rows, bias columns and outputs lie inside them
  Problem whole{h, W, B, d, bounds[n_chunks], 0, temp, bias, bias_row_stride, seed, step};
  FS_TRY(check_problem(whole, true, out_ids, out_max));
  FS_TRY(check_carry(B, carry_max, carry_ids));
  for (int i = 0; i < n_chunks; ++i) {
    const int flags = (i == 0 ? FS_CHUNK_FIRST : 0) | (i == n_chunks - 1 ? FS_CHUNK_LAST : 0);
    const void* W_chunk = static_cast<const uint16_t*>(W) + bounds[i] * d;
    const float* bias_chunk = bias != nullptr ? bias + bounds[i] : nullptr;
    FS_TRY(sample_chunk(h, W_chunk, B, d, bounds[i], bounds[i + 1], temp, bias_chunk, bias_row_stride, seed, step,
                        carry_max, carry_ids, flags, EarlyArgs{}, out_ids, out_max, stream, true));
  }
  return FS_OK;
}

fs_status fs_sample_chunked_early(const void* h, const void* W_chunk, int64_t B, int64_t d,
                                  int64_t v_begin, int64_t v_end, const float* temp,
                                  const float* bias_chunk, int64_t bias_row_stride,
                                  uint64_t seed, uint64_t step,
                                  float* carry_max, int64_t* carry_ids, int flags,
                                  const float* h_norms, float rest_w_norm, float rest_bias_max, int* done,
                                  int64_t* out_ids, float* out_max, void* stream) {
  g_last_error[0] = '\0';
  if (B > kEarlyMaxRows)
    return fail(FS_ERR_UNSUPPORTED, "early finalization handles B <= %d (got %lld)", kEarlyMaxRows, (long long)B);
  if (!(rest_w_norm >= 0.0f)) return fail(FS_ERR_INVALID_ARG, "rest_w_norm must be >= 0 and not NaN");
  if (rest_bias_max != rest_bias_max) return fail(FS_ERR_INVALID_ARG, "rest_bias_max is NaN");
  FS_TRY(check_device_ptr(done, "done"));
  FS_TRY(check_aligned(done, 4, "done"));
  if (B > 0) {
    FS_TRY(check_device_ptr(h_norms, "h_norms"));
    FS_TRY(check_aligned(h_norms, 4, "h_norms"));
  }
  EarlyArgs early;
  early.h_norms = h_norms;
  early.rest_w_norm = rest_w_norm;
  early.rest_bias_max = rest_bias_max;
  early.done = done;
  return sample_chunk(h, W_chunk, B, d, v_begin, v_end, temp, bias_chunk, bias_row_stride, seed, step, carry_max,
                      carry_ids, flags, early, out_ids, out_max, stream);
}

fs_status fs_row_norms(const void* X, int64_t n, int64_t d, float* out, void* stream) {
  g_last_error[0] = '\0';
  FS_TRY(check_shapes(0, d, n));
  if (n == 0) return FS_OK;
  FS_TRY(check_device_ptr(X, "X"));
  FS_TRY(check_aligned(X, 16, "X"));
  FS_TRY(check_device_ptr(out, "out"));
  FS_TRY(check_aligned(out, 4, "out"));
  cudaError_t e = launch_row_norms(X, n, d, out, nullptr, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "row-norm kernel launch");
  return FS_OK;
}

fs_status fs_chunk_rest_norms(const void* W, int64_t d, const int64_t* bounds, int64_t n_chunks,
                              float* rest_w_norm, void* stream_) {
  g_last_error[0] = '\0';
  if (n_chunks < 0) return fail(FS_ERR_INVALID_ARG, "n_chunks must be >= 0");
  if (n_chunks == 0) return FS_OK;
  if (bounds == nullptr || rest_w_norm == nullptr) return fail(FS_ERR_INVALID_ARG, "bounds / rest_w_norm is NULL");
  if (bounds[0] < 0) return fail(FS_ERR_INVALID_ARG, "bounds[0] must be >= 0");
  for (int64_t i = 0; i < n_chunks; ++i)
    if (bounds[i + 1] < bounds[i]) return fail(FS_ERR_INVALID_ARG, "bounds must be non-decreasing");
  FS_TRY(check_shapes(0, d, bounds[n_chunks]));
  if (bounds[n_chunks] > bounds[0]) {
    FS_TRY(check_device_ptr(W, "W"));
    FS_TRY(check_aligned(W, 16, "W"));
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  unsigned* seg = nullptr;
  cudaError_t e = cudaMalloc(&seg, static_cast<size_t>(n_chunks) * sizeof(unsigned));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(FS_ERR_WORKSPACE, "chunk maxima of %lld floats", (long long)n_chunks);
  }
  std::vector<unsigned> host(static_cast<size_t>(n_chunks), 0u);
  e = cudaMemsetAsync(seg, 0, static_cast<size_t>(n_chunks) * sizeof(unsigned), stream);
  for (int64_t i = 0; i < n_chunks && e == cudaSuccess; ++i)
    e = launch_row_norms(static_cast<const char*>(W) + bounds[i] * d * 2, bounds[i + 1] - bounds[i], d, nullptr,
                         seg + i, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(host.data(), seg, static_cast<size_t>(n_chunks) * sizeof(unsigned), cudaMemcpyDeviceToHost,
                        stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  cudaFree(seg);
  if (e != cudaSuccess) return cuda_fail(e, "chunk row norms");
  float rest = 0.0f;      // rows after the last chunk: none
  for (int64_t i = n_chunks - 1; i >= 0; --i) {
    rest_w_norm[i] = rest;
    float m;
    memcpy(&m, &host[static_cast<size_t>(i)], sizeof(m));
    rest = std::max(rest, m);
  }
  return FS_OK;
}

fs_status fs_sample_host(const void* h_host, const void* W, int64_t B, int64_t d, int64_t V,
                         const float* temp_host, const float* bias, int64_t bias_row_stride,
                         uint64_t seed, uint64_t step,
                         int64_t* out_ids_host, float* out_max_host, void* stream_) {
  g_last_error[0] = '\0';
  FS_TRY(check_shapes(B, d, V));
  if (B == 0) return FS_OK;
  if (!h_host || !temp_host || !out_ids_host || !out_max_host)
    return fail(FS_ERR_INVALID_ARG, "host buffers must not be NULL");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  FS_TRY(current_device(&dev));
  if (V > 0) {
    FS_TRY(check_device_ptr(W, "W"));
    FS_TRY(check_aligned(W, 16, "W"));
  }
  if (bias != nullptr) {
    if (bias_row_stride < 0 || (bias_row_stride != 0 && bias_row_stride < V))
      return fail(FS_ERR_INVALID_ARG, "bias_row_stride must be 0 or >= V");
    FS_TRY(check_device_ptr(bias, "bias"));
    FS_TRY(check_aligned(bias, 4, "bias"));
  }
  // device staging: [h | temp | ids, max] -- the results are contiguous so one
  // copy brings them back into a pinned landing area of the library
  const size_t h_bytes = static_cast<size_t>(B) * d * 2;
  const size_t off_temp = (h_bytes + 255) & ~size_t(255);
  const size_t off_ids = off_temp + ((static_cast<size_t>(B) * 4 + 255) & ~size_t(255));
  const size_t off_max = off_ids + static_cast<size_t>(B) * 8;
  const size_t out_bytes = static_cast<size_t>(B) * 12;
  const size_t total = off_ids + out_bytes;
  char* staging = nullptr;
  char* landing = nullptr;
  char* landing_dev = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace& ws = g_workspaces[{dev, stream}];
    FS_TRY(grow(&ws.staging, &ws.staging_bytes, total, stream));
    staging = static_cast<char*>(ws.staging);
    if (ws.host_out_bytes < out_bytes) {
      if (ws.host_out != nullptr) {
        cudaStreamSynchronize(stream);
        cudaFreeHost(ws.host_out);
        ws.host_out = nullptr;
        ws.host_out_bytes = 0;
      }
      ws.host_out_dev = nullptr;
      if (cudaHostAlloc(&ws.host_out, out_bytes, cudaHostAllocMapped) != cudaSuccess) {
        cudaGetLastError();
        ws.host_out = nullptr;
        return fail(FS_ERR_WORKSPACE, "pinned host landing area of %zu bytes", out_bytes);
      }
      if (cudaHostGetDevicePointer(&ws.host_out_dev, ws.host_out, 0) != cudaSuccess) {
        cudaGetLastError();
        ws.host_out_dev = nullptr;
      }
      ws.host_out_bytes = out_bytes;
    }
    landing = static_cast<char*>(ws.host_out);
    landing_dev = static_cast<char*>(ws.host_out_dev);
  }
  // Pinned, mapped host inputs (torch's pin_memory, cudaHostAlloc) are read
  // directly: a copy kernel moves h and T into device staging and the fused
  // kernel starts as its programmatic dependent, so its prologue and first W
  // loads overlap the copy; the results are written straight into the mapped
  // landing area.  Other host memory takes the copy-engine path.
  const void* h_map = mapped_device_pointer(h_host);
  const void* t_map = mapped_device_pointer(temp_host);
  const bool zero_copy = h_map != nullptr && t_map != nullptr && landing_dev != nullptr &&
                         reinterpret_cast<uintptr_t>(h_map) % 16 == 0 && reinterpret_cast<uintptr_t>(t_map) % 4 == 0;
  // staging pointers are the library's own device memory: no per-pointer queries
  Problem p{staging, W, B, d, V, 0, reinterpret_cast<const float*>(staging + off_temp), bias,
            bias_row_stride, seed, step};
  Finish f{};
  f.write_out = true;
  cudaError_t e = cudaSuccess;
  if (zero_copy) {
    e = launch_copy_in(h_map, staging, static_cast<int64_t>(h_bytes), static_cast<const float*>(t_map),
                       reinterpret_cast<float*>(staging + off_temp), B, stream);
    if (e != cudaSuccess) return cuda_fail(e, "copy-in kernel launch");
    p.pdl = g_launch_overlap.load() != 0;
    p.defer_inputs = p.pdl;
    f.out_ids = reinterpret_cast<int64_t*>(landing_dev);
    f.out_max = reinterpret_cast<float*>(landing_dev + static_cast<size_t>(B) * 8);
    FS_TRY(run(p, f, stream));
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  } else {
    e = cudaMemcpyAsync(staging, h_host, h_bytes, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(staging + off_temp, temp_host, static_cast<size_t>(B) * 4,
                          cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "host-to-device copy");
    f.out_ids = reinterpret_cast<int64_t*>(staging + off_ids);
    f.out_max = reinterpret_cast<float*>(staging + off_max);
    FS_TRY(run(p, f, stream));
    e = cudaMemcpyAsync(landing, staging + off_ids, out_bytes, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "device-to-host copy");
  }
  memcpy(out_ids_host, landing, static_cast<size_t>(B) * 8);
  memcpy(out_max_host, landing + static_cast<size_t>(B) * 8, static_cast<size_t>(B) * 4);
  return FS_OK;
}

fs_status fs_combine_shards(const float* shard_max, const int64_t* shard_ids, int64_t R, int64_t B,
                            int64_t* out_ids, float* out_max, void* stream) {
  g_last_error[0] = '\0';
  if (R < 0 || B < 0) return fail(FS_ERR_INVALID_ARG, "need R >= 0 and B >= 0 (got %lld, %lld)", (long long)R,
                                  (long long)B);
  if (B == 0) return FS_OK;
  if (R > 0) {
    FS_TRY(check_device_ptr(shard_max, "shard_max"));
    FS_TRY(check_aligned(shard_max, 4, "shard_max"));
    FS_TRY(check_device_ptr(shard_ids, "shard_ids"));
    FS_TRY(check_aligned(shard_ids, 8, "shard_ids"));
  }
  FS_TRY(check_device_ptr(out_ids, "out_ids"));
  FS_TRY(check_aligned(out_ids, 8, "out_ids"));
  FS_TRY(check_device_ptr(out_max, "out_max"));
  FS_TRY(check_aligned(out_max, 4, "out_max"));
  cudaError_t e = launch_combine_shards(shard_max, shard_ids, R, B, out_ids, out_max, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
  return FS_OK;
}

fs_status fs_sample_topk(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                         const float* temp, const float* bias, int64_t bias_row_stride,
                         uint64_t seed, uint64_t step, int k,
                         int64_t* out_ids, float* out_z, void* stream_) {
  g_last_error[0] = '\0';
  if (k < 1 || k > kTopKMax) return fail(FS_ERR_INVALID_ARG, "k must be in [1, %d] (got %d)", kTopKMax, k);
  Problem p{h, W, B, d, V, 0, temp, bias, bias_row_stride, seed, step};
  FS_TRY(check_problem(p, true, out_ids, out_z));
  if (B == 0) return FS_OK;
  if (B > kTopKMaxRows)
    return fail(FS_ERR_UNSUPPORTED, "fs_sample_topk handles B <= %d (got %lld)", kTopKMaxRows, (long long)B);
  if (V > 0 && d < 64) return fail(FS_ERR_UNSUPPORTED, "fs_sample_topk needs d >= 64 (got %lld)", (long long)d);
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  int dev;
  FS_TRY(current_device(&dev));
  const int K = k <= 4 ? 4 : (k <= 8 ? 8 : 16);
  // overlapped launch as for fs_sample_ex: W prefetched before the dependency
  // wait, h / temp / bias read and the shared partials written after it
  p.pdl = g_launch_overlap.load() != 0;
  p.defer_inputs = p.pdl;
  // B <= 64: the vocabulary-major kernel (one lane per batch column keeps the
  // lists); larger B: the kernel the sampler runs at that B (fs_set_path
  // included), CTA pairs or the batch-major one (one thread per batch row in
  // both); the vocabulary-major and CUDA-core families have no list epilogue
  // there, so those B take the batch-major one.
  const int family = B <= 64 ? kPathTcVocab
                     : (resolve_path(B, d) == kPathTcPair && B <= tc_pair_topk_max_rows(dev) ? kPathTcPair
                                                                                             : kPathTcBatch);
  const int parts = V <= 0 ? 0
                    : family == kPathTcVocab ? tc_vocab_topk_parts(V, dev)
                    : family == kPathTcPair  ? tc_pair_topk_parts(B, V, dev)
                                             : tc_topk_parts(B, V, dev);
  const size_t need = std::max<size_t>(static_cast<size_t>(B) * parts * K * sizeof(Partial), 256);
  Partial* partials = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace& ws = g_workspaces[{dev, stream}];
    FS_TRY(grow(&ws.topk, &ws.topk_bytes, need, stream));
    partials = static_cast<Partial*>(ws.topk);
  }
  cudaError_t e = cudaSuccess;
  if (V > 0) {
    int* err = nullptr;
    FS_TRY(error_word(&err, stream));
    e = family == kPathTcVocab ? launch_tc_vocab_topk(p, K, partials, err, stream)
        : family == kPathTcPair ? launch_tc_pair_topk(p, K, partials, err, stream)
                                : launch_tc_topk(p, K, partials, err, stream);
    if (e != cudaSuccess) return cuda_fail(e, "top-k kernel launch");
  }
  e = launch_topk_merge(partials, parts, K, B, k, out_ids, out_z, stream);
  if (e != cudaSuccess) return cuda_fail(e, "top-k merge launch");
  return FS_OK;
}

fs_status fs_sample_unfused(const void* h, const void* W, int64_t B, int64_t d, int64_t V,
                            const float* temp, const float* bias, int64_t bias_row_stride,
                            uint64_t seed, uint64_t step, int64_t* out_ids, float* out_max,
                            float* logits_out, void* stream_) {
  g_last_error[0] = '\0';
  Problem p{h, W, B, d, V, 0, temp, bias, bias_row_stride, seed, step};
  FS_TRY(check_problem(p, true, out_ids, out_max));
  if (B == 0) return FS_OK;
  if (d < 64) return fail(FS_ERR_UNSUPPORTED, "the unfused path needs d >= 64");
  if (logits_out != nullptr) {
    FS_TRY(check_device_ptr(logits_out, "logits_out"));
    FS_TRY(check_aligned(logits_out, 4, "logits_out"));
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (V == 0) {
    Finish f{};
    f.write_out = true;
    f.out_ids = out_ids;
    f.out_max = out_max;
    cudaError_t e = launch_reduce(f, B, stream);
    if (e != cudaSuccess) return cuda_fail(e, "reduction kernel launch");
    return FS_OK;
  }
  int dev;
  FS_TRY(current_device(&dev));
  const size_t plane = (static_cast<size_t>(B) * static_cast<size_t>(V) * 4 + 255) & ~size_t(255);
  char* buf = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace& ws = g_workspaces[{dev, stream}];
    FS_TRY(grow(&ws.unfused, &ws.unfused_bytes, (logits_out ? plane : 2 * plane) + unfused_partial_bytes(B),
                stream));
    buf = static_cast<char*>(ws.unfused);
  }
  float* logits = logits_out ? logits_out : reinterpret_cast<float*>(buf);
  float* probs = reinterpret_cast<float*>(logits_out ? buf : buf + plane);
  void* partials = logits_out ? buf + plane : buf + 2 * plane;
  int* err = nullptr;
  FS_TRY(error_word(&err, stream));
  cudaError_t e = launch_tc_logits(p, logits, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "logits GEMM launch");
  e = launch_unfused_tail(p, logits, probs, partials, out_ids, out_max, stream);
  if (e != cudaSuccess) return cuda_fail(e, "softmax / sample launch");
  return FS_OK;
}

size_t fs_workspace_bytes(int64_t B, int64_t V) {
  (void)V;
  return finish_bytes_for(B);
}

fs_status fs_workspace_reserve(int64_t B, int64_t V, void* stream) {
  g_last_error[0] = '\0';
  if (B < 0 || V < 0) return fail(FS_ERR_INVALID_ARG, "need B >= 0 and V >= 0");
  int* err = nullptr;
  FS_TRY(error_word(&err, static_cast<cudaStream_t>(stream)));   // once per device, never during capture
  Finish f{};
  return get_finish(static_cast<cudaStream_t>(stream), B, &f);
}

fs_status fs_workspace_release(void) {
  int dev;
  FS_TRY(current_device(&dev));
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  for (auto it = g_workspaces.begin(); it != g_workspaces.end();) {
    if (it->first.first == dev) {
      cudaStreamSynchronize(it->first.second);
      if (it->second.finish) cudaFree(it->second.finish);
      if (it->second.unfused) cudaFree(it->second.unfused);
      if (it->second.host_out) cudaFreeHost(it->second.host_out);
      if (it->second.staging) cudaFree(it->second.staging);
      if (it->second.topk) cudaFree(it->second.topk);
      it = g_workspaces.erase(it);
    } else {
      ++it;
    }
  }
  return FS_OK;
}

fs_status fs_set_path(int path) {
  if (path < FS_PATH_AUTO || path > FS_PATH_TC_PAIR) return fail(FS_ERR_INVALID_ARG, "unknown path %d", path);
  g_forced_path.store(path);
  return FS_OK;
}

fs_status fs_debug_set_fault(int kind) {
  g_last_error[0] = '\0';
  if (kind < FS_FAULT_NONE || kind > FS_FAULT_LAUNCH) return fail(FS_ERR_INVALID_ARG, "unknown fault kind %d", kind);
  g_fault.store(kind);
  return FS_OK;
}

fs_status fs_set_launch_overlap(int enable) {
  g_last_error[0] = '\0';
  if (enable != 0 && enable != 1) return fail(FS_ERR_INVALID_ARG, "enable must be 0 or 1 (got %d)", enable);
  g_launch_overlap.store(enable);
  return FS_OK;
}

int fs_path_for_batch(int64_t B) { return resolve_path(B, 4096); }

int fs_path_for_chunks(int64_t B, int64_t V_chunk, int step_chunks) {
  Problem p{};
  p.B = B;
  p.d = 4096;
  p.V_local = V_chunk;
  p.chunk = true;
  p.step_chunks = step_chunks;
  return resolve_call_path(p);
}

fs_status fs_profile_events(void* start, void* stop) {
  if ((start == nullptr) != (stop == nullptr))
    return fail(FS_ERR_INVALID_ARG, "pass both events or neither");
  g_prof_start = static_cast<cudaEvent_t>(start);
  g_prof_stop = static_cast<cudaEvent_t>(stop);
  return FS_OK;
}

fs_status fs_device_error(int* code) {
  if (code == nullptr) return fail(FS_ERR_INVALID_ARG, "code is NULL");
  *code = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  // the library's word, if any call on this device created it (reading
  // allocates nothing, so callers of fs_sample_noalloc may call this too)
  int* w = existing_error_word();
  if (w != nullptr) {
    e = cudaMemcpy(code, w, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(w, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  }
  // fs_sample_noalloc's word, in its static scratch
  int na = 0;
  e = noalloc_take_status(&na);
  if (e != cudaSuccess) return cuda_fail(e, "reading the allocation-free entry point's status word");
  if (*code == 0) *code = na;
  return FS_OK;
}

fs_status fs_debug_wait_timeout(uint64_t timeout_ns, void* stream) {
  g_last_error[0] = '\0';
  if (timeout_ns == 0 || timeout_ns > 1000000000ull)
    return fail(FS_ERR_INVALID_ARG, "timeout_ns must be in (0, 1e9]");
  int* err = nullptr;
  FS_TRY(error_word(&err, static_cast<cudaStream_t>(stream)));
  cudaError_t e = launch_debug_wait(err, timeout_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait kernel launch");
  return FS_OK;
}

const char* fs_status_string(fs_status s) {
  switch (s) {
    case FS_OK: return "FS_OK";
    case FS_ERR_INVALID_ARG: return "FS_ERR_INVALID_ARG";
    case FS_ERR_UNSUPPORTED: return "FS_ERR_UNSUPPORTED";
    case FS_ERR_CUDA: return "FS_ERR_CUDA";
    case FS_ERR_WORKSPACE: return "FS_ERR_WORKSPACE";
    case FS_ERR_DEVICE_TIMEOUT: return "FS_ERR_DEVICE_TIMEOUT";
  }
  return "FS_STATUS_UNKNOWN";
}

const char* fs_last_error(void) { return g_last_error; }

fs_status fs_debug_noise(uint64_t seed, uint64_t step, int64_t row0, int64_t n_rows,
                         int64_t v0, int64_t n_vocab, uint32_t* words, float* gumbel,
                         void* stream) {
  g_last_error[0] = '\0';
  if (row0 < 0 || n_rows < 0 || v0 < 0 || n_vocab < 0)
    return fail(FS_ERR_INVALID_ARG, "negative range");
  if (row0 + n_rows > (int64_t(1) << 32) || v0 + n_vocab > (int64_t(1) << 31))
    return fail(FS_ERR_UNSUPPORTED, "rows must be < 2^32 and vocabulary ids < 2^31");
  if (n_rows * n_vocab == 0) return FS_OK;
  if (words) FS_TRY(check_device_ptr(words, "words"));
  if (gumbel) FS_TRY(check_device_ptr(gumbel, "gumbel"));
  cudaError_t e = launch_debug_noise(seed, step, row0, n_rows, v0, n_vocab, words, gumbel,
                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "noise kernel launch");
  return FS_OK;
}

}  // extern "C"
