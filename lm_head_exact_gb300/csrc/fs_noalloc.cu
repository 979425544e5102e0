// fs_sample_noalloc: the tensor-core sampling path with its scratch memory in
// a fixed, statically allocated device array instead of the library's
// cudaMalloc'ed workspace.  It always runs the vocabulary-major tensor-core
// kernel, whatever the batch size (fs_sample picks the family from B).  The
// tensor-core families form the same logits bit for bit, so its results
// equal fs_sample's wherever fs_sample runs a tensor-core kernel (every
// 2 <= B <= 256 under the automatic rule) and agree with them within the
// parity tolerance at B = 1, where fs_sample runs the CUDA-core kernel.
//
// Why it exists: fs_sample finishes the sample through a small workspace (a
// ticket counter and one packed candidate key per batch row) that the
// library allocates with cudaMalloc the first time a (device, stream) needs
// it, and re-allocates when a larger batch arrives.
// Some callers cannot let a library do that: serving stacks whose allocator
// has already claimed the device memory budget (a library cudaMalloc then
// fails or fragments memory it does not own), and callers that must not pay
// for the device-wide synchronization cudaFree implies when a workspace is
// replaced.  This entry point never allocates or frees device memory.
//
// The scratch lives in `g_noalloc_scratch` below, a file-scope static
// __device__ array of kScratchBytes (2.3 KB: a 256-byte header holding the
// bounded-wait status word and the ticket counter, then 256 candidate keys)
// that every GPU loading the library keeps until the process exits.  Host
// code cannot use the array's name as a device address (it is a host-side
// stand-in), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, zeroes the whole array,
// and caches the pointer for later calls on that device.  Make that first
// call on each device before any stream capture begins.
//
// Every call on a device shares the one array and finds the previous call's
// contents in it.  The ticket and the keys must start each call at zero; the
// kernel's last CTA zeroes them again before the call completes, so they are
// zero for the next call.  Calls whose kernels overlap on the GPU (for
// example on two streams without ordering between them) race on the array
// and may return wrong samples: order them on one stream.
//
// The kernel's bounded waits report a timeout to the status word at the
// start of the array; fs_device_error() reads and clears it (together with
// the library's own error word) without allocating anything.
#include <cstdio>
#include <cstdint>
#include <mutex>

#include "flashsample.h"
#include "fs_internal.h"

namespace fs {
namespace {

// Largest batch this entry point accepts (the tensor-core vocabulary-major
// kernel's limit): one packed candidate key per batch row.
constexpr int64_t kNoAllocMaxBatch = 256;
constexpr size_t kHeaderBytes = 256;   // [0]: bounded-wait status word, [64]: ticket counter
constexpr size_t kCounterOffset = 64;
constexpr size_t kScratchBytes = kHeaderBytes + kNoAllocMaxBatch * sizeof(unsigned long long);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

fs_status noalloc_fail(fs_status s, const char* msg) {
  char buf[256];
  snprintf(buf, sizeof(buf), "fs_sample_noalloc: %s", msg);
  record_error(buf);
  return s;
}

// Device address of the static scratch on the current device; the first
// call per device resolves it and zeroes the whole array on `stream`, the
// stream of the call's kernel, so the kernel is ordered after the zeroing.
fs_status scratch_for_current_device(cudaStream_t stream, unsigned char** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(FS_ERR_CUDA, "cannot query the current device");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return noalloc_fail(FS_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    }
    e = cudaMemsetAsync(ptr, 0, kScratchBytes, stream);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return noalloc_fail(FS_ERR_CUDA, "clearing the static scratch failed");
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return FS_OK;
}

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

}  // namespace

cudaError_t noalloc_take_status(int* code) {
  *code = 0;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
  int* word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    word = static_cast<int*>(g_scratch_ptr[dev]);
  }
  if (word == nullptr) return cudaSuccess;          // the entry point never ran on this device
  e = cudaMemcpy(code, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(word, 0, sizeof(int));
  return e;
}

}  // namespace fs

using namespace fs;

extern "C" FS_API fs_status fs_sample_noalloc(const void* h, const void* W, int64_t B, int64_t d,
                                              int64_t V, const float* temp, uint64_t seed,
                                              uint64_t step, int64_t* out_ids, float* out_max,
                                              void* stream_) {
  record_error("");
  if (B < 0 || d <= 0 || V < 0) return noalloc_fail(FS_ERR_INVALID_ARG, "need B >= 0, d > 0, V >= 0");
  if (B > kNoAllocMaxBatch)
    return noalloc_fail(FS_ERR_UNSUPPORTED, "B exceeds 256, the static scratch's batch limit");
  if (d < 64) return noalloc_fail(FS_ERR_UNSUPPORTED, "d must be at least 64");
  if (d % 8 != 0) return noalloc_fail(FS_ERR_UNSUPPORTED, "d must be a multiple of 8");
  if (V >= (int64_t(1) << 31)) return noalloc_fail(FS_ERR_UNSUPPORTED, "V must be < 2^31");
  if (B == 0) return FS_OK;
  if (!h || !temp || !out_ids || !out_max || (V > 0 && !W))
    return noalloc_fail(FS_ERR_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(h) % 16 || reinterpret_cast<uintptr_t>(W) % 16)
    return noalloc_fail(FS_ERR_UNSUPPORTED, "h and W must be 16-byte aligned");
  // the kernel stores int64 ids and fp32 maxima and loads fp32 temperatures:
  // a misaligned pointer is rejected here rather than faulting on the device
  if (reinterpret_cast<uintptr_t>(temp) % 4)
    return noalloc_fail(FS_ERR_UNSUPPORTED, "temp must be 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(out_ids) % 8)
    return noalloc_fail(FS_ERR_UNSUPPORTED, "out_ids must be 8-byte aligned");
  if (reinterpret_cast<uintptr_t>(out_max) % 4)
    return noalloc_fail(FS_ERR_UNSUPPORTED, "out_max must be 4-byte aligned");
  if (!is_device_ptr(h) || !is_device_ptr(temp) || !is_device_ptr(out_ids) || !is_device_ptr(out_max) ||
      (V > 0 && !is_device_ptr(W)))
    return noalloc_fail(FS_ERR_INVALID_ARG, "h, W, temp, out_ids and out_max must be device memory");

  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  unsigned char* scratch = nullptr;
  fs_status s = scratch_for_current_device(stream, &scratch);
  if (s != FS_OK) return s;
  int* status_word = reinterpret_cast<int*>(scratch);
  Finish f{};
  f.counter = reinterpret_cast<unsigned int*>(scratch + kCounterOffset);
  f.keys = reinterpret_cast<unsigned long long*>(scratch + kHeaderBytes);
  f.write_out = true;
  f.out_ids = out_ids;
  f.out_max = out_max;
  Problem p{h, W, B, d, V, 0, temp, nullptr, 0, seed, step};
  cudaError_t e = V > 0 ? launch_tc_vocab(p, f, status_word, stream) : launch_reduce(f, B, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return noalloc_fail(FS_ERR_CUDA, "kernel launch failed");
  }
  return FS_OK;
}
