// Evaluates the library's own device noise transform (fs::gumbel_from_word,
// lm_head_exact_gb300/csrc/fs_device.cuh) on EVERY point of its uniform grid:
// the word m << 9 for m in [0, 2^23), i.e. u = (m + 1/2) 2^-23, the only
// values the sampler's u can take.  Writes the 2^23 fp32 Gumbel values, in
// order of m, to the file named by argv[1]; exit status 0 on success.
#include <cstdint>
#include <cstdio>
#include <vector>

#include "fs_device.cuh"

namespace {

constexpr uint32_t kGrid = 1u << 23;

__global__ void grid_kernel(float* out) {
  const uint32_t m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < kGrid) out[m] = fs::gumbel_from_word(m << 9);
}

}  // namespace

int main(int argc, char** argv) {
  if (argc != 2) {
    std::fprintf(stderr, "usage: %s OUT_FILE\n", argv[0]);
    return 2;
  }
  float* d = nullptr;
  if (cudaMalloc(&d, kGrid * sizeof(float)) != cudaSuccess) return 3;
  grid_kernel<<<kGrid / 256, 256>>>(d);
  std::vector<float> h(kGrid);
  const cudaError_t e = cudaMemcpy(h.data(), d, kGrid * sizeof(float), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) {
    std::fprintf(stderr, "CUDA error: %s\n", cudaGetErrorString(e));
    return 4;
  }
  FILE* f = std::fopen(argv[1], "wb");
  if (f == nullptr) return 5;
  const size_t n = std::fwrite(h.data(), sizeof(float), kGrid, f);
  std::fclose(f);
  return n == kGrid ? 0 : 6;
}
