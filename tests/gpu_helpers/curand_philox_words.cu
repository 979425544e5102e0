// Test helper (not part of the library): prints the Philox-4x32-10 words that
// cuRAND's device API returns, called as a library, for the (row, id, step)
// triples given on stdin.  Counter mapping used by the sampler: key =
// (seed lo, seed hi), counter = (id >> 2, row, step lo, step hi), word id & 3.
// cuRAND's curand_init(seed, subsequence, offset) sets the key from the seed,
// the counter's upper 64 bits from the subsequence and advances the lower 64
// bits by offset / 4 (word offset % 4), so subsequence = step and
// offset = (row << 34) + 4 * (id >> 2) reach the same counter.
#include <cstdio>
#include <cstdint>
#include <vector>
#include <curand_kernel.h>

__global__ void words_kernel(unsigned long long seed, const unsigned long long* row, const unsigned long long* id,
                             const unsigned long long* step, int n, unsigned int* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  curandStatePhilox4_32_10_t st;
  const unsigned long long offset = (row[i] << 34) + 4ull * (id[i] >> 2);
  curand_init(seed, step[i], offset, &st);
  const uint4 w = curand4(&st);
  const unsigned int k = static_cast<unsigned int>(id[i] & 3);
  out[i] = k == 0 ? w.x : k == 1 ? w.y : k == 2 ? w.z : w.w;
}

int main() {
  unsigned long long seed;
  int n;
  if (scanf("%llu %d", &seed, &n) != 2 || n <= 0 || n > 100000) return 2;
  std::vector<unsigned long long> row(n), id(n), step(n);
  for (int i = 0; i < n; ++i)
    if (scanf("%llu %llu %llu", &row[i], &id[i], &step[i]) != 3) return 2;
  unsigned long long *d_row, *d_id, *d_step;
  unsigned int* d_out;
  if (cudaMalloc(&d_row, n * 8) || cudaMalloc(&d_id, n * 8) || cudaMalloc(&d_step, n * 8) || cudaMalloc(&d_out, n * 4))
    return 3;
  cudaMemcpy(d_row, row.data(), n * 8, cudaMemcpyHostToDevice);
  cudaMemcpy(d_id, id.data(), n * 8, cudaMemcpyHostToDevice);
  cudaMemcpy(d_step, step.data(), n * 8, cudaMemcpyHostToDevice);
  words_kernel<<<(n + 127) / 128, 128>>>(seed, d_row, d_id, d_step, n, d_out);
  std::vector<unsigned int> out(n);
  if (cudaMemcpy(out.data(), d_out, n * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return 4;
  for (int i = 0; i < n; ++i) printf("%u\n", out[i]);
  return 0;
}
