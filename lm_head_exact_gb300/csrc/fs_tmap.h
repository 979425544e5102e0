// TMA tensor-map encoding for the tensor-core kernels (host side).
#pragma once

#include <cuda.h>

#include <cstdint>

namespace fs {

// Encode a 2-D tensor map over a row-major bf16 matrix [rows, d] whose boxes
// are box_cols elements (the contiguous K direction) by box_rows rows, stored
// in shared memory with the 128-byte swizzle the tcgen05 K-major descriptors
// expect.  Out-of-range rows / columns of a box read as zero.  Returns false
// if the driver entry point is unavailable or rejects the description.
bool encode_kmajor_bf16(CUtensorMap* tm, const void* base, int64_t rows, int64_t d, int box_cols,
                        int box_rows);

}  // namespace fs
