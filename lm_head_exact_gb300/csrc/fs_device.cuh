// Device primitives shared by every sampling kernel of libflashsample:
// the counter-based noise, the Gumbel transform, the per-row temperature
// mode and the total-order (max, argmax) combine.
//
// Method: FlashSampling: Fast and Memory-Efficient Exact Sampling -- summary
// page, "Method": each vocabulary tile gets per-element Gumbel noise, only
// one (max, argmax) per row and tile survives, and a small reduction over
// tiles finishes the sample; "Key claims": argmax decomposes over any
// partition of the vocabulary, so the result does not depend on the tiling.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace fs {

// Sentinel id of "no candidate yet" inside the kernels; it loses every
// comparison against a recorded candidate and is reported as id -1.
constexpr int32_t kNoId = 0x7fffffff;

// -------------------------------------------------------------------------
// Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11, section 4).  Ten rounds of two 32x32->64
// multiplies; the high halves are xored with the other words and the round
// key, the key advances by the Weyl increments between rounds.
// -------------------------------------------------------------------------
struct PhiloxKey {
  uint32_t k0, k1;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
  uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The four draws of vocabulary ids 4q .. 4q+3 for batch row b at a decode
// step: counter (q, b, step lo, step hi) under key (seed lo, seed hi); word
// j of the result belongs to vocabulary id 4q + j.
__device__ __forceinline__ uint4 noise_words(PhiloxKey key, uint32_t q, uint32_t b,
                                             uint32_t step_lo, uint32_t step_hi) {
  return philox4x32_10(make_uint4(q, b, step_lo, step_hi), key);
}

__device__ __forceinline__ uint32_t word_of(uint4 w, uint32_t j) {
  return j == 0 ? w.x : (j == 1 ? w.y : (j == 2 ? w.z : w.w));
}

// u = ((x >> 9) + 1/2) * 2^-23: the odd multiples of 2^-24 in (0, 1).  The
// fused multiply-add is exact here (a 23-bit integer times a power of two
// plus a smaller power of two), so u is the same value the fp64 reference
// forms.
__device__ __forceinline__ float uniform_from_word(uint32_t x) {
  return __fmaf_rn(__uint2float_rn(x >> 9), 0x1p-23f, 0x1p-24f);
}

// Standard Gumbel quantile g = -log(-log u).  The inner logarithm needs a
// small RELATIVE error near u = 1 (where -log u is about 6e-8), so it uses
// the accurate logf; the outer one only needs a small absolute error and
// uses the fast hardware logarithm.  Total error stays below ~1e-5 over the
// whole grid of u.
__device__ __forceinline__ float gumbel_from_uniform(float u) {
  return -__logf(-logf(u));
}

__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
  return gumbel_from_uniform(uniform_from_word(x));
}

// Upper bound of every value gumbel_from_word returns: the largest Gumbel
// value of the uniform grid, -log(-log(1 - 2^-24)) = 16.63553..., rounded up
// (the device transform is within 2e-6 of it and largest at the top grid
// point, checked over the whole grid).
constexpr float kGumbelMax = 16.6356f;

// -------------------------------------------------------------------------
// Per-row temperature mode.  T > 0: z = logit * (1/T) + g.  T == 0: greedy,
// z = logit.  T < 0 or NaN: the row has no valid sample (id -1).
// -------------------------------------------------------------------------
enum RowMode : int { kRowSample = 0, kRowGreedy = 1, kRowInvalid = 2 };

struct RowTemp {
  float inv_t;
  int mode;
};

__device__ __forceinline__ RowTemp row_temp(float t) {
  RowTemp r;
  if (t > 0.0f) {
    r.inv_t = 1.0f / t;
    r.mode = kRowSample;
  } else if (t == 0.0f) {
    r.inv_t = 1.0f;
    r.mode = kRowGreedy;
  } else {  // negative or NaN
    r.inv_t = 0.0f;
    r.mode = kRowInvalid;
  }
  return r;
}

// -------------------------------------------------------------------------
// Total order of candidates: a larger score wins; equal scores go to the
// smaller vocabulary id.  NaN and -inf never become candidates (the callers
// only record a score that beats the running best, which starts at -inf),
// so the recorded best always has z > -inf or is the (-inf, kNoId) identity.
// -------------------------------------------------------------------------
struct Best {
  float z;
  int32_t id;
};

__device__ __forceinline__ Best best_none() {
  Best b;
  b.z = -INFINITY;
  b.id = kNoId;
  return b;
}

__device__ __forceinline__ bool beats(float z, int32_t id, float bz, int32_t bid) {
  return z > bz || (z == bz && id < bid);
}

__device__ __forceinline__ Best combine(Best a, Best b) {
  return beats(b.z, b.id, a.z, a.id) ? b : a;
}

__device__ __forceinline__ Best warp_combine(Best b) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Best o;
    o.z = __shfl_xor_sync(0xffffffffu, b.z, off);
    o.id = __shfl_xor_sync(0xffffffffu, b.id, off);
    b = combine(b, o);
  }
  return b;
}

// One (max, argmax) candidate summary of a (row, part) pair, as stored in the
// partial buffer between the fused kernel and the cross-part reduction.
struct __align__(8) Partial {
  float z;
  int32_t id;
};

// -------------------------------------------------------------------------
// Packed candidate keys: one 64-bit word per row whose unsigned order is the
// total order above, so atomicMax over all CTAs' candidates is the cross-tile
// reduction (order-independent, hence deterministic).  High 32 bits: z mapped
// to an order-preserving unsigned; low 32 bits: 0xFFFFFFFF - id (a smaller id
// is larger).  0 means "no candidate" and is below every real key.  -0.0 is
// keyed as +0.0: the two scores are equal under the total order, so between
// them the smaller id must win, as it does in beats() and in the oracle.
// -------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long pack_key(float z, int32_t id) {
  if (id == kNoId) return 0ull;
  uint32_t u = __float_as_uint(z);
  if (u == 0x80000000u) u = 0u;
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(id));
}

__device__ __forceinline__ Best unpack_key(unsigned long long k) {
  if (k == 0ull) return best_none();
  uint32_t u = static_cast<uint32_t>(k >> 32);
  u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
  Best b;
  b.z = __uint_as_float(u);
  b.id = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k));
  return b;
}

// -------------------------------------------------------------------------
// Programmatic dependent launch.  A fused kernel lets the next kernel of its
// stream start as soon as every CTA has begun (launch_dependents), and waits
// for the previous kernel of its stream to complete (wait) only before it
// touches the cross-CTA finish area and the carry, which consecutive chunk
// launches share.  Without a programmatic launch both are no-ops.
// -------------------------------------------------------------------------
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Device error word: set by kernels whose bounded waits run out; read and
// cleared by the host through fs_device_error().
enum DeviceError : int {
  kDevOk = 0,
  kDevWaitTimeout = 1,
  kDevBadArgument = 2,
};

}  // namespace fs
