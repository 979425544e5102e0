// Tensor-core fused LM-head sampler, batch-major, one CTA per MMA: used for
// 64 < B <= 128 and for batches that do not fill 256-row CTA-pair tiles (the
// pair kernel, fs_tc_pair.cu, takes the rest).  W tiles are shared by the
// batch tiles of a CTA group through L2; from B ~ 300 on the contraction
// bounds the step.
//
// FlashSampling: Fast and Memory-Efficient Exact Sampling -- summary page,
// "Method": the logit tile is formed on chip, Gumbel noise is added in-tile,
// and only a per-row (max, argmax) survives; arXiv abstract: "keep only one
// maximizer per row and per vocabulary tile, and finish with a small
// reduction over tiles".
//
// Mapping on GB300 (sm_103a):
//   * Tile = 128 batch rows (MMA M; A = h tile) x 256 vocabulary rows (MMA N;
//     B = W tile), K = 64 per stage; tcgen05.mma kind::f16, fp32 accumulators
//     in TMEM, two 256-column accumulators (all 512 columns) so the epilogue
//     of one tile overlaps the MMAs of the next.
//   * CTA grouping: with nbt = ceil(B / 128) batch tiles, the grid is cut into
//     groups of nbt CTAs.  CTA c keeps batch tile c % nbt for its whole life
//     and walks the vocabulary tiles q, q + n_groups, ... (q = c / nbt).  The
//     nbt CTAs of a group read the same W tile at the same time, so W comes
//     from HBM once per group and from L2 for the others, and every epilogue
//     thread keeps ITS batch row's running (max, argmax) in registers across
//     all of the CTA's tiles and pushes one candidate per (row, CTA) at the
//     end; the last CTA to finish writes the sample (fs_finish.cuh).
//   * Warp roles: kEpi epilogue warps (TMEM lane = batch row; warps w, w + 4,
//     ... share lanes and split the 256 columns into kEpi / 4 parts), then
//     the TMA producer and the TMEM allocator + MMA issuer.  The sampler runs
//     16 epilogue warps when one batch tile covers the batch (B <= 128: the
//     last tile's epilogue is exposed there; 172 -> 167 us at B = 128 in
//     interleaved runs) and 8 above (B = 600: 471 vs 481 us with 16); the
//     top-k variants run 8 (at 18 warps a thread gets 96 registers, too few
//     for the lists).
//   * Epilogue per element: z = logit * (1/T) + Gumbel(Philox); one Philox
//     call serves the four consecutive vocabulary ids that share a counter.
#include <cuda.h>

#include <algorithm>

#include "fs_epilogue.cuh"
#include "fs_finish.cuh"
#include "fs_internal.h"
#include "fs_sm100.cuh"
#include "fs_tmap.h"

namespace fs {
namespace {

using namespace sm100;

template <int kEpiWarps>
struct BatchWarps {
  static constexpr int kEpi = kEpiWarps;
  static constexpr int kParts = kEpi / 4;
  static constexpr int kProducer = kEpi;
  static constexpr int kMma = kEpi + 1;
  static constexpr int kThreads = (kEpi + 2) * 32;
};
constexpr int kMaxColParts = 4;
constexpr int kBM = 128;            // batch rows per tile (MMA M)
constexpr int kBN = 256;            // vocabulary rows per tile (MMA N)
constexpr int kBK = 64;             // K per stage
constexpr int kStages = 4;
constexpr int kATileBytes = kBM * kBK * 2;     // 16 KB
constexpr int kBTileBytes = kBN * kBK * 2;     // 32 KB
constexpr int kTmemCols = 512;                 // two 256-column accumulators
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kATileBytes;
constexpr int kOffBars = kOffB + kStages * kBTileBytes;
constexpr int kNumBars = 2 * kStages + 5;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffHalf = kOffMisc + 16;                            // Best[parts - 1][128]: other parts' results
constexpr int kOffTopK = kOffHalf + (kMaxColParts - 1) * kBM * 8;  // top-k mode: Partial[128][K] of one part
constexpr int kSmemBytes = kOffTopK + 1024;
constexpr int smem_bytes(int top_k) { return kSmemBytes + kBM * top_k * 8; }

struct BatchArgs {
  Problem p;            // rows [0, p.B) of this launch's batch slice
  float* logits;        // store-logits mode: [B_slice, V_local] fp32 (row stride V_local)
  Finish f;             // sampling mode: cross-CTA finish of this slice's rows;
                        // top-k mode: f.partials [B, f.n_parts, K], part = CTA group
  int nbt;              // batch tiles of this launch
  int n_groups;         // CTA groups = gridDim.x / nbt
  int n_vt;             // vocabulary tiles = ceil(V_local / 256)
  int* err;
};

// kStoreLogits = false: fused sampling epilogue.  true: the unfused
// comparison path's plain GEMM epilogue, storing logits (+ bias) to HBM.
// kTopK > 0 (with kStoreLogits = false): Gumbel-top-k epilogue -- every
// thread keeps its batch row's K best perturbed scores, and each CTA writes
// its per-row list to f.partials for the merge kernel (no in-kernel finish).
template <bool kStoreLogits, int kTopK, int kEpi>
__global__ void __launch_bounds__(BatchWarps<kEpi>::kThreads, 1)
tc_batch_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
                const BatchArgs args) {
  constexpr int kEpiWarps = BatchWarps<kEpi>::kEpi;
  constexpr int kColParts = BatchWarps<kEpi>::kParts;
  constexpr int kProducerWarp = BatchWarps<kEpi>::kProducer;
  constexpr int kMmaWarp = BatchWarps<kEpi>::kMma;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty_bar = full_bar + kStages;
  uint64_t* tfull_bar = empty_bar + kStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* last_flag = reinterpret_cast<int*>(smem + kOffMisc + 8);
  if (!kStoreLogits && kTopK == 0 && early_done_cta(args.f, last_flag)) {
    early_skip_cta(args.f, args.p.B, args.p.pdl, last_flag);
    return;
  }
  Best* part_best = reinterpret_cast<Best*>(smem + kOffHalf);

  const Problem& p = args.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bt = blockIdx.x % args.nbt;
  const int q = blockIdx.x / args.nbt;
  const int n_tiles = q < args.n_vt ? (args.n_vt - 1 - q) / args.n_groups + 1 : 0;
  const int n_kb = static_cast<int>((p.d + kBK - 1) / kBK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], kEpiWarps * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmap_h);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem_base = *tmem_base_slot;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int64_t n_issued = 0;
      bool ok = true;
      // Deferred inputs: the first ring of stages (stage i = K step i mod
      // n_kb) gets its W boxes before the dependency wait, its h boxes after.
      bool h_ready = kStoreLogits || !p.defer_inputs;
      auto load_deferred_h = [&]() {
        pdl_wait();
        for (int64_t i = 0; i < n_issued; ++i)
          tma_load_2d(smem + kOffA + i * kATileBytes, &tmap_h, &full_bar[i], static_cast<int32_t>((i % n_kb) * kBK),
                      bt * kBM, pol_h);
        h_ready = true;
      };
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int vt = q + t * args.n_groups;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, args.err, abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_bar[stage], kATileBytes + kBTileBytes);
          if (h_ready)
            tma_load_2d(smem + kOffA + stage * kATileBytes, &tmap_h, &full_bar[stage], kb * kBK, bt * kBM,
                        pol_h);
          tma_load_2d(smem + kOffB + stage * kBTileBytes, &tmap_w, &full_bar[stage], kb * kBK, vt * kBN,
                      pol_w);
          ++n_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
          if (!h_ready && n_issued == kStages) load_deferred_h();
        }
      }
      if (!h_ready) load_deferred_h();   // fewer issues than stages (or an early stop)
      if (!ok) {
        volatile int no_abort = 0;
        for (int64_t i = std::max<int64_t>(0, n_issued - kStages); i < n_issued; ++i)
          mbar_wait(&full_bar[i % kStages], static_cast<uint32_t>((i / kStages) & 1), args.err, &no_abort);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int acc = t & 1;
        const uint32_t acc_phase = (t >> 1) & 1;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, args.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kBN;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, args.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + kOffA + stage * kATileBytes);
          const uint32_t b_addr = smem_u32(smem + kOffB + stage * kBTileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16(d_tmem, smem_desc_k128(a_addr + k * 32), smem_desc_k128(b_addr + k * 32), idesc,
                     (kb | k) != 0);
          mma_commit(&empty_bar[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (ok) mma_commit(&tfull_bar[acc]);
      }
      if (!ok) {
        mma_commit(drain_bar);
        volatile int no_abort = 0;
        mbar_wait(drain_bar, 0, args.err, &no_abort);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0 .. kEpi - 1)
    const int quad = warp & 3;                 // TMEM lane quadrant
    const int part = warp >> 2;                // column part of the 256-wide tile
    const int row_in_tile = quad * 32 + lane;
    const int64_t b = static_cast<int64_t>(bt) * kBM + row_in_tile;
    const bool row_ok = b < p.B;
    if (!kStoreLogits && p.defer_inputs) pdl_wait();   // temp (and bias) may come from the preceding kernel
    const RowTemp rt = row_temp(row_ok ? p.temp[b] : -1.0f);
    const bool active = row_ok && rt.mode != kRowInvalid;
    const bool greedy = rt.mode == kRowGreedy;
    const PhiloxKey key{static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32)};
    const uint32_t step_lo = static_cast<uint32_t>(p.step);
    const uint32_t step_hi = static_cast<uint32_t>(p.step >> 32);
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    RowScan scan;
    scan.key = key;
    scan.row = static_cast<uint32_t>(p.row_offset + b);
    scan.step_lo = step_lo;
    scan.step_hi = step_hi;
    scan.inv_t = rt.inv_t;
    scan.greedy = greedy;
    scan.bias_row = p.bias != nullptr ? p.bias + b * p.bias_stride : nullptr;
    Best best = best_none();
    TopList<(kTopK > 0 ? kTopK : 1)> list;
    topk_init(list);

    for (int t = 0; t < n_tiles; ++t) {
      const int acc = t & 1;
      const uint32_t acc_phase = (t >> 1) & 1;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, args.err, abort_flag)) break;
      tc_fence_after();
      const int vt = q + t * args.n_groups;
      const int64_t col0 = static_cast<int64_t>(vt) * kBN + part * (kBN / kColParts);   // local vocabulary row
#pragma unroll 1
      for (int c = 0; c < kBN / kColParts; c += 32) {
        uint32_t r[32];
        tmem_ld_32(tmem_base + lane_addr + acc * kBN + part * (kBN / kColParts) + c, r);
        tmem_ld_wait();
        const int64_t v0 = col0 + c;                       // local id of r[0]
        if (p.dbg_logits != nullptr && row_ok) {          // parity inspection only
#pragma unroll
          for (int j = 0; j < 32; ++j) {                   // unrolled: r stays in registers
            if (v0 + j < p.V_local) {
              float logit = __uint_as_float(r[j]);
              if (p.bias != nullptr) logit += p.bias[b * p.bias_stride + v0 + j];
              p.dbg_logits[b * p.V_local + v0 + j] = logit;
            }
          }
        }
        if constexpr (kStoreLogits) {
          if (row_ok && v0 < p.V_local) {
            float* dst = args.logits + b * p.V_local + v0;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (v0 + j < p.V_local) {
                float logit = __uint_as_float(r[j]);
                if (p.bias != nullptr) logit += p.bias[b * p.bias_stride + v0 + j];
                dst[j] = logit;
              }
            }
          }
        } else if (active && v0 < p.V_local) {
          if constexpr (kTopK > 0) {
            if (scan.bias_row != nullptr)
              scan32_topk<true>(r, v0, p.V_local, p.v_offset, scan, list);
            else
              scan32_topk<false>(r, v0, p.V_local, p.v_offset, scan, list);
          } else {
            if (scan.bias_row != nullptr)
              scan32<true>(r, v0, p.V_local, p.v_offset, scan, best);
            else
              scan32<false>(r, v0, p.V_local, p.v_offset, scan, best);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
    if constexpr (kTopK > 0) {
      // merge the column parts' lists into part 0's (one buffer, one part
      // at a time), then one list per (row, group)
      Partial* other = reinterpret_cast<Partial*>(smem + kOffTopK) + row_in_tile * kTopK;
#pragma unroll 1
      for (int src = 1; src < kColParts; ++src) {
        if (part == src) {
#pragma unroll
          for (int j = 0; j < kTopK; ++j) other[j] = Partial{list.z[j], list.id[j]};
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        if (part == 0) {
#pragma unroll
          for (int j = 0; j < kTopK; ++j) topk_offer(list, other[j].z, other[j].id);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      }
      if (p.pdl) pdl_wait();      // the previous call's merge kernel may still read the partials
      if (part == 0 && row_ok) {
        Partial* dst = args.f.partials + (b * args.f.n_parts + q) * kTopK;
#pragma unroll
        for (int j = 0; j < kTopK; ++j) dst[j] = Partial{list.z[j], list.id[j]};
      }
    }
    // combine the column parts of each row, then one candidate per (row, group)
    if constexpr (!kStoreLogits && kTopK == 0) {
      if (part != 0) part_best[(part - 1) * kBM + row_in_tile] = best;
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      if (part == 0) {
#pragma unroll
        for (int src = 1; src < kColParts; ++src) best = combine(best, part_best[(src - 1) * kBM + row_in_tile]);
      }
      // no dependency wait before the push: this launch's keys and ticket are
      // its own (only the grid's last CTA waits, in finish_grid)
      if (part == 0 && row_ok) push_candidate(args.f, b, best);
      finish_grid(args.f, p.B, threadIdx.x, kEpiWarps * 32, last_flag,
                  named_bar1_and<kEpiWarps * 32>);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace

// Geometry of one launch over a batch slice of B rows.
struct BatchGeometry {
  int nbt, n_groups, grid;
};

// Groups: at most SMs / nbt, then as few as give every group the same number
// of vocabulary tiles (measured: at B = 128, 501 tiles on 126 groups of 4
// instead of 152 groups of 3.3 cut the step from 179.5 to 171.9 us).
static BatchGeometry batch_geometry(int64_t B, int sms, int64_t n_vt) {
  BatchGeometry g;
  g.nbt = static_cast<int>((B + kBM - 1) / kBM);
  g.n_groups = std::max(1, sms / g.nbt);
  const int64_t per = (std::max<int64_t>(n_vt, 1) + g.n_groups - 1) / g.n_groups;
  g.n_groups = static_cast<int>(std::max<int64_t>(1, (std::max<int64_t>(n_vt, 1) + per - 1) / per));
  g.grid = g.n_groups * g.nbt;
  return g;
}

int64_t tc_batch_max_rows_per_launch(int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (sms <= 0) sms = 148;
  return static_cast<int64_t>(sms) * kBM;
}

static cudaError_t launch_batch_impl(const Problem& p, const Finish* f, float* logits, int* err,
                                     cudaStream_t stream) {
  if (p.d < kBK || p.V_local <= 0) return cudaErrorNotSupported;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  const bool store = logits != nullptr;
  cudaError_t e = cudaSuccess;
  if (store) {
    e = raise_smem_limit<tc_batch_kernel<true, 0, 16>>(dev, kSmemBytes);
  } else {
    e = raise_smem_limit<tc_batch_kernel<false, 0, 16>>(dev, kSmemBytes);
    if (e == cudaSuccess) e = raise_smem_limit<tc_batch_kernel<false, 0, 8>>(dev, kSmemBytes);
  }
  if (e != cudaSuccess) return e;
  CUtensorMap tw;
  if (!encode_kmajor_bf16(&tw, p.W, p.V_local, p.d, kBK, kBN)) return cudaErrorInvalidValue;
  const int64_t slice = tc_batch_max_rows_per_launch(dev);
  for (int64_t b0 = 0; b0 < p.B; b0 += slice) {
    Problem ps = p;
    ps.B = std::min<int64_t>(slice, p.B - b0);
    ps.h = static_cast<const uint16_t*>(p.h) + b0 * p.d;
    ps.temp = p.temp + b0;
    if (p.bias != nullptr) ps.bias = p.bias + b0 * p.bias_stride;
    ps.row_offset = p.row_offset + b0;
    if (p.dbg_logits != nullptr) ps.dbg_logits = p.dbg_logits + b0 * p.V_local;
    // The slices of one call share the ticket counter: a later slice starts
    // after the previous one has completed (and left the counter at zero).
    ps.pdl = p.pdl && b0 == 0;
    Finish fs_slice{};
    if (!store) {            // this launch finishes rows [b0, b0 + ps.B)
      fs_slice = *f;
      fs_slice.keys = f->keys + b0;
      if (f->carry_max != nullptr) {
        fs_slice.carry_max = f->carry_max + b0;
        fs_slice.carry_ids = f->carry_ids + b0;
      }
      if (f->write_out) {
        fs_slice.out_ids = f->out_ids + b0;
        fs_slice.out_max = f->out_max + b0;
      }
    }
    const BatchGeometry g = batch_geometry(ps.B, sms, (p.V_local + kBN - 1) / kBN);
    CUtensorMap th;
    if (!encode_kmajor_bf16(&th, ps.h, ps.B, p.d, kBK, kBM)) return cudaErrorInvalidValue;
    BatchArgs a{ps, store ? logits + b0 * p.V_local : nullptr, fs_slice, g.nbt, g.n_groups,
                static_cast<int>((p.V_local + kBN - 1) / kBN), err};
    if (store) {
      tc_batch_kernel<true, 0, 16><<<g.grid, BatchWarps<16>::kThreads, kSmemBytes, stream>>>(th, tw, a);
      e = cudaGetLastError();
    } else if (g.nbt == 1) {
      e = launch_kernel(tc_batch_kernel<false, 0, 16>, dim3(g.grid), dim3(BatchWarps<16>::kThreads), kSmemBytes,
                        stream, ps.pdl, th, tw, a);
    } else {
      e = launch_kernel(tc_batch_kernel<false, 0, 8>, dim3(g.grid), dim3(BatchWarps<8>::kThreads), kSmemBytes,
                        stream, ps.pdl, th, tw, a);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_tc_batch(const Problem& p, const Finish& f, int* err, cudaStream_t stream) {
  return launch_batch_impl(p, &f, nullptr, err, stream);
}

cudaError_t launch_tc_logits(const Problem& p, float* logits, int* err, cudaStream_t stream) {
  return launch_batch_impl(p, nullptr, logits, err, stream);
}

int tc_topk_parts(int64_t B, int64_t V, int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (sms <= 0) sms = 148;
  return batch_geometry(B, sms, (V + kBN - 1) / kBN).n_groups;
}

template <int K>
static cudaError_t launch_topk_k(const Problem& p, Partial* partials, int* err, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  if (p.B > static_cast<int64_t>(sms) * kBM) return cudaErrorNotSupported;   // one launch
  cudaError_t e = raise_smem_limit<tc_batch_kernel<false, K, 8>>(dev, smem_bytes(K));
  if (e != cudaSuccess) return e;
  CUtensorMap tw, th;
  if (!encode_kmajor_bf16(&tw, p.W, p.V_local, p.d, kBK, kBN)) return cudaErrorInvalidValue;
  if (!encode_kmajor_bf16(&th, p.h, p.B, p.d, kBK, kBM)) return cudaErrorInvalidValue;
  const BatchGeometry g = batch_geometry(p.B, sms, (p.V_local + kBN - 1) / kBN);
  Problem ps = p;
  Finish f{};
  f.partials = partials;
  f.n_parts = g.n_groups;
  BatchArgs a{ps, nullptr, f, g.nbt, g.n_groups, static_cast<int>((p.V_local + kBN - 1) / kBN), err};
  return launch_kernel(tc_batch_kernel<false, K, 8>, dim3(g.grid), dim3(BatchWarps<8>::kThreads), smem_bytes(K), stream,
                       ps.pdl, th,
                       tw, a);
}

cudaError_t launch_tc_topk(const Problem& p, int K, Partial* partials, int* err, cudaStream_t stream) {
  if (p.d < kBK || p.V_local <= 0) return cudaErrorNotSupported;
  switch (K) {
    case 4: return launch_topk_k<4>(p, partials, err, stream);
    case 8: return launch_topk_k<8>(p, partials, err, stream);
    case 16: return launch_topk_k<16>(p, partials, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fs
