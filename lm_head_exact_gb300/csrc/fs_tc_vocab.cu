// Tensor-core fused LM-head sampler, vocabulary-major: the small / medium
// batch path (B <= 256), where the step is bound by streaming W from HBM.
//
// FlashSampling: Fast and Memory-Efficient Exact Sampling -- summary page,
// "Method": the logit tile is formed on chip, Gumbel noise is added in-tile,
// and only a per-row (max, argmax) per tile survives; arXiv abstract: "keep
// only one maximizer per row and per vocabulary tile".
//
// Mapping on GB300 (sm_103a):
//   * One persistent CTA per SM takes the 128-row vocabulary tiles c, c + G,
//     c + 2G, ... (G = grid size): every tile is one 128-row TMA box of W per
//     K step (measured faster on GB300 than contiguous per-CTA ranges loaded
//     as 32-row boxes: 173 vs 178 us for the Llama-3-8B head at B = 16).
//   * MMA: D[v, b] = sum_k W[v, k] * h[b, k] with tcgen05.mma kind::f16,
//     M = 128 vocabulary rows (A = W tile), N = BN batch rows (B = h tile),
//     K = 64 per pipeline stage; fp32 accumulators in TMEM, double-buffered
//     so the epilogue of one tile overlaps the MMAs of the next.
//   * TMA streams W (evict-first) and h (evict-last) tiles, 128-byte swizzled,
//     through a STAGES-deep shared-memory ring guarded by mbarriers.
//   * Warp roles (192 threads): warps 0-3 epilogue (TMEM lane = vocabulary
//     row), warp 4 TMA producer, warp 5 TMEM allocator + MMA issuer.
//   * Epilogue: each warp transposes its 32 rows x 32 accumulator columns
//     through shared memory; lane j then scans batch column j over the rows in
//     increasing id order: z = logit * (1/T) + Gumbel(Philox), one Philox call
//     per four consecutive ids, running (max, argmax) in registers for the
//     whole CTA range; at the end the 4 warps are combined into one candidate
//     per (batch row, CTA).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "fs_epilogue.cuh"
#include "fs_finish.cuh"
#include "fs_internal.h"
#include "fs_sm100.cuh"
#include "fs_tmap.h"

namespace fs {
namespace {

using namespace sm100;

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kBM = 128;          // vocabulary rows per tile (MMA M)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr int kATileBytes = kBM * kBK * 2;

// kTopK > 0: Gumbel-top-k mode (BN <= 64): per-lane K-lists (one per
// accumulator chunk), one list per (row, CTA) written to partials, no
// in-kernel finish.
template <int BN, int kTopK = 0>
struct VocabCfg {
  static constexpr int kBTileBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes;
  static constexpr int kChunk = BN < 32 ? BN : 32;     // accumulator columns per transpose step
  static constexpr int kChunks = BN / kChunk;
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;     // two accumulators
  // everything but the stage ring: barriers (<= 29), tmem base / flags,
  // per-column 1/T and mode, per-warp bests, transpose tiles, alignment slack
  static constexpr int kTopKBytes = kTopK > 0 ? kEpiWarps * BN * kTopK * 8 : 0;   // per-warp lists
  static constexpr int kFixedBytes =
      29 * 8 + 16 + BN * 8 + kEpiWarps * BN * 8 + kEpiWarps * 32 * 33 * 4 + kTopKBytes + 1024;
  // Resident CTAs per SM: two for narrow batches (measured ~2% faster on
  // GB300 for B <= 32: two independent TMA streams per SM), one otherwise.
  // (Top-k lists need the registers: one CTA per SM there.)
  static constexpr int kCtasPerSm = (BN <= 32 && kTopK == 0) ? 2 : 1;
  static constexpr int kStages = std::min(12, (225 * 1024 / kCtasPerSm - kFixedBytes) / kStageBytes);
  // shared memory carve-up (offsets from a 1024-byte aligned base)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kATileBytes;
  static constexpr int kOffBars = kOffB + kStages * kBTileBytes;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;            // tmem base, abort flag, last-CTA flag
  static constexpr int kOffInvT = kOffMisc + 16;
  static constexpr int kOffMode = kOffInvT + BN * 4;
  static constexpr int kOffBest = kOffMode + BN * 4;
  static constexpr int kOffTr = kOffBest + kEpiWarps * BN * 8;     // per-warp 32 x 33 transpose tiles
  static constexpr int kOffTopK = kOffTr + kEpiWarps * 32 * 33 * 4;
  static constexpr int kSmemBytes = kOffTopK + kTopKBytes + 1024;   // + alignment slack
};

// Parity inspection (Problem::dbg_logits): the logits of batch column b at
// vocabulary rows row0 .. row0 + n - 1, from this lane's transposed column.
// Kept out of line so the sampling epilogue's register allocation is the
// same whether or not the store is compiled in.
__device__ __noinline__ void dump_column(const Problem& p, const float* col, int b, int64_t row0, int n) {
  for (int i = 0; i < n; ++i) {
    float logit = col[i];
    if (p.bias != nullptr) logit += p.bias[static_cast<int64_t>(b) * p.bias_stride + row0 + i];
    p.dbg_logits[static_cast<int64_t>(b) * p.V_local + row0 + i] = logit;
  }
}

struct VocabArgs {
  Problem p;
  Finish f;           // cross-CTA finish: packed keys, ticket, carry, outputs
  int64_t n_vt;       // vocabulary tiles: ceil(V_local / 128)
  int* err;
};

template <int BN, int kTopK = 0>
__global__ void __launch_bounds__(kThreads, VocabCfg<BN, kTopK>::kCtasPerSm)
tc_vocab_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_h,
                const VocabArgs args) {
  using C = VocabCfg<BN, kTopK>;
  static_assert(kTopK == 0 || C::kChunks <= 2, "top-k lists: at most two accumulator chunks per lane");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* tfull_bar = empty_bar + C::kStages;     // [2]
  uint64_t* tempty_bar = tfull_bar + 2;             // [2]
  uint64_t* drain_bar = tempty_bar + 2;             // abort path only
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  int* last_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
  if (kTopK == 0 && early_done_cta(args.f, last_flag)) {
    early_skip_cta(args.f, args.p.B, args.p.pdl, last_flag);
    return;
  }
  float* col_inv_t = reinterpret_cast<float*>(smem + C::kOffInvT);
  int* col_mode = reinterpret_cast<int*>(smem + C::kOffMode);
  Best* warp_best = reinterpret_cast<Best*>(smem + C::kOffBest);   // [kEpiWarps][BN]
  float* tr_all = reinterpret_cast<float*>(smem + C::kOffTr);       // [kEpiWarps][32][33]

  const Problem& p = args.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int B = static_cast<int>(p.B);

  // This CTA's tiles: global tile blockIdx.x + t * gridDim.x, rows [128 g, 128 g + 128) of W.
  const int n_tiles = blockIdx.x < args.n_vt ? static_cast<int>((args.n_vt - 1 - blockIdx.x) / gridDim.x + 1) : 0;
  auto tile_row = [&](int t) { return (static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(t) * gridDim.x) * kBM; };
  const int n_kb = static_cast<int>((p.d + kBK - 1) / kBK);

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
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
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_h);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_slot, C::kTmemCols);
    tmem_relinquish();
  }
  if (!p.defer_inputs) {
    for (int b = threadIdx.x; b < BN; b += kThreads) {
      const RowTemp rt = row_temp(b < B ? p.temp[b] : -1.0f);
      col_inv_t[b] = rt.inv_t;
      col_mode[b] = rt.mode;
    }
  }
  for (int i = threadIdx.x; i < kEpiWarps * BN; i += kThreads) warp_best[i] = best_none();
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
      // With deferred inputs the first ring of stages gets its W boxes before
      // the dependency wait and its h boxes after it (each stage's barrier
      // expects both from the start).  The first kStages issues are stages
      // 0, 1, ... and K steps 0, 1, ... modulo n_kb.
      bool h_ready = !p.defer_inputs;
      auto load_deferred_h = [&]() {
        pdl_wait();
        for (int64_t i = 0; i < n_issued; ++i)
          tma_load_2d(smem + C::kOffB + i * C::kBTileBytes, &tmap_h, &full_bar[i],
                      static_cast<int32_t>((i % n_kb) * kBK), 0, pol_h);
        h_ready = true;
      };
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int64_t row = tile_row(t);
        // rows past V (last tile) are zero-filled and still count as transferred bytes
        const uint32_t bytes = kATileBytes + C::kBTileBytes;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, args.err, abort_flag)) { ok = false; break; }
          uint8_t* a_dst = smem + C::kOffA + stage * kATileBytes;
          uint8_t* b_dst = smem + C::kOffB + stage * C::kBTileBytes;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          tma_load_2d(a_dst, &tmap_w, &full_bar[stage], kb * kBK, static_cast<int32_t>(row), pol_w);
          if (h_ready) tma_load_2d(b_dst, &tmap_h, &full_bar[stage], kb * kBK, 0, pol_h);
          ++n_issued;
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
          if (!h_ready && n_issued == C::kStages) load_deferred_h();
        }
      }
      if (!h_ready) load_deferred_h();   // fewer issues than stages (or an early stop)
      if (!ok) {
        // drain: never leave with copies in flight into this CTA's shared
        // memory -- wait (bounded) for the last load issued into every stage
        volatile int no_abort = 0;
        for (int64_t i = std::max<int64_t>(0, n_issued - C::kStages); i < n_issued; ++i)
          mbar_wait(&full_bar[i % C::kStages], static_cast<uint32_t>((i / C::kStages) & 1), args.err,
                    &no_abort);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int acc = t & 1;
        const uint32_t acc_phase = (t >> 1) & 1;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, args.err, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, args.err, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + C::kOffA + stage * kATileBytes);
          const uint32_t b_addr = smem_u32(smem + C::kOffB + stage * C::kBTileBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            mma_bf16(d_tmem, smem_desc_k128(a_addr + k * 32), smem_desc_k128(b_addr + k * 32), idesc,
                     (kb | k) != 0);
          mma_commit(&empty_bar[stage]);     // frees the stage once these MMAs have read it
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
        if (ok) mma_commit(&tfull_bar[acc]);   // accumulator ready for the epilogue
      }
      if (!ok) {
        // wait (bounded) until every MMA issued so far has finished before TMEM is freed
        mma_commit(drain_bar);
        volatile int no_abort = 0;
        mbar_wait(drain_bar, 0, args.err, &no_abort);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0-3)
    // Each warp owns 32 vocabulary rows (its TMEM lane quadrant).  Per chunk
    // of accumulator columns it transposes the 32 x chunk block through
    // shared memory so that lane j then owns batch column c0 + j and scans the
    // 32 rows in increasing id order: consecutive ids share one Philox call
    // and the running (max, argmax) of (warp, column) stays in registers
    // across all of the CTA's tiles -- no cross-lane reduction per tile.
    if (p.defer_inputs) {        // temp (and bias) may come from the preceding kernel
      pdl_wait();
      for (int b = threadIdx.x; b < BN; b += kEpiWarps * 32) {
        const RowTemp rt = row_temp(b < B ? p.temp[b] : -1.0f);
        col_inv_t[b] = rt.inv_t;
        col_mode[b] = rt.mode;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
    }
    const PhiloxKey key{static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32)};
    const uint32_t step_lo = static_cast<uint32_t>(p.step);
    const uint32_t step_hi = static_cast<uint32_t>(p.step >> 32);
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    float* tr = tr_all + warp * 32 * 33;
    float best_z[C::kChunks];
    int32_t best_id[C::kChunks];
    TopList<(kTopK > 0 ? kTopK : 1)> list[C::kChunks];   // top-k mode: this lane's column of each chunk
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c) topk_init(list[c]);
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c) {
      best_z[c] = -INFINITY;
      best_id[c] = kNoId;
    }
    for (int t = 0; t < n_tiles; ++t) {
      const int acc = t & 1;
      const uint32_t acc_phase = (t >> 1) & 1;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, args.err, abort_flag)) break;
      tc_fence_after();
      const int64_t row0 = tile_row(t) + warp * 32;                     // this warp's first row
      const int n_rows = static_cast<int>(std::max<int64_t>(0, std::min<int64_t>(32, p.V_local - row0)));
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const int c0 = c * C::kChunk;
        if (c0 < B) {                                                 // warp-uniform
          uint32_t r[C::kChunk];
          if constexpr (C::kChunk == 32) {
            tmem_ld_32(tmem_base + lane_addr + acc * BN + c0, r);
          } else {
            tmem_ld_16(tmem_base + lane_addr + acc * BN + c0, r);
          }
          tmem_ld_wait();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < C::kChunk; ++j) tr[j * 33 + lane] = __uint_as_float(r[j]);
          __syncwarp();
          const int b = c0 + lane;
          if (p.dbg_logits != nullptr && lane < C::kChunk && b < B)   // parity inspection only
            dump_column(p, tr + lane * 33, b, row0, n_rows);
          const int mode = (lane < C::kChunk && b < B) ? col_mode[b] : kRowInvalid;
          if (mode != kRowInvalid) {
            RowScan scan;
            scan.key = key;
            scan.row = static_cast<uint32_t>(b);
            scan.step_lo = step_lo;
            scan.step_hi = step_hi;
            scan.inv_t = col_inv_t[b];
            scan.greedy = mode == kRowGreedy;
            scan.bias_row = p.bias != nullptr ? p.bias + static_cast<int64_t>(b) * p.bias_stride : nullptr;
            uint32_t vals[32];
            const float* col = tr + lane * 33;
#pragma unroll
            for (int i = 0; i < 32; ++i) vals[i] = __float_as_uint(col[i]);
            const int64_t row_end = row0 + n_rows;
            if constexpr (kTopK > 0) {
              if (scan.bias_row != nullptr)
                scan32_topk<true>(vals, row0, row_end, p.v_offset, scan, list[c]);
              else
                scan32_topk<false>(vals, row0, row_end, p.v_offset, scan, list[c]);
            } else {
              Best bb;
              bb.z = best_z[c];
              bb.id = best_id[c];
              if (scan.bias_row != nullptr)
                scan32<true>(vals, row0, row_end, p.v_offset, scan, bb);
              else
                scan32<false>(vals, row0, row_end, p.v_offset, scan, bb);
              best_z[c] = bb.z;
              best_id[c] = bb.id;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
    if constexpr (kTopK > 0) {
      // merge the 4 epilogue warps' lists of each column, one list per (row, CTA)
      Partial* lists = reinterpret_cast<Partial*>(smem + C::kOffTopK);   // [kEpiWarps][BN][kTopK]
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const int b = c * C::kChunk + lane;
        if (lane < C::kChunk && b < B) {
#pragma unroll
          for (int j = 0; j < kTopK; ++j) lists[(warp * BN + b) * kTopK + j] = Partial{list[c].z[j], list[c].id[j]};
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      pdl_wait();                 // the previous call's merge kernel may still read the partials
      for (int b = threadIdx.x; b < B; b += kEpiWarps * 32) {
        TopList<(kTopK > 0 ? kTopK : 1)> m;
#pragma unroll
        for (int j = 0; j < kTopK; ++j) {
          m.z[j] = lists[b * kTopK + j].z;
          m.id[j] = lists[b * kTopK + j].id;
        }
        for (int w = 1; w < kEpiWarps; ++w) {
#pragma unroll
          for (int j = 0; j < kTopK; ++j) topk_offer(m, lists[(w * BN + b) * kTopK + j].z, lists[(w * BN + b) * kTopK + j].id);
        }
        Partial* dst = args.f.partials + (static_cast<int64_t>(b) * args.f.n_parts + blockIdx.x) * kTopK;
#pragma unroll
        for (int j = 0; j < kTopK; ++j) dst[j] = Partial{m.z[j], m.id[j]};
      }
    } else {
      // no dependency wait before the push: this launch's keys and ticket are
      // its own (only the grid's last CTA waits, in finish_grid)
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const int b = c * C::kChunk + lane;
        if (lane < C::kChunk && b < B) {
          Best bb;
          bb.z = best_z[c];
          bb.id = best_id[c];
          warp_best[warp * BN + b] = bb;
        }
      }
      // combine the 4 epilogue warps, push one candidate per (batch row, CTA)
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      for (int b = threadIdx.x; b < B; b += kEpiWarps * 32) {
        Best r = warp_best[b];
#pragma unroll
        for (int w = 1; w < kEpiWarps; ++w) r = combine(r, warp_best[w * BN + b]);
        push_candidate(args.f, b, r);
      }
      finish_grid(args.f, B, threadIdx.x, kEpiWarps * 32, last_flag, named_bar1_and<kEpiWarps * 32>);
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ------------------------------------------------------------------ host side
// Persistent CTAs: at most max_ctas, then as few as give every CTA the same
// number of tiles (measured: at B = 16, 1002 tiles on 251 CTAs of 4 instead of
// 304 CTAs of 3.3 cut the step from 159.2 to 154.4 us).
int vocab_grid(int64_t n_vt, int max_ctas) {
  const int64_t g0 = std::max<int64_t>(1, std::min<int64_t>(max_ctas, n_vt));
  const int64_t per = (std::max<int64_t>(n_vt, 1) + g0 - 1) / g0;
  return static_cast<int>(std::max<int64_t>(1, (std::max<int64_t>(n_vt, 1) + per - 1) / per));
}

template <int BN, int kTopK = 0>
cudaError_t launch_bn(const Problem& p, const Finish& f, int* err, cudaStream_t stream) {
  using C = VocabCfg<BN, kTopK>;
  static_assert(C::kStages >= 2, "pipeline needs at least two stages");
  static_assert(C::kSmemBytes * C::kCtasPerSm <= 228 * 1024, "shared memory budget");
  CUtensorMap tw, th;
  if (!encode_kmajor_bf16(&tw, p.W, p.V_local, p.d, kBK, kBM)) return cudaErrorInvalidValue;
  if (!encode_kmajor_bf16(&th, p.h, p.B, p.d, kBK, BN)) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaError_t e = raise_smem_limit<tc_vocab_kernel<BN, kTopK>>(dev, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 148;
  const int64_t n_vt = (p.V_local + kBM - 1) / kBM;
  const int grid = vocab_grid(n_vt, C::kCtasPerSm * sms);
  VocabArgs a{p, f, n_vt, err};
  return launch_kernel(tc_vocab_kernel<BN, kTopK>, dim3(grid), dim3(kThreads), C::kSmemBytes, stream, p.pdl, tw, th, a);
}

}  // namespace

int tc_vocab_bn(int64_t B) {
  return B <= 16 ? 16 : B <= 32 ? 32 : B <= 64 ? 64 : B <= 128 ? 128 : 256;
}

cudaError_t launch_tc_vocab(const Problem& p, const Finish& f, int* err, cudaStream_t stream) {
  if (p.B > 256 || p.d < kBK || p.V_local <= 0) return cudaErrorNotSupported;
  switch (tc_vocab_bn(p.B)) {
    case 16: return launch_bn<16>(p, f, err, stream);
    case 32: return launch_bn<32>(p, f, err, stream);
    case 64: return launch_bn<64>(p, f, err, stream);
    case 128: return launch_bn<128>(p, f, err, stream);
    default: return launch_bn<256>(p, f, err, stream);
  }
}

int tc_vocab_topk_parts(int64_t V, int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (sms <= 0) sms = 148;
  return vocab_grid((V + kBM - 1) / kBM, sms);   // top-k mode: one CTA per SM
}

template <int BN>
static cudaError_t launch_topk_bn(const Problem& p, int K, const Finish& f, int* err, cudaStream_t stream) {
  switch (K) {
    case 4: return launch_bn<BN, 4>(p, f, err, stream);
    case 8: return launch_bn<BN, 8>(p, f, err, stream);
    case 16: return launch_bn<BN, 16>(p, f, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_tc_vocab_topk(const Problem& p, int K, Partial* partials, int* err, cudaStream_t stream) {
  if (p.B > 64 || p.d < kBK || p.V_local <= 0) return cudaErrorNotSupported;
  int dev = 0;
  cudaGetDevice(&dev);
  Finish f{};
  f.partials = partials;
  f.n_parts = tc_vocab_topk_parts(p.V_local, dev);
  switch (tc_vocab_bn(p.B)) {
    case 16: return launch_topk_bn<16>(p, K, f, err, stream);
    case 32: return launch_topk_bn<32>(p, K, f, err, stream);
    default: return launch_topk_bn<64>(p, K, f, err, stream);
  }
}

}  // namespace fs
