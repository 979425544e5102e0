// Tensor-core fused LM-head sampler, batch-major over CTA PAIRS: the
// large-batch path in the contraction-bound regime.
//
// FlashSampling: Fast and Memory-Efficient Exact Sampling -- summary page,
// "Method": the logit tile is formed on chip, Gumbel noise is added in-tile,
// and only a per-row (max, argmax) survives; arXiv abstract: "keep only one
// maximizer per row and per vocabulary tile, and finish with a small
// reduction over tiles".
//
// Same tiling and epilogue as the single-CTA batch-major kernel, but each MMA
// spans a cluster of two CTAs (tcgen05 cta_group::2): M = 256 batch rows
// (128 per CTA, each CTA loads its own h rows) by N = 256 vocabulary rows
// (each CTA loads HALF of the W tile, 128 rows), K = 64 per stage.  Per CTA a
// stage is 32 KB instead of 48 KB, so seven stages fit and each CTA moves a
// third fewer bytes from L2 for the same MMA work.  The even CTA of the pair
// issues the MMAs and commits them to both CTAs' barriers; each CTA's TMEM
// holds the accumulators of its own 128 batch rows x 256 vocabulary rows, and
// each CTA's epilogue releases the accumulator by arriving on the even CTA's
// barrier.
//
// CTA grouping as in the single-CTA kernel: with npt = ceil(B / 256) pair
// tiles, groups of npt pairs walk the vocabulary tiles q, q + n_groups, ...
// in lockstep, so W comes from HBM once per group.
//
// Gumbel-top-k mode (kTopK > 0): every epilogue thread keeps its batch row's
// K best perturbed scores instead of the best one; the column parts
// merge through shared memory and each CTA writes one list per (row, group)
// for the merge kernel, with no in-kernel finish.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "fs_epilogue.cuh"
#include "fs_finish.cuh"
#include "fs_internal.h"
#include "fs_sm100.cuh"
#include "fs_tmap.h"

namespace fs {
namespace {

using namespace sm100;

// Warp roles: kEpi epilogue warps (kEpi / 4 per TMEM lane quarter, each
// scanning that share of the tile's columns), then the TMA producer and the
// MMA issuer.  The sampler runs 16 epilogue warps, four per scheduler (2.4%
// faster than 8 at B = 512, 1% at 1024 and 256, in interleaved runs); 18
// warps leave 96 registers a thread (the register file is split between the
// four schedulers), which made the top-k lists spill and the B = 256, k = 8
// call 2.5% slower, so the top-k variants keep 8.
//
// kLean: the instantiation for small vocabulary chunks of batches of several
// pair tiles (fs_sample_chunked; see launch_tc_pair): 3 stages, ONE 256-column accumulator
// and 8 epilogue warps, so that two CTAs fit on an SM (shared memory, TMEM
// and registers) and the next chunk's pairs stream and multiply while this
// chunk's run their epilogues.  Its MMAs (shapes, K order) and its scan are
// those of the full instantiation, so every logit and every sample is the
// same bit for bit; only the overlap differs.
template <int kTopK, bool kLean = false>
struct PairWarps {
  static constexpr int kEpi = (kTopK > 0 || kLean) ? 8 : 16;
  static constexpr int kParts = kEpi / 4;
  static constexpr int kProducer = kEpi;
  static constexpr int kMma = kEpi + 1;
  static constexpr int kThreads = (kEpi + 2) * 32;
};
constexpr int kMaxColParts = 4;
constexpr int kRowsPerCta = 128;    // batch rows of one CTA (half of the MMA M = 256)
constexpr int kBN = 256;            // vocabulary rows per tile (MMA N); each CTA loads 128
constexpr int kBK = 64;
constexpr int kATileBytes = kRowsPerCta * kBK * 2;     // 16 KB: this CTA's h rows
constexpr int kBTileBytes = (kBN / 2) * kBK * 2;       // 16 KB: this CTA's half of the W tile

template <bool kLean>
struct PairCfg {
  static constexpr int kStages = kLean ? 3 : 7;
  static constexpr int kAccs = kLean ? 1 : 2;          // 256-column TMEM accumulators
  static constexpr int kTmemCols = kAccs * kBN;
  static constexpr int kCtasPerSm = kLean ? 2 : 1;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kATileBytes;
  static constexpr int kOffBars = kOffB + kStages * kBTileBytes;
  static constexpr int kNumBars = 2 * kStages + 5;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  // The epilogue's merge buffers are used only after the CTA's last tile has
  // been waited for, when every MMA has completed and every TMA load has
  // landed, so they alias the first stages; that leaves room for a seventh
  // stage in the full instantiation (230.6 KB of the 232 KB a CTA may use).
  static constexpr int kOffHalf = kOffA;                                              // Best[parts - 1][128]
  static constexpr int kOffTopK = kOffHalf + (kMaxColParts - 1) * kRowsPerCta * 8;   // top-k mode: Partial[128][K]
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kOffHalf + (kMaxColParts - 1) * kRowsPerCta * 8 <= kOffBars, "merge buffers fit in the stages");
  static_assert(kLean || kOffTopK + kRowsPerCta * 16 * 8 <= kOffBars, "top-k buffers fit in the stages");
  static_assert(kSmemBytes * kCtasPerSm <= 232448, "shared memory per SM");
};
constexpr int kSmemBytes = PairCfg<false>::kSmemBytes;
constexpr int smem_bytes(int) { return kSmemBytes; }
constexpr uint16_t kPairMask = 0x3;

struct PairArgs {
  Problem p;            // rows [0, p.B) of this launch's batch slice
  Finish f;             // sampling mode: cross-CTA finish of this slice's rows;
                        // top-k mode: f.partials [B, f.n_parts, K], part = pair group
  int npt;              // pair tiles (256 batch rows each) of this launch
  int n_groups;         // groups of npt pairs
  int n_vt;             // vocabulary tiles = ceil(V_local / 256)
  int* err;
};

template <int kTopK = 0, bool kLean = false>
__global__ void __cluster_dims__(2, 1, 1)
__launch_bounds__(PairWarps<kTopK, kLean>::kThreads, PairCfg<kLean>::kCtasPerSm)
tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_h, const __grid_constant__ CUtensorMap tmap_w,
               const PairArgs args) {
  static_assert(!(kLean && kTopK > 0), "the lean instantiation samples only");
  using Cfg = PairCfg<kLean>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kAccs = Cfg::kAccs;
  constexpr int kTmemCols = Cfg::kTmemCols;
  constexpr int kOffA = Cfg::kOffA;
  constexpr int kOffB = Cfg::kOffB;
  constexpr int kOffBars = Cfg::kOffBars;
  constexpr int kOffMisc = Cfg::kOffMisc;
  constexpr int kOffHalf = Cfg::kOffHalf;
  constexpr int kOffTopK = Cfg::kOffTopK;
  constexpr int kEpiWarps = PairWarps<kTopK, kLean>::kEpi;
  constexpr int kColParts = PairWarps<kTopK, kLean>::kParts;
  constexpr int kProducerWarp = PairWarps<kTopK, kLean>::kProducer;
  constexpr int kMmaWarp = PairWarps<kTopK, kLean>::kMma;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kOffBars);   // used in the even CTA
  uint64_t* empty_bar = full_bar + kStages;                            // both CTAs
  uint64_t* tfull_bar = empty_bar + kStages;                           // both CTAs
  uint64_t* tempty_bar = tfull_bar + 2;                                // used in the even CTA
  uint64_t* drain_bar = tempty_bar + 2;                                // (2 + 2 slots; kAccs used)
  uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* last_flag = reinterpret_cast<int*>(smem + kOffMisc + 8);
  Best* part_best = reinterpret_cast<Best*>(smem + kOffHalf);
  if (kTopK == 0 && args.f.done != nullptr && args.f.carry_in) {
    // Early finalization: the two CTAs of a pair must take the same decision
    // (the running one would otherwise signal a peer that has left), so the
    // even CTA reads the flag once and stores it into both CTAs.
    cluster_sync();                                     // both CTAs have started: their shared memory is live
    if (cluster_ctarank() == 0 && threadIdx.x == 0) {
      const int skip = early_done(args.f) ? 1 : 0;
      *last_flag = skip;
      st_shared_cluster_u32(mapa_shared(smem_u32(last_flag), 1), static_cast<uint32_t>(skip));
    }
    cluster_sync();
    if (*last_flag != 0) {
      early_skip_cta(args.f, args.p.B, args.p.pdl, last_flag);
      return;
    }
  }

  const Problem& p = args.p;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();              // 0: issues the MMAs
  const int pair = blockIdx.x >> 1;
  const int pt = pair % args.npt;
  const int q = pair / args.npt;
  const int n_tiles = q < args.n_vt ? (args.n_vt - 1 - q) / args.n_groups + 1 : 0;
  const int n_kb = static_cast<int>((p.d + kBK - 1) / kBK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < kAccs; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 2 * kEpiWarps);        // one arrival per epilogue warp of both CTAs
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
    tmem_alloc_pair(tmem_base_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                       // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem_base = *tmem_base_slot;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_h = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int64_t n_issued = 0;
      bool ok = true;
      const int h_row = pt * 2 * kRowsPerCta + static_cast<int>(rank) * kRowsPerCta;
      // Deferred inputs: the first ring of stages (stage i = K step i mod
      // n_kb) gets its W boxes before the dependency wait, its h boxes after.
      bool h_ready = !p.defer_inputs;
      auto load_deferred_h = [&]() {
        pdl_wait();
        for (int64_t i = 0; i < n_issued; ++i)
          tma_load_2d_pair(smem + kOffA + i * kATileBytes, &tmap_h, mapa_shared(smem_u32(&full_bar[i]), 0),
                           static_cast<int32_t>((i % n_kb) * kBK), h_row, pol_h);
        h_ready = true;
      };
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int vt = q + t * args.n_groups;
        for (int kb = 0; kb < n_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, args.err, abort_flag)) { ok = false; break; }
          const uint32_t leader_full = mapa_shared(smem_u32(&full_bar[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * (kATileBytes + kBTileBytes));
          if (h_ready)
            tma_load_2d_pair(smem + kOffA + stage * kATileBytes, &tmap_h, leader_full, kb * kBK, h_row, pol_h);
          tma_load_2d_pair(smem + kOffB + stage * kBTileBytes, &tmap_w, leader_full, kb * kBK,
                           vt * kBN + static_cast<int>(rank) * (kBN / 2), pol_w);
          ++n_issued;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
          if (!h_ready && n_issued == kStages) load_deferred_h();
        }
      }
      if (!h_ready) load_deferred_h();   // fewer issues than stages (or an early stop)
      if (!ok && rank == 0) {
        volatile int no_abort = 0;
        for (int64_t i = std::max<int64_t>(0, n_issued - kStages); i < n_issued; ++i)
          mbar_wait(&full_bar[i % kStages], static_cast<uint32_t>((i / kStages) & 1), args.err, &no_abort);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer (even CTA only)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kRowsPerCta, kBN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int acc = t % kAccs;
        const uint32_t acc_phase = (t / kAccs) & 1;
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
            mma_bf16_pair(d_tmem, smem_desc_k128(a_addr + k * 32), smem_desc_k128(b_addr + k * 32), idesc,
                          (kb | k) != 0);
          mma_commit_pair_multicast(&empty_bar[stage], kPairMask);   // frees the stage in both CTAs
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (ok) mma_commit_pair_multicast(&tfull_bar[acc], kPairMask);
      }
      if (!ok) {
        mma_commit_pair_multicast(drain_bar, 0x1);
        volatile int no_abort = 0;
        mbar_wait(drain_bar, 0, args.err, &no_abort);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0-15, both CTAs)
    const int quad = warp & 3;
    const int part = warp >> 2;                         // column part of the tile
    const int row_in_tile = quad * 32 + lane;
    const int64_t b = static_cast<int64_t>(pt) * 2 * kRowsPerCta + static_cast<int64_t>(rank) * kRowsPerCta + row_in_tile;
    const bool row_ok = b < p.B;
    if (p.defer_inputs) pdl_wait();   // temp (and bias) may come from the preceding kernel
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
      const int acc = t % kAccs;
      const uint32_t acc_phase = (t / kAccs) & 1;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, args.err, abort_flag)) break;
      tc_fence_after();
      const int vt = q + t * args.n_groups;
      const int64_t col0 = static_cast<int64_t>(vt) * kBN + part * (kBN / kColParts);
#pragma unroll 1
      for (int c = 0; c < kBN / kColParts; c += 32) {
        uint32_t r[32];
        tmem_ld_32(tmem_base + lane_addr + acc * kBN + part * (kBN / kColParts) + c, r);
        tmem_ld_wait();
        const int64_t v0 = col0 + c;
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
        if (active && v0 < p.V_local) {
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
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
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
    } else {
      // combine the column parts of each row, then one candidate per (row, group)
      if (part != 0) part_best[(part - 1) * kRowsPerCta + row_in_tile] = best;
      asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
      if (part == 0) {
#pragma unroll
        for (int src = 1; src < kColParts; ++src) best = combine(best, part_best[(src - 1) * kRowsPerCta + row_in_tile]);
      }
      // no dependency wait before the push: this launch's keys and ticket are
      // its own (only the grid's last CTA waits, in finish_grid)
      if (part == 0 && row_ok) push_candidate(args.f, b, best);
      finish_grid(args.f, p.B, threadIdx.x, kEpiWarps * 32, last_flag,
                  named_bar1_and<kEpiWarps * 32>);
    }
  }

  // ---- teardown: neither CTA leaves (or frees TMEM) while the pair's MMAs or
  // the peer's signals may still touch it
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace

// CTA pairs that can be resident at once: a pair needs two SMs of one GPC,
// so with GPCs of odd SM counts this can be below SMs / 2 (per SM slot: the
// lean instantiation fits two CTAs on an SM).  A persistent grid larger than
// that would run its last pairs as a second wave.
template <bool kLean>
static int resident_pairs(int dev, int sms) {
  static std::atomic<int> cached[64];         // zero-initialized (static storage)
  if (dev >= 0 && dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  constexpr int per_sm = PairCfg<kLean>::kCtasPerSm;
  int n = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * per_sm * (sms / 2)));
  cfg.blockDim = dim3(PairWarps<0, kLean>::kThreads);
  cfg.dynamicSmemBytes = PairCfg<kLean>::kSmemBytes;
  if (cudaOccupancyMaxActiveClusters(&n, tc_pair_kernel<0, kLean>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = per_sm * (sms / 2);
  }
  n = std::min(n, per_sm * (sms / 2));
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

static int resident_pairs(int dev, int sms) { return resident_pairs<false>(dev, sms); }

// Geometry of one launch over a batch slice of B rows: npt pair tiles, then
// at most pairs / npt groups, as few as give every group the same number of
// vocabulary tiles.
struct PairGeometry {
  int npt, n_groups;
};

static PairGeometry pair_geometry(int64_t B, int pairs, int64_t n_vt, int min_per = 1) {
  PairGeometry g;
  g.npt = static_cast<int>((B + 2 * kRowsPerCta - 1) / (2 * kRowsPerCta));
  g.n_groups = std::max(1, pairs / g.npt);
  const int64_t tiles = std::max<int64_t>(n_vt, 1);
  const int64_t per = std::max<int64_t>(min_per, (tiles + g.n_groups - 1) / g.n_groups);
  g.n_groups = static_cast<int>(std::max<int64_t>(1, (tiles + per - 1) / per));
  return g;
}

static int device_sms(int* dev) {
  int sms = 0;
  cudaGetDevice(dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, *dev);
  return sms > 0 ? sms : 148;
}

template <bool kLean>
static cudaError_t launch_pair_sampler(const Problem& p, const Finish& f, int* err, cudaStream_t stream,
                                       int min_tiles_per_pair) {
  using Cfg = PairCfg<kLean>;
  int dev = 0;
  const int sms = device_sms(&dev);
  cudaError_t e = raise_smem_limit<tc_pair_kernel<0, kLean>>(dev, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int pairs = resident_pairs<kLean>(dev, sms);
  CUtensorMap tw;
  if (!encode_kmajor_bf16(&tw, p.W, p.V_local, p.d, kBK, kBN / 2)) return cudaErrorInvalidValue;
  const int64_t slice = static_cast<int64_t>(pairs) * 2 * kRowsPerCta;
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
    Finish fs_slice = f;
    fs_slice.keys = f.keys + b0;
    if (f.carry_max != nullptr) {
      fs_slice.carry_max = f.carry_max + b0;
      fs_slice.carry_ids = f.carry_ids + b0;
    }
    if (f.write_out) {
      fs_slice.out_ids = f.out_ids + b0;
      fs_slice.out_max = f.out_max + b0;
    }
    const int n_vt = static_cast<int>((p.V_local + kBN - 1) / kBN);
    const PairGeometry g = pair_geometry(ps.B, pairs, n_vt, min_tiles_per_pair);
    CUtensorMap th;
    if (!encode_kmajor_bf16(&th, ps.h, ps.B, p.d, kBK, kRowsPerCta)) return cudaErrorInvalidValue;
    PairArgs a{ps, fs_slice, g.npt, g.n_groups, n_vt, err};
    e = launch_kernel(tc_pair_kernel<0, kLean>, dim3(2 * g.npt * g.n_groups), dim3(PairWarps<0, kLean>::kThreads),
                      Cfg::kSmemBytes, stream, ps.pdl, th, tw, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Chunk calls.  Chunks of fewer than 24 tiles (32 chunks of a 128K
// vocabulary) run the full instantiation with 2 tiles per pair from 12 tiles
// on and 1 below; only chunks of fewer than 12 tiles of batches of several
// pair tiles run the lean instantiation (two CTAs per SM).  Measured on GB300
// (8B head, µs per step; one fs_sample_chunked_step call per step, steps back
// to back / the per-chunk calls replayed from a CUDA graph): B = 256, 24
// chunks (21 tiles): lean 254.8 / 282.5, k = 2 244.9 / 275.3; 32 chunks (16
// tiles): lean 299.1 / 277.4, k = 2 271.7 / 275.9, k = 1 274.5 / 303.8; 48
// chunks (11 tiles): lean 434.2 / 339.3, k = 1 319.9 / 349.2, k = 2 412.1 /
// 338.4; 64 chunks (8 tiles): lean 499.6 / 349.9, k = 1 364.9 / 340.7; 128
// chunks (4 tiles): lean 1201 / 681, k = 1 834 / 546.  B = 512, 32 chunks:
// lean 427.2 / 484.6, k = 2 414.4 / 471.7; 64 chunks: lean 580.9 / 528.8,
// k = 1 513.0 / 577.2.
// Chunks of at least 24 tiles run the full instantiation with k >= 4 tiles
// per pair: a pair's epilogues overlap its
// next tiles' MMAs and the chunks in flight take disjoint pairs.  Their cost
// follows waves of pairs: the step's chunks need n * ceil(T / k) * npt pairs
// (n chunks of T tiles, npt pair tiles of batch rows), run in
// ceil(pairs / resident) waves of k tile-times each, so k is the one in
// [4, 16] that minimizes waves * k (the smaller on ties), with n taken from
// the previous chunked step on the stream (k = 4 before there is one).
// Measured on GB300 (us per step, interleaved runs of one build, B = 256):
// 8B head, 8 chunks: k = 7 243, 8 244, 4 250, 2 273, 3 284, 5 296, 6 325
// (the model ranks them 7 < 4 = 8 < 3 < 5 < 6); Qwen3 head, 8 chunks: k = 4
// 266, 10 299, 7 397, 8 403 (model: 4 < 10 < 7 < 8); lean: 281 and 312.  The
// MMAs and the scan are the same in both instantiations, so the samples are
// too.
constexpr int64_t kChunkLeanMaxTiles = 24;
constexpr int64_t kChunkPairOfTwoMinTiles = 12;
constexpr int kChunkMinTilesPerPair = 4;
constexpr int kChunkMaxTilesPerPair = 16;

// Chunk grids launched on a stream (not from a CUDA graph) run at most 8 at a
// time on GB300, however many pairs stay idle: with 12 chunks of 6 pairs (72
// of the 76), a per-CTA timeline showed chunks 0-7 starting within 21 us and
// chunk 8 only when chunk 0 had exited, 180 us later (343 us per step against
// 216 on the batch-major kernel; 9 chunks of 8 pairs at B = 256: 357 us).
// Replayed from a graph the same 12 chunks ran side by side (229 us).  The
// waves of a step count both the pairs and, for stream launches, the grids.
constexpr int kStreamChunkGrids = 8;

static int64_t chunk_waves(int64_t need_pairs, int64_t pairs, int step_chunks, bool in_graph) {
  int64_t waves = (need_pairs + pairs - 1) / pairs;
  if (!in_graph) waves = std::max<int64_t>(waves, (step_chunks + kStreamChunkGrids - 1) / kStreamChunkGrids);
  return waves;
}

static int chunk_tiles_per_pair(int64_t n_vt, int64_t B, int step_chunks, bool in_graph, int pairs) {
  if (step_chunks <= 0) return kChunkMinTilesPerPair;
  const int64_t npt = (std::min<int64_t>(B, static_cast<int64_t>(pairs) * 2 * kRowsPerCta) + 2 * kRowsPerCta - 1) /
                      (2 * kRowsPerCta);
  int best_k = kChunkMinTilesPerPair;
  int64_t best_cost = -1;
  for (int k = kChunkMinTilesPerPair; k <= kChunkMaxTilesPerPair; ++k) {
    const int64_t need = static_cast<int64_t>(step_chunks) * ((n_vt + k - 1) / k) * npt;
    const int64_t cost = chunk_waves(need, pairs, step_chunks, in_graph) * k;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_k = k;
    }
  }
  return best_k;
}

// Whether a chunked step of step_chunks chunks like this one (V_local rows,
// B batch rows) runs on the pairs in ONE wave with at most
// kChunkFastTilesPerPair tiles per pair, which is where the pair kernel beats
// the single-CTA batch-major kernel for chunks of batches that fit one
// 128-row batch tile (8B head, B = 64 and 128, µs per step, pair vs batch-
// major: 4 chunks 215 / 218 vs 241, 6 chunks 217 / 221 vs 243, 8 chunks 219 /
// 223 vs 241, 12 chunks 229 / 232 vs 242 -- one wave of k = 7; 10 chunks
// 264 / 265 vs 242, 16 chunks 249 / 252 vs 237, 20 chunks 272 / 273 vs
// 249, 32 chunks 266 / 275 vs 233 -- two waves or the lean instantiation;
// times of per-chunk calls replayed from a CUDA graph).  Stream-launched
// steps must also fit the kStreamChunkGrids limit.
constexpr int kChunkFastTilesPerPair = 7;

bool tc_pair_chunk_one_wave(int64_t V_local, int64_t B, int step_chunks, bool in_graph, int device) {
  const int64_t n_vt = (V_local + kBN - 1) / kBN;
  if (step_chunks <= 0 || n_vt < kChunkLeanMaxTiles || B <= 0) return false;
  if (!in_graph && step_chunks > kStreamChunkGrids) return false;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  const int pairs = resident_pairs<false>(device, sms > 0 ? sms : 148);
  const int64_t npt = (std::min<int64_t>(B, static_cast<int64_t>(pairs) * 2 * kRowsPerCta) + 2 * kRowsPerCta - 1) /
                      (2 * kRowsPerCta);
  for (int k = kChunkMinTilesPerPair; k <= kChunkFastTilesPerPair; ++k)
    if (static_cast<int64_t>(step_chunks) * ((n_vt + k - 1) / k) * npt <= pairs) return true;
  return false;
}

cudaError_t launch_tc_pair(const Problem& p, const Finish& f, int* err, cudaStream_t stream) {
  if (p.d < kBK || p.V_local <= 0) return cudaErrorNotSupported;
  if (!p.chunk) return launch_pair_sampler<false>(p, f, err, stream, 1);
  const int64_t n_vt = (p.V_local + kBN - 1) / kBN;
  if (n_vt < kChunkLeanMaxTiles) {
    if (n_vt >= kChunkPairOfTwoMinTiles) return launch_pair_sampler<false>(p, f, err, stream, 2);
    if (p.B <= 2 * kRowsPerCta) return launch_pair_sampler<false>(p, f, err, stream, 1);
    return launch_pair_sampler<true>(p, f, err, stream, 1);
  }
  int dev = 0;
  const int sms = device_sms(&dev);
  const int k = chunk_tiles_per_pair(n_vt, p.B, p.step_chunks, p.in_graph, resident_pairs<false>(dev, sms));
  return launch_pair_sampler<false>(p, f, err, stream, k);
}

int64_t tc_pair_topk_max_rows(int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  return static_cast<int64_t>(resident_pairs(device, sms > 0 ? sms : 148)) * 2 * kRowsPerCta;
}

int tc_pair_topk_parts(int64_t B, int64_t V, int device) {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  const int pairs = resident_pairs(device, sms > 0 ? sms : 148);
  return pair_geometry(B, pairs, (V + kBN - 1) / kBN).n_groups;
}

template <int K>
static cudaError_t launch_pair_topk_k(const Problem& p, Partial* partials, int* err, cudaStream_t stream) {
  int dev = 0;
  const int sms = device_sms(&dev);
  const int pairs = resident_pairs(dev, sms);
  if (p.B > static_cast<int64_t>(pairs) * 2 * kRowsPerCta) return cudaErrorNotSupported;   // one launch
  cudaError_t e = raise_smem_limit<tc_pair_kernel<K>>(dev, smem_bytes(K));
  if (e != cudaSuccess) return e;
  CUtensorMap tw, th;
  if (!encode_kmajor_bf16(&tw, p.W, p.V_local, p.d, kBK, kBN / 2)) return cudaErrorInvalidValue;
  if (!encode_kmajor_bf16(&th, p.h, p.B, p.d, kBK, kRowsPerCta)) return cudaErrorInvalidValue;
  const int n_vt = static_cast<int>((p.V_local + kBN - 1) / kBN);
  const PairGeometry g = pair_geometry(p.B, pairs, n_vt);
  Finish f{};
  f.partials = partials;
  f.n_parts = g.n_groups;
  PairArgs a{p, f, g.npt, g.n_groups, n_vt, err};
  return launch_kernel(tc_pair_kernel<K>, dim3(2 * g.npt * g.n_groups), dim3(PairWarps<K>::kThreads), smem_bytes(K),
                       stream, p.pdl,
                       th, tw, a);
}

cudaError_t launch_tc_pair_topk(const Problem& p, int K, Partial* partials, int* err, cudaStream_t stream) {
  if (p.d < kBK || p.V_local <= 0) return cudaErrorNotSupported;
  switch (K) {
    case 4: return launch_pair_topk_k<4>(p, partials, err, stream);
    case 8: return launch_pair_topk_k<8>(p, partials, err, stream);
    case 16: return launch_pair_topk_k<16>(p, partials, err, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fs
