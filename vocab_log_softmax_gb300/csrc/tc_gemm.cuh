// A persistent tcgen05 GEMM mainloop with a pluggable epilogue:
//     C[M, Ncols] = A[M, K] * B[Ncols, K]^T,
// A and B 16-bit, fp32 accumulation in tensor memory.  Each operand is either
// K-major (stored [rows, K], K contiguous) or MN-major (stored [K, rows], its
// M or N index contiguous), chosen per launch, so a product whose operand
// sits transposed in memory needs no transpose.  The output tile is never
// stored by the mainloop: an epilogue object receives it, 32 columns of one
// row per thread at a time, and does what its operation needs (fold a
// softmax, form a gradient, store through TMA).
//
// Work is cut into units of (a row tile) x (a chunk of `chunk_tiles` column
// tiles of 256) x (a run of K blocks, with split-K), walked by a persistent
// grid.  Roles (192 threads): warp 0 issues TMA loads of 64-wide K slices of
// A and B into a shared-memory ring (128-byte swizzle); warp 1 owns 512
// tensor-memory columns and one of its threads issues kind::f16 MMAs into
// one of two accumulators; warps 2-5 read a finished accumulator (one row
// per thread) and hand it to the epilogue, then free it, so one tile's
// epilogue overlaps the next tile's MMAs.  Two forms: 128-row tiles on one
// SM (4 stages of 48 KB), and 256-row tiles on a CTA pair (cta_group::2, 6
// stages of 32 KB per CTA), the default.  Every wait is bounded
// (tc_device.cuh).
#pragma once

#include <atomic>

#include "tc_device.cuh"
#include "vls_device.cuh"

namespace vls {
namespace tcg {

constexpr int kBM = 128;            // rows per tile (MMA M)
constexpr int kBN = 256;            // columns per tile (MMA N)
constexpr int kBK = 64;             // K per stage: one 128-byte swizzled row of 16-bit elements
constexpr int kUK = 16;             // K per MMA instruction (kind::f16)
constexpr int kStages = 4;
constexpr int kThreads = 192;       // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
constexpr uint32_t kStageA = kBM * kBK * 2;   // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;   // 32 KB
constexpr uint32_t kTmemCols = 2 * kBN;       // two fp32 accumulators of 256 columns
constexpr int kNumBars = 2 * kStages + 4 + 1; // full, empty, acc_full x2, acc_empty x2, done
// epilogue staging (Epi::kStageBytes per epilogue warp) after the barriers, 1024-byte aligned
constexpr size_t kEpiOff = (kStages * (kStageA + kStageB) + kNumBars * 8 + 16 + 1023) & ~size_t(1023);

constexpr int kMaxDev = 64;   // devices the per-device launch caches cover

struct Sched {
  int64_t M;          // valid rows of the output
  int64_t Ncols;      // valid columns of the output
  int n_row_tiles, n_col_tiles, chunk_tiles, n_chunks, n_units, nk;
  int ksplit;         // K is cut into ksplit runs of nk_split K blocks (split-K; 1 = whole K)
  int nk_split;
  int n_units_k;      // units per K run: n_row_tiles x n_chunks
  int cols_fastest;   // unit order: 0 = row tiles fastest (B chunk shared by the CTAs in flight),
                      // 1 = column chunks fastest (A row panel shared)
  tc::WaitCtl wc;     // where a wait that runs out reports (tc::kStatusTimeout), and the wait limit

  // (row tile, column chunk, K run) of unit u; K runs outermost
  __device__ __forceinline__ void unit(int u, int& rt, int& chunk, int& ks) const {
    ks = u / n_units_k;
    u -= ks * n_units_k;
    if (cols_fastest) {
      rt = u / n_chunks;
      chunk = u - rt * n_chunks;
    } else {
      chunk = u / n_row_tiles;
      rt = u - chunk * n_row_tiles;
    }
  }
  // the K blocks [kb0, kb1) of K run ks
  __device__ __forceinline__ void k_range(int ks, int& kb0, int& kb1) const {
    kb0 = ks * nk_split;
    kb1 = min(kb0 + nk_split, nk);
  }
};

// rows_per_tile: 128 (1-SM form) or 256 (CTA pairs).  ksplit > 1 cuts K into
// that many runs of whole K blocks, one unit per (tile, chunk, run); the
// epilogue then sees partial sums and the run index (EpiWarp::ks).
inline Sched make_sched(int64_t M, int64_t Ncols, int64_t K, int chunk_tiles, const tc::WaitCtl& wc,
                        int rows_per_tile, int ksplit) {
  Sched s;
  s.M = M;
  s.Ncols = Ncols;
  s.n_row_tiles = static_cast<int>((M + rows_per_tile - 1) / rows_per_tile);
  s.n_col_tiles = static_cast<int>((Ncols + kBN - 1) / kBN);
  s.chunk_tiles = chunk_tiles;
  s.n_chunks = (s.n_col_tiles + chunk_tiles - 1) / chunk_tiles;
  s.nk = static_cast<int>((K + kBK - 1) / kBK);
  if (ksplit < 1) ksplit = 1;
  if (ksplit > s.nk) ksplit = s.nk;
  s.nk_split = (s.nk + ksplit - 1) / ksplit;
  s.ksplit = (s.nk + s.nk_split - 1) / s.nk_split;   // no empty run
  s.n_units_k = s.n_row_tiles * s.n_chunks;
  s.n_units = s.n_units_k * s.ksplit;
  s.cols_fastest = 0;
  s.wc = wc;
  return s;
}

// One stage of an operand: `rows` rows (of A, or columns of B) starting at r0,
// K slice k0 .. k0 + 63.  K-major: one TMA box of 64 x rows.  MN-major: rows
// / 64 boxes of 64 (M or N) x 64 (K), kMnBlockBytes apart.  PAIR issues the
// cta_group::2 form that completes on the pair leader's barrier.
template <bool MN, int ROWS, bool PAIR>
__device__ __forceinline__ void load_stage(uint32_t dst, const CUtensorMap* map, int32_t k0, int32_t r0,
                                           uint32_t bar) {
  if constexpr (!MN) {
    if constexpr (PAIR)
      tc::tma_load_2d_pair(dst, map, k0, r0, bar);
    else
      tc::tma_load_2d(dst, map, k0, r0, bar);
  } else {
#pragma unroll
    for (int j = 0; j < ROWS / 64; ++j) {
      if constexpr (PAIR)
        tc::tma_load_2d_pair(dst + j * tc::kMnBlockBytes, map, r0 + 64 * j, k0, bar);
      else
        tc::tma_load_2d(dst + j * tc::kMnBlockBytes, map, r0 + 64 * j, k0, bar);
    }
  }
}

// Descriptor of a stage and the step of its address field per 16-wide K
// slice: 32 bytes along a K-major row, two 8-row groups (2048 bytes) down an
// MN-major block.
template <bool MN>
__device__ __forceinline__ uint64_t stage_desc(uint32_t addr) {
  return MN ? tc::sdesc_sw128_mn(addr) : tc::sdesc_sw128(addr);
}
template <bool MN>
constexpr uint64_t kDescStep = MN ? (2048 >> 4) : (32 >> 4);

// What an epilogue warp owns: its shared-memory staging area (Epi::kStageBytes
// bytes, 1024-byte aligned; none when that is 0), the first of its 32 rows in
// the current unit, its lane, and a count the epilogue may keep (bulk stores
// issued, say).
struct EpiWarp {
  uint32_t stage;
  int64_t row0;
  int lane;
  uint32_t n;
  int ks;   // the unit's K run (0 without split-K)
};

// Epilogue interface (one object per launch, a __grid_constant__ kernel
// parameter, so a CUtensorMap member may serve TMA):
//   static constexpr uint32_t kStageBytes;                  shared memory per epilogue warp
//   struct State;                                           per-thread, per-unit state
//   State begin(int64_t row, bool row_ok, int chunk);       at each unit
//   void  cols(State&, const float (&v)[32], int64_t row, bool row_ok, int64_t col0, int nvalid, EpiWarp&);
//                                                           32 columns of the row (nvalid < 32 at the edge),
//                                                           called by the whole warp
//   void  end(State&, int64_t row, bool row_ok, int chunk); after the unit's last tile
//   void  finish(EpiWarp&);                                 once per warp before the CTA exits
template <bool BF16, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const Sched sc, const __grid_constant__ Epi epi) {
  extern __shared__ unsigned char smem_raw[];
  if (static_cast<int>(blockIdx.x) >= sc.n_units) return;  // whole CTA, before any barrier

  const uint32_t raw = tc::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase;                           // kStages x kStageA
  const uint32_t sB = sbase + kStages * kStageA;       // kStages x kStageB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * (kStageA + kStageB));
  const uint32_t bar0 = tc::smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kStages + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full(s), 1);
      tc::mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full(b), 1);
      tc::mbar_init(acc_empty(b), 4);   // one arrival per epilogue warp
    }
    tc::mbar_init(done_bar, 1);
    *abort_flag = 0u;
    tc::mbar_init_fence();
    tc::prefetch_tensormap(&tm_a);
    tc::prefetch_tensormap(&tm_b);
  }
  if (warp == 1) tc::tmem_alloc(tc::smem_u32(tmem_holder), kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;   // loads issued, for the drain below
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sc.n_units; u += gridDim.x) {
        int rt, chunk, ks, kb0, kb1;
        sc.unit(u, rt, chunk, ks);
        sc.k_range(ks, kb0, kb1);
        const int t_end = min((chunk + 1) * sc.chunk_tiles, sc.n_col_tiles);
        for (int t = chunk * sc.chunk_tiles; ok && t < t_end; ++t) {
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::wait(empty(stage), phase ^ 1u, abort_flag, sc.wc)) {
              ok = false;
              break;
            }
            tc::mbar_expect_tx(full(stage), kStageA + kStageB);
            load_stage<A_MN, kBM, false>(sA + stage * kStageA, &tm_a, kb * kBK, rt * kBM, full(stage));
            load_stage<B_MN, kBN, false>(sB + stage * kStageB, &tm_b, kb * kBK, t * kBN, full(stage));
            ++issued;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Before the CTA releases its shared memory, every load issued has
      // landed: the last one into each stage.  After a normal run the MMA
      // thread has waited for all of them and these waits return at once;
      // after an abort (this role's or another's) some may still be in flight.
      for (int s = 0; s < kStages; ++s) {
        if (issued > static_cast<uint32_t>(s)) {
          const uint32_t last = (issued - 1 - s) / kStages;   // index of the last load into stage s
          tc::wait_drain(full(s), last & 1u, sc.wc);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(BF16, kBM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tc_count = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sc.n_units; u += gridDim.x) {
        int rt, chunk, ks, kb0, kb1;
        sc.unit(u, rt, chunk, ks);
        sc.k_range(ks, kb0, kb1);
        const int t_end = min((chunk + 1) * sc.chunk_tiles, sc.n_col_tiles);
        for (int t = chunk * sc.chunk_tiles; ok && t < t_end; ++t, ++tc_count) {
          const uint32_t buf = tc_count & 1u, use = (tc_count >> 1) & 1u;
          if (!tc::wait(acc_empty(buf), use ^ 1u, abort_flag, sc.wc)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + buf * kBN;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::wait(full(stage), phase, abort_flag, sc.wc)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint64_t da = stage_desc<A_MN>(sA + stage * kStageA);
            const uint64_t db = stage_desc<B_MN>(sB + stage * kStageB);
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk)
              tc::mma_f16(d, da + kDescStep<A_MN> * kk, db + kDescStep<B_MN> * kk, idesc,
                          (kb > kb0 || kk > 0) ? 1u : 0u);
            tc::mma_commit(empty(stage));   // frees the stage once these MMAs have read it
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc::mma_commit(acc_full(buf));
        }
      }
      // every MMA this thread issued has completed before tensor memory is freed
      tc::mma_commit(done_bar);
      tc::wait_drain(done_bar, 0u, sc.wc);
    }
  } else {
    // ---------------- epilogue: warps 2-5 ----------------
    const int quarter = warp & 3;                 // the tensor-memory lanes this warp may read
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    EpiWarp ew{sbase + static_cast<uint32_t>(kEpiOff) + static_cast<uint32_t>(quarter) * Epi::kStageBytes, 0, lane, 0u, 0};
    uint32_t tc_count = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < sc.n_units; u += gridDim.x) {
      int rt, chunk, ks;
      sc.unit(u, rt, chunk, ks);
      ew.ks = ks;
      const int t_beg = chunk * sc.chunk_tiles, t_end = min(t_beg + sc.chunk_tiles, sc.n_col_tiles);
      const int64_t row = static_cast<int64_t>(rt) * kBM + r_in_tile;
      const bool row_ok = row < sc.M;
      ew.row0 = row - lane;
      typename Epi::State st = epi.begin(row, row_ok, chunk);
      for (int t = t_beg; t < t_end; ++t, ++tc_count) {
        const uint32_t buf = tc_count & 1u, use = (tc_count >> 1) & 1u;
        // one lane waits and the warp follows it, so the warp-wide tensor-memory
        // loads below are never reached by part of a warp
        const bool got = lane == 0 ? tc::wait(acc_full(buf), use, abort_flag, sc.wc) : true;
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        __syncwarp();
        tc::fence_after_sync();
        // chunk c + 1 is read from tensor memory while chunk c is folded
        auto fold = [&](const uint32_t (&r)[32], int c) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          const int64_t cbase = static_cast<int64_t>(t) * kBN + c * 32;
          const int64_t left = sc.Ncols - cbase;
          const int nvalid = left <= 0 ? 0 : (left >= 32 ? 32 : static_cast<int>(left));
          epi.cols(st, v, row, row_ok, cbase, nvalid, ew);
        };
        const uint32_t acc = lane_addr + buf * kBN;
        uint32_t ra[32], rb[32];
        tc::tmem_ld32_issue(acc, ra);
        tc::tmem_ld32_wait(ra);
        for (int c = 0; c < kBN / 32; c += 2) {
          tc::tmem_ld32_issue(acc + (c + 1) * 32, rb);
          fold(ra, c);
          tc::tmem_ld32_wait(rb);
          if (c + 2 < kBN / 32) tc::tmem_ld32_issue(acc + (c + 2) * 32, ra);
          fold(rb, c + 1);
          if (c + 2 < kBN / 32) tc::tmem_ld32_wait(ra);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty(buf));
      }
      if (ok) epi.end(st, row, row_ok, chunk);
    }
    epi.finish(ew);
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// The same GEMM on CTA pairs (2-SM MMA, tcgen05 cta_group::2).  A cluster of
// two CTAs computes 256 x 256 tiles: each CTA loads 128 rows of A and 128 of
// the tile's 256 columns of B, the pair's leader (rank 0) issues 256x256x16
// MMAs that read both CTAs' shared memory, and each CTA's tensor memory holds
// its own 128 rows of the accumulator.  Per CTA and K step this moves 32 KB
// into shared memory instead of 48 KB, which is what lets the tensor pipe
// run past the shared-memory bandwidth limit of the 1-SM form.
//   - loads of both CTAs complete on the leader's `full` barriers;
//   - MMA commits arrive on the `empty` / `acc_full` barriers of both CTAs;
//   - both CTAs' epilogue warps arrive on the leader's `acc_empty` (8 arrivals).
// ---------------------------------------------------------------------------

constexpr int kStages2 = 6;
constexpr uint32_t kStageA2 = kBM * kBK * 2;         // 16 KB: this CTA's 128 rows of A
constexpr uint32_t kStageB2 = (kBN / 2) * kBK * 2;   // 16 KB: this CTA's 128 columns of B
constexpr int kNumBars2 = 2 * kStages2 + 4 + 1;
constexpr size_t kEpiOff2 = (kStages2 * (kStageA2 + kStageB2) + kNumBars2 * 8 + 16 + 1023) & ~size_t(1023);

template <bool BF16, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const Sched sc, const __grid_constant__ Epi epi) {
  extern __shared__ unsigned char smem_raw[];
  const int pair = static_cast<int>(blockIdx.x >> 1), n_pairs = static_cast<int>(gridDim.x >> 1);
  if (pair >= sc.n_units) return;   // both CTAs of the pair, before any barrier
  const uint32_t rank = tc::cluster_rank();
  const bool leader = rank == 0;

  const uint32_t raw = tc::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase;
  const uint32_t sB = sbase + kStages2 * kStageA2;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages2 * (kStageA2 + kStageB2));
  const uint32_t bar0 = tc::smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kStages2 + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStages2 + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages2 + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kStages2 + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars2);
  volatile uint32_t* abort_flag = tmem_holder + 1;
  // written by the other CTA of the pair at the end: its abort flag and its
  // count of issued loads
  volatile uint32_t* peer_state = tmem_holder + 2;
  uint32_t issued = 0;   // loads this CTA's producer issued (thread 0)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages2; ++s) {
      tc::mbar_init(full(s), 1);    // the leader's: its expect_tx plus both CTAs' bytes
      tc::mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(acc_full(b), 1);
      tc::mbar_init(acc_empty(b), 8);   // the leader's: four epilogue warps in each CTA
    }
    tc::mbar_init(done_bar, 1);
    *abort_flag = 0u;
    tc::mbar_init_fence();
    tc::prefetch_tensormap(&tm_a);
    tc::prefetch_tensormap(&tm_b);
  }
  if (warp == 1) tc::tmem_alloc_pair(tc::smem_u32(tmem_holder), kTmemCols);
  tc::fence_before_sync();
  tc::cluster_sync_all();   // both CTAs' barriers initialised, tensor memory allocated in both
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = pair; ok && u < sc.n_units; u += n_pairs) {
        int rt, chunk, ks, kb0, kb1;
        sc.unit(u, rt, chunk, ks);
        sc.k_range(ks, kb0, kb1);
        const int t_end = min((chunk + 1) * sc.chunk_tiles, sc.n_col_tiles);
        for (int t = chunk * sc.chunk_tiles; ok && t < t_end; ++t) {
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::wait(empty(stage), phase ^ 1u, abort_flag, sc.wc)) {
              ok = false;
              break;
            }
            if (leader) tc::mbar_expect_tx(full(stage), 2 * (kStageA2 + kStageB2));
            const uint32_t lead_full = tc::map_to_rank(full(stage), 0);
            load_stage<A_MN, kBM, true>(sA + stage * kStageA2, &tm_a, kb * kBK, rt * 2 * kBM + rank * kBM, lead_full);
            load_stage<B_MN, kBN / 2, true>(sB + stage * kStageB2, &tm_b, kb * kBK, t * kBN + rank * (kBN / 2),
                                            lead_full);
            ++issued;
            if (++stage == kStages2) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the leader) ----------------
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = tc::idesc_f16(BF16, 2 * kBM, kBN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tc_count = 0;
      bool ok = true;
      for (int u = pair; ok && u < sc.n_units; u += n_pairs) {
        int rt, chunk, ks, kb0, kb1;
        sc.unit(u, rt, chunk, ks);
        sc.k_range(ks, kb0, kb1);
        const int t_end = min((chunk + 1) * sc.chunk_tiles, sc.n_col_tiles);
        for (int t = chunk * sc.chunk_tiles; ok && t < t_end; ++t, ++tc_count) {
          const uint32_t buf = tc_count & 1u, use = (tc_count >> 1) & 1u;
          if (!tc::wait(acc_empty(buf), use ^ 1u, abort_flag, sc.wc)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + buf * kBN;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!tc::wait(full(stage), phase, abort_flag, sc.wc)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint64_t da = stage_desc<A_MN>(sA + stage * kStageA2);
            const uint64_t db = stage_desc<B_MN>(sB + stage * kStageB2);
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk)
              tc::mma_f16_pair(d, da + kDescStep<A_MN> * kk, db + kDescStep<B_MN> * kk, idesc,
                               (kb > kb0 || kk > 0) ? 1u : 0u);
            tc::mma_commit_pair(empty(stage));   // frees this stage in both CTAs
            if (++stage == kStages2) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc::mma_commit_pair(acc_full(buf));
        }
      }
      // every pair MMA has completed before either CTA frees its memory
      tc::mma_commit_pair(done_bar);
      tc::wait_drain(done_bar, 0u, sc.wc);
    }
  } else {
    // ---------------- epilogue: warps 2-5 of both CTAs ----------------
    const int quarter = warp & 3;
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    EpiWarp ew{sbase + static_cast<uint32_t>(kEpiOff2) + static_cast<uint32_t>(quarter) * Epi::kStageBytes, 0, lane, 0u, 0};
    uint32_t tc_count = 0;
    bool ok = true;
    for (int u = pair; ok && u < sc.n_units; u += n_pairs) {
      int rt, chunk, ks;
      sc.unit(u, rt, chunk, ks);
      ew.ks = ks;
      const int t_beg = chunk * sc.chunk_tiles, t_end = min(t_beg + sc.chunk_tiles, sc.n_col_tiles);
      const int64_t row = static_cast<int64_t>(rt) * 2 * kBM + rank * kBM + r_in_tile;
      const bool row_ok = row < sc.M;
      ew.row0 = row - lane;
      typename Epi::State st = epi.begin(row, row_ok, chunk);
      for (int t = t_beg; t < t_end; ++t, ++tc_count) {
        const uint32_t buf = tc_count & 1u, use = (tc_count >> 1) & 1u;
        const bool got = lane == 0 ? tc::wait(acc_full(buf), use, abort_flag, sc.wc) : true;
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        __syncwarp();
        tc::fence_after_sync();
        // chunk c + 1 is read from tensor memory while chunk c is folded
        auto fold = [&](const uint32_t (&r)[32], int c) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          const int64_t cbase = static_cast<int64_t>(t) * kBN + c * 32;
          const int64_t left = sc.Ncols - cbase;
          const int nvalid = left <= 0 ? 0 : (left >= 32 ? 32 : static_cast<int>(left));
          epi.cols(st, v, row, row_ok, cbase, nvalid, ew);
        };
        const uint32_t acc = lane_addr + buf * kBN;
        uint32_t ra[32], rb[32];
        tc::tmem_ld32_issue(acc, ra);
        tc::tmem_ld32_wait(ra);
        for (int c = 0; c < kBN / 32; c += 2) {
          tc::tmem_ld32_issue(acc + (c + 1) * 32, rb);
          fold(ra, c);
          tc::tmem_ld32_wait(rb);
          if (c + 2 < kBN / 32) tc::tmem_ld32_issue(acc + (c + 2) * 32, ra);
          fold(rb, c + 1);
          if (c + 2 < kBN / 32) tc::tmem_ld32_wait(ra);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(tc::map_to_rank(acc_empty(buf), 0));
      }
      if (ok) epi.end(st, row, row_ok, chunk);
    }
    epi.finish(ew);
  }

  tc::fence_before_sync();
  __syncthreads();
  // Every role of this CTA is done.  Both CTAs' loads complete on the
  // leader's `full` barriers, so after an abort only the leader can tell when
  // a load still in flight has landed.  Each CTA tells the other its abort
  // flag and how many loads it issued, then the pair meets; no CTA leaves
  // while its pair may still read its memory.
  if (threadIdx.x == 0) {
    const uint32_t peer = rank ^ 1u;
    tc::st_cluster_u32(tc::map_to_rank(tc::smem_u32(const_cast<uint32_t*>(peer_state)), peer), *abort_flag);
    tc::st_cluster_u32(tc::map_to_rank(tc::smem_u32(const_cast<uint32_t*>(peer_state + 1)), peer), issued);
  }
  tc::cluster_sync_all();
  if (*abort_flag || peer_state[0]) {   // the same decision in both CTAs
    // After a normal run the MMA thread has waited for every load.  After an
    // abort the leader waits for the last load of each stage, both CTAs'
    // halves.  Per stage the two producers differ by at most one load (a
    // stage is refilled only after both halves of its previous load were
    // consumed), and a load only one of them issued is made whole: the
    // leader counts the missing half as done (complete_tx) or makes the
    // arrival its own producer never made (expect_tx of the peer's half).
    if (leader && threadIdx.x == 0) {
      const uint32_t peer_issued = peer_state[1];
      for (int s = 0; s < kStages2; ++s) {
        const uint32_t us = static_cast<uint32_t>(s);
        const uint32_t mine = issued > us ? (issued - 1 - us) / kStages2 + 1 : 0;
        const uint32_t theirs = peer_issued > us ? (peer_issued - 1 - us) / kStages2 + 1 : 0;
        if (mine == 0 && theirs == 0) continue;
        if (mine > theirs) tc::mbar_complete_tx(full(s), kStageA2 + kStageB2);
        else if (theirs > mine) tc::mbar_expect_tx(full(s), kStageA2 + kStageB2);
        const uint32_t last = (mine > theirs ? mine : theirs) - 1;
        tc::wait_drain(full(s), last & 1u, sc.wc);
      }
    }
    tc::cluster_sync_all();
  }
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Tensor map of a [rows, K] 16-bit row-major matrix with row stride ld
// (elements): a box of 64 x box_rows elements, 128-byte swizzle, zero fill
// outside the matrix.
bool encode_kmajor(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t K, int64_t ld,
                   int box_rows);

// Tensor map of the same operand stored MN-major: a [K, rows] 16-bit
// row-major matrix with row stride ld, boxes of 64 (rows) x 64 (K) elements,
// 128-byte swizzle, zero fill outside the matrix.
bool encode_mnmajor(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t K, int64_t ld);

// Tensor map of a [rows, cols] 16-bit row-major output with row stride ld for
// TMA stores of 32 x 32 boxes with 64-byte swizzle.  False when the base or
// the stride is not 16-byte aligned.
bool encode_store(CUtensorMap* map, void* base, bool bf16, int64_t rows, int64_t cols, int64_t ld);

// Either form, as the operand is stored.
inline bool encode_operand(CUtensorMap* map, bool mn, const void* base, bool bf16, int64_t rows, int64_t K,
                           int64_t ld, int box_rows) {
  return mn ? encode_mnmajor(map, base, bf16, rows, K, ld) : encode_kmajor(map, base, bf16, rows, K, ld, box_rows);
}

// 1 for the 1-SM kernel, 2 for CTA pairs (the default; a test build of the
// library can select the 1-SM form).  Defined by the C layer.
int cta_group();

template <bool BF16, bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm2(const void* A, int64_t lda, int64_t M, const void* Bm, int64_t ldb, int64_t Ncols,
                         int64_t K, int chunk_tiles, bool cols_fastest, const tc::WaitCtl& wc, const Epi& epi, int sms,
                         cudaStream_t s, int ksplit) {
  CUtensorMap tm_a, tm_b;
  if (!encode_operand(&tm_a, A_MN, A, BF16, M, K, lda, kBM) ||
      !encode_operand(&tm_b, B_MN, Bm, BF16, Ncols, K, ldb, kBN / 2))
    return cudaErrorInvalidValue;
  Sched sc = make_sched(M, Ncols, K, chunk_tiles, wc, 2 * kBM, ksplit);   // 256-row tiles
  sc.cols_fastest = cols_fastest ? 1 : 0;
  auto kern = gemm2_kernel<BF16, A_MN, B_MN, Epi>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  // per device and kernel, once: the shared-memory opt-in and the number of
  // resident pairs (runtime queries are kept out of stream capture)
  // (atomics: calls may come from several host threads; a repeated query is harmless)
  static std::atomic<int> resident_on[kMaxDev];
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  constexpr size_t smem = 1024 + kEpiOff2 + 4 * static_cast<size_t>(Epi::kStageBytes);
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // a persistent grid: only as many pairs as can be resident at once (a GPC
  // with an odd number of free SMs leaves one idle)
  int resident = resident_on[dev].load(std::memory_order_acquire);
  if (resident == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    if (cudaOccupancyMaxActiveClusters(&resident, kern, &cfg) != cudaSuccess || resident < 1) {
      cudaGetLastError();
      resident = sms / 2;
    }
    resident_on[dev].store(resident, std::memory_order_release);
  }
  const int pairs = sc.n_units < resident ? sc.n_units : resident;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  return cudaLaunchKernelEx(&cfg, kern, tm_a, tm_b, sc, epi);
}

// Split-K factor for an M x Ncols output (chunk_tiles 1) with K to reduce:
// the number of K runs, at most max_runs and each at least min_k_blocks K
// blocks long, that minimises a plain time model, or 1 when no split saves
// 3%.  The model charges the persistent grid's waves of units (tiles x runs
// over the resident CTAs or pairs) times the K blocks a unit walks, at the
// tensor rate, plus the fp32 partial sums' round trip through memory
// (written by every run and read by the reduction).  The rates are this
// GPU's: about 1.9 PFLOP/s dense bf16 and 6.8 TB/s.
inline int fill_ksplit(int64_t M, int64_t Ncols, int64_t K, int sms, int min_k_blocks, int64_t max_runs) {
  constexpr double kTensorFlops = 1.9e15, kHbmBytes = 6.8e12;
  const bool pair = cta_group() == 2 && sms >= 2;
  const int64_t rows = pair ? 2 * kBM : kBM;
  const int64_t slots = pair ? sms / 2 : sms;
  if (slots < 1) return 1;
  const int64_t tiles = ((M + rows - 1) / rows) * ((Ncols + kBN - 1) / kBN);
  const int64_t nk = (K + kBK - 1) / kBK;
  int64_t kmax = nk / (min_k_blocks > 0 ? min_k_blocks : 1);
  if (kmax > max_runs) kmax = max_runs;
  const double t_block = 2.0 * rows * kBN * kBK / (kTensorFlops / static_cast<double>(slots));
  auto time = [&](int64_t k) {
    const int64_t waves = (tiles * k + slots - 1) / slots;
    const int64_t blocks = (nk + k - 1) / k;
    const double partials = k > 1 ? 2.0 * static_cast<double>(k) * M * Ncols * 4.0 / kHbmBytes : 0.0;
    return static_cast<double>(waves * blocks) * t_block + partials;
  };
  const double t1 = time(1);
  int64_t best = 1;
  double best_t = t1;
  for (int64_t k = 2; k <= kmax; ++k) {
    const double t = time(k);
    if (t < best_t) {
      best = k;
      best_t = t;
    }
  }
  return best_t < 0.97 * t1 ? static_cast<int>(best) : 1;
}

// C = A B^T through the epilogue.  A_MN / B_MN: the operand is stored
// MN-major ([K, M] for A, [K, Ncols] for B, row stride lda / ldb), else
// K-major ([M, K], [Ncols, K]).  ksplit > 1: split-K (see make_sched).
template <bool BF16, bool A_MN = false, bool B_MN = false, class Epi>
cudaError_t launch_gemm(const void* A, int64_t lda, int64_t M, const void* Bm, int64_t ldb, int64_t Ncols,
                        int64_t K, int chunk_tiles, bool cols_fastest, const tc::WaitCtl& wc, const Epi& epi, int sms,
                        cudaStream_t s, int ksplit = 1) {
  if (cta_group() == 2 && sms >= 2)
    return launch_gemm2<BF16, A_MN, B_MN>(A, lda, M, Bm, ldb, Ncols, K, chunk_tiles, cols_fastest, wc, epi, sms,
                                          s, ksplit);
  CUtensorMap tm_a, tm_b;
  if (!encode_operand(&tm_a, A_MN, A, BF16, M, K, lda, kBM) || !encode_operand(&tm_b, B_MN, Bm, BF16, Ncols, K, ldb, kBN))
    return cudaErrorInvalidValue;
  Sched sc = make_sched(M, Ncols, K, chunk_tiles, wc, kBM, ksplit);
  sc.cols_fastest = cols_fastest ? 1 : 0;
  auto kern = gemm_kernel<BF16, A_MN, B_MN, Epi>;
  constexpr size_t smem = 1024 + kEpiOff + 4 * static_cast<size_t>(Epi::kStageBytes);
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  static std::atomic<bool> opted_in[kMaxDev];   // per device and kernel, once (or again, harmlessly)
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  const int grid = sc.n_units < sms ? sc.n_units : sms;
  kern<<<grid, kThreads, smem, s>>>(tm_a, tm_b, sc, epi);
  return cudaGetLastError();
}

}  // namespace tcg
}  // namespace vls
