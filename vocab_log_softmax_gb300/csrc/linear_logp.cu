// Fused linear head + target log-probabilities on the tcgen05 tensor cores.
//
// The logits z = h @ W^T (h: [N, D] hidden states, W: [V, D] head weights,
// both 16-bit) are never written to memory.  A persistent kernel walks work
// units of (128 rows) x (one vocabulary chunk of kLinChunkTiles tiles of 256
// columns).  For each tile, TMA streams 64-wide K slices of h and W into a
// 4-stage shared-memory ring, one thread issues 128x256x16 MMAs into a
// tensor-memory accumulator (two accumulators, so the epilogue of one tile
// overlaps the MMAs of the next), and four epilogue warps read the finished
// tile row by row from tensor memory and fold it into each row's online
// (max, sum of exponentials), capturing the logits of the row's target ids.
// Each unit ends by writing one vls_partial per row and the owned targets'
// logits: the same split-phase format as the vocabulary-parallel calls, so
// vls_logp_combine folds the chunks in order into logp and (m, log S).
//
// The linear head itself is the reading of the pages' linear_logp op
// ("perf(logp): fused zero-workspace backward ...", RL-Kernel PR #495,
// Summary); the statistics are those of the single-read logprob forward
// ("Add Triton kernels for vocab-parallel logprobs, entropy and KL",
// DeepSpeed PR #8838, Changes).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_device.cuh"
#include "vls_device.cuh"

namespace vls {

namespace {

constexpr int kLinBM = 128;            // rows per tile (MMA M)
constexpr int kLinBN = 256;            // vocabulary columns per tile (MMA N)
constexpr int kLinBK = 64;             // K per stage: one 128-byte swizzled row of 16-bit elements
constexpr int kLinUK = 16;             // K per MMA instruction (kind::f16)
constexpr int kLinStages = 4;
constexpr int kLinThreads = 192;       // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
constexpr uint32_t kStageA = kLinBM * kLinBK * 2;   // 16 KB
constexpr uint32_t kStageB = kLinBN * kLinBK * 2;   // 32 KB
constexpr uint32_t kTmemCols = 2 * kLinBN;          // two fp32 accumulators of 256 columns
constexpr int kNumBars = 2 * kLinStages + 4 + 1;    // full, empty, acc_full x2, acc_empty x2, done
constexpr size_t kLinSmem = 1024 /* alignment slack */ + kLinStages * (kStageA + kStageB) + kNumBars * 8 + 16;

struct LinArgs {
  int64_t N, D, V;
  const int64_t* ids;
  int32_t k;
  int64_t ignore_index;
  vls_partial* part;   // [S, N]
  float* zt;           // [S, N, k]
  uint32_t* status;    // device status word (tc::kStatusTimeout after a wait ran out)
  int n_row_tiles, n_vtiles, n_chunks, n_units, nk;
};

// logits of the id among v[0..31] at position loc (0 <= loc < 32)
__device__ __forceinline__ float pick32(const float (&v)[32], int loc) {
  float r = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) r = loc == i ? v[i] : r;
  return r;
}

template <bool BF16>
__global__ void __launch_bounds__(kLinThreads, 1)
    linear_logp_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                       const LinArgs a) {
  extern __shared__ unsigned char smem_raw[];
  if (static_cast<int>(blockIdx.x) >= a.n_units) return;  // whole CTA, before any barrier

  const uint32_t raw = tc::smem_u32(smem_raw);
  unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = tc::smem_u32(smem);
  const uint32_t sA = sbase;                                 // kLinStages x kStageA
  const uint32_t sB = sbase + kLinStages * kStageA;          // kLinStages x kStageB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLinStages * (kStageA + kStageB));
  const uint32_t bar0 = tc::smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (kLinStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kLinStages + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kLinStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kLinStages + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile uint32_t* abort_flag = tmem_holder + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kLinStages; ++s) {
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
    tc::prefetch_tensormap(&tm_h);
    tc::prefetch_tensormap(&tm_w);
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
      for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
        const int chunk = u / a.n_row_tiles, rt = u - chunk * a.n_row_tiles;
        const int t_end = min((chunk + 1) * kLinChunkTiles, a.n_vtiles);
        for (int t = chunk * kLinChunkTiles; ok && t < t_end; ++t) {
          for (int kb = 0; kb < a.nk; ++kb) {
            if (!tc::wait(empty(stage), phase ^ 1u, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc::mbar_expect_tx(full(stage), kStageA + kStageB);
            tc::tma_load_2d(sA + stage * kStageA, &tm_h, kb * kLinBK, rt * kLinBM, full(stage));
            tc::tma_load_2d(sB + stage * kStageB, &tm_w, kb * kLinBK, t * kLinBN, full(stage));
            ++issued;
            if (++stage == kLinStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // After an abort, wait for the loads still in flight before the CTA
      // releases its shared memory: the last load issued into each stage.
      if (!ok) {
        for (int s = 0; s < kLinStages; ++s) {
          if (issued > static_cast<uint32_t>(s)) {
            const uint32_t last = (issued - 1 - s) / kLinStages;   // loads into stage s before the last one
            tc::wait_drain(full(s), last & 1u, a.status);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16(BF16, kLinBM, kLinBN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tc_count = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
        const int chunk = u / a.n_row_tiles;
        const int t_end = min((chunk + 1) * kLinChunkTiles, a.n_vtiles);
        for (int t = chunk * kLinChunkTiles; ok && t < t_end; ++t, ++tc_count) {
          const uint32_t buf = tc_count & 1u, use = (tc_count >> 1) & 1u;
          if (!tc::wait(acc_empty(buf), use ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t d = tmem + buf * kLinBN;
          for (int kb = 0; kb < a.nk; ++kb) {
            if (!tc::wait(full(stage), phase, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint64_t da = tc::sdesc_sw128(sA + stage * kStageA);
            const uint64_t db = tc::sdesc_sw128(sB + stage * kStageB);
#pragma unroll
            for (int kk = 0; kk < kLinBK / kLinUK; ++kk) {
              // 16 elements = 32 bytes further along the swizzled row: +2 in the address field
              tc::mma_f16(d, da + 2ull * kk, db + 2ull * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            tc::mma_commit(empty(stage));   // frees the stage once these MMAs have read it
            if (++stage == kLinStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc::mma_commit(acc_full(buf));
        }
      }
      // every MMA this thread issued has completed before tensor memory is freed
      tc::mma_commit(done_bar);
      tc::wait_drain(done_bar, 0u, a.status);
    }
  } else {
    // ---------------- epilogue: warps 2-5 ----------------
    const int quarter = warp & 3;                 // the tensor-memory lanes this warp may read
    const int r_in_tile = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int k = a.k;
    uint32_t tc_count = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
      const int chunk = u / a.n_row_tiles, rt = u - chunk * a.n_row_tiles;
      const int t_beg = chunk * kLinChunkTiles, t_end = min(t_beg + kLinChunkTiles, a.n_vtiles);
      const int64_t row = static_cast<int64_t>(rt) * kLinBM + r_in_tile;
      const bool row_ok = row < a.N;
      int64_t id[kLinMaxTopk];
      float zt[kLinMaxTopk];
#pragma unroll
      for (int j = 0; j < kLinMaxTopk; ++j) {
        id[j] = (row_ok && j < k) ? a.ids[row * k + j] : -1;
        zt[j] = 0.0f;
      }
      float m = dev::neg_inf(), s = 0.0f;
      for (int t = t_beg; t < t_end; ++t, ++tc_count) {
        const uint32_t buf = tc_count & 1u, use = (tc_count >> 1) & 1u;
        // one lane waits and the warp follows it, so the warp-wide tensor-memory
        // loads below are never reached by part of a warp
        const bool got = lane == 0 ? tc::wait(acc_full(buf), use, abort_flag, a.status) : true;
        if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        __syncwarp();
        tc::fence_after_sync();
        for (int c = 0; c < kLinBN / 32; ++c) {
          float v[32];
          tc::tmem_ld32(lane_addr + buf * kLinBN + c * 32, v);
          const int64_t cbase = static_cast<int64_t>(t) * kLinBN + c * 32;
          const int64_t left = a.V - cbase;
          const int nvalid = left <= 0 ? 0 : (left >= 32 ? 32 : static_cast<int>(left));
          float cmax = dev::neg_inf();
#pragma unroll
          for (int i = 0; i < 32; ++i) cmax = i < nvalid ? fmaxf(cmax, v[i]) : cmax;
          if (cmax > m) {
            s = m == dev::neg_inf() ? 0.0f : s * dev::ex2((m - cmax) * dev::kLog2e);
            m = cmax;
          }
          float cs = 0.0f;   // z - m is formed first, as in the row sweeps
#pragma unroll
          for (int i = 0; i < 32; ++i) cs += i < nvalid ? dev::ex2((v[i] - m) * dev::kLog2e) : 0.0f;
          s += cs;
#pragma unroll
          for (int j = 0; j < kLinMaxTopk; ++j) {
            const int64_t loc = id[j] - cbase;
            if (loc >= 0 && loc < nvalid) zt[j] = pick32(v, static_cast<int>(loc));
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(acc_empty(buf));
      }
      if (ok && row_ok) {
        a.part[static_cast<int64_t>(chunk) * a.N + row] = vls_partial{m, s, 0.0f, 0.0f, 0.0f, 0u};
        float* z = a.zt + (static_cast<int64_t>(chunk) * a.N + row) * k;
#pragma unroll
        for (int j = 0; j < kLinMaxTopk; ++j)
          if (j < k) z[j] = zt[j];
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// Tensor map of a [rows, D] 16-bit matrix with row stride ld (elements): a
// box of 64 x box_rows elements, 128-byte swizzle, zero fill outside.
bool encode_2d(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t D, int64_t ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kLinBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int64_t linear_chunks(int64_t V) {
  const int64_t tiles = (V + kLinBN - 1) / kLinBN;
  return (tiles + kLinChunkTiles - 1) / kLinChunkTiles;
}

cudaError_t launch_linear_logp(const LinearArgs& la, int sms, cudaStream_t s) {
  const bool bf16 = la.dt == VLS_BF16;
  CUtensorMap tm_h, tm_w;
  if (!encode_2d(&tm_h, la.h, bf16, la.N, la.D, la.ldh, kLinBM) ||
      !encode_2d(&tm_w, la.W, bf16, la.V, la.D, la.ldw, kLinBN))
    return cudaErrorInvalidValue;
  LinArgs a;
  a.N = la.N;
  a.D = la.D;
  a.V = la.V;
  a.ids = la.ids;
  a.k = la.k;
  a.ignore_index = la.ignore_index;
  a.part = la.part;
  a.zt = la.zt;
  a.status = la.status;
  a.n_row_tiles = static_cast<int>((la.N + kLinBM - 1) / kLinBM);
  a.n_vtiles = static_cast<int>((la.V + kLinBN - 1) / kLinBN);
  a.n_chunks = static_cast<int>(linear_chunks(la.V));
  a.n_units = a.n_row_tiles * a.n_chunks;
  a.nk = static_cast<int>((la.D + kLinBK - 1) / kLinBK);
  auto kern = bf16 ? linear_logp_kernel<true> : linear_logp_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kLinSmem));
  if (e != cudaSuccess) return e;
  const int grid = a.n_units < sms ? a.n_units : sms;
  kern<<<grid, kLinThreads, kLinSmem, s>>>(tm_h, tm_w, a);
  return cudaGetLastError();
}

}  // namespace vls
