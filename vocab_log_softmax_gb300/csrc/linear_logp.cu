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
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc_gemm.cuh"

namespace vls {

namespace {

// logits of the id among v[0..31] at position loc (0 <= loc < 32)
__device__ __forceinline__ float pick32(const float (&v)[32], int loc) {
  float r = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) r = loc == i ? v[i] : r;
  return r;
}

// Epilogue of the forward: each row's online (max, sum of exponentials) over
// the unit's chunk of columns, the logits of its target ids, and at the end
// of the unit one vls_partial and the targets' logits.
struct LogpEpi {
  static constexpr uint32_t kStageBytes = 0;
  const int64_t* ids;
  int32_t k;
  int64_t N;
  vls_partial* part;   // [S, N]
  float* zt;           // [S, N, k]

  struct State {
    float m, s;
    int64_t id[kLinMaxTopk];
    float zt[kLinMaxTopk];
  };

  __device__ State begin(int64_t row, bool row_ok, int) const {
    State st;
    st.m = dev::neg_inf();
    st.s = 0.0f;
#pragma unroll
    for (int j = 0; j < kLinMaxTopk; ++j) {
      st.id[j] = (row_ok && j < k) ? ids[row * k + j] : -1;
      st.zt[j] = 0.0f;
    }
    return st;
  }

  __device__ void cols(State& st, const float (&v)[32], int64_t, bool, int64_t cbase, int nvalid,
                       tcg::EpiWarp&) const {
    float cmax = dev::neg_inf();
    float cs = 0.0f;   // z - m is formed first, as in the row sweeps
    if (nvalid == 32) {   // every chunk but the vocabulary's last
      cmax = v[0];
#pragma unroll
      for (int i = 1; i < 31; i += 2) cmax = dev::max3(cmax, v[i], v[i + 1]);
      cmax = fmaxf(cmax, v[31]);
      if (cmax > st.m) {
        st.s = st.m == dev::neg_inf() ? 0.0f : st.s * dev::ex2((st.m - cmax) * dev::kLog2e);
        st.m = cmax;
      }
      const dev::fp2 m2 = dev::splat(st.m), l2 = dev::splat(dev::kLog2e);
      dev::fp2 acc = dev::splat(0.0f);
#pragma unroll
      for (int i = 0; i < 32; i += 2)
        acc = dev::add2(acc, dev::ex2_2(dev::mul2(dev::sub2(dev::pk(v[i], v[i + 1]), m2), l2)));
      cs = dev::sum2(acc);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) cmax = i < nvalid ? fmaxf(cmax, v[i]) : cmax;
      if (cmax > st.m) {
        st.s = st.m == dev::neg_inf() ? 0.0f : st.s * dev::ex2((st.m - cmax) * dev::kLog2e);
        st.m = cmax;
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) cs += i < nvalid ? dev::ex2((v[i] - st.m) * dev::kLog2e) : 0.0f;
    }
    st.s += cs;
#pragma unroll
    for (int j = 0; j < kLinMaxTopk; ++j) {
      if (j >= k) break;   // k is uniform: the loop stops after the row's own ids
      const int64_t loc = st.id[j] - cbase;
      if (loc >= 0 && loc < nvalid) st.zt[j] = pick32(v, static_cast<int>(loc));
    }
  }

  __device__ void finish(tcg::EpiWarp&) const {}

  __device__ void end(State& st, int64_t row, bool row_ok, int chunk) const {
    if (!row_ok) return;
    part[static_cast<int64_t>(chunk) * N + row] = vls_partial{st.m, st.s, 0.0f, 0.0f, 0.0f, 0u};
    float* z = zt + (static_cast<int64_t>(chunk) * N + row) * k;
#pragma unroll
    for (int j = 0; j < kLinMaxTopk; ++j)
      if (j < k) z[j] = st.zt[j];
  }
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};   // looked up once (or again, harmlessly)
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (!f) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
      fn.store(f, std::memory_order_release);
    } else {
      cudaGetLastError();
    }
  }
  return f;
}

}  // namespace

namespace tcg {

bool encode_kmajor(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t K, int64_t ld,
                   int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_mnmajor(CUtensorMap* map, const void* base, bool bf16, int64_t rows, int64_t K, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(K)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBK)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_store(CUtensorMap* map, void* base, bool bf16, int64_t rows, int64_t cols, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcg

int64_t linear_chunks(int64_t V) {
  const int64_t tiles = (V + tcg::kBN - 1) / tcg::kBN;
  return (tiles + kLinChunkTiles - 1) / kLinChunkTiles;
}

cudaError_t launch_linear_logp(const LinearArgs& la, int sms, cudaStream_t s) {
  const LogpEpi epi{la.ids, la.k, la.N, la.part, la.zt};
  const tc::WaitCtl wc{la.status, la.sticky, la.wait_ns};
  return la.dt == VLS_BF16
             ? tcg::launch_gemm<true>(la.h, la.ldh, la.N, la.W, la.ldw, la.V, la.D, kLinChunkTiles, false, wc, epi, sms, s)
             : tcg::launch_gemm<false>(la.h, la.ldh, la.N, la.W, la.ldw, la.V, la.D, kLinChunkTiles, false, wc, epi, sms, s);
}

}  // namespace vls
