// Vocabulary-parallel combine: folds the R shards' partial states of a row
// in rank order 0..R-1 and finalises it with the same functions as the
// unsharded forward sweep (DeepSpeed PR #8838, Changes and review "Suggested
// change": local statistics re-centred on the global max).  One warp per
// row.  The lanes load 32 partials at a time and every lane folds them in
// rank order through shuffles, so the loads overlap while the fold keeps its
// one order.  Target logits: each id is owned by one shard (the others hold
// +0), so any order of their sum is exact.
#include <cstring>

#include "row_fwd.cuh"

namespace vls {

constexpr int kCombineThreads = 256;
constexpr int kCombineRows = kCombineThreads / 32;

template <int OP>
struct CombineState;
template <>
struct CombineState<kFwdLogp> { using type = LogpState; };
template <>
struct CombineState<kFwdEntropy> { using type = EntropyState; };
template <>
struct CombineState<kFwdKl> { using type = KlState; };

// v from lane src, field by field
template <class S>
__device__ __forceinline__ S shfl_state(const S& v, int src) {
  static_assert(sizeof(S) % 4 == 0, "states are made of 32-bit fields");
  constexpr int W = sizeof(S) / 4;
  uint32_t w[W];
  memcpy(w, &v, sizeof(S));
#pragma unroll
  for (int i = 0; i < W; ++i) w[i] = __shfl_sync(0xffffffffu, w[i], src);
  S r;
  memcpy(&r, w, sizeof(S));
  return r;
}

template <int OP, bool CAP>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
  using S = typename CombineState<OP>::type;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kCombineRows + warp;
  if (row >= a.rows) return;  // whole warps only
  S fin = S::identity();
  for (int base = 0; base < a.R; base += 32) {
    S mine = S::identity();
    if (base + lane < a.R) from_partial(a.parts[static_cast<int64_t>(base + lane) * a.rows + row], mine);
    const int cnt = a.R - base < 32 ? a.R - base : 32;
    for (int i = 0; i < cnt; ++i) fin = S::combine(fin, shfl_state(mine, i));
  }
  if constexpr (OP == kFwdLogp) {
    const CapK K = cap_consts(CAP ? a.cap : 1.0f);
    const float log_s = logf(fin.s);
    if (lane == 0) a.stats_x[row] = vls_rowstat{fin.m, log_s};
    if (a.R > 8) {
      // many shards: the lanes gather one id's R values at a time
      for (int j = 0; j < a.k; ++j) {
        const int64_t id = a.ids[row * a.k + j];
        float out = 0.0f;
        if (valid_id(id, a.vocab_total, a.ignore_index)) {
          float x = 0.0f;
          for (int r = lane; r < a.R; r += 32) x += a.zt[(static_cast<int64_t>(r) * a.rows + row) * a.k + j];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
          out = logp_of<CAP>(x, fin.m, log_s, K);
        }
        if (lane == 0) a.logp[row * a.k + j] = out;
      }
    } else {
      // few shards: each lane gathers its own ids
      for (int j = lane; j < a.k; j += 32) {
        const int64_t id = a.ids[row * a.k + j];
        float out = 0.0f;
        if (valid_id(id, a.vocab_total, a.ignore_index)) {
          float x = 0.0f;
          for (int r = 0; r < a.R; ++r) x += a.zt[(static_cast<int64_t>(r) * a.rows + row) * a.k + j];
          out = logp_of<CAP>(x, fin.m, log_s, K);
        }
        a.logp[row * a.k + j] = out;
      }
    }
  } else if constexpr (OP == kFwdEntropy) {
    if (lane == 0) {
      const float log_s = logf(fin.s);
      a.stats_x[row] = vls_rowstat{fin.m, log_s};
      a.out[row] = entropy_of(fin, log_s);
    }
  } else {
    if (lane == 0) {
      const float log_sp = logf(fin.sp), log_sq = logf(fin.sq);
      a.stats_x[row] = vls_rowstat{fin.mp, log_sp};
      a.stats_y[row] = vls_rowstat{fin.mq, log_sq};
      a.out[row] = kl_of(fin, log_sp, log_sq);
    }
  }
}

cudaError_t launch_combine(FwdOp op, const CombineArgs& a, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((a.rows + kCombineRows - 1) / kCombineRows);
  if (op == kFwdLogp) {
    if (a.cap > 0.0f)
      combine_kernel<kFwdLogp, true><<<grid, kCombineThreads, 0, s>>>(a);
    else
      combine_kernel<kFwdLogp, false><<<grid, kCombineThreads, 0, s>>>(a);
  } else if (op == kFwdEntropy) {
    combine_kernel<kFwdEntropy, false><<<grid, kCombineThreads, 0, s>>>(a);
  } else {
    combine_kernel<kFwdKl, false><<<grid, kCombineThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace vls
