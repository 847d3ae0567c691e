// One-read forward sweep: per-row max / sum-exp (and the entropy or KL
// weighted sum) in a single pass over the logits, then the row's outputs.
//
// Launch shape: a cluster of `cluster` CTAs per row (cluster size a function
// of V only), each CTA owning a contiguous run of 8-column vectors.  Inside a
// CTA, thread t owns vectors t, t + 256, t + 512, ... of that run and folds
// them in increasing order into its online state; the states are then
// combined by a fixed tree: lanes (xor 16..1), warps (xor 4..1 over 8
// warps), cluster ranks (xor 4..1 over up to 8 ranks, through distributed
// shared memory into rank 0).  Nothing in that order depends on N, on the
// row's position or on its alignment, so results are deterministic and batch
// invariant (the reduction-tree rule of "TP4 GDN, convolution and D=256
// attention mixers", RL-Kernel PR #507, and the one-block-per-row,
// fixed-tree rule of RL-Kernel PR #495, Summary).
#pragma once

#include "vls_device.cuh"

namespace vls {

template <int OP>
struct FwdState;
template <>
struct FwdState<kFwdLogp> { using type = dev::LogpState; };
template <>
struct FwdState<kFwdEntropy> { using type = dev::EntropyState; };
template <>
struct FwdState<kFwdKl> { using type = dev::KlState; };

template <class T, int OP, bool CAP>
__device__ __forceinline__ void fold_vec(typename FwdState<OP>::type& st, float (&zx)[8],
                                         float (&zy)[8], int nx, float cap, float rcap) {
  using namespace dev;
  apply_cap8<CAP>(zx, cap, rcap);
  if (nx < 8) mask_tail(zx, nx);
  if constexpr (OP == kFwdKl) {
    apply_cap8<CAP>(zy, cap, rcap);
    if (nx < 8) mask_tail(zy, nx);
    st.update(zx, zy);
  } else {
    st.update(zx);
  }
}

template <class T, int OP, bool CAP>
__global__ void __launch_bounds__(kRowThreads) row_fwd_kernel(const FwdArgs a) {
  using namespace dev;
  using S = typename FwdState<OP>::type;
  __shared__ S warp_part[kRowWarps];
  __shared__ S cta_part[kMaxCluster];
  __shared__ S row_state;

  const int C = a.cluster;
  const int64_t row = blockIdx.x / C;
  const int q = static_cast<int>(blockIdx.x - row * C);
  if (C > 1) cluster_arrive_relaxed();

  const T* xr = static_cast<const T*>(a.x) + row * a.ldx;
  const T* yr = OP == kFwdKl ? static_cast<const T*>(a.y) + row * a.ldy : nullptr;
  const int64_t V = a.vocab;
  const int64_t nvec = (V + 7) >> 3;
  const int64_t vb = static_cast<int64_t>(q) * a.vec_per_cta;
  const int64_t ve = min(vb + a.vec_per_cta, nvec);
  const int64_t vfull_end = min(ve, V >> 3);
  const bool al = aligned16(xr) && (OP != kFwdKl || aligned16(yr));

  S st = S::identity();
  int64_t v = vb + threadIdx.x;
  if (al) {
    // unrolled body: kUnroll 16-byte loads in flight per tensor before any use
    for (; v + (kUnroll - 1) * kRowThreads < vfull_end; v += kUnroll * kRowThreads) {
      float zx[kUnroll][8], zy[kUnroll][8];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        Elem<T>::load8(xr + 8 * (v + u * kRowThreads), zx[u]);
        if constexpr (OP == kFwdKl) Elem<T>::load8(yr + 8 * (v + u * kRowThreads), zy[u]);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) fold_vec<T, OP, CAP>(st, zx[u], zy[u], 8, a.cap, a.rcap);
    }
  }
  // remaining vectors, the partial last vector and unaligned rows: same
  // vectors, same order, same arithmetic
  for (; v < ve; v += kRowThreads) {
    float zx[8], zy[8];
    int nx = 8, ny = 8;
    load_vec(xr, v, V, al, zx, nx);
    if constexpr (OP == kFwdKl) load_vec(yr, v, V, al, zy, ny);
    fold_vec<T, OP, CAP>(st, zx, zy, nx, a.cap, a.rcap);
  }

  // ---- fixed-tree reduction: lanes, warps, cluster ranks ----
  st = warp_reduce(st);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_part[warp] = st;
  __syncthreads();
  S blk = S::identity();
  if (warp == 0) {
    blk = reduce8(lane < kRowWarps ? warp_part[lane] : S::identity());
    if (lane == 0 && C == 1) row_state = blk;
  }
  if (C > 1) {
    cluster_wait();  // every CTA of the cluster is resident: DSMEM is safe to use
    if (threadIdx.x == 0) {
      S* dst = cg::this_cluster().map_shared_rank(cta_part, 0);
      dst[q] = blk;
    }
    cluster_arrive();
    cluster_wait();  // all partials have landed in rank 0
    if (q != 0) return;
    if (warp == 0) {
      const S r = reduce8(lane < C ? cta_part[lane] : S::identity());
      if (lane == 0) row_state = r;
    }
  }
  __syncthreads();

  // ---- finalise (rank 0 of the row) ----
  const S fin = row_state;
  if constexpr (OP == kFwdLogp) {
    const float m = fin.m;
    const float log_s = logf(fin.s);
    if (threadIdx.x == 0) a.stats_x[row] = vls_rowstat{m, log_s};
    for (int j = threadIdx.x; j < a.k; j += kRowThreads) {
      const int64_t id = a.ids[row * a.k + j];
      float out = 0.0f;
      if (valid_id(id, V, a.ignore_index)) {
        float z = Elem<T>::load1(xr + id);
        if (CAP) z = softcap_z(z, a.cap, a.rcap);
        out = m == neg_inf() ? qnan() : (z - m) - log_s;
      }
      a.logp[row * a.k + j] = out;
    }
  } else if constexpr (OP == kFwdEntropy) {
    if (threadIdx.x == 0) {
      const float log_s = logf(fin.s);
      a.stats_x[row] = vls_rowstat{fin.m, log_s};
      a.out[row] = fin.m == neg_inf() ? qnan() : log_s - fin.w / fin.s;
    }
  } else {
    if (threadIdx.x == 0) {
      const float log_sp = logf(fin.sp), log_sq = logf(fin.sq);
      a.stats_x[row] = vls_rowstat{fin.mp, log_sp};
      a.stats_y[row] = vls_rowstat{fin.mq, log_sq};
      float kl;
      if (fin.mp == neg_inf() || fin.mq == neg_inf())
        kl = qnan();
      else if (fin.flag)
        kl = pos_inf();
      else
        kl = fin.w / fin.sp + (log_sq - log_sp);
      a.out[row] = kl;
    }
  }
}

template <class T, int OP, bool CAP>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.rows * a.cluster));
  cfg.blockDim = dim3(kRowThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, row_fwd_kernel<T, OP, CAP>, a);
}

template <int OP>
cudaError_t launch_fwd_op(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16)
    return cap ? launch_fwd_t<__nv_bfloat16, OP, true>(a, s) : launch_fwd_t<__nv_bfloat16, OP, false>(a, s);
  return cap ? launch_fwd_t<float, OP, true>(a, s) : launch_fwd_t<float, OP, false>(a, s);
}

}  // namespace vls
