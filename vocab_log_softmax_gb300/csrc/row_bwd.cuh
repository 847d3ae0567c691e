// Backward sweeps: with the forward's per-row (m, log S) saved, every
// gradient is a pointwise map of the row -- one read of the logits (two for
// KL) and one write of the gradient in the logits dtype, no workspace and no
// reduction over the row ("perf(logp): fused zero-workspace backward for the
// generic CUDA fused logp", RL-Kernel PR #495, Summary: dlogits =
// grad*(one_hot - softmax) written straight into the logits dtype).
//
// Launch shape: `chunks` CTAs per row, each owning a contiguous run of
// 8-column vectors.  The gradient of a column does not depend on which CTA
// computes it, so the chunking has no effect on results.
#pragma once

#include "vls_device.cuh"

namespace vls {

// p = exp((z - m) - log S), formed as 2^((z - m) log2 e - log S log2 e); z - m
// is exact for bf16 logits and keeps a large common offset out of the
// exponent.
__device__ __forceinline__ float prob(float z, float m, float log_s_l2e) {
  return dev::ex2(fmaf(z - m, dev::kLog2e, -log_s_l2e));
}

// Per-CTA prepared form of a row's top-k ids: G = sum of the upstream
// gradients of the valid ids (ascending j), and, for each distinct valid id
// that falls in this CTA's columns, the sum of its upstream gradients
// (ascending j).  DeepSpeed PR #8838, Changes: the top-k one-hot terms are
// added in fp32 before the single cast.
struct TopkPrep {
  float G;
  int nfix;
};

__device__ __forceinline__ TopkPrep prep_topk(const BwdArgs& a, int64_t row, int64_t col_beg,
                                              int64_t col_end, int64_t* s_id, float* s_g,
                                              int64_t* fix_id, float* fix_g, float* s_G,
                                              int* s_nfix) {
  const int k = a.k;
  const int64_t V = a.vocab;
  const int64_t* ids = a.ids + row * k;
  const float* g = a.g + row * k;
  if (threadIdx.x == 0) *s_nfix = 0;
  for (int j = threadIdx.x; j < k; j += kRowThreads) {
    s_id[j] = ids[j];
    s_g[j] = g[j];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float G = 0.0f;
    for (int j = 0; j < k; ++j)
      if (dev::valid_id(s_id[j], V, a.ignore_index)) G += s_g[j];
    *s_G = G;
  }
  for (int j = threadIdx.x; j < k; j += kRowThreads) {
    const int64_t id = s_id[j];
    if (!dev::valid_id(id, V, a.ignore_index) || id < col_beg || id >= col_end) continue;
    bool first = true;
    for (int i = 0; i < j && first; ++i) first = s_id[i] != id;
    if (!first) continue;
    float gs = 0.0f;
    for (int i = j; i < k; ++i)
      if (s_id[i] == id) gs += s_g[i];
    const int slot = atomicAdd(s_nfix, 1);
    fix_id[slot] = id;
    fix_g[slot] = gs;
  }
  __syncthreads();
  return TopkPrep{*s_G, *s_nfix};
}

template <class T, int OP, bool CAP>
__global__ void __launch_bounds__(kRowThreads) row_bwd_kernel(const BwdArgs a) {
  using namespace dev;
  const int64_t row = blockIdx.x / a.chunks;
  const int q = static_cast<int>(blockIdx.x - row * a.chunks);
  const int64_t V = a.vocab;
  const int64_t nvec = (V + 7) >> 3;
  const int64_t vb = static_cast<int64_t>(q) * a.vec_per_cta;
  const int64_t ve = min(vb + a.vec_per_cta, nvec);
  const T* xr = static_cast<const T*>(a.x) + row * a.ldx;
  const T* yr = OP >= kBwdKlReverse ? static_cast<const T*>(a.y) + row * a.ldy : nullptr;
  T* dr = static_cast<T*>(a.dx) + row * V;
  const bool al = aligned16(xr) && aligned16(dr) && (OP < kBwdKlReverse || aligned16(yr));

  const vls_rowstat sx = a.stats_x[row];
  const float m = sx.m, log_s_l2e = sx.log_s * kLog2e;

  // ---- per-row constants; rows whose gradient is a constant (zero / NaN) ----
  float G = 0.0f, K = 0.0f, gr = 0.0f;
  float mq = 0.0f, log_sq_l2e = 0.0f;
  int nfix = 0;
  bool nan_row = false, zero_row = false;
  constexpr int kFix = OP == kBwdLogp ? VLS_MAX_TOPK : 1;
  __shared__ int64_t fix_id[kFix];
  __shared__ float fix_g[kFix];
  if constexpr (OP == kBwdLogp) {
    __shared__ int64_t s_id[VLS_MAX_TOPK];
    __shared__ float s_g[VLS_MAX_TOPK];
    __shared__ float s_G;
    __shared__ int s_nfix;
    const int64_t col_beg = vb * 8, col_end = min(ve * 8, V);
    if (a.k == 1) {
      const int64_t id = a.ids[row];
      if (valid_id(id, V, a.ignore_index)) {
        G = a.g[row];
        if (id >= col_beg && id < col_end) {
          nfix = 1;
          if (threadIdx.x == 0) {
            fix_id[0] = id;
            fix_g[0] = G;
          }
        }
      } else {
        zero_row = true;
      }
    } else {
      const TopkPrep tp = prep_topk(a, row, col_beg, col_end, s_id, s_g, fix_id, fix_g, &s_G, &s_nfix);
      G = tp.G;
      nfix = tp.nfix;
      bool any_valid = false;
      for (int j = 0; j < a.k && !any_valid; ++j) any_valid = valid_id(s_id[j], V, a.ignore_index);
      zero_row = !any_valid;
    }
    G = -G;  // the streamed value is -G * p
  } else if constexpr (OP == kBwdEntropy) {
    const float H = a.fout[row];
    gr = -a.g[row];
    K = sx.log_s - H;  // log p + H = (z - m) - K
    nan_row = m == neg_inf() || isnan(H);
  } else {
    const vls_rowstat sy = a.stats_y[row];
    mq = sy.m;
    log_sq_l2e = sy.log_s * kLog2e;
    const float kl = a.fout[row];
    gr = a.g[row];
    if constexpr (OP == kBwdKlReverse) {
      K = (sx.log_s - sy.log_s) + kl;  // (log p_a - log p_b) - KL = (da - db) - K
      nan_row = !isfinite(kl);
    } else {
      nan_row = isnan(kl);
    }
  }

  if (zero_row || nan_row) {
    float c[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = nan_row ? qnan() : 0.0f;
    for (int64_t v = vb + threadIdx.x; v < ve; v += kRowThreads) store_vec(dr, v, V, al, c);
    return;
  }

  auto grad8 = [&](float (&x)[8], float (&y)[8], float (&out)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float z = x[j], chain = 1.0f;
      if (CAP) {
        const float u = x[j] * a.rcap;
        const float t = tanhf(u);
        z = a.cap * t;
        chain = softcap_dzdx(u, t);
      }
      float r;
      if constexpr (OP == kBwdLogp) {
        r = G * prob(z, m, log_s_l2e);
      } else if constexpr (OP == kBwdEntropy) {
        const float d = z - m;
        r = gr * ex2(fmaf(d, kLog2e, -log_s_l2e)) * (fmaxf(d, -kFltMax) - K);
      } else {
        const float zb = CAP ? softcap_z(y[j], a.cap, a.rcap) : y[j];
        const float da = z - m, db = zb - mq;
        const float pa = ex2(fmaf(da, kLog2e, -log_s_l2e));
        if constexpr (OP == kBwdKlReverse) {
          r = gr * pa * ((fmaxf(da, -kFltMax) - fmaxf(db, -kFltMax)) - K);
        } else {
          r = gr * (pa - ex2(fmaf(db, kLog2e, -log_sq_l2e)));
        }
      }
      out[j] = CAP ? r * chain : r;
    }
  };

  int64_t v = vb + threadIdx.x;
  const int64_t vfull_end = min(ve, V >> 3);
  if (al) {
    for (; v + (kUnroll - 1) * kRowThreads < vfull_end; v += kUnroll * kRowThreads) {
      float x[kUnroll][8], y[kUnroll][8];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        Elem<T>::load8(xr + 8 * (v + u * kRowThreads), x[u]);
        if constexpr (OP >= kBwdKlReverse) Elem<T>::load8(yr + 8 * (v + u * kRowThreads), y[u]);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        float out[8];
        grad8(x[u], y[u], out);
        Elem<T>::store8(dr + 8 * (v + u * kRowThreads), out);
      }
    }
  }
  for (; v < ve; v += kRowThreads) {
    float x[8], y[8], out[8];
    int nx = 8, ny = 8;
    load_vec(xr, v, V, al, x, nx);
    if constexpr (OP >= kBwdKlReverse) load_vec(yr, v, V, al, y, ny);
    grad8(x, y, out);
    store_vec(dr, v, V, al, out);
  }

  if constexpr (OP == kBwdLogp) {
    // one-hot columns: rewrite with (g_sum - G p) * dz/dx, one rounding
    if (nfix > 0) {
      __syncthreads();  // the streamed stores of this CTA precede the rewrites
      for (int f = threadIdx.x; f < nfix; f += kRowThreads) {
        const int64_t c = fix_id[f];
        const float x = Elem<T>::load1(xr + c);
        float z = x, chain = 1.0f;
        if (CAP) {
          const float u = x * a.rcap;
          const float t = tanhf(u);
          z = a.cap * t;
          chain = softcap_dzdx(u, t);
        }
        const float r = fmaf(G, prob(z, m, log_s_l2e), fix_g[f]);
        Elem<T>::store1(dr + c, CAP ? r * chain : r);
      }
    }
  }
}

template <class T, int OP, bool CAP>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.rows * a.chunks));
  row_bwd_kernel<T, OP, CAP><<<grid, kRowThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int OP>
cudaError_t launch_bwd_op(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16)
    return cap ? launch_bwd_t<__nv_bfloat16, OP, true>(a, s) : launch_bwd_t<__nv_bfloat16, OP, false>(a, s);
  return cap ? launch_bwd_t<float, OP, true>(a, s) : launch_bwd_t<float, OP, false>(a, s);
}

}  // namespace vls
