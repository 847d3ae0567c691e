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

using namespace dev;

// Ids are global vocabulary columns, valid against vocab_total; the CTA
// holds local columns [col_beg, col_end) of a shard that starts at global
// column vocab_offset (0 and V for an unsharded row).
//
// Per-CTA prepared form of a row's top-k ids (DeepSpeed PR #8838, Changes:
// the top-k one-hot terms are added in fp32 before the single cast):
//  - G, the sum of the upstream gradients of the valid ids, by a fixed tree
//    (each thread sums j = t, t+256, ... in order, then lanes xor 16..1,
//    then the 8 warp partials in order) -- the same bits in every CTA;
//  - the valid ids sorted as keys (id << 11 | j) by a shared-memory bitonic
//    sort, so duplicates sit together in ascending j; for each distinct id
//    in this CTA's columns, the sum of its upstream gradients in ascending j.
// Shared memory: keys[P] (P = next power of two >= k), fix_id[k], g[k],
// fix_g[k], and a bitmap of this CTA's 8-column vectors that hold a valid id
// (used by the top-k logprob map, which writes its one-hot columns inline):
// 8 P + 16 k + 4 ceil(vectors / 32) bytes.
struct TopkPrep {
  float G;
  int nfix;
  bool any_valid;
  const unsigned long long* key;   // the P sorted keys
  const float* g;                  // the k upstream gradients, by j
  const uint32_t* bitmap;          // vectors of this CTA that hold a valid id
  int P;
};

constexpr int kTopkJBits = 11;  // j < 2048 > VLS_MAX_TOPK

__host__ __device__ __forceinline__ int topk_pow2(int k) {
  int p = 1;
  while (p < k) p <<= 1;
  return p;
}

// keys[P] + fix_id[k] (8 bytes each) + g[k] + fix_g[k] (4 bytes each) + the
// vector bitmap
__host__ __device__ __forceinline__ size_t topk_smem_bytes(int k, int64_t vec_per_cta) {
  return 8 * static_cast<size_t>(topk_pow2(k)) + 16 * static_cast<size_t>(k) +
         4 * static_cast<size_t>((vec_per_cta + 31) / 32);
}

__device__ __forceinline__ TopkPrep prep_topk(const BwdArgs& a, int64_t row, int64_t col_beg, int64_t col_end,
                                              unsigned char* smem, int64_t*& fix_id, float*& fix_g,
                                              float* s_warp, int* s_nfix) {
  const int k = a.k;
  const int P = topk_pow2(k);
  const int64_t* ids = a.ids + row * k;
  const float* g = a.g + row * k;
  unsigned long long* key = reinterpret_cast<unsigned long long*>(smem);
  fix_id = reinterpret_cast<int64_t*>(key + P);
  float* s_g = reinterpret_cast<float*>(fix_id + k);
  fix_g = s_g + k;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(fix_g + k);
  constexpr unsigned long long kNone = ~0ull;

  if (threadIdx.x == 0) *s_nfix = 0;
  const int nwords = static_cast<int>((col_end - col_beg + 255) >> 8);   // one bit per 8-column vector
  for (int w = threadIdx.x; w < nwords; w += kRowThreads) bitmap[w] = 0u;
  float gpart = 0.0f;
  int any = 0;
  for (int j = threadIdx.x; j < P; j += kRowThreads) {
    unsigned long long kj = kNone;
    if (j < k) {
      const int64_t id = ids[j];
      const float gj = g[j];
      s_g[j] = gj;
      if (valid_id(id, a.vocab_total, a.ignore_index)) {
        kj = (static_cast<unsigned long long>(id) << kTopkJBits) | static_cast<unsigned long long>(j);
        gpart += gj;
        any = 1;
      }
    }
    key[j] = kj;
  }
  // G by a fixed tree
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) gpart += __shfl_xor_sync(0xffffffffu, gpart, off);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = gpart;
  const bool any_valid = __syncthreads_or(any) != 0;
  float G = 0.0f;
#pragma unroll
  for (int w = 0; w < kRowWarps; ++w) G += s_warp[w];

  // bitonic sort of the P keys, ascending
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < (P >> 1); t += kRowThreads) {
        const int lo = 2 * t - (t & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const unsigned long long x = key[lo], y = key[hi];
        if ((x > y) == up) {
          key[lo] = y;
          key[hi] = x;
        }
      }
      __syncthreads();
    }
  }

  // one fix-up entry per distinct id of this CTA's columns
  for (int s = threadIdx.x; s < k; s += kRowThreads) {
    const unsigned long long ks = key[s];
    if (ks == kNone) continue;
    const int64_t local = static_cast<int64_t>(ks >> kTopkJBits) - a.vocab_offset;
    if (s > 0 && (key[s - 1] >> kTopkJBits) == (ks >> kTopkJBits)) continue;
    if (local < col_beg || local >= col_end) continue;
    float gs = 0.0f;
    for (int t = s; t < k && (key[t] >> kTopkJBits) == (ks >> kTopkJBits); ++t)
      gs += s_g[key[t] & ((1ull << kTopkJBits) - 1)];
    const int slot = atomicAdd(s_nfix, 1);
    fix_id[slot] = local;
    fix_g[slot] = gs;
    const int64_t vi = (local - col_beg) >> 3;
    atomicOr(&bitmap[vi >> 5], 1u << (vi & 31));
  }
  __syncthreads();
  return TopkPrep{G, *s_nfix, any_valid, key, s_g, bitmap, P};
}

// One-hot columns of one 8-column vector of the top-k logprob map, written
// by the thread that has just stored the vector, from the raw values it
// holds: column c gets (the sum of g_j over the valid ids_j = c, ascending j)
// - G p_c with one rounding (times dz/dx with a cap), the arithmetic of the
// k = 1 map's fix-up.  gcol0: the vector's first global column.  Rare (a
// row has at most k such vectors), so it is not inlined into the sweep.
template <class T, bool CAP>
__device__ __noinline__ void onehot_vector(T* dst, const Raw8<T> x, int64_t gcol0, int nvalid,
                                           const unsigned long long* key, int P, const float* s_g, float m,
                                           float log_s, float G, float cap) {
  const unsigned long long first = static_cast<unsigned long long>(gcol0) << kTopkJBits;
  int lo = 0, hi = P;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (key[mid] < first)
      lo = mid + 1;
    else
      hi = mid;
  }
  const CapK K = cap_consts(CAP ? cap : 1.0f);
  int t = lo;
  while (t < P) {
    const unsigned long long id = key[t] >> kTopkJBits;   // the invalid keys (all ones) sort last, far beyond
    const int64_t e = static_cast<int64_t>(id) - gcol0;
    if (e >= nvalid) break;
    float gs = 0.0f;
    for (; t < P && (key[t] >> kTopkJBits) == id; ++t) gs += s_g[key[t] & ((1ull << kTopkJBits) - 1)];
    float xa, xb;
    upk(x.pair(static_cast<int>(e) >> 1), xa, xb);
    const float xe = (e & 1) ? xb : xa;
    float p, chain = 1.0f;
    if (CAP) {
      float E;
      const float r = cap_r_lim(xe, K, E);
      p = ex2(fmaf(r, K.a2, cap_b2_ls(m, log_s, K)));
      chain = 4.0f * E * r * r;
    } else {
      p = ex2(fmaf(xe - m, kLog2e, -log_s * kLog2e));
    }
    const float r = fmaf(-G, p, gs);
    Out8<T>::store1(dst + e, CAP ? r * chain : r);
  }
}

// Row constants of a backward map.
struct BwdRow {
  fp2 nm2;      // -m (of x)
  fp2 nls2;     // -log S * log2 e (of x); the softcapped logp map: (c - m - log S) log2 e
  fp2 coef2;    // logp: -G (times 4 with a cap); entropy: -g; KL: g
  fp2 k2;       // entropy: log S - H;  reverse KL: log S_a - log S_b + KL
  fp2 nmq2;     // KL: -m_b
  fp2 nlsq2;    // KL: -log S_b * log2 e
  // fused: gradient = p_a c0 + (p_a d_a) c1 + (p_a d_b) c2 + ngk p_b
  fp2 c1, c2, ngk;
};

template <int OP, int DIR>
constexpr bool bwd_reads_two() { return OP == kBwdKlReverse || OP == kBwdKlForward || (OP == kBwdFused && DIR != kFusedNoKl); }

// Gradient of pair i of a vector: x holds the logits (the policy for KL), y
// the reference (KL only).
template <class T, int OP, bool CAP, int DIR = kFusedNoKl>
__device__ __forceinline__ fp2 grad_pair(const Raw8<T>& x, const Raw8<T>& y, int i, const BwdRow& R,
                                         const CapK& K) {
  if constexpr (CAP && OP == kBwdLogp) {
    // -4 G p E r r; nls2 holds (c - m - log S) log2(e) here
    fp2 E;
    const fp2 r = cap_r_pair(x, i, K, E);
    const fp2 p = ex2_2(fma2(r, splat(K.a2), R.nls2));
    return mul2(mul2(p, R.coef2), mul2(mul2(E, r), r));
  }
  fp2 d, e2 = 0, r2 = 0;
  if (CAP) {
    d = fma2(cap_t2(x, i, K, e2, r2), splat(K.c), R.nm2);
  } else {
    d = add2(OP == kBwdLogp ? x.pair(i) : x.pair_clamped(i), R.nm2);
  }
  const fp2 p = ex2_2(fma2(d, splat(kLog2e), R.nls2));
  fp2 r;
  if constexpr (OP == kBwdLogp) {
    r = mul2(p, R.coef2);
  } else if constexpr (OP == kBwdEntropy) {
    r = mul2(mul2(p, R.coef2), sub2(d, R.k2));
  } else if constexpr (OP == kBwdFused) {
    // p c0 + (p d_a) c1 + (p d_b) c2 (+ ngk p_b); coef2 holds c0.  p is
    // multiplied in first, so masked columns (p = 0, d = -3.4e38) give 0.
    r = fma2(mul2(p, d), R.c1, mul2(p, R.coef2));
    if constexpr (DIR != kFusedNoKl) {
      fp2 db;
      if (CAP) {
        fp2 eq, rq;
        db = fma2(cap_t2(y, i, K, eq, rq), splat(K.c), R.nmq2);
      } else {
        db = add2(y.pair_clamped(i), R.nmq2);
      }
      if constexpr (DIR == kFusedKlReverse)
        r = fma2(mul2(p, db), R.c2, r);
      else
        r = fma2(ex2_2(fma2(db, splat(kLog2e), R.nlsq2)), R.ngk, r);
    }
  } else {
    fp2 dq;
    if (CAP) {
      fp2 eq, rq;
      dq = fma2(cap_t2(y, i, K, eq, rq), splat(K.c), R.nmq2);
    } else {
      dq = add2(y.pair_clamped(i), R.nmq2);
    }
    if constexpr (OP == kBwdKlReverse) {
      r = mul2(mul2(p, R.coef2), sub2(sub2(d, dq), R.k2));
    } else {
      r = mul2(sub2(p, ex2_2(fma2(dq, splat(kLog2e), R.nlsq2))), R.coef2);
    }
  }
  if (CAP) {
    // dz/dx = 4 e r^2 (the 4 is folded into coef for logp)
    r = mul2(mul2(r, e2), r2);
    r = mul2(r, OP == kBwdLogp ? r2 : mul2(r2, splat(4.0f)));
  }
  return r;
}

// Scalar form of the fused gradient at one column (the one-hot fix-up).
template <class T, bool CAP, int DIR>
__device__ __forceinline__ float fused_at(const T* xr, const T* yr, int64_t c, const vls_rowstat& sx, float mq,
                                          float log_sq, float c0, float c1, float c2, float ngk, float gsum,
                                          const CapK& K, float& chain) {
  const float x = load1(xr + c);
  float d;
  chain = 1.0f;
  if (CAP) {
    float e, r;
    d = cap_d(cap_t(x, K, e, r), K.c, sx.m);
    chain = 4.0f * e * r * r;
  } else {
    d = max_nan(x, kLowest) - sx.m;
  }
  const float p = ex2(fmaf(d, kLog2e, -sx.log_s * kLog2e));
  float r = fmaf(p * d, c1, fmaf(p, c0, gsum));
  if constexpr (DIR != kFusedNoKl) {
    const float y = load1(yr + c);
    const float db = CAP ? cap_d(cap_t(y, K), K.c, mq) : max_nan(y, kLowest) - mq;
    if constexpr (DIR == kFusedKlReverse) r = fmaf(p * db, c2, r);
    else r = fmaf(ex2(fmaf(db, kLog2e, -log_sq * kLog2e)), ngk, r);
  }
  return r;
}

// Six resident CTAs per SM (at most 40 registers a thread) keep enough
// loads in flight; with a larger register budget occupancy halves and the
// sweep slows down.  The 16-bit softcapped logprob map keeps six too: its
// software pipeline spills a little at 40 registers, and is still 6% faster
// than at 5 CTAs and 48 registers (and 8% faster than at 32); buffers of 3
// or 4 vectors at 4 or 5 CTAs were 1-9% slower at 151936 columns.  The other
// softcapped maps and the top-k map get kCapMinBlocks CTAs per SM.
// TOPK (logprob map with k > 1): the one-hot columns are written inline by
// the thread that stores their vector (onehot_vector) instead of by a
// post-pass that re-reads them after a barrier.
#ifndef VLS_CAP_LOGP_BWD_CTAS
#define VLS_CAP_LOGP_BWD_CTAS 6
#endif
// vectors per buffer of the softcapped maps' two-buffer pipeline (16-bit, one tensor)
#ifndef VLS_CAP_BWD_VECS
#define VLS_CAP_BWD_VECS 2
#endif
// The fused map with a KL term (two tensors, 16-bit) takes batches of 3
// vectors of each at 5 CTAs: 6.3% (reverse) and 2.5% (forward KL) faster
// than 2 at 6 CTAs; either change alone was slower, and without a KL term
// 5 CTAs were 3.9% slower.
template <class T, int OP, bool CAP, int DIR, bool TOPK>
constexpr int bwd_min_blocks() {
  if (TOPK) return kCapMinBlocks;
  if (!CAP) return (OP == kBwdFused && DIR != kFusedNoKl && sizeof(T) == 2) ? 5 : 6;
  return (OP == kBwdLogp && sizeof(T) == 2) ? VLS_CAP_LOGP_BWD_CTAS : kCapMinBlocks;
}

template <class T, int OP, bool CAP, int DIR = kFusedNoKl, bool TOPK = false>
__global__ void __launch_bounds__(kRowThreads, (bwd_min_blocks<T, OP, CAP, DIR, TOPK>())) row_bwd_kernel(const BwdArgs a) {
  constexpr bool KL = bwd_reads_two<OP, DIR>();
  const int64_t row = blockIdx.x / a.chunks;
  const int q = static_cast<int>(blockIdx.x - row * a.chunks);
  const int64_t V = a.vocab;
  const int64_t nvec = (V + 7) >> 3;
  const int64_t vb = static_cast<int64_t>(q) * a.vec_per_cta;
  const int64_t ve = min(vb + a.vec_per_cta, nvec);
  const T* xr = row_ptr<T>(a.x, a.rx, row);
  const T* yr = KL ? row_ptr<T>(a.y, a.ry, row) : xr;
  T* dr = static_cast<T*>(a.dx) + row * V;
  const bool al = aligned16(xr) && aligned16(dr) && aligned16(yr);
  const CapK K = cap_consts(CAP ? a.cap : 1.0f);

  const vls_rowstat sx = a.stats_x[row];
  BwdRow R;
  R.nm2 = splat(-sx.m);
  R.nls2 = splat((CAP && OP == kBwdLogp) ? cap_b2_ls(sx.m, sx.log_s, K) : -sx.log_s * kLog2e);
  R.k2 = 0;
  R.nmq2 = 0;
  R.nlsq2 = 0;
  R.c1 = 0;
  R.c2 = 0;
  R.ngk = 0;
  float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, ngk = 0.0f, mq = 0.0f, log_sq = 0.0f;

  // ---- per-row constants; rows whose gradient is a constant (zero / NaN) ----
  float G = 0.0f;
  int nfix = 0;
  bool nan_row = false, zero_row = false;
  int64_t* fix_id = nullptr;
  float* fix_g = nullptr;
  TopkPrep tp{};
  const bool has_logp = OP == kBwdLogp || (OP == kBwdFused && a.g != nullptr);
  if (OP == kBwdLogp || OP == kBwdFused) {
    // k = 1: one fixed slot; k > 1: sorted keys, upstream grads and the
    // fix-up list in dynamic shared memory
    __shared__ int64_t fix1_id;
    __shared__ float fix1_g;
    extern __shared__ __align__(16) unsigned char topk_smem[];
    __shared__ float s_warp[kRowWarps];
    __shared__ int s_nfix;
    const int64_t col_beg = vb * 8, col_end = min(ve * 8, V);
    if (!has_logp) {
      // fused backward without a logprob term
    } else if (a.k == 1) {
      fix_id = &fix1_id;
      fix_g = &fix1_g;
      const int64_t id = a.ids[row];
      if (valid_id(id, a.vocab_total, a.ignore_index)) {
        G = a.g[row];
        const int64_t local = id - a.vocab_offset;
        if (local >= col_beg && local < col_end) {
          nfix = 1;
          if (threadIdx.x == 0) {
            fix1_id = local;
            fix1_g = G;
          }
        }
      } else {
        zero_row = true;
      }
    } else {
      // the id preparation takes a few microseconds: start this thread's
      // first vectors on their way to L2 so that DRAM latency overlaps it
      if (al) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t pv = vb + threadIdx.x + u * kRowThreads;
          if (pv < (V >> 3) && pv < ve) prefetch_l2(xr + 8 * pv);
        }
      }
      tp = prep_topk(a, row, col_beg, col_end, topk_smem, fix_id, fix_g, s_warp, &s_nfix);
      G = tp.G;
      nfix = tp.nfix;
      zero_row = !tp.any_valid;
    }
    if constexpr (OP == kBwdLogp) {
      R.coef2 = splat(CAP ? -4.0f * G : -G);  // the streamed value is -G p (dz/dx)
    } else {
      // fused: p_a (c0 + c1 d_a + c2 d_b) + ngk p_b, one term per present gradient
      const bool has_h = a.g_h != nullptr, has_k = DIR != kFusedNoKl && a.g_kl != nullptr;
      if (has_logp) c0 = -G;
      if (has_h) {
        const float gh = a.g_h[row], H = a.h[row];
        c0 = fmaf(gh, sx.log_s - H, c0);  // -g_H p (d - (log S - H))
        c1 -= gh;
        nan_row |= isnan(H);
      }
      if constexpr (DIR != kFusedNoKl) {
        const vls_rowstat sy = a.stats_y[row];
        mq = sy.m;
        log_sq = sy.log_s;
        R.nmq2 = splat(-sy.m);
        R.nlsq2 = splat(-sy.log_s * kLog2e);
        if (has_k) {
          const float gk = a.g_kl[row], kl = a.kl[row];
          if constexpr (DIR == kFusedKlReverse) {
            c0 = fmaf(-gk, (sx.log_s - sy.log_s) + kl, c0);  // g_K p ((d_a - d_b) - (lS_a - lS_b + KL))
            c1 += gk;
            c2 = -gk;
            nan_row |= !isfinite(kl);
          } else {
            c0 += gk;  // g_K (p_a - p_b)
            ngk = -gk;
            nan_row |= isnan(kl);
          }
        }
      }
      nan_row |= sx.m == neg_inf() && (has_h || has_k);
      zero_row = zero_row && !has_h && !has_k;
      R.coef2 = splat(c0);
      R.c1 = splat(c1);
      R.c2 = splat(c2);
      R.ngk = splat(ngk);
    }
  } else if constexpr (OP == kBwdEntropy) {
    const float H = a.fout[row];
    R.coef2 = splat(-a.g[row]);
    R.k2 = splat(sx.log_s - H);  // log p + H = (z - m) - (log S - H)
    nan_row = sx.m == neg_inf() || isnan(H);
  } else {
    const vls_rowstat sy = a.stats_y[row];
    R.nmq2 = splat(-sy.m);
    R.nlsq2 = splat(-sy.log_s * kLog2e);
    const float kl = a.fout[row];
    R.coef2 = splat(a.g[row]);
    if constexpr (OP == kBwdKlReverse) {
      R.k2 = splat((sx.log_s - sy.log_s) + kl);  // (log p_a - log p_b) - KL = (da - db) - k
      nan_row = !isfinite(kl);
    } else {
      nan_row = isnan(kl);
    }
  }

  if (zero_row || nan_row) {
    const fp2 c = splat(nan_row ? qnan() : 0.0f);
    const fp2 o[4] = {c, c, c, c};
    for (int64_t v = vb + threadIdx.x; v < ve; v += kRowThreads) store_vec(dr, v, V, al, o);
    return;
  }

  // top-k: the one-hot columns of a stored vector, when the bitmap flags it
  const uint32_t* const bitmap = tp.bitmap;
  const unsigned long long* const tkey = tp.key;
  const float* const tg = tp.g;
  const int tP = tp.P;
  const float row_m = sx.m, row_ls = sx.log_s, row_G = G, row_cap = a.cap;
  const int64_t voff = a.vocab_offset;
  auto onehot_if_flagged = [=](int64_t vec, const Raw8<T>& xv, int nvalid) {
    const int64_t vi = vec - vb;
    if ((bitmap[vi >> 5] >> (vi & 31)) & 1u)
      onehot_vector<T, CAP>(dr + 8 * vec, xv, 8 * vec + voff, nvalid, tkey, tP, tg, row_m, row_ls, row_G, row_cap);
  };

  int64_t v = vb + threadIdx.x;
  const int64_t vfull_end = min(ve, V >> 3);
  if constexpr (CAP) {
    // Heavy per-element arithmetic (two exponentials and a reciprocal):
    // software-pipelined, the next batch's loads issued before the current
    // batch is computed, alternating between two register buffers.
    constexpr int U = (KL || sizeof(T) == 4) ? 1 : VLS_CAP_BWD_VECS;
    constexpr int64_t kStep = U * kRowThreads;
    if (al && v + (U - 1) * kRowThreads < vfull_end) {
      Raw8<T> xa[U], ya[U], xb[U], yb[U];
      auto load = [&](Raw8<T>(&x)[U], Raw8<T>(&y)[U], int64_t at) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          x[u].load(xr + 8 * (at + u * kRowThreads));
          if constexpr (KL) y[u].load(yr + 8 * (at + u * kRowThreads));
        }
      };
      auto work = [&](const Raw8<T>(&x)[U], const Raw8<T>(&y)[U], int64_t at) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          fp2 o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = grad_pair<T, OP, CAP, DIR>(x[u], KL ? y[u] : x[u], i, R, K);
          Out8<T>::store(dr + 8 * (at + u * kRowThreads), o);
          if constexpr (TOPK) onehot_if_flagged(at + u * kRowThreads, x[u], 8);
        }
      };
      load(xa, ya, v);
      for (;;) {
        bool more = v + kStep + (U - 1) * kRowThreads < vfull_end;
        if (more) load(xb, yb, v + kStep);
        work(xa, ya, v);
        v += kStep;
        if (!more) break;
        more = v + kStep + (U - 1) * kRowThreads < vfull_end;
        if (more) load(xa, ya, v + kStep);
        work(xb, yb, v);
        v += kStep;
        if (!more) break;
      }
    }
  } else {
    // light arithmetic: plain batches of U vectors in flight per thread; the
    // 16-bit KL maps take 3 of each tensor (1-3% faster than 2 at the same 40
    // registers), and so does the 16-bit fused map with a KL term (at 5 CTAs,
    // see bwd_min_blocks); fp32 two-tensor maps 2
    constexpr int U = KL ? (sizeof(T) == 2 ? 3 : 2) : 4;
    if (al) {
      for (; v + (U - 1) * kRowThreads < vfull_end; v += U * kRowThreads) {
        Raw8<T> x[U], y[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          x[u].load(xr + 8 * (v + u * kRowThreads));
          if constexpr (KL) y[u].load(yr + 8 * (v + u * kRowThreads));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          fp2 o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) o[i] = grad_pair<T, OP, CAP, DIR>(x[u], KL ? y[u] : x[u], i, R, K);
          Out8<T>::store(dr + 8 * (v + u * kRowThreads), o);
          if constexpr (TOPK) onehot_if_flagged(v + u * kRowThreads, x[u], 8);
        }
      }
    }
  }
  for (; v < ve; v += kRowThreads) {
    Raw8<T> x, y;
    int valid;
    load_raw(x, xr, v, V, al, valid);
    if constexpr (KL) load_raw(y, yr, v, V, al, valid);
    fp2 o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = grad_pair<T, OP, CAP, DIR>(x, KL ? y : x, i, R, K);
    store_vec(dr, v, V, al, o);
    if constexpr (TOPK) onehot_if_flagged(v, x, valid);
  }

  if constexpr (OP == kBwdFused) {
    // one-hot columns: rewrite with g_sum + (the streamed value), one rounding
    if (nfix > 0) {
      __syncthreads();  // the streamed stores of this CTA precede the rewrites
      for (int f = threadIdx.x; f < nfix; f += kRowThreads) {
        float chain;
        const float r = fused_at<T, CAP, DIR>(xr, yr, fix_id[f], sx, mq, log_sq, c0, c1, c2, ngk, fix_g[f], K, chain);
        Out8<T>::store1(dr + fix_id[f], CAP ? r * chain : r);
      }
    }
  }
  if constexpr (OP == kBwdLogp && !TOPK) {
    // one-hot columns: rewrite with (g_sum - G p) dz/dx, one rounding at the store
    if (nfix > 0) {
      __syncthreads();  // the streamed stores of this CTA precede the rewrites
      for (int f = threadIdx.x; f < nfix; f += kRowThreads) {
        const int64_t c = fix_id[f];
        const float x = load1(xr + c);
        float p, chain = 1.0f;
        if (CAP) {
          float E;
          const float r = cap_r_lim(x, K, E);
          p = ex2(fmaf(r, K.a2, cap_b2_ls(sx.m, sx.log_s, K)));
          chain = 4.0f * E * r * r;
        } else {
          p = ex2(fmaf(x - sx.m, kLog2e, -sx.log_s * kLog2e));
        }
        const float r = fmaf(-G, p, fix_g[f]);
        Out8<T>::store1(dr + c, CAP ? r * chain : r);
      }
    }
  }
}

template <class T, int OP, bool CAP, int DIR = kFusedNoKl>
cudaError_t launch_bwd_t(const BwdArgs& a, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.rows * a.chunks));
  const bool topk = (OP == kBwdLogp || (OP == kBwdFused && a.g != nullptr)) && a.k > 1;
  const size_t smem = topk ? topk_smem_bytes(a.k, a.vec_per_cta) : 0;
  if (OP == kBwdLogp && topk)
    row_bwd_kernel<T, OP, CAP, DIR, true><<<grid, kRowThreads, smem, s>>>(a);
  else
    row_bwd_kernel<T, OP, CAP, DIR, false><<<grid, kRowThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <class T, int OP, int DIR = kFusedNoKl>
cudaError_t launch_bwd_cap(bool cap, const BwdArgs& a, cudaStream_t s) {
  return cap ? launch_bwd_t<T, OP, true, DIR>(a, s) : launch_bwd_t<T, OP, false, DIR>(a, s);
}

template <int OP, int DIR = kFusedNoKl>
cudaError_t launch_bwd_op(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16) return launch_bwd_cap<__nv_bfloat16, OP, DIR>(cap, a, s);
  if (dt == VLS_F16) return launch_bwd_cap<__half, OP, DIR>(cap, a, s);
  return launch_bwd_cap<float, OP, DIR>(cap, a, s);
}

}  // namespace vls
