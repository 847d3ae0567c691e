// One-read forward sweep: per-row max / sum-exp (and the entropy or KL
// weighted sum) in a single pass over the logits, then the row's outputs.
//
// Launch shape: a cluster of `cluster` CTAs per row (cluster size a function
// of V only), each CTA owning a contiguous run of 8-column vectors.  Inside a
// CTA of T = kFwdThreads threads, thread t owns vectors t, t + T, t + 2T, ...
// of that run and folds them in increasing order into its online state; the
// states are then combined by a fixed tree: lanes (xor 16..1), warps (xor
// T/64..1 over the T/32 warps), cluster ranks (xor 4..1 over up to 8 ranks,
// through distributed shared memory into rank 0).  Nothing in that order
// depends on N, on the row's position or on its alignment, so results are
// deterministic and batch invariant (one block per row and a fixed reduction tree, "perf(logp): fused
// zero-workspace backward ...", RL-Kernel PR #495, Summary; a tree fixed
// regardless of the row count, "TP4 GDN, convolution and D=256 attention
// mixers", RL-Kernel PR #507).
#pragma once

#include <type_traits>

#include "vls_device.cuh"

namespace vls {

using namespace dev;

// With a softcap the row max is the cap of the raw max (tanh is
// increasing), so maxima are tracked on raw logits and only the new maximum
// is transformed.  `fresh` forces the first transform with a cap, where a
// vector of -inf still has a finite value (-c).
template <bool CAP>
__device__ __forceinline__ bool grows(float vmax_raw, float m_raw, float m) {
  return vmax_raw > m_raw || (CAP && m == neg_inf());
}

template <bool PARTIAL>
__device__ __forceinline__ fp2 keep(fp2 e, int i, int valid) {
  if (!PARTIAL) return e;
  float a, b;
  upk(e, a, b);
  return pk(2 * i < valid ? a : 0.0f, 2 * i + 1 < valid ? b : 0.0f);
}

template <class T, bool CAP>
struct LogpAcc {
  using State = LogpState;
  float m_raw = neg_inf(), m = neg_inf();
  // nm2: -m, or with a cap b2 = (c - m) log2(e) (cap_d2_pair)
  fp2 nm2 = 0, s2 = 0;

  // wa: with a cap, the warp's raw max over this vector's group (warp_max)
  template <bool PARTIAL, bool CLAMP = true>
  __device__ __forceinline__ void update(const Raw8<T>& v, const Raw8<T>&, int valid, const CapK& K, float wa = 0.0f,
                                         float = 0.0f) {
    if constexpr (CAP) {
      if (grows<CAP>(wa, m_raw, m)) {   // the same decision in every lane of the warp
        const float mn = cap_zr_rare(wa, K);
        s2 = mul2(s2, splat(rescale_rare(m, mn)));
        m_raw = wa;
        m = mn;
        nm2 = splat(cap_b2(mn, K));
      }
    } else {
      const float vm = v.max();
      if (grows<CAP>(vm, m_raw, m)) {
        s2 = mul2(s2, splat(rescale(m, vm)));
        m_raw = vm;
        m = vm;
        nm2 = splat(-vm);
      }
      if (m == neg_inf()) return;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const fp2 d2 = CAP ? cap_d2_pair<T, CLAMP>(v, i, K, nm2) : mul2(add2(v.pair(i), nm2), splat(kLog2e));
      s2 = add2(s2, keep<PARTIAL>(ex2_2(d2), i, valid));
    }
  }
  __device__ State state() const { return {m, sum2(s2)}; }
};

// With a cap, W is accumulated in log2 units (the weights' exponents come out
// of cap_d2_pair that way) and turned into natural units once, in state().
template <class T, bool CAP>
struct EntropyAcc {
  using State = EntropyState;
  float m_raw = neg_inf(), m = neg_inf();
  fp2 nm2 = 0, s2 = 0, w2 = 0;

  template <bool PARTIAL, bool CLAMP = true>
  __device__ __forceinline__ void update(const Raw8<T>& v, const Raw8<T>&, int valid, const CapK& K, float wa = 0.0f,
                                         float = 0.0f) {
    const float vm = CAP ? wa : v.max();   // with a cap, the warp's max: the same decision in every lane
    if (grows<CAP>(vm, m_raw, m)) {
      const float mn = CAP ? cap_zr_rare(vm, K) : vm;
      const float f = CAP ? rescale_rare(m, mn) : rescale(m, mn);
      const float shift = CAP ? (m - mn) * kLog2e : m - mn;
      w2 = m != neg_inf() ? mul2(fma2(s2, splat(shift), w2), splat(f)) : 0;
      s2 = mul2(s2, splat(f));
      m_raw = vm;
      m = mn;
      nm2 = splat(CAP ? cap_b2(mn, K) : -mn);
    }
    if (!CAP && m == neg_inf()) return;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      fp2 d, e;
      if (CAP) {
        d = cap_d2_pair<T, CLAMP>(v, i, K, nm2);
        e = keep<PARTIAL>(ex2_2(d), i, valid);
      } else {
        d = add2(v.pair_clamped(i), nm2);  // -inf columns: e = 0 and 0 * d = 0
        e = keep<PARTIAL>(ex2_2(mul2(d, splat(kLog2e))), i, valid);
      }
      s2 = add2(s2, e);
      w2 = fma2(e, d, w2);
    }
  }
  __device__ State state() const { return {m, sum2(s2), CAP ? sum2(w2) * kLn2 : sum2(w2)}; }
};

// KL(P||Q): `v` is a vector of P (first argument), `q` the same columns of Q.
// With a cap, W is accumulated in log2 units as in EntropyAcc.
template <class T, bool CAP>
struct KlAcc {
  using State = KlState;
  float mp_raw = neg_inf(), mp = neg_inf(), mq_raw = neg_inf(), mq = neg_inf();
  fp2 nmp2 = 0, nmq2 = 0, sp2 = 0, sq2 = 0, w2 = 0;
  uint32_t flag = 0;

  // wp, wq: with a cap, the warp's raw maxima over this vector's group of P and of Q
  template <bool PARTIAL, bool CLAMP = true>
  __device__ __forceinline__ void update(const Raw8<T>& v, const Raw8<T>& q, int valid, const CapK& K,
                                         float wp = 0.0f, float wq = 0.0f) {
    // with a cap, the warp's maxima: the same decisions in every lane
    const float vmp = CAP ? wp : v.max(), vmq = CAP ? wq : q.max();
    const bool up = grows<CAP>(vmp, mp_raw, mp), uq = grows<CAP>(vmq, mq_raw, mq);
    if (up || uq) {
      const float Mp = up ? (CAP ? cap_zr_rare(vmp, K) : vmp) : mp;
      const float Mq = uq ? (CAP ? cap_zr_rare(vmq, K) : vmq) : mq;
      const float fp = CAP ? rescale_rare(mp, Mp) : rescale(mp, Mp), fq = CAP ? rescale_rare(mq, Mq) : rescale(mq, Mq);
      const float shift = CAP ? ((mp - Mp) - (mq - Mq)) * kLog2e : (mp - Mp) - (mq - Mq);
      w2 = mp != neg_inf() ? mul2(fma2(sp2, splat(shift), w2), splat(fp)) : 0;
      sp2 = mul2(sp2, splat(fp));
      sq2 = mul2(sq2, splat(fq));
      if (up) { mp_raw = vmp; mp = Mp; nmp2 = splat(CAP ? cap_b2(Mp, K) : -Mp); }
      if (uq) { mq_raw = vmq; mq = Mq; nmq2 = splat(CAP ? cap_b2(Mq, K) : -Mq); }
    }
    if (!CAP) {
#pragma unroll
      for (int i = 0; i < 4; ++i) flag |= v.mismatch(i, q);
    }
    const bool p_ok = CAP || mp != neg_inf(), q_ok = CAP || mq != neg_inf();
    if (p_ok && q_ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        fp2 dp, dq, ep, eq;
        if (CAP) {
          dp = cap_d2_pair<T, CLAMP>(v, i, K, nmp2);
          dq = cap_d2_pair<T, CLAMP>(q, i, K, nmq2);
          ep = keep<PARTIAL>(ex2_2(dp), i, valid);
          eq = keep<PARTIAL>(ex2_2(dq), i, valid);
        } else {
          dp = add2(v.pair_clamped(i), nmp2);
          dq = add2(q.pair_clamped(i), nmq2);
          ep = keep<PARTIAL>(ex2_2(mul2(dp, splat(kLog2e))), i, valid);
          eq = keep<PARTIAL>(ex2_2(mul2(dq, splat(kLog2e))), i, valid);
        }
        sp2 = add2(sp2, ep);
        sq2 = add2(sq2, eq);
        w2 = fma2(ep, sub2(dp, dq), w2);
      }
    } else if (p_ok || q_ok) {
      // one side has seen only -inf so far (no W term: a finite P column
      // against an all -inf Q run is a mismatch, already flagged); never
      // with a cap, where no logit stays -inf
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (p_ok) sp2 = add2(sp2, keep<PARTIAL>(ex2_2(mul2(add2(v.pair_clamped(i), nmp2), splat(kLog2e))), i, valid));
        if (q_ok) sq2 = add2(sq2, keep<PARTIAL>(ex2_2(mul2(add2(q.pair_clamped(i), nmq2), splat(kLog2e))), i, valid));
      }
    }
  }
  __device__ State state() const { return {mp, sum2(sp2), mq, sum2(sq2), CAP ? sum2(w2) * kLn2 : sum2(w2), flag}; }
};

// Fused sweep over the policy a (`v`) and, with a KL term, the reference b
// (`q`): a's statistics and entropy W as EntropyAcc, b's as LogpAcc, and the
// KL W of direction DIR as KlAcc with P = a (reverse) or P = b (forward).
template <class T, bool CAP, int DIR>
struct FusedAcc {
  using State = FusedState<DIR>;
  static constexpr bool kHasB = DIR != kFusedNoKl;
  float ma_raw = neg_inf(), ma = neg_inf(), mb_raw = neg_inf(), mb = neg_inf();
  fp2 nma2 = 0, nmb2 = 0, sa2 = 0, wh2 = 0, sb2 = 0, wk2 = 0;
  uint32_t flag = 0;

  // wa, wb: with a cap, the warp's raw maxima over this vector's group of a and of b
  template <bool PARTIAL, bool CLAMP = true>
  __device__ __forceinline__ void update(const Raw8<T>& v, const Raw8<T>& q, int valid, const CapK& K,
                                         float wa = 0.0f, float wb = 0.0f) {
    const float vma = CAP ? wa : v.max();   // with a cap, the warp's max: the same decisions in every lane
    const bool ua = grows<CAP>(vma, ma_raw, ma);
    float vmb = neg_inf();
    bool ub = false;
    if constexpr (kHasB) {
      vmb = CAP ? wb : q.max();
      ub = grows<CAP>(vmb, mb_raw, mb);
    }
    if (ua || ub) {
      const float Ma = ua ? (CAP ? cap_zr_rare(vma, K) : vma) : ma;
      const float Mb = ub ? (CAP ? cap_zr_rare(vmb, K) : vmb) : mb;
      const float fa = CAP ? rescale_rare(ma, Ma) : rescale(ma, Ma), fb = CAP ? rescale_rare(mb, Mb) : rescale(mb, Mb);
      const float u = CAP ? kLog2e : 1.0f;   // units of W: log2 with a cap
      wh2 = ma != neg_inf() ? mul2(fma2(sa2, splat(CAP ? (ma - Ma) * kLog2e : ma - Ma), wh2), splat(fa)) : 0;
      if constexpr (DIR == kFusedKlReverse)
        wk2 = ma != neg_inf() ? mul2(fma2(sa2, splat(((ma - Ma) - (mb - Mb)) * u), wk2), splat(fa)) : 0;
      if constexpr (DIR == kFusedKlForward)
        wk2 = mb != neg_inf() ? mul2(fma2(sb2, splat(((mb - Mb) - (ma - Ma)) * u), wk2), splat(fb)) : 0;
      sa2 = mul2(sa2, splat(fa));
      sb2 = mul2(sb2, splat(fb));
      if (ua) { ma_raw = vma; ma = Ma; nma2 = splat(CAP ? cap_b2(Ma, K) : -Ma); }
      if (ub) { mb_raw = vmb; mb = Mb; nmb2 = splat(CAP ? cap_b2(Mb, K) : -Mb); }
    }
    if constexpr (kHasB && !CAP) {
#pragma unroll
      for (int i = 0; i < 4; ++i) flag |= DIR == kFusedKlReverse ? v.mismatch(i, q) : q.mismatch(i, v);
    }
    const bool a_ok = CAP || ma != neg_inf(), b_ok = CAP || mb != neg_inf();
    if (a_ok && (!kHasB || b_ok)) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        fp2 da, db = 0, ea, eb = 0;
        if (CAP) {
          da = cap_d2_pair<T, CLAMP>(v, i, K, nma2);
          ea = keep<PARTIAL>(ex2_2(da), i, valid);
          if constexpr (kHasB) {
            db = cap_d2_pair<T, CLAMP>(q, i, K, nmb2);
            eb = keep<PARTIAL>(ex2_2(db), i, valid);
          }
        } else {
          da = add2(v.pair_clamped(i), nma2);
          ea = keep<PARTIAL>(ex2_2(mul2(da, splat(kLog2e))), i, valid);
          if constexpr (kHasB) {
            db = add2(q.pair_clamped(i), nmb2);
            eb = keep<PARTIAL>(ex2_2(mul2(db, splat(kLog2e))), i, valid);
          }
        }
        sa2 = add2(sa2, ea);
        wh2 = fma2(ea, da, wh2);
        if constexpr (kHasB) {
          sb2 = add2(sb2, eb);
          if constexpr (DIR == kFusedKlReverse) wk2 = fma2(ea, sub2(da, db), wk2);
          else wk2 = fma2(eb, sub2(db, da), wk2);
        }
      }
    } else if (a_ok || b_ok) {
      // one side has seen only -inf so far: no cross term (a finite column
      // of the KL's first argument against an all -inf run is flagged);
      // never with a cap
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (a_ok) {
          const fp2 da = add2(v.pair_clamped(i), nma2);
          const fp2 ea = keep<PARTIAL>(ex2_2(mul2(da, splat(kLog2e))), i, valid);
          sa2 = add2(sa2, ea);
          wh2 = fma2(ea, da, wh2);
        }
        if (b_ok) sb2 = add2(sb2, keep<PARTIAL>(ex2_2(mul2(add2(q.pair_clamped(i), nmb2), splat(kLog2e))), i, valid));
      }
    }
  }
  __device__ State state() const {
    const float u = CAP ? kLn2 : 1.0f;
    return {ma, sum2(sa2), sum2(wh2) * u, mb, sum2(sb2), sum2(wk2) * u, flag};
  }
};

template <int OP, class T, bool CAP, int DIR>
struct FwdAccOf;
template <class T, bool CAP, int DIR>
struct FwdAccOf<kFwdLogp, T, CAP, DIR> { using type = LogpAcc<T, CAP>; };
template <class T, bool CAP, int DIR>
struct FwdAccOf<kFwdEntropy, T, CAP, DIR> { using type = EntropyAcc<T, CAP>; };
template <class T, bool CAP, int DIR>
struct FwdAccOf<kFwdKl, T, CAP, DIR> { using type = KlAcc<T, CAP>; };
template <class T, bool CAP, int DIR>
struct FwdAccOf<kFwdFused, T, CAP, DIR> { using type = FusedAcc<T, CAP, DIR>; };

// the sweep reads a second tensor
template <int OP, int DIR>
constexpr bool reads_two() { return OP == kFwdKl || (OP == kFwdFused && DIR != kFusedNoKl); }

// 16-byte loads in flight per thread before any is used: 4 vectors of one
// tensor; 3 vectors of each of the two 16-bit KL tensors (2.5-3.8% faster
// than 2 at the same 48 registers and 5 CTAs; 4, or 6 CTAs, spill), 2 of
// each in the other two-tensor sweeps.  The softcapped logp sweep, bound by
// its arithmetic rather than by memory, takes 4 at 6 resident CTAs (with the
// reciprocal of pairs 0, 2 and 3 on the FMA pipe: 1.0% faster than 6 vectors
// at 5 CTAs at 151936 columns, 2.8% at 262144; 8 at 4 CTAs was slower).
#ifndef VLS_CAP_LOGP_UNROLL
#define VLS_CAP_LOGP_UNROLL 4
#endif
#ifndef VLS_CAP_LOGP_CTAS
#define VLS_CAP_LOGP_CTAS 6
#endif
template <class T, int OP, int DIR, bool CAP>
constexpr int fwd_unroll() {
  if (reads_two<OP, DIR>()) return (OP == kFwdKl && !CAP && sizeof(T) == 2) ? 3 : 2;
  return (CAP && OP == kFwdLogp) ? VLS_CAP_LOGP_UNROLL : 4;
}

// Vectors per lane over which the softcapped sweeps take one warp max.
#ifndef VLS_CAP_MAX_GROUP
#define VLS_CAP_MAX_GROUP 2
#endif
constexpr int kCapMaxGroup = VLS_CAP_MAX_GROUP;

// Resident CTAs per SM the forward sweep is compiled for, at 256 threads.
// Without an explicit minimum, ptxas sized these kernels by heuristics that
// moved with the size of the argument struct (the bf16 entropy sweep went
// from 32 to 38 registers, the KL sweep from 44 to 56), costing 5-8% of
// bandwidth.  The bounds below keep the bf16 sweeps at 32 registers (one
// tensor), 40 (fp16 one-tensor, fused without a KL term, softcapped logp),
// 48 (softcapped entropy and fused, KL, and fused with a KL term: 4.7% and
// 2.5% faster there than at 64 registers and 4 CTAs for reverse and forward
// KL); fp16 two-tensor sweeps and fp32 vectors, which hold twice the
// registers, get 64.
template <class T, int OP, bool CAP, int DIR>
constexpr int fwd_ctas_at_256() {
  if (sizeof(T) == 4) return 4;
  if (reads_two<OP, DIR>())
    return (CAP || !std::is_same<T, __nv_bfloat16>::value) ? 4 : 5;
  if (CAP) return OP == kFwdLogp ? VLS_CAP_LOGP_CTAS : 5;
  return (OP == kFwdFused || std::is_same<T, __half>::value) ? 6 : 8;
}
template <class T, int OP, bool CAP, int DIR>
constexpr int fwd_min_blocks() {
  constexpr int b = fwd_ctas_at_256<T, OP, CAP, DIR>() * 256 / kFwdThreads;
  return b > 0 ? b : 1;
}

// ---- finalisation, shared with the vocabulary-parallel combine ----

// log p of a target from its raw logit x and the row's (m, log S); NaN for
// a row without a distribution.
// With a cap, z - m takes the sweeps' own form (cap_d2 times ln 2), so that
// the target's offset and the weights summed into S share their rounding.
template <bool CAP>
__device__ __forceinline__ float logp_of(float x, float m, float log_s, const CapK& K) {
  const float d = CAP ? cap_d2(x, K, cap_b2(m, K)) * kLn2 : x - m;
  return m == neg_inf() ? qnan() : d - log_s;
}
// H = log S - W/S
__device__ __forceinline__ float entropy_of(const EntropyState& f, float log_s) {
  return f.m == neg_inf() ? qnan() : log_s - f.w / f.s;
}
// KL = W/S_p - log S_p + log S_q; +inf on a support mismatch; NaN when a row
// of either tensor has no distribution
__device__ __forceinline__ float kl_of(const KlState& f, float log_sp, float log_sq) {
  if (f.mp == neg_inf() || f.mq == neg_inf()) return qnan();
  if (f.flag) return pos_inf();
  return f.w / f.sp + (log_sq - log_sp);
}

__device__ __forceinline__ vls_partial to_partial(const LogpState& s) { return {s.m, s.s, 0.0f, 0.0f, 0.0f, 0u}; }
__device__ __forceinline__ vls_partial to_partial(const EntropyState& s) { return {s.m, s.s, s.w, 0.0f, 0.0f, 0u}; }
__device__ __forceinline__ vls_partial to_partial(const KlState& s) { return {s.mp, s.sp, s.w, s.mq, s.sq, s.flag}; }
__device__ __forceinline__ void from_partial(const vls_partial& p, LogpState& s) { s = {p.m, p.s}; }
__device__ __forceinline__ void from_partial(const vls_partial& p, EntropyState& s) { s = {p.m, p.s, p.w}; }
__device__ __forceinline__ void from_partial(const vls_partial& p, KlState& s) {
  s = {p.m, p.s, p.mq, p.sq, p.w, p.flag};
}

template <class T, int OP, bool CAP, int DIR = kFusedNoKl>
__global__ void __launch_bounds__(kFwdThreads, (fwd_min_blocks<T, OP, CAP, DIR>())) row_fwd_kernel(const FwdArgs a) {
  using Acc = typename FwdAccOf<OP, T, CAP, DIR>::type;
  using S = typename Acc::State;
  constexpr int U = fwd_unroll<T, OP, DIR, CAP>();
  constexpr bool KL = reads_two<OP, DIR>();
  __shared__ S warp_part[kFwdWarps];
  __shared__ S cta_part[kMaxCluster];
  __shared__ S row_state;

  const int C = a.cluster;
  const int64_t row = blockIdx.x / C;
  const int q = static_cast<int>(blockIdx.x - row * C);
  if (C > 1) cluster_arrive_relaxed();

  const T* xr = row_ptr<T>(a.x, a.rx, row);
  const T* yr = KL ? row_ptr<T>(a.y, a.ry, row) : xr;
  const int64_t V = a.vocab;
  const int64_t nvec = (V + 7) >> 3;
  const int64_t vb = static_cast<int64_t>(q) * a.vec_per_cta;
  const int64_t ve = min(vb + a.vec_per_cta, nvec);
  const int64_t vfull_end = min(ve, V >> 3);
  const bool al = aligned16(xr) && aligned16(yr);
  const CapK K = cap_consts(CAP ? a.cap : 1.0f);
  if constexpr (!CAP) {
    // (the softcapped sweeps, bound by their arithmetic, are compiled without
    // it: it cost them 0.8% through register allocation)
    if (a.prefetch && al) {
      prefetch_l2_range(xr + 8 * vb, (vfull_end - vb) * 8 * static_cast<int64_t>(sizeof(T)));
      if constexpr (KL) prefetch_l2_range(yr + 8 * vb, (vfull_end - vb) * 8 * static_cast<int64_t>(sizeof(T)));
    }
  }

  // The row's first kFwdThreads target logits are loaded now by the CTA that
  // finalises the row (rank 0), so their latency overlaps the sweep instead
  // of following it (top-k rows gather up to k scattered columns).
  float xt0 = 0.0f;
  if constexpr (OP == kFwdLogp) {
    if (q == 0 && static_cast<int>(threadIdx.x) < a.k) {
      const int64_t id = a.ids[row * a.k + threadIdx.x];
      const int64_t local = id - a.vocab_offset;
      if (valid_id(id, a.vocab_total, a.ignore_index) && local >= 0 && local < V) xt0 = load1(xr + local);
    }
  }

  Acc acc;
  int64_t v = vb + threadIdx.x;
  if constexpr (!CAP) {
    if (al) {
      for (; v + (U - 1) * kFwdThreads < vfull_end; v += U * kFwdThreads) {
        Raw8<T> rx[U], ry[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          rx[u].load(xr + 8 * (v + u * kFwdThreads));
          if constexpr (KL) ry[u].load(yr + 8 * (v + u * kFwdThreads));
        }
#pragma unroll
        for (int u = 0; u < U; ++u) acc.template update<false>(rx[u], KL ? ry[u] : rx[u], 8, K);
      }
    }
    // remaining vectors, the partial last vector and unaligned rows: same
    // vectors, same order, same arithmetic
    for (; v < ve; v += kFwdThreads) {
      Raw8<T> rx, ry;
      int valid;
      load_raw(rx, xr, v, V, al, valid);
      if constexpr (KL) load_raw(ry, yr, v, V, al, valid);
      if (valid == 8)
        acc.template update<false>(rx, KL ? ry : rx, 8, K);
      else
        acc.template update<true>(rx, KL ? ry : rx, valid, K);
    }
  } else {
    // With a cap every lane of a warp runs the same iterations: the running
    // max is taken over the warp (warp_max), once per group of
    // kCapMaxGroup vectors of each lane (v, v + T, ...).  A lane past the end
    // of its run sees vectors of -inf with no valid column, which leave its
    // sums unchanged.  Batches (U a multiple of the group) and the tail
    // loop form the same groups, so aligned and unaligned rows get the same
    // bits.
    constexpr int G = kCapMaxGroup;
    static_assert(U % G == 0, "batches hold whole groups");
    const int lane = threadIdx.x & 31;
    if (al) {
      // whole batches for every lane of the warp (its last lane decides)
      for (; v - lane + 31 + (U - 1) * kFwdThreads < vfull_end; v += U * kFwdThreads) {
        Raw8<T> rx[U], ry[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          rx[u].load(xr + 8 * (v + u * kFwdThreads));
          if constexpr (KL) ry[u].load(yr + 8 * (v + u * kFwdThreads));
        }
#pragma unroll
        for (int g = 0; g < U; g += G) {
          const float wa = warp_max(group_max<T, G>(rx + g));
          const float wb = KL ? warp_max(group_max<T, G>(ry + g)) : 0.0f;
          if ((KL ? fmaxf(wa, wb) : wa) > K.xmax) {   // the same in every lane: rare
#pragma unroll
            for (int u = 0; u < G; ++u)
              acc.template update<false, true>(rx[g + u], KL ? ry[g + u] : rx[g + u], 8, K, wa, wb);
          } else {
#pragma unroll
            for (int u = 0; u < G; ++u)
              acc.template update<false, false>(rx[g + u], KL ? ry[g + u] : rx[g + u], 8, K, wa, wb);
          }
        }
      }
    }
    for (; v - lane < ve; v += G * kFwdThreads) {
      Raw8<T> rx[G], ry[G];
      int valid[G];
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const int64_t vu = v + u * kFwdThreads;
        valid[u] = 0;
        if (vu < ve) {
          load_raw(rx[u], xr, vu, V, al, valid[u]);
          if constexpr (KL) load_raw(ry[u], yr, vu, V, al, valid[u]);
        } else {   // no vector here: -inf, which adds nothing
          rx[u].load_scalar(xr, 0);
          if constexpr (KL) ry[u].load_scalar(yr, 0);
        }
      }
      const float wa = warp_max(group_max<T, G>(rx));
      const float wb = KL ? warp_max(group_max<T, G>(ry)) : 0.0f;
#pragma unroll
      for (int u = 0; u < G; ++u) {
        if (valid[u] == 8)
          acc.template update<false, true>(rx[u], KL ? ry[u] : rx[u], 8, K, wa, wb);
        else
          acc.template update<true, true>(rx[u], KL ? ry[u] : rx[u], valid[u], K, wa, wb);
      }
    }
  }

  // ---- fixed-tree reduction: lanes, warps, cluster ranks ----
  S st = warp_reduce(acc.state());
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_part[warp] = st;
  __syncthreads();
  S blk = S::identity();
  if (warp == 0) {
    blk = reduce_lanes<kFwdWarps>(lane < kFwdWarps ? warp_part[lane] : S::identity());
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
      const S r = reduce_lanes<kMaxCluster>(lane < C ? cta_part[lane] : S::identity());
      if (lane == 0) row_state = r;
    }
  }
  __syncthreads();

  // ---- finalise (rank 0 of the row) ----
  const S fin = row_state;
  if (OP != kFwdFused && a.part != nullptr) {
    // vocabulary-parallel partial: the state itself, and for logp the raw
    // logits of the target ids this shard owns (0 for the others)
    if constexpr (OP != kFwdFused) {
      if (threadIdx.x == 0) a.part[row] = to_partial(fin);
    }
    if constexpr (OP == kFwdLogp) {
      for (int j = threadIdx.x; j < a.k; j += kFwdThreads) {
        const int64_t id = a.ids[row * a.k + j];
        const int64_t local = id - a.vocab_offset;
        const bool own = valid_id(id, a.vocab_total, a.ignore_index) && local >= 0 && local < V;
        a.zt[row * a.k + j] = own ? (j < kFwdThreads ? xt0 : load1(xr + local)) : 0.0f;
      }
    }
    return;
  }
  if constexpr (OP == kFwdLogp) {
    const float m = fin.m;
    const float log_s = logf(fin.s);
    if (threadIdx.x == 0) a.stats_x[row] = vls_rowstat{m, log_s};
    for (int j = threadIdx.x; j < a.k; j += kFwdThreads) {
      const int64_t id = a.ids[row * a.k + j];
      a.logp[row * a.k + j] =
          valid_id(id, V, a.ignore_index) ? logp_of<CAP>(j < kFwdThreads ? xt0 : load1(xr + id), m, log_s, K) : 0.0f;
    }
  } else if constexpr (OP == kFwdEntropy) {
    if (threadIdx.x == 0) {
      const float log_s = logf(fin.s);
      a.stats_x[row] = vls_rowstat{fin.m, log_s};
      a.out[row] = entropy_of(fin, log_s);
    }
  } else if constexpr (OP == kFwdKl) {
    if (threadIdx.x == 0) {
      const float log_sp = logf(fin.sp), log_sq = logf(fin.sq);
      a.stats_x[row] = vls_rowstat{fin.mp, log_sp};
      a.stats_y[row] = vls_rowstat{fin.mq, log_sq};
      a.out[row] = kl_of(fin, log_sp, log_sq);
    }
  } else {
    // fused: stats_x / stats_y are a's and b's, whatever the direction
    const float log_sa = logf(fin.sa);
    if (a.logp != nullptr) {
      for (int j = threadIdx.x; j < a.k; j += kFwdThreads) {
        const int64_t id = a.ids[row * a.k + j];
        a.logp[row * a.k + j] = valid_id(id, V, a.ignore_index) ? logp_of<CAP>(load1(xr + id), fin.ma, log_sa, K) : 0.0f;
      }
    }
    if (threadIdx.x == 0) {
      a.stats_x[row] = vls_rowstat{fin.ma, log_sa};
      if (a.h != nullptr) a.h[row] = entropy_of(EntropyState{fin.ma, fin.sa, fin.wh}, log_sa);
      if constexpr (DIR != kFusedNoKl) {
        const float log_sb = logf(fin.sb);
        a.stats_y[row] = vls_rowstat{fin.mb, log_sb};
        if (a.kl != nullptr) {
          a.kl[row] = DIR == kFusedKlReverse
                          ? kl_of(KlState{fin.ma, fin.sa, fin.mb, fin.sb, fin.wk, fin.flag}, log_sa, log_sb)
                          : kl_of(KlState{fin.mb, fin.sb, fin.ma, fin.sa, fin.wk, fin.flag}, log_sb, log_sa);
        }
      }
    }
  }
}

template <class T, int OP, bool CAP, int DIR = kFusedNoKl>
cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.rows * a.cluster));
  cfg.blockDim = dim3(kFwdThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, row_fwd_kernel<T, OP, CAP, DIR>, a);
}

template <class T, int OP, int DIR = kFusedNoKl>
cudaError_t launch_fwd_cap(bool cap, const FwdArgs& a, cudaStream_t s) {
  return cap ? launch_fwd_t<T, OP, true, DIR>(a, s) : launch_fwd_t<T, OP, false, DIR>(a, s);
}

template <int OP, int DIR = kFusedNoKl>
cudaError_t launch_fwd_op(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16) return launch_fwd_cap<__nv_bfloat16, OP, DIR>(cap, a, s);
  if (dt == VLS_F16) return launch_fwd_cap<__half, OP, DIR>(cap, a, s);
  return launch_fwd_cap<float, OP, DIR>(cap, a, s);
}

}  // namespace vls
