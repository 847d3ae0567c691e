// Device building blocks shared by the row kernels: element loads/stores,
// the fp32 softcap, the single-read online statistics and their fixed-order
// reductions.
#pragma once

#include <cstdint>

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "vls_internal.h"

namespace vls {
namespace dev {

namespace cg = cooperative_groups;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFltMax = 3.402823466e38f;

__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000u); }
__device__ __forceinline__ float pos_inf() { return __int_as_float(0x7f800000u); }
__device__ __forceinline__ float qnan() { return __int_as_float(0x7fffffffu); }

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32): relative error
// of a few fp32 ulp; 2^-inf = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte read-only load that skips L1 (each logit is read once per sweep).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// --------------------------------------------------------------------------
// Element access.  A "vector" is 8 consecutive columns for every dtype, so
// the column -> thread map (and with it every reduction order) does not
// depend on the dtype: bf16 logits and their exact fp32 copies give the same
// bits.
// --------------------------------------------------------------------------
template <class T>
struct Elem;

template <>
struct Elem<float> {
  __device__ static float load1(const float* p) { return __ldg(p); }
  __device__ static void load8(const float* p, float (&v)[8]) {
    const uint4 a = ld_stream16(p), b = ld_stream16(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
  __device__ static void store1(float* p, float v) { *p = v; }
  __device__ static void store8(float* p, const float (&v)[8]) {
    st16(p, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                       __float_as_uint(v[3])));
    st16(p + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]),
                           __float_as_uint(v[7])));
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  // cvt.rn.bf16x2.f32: both halves rounded to nearest even
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <>
struct Elem<__nv_bfloat16> {
  __device__ static float load1(const __nv_bfloat16* p) {
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  __device__ static void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 w = ld_stream16(p);
    v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xffff0000u);
    v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xffff0000u);
    v[4] = __uint_as_float(w.z << 16); v[5] = __uint_as_float(w.z & 0xffff0000u);
    v[6] = __uint_as_float(w.w << 16); v[7] = __uint_as_float(w.w & 0xffff0000u);
  }
  __device__ static void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
  __device__ static void store8(__nv_bfloat16* p, const float (&v)[8]) {
    st16(p, make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                       pack_bf16x2(v[6], v[7])));
  }
};

// Loads the 8 columns [8*vec, 8*vec + 8) of a row.  `aligned` selects one
// 16-byte load per 16 bytes; otherwise scalar loads give the same values.
// Columns at or beyond V (only in the last, partial vector) are not read;
// `valid` reports how many columns are real.
template <class T>
__device__ __forceinline__ void load_vec(const T* row, int64_t vec, int64_t V, bool aligned,
                                         float (&v)[8], int& valid) {
  const int64_t c0 = vec * 8;
  if (aligned && c0 + 8 <= V) {
    Elem<T>::load8(row + c0, v);
    valid = 8;
    return;
  }
  const int64_t rem = V - c0;
  valid = rem < 8 ? static_cast<int>(rem) : 8;
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = j < valid ? Elem<T>::load1(row + c0 + j) : 0.0f;
}

template <class T>
__device__ __forceinline__ void store_vec(T* row, int64_t vec, int64_t V, bool aligned,
                                          const float (&v)[8]) {
  const int64_t c0 = vec * 8;
  if (aligned && c0 + 8 <= V) {
    Elem<T>::store8(row + c0, v);
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (c0 + j < V) Elem<T>::store1(row + c0 + j, v[j]);
}

// --------------------------------------------------------------------------
// Final-logit softcap z = c*tanh(x/c) in fp32 ("Final Logit Softcap",
// Summary).  x/c is formed as x*(1/c): within one ulp of the correctly
// rounded quotient.  tanh is CUDA's tanhf.
// --------------------------------------------------------------------------
__device__ __forceinline__ float softcap_z(float x, float cap, float rcap) {
  return cap * tanhf(x * rcap);
}

// dz/dx = 1 - tanh^2(x/c) = sech^2(x/c).  Near the origin 1 - t^2 has no
// cancellation; elsewhere it is formed as 4e/(1+e)^2 with e = exp(-2|u|),
// which keeps full relative accuracy where tanh rounds to +-1.
__device__ __forceinline__ float softcap_dzdx(float u, float t) {
  const float au = fabsf(u);
  if (au < 0.5f) return fmaf(-t, t, 1.0f);
  const float e = ex2(-2.0f * kLog2e * au);
  const float r = __frcp_rn(1.0f + e);
  return 4.0f * e * r * r;
}

template <bool CAP>
__device__ __forceinline__ void apply_cap8(float (&z)[8], float cap, float rcap) {
  if (CAP) {
#pragma unroll
    for (int j = 0; j < 8; ++j) z[j] = softcap_z(z[j], cap, rcap);
  }
}

// Columns past the end of the row take part as masked (-inf) logits; the
// mask goes after the softcap so that it stays -inf.
__device__ __forceinline__ void mask_tail(float (&z)[8], int valid) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j >= valid) z[j] = neg_inf();
}

__device__ __forceinline__ float max8(const float (&z)[8]) {
  return fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])),
               fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
}

// 2^((m_old - m_new) * log2 e): the factor that re-centres a sum taken
// around m_old onto m_new >= m_old; 0 when m_old = -inf.
__device__ __forceinline__ float rescale(float m_old, float m_new) {
  return ex2((m_old - m_new) * kLog2e);
}

// --------------------------------------------------------------------------
// Online statistics.  Each state is centred on its running max m:
//   S = sum e^{z-m};  entropy W = sum e^{z-m} (z-m);
//   KL(P||Q) W = sum e^{p-m_p} ((p-m_p) - (q-m_q)),
// re-centred when a max grows ("Add Triton kernels for vocab-parallel
// logprobs, entropy and KL", review "Suggested change"); when the max moves
// from m to M the entropy W becomes e^{m-M} (W + S (m-M)), and the KL W
// becomes e^{m_p-M_p} (W + S_p ((m_p-M_p) - (m_q-M_q))).
// --------------------------------------------------------------------------
struct LogpState {
  float m, s;
  __device__ static LogpState identity() { return {neg_inf(), 0.0f}; }
  __device__ __forceinline__ void update(const float (&z)[8]) {
    const float vm = max8(z);
    if (vm > m) {
      s *= rescale(m, vm);
      m = vm;
    }
    if (m != neg_inf()) {
      float e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = ex2((z[j] - m) * kLog2e);
      s += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    }
  }
  __device__ static LogpState combine(const LogpState& a, const LogpState& b) {
    const float M = fmaxf(a.m, b.m);
    if (M == neg_inf()) return identity();
    return {M, a.s * rescale(a.m, M) + b.s * rescale(b.m, M)};
  }
  __device__ LogpState shfl_xor(int lane_mask) const {
    return {__shfl_xor_sync(0xffffffffu, m, lane_mask), __shfl_xor_sync(0xffffffffu, s, lane_mask)};
  }
};

struct EntropyState {
  float m, s, w;
  __device__ static EntropyState identity() { return {neg_inf(), 0.0f, 0.0f}; }
  __device__ __forceinline__ void update(const float (&z)[8]) {
    const float vm = max8(z);
    if (vm > m) {
      const float f = rescale(m, vm);
      w = s > 0.0f ? f * fmaf(s, m - vm, w) : 0.0f;
      s *= f;
      m = vm;
    }
    if (m != neg_inf()) {
      float e[8], ed[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float d = z[j] - m;
        e[j] = ex2(d * kLog2e);
        // -inf columns: e = 0 and d is clamped so that 0 * d stays 0
        ed[j] = e[j] * fmaxf(d, -kFltMax);
      }
      s += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
      w += ((ed[0] + ed[1]) + (ed[2] + ed[3])) + ((ed[4] + ed[5]) + (ed[6] + ed[7]));
    }
  }
  __device__ static EntropyState combine(const EntropyState& a, const EntropyState& b) {
    const float M = fmaxf(a.m, b.m);
    if (M == neg_inf()) return identity();
    const float fa = rescale(a.m, M), fb = rescale(b.m, M);
    const float wa = a.s > 0.0f ? fa * fmaf(a.s, a.m - M, a.w) : 0.0f;
    const float wb = b.s > 0.0f ? fb * fmaf(b.s, b.m - M, b.w) : 0.0f;
    return {M, a.s * fa + b.s * fb, wa + wb};
  }
  __device__ EntropyState shfl_xor(int lane_mask) const {
    return {__shfl_xor_sync(0xffffffffu, m, lane_mask), __shfl_xor_sync(0xffffffffu, s, lane_mask),
            __shfl_xor_sync(0xffffffffu, w, lane_mask)};
  }
};

// KL(P||Q) with P the first argument.  `flag` records a column where P is
// finite and Q is -inf (decided on the logits).
struct KlState {
  float mp, sp, mq, sq, w;
  int flag;
  __device__ static KlState identity() { return {neg_inf(), 0.0f, neg_inf(), 0.0f, 0.0f, 0}; }
  __device__ __forceinline__ void update(const float (&p)[8], const float (&q)[8]) {
    const float vmp = max8(p), vmq = max8(q);
    if (vmp > mp || vmq > mq) {
      const float Mp = fmaxf(mp, vmp), Mq = fmaxf(mq, vmq);
      const float fp = rescale(mp, Mp), fq = rescale(mq, Mq);
      w = sp > 0.0f ? fp * fmaf(sp, (mp - Mp) - (mq - Mq), w) : 0.0f;
      sp *= fp;
      sq *= fq;
      mp = Mp;
      mq = Mq;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) flag |= (q[j] == neg_inf()) & (p[j] != neg_inf());
    if (mp != neg_inf()) {
      float e[8], dp[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        dp[j] = p[j] - mp;
        e[j] = ex2(dp[j] * kLog2e);
      }
      sp += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
      if (mq != neg_inf()) {
        float ew[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // clamps keep 0 * (-inf) and inf - inf out of W; a column where
          // only Q is -inf is caught by the flag
          const float a = fmaxf(dp[j], -kFltMax), b = fmaxf(q[j] - mq, -kFltMax);
          ew[j] = e[j] * (a - b);
        }
        w += ((ew[0] + ew[1]) + (ew[2] + ew[3])) + ((ew[4] + ew[5]) + (ew[6] + ew[7]));
      }
    }
    if (mq != neg_inf()) {
      float e[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = ex2((q[j] - mq) * kLog2e);
      sq += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    }
  }
  __device__ static KlState combine(const KlState& a, const KlState& b) {
    const float Mp = fmaxf(a.mp, b.mp), Mq = fmaxf(a.mq, b.mq);
    KlState r;
    r.mp = Mp;
    r.mq = Mq;
    r.flag = a.flag | b.flag;
    const float fpa = Mp == neg_inf() ? 0.0f : rescale(a.mp, Mp);
    const float fpb = Mp == neg_inf() ? 0.0f : rescale(b.mp, Mp);
    const float fqa = Mq == neg_inf() ? 0.0f : rescale(a.mq, Mq);
    const float fqb = Mq == neg_inf() ? 0.0f : rescale(b.mq, Mq);
    r.sp = a.sp * fpa + b.sp * fpb;
    r.sq = a.sq * fqa + b.sq * fqb;
    const float wa = a.sp > 0.0f ? fpa * fmaf(a.sp, (a.mp - Mp) - (a.mq - Mq), a.w) : 0.0f;
    const float wb = b.sp > 0.0f ? fpb * fmaf(b.sp, (b.mp - Mp) - (b.mq - Mq), b.w) : 0.0f;
    r.w = wa + wb;
    return r;
  }
  __device__ KlState shfl_xor(int lane_mask) const {
    KlState r;
    r.mp = __shfl_xor_sync(0xffffffffu, mp, lane_mask);
    r.sp = __shfl_xor_sync(0xffffffffu, sp, lane_mask);
    r.mq = __shfl_xor_sync(0xffffffffu, mq, lane_mask);
    r.sq = __shfl_xor_sync(0xffffffffu, sq, lane_mask);
    r.w = __shfl_xor_sync(0xffffffffu, w, lane_mask);
    r.flag = __shfl_xor_sync(0xffffffffu, flag, lane_mask);
    return r;
  }
};

// Butterfly over the 32 lanes of a warp, always xor 16, 8, 4, 2, 1.
template <class S>
__device__ __forceinline__ S warp_reduce(S s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s = S::combine(s, s.shfl_xor(off));
  return s;
}

// Butterfly over the first 8 lanes (xor 4, 2, 1); lanes 8..31 hold identities
// that never reach lanes 0..7.
template <class S>
__device__ __forceinline__ S reduce8(S s) {
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) s = S::combine(s, s.shfl_xor(off));
  return s;
}

// --------------------------------------------------------------------------
// Cluster barrier (split arrive / wait).
// --------------------------------------------------------------------------
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__device__ __forceinline__ bool valid_id(int64_t id, int64_t V, int64_t ignore_index) {
  return id != ignore_index && id >= 0 && id < V;
}

}  // namespace dev
}  // namespace vls
