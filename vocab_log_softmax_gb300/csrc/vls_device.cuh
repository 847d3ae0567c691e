// Device building blocks shared by the row kernels: raw 8-column vectors,
// packed fp32-pair arithmetic, the fp32 softcap, the single-read online
// statistics and their fixed-order reductions.
#pragma once

#include <cstdint>
#include <type_traits>

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "vls_internal.h"

namespace vls {
namespace dev {

namespace cg = cooperative_groups;

constexpr float kLog2e = 1.4426950408889634f;
// Lowest finite bfloat16 (bits 0xff7f).  Clamping a logit up to it changes
// nothing in any statistic -- its softmax weight is exactly 0 either way --
// but keeps -inf out of products such as 0 * (z - m).
constexpr float kLowest = -3.38953139e38f;
constexpr uint32_t kLowestBf16x2 = 0xff7fff7fu;
constexpr uint32_t kNegInfBf16x2 = 0xff80ff80u;

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

// 1/x on the special-function unit (PTX rcp.approx.ftz.f32).
__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// --------------------------------------------------------------------------
// Packed fp32 pairs (PTX .f32x2 arithmetic, two IEEE round-to-nearest
// operations per instruction: bit-identical to the scalar forms).
// --------------------------------------------------------------------------
using fp2 = unsigned long long;

__device__ __forceinline__ fp2 pk(float lo, float hi) {
  fp2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(fp2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ fp2 add2(fp2 a, fp2 b) {
  fp2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ fp2 sub2(fp2 a, fp2 b) {
  fp2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ fp2 mul2(fp2 a, fp2 b) {
  fp2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ fp2 fma2(fp2 a, fp2 b, fp2 c) {
  fp2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ fp2 splat(float v) { return pk(v, v); }
__device__ __forceinline__ fp2 ex2_2(fp2 y) {
  float a, b;
  upk(y, a, b);
  return pk(ex2(a), ex2(b));
}
__device__ __forceinline__ fp2 rcp2(fp2 y) {
  float a, b;
  upk(y, a, b);
  return pk(rcp(a), rcp(b));
}
// max of three (PTX max.f32 with three sources, sm_100 and later; a NaN
// source is dropped as by fmaxf)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float sum2(fp2 v) {
  float a, b;
  upk(v, a, b);
  return a + b;
}

// bfloat16x2 helpers on raw 32-bit words (two columns per word).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// 0xffff in each half where a == b, else 0
__device__ __forceinline__ uint32_t beq2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// float16x2 helpers on raw 32-bit words.
// max that returns NaN when either operand is NaN (the plain forms, like
// fmaxf, return the other): the clamp of -inf to the lowest finite value
// must not hide a NaN logit, which makes its whole row NaN.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t heq2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.eq.u32.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float h2f(uint32_t bits16) {
  float f;
  const unsigned short h = static_cast<unsigned short>(bits16);
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(h));
  return f;
}
constexpr uint32_t kNegInfF16x2 = 0xfc00fc00u;

// 16-byte read-only load that skips L1 (each logit is read once per sweep).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Starts pulling the 128-byte line at p into L2 (no register, no wait).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Starts pulling [p, p + bytes) into L2 with one bulk prefetch per 16 KiB,
// issued by the CTA's first threads (p 16-byte aligned, bytes a multiple of
// 16; no register, no wait).
__device__ __forceinline__ void prefetch_l2_range(const void* p, int64_t bytes) {
  constexpr int64_t kChunk = 16384;
  for (int64_t off = static_cast<int64_t>(threadIdx.x) * kChunk; off < bytes;
       off += static_cast<int64_t>(blockDim.x) * kChunk) {
    const int64_t n = bytes - off < kChunk ? bytes - off : kChunk;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(static_cast<const char*>(p) + off),
                 "r"(static_cast<uint32_t>(n))
                 : "memory");
  }
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// First element of row r of an operand addressed by a vls_rows descriptor:
// (r / group) * ld_group + (r % group) * ld.  Row indices stay below the
// 2^31 grid limit, so the split is a 32-bit division.  The C layer turns a
// single group (group 0) into group 2^31 - 1, so one branch-free path serves
// both forms (a branch here cost the register-bound backward maps spills).
template <class T>
__device__ __forceinline__ const T* row_ptr(const void* base, const vls_rows& l, int64_t r) {
  const uint32_t d = static_cast<uint32_t>(l.group);
  const uint32_t q = static_cast<uint32_t>(r) / d;
  const uint32_t t = static_cast<uint32_t>(r) - q * d;
  return static_cast<const T*>(base) + (static_cast<int64_t>(q) * l.ld_group + static_cast<int64_t>(t) * l.ld);
}

__device__ __forceinline__ bool valid_id(int64_t id, int64_t V, int64_t ignore_index) {
  return id != ignore_index && id >= 0 && id < V;
}

// --------------------------------------------------------------------------
// Raw 8-column vectors.  A vector is 8 consecutive columns for every dtype,
// so the column -> thread map (and every reduction order built on it) does
// not depend on the dtype: bf16 logits and their exact fp32 copies give the
// same bits.  `pair(i)` is columns 2i, 2i+1 as an fp32 pair.
// --------------------------------------------------------------------------
template <class T>
struct Raw8;

template <>
struct Raw8<__nv_bfloat16> {
  uint32_t w[4];
  __device__ __forceinline__ void load(const __nv_bfloat16* p) {
    const uint4 u = ld_stream16(p);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  }
  // columns j >= valid read as -inf
  __device__ __forceinline__ void load_scalar(const __nv_bfloat16* p, int valid) {
    const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = 2 * i < valid ? __ldg(q + 2 * i) : 0xff80u;
      const uint32_t hi = 2 * i + 1 < valid ? __ldg(q + 2 * i + 1) : 0xff80u;
      w[i] = lo | (hi << 16);
    }
  }
  __device__ __forceinline__ float max() const {
    const uint32_t m = bmax2(bmax2(w[0], w[1]), bmax2(w[2], w[3]));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
  __device__ __forceinline__ fp2 pair(int i) const {
    return pk(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  }
  __device__ __forceinline__ fp2 pair_clamped(int i) const {
    const uint32_t c = bmax2_nan(w[i], kLowestBf16x2);
    return pk(__uint_as_float(c << 16), __uint_as_float(c & 0xffff0000u));
  }
  __device__ __forceinline__ fp2 pair_abs(int i) const {
    const uint32_t a = w[i] & 0x7fff7fffu;
    return pk(__uint_as_float(a << 16), __uint_as_float(a & 0xffff0000u));
  }
  // sign bits of columns 2i, 2i+1 in bit 31 of each word
  __device__ __forceinline__ uint32_t sign_lo(int i) const { return w[i] << 16; }
  __device__ __forceinline__ uint32_t sign_hi(int i) const { return w[i]; }
  // nonzero iff some column of pair i has this = finite-or-+inf and q = -inf
  __device__ __forceinline__ uint32_t mismatch(int i, const Raw8& q) const {
    return beq2(q.w[i], kNegInfBf16x2) & ~beq2(w[i], kNegInfBf16x2);
  }
};

// float16: converted exactly to fp32 (cvt.f32.f16); -inf is clamped after
// the conversion, at the fp32 constant kLowest, far below any float16 value,
// so that it cannot collide with the lowest finite float16 (-65504).
template <>
struct Raw8<__half> {
  uint32_t w[4];
  __device__ __forceinline__ void load(const __half* p) {
    const uint4 u = ld_stream16(p);
    w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
  }
  __device__ __forceinline__ void load_scalar(const __half* p, int valid) {
    const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = 2 * i < valid ? __ldg(q + 2 * i) : 0xfc00u;
      const uint32_t hi = 2 * i + 1 < valid ? __ldg(q + 2 * i + 1) : 0xfc00u;
      w[i] = lo | (hi << 16);
    }
  }
  __device__ __forceinline__ float max() const {
    const uint32_t m = hmax2(hmax2(w[0], w[1]), hmax2(w[2], w[3]));
    return fmaxf(h2f(m & 0xffffu), h2f(m >> 16));
  }
  __device__ __forceinline__ fp2 pair(int i) const { return pk(h2f(w[i] & 0xffffu), h2f(w[i] >> 16)); }
  __device__ __forceinline__ fp2 pair_clamped(int i) const {
    return pk(max_nan(h2f(w[i] & 0xffffu), kLowest), max_nan(h2f(w[i] >> 16), kLowest));
  }
  __device__ __forceinline__ fp2 pair_abs(int i) const {
    const uint32_t a = w[i] & 0x7fff7fffu;
    return pk(h2f(a & 0xffffu), h2f(a >> 16));
  }
  __device__ __forceinline__ uint32_t sign_lo(int i) const { return w[i] << 16; }
  __device__ __forceinline__ uint32_t sign_hi(int i) const { return w[i]; }
  __device__ __forceinline__ uint32_t mismatch(int i, const Raw8& q) const {
    return heq2(q.w[i], kNegInfF16x2) & ~heq2(w[i], kNegInfF16x2);
  }
};

template <>
struct Raw8<float> {
  float v[8];
  __device__ __forceinline__ void load(const float* p) {
    const uint4 a = ld_stream16(p), b = ld_stream16(p + 4);
    v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
    v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
    v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
    v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
  }
  __device__ __forceinline__ void load_scalar(const float* p, int valid) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j < valid ? __ldg(p + j) : neg_inf();
  }
  __device__ __forceinline__ float max() const {
    return fmaxf(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])), fmaxf(fmaxf(v[4], v[5]), fmaxf(v[6], v[7])));
  }
  __device__ __forceinline__ fp2 pair(int i) const { return pk(v[2 * i], v[2 * i + 1]); }
  __device__ __forceinline__ fp2 pair_clamped(int i) const {
    return pk(max_nan(v[2 * i], kLowest), max_nan(v[2 * i + 1], kLowest));
  }
  __device__ __forceinline__ fp2 pair_abs(int i) const { return pk(fabsf(v[2 * i]), fabsf(v[2 * i + 1])); }
  __device__ __forceinline__ uint32_t sign_lo(int i) const { return __float_as_uint(v[2 * i]); }
  __device__ __forceinline__ uint32_t sign_hi(int i) const { return __float_as_uint(v[2 * i + 1]); }
  __device__ __forceinline__ uint32_t mismatch(int i, const Raw8& q) const {
    return ((q.v[2 * i] == neg_inf()) & (v[2 * i] != neg_inf())) |
           ((q.v[2 * i + 1] == neg_inf()) & (v[2 * i + 1] != neg_inf()));
  }
};

// Loads vector `vec` of a row: one or two 16-byte loads when the row start is
// 16-byte aligned and the vector is whole, else scalar loads (same values).
template <class T>
__device__ __forceinline__ void load_raw(Raw8<T>& r, const T* row, int64_t vec, int64_t V, bool aligned,
                                         int& valid) {
  const int64_t c0 = vec * 8;
  const int64_t rem = V - c0;
  valid = rem < 8 ? static_cast<int>(rem) : 8;
  if (aligned && valid == 8)
    r.load(row + c0);
  else
    r.load_scalar(row + c0, valid);
}

// --------------------------------------------------------------------------
// Final-logit softcap z = c tanh(x/c) in fp32 ("Final Logit Softcap",
// Summary), written with one exponential and one reciprocal:
//   a = |x|/c,  e = exp(-2a),  r = 1/(1+e),  tanh(a) = (1-e) r,
//   d tanh/du = 1 - tanh^2 = 4 e r^2,
// both with the sign of x.  1-e is exact for e in [1/2, 1] and the product
// carries an absolute error of a few 1e-7 * c; 4 e r^2 keeps full relative
// accuracy where tanh rounds to +-1.  x = -inf gives -c and slope 0.
// --------------------------------------------------------------------------
struct CapK {
  float c;     // cap
  float k;     // -2 log2(e) / c: exp(-2|x|/c) = 2^(|x| k)
  float k2;    // 2 log2(e) / c: exp(2x/c) = 2^(x k2)
  float a2;    // -2 c log2(e)
  // the largest x with x k2 <= 64 (so that exp(2x/c) <= 2^64), rounded down
  // to each input type: fp32, and packed pairs of bfloat16 and of float16
  float xmax;
  uint32_t xmax_bf16x2, xmax_f16x2;
};

__device__ __forceinline__ CapK cap_consts(float cap) {
  const float k2 = 2.0f * kLog2e / cap;
  const float xm = __fdiv_rd(64.0f, k2);
  const uint32_t b = __float_as_uint(xm) >> 16;                       // positive: truncation rounds down
  const uint32_t h = __half_as_ushort(__float2half_rd(xm));           // saturates at the largest finite half
  return {cap, -2.0f * kLog2e / cap, k2, -2.0f * cap * kLog2e, xm, b | (b << 16), h | (h << 16)};
}

// tanh(x/c) and e = exp(-2|x|/c), r = 1/(1+e) for the slope.
__device__ __forceinline__ float cap_t(float x, const CapK& K, float& e, float& r) {
  e = ex2(fabsf(x) * K.k);
  r = rcp(1.0f + e);
  const float t = (1.0f - e) * r;
  return __uint_as_float(__float_as_uint(t) | (__float_as_uint(x) & 0x80000000u));
}
__device__ __forceinline__ float cap_t(float x, const CapK& K) {
  float e, r;
  return cap_t(x, K, e, r);
}

// Packed form of cap_t for pair i of a raw vector (same operations).
template <class T>
__device__ __forceinline__ fp2 cap_t2(const Raw8<T>& v, int i, const CapK& K, fp2& e2, fp2& r2) {
  e2 = ex2_2(mul2(v.pair_abs(i), splat(K.k)));
  r2 = rcp2(add2(e2, splat(1.0f)));
  float t0, t1;
  upk(mul2(sub2(splat(1.0f), e2), r2), t0, t1);
  t0 = __uint_as_float(__float_as_uint(t0) | (v.sign_lo(i) & 0x80000000u));
  t1 = __uint_as_float(__float_as_uint(t1) | (v.sign_hi(i) & 0x80000000u));
  return pk(t0, t1);
}

// z - m for the softcapped logit: c t - m, one rounding.
__device__ __forceinline__ float cap_d(float t, float c, float m) { return fmaf(t, c, -m); }

// --------------------------------------------------------------------------
// The softcapped logit inside the forward sweeps, where only the softmax
// weights exp(z - m) and the target's z - m depend on it.  With
//   z = c tanh(x/c) = c - 2c r,   r = 1/(1 + E),   E = exp(2x/c) = 2^(x k2),
// the log2 weight is one FMA after the two special-function operations:
//   (z - m) log2(e) = a2 r + b2,   a2 = -2c log2(e),   b2 = (c - m) log2(e).
// The sign of x needs no handling: x = -inf gives E = 0 and r = 1 (z = -c),
// a large x gives E = +inf and r = 0 (z = c).  The absolute error of z is
// 2c r times the relative error of r, a few 1e-7 c, the same order as
// cap_t's; unlike cap_t it is not small relative to z near x = 0, which the
// standalone softcap output needs but a softmax weight does not.
// --------------------------------------------------------------------------
constexpr float kLn2 = 0.69314718055994531f;

// Pairs (of the four in an 8-column vector) whose reciprocal 1/(1 + E) runs
// on the FMA pipe (rcp2_fma_neg) instead of the special-function unit,
// which bounds the softcapped sweeps: bit i set for pair i.  A function of
// the column alone, so every sweep gets the same bits for the same column.
#ifndef VLS_CAP_FMA_PAIRS
#define VLS_CAP_FMA_PAIRS 0xD
#endif
constexpr uint32_t kCapFmaPairs = VLS_CAP_FMA_PAIRS;

// -1/(-nd) = 1/d for d in [1, 2^70] on the FMA pipe, from nd = -d: a seed
// from the bit pattern (0x7EF311C2 - bits(d), written 0xFEF311C2 - bits(nd);
// the constant fitted here to a relative error of at most 5.1% on that
// range), one third-order step r (1 + e + e^2) and one Newton-Raphson step
// r (1 + e), e = 1 - d r: each step multiplies the error's order, to within
// one fp32 ulp (0.77 ulp at most, checked on [1, 2^70]).
__device__ __forceinline__ fp2 rcp2_fma_neg(fp2 nd) {
  float a, b;
  upk(nd, a, b);
  fp2 r = pk(__uint_as_float(0xFEF311C2u - __float_as_uint(a)), __uint_as_float(0xFEF311C2u - __float_as_uint(b)));
  fp2 e = fma2(nd, r, splat(1.0f));
  r = fma2(r, fma2(e, e, e), r);
  e = fma2(nd, r, splat(1.0f));
  return fma2(r, e, r);
}

// Max over G vectors: one packed max tree over their words and one unpack
// for 16-bit types (the same value as the max of the vectors' maxima).
template <class T, int G>
__device__ __forceinline__ float group_max(const Raw8<T>* v) {
  if constexpr (sizeof(T) == 4) {
    float m = v[0].max();
#pragma unroll
    for (int u = 1; u < G; ++u) m = fmaxf(m, v[u].max());
    return m;
  } else {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    auto mx2 = [](uint32_t a, uint32_t b) { return kBf16 ? bmax2(a, b) : hmax2(a, b); };
    uint32_t m = mx2(mx2(v[0].w[0], v[0].w[1]), mx2(v[0].w[2], v[0].w[3]));
#pragma unroll
    for (int u = 1; u < G; ++u) m = mx2(m, mx2(mx2(v[u].w[0], v[u].w[1]), mx2(v[u].w[2], v[u].w[3])));
    if constexpr (kBf16) return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    else return fmaxf(h2f(m & 0xffffu), h2f(m >> 16));
  }
}

// The running max of the softcapped sweeps is taken over the 32 lanes of a
// warp (redux.sync.max.f32, sm_100 family), so that every lane sees the same
// running max.  Its growth, which costs three special-function operations
// (the cap of the new max and the rescale of the sums), is then a
// warp-uniform event, rare after the first vectors, instead of one that some
// lane of the warp meets at almost every vector.  A lane without a vector
// contributes -inf.
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}

// r = 1/(1 + exp(2x/c)) of one logit.
__device__ __forceinline__ float cap_r(float x, const CapK& K) { return rcp(1.0f + ex2(x * K.k2)); }

// The same special-function operations as volatile asm, for the rare growth
// step of a warp's running max: the compiler may not evaluate them
// speculatively ahead of the (warp-uniform) branch, where they would occupy
// the special-function unit at every group of vectors instead of only when
// the max grows.
__device__ __forceinline__ float ex2_rare(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_rare(float x) {
  float y;
  asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// cap_zr and rescale for that step (same operations, same bits)
__device__ __forceinline__ float cap_zr_rare(float x, const CapK& K) {
  return fmaf(rcp_rare(1.0f + ex2_rare(x * K.k2)), -2.0f * K.c, K.c);
}
// The softcapped value c - 2c r of one logit (the row max of a sweep).
__device__ __forceinline__ float cap_zr(float x, const CapK& K) { return fmaf(cap_r(x, K), -2.0f * K.c, K.c); }
// b2 = (c - m) log2(e) for the running max m.
__device__ __forceinline__ float cap_b2(float m, const CapK& K) { return (K.c - m) * kLog2e; }
// (z - m) log2(e) of one logit, given b2 of m.
__device__ __forceinline__ float cap_d2(float x, const CapK& K, float b2) { return fmaf(cap_r(x, K), K.a2, b2); }

// min(x, y) that returns NaN when either is NaN (fminf returns the other).
__device__ __forceinline__ float min_nan(float x, float y) {
  float r;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "f"(y));
  return r;
}

// Pair i of a raw vector with both values limited to K.xmax (one packed min
// for 16-bit types); -inf stays -inf and NaN stays NaN.
__device__ __forceinline__ fp2 pair_min(const Raw8<__nv_bfloat16>& v, int i, const CapK& K) {
  uint32_t w;
  asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(w) : "r"(v.w[i]), "r"(K.xmax_bf16x2));
  return pk(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ fp2 pair_min(const Raw8<__half>& v, int i, const CapK& K) {
  uint32_t w;
  asm("min.NaN.f16x2 %0, %1, %2;" : "=r"(w) : "r"(v.w[i]), "r"(K.xmax_f16x2));
  return pk(h2f(w & 0xffffu), h2f(w >> 16));
}
__device__ __forceinline__ fp2 pair_min(const Raw8<float>& v, int i, const CapK& K) {
  return pk(min_nan(v.v[2 * i], K.xmax), min_nan(v.v[2 * i + 1], K.xmax));
}

// (z - m) log2(e) for pair i of a raw vector, given b2 of m in both halves.
// With FMA_RCP the reciprocal runs on the FMA pipe (rcp2_fma_neg), on x
// limited to K.xmax so that 1 + E stays within its range; the reciprocal
// below 2^-64 it then gives in place of a smaller one only ever adds a term
// far below one ulp of c.
// CLAMP = false is for vectors known to hold nothing above K.xmax (the sweep
// checks the warp's max of the group): the limit is then skipped, with the
// same results.
template <class T, bool FMA_RCP, bool CLAMP>
__device__ __forceinline__ fp2 cap_d2_pair(const Raw8<T>& v, int i, const CapK& K, fp2 b2) {
  fp2 r;
  if constexpr (FMA_RCP) {
    r = rcp2_fma_neg(sub2(splat(-1.0f), ex2_2(mul2(CLAMP ? pair_min(v, i, K) : v.pair(i), splat(K.k2)))));
  } else {
    r = rcp2(add2(ex2_2(mul2(v.pair(i), splat(K.k2))), splat(1.0f)));
  }
  return fma2(r, splat(K.a2), b2);
}
template <class T, bool CLAMP = true>
__device__ __forceinline__ fp2 cap_d2_pair(const Raw8<T>& v, int i, const CapK& K, fp2 b2) {
  return ((kCapFmaPairs >> i) & 1u) ? cap_d2_pair<T, true, CLAMP>(v, i, K, b2) : cap_d2_pair<T, false, CLAMP>(v, i, K, b2);
}

// The logprob backward map's form.  There the logit enters through
// p = exp(z - m - log S) and the slope dz/dx = 1 - tanh(x/c)^2 = 4 E r^2:
//   log2 p = a2 r + (c - m - log S) log2(e),
// one FMA after E = exp(2x/c) and r = 1/(1 + E), with x limited to K.xmax
// so that E <= 2^64 and E r r stays finite (the slope it gives beyond that,
// below 2^-62, is as good as 0 next to any gradient; x = -inf gives E = 0,
// r = 1 and slope 0).  No sign handling and no 1 - e: three fewer packed
// operations a pair than cap_t2.  p carries the r-form's absolute error of z
// (a few 1e-7 c) as a relative error, which the gradient's bf16, fp16 and
// fp32 rounding rules all absorb.
// Pairs whose reciprocal runs on the FMA pipe in this map: 0 and 2 (bit i
// for pair i), 2% faster than none and than three; all four is 7% slower.
#ifndef VLS_CAP_BWD_FMA_PAIRS
#define VLS_CAP_BWD_FMA_PAIRS 0x5
#endif
constexpr uint32_t kCapBwdFmaPairs = VLS_CAP_BWD_FMA_PAIRS;

template <class T>
__device__ __forceinline__ fp2 cap_r_pair(const Raw8<T>& v, int i, const CapK& K, fp2& E) {
  E = ex2_2(mul2(pair_min(v, i, K), splat(K.k2)));
  return ((kCapBwdFmaPairs >> i) & 1u) ? rcp2_fma_neg(sub2(splat(-1.0f), E)) : rcp2(add2(E, splat(1.0f)));
}
// Scalar form (same operations as the special-function pairs).
__device__ __forceinline__ float cap_r_lim(float x, const CapK& K, float& E) {
  E = ex2(min_nan(x, K.xmax) * K.k2);
  return rcp(1.0f + E);
}
// (c - m - log S) log2(e) of a row.
__device__ __forceinline__ float cap_b2_ls(float m, float log_s, const CapK& K) {
  return ((K.c - m) - log_s) * kLog2e;
}

// The softcapped value of the row max (tanh is increasing, so the max of z
// is the cap of the max of x).
__device__ __forceinline__ float cap_z(float x, const CapK& K) { return K.c * cap_t(x, K); }

// --------------------------------------------------------------------------
// Online statistics (thread accumulators).  Each is centred on its running
// max m:  S = sum e^{z-m};  entropy W = sum e^{z-m} (z-m);
// KL(P||Q) W = sum e^{p-m_p} ((p-m_p) - (q-m_q)),
// re-centred when a max grows ("Add Triton kernels for vocab-parallel
// logprobs, entropy and KL", review "Suggested change"): when the max moves
// from m to M the entropy W becomes e^{m-M} (W + S (m-M)) and the KL W becomes
// e^{m_p-M_p} (W + S_p ((m_p-M_p) - (m_q-M_q))).  Even and odd columns of a
// vector accumulate in the two halves of a packed pair.
// --------------------------------------------------------------------------

// 2^((m_old - m_new) log2 e): re-centres a sum from m_old onto m_new >= m_old;
// 0 when m_old = -inf.
__device__ __forceinline__ float rescale(float m_old, float m_new) {
  return ex2((m_old - m_new) * kLog2e);
}
__device__ __forceinline__ float rescale_rare(float m_old, float m_new) {
  return ex2_rare((m_old - m_new) * kLog2e);
}

struct LogpState {
  float m, s;
  __device__ static LogpState identity() { return {neg_inf(), 0.0f}; }
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
  __device__ static EntropyState combine(const EntropyState& a, const EntropyState& b) {
    const float M = fmaxf(a.m, b.m);
    if (M == neg_inf()) return identity();
    const float fa = rescale(a.m, M), fb = rescale(b.m, M);
    const float wa = a.m != neg_inf() ? fa * fmaf(a.s, a.m - M, a.w) : 0.0f;
    const float wb = b.m != neg_inf() ? fb * fmaf(b.s, b.m - M, b.w) : 0.0f;
    return {M, a.s * fa + b.s * fb, wa + wb};
  }
  __device__ EntropyState shfl_xor(int lane_mask) const {
    return {__shfl_xor_sync(0xffffffffu, m, lane_mask), __shfl_xor_sync(0xffffffffu, s, lane_mask),
            __shfl_xor_sync(0xffffffffu, w, lane_mask)};
  }
};

// KL(P||Q) with P the first argument.  `flag` records a column where P is
// not -inf and Q is -inf (decided on the logits).
struct KlState {
  float mp, sp, mq, sq, w;
  uint32_t flag;
  __device__ static KlState identity() { return {neg_inf(), 0.0f, neg_inf(), 0.0f, 0.0f, 0u}; }
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
    const float wa = a.mp != neg_inf() ? fpa * fmaf(a.sp, (a.mp - Mp) - (a.mq - Mq), a.w) : 0.0f;
    const float wb = b.mp != neg_inf() ? fpb * fmaf(b.sp, (b.mp - Mp) - (b.mq - Mq), b.w) : 0.0f;
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

// Fused sweep (logprobs + entropy + KL of the same policy a): a's max and
// sum-exp, the entropy W of a, and (DIR != kFusedNoKl) b's max and sum-exp
// and the KL W in direction DIR (P = a for reverse, P = b for forward).
template <int DIR>
struct FusedState {
  float ma, sa, wh, mb, sb, wk;
  uint32_t flag;
  __device__ static FusedState identity() { return {neg_inf(), 0.0f, 0.0f, neg_inf(), 0.0f, 0.0f, 0u}; }
  __device__ static FusedState combine(const FusedState& x, const FusedState& y) {
    FusedState r;
    const float Ma = fmaxf(x.ma, y.ma), Mb = fmaxf(x.mb, y.mb);
    const float fax = Ma == neg_inf() ? 0.0f : rescale(x.ma, Ma);
    const float fay = Ma == neg_inf() ? 0.0f : rescale(y.ma, Ma);
    const float fbx = Mb == neg_inf() ? 0.0f : rescale(x.mb, Mb);
    const float fby = Mb == neg_inf() ? 0.0f : rescale(y.mb, Mb);
    r.ma = Ma;
    r.mb = Mb;
    r.sa = x.sa * fax + y.sa * fay;
    r.sb = x.sb * fbx + y.sb * fby;
    r.wh = (x.ma != neg_inf() ? fax * fmaf(x.sa, x.ma - Ma, x.wh) : 0.0f) +
           (y.ma != neg_inf() ? fay * fmaf(y.sa, y.ma - Ma, y.wh) : 0.0f);
    if (DIR == kFusedKlForward) {
      r.wk = (x.mb != neg_inf() ? fbx * fmaf(x.sb, (x.mb - Mb) - (x.ma - Ma), x.wk) : 0.0f) +
             (y.mb != neg_inf() ? fby * fmaf(y.sb, (y.mb - Mb) - (y.ma - Ma), y.wk) : 0.0f);
    } else {
      r.wk = (x.ma != neg_inf() ? fax * fmaf(x.sa, (x.ma - Ma) - (x.mb - Mb), x.wk) : 0.0f) +
             (y.ma != neg_inf() ? fay * fmaf(y.sa, (y.ma - Ma) - (y.mb - Mb), y.wk) : 0.0f);
    }
    r.flag = x.flag | y.flag;
    return r;
  }
  __device__ FusedState shfl_xor(int lane_mask) const {
    FusedState r;
    r.ma = __shfl_xor_sync(0xffffffffu, ma, lane_mask);
    r.sa = __shfl_xor_sync(0xffffffffu, sa, lane_mask);
    r.wh = __shfl_xor_sync(0xffffffffu, wh, lane_mask);
    r.mb = __shfl_xor_sync(0xffffffffu, mb, lane_mask);
    r.sb = __shfl_xor_sync(0xffffffffu, sb, lane_mask);
    r.wk = __shfl_xor_sync(0xffffffffu, wk, lane_mask);
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

// Butterfly over the first W lanes (xor W/2, ..., 1); lanes W..31 hold
// identities that never reach lanes 0..W-1.
template <int W, class S>
__device__ __forceinline__ S reduce_lanes(S s) {
#pragma unroll
  for (int off = W / 2; off > 0; off >>= 1) s = S::combine(s, s.shfl_xor(off));
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

// --------------------------------------------------------------------------
// Stores of 8 fp32 values as one vector of the output dtype.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  // cvt.rn.bf16x2.f32: both halves rounded to nearest even
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <class T>
struct Out8;

template <>
struct Out8<float> {
  __device__ static void store(float* p, const fp2 (&o)[4]) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) upk(o[i], v[2 * i], v[2 * i + 1]);
    st16(p, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3])));
    st16(p + 4,
         make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]), __float_as_uint(v[7])));
  }
  __device__ static void store1(float* p, float v) { *p = v; }
  __device__ static float nan_value() { return qnan(); }
};

template <>
struct Out8<__nv_bfloat16> {
  __device__ static void store(__nv_bfloat16* p, const fp2 (&o)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a, b;
      upk(o[i], a, b);
      w[i] = pack_bf16x2(a, b);
    }
    st16(p, make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static void store1(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

template <>
struct Out8<__half> {
  __device__ static void store(__half* p, const fp2 (&o)[4]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float a, b;
      upk(o[i], a, b);
      __half2 h = __floats2half2_rn(a, b);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    st16(p, make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static void store1(__half* p, float v) { *p = __float2half_rn(v); }
};

// Stores vector `vec` of an output row (whole and aligned: vector stores;
// otherwise element by element, columns < V only).
template <class T>
__device__ __forceinline__ void store_vec(T* row, int64_t vec, int64_t V, bool aligned, const fp2 (&o)[4]) {
  const int64_t c0 = vec * 8;
  if (aligned && c0 + 8 <= V) {
    Out8<T>::store(row + c0, o);
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a, b;
    upk(o[i], a, b);
    if (c0 + 2 * i < V) Out8<T>::store1(row + c0 + 2 * i, a);
    if (c0 + 2 * i + 1 < V) Out8<T>::store1(row + c0 + 2 * i + 1, b);
  }
}

// Scalar element load (gathers, fix-ups).
template <class T>
__device__ __forceinline__ float load1(const T* p);
template <>
__device__ __forceinline__ float load1<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load1<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
}
template <>
__device__ __forceinline__ float load1<__half>(const __half* p) {
  return h2f(__ldg(reinterpret_cast<const unsigned short*>(p)));
}

}  // namespace dev
}  // namespace vls
