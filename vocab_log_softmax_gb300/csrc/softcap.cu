// Standalone final-logit softcap ("Final Logit Softcap", Summary and Tensor
// and Precision Contract): y = c tanh(x/c) and gx = gy (1 - tanh^2(x/c)),
// fp32 math with one cast at the store, over a flat array of n elements.
//
// tanh and its slope come from one exponential and one reciprocal (see
// cap_t in vls_device.cuh).  For the output itself relative accuracy matters
// near 0, where (1 - e) loses digits, so |x/c| < 1/64 uses the odd cubic
// u - u^3/3 of the Taylor series instead (relative error below 2 u^4/15 <
// 1e-8 there).  The slope 4 e r^2 is accurate everywhere.
//
// Grid-stride kernels: the grid is one wave of resident CTAs (a multiple of
// the SM count) and each thread handles 8-element vectors (16-byte accesses
// for bf16, two for fp32) in batches; a misaligned pointer or the last
// n % 8 elements take scalar accesses with the same arithmetic.
#include "vls_device.cuh"

namespace vls {

using namespace dev;

constexpr int kCapThreads = 256;
constexpr float kCubicBelow = 1.0f / 64.0f;
// 8-element vectors each thread loads before mapping any: plain batches of
// 4 (16-bit; 2 for fp32, whose vectors take twice the registers) at 5
// resident CTAs (48 registers) in both directions.  Measured at 8192 x
// 151936 bf16: the forward 0.770 ms against 0.787 with a two-buffer software
// pipeline of 2 + 2, and against 0.801-0.835 with batches of 6 or 8 or at 4
// or 6 CTAs; the backward 1.157 ms against 1.168 at 6 CTAs.
template <class T>
constexpr int cap_unroll() { return sizeof(T) == 2 ? 4 : 2; }
constexpr int kSoftcapCtas = 5;

__device__ __forceinline__ float softcap_value(float x, const CapK& K, float rcap) {
  const float u = x * rcap;
  float t;
  if (fabsf(u) < kCubicBelow) {
    t = u * fmaf(u * u, -1.0f / 3.0f, 1.0f);
  } else {
    t = cap_t(x, K);
  }
  return K.c * t;
}

__device__ __forceinline__ float softcap_slope(float x, const CapK& K) {
  float e, r;
  cap_t(x, K, e, r);
  return 4.0f * e * r * r;
}

template <class T>
__device__ __forceinline__ fp2 softcap_pair(const Raw8<T>& v, int i, const CapK& K, float rcap) {
  fp2 e2, r2;
  const fp2 t2 = cap_t2(v, i, K, e2, r2);
  const fp2 u2 = mul2(v.pair(i), splat(rcap));
  const fp2 c2 = mul2(u2, fma2(mul2(u2, u2), splat(-1.0f / 3.0f), splat(1.0f)));
  float t0, t1, u0, u1, c0, c1;
  upk(t2, t0, t1);
  upk(u2, u0, u1);
  upk(c2, c0, c1);
  return mul2(pk(fabsf(u0) < kCubicBelow ? c0 : t0, fabsf(u1) < kCubicBelow ? c1 : t1), splat(K.c));
}

template <class T, class G>
__device__ __forceinline__ fp2 slope_pair(const Raw8<T>& v, const Raw8<G>& g, int i, const CapK& K) {
  fp2 e2, r2;
  cap_t2(v, i, K, e2, r2);
  return mul2(mul2(mul2(g.pair(i), e2), r2), mul2(r2, splat(4.0f)));
}

template <class T>
__global__ void __launch_bounds__(kCapThreads, kSoftcapCtas) softcap_fwd_kernel(const CapArgs a) {
  constexpr int kCapUnroll = cap_unroll<T>();
  const T* x = static_cast<const T*>(a.x);
  T* y = static_cast<T*>(a.out);
  const CapK K = cap_consts(a.cap);
  const int64_t nvec = a.n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCapThreads;
  const bool al = aligned16(x) && aligned16(y);
  int64_t v = static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  if (al) {
    for (; v + (kCapUnroll - 1) * stride < nvec; v += kCapUnroll * stride) {
      Raw8<T> r[kCapUnroll];
#pragma unroll
      for (int u = 0; u < kCapUnroll; ++u) r[u].load(x + 8 * (v + u * stride));
#pragma unroll
      for (int u = 0; u < kCapUnroll; ++u) {
        fp2 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = softcap_pair(r[u], i, K, a.rcap);
        Out8<T>::store(y + 8 * (v + u * stride), o);
      }
    }
    for (; v < nvec; v += stride) {
      Raw8<T> r;
      r.load(x + 8 * v);
      fp2 o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = softcap_pair(r, i, K, a.rcap);
      Out8<T>::store(y + 8 * v, o);
    }
    v = 8 * nvec + static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  }
  for (; v < a.n; v += stride) Out8<T>::store1(y + v, softcap_value(load1(x + v), K, a.rcap));
}

// The slope needs one exponential and one reciprocal per element; plain
// batches of 4 vectors of each input per thread (a software pipeline
// measured slower).
template <class T, class G>
__global__ void __launch_bounds__(kCapThreads, kSoftcapCtas) softcap_bwd_kernel(const CapArgs a) {
  constexpr int U = 4;
  const T* x = static_cast<const T*>(a.x);
  const G* gy = static_cast<const G*>(a.gy);
  T* gx = static_cast<T*>(a.out);
  const CapK K = cap_consts(a.cap);
  const int64_t nvec = a.n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCapThreads;
  const bool al = aligned16(x) && aligned16(gy) && aligned16(gx);
  int64_t v = static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  if (al) {
    for (; v + (U - 1) * stride < nvec; v += U * stride) {
      Raw8<T> r[U];
      Raw8<G> g[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        r[u].load(x + 8 * (v + u * stride));
        g[u].load(gy + 8 * (v + u * stride));
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        fp2 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = slope_pair(r[u], g[u], i, K);
        Out8<T>::store(gx + 8 * (v + u * stride), o);
      }
    }
    for (; v < nvec; v += stride) {
      Raw8<T> r;
      Raw8<G> g;
      r.load(x + 8 * v);
      g.load(gy + 8 * v);
      fp2 o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = slope_pair(r, g, i, K);
      Out8<T>::store(gx + 8 * v, o);
    }
    v = 8 * nvec + static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  }
  for (; v < a.n; v += stride) Out8<T>::store1(gx + v, load1(gy + v) * softcap_slope(load1(x + v), K));
}

// Grid-stride launch with exactly one wave: (resident CTAs per SM) x SMs,
// fewer when n is small.  `a.grid` holds the SM count on entry.
template <class K>
cudaError_t launch_one_wave(K kernel, CapArgs a, cudaStream_t s) {
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kCapThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t want = ((a.n >> 3) + kCapThreads - 1) / kCapThreads;
  const int64_t full = static_cast<int64_t>(a.grid) * per_sm;
  a.grid = static_cast<int>(want < 1 ? 1 : (want < full ? want : full));
  kernel<<<a.grid, kCapThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_softcap_fwd(vls_dtype dt, const CapArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16) return launch_one_wave(softcap_fwd_kernel<__nv_bfloat16>, a, s);
  if (dt == VLS_F16) return launch_one_wave(softcap_fwd_kernel<__half>, a, s);
  return launch_one_wave(softcap_fwd_kernel<float>, a, s);
}

cudaError_t launch_softcap_bwd(vls_dtype dt, const CapArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16) {
    if (a.gy_f32) return launch_one_wave(softcap_bwd_kernel<__nv_bfloat16, float>, a, s);
    return launch_one_wave(softcap_bwd_kernel<__nv_bfloat16, __nv_bfloat16>, a, s);
  }
  if (dt == VLS_F16) {
    if (a.gy_f32) return launch_one_wave(softcap_bwd_kernel<__half, float>, a, s);
    return launch_one_wave(softcap_bwd_kernel<__half, __half>, a, s);
  }
  return launch_one_wave(softcap_bwd_kernel<float, float>, a, s);
}

}  // namespace vls
