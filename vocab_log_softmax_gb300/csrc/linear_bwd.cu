// Backward of the fused linear head + logprobs: with z = h @ W^T and upstream
// gradients g [N, k],
//     dz = g (one-hot of the valid ids) - G p,   G = sum of the valid g,
//     dh = dz @ W,   dW = dz^T @ h,
// where p = softmax(z) comes from the forward's saved (m, log S) and logit
// tiles recomputed on the tensor cores (z is not stored by the forward).
//
// Steps, all on tcgen05 through the mainloop of tc_gemm.cuh, whose operands
// are K-major:
//  1. h^T [D, N] and W^T [D, V] by a shared-memory tiled transpose (64 x 64
//     tiles, 16-byte accesses);
//  2. the dz map: the forward's GEMM z = h @ W^T with an epilogue that forms
//     dz in fp32, casts it once to the operand dtype and writes it both as
//     dz [N, V] and as dz^T [V, N];
//  3. dh = dz @ (W^T)^T: M = N, columns D, K = V;
//  4. dW = dz^T @ (h^T)^T: M = V, columns D, K = N.
// The workspace (h^T, W^T, dz, dz^T) is the caller's.  Leading dimensions are
// padded to 8 elements (16 bytes, as TMA needs); the tensor maps carry the
// true K, so padding is never read.
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_gemm.cuh"

namespace vls {

namespace {

constexpr int64_t pad8(int64_t x) { return (x + 7) & ~int64_t(7); }
constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <class T>
__device__ __forceinline__ T to_t(float x);
template <>
__device__ __forceinline__ __nv_bfloat16 to_t<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }
template <>
__device__ __forceinline__ __half to_t<__half>(float x) { return __float2half_rn(x); }

// two values rounded to 16 bits and packed, the first in the low half
template <class T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  const __half2 r = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// one half of a packed pair to 16-bit memory
template <class T>
__device__ __forceinline__ void st_half(T* p, uint32_t w, int hi) {
  *reinterpret_cast<uint16_t*>(p) = static_cast<uint16_t>(hi ? w >> 16 : w);
}

// 32 values of one row to 16-bit memory: four 16-byte stores when the run is
// whole and aligned, else element by element.
template <class T>
__device__ __forceinline__ void store_row32(T* dst, const float (&v)[32], int nvalid) {
  if (nvalid == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const T lo = to_t<T>(v[8 * q + 2 * e]), hi = to_t<T>(v[8 * q + 2 * e + 1]);
        w[e] = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&lo)) |
               (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(&hi)) << 16);
      }
      dev::st16(dst + 8 * q, make_uint4(w[0], w[1], w[2], w[3]));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) dst[i] = to_t<T>(v[i]);
  }
}

// Epilogue of a plain GEMM: C[row, col] = the accumulator, cast once.
template <class T>
struct StoreEpi {
  T* C;
  int64_t ldc;
  struct State {};
  __device__ State begin(int64_t, bool, int) const { return {}; }
  __device__ void cols(State&, const float (&v)[32], int64_t row, bool row_ok, int64_t cbase, int nvalid) const {
    if (row_ok && nvalid > 0) store_row32(C + row * ldc + cbase, v, nvalid);
  }
  __device__ void end(State&, int64_t, bool, int) const {}
};

// Epilogue of the dz map: the logits tile becomes g one-hot - G p.
template <class T>
struct DzEpi {
  const int64_t* ids;
  int32_t k;
  int64_t ignore_index;
  int64_t V;
  const float* g;            // [N, k]
  const vls_rowstat* stats;  // [N]
  T* dz;                     // [N, ld_dz]
  int64_t ld_dz;
  T* dzt;                    // [V, ld_dzt]
  int64_t ld_dzt;

  struct State {
    float m, c, G;             // max, log S * log2(e), sum of the valid upstream gradients
    int64_t id[kLinMaxTopk];   // valid ids, -1 otherwise
    float gj[kLinMaxTopk];
  };

  __device__ State begin(int64_t row, bool row_ok, int) const {
    State st;
    st.m = 0.0f;
    st.c = 0.0f;
    st.G = 0.0f;
    if (row_ok) {
      const vls_rowstat rs = stats[row];
      st.m = rs.m;
      st.c = rs.log_s * dev::kLog2e;
    }
#pragma unroll
    for (int j = 0; j < kLinMaxTopk; ++j) {
      const int64_t id = (row_ok && j < k) ? ids[row * k + j] : -1;
      const bool ok = j < k && row_ok && dev::valid_id(id, V, ignore_index);
      st.id[j] = ok ? id : -1;
      st.gj[j] = ok ? g[row * k + j] : 0.0f;
      st.G += st.gj[j];   // ascending j
    }
    return st;
  }

  __device__ void cols(State& st, const float (&v)[32], int64_t row, bool row_ok, int64_t cbase, int nvalid) const {
    if (!row_ok || nvalid == 0) return;
    float oh[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) oh[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < kLinMaxTopk; ++j) {
      if (j >= k) break;   // k is uniform: the scan stops after the row's own ids
      const int64_t loc = st.id[j] - cbase;
      if (loc >= 0 && loc < nvalid) {
#pragma unroll
        for (int i = 0; i < 32; ++i) oh[i] += loc == i ? st.gj[j] : 0.0f;
      }
    }
    // p = 2^((z - m) log2(e) - log2(S)) and dz = g one-hot - G p, pairwise
    const dev::fp2 m2 = dev::splat(st.m), l2 = dev::splat(dev::kLog2e), c2 = dev::splat(-st.c),
                   g2 = dev::splat(-st.G);
    uint32_t w[16];   // dz as 16-bit pairs, column 2i in the low half
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const dev::fp2 p = dev::ex2_2(dev::fma2(dev::sub2(dev::pk(v[2 * i], v[2 * i + 1]), m2), l2, c2));
      float d0, d1;
      dev::upk(dev::fma2(g2, p, dev::pk(oh[2 * i], oh[2 * i + 1])), d0, d1);
      w[i] = pack2<T>(d0, d1);
    }
    T* dst = dz + row * ld_dz + cbase;
    if (nvalid == 32 && dev::aligned16(dst)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) dev::st16(dst + 8 * q, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nvalid) st_half(dst + i, w[i >> 1], i & 1);
    }
    T* col = dzt + cbase * ld_dzt + row;   // lanes hold consecutive rows: each column's store is coalesced
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) st_half(col + i * ld_dzt, w[i >> 1], i & 1);
  }

  __device__ void end(State&, int64_t, bool, int) const {}
};

// y[c, r] = x[r, c] for a [rows, cols] 16-bit matrix with row stride ldx
// into y with row stride ldy, through 64 x 64 shared-memory tiles: 16-byte
// loads along x's rows, 16-byte stores along y's rows (element by element at
// ragged edges).  x, y and both strides must be 16-byte aligned.
__global__ void __launch_bounds__(256) transpose_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                         int64_t ldx, uint16_t* __restrict__ y, int64_t ldy) {
  __shared__ __align__(16) uint16_t tile[64][72];   // 144-byte rows: 16-byte aligned, banks staggered
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64, c0 = static_cast<int64_t>(blockIdx.x) * 64;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int vec = threadIdx.x + 256 * i, r = vec >> 3, c8 = (vec & 7) * 8;
    const int64_t gr = r0 + r, gc = c0 + c8;
    if (gr < rows && gc + 8 <= cols) {
      *reinterpret_cast<uint4*>(&tile[r][c8]) = __ldg(reinterpret_cast<const uint4*>(x + gr * ldx + gc));
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[r][c8 + e] = (gr < rows && gc + e < cols) ? x[gr * ldx + gc + e] : 0;
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int vec = threadIdx.x + 256 * i, oc = vec >> 3, r8 = (vec & 7) * 8;
    const int64_t gc = c0 + oc, gr = r0 + r8;
    if (gc >= cols) continue;
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = tile[r8 + e][oc];
    if (gr + 8 <= rows) {
      uint4 w;
      w.x = v[0] | (static_cast<uint32_t>(v[1]) << 16);
      w.y = v[2] | (static_cast<uint32_t>(v[3]) << 16);
      w.z = v[4] | (static_cast<uint32_t>(v[5]) << 16);
      w.w = v[6] | (static_cast<uint32_t>(v[7]) << 16);
      *reinterpret_cast<uint4*>(y + gc * ldy + gr) = w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (gr + e < rows) y[gc * ldy + gr + e] = v[e];
    }
  }
}

cudaError_t transpose(const void* x, int64_t rows, int64_t cols, int64_t ldx, void* y, int64_t ldy,
                      cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((cols + 63) / 64), static_cast<unsigned>((rows + 63) / 64));
  transpose_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), rows, cols, ldx, static_cast<uint16_t*>(y),
                                        ldy);
  return cudaGetLastError();
}

struct Workspace {
  size_t hT, WT, dz, dzt, total;   // byte offsets and size
};

Workspace layout(int64_t N, int64_t D, int64_t V) {
  Workspace w;
  size_t off = 0;
  w.hT = off;
  off = align256(off + static_cast<size_t>(D) * pad8(N) * 2);
  w.WT = off;
  off = align256(off + static_cast<size_t>(D) * pad8(V) * 2);
  w.dz = off;
  off = align256(off + static_cast<size_t>(N) * pad8(V) * 2);
  w.dzt = off;
  off = align256(off + static_cast<size_t>(V) * pad8(N) * 2);
  w.total = off;
  return w;
}

template <bool BF16>
cudaError_t bwd_t(const LinearBwdArgs& a, int sms, cudaStream_t s) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const Workspace w = layout(a.N, a.D, a.V);
  unsigned char* ws = static_cast<unsigned char*>(a.workspace);
  T* hT = reinterpret_cast<T*>(ws + w.hT);
  T* WT = reinterpret_cast<T*>(ws + w.WT);
  T* dz = reinterpret_cast<T*>(ws + w.dz);
  T* dzt = reinterpret_cast<T*>(ws + w.dzt);
  const int64_t ldn = pad8(a.N), ldv = pad8(a.V);
  cudaError_t e;
  if ((e = transpose(a.h, a.N, a.D, a.ldh, hT, ldn, s)) != cudaSuccess) return e;
  if ((e = transpose(a.W, a.V, a.D, a.ldw, WT, ldv, s)) != cudaSuccess) return e;
  const DzEpi<T> dze{a.ids, a.k, a.ignore_index, a.V, a.g, a.stats, dz, ldv, dzt, ldn};
  if ((e = tcg::launch_gemm<BF16>(a.h, a.ldh, a.N, a.W, a.ldw, a.V, a.D, kLinChunkTiles, false, a.status, dze, sms, s)) !=
      cudaSuccess)
    return e;
  const StoreEpi<T> dhe{static_cast<T*>(a.dh), a.D};
  if ((e = tcg::launch_gemm<BF16>(dz, ldv, a.N, WT, ldv, a.D, a.V, 1, true, a.status, dhe, sms, s)) != cudaSuccess) return e;
  const StoreEpi<T> dwe{static_cast<T*>(a.dW), a.D};
  return tcg::launch_gemm<BF16>(dzt, ldn, a.V, hT, ldn, a.D, a.N, 1, true, a.status, dwe, sms, s);
}

}  // namespace

size_t linear_bwd_workspace(int64_t N, int64_t D, int64_t V) { return layout(N, D, V).total; }

cudaError_t launch_linear_logp_bwd(const LinearBwdArgs& a, int sms, cudaStream_t s) {
  return a.dt == VLS_BF16 ? bwd_t<true>(a, sms, s) : bwd_t<false>(a, sms, s);
}

}  // namespace vls
