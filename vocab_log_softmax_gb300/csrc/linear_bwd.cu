// Backward of the fused linear head + logprobs: with z = h @ W^T and upstream
// gradients g [N, k],
//     dz = g (one-hot of the valid ids) - G p,   G = sum of the valid g,
//     dh = dz @ W,   dW = dz^T @ h,
// where p = softmax(z) comes from the forward's saved (m, log S) and logit
// tiles recomputed on the tensor cores (z is not stored by the forward).
//
// Three launches of the tcgen05 mainloop in tc_gemm.cuh, each reading its
// operands where they already are:
//  1. the dz map: the forward's GEMM z = h @ W^T (both K-major) with an
//     epilogue that forms dz in fp32, rounds it once to the operand dtype and
//     stores it as dz [N, V];
//  2. dh = dz @ W: A = dz K-major (K = V), B = W read MN-major ([V, D] is
//     [K, columns]);
//  3. dW = dz^T @ h: A = dz read MN-major ([N, V] is [K, rows]), B = h read
//     MN-major ([N, D] is [K, columns]).
// The workspace (dz) is the caller's.  Its leading dimension is padded to 8
// elements (16 bytes, as TMA needs); the tensor maps carry the true sizes, so
// padding is never read.
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

// Epilogue of a plain GEMM: C[row, col] = the accumulator, cast once, stored
// by each thread (any C; the TMA form below is used where it applies).
template <class T>
struct StoreEpi {
  static constexpr uint32_t kStageBytes = 0;
  T* C;
  int64_t ldc;
  struct State {};
  __device__ State begin(int64_t, bool, int) const { return {}; }
  __device__ void cols(State&, const float (&v)[32], int64_t row, bool row_ok, int64_t cbase, int nvalid,
                       tcg::EpiWarp&) const {
    if (row_ok && nvalid > 0) store_row32(C + row * ldc + cbase, v, nvalid);
  }
  __device__ void end(State&, int64_t, bool, int) const {}
  __device__ void finish(tcg::EpiWarp&) const {}
};

// TMA stores from an epilogue warp.  The warp's 32 rows x 32 columns,
// already rounded to 16 bits (pk: lane = row, 16 packed pairs), go into one
// of two 2 KB boxes of its staging area; one lane then stores the box
// (cp.async.bulk.tensor, which clips the parts outside the tensor).  The
// boxes use the 64-byte swizzle: the 16-byte chunk q of box row r sits at
// chunk q ^ ((r >> 1) & 3), so each of the warp's 16-byte shared-memory
// writes spreads over all 32 banks.  A box is rewritten only after the store
// issued from it has read it.  Called by the whole warp.
constexpr uint32_t kBoxBytes = 32 * 32 * 2;
constexpr uint32_t kBoxStageBytes = 2 * kBoxBytes;

__device__ __forceinline__ void store_box(const CUtensorMap* map, tcg::EpiWarp& w, const uint32_t (&pk)[16],
                                          int64_t cbase) {
  const uint32_t box = w.stage + (w.n & 1u) * kBoxBytes;
  if (w.n >= 2) {
    if (w.lane == 0) tc::bulk_wait_read<1>();   // the store from this box, two boxes ago
    __syncwarp();
  }
  const uint32_t rowb = box + static_cast<uint32_t>(w.lane) * 64u;
  const uint32_t sw = (static_cast<uint32_t>(w.lane) >> 1) & 3u;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    tc::st_shared16(rowb + ((static_cast<uint32_t>(q) ^ sw) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                    pk[4 * q + 3]);
  tc::fence_proxy_async_shared();
  __syncwarp();
  if (w.lane == 0) {
    tc::tma_store_2d(map, box, static_cast<int32_t>(cbase), static_cast<int32_t>(w.row0));
    tc::bulk_commit();
  }
  ++w.n;
}

// the CTA's shared memory outlives no store that reads it
__device__ __forceinline__ void finish_boxes(tcg::EpiWarp& w) {
  if (w.lane == 0) tc::bulk_wait_all();
  __syncwarp();
}

// The plain GEMM epilogue through TMA stores (store_box).
template <class T>
struct TmaStoreEpi {
  static constexpr uint32_t kStageBytes = kBoxStageBytes;
  CUtensorMap map;   // C [M, Ncols]: tcg::encode_store
  int64_t M;
  struct State {};
  __device__ State begin(int64_t, bool, int) const { return {}; }
  __device__ void cols(State&, const float (&v)[32], int64_t, bool, int64_t cbase, int nvalid,
                       tcg::EpiWarp& w) const {
    if (nvalid <= 0 || w.row0 >= M) return;   // no column or no row of C here (the same in every lane)
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) pk[i] = pack2<T>(v[2 * i], v[2 * i + 1]);
    store_box(&map, w, pk, cbase);
  }
  __device__ void end(State&, int64_t, bool, int) const {}
  __device__ void finish(tcg::EpiWarp& w) const { finish_boxes(w); }
};

// Epilogue of a split-K product: the fp32 partial sums of K run ks go to
// P[ks] ([M, ld] fp32, ld a multiple of 4); splitk_reduce adds the runs.
struct PartialEpi {
  static constexpr uint32_t kStageBytes = 0;
  float* P;
  int64_t M, ld;
  struct State {};
  __device__ State begin(int64_t, bool, int) const { return {}; }
  __device__ void cols(State&, const float (&v)[32], int64_t row, bool row_ok, int64_t cbase, int nvalid,
                       tcg::EpiWarp& w) const {
    if (!row_ok || nvalid <= 0) return;
    float* dst = P + (static_cast<int64_t>(w.ks) * M + row) * ld + cbase;
    if (nvalid == 32) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        dev::st16(dst + 4 * q, make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                                          __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nvalid) dst[i] = v[i];
    }
  }
  __device__ void end(State&, int64_t, bool, int) const {}
  __device__ void finish(tcg::EpiWarp&) const {}
};

// out[e] = the runs' partial sums P[0][e] + P[1][e] + ... in that order,
// rounded once to T; n (a multiple of 4) elements, P and out 16- and 8-byte
// aligned.
template <class T>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float* __restrict__ P, int runs, int64_t n,
                                                            T* __restrict__ out) {
  const int64_t n4 = n >> 2;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    float4 acc = __ldg(reinterpret_cast<const float4*>(P) + i);
    for (int r = 1; r < runs; ++r) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(P + static_cast<int64_t>(r) * n) + i);
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    *reinterpret_cast<uint2*>(out + 4 * i) = make_uint2(pack2<T>(acc.x, acc.y), pack2<T>(acc.z, acc.w));
  }
}

// Epilogue of the dz map: the logits tile becomes g one-hot - G p, stored
// to dz through TMA boxes (store_box).
template <class T>
struct DzEpi {
  static constexpr uint32_t kStageBytes = kBoxStageBytes;
  const int64_t* ids;
  int32_t k;
  int64_t ignore_index;
  int64_t V;
  const float* g;            // [N, k]
  const vls_rowstat* stats;  // [N]
  int64_t N;
  CUtensorMap map;           // dz [N, ld_dz]: tcg::encode_store

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

  __device__ void cols(State& st, const float (&v)[32], int64_t row, bool row_ok, int64_t cbase, int nvalid,
                       tcg::EpiWarp& ew) const {
    // every lane takes part: a row past N holds zeros (its state is 0 and
    // its logits the zero fill) and the store clips it
    if (nvalid == 0) return;
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
    if (ew.row0 < N) store_box(&map, ew, w, cbase);   // the same in every lane
  }

  __device__ void end(State&, int64_t, bool, int) const {}
  __device__ void finish(tcg::EpiWarp& ew) const { finish_boxes(ew); }
};

// the workspace: dz [N, pad8(V)] in the operand dtype
size_t workspace_bytes(int64_t N, int64_t V) { return align256(static_cast<size_t>(N) * pad8(V) * 2); }

template <bool BF16>
cudaError_t bwd_t(const LinearBwdArgs& a, int sms, cudaStream_t s) {
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  T* dz = static_cast<T*>(a.workspace);
  const int64_t ldv = pad8(a.V);
  const tc::WaitCtl wc{a.status, a.sticky, a.wait_ns};
  cudaError_t e;
  // the dz map, dz through TMA stores (the workspace is 256-byte aligned and
  // its rows are padded to 16-byte multiples, so the map always encodes)
  DzEpi<T> dze;
  dze.ids = a.ids;
  dze.k = a.k;
  dze.ignore_index = a.ignore_index;
  dze.V = a.V;
  dze.g = a.g;
  dze.stats = a.stats;
  dze.N = a.N;
  if (!tcg::encode_store(&dze.map, dz, BF16, a.N, a.V, ldv)) return cudaErrorInvalidValue;
  if ((e = tcg::launch_gemm<BF16>(a.h, a.ldh, a.N, a.W, a.ldw, a.V, a.D, kLinChunkTiles, false, wc, dze, sms, s)) !=
      cudaSuccess)
    return e;
  // dh = dz W has K = V: at few rows its tiles leave SMs idle, and at some
  // row counts their last wave runs part full.  Then K is split into runs
  // (tcg::fill_ksplit) whose fp32 partial sums go to the dW buffer (written
  // only by the last product, and large enough: runs x N x 4 bytes per
  // column against V x 2), and a fixed-order sum of the runs gives dh.
  const int runs = (a.D % 4) == 0 ? tcg::fill_ksplit(a.N, a.D, a.V, sms, 16, a.V / (2 * a.N)) : 1;
  const bool split = runs > 1 && int64_t(runs) * a.N * 2 <= a.V &&
                     (reinterpret_cast<uintptr_t>(a.dW) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.dh) & 7u) == 0;
  if (split) {
    float* P = static_cast<float*>(a.dW);
    const PartialEpi pe{P, a.N, a.D};
    if ((e = tcg::launch_gemm<BF16, false, true>(dz, ldv, a.N, a.W, a.ldw, a.D, a.V, 1, true, wc, pe, sms, s,
                                                 runs)) != cudaSuccess)
      return e;
    const int64_t n = a.N * a.D;
    const int64_t blocks = (n / 4 + 255) / 256;
    const int grid = static_cast<int>(blocks < 4 * sms ? blocks : 4 * sms);
    splitk_reduce_kernel<T><<<grid > 0 ? grid : 1, 256, 0, s>>>(P, runs, n, static_cast<T*>(a.dh));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // dh and dW: TMA stores when the output allows them (16-byte aligned base
  // and rows), else per-thread stores
  TmaStoreEpi<T> dht, dwt;
  dht.M = a.N;
  dwt.M = a.V;
  if (tcg::encode_store(&dht.map, a.dh, BF16, a.N, a.D, a.D) && tcg::encode_store(&dwt.map, a.dW, BF16, a.V, a.D, a.D)) {
    if (!split &&
        (e = tcg::launch_gemm<BF16, false, true>(dz, ldv, a.N, a.W, a.ldw, a.D, a.V, 1, true, wc, dht, sms, s)) !=
            cudaSuccess)
      return e;
    return tcg::launch_gemm<BF16, true, true>(dz, ldv, a.V, a.h, a.ldh, a.D, a.N, 1, true, wc, dwt, sms, s);
  }
  const StoreEpi<T> dhe{static_cast<T*>(a.dh), a.D};
  if (!split &&
      (e = tcg::launch_gemm<BF16, false, true>(dz, ldv, a.N, a.W, a.ldw, a.D, a.V, 1, true, wc, dhe, sms, s)) !=
          cudaSuccess)
    return e;
  const StoreEpi<T> dwe{static_cast<T*>(a.dW), a.D};
  return tcg::launch_gemm<BF16, true, true>(dz, ldv, a.V, a.h, a.ldh, a.D, a.N, 1, true, wc, dwe, sms, s);
}

}  // namespace

size_t linear_bwd_workspace(int64_t N, int64_t, int64_t V) { return workspace_bytes(N, V); }

cudaError_t launch_linear_logp_bwd(const LinearBwdArgs& a, int sms, cudaStream_t s) {
  return a.dt == VLS_BF16 ? bwd_t<true>(a, sms, s) : bwd_t<false>(a, sms, s);
}

}  // namespace vls
