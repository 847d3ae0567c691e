// Standalone final-logit softcap ("Final Logit Softcap", Summary and Tensor
// and Precision Contract): y = c*tanh(x/c) and gx = gy*(1 - tanh^2(x/c)),
// fp32 math with one cast at the store, over a flat array of n elements.
//
// Grid-stride kernels: the grid is a multiple of the SM count and each
// thread handles 8-element vectors (16-byte accesses for bf16, two for
// fp32); a misaligned pointer or the last n % 8 elements take scalar
// accesses with the same arithmetic.
#include "vls_device.cuh"

namespace vls {

constexpr int kCapThreads = 256;

template <class T>
__global__ void __launch_bounds__(kCapThreads) softcap_fwd_kernel(const CapArgs a) {
  using namespace dev;
  const T* x = static_cast<const T*>(a.x);
  T* y = static_cast<T*>(a.out);
  const int64_t nvec = a.n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCapThreads;
  const bool al = aligned16(x) && aligned16(y);
  int64_t v = static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  if (al) {
    for (; v < nvec; v += stride) {
      float z[8];
      Elem<T>::load8(x + 8 * v, z);
#pragma unroll
      for (int j = 0; j < 8; ++j) z[j] = softcap_z(z[j], a.cap, a.rcap);
      Elem<T>::store8(y + 8 * v, z);
    }
    v = 8 * nvec + static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  }
  for (; v < a.n; v += stride) Elem<T>::store1(y + v, softcap_z(Elem<T>::load1(x + v), a.cap, a.rcap));
}

template <class T, class G>
__global__ void __launch_bounds__(kCapThreads) softcap_bwd_kernel(const CapArgs a) {
  using namespace dev;
  const T* x = static_cast<const T*>(a.x);
  const G* gy = static_cast<const G*>(a.gy);
  T* gx = static_cast<T*>(a.out);
  const int64_t nvec = a.n >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCapThreads;
  const bool al = aligned16(x) && aligned16(gy) && aligned16(gx);
  int64_t v = static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  if (al) {
    for (; v < nvec; v += stride) {
      float z[8], g[8];
      Elem<T>::load8(x + 8 * v, z);
      Elem<G>::load8(gy + 8 * v, g);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float u = z[j] * a.rcap;
        z[j] = g[j] * softcap_dzdx(u, tanhf(u));
      }
      Elem<T>::store8(gx + 8 * v, z);
    }
    v = 8 * nvec + static_cast<int64_t>(blockIdx.x) * kCapThreads + threadIdx.x;
  }
  for (; v < a.n; v += stride) {
    const float u = Elem<T>::load1(x + v) * a.rcap;
    Elem<T>::store1(gx + v, Elem<G>::load1(gy + v) * softcap_dzdx(u, tanhf(u)));
  }
}

cudaError_t launch_softcap_fwd(vls_dtype dt, const CapArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16)
    softcap_fwd_kernel<__nv_bfloat16><<<a.grid, kCapThreads, 0, s>>>(a);
  else
    softcap_fwd_kernel<float><<<a.grid, kCapThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_softcap_bwd(vls_dtype dt, const CapArgs& a, cudaStream_t s) {
  if (dt == VLS_BF16) {
    if (a.gy_f32)
      softcap_bwd_kernel<__nv_bfloat16, float><<<a.grid, kCapThreads, 0, s>>>(a);
    else
      softcap_bwd_kernel<__nv_bfloat16, __nv_bfloat16><<<a.grid, kCapThreads, 0, s>>>(a);
  } else {
    softcap_bwd_kernel<float, float><<<a.grid, kCapThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace vls
