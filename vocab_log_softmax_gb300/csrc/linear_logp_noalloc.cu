// vls_linear_logp_fwd_noalloc: the fused linear-head logprob forward for
// callers that cannot allocate device memory.
//
// The ordinary route (vls_linear_logp_partial, then vls_logp_combine) needs
// two intermediate buffers between its kernels: one vls_partial per
// vocabulary chunk and row, and the chunks' target logits.  Some callers have
// no way to provide them: a serving engine that has handed all device memory
// to its own pool up front (its KV-cache arena, say) and forbids further
// cudaMalloc calls, or a host program that runs under a fixed device-memory
// budget it may not exceed.  For them this entry point keeps the two buffers
// in one fixed array in the library's own device memory, so a call needs
// only the inputs and the outputs.
//
// The array (kScratchBytes = 32 MiB) lives for as long as the library is
// loaded, on every GPU where this file's module is loaded: with CUDA's lazy
// module loading (the default) that is each GPU where this entry point has
// been called, with eager loading every GPU of the process.  Every call
// shares it, so two calls whose kernels overlap on the GPU (on different
// streams, or from different host threads) race on it and may return each
// other's results.
#include <mutex>

#include "vls_internal.h"

namespace {

// vls_partial entries (24 MiB) and fp32 target logits (8 MiB) the array holds
constexpr int64_t kNoAllocPartials = int64_t(1) << 20;
constexpr int64_t kNoAllocTargets = int64_t(1) << 21;
constexpr size_t kPartBytes = static_cast<size_t>(kNoAllocPartials) * sizeof(vls_partial);
constexpr size_t kScratchBytes = kPartBytes + static_cast<size_t>(kNoAllocTargets) * sizeof(float);

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices];   // the array's device address, per device, once looked up

// The device address of g_scratch on `dev`.  In host code the name g_scratch
// only stands for the symbol: its address must be asked of the runtime, once
// per device, with that device current.
int scratch_on(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return VLS_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
    if (prev != dev) cudaSetDevice(prev);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return VLS_OK;
}

}  // namespace

extern "C" int vls_linear_logp_fwd_noalloc(const void* h, int64_t ldh, const void* W, int64_t ldw, vls_dtype dt,
                                           int64_t N, int64_t D, int64_t V, const int64_t* ids, int32_t k,
                                           int64_t ignore_index, float* logp, vls_rowstat* stats,
                                           uint32_t* status, void* stream) {
  if (N < 0 || D < 1 || V < 1 || k < 1 || k > VLS_LINEAR_MAX_TOPK) return VLS_ERR_SHAPE;
  const int64_t chunks = vls_linear_logp_chunks(V);
  if (N > kNoAllocPartials / chunks || N * chunks * k > kNoAllocTargets) return VLS_ERR_TOO_LARGE;
  if (N == 0) return VLS_OK;
  if (!h) return VLS_ERR_NULL;
  // the device the launch goes to, chosen as for every other call
  int dev = -1;
  if (int e = vls::launch_device(h, stream, &dev)) return e;
  void* base = nullptr;
  if (int e = scratch_on(dev, &base)) return e;
  vls_partial* part = static_cast<vls_partial*>(base);
  float* zt = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kPartBytes);
  // every partial and target entry of [chunks, N(, k)] is written by the first
  // kernel before the second reads it, so nothing left by an earlier call is read
  if (int e = vls_linear_logp_partial(h, ldh, W, ldw, dt, N, D, V, ids, k, ignore_index, part, zt, status,
                                      stream))
    return e;
  return vls_logp_combine(part, zt, static_cast<int32_t>(chunks), N, ids, k, V, ignore_index, 0.0f, logp, stats,
                          stream);
}
