// C ABI of libvls (declared in include/vls.h): argument validation, the
// device guard, the launch-geometry policy and dispatch to the kernels.
//
// Validation order for every call: shapes, dtypes and cap first (no CUDA
// call), then the empty-input fast return, then NULL pointers, then the
// device of every pointer and of the stream, then the launch.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <initializer_list>

#include "vls_internal.h"
#include "vls_test.h"

namespace vls {
namespace {

constexpr int64_t kMaxGrid = 0x7fffffff;

bool dtype_ok(int dt) { return dt == VLS_F32 || dt == VLS_BF16 || dt == VLS_F16; }

// cap == 0 disables the softcap in the row calls; NaN, inf and negative
// values are rejected ("Final Logit Softcap", Summary: the cap must be finite
// and positive).
int check_row_cap(float cap) { return (std::isfinite(cap) && cap >= 0.0f) ? VLS_OK : VLS_ERR_CAP; }
int check_softcap_cap(float cap) { return (std::isfinite(cap) && cap > 0.0f) ? VLS_OK : VLS_ERR_CAP; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Tuning and fault injection.  The product library has fixed values.  The
// test build (VLS_TEST_HOOKS, lib/libvls_test.so, hooks in include/vls_test.h)
// lets a test choose other launch geometries, the 1-SM tensor-core form and
// a shorter wait limit, and make a call fail on purpose on the host, so that
// error paths can be exercised without a GPU fault.
// ---------------------------------------------------------------------------
constexpr int64_t kFwdVecPerCta = 24576;
constexpr int64_t kBwdVecPerCta = 4096;

#ifdef VLS_TEST_HOOKS
std::atomic<int> g_fault{VLS_TEST_FAULT_NONE};
std::atomic<uint64_t> g_wait_ns{0};
std::atomic<int64_t> g_fwd_vec{0}, g_bwd_vec{0};
std::atomic<int> g_cta_group{0};
int64_t fwd_vec_target() {
  const int64_t v = g_fwd_vec.load(std::memory_order_relaxed);
  return v > 0 ? v : kFwdVecPerCta;
}
int64_t bwd_vec_target() {
  const int64_t v = g_bwd_vec.load(std::memory_order_relaxed);
  return v > 0 ? v : kBwdVecPerCta;
}
bool fault_is(int mode) { return g_fault.load(std::memory_order_relaxed) == mode; }
#else
constexpr int64_t fwd_vec_target() { return kFwdVecPerCta; }
constexpr int64_t bwd_vec_target() { return kBwdVecPerCta; }
constexpr bool fault_is(int) { return false; }
#endif

// Forward geometry: a function of V only.  One CTA per row up to 24576
// vectors (196608 columns), then a cluster of up to 8 CTAs.  Fewer, longer
// CTAs win at the row counts this path serves (thousands of rows): every CTA
// of a cluster waits at the cluster barrier for its slowest sibling.
void fwd_geometry(int64_t V, int* cluster, int64_t* vec_per_cta) {
  const int64_t target = fwd_vec_target();
  const int64_t nvec = ceil_div(V, 8);
  int64_t c = ceil_div(nvec, target);
  if (c < 1) c = 1;
  if (c > kMaxCluster) c = kMaxCluster;
  *cluster = static_cast<int>(c);
  *vec_per_cta = ceil_div(nvec, c);
}

// Backward geometry: results do not depend on it (pure map).  Top-k rows
// prepare their id list once per CTA, so they take whole rows up to 262144
// columns.  A piece's run of vectors is rounded up to a multiple of
// kBwdVecRound (two batches of one vector per thread), so that the sweeps'
// batched loops cover it whole and only a row's last piece ends in the
// one-vector-at-a-time tail: at 151936 columns that made the maps 2-4%
// faster (4096 + 4096 + 4096 + 4096 + 2608 vectors instead of 5 x 3799).
constexpr int64_t kBwdVecRound = 512;
void bwd_geometry(int64_t V, int32_t k, int* chunks, int64_t* vec_per_cta) {
  const int64_t target = bwd_vec_target();
  const int64_t nvec = ceil_div(V, 8);
  const int64_t t = k > 1 ? 8 * target : target;
  int64_t c = ceil_div(nvec, t);
  if (c < 1) c = 1;
  int64_t per = ceil_div(ceil_div(nvec, c), kBwdVecRound) * kBwdVecRound;
  if (per > nvec) per = nvec;
  *chunks = static_cast<int>(ceil_div(nvec, per));
  *vec_per_cta = per;
}

// Small batches: when the rows alone would leave SMs idle, the backward's
// rows are cut into more pieces (of at least 256 vectors, one per thread)
// until the grid covers every SM twice.  The backward is a map, so its split
// changes no result.  Top-k rows keep whole-row pieces: each CTA prepares
// the row's id list.
void widen_bwd(BwdArgs& a, int sms) {
  if (a.k > 1 || a.rows < 1) return;
  const int64_t nvec = ceil_div(a.vocab, 8);
  const int64_t want = ceil_div(2 * static_cast<int64_t>(sms), a.rows);
  const int64_t most = ceil_div(nvec, 256);
  const int64_t c = want < most ? want : most;
  if (c > a.chunks) {
    a.chunks = static_cast<int>(c);
    a.vec_per_cta = ceil_div(nvec, c);
  }
}

int sm_count(int dev) {
  static std::atomic<int> cache[64];   // several host threads may ask; a repeated query is harmless
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = 1;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Few rows (the small-batch workloads): a forward launch with at most one
// CTA per SM leaves most of the GPU idle, and each CTA waits on DRAM latency
// batch after batch.  Then every CTA first asks L2 for its whole run, when
// the launch's inputs take at most a quarter of L2.  A prefetch changes no
// result.  (The backward maps are already cut into small pieces at few rows,
// see widen_bwd, and gained nothing from it.)
#ifndef VLS_PREFETCH_MAX_BYTES
#define VLS_PREFETCH_MAX_BYTES (32ll << 20)
#endif
constexpr int64_t kPrefetchMaxBytes = VLS_PREFETCH_MAX_BYTES;
int64_t input_bytes(int64_t N, int64_t V, vls_dtype dt, bool two) {
  return N * V * (dt == VLS_F32 ? 4 : 2) * (two ? 2 : 1);
}
void few_rows_prefetch(FwdArgs& a, vls_dtype dt, int dev) {
  a.prefetch = a.rows * a.cluster <= sm_count(dev) &&
               input_bytes(a.rows, a.vocab, dt, a.y != nullptr) <= kPrefetchMaxBytes;
}

// Finds the one device that holds every non-NULL pointer and owns the stream.
int resolve_device(std::initializer_list<const void*> ptrs, void* stream, int* dev_out) {
  // test build: the device check fails before any CUDA call
  if (fault_is(VLS_TEST_FAULT_VALIDATE)) return VLS_ERR_ARG;
  if (fault_is(VLS_TEST_FAULT_DEVICE)) return VLS_ERR_DEVICE;
  // While a stream is being captured into a CUDA graph the runtime refuses
  // pointer-attribute and stream-device queries, and the refusal would end the
  // capture: take the current device, which the capturing caller has made the
  // stream's (that is what CUDA requires of a launch into a capture anyway).
  if (reinterpret_cast<uintptr_t>(stream) > 2) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    if (cs != cudaStreamCaptureStatusNone) {
      int cur = -1;
      if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return VLS_ERR_DEVICE;
      }
      *dev_out = cur;
      return VLS_OK;
    }
  }
  int dev = -1;
  for (const void* p : ptrs) {
    if (!p) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) return VLS_ERR_DEVICE;
    if (dev < 0) dev = at.device;
    if (at.device != dev) return VLS_ERR_DEVICE;
  }
  if (dev < 0) return VLS_ERR_DEVICE;
  // NULL, cudaStreamLegacy (1) and cudaStreamPerThread (2) are per-device
  // handles: they refer to the device made current by the guard.
  if (reinterpret_cast<uintptr_t>(stream) > 2) {
    int sdev = -1;
    if (cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev) != cudaSuccess) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    if (sdev != dev) return VLS_ERR_DEVICE;
  }
  *dev_out = dev;
  return VLS_OK;
}

// Makes `dev` current for the launch and restores the caller's device.
class DeviceGuard {
 public:
  int enter(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) {
      cudaGetLastError();
      return VLS_ERR_DEVICE;
    }
    if (prev_ != dev) {
      if (cudaSetDevice(dev) != cudaSuccess) {
        cudaGetLastError();
        return VLS_ERR_DEVICE;
      }
      switched_ = true;
    }
    return VLS_OK;
  }
  ~DeviceGuard() {
    if (switched_) cudaSetDevice(prev_);
  }

 private:
  int prev_ = -1;
  bool switched_ = false;
};

int launch_status(cudaError_t e) {
  if (e == cudaSuccess) e = cudaGetLastError();
  else cudaGetLastError();
  return e == cudaSuccess ? VLS_OK : VLS_ERR_LAUNCH;
}

// The launch of a call and its status.  In the test build a launch fault
// skips the launch (outputs are left as they were) and reports VLS_ERR_LAUNCH.
#define VLS_LAUNCH(call) (fault_is(VLS_TEST_FAULT_LAUNCH) ? VLS_ERR_LAUNCH : launch_status(call))

int check_rows(int64_t N, int64_t V) {
  if (N < 0 || V < 1) return VLS_ERR_SHAPE;
  return VLS_OK;
}

// A row descriptor of an operand with V columns: NULL, a row stride below V,
// a negative group or (with groups) a group stride below V are rejected.
int check_layout(const vls_rows* r, int64_t V) {
  if (!r) return VLS_ERR_NULL;
  if (r->ld < V || r->group < 0 || (r->group > 0 && r->ld_group < V)) return VLS_ERR_SHAPE;
  return VLS_OK;
}

// The kernels' form of a checked descriptor: one group (group 0, or a group
// of at least 2^31 - 1 rows) becomes group 2^31 - 1, above every row index.
constexpr int64_t kOneGroup = 0x7fffffff;
vls_rows kernel_rows(const vls_rows& r) {
  if (r.group == 0 || r.group >= kOneGroup) return vls_rows{r.ld, kOneGroup, 0};
  return r;
}

FwdArgs fwd_args(int64_t N, int64_t V, float cap) {
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.rows = N;
  a.vocab = V;
  a.cap = cap;
  a.rcap = cap > 0.0f ? 1.0f / cap : 0.0f;
  a.rx = a.ry = vls_rows{0, kOneGroup, 0};  // until the call sets its operands
  a.vocab_offset = 0;
  a.vocab_total = V;
  fwd_geometry(V, &a.cluster, &a.vec_per_cta);
  return a;
}

BwdArgs bwd_args(int64_t N, int64_t V, int32_t k, float cap) {
  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.rows = N;
  a.vocab = V;
  a.cap = cap;
  a.rcap = cap > 0.0f ? 1.0f / cap : 0.0f;
  a.rx = a.ry = vls_rows{0, kOneGroup, 0};  // until the call sets its operands
  a.k = k;
  a.vocab_offset = 0;
  a.vocab_total = V;
  bwd_geometry(V, k, &a.chunks, &a.vec_per_cta);
  return a;
}

// A shard [offset, offset + V_shard) of a V_total-column vocabulary.
int check_shard(int64_t N, int64_t V_shard, int64_t offset, int64_t V_total) {
  if (N < 0 || V_shard < 0 || V_total < 1 || offset < 0 || offset + V_shard > V_total)
    return VLS_ERR_SHAPE;
  return VLS_OK;
}

// Bit 0 (tc::kStatusTimeout): a bounded wait in a tensor-core kernel ran
// out on this device since the last vls_check_device_error.  A __device__
// variable exists once on every device that loads this module.
__device__ uint32_t g_device_status;

std::atomic<uint32_t*> g_status_addr[64];   // its address per device, once looked up

}  // namespace

int launch_device(const void* p, void* stream, int* dev) { return resolve_device({p}, stream, dev); }

uint32_t* tc_sticky_status() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  uint32_t* p = g_status_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    // in host code the variable's name only stands for the symbol: its
    // device address is asked of the runtime, with the device current
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    p = static_cast<uint32_t*>(a);
    g_status_addr[dev].store(p, std::memory_order_release);
  }
  return p;
}

uint64_t tc_wait_ns() {
#ifdef VLS_TEST_HOOKS
  const uint64_t v = g_wait_ns.load(std::memory_order_relaxed);
  if (v > 0) return v;
#endif
  return kTcWaitNs;
}

namespace tcg {
int cta_group() {
#ifdef VLS_TEST_HOOKS
  if (g_cta_group.load(std::memory_order_relaxed) == 1) return 1;
#endif
  return 2;
}
}  // namespace tcg

}  // namespace vls

using namespace vls;

extern "C" {

int vls_version(void) { return 101; }

int vls_check_device_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return VLS_ERR_LAUNCH;
  }
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)) != cudaSuccess) {
    cudaGetLastError();
    return VLS_ERR_LAUNCH;
  }
  if (v == 0) return VLS_OK;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess) cudaGetLastError();
  return VLS_ERR_TIMEOUT;
}

#ifdef VLS_TEST_HOOKS
int vls_test_set_fault(int mode) {
  if (mode < VLS_TEST_FAULT_NONE || mode > VLS_TEST_FAULT_DEVICE) return VLS_ERR_ARG;
  g_fault.store(mode, std::memory_order_relaxed);
  return VLS_OK;
}

int vls_test_set_wait_ns(uint64_t ns) {
  g_wait_ns.store(ns, std::memory_order_relaxed);
  return VLS_OK;
}

int vls_test_set_tuning(int64_t fwd_vec_per_cta, int64_t bwd_vec_per_cta, int tc_cta_group) {
  if (fwd_vec_per_cta < 0 || bwd_vec_per_cta < 0 || tc_cta_group < 0 || tc_cta_group > 2) return VLS_ERR_ARG;
  g_fwd_vec.store(fwd_vec_per_cta, std::memory_order_relaxed);
  g_bwd_vec.store(bwd_vec_per_cta, std::memory_order_relaxed);
  g_cta_group.store(tc_cta_group, std::memory_order_relaxed);
  return VLS_OK;
}
#endif

const char* vls_status_string(int status) {
  switch (status) {
    case VLS_OK: return "VLS_OK";
    case VLS_ERR_NULL: return "VLS_ERR_NULL: a required pointer is NULL";
    case VLS_ERR_SHAPE: return "VLS_ERR_SHAPE: bad N, V, row layout, k or n";
    case VLS_ERR_DTYPE: return "VLS_ERR_DTYPE: unsupported dtype";
    case VLS_ERR_CAP: return "VLS_ERR_CAP: cap must be finite and non-negative (softcap calls: positive)";
    case VLS_ERR_DEVICE:
      return "VLS_ERR_DEVICE: pointer not device memory, or pointers/stream on different devices";
    case VLS_ERR_LAUNCH: return "VLS_ERR_LAUNCH: CUDA launch failed";
    case VLS_ERR_ARG: return "VLS_ERR_ARG: bad argument";
    case VLS_ERR_TOO_LARGE: return "VLS_ERR_TOO_LARGE: the call needs more than the no-alloc call's fixed scratch";
    case VLS_ERR_TIMEOUT: return "VLS_ERR_TIMEOUT: a bounded wait in a tensor-core kernel ran out";
    default: return "VLS_ERR_UNKNOWN";
  }
}

int vls_softcap_fwd(const void* x, void* y, int64_t n, vls_dtype dt, float cap, void* stream) {
  if (n < 0) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_softcap_cap(cap)) return e;
  if (n == 0) return VLS_OK;
  if (!x || !y) return VLS_ERR_NULL;
  int dev;
  if (int e = resolve_device({x, y}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  CapArgs a{x, nullptr, 0, y, n, cap, 1.0f / cap, 0};
  a.grid = sm_count(dev);
  return VLS_LAUNCH(launch_softcap_fwd(dt, a, static_cast<cudaStream_t>(stream)));
}

int vls_softcap_bwd(const void* x, const void* gy, vls_dtype gy_dt, void* gx, int64_t n, vls_dtype dt,
                    float cap, void* stream) {
  if (n < 0) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt) || !dtype_ok(gy_dt) || (gy_dt != VLS_F32 && gy_dt != dt)) return VLS_ERR_DTYPE;
  if (int e = check_softcap_cap(cap)) return e;
  if (n == 0) return VLS_OK;
  if (!x || !gy || !gx) return VLS_ERR_NULL;
  int dev;
  if (int e = resolve_device({x, gy, gx}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  CapArgs a{x, gy, gy_dt == VLS_F32 ? 1 : 0, gx, n, cap, 1.0f / cap, 0};
  a.grid = sm_count(dev);
  return VLS_LAUNCH(launch_softcap_bwd(dt, a, static_cast<cudaStream_t>(stream)));
}

int vls_logp_fwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V,
                 const int64_t* ids, int32_t k, int64_t ignore_index, float cap, float* logp,
                 vls_rowstat* stats,
                 void* stream) {
  if (int e = check_rows(N, V)) return e;
  if (k < 1 || k > VLS_MAX_TOPK) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows, V)) return e;
  if (!logits || !ids || !logp || !stats) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({logits, ids, logp, stats}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  a.x = logits;
  a.rx = kernel_rows(*rows);
  a.ids = ids;
  a.k = k;
  a.ignore_index = ignore_index;
  a.logp = logp;
  a.stats_x = stats;
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_logp(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_logp_bwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V,
                 const int64_t* ids, int32_t k, int64_t ignore_index, float cap, const float* g,
                 const vls_rowstat* stats,
                 void* dlogits, void* stream) {
  if (int e = check_rows(N, V)) return e;
  if (k < 1 || k > VLS_MAX_TOPK) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows, V)) return e;
  if (!logits || !ids || !g || !stats || !dlogits) return VLS_ERR_NULL;
  BwdArgs a = bwd_args(N, V, k, cap);
  if (N * a.chunks > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({logits, ids, g, stats, dlogits}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  widen_bwd(a, sm_count(dev));
  a.x = logits;
  a.rx = kernel_rows(*rows);
  a.ids = ids;
  a.ignore_index = ignore_index;
  a.g = g;
  a.stats_x = stats;
  a.dx = dlogits;
  return VLS_LAUNCH(launch_bwd_logp(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_entropy_fwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V, float cap,
                    float* H, vls_rowstat* stats, void* stream) {
  if (int e = check_rows(N, V)) return e;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows, V)) return e;
  if (!logits || !H || !stats) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({logits, H, stats}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  a.x = logits;
  a.rx = kernel_rows(*rows);
  a.out = H;
  a.stats_x = stats;
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_entropy(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_entropy_bwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V, float cap,
                    const float* g, const float* H, const vls_rowstat* stats, void* dlogits,
                    void* stream) {
  if (int e = check_rows(N, V)) return e;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows, V)) return e;
  if (!logits || !g || !H || !stats || !dlogits) return VLS_ERR_NULL;
  BwdArgs a = bwd_args(N, V, 1, cap);
  if (N * a.chunks > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({logits, g, H, stats, dlogits}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  widen_bwd(a, sm_count(dev));
  a.x = logits;
  a.rx = kernel_rows(*rows);
  a.g = g;
  a.fout = H;
  a.stats_x = stats;
  a.dx = dlogits;
  return VLS_LAUNCH(launch_bwd_entropy(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_kl_fwd(const void* pa, const vls_rows* rows_a, const void* pb, const vls_rows* rows_b,
               vls_dtype dt, int64_t N, int64_t V,
               vls_kl_dir dir, float cap, float* kl, vls_rowstat* stats_a, vls_rowstat* stats_b,
               void* stream) {
  if (int e = check_rows(N, V)) return e;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (dir != VLS_KL_REVERSE && dir != VLS_KL_FORWARD) return VLS_ERR_ARG;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows_a, V)) return e;
  if (int e = check_layout(rows_b, V)) return e;
  if (!pa || !pb || !kl || !stats_a || !stats_b) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({pa, pb, kl, stats_a, stats_b}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  // the sweep's first argument is the distribution the expectation is over
  const bool rev = dir == VLS_KL_REVERSE;
  a.x = rev ? pa : pb;
  a.rx = kernel_rows(rev ? *rows_a : *rows_b);
  a.y = rev ? pb : pa;
  a.ry = kernel_rows(rev ? *rows_b : *rows_a);
  a.stats_x = rev ? stats_a : stats_b;
  a.stats_y = rev ? stats_b : stats_a;
  a.out = kl;
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_kl(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_kl_bwd(const void* pa, const vls_rows* rows_a, const void* pb, const vls_rows* rows_b,
               vls_dtype dt, int64_t N, int64_t V,
               vls_kl_dir dir, float cap, const float* g, const float* kl, const vls_rowstat* stats_a,
               const vls_rowstat* stats_b, void* da, void* stream) {
  if (int e = check_rows(N, V)) return e;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (dir != VLS_KL_REVERSE && dir != VLS_KL_FORWARD) return VLS_ERR_ARG;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows_a, V)) return e;
  if (int e = check_layout(rows_b, V)) return e;
  if (!pa || !pb || !g || !kl || !stats_a || !stats_b || !da) return VLS_ERR_NULL;
  BwdArgs a = bwd_args(N, V, 1, cap);
  if (N * a.chunks > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({pa, pb, g, kl, stats_a, stats_b, da}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  widen_bwd(a, sm_count(dev));
  a.x = pa;
  a.rx = kernel_rows(*rows_a);
  a.y = pb;
  a.ry = kernel_rows(*rows_b);
  a.g = g;
  a.fout = kl;
  a.stats_x = stats_a;
  a.stats_y = stats_b;
  a.dx = da;
  return VLS_LAUNCH(
      launch_bwd_kl(dir == VLS_KL_REVERSE, dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}


// ---------------------------------------------------------------------------
// fused statistics
// ---------------------------------------------------------------------------

int vls_fused_fwd(const void* pa, const vls_rows* rows_a, const void* pb, const vls_rows* rows_b,
                  vls_dtype dt, int64_t N, int64_t V,
                  const int64_t* ids, int32_t k, int64_t ignore_index, vls_kl_dir dir, float cap, float* logp,
                  float* H, float* kl, vls_rowstat* stats_a, vls_rowstat* stats_b, void* stream) {
  if (int e = check_rows(N, V)) return e;
  const bool want_kl = kl != nullptr;
  if (logp && (k < 1 || k > VLS_MAX_TOPK)) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (want_kl && dir != VLS_KL_REVERSE && dir != VLS_KL_FORWARD) return VLS_ERR_ARG;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows_a, V)) return e;
  if (want_kl) {
    if (int e = check_layout(rows_b, V)) return e;
  }
  if (!pa || !stats_a || (logp && !ids) || (want_kl && (!pb || !stats_b))) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({pa, want_kl ? pb : nullptr, logp ? ids : nullptr, logp, H, kl, stats_a,
                              want_kl ? stats_b : nullptr},
                             stream, &dev))
    return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  a.x = pa;
  a.rx = kernel_rows(*rows_a);
  a.y = want_kl ? pb : nullptr;
  if (want_kl) a.ry = kernel_rows(*rows_b);
  a.ids = ids;
  a.k = logp ? k : 0;
  a.ignore_index = ignore_index;
  a.logp = logp;
  a.h = H;
  a.kl = kl;
  a.stats_x = stats_a;
  a.stats_y = stats_b;
  const FusedKl fk = !want_kl ? kFusedNoKl : (dir == VLS_KL_REVERSE ? kFusedKlReverse : kFusedKlForward);
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_fused(fk, dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_fused_bwd(const void* pa, const vls_rows* rows_a, const void* pb, const vls_rows* rows_b,
                  vls_dtype dt, int64_t N, int64_t V,
                  const int64_t* ids, int32_t k, int64_t ignore_index, vls_kl_dir dir, float cap,
                  const float* g_logp, const float* g_H, const float* g_kl, const float* H, const float* kl,
                  const vls_rowstat* stats_a, const vls_rowstat* stats_b, void* da, void* stream) {
  if (int e = check_rows(N, V)) return e;
  const bool want_kl = g_kl != nullptr;
  if (g_logp && (k < 1 || k > VLS_MAX_TOPK)) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (!g_logp && !g_H && !g_kl) return VLS_ERR_ARG;
  if (want_kl && dir != VLS_KL_REVERSE && dir != VLS_KL_FORWARD) return VLS_ERR_ARG;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (int e = check_layout(rows_a, V)) return e;
  if (want_kl) {
    if (int e = check_layout(rows_b, V)) return e;
  }
  if (!pa || !stats_a || !da || (g_logp && !ids) || (g_H && !H) || (want_kl && (!pb || !kl || !stats_b)))
    return VLS_ERR_NULL;
  BwdArgs a = bwd_args(N, V, g_logp ? k : 1, cap);
  if (N * a.chunks > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({pa, want_kl ? pb : nullptr, g_logp ? ids : nullptr, g_logp, g_H, g_kl, H, kl,
                              stats_a, want_kl ? stats_b : nullptr, da},
                             stream, &dev))
    return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  widen_bwd(a, sm_count(dev));
  a.x = pa;
  a.rx = kernel_rows(*rows_a);
  a.y = want_kl ? pb : nullptr;
  if (want_kl) a.ry = kernel_rows(*rows_b);
  a.ids = ids;
  a.k = g_logp ? k : 1;
  a.ignore_index = ignore_index;
  a.g = g_logp;
  a.g_h = g_H;
  a.g_kl = g_kl;
  a.h = H;
  a.kl = kl;
  a.stats_x = stats_a;
  a.stats_y = stats_b;
  a.dx = da;
  const FusedKl fk = !want_kl ? kFusedNoKl : (dir == VLS_KL_REVERSE ? kFusedKlReverse : kFusedKlForward);
  return VLS_LAUNCH(launch_bwd_fused(fk, dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// vocabulary-parallel split phase
// ---------------------------------------------------------------------------

int vls_logp_partial(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V_shard,
                     int64_t vocab_offset, int64_t V_total, const int64_t* ids, int32_t k,
                     int64_t ignore_index, float cap, vls_partial* part, float* zt, void* stream) {
  if (int e = check_shard(N, V_shard, vocab_offset, V_total)) return e;
  if (k < 1 || k > VLS_MAX_TOPK) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (V_shard > 0) {
    if (int e = check_layout(rows, V_shard)) return e;
  }
  if ((!logits && V_shard > 0) || !ids || !part || !zt) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V_shard, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({V_shard > 0 ? logits : nullptr, ids, part, zt}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  a.x = logits;
  if (V_shard > 0) a.rx = kernel_rows(*rows);
  a.ids = ids;
  a.k = k;
  a.ignore_index = ignore_index;
  a.vocab_offset = vocab_offset;
  a.vocab_total = V_total;
  a.part = part;
  a.zt = zt;
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_logp(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_logp_combine(const vls_partial* parts, const float* zt, int32_t R, int64_t N, const int64_t* ids,
                     int32_t k, int64_t V_total, int64_t ignore_index, float cap, float* logp,
                     vls_rowstat* stats, void* stream) {
  if (N < 0 || R < 1 || V_total < 1 || k < 1 || k > VLS_MAX_TOPK) return VLS_ERR_SHAPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (!parts || !zt || !ids || !logp || !stats) return VLS_ERR_NULL;
  int dev;
  if (int e = resolve_device({parts, zt, ids, logp, stats}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  CombineArgs a;
  std::memset(&a, 0, sizeof(a));
  a.parts = parts;
  a.zt = zt;
  a.R = R;
  a.rows = N;
  a.ids = ids;
  a.k = k;
  a.vocab_total = V_total;
  a.ignore_index = ignore_index;
  a.cap = cap;
  a.logp = logp;
  a.stats_x = stats;
  return VLS_LAUNCH(launch_combine(kFwdLogp, a, static_cast<cudaStream_t>(stream)));
}

int vls_logp_bwd_shard(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V_shard,
                       int64_t vocab_offset, int64_t V_total, const int64_t* ids, int32_t k,
                       int64_t ignore_index, float cap, const float* g, const vls_rowstat* stats,
                       void* dlogits, void* stream) {
  if (int e = check_shard(N, V_shard, vocab_offset, V_total)) return e;
  if (k < 1 || k > VLS_MAX_TOPK) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0 || V_shard == 0) return VLS_OK;
  if (int e = check_layout(rows, V_shard)) return e;
  if (!logits || !ids || !g || !stats || !dlogits) return VLS_ERR_NULL;
  BwdArgs a = bwd_args(N, V_shard, k, cap);
  if (N * a.chunks > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({logits, ids, g, stats, dlogits}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  widen_bwd(a, sm_count(dev));
  a.x = logits;
  a.rx = kernel_rows(*rows);
  a.ids = ids;
  a.ignore_index = ignore_index;
  a.g = g;
  a.stats_x = stats;
  a.dx = dlogits;
  a.vocab_offset = vocab_offset;
  a.vocab_total = V_total;
  return VLS_LAUNCH(launch_bwd_logp(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_entropy_partial(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V_shard,
                        float cap,
                        vls_partial* part, void* stream) {
  if (N < 0 || V_shard < 0) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (V_shard > 0) {
    if (int e = check_layout(rows, V_shard)) return e;
  }
  if ((!logits && V_shard > 0) || !part) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V_shard, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({V_shard > 0 ? logits : nullptr, part}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  a.x = logits;
  if (V_shard > 0) a.rx = kernel_rows(*rows);
  a.part = part;
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_entropy(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_entropy_combine(const vls_partial* parts, int32_t R, int64_t N, float* H, vls_rowstat* stats,
                        void* stream) {
  if (N < 0 || R < 1) return VLS_ERR_SHAPE;
  if (N == 0) return VLS_OK;
  if (!parts || !H || !stats) return VLS_ERR_NULL;
  int dev;
  if (int e = resolve_device({parts, H, stats}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  CombineArgs a;
  std::memset(&a, 0, sizeof(a));
  a.parts = parts;
  a.R = R;
  a.rows = N;
  a.out = H;
  a.stats_x = stats;
  return VLS_LAUNCH(launch_combine(kFwdEntropy, a, static_cast<cudaStream_t>(stream)));
}

int vls_kl_partial(const void* pa, const vls_rows* rows_a, const void* pb, const vls_rows* rows_b,
                   vls_dtype dt, int64_t N,
                   int64_t V_shard, vls_kl_dir dir, float cap, vls_partial* part, void* stream) {
  if (N < 0 || V_shard < 0) return VLS_ERR_SHAPE;
  if (!dtype_ok(dt)) return VLS_ERR_DTYPE;
  if (dir != VLS_KL_REVERSE && dir != VLS_KL_FORWARD) return VLS_ERR_ARG;
  if (int e = check_row_cap(cap)) return e;
  if (N == 0) return VLS_OK;
  if (V_shard > 0) {
    if (int e = check_layout(rows_a, V_shard)) return e;
    if (int e = check_layout(rows_b, V_shard)) return e;
  }
  if (((!pa || !pb) && V_shard > 0) || !part) return VLS_ERR_NULL;
  FwdArgs a = fwd_args(N, V_shard, cap);
  if (N * a.cluster > kMaxGrid) return VLS_ERR_SHAPE;
  int dev;
  if (int e = resolve_device({V_shard > 0 ? pa : nullptr, V_shard > 0 ? pb : nullptr, part}, stream, &dev))
    return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  const bool rev = dir == VLS_KL_REVERSE;
  a.x = rev ? pa : pb;
  a.y = rev ? pb : pa;
  if (V_shard > 0) {
    a.rx = kernel_rows(rev ? *rows_a : *rows_b);
    a.ry = kernel_rows(rev ? *rows_b : *rows_a);
  }
  a.part = part;
  few_rows_prefetch(a, dt, dev);
  return VLS_LAUNCH(launch_fwd_kl(dt, cap > 0.0f, a, static_cast<cudaStream_t>(stream)));
}

int vls_kl_combine(const vls_partial* parts, int32_t R, int64_t N, vls_kl_dir dir, float* kl,
                   vls_rowstat* stats_a, vls_rowstat* stats_b, void* stream) {
  if (N < 0 || R < 1) return VLS_ERR_SHAPE;
  if (dir != VLS_KL_REVERSE && dir != VLS_KL_FORWARD) return VLS_ERR_ARG;
  if (N == 0) return VLS_OK;
  if (!parts || !kl || !stats_a || !stats_b) return VLS_ERR_NULL;
  int dev;
  if (int e = resolve_device({parts, kl, stats_a, stats_b}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  CombineArgs a;
  std::memset(&a, 0, sizeof(a));
  a.parts = parts;
  a.R = R;
  a.rows = N;
  a.out = kl;
  const bool rev = dir == VLS_KL_REVERSE;
  a.stats_x = rev ? stats_a : stats_b;
  a.stats_y = rev ? stats_b : stats_a;
  return VLS_LAUNCH(launch_combine(kFwdKl, a, static_cast<cudaStream_t>(stream)));
}

// ---------------------------------------------------------------------------
// fused linear head + logprobs
// ---------------------------------------------------------------------------

// TMA coordinates are 32-bit and a tile's last coordinate runs up to 511
// past the end of its matrix
constexpr int64_t kMaxLinear = kMaxGrid - 511;

int64_t vls_linear_logp_chunks(int64_t V) { return V < 1 ? -1 : linear_chunks(V); }

int vls_linear_logp_partial(const void* h, int64_t ldh, const void* W, int64_t ldw, vls_dtype dt, int64_t N,
                            int64_t D, int64_t V, const int64_t* ids, int32_t k, int64_t ignore_index,
                            vls_partial* part, float* zt, uint32_t* status, void* stream) {
  if (N < 0 || D < 1 || V < 1 || ldh < D || ldw < D || k < 1 || k > VLS_LINEAR_MAX_TOPK) return VLS_ERR_SHAPE;
  if (N > kMaxLinear || V > kMaxLinear || D > kMaxLinear) return VLS_ERR_SHAPE;
  if (dt != VLS_BF16 && dt != VLS_F16) return VLS_ERR_DTYPE;
  if (N == 0) return VLS_OK;
  if (!h || !W || !ids || !part || !zt || !status) return VLS_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(W)) & 15u) return VLS_ERR_ARG;
  if ((ldh % 8) || (ldw % 8)) return VLS_ERR_ARG;
  int dev;
  if (int e = resolve_device({h, W, ids, part, zt, status}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  LinearArgs a{h, ldh, W, ldw, dt, N, D, V, ids, k, ignore_index, part, zt, status, tc_sticky_status(), tc_wait_ns()};
  return VLS_LAUNCH(launch_linear_logp(a, sm_count(dev), static_cast<cudaStream_t>(stream)));
}

int64_t vls_linear_logp_bwd_workspace(int64_t N, int64_t D, int64_t V) {
  if (N < 0 || D < 1 || V < 1 || N > kMaxLinear || V > kMaxLinear || D > kMaxLinear) return -1;
  return static_cast<int64_t>(linear_bwd_workspace(N, D, V));
}

int vls_linear_logp_bwd(const void* h, int64_t ldh, const void* W, int64_t ldw, vls_dtype dt, int64_t N, int64_t D,
                        int64_t V, const int64_t* ids, int32_t k, int64_t ignore_index, const float* g,
                        const vls_rowstat* stats, void* dh, void* dW, void* workspace, int64_t workspace_bytes,
                        uint32_t* status, void* stream) {
  if (N < 0 || D < 1 || V < 1 || ldh < D || ldw < D || k < 1 || k > VLS_LINEAR_MAX_TOPK) return VLS_ERR_SHAPE;
  if (N > kMaxLinear || V > kMaxLinear || D > kMaxLinear) return VLS_ERR_SHAPE;
  if (dt != VLS_BF16 && dt != VLS_F16) return VLS_ERR_DTYPE;
  if (N == 0) return VLS_OK;
  if (!h || !W || !ids || !g || !stats || !dh || !dW || !workspace || !status) return VLS_ERR_NULL;
  if (workspace_bytes < vls_linear_logp_bwd_workspace(N, D, V)) return VLS_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(h) | reinterpret_cast<uintptr_t>(W)) & 15u) return VLS_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return VLS_ERR_ARG;
  if ((ldh % 8) || (ldw % 8)) return VLS_ERR_ARG;
  int dev;
  if (int e = resolve_device({h, W, ids, g, stats, dh, dW, workspace, status}, stream, &dev)) return e;
  DeviceGuard guard;
  if (int e = guard.enter(dev)) return e;
  LinearBwdArgs a{h, ldh, W, ldw, dt, N, D, V, ids, k, ignore_index, g, stats, dh, dW, workspace, status,
                  tc_sticky_status(), tc_wait_ns()};
  return VLS_LAUNCH(launch_linear_logp_bwd(a, sm_count(dev), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
