// Internal declarations shared by the C-ABI layer (api.cpp) and the kernel
// translation units.  Nothing here is part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "vls.h"

namespace vls {

// Statistic computed by the one-read forward sweep.
enum FwdOp { kFwdLogp = 0, kFwdEntropy = 1, kFwdKl = 2, kFwdFused = 3 };
// Gradient map applied by the backward sweep.
enum BwdOp { kBwdLogp = 0, kBwdEntropy = 1, kBwdKlReverse = 2, kBwdKlForward = 3, kBwdFused = 4 };
// KL term of the fused sweeps
enum FusedKl { kFusedNoKl = 0, kFusedKlReverse = 1, kFusedKlForward = 2 };

// Threads per CTA of the row kernels.  Each thread owns whole 8-column
// vectors; the reduction tree (lanes, then warps, then cluster ranks) is a
// function of this constant and of the cluster size, never of N.
constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
// Threads per CTA of the forward sweep (its reduction tree: lanes, then the
// kFwdWarps warps, then cluster ranks).
#ifndef VLS_FWD_THREADS
#define VLS_FWD_THREADS 256
#endif
constexpr int kFwdThreads = VLS_FWD_THREADS;
constexpr int kFwdWarps = kFwdThreads / 32;
static_assert(kFwdThreads == 256 || kFwdThreads == 512 || kFwdThreads == 1024, "forward CTA width");
// Resident CTAs per SM the softcapped maps (capped backward, standalone
// softcap) are compiled for; their software-pipelined loops need more
// registers than the plain maps (6 CTAs, 40 registers).
#ifndef VLS_CAP_MIN_BLOCKS
#define VLS_CAP_MIN_BLOCKS 5
#endif
constexpr int kCapMinBlocks = VLS_CAP_MIN_BLOCKS;
// Vectors each thread loads before using any of them (memory-level
// parallelism).  Changing it does not change results: every thread still
// visits its vectors in increasing order.
constexpr int kUnroll = 4;
constexpr int kMaxCluster = 8;
// Nanoseconds one protocol wait of a tensor-core kernel may take before the
// kernel gives up (a legitimate wait lasts microseconds).
constexpr uint64_t kTcWaitNs = 4000000000ull;

struct FwdArgs {
  // logits (logp / entropy), or the first KL argument: the distribution the
  // expectation is taken over (a for reverse KL, b for forward KL)
  const void* x;
  vls_rows rx;
  // second KL argument (KL only)
  const void* y;
  vls_rows ry;
  int64_t rows;
  int64_t vocab;
  float cap;   // 0 = no softcap
  float rcap;  // 1/cap rounded once (0 when cap == 0)
  // logp
  const int64_t* ids;
  int32_t k;
  int64_t ignore_index;
  float* logp;
  // entropy H or KL value per row
  float* out;
  // per-row stats of x and (KL) of y
  vls_rowstat* stats_x;
  vls_rowstat* stats_y;
  // launch geometry: CTAs per row (= cluster size) and 8-column vectors per CTA
  int cluster;
  int64_t vec_per_cta;
  // vocabulary-parallel partial mode (part != nullptr): the rows hold the
  // columns [vocab_offset, vocab_offset + vocab) of a vocab_total-column
  // vocabulary; the kernel writes its per-row state to part and (logp) the
  // raw logits of the owned target ids to zt instead of finalising
  int64_t vocab_offset;
  int64_t vocab_total;
  vls_partial* part;
  float* zt;
  // fused sweep: entropy and KL outputs (either may be null)
  float* h;
  float* kl;
  // few rows: every CTA first asks L2 for its whole run (changes no result)
  int prefetch;
};

struct BwdArgs {
  const void* x;  // logits / policy a
  vls_rows rx;
  const void* y;  // reference b (KL only)
  vls_rows ry;
  int64_t rows;
  int64_t vocab;
  float cap;
  float rcap;
  const int64_t* ids;
  int32_t k;
  int64_t ignore_index;
  const float* g;      // upstream gradient: [N, k] (logp) or [N]
  const float* fout;   // forward value per row: H (entropy) or KL
  const vls_rowstat* stats_x;
  const vls_rowstat* stats_y;
  void* dx;            // [N, V] contiguous gradient, dtype of x
  int chunks;          // CTAs per row
  int64_t vec_per_cta;
  // logp over a vocabulary shard: ids are global columns, valid against
  // vocab_total; this shard holds [vocab_offset, vocab_offset + vocab)
  int64_t vocab_offset;
  int64_t vocab_total;
  // fused backward: upstream gradients (null = term left out) and the
  // forward's H and KL
  const float* g_h;
  const float* g_kl;
  const float* h;
  const float* kl;
};

struct CombineArgs {
  const vls_partial* parts;  // [R, N]
  const float* zt;           // logp: [R, N, k]
  int32_t R;
  int64_t rows;
  const int64_t* ids;
  int32_t k;
  int64_t vocab_total;
  int64_t ignore_index;
  float cap;
  float* logp;
  float* out;                // H or KL
  vls_rowstat* stats_x;
  vls_rowstat* stats_y;      // KL: stats of the second argument
};

struct CapArgs {
  const void* x;
  const void* gy;   // backward only
  int gy_f32;       // gy is fp32 (else the dtype of x)
  void* out;        // y (forward) or gx (backward)
  int64_t n;
  float cap;
  float rcap;
  int grid;         // the SM count on entry to the launcher, the grid size after
};

// Fused linear head + logprobs (tcgen05): vocabulary chunks of
// kLinChunkTiles tiles of 256 columns each give one vls_partial per row.
constexpr int kLinChunkTiles = 8;
constexpr int kLinMaxTopk = VLS_LINEAR_MAX_TOPK;

struct LinearArgs {
  const void* h;       // [N, D], row stride ldh
  int64_t ldh;
  const void* W;       // [V, D], row stride ldw
  int64_t ldw;
  vls_dtype dt;        // VLS_BF16 or VLS_F16
  int64_t N, D, V;
  const int64_t* ids;  // [N, k]
  int32_t k;
  int64_t ignore_index;
  vls_partial* part;   // [S, N]
  float* zt;           // [S, N, k]
  uint32_t* status;    // the caller's status word
  uint32_t* sticky;    // the library's status word on this device (tc_sticky_status)
  uint64_t wait_ns;    // limit of one protocol wait (tc_wait_ns)
};

int64_t linear_chunks(int64_t V);

struct LinearBwdArgs {
  const void* h;
  int64_t ldh;
  const void* W;
  int64_t ldw;
  vls_dtype dt;
  int64_t N, D, V;
  const int64_t* ids;        // [N, k]
  int32_t k;
  int64_t ignore_index;
  const float* g;            // [N, k]
  const vls_rowstat* stats;  // [N], from the forward
  void* dh;                  // [N, D] contiguous, dtype dt
  void* dW;                  // [V, D] contiguous, dtype dt
  void* workspace;           // linear_bwd_workspace(N, D, V) bytes, 256-byte aligned
  uint32_t* status;
  uint32_t* sticky;
  uint64_t wait_ns;
};

size_t linear_bwd_workspace(int64_t N, int64_t D, int64_t V);

// Defined by the C layer (api.cu): the address of the library's device
// status word on the current device (null if it cannot be had), the limit of
// one protocol wait in the tensor-core kernels, and their CTA-group form.
uint32_t* tc_sticky_status();
// The device a call whose first input pointer is p launches on: p's device,
// or the current device while `stream` is being captured (as every call of
// the C layer chooses it); VLS_ERR_DEVICE when p is not device memory.
int launch_device(const void* p, void* stream, int* dev);
uint64_t tc_wait_ns();
namespace tcg {
int cta_group();
}

// Launchers: one per kernel family, dispatching on dtype and softcap.  They
// return a cudaError_t of the launch.
cudaError_t launch_fwd_logp(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_fwd_entropy(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_fwd_kl(vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_logp(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_entropy(vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_kl(bool reverse, vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_combine(FwdOp op, const CombineArgs& a, cudaStream_t s);
cudaError_t launch_fwd_fused(FusedKl kl, vls_dtype dt, bool cap, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_fused(FusedKl kl, vls_dtype dt, bool cap, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_softcap_fwd(vls_dtype dt, const CapArgs& a, cudaStream_t s);
cudaError_t launch_softcap_bwd(vls_dtype dt, const CapArgs& a, cudaStream_t s);
cudaError_t launch_linear_logp(const LinearArgs& a, int sms, cudaStream_t s);
cudaError_t launch_linear_logp_bwd(const LinearBwdArgs& a, int sms, cudaStream_t s);

}  // namespace vls
