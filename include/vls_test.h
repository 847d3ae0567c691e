/*
 * vls_test.h -- hooks of the TEST BUILD of libvls.
 *
 * The build makes two libraries from the same sources: lib/libvls.so, the
 * product, and lib/libvls_test.so, compiled with VLS_TEST_HOOKS.  Only the
 * test build exports the calls below; everything else (include/vls.h) is
 * the same in both.  The product library reads no environment variable and
 * has none of these settings: its launch geometry, and with it every result
 * bit, is fixed.
 *
 * The hooks let a test reach error paths without faulting a GPU: a call that
 * fails on the host as if its launch or its argument checks had failed, a
 * tensor-core kernel whose protocol waits run out (so that its abort and
 * drain path runs and reports through the status words), and other launch
 * geometries.  Each setting applies to every later call of the process
 * until it is changed; none is meant to be changed while calls run on other
 * threads.
 */
#ifndef VLS_TEST_H_
#define VLS_TEST_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  VLS_TEST_FAULT_NONE = 0,
  VLS_TEST_FAULT_LAUNCH = 1,   /* every call returns VLS_ERR_LAUNCH in place of its launch
                                  (after its argument checks); nothing is enqueued */
  VLS_TEST_FAULT_VALIDATE = 2, /* every call with valid arguments returns VLS_ERR_ARG at its
                                  device check, before any CUDA call */
  VLS_TEST_FAULT_DEVICE = 3    /* the same with VLS_ERR_DEVICE */
};

/* Selects the injected fault (VLS_TEST_FAULT_*); VLS_ERR_ARG for another mode. */
int vls_test_set_fault(int mode);

/* Limit of one protocol wait in the tensor-core kernels, in nanoseconds;
 * 0 restores the default (4 s).  Waits that drain work already issued keep
 * the default whatever this says. */
int vls_test_set_wait_ns(uint64_t ns);

/* Launch geometry: 8-column vectors per CTA of the forward sweeps (which
 * sets the cluster size for a V, and so the reduction tree and the result
 * bits) and of the backward maps (results do not depend on it), and the
 * tensor-core form (1: one SM per tile, 2: CTA pairs).  0 restores each
 * default (24576, 4096, 2); negative values or a form other than 0, 1, 2
 * return VLS_ERR_ARG. */
int vls_test_set_tuning(int64_t fwd_vec_per_cta, int64_t bwd_vec_per_cta, int tc_cta_group);

#ifdef __cplusplus
}
#endif

#endif /* VLS_TEST_H_ */
