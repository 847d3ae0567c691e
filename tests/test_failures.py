"""Failure paths, exercised without faulting a GPU.

The product library has no way to fail on purpose.  Its test build,
libvls_test.so (include/vls_test.h), adds hooks that make a call fail on the
host exactly where a real failure would surface, and that shorten the limit
of the tensor-core kernels' protocol waits so that a real kernel runs out of
time, takes its abort path and reports it.  A failed call must be visible
to the caller, never replaced by another path ("Final Logit Softcap",
section Backends: a failed launch is not retried with another backend)."""

import ctypes
import math
import os

import numpy as np
import pytest
import torch

import oracle
from vls_compare import assert_fp32_close, bitwise_equal, to_f64
from vocab_log_softmax_gb300 import _lib, build
from vocab_log_softmax_gb300 import binding as B

P = 0x1000   # a non-NULL pointer value; never dereferenced (every path tested on CPU returns first)
BF16 = _lib.VLS_BF16
ARG, DEVICE, LAUNCH = 7, 5, 6


@pytest.fixture(scope="module")
def tlib():
    build.build()
    lib = _lib.load_test()
    yield lib
    lib.vls_test_set_fault(_lib.VLS_TEST_FAULT_NONE)
    lib.vls_test_set_wait_ns(0)
    lib.vls_test_set_tuning(0, 0, 0)


def test_only_the_test_build_exports_hooks(tlib):
    prod = _lib.load()
    for name in _lib.TEST_SIGNATURES:
        assert hasattr(tlib, name)
        with pytest.raises(AttributeError):
            getattr(prod, name)


def test_hooks_reject_bad_settings(tlib):
    assert tlib.vls_test_set_fault(4) == ARG and tlib.vls_test_set_fault(-1) == ARG
    assert tlib.vls_test_set_tuning(-1, 0, 0) == ARG and tlib.vls_test_set_tuning(0, 0, 3) == ARG
    assert tlib.vls_test_set_fault(0) == 0 and tlib.vls_test_set_tuning(0, 0, 0) == 0


@pytest.mark.parametrize("mode,code", [(_lib.VLS_TEST_FAULT_VALIDATE, ARG), (_lib.VLS_TEST_FAULT_DEVICE, DEVICE)])
def test_injected_check_failures_come_back_before_any_cuda_call(tlib, mode, code):
    """Valid arguments reach the device check, where the injected failure
    returns first: every family of calls reports it (runs on CPU hosts)."""
    R = _lib.rows
    assert tlib.vls_test_set_fault(mode) == 0
    try:
        assert tlib.vls_logp_fwd(P, R(10), BF16, 4, 10, P, 1, -100, 0.0, P, P, None) == code
        assert tlib.vls_entropy_bwd(P, R(10), BF16, 4, 10, 0.0, P, P, P, P, None) == code
        assert tlib.vls_kl_fwd(P, R(10), P, R(10), BF16, 4, 10, 0, 0.0, P, P, P, None) == code
        assert tlib.vls_softcap_fwd(P, P, 8, BF16, 30.0, None) == code
        assert tlib.vls_logp_combine(P, P, 2, 4, P, 1, 10, -100, 0.0, P, P, None) == code
        assert tlib.vls_linear_logp_partial(P, 64, P, 64, BF16, 4, 64, 100, P, 1, -100, P, P, P, None) == code
        assert tlib.vls_linear_logp_fwd_noalloc(P, 64, P, 64, BF16, 4, 64, 100, P, 1, -100, P, P, P, None) == code
        # argument errors still win: they are found first
        assert tlib.vls_logp_fwd(P, R(10), BF16, 4, 10, P, 0, -100, 0.0, P, P, None) == 2
    finally:
        tlib.vls_test_set_fault(_lib.VLS_TEST_FAULT_NONE)


def test_status_codes_map_to_python_exceptions():
    """Argument errors are ValueErrors; device, launch and in-kernel failures
    are RuntimeErrors that are not ValueErrors."""
    for code in (1, 2, 3, 4, 7, 8):
        with pytest.raises(ValueError):
            _lib.check("f", code)
    for code, cls in ((5, _lib.VlsError), (6, _lib.VlsError), (9, _lib.VlsDeviceError)):
        with pytest.raises(cls) as e:
            _lib.check("f", code)
        assert isinstance(e.value, RuntimeError) and not isinstance(e.value, ValueError)
        assert e.value.status == code and _lib.STATUS[code] in str(e.value)


# ---------------------------------------------------------------------------
# on the GPU
# ---------------------------------------------------------------------------

DEV = "cuda"


@pytest.mark.gpu
def test_injected_launch_failure_raises_and_enqueues_nothing(tlib):
    import vocab_log_softmax_gb300 as V
    g = torch.Generator(device=DEV).manual_seed(5)
    x = (3.0 * torch.randn((6, 3001), generator=g, device=DEV)).to(torch.bfloat16)
    ids = torch.randint(0, 3001, (6, 1), generator=g, device=DEV)
    lp = torch.full((6, 1), 7.0, device=DEV)
    st = torch.full((6, 2), 7.0, device=DEV)
    with _lib.using(tlib):
        tlib.vls_test_set_fault(_lib.VLS_TEST_FAULT_LAUNCH)
        try:
            for f in (lambda: B.vls_logp_fwd(x, ids, logp=lp, stats=st),
                      lambda: B.vls_entropy_fwd(x),
                      lambda: B.vls_kl_fwd(x, x),
                      lambda: B.vls_softcap_fwd(x, 30.0),
                      lambda: V.logprobs(x, ids)):
                with pytest.raises(_lib.VlsError) as e:
                    f()
                assert e.value.status == LAUNCH and not isinstance(e.value, ValueError)
            torch.cuda.synchronize()
            assert bool((lp == 7.0).all()) and bool((st == 7.0).all())   # nothing ran
        finally:
            tlib.vls_test_set_fault(_lib.VLS_TEST_FAULT_NONE)
        lp1, st1 = B.vls_logp_fwd(x, ids)
    lp0, st0 = B.vls_logp_fwd(x, ids)   # the product library
    assert bitwise_equal(lp0, lp1) and bitwise_equal(st0, st1)


def _linear_case(n, d, v, seed):
    """Small-integer h and W: every logit is exact in fp32."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    h = torch.randint(-1, 2, (n, d), generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randint(-1, 2, (v, d), generator=g, device=DEV).to(torch.bfloat16)
    ids = torch.randint(0, v, (n, 1), generator=g, device=DEV)
    return h, w, ids


def _expire_and_recover(tlib, form):
    """A real tensor-core kernel whose protocol waits may last only 1 us:
    its first wait for a tile of products (K = 4096 takes far longer) runs
    out, the kernel drains what it has in flight and returns.  The call's
    status word and the library's word report it; the next normal call on
    the same GPU is correct."""
    import vocab_log_softmax_gb300 as V
    h, w, ids = _linear_case(256, 4096, 4096, 11)
    assert tlib.vls_test_set_tuning(0, 0, form) == 0
    try:
        with _lib.using(tlib):
            assert tlib.vls_check_device_error() == 0   # nothing pending from earlier tests
            assert tlib.vls_test_set_wait_ns(1000) == 0
            try:
                _, _, status = B.vls_linear_logp_fwd(h, w, ids)
                torch.cuda.synchronize()                   # the kernels returned
                assert int(status.item()) & 1, "no wait ran out"
                assert tlib.vls_check_device_error() == _lib.VLS_ERR_TIMEOUT
                assert tlib.vls_check_device_error() == 0   # the report was cleared
                with pytest.raises(_lib.VlsDeviceError):
                    B.vls_linear_logp_fwd(h, w, ids, check=True)
                hh = h.detach().clone().requires_grad_(True)
                with pytest.raises(_lib.VlsDeviceError):
                    V.linear_logprobs(hh, w, ids)
                B.vls_linear_logp_fwd(h, w, ids)
                with pytest.raises(_lib.VlsDeviceError):
                    B.vls_check_device_error()
            finally:
                tlib.vls_test_set_wait_ns(0)
            logp, stats, status = B.vls_linear_logp_fwd(h, w, ids, check=True)
            assert tlib.vls_check_device_error() == 0 and int(status.item()) == 0
    finally:
        tlib.vls_test_set_tuning(0, 0, 0)
    ref = oracle.linear_logp_fwd(to_f64(h), to_f64(w), ids.cpu().numpy())
    assert_fp32_close(logp, ref, f"after an expired wait ({form}-SM form)")
    lp0, st0, s0 = B.vls_linear_logp_fwd(h, w, ids, check=True)   # the product library
    assert int(s0.item()) == 0


@pytest.mark.gpu
def test_expired_wait_one_sm_form(tlib):
    _expire_and_recover(tlib, 1)


@pytest.mark.gpu
def test_expired_wait_cta_pairs(tlib):
    """The same on the default form, where both CTAs' loads complete on the
    leader's barriers: after the abort the pair exchanges its issue counts
    and the leader waits for every load of both CTAs before the pair leaves."""
    _expire_and_recover(tlib, 2)
