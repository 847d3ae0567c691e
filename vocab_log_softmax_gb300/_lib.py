"""Loads libvls.so and declares its C ABI (include/vls.h) for ctypes.

There is no fallback: if the library is missing or cannot be loaded, every
entry point raises.  Build it with ``python -m vocab_log_softmax_gb300.build``
(``__graft_entry__.build()`` does the same).

``load_test()`` loads the test build, libvls_test.so (the same ABI plus the
hooks of include/vls_test.h), and ``using(lib)`` routes the ``binding``
functions through it for the duration of a ``with`` block; tests use them to
inject failures.  Nothing else does.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libvls.so")
TEST_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libvls_test.so")

VLS_F32 = 0
VLS_BF16 = 1
VLS_F16 = 2
VLS_KL_REVERSE = 0
VLS_KL_FORWARD = 1
VLS_MAX_TOPK = 1024

STATUS = {
    0: "VLS_OK",
    1: "VLS_ERR_NULL",
    2: "VLS_ERR_SHAPE",
    3: "VLS_ERR_DTYPE",
    4: "VLS_ERR_CAP",
    5: "VLS_ERR_DEVICE",
    6: "VLS_ERR_LAUNCH",
    7: "VLS_ERR_ARG",
    8: "VLS_ERR_TOO_LARGE",
    9: "VLS_ERR_TIMEOUT",
}
VLS_ERR_LAUNCH = 6
VLS_ERR_TIMEOUT = 9

# include/vls_test.h
VLS_TEST_FAULT_NONE = 0
VLS_TEST_FAULT_LAUNCH = 1
VLS_TEST_FAULT_VALIDATE = 2
VLS_TEST_FAULT_DEVICE = 3

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_int = ctypes.c_int
_f = ctypes.c_float


class VlsRows(ctypes.Structure):
    """vls_rows: row r of an operand starts (r // group) * ld_group + (r % group) * ld
    elements after its base pointer (group 0: r * ld)."""

    _fields_ = [("ld", ctypes.c_int64), ("group", ctypes.c_int64), ("ld_group", ctypes.c_int64)]


def rows(ld: int, group: int = 0, ld_group: int = 0) -> VlsRows:
    return VlsRows(ld, group, ld_group)


_r = ctypes.POINTER(VlsRows)

# name -> argument types, in the order of include/vls.h
SIGNATURES = {
    "vls_softcap_fwd": [_p, _p, _i64, _int, _f, _p],
    "vls_softcap_bwd": [_p, _p, _int, _p, _i64, _int, _f, _p],
    "vls_logp_fwd": [_p, _r, _int, _i64, _i64, _p, _i32, _i64, _f, _p, _p, _p],
    "vls_logp_bwd": [_p, _r, _int, _i64, _i64, _p, _i32, _i64, _f, _p, _p, _p, _p],
    "vls_entropy_fwd": [_p, _r, _int, _i64, _i64, _f, _p, _p, _p],
    "vls_entropy_bwd": [_p, _r, _int, _i64, _i64, _f, _p, _p, _p, _p, _p],
    "vls_kl_fwd": [_p, _r, _p, _r, _int, _i64, _i64, _int, _f, _p, _p, _p, _p],
    "vls_kl_bwd": [_p, _r, _p, _r, _int, _i64, _i64, _int, _f, _p, _p, _p, _p, _p, _p],
    "vls_fused_fwd": [_p, _r, _p, _r, _int, _i64, _i64, _p, _i32, _i64, _int, _f, _p, _p, _p, _p, _p, _p],
    "vls_fused_bwd": [_p, _r, _p, _r, _int, _i64, _i64, _p, _i32, _i64, _int, _f, _p, _p, _p, _p, _p, _p, _p,
                      _p, _p],
    "vls_logp_partial": [_p, _r, _int, _i64, _i64, _i64, _i64, _p, _i32, _i64, _f, _p, _p, _p],
    "vls_logp_combine": [_p, _p, _i32, _i64, _p, _i32, _i64, _i64, _f, _p, _p, _p],
    "vls_logp_bwd_shard": [_p, _r, _int, _i64, _i64, _i64, _i64, _p, _i32, _i64, _f, _p, _p, _p, _p],
    "vls_entropy_partial": [_p, _r, _int, _i64, _i64, _f, _p, _p],
    "vls_entropy_combine": [_p, _i32, _i64, _p, _p, _p],
    "vls_kl_partial": [_p, _r, _p, _r, _int, _i64, _i64, _int, _f, _p, _p],
    "vls_kl_combine": [_p, _i32, _i64, _int, _p, _p, _p, _p],
    "vls_linear_logp_chunks": [_i64],
    "vls_linear_logp_partial": [_p, _i64, _p, _i64, _int, _i64, _i64, _i64, _p, _i32, _i64, _p, _p, _p, _p],
    "vls_linear_logp_bwd_workspace": [_i64, _i64, _i64],
    "vls_linear_logp_bwd": [_p, _i64, _p, _i64, _int, _i64, _i64, _i64, _p, _i32, _i64, _p, _p, _p, _p, _p, _i64,
                            _p, _p],
    "vls_linear_logp_fwd_noalloc": [_p, _i64, _p, _i64, _int, _i64, _i64, _i64, _p, _i32, _i64, _p, _p, _p, _p],
    "vls_status_string": [_int],
    "vls_check_device_error": [],
    "vls_version": [],
}

# the test build's hooks (include/vls_test.h)
TEST_SIGNATURES = {
    "vls_test_set_fault": [_int],
    "vls_test_set_wait_ns": [ctypes.c_uint64],
    "vls_test_set_tuning": [_i64, _i64, _int],
}

RESTYPES = {"vls_status_string": ctypes.c_char_p, "vls_linear_logp_chunks": ctypes.c_int64,
            "vls_linear_logp_bwd_workspace": ctypes.c_int64}
VLS_LINEAR_MAX_TOPK = 16

_lib = None


class VlsError(RuntimeError):
    """A libvls call returned a status other than VLS_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


class VlsArgumentError(VlsError, ValueError):
    """A libvls call rejected its arguments (shape, dtype, cap, NULL pointer)."""


class VlsDeviceError(VlsError):
    """Work already enqueued failed on the GPU: a bounded wait in a
    tensor-core kernel ran out (VLS_ERR_TIMEOUT), whose outputs are then
    invalid."""


_test_lib = None


def _declare(lib: ctypes.CDLL, signatures: dict) -> None:
    for name, argtypes in signatures.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = RESTYPES.get(name, ctypes.c_int)


def load() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libvls.so not found at {LIB_PATH}; build it with "
            "`python -m vocab_log_softmax_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(LIB_PATH)
    _declare(lib, SIGNATURES)
    _lib = lib
    return lib


def load_test() -> ctypes.CDLL:
    """The test build, libvls_test.so (loaded once): the ABI of libvls.so plus
    the hooks of include/vls_test.h."""
    global _test_lib
    if _test_lib is not None:
        return _test_lib
    if not os.path.exists(TEST_LIB_PATH):
        raise RuntimeError(f"libvls_test.so not found at {TEST_LIB_PATH}; build it with "
                           "`python -m vocab_log_softmax_gb300.build`")
    lib = ctypes.CDLL(TEST_LIB_PATH)
    _declare(lib, SIGNATURES)
    _declare(lib, TEST_SIGNATURES)
    _test_lib = lib
    return lib


@contextlib.contextmanager
def using(lib: ctypes.CDLL):
    """Routes every ``binding`` call through `lib` inside the block."""
    global _lib
    prev = load()
    _lib = lib
    try:
        yield lib
    finally:
        _lib = prev


def check(fn: str, status: int) -> None:
    if status == 0:
        return
    if status in (1, 2, 3, 4, 7, 8):
        raise VlsArgumentError(fn, status)
    if status == VLS_ERR_TIMEOUT:
        raise VlsDeviceError(fn, status)
    raise VlsError(fn, status)
