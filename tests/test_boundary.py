"""The C ABI boundary: every symbol include/vls.h declares is exported, and
argument errors come back as status codes without any CUDA call (these run
on CPU-only hosts).  The device-pointer checks need a GPU."""

import ctypes
import math
import os
import re

import pytest

from vocab_log_softmax_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vls.h")

OK, NULL, SHAPE, DTYPE, CAP, DEVICE, LAUNCH, ARG = range(8)
F32, BF16 = 0, 1
P = 0x1000   # a non-NULL pointer value; never dereferenced (errors precede any access)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vls_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_eight_calls():
    names = declared_functions()
    for op in ("softcap", "logp", "entropy", "kl"):
        for d in ("fwd", "bwd"):
            assert f"vls_{op}_{d}" in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.vls_status_string(code).decode().startswith(name)
    assert lib.vls_status_string(99).decode() == "VLS_ERR_UNKNOWN"
    assert lib.vls_version() >= 100


def test_logp_argument_errors(lib):
    f = lib.vls_logp_fwd
    #        logits ld  dt    N  V  ids k  ign  cap  logp stats stream
    assert f(None, 10, BF16, 4, 10, None, 1, -100, 0.0, None, None, None) == NULL
    assert f(P, 10, BF16, -1, 10, P, 1, -100, 0.0, P, P, None) == SHAPE
    assert f(P, 10, BF16, 4, 0, P, 1, -100, 0.0, P, P, None) == SHAPE
    assert f(P, 9, BF16, 4, 10, P, 1, -100, 0.0, P, P, None) == SHAPE       # ld < V
    assert f(P, 10, BF16, 4, 10, P, 0, -100, 0.0, P, P, None) == SHAPE      # k < 1
    assert f(P, 10, BF16, 4, 10, P, _lib.VLS_MAX_TOPK + 1, -100, 0.0, P, P, None) == SHAPE
    assert f(P, 10, 7, 4, 10, P, 1, -100, 0.0, P, P, None) == DTYPE
    for bad in (math.nan, math.inf, -1.0):
        assert f(P, 10, BF16, 4, 10, P, 1, -100, bad, P, P, None) == CAP
    assert f(None, 10, BF16, 0, 10, None, 1, -100, 0.0, None, None, None) == OK   # empty: no launch
    g = lib.vls_logp_bwd
    assert g(P, 10, BF16, 4, 10, P, 1, -100, 0.0, None, P, P, None) == NULL
    assert g(P, 10, F32, 4, 10, P, 1, -100, -3.0, P, P, P, None) == CAP


def test_entropy_kl_argument_errors(lib):
    assert lib.vls_entropy_fwd(P, 10, F32, 4, 10, 0.0, None, P, None) == NULL
    assert lib.vls_entropy_bwd(P, 5, F32, 4, 10, 0.0, P, P, P, P, None) == SHAPE
    assert lib.vls_entropy_fwd(None, 10, F32, 0, 10, 0.0, None, None, None) == OK
    kf = lib.vls_kl_fwd
    assert kf(P, 10, P, 9, BF16, 4, 10, 0, 0.0, P, P, P, None) == SHAPE          # ldb < V
    assert kf(P, 10, P, 10, BF16, 4, 10, 2, 0.0, P, P, P, None) == ARG           # bad direction
    assert kf(P, 10, None, 10, BF16, 4, 10, 0, 0.0, P, P, P, None) == NULL
    assert kf(P, 10, P, 10, 3, 4, 10, 0, 0.0, P, P, P, None) == DTYPE
    kb = lib.vls_kl_bwd
    assert kb(P, 10, P, 10, BF16, 4, 10, 1, math.inf, P, P, P, P, P, None) == CAP


def test_softcap_argument_errors(lib):
    f, b = lib.vls_softcap_fwd, lib.vls_softcap_bwd
    assert f(P, P, -1, BF16, 30.0, None) == SHAPE
    for bad in (0.0, -30.0, math.nan, math.inf):        # the softcap call needs cap > 0
        assert f(P, P, 10, BF16, bad, None) == CAP
    assert f(None, P, 10, BF16, 30.0, None) == NULL
    assert f(None, None, 0, BF16, 30.0, None) == OK
    assert b(P, P, BF16, P, 10, F32, 30.0, None) == DTYPE     # gy bf16 with fp32 x
    assert b(P, None, F32, P, 10, BF16, 30.0, None) == NULL


def test_binding_rejects_bad_layouts():
    import torch

    from vocab_log_softmax_gb300 import binding as B
    x = torch.zeros((4, 6), dtype=torch.float64)
    with pytest.raises(TypeError):
        B.vls_entropy_fwd(x)
    with pytest.raises(ValueError):
        B.vls_entropy_fwd(torch.zeros((6, 4)).t())          # strided vocabulary dimension
    with pytest.raises(ValueError):
        B.vls_entropy_fwd(torch.zeros((3,)))                # not [N, V]


@pytest.mark.gpu
def test_host_pointer_is_rejected(lib):
    import torch
    host = torch.zeros((4, 10))
    out = torch.empty(4, device="cuda")
    st = torch.empty((4, 2), device="cuda")
    r = lib.vls_entropy_fwd(host.data_ptr(), 10, F32, 4, 10, 0.0, out.data_ptr(), st.data_ptr(), None)
    assert r == DEVICE


@pytest.mark.gpu
def test_side_stream_and_current_device_restored():
    import torch

    from vocab_log_softmax_gb300 import binding as B
    x = torch.randn((8, 4000), device="cuda")
    h0, _ = B.vls_entropy_fwd(x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        h1, _ = B.vls_entropy_fwd(x)
    s.synchronize()
    assert torch.equal(h0, h1)
    assert torch.cuda.current_device() == 0


def test_library_missing_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()


def test_ctypes_signature_count_matches_header():
    assert len(declared_functions()) == len(_lib.SIGNATURES)
    assert all(isinstance(t, list) for t in _lib.SIGNATURES.values())
    assert ctypes.sizeof(ctypes.c_int64) == 8
