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
TEST_HEADER = os.path.join(ROOT, "include", "vls_test.h")

OK, NULL, SHAPE, DTYPE, CAP, DEVICE, LAUNCH, ARG = range(8)
F32, BF16 = 0, 1
P = 0x1000   # a non-NULL pointer value; never dereferenced (errors precede any access)
R = _lib.rows


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions(header=HEADER):
    text = open(header).read()
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


def test_test_build_exports_both_headers_and_the_product_only_its_own(lib):
    tlib = _lib.load_test()
    hooks = declared_functions(TEST_HEADER)
    assert sorted(hooks) == sorted(_lib.TEST_SIGNATURES)
    for name in declared_functions() + hooks:
        assert hasattr(tlib, name), name
    for name in hooks:
        assert not hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.vls_status_string(code).decode().startswith(name)
    assert lib.vls_status_string(99).decode() == "VLS_ERR_UNKNOWN"
    assert lib.vls_version() >= 100


def test_logp_argument_errors(lib):
    f = lib.vls_logp_fwd
    #        logits rows dt    N  V  ids k  ign  cap  logp stats stream
    assert f(None, R(10), BF16, 4, 10, None, 1, -100, 0.0, None, None, None) == NULL
    assert f(P, R(10), BF16, -1, 10, P, 1, -100, 0.0, P, P, None) == SHAPE
    assert f(P, R(10), BF16, 4, 0, P, 1, -100, 0.0, P, P, None) == SHAPE
    assert f(P, R(9), BF16, 4, 10, P, 1, -100, 0.0, P, P, None) == SHAPE       # ld < V
    assert f(P, R(10), BF16, 4, 10, P, 0, -100, 0.0, P, P, None) == SHAPE      # k < 1
    assert f(P, R(10), BF16, 4, 10, P, _lib.VLS_MAX_TOPK + 1, -100, 0.0, P, P, None) == SHAPE
    assert f(P, R(10), 7, 4, 10, P, 1, -100, 0.0, P, P, None) == DTYPE
    for bad in (math.nan, math.inf, -1.0):
        assert f(P, R(10), BF16, 4, 10, P, 1, -100, bad, P, P, None) == CAP
    assert f(None, None, BF16, 0, 10, None, 1, -100, 0.0, None, None, None) == OK   # empty: no launch
    g = lib.vls_logp_bwd
    assert g(P, R(10), BF16, 4, 10, P, 1, -100, 0.0, None, P, P, None) == NULL
    assert g(P, R(10), F32, 4, 10, P, 1, -100, -3.0, P, P, P, None) == CAP


def test_entropy_kl_argument_errors(lib):
    assert lib.vls_entropy_fwd(P, R(10), F32, 4, 10, 0.0, None, P, None) == NULL
    assert lib.vls_entropy_bwd(P, R(5), F32, 4, 10, 0.0, P, P, P, P, None) == SHAPE
    assert lib.vls_entropy_fwd(None, None, F32, 0, 10, 0.0, None, None, None) == OK
    kf = lib.vls_kl_fwd
    assert kf(P, R(10), P, R(9), BF16, 4, 10, 0, 0.0, P, P, P, None) == SHAPE          # b: ld < V
    assert kf(P, R(10), P, R(10), BF16, 4, 10, 2, 0.0, P, P, P, None) == ARG           # bad direction
    assert kf(P, R(10), None, R(10), BF16, 4, 10, 0, 0.0, P, P, P, None) == NULL
    assert kf(P, R(10), P, R(10), 3, 4, 10, 0, 0.0, P, P, P, None) == DTYPE
    kb = lib.vls_kl_bwd
    assert kb(P, R(10), P, R(10), BF16, 4, 10, 1, math.inf, P, P, P, P, P, None) == CAP


def test_row_layout_errors(lib):
    f = lib.vls_entropy_fwd
    assert f(P, None, F32, 4, 10, 0.0, P, P, None) == NULL                 # descriptor missing
    assert f(P, R(10, -1, 40), F32, 4, 10, 0.0, P, P, None) == SHAPE       # negative group
    assert f(P, R(10, 2, 9), F32, 4, 10, 0.0, P, P, None) == SHAPE         # group stride < V
    assert f(P, R(9, 2, 40), F32, 4, 10, 0.0, P, P, None) == SHAPE         # row stride < V
    kf = lib.vls_kl_fwd
    assert kf(P, R(10, 2, 40), P, R(10, 3, 5), BF16, 4, 10, 0, 0.0, P, P, P, None) == SHAPE
    assert kf(P, R(10), P, None, BF16, 4, 10, 0, 0.0, P, P, P, None) == NULL
    # an empty vocabulary shard needs neither logits nor a descriptor
    assert lib.vls_entropy_partial(None, None, BF16, 4, 0, 0.0, None, None) == NULL   # part missing


def test_linear_backward_workspace_size(lib):
    """The backward's workspace is dz alone: N rows of V padded to 8
    elements, 16-bit, rounded up to 256 bytes; sizes out of range give -1."""
    ws = lib.vls_linear_logp_bwd_workspace
    for n, d, v in ((300, 200, 3001), (1, 8, 1), (8192, 4096, 151936), (0, 64, 256)):
        want = (n * ((v + 7) // 8 * 8) * 2 + 255) // 256 * 256
        assert ws(n, d, v) == want, (n, d, v)
    for n, d, v in ((-1, 8, 8), (8, 0, 8), (8, 8, 0), (2 ** 31, 8, 8), (8, 8, 2 ** 31), (8, 2 ** 31, 8)):
        assert ws(n, d, v) == -1, (n, d, v)


def test_rows_struct_matches_header():
    text = open(HEADER).read()
    assert re.search(r"typedef struct \{ int64_t ld; int64_t group; int64_t ld_group; \} vls_rows;", text)
    assert ctypes.sizeof(_lib.VlsRows) == 24
    assert [f[0] for f in _lib.VlsRows._fields_] == ["ld", "group", "ld_group"]


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
    with pytest.raises(ValueError):
        B.vls_entropy_fwd(torch.zeros((2, 6)).expand(3, 2, 6))   # broadcast rows overlap


def test_binding_row_descriptors():
    """[N, V] and [B, T, V] views map to the C ABI's vls_rows; a view whose
    leading dims collapse to one stride uses the single-stride form."""
    import torch

    from vocab_log_softmax_gb300 import binding as B

    def desc(t):
        n, v, r = B._rows(t)
        return n, v, (r.ld, r.group, r.ld_group)

    x = torch.zeros((4, 9, 16))
    assert desc(x) == (36, 16, (16, 0, 0))                  # contiguous: one stride
    assert desc(x[:, :-1]) == (32, 16, (16, 8, 144))        # shifted sequence: two strides
    assert desc(x[:, 1:, :8]) == (32, 8, (16, 8, 144))      # and a vocabulary slice
    assert desc(x[1:2, :-1]) == (8, 16, (16, 0, 0))         # one batch entry
    assert desc(x[:, 2:3]) == (4, 16, (144, 0, 0))          # one position per batch entry
    assert desc(x.reshape(36, 16)[::2]) == (18, 16, (32, 0, 0))
    assert desc(torch.zeros((1, 5))) == (1, 5, (5, 0, 0))


def test_as_rows_keeps_addressable_views():
    import torch

    import vocab_log_softmax_gb300 as V
    base = torch.zeros((4, 9, 16))
    for view in (base, base[:, :-1], base[:, 1:, :8], base[..., :8]):
        rows = V._as_rows(view)
        assert rows.data_ptr() == view.data_ptr() and rows.dim() in (2, 3)
    y = V._as_rows(torch.zeros((2, 3, 4, 16))[:, :, :-1])   # [2, 3, 3, 16]: leading dims merge to [6, 3]
    assert tuple(y.shape) == (6, 3, 16) and y.stride() == (64, 16, 1)
    t = V._as_rows(torch.zeros((16, 4)).t())               # strided vocabulary: copied
    assert t.is_contiguous()
    e = V._as_rows(torch.zeros((1, 16)).expand(5, 16))      # broadcast rows: copied
    assert e.is_contiguous() and e.shape == (5, 16)


@pytest.mark.gpu
def test_host_pointer_is_rejected(lib):
    import torch
    host = torch.zeros((4, 10))
    out = torch.empty(4, device="cuda")
    st = torch.empty((4, 2), device="cuda")
    r = lib.vls_entropy_fwd(host.data_ptr(), R(10), F32, 4, 10, 0.0, out.data_ptr(), st.data_ptr(), None)
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


@pytest.mark.gpu
def test_concurrent_host_threads():
    """Several host threads, each on its own stream, call the row sweeps and
    the tensor-core linear head at once (when this test runs first in its
    process, they also race on the linear head's one-time launch setup).
    Every result equals the one-thread result bit for bit."""
    import threading

    import torch

    from vocab_log_softmax_gb300 import binding as B
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn((64, 30000), generator=g, device="cuda").to(torch.bfloat16)
    ids = torch.randint(0, 30000, (64, 1), generator=g, device="cuda")
    h = torch.randn((300, 512), generator=g, device="cuda").to(torch.bfloat16)
    w = (0.1 * torch.randn((5000, 512), generator=g, device="cuda")).to(torch.bfloat16)
    lids = torch.randint(0, 5000, (300, 1), generator=g, device="cuda")
    torch.cuda.synchronize()
    out = [None] * 6
    errors = []

    def work(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                lp, st = B.vls_logp_fwd(x, ids)
                llp, lst, status = B.vls_linear_logp_fwd(h, w, lids)
            s.synchronize()
            out[i] = (lp, st, llp, lst, int(status.item()))
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(out))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    ref = (*B.vls_logp_fwd(x, ids), *B.vls_linear_logp_fwd(h, w, lids)[:2])
    torch.cuda.synchronize()
    for o in out:
        assert o[4] == 0
        for a, b in zip(o[:4], ref):
            assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                               b.view(torch.int32) if b.dtype == torch.float32 else b)


def test_library_missing_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()


def test_ctypes_signature_count_matches_header():
    assert len(declared_functions()) == len(_lib.SIGNATURES)
    assert all(isinstance(t, list) for t in _lib.SIGNATURES.values())
    assert ctypes.sizeof(ctypes.c_int64) == 8
