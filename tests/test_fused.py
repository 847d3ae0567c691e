"""Fused statistics: logprobs + entropy (+ KL) from one read of the policy,
and one backward pass for any weighted sum of them.  Forward outputs must
equal the single calls bit for bit (same arithmetic per field) and match the
oracle; the fused gradient must match the sum of the oracle's gradients."""

import pytest
import torch

import oracle
import workloads
from vls_compare import assert_fp32_close, assert_grad_close, bitwise_equal, to_f64
from vocab_log_softmax_gb300 import binding as B
from vocab_log_softmax_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
V = 151936


@pytest.fixture(scope="module")
def data():
    w = workloads.kl_masked(DEV, n=66, v=V)
    g = torch.Generator(device=DEV).manual_seed(21)
    ids = torch.randint(0, V, (66, 3), generator=g, device=DEV)
    ids[:, 2] = ids[:, 0]
    ids[3, 1] = -100
    ids[4, :] = -100
    gl = torch.randn((66, 3), generator=g, device=DEV)
    gh = torch.randn((66,), generator=g, device=DEV)
    gk = torch.randn((66,), generator=g, device=DEV)
    return w["a"], w["b"], ids, gl, gh, gk


def _np(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("direction", [None, "reverse", "forward"])
@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_fused_forward(data, direction, cap):
    a, b, ids, *_ = data
    out = B.vls_fused_fwd(a, b if direction else None, ids, direction=direction or "reverse", cap=cap)
    torch.cuda.synchronize()
    xa, xb = to_f64(a), to_f64(b)
    assert_fp32_close(out["logp"], oracle.logp_fwd(xa, _np(ids), -100, cap), "fused logp")
    assert_fp32_close(out["H"], oracle.entropy_fwd(xa, cap), "fused H")
    lp, st = B.vls_logp_fwd(a, ids, -100, cap)
    H, sh = B.vls_entropy_fwd(a, cap)
    assert bitwise_equal(out["logp"], lp) and bitwise_equal(out["stats_a"], st)
    assert bitwise_equal(out["H"], H)
    if direction:
        assert_fp32_close(out["kl"], oracle.kl_fwd(xa, xb, direction, cap), f"fused kl {direction}")
        kl, sa, sb = B.vls_kl_fwd(a, b, direction, cap)
        assert bitwise_equal(out["kl"], kl) and bitwise_equal(out["stats_b"], sb)


TERMS = {
    "logp": ("l",), "entropy": ("h",), "kl": ("k",), "logp+entropy": ("l", "h"), "all three": ("l", "h", "k"),
}


@pytest.mark.parametrize("terms", sorted(TERMS))
@pytest.mark.parametrize("direction", ["reverse", "forward"])
@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_fused_backward(data, terms, direction, cap):
    a, b, ids, gl, gh, gk = data
    t = TERMS[terms]
    with_kl = "k" in t
    out = B.vls_fused_fwd(a, b if with_kl else None, ids, direction=direction, cap=cap)
    da = B.vls_fused_bwd(a, out, b if with_kl else None, ids, g_logp=gl if "l" in t else None,
                         g_H=gh if "h" in t else None, g_kl=gk if with_kl else None, direction=direction, cap=cap)
    torch.cuda.synchronize()
    xa, xb = to_f64(a), to_f64(b)
    ref = 0.0
    if "l" in t:
        ref = ref + oracle.logp_bwd(xa, _np(ids), _np(gl), -100, cap)
    if "h" in t:
        ref = ref + oracle.entropy_bwd(xa, _np(gh), cap)
    if with_kl:
        ref = ref + oracle.kl_bwd(xa, xb, _np(gk), direction, cap)
    assert_grad_close(da, ref, f"fused bwd {terms} {direction} cap={cap}")


def test_fused_topk_and_fp32(data):
    a, b, _, _, gh, gk = data
    a32, b32 = a[:8].float(), b[:8].float()
    g = torch.Generator(device=DEV).manual_seed(3)
    ids = torch.randint(0, V, (8, 64), generator=g, device=DEV)
    ids[:, 32:] = ids[:, :32]
    gl = torch.randn((8, 64), generator=g, device=DEV)
    out = B.vls_fused_fwd(a32, b32, ids)
    da = B.vls_fused_bwd(a32, out, b32, ids, g_logp=gl, g_H=gh[:8].contiguous(), g_kl=gk[:8].contiguous())
    torch.cuda.synchronize()
    xa, xb = to_f64(a32), to_f64(b32)
    ref = (oracle.logp_bwd(xa, _np(ids), _np(gl)) + oracle.entropy_bwd(xa, _np(gh[:8]))
           + oracle.kl_bwd(xa, xb, _np(gk[:8]), "reverse"))
    assert_grad_close(da, ref, "fused top-64 fp32")


def test_fused_needs_a_term(data):
    a = data[0]
    out = B.vls_fused_fwd(a)
    with pytest.raises(_lib.VlsArgumentError):
        B.vls_fused_bwd(a, out)
