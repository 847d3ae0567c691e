"""The public autograd API (logprobs, entropy, kl, softcap, stats) on the
GPU: values and gradients against the CPU oracle, through torch.autograd,
with [B, T, V] inputs and a strided slice."""

import numpy as np
import pytest
import torch

import oracle
import vocab_log_softmax_gb300 as vls
from vls_compare import assert_fp32_close, assert_grad_close, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(dtype=torch.bfloat16, seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    a = (3 * torch.randn((2, 5, 3001), generator=g, device=DEV)).to(dtype)
    b = (a.float() + 0.5 * torch.randn(a.shape, generator=g, device=DEV)).to(dtype)
    ids = torch.randint(0, 3001, (2, 5), generator=g, device=DEV)
    ids[0, 1] = -100
    return a, b, ids, g


@pytest.mark.parametrize("cap", [None, 25.0])
def test_logprobs_autograd(cap):
    a, _, ids, g = _inputs()
    x = a.clone().requires_grad_(True)
    lp = vls.logprobs(x, ids, softcap=cap)
    gy = torch.randn(lp.shape, generator=g, device=DEV)
    (lp * gy).sum().backward()
    xa = to_f64(a.reshape(-1, 3001))
    c = cap or 0.0
    assert_fp32_close(lp.reshape(-1, 1), oracle.logp_fwd(xa, ids.reshape(-1, 1).cpu().numpy(), -100, c), "logprobs")
    assert_grad_close(x.grad.reshape(-1, 3001), oracle.logp_bwd(xa, ids.reshape(-1, 1).cpu().numpy(),
                                                                  gy.reshape(-1, 1).cpu().numpy(), -100, c), "dlogprobs")


def test_entropy_kl_autograd_on_a_slice():
    a, b, _, g = _inputs(torch.float32, 1)
    wide = torch.cat([a, a[..., :7]], dim=-1)                 # [2, 5, 3008]
    x = wide.clone().requires_grad_(True)
    view = x[..., :3001]                                      # strided rows read in place
    H = vls.entropy(view)
    kl = vls.kl(view, b, "reverse")
    gh = torch.randn(H.shape, generator=g, device=DEV)
    gk = torch.randn(kl.shape, generator=g, device=DEV)
    ((H * gh).sum() + (kl * gk).sum()).backward()
    xa, xb = to_f64(a.reshape(-1, 3001)), to_f64(b.reshape(-1, 3001))
    assert_fp32_close(H.reshape(-1), oracle.entropy_fwd(xa), "entropy")
    assert_fp32_close(kl.reshape(-1), oracle.kl_fwd(xa, xb, "reverse"), "kl")
    ref = oracle.entropy_bwd(xa, gh.reshape(-1).cpu().numpy()) + oracle.kl_bwd(xa, xb, gk.reshape(-1).cpu().numpy())
    assert_grad_close(x.grad[..., :3001].reshape(-1, 3001), ref, "entropy+kl grad")
    assert torch.count_nonzero(x.grad[..., 3001:]) == 0


def test_softcap_autograd():
    a, _, _, g = _inputs()
    x = (a.float() * 10).to(torch.bfloat16).requires_grad_(True)
    y = vls.softcap(x, 30.0)
    gy = torch.randn(y.shape, generator=g, device=DEV).to(torch.bfloat16)
    y.backward(gy)
    xs = to_f64(x.detach())
    assert_grad_close(y, oracle.softcap(xs, 30.0), "softcap")
    assert_grad_close(x.grad, oracle.softcap_grad(xs, to_f64(gy), 30.0), "dsoftcap")


@pytest.mark.parametrize("direction", ["reverse", "forward"])
def test_stats_fused_autograd(direction):
    a, b, ids, g = _inputs()
    x = a.clone().requires_grad_(True)
    lp, H, kl = vls.stats(x, ids, b, direction)
    gl = torch.randn(lp.shape, generator=g, device=DEV)
    gh = torch.randn(H.shape, generator=g, device=DEV)
    gk = torch.randn(kl.shape, generator=g, device=DEV)
    ((lp * gl).sum() + (H * gh).sum() + (kl * gk).sum()).backward()
    xa, xb = to_f64(a.reshape(-1, 3001)), to_f64(b.reshape(-1, 3001))
    i2 = ids.reshape(-1, 1).cpu().numpy()
    ref = (oracle.logp_bwd(xa, i2, gl.reshape(-1, 1).cpu().numpy()) + oracle.entropy_bwd(xa, gh.reshape(-1).cpu().numpy())
           + oracle.kl_bwd(xa, xb, gk.reshape(-1).cpu().numpy(), direction))
    assert_fp32_close(kl.reshape(-1), oracle.kl_fwd(xa, xb, direction), "stats kl")
    assert_grad_close(x.grad.reshape(-1, 3001), ref, "stats grad")
    # a loss that uses only the entropy leaves the other terms out
    y = a.clone().requires_grad_(True)
    _, H2, _ = vls.stats(y, ids, b, direction)
    (H2 * gh).sum().backward()
    assert_grad_close(y.grad.reshape(-1, 3001), oracle.entropy_bwd(xa, gh.reshape(-1).cpu().numpy()), "entropy only")
    assert np.isfinite(to_f64(y.grad)).all()
