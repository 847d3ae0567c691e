"""Two-stride row layouts: a [B, T, V] tensor read as N = B*T rows, with
slices such as x[:, :-1] (the shifted sequence of a language-model loss) read
in place instead of copied ("Add Triton kernels for vocab-parallel
logprobs, entropy and KL", DeepSpeed PR #8838, review "Suggested change":
rows addressed with up to two strides, the shifted slice with no extra
peak memory).  Every value outside the view is NaN, so a stray read shows;
results must be bit-identical to the contiguous copy, which is itself held
to the oracle here and in the parity tests."""

import numpy as np
import pytest
import torch

import oracle
import vocab_log_softmax_gb300 as V
from vls_compare import assert_fp32_close, assert_grad_close, bitwise_equal, to_f64
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _views(bsz, t, v, dtype, seed, shift_t=1, col0=0, pad=0):
    """x[:, :T-shift_t, col0:col0+v] of NaN-filled [B, T, col0+v+pad] buffers,
    for a policy and a reference (policy + noise), with contiguous copies."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    pol = 3.0 * torch.randn((bsz, t, v), generator=g, device=DEV)
    ref = pol + 0.5 * torch.randn((bsz, t, v), generator=g, device=DEV)
    out = []
    for vals in (pol, ref):
        buf = torch.full((bsz, t, col0 + v + pad), float("nan"), dtype=dtype, device=DEV)
        buf[:, :, col0:col0 + v] = vals.to(dtype)
        view = buf[:, : t - shift_t, col0:col0 + v]
        out.append((view, view.contiguous()))
    return out


CASES = [  # B, T, V, shift, first column, padding
    (4, 9, 1031, 1, 0, 0),
    (3, 17, 4096, 1, 3, 5),
    (2, 65, 151936, 1, 0, 0),
    (5, 6, 37, 2, 1, 2),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("bsz,t,v,shift,col0,pad", CASES)
def test_two_stride_views_are_bitwise_the_contiguous_copy(bsz, t, v, shift, col0, pad, dtype):
    (a, ac), (b, bc) = _views(bsz, t, v, dtype, seed=v + t, shift_t=shift, col0=col0, pad=pad)
    n = bsz * (t - shift)
    lay = B._rows(a)[2]
    assert lay.group == t - shift and lay.ld_group == t * (col0 + v + pad)   # really two strides
    g = torch.Generator(device=DEV).manual_seed(1)
    ids = torch.randint(0, v, (n, 3), generator=g, device=DEV)
    gk = torch.randn((n, 3), generator=g, device=DEV)
    gr = torch.randn((n,), generator=g, device=DEV)
    for cap in (0.0, 20.0):
        lp0, st0 = B.vls_logp_fwd(ac.reshape(n, v), ids, cap=cap)
        lp1, st1 = B.vls_logp_fwd(a, ids, cap=cap)
        assert bitwise_equal(lp0, lp1) and bitwise_equal(st0, st1)
        assert bitwise_equal(B.vls_logp_bwd(ac.reshape(n, v), ids, gk, st0, cap=cap),
                             B.vls_logp_bwd(a, ids, gk, st1, cap=cap))
        h0, s0 = B.vls_entropy_fwd(ac.reshape(n, v), cap)
        h1, s1 = B.vls_entropy_fwd(a, cap)
        assert bitwise_equal(h0, h1)
        assert bitwise_equal(B.vls_entropy_bwd(ac.reshape(n, v), gr, h0, s0, cap),
                             B.vls_entropy_bwd(a, gr, h1, s1, cap))
        for d in ("reverse", "forward"):
            k0, sa0, sb0 = B.vls_kl_fwd(ac.reshape(n, v), bc.reshape(n, v), d, cap)
            k1, sa1, sb1 = B.vls_kl_fwd(a, b, d, cap)
            assert bitwise_equal(k0, k1)
            assert bitwise_equal(B.vls_kl_bwd(ac.reshape(n, v), bc.reshape(n, v), gr, k0, sa0, sb0, d, cap),
                                 B.vls_kl_bwd(a, b, gr, k1, sa1, sb1, d, cap))
        f0 = B.vls_fused_fwd(ac.reshape(n, v), bc.reshape(n, v), ids, cap=cap)
        f1 = B.vls_fused_fwd(a, b, ids, cap=cap)
        for key in f0:
            assert bitwise_equal(f0[key], f1[key]), key
        assert bitwise_equal(
            B.vls_fused_bwd(ac.reshape(n, v), f0, bc.reshape(n, v), ids, g_logp=gk, g_H=gr, g_kl=gr, cap=cap),
            B.vls_fused_bwd(a, f1, b, ids, g_logp=gk, g_H=gr, g_kl=gr, cap=cap))
    p0 = B.vls_entropy_partial(ac.reshape(n, v))
    p1 = B.vls_entropy_partial(a)
    assert bitwise_equal(p0, p1)


def test_two_stride_view_against_the_oracle():
    (a, ac), (b, bc) = _views(3, 33, 5003, torch.bfloat16, seed=7, col0=2, pad=3)
    n, v = a.shape[0] * a.shape[1], a.shape[2]
    g = torch.Generator(device=DEV).manual_seed(2)
    ids = torch.randint(0, v, (n, 1), generator=g, device=DEV)
    ids[::7] = -100
    gk = torch.randn((n, 1), generator=g, device=DEV)
    gr = torch.randn((n,), generator=g, device=DEV)
    lp, st = B.vls_logp_fwd(a, ids)
    dl = B.vls_logp_bwd(a, ids, gk, st)
    kl, sa, sb = B.vls_kl_fwd(a, b, "reverse")
    dk = B.vls_kl_bwd(a, b, gr, kl, sa, sb, "reverse")
    torch.cuda.synchronize()
    x, y = to_f64(ac).reshape(n, v), to_f64(bc).reshape(n, v)
    idn, gkn, grn = ids.cpu().numpy(), gk.cpu().numpy().astype(np.float64), gr.cpu().numpy().astype(np.float64)
    assert_fp32_close(lp, oracle.logp_fwd(x, idn, -100, 0.0), "two-stride logp fwd")
    assert_grad_close(dl, oracle.logp_bwd(x, idn, gkn, -100, 0.0), "two-stride logp bwd")
    assert_fp32_close(kl, oracle.kl_fwd(x, y, "reverse", 0.0), "two-stride KL fwd")
    assert_grad_close(dk, oracle.kl_bwd(x, y, grn, "reverse", 0.0), "two-stride KL bwd")


def test_autograd_reads_the_shifted_slice_in_place():
    """reverse KL and logprobs of logits[:, :-1] through the autograd API: the
    same bits as on a contiguous copy, and no copy of the slice in between."""
    g = torch.Generator(device=DEV).manual_seed(3)
    leaf = (3.0 * torch.randn((4, 257, 32768), generator=g, device=DEV)).to(torch.bfloat16).requires_grad_(True)
    ref = (3.0 * torch.randn((4, 256, 32768), generator=g, device=DEV)).to(torch.bfloat16)
    ids = torch.randint(0, 32768, (4, 256), generator=g, device=DEV)
    view = leaf[:, :-1]
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    before = torch.cuda.memory_allocated()
    kl = V.kl(view, ref, "reverse")
    lp = V.logprobs(view, ids)
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - before
    assert extra < view.numel() * view.element_size() // 4, extra   # no [B, T-1, V] copy
    (kl.sum() + lp.sum()).backward()

    copy = view.detach().contiguous().requires_grad_(True)
    kl0 = V.kl(copy, ref, "reverse")
    lp0 = V.logprobs(copy, ids)
    (kl0.sum() + lp0.sum()).backward()
    assert bitwise_equal(kl, kl0) and bitwise_equal(lp, lp0)
    assert bitwise_equal(leaf.grad[:, :-1], copy.grad)
    assert bool(torch.all(leaf.grad[:, -1] == 0))
