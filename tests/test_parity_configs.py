"""CUDA path vs the CPU fp64 oracle, element by element, on the five
workloads: the small logprob workload at full size, the other four as
reduced copies (fewer rows, the full vocabulary, the same recipe and the
same special rows).  Every call goes through the C ABI (``binding``)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from vls_compare import assert_fp32_close, assert_grad_close, to_f64
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _np(t):
    return t.detach().cpu().numpy()


def check_logp(logits, ids, g, cap=0.0, ignore=-100, what="logp"):
    logp, stats = B.vls_logp_fwd(logits, ids, ignore, cap)
    d = B.vls_logp_bwd(logits, ids, g, stats, ignore, cap)
    torch.cuda.synchronize()
    x = to_f64(logits)
    assert_fp32_close(logp, oracle.logp_fwd(x, _np(ids), ignore, cap), what + " fwd")
    assert_grad_close(d, oracle.logp_bwd(x, _np(ids), _np(g), ignore, cap), what + " bwd")
    return logp, d


def check_entropy(logits, g, cap=0.0, what="entropy"):
    H, stats = B.vls_entropy_fwd(logits, cap)
    d = B.vls_entropy_bwd(logits, g, H, stats, cap)
    torch.cuda.synchronize()
    x = to_f64(logits)
    assert_fp32_close(H, oracle.entropy_fwd(x, cap), what + " fwd")
    assert_grad_close(d, oracle.entropy_bwd(x, _np(g), cap), what + " bwd")


def check_kl(a, b, g, direction, cap=0.0, what="kl"):
    kl, sa, sb = B.vls_kl_fwd(a, b, direction, cap)
    d = B.vls_kl_bwd(a, b, g, kl, sa, sb, direction, cap)
    torch.cuda.synchronize()
    xa, xb = to_f64(a), to_f64(b)
    assert_fp32_close(kl, oracle.kl_fwd(xa, xb, direction, cap), f"{what} {direction} fwd")
    assert_grad_close(d, oracle.kl_bwd(xa, xb, _np(g), direction, cap), f"{what} {direction} bwd")
    return kl


def test_logp_small_full():
    w = workloads.logp_small(DEV)
    check_logp(w["logits"], w["ids"], w["g"], what="logp_small")


def test_logp_offset_reduced():
    w = workloads.logp_offset(DEV, n=100)
    ids = w["ids"].cpu()
    assert (ids == -100).sum() == 5 and (ids >= 151936).sum() == 1
    check_logp(w["logits"], w["ids"], w["g"], what="logp_offset")


def test_entropy_kl_masked_reduced():
    w = workloads.kl_masked(DEV, n=130)
    check_entropy(w["a"], w["g"], what="entropy(a)")
    for direction in ("reverse", "forward"):
        kl = check_kl(w["a"], w["b"], w["g"], direction)
        kl = kl.cpu()
        if direction == "reverse":
            assert torch.isinf(kl[[0, 64, 128]]).all()      # support mismatch rows
        assert torch.isnan(kl[129])                         # all -inf row


@pytest.mark.parametrize("cap", [30.0, 20.0])
def test_softcap_fused_logp_reduced(cap):
    w = workloads.softcap_wide(DEV, n=12)
    check_logp(w["logits"], w["ids"], w["g"], cap=cap, what=f"softcap{cap:g} logp")


@pytest.mark.parametrize("cap", [30.0, 20.0])
def test_softcap_standalone_reduced(cap):
    w = workloads.softcap_wide(DEV, n=6)
    x = w["logits"]
    xs = to_f64(x)
    y = B.vls_softcap_fwd(x, cap)
    for gy in (w["gy_bf16"], workloads.softcap_gy_f32(w, DEV)):
        gx = B.vls_softcap_bwd(x, gy, cap)
        torch.cuda.synchronize()
        assert gx.dtype == x.dtype
        assert_grad_close(gx, oracle.softcap_grad(xs, to_f64(gy), cap), f"softcap{cap:g} bwd gy={gy.dtype}")
    assert_grad_close(y, oracle.softcap(xs, cap), f"softcap{cap:g} fwd")


def test_long_seq_reduced():
    w = workloads.long_seq(DEV, n=20)
    check_logp(w["logits"], w["ids1"], w["g1"], what="long k=1")
    logp, _ = check_logp(w["logits"], w["idsk"], w["gk"], what="long k=256")
    check_entropy(w["logits"], w["g_row"], what="long entropy")
    # duplicates carry the same log-probability
    ids = w["idsk"].cpu().numpy()
    lp = logp.cpu().numpy()
    for r in range(ids.shape[0]):
        for i in np.unique(ids[r]):
            vals = lp[r][ids[r] == i]
            assert np.all(vals == vals[0])


def test_fp32_logits_all_ops():
    """fp32 logits through every op (the fp32 rows of the tolerance rules)."""
    g = torch.Generator(device=DEV).manual_seed(77)
    a = 4.0 * torch.randn((9, 5003), generator=g, device=DEV)
    b = a + 0.5 * torch.randn((9, 5003), generator=g, device=DEV)
    a[:, 17] = float("-inf")
    b[:, 17] = float("-inf")
    b[3, 40] = float("-inf")
    ids = torch.randint(0, 5003, (9, 3), generator=g, device=DEV)
    ids[2, 1] = -100
    gk = torch.randn((9, 3), generator=g, device=DEV)
    gr = torch.randn((9,), generator=g, device=DEV)
    for cap in (0.0, 7.5):
        check_logp(a, ids, gk, cap=cap, what=f"fp32 logp cap={cap}")
        check_entropy(a, gr, cap=cap, what=f"fp32 entropy cap={cap}")
        for direction in ("reverse", "forward"):
            check_kl(a, b, gr, direction, cap=cap, what=f"fp32 kl cap={cap}")
