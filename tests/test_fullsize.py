"""Full-size workloads in the launch configuration the benchmark times,
checked on sampled rows (the oracle computes them one by one) and on
properties that hold at any size; plus the zero-workspace check: the calls
allocate no device memory beyond their outputs (the long-sequence case,
"perf(logp): fused zero-workspace backward ...", RL-Kernel PR #495, Tests: the
fused path's memory check)."""

import gc

import pytest
import torch

import oracle
import workloads
from vls_compare import assert_fp32_close, assert_grad_close, to_f64
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(n, special=()):
    g = torch.Generator().manual_seed(n)
    pick = {0, n - 1, *special, *torch.randint(0, n, (4,), generator=g).tolist()}
    return sorted(pick)


def _np(t):
    return t.detach().cpu().numpy()


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def test_logp_offset_full():
    w = workloads.logp_offset(DEV)
    x, ids, g = w["logits"], w["ids"], w["g"]
    lp, st = B.vls_logp_fwd(x, ids)
    d = B.vls_logp_bwd(x, ids, g, st)
    ign = torch.nonzero(ids[:, 0] == -100)[0, 0].item()
    oob = torch.nonzero(ids[:, 0] >= x.shape[1])[0, 0].item()
    rows = _rows(x.shape[0], (ign, oob))
    xs = to_f64(x[rows])
    assert_fp32_close(lp[rows], oracle.logp_fwd(xs, _np(ids[rows])), "logp fwd")
    assert_grad_close(d[rows], oracle.logp_bwd(xs, _np(ids[rows]), _np(g[rows])), "logp bwd")
    assert torch.isfinite(lp).all()
    valid = (ids[:, 0] >= 0) & (ids[:, 0] < x.shape[1])
    assert (lp[~valid] == 0).all() and (lp[valid] < 0).all()
    del w, x, d
    _free()


def test_kl_masked_full():
    w = workloads.kl_masked(DEV)
    a, b, g = w["a"], w["b"], w["g"]
    n = a.shape[0]
    rows = _rows(n, (64, 8191, 4096))
    xa, xb = to_f64(a[rows]), to_f64(b[rows])
    H, se = B.vls_entropy_fwd(a)
    dH = B.vls_entropy_bwd(a, g, H, se)
    assert_fp32_close(H[rows], oracle.entropy_fwd(xa), "entropy fwd")
    assert_grad_close(dH[rows], oracle.entropy_bwd(xa, _np(g[rows])), "entropy bwd")
    del dH
    for direction in ("reverse", "forward"):
        kl, sa, sb = B.vls_kl_fwd(a, b, direction)
        da = B.vls_kl_bwd(a, b, g, kl, sa, sb, direction)
        assert_fp32_close(kl[rows], oracle.kl_fwd(xa, xb, direction), f"kl {direction} fwd")
        assert_grad_close(da[rows], oracle.kl_bwd(xa, xb, _np(g[rows]), direction), f"kl {direction} bwd")
        ok = torch.ones(n, dtype=torch.bool, device=DEV)
        ok[n - 1] = False
        if direction == "reverse":
            ok[torch.arange(0, n, 64, device=DEV)] = False
            assert torch.isposinf(kl[0:n - 1:64]).all()
        assert torch.isnan(kl[n - 1])
        assert torch.isfinite(kl[ok]).all() and (kl[ok] >= -1e-5).all()      # Gibbs
        del da
    del w, a, b
    _free()


@pytest.mark.parametrize("cap", [30.0, 20.0])
def test_softcap_wide_full(cap):
    w = workloads.softcap_wide(DEV)
    x, ids, g = w["logits"], w["ids"], w["g"]
    rows = _rows(x.shape[0])
    xs = to_f64(x[rows])
    lp, st = B.vls_logp_fwd(x, ids, -100, cap)
    d = B.vls_logp_bwd(x, ids, g, st, -100, cap)
    assert_fp32_close(lp[rows], oracle.logp_fwd(xs, _np(ids[rows]), -100, cap), "capped logp fwd")
    assert_grad_close(d[rows], oracle.logp_bwd(xs, _np(ids[rows]), _np(g[rows]), -100, cap), "capped logp bwd")
    del d
    y = B.vls_softcap_fwd(x, cap)
    assert_grad_close(y[rows], oracle.softcap(xs, cap), "softcap fwd")
    assert (y.float().abs() <= cap).all()
    del y
    for gy in (w["gy_bf16"], None):
        if gy is None:
            gy = workloads.softcap_gy_f32(w, DEV)
        gx = B.vls_softcap_bwd(x, gy, cap)
        assert_grad_close(gx[rows], oracle.softcap_grad(xs, to_f64(gy[rows]), cap), f"softcap bwd {gy.dtype}")
        del gx, gy
    del w, x
    _free()


def test_long_seq_full_and_zero_workspace():
    w = workloads.long_seq(DEV)
    x = w["logits"]
    n, v = x.shape
    rows = _rows(n)
    xs = to_f64(x[rows])
    ids1, idsk, g1, gk, gr = (_np(w[k][rows]) for k in ("ids1", "idsk", "g1", "gk", "g_row"))
    # outputs preallocated, so any allocation by the calls would show in the peak
    lp1 = torch.empty((n, 1), device=DEV)
    lpk = torch.empty((n, w["idsk"].shape[1]), device=DEV)
    st = torch.empty((n, 2), device=DEV)
    H = torch.empty((n,), device=DEV)
    d = torch.empty((n, v), dtype=x.dtype, device=DEV)

    def sample(t):  # per-row views copied to the host: no device allocation
        return torch.stack([t[r].cpu() for r in rows])

    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    got = {}
    B.vls_logp_fwd(x, w["ids1"], logp=lp1, stats=st)
    B.vls_logp_bwd(x, w["ids1"], w["g1"], st, dlogits=d)
    got["k1"] = sample(lp1), sample(d)
    B.vls_logp_fwd(x, w["idsk"], logp=lpk, stats=st)
    B.vls_logp_bwd(x, w["idsk"], w["gk"], st, dlogits=d)
    got["k256"] = sample(lpk), sample(d)
    B.vls_entropy_fwd(x, H=H, stats=st)
    B.vls_entropy_bwd(x, w["g_row"], H, st, dlogits=d)
    got["entropy"] = sample(H), sample(d)
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - base
    free1 = torch.cuda.mem_get_info()[0]
    assert extra == 0, f"the calls allocated {extra} bytes through torch"
    # nothing allocated behind torch's back either (allocation granularity 2 MiB)
    assert free0 - free1 < (2 << 20), free0 - free1

    assert_fp32_close(got["k1"][0], oracle.logp_fwd(xs, ids1), "k=1 fwd")
    assert_grad_close(got["k1"][1], oracle.logp_bwd(xs, ids1, g1), "k=1 bwd")
    assert_fp32_close(got["k256"][0], oracle.logp_fwd(xs, idsk), "k=256 fwd")
    assert_grad_close(got["k256"][1], oracle.logp_bwd(xs, idsk, gk), "k=256 bwd")
    assert_fp32_close(got["entropy"][0], oracle.entropy_fwd(xs), "entropy fwd")
    assert_grad_close(got["entropy"][1], oracle.entropy_bwd(xs, gr), "entropy bwd")
    del w, x, d
    _free()
