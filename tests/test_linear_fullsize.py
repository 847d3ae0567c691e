"""The fused linear head at the shape the bench times (N = 8192 rows, D =
4096, V = 151936, bf16) and at N = 1024, on outputs the fp64 oracle can
compute one at a time: sampled rows of logp and dh (each needs its own
row's logits only), and sampled vocabulary columns of dW (each needs one
column of dz over all rows, so the oracle forms every row's logits: N = 1024
keeps that to about a minute of fp64 work).  These reach the launch shapes
the small cases do not: 75 vocabulary chunks on CTA pairs with K = 4096 in
the forward and the dz map, the 2.5 GB dz workspace with its column-fastest
raster and TMA-store epilogues, dh with no K split (N = 8192) and with one
(N = 1024).

Tolerances are those of tests/test_linear_logp.py: the logprob rule plus the
fp32 summation bound of the logits (none with integer inputs, whose logits
are exact), and for dh / dW the bound of a dz formed in fp32, rounded once
to bf16 and summed in fp32 over K = V (dh) or K = N (dW)."""

import numpy as np
import pytest
import torch

import oracle
from vls_compare import assert_fp32_close, to_f64, ulp_bf16
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24
D, V = 4096, 151936


def _inputs(n, seed, integer=False, k=1, ignore_frac=0.05):
    g = torch.Generator(device=DEV).manual_seed(seed)
    if integer:
        h = torch.randint(-1, 2, (n, D), generator=g, device=DEV).to(torch.bfloat16)
        w = torch.randint(-1, 2, (V, D), generator=g, device=DEV).to(torch.bfloat16)
    else:
        h = torch.randn((n, D), generator=g, device=DEV).to(torch.bfloat16)
        w = (3.0 / D ** 0.5 * torch.randn((V, D), generator=g, device=DEV)).to(torch.bfloat16)
    ids = torch.randint(0, V, (n, k), generator=g, device=DEV)
    ids[torch.rand((n, k), generator=g, device=DEV) < ignore_frac] = -100
    gr = torch.randn((n, k), generator=g, device=DEV)
    return h, w, ids, gr


def _logit_bound(x, wf):
    """Per row: D 2^-24 max_c sum_i |h_ri W_ci|, bounded by Cauchy-Schwarz
    (||h_r|| max_c ||W_c||) so that no second product over V is needed."""
    return D * U * np.linalg.norm(x, axis=1) * np.linalg.norm(wf, axis=1).max()


def _dz_err(z, dz, idn, gn, bz):
    """Bound on |dz_gpu - dz| per element: the bf16 rounding of dz (taken as
    2^-8 relative) plus the softmax term moved by the logits' error."""
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    valid = (idn != -100) & (idn >= 0) & (idn < V)
    G = np.abs((gn * valid).sum(axis=1))
    return np.abs(dz) * 2.0 ** -8 + G[:, None] * p * (2.0 * bz[:, None] + 2.0 ** -20)


def _assert_within(got, ref, bound, what):
    bound = bound + ulp_bf16(ref) + 1e-6
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} out of bound; worst {np.max(err - bound):.3e}"


def test_forward_exact_integers_at_bench_shape():
    """h, W in {-1, 0, 1}: every logit is an integer, exact in fp32 in any
    summation order, so sampled rows meet the plain logprob rule."""
    n = 8192
    h, w, ids, _ = _inputs(n, 101, integer=True, k=2)
    logp, stats, _ = B.vls_linear_logp_fwd(h, w, ids, check=True)
    rows = [0, 1, 255, 256, 4095, 4096, 8190, 8191]
    wf = to_f64(w)
    x = to_f64(h[rows])
    ref = oracle.linear_logp_fwd(x, wf, ids[rows].cpu().numpy())
    assert_fp32_close(logp[rows], ref, "integer logp, bench shape")
    z = oracle.linear_logits(x, wf)
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    st = stats[rows].double().cpu().numpy()
    assert np.all(np.abs(st[:, 0] + st[:, 1] - lse) <= 1e-5 + 1e-5 * np.abs(lse))
    assert np.array_equal(st[:, 0], m)   # the max of exact logits is exact


def test_backward_dh_sampled_rows_at_bench_shape():
    n = 8192
    h, w, ids, gr = _inputs(n, 102)
    _, stats, _ = B.vls_linear_logp_fwd(h, w, ids, check=True)
    dh, _, _ = B.vls_linear_logp_bwd(h, w, ids, gr, stats, check=True)
    rows = [0, 1, 255, 256, 4095, 4096, 8190, 8191]
    wf = to_f64(w)
    x = to_f64(h[rows])
    idn, gn = ids[rows].cpu().numpy(), gr[rows].double().cpu().numpy()
    ref_dh, _ = oracle.linear_logp_bwd(x, wf, idn, gn)
    z = oracle.linear_logits(x, wf)
    dz = oracle.logp_bwd(z, idn, gn)
    err = _dz_err(z, dz, idn, gn, _logit_bound(x, wf))
    awf = np.abs(wf)
    bound = err @ awf + V * U * (np.abs(dz) @ awf)
    _assert_within(to_f64(dh[rows]), ref_dh, bound, "dh rows, bench shape")


def test_backward_dw_sampled_columns_n1024():
    """dW columns need every row's softmax: the oracle forms all 1024 x
    151936 logits in fp64.  dh at this size is summed in several K runs."""
    n = 1024
    h, w, ids, gr = _inputs(n, 103, k=2)
    ids[:, 1] = ids[:, 0]                    # duplicate ids add their gradients
    _, stats, _ = B.vls_linear_logp_fwd(h, w, ids, check=True)
    dh, dw, _ = B.vls_linear_logp_bwd(h, w, ids, gr, stats, check=True)
    x, wf = to_f64(h), to_f64(w)
    idn, gn = ids.cpu().numpy(), gr.double().cpu().numpy()
    z = oracle.linear_logits(x, wf)
    dz = oracle.logp_bwd(z, idn, gn)
    err = _dz_err(z, dz, idn, gn, _logit_bound(x, wf))
    # sampled columns: both ends, tile and chunk edges, some targets (their
    # one-hot terms), and random ones
    rs = np.random.default_rng(0)
    targets = idn[:6, 0][idn[:6, 0] >= 0]
    cols = np.unique(np.concatenate([[0, 1, 255, 256, 2047, 2048, V - 1], targets, rs.integers(0, V, 24)]))
    ax = np.abs(x)
    ref_dw = dz[:, cols].T @ x
    bound = err[:, cols].T @ ax + n * U * (np.abs(dz[:, cols]).T @ ax)
    _assert_within(to_f64(dw[cols]), ref_dw, bound, "dW columns, N=1024")
    rows = [0, 1, 127, 128, 511, 512, 1022, 1023]
    awf = np.abs(wf)
    ref_dh = dz[rows] @ wf
    bound = err[rows] @ awf + V * U * (np.abs(dz[rows]) @ awf)
    _assert_within(to_f64(dh[rows]), ref_dh, bound, "dh rows, N=1024")
