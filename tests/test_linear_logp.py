"""Fused linear head + logprobs on the tensor cores against the oracle
(logits z = h @ W^T formed in fp64 there, never stored on the GPU).

Tolerance.  The logits are fp32 sums of D exact bf16 / fp16 products, in an
order the tensor cores fix.  Any order of an fp32 sum of D terms is within
D * 2^-24 * sum |terms| of the exact sum (the standard worst-case bound of
recursive summation), so a log-probability, which is z_target - max z - log S,
moves by at most twice the largest such bound over the row's columns.  The
tests add that bound to the logprob rule of the other calls
(1e-5 + 1e-5 |ref|).  With small integer inputs every logit is exact in fp32,
the bound is 0, and the plain rule applies: any misplaced product, tile or
chunk changes an integer and fails.
"""

import numpy as np
import pytest
import torch

import oracle
from vls_compare import assert_fp32_close, bitwise_equal, to_f64
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


def _gen(seed):
    return torch.Generator(device=DEV).manual_seed(seed)


def _ids(n, v, k, seed, ignore_frac=0.0):
    g = _gen(seed)
    ids = torch.randint(0, v, (n, k), generator=g, device=DEV)
    if ignore_frac:
        mask = torch.rand((n, k), generator=g, device=DEV) < ignore_frac
        ids[mask] = -100
    return ids


def _summation_bound(h, w):
    """Per row: 2 * D * 2^-24 * max_c sum_i |h_ri W_ci| (float64)."""
    hh, ww = np.abs(to_f64(h)), np.abs(to_f64(w))
    return 2.0 * h.shape[1] * U * (hh @ ww.T).max(axis=1)


def _check(h, w, ids, what, ignore=-100, exact=False):
    logp, stats, status = B.vls_linear_logp_fwd(h, w, ids, ignore)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"{what}: a wait in the kernel ran out"
    ref = oracle.linear_logp_fwd(to_f64(h), to_f64(w), ids.cpu().numpy(), ignore)
    extra = 0.0 if exact else _summation_bound(h, w)[:, None]
    assert_fp32_close(logp, ref, what, atol=1e-5 + extra)
    z = oracle.linear_logits(to_f64(h), to_f64(w))
    m_ref = z.max(axis=1)
    lse = m_ref + np.log(np.exp(z - m_ref[:, None]).sum(axis=1))
    got = stats.cpu().numpy().astype(np.float64)
    tol = 1e-5 + 1e-5 * np.abs(lse) + (0.0 if exact else _summation_bound(h, w))
    assert np.all(np.abs(got[:, 0] + got[:, 1] - lse) <= tol), what + " stats"
    return logp, stats


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_exact_integer_inputs(dtype):
    """Entries in {-1, 0, 1}: every logit is an exact integer in fp32."""
    n, d, v = 300, 200, 5000          # 3 row tiles (ragged), D not a multiple of 64, 3 chunks, ragged last tile
    g = _gen(1)
    h = torch.randint(-1, 2, (n, d), generator=g, device=DEV).to(dtype)
    w = torch.randint(-1, 2, (v, d), generator=g, device=DEV).to(dtype)
    _check(h, w, _ids(n, v, 1, 2, 0.1), "integer linear logp", exact=True)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("n,d,v", [(129, 1000, 2049), (8, 64, 256), (1, 8, 1), (520, 4096, 16000)])
def test_random_inputs(n, d, v, dtype):
    g = _gen(n + d + v)
    h = torch.randn((n, d), generator=g, device=DEV).to(dtype)
    w = (3.0 / d ** 0.5 * torch.randn((v, d), generator=g, device=DEV)).to(dtype)
    _check(h, w, _ids(n, v, 1, 3, 0.05), f"linear logp N={n} D={d} V={v}")


def test_topk_duplicates_ignores_out_of_range():
    n, d, v = 200, 128, 3000
    g = _gen(7)
    h = torch.randn((n, d), generator=g, device=DEV).to(torch.bfloat16)
    w = (0.3 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16)
    ids = _ids(n, v, 16, 8, 0.1)
    ids[:, 5] = ids[:, 4]                  # duplicates
    ids[::3, 7] = v + 5                    # out of range
    ids[1::7, 9] = -7                      # negative
    _check(h, w, ids, "linear logp top-16")
    _check(h, w, ids, "linear logp ignore=3", ignore=3)


def test_strided_rows_and_batch_invariance():
    """Rows read in place from wider buffers; any subset or order of rows
    gives the same bits (each row's statistics depend on that row only)."""
    n, d, v = 300, 256, 4100
    g = _gen(11)
    hbuf = torch.randn((n, d + 8), generator=g, device=DEV).to(torch.bfloat16)
    wbuf = (0.2 * torch.randn((v, d + 16), generator=g, device=DEV)).to(torch.bfloat16)
    h, w = hbuf[:, :d], wbuf[:, :d]
    ids = _ids(n, v, 2, 12)
    lp, st = _check(h, w, ids, "strided linear logp")
    lpc, stc, _ = B.vls_linear_logp_fwd(h.contiguous(), w.contiguous(), ids)
    assert bitwise_equal(lp, lpc) and bitwise_equal(st, stc)
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(0)).to(DEV)
    for rows in (perm, perm[:1], perm[:130], torch.arange(n - 1, -1, -1, device=DEV)):
        lps, sts, _ = B.vls_linear_logp_fwd(h[rows].contiguous(), w, ids[rows].contiguous())
        assert bitwise_equal(lps, lp[rows]) and bitwise_equal(sts, st[rows])


def test_chunk_count_depends_on_v_only():
    assert B.vls_linear_logp_chunks(1) == 1
    assert B.vls_linear_logp_chunks(2048) == 1
    assert B.vls_linear_logp_chunks(2049) == 2
    assert B.vls_linear_logp_chunks(151936) == 75


def test_full_size_sampled_rows():
    """N=8192, D=4096, V=151936 (a Qwen-size head) in the launch shape the
    bench times; 6 sampled rows checked against the oracle one by one."""
    n, d, v = 8192, 4096, 151936
    g = _gen(21)
    h = torch.randn((n, d), generator=g, device=DEV).to(torch.bfloat16)
    w = (3.0 / d ** 0.5 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16)
    ids = _ids(n, v, 1, 22, 0.05)
    logp, stats, status = B.vls_linear_logp_fwd(h, w, ids)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    wf = to_f64(w)
    for r in (0, 1, 127, 128, 4097, n - 1):
        hr = to_f64(h[r:r + 1])
        ref = oracle.linear_logp_fwd(hr, wf, ids[r:r + 1].cpu().numpy())
        bound = 2.0 * d * U * (np.abs(hr) @ np.abs(wf).T).max()
        assert_fp32_close(logp[r:r + 1], ref, f"row {r}", atol=1e-5 + bound)


# ---------------------------------------------------------------------------
# backward: dh = dz @ W, dW = dz^T @ h with dz = g one-hot - G p
# ---------------------------------------------------------------------------

def _ulp16(r, dtype):
    from vls_compare import ulp_bf16, ulp_f16
    return ulp_bf16(r) if dtype == torch.bfloat16 else ulp_f16(r)


def _check_bwd(h, w, ids, g, what, ignore=-100):
    """dh and dW against the oracle.  Bound: dz is formed in fp32 from logits
    within the summation bound, then rounded once to the 16-bit dtype
    (relative 2^-9 for bf16, 2^-11 for fp16; taken as 2^-8 and 2^-10); the
    products sum in fp32 (K 2^-24 sum |terms|), then round once more."""
    logp, stats, st0 = B.vls_linear_logp_fwd(h, w, ids, ignore)
    dh, dw, st1 = B.vls_linear_logp_bwd(h, w, ids, g, stats, ignore)
    torch.cuda.synchronize()
    assert int(st0.item()) == 0 and int(st1.item()) == 0, what + ": a wait ran out"
    x, wf = to_f64(h), to_f64(w)
    idn, gn = ids.cpu().numpy(), g.cpu().numpy().astype(np.float64)
    ref_dh, ref_dw = oracle.linear_logp_bwd(x, wf, idn, gn, ignore)
    z = oracle.linear_logits(x, wf)
    dz = oracle.logp_bwd(z, idn, gn, ignore)
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    valid = (idn != ignore) & (idn >= 0) & (idn < wf.shape[0])
    G = np.abs((gn * valid).sum(axis=1))
    rel = 2.0 ** -8 if h.dtype == torch.bfloat16 else 2.0 ** -10
    bz = h.shape[1] * U * (np.abs(x) @ np.abs(wf).T).max(axis=1)
    err_dz = np.abs(dz) * rel + G[:, None] * p * (2.0 * bz[:, None] + 2.0 ** -20)
    tol_dh = err_dz @ np.abs(wf) + wf.shape[0] * U * (np.abs(dz) @ np.abs(wf))
    tol_dw = err_dz.T @ np.abs(x) + x.shape[0] * U * (np.abs(dz).T @ np.abs(x))
    for got, ref, tol, name in ((dh, ref_dh, tol_dh, "dh"), (dw, ref_dw, tol_dw, "dW")):
        gotn = to_f64(got)
        bound = tol + _ulp16(ref, h.dtype) + 1e-6
        bad = np.abs(gotn - ref) > bound
        assert not bad.any(), (f"{what} {name}: {int(bad.sum())} of {bad.size} out of bound; worst "
                               f"{np.max(np.abs(gotn - ref) - bound):.3e}")
    return dh, dw


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
@pytest.mark.parametrize("n,d,v,k", [(300, 256, 5003, 2), (129, 1000, 2049, 1), (8, 64, 256, 3)])
def test_backward(n, d, v, k, dtype):
    g = _gen(n * 7 + v)
    h = torch.randn((n, d), generator=g, device=DEV).to(dtype)
    w = (3.0 / d ** 0.5 * torch.randn((v, d), generator=g, device=DEV)).to(dtype)
    ids = _ids(n, v, k, 31, 0.1)
    if k > 1:
        ids[:, 1] = ids[:, 0]               # duplicates add their upstream gradients
    gr = torch.randn((n, k), generator=g, device=DEV)
    _check_bwd(h, w, ids, gr, f"linear bwd N={n} D={d} V={v} k={k}")


def test_backward_many_k_runs():
    """Few rows over a long vocabulary: dh is summed in dozens of K runs
    (32 here) whose partial sums sit in dW's memory before dW is written."""
    n, d, v = 64, 512, 32768
    g = _gen(71)
    h = torch.randn((n, d), generator=g, device=DEV).to(torch.bfloat16)
    w = (3.0 / d ** 0.5 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16)
    ids = _ids(n, v, 2, 72, 0.1)
    gr = torch.randn((n, 2), generator=g, device=DEV)
    _check_bwd(h, w, ids, gr, "linear bwd, many K runs")


def test_backward_ignored_rows_give_zero_dh():
    n, d, v = 200, 128, 3000
    g = _gen(41)
    h = torch.randn((n, d), generator=g, device=DEV).to(torch.bfloat16)
    w = (0.3 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16)
    ids = _ids(n, v, 1, 42)
    ids[::4] = -100
    ids[1::9] = v + 3
    gr = torch.randn((n, 1), generator=g, device=DEV)
    dh, _ = _check_bwd(h, w, ids, gr, "linear bwd with ignored rows")
    dead = ((ids[:, 0] == -100) | (ids[:, 0] >= v)).nonzero().flatten()
    assert bool(torch.all(dh[dead] == 0))


@pytest.mark.parametrize("d", [200, 100])
def test_backward_strided_operands(d):
    """h and W read in place from wider buffers: the products take W and h
    as stored (their rows are the reduction index of dh and dW), so the row
    strides reach the tensor maps directly.  Same bits as contiguous copies,
    and within the oracle bound.  With D = 100 the rows of dh and dW are not
    16-byte multiples, so their products store through the threads instead
    of TMA."""
    n, v = 300, 3001
    g = _gen(61)
    d8 = (d + 7) // 8 * 8
    hbuf = torch.randn((n, d8 + 8), generator=g, device=DEV).to(torch.bfloat16)
    wbuf = (0.2 * torch.randn((v, d8 + 24), generator=g, device=DEV)).to(torch.bfloat16)
    h, w = hbuf[:, :d], wbuf[:, :d]
    ids = _ids(n, v, 2, 62, 0.1)
    gr = torch.randn((n, 2), generator=g, device=DEV)
    dh, dw = _check_bwd(h, w, ids, gr, "strided linear bwd")
    # the same values under other row strides (multiples of 8 elements, as TMA needs)
    h2 = torch.zeros((n, d8 + 24), dtype=h.dtype, device=DEV)[:, :d]
    w2 = torch.zeros((v, d8 + 8), dtype=w.dtype, device=DEV)[:, :d]
    h2.copy_(h)
    w2.copy_(w)
    _, st, _ = B.vls_linear_logp_fwd(h2, w2, ids)
    dhc, dwc, status = B.vls_linear_logp_bwd(h2, w2, ids, gr, st)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert bitwise_equal(dh, dhc) and bitwise_equal(dw, dwc)


def test_autograd_linear_logprobs():
    import vocab_log_softmax_gb300 as V
    n, d, v = 2 * 96, 256, 4100
    g = _gen(51)
    h = torch.randn((2, 96, d), generator=g, device=DEV).to(torch.bfloat16).requires_grad_(True)
    w = (0.2 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16).requires_grad_(True)
    ids = _ids(n, v, 1, 52).reshape(2, 96)
    gr = torch.randn((2, 96), generator=g, device=DEV)
    lp = V.linear_logprobs(h, w, ids)
    (lp * gr).sum().backward()
    ref_lp, st, _ = B.vls_linear_logp_fwd(h.detach().reshape(n, d), w.detach(), ids.reshape(n, 1))
    dh, dw, _ = B.vls_linear_logp_bwd(h.detach().reshape(n, d), w.detach(), ids.reshape(n, 1),
                                      gr.reshape(n, 1).contiguous(), st)
    assert bitwise_equal(lp.reshape(n, 1), ref_lp)
    assert bitwise_equal(h.grad.reshape(n, d), dh) and bitwise_equal(w.grad, dw)


def test_one_sm_kernel():
    """The 1-SM form of the tensor-core GEMM (selected through the test
    build's tuning hook; the product library always takes CTA pairs) passes
    the exact-integer and backward parity checks too."""
    from vocab_log_softmax_gb300 import _lib
    tlib = _lib.load_test()
    assert tlib.vls_test_set_tuning(0, 0, 1) == 0
    try:
        with _lib.using(tlib):
            test_exact_integer_inputs(torch.bfloat16)
            test_backward(300, 256, 5003, 2, torch.bfloat16)
            test_backward_strided_operands(200)
    finally:
        tlib.vls_test_set_tuning(0, 0, 0)
