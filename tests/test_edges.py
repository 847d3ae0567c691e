"""Edge cases of the CUDA path against the oracle: tiny and ragged
vocabularies, misaligned and strided rows (with NaN outside the view, so a
stray read shows), masked columns and rows, ignored and out-of-range ids,
duplicate ids, the top-k limit and empty input."""

import numpy as np
import pytest
import torch

import oracle
from test_parity_configs import check_entropy, check_kl, check_logp
from vls_compare import assert_fp32_close, assert_grad_close, bitwise_equal, to_f64
from vocab_log_softmax_gb300 import binding as B
from vocab_log_softmax_gb300 import _lib

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.float32, torch.bfloat16, torch.float16]


def _gen(seed):
    return torch.Generator(device=DEV).manual_seed(seed)


def _data(n, v, dtype, seed, scale=3.0):
    g = _gen(seed)
    a = (scale * torch.randn((n, v), generator=g, device=DEV)).to(dtype)
    b = (a.float() + 0.5 * torch.randn((n, v), generator=g, device=DEV)).to(dtype)
    ids = torch.randint(0, v, (n, 2), generator=g, device=DEV)
    gk = torch.randn((n, 2), generator=g, device=DEV)
    gr = torch.randn((n,), generator=g, device=DEV)
    return a, b, ids, gk, gr


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("v", [1, 2, 7, 8, 9, 255, 1031, 4097, 16385])
def test_vocab_sizes(v, dtype):
    a, b, ids, gk, gr = _data(5, v, dtype, seed=v)
    check_logp(a, ids, gk, what=f"V={v} logp")
    check_entropy(a, gr, what=f"V={v} entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, what=f"V={v} kl")
    check_logp(a, ids, gk, cap=5.0, what=f"V={v} logp cap")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("v", [262144, 600001, 2000003])
def test_cluster_rows(v, dtype):
    """Rows wider than one CTA's share of 24576 vectors: the forward sweep runs
    on a cluster of 2, 4 and 8 CTAs (the last with more than 24576 vectors
    each), whose states combine through distributed shared memory in rank
    order; the backward cuts the row into many pieces."""
    a, b, ids, gk, gr = _data(2, v, dtype, seed=v % 1009)
    check_logp(a, ids, gk, what=f"V={v} logp")
    check_entropy(a, gr, what=f"V={v} entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, what=f"V={v} kl {d}")
    check_logp(a, ids, gk, cap=20.0, what=f"V={v} logp cap")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("v,pad,shift", [(1031, 3, 0), (1031, 5, 1), (4096, 1, 1), (37, 11, 3), (151936, 8, 1)])
def test_strided_and_misaligned_rows(v, pad, shift, dtype):
    """Rows read in place from a wider buffer (row stride v + pad, start shifted
    by `shift` elements); everything outside the view is NaN.  Results must be
    bit-identical to the contiguous copy."""
    n = 6
    a, b, ids, gk, gr = _data(n, v, dtype, seed=v + pad)
    wide_a = torch.full((n, v + pad + shift), float("nan"), dtype=dtype, device=DEV)
    wide_b = torch.full((n, v + pad + shift), float("nan"), dtype=dtype, device=DEV)
    wide_a[:, shift:shift + v] = a
    wide_b[:, shift:shift + v] = b
    va, vb = wide_a[:, shift:shift + v], wide_b[:, shift:shift + v]
    assert va.stride(0) == v + pad + shift and va.stride(1) == 1

    lp0, st0 = B.vls_logp_fwd(a, ids)
    lp1, st1 = B.vls_logp_fwd(va, ids)
    assert bitwise_equal(lp0, lp1) and bitwise_equal(st0, st1)
    assert bitwise_equal(B.vls_logp_bwd(a, ids, gk, st0), B.vls_logp_bwd(va, ids, gk, st1))
    h0, s0 = B.vls_entropy_fwd(a)
    h1, s1 = B.vls_entropy_fwd(va)
    assert bitwise_equal(h0, h1)
    assert bitwise_equal(B.vls_entropy_bwd(a, gr, h0, s0), B.vls_entropy_bwd(va, gr, h1, s1))
    for d in ("reverse", "forward"):
        k0, sa0, sb0 = B.vls_kl_fwd(a, b, d)
        k1, sa1, sb1 = B.vls_kl_fwd(va, vb, d)
        assert bitwise_equal(k0, k1)
        assert bitwise_equal(B.vls_kl_bwd(a, b, gr, k0, sa0, sb0, d), B.vls_kl_bwd(va, vb, gr, k1, sa1, sb1, d))
    check_logp(va, ids, gk, what="strided logp")


@pytest.mark.parametrize("dtype", DTYPES)
def test_masks_and_ignores(dtype):
    v = 3000
    a, b, ids, gk, gr = _data(8, v, dtype, seed=5)
    a[:, 100:140] = float("-inf")          # masked vocabulary block
    b[:, 100:140] = float("-inf")
    a[1, v - 200:] = float("-inf")         # masked tail
    b[1, v - 200:] = float("-inf")
    a[2] = float("-inf")                   # all -inf row (policy only)
    b[3] = float("-inf")                   # all -inf row (reference only)
    a[4], b[4] = float("-inf"), float("-inf")
    b[5, 7] = float("-inf")                # mismatch, policy weight underflows fp32
    a[5, 7] = a[5].float().max().to(dtype) - 120.0
    ids[0, 0], ids[0, 1] = -100, 120       # ignored id; id on a masked column
    ids[6, 0], ids[6, 1] = v, v + 5        # out of range only: zero row
    ids[7, 0] = ids[7, 1] = 11             # duplicate
    check_logp(a, ids, gk, what="masked logp")
    check_logp(a, ids, gk, ignore=11, what="masked logp ignore=11")
    check_entropy(a, gr, what="masked entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, what="masked kl")
    # softcap turns -inf into -cap: no masked columns remain
    check_logp(a, ids, gk, cap=4.0, what="masked logp cap")
    check_entropy(a, gr, cap=4.0, what="masked entropy cap")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, cap=4.0, what="masked kl cap")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_nan_logit_makes_its_row_nan(cap, dtype):
    """A NaN logit makes every statistic of its row NaN, and every gradient
    of that row, as in the oracle; the other rows are untouched.  With a cap,
    logits above about 22 c are limited before the exponential: a NaN beside
    such a value (in the same pair, the same vector, or the ragged tail) must
    stay NaN through that limit."""
    v = 4099
    a, b, ids, gk, gr = _data(6, v, dtype, seed=31)
    nan = float("nan")
    a[0, 0], a[0, 1] = nan, 1e4            # same pair as a limited value
    a[1, 2000], a[1, 2003] = nan, 1e4      # same vector
    a[2, v - 1] = nan                      # ragged tail
    a[3, 10] = 1e4                         # limited value, finite row
    b[4, 77] = nan                         # reference only (KL)
    check_logp(a, ids, gk, cap=cap, what="nan logp")
    check_logp(a, ids[:, :1].contiguous(), gk[:, :1].contiguous(), cap=cap, what="nan logp k=1")
    check_entropy(a, gr, cap=cap, what="nan entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, cap=cap, what="nan kl")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
@pytest.mark.parametrize("cap", [50.0, 100.0])
def test_large_caps(cap, dtype):
    """Caps above the pages' 20 and 30 (50 is another common softcap).  The
    capped logit carries an absolute error of a few 1e-7 * cap, so the
    results still meet the fp32 rule at these caps, in a short row and a
    full-width one, with logits spread enough to reach the cap's bend."""
    for n, v, scale in ((6, 4099, 40.0), (3, 151936, 25.0)):
        a, b, ids, gk, gr = _data(n, v, dtype, seed=int(cap) + v % 97, scale=scale)
        check_logp(a, ids, gk, cap=cap, what=f"cap={cap} V={v} logp")
        check_entropy(a, gr, cap=cap, what=f"cap={cap} V={v} entropy")
        for d in ("reverse", "forward"):
            check_kl(a, b, gr, d, cap=cap, what=f"cap={cap} V={v} kl")


def test_zero_rows_are_exact():
    a, _, ids, gk, _ = _data(4, 777, torch.bfloat16, seed=9)
    ids[:] = -100
    lp, st = B.vls_logp_fwd(a, ids)
    d = B.vls_logp_bwd(a, ids, gk, st)
    assert torch.count_nonzero(lp) == 0
    assert torch.equal(d.view(torch.int16), torch.zeros_like(d).view(torch.int16))   # +0.0 bits


@pytest.mark.parametrize("k", [1, 3, 64, 256, _lib.VLS_MAX_TOPK])
def test_topk(k):
    v = 5000
    a, _, _, _, _ = _data(3, v, torch.bfloat16, seed=k)
    g = _gen(k + 1)
    ids = torch.randint(0, v, (3, k), generator=g, device=DEV)
    if k > 2:
        ids[0, k // 2:] = ids[0, : k - k // 2].clone()   # many duplicates
        ids[1, ::3] = -100
        ids[2, 1] = v + 1
    gk = torch.randn((3, k), generator=g, device=DEV)
    check_logp(a, ids, gk, what=f"top-{k}")


def test_topk_full_vocab_sums_to_one():
    v = 1000
    a, _, _, _, _ = _data(2, v, torch.float32, seed=3)
    ids = torch.arange(v, device=DEV).repeat(2, 1)
    lp, _ = B.vls_logp_fwd(a, ids)
    s = torch.exp(lp.double()).sum(dim=1)
    assert torch.allclose(s, torch.ones_like(s), atol=1e-5)


def test_empty_inputs():
    x = torch.empty((0, 100), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty((0, 1), dtype=torch.int64, device=DEV)
    lp, st = B.vls_logp_fwd(x, ids)
    assert lp.shape == (0, 1)
    d = B.vls_logp_bwd(x, ids, torch.empty((0, 1), device=DEV), st)
    assert d.shape == (0, 100)
    h, _ = B.vls_entropy_fwd(x)
    assert h.shape == (0,)
    y = B.vls_softcap_fwd(torch.empty(0, dtype=torch.bfloat16, device=DEV), 30.0)
    assert y.numel() == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("n", [1, 7, 8, 9, 1023, 4097])
def test_softcap_ragged_and_misaligned(n, dtype):
    g = _gen(n)
    buf = (40.0 * torch.randn(n + 1, generator=g, device=DEV)).to(dtype)
    buf[0] = float("-inf")
    for x in (buf[:n], buf[1:]):               # aligned, then one element off
        for cap in (20.0, 30.0):
            y = B.vls_softcap_fwd(x, cap)
            gy = torch.randn(x.shape, generator=g, device=DEV)
            gx = B.vls_softcap_bwd(x, gy, cap)
            torch.cuda.synchronize()
            xs = to_f64(x)
            assert_grad_close(y, oracle.softcap(xs, cap), "softcap fwd")
            assert_grad_close(gx, oracle.softcap_grad(xs, to_f64(gy), cap), "softcap bwd")


def test_large_offset():
    """+1000 common offset with -inf masks (the pages' large-offset case)."""
    a, b, ids, gk, gr = _data(4, 32000, torch.float32, seed=21)
    a += 1000.0
    b += 1000.0
    a[:, :50] = float("-inf")
    b[:, :50] = float("-inf")
    check_logp(a, ids, gk, what="offset logp")
    check_entropy(a, gr, what="offset entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, what="offset kl")


def test_kl_self_is_zero_bitwise():
    a, _, _, _, gr = _data(6, 75968, torch.bfloat16, seed=4)
    for d in ("reverse", "forward"):
        kl, sa, sb = B.vls_kl_fwd(a, a, d)
        da = B.vls_kl_bwd(a, a, gr, kl, sa, sb, d)
        assert torch.all(kl == 0)
        assert torch.count_nonzero(da.float()) == 0


def test_uniform_rows_closed_form():
    v = 151936
    x = torch.full((3, v), 1.5, dtype=torch.bfloat16, device=DEV)
    ids = torch.tensor([[0], [v - 1], [77]], device=DEV)
    lp, _ = B.vls_logp_fwd(x, ids)
    h, _ = B.vls_entropy_fwd(x)
    assert_fp32_close(lp, np.full((3, 1), -np.log(v)), "uniform logp")
    assert_fp32_close(h, np.full(3, np.log(v)), "uniform entropy")


def test_float16_range_limits():
    """float16 logits at the ends of its range, next to -inf masks: the
    lowest finite float16 (-65504) is a real logit, not a mask."""
    v = 4001
    g = _gen(65504)
    a = (3.0 * torch.randn((6, v), generator=g, device=DEV)).to(torch.float16)
    b = (a.float() + 0.5 * torch.randn((6, v), generator=g, device=DEV)).to(torch.float16)
    a[0, :] = -65504.0                          # a whole row at the lowest finite value: uniform
    a[0, 17] = float("-inf")
    b[0, :] = -65504.0
    b[0, 17] = float("-inf")
    a[1, 5] = 65504.0                           # the largest finite value dominates the row
    a[2, 100:110] = -65504.0
    b[2, 100:110] = float("-inf")               # mismatch against finite (if tiny) policy weight
    ids = torch.randint(0, v, (6, 2), generator=g, device=DEV)
    gk = torch.randn((6, 2), generator=g, device=DEV)
    gr = torch.randn((6,), generator=g, device=DEV)
    check_logp(a, ids, gk, what="f16 limits logp")
    check_entropy(a, gr, what="f16 limits entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, what="f16 limits kl")
