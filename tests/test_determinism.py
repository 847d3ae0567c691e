"""Determinism and batch invariance, bit for bit: repeated calls, row
subsets, permutations, padding rows, N=1 against the full batch, and bf16
logits against their exact fp32 copy ("perf(logp): fused zero-workspace
backward ...", RL-Kernel PR #495, Summary: deterministic and batch-invariant,
one block per row and a fixed reduction tree; "Final Logit Softcap",
Accuracy and Invariance: bitwise equality under repetition, slicing and
padding)."""

import pytest
import torch

import workloads
from vls_compare import bitwise_equal
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _all_outputs(a, b, ids, gk, gr, cap=0.0):
    """Every forward output and gradient of every op, per row (row-indexed tensors)."""
    lp, st = B.vls_logp_fwd(a, ids, -100, cap)
    dl = B.vls_logp_bwd(a, ids, gk, st, -100, cap)
    h, se = B.vls_entropy_fwd(a, cap)
    de = B.vls_entropy_bwd(a, gr, h, se, cap)
    # k = 1: at a few rows the backward cuts each row into more pieces than
    # at many rows (the split follows N there); the bits must not move
    dl1 = B.vls_logp_bwd(a, ids[:, :1].contiguous(), gk[:, :1].contiguous(), st, -100, cap)
    out = {"logp": lp, "stats": st, "dlogp": dl, "dlogp_k1": dl1, "H": h, "dH": de}
    for d in ("reverse", "forward"):
        kl, sa, sb = B.vls_kl_fwd(a, b, d, cap)
        out["kl_" + d] = kl
        out["dkl_" + d] = B.vls_kl_bwd(a, b, gr, kl, sa, sb, d, cap)
    torch.cuda.synchronize()
    return out


@pytest.fixture(scope="module")
def batch():
    w = workloads.kl_masked(DEV, n=70, v=151936)
    g = torch.Generator(device=DEV).manual_seed(5)
    ids = torch.randint(0, 151936, (70, 4), generator=g, device=DEV)
    ids[3, 1] = -100
    gk = torch.randn((70, 4), generator=g, device=DEV)
    return w["a"], w["b"], ids, gk, w["g"]


@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_repeat(batch, cap):
    o1 = _all_outputs(*batch, cap=cap)
    o2 = _all_outputs(*batch, cap=cap)
    for k in o1:
        assert bitwise_equal(o1[k], o2[k]), k


@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_row_subsets_permutation_padding(batch, cap):
    a, b, ids, gk, gr = batch
    full = _all_outputs(a, b, ids, gk, gr, cap)
    n = a.shape[0]
    perm = torch.randperm(n, generator=torch.Generator().manual_seed(1)).to(DEV)
    cases = {
        "single rows": [torch.tensor([i], device=DEV) for i in (0, 1, 64, n - 1)],
        "subset": [torch.arange(10, 40, 3, device=DEV)],
        "permutation": [perm],
    }
    for name, idx_list in cases.items():
        for idx in idx_list:
            sub = _all_outputs(a[idx].contiguous(), b[idx].contiguous(), ids[idx].contiguous(),
                               gk[idx].contiguous(), gr[idx].contiguous(), cap)
            for k in full:
                assert bitwise_equal(full[k][idx], sub[k]), (name, k)
    # padding: the batch followed by extra rows
    pad = torch.cat([a, a[:5] * 0.5]), torch.cat([b, b[:5]]), torch.cat([ids, ids[:5]]), \
        torch.cat([gk, gk[:5]]), torch.cat([gr, gr[:5]])
    padded = _all_outputs(*pad, cap=cap)
    for k in full:
        assert bitwise_equal(full[k], padded[k][:n]), ("padding", k)


def test_bf16_equals_exact_fp32_copy(batch):
    """Thread <-> column map is defined in columns, so bf16 logits and their
    exact fp32 copies give identical forward bits, and the bf16 gradient is the
    round-to-nearest-even of the fp32 one."""
    a, b, ids, gk, gr = batch
    ob = _all_outputs(a, b, ids, gk, gr)
    of = _all_outputs(a.float(), b.float(), ids, gk, gr)
    for k in ("logp", "stats", "H", "kl_reverse", "kl_forward"):
        assert bitwise_equal(ob[k], of[k]), k
    for k in ("dlogp", "dH", "dkl_reverse", "dkl_forward"):
        assert bitwise_equal(ob[k], of[k].to(torch.bfloat16)), k


def test_f16_equals_exact_fp32_copy(batch):
    """The same for float16 logits (values rescaled into float16's range)."""
    a, b, ids, gk, gr = batch
    a16 = (a.float() * 0.25).to(torch.float16)
    b16 = (b.float() * 0.25).to(torch.float16)
    oh = _all_outputs(a16, b16, ids, gk, gr)
    of = _all_outputs(a16.float(), b16.float(), ids, gk, gr)
    for k in ("logp", "stats", "H", "kl_reverse", "kl_forward"):
        assert bitwise_equal(oh[k], of[k]), k
    for k in ("dlogp", "dH", "dkl_reverse", "dkl_forward"):
        assert bitwise_equal(oh[k], of[k].to(torch.float16)), k


def test_k1_equals_same_id_in_topk(batch):
    a = batch[0]
    w = workloads.long_seq(DEV, n=8, v=a.shape[1])
    ids_k = w["idsk"]
    lpk, _ = B.vls_logp_fwd(w["logits"], ids_k)
    for j in (0, 17, 255):
        lp1, _ = B.vls_logp_fwd(w["logits"], ids_k[:, j:j + 1].contiguous())
        assert bitwise_equal(lp1[:, 0], lpk[:, j])
