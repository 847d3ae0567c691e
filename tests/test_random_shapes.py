"""A seeded sweep of random small shapes against the oracle: every op, with
ragged vocabularies, all three dtypes, softcap on and off, rows read in place
from a wider buffer, ignored and out-of-range ids, and duplicate top-k ids.
The cases come from one fixed seed, so a failure names a case that can be
rerun alone (``-k "case07"``)."""

import numpy as np
import pytest
import torch

from test_parity_configs import check_entropy, check_kl, check_logp

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.float32, torch.bfloat16, torch.float16]


def _cases(count=24, seed=1234):
    rs = np.random.RandomState(seed)
    out = []
    for i in range(count):
        n = int(rs.randint(1, 34))
        v = int(rs.choice([int(rs.randint(1, 64)), int(rs.randint(64, 5000)), int(rs.randint(5000, 40000))]))
        k = int(rs.randint(1, 7))
        dtype = DTYPES[int(rs.randint(0, 3))]
        cap = float(rs.choice([0.0, 0.0, 15.0]))
        pad = int(rs.choice([0, 0, 8, 13]))   # extra columns per row of the buffer the rows are read from
        out.append(pytest.param(i, n, v, k, dtype, cap, pad, id=f"case{i:02d}"))
    return out


@pytest.mark.parametrize("i,n,v,k,dtype,cap,pad", _cases())
def test_random_shape(i, n, v, k, dtype, cap, pad):
    g = torch.Generator(device=DEV).manual_seed(1000 + i)
    buf = (4.0 * torch.randn((n, v + pad), generator=g, device=DEV)).to(dtype)
    a = buf[:, :v]
    b = (a.float() + 0.7 * torch.randn((n, v), generator=g, device=DEV)).to(dtype)
    ids = torch.randint(0, v, (n, k), generator=g, device=DEV)
    if k > 1:
        ids[:, -1] = ids[:, 0]                         # a duplicate id in every row
    flip = torch.rand((n, k), generator=g, device=DEV)
    ids[flip < 0.1] = -100                             # ignored
    ids[(flip >= 0.1) & (flip < 0.15)] = v + 7          # out of range, ignored too
    gk = torch.randn((n, k), generator=g, device=DEV)
    gr = torch.randn((n,), generator=g, device=DEV)
    what = f"case{i:02d} N={n} V={v} k={k} {dtype} cap={cap} pad={pad}"
    check_logp(a, ids, gk, cap=cap, what=what + " logp")
    check_entropy(a, gr, cap=cap, what=what + " entropy")
    for d in ("reverse", "forward"):
        check_kl(a, b, gr, d, cap=cap, what=what + f" kl {d}")
