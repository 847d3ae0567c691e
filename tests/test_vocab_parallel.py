"""Vocabulary-parallel split phase on one GPU: the vocabulary is cut into R
shards (equal, uneven with an empty shard, a single shard), each shard's
partial is computed from a strided view of the full logits, the partials
are stacked in rank order and combined; the result is compared with the
CPU oracle and with the unsharded call, and the per-shard backward
gradients, concatenated, with the oracle ("Add Triton kernels for
vocab-parallel logprobs, entropy and KL", DeepSpeed PR #8838, Tests: TP=2
with uneven and empty shards)."""

import numpy as np
import pytest
import torch

import oracle
import workloads
from vls_compare import assert_fp32_close, assert_grad_close, bitwise_equal, to_f64
from vocab_log_softmax_gb300 import binding as B
from vocab_log_softmax_gb300.vocab_parallel import shard_bounds

pytestmark = pytest.mark.gpu
DEV = "cuda"
V = 151936
SHARDINGS = {
    "two equal": [75968, 75968],
    "uneven with an empty shard": [40000, 0, 70001, 41935],
    "eight": [shard_bounds(V, 8, r)[1] for r in range(8)],
}


def _shards(x, widths):
    out, off = [], 0
    for w in widths:
        out.append((off, x[:, off:off + w]))
        off += w
    assert off == x.shape[1]
    return out


@pytest.fixture(scope="module")
def data():
    w = workloads.kl_masked(DEV, n=66, v=V)
    g = torch.Generator(device=DEV).manual_seed(9)
    ids = torch.randint(0, V, (66, 4), generator=g, device=DEV)
    ids[:, 3] = ids[:, 0]                     # duplicate
    ids[5, 1] = -100
    ids[6, 2] = V + 7                         # out of range
    ids[7, :] = -100                          # no valid id
    ids[8, 1] = 40000                         # first column of the third shard
    ids[8, 2] = 39999                         # last column of the first
    gk = torch.randn((66, 4), generator=g, device=DEV)
    return w["a"], w["b"], ids, gk, w["g"]


def _np(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("sharding", sorted(SHARDINGS))
@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_logp_sharded(data, sharding, cap):
    a, _, ids, gk, _ = data
    sh = _shards(a, SHARDINGS[sharding])
    parts, zts = zip(*[B.vls_logp_partial(x, ids, off, V, -100, cap) for off, x in sh])
    lp, st = B.vls_logp_combine(torch.stack(parts), torch.stack(zts), ids, V, -100, cap)
    d = torch.cat([B.vls_logp_bwd_shard(x, ids, gk, st, off, V, -100, cap) for off, x in sh], dim=1)
    torch.cuda.synchronize()
    xa = to_f64(a)
    assert_fp32_close(lp, oracle.logp_fwd(xa, _np(ids), -100, cap), f"{sharding} logp")
    assert_grad_close(d, oracle.logp_bwd(xa, _np(ids), _np(gk), -100, cap), f"{sharding} logp bwd")
    lp0, st0 = B.vls_logp_fwd(a, ids, -100, cap)
    assert_fp32_close(lp, to_f64(lp0), "sharded vs unsharded logp")


@pytest.mark.parametrize("sharding", sorted(SHARDINGS))
def test_entropy_sharded(data, sharding):
    a, _, _, _, gr = data
    sh = _shards(a, SHARDINGS[sharding])
    H, st = B.vls_entropy_combine(torch.stack([B.vls_entropy_partial(x) for _, x in sh]))
    d = torch.cat([B.vls_entropy_bwd(x, gr, H, st) if x.shape[1] else x.new_empty(x.shape) for _, x in sh], dim=1)
    torch.cuda.synchronize()
    xa = to_f64(a)
    assert_fp32_close(H, oracle.entropy_fwd(xa), f"{sharding} entropy")
    assert_grad_close(d, oracle.entropy_bwd(xa, _np(gr)), f"{sharding} entropy bwd")


@pytest.mark.parametrize("sharding", sorted(SHARDINGS))
@pytest.mark.parametrize("direction", ["reverse", "forward"])
def test_kl_sharded(data, sharding, direction):
    a, b, _, _, gr = data
    sa, sb = _shards(a, SHARDINGS[sharding]), _shards(b, SHARDINGS[sharding])
    parts = torch.stack([B.vls_kl_partial(x, y, direction) for (_, x), (_, y) in zip(sa, sb)])
    kl, stats_a, stats_b = B.vls_kl_combine(parts, direction)
    d = torch.cat([B.vls_kl_bwd(x, y, gr, kl, stats_a, stats_b, direction) if x.shape[1] else x.new_empty(x.shape)
                   for (_, x), (_, y) in zip(sa, sb)], dim=1)
    torch.cuda.synchronize()
    xa, xb = to_f64(a), to_f64(b)
    assert_fp32_close(kl, oracle.kl_fwd(xa, xb, direction), f"{sharding} kl {direction}")
    assert_grad_close(d, oracle.kl_bwd(xa, xb, _np(gr), direction), f"{sharding} kl {direction} bwd")


def test_single_shard_is_the_unsharded_forward_bitwise(data):
    """R = 1: folding one partial into the identity is exact, so combine
    reproduces the unsharded forward bit for bit."""
    a, b, ids, gk, gr = data
    part, zt = B.vls_logp_partial(a, ids, 0, V)
    lp, st = B.vls_logp_combine(part[None], zt[None], ids, V)
    lp0, st0 = B.vls_logp_fwd(a, ids)
    assert bitwise_equal(lp, lp0) and bitwise_equal(st, st0)
    H, sh = B.vls_entropy_combine(B.vls_entropy_partial(a)[None])
    H0, sh0 = B.vls_entropy_fwd(a)
    assert bitwise_equal(H, H0) and bitwise_equal(sh, sh0)
    for d in ("reverse", "forward"):
        kl, s1, s2 = B.vls_kl_combine(B.vls_kl_partial(a, b, d)[None], d)
        kl0, t1, t2 = B.vls_kl_fwd(a, b, d)
        assert bitwise_equal(kl, kl0) and bitwise_equal(s1, t1) and bitwise_equal(s2, t2)


def test_sharded_is_deterministic(data):
    a, _, ids, _, _ = data
    sh = _shards(a, SHARDINGS["uneven with an empty shard"])
    runs = []
    for _ in range(2):
        parts, zts = zip(*[B.vls_logp_partial(x, ids, off, V) for off, x in sh])
        runs.append(B.vls_logp_combine(torch.stack(parts), torch.stack(zts), ids, V))
    assert bitwise_equal(runs[0][0], runs[1][0]) and bitwise_equal(runs[0][1], runs[1][1])


def test_empty_shard_partial_is_identity(data):
    a = data[0]
    p = B.vls_entropy_partial(a[:, 100:100])
    torch.cuda.synchronize()
    v = p.cpu().numpy()
    assert np.all(np.isneginf(v[:, 0])) and np.all(v[:, 1] == 0) and np.all(v[:, 2] == 0)
