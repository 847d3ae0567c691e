"""Seeded synthetic inputs for the five workloads of the vocabulary-statistics
path.  Used by the tests, the benchmark and the smoke check; it holds none of
the method's arithmetic (no softmax, no statistic), only random draws.

Values are drawn in fp32 with ``torch.Generator`` on the target device, in
blocks of 1024 rows seeded ``seed * 1_000_003 + block``, then cast once
(round to nearest even) to the logits dtype.  The same call on the same
device and torch version gives the same bits.  There is no public dataset
behind these workloads; the shapes are the pages' own (Qwen vocabulary
151936 and its TP2 shard 75968, a 262144-column vocabulary for the softcap,
32k rows for the long-sequence case).

Workloads (rows N x vocabulary V):

* ``logp_small``  64 x 32000 fp32, N(0, 2^2); targets uniform, 10% of rows
  -100; upstream grad N(0, 1) per row.  (seed 0)
* ``logp_offset`` 8192 x 151936 bf16, N(0, 3^2) plus a per-row offset
  uniform in [-50, 50]; targets uniform, 5% of rows -100, another 1% at
  V + randint(0, 1000); grad N(0, 1).  (seed 1)
* ``kl_masked``   8192 x 75968 bf16 policy a ~ N(0, 3^2), reference
  b = a + N(0, 0.5^2) (both rounded from the same fp32 draw of a); 1% of the
  columns -inf in both; rows i % 64 == 0 get 16 more -inf columns in b only
  (support mismatch); the last row is -inf everywhere in both; grad N(0, 1).
  (seed 2)
* ``softcap_wide`` 4096 x 262144 bf16, N(0, 15^2) (tanh saturates at caps
  30 and 20); targets uniform; grad N(0, 1); softcap upstream gy N(0, 1) in
  bf16 and in fp32.  (seed 3)
* ``long_seq``    32768 x 151936 bf16, N(0, 3^2); k=1 uniform targets;
  k=256 ids per row = 224 distinct ids + 32 repeats of some of them,
  shuffled; grads N(0, 1).  (seed 4)

* ``linear_head`` h: 8192 x 4096 bf16 hidden states N(0, 1); W: 151936 x
  4096 bf16 head weights N(0, 9 / 4096), so the logits h @ W^T are about
  N(0, 3^2); a Qwen-size head (vocabulary 151936, hidden 4096); targets
  uniform, 5% of rows -100; grad N(0, 1).  (seed 5)

Every builder takes ``n`` and ``v`` overrides so that reduced copies of a
workload (the parity tests' sizes) follow the same recipe.
"""

from __future__ import annotations

import torch

BLOCK = 1024


def _gen(device, seed: int, block: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + block)
    return g


def _blocks(n: int):
    for b in range(0, max(n, 0), BLOCK):
        yield b // BLOCK, b, min(n, b + BLOCK)


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def logp_small(device="cuda", n: int = 64, v: int = 32000, seed: int = 0) -> dict:
    g = _gen(device, seed, 0)
    logits = 2.0 * _randn((n, v), g, device)
    ids = torch.randint(0, v, (n, 1), generator=g, device=device, dtype=torch.int64)
    n_ign = int(round(0.10 * n))
    rows = torch.randperm(n, generator=g, device=device)[:n_ign]
    ids[rows, 0] = -100
    grad = _randn((n, 1), g, device)
    return {"logits": logits, "ids": ids, "g": grad}


def logp_offset(device="cuda", n: int = 8192, v: int = 151936, seed: int = 1) -> dict:
    logits = torch.empty((n, v), dtype=torch.bfloat16, device=device)
    for blk, r0, r1 in _blocks(n):
        g = _gen(device, seed, blk)
        off = torch.rand((r1 - r0, 1), generator=g, device=device) * 100.0 - 50.0
        logits[r0:r1] = (3.0 * _randn((r1 - r0, v), g, device) + off).to(torch.bfloat16)
    g = _gen(device, seed, 1 << 20)
    ids = torch.randint(0, v, (n, 1), generator=g, device=device, dtype=torch.int64)
    perm = torch.randperm(n, generator=g, device=device)
    n_ign, n_oob = int(round(0.05 * n)), int(round(0.01 * n))
    ids[perm[:n_ign], 0] = -100
    oob = perm[n_ign:n_ign + n_oob]
    ids[oob, 0] = v + torch.randint(0, 1000, (oob.numel(),), generator=g, device=device)
    grad = _randn((n, 1), g, device)
    return {"logits": logits, "ids": ids, "g": grad}


def kl_masked(device="cuda", n: int = 8192, v: int = 75968, seed: int = 2) -> dict:
    a = torch.empty((n, v), dtype=torch.bfloat16, device=device)
    b = torch.empty((n, v), dtype=torch.bfloat16, device=device)
    for blk, r0, r1 in _blocks(n):
        g = _gen(device, seed, blk)
        a32 = 3.0 * _randn((r1 - r0, v), g, device)
        b32 = a32 + 0.5 * _randn((r1 - r0, v), g, device)
        a[r0:r1] = a32.to(torch.bfloat16)
        b[r0:r1] = b32.to(torch.bfloat16)
    g = _gen(device, seed, 1 << 20)
    cols = torch.randperm(v, generator=g, device=device)
    n_mask = max(1, int(round(0.01 * v)))
    masked = cols[:n_mask]
    a[:, masked] = float("-inf")
    b[:, masked] = float("-inf")
    unmasked = cols[n_mask:]
    for r in range(0, n, 64):
        pick = torch.randperm(unmasked.numel(), generator=g, device=device)[:16]
        b[r, unmasked[pick]] = float("-inf")
    a[n - 1] = float("-inf")
    b[n - 1] = float("-inf")
    grad = _randn((n,), g, device)
    return {"a": a, "b": b, "g": grad, "mismatch_rows": list(range(0, n, 64)), "masked_row": n - 1}


def softcap_wide(device="cuda", n: int = 4096, v: int = 262144, seed: int = 3) -> dict:
    x = torch.empty((n, v), dtype=torch.bfloat16, device=device)
    gy = torch.empty((n, v), dtype=torch.bfloat16, device=device)
    for blk, r0, r1 in _blocks(n):
        g = _gen(device, seed, blk)
        x[r0:r1] = (15.0 * _randn((r1 - r0, v), g, device)).to(torch.bfloat16)
        gy[r0:r1] = _randn((r1 - r0, v), g, device).to(torch.bfloat16)
    g = _gen(device, seed, 1 << 20)
    ids = torch.randint(0, v, (n, 1), generator=g, device=device, dtype=torch.int64)
    grad = _randn((n, 1), g, device)
    return {"logits": x, "ids": ids, "g": grad, "gy_bf16": gy, "caps": (30.0, 20.0)}


def softcap_gy_f32(data: dict, device="cuda", seed: int = 3) -> torch.Tensor:
    """The fp32 upstream-gradient variant of ``softcap_wide`` (same shape)."""
    n, v = data["logits"].shape
    out = torch.empty((n, v), dtype=torch.float32, device=device)
    for blk, r0, r1 in _blocks(n):
        out[r0:r1] = _randn((r1 - r0, v), _gen(device, seed + 100, blk), device)
    return out


def topk_ids(n: int, v: int, gen: torch.Generator, device, k_distinct: int = 224,
             k_dup: int = 32) -> torch.Tensor:
    """Per row: k_distinct distinct ids plus k_dup repeats of some of them, shuffled."""
    ids = torch.empty((n, k_distinct + k_dup), dtype=torch.int64, device=device)
    for _, r0, r1 in _blocks(n):
        m = r1 - r0
        keys = torch.rand((m, v), generator=gen, device=device)
        distinct = keys.topk(k_distinct, dim=1).indices
        rep = torch.randint(0, k_distinct, (m, k_dup), generator=gen, device=device)
        allid = torch.cat([distinct, distinct.gather(1, rep)], dim=1)
        order = torch.rand((m, k_distinct + k_dup), generator=gen, device=device).argsort(dim=1)
        ids[r0:r1] = allid.gather(1, order)
    return ids


def long_seq(device="cuda", n: int = 32768, v: int = 151936, seed: int = 4, k: int = 256) -> dict:
    logits = torch.empty((n, v), dtype=torch.bfloat16, device=device)
    for blk, r0, r1 in _blocks(n):
        g = _gen(device, seed, blk)
        logits[r0:r1] = (3.0 * _randn((r1 - r0, v), g, device)).to(torch.bfloat16)
    g = _gen(device, seed, 1 << 20)
    ids1 = torch.randint(0, v, (n, 1), generator=g, device=device, dtype=torch.int64)
    idsk = topk_ids(n, v, g, device, k_distinct=k - k // 8, k_dup=k // 8)
    return {
        "logits": logits,
        "ids1": ids1,
        "g1": _randn((n, 1), g, device),
        "idsk": idsk,
        "gk": _randn((n, k), g, device),
        "g_row": _randn((n,), g, device),
    }


def linear_head(device="cuda", n: int = 8192, d: int = 4096, v: int = 151936, seed: int = 5) -> dict:
    h = torch.empty((n, d), dtype=torch.bfloat16, device=device)
    for blk, r0, r1 in _blocks(n):
        h[r0:r1] = _randn((r1 - r0, d), _gen(device, seed, blk), device).to(torch.bfloat16)
    w = torch.empty((v, d), dtype=torch.bfloat16, device=device)
    scale = 3.0 / d ** 0.5
    for blk, r0, r1 in _blocks(v):
        w[r0:r1] = (scale * _randn((r1 - r0, d), _gen(device, seed, (1 << 16) + blk), device)).to(torch.bfloat16)
    g = _gen(device, seed, 1 << 20)
    ids = torch.randint(0, v, (n, 1), generator=g, device=device, dtype=torch.int64)
    ign = torch.randperm(n, generator=g, device=device)[: n // 20]
    ids[ign] = -100
    return {"h": h, "w": w, "ids": ids, "g": _randn((n, 1), g, device)}
