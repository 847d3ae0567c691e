"""Pins for the CPU oracle: checks against facts fixed by the pages and by
mathematics, never against the oracle itself.

Each ``check_*`` takes an implementation namespace (normally the ``oracle``
package) and raises AssertionError on a failure, so that
``test_oracle_mutations.py`` can show that plausible mistakes planted in a
copy of the oracle are caught.  The pins are:

* closed forms from ``tests/golden/closed_forms.json`` (uniform rows,
  Bernoulli rows, masked columns, KL(p||p) = 0, tanh(log(3)/2) = 1/2);
* library routines on special cases: scipy's ``log_softmax``,
  ``scipy.stats.entropy`` (entropy and KL), torch fp64 autograd of
  ``log_softmax`` + ``gather``;
* invariants: shift invariance, sum of probabilities = 1, zero row sums of
  gradients, Gibbs' inequality, odd symmetry of the softcap;
* central finite differences in fp64 on tiny rows for every backward;
* for the linear head, dot products and log-sum-exp written out with
  Python's math on a tiny case, and torch fp64 autograd.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")

_MATH = {"log": math.log, "exp": math.exp, "inf": math.inf, "sqrt": math.sqrt}


def closed_form(expr) -> float:
    """Evaluate a closed-form expression from the fixture with Python's math."""
    if isinstance(expr, (int, float)):
        return float(expr)
    return float(eval(expr, {"__builtins__": {}}, _MATH))  # fixture text only


def _vec(xs) -> np.ndarray:
    return np.array([closed_form(x) for x in xs], dtype=np.float64)


def load_golden() -> dict:
    with open(GOLDEN) as f:
        return json.load(f)


def _close(a, b, rtol=1e-12, atol=1e-12) -> bool:
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    same_nonfinite = np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        np.where(np.isinf(a), a, 0.0), np.where(np.isinf(b), b, 0.0))
    fa, fb = np.isfinite(a), np.isfinite(b)
    return bool(same_nonfinite and np.array_equal(fa, fb)
                and np.all(np.abs(a[fa] - b[fb]) <= atol + rtol * np.abs(b[fb])))


def _fd(f, x: np.ndarray, h: float = 1e-6) -> np.ndarray:
    """Central finite differences of the scalar function f at x (fp64)."""
    grad = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        grad[idx] = (f(xp) - f(xm)) / (2.0 * h)
    return grad


# ----------------------------------------------------------------------------
# closed forms (golden fixture)
# ----------------------------------------------------------------------------

def check_golden_logp(impl):
    for case in load_golden()["logp"]:
        z = _vec(case["logits"])[None, :]
        ids = np.array(case["ids"], dtype=np.int64)[None, :]
        got = impl.logp_fwd(z, ids, -100)[0]
        want = _vec(case["expected"])
        assert _close(got, want, 1e-12, 1e-12), (case["name"], got, want)


def check_golden_entropy(impl):
    for case in load_golden()["entropy"]:
        z = _vec(case["logits"])[None, :]
        got = impl.entropy_fwd(z)[0]
        want = closed_form(case["expected"])
        assert abs(got - want) <= 1e-12, (case["name"], got, want)


def check_golden_kl(impl):
    for case in load_golden()["kl"]:
        a, b = _vec(case["a"])[None, :], _vec(case["b"])[None, :]
        for direction in ("reverse", "forward"):
            got = impl.kl_fwd(a, b, direction)[0]
            want = closed_form(case[direction])
            if math.isinf(want):
                assert got == want, (case["name"], direction, got)
            else:
                assert abs(got - want) <= 1e-12 + 1e-10 * abs(want), (case["name"], direction, got, want)


def check_golden_softcap(impl):
    for case in load_golden()["softcap"]:
        c = case["cap"]
        x = np.array([closed_form(case["x"])])
        y = impl.softcap(x, c)[0]
        dydx = impl.softcap_grad(x, np.ones(1), c)[0]
        assert abs(y - closed_form(case["y"])) <= 1e-12 * c, (case["name"], y)
        assert abs(dydx - closed_form(case["dydx"])) <= 1e-12, (case["name"], dydx)


# ----------------------------------------------------------------------------
# logp
# ----------------------------------------------------------------------------

def check_logp_uniform(impl):
    for v in (1, 5, 1000, 151936):
        z = np.full((1, v), -3.25)
        ids = np.array([[0, v - 1]])
        got = impl.logp_fwd(z, ids)
        assert np.allclose(got, -math.log(v), rtol=0, atol=1e-12), (v, got)


def check_logp_shift_invariance(impl):
    rng = np.random.default_rng(11)
    z = rng.normal(0, 3, size=(3, 257))
    ids = rng.integers(0, 257, size=(3, 4))
    base = impl.logp_fwd(z, ids)
    for c in (-50.0, 50.0, 1000.0):
        got = impl.logp_fwd(z + c, ids)
        assert np.allclose(got, base, rtol=0, atol=1e-9 * (1 + abs(c))), c


def check_logp_normalised(impl):
    rng = np.random.default_rng(12)
    v = 97
    z = rng.normal(0, 4, size=(2, v))
    ids = np.tile(np.arange(v), (2, 1))
    lp = impl.logp_fwd(z, ids)
    assert np.allclose(np.exp(lp).sum(axis=1), 1.0, rtol=0, atol=1e-12)


def check_logp_vs_scipy(impl):
    from scipy.special import log_softmax
    rng = np.random.default_rng(13)
    z = rng.normal(0, 3, size=(4, 1031)) + rng.uniform(-50, 50, size=(4, 1))
    ids = rng.integers(0, 1031, size=(4, 8))
    want = np.take_along_axis(log_softmax(z, axis=1), ids, axis=1)
    assert np.allclose(impl.logp_fwd(z, ids), want, rtol=1e-12, atol=1e-12)


def check_logp_ignored(impl):
    rng = np.random.default_rng(14)
    z = rng.normal(size=(3, 10))
    ids = np.array([[-100, 10, 15], [-7, 3, -100], [2, 2, 9]])
    lp = impl.logp_fwd(z, ids, -100)
    assert lp[0].tolist() == [0.0, 0.0, 0.0]
    assert lp[1, 0] == 0.0 and lp[1, 2] == 0.0 and lp[1, 1] != 0.0
    lp3 = impl.logp_fwd(z, ids, 3)        # an in-range ignore index is ignored too
    assert lp3[1].tolist() == [0.0, 0.0, 0.0]
    assert lp3[2, 0] != 0.0
    g = rng.normal(size=ids.shape)
    d = impl.logp_bwd(z, ids, g, -100)
    assert np.all(d[0] == 0.0)            # no valid id: exact zeros
    assert np.all(np.isfinite(d))


def _logp_loss(impl, ids, g, cap=0.0):
    def f(x):
        return float(np.sum(g * impl.logp_fwd(x[None, :], ids[None, :], -100, cap)[0]))
    return f


def check_logp_bwd_fd(impl):
    rng = np.random.default_rng(15)
    for cap in (0.0, 3.0):
        v = 9
        x = rng.normal(0, 2, size=v)
        ids = np.array([2, 5, 2, -100, 11, 0])          # duplicate, ignored, out of range
        g = rng.normal(size=ids.size)
        want = _fd(_logp_loss(impl, ids, g, cap), x)
        got = impl.logp_bwd(x[None, :], ids[None, :], g[None, :], -100, cap)[0]
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7), (cap, got, want)


def check_logp_bwd_rowsum(impl):
    rng = np.random.default_rng(16)
    z = rng.normal(0, 3, size=(4, 333))
    ids = rng.integers(0, 333, size=(4, 5))
    g = rng.normal(size=(4, 5))
    d = impl.logp_bwd(z, ids, g)
    assert np.allclose(d.sum(axis=1), 0.0, atol=1e-12)


def check_logp_bwd_vs_torch(impl):
    import torch
    rng = np.random.default_rng(17)
    z = rng.normal(0, 3, size=(3, 64))
    ids = rng.integers(0, 64, size=(3, 6))
    ids[1, 3] = ids[1, 1]                                # duplicate
    g = rng.normal(size=(3, 6))
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    lp = torch.log_softmax(zt, dim=1).gather(1, torch.tensor(ids))
    (lp * torch.tensor(g)).sum().backward()
    assert np.allclose(impl.logp_bwd(z, ids, g), zt.grad.numpy(), rtol=1e-12, atol=1e-12)


def check_logp_masked(impl):
    z = np.array([[0.0, -np.inf, 0.0, 1.0]])
    ids = np.array([[1]])
    assert impl.logp_fwd(z, ids)[0, 0] == -np.inf
    d = impl.logp_bwd(z, ids, np.array([[2.0]]))[0]
    assert d[1] == 2.0                                   # p = 0 at the -inf column
    assert np.all(np.isfinite(d))
    full = np.full((1, 5), -np.inf)
    assert np.isnan(impl.logp_fwd(full, np.array([[1]]))[0, 0])
    assert np.all(np.isnan(impl.logp_bwd(full, np.array([[1]]), np.array([[1.0]]))))
    assert impl.logp_fwd(full, np.array([[-100]]))[0, 0] == 0.0
    assert np.all(impl.logp_bwd(full, np.array([[-100]]), np.array([[1.0]])) == 0.0)


# ----------------------------------------------------------------------------
# entropy
# ----------------------------------------------------------------------------

def check_entropy_uniform(impl):
    for v in (1, 7, 32000):
        z = np.full((1, v), 0.125)
        assert abs(impl.entropy_fwd(z)[0] - math.log(v)) <= 1e-12 * max(1.0, math.log(v))
        d = impl.entropy_bwd(z, np.array([1.5]))
        assert np.allclose(d, 0.0, atol=1e-14)


def check_entropy_vs_scipy(impl):
    from scipy.stats import entropy
    rng = np.random.default_rng(21)
    z = rng.normal(0, 3, size=(4, 500))
    z[:, ::37] = -np.inf
    p = np.exp(z - z.max(axis=1, keepdims=True))
    want = entropy(p, axis=1)
    assert np.allclose(impl.entropy_fwd(z), want, rtol=1e-12, atol=1e-12)


def _entropy_loss(impl, g, cap=0.0):
    return lambda x: float(g * impl.entropy_fwd(x[None, :], cap)[0])


def check_entropy_bwd_fd(impl):
    rng = np.random.default_rng(22)
    for cap in (0.0, 2.5):
        x = rng.normal(0, 2, size=11)
        g = float(rng.normal())
        want = _fd(_entropy_loss(impl, g, cap), x)
        got = impl.entropy_bwd(x[None, :], np.array([g]), cap)[0]
        assert np.allclose(got, want, rtol=1e-6, atol=1e-7), (cap, got, want)
    x = rng.normal(0, 2, size=12)
    x[[3, 7]] = -np.inf                                   # masked columns: zero gradient there
    got = impl.entropy_bwd(x[None, :], np.array([1.0]))[0]
    assert got[3] == 0.0 and got[7] == 0.0
    keep = np.isfinite(x)
    sub = _fd(lambda y: float(impl.entropy_fwd(y[None, :])[0]), x[keep])
    assert np.allclose(got[keep], sub, rtol=1e-6, atol=1e-7)
    assert abs(got.sum()) < 1e-12


def check_entropy_masked(impl):
    assert np.isnan(impl.entropy_fwd(np.full((1, 4), -np.inf))[0])
    assert np.all(np.isnan(impl.entropy_bwd(np.full((1, 4), -np.inf), np.array([1.0]))))


# ----------------------------------------------------------------------------
# KL
# ----------------------------------------------------------------------------

def check_kl_self_zero(impl):
    rng = np.random.default_rng(31)
    z = rng.normal(0, 3, size=(3, 200))
    z[:, 5] = -np.inf
    for direction in ("reverse", "forward"):
        assert np.allclose(impl.kl_fwd(z, z, direction), 0.0, atol=1e-13)
        assert np.allclose(impl.kl_bwd(z, z, np.ones(3), direction), 0.0, atol=1e-14)


def check_kl_vs_scipy(impl):
    from scipy.stats import entropy
    rng = np.random.default_rng(32)
    a = rng.normal(0, 3, size=(4, 300))
    b = a + rng.normal(0, 0.5, size=(4, 300)) + 7.0
    pa = np.exp(a - a.max(axis=1, keepdims=True))
    pb = np.exp(b - b.max(axis=1, keepdims=True))
    assert np.allclose(impl.kl_fwd(a, b, "reverse"), entropy(pa, pb, axis=1), rtol=1e-10, atol=1e-13)
    assert np.allclose(impl.kl_fwd(a, b, "forward"), entropy(pb, pa, axis=1), rtol=1e-10, atol=1e-13)


def check_kl_gibbs_and_shift(impl):
    rng = np.random.default_rng(33)
    a = rng.normal(0, 3, size=(5, 64))
    b = rng.normal(0, 3, size=(5, 64))
    for direction in ("reverse", "forward"):
        kl = impl.kl_fwd(a, b, direction)
        assert np.all(kl > 0)
        shifted = impl.kl_fwd(a + 40.0, b - 13.0, direction)
        assert np.allclose(kl, shifted, rtol=1e-9, atol=1e-12)


def check_kl_mismatch(impl):
    a = np.array([[0.0, -200.0, 1.0]])        # p_a of column 1 underflows fp32, still supported
    b = np.array([[0.0, -np.inf, 1.0]])
    assert impl.kl_fwd(a, b, "reverse")[0] == np.inf
    assert np.all(np.isnan(impl.kl_bwd(a, b, np.ones(1), "reverse")))
    fwd = impl.kl_fwd(a, b, "forward")[0]
    assert np.isfinite(fwd) and fwd >= 0.0
    assert impl.kl_fwd(b, a, "forward")[0] == np.inf      # B supports what A masks
    assert np.all(np.isfinite(impl.kl_bwd(b, a, np.ones(1), "forward")))
    full = np.full((1, 3), -np.inf)
    for direction in ("reverse", "forward"):
        assert np.isnan(impl.kl_fwd(full, full, direction)[0])
        assert np.all(np.isnan(impl.kl_bwd(full, full, np.ones(1), direction)))


def check_kl_bwd_fd(impl):
    rng = np.random.default_rng(34)
    for direction in ("reverse", "forward"):
        for cap in (0.0, 2.0):
            a = rng.normal(0, 2, size=8)
            b = a + rng.normal(0, 1, size=8)
            g = float(rng.normal())
            f = lambda x: float(g * impl.kl_fwd(x[None, :], b[None, :], direction, cap)[0])  # noqa: E731
            want = _fd(f, a)
            got = impl.kl_bwd(a[None, :], b[None, :], np.array([g]), direction, cap)[0]
            assert np.allclose(got, want, rtol=1e-6, atol=1e-7), (direction, cap, got, want)


# ----------------------------------------------------------------------------
# softcap
# ----------------------------------------------------------------------------

def check_softcap_properties(impl):
    x = np.linspace(-400, 400, 2001)
    for c in (20.0, 30.0):
        y = impl.softcap(x, c)
        assert np.array_equal(impl.softcap(-x, c), -y)                  # odd
        assert np.all(np.abs(y) <= c) and np.all(np.abs(y[np.abs(x) < 100]) < c)
        small = np.array([1e-3, -2e-3, 1e-2])
        assert np.allclose(impl.softcap(small, c), small - small**3 / (3 * c * c), rtol=1e-12)


def check_softcap_grad_fd(impl):
    rng = np.random.default_rng(41)
    for c in (20.0, 30.0):
        x = rng.normal(0, c, size=9)
        gy = rng.normal(size=9)
        want = np.array([(impl.softcap(xi + 1e-6, c) - impl.softcap(xi - 1e-6, c)) / 2e-6 for xi in x]) * gy
        assert np.allclose(impl.softcap_grad(x, gy, c), want, rtol=1e-6, atol=1e-9)


def check_softcap_grad_cap_free(impl):
    u = np.linspace(-3, 3, 13)
    d20 = impl.softcap_grad(20.0 * u, np.ones_like(u), 20.0)
    d30 = impl.softcap_grad(30.0 * u, np.ones_like(u), 30.0)
    assert np.allclose(d20, d30, rtol=1e-14, atol=0)


# ---- fused linear head + logprobs (z = h @ W^T) ----

def _tiny_linear():
    h = np.array([[1.0, -2.0, 0.5], [0.0, 3.0, -1.0]])
    w = np.array([[2.0, 0.0, -1.0], [1.0, 1.0, 1.0], [-3.0, 0.5, 2.0], [0.0, -1.0, 4.0]])
    ids = np.array([[2], [0]])
    return h, w, ids


def check_linear_logp_brute_force(impl):
    """Dot products and log-sum-exp written out with Python's math on a 2 x 3 x 4 case."""
    h, w, ids = _tiny_linear()
    got = impl.linear_logp_fwd(h, w, ids)
    for i in range(2):
        z = [sum(h[i, d] * w[c, d] for d in range(3)) for c in range(4)]
        lse = max(z) + math.log(sum(math.exp(t - max(z)) for t in z))
        assert abs(got[i, 0] - (z[int(ids[i, 0])] - lse)) < 1e-12


def check_linear_logp_zero_hidden(impl):
    """h = 0 gives uniform logits: log p = -ln V for every valid id, 0 for ignored ones."""
    w = np.random.default_rng(3).standard_normal((37, 8))
    ids = np.array([[5, -100], [36, 0]])
    got = impl.linear_logp_fwd(np.zeros((2, 8)), w, ids)
    assert _close(got, [[-math.log(37), 0.0], [-math.log(37), -math.log(37)]])


def check_linear_logp_vs_torch(impl):
    """torch fp64 autograd of log_softmax(h @ W^T).gather: forward, dh and dW."""
    import torch
    rng = np.random.default_rng(11)
    h, w = rng.standard_normal((5, 6)), 0.7 * rng.standard_normal((9, 6))
    ids = np.array([[1, 1], [8, -100], [0, 3], [4, 4], [7, 2]])
    g = rng.standard_normal((5, 2))
    th, tw = torch.tensor(h, requires_grad=True), torch.tensor(w, requires_grad=True)
    tid = torch.tensor(np.where(ids < 0, 0, ids))
    lp = torch.log_softmax(th @ tw.T, dim=1).gather(1, tid) * torch.tensor(ids >= 0, dtype=torch.float64)
    (lp * torch.tensor(g)).sum().backward()
    assert _close(impl.linear_logp_fwd(h, w, ids), lp.detach().numpy(), rtol=1e-12, atol=1e-12)
    dh, dw = impl.linear_logp_bwd(h, w, ids, g)
    assert _close(dh, th.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert _close(dw, tw.grad.numpy(), rtol=1e-10, atol=1e-12)


def check_linear_logp_bwd_fd(impl):
    """Central finite differences of sum(g * logp) in h and in W."""
    h, w, ids = _tiny_linear()
    g = np.array([[0.7], [-1.3]])
    dh, dw = impl.linear_logp_bwd(h, w, ids, g)
    fh = _fd(lambda x: float(np.sum(g * impl.linear_logp_fwd(x, w, ids))), h.copy())
    fw = _fd(lambda x: float(np.sum(g * impl.linear_logp_fwd(h, x, ids))), w.copy())
    assert np.allclose(dh, fh, rtol=1e-6, atol=1e-7) and np.allclose(dw, fw, rtol=1e-6, atol=1e-7)


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
