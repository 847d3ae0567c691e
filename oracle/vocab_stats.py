"""Plain CPU fp64 oracle for row-wise vocabulary log-softmax statistics.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may call it.  It shares no code with
the CUDA library and imports nothing from it.

Every function works on float64 numpy arrays, one row at a time, with the
plain two-pass definition (max, then sum of exponentials) rather than the
single-pass online statistics the GPU uses: both reach the same value up to
rounding, and the two-pass form is the one a reader can check by eye.

Sources (titles of the pages the method is described on):

* "Final Logit Softcap" (RL-Kernel operator docs), section Summary:
  ``y = c*tanh(x/c)`` and ``dy/dx = 1 - tanh^2(x/c)``; section Accuracy and
  Invariance: the fp64 reference derivative is written ``1/cosh^2(x/c)``.
* "Add Triton kernels for vocab-parallel logprobs, entropy and KL"
  (DeepSpeed PR #8838), section Changes: target log-probabilities and the
  logprob backward ``g*(one_hot - softmax)`` with top-k one-hot terms;
  section Tests: all -inf rows, support mismatch, duplicate / ignored top-k
  ids; review "Suggested change": ``H = log S - W/S`` and
  ``KL = W/S_A - log S_A + log S_B`` with sums centred on the max, and the
  support-mismatch flag decided on the logits.
* "perf(logp): fused zero-workspace backward for the generic CUDA fused
  logp" (RL-Kernel PR #495), sections Summary and Behavior changes:
  ``dlogits = grad*(one_hot - softmax)``; targets outside ``[0, V)``
  (including the ignore index -100) give log-probability 0 and an exactly
  zero gradient row.

Readings where the pages are silent (each also listed in the design notes):

* A row whose logits are all -inf has no distribution: every statistic of
  it is NaN and its gradient row is NaN.  The one exception is a logprob
  row whose ids are all ignored: 0 and a zero gradient row, as for any
  row without a valid id.
* Reverse KL(A||B) with a column where A is finite and B is -inf is +inf;
  its gradient row is NaN (the derivative needs inf - inf).  Forward
  KL(B||A) with a column where B is finite and A is -inf is +inf; its
  gradient ``g*(p_A - p_B)`` stays finite.  A KL of a row where either
  tensor is all -inf is NaN, with a NaN gradient row.
* With a softcap, -inf logits become ``c*tanh(-inf) = -c``: the cap is
  applied first and masks are seen through it.
* Top-k ids: each id's log-probability is reported at its own position;
  duplicate valid ids add their upstream gradients in the one-hot term,
  and the softmax term is weighted by the sum of all valid upstream
  gradients.  With k = 1 this is ``g*(one_hot - softmax)``.

* Fused linear + logprobs: the pages name a ``linear_logp`` op ("perf(logp):
  fused zero-workspace backward ...", RL-Kernel PR #495, Summary, listed as
  not touched) without defining it.  The plainest reading is the target
  log-probabilities of the logits a linear vocabulary head produces,
  ``z = h @ W^T`` (h: [N, D] hidden states, W: [V, D] head weights), with
  the gradient flowing to both h and W.

Parity pins for every function here are the checks in ``tests/oracle_pins.py``
(closed forms, library routines, invariants, finite differences), run by
``tests/test_oracle.py``; ``tests/test_oracle_mutations.py`` plants mistakes in
a copy of this module and checks that a pin catches each.
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


# ----------------------------------------------------------------------------
# input decoding
# ----------------------------------------------------------------------------

def decode_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16 / int16) -> exact float64 values.

    A bfloat16 is the high half of an IEEE float32, so shifting the 16 bits
    into the top of a 32-bit word gives the float32 with the same value.
    """
    u16 = np.asarray(bits).view(np.uint16).astype(np.uint32)
    with np.errstate(invalid="ignore"):
        return (u16 << np.uint32(16)).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# softcap  ("Final Logit Softcap", Summary)
# ----------------------------------------------------------------------------

def softcap(x: np.ndarray, cap: float) -> np.ndarray:
    """y = c * tanh(x / c), elementwise, in float64."""
    x = np.asarray(x, dtype=np.float64)
    return cap * np.tanh(x / cap)


def softcap_grad(x: np.ndarray, gy: np.ndarray, cap: float) -> np.ndarray:
    """g_x = g_y * (1 - tanh^2(x/c)), written as g_y / cosh^2(x/c).

    The 1/cosh^2 form is the one the page's fp64 reference uses
    ("Final Logit Softcap", Accuracy and Invariance); the cap cancels.
    """
    x = np.asarray(x, dtype=np.float64)
    gy = np.asarray(gy, dtype=np.float64)
    with np.errstate(over="ignore"):
        ch = np.cosh(x / cap)
    return gy / (ch * ch)


def _apply_cap(x: np.ndarray, cap: float) -> np.ndarray:
    """The row seen by the softmax: the raw logits, or their softcap if cap > 0."""
    return softcap(x, cap) if cap > 0.0 else np.asarray(x, dtype=np.float64)


def _cap_chain(x: np.ndarray, cap: float) -> np.ndarray:
    """dz/dx for z = softcap(x) (1 when there is no cap)."""
    if cap > 0.0:
        return softcap_grad(x, np.ones_like(x, dtype=np.float64), cap)
    return np.ones_like(x, dtype=np.float64)


# ----------------------------------------------------------------------------
# per-row softmax statistics (two-pass definition)
# ----------------------------------------------------------------------------

def row_stats(z: np.ndarray) -> tuple[float, float]:
    """(m, log S) of one row: m = max_j z_j, S = sum over finite z_j of exp(z_j - m).

    A row with no finite entry has m = -inf; its log S is reported as NaN
    (the row has no distribution).
    """
    z = np.asarray(z, dtype=np.float64)
    m = float(np.max(z)) if z.size else NEG_INF
    if m == NEG_INF:
        return NEG_INF, float("nan")
    finite = z > NEG_INF
    s = float(np.sum(np.exp(z[finite] - m)))
    return m, float(np.log(s))


def row_log_softmax(z: np.ndarray) -> np.ndarray:
    """log p_j = (z_j - m) - log S; -inf where z_j = -inf; NaN for an all -inf row."""
    m, log_s = row_stats(z)
    if m == NEG_INF:
        return np.full(z.shape, np.nan)
    with np.errstate(invalid="ignore"):
        return (np.asarray(z, dtype=np.float64) - m) - log_s


def is_valid_id(i: int, vocab: int, ignore_index: int) -> bool:
    """An id takes part iff it is not the ignore index and lies in [0, V)
    ("perf(logp): fused zero-workspace backward ...", Behavior changes)."""
    return i != ignore_index and 0 <= i < vocab


# ----------------------------------------------------------------------------
# target log-probabilities
# ----------------------------------------------------------------------------

def logp_fwd(logits: np.ndarray, ids: np.ndarray, ignore_index: int = -100,
             cap: float = 0.0) -> np.ndarray:
    """logp[i, j] = log_softmax(z_i)[ids[i, j]] for valid ids, exactly 0 otherwise.

    logits: [N, V] float64 (already decoded); ids: [N, k] integers.
    DeepSpeed PR #8838, Changes; RL-Kernel PR #495, Behavior changes.
    """
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    ids = np.asarray(ids).reshape(logits.shape[0], -1)
    n, v = logits.shape
    out = np.zeros(ids.shape, dtype=np.float64)
    for i in range(n):
        valid = [j for j in range(ids.shape[1]) if is_valid_id(int(ids[i, j]), v, ignore_index)]
        if not valid:
            continue
        lp = row_log_softmax(_apply_cap(logits[i], cap))
        for j in valid:
            out[i, j] = lp[int(ids[i, j])]
    return out


def logp_bwd(logits: np.ndarray, ids: np.ndarray, g: np.ndarray,
             ignore_index: int = -100, cap: float = 0.0) -> np.ndarray:
    """Vector-Jacobian product of logp_fwd: d logits for upstream g [N, k].

    Row i: d_c = sum over valid j with ids[i,j] = c of g[i,j]  -  G * p_c,
    G = sum over valid j of g[i,j], p = softmax(z_i).  A row without a valid
    id is exactly zero.  With a cap the result is multiplied by dz/dx.
    DeepSpeed PR #8838, Changes (top-k one-hot terms); RL-Kernel PR #495,
    Summary (grad * (one_hot - softmax)) and Behavior changes (zero rows).
    """
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    ids = np.asarray(ids).reshape(logits.shape[0], -1)
    g = np.asarray(g, dtype=np.float64).reshape(ids.shape)
    n, v = logits.shape
    d = np.zeros((n, v), dtype=np.float64)
    for i in range(n):
        valid = [j for j in range(ids.shape[1]) if is_valid_id(int(ids[i, j]), v, ignore_index)]
        if not valid:
            continue
        z = _apply_cap(logits[i], cap)
        with np.errstate(invalid="ignore"):
            p = np.exp(row_log_softmax(z))
        one_hot = np.zeros(v, dtype=np.float64)
        total = 0.0
        for j in valid:                      # ascending j
            one_hot[int(ids[i, j])] += g[i, j]
            total += g[i, j]
        with np.errstate(invalid="ignore"):
            d[i] = (one_hot - total * p) * _cap_chain(logits[i], cap)
    return d


# ----------------------------------------------------------------------------
# entropy  (DeepSpeed PR #8838, review "Suggested change")
# ----------------------------------------------------------------------------

def entropy_fwd(logits: np.ndarray, cap: float = 0.0) -> np.ndarray:
    """H_i = -sum over finite z_j of p_j log p_j  (0 log 0 := 0); NaN for an all -inf row."""
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    out = np.empty(logits.shape[0], dtype=np.float64)
    for i in range(logits.shape[0]):
        z = _apply_cap(logits[i], cap)
        lp = row_log_softmax(z)
        finite = z > NEG_INF
        if not np.any(finite):
            out[i] = np.nan
            continue
        out[i] = -float(np.sum(np.exp(lp[finite]) * lp[finite]))
    return out


def entropy_bwd(logits: np.ndarray, g: np.ndarray, cap: float = 0.0) -> np.ndarray:
    """dH/dz_c = -p_c (log p_c + H), times g[i] (and dz/dx with a cap).

    0 on -inf columns; a NaN row for an all -inf row.  The derivative is not
    printed on the pages; it follows from H = -sum p log p and
    dp_c/dz_j = p_c (delta_cj - p_j).
    """
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    g = np.asarray(g, dtype=np.float64).reshape(-1)
    h = entropy_fwd(logits, cap)
    d = np.zeros(logits.shape, dtype=np.float64)
    for i in range(logits.shape[0]):
        if np.isnan(h[i]):
            d[i] = np.nan
            continue
        z = _apply_cap(logits[i], cap)
        lp = row_log_softmax(z)
        finite = z > NEG_INF
        row = np.zeros(z.shape, dtype=np.float64)
        p = np.exp(lp[finite])
        row[finite] = -g[i] * p * (lp[finite] + h[i])
        d[i] = row * _cap_chain(logits[i], cap)
    return d


# ----------------------------------------------------------------------------
# KL divergence  (DeepSpeed PR #8838, review "Suggested change")
# ----------------------------------------------------------------------------

def _kl_row(first: np.ndarray, second: np.ndarray) -> float:
    """KL(P_first || P_second) = sum over first_j > -inf of p_j (log p_j - log q_j).

    NaN if either row is all -inf; +inf if some column has first finite and
    second -inf (support mismatch, decided on the logits).
    """
    if not np.any(first > NEG_INF) or not np.any(second > NEG_INF):
        return float("nan")
    support = first > NEG_INF
    if np.any(support & (second == NEG_INF)):
        return float("inf")
    lp = row_log_softmax(first)
    lq = row_log_softmax(second)
    return float(np.sum(np.exp(lp[support]) * (lp[support] - lq[support])))


def kl_fwd(a: np.ndarray, b: np.ndarray, direction: str = "reverse",
           cap: float = 0.0) -> np.ndarray:
    """Per-row KL between softmax(a) (policy) and softmax(b) (reference).

    direction "reverse": KL(p_a || p_b); "forward": KL(p_b || p_a).
    """
    a = np.atleast_2d(np.asarray(a, dtype=np.float64))
    b = np.atleast_2d(np.asarray(b, dtype=np.float64))
    out = np.empty(a.shape[0], dtype=np.float64)
    for i in range(a.shape[0]):
        za, zb = _apply_cap(a[i], cap), _apply_cap(b[i], cap)
        out[i] = _kl_row(za, zb) if direction == "reverse" else _kl_row(zb, za)
    return out


def kl_bwd(a: np.ndarray, b: np.ndarray, g: np.ndarray, direction: str = "reverse",
           cap: float = 0.0) -> np.ndarray:
    """Gradient of g[i] * KL_i with respect to the policy logits a (b is detached).

    reverse KL(p_a||p_b): d_c = g p_a,c ((log p_a,c - log p_b,c) - KL), 0 where
    a_c = -inf, and a NaN row when KL is +inf or NaN.
    forward KL(p_b||p_a): d_c = g (p_a,c - p_b,c), a NaN row only when a row
    of a or b is all -inf.
    Neither derivative is printed on the pages; both follow from
    dp_c/dz_j = p_c (delta_cj - p_j).
    """
    a = np.atleast_2d(np.asarray(a, dtype=np.float64))
    b = np.atleast_2d(np.asarray(b, dtype=np.float64))
    g = np.asarray(g, dtype=np.float64).reshape(-1)
    kl = kl_fwd(a, b, direction, cap)
    d = np.zeros(a.shape, dtype=np.float64)
    for i in range(a.shape[0]):
        za, zb = _apply_cap(a[i], cap), _apply_cap(b[i], cap)
        if np.isnan(kl[i]):
            d[i] = np.nan
            continue
        lpa, lpb = row_log_softmax(za), row_log_softmax(zb)
        if direction == "reverse":
            if np.isinf(kl[i]):
                d[i] = np.nan
                continue
            sup = za > NEG_INF
            row = np.zeros(za.shape, dtype=np.float64)
            row[sup] = g[i] * np.exp(lpa[sup]) * ((lpa[sup] - lpb[sup]) - kl[i])
        else:
            row = g[i] * (np.exp(lpa) - np.exp(lpb))
        d[i] = row * _cap_chain(a[i], cap)
    return d


# ----------------------------------------------------------------------------
# fused linear head + target log-probabilities (reading: z = h @ W^T)
# ----------------------------------------------------------------------------

def linear_logits(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """z = h @ W^T in float64: h [N, D], W [V, D] -> [N, V]."""
    h = np.atleast_2d(np.asarray(h, dtype=np.float64))
    w = np.atleast_2d(np.asarray(w, dtype=np.float64))
    return h @ w.T


def linear_logp_fwd(h: np.ndarray, w: np.ndarray, ids: np.ndarray, ignore_index: int = -100) -> np.ndarray:
    """logp_fwd of the logits z = h @ W^T (never formed on the GPU)."""
    return logp_fwd(linear_logits(h, w), ids, ignore_index)


def linear_logp_bwd(h: np.ndarray, w: np.ndarray, ids: np.ndarray, g: np.ndarray,
                    ignore_index: int = -100) -> tuple[np.ndarray, np.ndarray]:
    """(dh, dW) for upstream g [N, k]: with dz = logp_bwd(z, ids, g) [N, V],
    dh = dz @ W and dW = dz^T @ h (the chain rule through z = h @ W^T)."""
    h = np.atleast_2d(np.asarray(h, dtype=np.float64))
    w = np.atleast_2d(np.asarray(w, dtype=np.float64))
    dz = logp_bwd(linear_logits(h, w), ids, g, ignore_index)
    return dz @ w, dz.T @ h
