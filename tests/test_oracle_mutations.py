"""Plausible mistakes planted in a copy of the oracle (on the CPU) must each
fail at least one pin.  This is what makes the pins trustworthy."""

import types

import numpy as np
import pytest

import oracle
import oracle_pins
from oracle import vocab_stats as vs


def _mutant(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(oracle, k) for k in dir(oracle) if not k.startswith("_")})
    for k, v in overrides.items():
        setattr(ns, k, v)
    return ns


def _fails_some_pin(impl):
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(impl)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            return True
    return False


def _logp_bwd_without_softmax_term(logits, ids, g, ignore_index=-100, cap=0.0):
    logits = np.atleast_2d(logits)
    ids = np.asarray(ids).reshape(logits.shape[0], -1)
    g = np.asarray(g, dtype=np.float64).reshape(ids.shape)
    d = np.zeros(logits.shape)
    for i in range(logits.shape[0]):
        for j in range(ids.shape[1]):
            if vs.is_valid_id(int(ids[i, j]), logits.shape[1], ignore_index):
                d[i, int(ids[i, j])] += g[i, j]
    return d


def _logp_bwd_sign_flip(logits, ids, g, ignore_index=-100, cap=0.0):
    return -vs.logp_bwd(logits, ids, g, ignore_index, cap)


def _logp_bwd_first_g_only(logits, ids, g, ignore_index=-100, cap=0.0):
    # weights the softmax term by the first upstream gradient instead of their sum
    g = np.asarray(g, dtype=np.float64).reshape(np.asarray(ids).shape)
    g_first = np.zeros_like(g)
    g_first[:, 0] = g[:, 0]
    softmax_term = (vs.logp_bwd(logits, ids, g_first, ignore_index)
                    - _logp_bwd_without_softmax_term(logits, ids, g_first, ignore_index))
    return _logp_bwd_without_softmax_term(logits, ids, g, ignore_index) + softmax_term


def _logp_fwd_no_max(logits, ids, ignore_index=-100, cap=0.0):
    out = vs.logp_fwd(logits, ids, ignore_index, cap)
    m = np.max(np.atleast_2d(logits), axis=1, keepdims=True)
    return np.where(out != 0.0, out + m, out)


def _logp_fwd_ignore_only_minus100(logits, ids, ignore_index=-100, cap=0.0):
    ids = np.where(np.asarray(ids) == ignore_index, ignore_index, np.asarray(ids) % np.atleast_2d(logits).shape[1])
    return vs.logp_fwd(logits, ids, ignore_index, cap)


def _entropy_bwd_minus_h(logits, g, cap=0.0):
    logits = np.atleast_2d(logits)
    h = vs.entropy_fwd(logits, cap)
    out = vs.entropy_bwd(logits, g, cap)
    # d = -g p (log p - H) instead of -g p (log p + H)
    p = np.exp(np.array([vs.row_log_softmax(r) for r in logits]))
    return out + 2.0 * np.asarray(g).reshape(-1, 1) * p * h.reshape(-1, 1)


def _entropy_fwd_natural_sum(logits, cap=0.0):
    # forgets the minus sign
    return -vs.entropy_fwd(logits, cap)


def _kl_fwd_swapped(a, b, direction="reverse", cap=0.0):
    return vs.kl_fwd(a, b, "forward" if direction == "reverse" else "reverse", cap)


def _kl_bwd_swapped(a, b, g, direction="reverse", cap=0.0):
    return vs.kl_bwd(a, b, g, "forward" if direction == "reverse" else "reverse", cap)


def _kl_fwd_no_mismatch(a, b, direction="reverse", cap=0.0):
    a2 = np.where(np.isneginf(a), -1e30, a)
    b2 = np.where(np.isneginf(b), -1e30, b)
    return vs.kl_fwd(a2, b2, direction, cap)


def _kl_bwd_without_kl_term(a, b, g, direction="reverse", cap=0.0):
    out = vs.kl_bwd(a, b, g, direction, cap)
    if direction != "reverse":
        return out
    kl = vs.kl_fwd(a, b, direction, cap)
    pa = np.exp(np.array([vs.row_log_softmax(r) for r in np.atleast_2d(a)]))
    return out + np.asarray(g).reshape(-1, 1) * pa * kl.reshape(-1, 1)


def _softcap_grad_no_square(x, gy, cap):
    return np.asarray(gy) * (1.0 - np.abs(np.tanh(np.asarray(x) / cap)))


def _softcap_grad_keeps_cap(x, gy, cap):
    return cap * vs.softcap_grad(x, gy, cap)


def _softcap_no_outer_cap(x, cap):
    return np.tanh(np.asarray(x, dtype=np.float64) / cap)


def _linear_logp_fwd_scaled(h, w, ids, ignore_index=-100):
    # logits scaled by 1/sqrt(D), as an attention score would be
    h = np.atleast_2d(np.asarray(h, dtype=np.float64))
    return vs.logp_fwd(vs.linear_logits(h, w) / np.sqrt(h.shape[1]), ids, ignore_index)


def _linear_logp_bwd_dw_rows_reversed(h, w, ids, g, ignore_index=-100):
    # the vocabulary index of dW taken in the wrong order
    dh, dw = vs.linear_logp_bwd(h, w, ids, g, ignore_index)
    return dh, dw[::-1]


def _linear_logp_bwd_dh_without_softmax(h, w, ids, g, ignore_index=-100):
    # dh from the one-hot term only
    z = vs.linear_logits(h, w)
    dz = _logp_bwd_without_softmax_term(z, ids, g, ignore_index)
    return dz @ np.asarray(w, dtype=np.float64), vs.linear_logp_bwd(h, w, ids, g, ignore_index)[1]


MUTANTS = {
    "linear_logp_fwd: logits scaled by 1/sqrt(D)": dict(linear_logp_fwd=_linear_logp_fwd_scaled),
    "linear_logp_bwd: dW vocabulary rows reversed": dict(linear_logp_bwd=_linear_logp_bwd_dw_rows_reversed),
    "linear_logp_bwd: dh without the softmax term": dict(linear_logp_bwd=_linear_logp_bwd_dh_without_softmax),
    "logp_bwd: softmax term dropped": dict(logp_bwd=_logp_bwd_without_softmax_term),
    "logp_bwd: sign flipped": dict(logp_bwd=_logp_bwd_sign_flip),
    "logp_bwd: softmax weight = first g": dict(logp_bwd=_logp_bwd_first_g_only),
    "logp_fwd: max not subtracted": dict(logp_fwd=_logp_fwd_no_max),
    "logp_fwd: out-of-range ids wrapped": dict(logp_fwd=_logp_fwd_ignore_only_minus100),
    "entropy_bwd: -H instead of +H": dict(entropy_bwd=_entropy_bwd_minus_h),
    "entropy_fwd: sign dropped": dict(entropy_fwd=_entropy_fwd_natural_sum),
    "kl_fwd: directions swapped": dict(kl_fwd=_kl_fwd_swapped),
    "kl_bwd: directions swapped": dict(kl_bwd=_kl_bwd_swapped),
    "kl_fwd: support mismatch ignored": dict(kl_fwd=_kl_fwd_no_mismatch),
    "kl_bwd: -KL term dropped": dict(kl_bwd=_kl_bwd_without_kl_term),
    "softcap_grad: 1-|tanh| instead of 1-tanh^2": dict(softcap_grad=_softcap_grad_no_square),
    "softcap_grad: cap not cancelled": dict(softcap_grad=_softcap_grad_keeps_cap),
    "softcap: outer cap dropped": dict(softcap=_softcap_no_outer_cap),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert _fails_some_pin(_mutant(**MUTANTS[name])), name


def test_real_oracle_passes_all_pins():
    assert not _fails_some_pin(_mutant())
