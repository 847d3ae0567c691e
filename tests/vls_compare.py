"""Comparison rules between the CUDA path and the CPU fp64 oracle.

* fp32 forward outputs (logp, H, KL): |gpu - ref| <= 1e-5 + 1e-5 |ref|.
* bf16 gradients and bf16 softcap outputs: |gpu - ref| <= ulp_bf16(ref) + 1e-6,
  ulp_bf16(r) = 2^(floor(log2 |r|) - 7) (one unit in the last place of a
  bfloat16 with magnitude |r|).
* fp16 gradients and fp16 softcap outputs: the same rule with one float16
  unit, ulp_f16(r) = 2^(max(floor(log2 |r|), -14) - 10) (the float16 spacing,
  2^-24 in the subnormal range).
* fp32 gradients and fp32 softcap outputs: 1e-5 + 1e-5 |ref|.
* Non-finite values match exactly: NaN, +inf and -inf in the same places.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle

FWD_RTOL = 1e-5
FWD_ATOL = 1e-5
BF16_ATOL = 1e-6


def to_f64(t) -> np.ndarray:
    """Exact float64 copy of a CPU/GPU tensor (bf16 decoded bit for bit)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return oracle.decode_bf16_bits(t.view(torch.int16).numpy())
    return t.to(torch.float64).numpy()


def _nonfinite_match(got: np.ndarray, ref: np.ndarray, what: str) -> np.ndarray:
    for name, f in (("NaN", np.isnan), ("+inf", np.isposinf), ("-inf", np.isneginf)):
        g, r = f(got), f(ref)
        if not np.array_equal(g, r):
            idx = np.argwhere(g != r)[:5]
            raise AssertionError(f"{what}: {name} pattern differs at {idx.tolist()} "
                                 f"(gpu {got[tuple(idx[0])]!r}, ref {ref[tuple(idx[0])]!r})")
    return np.isfinite(ref)


def _report(what, got, ref, tol, fin):
    err = np.abs(got[fin] - ref[fin])
    bad = err > tol
    if np.any(bad):
        i = np.argmax(err - tol)
        pos = np.argwhere(fin)[i].tolist()
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} values out of tolerance; worst at {pos}: "
            f"gpu {got[fin][i]!r} ref {ref[fin][i]!r} err {err[i]:.3e} tol {tol[i]:.3e}")


def assert_fp32_close(got, ref, what: str = "", rtol: float = FWD_RTOL, atol=FWD_ATOL):
    """atol may be an array that broadcasts against ref (a per-row bound)."""
    got, ref = to_f64(got), np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    fin = _nonfinite_match(got, ref, what)
    atol = np.broadcast_to(np.asarray(atol, dtype=np.float64), ref.shape)[fin]
    _report(what, got, ref, atol + rtol * np.abs(ref[fin]), fin)


def ulp_bf16(r: np.ndarray) -> np.ndarray:
    a = np.abs(r)
    out = np.zeros_like(a)
    nz = a > 0
    out[nz] = np.exp2(np.floor(np.log2(a[nz])) - 7.0)
    return out


def ulp_f16(r: np.ndarray) -> np.ndarray:
    a = np.abs(r)
    out = np.full_like(a, 2.0 ** -24)
    nz = a > 0
    out[nz] = np.exp2(np.maximum(np.floor(np.log2(a[nz])), -14.0) - 10.0)
    return out


def assert_grad_close(got: torch.Tensor, ref, what: str = ""):
    """Gradient / softcap-output rule for the tensor's own dtype."""
    ref = np.asarray(ref, dtype=np.float64)
    if got.dtype in (torch.bfloat16, torch.float16):
        g = to_f64(got)
        assert g.shape == ref.shape, (what, g.shape, ref.shape)
        fin = _nonfinite_match(g, ref, what)
        ulp = ulp_bf16 if got.dtype == torch.bfloat16 else ulp_f16
        _report(what, g, ref, ulp(ref[fin]) + BF16_ATOL, fin)
    else:
        assert_fp32_close(got, ref, what)


def bitwise_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bit-for-bit equality (NaNs with equal payloads compare equal)."""
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    ia = a.detach().contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.detach().contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32)
    return bool(torch.equal(ia, ib))
