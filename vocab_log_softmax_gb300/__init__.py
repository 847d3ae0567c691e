"""vocab_log_softmax_gb300: row-wise vocabulary log-softmax statistics on
GB300 (sm_103a).

Two layers over the CUDA library libvls (C ABI in include/vls.h):

* ``binding``: ``vls_*`` functions with the C ABI's names, argument
  marshalling only (tensors in, raw pointers to the library);
* the autograd functions below -- ``logprobs``, ``entropy``, ``kl`` and
  ``softcap`` -- which save the forward's per-row statistics so that each
  backward is one read of the logits and one write of the gradient.

Every computation runs in the library's kernels; there is no CPU or eager
fallback, and a missing library raises.
"""

from __future__ import annotations

import torch

from ._lib import VlsArgumentError, VlsDeviceError, VlsError  # noqa: F401
from .binding import (  # noqa: F401
    vls_check_device_error,
    vls_linear_logp_bwd,
    vls_linear_logp_fwd,
    vls_entropy_bwd,
    vls_entropy_fwd,
    vls_fused_bwd,
    vls_fused_fwd,
    vls_kl_bwd,
    vls_kl_fwd,
    vls_logp_bwd,
    vls_logp_fwd,
    vls_softcap_bwd,
    vls_softcap_fwd,
    vls_status_string,
    vls_version,
)

__all__ = ["logprobs", "entropy", "kl", "softcap", "stats", "linear_logprobs", "check_device_error"]


def check_device_error() -> None:
    """Raises VlsDeviceError if a bounded wait of a tensor-core kernel ran out
    on the current device since the last check (synchronises the device)."""
    vls_check_device_error()


def _addressable(rows: torch.Tensor) -> bool:
    """Whether the kernels can read a [N, V] or [B, T, V] view in place: every
    row stride at least V (broadcast rows, for one, are not)."""
    v = rows.shape[-1]
    return all(size <= 1 or stride >= v for size, stride in zip(rows.shape[:-1], rows.stride()[:-1]))


def _as_rows(x: torch.Tensor) -> torch.Tensor:
    """[..., V] -> a [N, V] view, or a [B, T, V] view read with two row strides
    (a slice such as ``x[:, :-1]`` stays in place); layouts the kernels cannot
    address, such as a strided vocabulary dimension, are copied first."""
    if x.dim() == 0:
        raise ValueError("expected at least one dimension (the vocabulary)")
    v = x.shape[-1]
    if x.dim() == 1:
        x = x.reshape(1, v)
    if v > 1 and x.stride(-1) != 1:
        x = x.contiguous()
    try:
        rows = x.view(-1, v)
    except RuntimeError:
        try:
            rows = x.view(-1, x.shape[-2], v)
        except RuntimeError:
            rows = x.reshape(-1, v)
    return rows if _addressable(rows) else rows.contiguous()


def _nrows(rows: torch.Tensor) -> int:
    return rows.shape[:-1].numel()


def _ids_rows(ids: torch.Tensor, n: int) -> torch.Tensor:
    """ids shaped like the logits' leading dims (k = 1) or with a trailing k -> [N, k] int64."""
    if n == 0 or ids.numel() % n != 0:
        if n == 0:
            return ids.reshape(0, ids.shape[-1] if ids.dim() > 0 else 1).to(torch.int64)
        raise ValueError(f"ids with {ids.numel()} elements do not divide into {n} rows")
    return ids.reshape(n, ids.numel() // n).to(torch.int64).contiguous()


def _cap(softcap) -> float:
    if softcap is None:
        return 0.0
    c = float(softcap)
    if not (c > 0.0 and c != float("inf")):
        raise ValueError("softcap must be finite and positive")
    return c


class _Logprobs(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, ids, ignore_index, cap):
        rows = _as_rows(logits)
        ids2 = _ids_rows(ids, _nrows(rows))
        logp, stats = vls_logp_fwd(rows, ids2, ignore_index, cap)
        ctx.save_for_backward(rows, ids2, stats)
        ctx.meta = (ignore_index, cap, logits.shape)
        return logp.reshape(ids.shape)

    @staticmethod
    def backward(ctx, grad):
        rows, ids2, stats = ctx.saved_tensors
        ignore_index, cap, shape = ctx.meta
        g = grad.reshape(ids2.shape).to(torch.float32).contiguous()
        d = vls_logp_bwd(rows, ids2, g, stats, ignore_index, cap)
        return d.reshape(shape), None, None, None


class _Entropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, cap):
        rows = _as_rows(logits)
        H, stats = vls_entropy_fwd(rows, cap)
        ctx.save_for_backward(rows, H, stats)
        ctx.meta = (cap, logits.shape)
        return H.reshape(logits.shape[:-1])

    @staticmethod
    def backward(ctx, grad):
        rows, H, stats = ctx.saved_tensors
        cap, shape = ctx.meta
        g = grad.reshape(-1).to(torch.float32).contiguous()
        return vls_entropy_bwd(rows, g, H, stats, cap).reshape(shape), None


class _KL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, policy, reference, direction, cap):
        a, b = _as_rows(policy), _as_rows(reference.detach())
        kl, sa, sb = vls_kl_fwd(a, b, direction, cap)
        ctx.save_for_backward(a, b, kl, sa, sb)
        ctx.meta = (direction, cap, policy.shape)
        return kl.reshape(policy.shape[:-1])

    @staticmethod
    def backward(ctx, grad):
        a, b, kl, sa, sb = ctx.saved_tensors
        direction, cap, shape = ctx.meta
        g = grad.reshape(-1).to(torch.float32).contiguous()
        return vls_kl_bwd(a, b, g, kl, sa, sb, direction, cap).reshape(shape), None, None, None


class _Softcap(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, cap):
        xc = x.contiguous()
        ctx.save_for_backward(xc)
        ctx.cap = cap
        return vls_softcap_fwd(xc, cap)

    @staticmethod
    def backward(ctx, gy):
        (xc,) = ctx.saved_tensors
        if gy.dtype not in (torch.float32, xc.dtype):
            gy = gy.to(torch.float32)
        return vls_softcap_bwd(xc, gy.contiguous(), ctx.cap), None


class _Stats(torch.autograd.Function):
    @staticmethod
    def forward(ctx, policy, reference, ids, direction, ignore_index, cap):
        a = _as_rows(policy)
        b = _as_rows(reference.detach()) if reference is not None else None
        ids2 = None
        if ids is not None:
            ids2 = _ids_rows(ids, _nrows(a))
        out = vls_fused_fwd(a, b, ids2, logp=ids is not None, entropy=True, direction=direction,
                            ignore_index=ignore_index, cap=cap)
        ctx.save_for_backward(a, b, ids2, out["stats_a"], out.get("stats_b"), out["H"], out.get("kl"))
        ctx.meta = (direction, ignore_index, cap, policy.shape, ids.shape if ids is not None else None)
        lead = policy.shape[:-1]
        empty = a.new_empty(0, dtype=torch.float32)
        logp = out["logp"].reshape(ids.shape) if ids is not None else empty
        klv = out["kl"].reshape(lead) if b is not None else empty
        return logp, out["H"].reshape(lead), klv

    @staticmethod
    def backward(ctx, g_logp, g_H, g_kl):
        a, b, ids2, sa, sb, H, kl = ctx.saved_tensors
        direction, ignore_index, cap, shape, ids_shape = ctx.meta
        f32 = lambda g, shp: None if g is None else g.reshape(shp).to(torch.float32).contiguous()  # noqa: E731
        gl = f32(g_logp, ids2.shape) if ids2 is not None else None
        gh = f32(g_H, (-1,))
        gk = f32(g_kl, (-1,)) if b is not None else None
        if gl is None and gh is None and gk is None:
            return None, None, None, None, None, None
        fwd = {"stats_a": sa, "stats_b": sb, "H": H, "kl": kl}
        da = vls_fused_bwd(a, fwd, b, ids2, g_logp=gl, g_H=gh, g_kl=gk, direction=direction,
                           ignore_index=ignore_index, cap=cap)
        return da.reshape(shape), None, None, None, None, None


def stats(policy: torch.Tensor, ids: torch.Tensor | None = None, reference: torch.Tensor | None = None,
          direction: str = "reverse", ignore_index: int = -100, softcap: float | None = None):
    """(logp, entropy, kl) of softmax(softcap(policy)) from one read of the
    policy (and one of the reference): logp like ``logprobs`` (empty without
    ids), entropy per row, KL against the detached reference (empty without
    one).  The backward of any weighted sum of the three is one pass."""
    if direction not in ("reverse", "forward"):
        raise ValueError("direction must be 'reverse' or 'forward'")
    return _Stats.apply(policy, reference, ids, direction, int(ignore_index), _cap(softcap))


def logprobs(logits: torch.Tensor, ids: torch.Tensor, ignore_index: int = -100,
             softcap: float | None = None) -> torch.Tensor:
    """log_softmax(softcap(logits))[..., ids]: fp32, shaped like ``ids`` ([..., k] or [...]).

    Ids equal to ``ignore_index`` or outside [0, V) give 0 and no gradient.
    """
    return _Logprobs.apply(logits, ids, int(ignore_index), _cap(softcap))


def entropy(logits: torch.Tensor, softcap: float | None = None) -> torch.Tensor:
    """Entropy of softmax(softcap(logits)) per row (fp32, shape logits.shape[:-1])."""
    return _Entropy.apply(logits, _cap(softcap))


def kl(policy: torch.Tensor, reference: torch.Tensor, direction: str = "reverse",
       softcap: float | None = None) -> torch.Tensor:
    """Per-row KL between softmax(policy) and softmax(reference).

    ``direction="reverse"``: KL(p_policy || p_reference); ``"forward"``:
    KL(p_reference || p_policy).  The gradient flows to ``policy`` only.
    """
    if direction not in ("reverse", "forward"):
        raise ValueError("direction must be 'reverse' or 'forward'")
    return _KL.apply(policy, reference, direction, _cap(softcap))


def softcap(x: torch.Tensor, cap: float = 30.0) -> torch.Tensor:
    """cap * tanh(x / cap), elementwise, in x's dtype."""
    return _Softcap.apply(x, _cap(cap))


class _LinearLogprobs(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, ids, ignore_index, check):
        h = hidden.reshape(-1, hidden.shape[-1])
        if h.shape[-1] > 1 and h.stride(-1) != 1:
            h = h.contiguous()
        w = weight if weight.stride(-1) == 1 else weight.contiguous()
        ids2 = _ids_rows(ids, h.shape[0])
        logp, st, _ = vls_linear_logp_fwd(h, w, ids2, ignore_index, check=check)
        ctx.save_for_backward(h, w, ids2, st)
        ctx.meta = (ignore_index, hidden.shape, check)
        return logp.reshape(ids.shape)

    @staticmethod
    def backward(ctx, grad):
        h, w, ids2, st = ctx.saved_tensors
        ignore_index, shape, check = ctx.meta
        g = grad.reshape(ids2.shape).to(torch.float32).contiguous()
        dh, dw, _ = vls_linear_logp_bwd(h, w, ids2, g, st, ignore_index, check=check)
        return dh.reshape(shape), dw, None, None, None


def linear_logprobs(hidden: torch.Tensor, weight: torch.Tensor, ids: torch.Tensor,
                    ignore_index: int = -100, check: bool = True) -> torch.Tensor:
    """log_softmax(hidden @ weight^T)[..., ids] without storing the logits.

    hidden: [..., D] and weight: [V, D], both bfloat16 or both float16; ids
    shaped like hidden's leading dims ([...] or [..., k], k <= 16).  The
    gradient flows to hidden and weight.

    Every wait inside the tensor-core kernels is bounded; one that runs out
    makes the kernel return early with invalid outputs and sets a status
    word.  With check=True (the default) the forward and the backward each
    synchronise the device after their kernels, read that word and raise
    VlsDeviceError when it is set.  check=False skips the synchronisation
    (the calls stay asynchronous); ``check_device_error()`` then reports
    the same failures later, for any number of calls at once.
    """
    return _LinearLogprobs.apply(hidden, weight, ids, int(ignore_index), bool(check))
