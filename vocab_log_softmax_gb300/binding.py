"""Thin torch binding of the C ABI: one function per ``vls_*`` entry point,
same names, argument marshalling only.

Each function takes CUDA tensors, allocates its outputs with torch when they
are not given, and passes raw pointers, sizes and the current CUDA stream of
the inputs' device to libvls.  No arithmetic of the method happens here.

Row layout: a logits tensor is [N, V], or [B, T, V] read as N = B*T rows,
with a contiguous last dimension.  Its row strides may exceed V, so slices
such as ``logits[:, :V]`` or ``logits[:, :-1, :]`` are read in place through
the C ABI's two-stride row descriptor (vls_rows).  Gradients are returned
contiguous [N, V].
"""

from __future__ import annotations

import torch

from . import _lib

_DT = {torch.float32: _lib.VLS_F32, torch.bfloat16: _lib.VLS_BF16, torch.float16: _lib.VLS_F16}
_DIR = {"reverse": _lib.VLS_KL_REVERSE, "forward": _lib.VLS_KL_FORWARD}


def _dtype(t: torch.Tensor) -> int:
    try:
        return _DT[t.dtype]
    except KeyError:
        raise TypeError(f"libvls supports float32, bfloat16 and float16 tensors, not {t.dtype}") from None


def _rows(t: torch.Tensor) -> tuple[int, int, _lib.VlsRows]:
    """(N, V, vls_rows) of a [N, V] tensor, or of a [B, T, V] tensor read as
    N = B*T rows with two row strides; the last dimension is contiguous."""
    if t.dim() not in (2, 3):
        raise ValueError(f"expected a [N, V] or [B, T, V] tensor, got shape {tuple(t.shape)}")
    v = t.shape[-1]
    if v > 1 and t.stride(-1) != 1:
        raise ValueError("the vocabulary dimension must be contiguous (stride 1)")
    if t.dim() == 2:
        n = t.shape[0]
        ld = t.stride(0) if n > 1 else v
        if ld < v:
            raise ValueError("rows overlap (row stride smaller than V)")
        return n, v, _lib.rows(ld)
    b, tt = t.shape[0], t.shape[1]
    if b == 1 or tt == 1:  # one leading dim of size 1: one row stride
        return _rows(t[0] if b == 1 else t[:, 0])
    ld, ldg = t.stride(1), t.stride(0)
    if ld < v or ldg < v:
        raise ValueError("rows overlap (row stride smaller than V)")
    if ldg == tt * ld:  # the leading dims collapse
        return b * tt, v, _lib.rows(ld)
    return b * tt, v, _lib.rows(ld, tt, ldg)


def _ids2d(ids: torch.Tensor, n: int) -> torch.Tensor:
    """ids as [N, k] (a 1-D tensor is [N] with k = 1)."""
    k = ids.shape[-1] if ids.dim() >= 2 else 1
    return ids.reshape(n, k)


def _stream(t: torch.Tensor, stream) -> int:
    if stream is not None:
        return int(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)
    return int(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _raise_on_status(fn: str, status: torch.Tensor) -> None:
    """check=True of the tensor-core calls: synchronises the device, reads the
    call's status word and raises VlsDeviceError when a bounded wait in the
    kernel ran out (the call's outputs are then invalid)."""
    torch.cuda.synchronize(status.device)
    if int(status.item()) & 1:
        raise _lib.VlsDeviceError(fn, _lib.VLS_ERR_TIMEOUT)


def _stats(n: int, device, out=None) -> torch.Tensor:
    """vls_rowstat [N]: (m, log S) pairs as a float32 [N, 2] tensor."""
    if out is not None:
        return out
    return torch.empty((n, 2), dtype=torch.float32, device=device)


def vls_softcap_fwd(x: torch.Tensor, cap: float = 30.0, *, y=None, stream=None) -> torch.Tensor:
    lib = _lib.load()
    y = torch.empty_like(x, memory_format=torch.contiguous_format) if y is None else y
    if not x.is_contiguous() or not y.is_contiguous():
        raise ValueError("vls_softcap_fwd needs contiguous tensors")
    st = lib.vls_softcap_fwd(_ptr(x), _ptr(y), x.numel(), _dtype(x), float(cap), _stream(x, stream))
    _lib.check("vls_softcap_fwd", st)
    return y


def vls_softcap_bwd(x: torch.Tensor, gy: torch.Tensor, cap: float = 30.0, *, gx=None,
                    stream=None) -> torch.Tensor:
    lib = _lib.load()
    gx = torch.empty_like(x, memory_format=torch.contiguous_format) if gx is None else gx
    if not (x.is_contiguous() and gy.is_contiguous() and gx.is_contiguous()):
        raise ValueError("vls_softcap_bwd needs contiguous tensors")
    if gy.numel() != x.numel():
        raise ValueError("gy must have as many elements as x")
    st = lib.vls_softcap_bwd(_ptr(x), _ptr(gy), _dtype(gy), _ptr(gx), x.numel(), _dtype(x),
                             float(cap), _stream(x, stream))
    _lib.check("vls_softcap_bwd", st)
    return gx


def vls_logp_fwd(logits: torch.Tensor, ids: torch.Tensor, ignore_index: int = -100, cap: float = 0.0,
                 *, logp=None, stats=None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Returns (logp [N, k] float32, stats [N, 2] float32)."""
    lib = _lib.load()
    n, v, lay = _rows(logits)
    ids = _ids2d(ids, n)
    if ids.dtype != torch.int64 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous int64 [N, k] tensor")
    k = ids.shape[1]
    logp = torch.empty((n, k), dtype=torch.float32, device=logits.device) if logp is None else logp
    stats = _stats(n, logits.device, stats)
    st = lib.vls_logp_fwd(_ptr(logits), lay, _dtype(logits), n, v, _ptr(ids), k, int(ignore_index),
                          float(cap), _ptr(logp), _ptr(stats), _stream(logits, stream))
    _lib.check("vls_logp_fwd", st)
    return logp, stats


def vls_logp_bwd(logits: torch.Tensor, ids: torch.Tensor, g: torch.Tensor, stats: torch.Tensor,
                 ignore_index: int = -100, cap: float = 0.0, *, dlogits=None,
                 stream=None) -> torch.Tensor:
    lib = _lib.load()
    n, v, lay = _rows(logits)
    ids = _ids2d(ids, n)
    k = ids.shape[1]
    g = g.reshape(n, k)
    if g.dtype != torch.float32 or not g.is_contiguous():
        raise ValueError("g must be a contiguous float32 [N, k] tensor")
    if dlogits is None:
        dlogits = torch.empty((n, v), dtype=logits.dtype, device=logits.device)
    st = lib.vls_logp_bwd(_ptr(logits), lay, _dtype(logits), n, v, _ptr(ids), k, int(ignore_index),
                          float(cap), _ptr(g), _ptr(stats), _ptr(dlogits), _stream(logits, stream))
    _lib.check("vls_logp_bwd", st)
    return dlogits


def vls_entropy_fwd(logits: torch.Tensor, cap: float = 0.0, *, H=None, stats=None,
                    stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    lib = _lib.load()
    n, v, lay = _rows(logits)
    H = torch.empty((n,), dtype=torch.float32, device=logits.device) if H is None else H
    stats = _stats(n, logits.device, stats)
    st = lib.vls_entropy_fwd(_ptr(logits), lay, _dtype(logits), n, v, float(cap), _ptr(H), _ptr(stats),
                             _stream(logits, stream))
    _lib.check("vls_entropy_fwd", st)
    return H, stats


def vls_entropy_bwd(logits: torch.Tensor, g: torch.Tensor, H: torch.Tensor, stats: torch.Tensor,
                    cap: float = 0.0, *, dlogits=None, stream=None) -> torch.Tensor:
    lib = _lib.load()
    n, v, lay = _rows(logits)
    if g.dtype != torch.float32 or not g.is_contiguous():
        raise ValueError("g must be a contiguous float32 [N] tensor")
    if dlogits is None:
        dlogits = torch.empty((n, v), dtype=logits.dtype, device=logits.device)
    st = lib.vls_entropy_bwd(_ptr(logits), lay, _dtype(logits), n, v, float(cap), _ptr(g), _ptr(H),
                             _ptr(stats), _ptr(dlogits), _stream(logits, stream))
    _lib.check("vls_entropy_bwd", st)
    return dlogits


def vls_kl_fwd(a: torch.Tensor, b: torch.Tensor, direction: str = "reverse", cap: float = 0.0, *,
               kl=None, stats_a=None, stats_b=None,
               stream=None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Returns (kl [N], stats_a [N, 2], stats_b [N, 2])."""
    lib = _lib.load()
    n, v, lay_a = _rows(a)
    nb, vb, lay_b = _rows(b)
    if (nb, vb) != (n, v):
        raise ValueError("a and b must have the same shape")
    if a.dtype != b.dtype:
        raise TypeError("a and b must have the same dtype")
    kl = torch.empty((n,), dtype=torch.float32, device=a.device) if kl is None else kl
    stats_a = _stats(n, a.device, stats_a)
    stats_b = _stats(n, a.device, stats_b)
    st = lib.vls_kl_fwd(_ptr(a), lay_a, _ptr(b), lay_b, _dtype(a), n, v, _DIR[direction], float(cap), _ptr(kl),
                        _ptr(stats_a), _ptr(stats_b), _stream(a, stream))
    _lib.check("vls_kl_fwd", st)
    return kl, stats_a, stats_b


def vls_kl_bwd(a: torch.Tensor, b: torch.Tensor, g: torch.Tensor, kl: torch.Tensor, stats_a: torch.Tensor,
               stats_b: torch.Tensor, direction: str = "reverse", cap: float = 0.0, *, da=None,
               stream=None) -> torch.Tensor:
    lib = _lib.load()
    n, v, lay_a = _rows(a)
    _, _, lay_b = _rows(b)
    if g.dtype != torch.float32 or not g.is_contiguous():
        raise ValueError("g must be a contiguous float32 [N] tensor")
    if da is None:
        da = torch.empty((n, v), dtype=a.dtype, device=a.device)
    st = lib.vls_kl_bwd(_ptr(a), lay_a, _ptr(b), lay_b, _dtype(a), n, v, _DIR[direction], float(cap), _ptr(g),
                        _ptr(kl), _ptr(stats_a), _ptr(stats_b), _ptr(da), _stream(a, stream))
    _lib.check("vls_kl_bwd", st)
    return da


# ---------------------------------------------------------------------------
# fused statistics
# ---------------------------------------------------------------------------

def vls_fused_fwd(a: torch.Tensor, b: torch.Tensor | None = None, ids: torch.Tensor | None = None, *,
                  logp: bool = True, entropy: bool = True, kl: bool | None = None, direction: str = "reverse",
                  ignore_index: int = -100, cap: float = 0.0, stream=None) -> dict:
    """One read of the policy a (and of the reference b for KL).  Returns a
    dict with 'logp' [N, k] (when ids are given and logp), 'H' [N] (entropy),
    'kl' [N] (when b is given), 'stats_a' and 'stats_b' [N, 2]."""
    lib = _lib.load()
    n, v, lay_a = _rows(a)
    want_kl = (b is not None) if kl is None else bool(kl)
    lay_b = None
    if want_kl:
        nb, vb, lay_b = _rows(b)
        if (nb, vb) != (n, v) or b.dtype != a.dtype:
            raise ValueError("a and b must have the same shape and dtype")
    f32 = dict(dtype=torch.float32, device=a.device)
    out = {"stats_a": torch.empty((n, 2), **f32)}
    k = 0
    if logp and ids is not None:
        ids = _ids2d(ids, n)
        if ids.dtype != torch.int64 or not ids.is_contiguous():
            raise ValueError("ids must be a contiguous int64 [N, k] tensor")
        k = ids.shape[1]
        out["logp"] = torch.empty((n, k), **f32)
    if entropy:
        out["H"] = torch.empty((n,), **f32)
    if want_kl:
        out["kl"] = torch.empty((n,), **f32)
        out["stats_b"] = torch.empty((n, 2), **f32)
    st = lib.vls_fused_fwd(_ptr(a), lay_a, _ptr(b) if want_kl else None, lay_b, _dtype(a), n, v,
                           _ptr(ids) if k else None, k, int(ignore_index), _DIR[direction], float(cap),
                           _ptr(out.get("logp")), _ptr(out.get("H")), _ptr(out.get("kl")), _ptr(out["stats_a"]),
                           _ptr(out.get("stats_b")), _stream(a, stream))
    _lib.check("vls_fused_fwd", st)
    return out


def vls_fused_bwd(a: torch.Tensor, fwd: dict, b: torch.Tensor | None = None, ids: torch.Tensor | None = None, *,
                  g_logp: torch.Tensor | None = None, g_H: torch.Tensor | None = None,
                  g_kl: torch.Tensor | None = None, direction: str = "reverse", ignore_index: int = -100,
                  cap: float = 0.0, da=None, stream=None) -> torch.Tensor:
    """Gradient w.r.t. a of sum(g_logp * logp) + sum(g_H * H) + sum(g_kl * KL);
    `fwd` is vls_fused_fwd's result; absent gradients leave their term out."""
    lib = _lib.load()
    n, v, lay_a = _rows(a)
    lay_b = _rows(b)[2] if g_kl is not None else None
    k = 1
    if g_logp is not None:
        ids = _ids2d(ids, n)
        k = ids.shape[1]
        g_logp = g_logp.reshape(n, k)
    for t in (g_logp, g_H, g_kl):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous()):
            raise ValueError("upstream gradients must be contiguous float32")
    if da is None:
        da = torch.empty((n, v), dtype=a.dtype, device=a.device)
    st = lib.vls_fused_bwd(_ptr(a), lay_a, _ptr(b) if g_kl is not None else None, lay_b, _dtype(a), n, v,
                           _ptr(ids) if g_logp is not None else None, k, int(ignore_index), _DIR[direction],
                           float(cap), _ptr(g_logp), _ptr(g_H), _ptr(g_kl),
                           _ptr(fwd.get("H")) if g_H is not None else None,
                           _ptr(fwd.get("kl")) if g_kl is not None else None, _ptr(fwd["stats_a"]),
                           _ptr(fwd.get("stats_b")) if g_kl is not None else None, _ptr(da), _stream(a, stream))
    _lib.check("vls_fused_bwd", st)
    return da


# ---------------------------------------------------------------------------
# vocabulary-parallel split phase
# ---------------------------------------------------------------------------

PARTIAL_FIELDS = 6  # vls_partial: m, s, w, mq, sq, flag (4 bytes each)


def _partials(shape, device, out=None) -> torch.Tensor:
    """vls_partial arrays as float32 [..., 6] tensors (the flag word keeps its bits)."""
    if out is not None:
        return out
    return torch.empty((*shape, PARTIAL_FIELDS), dtype=torch.float32, device=device)


def _shard_rows(t: torch.Tensor) -> tuple[int, int, _lib.VlsRows | None]:
    """Like _rows, but a shard may have 0 columns (no descriptor then)."""
    if t.dim() not in (2, 3):
        raise ValueError(f"expected a [N, V_shard] or [B, T, V_shard] tensor, got shape {tuple(t.shape)}")
    if t.shape[-1] == 0:
        return t.shape[:-1].numel(), 0, None
    return _rows(t)


def _ptr_or_none(t: torch.Tensor):
    return t.data_ptr() if t.numel() > 0 else None


def vls_logp_partial(logits: torch.Tensor, ids: torch.Tensor, vocab_offset: int, vocab_total: int,
                     ignore_index: int = -100, cap: float = 0.0, *, part=None, zt=None,
                     stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Returns (part [N, 6], zt [N, k]) for the shard [vocab_offset, vocab_offset + V_shard)."""
    lib = _lib.load()
    n, v, lay = _shard_rows(logits)
    ids = _ids2d(ids, n)
    if ids.dtype != torch.int64 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous int64 [N, k] tensor")
    k = ids.shape[1]
    part = _partials((n,), ids.device, part)
    zt = torch.empty((n, k), dtype=torch.float32, device=ids.device) if zt is None else zt
    st = lib.vls_logp_partial(_ptr_or_none(logits), lay, _dtype(logits), n, v, int(vocab_offset), int(vocab_total),
                              _ptr(ids), k, int(ignore_index), float(cap), _ptr(part), _ptr(zt),
                              _stream(ids, stream))
    _lib.check("vls_logp_partial", st)
    return part, zt


def vls_logp_combine(parts: torch.Tensor, zt: torch.Tensor, ids: torch.Tensor, vocab_total: int,
                     ignore_index: int = -100, cap: float = 0.0, *, logp=None, stats=None,
                     stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """parts [R, N, 6] and zt [R, N, k] in rank order -> (logp [N, k], stats [N, 2])."""
    lib = _lib.load()
    r, n = parts.shape[0], parts.shape[1]
    ids = _ids2d(ids, n)
    k = ids.shape[1]
    if not (parts.is_contiguous() and zt.is_contiguous() and tuple(zt.shape) == (r, n, k)):
        raise ValueError("parts must be contiguous [R, N, 6] and zt contiguous [R, N, k]")
    logp = torch.empty((n, k), dtype=torch.float32, device=parts.device) if logp is None else logp
    stats = _stats(n, parts.device, stats)
    st = lib.vls_logp_combine(_ptr(parts), _ptr(zt), r, n, _ptr(ids), k, int(vocab_total), int(ignore_index),
                              float(cap), _ptr(logp), _ptr(stats), _stream(parts, stream))
    _lib.check("vls_logp_combine", st)
    return logp, stats


def vls_logp_bwd_shard(logits: torch.Tensor, ids: torch.Tensor, g: torch.Tensor, stats: torch.Tensor,
                       vocab_offset: int, vocab_total: int, ignore_index: int = -100, cap: float = 0.0, *,
                       dlogits=None, stream=None) -> torch.Tensor:
    lib = _lib.load()
    n, v, lay = _shard_rows(logits)
    ids = _ids2d(ids, n)
    k = ids.shape[1]
    g = g.reshape(n, k)
    if g.dtype != torch.float32 or not g.is_contiguous():
        raise ValueError("g must be a contiguous float32 [N, k] tensor")
    if dlogits is None:
        dlogits = torch.empty((n, v), dtype=logits.dtype, device=ids.device)
    st = lib.vls_logp_bwd_shard(_ptr_or_none(logits), lay, _dtype(logits), n, v, int(vocab_offset),
                                int(vocab_total), _ptr(ids), k, int(ignore_index), float(cap), _ptr(g),
                                _ptr(stats), _ptr_or_none(dlogits), _stream(ids, stream))
    _lib.check("vls_logp_bwd_shard", st)
    return dlogits


def vls_entropy_partial(logits: torch.Tensor, cap: float = 0.0, *, part=None, stream=None) -> torch.Tensor:
    lib = _lib.load()
    n, v, lay = _shard_rows(logits)
    part = _partials((n,), logits.device, part)
    st = lib.vls_entropy_partial(_ptr_or_none(logits), lay, _dtype(logits), n, v, float(cap), _ptr(part),
                                 _stream(part, stream))
    _lib.check("vls_entropy_partial", st)
    return part


def vls_entropy_combine(parts: torch.Tensor, *, H=None, stats=None, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    lib = _lib.load()
    r, n = parts.shape[0], parts.shape[1]
    H = torch.empty((n,), dtype=torch.float32, device=parts.device) if H is None else H
    stats = _stats(n, parts.device, stats)
    st = lib.vls_entropy_combine(_ptr(parts), r, n, _ptr(H), _ptr(stats), _stream(parts, stream))
    _lib.check("vls_entropy_combine", st)
    return H, stats


def vls_kl_partial(a: torch.Tensor, b: torch.Tensor, direction: str = "reverse", cap: float = 0.0, *, part=None,
                   stream=None) -> torch.Tensor:
    lib = _lib.load()
    n, v, lay_a = _shard_rows(a)
    _, vb, lay_b = _shard_rows(b)
    if vb != v or a.dtype != b.dtype:
        raise ValueError("a and b shards must have the same shape and dtype")
    part = _partials((n,), a.device, part)
    st = lib.vls_kl_partial(_ptr_or_none(a), lay_a, _ptr_or_none(b), lay_b, _dtype(a), n, v, _DIR[direction],
                            float(cap), _ptr(part), _stream(part, stream))
    _lib.check("vls_kl_partial", st)
    return part


def vls_kl_combine(parts: torch.Tensor, direction: str = "reverse", *, kl=None, stats_a=None, stats_b=None,
                   stream=None) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    lib = _lib.load()
    r, n = parts.shape[0], parts.shape[1]
    kl = torch.empty((n,), dtype=torch.float32, device=parts.device) if kl is None else kl
    stats_a = _stats(n, parts.device, stats_a)
    stats_b = _stats(n, parts.device, stats_b)
    st = lib.vls_kl_combine(_ptr(parts), r, n, _DIR[direction], _ptr(kl), _ptr(stats_a), _ptr(stats_b),
                            _stream(parts, stream))
    _lib.check("vls_kl_combine", st)
    return kl, stats_a, stats_b


# ---------------------------------------------------------------------------
# fused linear head + logprobs
# ---------------------------------------------------------------------------

def vls_linear_logp_chunks(vocab: int) -> int:
    return int(_lib.load().vls_linear_logp_chunks(int(vocab)))


def _matrix(t: torch.Tensor, what: str) -> tuple[int, int, int]:
    """(rows, D, row stride) of a 2-D tensor with a contiguous last dimension."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{what} must be a 2-D tensor with a contiguous last dimension")
    return t.shape[0], t.shape[1], (t.stride(0) if t.shape[0] > 1 else t.shape[1])


def vls_linear_logp_partial(h: torch.Tensor, w: torch.Tensor, ids: torch.Tensor, ignore_index: int = -100, *,
                            part=None, zt=None, status=None, stream=None, check=False):
    """(part [S, N, 6], zt [S, N, k], status [1] int32) of the linear head z = h @ w^T.

    The call only enqueues its kernel; `status` gets bit 0 if one of the
    kernel's bounded waits ran out.  check=True synchronises the device and
    raises VlsDeviceError in that case."""
    lib = _lib.load()
    n, d, ldh = _matrix(h, "h")
    v, dw, ldw = _matrix(w, "W")
    if dw != d:
        raise ValueError(f"h has D={d} but W has D={dw}")
    if h.dtype != w.dtype or h.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("h and W must both be bfloat16 or both float16")
    ids = _ids2d(ids, n)
    if ids.dtype != torch.int64 or not ids.is_contiguous():
        raise ValueError("ids must be a contiguous int64 [N, k] tensor")
    k = ids.shape[1]
    s = vls_linear_logp_chunks(v) if v > 0 else 0
    part = _partials((s, n), h.device, part)
    zt = torch.empty((s, n, k), dtype=torch.float32, device=h.device) if zt is None else zt
    status = torch.zeros(1, dtype=torch.int32, device=h.device) if status is None else status
    st = lib.vls_linear_logp_partial(_ptr(h), ldh, _ptr(w), ldw, _dtype(h), n, d, v, _ptr(ids), k,
                                     int(ignore_index), _ptr(part), _ptr(zt), _ptr(status), _stream(h, stream))
    _lib.check("vls_linear_logp_partial", st)
    if check:
        _raise_on_status("vls_linear_logp_partial", status)
    return part, zt, status


def vls_linear_logp_fwd(h: torch.Tensor, w: torch.Tensor, ids: torch.Tensor, ignore_index: int = -100, *,
                        stream=None, check=False) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(logp [N, k], stats [N, 2], status [1]): the two C calls in sequence
    (check as for vls_linear_logp_partial)."""
    part, zt, status = vls_linear_logp_partial(h, w, ids, ignore_index, stream=stream)
    logp, stats = vls_logp_combine(part, zt, ids, w.shape[0], ignore_index, 0.0, stream=stream)
    if check:
        _raise_on_status("vls_linear_logp_partial", status)
    return logp, stats, status


def vls_linear_logp_bwd_workspace(n: int, d: int, v: int) -> int:
    return int(_lib.load().vls_linear_logp_bwd_workspace(int(n), int(d), int(v)))


def vls_linear_logp_bwd(h: torch.Tensor, w: torch.Tensor, ids: torch.Tensor, g: torch.Tensor, stats: torch.Tensor,
                        ignore_index: int = -100, *, dh=None, dW=None, workspace=None, status=None, stream=None,
                        check=False):
    """(dh [N, D], dW [V, D], status [1]) of sum(g * logp) for the linear head
    z = h @ w^T; `stats` is vls_linear_logp_fwd's (check as for
    vls_linear_logp_partial)."""
    lib = _lib.load()
    n, d, ldh = _matrix(h, "h")
    v, dw, ldw = _matrix(w, "W")
    if dw != d or h.dtype != w.dtype:
        raise ValueError("h and W must share D and dtype")
    ids = _ids2d(ids, n)
    k = ids.shape[1]
    g = g.reshape(n, k)
    if g.dtype != torch.float32 or not g.is_contiguous():
        raise ValueError("g must be a contiguous float32 [N, k] tensor")
    dh = torch.empty((n, d), dtype=h.dtype, device=h.device) if dh is None else dh
    dW = torch.empty((v, d), dtype=h.dtype, device=h.device) if dW is None else dW
    need = vls_linear_logp_bwd_workspace(n, d, v)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=h.device)
    status = torch.zeros(1, dtype=torch.int32, device=h.device) if status is None else status
    st = lib.vls_linear_logp_bwd(_ptr(h), ldh, _ptr(w), ldw, _dtype(h), n, d, v, _ptr(ids), k, int(ignore_index),
                                 _ptr(g), _ptr(stats), _ptr(dh), _ptr(dW), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), _ptr(status), _stream(h, stream))
    _lib.check("vls_linear_logp_bwd", st)
    if check:
        _raise_on_status("vls_linear_logp_bwd", status)
    return dh, dW, status


def vls_linear_logp_fwd_noalloc(h: torch.Tensor, w: torch.Tensor, ids: torch.Tensor, ignore_index: int = -100, *,
                                logp=None, stats=None, status=None, stream=None, check=False):
    """vls_linear_logp_fwd through the C entry point that needs no buffer
    beyond the inputs and outputs (its intermediates sit in a fixed array of
    the library).  Returns (logp [N, k], stats [N, 2], status [1]) (check as
    for vls_linear_logp_partial)."""
    lib = _lib.load()
    n, d, ldh = _matrix(h, "h")
    v, dw, ldw = _matrix(w, "W")
    if dw != d:
        raise ValueError(f"h has D={d} but W has D={dw}")
    ids = _ids2d(ids, n)
    k = ids.shape[1]
    logp = torch.empty((n, k), dtype=torch.float32, device=h.device) if logp is None else logp
    stats = _stats(n, h.device, stats)
    status = torch.zeros(1, dtype=torch.int32, device=h.device) if status is None else status
    st = lib.vls_linear_logp_fwd_noalloc(_ptr(h), ldh, _ptr(w), ldw, _dtype(h), n, d, v, _ptr(ids), k,
                                         int(ignore_index), _ptr(logp), _ptr(stats), _ptr(status),
                                         _stream(h, stream))
    _lib.check("vls_linear_logp_fwd_noalloc", st)
    if check:
        _raise_on_status("vls_linear_logp_fwd_noalloc", status)
    return logp, stats, status


def vls_check_device_error() -> None:
    """Synchronises the current device and raises VlsDeviceError when a
    bounded wait of a tensor-core kernel ran out there since the last check
    (VlsError for a CUDA error of earlier work).  Clears the report."""
    _lib.check("vls_check_device_error", _lib.load().vls_check_device_error())


def vls_status_string(status: int) -> str:
    return _lib.load().vls_status_string(int(status)).decode()


def vls_version() -> int:
    return int(_lib.load().vls_version())
