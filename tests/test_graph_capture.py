"""The calls can be recorded into a CUDA graph (torch's default, global
capture mode) and replayed: every launch goes to the caller's stream, and no
call makes a runtime query that a capture refuses.  Replays must give the
eager results bit for bit."""

import pytest
import torch

from vls_compare import bitwise_equal
from vocab_log_softmax_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs():
    g = torch.Generator(device=DEV).manual_seed(77)
    n, v = 96, 30011
    a = (3.0 * torch.randn((n, v), generator=g, device=DEV)).to(torch.bfloat16)
    b = (a.float() + 0.5 * torch.randn((n, v), generator=g, device=DEV)).to(torch.bfloat16)
    ids = torch.randint(0, v, (n, 2), generator=g, device=DEV)
    gk = torch.randn((n, 2), generator=g, device=DEV)
    gr = torch.randn((n,), generator=g, device=DEV)
    h = torch.randn((130, 256), generator=g, device=DEV).to(torch.bfloat16)
    w = (0.2 * torch.randn((3001, 256), generator=g, device=DEV)).to(torch.bfloat16)
    lid = torch.randint(0, 3001, (130, 1), generator=g, device=DEV)
    lg = torch.randn((130, 1), generator=g, device=DEV)
    return a, b, ids, gk, gr, h, w, lid, lg


def _outputs(a, ids, h, w, lid):
    f32 = dict(dtype=torch.float32, device=DEV)
    n, v = a.shape
    s = B.vls_linear_logp_chunks(w.shape[0])
    return {
        "lp": torch.empty((n, 2), **f32), "st": torch.empty((n, 2), **f32), "st2": torch.empty((n, 2), **f32),
        "H": torch.empty((n,), **f32), "kl": torch.empty((n,), **f32),
        "d1": torch.empty_like(a), "d2": torch.empty_like(a), "d3": torch.empty_like(a), "y": torch.empty_like(a),
        "d4": torch.empty_like(a),
        "part": torch.empty((s, 130, 6), **f32), "zt": torch.empty((s, 130, 1), **f32),
        "llp": torch.empty((130, 1), **f32), "lst": torch.empty((130, 2), **f32),
        "status": torch.zeros(1, dtype=torch.int32, device=DEV),
        "dh": torch.empty_like(h), "dw": torch.empty_like(w),
        "ws": torch.empty((B.vls_linear_logp_bwd_workspace(130, 256, 3001),), dtype=torch.uint8, device=DEV),
    }


def _run(o, a, b, ids, gk, gr, h, w, lid, lg):
    B.vls_logp_fwd(a, ids, logp=o["lp"], stats=o["st"])
    B.vls_logp_bwd(a, ids, gk, o["st"], dlogits=o["d1"])
    B.vls_entropy_fwd(a, H=o["H"], stats=o["st"])
    B.vls_entropy_bwd(a, gr, o["H"], o["st"], dlogits=o["d2"])
    B.vls_kl_fwd(a, b, "reverse", 30.0, kl=o["kl"], stats_a=o["st"], stats_b=o["st2"])
    B.vls_kl_bwd(a, b, gr, o["kl"], o["st"], o["st2"], "reverse", 30.0, da=o["d3"])
    B.vls_softcap_fwd(a, 20.0, y=o["y"])
    B.vls_softcap_bwd(a, o["y"], 20.0, gx=o["d4"])
    B.vls_linear_logp_partial(h, w, lid, part=o["part"], zt=o["zt"], status=o["status"])
    B.vls_logp_combine(o["part"], o["zt"], lid, w.shape[0], logp=o["llp"], stats=o["lst"])
    B.vls_linear_logp_bwd(h, w, lid, lg, o["lst"], dh=o["dh"], dW=o["dw"], workspace=o["ws"], status=o["status"])


def test_capture_and_replay_bitwise():
    args = _inputs()
    a, b, ids, gk, gr, h, w, lid, lg = args
    eager = _outputs(a, ids, h, w, lid)
    _run(eager, *args)                                   # also the first call of each kernel on this device
    torch.cuda.synchronize()
    o = _outputs(a, ids, h, w, lid)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _run(o, *args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):                        # global capture mode
        _run(o, *args)
    for _ in range(2):
        for t in o.values():
            if t.dtype != torch.uint8:
                t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert int(o["status"].item()) == 0
        for key in eager:
            if key in ("ws",):
                continue
            assert bitwise_equal(o[key], eager[key]), key
