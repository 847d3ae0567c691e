"""The linear-head logprob forward for callers that cannot allocate device
memory (a serving engine whose memory all belongs to its own pool, a program
held to a fixed device-memory budget): vls_linear_logp_fwd_noalloc keeps its
intermediate partials in a fixed array of the library instead of buffers
from the caller.  Its results must match the ordinary two-call route.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""

import ctypes

import pytest
import torch

from vls_compare import assert_fp32_close
from vocab_log_softmax_gb300 import _lib
from vocab_log_softmax_gb300 import binding as B

DEV = "cuda"


def _noalloc(lib, h, w, ids, logp, stats, status):
    """One call straight through the C ABI (no Python-side allocation)."""
    stream = torch.cuda.current_stream().cuda_stream
    return lib.vls_linear_logp_fwd_noalloc(h.data_ptr(), h.stride(0), w.data_ptr(), w.stride(0), _lib.VLS_BF16,
                                           h.shape[0], h.shape[1], w.shape[0], ids.data_ptr(), ids.shape[1], -100,
                                           logp.data_ptr(), stats.data_ptr(), status.data_ptr(), stream)


@pytest.mark.gpu
def test_noalloc_matches_the_two_call_route_on_two_calls_in_a_row():
    lib = _lib.load()
    # two different problems back to back: the second must not see the first's partials
    for n, d, v, seed in ((300, 512, 20000, 1), (129, 256, 5003, 2)):
        g = torch.Generator(device=DEV).manual_seed(seed)
        h = torch.randn((n, d), generator=g, device=DEV).to(torch.bfloat16)
        w = (3.0 / d ** 0.5 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16)
        ids = torch.randint(0, v, (n, 2), generator=g, device=DEV)
        ids[::5, 1] = -100
        ref_logp, ref_stats, ref_status = B.vls_linear_logp_fwd(h, w, ids)
        logp = torch.empty((n, 2), dtype=torch.float32, device=DEV)
        stats = torch.empty((n, 2), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _noalloc(lib, h, w, ids, logp, stats, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(ref_status.item()) == 0
        assert_fp32_close(logp, ref_logp.double().cpu().numpy(), f"no-alloc logp N={n}")
        assert_fp32_close(stats, ref_stats.double().cpu().numpy(), f"no-alloc stats N={n}")


def test_noalloc_rejects_calls_beyond_its_scratch():
    """The size check comes before any CUDA call, so it runs on any host."""
    lib = _lib.load()
    p = ctypes.c_void_p(0x1000)
    # V = 151936 gives 75 chunks: 13981 rows fit at k = 1, 14000 do not
    rc = lib.vls_linear_logp_fwd_noalloc(p, 4096, p, 4096, _lib.VLS_BF16, 14000, 4096, 151936, p, 1, -100,
                                         p, p, p, None)
    assert rc == 8 and lib.vls_status_string(rc).decode().startswith("VLS_ERR_TOO_LARGE")
    rc = lib.vls_linear_logp_fwd_noalloc(p, 4096, p, 4096, _lib.VLS_BF16, 8000, 4096, 151936, p, 16, -100,
                                         p, p, p, None)
    assert rc == 8       # 8000 x 75 x 16 target logits exceed 2^21
