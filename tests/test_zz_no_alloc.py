"""The linear-head logprob forward for callers that cannot allocate device
memory (a serving engine whose memory all belongs to its own pool, a program
held to a fixed device-memory budget): vls_linear_logp_fwd_noalloc keeps its
intermediate partials in a fixed array of the library instead of buffers
from the caller.  It runs the same two kernels on the same inputs as the
ordinary two-call route, so its results must be the same bits.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test."""

import ctypes

import pytest
import torch

from vls_compare import bitwise_equal
from vocab_log_softmax_gb300 import _lib, build
from vocab_log_softmax_gb300 import binding as B

DEV = "cuda"


def _noalloc(lib, h, w, ids, logp, stats, status):
    """One call straight through the C ABI (no Python-side allocation)."""
    stream = torch.cuda.current_stream().cuda_stream
    return lib.vls_linear_logp_fwd_noalloc(h.data_ptr(), h.stride(0), w.data_ptr(), w.stride(0), _lib.VLS_BF16,
                                           h.shape[0], h.shape[1], w.shape[0], ids.data_ptr(), ids.shape[1], -100,
                                           logp.data_ptr(), stats.data_ptr(), status.data_ptr(), stream)


def _case(n, d, v, k, seed):
    g = torch.Generator(device=DEV).manual_seed(seed)
    h = torch.randn((n, d), generator=g, device=DEV).to(torch.bfloat16)
    w = (3.0 / d ** 0.5 * torch.randn((v, d), generator=g, device=DEV)).to(torch.bfloat16)
    ids = torch.randint(0, v, (n, k), generator=g, device=DEV)
    ids[::5, k - 1] = -100
    return h, w, ids


@pytest.mark.gpu
def test_noalloc_matches_the_two_call_route_bit_for_bit():
    """Calls in a row, each a different problem, so that a later call cannot
    pass on an earlier call's partials: two small ones, then two at the
    array's limits (V = 151936 has 75 chunks: 13981 rows x 75 chunks is one
    partial below 2^20, and with k = 2 the targets are two below 2^21)."""
    lib = _lib.load()
    for n, d, v, k, seed in ((300, 512, 20000, 2, 1), (129, 256, 5003, 1, 2),
                             (13981, 256, 151936, 1, 3), (13981, 256, 151936, 2, 4)):
        h, w, ids = _case(n, d, v, k, seed)
        ref_logp, ref_stats, ref_status = B.vls_linear_logp_fwd(h, w, ids)
        logp = torch.full((n, k), float("nan"), dtype=torch.float32, device=DEV)
        stats = torch.full((n, 2), float("nan"), dtype=torch.float32, device=DEV)
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        assert _noalloc(lib, h, w, ids, logp, stats, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0 and int(ref_status.item()) == 0
        assert bitwise_equal(logp, ref_logp), f"no-alloc logp N={n} k={k}"
        assert bitwise_equal(stats, ref_stats), f"no-alloc stats N={n} k={k}"
        # the Python wrapper of the same entry point gives the same bits
        lp2, st2, s2 = B.vls_linear_logp_fwd_noalloc(h, w, ids, check=True)
        assert bitwise_equal(lp2, ref_logp) and bitwise_equal(st2, ref_stats) and int(s2.item()) == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    """The size check comes before any CUDA call, so it runs on any host."""
    build.build()
    lib = _lib.load()
    p = ctypes.c_void_p(0x1000)
    # V = 151936 gives 75 chunks: 13981 rows fit at k = 1, 13982 do not
    rc = lib.vls_linear_logp_fwd_noalloc(p, 4096, p, 4096, _lib.VLS_BF16, 13982, 4096, 151936, p, 1, -100,
                                         p, p, p, None)
    assert rc == 8 and lib.vls_status_string(rc).decode().startswith("VLS_ERR_TOO_LARGE")
    rc = lib.vls_linear_logp_fwd_noalloc(p, 4096, p, 4096, _lib.VLS_BF16, 8000, 4096, 151936, p, 16, -100,
                                         p, p, p, None)
    assert rc == 8       # 8000 x 75 x 16 target logits exceed 2^21
