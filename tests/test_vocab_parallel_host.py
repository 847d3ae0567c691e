"""Host side of the vocabulary-parallel path on CPU: shard bounds, and the
rank-ordered all-gather of partial states on a two-rank gloo group."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from vocab_log_softmax_gb300.vocab_parallel import gather_partials, shard_bounds


@pytest.mark.parametrize("vocab,world", [(151936, 2), (151936, 3), (10, 4), (3, 8), (75968, 8)])
def test_shard_bounds_tile_the_vocabulary(vocab, world):
    spans = [shard_bounds(vocab, world, r) for r in range(world)]
    off = 0
    for o, w in spans:
        assert o == off and w >= 0
        off += w
    assert off == vocab
    assert max(w for _, w in spans) - min(w for _, w in spans) <= 1


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    part = torch.full((5, 6), float(rank)) + torch.arange(5.0)[:, None]
    out = gather_partials(part)
    q.put((rank, out.numpy()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_gather_partials_rank_order_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for r in range(2):
        out = res[r]
        assert out.shape == (2, 5, 6)
        for src in range(2):
            assert (out[src] == src + torch.arange(5.0)[:, None].numpy()).all()
