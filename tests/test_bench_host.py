"""Host logic of bench.py that needs no GPU: the algorithmic byte model and
the multi-rank timing (max over ranks, whole-job throughput) on a gloo
process group of two ranks."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_byte_model():
    n, v = 8192, 151936
    nv = n * v * 2
    b = bench.op_bytes("logp", n, v)
    assert nv < b["fwd"] < 1.01 * nv and 2 * nv < b["bwd"] < 1.01 * 2 * nv
    kl = bench.op_bytes("kl_reverse", n, v)
    assert 2 * nv < kl["fwd"] < 1.01 * 2 * nv and 3 * nv < kl["bwd"] < 1.01 * 3 * nv
    assert bench.op_bytes("softcap", n, v) == {"fwd": 2 * nv, "bwd": 3 * nv}
    # logp 3 + entropy 3 + two KL 5 + capped logp 3 + softcap 5 passes of N*V*2 bytes
    assert abs(bench.step_bytes(n, v) / nv - 24) < 0.05


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(10.0 + 5.0 * rank)
    bench.barrier()
    q.put((rank, t, bench.aggregate(1_000_000_000_000, world, t / 1e3)))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]           # both ranks see the slowest time
    assert all(abs(r[2] - 2 * 1.0 / 0.015) < 1e-9 for r in res)   # 2 ranks x 1 TB in 15 ms


def test_single_process_helpers():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.dist_env()[1] >= 1
