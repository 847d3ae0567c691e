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


def test_config_summary_groups_forward_and_backward():
    """The per-config block: each op's forward and backward, its fwd+bwd
    throughput from the two launches' bytes, comparison launches left out."""
    peak = 6000.0
    line = {"workload": "x", "rows": 8, "vocab": 10, "steps": 3, "fwd_bwd_ms": 3.0, "tbs": 2.0, "peak_gbs": peak,
            "l2": "no flush", "comparison_ops": ["other fwd"],
            "ops": {"a fwd": {"ms_median": 1.0, "tbs": 1.0, "frac_of_measured": 1.0 / 6, "bytes": 1e9},
                    "a bwd": {"ms_median": 2.0, "tbs": 1.5, "frac_of_measured": 0.25, "bytes": 3e9},
                    "other fwd": {"ms_median": 9.0, "tbs": 0.1, "frac_of_measured": 0.0, "bytes": 1e9}},
            "fwd_bwd_back_to_back": {}, "autograd": {}, "graph_replay": {"ms_median": 0.5, "tbs": 8.0}}
    out = bench.config_summary(line)
    assert set(out["ops"]) == {"a"}
    a = out["ops"]["a"]
    assert a["fwd_ms"] == 1.0 and a["bwd_ms"] == 2.0 and a["fwd_bwd_ms"] == 3.0
    assert abs(a["fwd_bwd_tbs"] - 4e9 / 3.0 / 1e9) < 1e-3 and abs(a["fwd_bwd_frac"] - 4e9 / 3.0 / 1e6 / peak) < 1e-3
    assert out["graph_replay"] == {"ms_median": 0.5, "tbs": 8.0}
    assert abs(out["frac_of_measured"] - 2.0 * 1e3 / peak) < 1e-4
    assert [k for k, *_ in bench.CONFIGS] == ["C1", "C2", "C3", "C4", "C5"]


@pytest.mark.timeout(300)
def test_oracle_pool_sizes_its_sample(monkeypatch):
    """The CPU legs time the oracle over a spawned pool: rows sized from a
    probe timed in every process at once, within the time budget, the row
    limit and the host-memory cap (here forced to two rows)."""
    v = 2048
    rows, dt = bench.oracle_pool(v, 1, 0, 2, budget_s=0.5, max_rows=64)
    assert 1 <= rows <= 64 and dt > 0
    monkeypatch.setattr(bench, "host_memory_available", lambda: int(2 * 2 * bench.ORACLE_BYTES_PER_COLUMN * v / 0.4) + 1)
    rows, dt = bench.oracle_pool(v, 1, 0, 2, budget_s=60.0, max_rows=64)
    assert rows == 2 and dt > 0


def test_both_arms_share_the_workload_config():
    c = bench.step_config(8192, 151936, 1)
    assert c == bench.step_config(8192, 151936, 1) and c["rows_per_gpu"] == 8192 and c["global_rows"] == 8192
    assert "per_op" not in c and c["bytes_per_step_per_gpu"] == bench.step_bytes(8192, 151936)
