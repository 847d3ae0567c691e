#!/usr/bin/env python3
"""Benchmark of the vocabulary-statistics hot path on one or more GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--rows N]

One step is one pass of the whole path over one batch of synthetic input,
N = 8192 rows x V = 151936 bf16 logits (the Qwen vocabulary), forward and
backward of every statistic:

  1. target logprob, k = 1        (logits N(0,3^2) + per-row offset U[-50,50];
                                   5% ignored rows, 1% out-of-range targets)
  2. entropy                      (policy a ~ N(0,3^2), 1% masked columns,
  3. reverse KL(a||b)              reference b = a + N(0,0.5^2), mismatch rows,
  4. forward KL(b||a)              one all -inf row)
  5. softcap-fused logprob, cap 30 (logits N(0,15^2))
  6. standalone softcap, cap 30, bf16 upstream gradient

The metric is fwd+bwd achieved HBM bandwidth: the algorithmic bytes of the
step (every logit read once per sweep that reads it, every gradient written
once, plus ids, upstream gradients, outputs and per-row stats) divided by the
device time of the step; per-op ms and TB/s are reported alongside.  Inputs
(2.5 GB per tensor) are far larger than L2, so no flush is needed between
steps.  Multi-GPU runs (torchrun) give each rank its own batch (weak scaling;
rows are independent, no collective on the data path); the time is the
maximum over ranks.

``--impl reference`` times the CPU fp64 oracle on a bounded sample of the
same workload (this is the baseline arm; no GPU is used).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

N_ROWS = 8192
VOCAB = 151936
CAP = 30.0
METRIC = "fwd+bwd achieved HBM TB/s, logp/entropy/KL/softcap, V=151936 bf16"
WORKLOAD = ("fwd+bwd of logp k=1, entropy, reverse KL, forward KL, softcap-fused logp (cap 30) "
            "and standalone softcap (cap 30), N=8192 x V=151936 bf16")
OPS = ["logp", "entropy", "kl_reverse", "kl_forward", "cap_logp", "softcap"]
KERNEL_NAMES = {  # op, pass -> CUDA kernel (for the ncu launch list)
    ("logp", "fwd"): "row_fwd_kernel<bf16, logp, nocap>",
    ("logp", "bwd"): "row_bwd_kernel<bf16, logp, nocap>",
    ("entropy", "fwd"): "row_fwd_kernel<bf16, entropy, nocap>",
    ("entropy", "bwd"): "row_bwd_kernel<bf16, entropy, nocap>",
    ("kl_reverse", "fwd"): "row_fwd_kernel<bf16, kl, nocap>",
    ("kl_reverse", "bwd"): "row_bwd_kernel<bf16, kl_reverse, nocap>",
    ("kl_forward", "fwd"): "row_fwd_kernel<bf16, kl, nocap>",
    ("kl_forward", "bwd"): "row_bwd_kernel<bf16, kl_forward, nocap>",
    ("cap_logp", "fwd"): "row_fwd_kernel<bf16, logp, cap>",
    ("cap_logp", "bwd"): "row_bwd_kernel<bf16, logp, cap>",
    ("softcap", "fwd"): "softcap_fwd_kernel<bf16>",
    ("softcap", "bwd"): "softcap_bwd_kernel<bf16, bf16>",
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ----------------------------------------------------------------------------
# algorithmic bytes
# ----------------------------------------------------------------------------

def op_bytes(op: str, n: int, v: int, es: int = 2, k: int = 1) -> dict:
    """Algorithmic bytes of one forward and one backward launch of `op`:
    each logit read once per sweep, each gradient element written once, plus
    the small per-row tensors (ids, upstream gradients, outputs, stats)."""
    nv = n * v * es
    stat = 8 * n
    if op in ("logp", "cap_logp"):
        small = n * k * (8 + 4)          # ids, logp (fwd) / ids, g (bwd)
        return {"fwd": nv + small + stat, "bwd": 2 * nv + small + stat}
    if op == "entropy":
        return {"fwd": nv + 4 * n + stat, "bwd": 2 * nv + 8 * n + stat}
    if op in ("kl_reverse", "kl_forward"):
        return {"fwd": 2 * nv + 4 * n + 2 * stat, "bwd": 3 * nv + 8 * n + 2 * stat}
    if op == "softcap":
        return {"fwd": 2 * nv, "bwd": 3 * nv}
    raise KeyError(op)


def step_bytes(n: int, v: int) -> int:
    return sum(sum(op_bytes(op, n, v).values()) for op in OPS)


# ----------------------------------------------------------------------------
# distributed helpers (host logic; covered by a gloo test)
# ----------------------------------------------------------------------------

def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(bytes_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job throughput in TB/s: the bytes all ranks processed over the
    slowest rank's time (each rank runs the same per-GPU workload)."""
    return bytes_per_rank * world / seconds / 1e12


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling every 200 ms while the timed region runs."""

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = None
        if gpu_id is None:
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(CLOCK_FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", gpu_id], stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == len(CLOCK_FIELDS):
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        reasons = []
        for i, name in ((5, "hw_slowdown"), (6, "hw_thermal_slowdown"), (7, "sw_thermal_slowdown"),
                        (8, "sw_power_cap")):
            if any(r[i].lower().startswith("active") for r in rows):
                reasons.append(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(rows)}


def gpu_id_for(device) -> str | None:
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return None


# ----------------------------------------------------------------------------
# peaks and ncu traffic
# ----------------------------------------------------------------------------

def hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def tensor_peak() -> tuple[float, str]:
    """Dense bf16 tensor-core peak in TFLOP/s: the measured burst figure, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def source_hash() -> str:
    """Hash of the sources the row kernels and their launches are built from
    (everything in csrc/ but the tensor-core linear head), which the committed
    traffic record must match."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "vocab_log_softmax_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith(("linear_", "tc_")):
            continue
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, n: int) -> float | None:
    """DRAM bytes per launch from the committed ncu capture, scaled to n rows;
    None when there is no capture or the kernels changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_hash") != source_hash():
        return None
    e = t.get("kernels", {}).get(kernel)
    if not e:
        return None
    return e["dram_bytes_per_launch"] * n / e["rows"]


# ----------------------------------------------------------------------------
# the step
# ----------------------------------------------------------------------------

class Step:
    """Device inputs, preallocated outputs, and the 12 launches of one step."""

    def __init__(self, device, n: int, v: int, seed_offset: int = 0):
        import torch

        import workloads
        self.n, self.v = n, v
        c2 = workloads.logp_offset(device, n=n, v=v, seed=1 + seed_offset)
        c3 = workloads.kl_masked(device, n=n, v=v, seed=2 + seed_offset)
        c4 = workloads.softcap_wide(device, n=n, v=v, seed=3 + seed_offset)
        self.inp = {
            "x": c2["logits"], "ids": c2["ids"], "g": c2["g"],
            "a": c3["a"], "b": c3["b"], "g_row": c3["g"],
            "xc": c4["logits"], "ids_c": c4["ids"], "g_c": c4["g"], "gy": c4["gy_bf16"],
        }
        f32 = dict(dtype=torch.float32, device=device)
        self.out = {
            "lp": torch.empty((n, 1), **f32), "st": torch.empty((n, 2), **f32),
            "st2": torch.empty((n, 2), **f32), "val": torch.empty((n,), **f32),
            "H": torch.empty((n,), **f32), "klr": torch.empty((n,), **f32), "klf": torch.empty((n,), **f32),
            "lpc": torch.empty((n, 1), **f32),
            "d": torch.empty((n, v), dtype=torch.bfloat16, device=device),
            "y": torch.empty((n, v), dtype=torch.bfloat16, device=device),
        }

    def launches(self):
        """(op, pass, thunk) for the 12 launches of one step, in order."""
        from vocab_log_softmax_gb300 import binding as B
        i, o = self.inp, self.out
        return [
            ("logp", "fwd", lambda: B.vls_logp_fwd(i["x"], i["ids"], -100, 0.0, logp=o["lp"], stats=o["st"])),
            ("logp", "bwd", lambda: B.vls_logp_bwd(i["x"], i["ids"], i["g"], o["st"], -100, 0.0, dlogits=o["d"])),
            ("entropy", "fwd", lambda: B.vls_entropy_fwd(i["a"], 0.0, H=o["H"], stats=o["st"])),
            ("entropy", "bwd", lambda: B.vls_entropy_bwd(i["a"], i["g_row"], o["H"], o["st"], 0.0, dlogits=o["d"])),
            ("kl_reverse", "fwd", lambda: B.vls_kl_fwd(i["a"], i["b"], "reverse", 0.0, kl=o["klr"],
                                                       stats_a=o["st"], stats_b=o["st2"])),
            ("kl_reverse", "bwd", lambda: B.vls_kl_bwd(i["a"], i["b"], i["g_row"], o["klr"], o["st"], o["st2"],
                                                       "reverse", 0.0, da=o["d"])),
            ("kl_forward", "fwd", lambda: B.vls_kl_fwd(i["a"], i["b"], "forward", 0.0, kl=o["klf"],
                                                       stats_a=o["st"], stats_b=o["st2"])),
            ("kl_forward", "bwd", lambda: B.vls_kl_bwd(i["a"], i["b"], i["g_row"], o["klf"], o["st"], o["st2"],
                                                       "forward", 0.0, da=o["d"])),
            ("cap_logp", "fwd", lambda: B.vls_logp_fwd(i["xc"], i["ids_c"], -100, CAP, logp=o["lpc"], stats=o["st"])),
            ("cap_logp", "bwd", lambda: B.vls_logp_bwd(i["xc"], i["ids_c"], i["g_c"], o["st"], -100, CAP,
                                                       dlogits=o["d"])),
            ("softcap", "fwd", lambda: B.vls_softcap_fwd(i["xc"], CAP, y=o["y"])),
            ("softcap", "bwd", lambda: B.vls_softcap_bwd(i["xc"], i["gy"], CAP, gx=o["d"])),
        ]

    def results(self):
        """The step's results a caller reads back: every forward output and
        gradient (the gradient buffer is shared, so it is read after each op)."""
        o = self.out
        return [o["lp"], o["H"], o["klr"], o["klf"], o["lpc"], o["y"], o["d"]]


def time_device(step: Step, steps: int, warmup: int, device):
    import torch
    launches = step.launches()
    for _ in range(warmup):
        for _, _, f in launches:
            f()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)] for _ in range(steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_id_for(device))
    time.sleep(0.6)                      # let the sampler start before the timed region
    start.record(stream)
    for s in range(steps):
        for j, (_, _, f) in enumerate(launches):
            ev[s][j].record(stream)
            f()
        ev[s][-1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier()
    total_ms = start.elapsed_time(stop)
    per = {}
    for j, (op, ps, _) in enumerate(launches):
        per[(op, ps)] = statistics.mean(ev[s][j].elapsed_time(ev[s][j + 1]) for s in range(steps))
    return total_ms, per, clk


class ConfigRun:
    """One of the five workloads, fwd+bwd of its ops, for per-config numbers
    (``--workload``).  Not the headline step; the same kernels and geometry."""

    def __init__(self, name: str, device, rows: int | None = None):
        import torch

        import workloads
        from vocab_log_softmax_gb300 import binding as B
        self.name = name
        f32 = dict(dtype=torch.float32, device=device)
        L = []                                       # (label, bytes, thunk[, flops])
        # launches timed only for comparison (another route to the same
        # outputs); they stay out of the workload's totals
        self.compare = set()
        if name == "logp_small":
            w = workloads.logp_small(device)
            x, ids, g = w["logits"], w["ids"], w["g"]
            n, v = x.shape
            lp, st, d = torch.empty((n, 1), **f32), torch.empty((n, 2), **f32), torch.empty_like(x)
            b = op_bytes("logp", n, v, es=4)
            L += [("logp fwd", b["fwd"], lambda: B.vls_logp_fwd(x, ids, logp=lp, stats=st)),
                  ("logp bwd", b["bwd"], lambda: B.vls_logp_bwd(x, ids, g, st, dlogits=d))]
        elif name == "logp_offset":
            w = workloads.logp_offset(device)
            x, ids, g = w["logits"], w["ids"], w["g"]
            n, v = x.shape
            lp, st, d = torch.empty((n, 1), **f32), torch.empty((n, 2), **f32), torch.empty_like(x)
            b = op_bytes("logp", n, v)
            L += [("logp fwd", b["fwd"], lambda: B.vls_logp_fwd(x, ids, logp=lp, stats=st)),
                  ("logp bwd", b["bwd"], lambda: B.vls_logp_bwd(x, ids, g, st, dlogits=d))]
        elif name == "kl_masked":
            w = workloads.kl_masked(device)
            a_, b_, g = w["a"], w["b"], w["g"]
            n, v = a_.shape
            H, kl, sa, sb = (torch.empty((n,), **f32), torch.empty((n,), **f32), torch.empty((n, 2), **f32),
                             torch.empty((n, 2), **f32))
            d = torch.empty_like(a_)
            be, bk = op_bytes("entropy", n, v), op_bytes("kl_reverse", n, v)
            L += [("entropy fwd", be["fwd"], lambda: B.vls_entropy_fwd(a_, H=H, stats=sa)),
                  ("entropy bwd", be["bwd"], lambda: B.vls_entropy_bwd(a_, g, H, sa, dlogits=d))]
            for dr in ("forward", "reverse"):
                L += [(f"{dr} KL fwd", bk["fwd"], lambda dr=dr: B.vls_kl_fwd(a_, b_, dr, kl=kl, stats_a=sa, stats_b=sb)),
                      (f"{dr} KL bwd", bk["bwd"], lambda dr=dr: B.vls_kl_bwd(a_, b_, g, kl, sa, sb, dr, da=d))]
        elif name == "softcap_wide":
            w = workloads.softcap_wide(device)
            x, ids, g, gy = w["logits"], w["ids"], w["g"], w["gy_bf16"]
            n, v = x.shape
            lp, st, d, y = torch.empty((n, 1), **f32), torch.empty((n, 2), **f32), torch.empty_like(x), torch.empty_like(x)
            b, bs = op_bytes("cap_logp", n, v), op_bytes("softcap", n, v)
            for c in w["caps"]:
                L += [(f"cap{c:g} logp fwd", b["fwd"], lambda c=c: B.vls_logp_fwd(x, ids, -100, c, logp=lp, stats=st)),
                      (f"cap{c:g} logp bwd", b["bwd"], lambda c=c: B.vls_logp_bwd(x, ids, g, st, -100, c, dlogits=d))]
            L += [("softcap fwd", bs["fwd"], lambda: B.vls_softcap_fwd(x, 30.0, y=y)),
                  ("softcap bwd", bs["bwd"], lambda: B.vls_softcap_bwd(x, gy, 30.0, gx=d))]
        elif name == "long_seq":
            w = workloads.long_seq(device)
            x = w["logits"]
            n, v = x.shape
            k = w["idsk"].shape[1]
            lp1, lpk = torch.empty((n, 1), **f32), torch.empty((n, k), **f32)
            st, H, d = torch.empty((n, 2), **f32), torch.empty((n,), **f32), torch.empty_like(x)
            b1, bk, be = op_bytes("logp", n, v), op_bytes("logp", n, v, k=k), op_bytes("entropy", n, v)
            L += [("k=1 logp fwd", b1["fwd"], lambda: B.vls_logp_fwd(x, w["ids1"], logp=lp1, stats=st)),
                  ("k=1 logp bwd", b1["bwd"], lambda: B.vls_logp_bwd(x, w["ids1"], w["g1"], st, dlogits=d)),
                  ("k=256 logp fwd", bk["fwd"], lambda: B.vls_logp_fwd(x, w["idsk"], logp=lpk, stats=st)),
                  ("k=256 logp bwd", bk["bwd"], lambda: B.vls_logp_bwd(x, w["idsk"], w["gk"], st, dlogits=d)),
                  ("entropy fwd", be["fwd"], lambda: B.vls_entropy_fwd(x, H=H, stats=st)),
                  ("entropy bwd", be["bwd"], lambda: B.vls_entropy_bwd(x, w["g_row"], H, st, dlogits=d))]

            def peak_extra():
                """Device memory the calls need beyond their inputs, the returned
                gradient and the forward outputs: the saved per-row stats
                (8 B per row) plus whatever the calls allocate, measured
                through torch's allocator and through the device's free memory
                (2 MiB granularity).  Also through the autograd API, where
                the stats are saved by the function and the gradient and
                outputs are allocated by it."""
                import vocab_log_softmax_gb300 as Vl
                launches = [f for _, _, f in L]
                torch.cuda.synchronize()
                torch.cuda.reset_peak_memory_stats()
                base, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
                for f in launches:
                    f()
                torch.cuda.synchronize()
                by_calls = torch.cuda.max_memory_allocated() - base
                free_delta = max(0, free0 - torch.cuda.mem_get_info()[0])
                leaf = x.detach().requires_grad_(True)
                g1 = w["g1"].reshape(w["ids1"].shape)
                torch.cuda.synchronize()
                torch.cuda.reset_peak_memory_stats()
                base = torch.cuda.memory_allocated()
                out = Vl.logprobs(leaf, w["ids1"])
                out.backward(g1)
                torch.cuda.synchronize()
                autograd_extra = (torch.cuda.max_memory_allocated() - base - leaf.grad.numel() * leaf.grad.element_size()
                                  - out.numel() * out.element_size())
                del out, leaf
                stats_bytes = n * 8
                return {"saved_stats_bytes": stats_bytes, "allocated_by_calls_bytes": by_calls,
                        "device_free_delta_bytes": free_delta,
                        "peak_extra_bytes": stats_bytes + max(by_calls, free_delta),
                        "autograd_k1_peak_extra_bytes": autograd_extra, "limit_bytes": 1 << 20}
            self.peak_extra = peak_extra
        elif name == "fused":
            # logprobs + entropy + reverse KL of one policy: fused calls vs the six separate calls
            w = workloads.kl_masked(device, n=N_ROWS, v=VOCAB)
            wl = workloads.logp_offset(device, n=N_ROWS, v=VOCAB)
            a_, b_, g = w["a"], w["b"], w["g"]
            ids, gl = wl["ids"], wl["g"]
            n, v = a_.shape
            out = {}
            d = torch.empty_like(a_)
            nv = n * v * 2
            small = n * (8 + 4 + 4 + 4 + 16)

            def ffwd():
                out.update(B.vls_fused_fwd(a_, b_, ids))

            L += [("fused fwd (logp+H+KL)", 2 * nv + small, ffwd),
                  ("fused bwd (logp+H+KL)", 3 * nv + small,
                   lambda: B.vls_fused_bwd(a_, out, b_, ids, g_logp=gl, g_H=g, g_kl=g, da=d))]
            lp, H, kl = torch.empty((n, 1), **f32), torch.empty((n,), **f32), torch.empty((n,), **f32)
            st1, st2, st3 = (torch.empty((n, 2), **f32) for _ in range(3))
            bl, be, bk = op_bytes("logp", n, v), op_bytes("entropy", n, v), op_bytes("kl_reverse", n, v)
            L += [("separate logp fwd", bl["fwd"], lambda: B.vls_logp_fwd(a_, ids, logp=lp, stats=st1)),
                  ("separate entropy fwd", be["fwd"], lambda: B.vls_entropy_fwd(a_, H=H, stats=st1)),
                  ("separate KL fwd", bk["fwd"], lambda: B.vls_kl_fwd(a_, b_, kl=kl, stats_a=st2, stats_b=st3)),
                  ("separate logp bwd", bl["bwd"], lambda: B.vls_logp_bwd(a_, ids, gl, st1, dlogits=d)),
                  ("separate entropy bwd", be["bwd"], lambda: B.vls_entropy_bwd(a_, g, H, st1, dlogits=d)),
                  ("separate KL bwd", bk["bwd"], lambda: B.vls_kl_bwd(a_, b_, g, kl, st2, st3, da=d))]
            self.compare |= {label for label, *_ in L if label.startswith("separate ")}
        elif name == "linear_logp":
            # fused linear head + logprobs on the tensor cores, against cuBLAS logits + the logp sweep
            # rows: the batch (8192 by default; --rows sets it for this workload)
            w = workloads.linear_head(device) if rows is None else workloads.linear_head(device, n=rows)
            h, wt, ids = w["h"], w["w"], w["ids"]
            n, dd = h.shape
            v = wt.shape[0]
            s = B.vls_linear_logp_chunks(v)
            part = torch.empty((s, n, 6), **f32)
            zt = torch.empty((s, n, 1), **f32)
            status = torch.zeros(1, dtype=torch.int32, device=device)
            lp, st = torch.empty((n, 1), **f32), torch.empty((n, 2), **f32)
            z = torch.empty((n, v), dtype=torch.bfloat16, device=device)
            flops = 2 * n * v * dd
            io = (n + v) * dd * 2

            def fused():
                B.vls_linear_logp_partial(h, wt, ids, part=part, zt=zt, status=status)
                B.vls_logp_combine(part, zt, ids, v, logp=lp, stats=st)

            g = w["g"]
            dh, dw = torch.empty_like(h), torch.empty_like(wt)
            ws = torch.empty((B.vls_linear_logp_bwd_workspace(n, dd, v),), dtype=torch.uint8, device=device)
            # backward bytes: h and W read twice over the three products, dz
            # written once and read twice, dh and dW written
            L += [("fused linear logp fwd", io, fused, flops),
                  ("fused linear logp bwd", 3 * io + 3 * n * v * 2,
                   lambda: B.vls_linear_logp_bwd(h, wt, ids, g, st, dh=dh, dW=dw, workspace=ws, status=status),
                   3 * flops),
                  ("cuBLAS h @ W^T to bf16 logits", io + n * v * 2, lambda: torch.mm(h, wt.t(), out=z), flops),
                  ("logp fwd over those logits", n * v * 2, lambda: B.vls_logp_fwd(z, ids, logp=lp, stats=st))]
            self.compare |= {"cuBLAS h @ W^T to bf16 logits", "logp fwd over those logits"}
            self.status = status
        else:
            raise SystemExit(f"unknown workload {name}")
        self.launches = L
        self.rows, self.vocab = n, v
        self.small = name == "logp_small"   # 8 MB of inputs: inside L2
        if name == "fused":
            w = {"a": w["a"], "b": w["b"], "g": w["g"], "ids": wl["ids"], "gl": wl["g"]}
        self.autograd = self._autograd_thunks(name, w, device)

    @staticmethod
    def _autograd_thunks(name, w, device):
        """(label, bytes, thunk): the public autograd API, forward and backward,
        for the workload's main op -- the path a training loop calls."""
        import torch

        import vocab_log_softmax_gb300 as V

        leaves = []

        def fwd_bwd(make):
            def run():
                for t in leaves:        # a training step starts from cleared gradients
                    t.grad = None
                out, g = make()
                out.backward(g)
            return run

        def leaf(t):
            t = t.detach().requires_grad_(True)
            leaves.append(t)
            return t

        if name in ("logp_small", "logp_offset", "long_seq"):
            x = leaf(w["logits"])
            ids = w["ids"] if "ids" in w else w["ids1"]
            g = (w["g"] if "g" in w else w["g1"]).reshape(ids.shape)
            n, v = x.shape
            b = op_bytes("logp", n, v, es=x.element_size())
            return [("autograd logprobs fwd+bwd", b["fwd"] + b["bwd"], fwd_bwd(lambda: (V.logprobs(x, ids), g)))]
        if name == "kl_masked":
            a = leaf(w["a"])
            n, v = a.shape
            be, bk = op_bytes("entropy", n, v), op_bytes("kl_reverse", n, v)
            return [("autograd entropy fwd+bwd", be["fwd"] + be["bwd"], fwd_bwd(lambda: (V.entropy(a), w["g"]))),
                    ("autograd reverse KL fwd+bwd", bk["fwd"] + bk["bwd"],
                     fwd_bwd(lambda: (V.kl(a, w["b"], "reverse"), w["g"])))]
        if name == "softcap_wide":
            x = leaf(w["logits"])
            n, v = x.shape
            b, bs = op_bytes("cap_logp", n, v), op_bytes("softcap", n, v)
            g = w["g"].reshape(w["ids"].shape)
            return [("autograd cap30 logprobs fwd+bwd", b["fwd"] + b["bwd"],
                     fwd_bwd(lambda: (V.logprobs(x, w["ids"], softcap=30.0), g))),
                    ("autograd softcap fwd+bwd", bs["fwd"] + bs["bwd"],
                     fwd_bwd(lambda: (V.softcap(x, 30.0), w["gy_bf16"])))]
        if name == "fused":
            a = leaf(w["a"])
            n, v = a.shape
            gl = w["gl"].reshape(w["ids"].shape)

            def stats_run():
                a.grad = None
                lp, H, kl = V.stats(a, w["ids"], reference=w["b"])
                torch.autograd.backward([lp, H, kl], [gl, w["g"], w["g"]])
            return [("autograd stats (logp+H+KL) fwd+bwd", 5 * n * v * 2, stats_run)]
        if name == "linear_logp":
            h = leaf(w["h"])
            wt = leaf(w["w"])
            g = w["g"].reshape(w["ids"].shape)
            n, d = h.shape
            return [("autograd linear_logprobs fwd+bwd", (n + wt.shape[0]) * d * 2 * 3,
                     fwd_bwd(lambda: (V.linear_logprobs(h, wt, w["ids"]), g)),
                     4 * 2 * n * wt.shape[0] * d)]
        return []


def run_config(args) -> None:
    """Per-config fwd / bwd times (median over steps) and TB/s for every op."""
    import torch
    device = torch.device("cuda", 0)
    rows = args.rows if args.workload == "linear_logp" and args.rows != N_ROWS else None
    print(json.dumps(measure_workload(args.workload, device, args.steps, args.warmup, rows)), flush=True)


def l2_flusher(device):
    """Writes a buffer twice the size of L2 (129 MB) between timed steps of a
    workload small enough to stay in L2, so that each step starts cold."""
    import torch
    buf = torch.empty((64 << 20,), dtype=torch.float32, device=device)   # 256 MB
    return lambda: buf.zero_()


def measure_workload(name: str, device, steps: int, warmup: int, rows: int | None = None) -> dict:
    """One workload's launches timed with CUDA events: per-op median ms,
    TB/s and fraction of the measured copy bandwidth, fwd+bwd back to back,
    the autograd API, and (C1) CUDA-graph replay.  Workloads smaller than L2
    (C1) flush it between timed steps, outside the timed launches."""
    import torch
    run = ConfigRun(name, device, rows)
    flush = l2_flusher(device) if run.small else None
    for _ in range(warmup):
        for _, _, f, *_ in run.launches:
            f()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(run.launches) + 1)] for _ in range(steps)]
    for s in range(steps):
        if flush:
            flush()
        for j, (_, _, f, *_) in enumerate(run.launches):
            ev[s][j].record(stream)
            f()
        ev[s][-1].record(stream)
    torch.cuda.synchronize()
    peak, kind = hbm_peak()
    tpeak, tkind = tensor_peak()
    ops = {}
    for j, (label, nbytes, _, *fl) in enumerate(run.launches):
        ts = sorted(ev[s][j].elapsed_time(ev[s][j + 1]) for s in range(steps))
        med = ts[len(ts) // 2]
        ops[label] = {"ms_median": round(med, 4), "ms_p10": round(ts[len(ts) // 10], 4),
                      "ms_p90": round(ts[(9 * len(ts)) // 10], 4), "tbs": round(nbytes / med / 1e9, 3),
                      "frac_of_measured": round(nbytes / med / 1e6 / peak, 4), "bytes": nbytes}
        if fl:   # a contraction: its tensor-core roofline
            ops[label].update({"tflops": round(fl[0] / med / 1e9, 1), "flops": fl[0],
                               "frac_of_bf16_peak": round(fl[0] / med / 1e9 / tpeak, 4), "bf16_peak_kind": tkind})
    if getattr(run, "status", None) is not None and int(run.status.item()) != 0:
        raise SystemExit(f"{run.name}: a bounded wait in the kernel ran out (status {int(run.status.item())})")
    own = [(label, b, fl) for label, b, _, *fl in run.launches if label not in run.compare]
    total_b = sum(b for _, b, _ in own)
    total_ms = sum(ops[label]["ms_median"] for label, _, _ in own)
    total_fl = sum(fl[0] for _, _, fl in own if fl)
    # an op's forward and backward timed back to back (one event pair around both)
    pairs = {}
    for j in range(len(run.launches) - 1):
        lf, lb = run.launches[j][0], run.launches[j + 1][0]
        if lf.endswith(" fwd") and lb == lf[:-4] + " bwd":
            ts = sorted(ev[s][j].elapsed_time(ev[s][j + 2]) for s in range(steps))
            nb = run.launches[j][1] + run.launches[j + 1][1]
            pairs[lf[:-4] + " fwd+bwd"] = {"ms_median": round(ts[len(ts) // 2], 4), "ms_p10": round(ts[len(ts) // 10], 4),
                                           "ms_p90": round(ts[(9 * len(ts)) // 10], 4),
                                           "tbs": round(nb / ts[len(ts) // 2] / 1e9, 3)}
    autograd = {}
    for label, nbytes, f, *fl in run.autograd:
        ts = time_thunk(f, steps, warmup, stream, flush)
        med = ts[len(ts) // 2]
        autograd[label] = {"ms_median": round(med, 4), "ms_p10": round(ts[len(ts) // 10], 4),
                           "ms_p90": round(ts[(9 * len(ts)) // 10], 4), "tbs": round(nbytes / med / 1e9, 3)}
        if fl:
            autograd[label]["tflops"] = round(fl[0] / med / 1e9, 1)
    graph = graph_replay(run, steps, stream, flush) if run.name == "logp_small" else None
    line = {"workload": run.name, "rows": run.rows, "vocab": run.vocab, "steps": steps,
            "fwd_bwd_ms": round(total_ms, 4), "tbs": round(total_b / total_ms / 1e9, 3),
            "peak_gbs": peak, "peak_kind": kind,
            "l2": "flushed between timed steps (inputs fit in L2)" if flush else "inputs larger than L2; no flush"}
    if total_fl:   # a tensor-bound workload: its throughput against the bf16 peak
        line.update({"tflops": round(total_fl / total_ms / 1e9, 1),
                     "frac_of_bf16_peak": round(total_fl / total_ms / 1e9 / tpeak, 4), "bf16_peak_kind": tkind})
    line.update({"comparison_ops": sorted(run.compare), "ops": ops, "fwd_bwd_back_to_back": pairs,
                 "autograd": autograd, "graph_replay": graph})
    if getattr(run, "peak_extra", None) is not None:
        line["peak_extra_memory"] = run.peak_extra()
    return line


def time_thunk(f, steps: int, warmup: int, stream, flush=None) -> list:
    """Sorted CUDA-event times (ms) of f() over `steps` calls after `warmup`
    (flush(), if given, runs before each timed call, outside its events)."""
    import torch
    for _ in range(warmup):
        f()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        if flush:
            flush()
        a.record(stream)
        f()
        b.record(stream)
    torch.cuda.synchronize()
    return sorted(a.elapsed_time(b) for a, b in ev)


def graph_replay(run, steps: int, stream, flush=None) -> dict:
    """The workload's launches captured once in a CUDA graph and replayed: the
    per-replay time without host launch overhead (for launch-bound sizes)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            for _, _, f, *_ in run.launches:
                f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(graph):
            for _, _, f, *_ in run.launches:
                f()
    except RuntimeError as e:
        return {"unavailable": str(e).splitlines()[0][:200]}
    ts = time_thunk(graph.replay, steps, 3, torch.cuda.current_stream(), flush)
    nb = sum(b for _, b, *_ in run.launches)
    med = ts[len(ts) // 2]
    return {"launches_per_replay": len(run.launches), "ms_median": round(med, 4), "ms_p10": round(ts[len(ts) // 10], 4),
            "ms_p90": round(ts[(9 * len(ts)) // 10], 4), "tbs": round(nb / med / 1e9, 3)}


E2E_CHUNKS = 8
E2E_COPY_STREAMS = 1


def time_e2e(step: Step, steps: int, device, chunks: int = E2E_CHUNKS, copy_streams: int = E2E_COPY_STREAMS):
    """The same step through the same calls with HOST buffers: every input is
    copied in from pinned host memory and every result (forward outputs, each
    op's gradient, the softcap output) is copied back to pinned host memory
    inside the timed region.  Rows are independent, so the batch is cut into
    row chunks pipelined over three streams: chunk c's inputs are copied in
    while chunk c-1 computes and chunk c-2's results are copied out (the two
    copy directions run on separate copy engines; ``copy_streams`` > 1 deals
    the chunks round-robin over that many streams per direction).  Each op
    writes its own gradient buffer, so no readback waits for a later op."""
    import torch
    n = step.n
    bounds = [(n * c // chunks, n * (c + 1) // chunks) for c in range(chunks)]
    pinned_in = {k: t.detach().cpu().pin_memory() for k, t in step.inp.items()}
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    i, o = step.inp, step.out
    grad = {op: torch.empty_like(o["d"]) for op in OPS}
    dev_out = {"lp": o["lp"], "H": o["H"], "klr": o["klr"], "klf": o["klf"], "lpc": o["lpc"], "y": o["y"]}
    dev_out.update({"d_" + op: grad[op] for op in OPS})
    host_out = {k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for k, t in dev_out.items()}
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    from vocab_log_softmax_gb300 import binding as B

    def launches(lo, hi):
        r = slice(lo, hi)
        st, st2 = o["st"][r], o["st2"][r]
        B.vls_logp_fwd(i["x"][r], i["ids"][r], -100, 0.0, logp=o["lp"][r], stats=st)
        B.vls_logp_bwd(i["x"][r], i["ids"][r], i["g"][r], st, -100, 0.0, dlogits=grad["logp"][r])
        B.vls_entropy_fwd(i["a"][r], 0.0, H=o["H"][r], stats=st)
        B.vls_entropy_bwd(i["a"][r], i["g_row"][r], o["H"][r], st, 0.0, dlogits=grad["entropy"][r])
        for op, d, kl in (("kl_reverse", "reverse", o["klr"]), ("kl_forward", "forward", o["klf"])):
            B.vls_kl_fwd(i["a"][r], i["b"][r], d, 0.0, kl=kl[r], stats_a=st, stats_b=st2)
            B.vls_kl_bwd(i["a"][r], i["b"][r], i["g_row"][r], kl[r], st, st2, d, 0.0, da=grad[op][r])
        B.vls_logp_fwd(i["xc"][r], i["ids_c"][r], -100, CAP, logp=o["lpc"][r], stats=st)
        B.vls_logp_bwd(i["xc"][r], i["ids_c"][r], i["g_c"][r], st, -100, CAP, dlogits=grad["cap_logp"][r])
        B.vls_softcap_fwd(i["xc"][r], CAP, y=o["y"][r])
        B.vls_softcap_bwd(i["xc"][r], i["gy"][r], CAP, gx=grad["softcap"][r])

    comp = torch.cuda.current_stream(device)
    s_ins = [torch.cuda.Stream(device) for _ in range(copy_streams)]
    s_outs = [torch.cuda.Stream(device) for _ in range(copy_streams)]
    ev = {k: [torch.cuda.Event() for _ in bounds] for k in ("in", "comp", "out")}

    def one():
        for c, (lo, hi) in enumerate(bounds):
            s_in, s_out = s_ins[c % copy_streams], s_outs[c % copy_streams]
            s_in.wait_event(ev["comp"][c])            # the previous step has read chunk c's inputs
            with torch.cuda.stream(s_in):
                for k, t in pinned_in.items():
                    i[k][lo:hi].copy_(t[lo:hi], non_blocking=True)
            ev["in"][c].record(s_in)
            comp.wait_event(ev["in"][c])
            comp.wait_event(ev["out"][c])             # the previous step's chunk c results are read back
            launches(lo, hi)
            ev["comp"][c].record(comp)
            s_out.wait_event(ev["comp"][c])
            with torch.cuda.stream(s_out):
                for k, t in dev_out.items():
                    host_out[k][lo:hi].copy_(t[lo:hi], non_blocking=True)
            ev["out"][c].record(s_out)

    one()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(comp)
    for st in s_ins + s_outs:
        st.wait_event(t0)
    for _ in range(steps):
        one()
    for e in ev["out"]:
        comp.wait_event(e)
    t1.record(comp)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps, h2d, d2h


# ----------------------------------------------------------------------------
# the five configurations, each on its own (reported beside the headline step)
# ----------------------------------------------------------------------------

CONFIGS = [
    ("C1", "logp_small", "logprobs k=1, 64 x 32000 fp32 (launch-bound: CUDA-graph replay reported too)"),
    ("C2", "logp_offset", "logprobs k=1, 8192 x 151936 bf16, offset rows, ignored and out-of-range targets"),
    ("C3", "kl_masked", "entropy, forward KL and reverse KL, 8192 x 75968 bf16, masked columns, mismatch rows"),
    ("C4", "softcap_wide", "softcap-fused logprobs at caps 30 and 20, and the standalone softcap, 4096 x 262144 bf16"),
    ("C5", "long_seq", "logprobs k=1 and k=256, entropy, 32768 x 151936 bf16; peak extra device memory"),
]


def config_summary(line: dict) -> dict:
    """The compact per-config record of the bench line: per op its forward
    and backward median ms, TB/s and fraction of the measured copy
    bandwidth, and the config's fwd+bwd totals."""
    peak = line["peak_gbs"]
    ops = {}
    for label, v in line["ops"].items():
        if label in line["comparison_ops"]:
            continue
        op, ps = label.rsplit(" ", 1)
        e = ops.setdefault(op, {})
        e[f"{ps}_ms"] = v["ms_median"]
        e[f"{ps}_tbs"] = v["tbs"]
        e[f"{ps}_frac"] = v["frac_of_measured"]
    for op, e in ops.items():
        if "fwd_ms" in e and "bwd_ms" in e:
            b = line["ops"][op + " fwd"]["bytes"] + line["ops"][op + " bwd"]["bytes"]
            ms = e["fwd_ms"] + e["bwd_ms"]
            e.update({"fwd_bwd_ms": round(ms, 4), "fwd_bwd_tbs": round(b / ms / 1e9, 3),
                      "fwd_bwd_frac": round(b / ms / 1e6 / peak, 4)})
    out = {"workload": line["workload"], "rows": line["rows"], "vocab": line["vocab"], "steps": line["steps"],
           "fwd_bwd_ms": line["fwd_bwd_ms"], "tbs": line["tbs"], "frac_of_measured": round(line["tbs"] * 1e3 / peak, 4),
           "l2": line["l2"], "ops": ops}
    if line.get("graph_replay"):
        out["graph_replay"] = {k: line["graph_replay"][k] for k in ("ms_median", "tbs") if k in line["graph_replay"]}
    if line.get("peak_extra_memory"):
        out["peak_extra_memory"] = line["peak_extra_memory"]
    return out


def measure_configs(device, steps: int, warmup: int) -> dict:
    import torch
    res = {}
    for key, name, what in CONFIGS:
        line = measure_workload(name, device, steps, warmup)
        res[key] = {"what": what, **config_summary(line)}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------
# CPU oracle (baseline arm)
# ----------------------------------------------------------------------------

def oracle_step(rows: dict) -> None:
    """One pass of the whole path on the CPU fp64 oracle over the given rows."""
    import oracle
    x, ids, g = rows["x"], rows["ids"], rows["g"]
    oracle.logp_fwd(x, ids)
    oracle.logp_bwd(x, ids, g)
    oracle.entropy_fwd(rows["a"])
    oracle.entropy_bwd(rows["a"], rows["g_row"])
    for d in ("reverse", "forward"):
        oracle.kl_fwd(rows["a"], rows["b"], d)
        oracle.kl_bwd(rows["a"], rows["b"], rows["g_row"], d)
    oracle.logp_fwd(rows["xc"], rows["ids_c"], -100, CAP)
    oracle.logp_bwd(rows["xc"], rows["ids_c"], rows["g_c"], -100, CAP)
    oracle.softcap(rows["xc"], CAP)
    oracle.softcap_grad(rows["xc"], rows["gy"], CAP)


def host_rows(inp: dict, lo: int, hi: int) -> dict:
    """Rows [lo, hi) of every input, decoded to float64 numpy on the host."""
    import numpy as np
    import torch

    import oracle
    out = {}
    for k, t in inp.items():
        s = t[lo:hi].detach().cpu()
        if s.dtype == torch.bfloat16:
            out[k] = oracle.decode_bf16_bits(s.view(torch.int16).numpy())
        elif s.dtype.is_floating_point:
            out[k] = s.to(torch.float64).numpy()
        else:
            out[k] = np.ascontiguousarray(s.numpy())
    return out


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


_BARRIER = None


def _oracle_init(barrier) -> None:
    global _BARRIER
    _BARRIER = barrier
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"


def _oracle_worker(job: tuple) -> tuple:
    """One process of the oracle pool: builds its own block of rows of the
    workload on the CPU (same recipe, its own seed), waits for the others,
    then runs the whole path on it `warmup + steps` times; returns the
    start and end of the timed steps on the system-wide monotonic clock."""
    rows, v, worker, steps, warmup = job
    import workloads
    inp = host_rows(_cpu_inputs(workloads, rows, v, seed_offset=100 * (worker + 1)), 0, rows)
    _BARRIER.wait()
    for _ in range(warmup):
        oracle_step(inp)
    _BARRIER.wait()
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(inp)
    return t0, time.perf_counter()


def _oracle_calibrate(v: int) -> float:
    """Seconds of one row of the whole path on the oracle in one process of
    the pool, timed while every other process runs the same probe (the
    processes share the host's memory bandwidth)."""
    import workloads
    rows = 8                 # more than the host's caches hold, as in the timed passes
    probe = host_rows(_cpu_inputs(workloads, rows, v), 0, rows)
    _BARRIER.wait()
    oracle_step(probe)
    t0 = time.perf_counter()
    oracle_step(probe)
    return (time.perf_counter() - t0) / rows


def host_memory_available() -> int:
    """Bytes of host memory available now (MemAvailable), 8 GiB if unknown."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 8 << 30


ORACLE_BYTES_PER_COLUMN = 96   # peak host memory of one oracle row of the whole path, per column (measured ~70)


def oracle_pool(v: int, steps: int, warmup: int, workers: int, budget_s: float, max_rows: int) -> tuple:
    """The oracle over `workers` processes, each on its own block of rows,
    sized so that its warm-up and timed passes take about budget_s seconds
    under contention and all blocks together stay within 40% of the host's
    available memory.  Returns (rows per worker, seconds per step: the wall
    time from the first worker's start to the last worker's end).  Processes
    are spawned (never forked after CUDA)."""
    import multiprocessing as mp
    mem_rows = int(0.4 * host_memory_available() / (workers * ORACLE_BYTES_PER_COLUMN * v))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(workers)
    with ctx.Pool(workers, initializer=_oracle_init, initargs=(barrier,)) as pool:
        per_row = max(pool.map(_oracle_calibrate, [v] * workers))
        rows = int(max(1, min(max_rows, mem_rows, budget_s / (steps + warmup) / max(per_row, 1e-6))))
        spans = pool.map(_oracle_worker, [(rows, v, w, steps, warmup) for w in range(workers)])
    return rows, (max(t1 for _, t1 in spans) - min(t0 for t0, _ in spans)) / steps


def cpu_baseline(n: int, v: int, budget_s: float = 12.0) -> dict:
    """The oracle, as it stands, on every host core: one process per core,
    each on its own block of rows of the workload (about budget_s seconds of
    work each)."""
    cores = host_cores()
    rows, dt = oracle_pool(v, 1, 0, cores, budget_s, n)
    total = rows * cores
    return {"value": round(step_bytes(total, v) / dt / 1e12, 6), "unit": "TB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes x {rows} rows of the workload's recipe (each its own seeded block), "
                      f"full V={v}; the whole path once; numpy fp64",
            "seconds": round(dt, 2)}


def step_config(n: int, v: int, world: int) -> dict:
    """The workload the step line is quoted on; both arms print it as is."""
    return {"workload": WORKLOAD, "rows_per_gpu": n, "vocab": v, "global_rows": n * world,
            "parallelism": f"dp{world} (row shards, no collective)",
            "l2": "inputs (2.5 GB per tensor) larger than L2; no flush",
            "bytes_per_step_per_gpu": step_bytes(n, v)}


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    n, v = args.rows, VOCAB
    cores = host_cores()
    rows, dt = oracle_pool(v, args.steps, args.warmup, cores, 120.0, n)   # about 2-3 minutes for the whole run
    s = rows * cores
    value = step_bytes(s, v) / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(n, v, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{cores} processes x {rows} of the {n} rows per step ({s} rows, a bounded "
                                   f"sample of the batch; value = their algorithmic bytes / time), full V={v}"},
        "e2e": {"value": round(value, 6), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _cpu_inputs(workloads, n: int, v: int, seed_offset: int = 0) -> dict:
    c2 = workloads.logp_offset("cpu", n=n, v=v, seed=1 + seed_offset)
    c3 = workloads.kl_masked("cpu", n=max(n, 2), v=v, seed=2 + seed_offset)
    c4 = workloads.softcap_wide("cpu", n=n, v=v, seed=3 + seed_offset)
    return {"x": c2["logits"], "ids": c2["ids"], "g": c2["g"], "a": c3["a"][:n], "b": c3["b"][:n],
            "g_row": c3["g"][:n], "xc": c4["logits"], "ids_c": c4["ids"], "g_c": c4["g"], "gy": c4["gy_bf16"]}


# ----------------------------------------------------------------------------
# main
# ----------------------------------------------------------------------------

def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--rows", type=int, default=N_ROWS, help="rows per GPU (default 8192)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--e2e-chunks", type=int, default=E2E_CHUNKS, help="row chunks of the host-buffer pipeline")
    ap.add_argument("--e2e-copy-streams", type=int, default=E2E_COPY_STREAMS,
                    help="copy streams per direction in the host-buffer pipeline")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config block (C1-C5)")
    ap.add_argument("--config-steps", type=int, default=20, help="timed steps per config in the per-config block")
    ap.add_argument("--config-warmup", type=int, default=3, help="warm-up steps per config (at least 3)")
    ap.add_argument("--workload", default="step",
                    choices=["step", "logp_small", "logp_offset", "kl_masked", "softcap_wide", "long_seq", "fused",
                             "linear_logp"],
                    help="step (default): the benchmark step; otherwise per-op times of one workload")
    args = ap.parse_args()
    if args.workload != "step" and args.impl == "ours":
        run_config(args)
        return

    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import torch.distributed as dist
    rank, world, local_rank = dist_env()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(device)

    import vocab_log_softmax_gb300 as vls
    vls.vls_version()                                     # fails loudly if libvls is missing
    n, v = args.rows, VOCAB
    step = Step(device, n, v, seed_offset=rank * 10)
    torch.cuda.synchronize()

    launches_per_step = len(step.launches())
    total_ms, per, clk = time_device(step, args.steps, args.warmup, device)
    total_ms = max_over_ranks(total_ms, device)
    ms = total_ms / args.steps
    sb = step_bytes(n, v)
    value = aggregate(sb, world, ms / 1e3)

    per_op = {}
    for op in OPS:
        b = op_bytes(op, n, v)
        f, bw = per[(op, "fwd")], per[(op, "bwd")]
        per_op[op] = {"fwd_ms": round(f, 4), "bwd_ms": round(bw, 4), "fwd_bwd_ms": round(f + bw, 4),
                      "fwd_tbs": round(b["fwd"] / f / 1e9, 3), "bwd_tbs": round(b["bwd"] / bw / 1e9, 3),
                      "fwd_bwd_tbs": round((b["fwd"] + b["bwd"]) / (f + bw) / 1e9, 3)}
    # dominant kernel: the launch with the largest share of the step's device time
    kernel_time = {}
    for (op, ps), t in per.items():
        kernel_time.setdefault(KERNEL_NAMES[(op, ps)], []).append((op, ps, t))
    dom_name, dom = max(kernel_time.items(), key=lambda kv: sum(t for _, _, t in kv[1]))
    dom_bytes = sum(op_bytes(op, n, v)[ps] for op, ps, _ in dom)
    dom_ms = sum(t for _, _, t in dom)
    peak, peak_kind = hbm_peak()
    achieved = dom_bytes / len(dom) / (dom_ms / len(dom)) / 1e6     # GB/s
    tr = traffic_for(dom_name, n)
    roofline = {"bound": "hbm", "kernel": dom_name, "achieved": round(achieved, 1), "peak": peak,
                "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": None if tr is None else round(tr), "bytes_per_launch": dom_bytes // len(dom),
                "share_of_step": round(dom_ms / ms, 4),
                "step_frac": round(sb / (ms / 1e3) / 1e9 / peak, 4)}

    e2e_ms, h2d, d2h = time_e2e(step, args.e2e_steps, device, args.e2e_chunks, args.e2e_copy_streams)
    e2e_ms = max_over_ranks(e2e_ms, device)
    e2e = {"value": round(aggregate(sb, world, e2e_ms / 1e3), 4), "unit": "TB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3), "steps": args.e2e_steps,
           "pipeline": {"row_chunks": args.e2e_chunks, "copy_streams_per_direction": args.e2e_copy_streams}}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(n, v)

    configs = None
    if not args.no_configs:
        del step
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        configs = measure_configs(device, args.config_steps, max(3, args.config_warmup))

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": step_config(n, v, world),
            "per_op": per_op,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
