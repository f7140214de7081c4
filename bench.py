#!/usr/bin/env python
"""Benchmark of the bitwise-aligned causal GQA attention hot path on GB300.

One step = one causal prefill (B=4, S=16384) and one one-token decode
(B=16, ctx=8192), Hq=32, Hkv=8, D=128, bf16, through the library's C ABI.
Inputs are synthetic (iid N(0,1) rounded to bf16, seeded) and larger than L2.

Prints ONE JSON line.  `value` is prefill throughput in causal TFLOP/s
(4*B*Hq*D*S(S+1)/2 per call) summed over ranks; the decode leg's KV GB/s sits
under "decode".  `--impl reference` times the fp64 CPU oracle instead, on a
bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]
For N>1 launch one process per GPU with torch.distributed.run.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill causal TFLOP/s & decode KV GB/s at 1 GB300 (% roofline), bitwise-aligned"
HQ, HKV, D = 32, 8, 128
# full: the headline workload; small: the same kernels at a size an ncu
# replay handles quickly (inputs still larger than L2)
WORKLOADS = {"full": (4, 16384, 16, 8192), "small": (4, 4096, 16, 8192)}
PREFILL_B, PREFILL_S, DECODE_B, DECODE_CTX = WORKLOADS["full"]
SEED_PREFILL = 7_000_001
SEED_DECODE = 7_000_002
SEED_BACKWARD = 7_000_003


def workload_name():
    return (f"causal GQA prefill B={PREFILL_B} S={PREFILL_S} + one-token decode B={DECODE_B} ctx={DECODE_CTX}, "
            f"Hq={HQ} Hkv={HKV} D={D} bf16")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# ncu dram bytes (read + write) per launch, each with the hash of the kernel
# sources it was captured on and the profile summary that records it.  When
# the sources differ from that hash, the figure no longer describes the timed
# build and the bench line reports traffic as null.
NCU_TRAFFIC = {
    "prefill": {"bytes": 806.31e6 + 503.93e6, "sources": "9ffdbcc262b023f9",
                "profile": "profiles/launch_list_bench_full.md"},
    "decode": {"bytes": 537.09e6 + 0.22e6, "sources": "fcbe3f1dc60b9ee3",
               "profile": "profiles/launch_list_bench_full.md"},
    # one kb_attn_backward call: the delta, dq and dk/dv kernels together
    "backward": {"bytes": 3832.15e6 + 774.73e6, "sources": "0195856a1fa6798b",
                 "profile": "profiles/launch_list_bench_full.md"},
}
KERNEL_SOURCES = {
    "prefill": ["kb_prefill2.cu", "kb_contract.cuh", "kb_ptx.cuh", "kb_launch.h", "kb_host.cu"],
    "decode": ["kb_decode.cu", "kb_contract.cuh", "kb_ptx.cuh", "kb_launch.h", "kb_host.cu"],
    "backward": ["kb_backward.cu", "kb_contract.cuh", "kb_ptx.cuh", "kb_launch.h", "kb_host.cu"],
}


def sources_hash(kernel: str) -> str:
    """sha256 (16 hex digits) over the CUDA sources that define a kernel and its launch."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bitwise_aligned_causal_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic(kernel: str):
    """(bytes or None, provenance dict) of the ncu DRAM traffic for the current sources."""
    rec = NCU_TRAFFIC[kernel]
    cur = sources_hash(kernel)
    fresh = rec["bytes"] is not None and rec["sources"] == cur
    return (rec["bytes"] if fresh else None), {"profile": rec["profile"], "captured_on_sources": rec["sources"],
                                               "current_sources": cur, "fresh": fresh}


def prefill_flops(B: int, S: int) -> int:
    """Algorithmic causal FLOPs: Q K^T and P V over the S(S+1)/2 visible pairs."""
    return 4 * B * HQ * D * S * (S + 1) // 2


def decode_bytes(B: int, ctx: int) -> int:
    """Algorithmic bytes: K and V of the context read once per KV head, q read and o written."""
    return 2 * B * HKV * ctx * D * 2 + 2 * B * HQ * D * 2


# ------------------------------------------------------------------ environment

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                raw = json.load(f)
            flat = {}

            def walk(d):
                for kk, vv in d.items():
                    if isinstance(vv, dict):
                        walk(vv)
                    elif isinstance(vv, (int, float)):
                        flat.setdefault(kk, float(vv))

            walk(raw)
            if "hbm_gbs" in flat and "bf16_tflops" in flat:
                out = {"hbm_gbs": flat["hbm_gbs"], "bf16_tflops": flat["bf16_tflops"],
                       "bf16_tflops_sustained": flat.get("bf16_tflops_sustained", flat["bf16_tflops"]),
                       "source": "measured"}
                return out
        except Exception:  # noqa: BLE001 - fall through to the fallback figures
            pass
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="kb_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ distributed glue

def dist_setup(n_gpus: int):
    """(rank, world, local_rank) -- one process per GPU under torch.distributed.run."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if n_gpus > 1 and world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} needs a torch.distributed.run launch with {n_gpus} processes")
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = os.environ.get("KB_DIST_BACKEND", "nccl")
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist

        if dist.get_backend() == "nccl" and device is not None:
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def reduce_max(value: float, world: int, device: str = "cpu") -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_units: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank processed `per_rank_units`; the job took the slowest rank's time."""
    return per_rank_units * world / max_seconds


# ------------------------------------------------------------------ CPU oracle legs

def oracle_sample_rate(x_pre, budget_s: float, seed: int, n_threads: int | None = None):
    """Time the oracle on random prefill rows of the workload for ~budget_s; return (flop/s, rows, threads)."""
    import numpy as np

    import oracle

    rng = np.random.default_rng(seed)
    B, _, S, _ = x_pre.q.shape
    nt = oracle.default_threads() if n_threads is None else n_threads
    flops = 0
    rows_done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        n = max(nt, 32)
        rows = np.stack([rng.integers(0, B, n), rng.integers(0, HQ, n), rng.integers(0, S, n)], axis=1)
        oracle.attention_rows(x_pre.q, x_pre.k, x_pre.v, rows, n_threads=nt)
        flops += int(sum(4 * D * (int(i) + 1) for i in rows[:, 2]))
        rows_done += n
    dt = time.perf_counter() - t0
    return flops / dt, rows_done, nt, dt


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is a bounded sample of the same workload."""
    if rank != 0:
        return
    from bitwise_aligned_causal_gb300 import inputs

    x = inputs.make_qkv(PREFILL_B, PREFILL_S, SEED_PREFILL)
    for _ in range(args.warmup):
        oracle_sample_rate(x, 0.5, seed=11)
    rates, secs, rows, nt = [], [], 0, 1
    for s in range(args.steps):
        r, n, nt, dt = oracle_sample_rate(x, 2.0, seed=100 + s)
        rates.append(r)
        secs.append(dt)
        rows += n
    value = statistics.mean(rates) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: iid N(0,1) rounded to bf16 (numpy default_rng)",
        "config": {"workload": workload_name(), "parallelism": "none (CPU oracle, rank 0 only)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
                         "sample": f"{rows} random prefill query rows of the workload (about 2 s of oracle work per step)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from bitwise_aligned_causal_gb300 import build, inputs

    torch.cuda.set_device(local)
    build.build()
    from bitwise_aligned_causal_gb300 import kb_attn

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    x = inputs.make_qkv(PREFILL_B, PREFILL_S, SEED_PREFILL + 1000 * rank)
    y = inputs.make_qkv(DECODE_B, DECODE_CTX, SEED_DECODE + 1000 * rank, Lq=1)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    qd, kd, vd = to_dev(y.q), to_dev(y.k), to_dev(y.v)
    o = torch.empty_like(q)
    od = torch.empty_like(qd)

    def step():
        kb_attn.prefill(q, k, v, out=o)
        kb_attn.decode(qd, kd, vd, DECODE_CTX, out=od)

    for _ in range(max(args.warmup, 3)):
        step()
    kb_attn.check_device_status()

    # --- timed region: device-resident inputs, events per kernel on the launching stream
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    barrier(world, local)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(n):
            ev[i][0].record(stream)
            kb_attn.prefill(q, k, v, out=o)
            ev[i][1].record(stream)
            kb_attn.decode(qd, kd, vd, DECODE_CTX, out=od)
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world, local)
    clocks = clk.summary()
    kb_attn.check_device_status()
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    dec_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    step_ms_max = reduce_max(total_ms / n, world, "cuda" if world > 1 else "cpu")
    pre_ms_max = reduce_max(pre_ms, world, "cuda" if world > 1 else "cpu")
    dec_ms_max = reduce_max(dec_ms, world, "cuda" if world > 1 else "cpu")

    pf = prefill_flops(PREFILL_B, PREFILL_S)
    db = decode_bytes(DECODE_B, DECODE_CTX)
    pre_tflops = aggregate(pf, world, pre_ms_max / 1e3) / 1e12
    dec_gbs = aggregate(db, world, dec_ms_max / 1e3) / 1e9

    # --- end to end: pinned host inputs copied in, result copied out, every step
    if args.no_e2e:
        e2e = None
    else:
        e2e = run_e2e(args, x, y, q, k, v, o, qd, kd, vd, od, stream, world, local, kb_attn)
    bwd = None if args.no_backward else run_backward(args, q, k, v, stream, world, local, rank, kb_attn)
    grid = None
    if not args.no_grid:
        barrier(world, local)
        grid = grid_summary(time_grid(kb_attn, load_peaks(), (1,), dev), load_peaks())
    if rank != 0:
        return
    emit_line(args, world, n, step_ms_max, pre_ms, dec_ms, pre_ms_max, dec_ms_max, pre_tflops, dec_gbs, e2e, clocks, x,
              bwd, grid)


def run_backward(args, q, k, v, stream, world, local, rank, kb_attn):
    """The training pair on the prefill workload: kb_attn_prefill_lse, then
    kb_attn_backward for a seeded N(0,1) output gradient, each timed alone
    (CUDA events on the launching stream, device-resident inputs)."""
    import numpy as np
    import torch

    from bitwise_aligned_causal_gb300 import inputs

    dob = inputs.make_qkv(PREFILL_B, PREFILL_S, SEED_BACKWARD + 1000 * rank).q
    do = torch.from_numpy(np.ascontiguousarray(dob).view(np.int16)).view(torch.bfloat16).to(q.device)
    o, lse = kb_attn.prefill_lse(q, k, v)
    dq, dk, dv, delta = kb_attn.backward(q, k, v, o, do, lse)
    reps = max(3, min(args.steps, 10))

    def timed(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    barrier(world, local)
    fwd_ms = timed(lambda: kb_attn.prefill_lse(q, k, v, out=o, lse=lse))
    bwd_ms = timed(lambda: kb_attn.backward(q, k, v, o, do, lse, delta=delta, dq=dq, dk=dk, dv=dv))
    kb_attn.check_device_status()
    dev = "cuda" if world > 1 else "cpu"
    return {"fwd_ms": reduce_max(fwd_ms, world, dev), "bwd_ms": reduce_max(bwd_ms, world, dev), "reps": reps,
            "fwd_ms_local": fwd_ms, "bwd_ms_local": bwd_ms}


def pipelined_e2e(n, host_in, dev_sets, host_out, launch):
    """Per-step time (ms) of n steps, each copying its inputs from pinned host
    memory, computing, and copying its result back.  Two device buffer sets
    and two copy streams let step i+1's upload and step i-1's download run
    under step i's kernels; every byte of every step still crosses inside the
    timed region."""
    import torch

    cs = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(n)]
    ev_comp = [torch.cuda.Event() for _ in range(n)]
    ev_down = [torch.cuda.Event() for _ in range(n)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(up)
    for i in range(n):
        s = i % 2
        ins, out = dev_sets[s]
        if i >= 2:
            up.wait_event(ev_comp[i - 2])          # buffer set s is free once step i-2 has computed
        with torch.cuda.stream(up):
            for d, h in zip(ins, host_in):
                d.copy_(h, non_blocking=True)
        ev_up[i].record(up)
        cs.wait_event(ev_up[i])
        if i >= 2:
            cs.wait_event(ev_down[i - 2])          # ... and its result has been read back
        launch(ins, out)
        ev_comp[i].record(cs)
        down.wait_event(ev_comp[i])
        with torch.cuda.stream(down):
            host_out[s].copy_(out, non_blocking=True)
        ev_down[i].record(down)
    t1.record(down)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n


def link_bandwidth(host_in, dev_in, host_out, dev_out):
    """Host<->device copy bandwidth alone (GB/s): the prefill inputs uploaded,
    its output downloaded, each timed on its own."""
    import torch

    st = torch.cuda.Stream()
    e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        e0.record(st)
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        e1.record(st)
        host_out.copy_(dev_out, non_blocking=True)
        e2.record(st)
    torch.cuda.synchronize()
    up = sum(h.numel() * h.element_size() for h in host_in)
    down = host_out.numel() * host_out.element_size()
    return up / (e0.elapsed_time(e1) * 1e6), down / (e1.elapsed_time(e2) * 1e6)


def run_e2e(args, x, y, q, k, v, o, qd, kd, vd, od, stream, world, local, kb_attn):
    import numpy as np
    import torch

    n = max(4, min(args.steps, 12))
    pf = prefill_flops(PREFILL_B, PREFILL_S)
    db = decode_bytes(DECODE_B, DECODE_CTX)

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = pinned(x.q), pinned(x.k), pinned(x.v)
    hqd, hkd, hvd = pinned(y.q), pinned(y.k), pinned(y.v)
    ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    hod = [torch.empty(od.shape, dtype=od.dtype).pin_memory() for _ in range(2)]
    pre_sets = [([q, k, v], o), ([torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)], torch.empty_like(o))]
    dec_sets = [([qd, kd, vd], od),
                ([torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)], torch.empty_like(od))]
    pre_launch = lambda ins, out: kb_attn.prefill(ins[0], ins[1], ins[2], out=out)  # noqa: E731
    dec_launch = lambda ins, out: kb_attn.decode(ins[0], ins[1], ins[2], DECODE_CTX, out=out)  # noqa: E731
    # untimed warm-up of the same pipeline: the first copies out of freshly
    # pinned host buffers are slower than the steady state
    pipelined_e2e(2, [hq, hk, hv], pre_sets, ho, pre_launch)
    pipelined_e2e(2, [hqd, hkd, hvd], dec_sets, hod, dec_launch)
    barrier(world, local)
    # three runs of the pipeline, the median reported: the host side of the
    # link is shared with the machine's other work, and a run where the
    # upload and the download stop overlapping reads far lower than the rest
    pre_runs = [pipelined_e2e(n, [hq, hk, hv], pre_sets, ho, pre_launch) for _ in range(3)]
    dec_runs = [pipelined_e2e(n, [hqd, hkd, hvd], dec_sets, hod, dec_launch) for _ in range(3)]
    pre_ms = sorted(pre_runs)[1]
    dec_ms = sorted(dec_runs)[1]
    kb_attn.check_device_status()
    h2d_gbs, d2h_gbs = link_bandwidth([hq, hk, hv], pre_sets[1][0], ho[0], o)
    # the downloaded results are the kernels' results
    assert torch.equal(ho[(n - 1) % 2].view(torch.int16), o.view(torch.int16).cpu())
    e2e_pre_ms = reduce_max(pre_ms, world, "cuda" if world > 1 else "cpu")
    e2e_dec_ms = reduce_max(dec_ms, world, "cuda" if world > 1 else "cpu")
    h2d = sum(t.numel() * 2 for t in (hq, hk, hv, hqd, hkd, hvd))
    d2h = (ho[0].numel() + hod[0].numel()) * 2
    return {"value": aggregate(pf, world, e2e_pre_ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "decode_gbs": aggregate(db, world, e2e_dec_ms / 1e3) / 1e9, "steps": n,
            "runs_ms": {"prefill": [round(t, 4) for t in pre_runs], "decode": [round(t, 4) for t in dec_runs]},
            "of_runs": "median of three pipelined runs of `steps` steps",
            "copy_only_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs},
            "note": ("every step uploads its inputs from pinned host memory and downloads its output; "
                     "two buffer sets let one step's copies overlap the neighbouring step's kernels; "
                     "bound by the host link when (h2d + d2h bytes) / copy_only_gbs exceeds the kernel time")}


def emit_line(args, world, n, step_ms_max, pre_ms, dec_ms, pre_ms_max, dec_ms_max, pre_tflops, dec_gbs, e2e, clocks,
              x, bwd=None, grid=None):
    pf = prefill_flops(PREFILL_B, PREFILL_S)
    db = decode_bytes(DECODE_B, DECODE_CTX)
    peaks = load_peaks()
    pre_per_launch = pf / (pre_ms / 1e3) / 1e12
    dec_per_launch = db / (dec_ms / 1e3) / 1e9
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, rows, nt, dt = oracle_sample_rate(x, args.cpu_seconds, seed=99)
        cpu = {"value": rate / 1e12, "unit": "TFLOP/s", "cores": nt, "kind": "oracle",
               "sample": f"{rows} random prefill query rows of the workload, {dt:.1f} s of oracle work on "
                         f"{os.cpu_count()} host cores"}
    tr_pre, tr_pre_src = traffic("prefill")
    tr_dec, tr_dec_src = traffic("decode")
    line = {
        "metric": METRIC,
        "value": pre_tflops,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": n,
        "warmup": max(args.warmup, 3),
        "ms_per_step": step_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: iid N(0,1) rounded to bf16 (numpy default_rng, seeds 7000001/7000002 + 1000*rank)",
        "config": {
            "workload": workload_name(),
            "prefill": {"B": PREFILL_B, "S": PREFILL_S, "Hq": HQ, "Hkv": HKV, "D": D},
            "decode": {"B": DECODE_B, "ctx": DECODE_CTX, "Hq": HQ, "Hkv": HKV, "D": D},
            "parallelism": f"replicas x{world} (independent batches per GPU)",
            "l2": (f"inputs larger than L2 (prefill q/k/v {3 * PREFILL_B * HQ * PREFILL_S * D * 2 // 2 // 1000000} MB, "
                   f"decode K/V {2 * DECODE_B * HKV * DECODE_CTX * D * 2 // 1000000} MB per step), no flush"),
        },
        "decode": {
            "value": dec_gbs, "unit": "GB/s", "ms": dec_ms_max,
            "roofline": {"bound": "hbm", "achieved": dec_per_launch, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": dec_per_launch / peaks["hbm_gbs"],
                         "traffic": tr_dec, "traffic_source": tr_dec_src, "peak_source": peaks["source"]},
        },
        "roofline": {
            "bound": "tensor", "achieved": pre_per_launch, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": pre_per_launch / peaks["bf16_tflops"], "traffic": tr_pre, "traffic_source": tr_pre_src,
            "kernel": "kb_prefill_kernel_s2", "peak_source": peaks["source"] + " burst bf16",
            "frac_of_sustained": pre_per_launch / peaks["bf16_tflops_sustained"],
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 2 * n,
        "clocks": clocks,
    }
    if bwd is not None:
        bf = 2.5 * pf                                   # dq, dk, dv: five products of the forward's size
        per_launch = bf / (bwd["bwd_ms_local"] / 1e3) / 1e12
        tr_bwd, tr_bwd_src = traffic("backward")
        line["backward"] = {
            "value": 2.5 * aggregate(pf, world, bwd["bwd_ms"] / 1e3) / 1e12, "unit": "TFLOP/s", "ms": bwd["bwd_ms"],
            "flops": "algorithmic 2.5 x the forward's (five products over the visible pairs)",
            "workload": f"kb_attn_backward on the prefill workload (B={PREFILL_B} S={PREFILL_S}), dO ~ N(0,1)",
            "forward_with_lse": {"value": aggregate(pf, world, bwd["fwd_ms"] / 1e3) / 1e12, "unit": "TFLOP/s",
                                 "ms": bwd["fwd_ms"]},
            "reps": bwd["reps"],
            "roofline": {"bound": "tensor", "achieved": per_launch, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": per_launch / peaks["bf16_tflops"], "traffic": tr_bwd, "traffic_source": tr_bwd_src,
                         "kernel": "kb_bwd_delta_kernel + kb_bwd_dq_kernel + kb_bwd_dkdv_kernel (one call)",
                         "peak_source": peaks["source"] + " burst bf16"},
        }
    if grid is not None:
        line["grid"] = grid
    print(json.dumps(line), flush=True)


GRID_PREFILL_S = (1024, 4096, 8192, 16384)
GRID_LONG_DECODE = ((1, 16384), (1, 32768), (1, 65536), (2, 32768))
GRID_DECODE_CTX = (128, 1024, 4096, 8192)
GRID_B = (1, 4, 8, 16)


L2_BYTES = 129e6      # GB300 L2


def rotating_launch_ms(make, launch, bytes_per_copy, device, min_launches=48):
    """Mean device time (ms) of one launch, timed over back-to-back launches on
    rotating copies of the inputs that together exceed L2 twice over (so no
    launch finds its inputs in L2 and no flush kernel runs between launches).
    The launches are captured in a CUDA graph when the stream allows it, so
    host-side launch cost does not enter; otherwise they are enqueued
    directly.  Returns (ms, copies, method)."""
    import torch

    R = max(1, min(256, int(2 * L2_BYTES // max(1, bytes_per_copy)) + 1))
    bufs = [make() for _ in range(R)]
    for bb in bufs[: min(R, 3)]:
        launch(bb)
    torch.cuda.synchronize(device)
    reps = max(1, (min_launches + R - 1) // R)
    method = "graph"
    try:
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream(device)
        with torch.cuda.stream(st):
            for bb in bufs:
                launch(bb)
            torch.cuda.synchronize(device)
            with torch.cuda.graph(g, stream=st):
                for bb in bufs:
                    launch(bb)
        torch.cuda.synchronize(device)
        g.replay()
        torch.cuda.synchronize(device)

        def run():
            for _ in range(reps):
                g.replay()
    except Exception:  # noqa: BLE001 - capture unsupported: enqueue the launches directly
        method = "stream"
        torch.cuda.synchronize(device)

        def run():
            for _ in range(reps):
                for bb in bufs:
                    launch(bb)
    a = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    a.record()
    run()
    e.record()
    torch.cuda.synchronize(device)
    return a.elapsed_time(e) / (reps * R), R, method


def time_grid(kb_attn, peaks, prefill_batches, device):
    """The configuration grid of the KernelBraid README ("Performance":
    prefill at S in 1K..16K, decode at B in 1..16 x ctx in 128..8K).  Each
    configuration is timed as back-to-back launches over rotating input copies
    larger than L2 (rotating_launch_ms).  Returns one record per configuration."""
    import torch

    gen = torch.Generator(device=device)
    out = []

    def randn(shape):
        return torch.randn(shape, device=device, dtype=torch.bfloat16, generator=gen)

    for S in GRID_PREFILL_S:
        for B in prefill_batches:
            gen.manual_seed(8_000_000 + 100 * (S // 1024) + B)
            per_copy = (2 * B * HQ * S + 2 * B * HKV * S) * D * 2
            ms, R, how = rotating_launch_ms(
                lambda: (randn((B, HQ, S, D)), randn((B, HKV, S, D)), randn((B, HKV, S, D)),
                         torch.empty((B, HQ, S, D), device=device, dtype=torch.bfloat16)),
                lambda t: kb_attn.prefill(t[0], t[1], t[2], out=t[3]), per_copy, device)
            tf = prefill_flops(B, S) / (ms / 1e3) / 1e12
            out.append({"kind": "prefill", "S": S, "B": B, "ms": ms, "TFLOP/s": tf, "frac": tf / peaks["bf16_tflops"],
                        "copies": R, "timing": how})
            torch.cuda.empty_cache()
    for ctx in GRID_DECODE_CTX:
        for B in GRID_B:
            gen.manual_seed(9_000_000 + ctx + B)
            per_copy = decode_bytes(B, ctx)
            ms, R, how = rotating_launch_ms(
                lambda: (randn((B, HQ, 1, D)), randn((B, HKV, ctx, D)), randn((B, HKV, ctx, D)),
                         torch.empty((B, HQ, 1, D), device=device, dtype=torch.bfloat16)),
                lambda t: kb_attn.decode(t[0], t[1], t[2], ctx, out=t[3]), per_copy, device)
            gbs = decode_bytes(B, ctx) / (ms / 1e3) / 1e9
            out.append({"kind": "decode", "ctx": ctx, "B": B, "us": ms * 1e3, "GB/s": gbs,
                        "frac": gbs / peaks["hbm_gbs"], "copies": R, "timing": how})
            torch.cuda.empty_cache()
    # beyond the README grid: long-context decode of small batches, where the
    # segments of one sequence spread over a cluster and meet in one CTA
    for B, ctx in GRID_LONG_DECODE:
        gen.manual_seed(9_500_000 + ctx + B)
        per_copy = decode_bytes(B, ctx)
        ms, R, how = rotating_launch_ms(
            lambda: (randn((B, HQ, 1, D)), randn((B, HKV, ctx, D)), randn((B, HKV, ctx, D)),
                     torch.empty((B, HQ, 1, D), device=device, dtype=torch.bfloat16)),
            lambda t: kb_attn.decode(t[0], t[1], t[2], ctx, out=t[3]), per_copy, device, min_launches=24)
        gbs = decode_bytes(B, ctx) / (ms / 1e3) / 1e9
        out.append({"kind": "decode_long", "ctx": ctx, "B": B, "us": ms * 1e3, "GB/s": gbs,
                    "frac": gbs / peaks["hbm_gbs"], "copies": R, "timing": how})
        torch.cuda.empty_cache()
    kb_attn.check_device_status()
    return out


def grid_summary(records, peaks):
    """The grid as the KernelBraid README ("Performance") reports it: the prefill bar over S at B=1 and the
    decode bar over all 16 (B, ctx) cells, here as mean fractions of roofline."""
    pre = [r for r in records if r["kind"] == "prefill" and r["B"] == 1]
    dec = [r for r in records if r["kind"] == "decode"]
    long_ctx = [r for r in records if r["kind"] == "decode_long"]
    return {
        "workload": ("KernelBraid README grid: prefill B=1, S in 1K/4K/8K/16K; decode B in 1/4/8/16 x ctx in 128/1K/4K/8K; "
                     "Hq=32 Hkv=8 D=128 bf16, torch.randn inputs; each configuration timed over back-to-back "
                     "launches (a CUDA graph) on rotating input copies that together exceed L2 twice over, "
                     "so no launch finds its inputs in L2"),
        "timing": sorted({r["timing"] for r in records}),
        "prefill_b1": {str(r["S"]): {"TFLOP/s": round(r["TFLOP/s"], 1), "frac": round(r["frac"], 4)} for r in pre},
        "decode": {f"B{r['B']}_ctx{r['ctx']}": {"GB/s": round(r["GB/s"], 1), "us": round(r["us"], 2),
                                                "frac": round(r["frac"], 4)} for r in dec},
        "prefill_bar_mean_frac": statistics.mean(r["frac"] for r in pre),
        "decode_bar_mean_frac": statistics.mean(r["frac"] for r in dec),
        "decode_long_ctx": {f"B{r['B']}_ctx{r['ctx']}": {"GB/s": round(r["GB/s"], 1), "us": round(r["us"], 2),
                                                        "frac": round(r["frac"], 4)} for r in long_ctx},
        "peaks": {"bf16_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"], "source": peaks["source"]},
    }


def run_sweep(args, local):
    """Time the whole grid (prefill S x B, decode ctx x B), one JSON line per configuration."""
    import torch

    from bitwise_aligned_causal_gb300 import build

    torch.cuda.set_device(local)
    build.build()
    from bitwise_aligned_causal_gb300 import kb_attn

    peaks = load_peaks()
    for r in time_grid(kb_attn, peaks, GRID_B, torch.device("cuda", local)):
        print(json.dumps(dict(r, peak_source=peaks["source"])), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true", help="skip timing the training forward + backward")
    ap.add_argument("--no-grid", action="store_true", help="skip timing the README's configuration grid")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="full")
    ap.add_argument("--sweep", action="store_true",
                    help="time every prefill (S x B) and decode (ctx x B) configuration of the grid instead")
    args = ap.parse_args()
    global PREFILL_B, PREFILL_S, DECODE_B, DECODE_CTX
    PREFILL_B, PREFILL_S, DECODE_B, DECODE_CTX = WORKLOADS[args.workload]
    rank, world, local = dist_setup(args.gpus)
    try:
        if args.sweep:
            if rank == 0:
                run_sweep(args, local)
        elif args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
