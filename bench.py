#!/usr/bin/env python3
"""Throughput of one FlashAttention-2 training step (forward + backward) on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
fa2_fwd (O, L) then fa2_bwd (D preprocessing, then one launch of the K/V-outer dK/dV workers and the
Q-outer dQ workers). The metric is TFLOP/s with the usual FLOP convention
(forward 4*B*H*N^2*d, halved under the causal mask; backward 2.5x forward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl fa2|reference]

Prints one JSON line (rank 0). Under torchrun each rank runs the same
workload on its own GPU with its own seed (independent heads, no collective
on the data path); the timed region is bracketed by a barrier and
torch.cuda.synchronize() and the slowest rank's time is used.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "attention fwd/bwd TFLOPS on 1 GB300 (causal & not); % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
PROFILE_TRAFFIC = ROOT / "profiles" / "traffic.json"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=None)
    p.add_argument("--impl", default="fa2", choices=["fa2", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-sample-heads", type=int, default=6)
    p.add_argument("--no-configs", action="store_true",
                   help="skip the forward/backward lines of the other configurations")
    p.add_argument("--fwd-splits", default="auto",
                   help="K/V parts per forward worker: an integer, or 'auto' for the library's "
                        "rule (the default of forward())")
    p.add_argument("--record-traffic", metavar="NCU_REP", default=None,
                   help="write profiles/traffic.json from an ncu report of --workload "
                        "(dram__bytes_read.sum + dram__bytes_write.sum per kernel launch, scaled "
                        "to the headline workload by heads) and exit")
    p.add_argument("--e2e-heads-per-chunk", type=int, default=0,
                   help="heads per pipelined chunk of the end-to-end leg (fa2_step_host; 0 = auto)")
    p.add_argument("--bwd", default="split", choices=["split", "atomic"],
                   help="backward: split (fa2_bwd: dK/dV workers and dQ workers, no atomics) or "
                        "atomic (fa2_bwd_atomic: column workers with fp32 dQ reduce-adds)")
    p.add_argument("--fwd-order", default="fa2", choices=["fa2", "kv_outer"],
                   help="forward loop order: fa2 (Q outer) or kv_outer (the FlashAttention-1 "
                        "order, fa2_fwd_kv_outer), for measuring the loop order")
    return p.parse_args()


def peaks():
    f = ROOT / "MEASURED_PEAKS.json"
    if f.exists():
        d = json.loads(f.read_text())
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def source_sha(files) -> str:
    """Hash of a kernel's CUDA sources: recorded ncu counters are only used
    while it matches."""
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        h.update((ROOT / "exact_attention_64_gb300" / "csrc" / f).read_bytes())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def slowest_rank_ms(ms: float, dist=None, device=None) -> float:
    """The timed region's duration on the slowest rank (the max over ranks)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch

    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank_step: float, world: int, steps: int, ms: float) -> float:
    """Whole-job throughput: work of all ranks over the slowest rank's time
    (weak scaling: every rank processes its own heads)."""
    return flops_per_rank_step * world * steps / (ms * 1e-3) / 1e12


def cpu_baseline(w, heads: int):
    """The fp64 oracle, as it stands, on a bounded sample of the workload: the
    first `heads` heads, forward and backward timed separately. Returns
    TFLOP/s in the metric's FLOP convention (fwd+bwd, and each on its own)."""
    import torch

    import oracle
    from exact_attention_64_gb300.workloads import make_inputs

    q, k, v, do = make_inputs(1, heads, w.N, w.d, w.torch_dtype, w.q_std, seed=0)
    f = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    q, k, v, do = map(f, (q, k, v, do))
    t0 = time.perf_counter()
    oracle.forward(q, k, v, causal=w.causal, scale=w.scale)
    t1 = time.perf_counter()
    oracle.backward(q, k, v, do, causal=w.causal, scale=w.scale)
    t2 = time.perf_counter()
    fwd_s, bwd_s = t1 - t0, t2 - t1
    per_head_f = w.fwd_flops() / (w.B * w.H)
    per_head_b = w.bwd_flops() / (w.B * w.H)
    return {"value": (per_head_f + per_head_b) * heads / (fwd_s + bwd_s) / 1e12, "unit": UNIT,
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} heads (N={w.N}, d={w.d}), fwd and bwd in fp64 "
                      f"NumPy, {fwd_s:.2f} s + {bwd_s:.2f} s",
            "fwd_tflops": per_head_f * heads / fwd_s / 1e12,
            "bwd_tflops": per_head_b * heads / bwd_s / 1e12,
            "seconds": fwd_s + bwd_s}


def run_reference(args, w, rank, world):
    """The reference arm: the fp64 oracle on the host cores, one head per step."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_baseline(w, 1)
    steps = [cpu_baseline(w, 1) for _ in range(args.steps)]
    total = sum(s["seconds"] for s in steps)
    per_head = (w.fwd_flops() + w.bwd_flops()) / (w.B * w.H)
    value = per_head * len(steps) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "q_std": w.q_std, "step": "one (batch, head) of the workload, fwd+bwd"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "one head of the workload per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


TRAFFIC_FILES = {
    "fa2_fwd_kernel": ["fa2_fwd.cu", "fa2_common.cuh", "sm103_ptx.cuh"],
    "fa2_fwd_persist_kernel": ["fa2_fwd.cu", "fa2_fwd_persist.cuh", "fa2_common.cuh", "sm103_ptx.cuh"],
    "fa2_bwd_main_kernel": ["fa2_bwd.cu", "fa2_bwd_persist.cuh", "fa2_bwd_parts.cuh", "fa2_common.cuh",
                            "sm103_ptx.cuh"],
    "fa2_bwd_fused_kernel": ["fa2_bwd_fused.cu", "fa2_bwd_parts.cuh", "fa2_common.cuh",
                             "sm103_ptx.cuh"],
    "fa2_bwd_pre_kernel": ["fa2_bwd.cu", "fa2_bwd_persist.cuh", "fa2_bwd_parts.cuh", "fa2_common.cuh",
                           "sm103_ptx.cuh"],
    "fa2_bwd_dq_convert_kernel": ["fa2_bwd_fused.cu", "fa2_bwd_parts.cuh", "fa2_common.cuh",
                                  "sm103_ptx.cuh"],
}


def parse_ncu_dram(text: str) -> dict:
    """{kernel base name: (DRAM bytes read, DRAM bytes written)} of the first
    launch of each kernel in an `ncu --page raw --csv` export (a header row, a
    units row, then one row per launch)."""
    import csv
    import io

    rows = list(csv.reader(io.StringIO(text)))
    hdr, units, data = rows[0], rows[1], rows[2:]
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}

    def col(row, name):
        i = hdr.index(name)
        return float(row[i]) * scale[units[i]]

    out = {}
    for row in data:
        name = row[hdr.index("Kernel Name")].split("(")[0].split("<")[0].split()[-1].split("::")[-1]
        if name not in out:
            out[name] = (col(row, "dram__bytes_read.sum"), col(row, "dram__bytes_write.sum"))
    return out


def record_traffic(rep: str, measured) -> None:
    """profiles/traffic.json from one ncu capture of `measured` (one launch per
    kernel): DRAM bytes read + written per launch, scaled to the headline
    workload by the heads processed (same sequence length: each kernel reads its
    inputs once and writes its outputs once, so traffic grows with B*H), with
    the hash of the kernel's sources at the time of the capture."""
    from exact_attention_64_gb300.workloads import HEADLINE, WORKLOADS

    head = WORKLOADS[HEADLINE]
    if (measured.N, measured.d, measured.causal) != (head.N, head.d, head.causal):
        raise SystemExit("the measured workload must share the headline's N, d and mask")
    factor = (head.B * head.H) / (measured.B * measured.H)
    text = subprocess.run(["ncu", "-i", rep, "--page", "raw", "--csv"], capture_output=True,
                          text=True, check=True).stdout
    kernels = {}
    for name, (rd, wr) in parse_ncu_dram(text).items():
        if name not in TRAFFIC_FILES:
            continue
        kernels[name] = {
            "workload": head.name,
            "bytes_per_launch": int(round((rd + wr) * factor)),
            "measured": {"workload": measured.name, "dram_read_bytes": int(round(rd)),
                         "dram_write_bytes": int(round(wr))},
            "source_sha": source_sha(TRAFFIC_FILES[name]),
            "files": TRAFFIC_FILES[name],
        }
    note = (f"dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture of "
            f"{measured.name} (B={measured.B} H={measured.H}), scaled to {head.name} by the heads "
            f"processed (x{factor:g}): each kernel reads its inputs from DRAM once and writes its "
            f"outputs once, so traffic grows with B*H at fixed N. Written by "
            f"`python bench.py --workload {measured.name} --record-traffic <report>`.")
    PROFILE_TRAFFIC.write_text(json.dumps({"note": note, "kernels": kernels}, indent=1) + "\n")
    print(json.dumps({k: v["bytes_per_launch"] for k, v in kernels.items()}))


DETAIL_CONFIGS = ["causal_bf16_b2h4_n1024_d64", "bf16_b8h16_n2048_d128",
                  "causal_bf16_b8h16_n2048_d128", "causal_bf16_b1h2_n16384_d128"]


def time_fwd_bwd(fa2, lib, w, dev, steps: int, warmup: int, fwd_splits):
    """Mean forward and backward times (ms, CUDA events on the launching
    stream) of workload w, and the split count the forward used. Inputs that
    fit in L2 get a 256 MiB buffer overwritten before every step, outside the
    events. fwd_splits: an integer, or "auto" for the library's own choice
    (the product default of forward())."""
    import torch

    from exact_attention_64_gb300.workloads import workload_inputs

    B, H, N, d = w.B, w.H, w.N, w.d
    dt_code = 1 if w.dtype == "bf16" else 0
    q, k, v, do = (t.to(dev) for t in workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa2.bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    causal = int(w.causal)
    if fwd_splits == "auto":
        fwd_splits = fa2.num_splits(B, H, N, d, w.causal,
                                    torch.cuda.get_device_properties(dev).multi_processor_count)
    fwd_splits = int(fwd_splits)
    split_bytes = lib.fa2_fwd_split_workspace_size(B, H, N, d, fwd_splits) if fwd_splits > 1 else 0
    split_ws = torch.empty(max(split_bytes, 1), dtype=torch.uint8, device=dev)

    def fwd():
        if fwd_splits > 1:
            c = lib.fa2_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, N, d, causal, w.scale, dt_code, fwd_splits,
                                  split_ws.data_ptr(), split_bytes, sp)
        else:
            c = lib.fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, causal, w.scale, dt_code, sp)
        if c:
            raise fa2.FA2Error("fa2_fwd", c)

    def bwd():
        c = lib.fa2_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                        causal, w.scale, dt_code, ws.data_ptr(), ws_bytes, sp)
        if c:
            raise fa2.FA2Error("fa2_bwd", c)

    step_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do, o, dq, dk, dv))
    flush = step_bytes <= 2 * L2_BYTES
    scratch = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev) if flush else None
    for _ in range(warmup):
        fwd()
        bwd()
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev = [(E(), E(), E()) for _ in range(steps)]
    torch.cuda.synchronize()
    for s, (a, b, c) in enumerate(ev):
        if flush:
            scratch.fill_(s & 0xFF)
        a.record(stream)
        fwd()
        b.record(stream)
        bwd()
        c.record(stream)
    torch.cuda.synchronize()
    st = fa2.device_status()
    if st != 0:
        raise SystemExit(f"device status {fa2.status_string(st)} while timing {w.name}")
    t_f = statistics.mean(a.elapsed_time(b) for a, b, _ in ev)
    t_b = statistics.mean(b.elapsed_time(c) for _, b, c in ev)
    return t_f, t_b, fwd_splits, flush


def config_line(fa2, lib, w, dev, steps, warmup, peak, fwd_splits="auto"):
    """Forward and backward TFLOP/s of workload w and their fractions of the
    burst bf16 peak (a launch of microseconds to milliseconds is a burst)."""
    t_f, t_b, S, flush = time_fwd_bwd(fa2, lib, w, dev, steps, warmup, fwd_splits)
    f_tf = w.fwd_flops() / (t_f * 1e-3) / 1e12
    b_tf = w.bwd_flops() / (t_b * 1e-3) / 1e12
    return {"B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal, "dtype": w.dtype,
            "fwd_splits": S, "fwd_ms": t_f, "bwd_ms": t_b, "fwd_tflops": f_tf,
            "bwd_tflops": b_tf, "fwd_frac_of_peak": f_tf / peak, "bwd_frac_of_peak": b_tf / peak,
            "l2_flushed": flush}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from exact_attention_64_gb300.workloads import HEADLINE, WORKLOADS

    w = WORKLOADS[args.workload or HEADLINE]
    if args.record_traffic:
        return record_traffic(args.record_traffic, w)
    if args.impl == "reference":
        return run_reference(args, w, rank, world)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    import torch.distributed as dist

    import exact_attention_64_gb300 as fa2
    from exact_attention_64_gb300 import build as _build
    from exact_attention_64_gb300.workloads import workload_inputs

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    _build.build()
    lib = fa2.load_library()

    B, H, N, d = w.B, w.H, w.N, w.d
    dt_code = 1 if w.dtype == "bf16" else 0
    q, k, v, do = (t.to(dev) for t in workload_inputs(w, seed=rank))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    det = args.bwd == "split"
    ws_bytes = fa2.bwd_workspace_size(B, H, N, d, not det)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    scale = w.scale
    causal = int(w.causal)

    if args.fwd_splits == "auto":
        fwd_splits = fa2.num_splits(B, H, N, d, bool(causal),
                                    torch.cuda.get_device_properties(dev).multi_processor_count)
    else:
        fwd_splits = int(args.fwd_splits)
    split_bytes = lib.fa2_fwd_split_workspace_size(B, H, N, d, fwd_splits) if fwd_splits > 1 else 0
    split_ws = torch.empty(max(split_bytes, 1), dtype=torch.uint8, device=dev)

    kv_outer = args.fwd_order == "kv_outer"
    if kv_outer and fwd_splits > 1:
        raise SystemExit("--fwd-order kv_outer takes no K/V split")
    fa1_bytes = lib.fa2_fwd_kv_outer_workspace_size(B, H, N, d) if kv_outer else 0
    fa1_ws = torch.empty(max(fa1_bytes, 1), dtype=torch.uint8, device=dev)

    def fwd():
        if kv_outer:
            c = lib.fa2_fwd_kv_outer(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), B, H, N, d, causal, scale, dt_code,
                                     fa1_ws.data_ptr(), fa1_bytes, sp)
        elif fwd_splits > 1:
            c = lib.fa2_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, N, d, causal, scale, dt_code, fwd_splits,
                                  split_ws.data_ptr(), split_bytes, sp)
        else:
            c = lib.fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, causal, scale, dt_code, sp)
        if c:
            raise fa2.FA2Error("fa2_fwd", c)

    def bwd(ev_handles=None):
        evp = None
        if ev_handles is not None:
            arr = (ctypes.c_void_p * 4)(*ev_handles)
            evp = ctypes.cast(arr, ctypes.c_void_p)
        fn = lib.fa2_bwd_timed if det else lib.fa2_bwd_atomic_timed
        c = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
               do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, causal,
               scale, dt_code, ws.data_ptr(), ws_bytes, evp, sp)
        if c:
            raise fa2.FA2Error("fa2_bwd", c)

    for _ in range(args.warmup):
        fwd()
        bwd()
    torch.cuda.synchronize()
    st = fa2.device_status()
    if st != 0:
        raise SystemExit(f"device status {fa2.status_string(st)} during warm-up")

    # ---- timed region: K steps, per-kernel events on the launching stream ----
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    fwd_ev = [(E(), E()) for _ in range(args.steps)]
    bwd_ev = [[E(), E(), E(), E()] for _ in range(args.steps)]
    t0, t1 = E(), E()
    # torch creates an event's CUDA handle on its first record(): record every
    # event once here so the handles passed to the library are valid.
    for ev in [t0, t1] + [x for pair in fwd_ev for x in pair] + [x for l4 in bwd_ev for x in l4]:
        ev.record(stream)
    # Inputs smaller than L2 would stay cached from one step to the next: then
    # a 256 MiB buffer is overwritten between steps, outside the per-step
    # events, and the step time is the sum of the per-step event spans.
    step_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do, o, dq, dk, dv))
    flush = step_bytes <= 2 * L2_BYTES
    scratch = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev) if flush else None
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    nvtx = torch.cuda.nvtx
    with ClockSampler(local) as clk:
        nvtx.range_push("timed region")
        t0.record(stream)
        for s in range(args.steps):
            if flush:
                scratch.fill_(s & 0xFF)
            fwd_ev[s][0].record(stream)
            nvtx.range_push("forward")
            fwd()
            nvtx.range_pop()
            fwd_ev[s][1].record(stream)
            nvtx.range_push("backward")
            bwd([e.cuda_event for e in bwd_ev[s]])
            nvtx.range_pop()
        t1.record(stream)
        torch.cuda.synchronize()
        nvtx.range_pop()
    if world > 1:
        dist.barrier()
    if flush:
        elapsed_ms = sum(f[0].elapsed_time(b[3]) for f, b in zip(fwd_ev, bwd_ev))
    else:
        elapsed_ms = t0.elapsed_time(t1)
    st = fa2.device_status()
    if st != 0:
        raise SystemExit(f"device status {fa2.status_string(st)} in the timed region")
    t_fwd = [a.elapsed_time(b) for a, b in fwd_ev]
    t_pre = [e[0].elapsed_time(e[1]) for e in bwd_ev]
    t_kv = [e[1].elapsed_time(e[2]) for e in bwd_ev]
    t_conv = [e[2].elapsed_time(e[3]) for e in bwd_ev]
    elapsed_ms = slowest_rank_ms(elapsed_ms, dist if world > 1 else None, dev)

    flops_step = w.fwd_flops() + w.bwd_flops()
    value = job_tflops(flops_step, world, args.steps, elapsed_ms)
    pk = peaks()
    mean = statistics.mean
    # Algorithmic work per launch. The convention counts the forward as two
    # N x N x d GEMM units (S, PV) and the backward as five (2.5x). The
    # backward's main launch runs the dK/dV workers (S^T, dP^T, dV, dK: four
    # units) and the dQ workers (dQ, plus the recomputed S and dP that the
    # convention does not count): five units credited. fa2_bwd_atomic's main
    # launch (the column workers) executes exactly the five. The
    # preprocessing pass reads O and dO and writes D and L*log2e (and, for
    # fa2_bwd_atomic, zeroes the fp32 dQ accumulator); that variant's
    # conversion reads the accumulator and writes dQ.
    fw = w.fwd_flops()
    n_pad = -(-N // 128) * 128
    pre_bytes = B * H * N * (2 * d * 2 + 4 + 8) + (0 if det else B * H * n_pad * d * 4)
    kernels = {
        ("fa1_order_fwd_kernel" if kv_outer else
         "fa2_fwd_kernel" if fwd_splits > 1 else "fa2_fwd_persist_kernel"): (mean(t_fwd), fw, "tensor"),
        ("fa2_bwd_main_kernel" if det else "fa2_bwd_fused_kernel"): (mean(t_kv), 2.5 * fw, "tensor"),
        "fa2_bwd_pre_kernel": (mean(t_pre), pre_bytes, "hbm"),
    }
    if not det:
        kernels["fa2_bwd_dq_convert_kernel"] = (mean(t_conv), B * H * N * d * (4 + 2), "hbm")
    dom = max(kernels, key=lambda n: kernels[n][0])
    ms, work, bound = kernels[dom]
    traffic = None
    if PROFILE_TRAFFIC.exists():
        tr = json.loads(PROFILE_TRAFFIC.read_text())
        ent = tr.get("kernels", {}).get(dom)
        if (ent and ent.get("workload") == w.name
                and ent.get("source_sha") == source_sha(ent.get("files", []))):
            traffic = ent.get("bytes_per_launch")
    if bound == "tensor":
        # The timed region is a fraction of a second of back-to-back launches
        # of milliseconds each, not a seconds-long loop: the burst peak applies.
        achieved = work / (ms * 1e-3) / 1e12
        peak = pk["bf16"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                "peak_kind": f"bf16 burst ({pk['source']})"}
    else:
        achieved = work / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": traffic, "kernel": dom,
                "peak_kind": f"hbm copy ({pk['source']})"}
    tot = sum(x[0] for x in kernels.values())
    per_kernel = {n: {"ms": t, "share": t / tot} for n, (t, _, _) in kernels.items()}
    fwd_tf = fw / (mean(t_fwd) * 1e-3) / 1e12
    bwd_tf = w.bwd_flops() / ((mean(t_pre) + mean(t_kv) + mean(t_conv)) * 1e-3) / 1e12

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (t.cpu().pin_memory() for t in (q, k, v, do))
        ho, hdq, hdk, hdv = (torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(4))
        hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

        hpc = args.e2e_heads_per_chunk
        e2e_ws_bytes = lib.fa2_step_host_workspace_size(B, H, N, d, hpc)
        e2e_ws = torch.empty(e2e_ws_bytes, dtype=torch.uint8, device=dev)

        def e2e_step():
            # One call of the public host-buffer entry point: uploads, kernels
            # and downloads of the step, pipelined by head chunks.
            c = lib.fa2_step_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), hdo.data_ptr(),
                                  ho.data_ptr(), hlse.data_ptr(), hdq.data_ptr(), hdk.data_ptr(),
                                  hdv.data_ptr(), B, H, N, d, causal, scale, dt_code, hpc,
                                  e2e_ws.data_ptr(), e2e_ws_bytes, sp)
            if c:
                raise fa2.FA2Error("fa2_step_host", c)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        a, b = E(), E()
        nvtx.range_push("end to end (host buffers)")
        a.record(stream)
        for _ in range(args.steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        nvtx.range_pop()
        st = fa2.device_status()
        if st != 0:
            raise SystemExit(f"device status {fa2.status_string(st)} in the end-to-end leg")
        e_ms = slowest_rank_ms(a.elapsed_time(b), dist if world > 1 else None, dev)
        e2e = {"value": job_tflops(flops_step, world, args.steps, e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / args.steps, "api": "fa2_step_host",
               "heads_per_chunk": hpc or -(-(B * H) // 8)}

    # ---- every other configuration of the metric, causal and not ----
    configs = {}
    if not args.no_configs and args.workload is None:
        for name in DETAIL_CONFIGS:
            cw = WORKLOADS[name]
            configs[name] = config_line(fa2, lib, cw, dev, 10, 3, pk["bf16"])
            if cw.causal and configs[name]["fwd_splits"] != 1:
                unsplit = config_line(fa2, lib, cw, dev, 10, 3, pk["bf16"], fwd_splits=1)
                configs[name]["fwd_unsplit"] = {k: unsplit[k] for k in
                                                ("fwd_ms", "fwd_tflops", "fwd_frac_of_peak")}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_sample_heads)
        cpu.pop("seconds", None)
        if configs:
            # The oracle on one head of every other configuration, forward and
            # backward timed separately.
            cpu["configs"] = {}
            for name in configs:
                c1 = cpu_baseline(WORKLOADS[name], 1)
                cpu["configs"][name] = {k: c1[k] for k in ("fwd_tflops", "bwd_tflops", "sample")}

    l2_note = (f"L2 flushed between steps (256 MiB written; {step_bytes / 2**20:.0f} MiB touched "
               f"per step fits in L2); step time = sum of per-step event spans" if flush else
               f"inputs larger than L2 ({step_bytes / 2**20:.0f} MiB touched per step "
               f"> {L2_BYTES / 2**20:.0f} MiB)")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "q_std": w.q_std, "parallelism": f"head-sharded replicas x{world}",
                   "l2": l2_note, "fwd_splits": fwd_splits, "fwd_order": args.fwd_order,
                   "bwd": args.bwd},
        "detail": {"fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
                   "fwd_frac_of_peak": fwd_tf / pk["bf16"],
                   "bwd_frac_of_peak": bwd_tf / pk["bf16"],
                   "peak_tflops": pk["bf16"], "peak_kind": f"bf16 burst ({pk['source']})",
                   "per_kernel": per_kernel, "configs": configs},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per step: the forward (a split forward adds a counter memset, not a
        # kernel), the backward's preprocessing, its main launch and, for
        # fa2_bwd_atomic, the dQ conversion
        "gpu_launches": (3 if det else 4) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
