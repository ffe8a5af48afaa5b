#!/usr/bin/env python
"""Benchmark: complex SSD tokens/s (B*T*H) on GB300.

One step = one pass of the whole hot path on the mamba2_layer workload
(batch 4, T 2048, 24 heads, N = P = 64, chunk 64): the chunked forward over
the batch (discretise, chunk decays, intra-chunk contraction, chunk states,
inter-chunk scan, output combine) followed by one decode step that continues
from the forward's final state, launched as one replayed CUDA graph.  Units
per step: Bz*T*H + Bz*H token-heads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run, one independent replica per rank
(weak scaling, no collective on the data path).  Rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "complex SSD scan tokens/s (B·T·H) at 1 GB300; % tensor-pipe / % HBM roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-long", action="store_true", help="skip the long_seq forward measurement")
    ap.add_argument("--no-cayley", action="store_true", help="skip the per-coordinate Cayley scan measurement")
    ap.add_argument("--no-born", action="store_true", help="skip the causal Born attention measurement")
    ap.add_argument("--no-backward", action="store_true", help="skip the gradient (backward) measurement")
    ap.add_argument("--no-precise", action="store_true", help="skip the split-precision forward measurement")
    ap.add_argument("--no-tf32", action="store_true", help="skip the TF32-operand forward measurement")
    ap.add_argument("--no-small", action="store_true", help="skip the dstate = headdim = 32 forward measurement")
    ap.add_argument("--no-pam", action="store_true", help="skip the PAM-workload forward measurement")
    ap.add_argument("--long-seqlen", type=int, default=0,
                    help="tokens of the long_seq forward (default: the workload's 65536; smaller for profiling)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- multi-rank helpers
def reduce_max(pg, value: float, device) -> float:
    """Max of `value` over all ranks (the slowest rank sets the step time)."""
    if pg is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: int, ms_per_step: float) -> float:
    """Units processed by all ranks per second, each rank doing its own replica."""
    return world * units_per_rank / (ms_per_step / 1e3)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- traffic record
# Sources that define each kernel with recorded DRAM traffic: the counters in
# profiles/dram_traffic.json hold only while these files are unchanged.
# Files that hold each kernel's device code (its .cu and the device headers it
# includes; cssd_internal.h only declares host launchers).
KERNEL_SOURCES = {
    "fused_chunk_kernel_h16": ("forward_tc.cu", "tcgen05.cuh", "cssd_common.cuh"),
    "fused_chunk_kernel_split": ("forward_tc.cu", "tcgen05.cuh", "cssd_common.cuh"),
    "fused_chunk_kernel_dstate128": ("forward_tc.cu", "tcgen05.cuh", "cssd_common.cuh"),
    "fused_chunk_kernel_tf32": ("forward_tc.cu", "tcgen05.cuh", "cssd_common.cuh"),
    "step_kernel": ("step.cu", "cssd_common.cuh"),
    "cayley_scan_kernel": ("cayley.cu", "cssd_common.cuh"),
    "born_kernel": ("born.cu", "tcgen05.cuh", "cssd_common.cuh"),
}


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments (string and character literals
    kept as they are), so that a comment-only edit leaves the hash alone."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_sha(kernel: str) -> str:
    """Hash of the kernel's sources without comments and with whitespace runs
    collapsed: the traffic record of a kernel counts only while its code is the
    one the counters were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "complex_valued_state_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = " ".join(strip_comments(f.read()).split())  # whitespace runs as one space
            h.update(name.encode() + code.encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, units: int):
    """DRAM bytes per launch from a committed ncu summary, if taken on this source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("source_sha") != kernel_source_sha(kernel):
        return None
    return float(rec["bytes_per_unit"]) * units


# ---------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch

    from complex_valued_state_gb300 import build as cbuild
    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    if rank == 0 or world == 1:
        cbuild.build()
    if pg:
        pg.barrier()
    cssd.load()

    w = wl.MAMBA2_LAYER
    Bz, T, H, N, P, ch = w.batch, w.seqlen, w.nheads, w.dstate, w.headdim, w.chunk
    host = wl.make_inputs(w, seed=w.seed + rank)
    tok = wl.decode_token(w.with_(kind="decode"), rank)
    keys = ("x", "dt", "A", "B", "C", "D")
    g = {k: torch.from_numpy(host[k]).to(dev) for k in keys}
    gt = {k: torch.from_numpy(tok[k]).to(dev) for k in ("x", "dt", "B", "C")}
    y = torch.empty((Bz, T, H, P), dtype=torch.complex64, device=dev)
    h = torch.empty((Bz, H, N, P), dtype=torch.complex64, device=dev)
    y1 = torch.empty((Bz, H, P), dtype=torch.complex64, device=dev)
    ws = torch.empty(cssd.workspace_bytes(Bz, T, H, N, P, ch), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    units = Bz * T * H + Bz * H
    launches = cssd.forward_launches(Bz, T, H, N, P, ch) + 1

    def step():
        cssd.chunked_forward(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk=ch, y=y, h_final=h, workspace=ws)
        cssd.step(h, gt["x"], gt["dt"], g["A"], gt["B"], gt["C"], g["D"], y=y1)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # Per-launch events around the dominant kernel (recorded by the library on
    # this stream), plus events around the whole timed region.
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in kb + ke:  # creates the events; the library re-records them later
        e.record(stream)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for i in range(args.steps):
        cssd.profile_events(kb[i], ke[i])
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    cssd.profile_events(None, None)
    if pg:
        pg.barrier()
    ms_stream = t0.elapsed_time(t1) / args.steps
    k_ms = sum(kb[i].elapsed_time(ke[i]) for i in range(args.steps)) / args.steps

    # The same step captured once into a CUDA graph (the entry points are
    # capturable; every per-device cache was filled by the calls above) and
    # replayed: the four launches of a step then run back to back without the
    # host's per-call work between them.  This is the timed step of `value`.
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        g0.record(stream)
        for i in range(args.steps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        if pg:
            pg.barrier()
    ms = g0.elapsed_time(g1) / args.steps
    ms = reduce_max(pg, ms, dev)
    ms_stream = reduce_max(pg, ms_stream, dev)
    value = whole_job_rate(world, units, ms)

    # end to end through the host-buffer entry point: the prefill's inputs live
    # in pinned host memory and stream through the device in pieces (copies
    # overlapping the compute), y comes back to pinned host memory and the
    # final state stays on the device for the decode token, whose inputs are
    # copied in and whose output is read back
    pin = {k: torch.from_numpy(host[k]).pin_memory() for k in keys}
    pint = {k: torch.from_numpy(tok[k]).pin_memory() for k in ("x", "dt", "B", "C")}
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    y1_host = torch.empty(y1.shape, dtype=y1.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in list(pin.values()) + list(pint.values()))
    d2h = y_host.numel() * y_host.element_size() + y1_host.numel() * y1_host.element_size()
    hbuf = torch.empty(cssd.host_forward_device_bytes(Bz, T, H, N, P, ch), dtype=torch.uint8, device=dev)

    def e2e_step():
        cssd.chunked_forward_host(**pin, chunk=ch, y=y_host, h_final=h, device_buffer=hbuf, device=dev)
        for k in pint:
            gt[k].copy_(pint[k], non_blocking=True)
        cssd.step(h, gt["x"], gt["dt"], g["A"], gt["B"], gt["C"], g["D"], y=y1)
        y1_host.copy_(y1, non_blocking=True)

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(3, args.steps // 2)
    e0.record(stream)
    for _ in range(e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e_ms = e0.elapsed_time(e1) / e_steps
    e_ms = reduce_max(pg, e_ms, dev)
    link = host_link(dev, h2d, d2h, e_ms)

    decode = const_input = cayley = born = backward = None
    if not args.no_decode:
        decode = bench_decode(args, dev)
        const_input = bench_const_input(args, dev)
    if not args.no_cayley:
        cayley = bench_cayley(args, dev)
    if not args.no_born:
        born = bench_born(args, dev)
    if not args.no_backward:
        backward = bench_backward(args, dev)
    precise = None if args.no_precise else bench_precise(args, dev)
    tf32 = None if args.no_tf32 else bench_tf32(args, dev)
    small = None if args.no_small else bench_small(args, dev)
    pam = None if args.no_pam else bench_pam(args, dev)
    long_seq = None
    if not args.no_long:
        long_seq = bench_long_seq(args, dev)

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    hbm, peak_kind = peaks()
    fwd_units = Bz * T * H
    alg_bytes = fwd_units * (8 * P + 16 * N + 4 + 8 * P)  # x, B, C, dt in; y out
    achieved = alg_bytes / (k_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "kernel": "fused_chunk_kernel_h16", "achieved": round(achieved, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(achieved / hbm, 4), "peak_kind": peak_kind,
            "traffic": recorded_traffic("fused_chunk_kernel_h16", fwd_units), "kernel_ms": round(k_ms, 5),
            "alg_bytes_per_launch": alg_bytes, "tensor": fused_tensor(fwd_units, N, k_ms, operand="f16")}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "step_launch": "one CUDA graph per step (forward prep, chunk kernel, decode step), replayed",
        "ms_per_step_stream_launches": round(ms_stream, 5),
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "precision": "GEMM operands IEEE half with a power-of-two scale per tile and operand, fp32 accumulation; "
                     "decays, rotations, hand-off and output in fp32",
        "config": {"workload": f"mamba2_layer prefill Bz{Bz} T{T} H{H} N{N} P{P} chunk{ch} + 1 decode token",
                   "batch": Bz, "seqlen": T, "nheads": H, "dstate": N, "headdim": P, "chunk": ch,
                   "units_per_step": units, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (%.2f GB read+written per step)" % (alg_bytes / 1e9)},
        "roofline": roof,
        "e2e": {"value": round(whole_job_rate(world, units, e_ms), 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 5),
                "path": "cssd_chunked_forward_host (pinned host tensors streamed in pieces) + cssd_step",
                "link": link},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    if decode:
        out["decode"] = decode
    if const_input:
        out["const_input"] = const_input
    if cayley:
        out["cayley_scan"] = cayley
    if born:
        out["born_attention"] = born
    if backward:
        out["backward"] = backward
    if precise:
        out["precise_forward"] = precise
    if tf32:
        out["tf32_forward"] = tf32
    if small:
        out["small_widths"] = small
    if pam:
        out["pam_forward"] = pam
    if long_seq:
        out["long_seq"] = long_seq
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(host, tok)
    print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


def host_link(dev, h2d_bytes, d2h_bytes, e2e_ms):
    """The host link alone on the step's bytes, timed in the same run as e2e:
    one pinned-to-device copy of the step's inputs and one device-to-pinned copy
    of its outputs, each alone and then both at once on two streams (what a
    step that hides all compute under the copies would take).  `frac` = that
    concurrent copy time / the e2e step time (1.0: e2e runs at the link's rate)."""
    import torch

    src = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
    dst_h = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, reps=5):
        for _ in range(2):
            fn()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(reps):
            t = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, (time.perf_counter() - t) * 1e3)
        return best

    def h2d():
        with torch.cuda.stream(s_in):
            d_in.copy_(src, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s_out):
            dst_h.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    h_ms, d_ms, b_ms = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": round(h2d_bytes / h_ms / 1e6, 1), "d2h_gbs": round(d2h_bytes / d_ms / 1e6, 1),
            "h2d_ms": round(h_ms, 4), "d2h_ms": round(d_ms, 4), "both_ms": round(b_ms, 4),
            "link_gbs": round((h2d_bytes + d2h_bytes) / b_ms / 1e6, 1), "link_frac": round(b_ms / e2e_ms, 4),
            "note": "pinned copies of the step's bytes, best of 5 host-timed reps; link_frac = both_ms / e2e ms"}


def bench_decode(args, dev):
    """Decode workload (batch 256, 32 heads, N 128, P 64): one token per call."""
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.DECODE
    fx = wl.decode_fixed(w)
    h = torch.from_numpy(fx["h"]).to(dev)
    A, D = torch.from_numpy(fx["A"]).to(dev), torch.from_numpy(fx["D"]).to(dev)
    toks = []
    for s in range(4):
        t = wl.decode_token(w, s)
        toks.append({k: torch.from_numpy(t[k]).to(dev) for k in t})
    y = torch.empty((w.batch, w.nheads, w.headdim), dtype=torch.complex64, device=dev)
    stream = torch.cuda.current_stream(dev)
    for i in range(max(3, args.warmup)):
        t = toks[i % 4]
        cssd.step(h, t["x"], t["dt"], A, t["B"], t["C"], D, y=y)
    torch.cuda.synchronize(dev)
    n = max(20, 5 * args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        t = toks[i % 4]
        cssd.step(h, t["x"], t["dt"], A, t["B"], t["C"], D, y=y)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / n
    units = w.batch * w.nheads
    N, P = w.dstate, w.headdim
    alg = units * (2 * 8 * N * P + 8 * P + 16 * N + 4 + 8 * P)  # state read+write, x, B, C, dt, y
    hbm, kind = peaks()
    gbs = alg / (us / 1e6) / 1e9
    return {"workload": f"decode Bz{w.batch} H{w.nheads} N{N} P{P}, one token per call",
            "value": round(units / (us / 1e6), 1), "unit": UNIT, "us_per_step": round(us, 3), "steps": n,
            "roofline": {"bound": "hbm", "kernel": "step_kernel", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "peak_kind": kind,
                         "traffic": recorded_traffic("step_kernel", units), "alg_bytes_per_launch": alg}}


def bench_const_input(args, dev):
    """Constant-input shortcuts on the decode shapes: cssd_step_n with the
    4096-step run of the decode workload (one call), and cssd_step_infinite."""
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.DECODE
    nsteps = 4096
    fx = wl.decode_fixed(w)
    h = torch.from_numpy(fx["h"]).to(dev)
    A, D = torch.from_numpy(fx["A"]).to(dev), torch.from_numpy(fx["D"]).to(dev)
    t = {k: torch.from_numpy(v).to(dev) for k, v in wl.decode_token(w, 0).items()}
    y = torch.empty((w.batch, w.nheads, w.headdim), dtype=torch.complex64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn, n):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / n

    n = max(20, 5 * args.steps)
    us_n = timed(lambda: cssd.step_n(h, t["x"], t["dt"], A, t["B"], t["C"], D, nsteps, y=y), n)
    us_inf = timed(lambda: cssd.step_infinite(t["x"], t["dt"], A, t["B"], t["C"], D, y=y), n)
    # the same call replayed from a CUDA graph of `reps` launches: the kernel's own
    # time, without the per-call host checks (the inputs stay resident in L2)
    reps = 50
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        cssd.step_infinite(t["x"], t["dt"], A, t["B"], t["C"], D, y=y)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            cssd.step_infinite(t["x"], t["dt"], A, t["B"], t["C"], D, y=y)
    graph.replay()
    torch.cuda.synchronize(dev)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(5):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    us_inf_kernel = g0.elapsed_time(g1) * 1e3 / (5 * reps)
    units = w.batch * w.nheads
    N, P = w.dstate, w.headdim
    alg_n = units * (2 * 8 * N * P + 8 * P + 16 * N + 4 + 8 * P)  # state read+write, x, B, C, dt, y
    alg_inf = units * (8 * P + 16 * N + 4 + 8 * P)  # x, B, C, dt, y: no state
    hbm, kind = peaks()
    gbs_n, gbs_inf = alg_n / (us_n / 1e6) / 1e9, alg_inf / (us_inf / 1e6) / 1e9
    return {"workload": f"decode Bz{w.batch} H{w.nheads} N{N} P{P}, one token held for {nsteps} steps",
            "metric": "token-heads/s folded into the state (nsteps x heads per call)",
            "value": round(units * nsteps / (us_n / 1e6), 1), "us_per_call": round(us_n, 3), "calls": n,
            "roofline": {"bound": "hbm", "kernel": "step_kernel (closed form)", "achieved": round(gbs_n, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs_n / hbm, 4), "peak_kind": kind,
                         "alg_bytes_per_launch": alg_n},
            "infinite": {"us_per_call": round(us_inf, 3), "kernel": "step_infinite_kernel",
                         "us_per_launch_in_graph": round(us_inf_kernel, 3),
                         "achieved": round(alg_inf / (us_inf_kernel / 1e6) / 1e9, 1), "unit": "GB/s",
                         "alg_bytes_per_launch": alg_inf,
                         "note": "us_per_call: back-to-back calls, each with the binding's and the library's "
                                 "host argument and pointer checks, so the host sets the rate; "
                                 "us_per_launch_in_graph: %d calls captured in one CUDA graph and replayed; the "
                                 "inputs (%.1f MB) stay in L2, so achieved is an L2 rate, not an HBM fraction"
                                 % (reps, alg_inf / 1e6)}}


def bench_cayley(args, dev):
    """Per-coordinate Cayley-phase scan at the H-Mamba shapes (batch 256, T 1024,
    16 heads of 16 coordinates, chunk 64): the paper's clamped chunked scan
    (log clamp -30) and the exact recurrence."""
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.HMAMBA_SCAN
    host = wl.make_cayley_inputs(w)
    g = {k: torch.from_numpy(v).to(dev) for k, v in host.items()}
    del host
    Bz, T, H, N = w.batch, w.seqlen, w.nheads, w.dstate
    y = torch.empty((Bz, T, H, N), dtype=torch.complex64, device=dev)
    pf = torch.empty((Bz, H, N), dtype=torch.complex64, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {"workload": f"hmamba_scan Bz{Bz} T{T} H{H} N{N} chunk{w.chunk}",
           "metric": "tokens/s through one layer's scan (all heads)"}
    alg = Bz * T * H * N * (4 + 4 + 8 + 8 + 8) + Bz * H * N * 16  # phi, u, b, C in; y out; psi0 in, psi_final out
    hbm, kind = peaks()
    for name, lo in (("clamped", -30.0), ("exact", float("-inf"))):
        def call():
            cssd.cayley_scan(g["phi"], g["u"], g["b"], g["C"], psi0=g["psi0"], chunk=w.chunk, log_clamp=lo, y=y,
                             psi_final=pf)
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize(dev)
        n = max(10, args.steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        us = e0.elapsed_time(e1) * 1e3 / n
        gbs = alg / (us / 1e6) / 1e9
        out[name] = {"log_clamp": lo if lo > float("-inf") else "-inf", "us_per_call": round(us, 2), "calls": n,
                     "value": round(Bz * T / (us / 1e6), 1), "unit": "tokens/s",
                     "roofline": {"bound": "hbm", "kernel": "cayley_scan_kernel", "achieved": round(gbs, 1),
                                  "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_kind": kind,
                                  "alg_bytes_per_launch": alg,
                                  "traffic": recorded_traffic("cayley_scan_kernel", Bz * T * H * N)}}
    out["context"] = "the paper's ~48,000 tokens/s is a whole 253M-parameter model training on an A100, not this scan"
    return out


def tf32_peak():
    """Dense TF32 tensor peak: the measured bf16 burst figure times the nominal
    TF32 / bf16 ratio (1.1 / 2.25 PFLOP/s), else the fallback bf16 figure times it."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    ratio = 1.1 / 2.25
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]) * ratio, "measured bf16 burst x nominal tf32/bf16 (1.1/2.25)"
    return 1900.0 * ratio, "fallback bf16 x nominal tf32/bf16 (1.1/2.25)"


def bench_born(args, dev):
    """Causal Born attention at the H-Transformer shapes (batch 256, T 1024,
    16 heads of width 16).  Tensor-bound: the roofline counts the algorithmic
    flops of the causal pairs (<q|k>, its squared modulus, s v and the score
    sum); the MMA flops the kernel executes (128-query blocks against 32-key
    blocks up to the diagonal: Re G and Im G together 128x64x(2D), the value
    GEMM 128x(2D+16)x32 with its row of ones) are reported beside them."""
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.HTRANSFORMER_ATTN
    host = wl.make_born_inputs(w)
    g = {k: torch.from_numpy(host[k]).to(dev) for k in ("q", "k", "v")}
    del host
    Bz, T, H, D = w.batch, w.seqlen, w.nheads, w.dstate
    psi = torch.empty_like(g["q"])
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        cssd.born_attention(g["q"], g["k"], g["v"], psi=psi)
    torch.cuda.synchronize(dev)
    n = max(10, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        cssd.born_attention(g["q"], g["k"], g["v"], psi=psi)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n
    nqb, nkb = (T + 127) // 128, (T + 31) // 32
    blocks = Bz * H * sum(min(4 * (qb + 1), nkb) for qb in range(nqb))  # (128 queries, 32 keys) pairs visited
    executed = blocks * (2 * 128 * 64 * (2 * D) + 2 * 128 * (2 * D + 16) * 32)
    pairs = Bz * H * T * (T + 1) // 2
    minimal = pairs * (8 * D + 3 + 4 * D + 1)  # <q|k>, |.|^2, s v and the score sum
    peak, kind = tf32_peak()
    tf = minimal / (ms / 1e3) / 1e12
    return {"workload": f"htransformer_attn Bz{Bz} T{T} H{H} D{D}", "ms_per_call": round(ms, 4), "calls": n,
            "value": round(Bz * T * H / (ms / 1e3), 1), "unit": "token-heads/s",
            "roofline": {"bound": "tensor", "kernel": "born_kernel_ws<16>", "achieved": round(tf, 1),
                         "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(tf / peak, 4), "peak_kind": kind,
                         "flops_per_launch": minimal, "flops": "algorithmic: the causal pairs",
                         "executed_flops_per_launch": executed,
                         "executed_tflops": round(executed / (ms / 1e3) / 1e12, 1),
                         "executed_frac": round(executed / (ms / 1e3) / 1e12 / peak, 4)},
            "hbm_bytes_per_launch": 4 * Bz * T * H * D * 8,
            "traffic": recorded_traffic("born_kernel", Bz * T * H),
            "context": "the paper's ~80,000 tokens/s is a whole 253M-parameter H-Transformer training on A100s, not this kernel"}


def bench_backward(args, dev):
    """Gradients of the mamba2_layer forward (cssd_chunked_backward: y and the
    x-gradient run on the split-precision half-operand kernel, the B and C
    gradients on the plain half-operand kernel, each with the index and sign
    modes).  HBM roofline on the algorithmic bytes: x, dt, B, C, dy in and gx,
    gdt, gB, gC out."""
    import numpy as np
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.MAMBA2_LAYER
    host = wl.make_inputs(w)
    g = {k: torch.from_numpy(host[k]).to(dev) for k in ("x", "dt", "A", "B", "C", "D")}
    rng = np.random.default_rng(w.seed + 1000)
    shape = (w.batch, w.seqlen, w.nheads, w.headdim)
    dy = torch.from_numpy(((rng.standard_normal(shape) + 1j * rng.standard_normal(shape)) / np.sqrt(2))
                          .astype(np.complex64)).to(dev)
    ws = torch.empty(cssd.backward_workspace_bytes(w.batch, w.seqlen, w.nheads, w.dstate, w.headdim, w.chunk),
                     dtype=torch.uint8, device=dev)
    out = cssd.chunked_backward(**g, dy=dy, chunk=w.chunk, workspace=ws)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        cssd.chunked_backward(**g, dy=dy, chunk=w.chunk, workspace=ws, grads=out)
    torch.cuda.synchronize(dev)
    n = max(10, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        cssd.chunked_backward(**g, dy=dy, chunk=w.chunk, workspace=ws, grads=out)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / n
    N, P = w.dstate, w.headdim
    alg = w.units * (8 * P + 4 + 16 * N + 8 * P + 8 * P + 4 + 16 * N)
    hbm, kind = peaks()
    gbs = alg / (ms / 1e3) / 1e9
    return {"workload": f"mamba2_layer backward Bz{w.batch} T{w.seqlen} H{w.nheads} N{N} P{P} chunk{w.chunk}",
            "ms_per_call": round(ms, 4), "calls": n, "value": round(w.units / (ms / 1e3), 1), "unit": "token-heads/s",
            "roofline": {"bound": "hbm", "kernel": "whole backward (12 launches)", "achieved": round(gbs, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_kind": kind,
                         "alg_bytes_per_call": alg},
            "workspace_bytes": int(ws.numel())}


def bench_long_seq(args, dev):
    """Forward on the long_seq workload (batch 1, T 65536, 32 heads, N 128, P 64, chunk 128)."""
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.LONG_SEQ if args.long_seqlen <= 0 else wl.LONG_SEQ.with_(seqlen=args.long_seqlen)
    host = wl.make_inputs(w)
    g = {k: torch.from_numpy(host[k]).to(dev) for k in ("x", "dt", "A", "B", "C", "D")}
    del host
    Bz, T, H, N, P, ch = w.batch, w.seqlen, w.nheads, w.dstate, w.headdim, w.chunk
    y = torch.empty((Bz, T, H, P), dtype=torch.complex64, device=dev)
    h = torch.empty((Bz, H, N, P), dtype=torch.complex64, device=dev)
    ws = torch.empty(cssd.workspace_bytes(Bz, T, H, N, P, ch), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        cssd.chunked_forward(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk=ch, y=y, h_final=h, workspace=ws)

    for _ in range(3):
        fwd()
    torch.cuda.synchronize(dev)
    n = 5
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in kb + ke:
        e.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(n):
        cssd.profile_events(kb[i], ke[i])
        fwd()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    cssd.profile_events(None, None)
    ms = e0.elapsed_time(e1) / n
    k_ms = sum(kb[i].elapsed_time(ke[i]) for i in range(n)) / n
    units = Bz * T * H
    alg = units * (8 * P + 16 * N + 4 + 8 * P)
    hbm, kind = peaks()
    gbs = alg / (k_ms / 1e3) / 1e9
    return {"workload": f"long_seq Bz{Bz} T{T} H{H} N{N} P{P} chunk{ch}, forward only",
            "value": round(units / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4), "steps": n,
            "roofline": {"bound": "hbm", "kernel": "fused_chunk_kernel_h16w (dstate 128, half operands)",
                         "achieved": round(gbs, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_kind": kind, "kernel_ms": round(k_ms, 4),
                         "traffic": recorded_traffic("fused_chunk_kernel_dstate128", units),
                         "alg_bytes_per_launch": alg, "tensor": fused_tensor(units, N, k_ms, operand="f16")}}


def f16_peak():
    """Dense f16 tensor peak: the measured bf16 burst figure (f16 and bf16 run at
    the same rate), else the fallback bf16 figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16 burst (the f16 rate)"
    return 1900.0, "fallback bf16 (the f16 rate)"


def fused_tensor(units, dstate, k_ms, passes=1, operand="tf32"):
    """Tensor pipe of the fused chunk kernel on its executed MMA work: per 64-token
    tile, three complex 64x64x64 GEMMs per 64-row state half (chunk state, scores,
    carried-in readout) and one for the masked scores times X, 8 real flops per
    complex multiply-add; `passes` = 3 with split-precision operands; `operand`
    is the MMA input type (tf32, or f16 for the half-operand kernel)."""
    nh = dstate // 64
    flops = passes * units * (3 * nh + 1) * 64 * 64 * 8
    tf = flops / (k_ms / 1e3) / 1e12
    peak, kind = f16_peak() if operand == "f16" else tf32_peak()
    return {"executed_tflops": round(tf, 1), "peak": round(peak, 1), "peak_kind": kind, "frac": round(tf / peak, 4),
            "flops_per_launch": flops}


def bench_precise(args, dev):
    """Split-precision forward (cssd_chunked_forward_precise) on the mamba2_layer workload."""
    return bench_operand_variant(args, dev, "precise")


def bench_tf32(args, dev):
    """TF32-operand forward (cssd_chunked_forward_tf32, the TF32 fused kernel at
    dstate 64) on the mamba2_layer workload, beside the half-operand headline."""
    return bench_operand_variant(args, dev, "tf32")


def bench_small(args, dev):
    """dstate = headdim = 32 at the mamba2_layer's batch, length and heads: the
    half-operand chunk kernel on tiles padded to 64 (the tensor-core path of the
    widths below 64)."""
    from complex_valued_state_gb300 import workloads as wl

    w = wl.MAMBA2_LAYER.with_(dstate=32, headdim=32)
    return bench_forward_shape(
        dev, w, f"mamba2_layer batch, length and heads at Bz{w.batch} T{w.seqlen} H{w.nheads} N{w.dstate} P{w.headdim} "
        f"chunk{w.chunk}", "fused_chunk_kernel_h16 on tiles padded to 64", "fused_chunk_kernel_h16 (padded)")


def bench_pam(args, dev):
    """The PAM workload (Bz 8, T 1024, H 12, N = P = 64; queries, keys and values
    mapped onto C, B and x, decay from the retention rates): the default
    forward, the half-operand chunk kernel."""
    from complex_valued_state_gb300 import workloads as wl

    w = wl.PAM
    return bench_forward_shape(
        dev, w, f"pam Bz{w.batch} T{w.seqlen} H{w.nheads} N{w.dstate} P{w.headdim} chunk{w.chunk}",
        "fused_chunk_kernel_h16", "fused_chunk_kernel_h16")


def bench_forward_shape(dev, w, workload, kernel, roof_kernel):
    """cssd_chunked_forward on one workload's inputs: whole-call time and the
    chunk kernel's own time (the library's event hook), HBM roofline on the
    algorithmic bytes (x, B, C, dt in; y out)."""
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    host = wl.make_inputs(w)
    g = {k: torch.from_numpy(host[k]).to(dev) for k in ("x", "dt", "A", "B", "C", "D")}
    del host
    Bz, T, H, N, P, ch = w.batch, w.seqlen, w.nheads, w.dstate, w.headdim, w.chunk
    y = torch.empty((Bz, T, H, P), dtype=torch.complex64, device=dev)
    h = torch.empty((Bz, H, N, P), dtype=torch.complex64, device=dev)
    ws = torch.empty(cssd.workspace_bytes(Bz, T, H, N, P, ch), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        cssd.chunked_forward(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk=ch, y=y, h_final=h, workspace=ws)

    for _ in range(3):
        fwd()
    torch.cuda.synchronize(dev)
    n = 20
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in kb + ke:
        e.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(n):
        cssd.profile_events(kb[i], ke[i])
        fwd()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    cssd.profile_events(None, None)
    ms = e0.elapsed_time(e1) / n
    k_ms = sum(kb[i].elapsed_time(ke[i]) for i in range(n)) / n
    units = Bz * T * H
    alg = units * (8 * P + 16 * N + 4 + 8 * P)
    hbm, kind = peaks()
    gbs = alg / (k_ms / 1e3) / 1e9
    return {"workload": workload,
            "value": round(units / (ms / 1e3), 1), "unit": UNIT, "ms_per_call": round(ms, 4), "calls": n,
            "kernel": kernel,
            "roofline": {"bound": "hbm", "kernel": roof_kernel, "achieved": round(gbs, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_kind": kind,
                         "kernel_ms": round(k_ms, 4), "alg_bytes_per_launch": alg},
            "tensor": fused_tensor(units, 64, k_ms, operand="f16")}


def bench_operand_variant(args, dev, variant):
    import torch

    from complex_valued_state_gb300 import cssd
    from complex_valued_state_gb300 import workloads as wl

    w = wl.MAMBA2_LAYER
    host = wl.make_inputs(w)
    g = {k: torch.from_numpy(host[k]).to(dev) for k in ("x", "dt", "A", "B", "C", "D")}
    del host
    Bz, T, H, N, P, ch = w.batch, w.seqlen, w.nheads, w.dstate, w.headdim, w.chunk
    y = torch.empty((Bz, T, H, P), dtype=torch.complex64, device=dev)
    h = torch.empty((Bz, H, N, P), dtype=torch.complex64, device=dev)
    ws = torch.empty(cssd.workspace_bytes(Bz, T, H, N, P, ch), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        cssd.chunked_forward(g["x"], g["dt"], g["A"], g["B"], g["C"], g["D"], chunk=ch, y=y, h_final=h, workspace=ws,
                             precise=variant == "precise", tf32=variant == "tf32")

    for _ in range(3):
        fwd()
    torch.cuda.synchronize(dev)
    n = 20
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in kb + ke:
        e.record(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for i in range(n):
        cssd.profile_events(kb[i], ke[i])
        fwd()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    cssd.profile_events(None, None)
    ms = e0.elapsed_time(e1) / n
    k_ms = sum(kb[i].elapsed_time(ke[i]) for i in range(n)) / n
    units = Bz * T * H
    alg = units * (8 * P + 16 * N + 4 + 8 * P)
    hbm, kind = peaks()
    gbs = alg / (k_ms / 1e3) / 1e9
    if variant == "precise":
        tensor = fused_tensor(units, N, k_ms, passes=3, operand="f16")  # hi.hi, hi.lo, lo.hi of half parts
        label, kname, tkey = "split-precision forward", "fused_chunk_kernel_h16 (split)", "fused_chunk_kernel_split"
    else:
        tensor = fused_tensor(units, N, k_ms)
        label, kname, tkey = "TF32-operand forward", "fused_chunk_kernel (tf32)", "fused_chunk_kernel_tf32"
    return {"workload": f"mamba2_layer Bz{Bz} T{T} H{H} N{N} P{P} chunk{ch}, {label}",
            "value": round(units / (ms / 1e3), 1), "unit": UNIT, "ms_per_call": round(ms, 4), "calls": n,
            "dtype": "f32 (split half operands)" if variant == "precise" else "tf32",
            "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(gbs, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_kind": kind,
                         "traffic": recorded_traffic(tkey, units),
                         "kernel_ms": round(k_ms, 4), "alg_bytes_per_launch": alg},
            "tensor": tensor}


# ---------------------------------------------------------------- CPU oracle
def _oracle_step(o, arrays, tok_arrays):
    y, hf = o.cssd_naive(*arrays)
    o.cssd_step(hf, *tok_arrays)


def _oracle_inputs(host, tok):
    c = lambda a: np.ascontiguousarray(a, dtype=np.complex128)
    r = lambda a: np.ascontiguousarray(a, dtype=np.float64)
    arrays = (c(host["x"]), r(host["dt"]), c(host["A"]), c(host["B"]), c(host["C"]), r(host["D"]))
    tok_arrays = (c(tok["x"]), r(tok["dt"]), c(host["A"]), c(tok["B"]), c(tok["C"]), r(host["D"]))
    return arrays, tok_arrays


def cpu_baseline(host, tok, budget_s: float = 12.0):
    """The oracle as it stands on this host's cores, on the same workload."""
    import oracle

    oracle.build()
    arrays, tok_arrays = _oracle_inputs(host, tok)
    Bz, T, H, _ = host["x"].shape
    units = Bz * T * H + Bz * H
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(oracle, arrays, tok_arrays)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 100:
            break
    return {"value": round(reps * units / el, 1), "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": f"full mamba2_layer step (prefill + 1 decode token) x{reps}, {el:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle, timed as it stands on the host cores."""
    if rank != 0:
        return
    import oracle

    from complex_valued_state_gb300 import workloads as wl

    oracle.build()
    w = wl.MAMBA2_LAYER
    host = wl.make_inputs(w)
    tok = wl.decode_token(w.with_(kind="decode"), 0)
    arrays, tok_arrays = _oracle_inputs(host, tok)
    Bz, T, H = w.batch, w.seqlen, w.nheads
    # bounded sample per step: a slice of heads, sized to keep the run to minutes
    hs = max(1, H // 6)
    sub = tuple(a[:, :, :hs] if a.ndim == 4 or a.ndim == 3 else a[:hs] for a in arrays)
    sub_tok = tuple(a[:, :hs] if a.ndim >= 2 else a[:hs] for a in tok_arrays)
    sub = tuple(np.ascontiguousarray(a) for a in sub)
    sub_tok = tuple(np.ascontiguousarray(a) for a in sub_tok)
    units = Bz * T * hs + Bz * hs
    for _ in range(args.warmup):
        _oracle_step(oracle, sub, sub_tok)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(oracle, sub, sub_tok)
    el = time.perf_counter() - t0
    ms = el * 1e3 / args.steps
    value = units / (ms / 1e3)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"mamba2_layer prefill Bz{Bz} T{T} H{H} N{w.dstate} P{w.headdim} chunk{w.chunk} "
                                  f"+ 1 decode token", "parallelism": "host cores"},
           "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                            "sample": f"{hs} of {H} heads, all {Bz} batch rows and {T} tokens, per step"},
           "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
