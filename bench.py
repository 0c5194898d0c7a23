"""Benchmark: fused residual Add + RMSNorm and RMSNorm backward on GB300, as achieved HBM GB/s.

One step is one pass of the whole hot path over one batch of synthetic input:
    add_rmsnorm_fwd  (x, residual -> residual_out, y, rstd)              16384 x 4096 bf16
    rmsnorm_bwd      (dy, x, w, rstd -> dx, dw; stage 1 + stage 2)       16384 x 4096 bf16
Throughput is counted in minimum HBM bytes (every input read once, every output written once):
536,944,640 B for the forward and 402,743,296 B for the backward, 939,687,936 B per step.

Output: one JSON line on rank 0 (see the keys below). ``--impl reference`` times the CPU fp64
oracle on a bounded sample of the same workload instead (the reference arm).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the step on its own GPU (rows are
independent; no data-path collective), and the timed region is bracketed by barriers.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "fused Add+RMSNorm bf16 achieved HBM GB/s and % of GB300 peak, by M×N"
FWD_WL = "add_rmsnorm_fwd_16384x4096_bf16"
BWD_WL = "rmsnorm_bwd_16384x4096_bf16"
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "residual_rmsnorm_row_gb300", "csrc")
# The sources the timed forward kernel (fwd_row_cta, fused, bf16) is built from; the ncu DRAM
# traffic below holds only while their hash matches (else `traffic` is reported as null).
FWD_SOURCES = ("common.cuh", "launch.h", "fwd_kernels.cuh", "fwd_bf16.cu", "tma.cuh")
# dram__bytes_read.sum + dram__bytes_write.sum of one fwd_row_cta<bf16, 4, fused> launch on the
# 16384 x 4096 workload (ncu metric capture, summarised under profiles/: 268,479,488 read +
# 213,795,840 written) and the source hash it was taken at.
NCU_FWD_TRAFFIC = {"bytes": 482275328, "sources_sha": "694046472883c4ea"}


# ------------------------------------------------------------------ helpers
def kernel_source_hash(files=FWD_SOURCES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic():
    """ncu DRAM bytes per launch of the timed forward kernel, if its sources are unchanged."""
    if NCU_FWD_TRAFFIC["bytes"] and NCU_FWD_TRAFFIC["sources_sha"] == kernel_source_hash():
        return NCU_FWD_TRAFFIC["bytes"]
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while the benchmark runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        self.file.close()
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summarise(rows, t0, t1):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[1] for r in use])), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole run"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def as_dev(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def step_bytes():
    fwd = synth.min_bytes(synth.get(FWD_WL))
    bwd = synth.min_bytes(synth.get(BWD_WL))
    return fwd, bwd


def base_config(world):
    f, b = synth.get(FWD_WL), synth.get(BWD_WL)
    return {
        "workload": f"fused Add+RMSNorm forward {f.M}x{f.N} bf16 (eps {f.eps}) + RMSNorm backward "
                    f"{b.M}x{b.N} bf16 per step",
        "M": f.M, "N": f.N,
        "step": "add_rmsnorm_fwd then rmsnorm_bwd (two-stage dw)",
        "bytes_per_step": sum(step_bytes()),
        "l2": "inputs larger than L2: two rotating buffer sets, 1.8 GB per set pair",
        "parallelism": "replicas" if world == 1 else f"dp{world} replicas (rows sharded, no collective)",
        "inputs": "seeded synthetic: x, residual, dy ~ N(0,1); w ~ 1+0.1 N(0,1)",
    }


# ------------------------------------------------------------------ our arm
def run_ours(args, world, rank, local):
    import residual_rmsnorm_row_gb300 as rrn

    rrn.load_library()
    dev = torch.device("cuda", local)
    fw, bw = synth.get(FWD_WL), synth.get(BWD_WL)
    hf = synth.make(fw)
    hb = synth.make(bw)
    w = as_dev(hf["w"], dev)
    wb = as_dev(hb["w"], dev)
    sets = []
    for s in range(2):
        x = as_dev(hf["x"], dev)
        res = as_dev(hf["residual"], dev)
        xb = as_dev(hb["x"], dev)
        dy = as_dev(hb["dy"], dev)
        if s == 1:   # a second, different buffer set (rows rolled) so no step re-reads L2 lines
            x, res, xb, dy = (t.roll(1, 0).contiguous() for t in (x, res, xb, dy))
        _, rstd_b = rrn.rms_norm(xb, wb, bw.eps)
        sets.append(dict(x=x, res=res, ro=torch.empty_like(x), y=torch.empty_like(x),
                         rstd=torch.empty(fw.M, device=dev), xb=xb, dy=dy, rstd_b=rstd_b,
                         dx=torch.empty_like(xb), dw=torch.empty(bw.N, device=dev)))
    ws = torch.empty(max(rrn.rmsnorm_bwd_workspace_bytes(bw.M, bw.N, torch.bfloat16), 16) // 4,
                     device=dev)
    stream = torch.cuda.current_stream(dev)
    fwd_plan = rrn.plan_fwd(sets[0]["x"], sets[0]["res"], sets[0]["ro"], w, sets[0]["y"])
    bwd_plan = rrn.plan_bwd(sets[0]["dy"], sets[0]["xb"], wb, sets[0]["dx"])

    do_fwd = args.only in ("step", "fwd")
    do_bwd = args.only in ("step", "bwd")

    def step(i, ev=None):
        s = sets[i & 1]
        if ev is not None:
            ev[0].record(stream)
        if do_fwd:
            rrn.add_rmsnorm_fwd(s["x"], s["res"], s["ro"], w, s["y"], s["rstd"], fw.eps, stream)
        if ev is not None:
            ev[1].record(stream)
        if do_bwd:
            rrn.rmsnorm_bwd(s["dy"], s["xb"], wb, s["rstd_b"], s["dx"], s["dw"], ws, bw.eps, stream)
        if ev is not None:
            ev[2].record(stream)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(args.warmup + i, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    elapsed_ms = max_over_ranks(world, start.elapsed_time(end))
    fwd_ms = [e[0].elapsed_time(e[1]) for e in evs]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    clocks = ClockSampler.summarise(sampler.stop(), t0, t1) if sampler else None

    # End to end through the public API, every step: pinned host inputs (x, residual, dy) ->
    # device, fused forward + fused-input backward (dy at y, x = the step's residual_out), results
    # (y, residual_out, dx, dw) -> pinned host. Steps are pipelined the way a streaming caller
    # would run them: uploads on one stream, compute on another, downloads on a third, two
    # buffer sets, so step i+1's upload and step i-1's download overlap step i's compute.
    e2e_steps = 0 if args.no_e2e else max(2, min(args.steps, 40))
    e2e_ms = 0.0
    h2d = d2h = 0
    if e2e_steps:
        nb = 2
        pin = lambda t: t.cpu().pin_memory()  # noqa: E731
        hin = [dict(x=pin(sets[b]["x"]), res=pin(sets[b]["res"]), dy=pin(sets[b]["dy"])) for b in range(nb)]
        hout = [dict(y=torch.empty_like(hin[0]["x"]).pin_memory(), ro=torch.empty_like(hin[0]["x"]).pin_memory(),
                     dx=torch.empty_like(hin[0]["x"]).pin_memory(), dw=torch.empty(bw.N).pin_memory())
                for _ in range(nb)]
        dbuf = [dict(x=torch.empty_like(sets[0]["x"]), res=torch.empty_like(sets[0]["x"]),
                     dy=torch.empty_like(sets[0]["x"]), ro=torch.empty_like(sets[0]["x"]),
                     y=torch.empty_like(sets[0]["x"]), dx=torch.empty_like(sets[0]["x"]),
                     rstd=torch.empty(fw.M, device=dev), dw=torch.empty(bw.N, device=dev))
                for _ in range(nb)]
        up, comp, down = (torch.cuda.Stream(dev) for _ in range(3))
        uploaded = [torch.cuda.Event() for _ in range(nb)]
        computed = [torch.cuda.Event() for _ in range(nb)]
        downloaded = [torch.cuda.Event() for _ in range(nb)]
        for e in downloaded:
            e.record(down)
        for e in computed:
            e.record(comp)

        def e2e_step(i):
            b = i % nb
            hi, ho, d = hin[b], hout[b], dbuf[b]
            with torch.cuda.stream(up):
                up.wait_event(computed[b])        # the previous user of buffer b has computed
                for k in ("x", "res", "dy"):
                    d[k].copy_(hi[k], non_blocking=True)
                uploaded[b].record(up)
            comp.wait_event(uploaded[b])
            comp.wait_event(downloaded[b])        # its outputs have been downloaded
            rrn.add_rmsnorm_fwd(d["x"], d["res"], d["ro"], w, d["y"], d["rstd"], fw.eps, comp)
            rrn.rmsnorm_bwd(d["dy"], d["ro"], w, d["rstd"], d["dx"], d["dw"], ws, bw.eps, comp)
            computed[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                for k in ("y", "ro", "dx", "dw"):
                    ho[k].copy_(d[k], non_blocking=True)
                downloaded[b].record(down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(world)
        t_e0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(world, (time.perf_counter() - t_e0) * 1e3)
        barrier(world)
        h2d = sum(t.numel() * t.element_size() for t in hin[0].values())
        d2h = sum(t.numel() * t.element_size() for t in hout[0].values())

    fb, bb = step_bytes()
    per_step = (fb if do_fwd else 0) + (bb if do_bwd else 0)
    ms_per_step = elapsed_ms / args.steps
    value = per_step * args.steps * world / (elapsed_ms * 1e-3) / 1e9
    fwd_us = float(np.mean(fwd_ms)) * 1e3 if do_fwd else float("nan")
    bwd_us = float(np.mean(bwd_ms)) * 1e3 if do_bwd else float("nan")
    peak, peak_kind = hbm_peak()
    fwd_gbs = fb / (fwd_us * 1e-6) / 1e9
    bwd_gbs = bb / (bwd_us * 1e-6) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": base_config(world),
        "kernels": {
            "add_rmsnorm_fwd": {"us": round(fwd_us, 2), "gbps": round(fwd_gbs, 1),
                                "frac_of_peak": round(fwd_gbs / peak, 4),
                                "rows_per_s": round(fw.M / (fwd_us * 1e-6), 1),
                                "launch": fwd_plan.name, "launches_per_step": 1},
            "rmsnorm_bwd": {"us": round(bwd_us, 2), "gbps": round(bwd_gbs, 1),
                            "frac_of_peak": round(bwd_gbs / peak, 4),
                            "rows_per_s": round(bw.M / (bwd_us * 1e-6), 1),
                            "launch": bwd_plan.name, "launches_per_step": 2},
        },
        "roofline": {"bound": "hbm", "kernel": "add_rmsnorm_fwd (fwd_row_cta)",
                     "achieved": round(fwd_gbs, 1), "peak": peak, "peak_kind": f"{peak_kind} hbm_gbs",
                     "unit": "GB/s", "frac": round(fwd_gbs / peak, 4),
                     "traffic": recorded_traffic(),
                     "algorithmic_bytes": fb},
        "e2e": ({"value": round((fb + bb) * e2e_steps * world / (e2e_ms * 1e-3) / 1e9, 1),
                 "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                 "steps": e2e_steps, "ms_per_step": round(e2e_ms / e2e_steps, 4),
                 "timing": "host wall clock around the pipelined steps, synchronised on both sides",
                 "pipeline": "upload / compute / download streams, two buffer sets"}
                if e2e_steps else None),
        "gpu_launches": (int(do_fwd) + 2 * int(do_bwd)) * args.steps,
        "clocks": clocks,
    }
    return out


# ------------------------------------------------------------------ per-shape table
BY_SHAPE = [
    "rmsnorm_fwd_256x1024_bf16", "add_rmsnorm_fwd_4096x4096_bf16",
    "add_rmsnorm_fwd_16384x4096_bf16", "add_rmsnorm_fwd_16384x7168_bf16",
    "rmsnorm_fwd_1x8192_bf16", "rmsnorm_fwd_8x8192_bf16", "rmsnorm_fwd_32x8192_bf16",
    "rmsnorm_fwd_64x8192_bf16", "rmsnorm_fwd_1x8192_f32", "rmsnorm_fwd_8x8192_f32",
    "rmsnorm_fwd_32x8192_f32", "rmsnorm_fwd_64x8192_f32", "rmsnorm_fwd_65536x2048_bf16",
    "rmsnorm_fwd_65536x2048_f32", "rmsnorm_bwd_16384x4096_bf16", "add_rmsnorm_bwd_16384x4096_bf16",
    "add_layernorm_fwd_16384x4096_bf16", "layernorm_bwd_16384x4096_bf16",
    "layernorm_bwd_plain_16384x4096_bf16",
    "add_rmsnorm_fp8_16384x4096_bf16", "add_rmsnorm_fwd_16384x16384_bf16",
    "add_rmsnorm_fwd_4096x65536_bf16", "rmsnorm_bwd_8192x16384_bf16", "add_rmsnorm_bwd_8192x16384_bf16",
    "layernorm_bwd_8192x16384_bf16", "add_rmsnorm_fp8_16384x16384_bf16",
    "add_layernorm_fwd_65536x1024_bf16", "add_layernorm_fwd_8192x8192_bf16",
    "add_rmsnorm_fp8_65536x1024_bf16", "rmsnorm_bwd_131072x512_bf16",
    "layernorm_bwd_plain_65536x1024_bf16",
]
L2_BYTES = 129 * 2 ** 20
SMALL_BYTES = 8 * 2 ** 20     # below this a launch takes a few microseconds: time it in a graph
GRAPH_LAUNCHES = 32


def dev_tensor(a: np.ndarray, device) -> torch.Tensor:
    if a.dtype == np.float32:
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return as_dev(a, device)


def measure_shape(name: str, dev, reps: int):
    """Per-launch time of one workload through the C ABI (automatic launch): launches back to
    back between two events (`us`), and the median of single launches each between its own pair
    of events (`us_single`: adds the launch latency the stream hides). Inputs are rotated across
    enough buffer sets to exceed 3x L2, or L2 is flushed (a 512 MB write outside the timed launch,
    single launches only) when one set is too small for that. Below 8 MiB: a CUDA graph of
    back-to-back launches with the inputs L2-resident."""
    import residual_rmsnorm_row_gb300 as rrn

    wl = synth.get(name)
    h = synth.make(wl)
    nbytes = synth.min_bytes(wl)
    nsets = int(min(8, max(1, -(-3 * L2_BYTES // max(nbytes, 1)))))
    flush = nbytes * nsets < 3 * L2_BYTES and nbytes >= SMALL_BYTES
    scrub = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev) if flush else None
    w = dev_tensor(h["w"], dev)
    b = dev_tensor(h["b"], dev) if "b" in h else None
    M, N = wl.M, wl.N
    sets = []
    for k in range(nsets):
        t = {key: dev_tensor(h[key], dev).roll(k, 0).contiguous()
             for key in ("x", "residual", "dy", "d_ro") if key in h}
        sets.append(t)
    bwd = wl.op in ("rmsnorm_bwd", "add_rmsnorm_bwd", "layernorm_bwd")
    ws = torch.empty(max(rrn.rmsnorm_bwd_workspace_bytes(M, N, w.dtype),
                         rrn.layernorm_bwd_workspace_bytes(M, N, w.dtype), 16) // 4 if bwd else 4,
                     device=dev)
    f32 = lambda n: torch.empty(n, device=dev)  # noqa: E731
    outs = [dict(y=torch.empty_like(s["x"]), ro=torch.empty_like(s["x"]), rstd=f32(M), mean=f32(M),
                 dw=f32(N), db=f32(N)) for s in sets]
    if wl.op == "add_rmsnorm_fp8":
        for o in outs:
            o["q"] = torch.empty(M, N, dtype=torch.uint8, device=dev)
            o["scale"] = f32(M)
    if wl.op in ("rmsnorm_bwd", "add_rmsnorm_bwd", "layernorm_bwd"):
        for s in sets:   # the forward statistics the backward consumes
            if wl.op == "layernorm_bwd":
                _, s["mean"], s["rstd"] = rrn.layer_norm(s["x"], w, None, wl.eps)
            else:
                _, s["rstd"] = rrn.rms_norm(s["x"], w, wl.eps)

    def run(i):
        s, o = sets[i % nsets], outs[i % nsets]
        if wl.op == "rmsnorm_fwd":
            rrn.rmsnorm_fwd(s["x"], w, o["y"], o["rstd"], wl.eps)
        elif wl.op == "add_rmsnorm_fwd":
            rrn.add_rmsnorm_fwd(s["x"], s["residual"], o["ro"], w, o["y"], o["rstd"], wl.eps)
        elif wl.op == "rmsnorm_bwd":
            rrn.rmsnorm_bwd(s["dy"], s["x"], w, s["rstd"], o["y"], o["dw"], ws, wl.eps)
        elif wl.op == "add_rmsnorm_bwd":
            rrn.add_rmsnorm_bwd(s["dy"], s["d_ro"], s["x"], w, s["rstd"], o["y"], o["dw"], ws, wl.eps)
        elif wl.op == "add_layernorm_fwd":
            rrn.layernorm_fwd(s["x"], w, b, o["y"], o["mean"], o["rstd"], wl.eps,
                              residual=s["residual"], residual_out=o["ro"])
        elif wl.op == "layernorm_bwd":
            rrn.layernorm_bwd(s["dy"], s.get("d_ro"), s["x"], w, s["mean"], s["rstd"], o["y"], o["dw"],
                              o["db"], ws, wl.eps)
        elif wl.op == "add_rmsnorm_fp8":
            rrn.rmsnorm_fwd_fp8(s["x"], s["residual"], o["ro"], w, o["q"], o["scale"], None, wl.eps)

    for i in range(3):
        run(i)
    torch.cuda.synchronize()
    if nbytes < SMALL_BYTES:
        # Launch-latency-bound shapes: time a CUDA graph of GRAPH_LAUNCHES back-to-back launches
        # (rotating over the buffer sets, which then stay in L2) so host launch overhead is out.
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(GRAPH_LAUNCHES):
                run(i)
        g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            ev[i][0].record()
            g.replay()
            ev[i][1].record()
        torch.cuda.synchronize()
        us = float(np.median([a.elapsed_time(c) for a, c in ev])) * 1e3 / GRAPH_LAUNCHES
        l2_note = "L2-resident: CUDA graph of %d back-to-back launches" % GRAPH_LAUNCHES
        us_single = None
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for i in range(reps):
            if flush:
                scrub.zero_()
            ev[i][0].record()
            run(i)
            ev[i][1].record()
        torch.cuda.synchronize()
        us_single = float(np.median([a.elapsed_time(c) for a, c in ev])) * 1e3
        us = us_single
        l2_note = "flushed" if flush else "%d rotating sets" % nsets
        if not flush:
            # The same launches back to back, as a training or serving loop issues them: one
            # event pair around `reps` launches (each kernel's launch and CTA start-up overlap the
            # previous kernel's tail). The table's figure; the isolated launch is kept beside it.
            a, c = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(reps):
                run(i)
            c.record()
            torch.cuda.synchronize()
            us = a.elapsed_time(c) * 1e3 / reps
            l2_note += ", back-to-back launches"
    peak, _ = hbm_peak()
    gbs = nbytes / (us * 1e-6) / 1e9
    if wl.op == "add_layernorm_fwd":
        plan = rrn.plan_layernorm_fwd(sets[0]["x"], w, outs[0]["y"], b, sets[0]["residual"], outs[0]["ro"]).name
    elif wl.op == "layernorm_bwd":
        plan = rrn.plan_layernorm_bwd(sets[0]["dy"], sets[0]["x"], w, outs[0]["y"], sets[0].get("d_ro")).name
    elif wl.op == "add_rmsnorm_fp8":
        plan = rrn.plan_fwd_fp8(sets[0]["x"], w, outs[0]["q"], sets[0]["residual"], outs[0]["ro"]).name
    elif wl.op in ("rmsnorm_bwd", "add_rmsnorm_bwd"):
        plan = rrn.plan_bwd(sets[0]["dy"], sets[0]["x"], w, outs[0]["y"], sets[0].get("d_ro")).name
    else:
        plan = rrn.plan_fwd(sets[0]["x"], sets[0].get("residual"), outs[0]["ro"], w, outs[0]["y"]).name
    return {"workload": name, "op": wl.op, "M": M, "N": N, "dtype": wl.dtype, "us": round(us, 2),
            "us_single": None if us_single is None else round(us_single, 2),
            "frac_single": None if us_single is None else round(nbytes / (us_single * 1e-6) / 1e9 / peak, 4),
            "gbps": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "rows_per_s": round(M / (us * 1e-6), 1), "min_bytes": nbytes,
            "l2": l2_note, "launch": plan}


# ------------------------------------------------------------------ the oracle (CPU)
def host_threads() -> int:
    """Host cores this process may run on (the threads the CPU baseline uses)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


class OracleStep:
    """One fused forward + backward of the CPU oracle (as it stands: single-threaded C per call)
    over `rows` rows, run as `threads` calls on contiguous row blocks at once (the C code runs
    without the GIL); the blocks' dw sums are added in block order."""

    def __init__(self, rows: int, threads: int):
        import concurrent.futures as cf

        fw, bw = synth.get(FWD_WL), synth.get(BWD_WL)
        self.eps_f, self.eps_b = fw.eps, bw.eps
        self.hf = synth.make(fw.with_shape(rows))
        self.hb = synth.make(bw.with_shape(rows))
        self.threads = max(1, min(threads, rows))
        cuts = np.linspace(0, rows, self.threads + 1).astype(int)
        self.blocks = [(int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:])]
        self.pool = cf.ThreadPoolExecutor(max_workers=self.threads)
        self.rows = rows

    def _block(self, ab):
        import oracle

        a, b = ab
        hf, hb = self.hf, self.hb
        oracle.add_rmsnorm_fwd(hf["x"][a:b], hf["residual"][a:b], hf["w"], self.eps_f)
        return oracle.rmsnorm_bwd(hb["dy"][a:b], hb["x"][a:b], hb["w"], self.eps_b)[1]

    def __call__(self):
        dws = list(self.pool.map(self._block, self.blocks))
        return np.sum(np.stack(dws), axis=0)

    def close(self):
        self.pool.shutdown()


def oracle_sample(target_s: float):
    """Time the fp64 CPU oracle on row samples of the same workload, on every host core, until
    about target_s seconds have passed."""
    fw = synth.get(FWD_WL)
    threads = host_threads()
    step = OracleStep(rows=min(fw.M, 128 * threads), threads=threads)
    fb, bb = step_bytes()
    step()  # warm-up (thread start, first touch)
    t0 = time.perf_counter()
    n = 0
    while True:
        step()
        n += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    step.close()
    bytes_done = n * step.rows * (fb + bb) / fw.M
    return {"value": round(bytes_done / el / 1e9, 4), "unit": "GB/s", "cores": step.threads,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} x {step.rows} of {fw.M} rows (fused fwd + bwd, N={fw.N}, bf16 in, fp64 "
                      f"arithmetic), the C oracle on {step.threads} threads over contiguous row "
                      f"blocks, {el:.1f} s wall, on a host with {os.cpu_count()} cores"}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, timed step by step on every host core."""
    if rank != 0:
        return None
    fw = synth.get(FWD_WL)
    fb, bb = step_bytes()
    threads = host_threads()
    # size each step so warmup + steps end within about two minutes
    probe = OracleStep(rows=min(fw.M, 8 * threads), threads=threads)
    probe()
    t = time.perf_counter()
    probe()
    per_row = (time.perf_counter() - t) / probe.rows
    probe.close()
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(threads, min(fw.M, budget / max(per_row, 1e-9))))
    step = OracleStep(rows=rows, threads=threads)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    step.close()
    bytes_done = args.steps * rows * (fb + bb) / fw.M
    value = bytes_done / el / 1e9
    sample = (f"{rows} of {fw.M} rows per step (fused fwd + bwd, N={fw.N}, bf16 in, fp64 "
              f"arithmetic), the C oracle on {step.threads} threads over contiguous row blocks, "
              f"on a host with {os.cpu_count()} cores")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": base_config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": step.threads,
                         "host_cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0,
                    help="seconds of CPU oracle work for cpu_baseline (0: skip)")
    ap.add_argument("--only", choices=["step", "fwd", "bwd"], default="step",
                    help="time the whole step (default) or one kernel alone (for profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--no-by-shape", action="store_true",
                    help="skip the per-shape table (every named workload timed alone)")
    ap.add_argument("--by-shape-reps", type=int, default=50)
    ap.add_argument("--shape", choices=BY_SHAPE, default=None,
                    help="time one workload of the per-shape table alone and print its entry "
                         "(3 untimed launches, then --by-shape-reps timed ones; for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.shape:
        import residual_rmsnorm_row_gb300 as rrn

        rrn.load_library()
        print(json.dumps(measure_shape(args.shape, torch.device("cuda", 0), args.by_shape_reps)),
              flush=True)
        return
    world, rank, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    out = run_ours(args, world, rank, local)
    if not args.no_by_shape and args.only == "step":
        dev = torch.device("cuda", local)
        out["by_shape"] = [measure_shape(n, dev, args.by_shape_reps) for n in BY_SHAPE]
        torch.cuda.empty_cache()
    if rank == 0:
        out["cpu_baseline"] = (oracle_sample(args.cpu_baseline_seconds)
                               if world == 1 and args.cpu_baseline_seconds > 0 else None)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
