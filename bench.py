"""Benchmark of the MoE SwiGLU layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one whole layer forward (router GEMM, top-k, dispatch, gate/up grouped GEMM, down
grouped GEMM, combine) over one batch of T synthetic tokens whose inputs are resident in HBM.
Default workload: the DeepSeek-V4-Flash-shaped layer at T=8192 (prefill), also with FP8 expert
weights ("fp8_weights") and MXFP4 expert weights ("mxfp4_weights"); the same line carries the same layer with Zipf-skewed routing under
"skewed", a T=64 (decode) measurement under "decode" and a T=1024 batch of the main workload's
shapes under "small_prefill" (24 rows per routed expert: the weight-streaming single-CTA
kernels), each with the same layer on FP8 expert weights ("fp8_weights") and on MXFP4 expert
weights ("mxfp4_weights": the one-time conversion to the FP8 form, the forward on the converted
tiles, and the native forward on the 4-bit codes).
Multi-GPU runs are independent replicas (one process per GPU, each with its own token batch; no
collective on the data path).

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle instead, on bounded
samples of the same workload, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

_NCORES = len(os.sched_getaffinity(0))
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_NCORES))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from routed_expert_swiglu_gb300 import cost, inputs, workloads  # noqa: E402

PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ["router_gemm", "topk", "dispatch", "gate_up_gemm", "down_gemm", "combine"]


def load_peaks():
    try:
        with open(PEAKS_PATH) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- distributed

def _free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_replicas(n: int) -> int:
    """`--gpus N` without a launcher's environment: start N rank processes of this same command
    (torch.distributed.run, one process per GPU, rendezvous on 127.0.0.1) and return their
    exit status.  Rank 0 prints the JSON line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        """The raw samples go to $MOE_CLOCKS_DIR/clocks_gpu<i>.csv (the system temp directory by
        default); the bench line carries their summary."""
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        out_dir = os.environ.get("MOE_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_gpu{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- our arm

def time_layer(layer, x, token_ids, steps, warmup, stream, with_stages=True, fwd=None):
    """Device time of `steps` forwards (after `warmup`), with per-stage event times.  `fwd`
    replaces layer.forward (same arguments), e.g. the FP8-weight forward."""
    nstage = len(STAGES)
    if fwd is None:
        fwd = layer.forward
    for _ in range(warmup):
        fwd(x, token_ids, out=layer._out)
    torch.cuda.synchronize()
    evsets = []
    if with_stages:
        for _ in range(steps):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(nstage + 1)]
            for e in evs:
                e.record(stream)  # materialise the CUDA events before handing them to the library
            evsets.append(evs)
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        if with_stages:
            layer.set_events(evsets[i])
        fwd(x, token_ids, out=layer._out)
    end.record(stream)
    torch.cuda.synchronize()
    layer.set_events(None)
    total_ms = start.elapsed_time(end)
    stage_ms = None
    if with_stages:
        stage_ms = [sum(evs[j].elapsed_time(evs[j + 1]) for evs in evsets) / steps for j in range(nstage)]
    return total_ms, stage_ms


def measure_workload(w, steps, warmup, device, seed, world, rank):
    from routed_expert_swiglu_gb300 import binding
    inp = inputs.make_layer_inputs(w, seed=seed, device=device)
    layer = binding.MoELayer(w, inp)
    layer._out = torch.empty((w.T, w.d), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream()
    barrier(world)
    torch.cuda.synchronize()
    total_ms, stage_ms = time_layer(layer, inp.x, inp.token_ids, steps, warmup, stream)
    torch.cuda.synchronize()
    barrier(world)
    st = layer.check_status()
    if st != 0:
        raise RuntimeError(f"device status {binding.STATUS_NAMES.get(st, st)} on {w.name}")
    counts = layer.views(w.T)["counts"].cpu().numpy()
    active = int((counts > 0).sum())
    launches = binding.moe_forward_launch_count(layer.plan, w.T)
    return layer, inp, total_ms, stage_ms, active, launches


def measure_fp8(layer, inp, w, steps, warmup, active, bf16_ms, hbm_peak, world):
    """The same layer with FP8 (E4M3) expert weights, one power-of-two scale per 128 x 128
    tile: quantised once before timing (static weights), then moe_forward_fp8 timed like the
    bf16 forward.  Bytes = the bf16 layer's with one byte per expert weight plus the tile
    exponents."""
    from routed_expert_swiglu_gb300 import binding
    q = layer.quantize_fp8()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    fwd = lambda x, tok, out: layer.forward_fp8(x, q, tok, out=out)  # noqa: E731
    ms, stage = time_layer(layer, inp.x, inp.token_ids, steps, warmup, stream, fwd=fwd)
    st = layer.check_status()
    if st != 0:
        raise RuntimeError(f"device status {binding.STATUS_NAMES.get(st, st)} on {w.name} (fp8 weights)")
    ms = max_over_ranks(ms, world) / steps
    n_mat = active + w.n_shared
    exps = n_mat * (-(-2 * w.d_ff // 128) * -(-w.d // 128) + -(-w.d // 128) * -(-w.d_ff // 128))
    nbytes = cost.layer_bytes(w, active) - n_mat * 3 * w.d * w.d_ff + exps
    return {"weights": "fp8 e4m3, one power-of-two scale per 128x128 tile", "ms_per_step": round(ms, 4),
            "tokens_per_s": round(world * w.T / (ms / 1e3), 1), "layer_bytes": int(nbytes),
            "hbm_gbs_layer": round(nbytes / (ms / 1e3) / 1e9, 1),
            "hbm_frac_layer": round(nbytes / (ms / 1e3) / 1e9 / hbm_peak, 4),
            "speedup_vs_bf16": round(bf16_ms / ms, 3),
            "stage_ms": {s: round(v, 4) for s, v in zip(STAGES, stage)}}


def measure_mxfp4(layer, inp, w, steps, warmup, fp8_ms, bf16_ms, world):
    """The same layer with MXFP4 (E2M1, 1 x 32 sub-block scales) expert weights: quantised once,
    converted losslessly to the FP8 tile form once per weight set (timed: conversion_ms), then
    the forward on the converted tiles timed like the FP8 forward."""
    from routed_expert_swiglu_gb300 import binding
    q4 = layer.quantize_mxfp4()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    layer.mxfp4_to_fp8(q4)  # warm-up
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    q8 = layer.mxfp4_to_fp8(q4)
    end.record(stream)
    torch.cuda.synchronize()
    conv_ms = start.elapsed_time(end)
    fwd = lambda x, tok, out: layer.forward_fp8(x, q8, tok, out=out)  # noqa: E731
    ms, _ = time_layer(layer, inp.x, inp.token_ids, steps, warmup, stream, fwd=fwd, with_stages=False)
    st = layer.check_status()
    if st != 0:
        raise RuntimeError(f"device status {binding.STATUS_NAMES.get(st, st)} on {w.name} (mxfp4 weights)")
    ms = max_over_ranks(ms, world) / steps
    at_rest = sum(c.numel() + e.numel() for c, e in q4.values())
    res = {"weights": "mxfp4 e2m1, one power-of-two scale per 1x32 sub-block", "bytes_at_rest": int(at_rest),
           "conversion_ms": round(max_over_ranks(conv_ms, world), 4),
           "converted": {"ms_per_step": round(ms, 4), "tokens_per_s": round(world * w.T / (ms / 1e3), 1),
                         "what": "moe_forward_fp8 on the losslessly converted fp8 tiles"}}
    if w.d % 128 == 0 and w.d_ff % 128 == 0:
        fwd = lambda x, tok, out: layer.forward_mxfp4(x, q4, tok, out=out)  # noqa: E731
        nms, nstage = time_layer(layer, inp.x, inp.token_ids, steps, warmup, stream, fwd=fwd)
        st = layer.check_status()
        if st != 0:
            raise RuntimeError(f"device status {binding.STATUS_NAMES.get(st, st)} on {w.name} (native mxfp4)")
        nms = max_over_ranks(nms, world) / steps
        res["native"] = {"ms_per_step": round(nms, 4), "tokens_per_s": round(world * w.T / (nms / 1e3), 1),
                         "speedup_vs_fp8": round(fp8_ms / nms, 3), "speedup_vs_bf16": round(bf16_ms / nms, 3),
                         "stage_ms": {s: round(v, 4) for s, v in zip(STAGES, nstage)},
                         "what": "moe_forward_mxfp4: 4-bit codes fed to the block-scaled MMA with their 1x32 scales"}
    return res


def measure_leg(wl, args, device, rank, world, peaks, hbm_peak):
    """One more workload on the same line: the bf16 layer (stage times, HBM bytes and the
    layer roofline) and, unless --no-fp8, the same layer on FP8 and on MXFP4 expert weights."""
    steps = max(args.steps, 10)
    ll, linp, lms, lstage, lactive, _ = measure_workload(wl, steps, args.warmup, device, seed=rank, world=world,
                                                         rank=rank)
    lms = max_over_ranks(lms, world) / steps
    lbytes = cost.layer_bytes(wl, lactive)
    roof = cost.roofline_seconds(cost.layer_flops(wl), lbytes, float(peaks["bf16_tflops_sustained"]), hbm_peak)
    leg = {"workload": wl.name, "T": wl.T, "rows_per_expert": round(wl.T * wl.k / wl.E, 2),
           "ms_per_step": round(lms, 4), "tokens_per_s": round(world * wl.T / (lms / 1e3), 1),
           "active_experts": lactive, "layer_bytes": int(lbytes),
           "hbm_gbs_layer": round(lbytes / (lms / 1e3) / 1e9, 1),
           "hbm_frac_layer": round(lbytes / (lms / 1e3) / 1e9 / hbm_peak, 4),
           "layer_roofline_ms": round(roof * 1e3, 4), "layer_roofline_frac": round(roof * 1e3 / lms, 4),
           "stage_ms": {s: round(v, 4) for s, v in zip(STAGES, lstage)}}
    if not args.no_fp8:
        leg["fp8_weights"] = measure_fp8(ll, linp, wl, steps, args.warmup, lactive, lms, hbm_peak, world)
        leg["mxfp4_weights"] = measure_mxfp4(ll, linp, wl, steps, args.warmup, leg["fp8_weights"]["ms_per_step"],
                                             lms, world)
    ll.close()
    del ll, linp
    torch.cuda.empty_cache()
    return leg


def measure_e2e(layer, inp, w, steps, warmup, world):
    """Same metric through moe_forward_host: pinned host x in, pinned host y out, copies timed."""
    from routed_expert_swiglu_gb300 import binding
    x_h = inp.x.cpu().pin_memory()
    tok_h = inp.token_ids.cpu().pin_memory() if inp.token_ids is not None else None
    y_h = torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.current_stream()

    def step():
        binding.moe_forward_host(layer.plan, w.T, x_h, tok_h, inp.w_r, inp.bias, inp.w13, inp.w2, inp.w13_sh,
                                 inp.w2_sh, y_h, layer.ws, stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(end), world)
    h2d = w.T * w.d * 2 + (w.T * 4 if inp.token_ids is not None else 0)
    d2h = w.T * w.d * 2
    return ms, h2d, d2h


# The sources the bf16 grouped-GEMM kernels are compiled from (the FP8 kernels live elsewhere).
GEMM_SOURCES = ("common.cuh", "gemm_common.cuh", "grouped_gemm.cu")


def gemm_source_sha():
    """sha256 prefix of the bf16 grouped-GEMM sources, concatenated in GEMM_SOURCES order."""
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "routed_expert_swiglu_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload_name):
    """DRAM bytes per gate/up launch from the committed ncu capture, or None when there is no
    capture for this workload or the kernel sources changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "gate_up_traffic.json")) as fh:
            rec = json.load(fh)
        sha = gemm_source_sha()
    except (OSError, ValueError):
        return None
    if rec.get("source_sha256_prefix") != sha:
        return None
    v = rec.get("scaled_bytes_per_launch", {}).get(workload_name)
    if v is None:
        v = rec.get("measured_bytes_per_launch", {}).get(workload_name)
    return None if v is None else int(v)


def gate_up_bytes(w, active):
    """Algorithmic HBM bytes of one gate/up grouped-GEMM launch: the w13 slabs of the active
    experts (+ shared) and the layer input x, read once.  The dispatched rows it reads and the
    activations it writes are intermediates of this implementation, reported separately
    (gate_up_intermediate_bytes)."""
    bf = 2
    return (active + w.n_shared) * 2 * w.d * w.d_ff * bf + w.T * w.d * bf


def gate_up_intermediate_bytes(w):
    """Bytes the gate/up launch moves beyond its algorithmic ones: the dispatched routed rows
    read (the shared expert reads x itself) and the (hi, lo) activation pair written."""
    bf = 2
    return w.N * w.d * bf + (w.N + w.n_shared * w.T) * 2 * w.d_ff * bf


def run_ours(args, world, rank, local):
    from routed_expert_swiglu_gb300 import binding, build
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    build.build()  # recompiles whatever is older than its sources; a no-op when up to date
    binding.load()
    peaks, peak_src = load_peaks()
    w = workloads.BY_NAME[args.workload]

    with ClockSampler(local) as clk:
        layer, inp, total_ms, stage_ms, active, launches = measure_workload(
            w, args.steps, args.warmup, device, seed=rank, world=world, rank=rank)
    clocks = clk.summary()
    ms_max = max_over_ranks(total_ms, world)
    ms_per_step = ms_max / args.steps
    tokens_per_s = world * w.T * args.steps / (ms_max / 1e3)

    # dominant kernel: the gate/up grouped GEMM
    g1_ms = stage_ms[STAGES.index("gate_up_gemm")]
    g1_bytes = gate_up_bytes(w, active)
    g1_gbs = g1_bytes / (g1_ms / 1e3) / 1e9
    hbm_peak = float(peaks["hbm_gbs"])
    layer_flops = cost.layer_flops(w)
    layer_bytes = cost.layer_bytes(w, active)
    roof_s = cost.roofline_seconds(layer_flops, layer_bytes, float(peaks["bf16_tflops_sustained"]), hbm_peak)
    gemm_ms = stage_ms[STAGES.index("gate_up_gemm")] + stage_ms[STAGES.index("down_gemm")]
    gemm_roof_s = cost.roofline_seconds(cost.expert_gemm_flops(w), cost.expert_gemm_bytes(w, active),
                                        float(peaks["bf16_tflops_sustained"]), hbm_peak)
    e2e_ms, h2d, d2h = measure_e2e(layer, inp, w, args.steps, args.warmup, world)
    prefill_fp8 = prefill_mxfp4 = None
    if not args.no_fp8:
        prefill_fp8 = measure_fp8(layer, inp, w, max(args.steps // 2, 5), args.warmup, active, ms_per_step,
                                  hbm_peak, world)
        prefill_mxfp4 = measure_mxfp4(layer, inp, w, max(args.steps // 2, 5), args.warmup,
                                      prefill_fp8["ms_per_step"], ms_per_step, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, min(args.cpu_tokens, w.T))
    layer.close()
    del layer, inp
    torch.cuda.empty_cache()

    skewed = None
    if args.skew_workload not in ("none", args.workload):
        ws = workloads.BY_NAME[args.skew_workload]
        sl, sinp, sms_, sstage, sactive, _ = measure_workload(ws, max(args.steps // 2, 5), args.warmup, device,
                                                              seed=rank, world=world, rank=rank)
        sms_ = max_over_ranks(sms_, world) / max(args.steps // 2, 5)
        s_roof = cost.roofline_seconds(cost.layer_flops(ws), cost.layer_bytes(ws, sactive),
                                       float(peaks["bf16_tflops_sustained"]), hbm_peak)
        counts = sl.views(ws.T)["counts"].cpu().numpy()
        skewed = {"workload": ws.name, "T": ws.T, "ms_per_step": round(sms_, 4),
                  "tokens_per_s": round(world * ws.T / (sms_ / 1e3), 1), "active_experts": sactive,
                  "rows_hottest_expert": int(counts.max()), "rows_median_expert": int(np.median(counts)),
                  "layer_roofline_ms": round(s_roof * 1e3, 4), "layer_roofline_frac": round(s_roof * 1e3 / sms_, 4),
                  "stage_ms": {s: round(v, 4) for s, v in zip(STAGES, sstage)}}
        sl.close()
        del sl, sinp
        torch.cuda.empty_cache()

    decode = None
    if args.decode_workload not in ("none", args.workload):
        wd = workloads.BY_NAME[args.decode_workload]
        dl, dinp, dms, dstage, dactive, _ = measure_workload(wd, max(args.steps, 10), args.warmup, device,
                                                             seed=rank, world=world, rank=rank)
        dms = max_over_ranks(dms, world) / max(args.steps, 10)
        dbytes = cost.layer_bytes(wd, dactive)
        decode = {"workload": wd.name, "T": wd.T, "ms_per_step": round(dms, 4),
                  "tokens_per_s": round(world * wd.T / (dms / 1e3), 1), "active_experts": dactive,
                  "layer_bytes": int(dbytes), "hbm_gbs_layer": round(dbytes / (dms / 1e3) / 1e9, 1),
                  "hbm_frac_layer": round(dbytes / (dms / 1e3) / 1e9 / hbm_peak, 4),
                  "stage_ms": {s: round(v, 4) for s, v in zip(STAGES, dstage)}}
        if not args.no_fp8:
            decode["fp8_weights"] = measure_fp8(dl, dinp, wd, max(args.steps, 10), args.warmup, dactive, dms,
                                                hbm_peak, world)
            decode["mxfp4_weights"] = measure_mxfp4(dl, dinp, wd, max(args.steps, 10), args.warmup,
                                                    decode["fp8_weights"]["ms_per_step"], dms, world)
        dl.close()
        del dl, dinp
        torch.cuda.empty_cache()

    small = None
    if 0 < args.small_prefill_tokens != w.T:
        small = measure_leg(w.with_T(args.small_prefill_tokens), args, device, rank, world, peaks, hbm_peak)

    line = {
        "metric": "MoE-layer tokens/s (V4-Flash shape)",
        "value": round(tokens_per_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "d_ff": w.d_ff, "E": w.E, "k": w.k,
                   "n_shared": w.n_shared, "score": w.score, "bias": w.use_bias,
                   "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (expert weights "
                   f"{(w.E + w.n_shared) * 3 * w.d * w.d_ff * 2 / 1e9:.1f} GB)"},
        "roofline": {"kernel": "gate_up_gemm", "bound": "hbm", "achieved": round(g1_gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(g1_gbs / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": measured_traffic(w.name), "algorithmic_bytes": int(g1_bytes),
                     "intermediate_bytes": int(gate_up_intermediate_bytes(w)), "avg_ms": round(g1_ms, 4)},
        "layer_roofline": {"flops": int(layer_flops), "bytes": int(layer_bytes), "active_experts": active,
                           "roofline_ms": round(roof_s * 1e3, 4), "frac": round(roof_s * 1e3 / ms_per_step, 4),
                           "peaks": f"{peaks['bf16_tflops_sustained']} TFLOP/s sustained bf16, {hbm_peak} GB/s "
                                    f"({peak_src})"},
        "grouped_gemm_tflops": round(cost.expert_gemm_flops(w) / (gemm_ms / 1e3) / 1e12, 1),
        "grouped_gemm_roofline": {"ms": round(gemm_roof_s * 1e3, 4), "measured_ms": round(gemm_ms, 4),
                                  "frac": round(gemm_roof_s * 1e3 / gemm_ms, 4),
                                  "what": "gate/up + down GEMMs against max(their FLOPs / sustained bf16, "
                                          "activated expert weights + token rows in and out / HBM)"},
        "stage_ms": {s: round(v, 4) for s, v in zip(STAGES, stage_ms)},
        "e2e": {"value": round(world * w.T * args.steps / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms / args.steps, 4), "api": "moe_forward_host"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "fp8_weights": prefill_fp8,
        "mxfp4_weights": prefill_mxfp4,
        "decode": decode,
        "small_prefill": small,
        "skewed": skewed,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- CPU oracle

class HostLayer:
    """The layer's inputs copied to host memory as bf16 (what a CPU implementation holds);
    the oracle widens what it touches to fp64 as part of its own work."""

    def __init__(self, inp, ntok):
        c = lambda t: None if t is None else t.detach().cpu()  # noqa: E731
        self.x = inp.x[:ntok].detach().cpu()
        self.w_r, self.w13, self.w2 = c(inp.w_r), c(inp.w13), c(inp.w2)
        self.w13_sh, self.w2_sh, self.bias = c(inp.w13_sh), c(inp.w2_sh), c(inp.bias)
        self.tid2eid = c(inp.tid2eid)
        self.token_ids = None if inp.token_ids is None else inp.token_ids[:ntok].detach().cpu()


def _oracle_sample(w, h: HostLayer):
    """Oracle on the host copy: router logits, routing, every selected expert, shared, combine."""
    import oracle
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()  # noqa: E731
    x64 = f64(h.x)
    logits = oracle.router_logits(x64, f64(h.w_r))
    ids, wts, _ = oracle.route(logits, w.k, w.score, bias=f64(h.bias), n_groups=w.n_groups,
                               topk_groups=w.topk_groups, group_topk=w.group_topk,
                               token_ids=None if h.token_ids is None else h.token_ids.numpy(),
                               tid2eid=None if h.tid2eid is None else h.tid2eid.numpy())
    shared = None if h.w13_sh is None else (f64(h.w13_sh), f64(h.w2_sh))
    return oracle.forward(x64, ids, wts, lambda e: (f64(h.w13[e]), f64(h.w2[e])), shared)


def _oracle_routing(w, h: HostLayer):
    """Oracle routing alone (router logits + scoring + top-k) on the host copy."""
    import oracle
    f64 = lambda t: None if t is None else t.to(torch.float64).numpy()  # noqa: E731
    logits = oracle.router_logits(f64(h.x), f64(h.w_r))
    return oracle.route(logits, w.k, w.score, bias=f64(h.bias), n_groups=w.n_groups,
                        topk_groups=w.topk_groups, group_topk=w.group_topk,
                        token_ids=None if h.token_ids is None else h.token_ids.numpy(),
                        tid2eid=None if h.tid2eid is None else h.tid2eid.numpy())


def cpu_baseline(w, inp, ntok):
    h = HostLayer(inp, ntok)
    t0 = time.perf_counter()
    _oracle_sample(w, h)
    dt = time.perf_counter() - t0
    t0 = time.perf_counter()
    _oracle_routing(w, h)
    dr = time.perf_counter() - t0
    return {"value": round(ntok / dt, 3), "unit": "tokens/s", "cores": _NCORES, "kind": "oracle",
            "sample": f"{ntok} tokens of {w.name} (routing + every selected expert + shared + combine), "
                      f"fp64 numpy on host copies of the bf16 inputs", "seconds": round(dt, 2),
            "routing_tokens_per_s": round(ntok / dr, 1)}


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workloads.BY_NAME[args.workload]
    ntok = args.ref_tokens
    dev = "cuda:0" if torch.cuda.is_available() else "cpu"
    inp = inputs.make_layer_inputs(w, seed=0, device=dev, T=ntok)   # input synthesis only
    h = HostLayer(inp, ntok)
    del inp
    if dev != "cpu":
        torch.cuda.empty_cache()
    for _ in range(args.warmup):
        hw = HostLayer.__new__(HostLayer)
        hw.__dict__.update(h.__dict__)
        hw.x = h.x[:1]
        hw.token_ids = None if h.token_ids is None else h.token_ids[:1]
        _oracle_sample(w, hw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample(w, h)
    dt = time.perf_counter() - t0
    value = args.steps * ntok / dt
    line = {"impl": "reference", "metric": "MoE-layer tokens/s (V4-Flash shape)", "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "d_ff": w.d_ff, "E": w.E, "k": w.k,
                       "n_shared": w.n_shared, "sample_tokens_per_step": ntok},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": _NCORES, "kind": "oracle",
                             "sample": f"{ntok} tokens of {w.name} per step"},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="v4flash_T8192", choices=sorted(workloads.BY_NAME))
    ap.add_argument("--decode-workload", default="v4flash_T64", help="second (decode) workload, or none")
    ap.add_argument("--small-prefill-tokens", type=int, default=1024,
                    help="T of a small prefill batch on the main workload's shapes (0: none)")
    ap.add_argument("--skew-workload", default="v4flash_zipf_T8192",
                    help="the same layer with Zipf-skewed routing, timed alongside (or none)")
    ap.add_argument("--cpu-tokens", type=int, default=8192,
                    help="tokens of the workload the CPU-baseline oracle runs, at most T (the whole "
                         "V4-Flash T=8192 batch: about 10 s on 16 Grace cores)")
    ap.add_argument("--ref-tokens", type=int, default=240,
                    help="tokens per step of the reference arm (the oracle; about 3 s per step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8- and MXFP4-weight measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_replicas(args.gpus))
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
