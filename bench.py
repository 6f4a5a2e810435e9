"""Benchmark of the bit-exact block-scaled int8 GEMM on GB300.

One step = one pass of the whole hot path over one batch: the three
GPT-2-small linears at M = 8192 tokens -- QKV (K 768 -> N 2304), fc
(768 -> 3072, fused ReLU), proj (3072 -> 768) -- each a full bsgemm_i8
(per-row quantize of A, per-column quantize of B, exact int8 contraction on
the tensor cores, f32 epilogue), plus the step's probe hash (the seeded
1024^3 GEMM hashed to 32 bytes).  Throughput counts 2*M*N*K operations per
GEMM.  Inputs are synthetic (seeded, GPT-2-small-shaped), resident in HBM
before the timed region; L2 is flushed between timed steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `--impl reference` times the CPU oracle on a bounded
sample of the same workload on this host's cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "bit-exact block-scaled int8 GEMM TOPS and % of GB300 dense INT8 peak"
WORKLOAD = "gpt2_small_linears_M8192_qkv_fc_proj+probe1024"
PROBE = (1024, 1024, 1024)
PROBE_SEED = 0
L2_FLUSH_BYTES = 256 << 20
STAGE_REPEAT = 8          # launches per stage graph for the per-kernel durations
GEMM_SOURCES = ("verifiable_quantize_rows_gb300/csrc/gemm_tc.cu",
                "verifiable_quantize_rows_gb300/csrc/bsg_ptx.cuh")
GEMM_PROFILE = "profiles/gemm_tc_gpt2_linears.md"


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def step_ops():
    from verifiable_quantize_rows_gb300 import inputs
    ops = sum(2 * M * N * K for _, M, N, K, _, _ in inputs.GPT2_LINEARS)
    return ops + 2 * PROBE[0] * PROBE[1] * PROBE[2]


def config_dict(n_gpus):
    from verifiable_quantize_rows_gb300 import inputs
    return {
        "workload": WORKLOAD,
        "gemms": [{"name": n, "M": M, "N": N, "K": K, "relu": r}
                  for n, M, N, K, r, _ in inputs.GPT2_LINEARS]
                 + [{"name": "probe", "M": PROBE[0], "N": PROBE[1], "K": PROBE[2], "relu": False}],
        "inputs": "activations N(0,1) with 0.1% x20 outliers, weights N(0,0.02), seeded",
        "l2": "flushed between timed steps (256 MiB write); inputs resident in HBM",
        "parallelism": f"replicas x{n_gpus} (weak: each GPU runs the full step)",
    }


def code_digest(texts):
    """SHA-256 (16 hex digits) of C/C++ sources with comments and blank lines
    removed: an edit of comments alone keeps the digest."""
    import hashlib
    import re
    h = hashlib.sha256()
    for text in texts:
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def gemm_source_hash():
    """Digest of the GEMM's code (see code_digest), as recorded in the
    committed ncu summary."""
    texts = []
    for rel in GEMM_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            texts.append(f.read())
    return code_digest(texts)


def profiled_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current GEMM source (else None: the counters are stale)."""
    p = os.path.join(ROOT, GEMM_PROFILE)
    if not os.path.exists(p):
        return None
    src, per = None, {}
    with open(p) as f:
        for line in f:
            parts = line.strip().strip("`").split()
            if len(parts) == 2 and parts[0] == "source-sha256:":
                src = parts[1]
            elif len(parts) == 3 and parts[0] == "dram-bytes-per-launch":
                per[parts[1].rstrip(":")] = int(parts[2])
    if src != gemm_source_hash() or not per:
        return None
    return per


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# -------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the raw samples: a temporary file unless BSG_CLOCKS_DIR names a
        # folder to keep them in
        import tempfile
        folder = os.environ.get("BSG_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(folder, f"bsg_clocks_gpu{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_selector(local_rank):
    """nvidia-smi -i argument for this process's GPU (its UUID when known)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        if u:
            return u if u.startswith("GPU-") else f"GPU-{u}"
    except Exception:
        pass
    return str(local_rank)


# -------------------------------------------------------------- GPU arm
def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import verifiable_quantize_rows_gb300 as bsg
    from verifiable_quantize_rows_gb300 import build as bsg_build
    from verifiable_quantize_rows_gb300 import inputs

    if not os.path.exists(bsg.LIB_PATH):
        bsg_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    lib = bsg.load()

    # resident inputs and outputs
    lin = []
    for name, M, N, K, relu, seed in inputs.GPT2_LINEARS:
        A, B, _ = inputs.gpt2_linear_inputs(name)
        ws = bsg.Workspace(dev)
        ws.get(lib.bsgemm_i8_workspace_size(M, N, K))
        lin.append(dict(name=name, M=M, N=N, K=K, relu=relu, A=A.to(dev), B=B.to(dev),
                        C=torch.empty(M, N, device=dev), ws=ws, Ah=A.pin_memory(),
                        Bh=B.pin_memory(), Ch=torch.empty(M, N, pin_memory=True)))
    pws = bsg.Workspace(dev)
    pws.get(lib.bsg_probe_workspace_size(*PROBE))
    probe_out = torch.empty(32, dtype=torch.uint8, device=dev)
    dstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    host_ws = bsg.Workspace(dev)
    host_ws.get(sum((lib.bsgemm_i8_host_workspace_size(L["M"], L["N"], L["K"]) + 255) // 256 * 256
                    for L in lin))

    side = torch.cuda.Stream(device=dev)

    def stage_quantize(L):
        bsg.bsgemm_i8_quantize(L["A"], L["B"], L["ws"], dstatus=dstatus)

    def stage_contract(L):
        bsg.bsgemm_i8_contract(L["M"], L["N"], L["K"], L["C"], L["ws"], relu=L["relu"],
                               dstatus=dstatus)

    def stage_probe():
        bsg.probe_hash_async(PROBE_SEED, *PROBE, out=probe_out, dstatus=dstatus, workspace=pws)

    def step_body():
        """One step on the current stream; the probe runs on a side stream
        forked from it and joined at the end, so it overlaps the linears."""
        cur = torch.cuda.current_stream()
        if args.probe_overlap:
            side.wait_stream(cur)
            with torch.cuda.stream(side):
                stage_probe()
        for L in lin:
            stage_quantize(L)
            stage_contract(L)
        if args.probe_overlap:
            cur.wait_stream(side)
        else:
            stage_probe()

    # Per-kernel launch durations: each stage is captured STAGE_REPEAT times
    # back to back in one graph, timed with events around the replay and
    # divided by the repeat count (a one-launch graph would add the graph's
    # own launch latency to every number).  Quantize stages rotate over
    # STAGE_REPEAT copies of their inputs, so that every launch reads A and B
    # from HBM as in the step; GEMM stages re-run on the operands their
    # quantize stage wrote, which sit in L2 as they do in the step.
    R = STAGE_REPEAT
    for L in lin:
        L["copies"] = [(L["A"].clone(), L["B"].clone()) for _ in range(R - 1)] + [(L["A"], L["B"])]

    def stage_quantize_r(L):
        for A_, B_ in L["copies"]:
            bsg.bsgemm_i8_quantize(A_, B_, L["ws"], dstatus=dstatus)

    def stage_contract_r(L):
        for _ in range(R):
            stage_contract(L)

    def stage_probe_r():
        for _ in range(R):
            stage_probe()

    stages = []
    for L in lin:
        stages.append(("quantize_" + L["name"], (lambda L=L: stage_quantize_r(L))))
        stages.append(("gemm_" + L["name"], (lambda L=L: stage_contract_r(L))))
    stages.append(("probe", stage_probe_r))

    def barrier():
        if world > 1:
            dist.barrier()

    # warm up eagerly (first calls set kernel attributes), then capture graphs
    for _ in range(args.warmup):
        step_body()
    torch.cuda.synchronize()
    capture = torch.cuda.Stream(device=dev)
    n0 = bsg.launch_count()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=capture):
        step_body()
    launches_step = bsg.launch_count() - n0
    g_stages = []
    launches_stages = 0
    for name, fn in stages:
        g = torch.cuda.CUDAGraph()
        n0 = bsg.launch_count()
        with torch.cuda.graph(g, stream=capture):
            fn()
        launches_stages += bsg.launch_count() - n0
        g_stages.append((name, g))
    for _ in range(args.warmup):
        g_step.replay()
        for _, g in g_stages:
            g.replay()
    torch.cuda.synchronize()

    # ---- timed region: device-resident inputs, L2 flushed between steps
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    stage_steps = max(10, min(args.steps, 50))
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(len(g_stages))] for _ in range(stage_steps)]
    clocks = ClockSampler(gpu_selector(local_rank))
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()                      # L2 flush, outside the timed pair
        ev_step[s][0].record(stream)
        g_step.replay()
        ev_step[s][1].record(stream)
    for s in range(stage_steps):
        for k, (name, g) in enumerate(g_stages):
            if not name.startswith("gemm_"):   # a GEMM reads what its quantize just wrote
                flush.zero_()
            e0, e1 = evs[s][k]
            e0.record(stream)
            g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    launches = launches_step * args.steps + launches_stages * stage_steps
    clk = clocks.stop()

    step_ms_list = [a.elapsed_time(b) for a, b in ev_step]
    stage_ms = [[a.elapsed_time(b) / R for a, b in row] for row in evs]
    ms_per_step = statistics.mean(step_ms_list)
    probe_hex = bytes(probe_out.cpu().tolist()).hex()
    # ---- end-to-end through the host-buffer entry points (copies inside):
    # the probe starts on a side stream (device work only), the three linears
    # run as one pipelined batch call (bound by the host link), then the
    # probe's 32-byte hash is read back to the host
    e2e_hash = torch.empty(32, dtype=torch.uint8, device=dev)
    e2e_hash_host = torch.empty(32, dtype=torch.uint8, pin_memory=True)

    def e2e_step():
        side.wait_stream(torch.cuda.current_stream())
        bsg.probe_hash_async(PROBE_SEED, *PROBE, out=e2e_hash, stream=side, dstatus=dstatus,
                             workspace=pws)
        _, st = bsg.bsgemm_i8_host_batch([(L["Ah"], L["Bh"], L["relu"], L["Ch"]) for L in lin],
                                         workspace=host_ws)
        if st:
            raise RuntimeError(f"device status {st} in the end-to-end step")
        with torch.cuda.stream(side):
            e2e_hash_host.copy_(e2e_hash, non_blocking=True)
        side.synchronize()
        return bytes(e2e_hash_host.tolist())

    def e2e_step_calls():
        """The same work as one bsgemm_i8_host call per linear (for comparison)."""
        for L in lin:
            bsg.bsgemm_i8_host(L["Ah"], L["Bh"], relu=L["relu"], out=L["Ch"], workspace=host_ws)
        return bsg.probe_hash(PROBE_SEED, *PROBE, workspace=pws)

    for _ in range(max(1, args.warmup // 2)):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e2e_times = []
    e2e_hex = ""
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t = time.perf_counter()
        e2e_hex = e2e_step().hex()         # synchronizes: C and the hash are on the host
        e2e_times.append(time.perf_counter() - t)
    barrier()
    e2e_ms = statistics.mean(e2e_times) * 1e3
    calls_times = []
    for _ in range(min(args.steps, 50)):
        flush.zero_()
        torch.cuda.synchronize()
        t = time.perf_counter()
        e2e_step_calls()
        calls_times.append(time.perf_counter() - t)
    e2e_calls_ms = statistics.mean(calls_times) * 1e3

    # ---- max over ranks, and the replicas' probe hashes (the pages' cross-device check)
    from verifiable_quantize_rows_gb300.replicas import max_over_ranks, probe_hashes_agree
    ms_max, e2e_max = max_over_ranks([ms_per_step, e2e_ms], device=dev)
    golden = None
    gpath = os.path.join(ROOT, "tests", "golden", "probe_hash.txt")
    if os.path.exists(gpath):
        for line in open(gpath):
            p = line.split()
            if len(p) == 5 and p[:4] == [str(PROBE_SEED), *map(str, PROBE)]:
                golden = p[4]
    replicas_agree, _ = probe_hashes_agree(bytes.fromhex(probe_hex), device=dev)
    torch.cuda.synchronize()
    dstat = int(dstatus.item())

    if rank != 0:
        return None

    ops = step_ops()
    peaks, peak_kind = load_peaks()
    prof = profiled_traffic()
    traffic = (round(sum(prof[L["name"]] for L in lin) / len(lin))
               if prof and all(L["name"] in prof for L in lin) else None)
    # f16 operands read once, f32 C written once
    algo_bytes = round(sum(2 * (L["M"] + L["N"]) * L["K"] + 4 * L["M"] * L["N"] for L in lin)
                       / len(lin))
    # dominant kernel: the tensor-core contraction (one launch per linear),
    # timed per stage graph in the second half of the timed region
    gemm_ms = [statistics.mean(sm[2 * i + 1] for sm in stage_ms) for i in range(len(lin))]
    quant_ms = [statistics.mean(sm[2 * i] for sm in stage_ms) for i in range(len(lin))]
    probe_ms = statistics.mean(sm[-1] for sm in stage_ms)
    gemm_ops = [2 * L["M"] * L["N"] * L["K"] for L in lin]
    achieved = sum(gemm_ops) / (sum(gemm_ms) * 1e-3) / 1e12      # TFLOP/s (f16 pipe)
    peak = float(peaks.get("bf16_tflops", 1900.0))
    quant_bytes = [4 * (L["M"] * L["K"] + L["K"] * L["N"]) + 2 * (L["M"] * L["K"] + L["K"] * L["N"])
                   for L in lin]
    quant_gbs = sum(quant_bytes) / (sum(quant_ms) * 1e-3) / 1e9
    value = ops * world / (ms_max * 1e-3) / 1e12
    h2d = sum(4 * (L["M"] * L["K"] + L["K"] * L["N"]) for L in lin)
    d2h = sum(4 * L["M"] * L["N"] for L in lin) + 32
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic",
        "config": config_dict(world),
        "roofline": {
            "bound": "tensor",
            "kernel": "gemm_tc_kernel (tcgen05 kind::f16, exact int8 contraction + epilogue)",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} bf16 burst (f16 dense rate = bf16 nominal)",
            "traffic": traffic,
            "traffic_note": ("DRAM bytes read + written per GEMM launch (mean of the three "
                             "linears) from the committed ncu summary " + GEMM_PROFILE +
                             ", taken on this GEMM source; null if the source has changed "
                             "since"),
            "algorithmic_bytes": algo_bytes,
            "per_gemm_ms": {L["name"]: round(g, 4) for L, g in zip(lin, gemm_ms)},
        },
        "quantize": {
            "bound": "hbm",
            "achieved_gbs": round(quant_gbs, 1),
            "peak_gbs": float(peaks.get("hbm_gbs", 6800.0)),
            "frac": round(quant_gbs / float(peaks.get("hbm_gbs", 6800.0)), 4),
            "bytes": "4 B read + 2 B f16 operand write per element of A and B",
            "per_gemm_ms": {L["name"]: round(q, 4) for L, q in zip(lin, quant_ms)},
        },
        "probe_ms": round(probe_ms, 4),
        "int8_peak_note": ("sm_103a has no int8 tensor-core MMA (ptxas rejects tcgen05 "
                           "kind::i8); the exact contraction runs on the f16 pipe, so the "
                           "roofline peak is the measured 16-bit dense rate"),
        "e2e": {"value": round(ops * world / (e2e_max * 1e-3) / 1e12, 3), "unit": "TOPS",
                "ms_per_step": round(e2e_max, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "bsgemm_i8_host_batch of the three linears (pinned host A, B in; C out) "
                       "+ bsg_probe_hash",
                "one_call_per_linear_ms_per_step": round(e2e_calls_ms, 4),
                "probe_hash_matches_golden": (golden == e2e_hex) if golden else None},
        "clocks": clk,
        "gpu_launches": launches,
        "wall_s_timed": round(wall, 4),
        "timing": ("value/ms_per_step: the whole step replayed as one CUDA graph, CUDA events "
                   "around each replay, L2 flushed before each; roofline/quantize/probe: per "
                   f"launch, each stage captured {R}x back to back in one graph and timed with "
                   f"events around its replay / {R}, quantize over {R} input copies (reads from "
                   "HBM), GEMM on the operands its quantize wrote (in L2, as in the step)"),
        "probe_overlap": bool(args.probe_overlap),
        "stage_sum_ms": round(statistics.mean(sum(x) for x in stage_ms), 4),
        "probe_hash": probe_hex,
        "probe_hash_matches_golden": (golden == probe_hex) if golden else None,
        "replicas_agree": replicas_agree,
        "device_status": dstat,
    }
    return line


# -------------------------------------------------------------- config sweep
def run_configs(args):
    """Device time of the unit on every workload of the measurement plan
    (inputs resident in HBM, L2 flushed between timed replays): one JSON line
    per workload.  Each timing is a graph of R back-to-back calls, replayed
    10 times; the median replay / R is reported."""
    import torch
    import verifiable_quantize_rows_gb300 as bsg
    from verifiable_quantize_rows_gb300 import inputs
    dev = torch.device("cuda", 0)
    peaks, _ = load_peaks()
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    dstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    capture = torch.cuda.Stream(device=dev)

    def timed(fn, target_us=400.0):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); fn(); e1.record(); torch.cuda.synchronize()
        R = int(max(1, min(8, target_us // max(e0.elapsed_time(e1) * 1e3, 1.0))))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=capture):
            for _ in range(R):
                fn()
        g.replay()
        ts = []
        for _ in range(10):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); g.replay(); b.record(); torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / R)
        return statistics.median(ts)

    def timed_copies(fns):
        """Median device time per call of a graph that calls each fn once."""
        for fn in fns:
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=capture):
            for fn in fns:
                fn()
        g.replay()
        ts = []
        for _ in range(10):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(); g.replay(); b.record(); torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) * 1e3 / len(fns))
        return statistics.median(ts)

    def unit_line(name, A, B, relu=False):
        M, K = A.shape
        N = B.shape[1]
        ws = bsg.Workspace(dev)
        ws.get(bsg.workspace_size(M, N, K))
        C = torch.empty(M, N, device=dev)
        if (M * K + K * N) * 4 * 8 <= (1 << 30):
            # inputs this small are timed over 8 copies, so that every call
            # reads its inputs from HBM, as in a model
            copies = [(A.clone(), B.clone()) for _ in range(7)] + [(A, B)]
            q_us = timed_copies([(lambda A_=A_, B_=B_: bsg.bsgemm_i8_quantize(
                A_, B_, ws, dstatus=dstatus)) for A_, B_ in copies])
            del copies
        else:
            q_us = timed(lambda: bsg.bsgemm_i8_quantize(A, B, ws, dstatus=dstatus))
        g_us = timed(lambda: bsg.bsgemm_i8_contract(M, N, K, C, ws, relu=relu, dstatus=dstatus))
        u_us = timed(lambda: bsg.bsgemm_i8(A, B, relu=relu, out=C, dstatus=dstatus, workspace=ws))
        ops = 2 * M * N * K
        qbytes = 6 * (M * K + K * N)
        return {"config": name, "M": M, "N": N, "K": K, "relu": relu,
                "unit_us": round(u_us, 2), "unit_tops": round(ops / u_us / 1e6, 1),
                "gemm_us": round(g_us, 2), "gemm_tflops": round(ops / g_us / 1e6, 1),
                "gemm_frac_of_measured_bf16": round(ops / g_us / 1e6 / tc_peak, 3),
                "quantize_us": round(q_us, 2), "quantize_gbs": round(qbytes / q_us / 1e3, 1),
                "quantize_frac_of_measured_hbm": round(qbytes / q_us / 1e3 / hbm_peak, 3)}

    lines = []
    lines.append(unit_line("c0 256^3", inputs.normal((256, 256), 1.0, 0).to(dev),
                           inputs.normal((256, 256), 1.0, 1).to(dev)))
    for name, M, N, K, relu, seed in inputs.GPT2_LINEARS:
        A, B, _ = inputs.gpt2_linear_inputs(name)
        lines.append(unit_line("c1 " + name, A.to(dev), B.to(dev), relu))
    lines.append(unit_line("c2 lm head", inputs.gpt2_activations(8192, 768, 4).to(dev),
                           inputs.gpt2_weights(768, 50304, 4).to(dev)))
    pws = bsg.Workspace(dev)
    pws.get(bsg.load().bsg_probe_workspace_size(*PROBE))
    pout = torch.empty(32, dtype=torch.uint8, device=dev)
    p_us = timed(lambda: bsg.probe_hash_async(PROBE_SEED, *PROBE, out=pout, dstatus=dstatus,
                                              workspace=pws))
    lines.append({"config": "c2 probe 1024^3 (fill, unit, hash)", "unit_us": round(p_us, 2),
                  "unit_tops": round(2 * 1024 ** 3 / p_us / 1e6, 1)})
    X, W, dY = (t.to(dev) for t in inputs.train_trio())
    trio = [(X, W, False, False, False), (dY, W, False, True, False), (X, dY, True, False, False)]
    gws = bsg.Workspace(dev)
    g_us = timed(lambda: bsg.bsgemm_i8_group(trio, dstatus=dstatus, workspace=gws))
    s_us = timed(lambda: [bsg.bsgemm_i8_ex(A, B, transA=tA, transB=tB, relu=r, dstatus=dstatus)
                          for A, B, tA, tB, r in trio])
    ops = 3 * 2 * 8192 * 3072 * 768
    lines.append({"config": "c3 training trio 8192x3072x768", "grouped_us": round(g_us, 1),
                  "grouped_tops": round(ops / g_us / 1e6, 1), "separate_us": round(s_us, 1),
                  "separate_tops": round(ops / s_us / 1e6, 1)})
    del X, W, dY, trio
    for n in (4096, 8192, 16384):
        lines.append(unit_line(f"c4 {n}^3", inputs.uniform((n, n), -1, 1, 7).to(dev),
                               inputs.uniform((n, n), -1, 1, 8).to(dev)))
        torch.cuda.empty_cache()
    lines.append(unit_line("c4 ragged", inputs.uniform((4097, 8191), -1, 1, 9).to(dev),
                           inputs.uniform((8191, 12289), -1, 1, 10).to(dev)))
    lines.append(unit_line("c4 adversarial 4096^3", inputs.adversarial(4096, 4096, 11).to(dev),
                           inputs.adversarial(4096, 4096, 12, along_rows=False).to(dev)))
    torch.cuda.synchronize()
    if int(dstatus.item()) & ~1:  # the adversarial mix sets the non-finite bit by design
        raise RuntimeError(f"device status {int(dstatus.item())}")
    return lines


# -------------------------------------------------------------- CPU oracle
def oracle_inputs():
    """The step's inputs for the oracle, generated once (the same seeded
    tensors the GPU arm uses)."""
    from verifiable_quantize_rows_gb300 import inputs
    out = []
    for name, M, N, K, relu, seed in inputs.GPT2_LINEARS:
        A, B, _ = inputs.gpt2_linear_inputs(name)
        out.append((A.numpy(), B.numpy(), relu))
    return out


PARTS = ("qkv", "fc", "proj", "probe")


def oracle_part(orc, data, part, rows):
    """Part `part` of the step on the oracle: a GPT-2 linear on the first
    `rows` rows of its A (full N, K), or (part 3) the probe with M = `rows`
    (N = K = 1024, hash included).  Returns (ops, seconds)."""
    if part < 3:
        A, B, relu = data[part]
        a = np.ascontiguousarray(A[:rows])
        t0 = time.perf_counter()
        orc.bsgemm_i8(a, B, relu)
        return 2 * a.shape[0] * B.shape[1] * B.shape[0], time.perf_counter() - t0
    t0 = time.perf_counter()
    orc.probe_hash(PROBE_SEED, rows, PROBE[1], PROBE[2])
    return 2 * rows * PROBE[1] * PROBE[2], time.perf_counter() - t0


def sample_rows(orc, data, seconds):
    """Rows per part for about `seconds` of oracle work each, scaled from a
    256-row calibration run of every part."""
    rows = []
    for part in range(len(PARTS)):
        _, t = oracle_part(orc, data, part, 256)
        cap = 8192 if part < 3 else PROBE[0]
        rows.append(max(8, int(min(cap, max(8, 256 * seconds / max(t, 1e-3)))) // 8 * 8))
    return rows


def sample_text(rows):
    return (f"qkv, fc, proj on their first {rows[0]}, {rows[1]}, {rows[2]} of 8192 rows "
            f"(full N, K) and the probe at M = {rows[3]} of 1024 (N = K = 1024, hash included)")


def cpu_baseline(budget_s=12.0):
    import oracle
    orc = oracle.load()
    data = oracle_inputs()
    rows = sample_rows(orc, data, budget_s / len(PARTS))
    # repeat the four parts until about budget_s of CPU work (when even the
    # whole workload takes less)
    total_ops, total_t, reps = 0, 0.0, 0
    while total_t < 0.8 * budget_s or reps == 0:
        for part in range(len(PARTS)):
            ops, t = oracle_part(orc, data, part, rows[part])
            total_ops, total_t = total_ops + ops, total_t + t
        reps += 1
    return {"value": round(total_ops / total_t / 1e12, 6), "unit": "TOPS",
            "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{sample_text(rows)}, {reps}x: {total_ops / 1e9:.1f} G ops in "
                      f"{total_t:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    orc = oracle.load()
    data = oracle_inputs()
    # About two minutes of oracle work for the whole run, whatever K and W
    # are: step i runs part i mod 4 of the workload (qkv, fc, proj, probe),
    # each on a row sample sized to the per-step budget.
    total_budget = 120.0
    per_step = min(10.0, total_budget / max(1, args.steps + args.warmup))
    rows = sample_rows(orc, data, per_step)
    for i in range(args.warmup):
        oracle_part(orc, data, i % len(PARTS), rows[i % len(PARTS)])
    total_ops, total_t = 0, 0.0
    for i in range(args.steps):
        ops, t = oracle_part(orc, data, i % len(PARTS), rows[i % len(PARTS)])
        total_ops, total_t = total_ops + ops, total_t + t
    value = total_ops / total_t / 1e12
    ms = total_t / max(1, args.steps) * 1e3
    sample = (f"step i runs part i mod 4 of the step: {sample_text(rows)}; "
              f"{total_ops / 1e9:.2f} G ops in {total_t:.1f} s over {args.steps} steps")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8", "data": "synthetic", "config": config_dict(world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probe-overlap", type=int, default=1,
                    help="1: the probe runs on a side stream alongside the linears")
    ap.add_argument("--configs", action="store_true",
                    help="time the unit on every workload of the measurement plan instead "
                         "(one JSON line each)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local_rank = env_int("LOCAL_RANK", 0)

    if args.configs:
        for line in run_configs(args):
            print(json.dumps(line), flush=True)
        return

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_gpu(args, rank, world, local_rank)
    if line is not None:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
