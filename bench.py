"""Benchmark of the bit-exact block-scaled int8 GEMM on GB300.

One step = one pass of the whole hot path over one batch of the large and
adversarial GEMMs: 4096^3, 8192^3 and 16384^3 with U(-1, 1) values, and the
ragged 4097 x 12289 x 8191 whose rows of A and columns of B mix the
adversarial cases (all-zero and -0 vectors, exact quantize ties, subnormals,
1e30 and 1e-30 magnitudes) -- each a full bsgemm_i8 (per-row quantize of A,
per-column quantize of B, exact int8 contraction on the tensor cores, f32
epilogue) -- plus the step's probe hash (the seeded 1024^3 GEMM hashed to 32
bytes) on a side stream.  Throughput counts 2*M*N*K operations per GEMM.
Inputs are synthetic (seeded), resident in HBM before the timed region; L2
is flushed between timed steps.  The GPT-2-small linears at M = 8192 (QKV,
fc + ReLU, proj, with the probe) are measured the same way and reported
under "gpt2_linears".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `--impl reference` times the CPU oracle on a bounded
sample of the same workload on this host's cores.  `--configs` times the unit
on every workload of the measurement plan instead (one line each).
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
WORKLOAD = "large_gemms_4096^3+8192^3+16384^3+ragged_4097x12289x8191_adversarial+probe1024"
SMALL_WORKLOAD = "gpt2_small_linears_M8192_qkv_fc_proj+probe1024"
PROBE = (1024, 1024, 1024)
PROBE_SEED = 0
L2_FLUSH_BYTES = 256 << 20
GEMM_SOURCES = ("verifiable_quantize_rows_gb300/csrc/gemm_tc.cu",
                "verifiable_quantize_rows_gb300/csrc/bsg_ptx.cuh")
GEMM_PROFILE = "profiles/gemm_tc_large_gemms.md"
SMALL_GEMM_PROFILE = "profiles/gemm_tc_gpt2_linears.md"
HBM_NOMINAL_GBS = 8000.0
# The INT8 tensor figure NVIDIA publishes for the GB300 NVL72 rack, 23 POPS
# over 72 GPUs.  Blackwell Ultra cut INT8 tensor throughput far below its
# 16-bit rate, and CUDA 13.0's ptxas has no int8 tensor-core MMA for sm_103a
# at all, so the exact contraction runs on the 16-bit pipe; the fraction of
# this figure is reported because the metric names it.
INT8_DATASHEET_TOPS = 23000.0 / 72
INT8_DATASHEET_SOURCE = ("NVIDIA GB300 NVL72 specifications: INT8 Tensor Core 23 POPS for 72 "
                         "GPUs (quoted without network access here; per GPU 319.4 TOPS)")
MMA_CEILING_ITERS = 8192


def unit_list(kind):
    """(name, M, N, K, relu, loader) of the step's GEMMs."""
    from verifiable_quantize_rows_gb300 import inputs
    if kind == "large":
        return [(n, M, N, K, r, (lambda n=n: inputs.large_gemm_inputs(n)[:2]))
                for n, M, N, K, r, _ in inputs.LARGE_GEMMS]
    return [(n, M, N, K, r, (lambda n=n: inputs.gpt2_linear_inputs(n)[:2]))
            for n, M, N, K, r, _ in inputs.GPT2_LINEARS]


def step_ops(kind="large"):
    ops = sum(2 * M * N * K for _, M, N, K, _, _ in unit_list(kind))
    return ops + 2 * PROBE[0] * PROBE[1] * PROBE[2]


def quant_algo_bytes(M, N, K):
    """Quantize's algorithmic bytes for one unit: 4 B read + 1 B int8 code
    written per element of A and B, and 4 B per scale."""
    return 5 * (M * K + K * N) + 4 * (M + N)


def config_dict(n_gpus, kind="large"):
    if kind == "large":
        workload = WORKLOAD
        vals = ("squares U(-1,1) (A seed 6/7/8, B seed+1); ragged A rows / B columns: the "
                "adversarial mix (a third of the vectors all-zero, -0, exact ties, subnormal, "
                "subnormal-mixed, 1e30, 1e-30, negative-max, spike; the rest U(-1,1)), seeded")
        l2 = "flushed between timed steps (256 MiB write); inputs resident in HBM, larger than L2"
    else:
        workload = SMALL_WORKLOAD
        vals = "activations N(0,1) with 0.1% x20 outliers, weights N(0,0.02), seeded"
        l2 = "flushed between timed steps (256 MiB write); inputs resident in HBM"
    return {
        "workload": workload,
        "gemms": [{"name": n, "M": M, "N": N, "K": K, "relu": r}
                  for n, M, N, K, r, _ in unit_list(kind)]
                 + [{"name": "probe", "M": PROBE[0], "N": PROBE[1], "K": PROBE[2], "relu": False}],
        "inputs": vals,
        "l2": l2,
        "parallelism": f"replicas x{n_gpus} (weak: each GPU runs the full step)",
    }


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


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


def parse_profile(profile):
    """(source digest, {gemm name: DRAM bytes per launch}) recorded in a
    committed ncu summary, or (None, {}) if there is none."""
    p = os.path.join(ROOT, profile)
    src, per = None, {}
    if not os.path.exists(p):
        return src, per
    with open(p) as f:
        for line in f:
            parts = line.strip().strip("`").split()
            if len(parts) == 2 and parts[0] == "source-sha256:":
                src = parts[1]
            elif len(parts) == 3 and parts[0] == "dram-bytes-per-launch":
                per[parts[1].rstrip(":")] = int(parts[2])
    return src, per


def profiled_traffic(profile=GEMM_PROFILE):
    """DRAM bytes per GEMM launch from a committed ncu summary, if it was
    taken on the current GEMM source (else None: the counters are stale)."""
    src, per = parse_profile(profile)
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
class Workload:
    """Device-resident inputs, outputs and workspaces of one step's GEMMs,
    with the step and its per-stage graphs."""

    def __init__(self, kind, dev, lib, side, dstatus, probe_out, probe_ws, with_host):
        import torch
        import verifiable_quantize_rows_gb300 as bsg
        self.kind = kind
        self.dev = dev
        self.side = side
        self.dstatus = dstatus
        self.probe_out = probe_out
        self.probe_ws = probe_ws
        self.units = []
        for name, M, N, K, relu, load in unit_list(kind):
            A, B = load()
            ws = bsg.Workspace(dev)
            ws.get(lib.bsgemm_i8_workspace_size(M, N, K))
            u = dict(name=name, M=M, N=N, K=K, relu=relu, A=A.to(dev), B=B.to(dev),
                     C=torch.empty(M, N, device=dev), ws=ws)
            if with_host:
                u.update(Ah=A.pin_memory(), Bh=B.pin_memory(),
                         Ch=torch.empty(M, N, pin_memory=True))
            del A, B
            # Small inputs are timed per stage over 8 copies so that every
            # quantize launch reads them from HBM as in the step; large ones
            # (beyond L2) repeat on the same copy, twice.
            in_bytes = 4 * (M * K + K * N)
            if in_bytes <= (256 << 20):
                u["copies"] = [(u["A"].clone(), u["B"].clone()) for _ in range(7)] + [(u["A"], u["B"])]
            else:
                u["copies"] = [(u["A"], u["B"])] * 2
            self.units.append(u)

    # ---- the step
    def quantize(self, u, A=None, B=None):
        import verifiable_quantize_rows_gb300 as bsg
        bsg.bsgemm_i8_quantize(u["A"] if A is None else A, u["B"] if B is None else B, u["ws"],
                               dstatus=self.dstatus)

    def contract(self, u):
        import verifiable_quantize_rows_gb300 as bsg
        bsg.bsgemm_i8_contract(u["M"], u["N"], u["K"], u["C"], u["ws"], relu=u["relu"],
                               dstatus=self.dstatus)

    def probe(self):
        import verifiable_quantize_rows_gb300 as bsg
        bsg.probe_hash_async(PROBE_SEED, *PROBE, out=self.probe_out, dstatus=self.dstatus,
                             workspace=self.probe_ws)

    def step(self):
        """One step on the current stream; the probe runs on a side stream
        forked from it and joined at the end, so it overlaps the GEMMs."""
        import torch
        cur = torch.cuda.current_stream()
        self.side.wait_stream(cur)
        with torch.cuda.stream(self.side):
            self.probe()
        for u in self.units:
            self.quantize(u)
            self.contract(u)
        cur.wait_stream(self.side)

    def stages(self):
        """(name, fn, repeat) per stage: each is captured `repeat` times back
        to back in one graph and timed per launch."""
        out = []
        for u in self.units:
            out.append(("quantize_" + u["name"],
                        (lambda u=u: [self.quantize(u, A_, B_) for A_, B_ in u["copies"]]),
                        len(u["copies"])))
            reps = len(u["copies"])
            out.append(("gemm_" + u["name"], (lambda u=u, r=reps: [self.contract(u)
                                                                    for _ in range(r)]), reps))
        out.append(("probe", lambda: [self.probe() for _ in range(4)], 4))
        return out


def time_workload(W, steps, warmup, flush, stream, barrier, stage_steps):
    """Time W's step (graph replays, L2 flushed before each) and each stage
    (per launch).  Returns step times (ms), stage times (ms per launch, one
    row per stage round) and the number of this library's kernel launches."""
    import torch
    import verifiable_quantize_rows_gb300 as bsg
    dev = W.dev
    for _ in range(warmup):           # eager first calls set kernel attributes
        W.step()
    torch.cuda.synchronize()
    capture = torch.cuda.Stream(device=dev)
    n0 = bsg.launch_count()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=capture):
        W.step()
    launches_step = bsg.launch_count() - n0
    g_stages = []
    launches_stages = 0
    for name, fn, reps in W.stages():
        g = torch.cuda.CUDAGraph()
        n0 = bsg.launch_count()
        with torch.cuda.graph(g, stream=capture):
            fn()
        launches_stages += bsg.launch_count() - n0
        g_stages.append((name, g, reps))
    for _ in range(warmup):
        g_step.replay()
        for _, g, _ in g_stages:
            g.replay()
    torch.cuda.synchronize()

    def ev():
        return torch.cuda.Event(enable_timing=True)
    ev_step = [(ev(), ev()) for _ in range(steps)]
    evs = [[(ev(), ev()) for _ in g_stages] for _ in range(stage_steps)]
    barrier()
    torch.cuda.synchronize()
    for s in range(steps):
        flush.zero_()                      # L2 flush, outside the timed pair
        ev_step[s][0].record(stream)
        g_step.replay()
        ev_step[s][1].record(stream)
    for s in range(stage_steps):
        for k, (name, g, _) in enumerate(g_stages):
            if not name.startswith("gemm_"):   # a GEMM reads what its quantize just wrote
                flush.zero_()
            e0, e1 = evs[s][k]
            e0.record(stream)
            g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    stage_ms = {name: [evs[s][k][0].elapsed_time(evs[s][k][1]) / reps for s in range(stage_steps)]
                for k, (name, _, reps) in enumerate(g_stages)}
    launches = launches_step * steps + launches_stages * stage_steps
    del g_step, g_stages
    return step_ms, stage_ms, launches


def mma_ceiling(stream, dstatus, reps=5):
    """TFLOP/s of the tensor-pipe ceiling kernel (median of `reps` launches)."""
    import torch
    import verifiable_quantize_rows_gb300 as bsg
    bsg.mma_ceiling(MMA_CEILING_ITERS, dstatus=dstatus)
    torch.cuda.synchronize()
    ts, flops = [], 0.0
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        flops = bsg.mma_ceiling(MMA_CEILING_ITERS, dstatus=dstatus)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return flops / (statistics.median(ts) * 1e-3) / 1e12


def summarize(W, step_ms, stage_ms, peaks, peak_kind, ms_max, world, profile):
    """Roofline of the GEMM (dominant kernel) and quantize figures."""
    units = W.units
    mean = statistics.mean
    gemm_ms = [mean(stage_ms["gemm_" + u["name"]]) for u in units]
    quant_ms = [mean(stage_ms["quantize_" + u["name"]]) for u in units]
    gemm_ops = [2 * u["M"] * u["N"] * u["K"] for u in units]
    achieved = sum(gemm_ops) / (sum(gemm_ms) * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", 1900.0))
    peak_sus = float(peaks.get("bf16_tflops_sustained", 1700.0))
    prof = profiled_traffic(profile)
    traffic = (round(sum(prof[u["name"]] for u in units) / len(units))
               if prof and all(u["name"] in prof for u in units) else None)
    algo_bytes = round(sum(2 * (u["M"] + u["N"]) * u["K"] + 4 * u["M"] * u["N"] for u in units)
                       / len(units))
    qbytes = [quant_algo_bytes(u["M"], u["N"], u["K"]) for u in units]
    f16_extra = [2 * (u["M"] * u["K"] + u["K"] * u["N"]) for u in units]
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    q_gbs = sum(qbytes) / (sum(quant_ms) * 1e-3) / 1e9
    # bytes the kernels move to and from HBM: each operand read once and its
    # f16 operand written, 6 B per element (columns longer than the strip
    # kernel holds are read a second time, from L2)
    moved = [6 * (u["M"] * u["K"] + u["K"] * u["N"]) for u in units]
    roof = {
        "bound": "tensor",
        "kernel": "gemm_tc_kernel (tcgen05 kind::f16, exact int8 contraction + epilogue)",
        "achieved": round(achieved, 2),
        "peak": peak,
        "unit": "TFLOP/s",
        "frac": round(achieved / peak, 4),
        "peak_source": f"{peak_kind} bf16 burst (f16 dense rate = bf16 nominal)",
        "frac_of_sustained": round(achieved / peak_sus, 4),
        "traffic": traffic,
        "traffic_note": ("DRAM bytes read + written per GEMM launch (mean over the step's "
                         "GEMMs) from the committed ncu summary " + profile + ", taken on this "
                         "GEMM source; null if the source has changed since"),
        "algorithmic_bytes": algo_bytes,
        "per_gemm_ms": {u["name"]: round(g, 4) for u, g in zip(units, gemm_ms)},
        "per_gemm_frac": {u["name"]: round(o / (g * 1e-3) / 1e12 / peak, 4)
                          for u, o, g in zip(units, gemm_ops, gemm_ms)},
    }
    quant = {
        "bound": "hbm",
        "achieved_gbs": round(q_gbs, 1),
        "peak_gbs": hbm,
        "frac": round(q_gbs / hbm, 4),
        "frac_of_nominal_8tbs": round(q_gbs / HBM_NOMINAL_GBS, 4),
        "bytes": "4 B read + 1 B int8 code per element of A and B + 4 B per scale",
        "f16_operand_extra_bytes": sum(f16_extra),
        "achieved_gbs_incl_f16_operand": round((sum(qbytes) + sum(f16_extra))
                                               / (sum(quant_ms) * 1e-3) / 1e9, 1),
        "moved_bytes": sum(moved),
        "moved_gbs": round(sum(moved) / (sum(quant_ms) * 1e-3) / 1e9, 1),
        "moved_frac": round(sum(moved) / (sum(quant_ms) * 1e-3) / 1e9 / hbm, 4),
        "moved_note": ("HBM bytes the kernels move: A and B read once + their f16 operands "
                       "written (6 B per element); B's columns longer than 4096 rows are read "
                       "again from L2"),
        "per_gemm_ms": {u["name"]: round(q, 4) for u, q in zip(units, quant_ms)},
        "per_gemm_frac": {u["name"]: round(b / (q * 1e-3) / 1e9 / hbm, 4)
                          for u, b, q in zip(units, qbytes, quant_ms)},
    }
    return roof, quant, mean(stage_ms["probe"])


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import verifiable_quantize_rows_gb300 as bsg
    from verifiable_quantize_rows_gb300 import build as bsg_build
    from verifiable_quantize_rows_gb300.replicas import max_over_ranks, probe_hashes_agree

    if not os.path.exists(bsg.LIB_PATH):
        bsg_build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    lib = bsg.load()
    side = torch.cuda.Stream(device=dev)
    pws = bsg.Workspace(dev)
    pws.get(lib.bsg_probe_workspace_size(*PROBE))
    probe_out = torch.empty(32, dtype=torch.uint8, device=dev)
    dstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    W = Workload("large", dev, lib, side, dstatus, probe_out, pws, with_host=True)
    clocks = ClockSampler(gpu_selector(local_rank))
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    step_ms, stage_ms, launches = time_workload(W, args.steps, args.warmup, flush, stream,
                                                barrier, stage_steps=5)
    wall = time.perf_counter() - wall0
    ceiling = mma_ceiling(stream, dstatus)
    clk = clocks.stop()
    ms_per_step = statistics.mean(step_ms)
    probe_hex = bytes(probe_out.cpu().tolist()).hex()

    # ---- end to end through the host-buffer entry points (copies inside):
    # the probe starts on a side stream, the GEMMs run as one pipelined
    # bsgemm_i8_host_batch call (bound by the host link), then the probe's
    # 32-byte hash is read back to the host
    host_ws = bsg.Workspace(dev)
    host_ws.get(sum((lib.bsgemm_i8_host_workspace_size(u["M"], u["N"], u["K"]) + 255) // 256 * 256
                    for u in W.units))
    e2e_hash = torch.empty(32, dtype=torch.uint8, device=dev)
    e2e_hash_host = torch.empty(32, dtype=torch.uint8, pin_memory=True)

    def e2e_step():
        side.wait_stream(torch.cuda.current_stream())
        bsg.probe_hash_async(PROBE_SEED, *PROBE, out=e2e_hash, stream=side, dstatus=dstatus,
                             workspace=pws)
        _, st = bsg.bsgemm_i8_host_batch([(u["Ah"], u["Bh"], u["relu"], u["Ch"])
                                          for u in W.units], workspace=host_ws)
        if st & ~1:
            raise RuntimeError(f"device status {st} in the end-to-end step")
        with torch.cuda.stream(side):
            e2e_hash_host.copy_(e2e_hash, non_blocking=True)
        side.synchronize()
        return bytes(e2e_hash_host.tolist())

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e2e_times, e2e_hex = [], ""
    import gc
    gc.collect()
    gc.disable()    # no collector pause inside a timed host step
    for _ in range(e2e_steps):
        flush.zero_()
        torch.cuda.synchronize()
        t = time.perf_counter()
        e2e_hex = e2e_step().hex()         # synchronizes: C and the hash are on the host
        e2e_times.append(time.perf_counter() - t)
    gc.enable()
    barrier()
    # the median: a host-side stall (seen: 51 and 157 ms steps among 18 ms
    # ones) would otherwise decide the figure; the mean and every step are
    # reported beside it
    e2e_ms = statistics.median(e2e_times) * 1e3
    e2e_mean_ms = statistics.mean(e2e_times) * 1e3
    e2e_all_ms = [round(t * 1e3, 3) for t in e2e_times]
    h2d = sum(4 * (u["M"] * u["K"] + u["K"] * u["N"]) for u in W.units)
    d2h = sum(4 * u["M"] * u["N"] for u in W.units) + 32
    peaks, peak_kind = load_peaks()
    ms_max, e2e_max, e2e_mean_max = max_over_ranks([ms_per_step, e2e_ms, e2e_mean_ms],
                                                   device=dev)
    roof, quant, probe_ms = summarize(W, step_ms, stage_ms, peaks, peak_kind, ms_max, world,
                                      GEMM_PROFILE)
    dstat_large = int(dstatus.item())
    del W, host_ws
    torch.cuda.empty_cache()

    # ---- the GPT-2-small linears, the same way (reported beside the headline)
    dstatus.zero_()
    Ws = Workload("small", dev, lib, side, dstatus, probe_out, pws, with_host=False)
    s_steps = max(10, min(args.steps * 4, 400))
    s_step_ms, s_stage_ms, s_launches = time_workload(Ws, s_steps, args.warmup, flush, stream,
                                                      barrier, stage_steps=20)
    s_ms = statistics.mean(s_step_ms)
    (s_ms_max,) = max_over_ranks([s_ms], device=dev)
    s_roof, s_quant, _ = summarize(Ws, s_step_ms, s_stage_ms, peaks, peak_kind, s_ms_max, world,
                                   SMALL_GEMM_PROFILE)
    dstat_small = int(dstatus.item())
    del Ws
    torch.cuda.empty_cache()

    golden = None
    gpath = os.path.join(ROOT, "tests", "golden", "probe_hash.txt")
    if os.path.exists(gpath):
        for line in open(gpath):
            p = line.split()
            if len(p) == 5 and p[:4] == [str(PROBE_SEED), *map(str, PROBE)]:
                golden = p[4]
    replicas_agree, _ = probe_hashes_agree(bytes.fromhex(probe_hex), device=dev)
    if rank != 0:
        return None
    return build_line(args, world, ms_max, roof, quant, probe_ms, ceiling, clk, launches,
                      s_launches, s_steps, wall, (e2e_max, e2e_mean_max), e2e_all_ms, h2d, d2h,
                      golden, e2e_hex,
                      probe_hex, replicas_agree, dstat_large, dstat_small, s_ms_max, s_roof,
                      s_quant)


def build_line(args, world, ms_max, roof, quant, probe_ms, ceiling, clk, launches, s_launches,
               s_steps, wall, e2e_ms2, e2e_all_ms, h2d, d2h, golden, e2e_hex, probe_hex,
               replicas_agree, dstat_large, dstat_small, s_ms_max, s_roof, s_quant):
    ops = step_ops("large")
    value = ops * world / (ms_max * 1e-3) / 1e12
    e2e_max, e2e_mean_max = e2e_ms2
    roof = dict(roof)
    roof["mma_ceiling_tflops"] = round(ceiling, 1)
    roof["frac_of_mma_ceiling"] = round(roof["achieved"] / ceiling, 4)
    roof["mma_ceiling_note"] = ("bsg_mma_ceiling: pair kind::f16 MMAs 256x256x16 issued back to "
                                "back from shared memory on every resident SM pair, no operand "
                                "copies or epilogue; median of 5 launches, CUDA events")
    s_ops = step_ops("small")
    return {
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
        "config": config_dict(world, "large"),
        "roofline": roof,
        "int8_datasheet": {
            "tops_per_gpu": round(INT8_DATASHEET_TOPS, 1),
            "source": INT8_DATASHEET_SOURCE,
            "frac_step": round(value / world / INT8_DATASHEET_TOPS, 3),
            "frac_gemm": round(roof["achieved"] / INT8_DATASHEET_TOPS, 3),
            "note": ("sm_103a has no int8 tensor-core MMA (ptxas rejects tcgen05 kind::i8); the "
                     "exact contraction runs on the f16 pipe, whose measured rate is the "
                     "roofline peak; the datasheet INT8 figure is far below it"),
        },
        "quantize": quant,
        "probe_ms": round(probe_ms, 4),
        "e2e": {"value": round(ops * world / (e2e_max * 1e-3) / 1e12, 3), "unit": "TOPS",
                "ms_per_step": round(e2e_max, 4), "statistic": "median over the steps",
                "mean_ms_per_step": round(e2e_mean_max, 4),
                "value_from_mean": round(ops * world / (e2e_mean_max * 1e-3) / 1e12, 3),
                "steps": len(e2e_all_ms), "step_ms": e2e_all_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "bsgemm_i8_host_batch of the step's four GEMMs (pinned host A, B in; "
                       "C out) + bsg_probe_hash_async with its 32 bytes read back",
                "probe_hash_matches_golden": (golden == e2e_hex) if golden else None},
        "clocks": clk,
        "gpu_launches": launches,
        "wall_s_timed": round(wall, 4),
        "timing": ("value/ms_per_step: the whole step replayed as one CUDA graph, CUDA events "
                   "around each replay, L2 flushed before each; roofline/quantize/probe: per "
                   "launch, each stage captured 2x (8x, over 8 input copies, for inputs under "
                   "256 MiB) back to back in one graph and timed with events around its replay; "
                   "the GEMM runs on the operands its quantize wrote"),
        "probe_hash": probe_hex,
        "probe_hash_matches_golden": (golden == probe_hex) if golden else None,
        "replicas_agree": replicas_agree,
        "device_status": dstat_large,
        "device_status_note": "bit 0 (non-finite input) is not expected; bit 1 is a timeout",
        "gpt2_linears": {
            "workload": SMALL_WORKLOAD,
            "config": config_dict(world, "small"),
            "value": round(s_ops * world / (s_ms_max * 1e-3) / 1e12, 3),
            "unit": "TOPS",
            "steps": s_steps,
            "ms_per_step": round(s_ms_max, 4),
            "roofline": s_roof,
            "quantize": s_quant,
            "gpu_launches": s_launches,
            "device_status": dstat_small,
        },
    }


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
        qbytes = quant_algo_bytes(M, N, K)
        return {"config": name, "M": M, "N": N, "K": K, "relu": relu,
                "unit_us": round(u_us, 2), "unit_tops": round(ops / u_us / 1e6, 1),
                "gemm_us": round(g_us, 2), "gemm_tflops": round(ops / g_us / 1e6, 1),
                "gemm_frac_of_measured_bf16": round(ops / g_us / 1e6 / tc_peak, 3),
                "quantize_us": round(q_us, 2), "quantize_gbs": round(qbytes / q_us / 1e3, 1),
                "quantize_frac_of_measured_hbm": round(qbytes / q_us / 1e3 / hbm_peak, 3),
                "quantize_frac_of_nominal_8tbs": round(qbytes / q_us / 1e3 / HBM_NOMINAL_GBS, 3),
                "quantize_bytes": "4 B read + 1 B code per element + 4 B per scale (the f16 "
                                  "operand's 2 B per element not counted)"}

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
    # the chained units: the GPT-2 MLP (fc + ReLU, then proj) as one chain
    # against two units, and one unit + its C's per-row codes against a unit
    # then a row quantize of C
    Xm = inputs.gpt2_activations(8192, 768, 2).to(dev)
    W1 = inputs.gpt2_weights(768, 3072, 2).to(dev)
    W2 = inputs.gpt2_weights(3072, 768, 3).to(dev)
    cws, uws1, uws2 = bsg.Workspace(dev), bsg.Workspace(dev), bsg.Workspace(dev)
    C1 = torch.empty(8192, 3072, device=dev)
    C2 = torch.empty(8192, 768, device=dev)
    ch_us = timed(lambda: bsg.bsgemm_i8_chain(Xm, W1, W2, True, False, out1=C1, out2=C2,
                                              dstatus=dstatus, workspace=cws))
    two_us = timed(lambda: bsg.bsgemm_i8(bsg.bsgemm_i8(Xm, W1, relu=True, out=C1, dstatus=dstatus,
                                                       workspace=uws1),
                                         W2, out=C2, dstatus=dstatus, workspace=uws2))
    rq_us = timed(lambda: bsg.bsgemm_i8_requant(Xm, W1, relu=True, dstatus=dstatus,
                                                workspace=cws))
    uq_us = timed(lambda: bsg.quantize_rows(bsg.bsgemm_i8(Xm, W1, relu=True, out=C1,
                                                          dstatus=dstatus, workspace=uws1),
                                            dstatus=dstatus))
    lines.append({"config": "f1 gpt2 mlp chain 8192x768 -> 3072 (ReLU) -> 768",
                  "chain_us": round(ch_us, 1), "two_units_us": round(two_us, 1),
                  "requant_us": round(rq_us, 1), "unit_then_quantize_rows_us": round(uq_us, 1)})
    del Xm, W1, W2, C1, C2, cws, uws1, uws2
    # the live audit (f2): 4096 seeded cells of a finished qkv unit, and the
    # init gate (probe + known answer + audit of 4096 cells), per call
    A, B, _ = inputs.gpt2_linear_inputs("qkv")
    A, B = A.to(dev), B.to(dev)
    Cq = bsg.bsgemm_i8(A, B)
    mism = torch.zeros(1, dtype=torch.int32, device=dev)
    a_us = timed(lambda: bsg.audit(A, B, Cq, nsamples=4096, mismatches=mism))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        bsg.selftest()
    st_ms = (time.perf_counter() - t0) / 5 * 1e3
    lines.append({"config": "f2 live audit, 4096 cells of qkv 8192x2304x768",
                  "audit_us": round(a_us, 1), "mismatches": int(mism.item()),
                  "selftest_ms_host": round(st_ms, 2)})
    del A, B, Cq
    # the weight storage (f4): codes and stored weights of a GPT-2 fc weight
    # and of an 8192 x 8192 one.  Bytes: the weight read once + codes written;
    # codes read + f32 written.
    for K, N in ((768, 3072), (8192, 8192)):
        Wt = inputs.gpt2_weights(K, N, 5).to(dev)
        for bits in (8, 4):
            cb = 1.0 if bits == 8 else 0.5
            q_us = timed(lambda: bsg.wquant_cols(Wt, bits=bits))
            Q, sc = bsg.wquant_cols(Wt, bits=bits)
            d_us = timed(lambda: bsg.wdequant_cols(Q, sc, N, bits=bits))
            qb = K * N * (4 + cb)
            db = K * N * (cb + 4)
            lines.append({"config": f"f4 weight storage int{bits} {K}x{N}",
                          "wquant_us": round(q_us, 2), "wquant_gbs": round(qb / q_us / 1e3, 1),
                          "wquant_frac_of_measured_hbm": round(qb / q_us / 1e3 / hbm_peak, 3),
                          "wdequant_us": round(d_us, 2), "wdequant_gbs": round(db / d_us / 1e3, 1),
                          "wdequant_frac_of_measured_hbm": round(db / d_us / 1e3 / hbm_peak, 3),
                          "bytes": "wquant: 4 B read + code bytes; wdequant: code bytes + 4 B"})
        del Wt
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
    for name, *_ in inputs.LARGE_GEMMS:
        A, B, relu = inputs.large_gemm_inputs(name)
        lines.append(unit_line("c4 " + name, A.to(dev), B.to(dev), relu))
        del A, B
        torch.cuda.empty_cache()
    lines.append(unit_line("c4 adversarial 4096^3", inputs.adversarial(4096, 4096, 11).to(dev),
                           inputs.adversarial(4096, 4096, 12, along_rows=False).to(dev)))
    torch.cuda.synchronize()
    if int(dstatus.item()) & ~1:  # the adversarial mix sets the non-finite bit by design
        raise RuntimeError(f"device status {int(dstatus.item())}")
    return lines


# -------------------------------------------------------------- CPU oracle
PARTS = ("sq4096", "sq8192", "sq16384", "ragged_adversarial", "probe")
CLOCK = time.perf_counter   # the oracle sample's clock (tests replace it)


def oracle_inputs():
    """The step's GEMM inputs for the oracle, generated once (the same seeded
    tensors the GPU arm uses): {name: (A, B, relu)} as numpy arrays."""
    from verifiable_quantize_rows_gb300 import inputs
    out = {}
    for name, *_ in inputs.LARGE_GEMMS:
        A, B, relu = inputs.large_gemm_inputs(name)
        out[name] = (A.numpy(), B.numpy(), relu)
    return out


class OracleSample:
    """Part `part` of the step on the oracle, on a sub-block: the first r
    rows of A and the first r columns of B (full K: every sampled output
    cell is computed exactly as in the full GEMM, scales included), or, for
    the probe, M = r rows (N = K = 1024, hash included)."""

    def __init__(self, orc, data):
        self.orc = orc
        self.data = data
        self.cache = {}

    def prepare(self, part, r):
        name = PARTS[part]
        if name == "probe" or (part, r) in self.cache:
            return
        A, B, relu = self.data[name]
        rr, cc = min(r, A.shape[0]), min(r, B.shape[1])
        self.cache[(part, r)] = (np.ascontiguousarray(A[:rr]), np.ascontiguousarray(B[:, :cc]),
                                 relu)

    def run(self, part, r):
        """Returns (ops, seconds) of one oracle call."""
        if PARTS[part] == "probe":
            t0 = CLOCK()
            self.orc.probe_hash(PROBE_SEED, r, PROBE[1], PROBE[2])
            return 2 * r * PROBE[1] * PROBE[2], CLOCK() - t0
        self.prepare(part, r)
        a, b, relu = self.cache[(part, r)]
        t0 = CLOCK()
        self.orc.bsgemm_i8(a, b, relu)
        return 2 * a.shape[0] * b.shape[1] * a.shape[1], CLOCK() - t0

    def sizes(self, seconds):
        """r per part for about `seconds` of oracle work each, scaled from a
        64-row calibration call (work grows as r^2 for the GEMMs)."""
        rows = []
        for part, name in enumerate(PARTS):
            _, t = self.run(part, 64)
            if name == "probe":
                r = int(64 * seconds / max(t, 1e-4))
                cap = PROBE[0]
            else:
                r = int(64 * (seconds / max(t, 1e-4)) ** 0.5)
                A, B, _ = self.data[name]
                cap = max(A.shape[0], B.shape[1])
            rows.append(max(8, min(cap, r)) // 8 * 8)
        return rows


def sample_text(rows):
    parts = [f"{n} on a {r}x{r} block of C (first rows of A, first columns of B, full K)"
             for n, r in zip(PARTS[:-1], rows[:-1])]
    return "; ".join(parts) + f"; the probe at M = {rows[-1]} of 1024 (N = K = 1024, hash included)"


def cpu_baseline(budget_s=15.0):
    import oracle
    orc = oracle.load()
    smp = OracleSample(orc, oracle_inputs())
    rows = smp.sizes(budget_s / len(PARTS))
    for part in range(len(PARTS)):
        smp.prepare(part, rows[part])
    total_ops, total_t, reps = 0, 0.0, 0
    while total_t < 0.8 * budget_s or reps == 0:
        for part in range(len(PARTS)):
            ops, t = smp.run(part, rows[part])
            total_ops, total_t = total_ops + ops, total_t + t
        reps += 1
    return {"value": round(total_ops / total_t / 1e12, 6), "unit": "TOPS",
            "cores": orc.num_threads(), "kind": "oracle",
            "sample": f"{sample_text(rows)}; {reps}x: {total_ops / 1e9:.1f} G ops in "
                      f"{total_t:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    if world > 1:
        # torchrun sets OMP_NUM_THREADS=1 for every rank; rank 0 runs the
        # oracle alone, on the host's cores as at N = 1 (read when the
        # oracle's OpenMP runtime loads, below)
        os.environ["OMP_NUM_THREADS"] = str(len(os.sched_getaffinity(0)))
    import oracle
    orc = oracle.load()
    smp = OracleSample(orc, oracle_inputs())
    # About two minutes of oracle work for the whole run, whatever K and W
    # are: step i runs part i mod 5 of the workload (the four GEMMs, the
    # probe), each on a sample sized to the per-step budget.
    total_budget = 120.0
    per_step = min(10.0, total_budget / max(1, args.steps + args.warmup))
    rows = smp.sizes(per_step)
    for part in range(len(PARTS)):
        smp.prepare(part, rows[part])
    n = len(PARTS)
    for i in range(args.warmup):
        smp.run(i % n, rows[i % n])
    total_ops, total_t = 0, 0.0
    for i in range(args.steps):
        ops, t = smp.run(i % n, rows[i % n])
        total_ops, total_t = total_ops + ops, total_t + t
    value = total_ops / total_t / 1e12
    ms = total_t / max(1, args.steps) * 1e3
    sample = (f"step i runs part i mod {n} of the step: {sample_text(rows)}; "
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


# -------------------------------------------------------------- single workloads
def run_single(args):
    """`--only small`: the GPT-2 linears step alone; `--unit M,N,K[,relu]`:
    one bsgemm_i8 of U(-1, 1) inputs, called --steps times after --warmup
    (CUDA events, L2 flushed before each call); `--wquant K,N[,bits]`: the
    weight-storage quantize of a seeded N(0, 0.02) weight, the same way.  One
    JSON line; used to run small cases under a profiler."""
    import torch
    import verifiable_quantize_rows_gb300 as bsg
    from verifiable_quantize_rows_gb300 import build as bsg_build
    from verifiable_quantize_rows_gb300 import inputs
    if not os.path.exists(bsg.LIB_PATH):
        bsg_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    lib = bsg.load()
    dstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    if args.only == "small":
        side = torch.cuda.Stream(device=dev)
        pws = bsg.Workspace(dev)
        pws.get(lib.bsg_probe_workspace_size(*PROBE))
        probe_out = torch.empty(32, dtype=torch.uint8, device=dev)
        W = Workload("small", dev, lib, side, dstatus, probe_out, pws, with_host=False)
        step_ms, stage_ms, launches = time_workload(W, args.steps, args.warmup, flush, stream,
                                                    lambda: None, stage_steps=20)
        ms = statistics.mean(step_ms)
        peaks, peak_kind = load_peaks()
        roof, quant, _ = summarize(W, step_ms, stage_ms, peaks, peak_kind, ms, 1,
                                   SMALL_GEMM_PROFILE)
        return {"workload": SMALL_WORKLOAD, "ms_per_step": round(ms, 4),
                "value": round(step_ops("small") / (ms * 1e-3) / 1e12, 3), "unit": "TOPS",
                "gemm_frac": roof["frac"], "gemm_ms": roof["per_gemm_ms"],
                "quantize_ms": quant["per_gemm_ms"],
                "gpu_launches": launches, "device_status": int(dstatus.item())}
    if args.wquant:
        parts = [int(v) for v in args.wquant.split(",")]
        K, N = parts[:2]
        bits = parts[2] if len(parts) > 2 else 8
        Wt = inputs.gpt2_weights(K, N, 5).to(dev)
        wws = bsg.Workspace(dev)
        for _ in range(args.warmup):
            bsg.wquant_cols(Wt, bits=bits, dstatus=dstatus, workspace=wws)
        ts = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            bsg.wquant_cols(Wt, bits=bits, dstatus=dstatus, workspace=wws)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts)
        return {"wquant": f"{K}x{N} int{bits}", "ms": round(ms, 4),
                "gbs": round(K * N * (4 + bits / 8) / (ms * 1e-3) / 1e9, 1),
                "device_status": int(dstatus.item())}
    parts = [int(v) for v in args.unit.split(",")]
    M, N, K = parts[:3]
    relu = bool(parts[3]) if len(parts) > 3 else False
    A = inputs.uniform((M, K), -1, 1, 1).to(dev)
    B = inputs.uniform((K, N), -1, 1, 2).to(dev)
    C = torch.empty(M, N, device=dev)
    ws = bsg.Workspace(dev)
    ws.get(lib.bsgemm_i8_workspace_size(M, N, K))
    for _ in range(args.warmup):
        bsg.bsgemm_i8(A, B, relu=relu, out=C, dstatus=dstatus, workspace=ws)
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bsg.bsgemm_i8(A, B, relu=relu, out=C, dstatus=dstatus, workspace=ws)
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    ms = statistics.median(ts)
    return {"unit": f"{M}x{N}x{K}", "relu": relu, "ms": round(ms, 4),
            "tops": round(2 * M * N * K / (ms * 1e-3) / 1e12, 2),
            "device_status": int(dstatus.item())}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["small"], default=None,
                    help="run the GPT-2 linears step alone (one JSON line)")
    ap.add_argument("--unit", default=None, metavar="M,N,K[,relu]",
                    help="time one bsgemm_i8 of this shape instead (one JSON line)")
    ap.add_argument("--wquant", default=None, metavar="K,N[,bits]",
                    help="time one weight-storage quantize of this shape instead (one JSON line)")
    ap.add_argument("--configs", action="store_true",
                    help="time the unit on every workload of the measurement plan instead "
                         "(one JSON line each)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local_rank = env_int("LOCAL_RANK", 0)

    if args.only or args.unit or args.wquant:
        print(json.dumps(run_single(args)), flush=True)
        return

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
        if not args.no_cpu_baseline and world == 1:   # the CPU baseline is an N = 1 figure
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
