"""Benchmark of the Mamba-2 SSD chunked forward on one or more GB300s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores

A step is one call of ``ssd_chunked_fwd`` (all four stages) on one batch of
the workload's synthetic inputs, resident in HBM.  Under torchrun every rank
runs its own batch of the same shape (independent (batch, head) slabs: no
collective), so ``value`` is the tokens of all ranks over the slowest rank's
time ("weak" scaling).  Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from state_space_model_gb300 import inputs as gen  # noqa: E402

METRIC = "SSD chunked-forward tokens/s at Mamba-2 2.7B layer shape; % of roofline"
L2_BYTES = 129 * 1024 * 1024


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# algorithmic work (compulsory HBM bytes, flops) of the path and of each step


def path_work(w):
    B, L, H, P, N, G, Q = (w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                           w.chunk_size)
    es = 2 if w.dtype == "bf16" else 4
    T = B * L
    rd = T * H * P * es + 2 * T * G * N * es + T * H * 4 + 2 * H * 4
    if w.init_states:
        rd += B * H * P * N * 4
    wr = T * H * P * es + B * H * P * N * 4
    flops = T * H * (2 * N * P + 2 * N * P + (Q + 1) * P + 2 * N * P / Q) + T * G * (Q + 1) * N
    return rd + wr, flops


def stage_bytes(w):
    """Bytes each step reads and writes once as a standalone kernel."""
    B, L, H, P, N, G, Q = (w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups,
                           w.chunk_size)
    es = 2 if w.dtype == "bf16" else 4
    nc = -(-L // Q)
    T = B * L
    x, bc, dt = T * H * P * es, T * G * N * es, T * H * 4
    g = B * H * nc * Q * 4
    s = B * nc * H * P * N * 4
    hp = B * nc * H * P * N * es
    fin = B * H * P * N * 4
    h0 = fin if w.init_states else 0
    return {
        "chunk_cumsum": dt + g,
        "chunk_state": x + bc + dt + g + s,
        "state_passing": s + B * H * nc * 4 + h0 + hp + fin,
        "chunk_scan": x + dt + g + 2 * bc + hp + x,
    }


# ---------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.idx)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t_on and self.t_on - 0.15 <= r[0] <= self.t_off + 0.15]
        use = inside if len(inside) >= 3 else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for name, v in zip(names, r[3][1:5]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in use),
                "sm_max_mhz": max(r[2] for r in use), "reasons": sorted(reasons),
                "samples": len(use),
                "window": "timed region" if use is inside else "whole run (timed region too short)"}


# ---------------------------------------------------------------------------
# traffic from a committed ncu summary, valid only for the kernel source it was taken on


# the sources each recorded kernel is built from (a change elsewhere leaves
# its DRAM traffic record valid)
KERNEL_SOURCES = {   # each kernel's translation unit and the headers it includes
    "k_ssd_fused": ["ssd_fused.cu", "ssd_block_math.cuh", "ptx_sm100.cuh", "ssd_tc.cuh",
                    "ssd_tmap.h", "ssd_internal.h", "ssd_common.h"],
    "k_ssd_pair": ["ssd_pair.cu", "ssd_block_math.cuh", "ptx_sm100.cuh", "ssd_tc.cuh",
                   "ssd_tmap.h", "ssd_internal.h", "ssd_common.h"],
    "k_ssu_tokens": ["ssd_ssu.cu", "ptx_sm100.cuh", "ssd_decode.h", "ssd_common.h"],
    "k_conv_prologue": ["ssd_mixer.cu", "ssd_mixer.h", "ssd_common.h"],
}


def code_tokens(src: str) -> str:
    """C/C++/CUDA source with its comments removed and every run of
    whitespace outside string and character literals collapsed to one space,
    so that editing a comment or re-indenting leaves the result unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c == "/" and src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif c == "/" and src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            if out and out[-1] != " ":
                out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif c.isspace():
            while i < n and src[i].isspace():
                i += 1
            if out and out[-1] != " ":
                out.append(" ")
        else:
            out.append(c)
            i += 1
    return "".join(out).strip()


def kernel_source_hash(stage: str) -> str:
    """Hash of the code (comments and layout ignored) of the files a kernel
    is built from: a recorded DRAM traffic figure stays valid while it holds."""
    csrc = os.path.join(ROOT, "state_space_model_gb300", "csrc")
    names = KERNEL_SOURCES.get(stage) or sorted(
        n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(stage: str, workload: str):
    """Per-launch dram read+write bytes recorded in profiles/traffic.txt as
    `stage workload source_hash bytes`; None if absent or taken on other source."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    want = kernel_source_hash(stage)
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and parts[0] == stage and parts[1] == workload and \
                    parts[2] == want:
                return float(parts[3])
    return None


# ---------------------------------------------------------------------------


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if (torch.cuda.is_available() and args.impl == "ours") else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, w, world, rank):
    """The fp64 oracle on the host cores: each step a bounded sample of the
    workload's (batch, head) slabs; value = equivalent tokens/s."""
    if rank != 0:
        return
    from oracle import oracle as orc
    inp = gen.make_inputs(w)
    cores = orc.max_threads()
    slabs_all = [(b, h) for b in range(w.batch) for h in range(w.nheads)]
    t0 = time.perf_counter()
    orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                   inp["initial_states"], ngroups=w.ngroups, slabs=slabs_all[:cores])
    per_slab = max((time.perf_counter() - t0) / cores, 1e-4)  # wall per slab at full width
    budget = args.ref_seconds / max(args.steps + args.warmup, 1)
    n = int(max(1, min(len(slabs_all), budget / per_slab)))
    sample = slabs_all[:n]
    step = lambda: orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                                  inp["initial_states"], ngroups=w.ngroups, slabs=sample)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    tokens = n * w.seqlen / w.nheads  # a token is all heads of one position
    value = tokens / dt
    desc = f"{n} of {len(slabs_all)} (batch, head) slabs x {w.seqlen} tokens per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen,
                       "nheads": w.nheads, "headdim": w.headdim, "dstate": w.dstate,
                       "ngroups": w.ngroups, "chunk_size": w.chunk_size},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(w, inp):
    from oracle import oracle as orc
    cores = orc.max_threads()
    slabs_all = [(b, h) for b in range(w.batch) for h in range(w.nheads)]
    # about 10-30 s of CPU work: estimate from a probe of one slab per core
    t0 = time.perf_counter()
    orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                   inp["initial_states"], ngroups=w.ngroups, slabs=slabs_all[:cores])
    per_slab_cpu = (time.perf_counter() - t0)  # core-seconds per slab ~ wall of the probe
    n = int(max(1, min(len(slabs_all), 20.0 / max(per_slab_cpu, 1e-4))))
    sample = slabs_all[:n]
    t0 = time.perf_counter()
    orc.recurrence(inp["x"], inp["dt"], inp["A"], inp["B"], inp["C"], inp["D"],
                   inp["initial_states"], ngroups=w.ngroups, slabs=sample)
    dt = time.perf_counter() - t0
    return {"value": n * w.seqlen / w.nheads / dt, "unit": "tokens/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} of {len(slabs_all)} (batch, head) slabs x {w.seqlen} tokens "
                      f"({dt:.1f} s wall)"}


SSU_METRIC = "SSU decode tokens/s at the Nemotron hybrid layer shape; % of HBM roofline"


def ssu_bytes(Bn, H, P, N, G, T=1, cached=False, state_bytes=4):
    """Compulsory HBM bytes of one decode call of T tokens: the state (fp32, or
    bf16 with state_bytes = 2) read and written once, the per-token state cache
    written when kept, and per token x, z and out (bf16), B and C (bf16), dt
    (f32); plus A, D, dt_bias."""
    sb = state_bytes
    return 2 * Bn * H * P * N * sb + (T * Bn * H * P * N * sb if cached else 0) + \
        T * (3 * Bn * H * P * 2 + 2 * Bn * G * N * 2 + Bn * H * 4) + 3 * H * 4


def run_ssu(args, world, rank, local):
    """One decode call per timed iteration, state updated in place (so the
    state carried from step to step is real): ssd_state_update, or with
    --tokens T > 1 ssd_state_update_tokens over T tokens per sequence keeping
    the per-token state cache (the verification pass of speculative decoding
    with T draft tokens)."""
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    from state_space_model_gb300 import build, ssd
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sh = dict(gen.SSU_SHAPE)
    if args.batch is not None:
        sh["batch"] = args.batch
    Bn, H, P, N, G = sh["batch"], sh["nheads"], sh["headdim"], sh["dstate"], sh["ngroups"]
    T = args.tokens
    cpu = gen.make_ssu_inputs(Bn, H, P, N, G, seed=20270 + rank, tokens=T if T > 1 else None)
    sdt = torch.bfloat16 if args.state_dtype == "bf16" else torch.float32
    sbytes = 2 if args.state_dtype == "bf16" else 4
    cpu["state"] = cpu["state"].to(sdt)
    d = {k: (None if v is None else v.to(dev)) for k, v in cpu.items()}
    # the state must not stay in L2 from one call to the next: calls rotate over
    # nbuf state buffers (other sequences' states) holding together at least
    # twice L2
    sbytes_all = Bn * H * P * N * sbytes
    nbuf = min(8, max(1, -(-2 * L2_BYTES // sbytes_all)))
    states = [d["state"]] + [d["state"].clone() for _ in range(nbuf - 1)]
    if T > 1:
        out = torch.empty((Bn, T, H, P), dtype=torch.bfloat16, device=dev)
        inter = torch.empty((Bn, T, H, P, N), dtype=sdt, device=dev)

        def call(st):
            ssd.state_update_tokens(st, d["x"], d["dt"], d["A"], d["B"], d["C"],
                                    D=d["D"], z=d["z"], dt_bias=d["dt_bias"], dt_softplus=True,
                                    ngroups=G, intermediate_states=inter, out=out)
    else:
        out = torch.empty((Bn, H, P), dtype=torch.bfloat16, device=dev)

        def call(st):
            ssd.state_update(st, d["x"], d["dt"], d["A"], d["B"], d["C"], D=d["D"],
                             z=d["z"], dt_bias=d["dt_bias"], dt_softplus=True, ngroups=G,
                             out=out)

    def step():
        for st in states:
            call(st)

    # a decode step is a few microseconds of GPU work at small batch, less than
    # the Python call that launches it: replay it from a CUDA graph, as a
    # serving loop does, so the timed region holds GPU work and launch gaps only
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_on()
    ev0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / (args.steps * nbuf), world)   # per call
    clk = clocks.stop()
    pk = peaks()
    nbytes = ssu_bytes(Bn, H, P, N, G, T, cached=T > 1, state_bytes=sbytes)
    wname = "ssu_decode" if T == 1 else f"ssu_decode_{T}_tokens"
    if Bn != gen.SSU_SHAPE["batch"]:
        wname += f"_b{Bn}"
    if sbytes == 2:
        wname += "_bf16_state"
    achieved = nbytes / (ms / 1e3) / 1e9
    if rank == 0:
        line = {
            "metric": SSU_METRIC, "value": world * Bn * T / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; see state_space_model_gb300/inputs.py)",
            "config": {"workload": wname, "state_dtype": args.state_dtype,
                       "batch": Bn, "tokens": T, "nheads": H, "headdim": P,
                       "dstate": N, "ngroups": G, "gated": True, "dt_softplus": True,
                       "state_cache": T > 1,
                       "l2": f"calls rotate over {nbuf} state buffer(s) of "
                             f"{sbytes_all / 1e6:.0f} MB, {nbuf * sbytes_all / 1e6:.0f} MB "
                             f"together, at least twice L2"},
            "roofline": {"bound": "hbm", "kernel": "k_ssu_tokens", "achieved": achieved,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                         "traffic": recorded_traffic("k_ssu_tokens", wname),
                         "algorithmic_bytes": nbytes, "kernel_ms": ms,
                         "peak_source": pk["source"]},
            "gpu_launches": args.steps * nbuf,
            "launch": f"CUDA graph replay of {nbuf} call(s), one kernel per call; "
                      "ms_per_step is per call",
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)


PROLOGUE_METRIC = ("mixer prologue (conv1d + SiLU + x/B/C split + dt softplus) tokens/s at "
                   "Mamba-2 2.7B layer shape; % of HBM roofline")


def prologue_bytes(Bn, L, H, P, G, N, W, es=2):
    """Compulsory HBM bytes of one prologue call: xBC read and x, B, C written
    (es bytes each), raw dt read and dt' written (f32), the conv state read and
    written, the conv weights and biases, dt_bias."""
    Dc = H * P + 2 * G * N
    return 2 * Bn * L * Dc * es + 2 * Bn * L * H * 4 + 2 * Bn * Dc * W * es + Dc * (W + 1) * 4 \
        + H * 4


def run_prologue(args, world, rank, local):
    """One ssd_mixer_prologue call per timed iteration on the Mamba-2 2.7B mixer
    shape (d_inner 5120 = 80 heads x 64, one group of 128 states, width-4
    convolution), conv state carried in place."""
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    from state_space_model_gb300 import build, ssd
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    w = gen.WORKLOADS[args.workload]
    Bn = args.batch if args.batch is not None else w.batch
    L, H, P, G, N, W = w.seqlen, w.nheads, w.headdim, w.ngroups, w.dstate, 4
    cpu = gen.make_prologue_inputs(Bn, L, H, P, G, N, W, seed=20280 + rank)
    d = {k: v.to(dev) for k, v in cpu.items()}
    outs = (torch.empty((Bn, L, H, P), dtype=torch.bfloat16, device=dev),
            torch.empty((Bn, L, G, N), dtype=torch.bfloat16, device=dev),
            torch.empty((Bn, L, G, N), dtype=torch.bfloat16, device=dev),
            torch.empty((Bn, L, H), dtype=torch.float32, device=dev))

    def step():
        ssd.mixer_prologue(d["xBC"], d["conv_weight"], d["dt"], H, P, G, N,
                           conv_bias=d["conv_bias"], conv_state=d["conv_state"],
                           dt_bias=d["dt_bias"], dt_softplus=True, out=outs)

    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark_on()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    clk = clocks.stop()
    pk = peaks()
    nbytes = prologue_bytes(Bn, L, H, P, G, N, W)
    achieved = nbytes / (ms / 1e3) / 1e9
    in_bytes = Bn * L * (H * P + 2 * G * N) * 2
    if rank == 0:
        line = {
            "metric": PROLOGUE_METRIC, "value": world * Bn * L / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; see state_space_model_gb300/inputs.py)",
            "config": {"workload": f"prologue_{w.name}", "batch": Bn, "seqlen": L, "nheads": H,
                       "headdim": P, "ngroups": G, "dstate": N, "conv_width": W,
                       "conv_state": True, "dt_softplus": True,
                       "l2": f"xBC {in_bytes / 1e6:.0f} MB, larger than L2"
                       if in_bytes > L2_BYTES else "xBC smaller than L2"},
            "roofline": {"bound": "hbm", "kernel": "k_conv_prologue", "achieved": achieved,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                         "traffic": recorded_traffic("k_conv_prologue", f"prologue_{w.name}"),
                         "algorithmic_bytes": nbytes, "kernel_ms": ms,
                         "peak_source": pk["source"]},
            "gpu_launches": 2 * args.steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["prefill", "ssu", "prologue"], default="prefill",
                    help="prefill: ssd_chunked_fwd (the headline); ssu: one decode step; "
                         "prologue: ssd_mixer_prologue on the workload's mixer shape")
    ap.add_argument("--workload", default=gen.HEADLINE, choices=sorted(gen.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--gate", action="store_true",
                    help="prefill: gate the output, y * silu(z) (ssd_chunked_fwd_gated)")
    ap.add_argument("--tokens", type=int, default=1,
                    help="--op ssu: decode tokens per sequence and call (T > 1 keeps the "
                         "per-token state cache)")
    ap.add_argument("--state-dtype", choices=["f32", "bf16"], default="f32",
                    help="--op ssu: dtype the decode state is kept in")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (a smaller case of the same shape)")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="wall-time budget of the whole --impl reference run")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = gen.WORKLOADS[args.workload]
    if args.batch is not None:
        w = w.with_(batch=args.batch)
    world, rank, local = dist_setup(args)

    if args.impl == "reference":
        run_reference(args, w, world, rank)
        return
    if args.op in ("ssu", "prologue"):
        (run_ssu if args.op == "ssu" else run_prologue)(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the CUDA path has no CPU fallback)")
    from state_space_model_gb300 import build, ssd
    build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    inp_cpu = gen.make_inputs(w, seed=w.seed + rank)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp_cpu.items()}
    B, L, H, P, N = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate
    y = torch.empty((B, L, H, P), dtype=w.torch_dtype, device=dev)
    fin = torch.empty((B, H, P, N), dtype=torch.float32, device=dev)
    ws = torch.empty(ssd.workspace_size(B, L, H, P, N, w.ngroups, w.chunk_size, w.torch_dtype),
                     dtype=torch.uint8, device=dev)
    # --gate: the mixer's output gate fused in, y * silu(z) (z ~ N(0, 1), dtype of x)
    z = (torch.randn((B, L, H, P), generator=torch.Generator().manual_seed(w.seed + 7 + rank))
         .to(w.torch_dtype).to(dev) if args.gate else None)
    z_bytes = 0 if z is None else z.numel() * z.element_size()

    def step():
        ssd.chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["D"], d["initial_states"],
                        w.chunk_size, w.ngroups, y=y, final_states=fin, workspace=ws, z=z)

    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local)
    clocks.start()
    # inputs that fit in L2 would be re-read from it: then every timed step gets
    # its own events and a write of twice L2 runs before it, outside the timing
    in_bytes = sum(v.numel() * v.element_size() for v in inp_cpu.values() if v is not None)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) \
        if in_bytes <= L2_BYTES else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark_on()
    if flush is None:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1) / args.steps
        # the spread: steps timed one by one (each its own event pair, back to
        # back, no flush: the inputs exceed L2), after the timed window
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(50, min(args.steps, 200)))]
        for ea, eb in evs:
            ea.record(stream)
            step()
            eb.record(stream)
        torch.cuda.synchronize()
        per_step = sorted(ea.elapsed_time(eb) for ea, eb in evs)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i, (ea, eb) in enumerate(evs):
            flush.fill_(i & 255)
            ea.record(stream)
            step()
            eb.record(stream)
        torch.cuda.synchronize()
        per_step = sorted(ea.elapsed_time(eb) for ea, eb in evs)
        ms = sum(per_step) / args.steps
    clocks.mark_off()
    q = lambda f: per_step[min(len(per_step) - 1, int(f * len(per_step)))]
    step_stats = {"median_ms": statistics.median(per_step), "p10_ms": q(0.1), "p90_ms": q(0.9),
                  "min_ms": per_step[0], "max_ms": per_step[-1], "n": len(per_step),
                  "how": ("each step its own event pair after a write of twice L2"
                          if flush is not None else
                          "each step its own event pair, back to back, after the timed window")}
    barrier(world)
    torch.cuda.synchronize()
    ms = max_over_ranks(ms, world)
    clk = clocks.stop()
    tokens = B * L
    value = world * tokens / (ms / 1e3)

    plan = ssd.describe_plan(B, L, H, P, N, w.ngroups, w.chunk_size, w.torch_dtype)
    fused = plan.startswith("fused")
    reps = max(10, min(args.steps, 200))
    sb = stage_bytes(w)
    if args.gate and not fused:
        raise SystemExit("bench.py: --gate times the fused plan; this workload runs four steps")
    # launches per step: the fused kernel, plus its states-only pass and the
    # combine when the plan splits the last partial wave by sequence
    split = "segments" in plan
    launches = (3 if split else 1) if fused else 4
    if fused:
        # the step's launches back to back: their total is the timed region's
        # (events on the launching stream); the dominant kernel's figures below
        # are charged the whole step (gated: the gate pass too)
        kname = "k_ssd_pair" if "k_ssd_pair" in plan else "k_ssd_fused"
        if split:
            kname += " (+ states-only pass + combine)"
        if args.gate:
            kname += " + k_gate"
        kstats = {kname: ms}
        sb[kname] = path_work(w)[0] + z_bytes
    else:
        # the four stage entry points, events between them
        nc = -(-L // w.chunk_size)
        G = torch.empty((B, H, nc * w.chunk_size), dtype=torch.float32, device=dev)
        S = torch.empty((B, nc, H, P, N), dtype=torch.float32, device=dev)
        hp = torch.empty((B, nc, H, P, N), dtype=w.torch_dtype, device=dev)
        kstats = {k: 0.0 for k in ("chunk_cumsum", "chunk_state", "state_passing", "chunk_scan")}
        for it in range(reps + 3):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            if flush is not None:
                flush.fill_(it & 255)
            evs[0].record(stream)
            ssd.chunk_cumsum(d["dt"], d["A"], w.chunk_size, out=G)
            evs[1].record(stream)
            ssd.chunk_state(d["x"], d["B"], d["dt"], G, w.chunk_size, w.ngroups, out=S)
            evs[2].record(stream)
            ssd.state_passing(S, G, d["initial_states"], w.chunk_size, out=(hp, fin))
            evs[3].record(stream)
            ssd.chunk_scan(d["x"], d["dt"], G, d["B"], d["C"], d["D"], hp, w.chunk_size,
                           w.ngroups, out=y)
            evs[4].record(stream)
            torch.cuda.synchronize()
            if it >= 3:
                for i, k in enumerate(kstats):
                    kstats[k] += evs[i].elapsed_time(evs[i + 1]) / reps
    dom = max(kstats, key=kstats.get)
    pk = peaks()
    achieved = sb[dom] / (kstats[dom] / 1e3) / 1e9
    # recorded per step: every launch of the step (the dominant kernel's name
    # is the record's key)
    traffic = recorded_traffic(dom.split()[0], w.name)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                "algorithmic_bytes": sb[dom], "kernel_ms": kstats[dom],
                "peak_source": pk["source"],
                "kernel_ms_all": {k: round(v, 4) for k, v in kstats.items()}}
    pbytes, pflops = path_work(w)
    pbytes += z_bytes
    t_roof = max(pbytes / (pk["hbm_gbs"] * 1e9), pflops / (pk["bf16_tflops"] * 1e12))
    path_roof = {"t_roof_us": t_roof * 1e6, "t_step_us": ms * 1e3,
                 "frac": t_roof / (ms / 1e3), "bytes": pbytes, "flops": pflops,
                 "peak_source": pk["source"]}

    # end to end: pinned host inputs -> device, the call, results -> pinned host
    e2e = None
    if not args.no_e2e and not args.gate:   # (the gated line is a kernel measurement)
        host = {k: (None if v is None else v.pin_memory()) for k, v in inp_cpu.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = y.numel() * y.element_size() + fin.numel() * fin.element_size()

        # Every step uploads its inputs, runs the forward and downloads y and
        # final_states.  The batch goes through in up to eight chunks on three
        # streams -- uploads, scans, downloads, joined by events -- so chunk
        # i + 1's upload, chunk i's scan and chunk i - 1's download run at
        # once; and consecutive steps use two sets of device and host buffers,
        # so step j + 1's uploads run under step j's downloads (the host link
        # carries both directions at once and bounds this measurement).
        nch = min(B, 8)
        cuts = [(B * i) // nch for i in range(nch + 1)]
        s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        per_batch = [k for k, v in host.items() if v is not None and v.dim() > 1]
        shared = [k for k, v in host.items() if v is not None and v.dim() <= 1]
        bmax = max(cuts[i + 1] - cuts[i] for i in range(nch))
        ws_e2e = torch.empty(max(1, ssd.workspace_size(bmax, L, H, P, N, w.ngroups, w.chunk_size,
                                                       w.torch_dtype)),
                             dtype=torch.uint8, device=dev)
        sets = []
        for j in range(2):
            dj = d if j == 0 else {k: (None if v is None else torch.empty_like(v))
                                   for k, v in d.items()}
            sets.append((dj, y if j == 0 else torch.empty_like(y),
                         fin if j == 0 else torch.empty_like(fin),
                         torch.empty(y.shape, dtype=y.dtype, pin_memory=True),
                         torch.empty(fin.shape, dtype=fin.dtype, pin_memory=True)))
        ev_in = [torch.cuda.Event() for _ in range(nch)]
        ev_run = [torch.cuda.Event() for _ in range(nch)]
        # per buffer set: its inputs consumed by its last scans, its outputs read back
        ev_scanned = [torch.cuda.Event() for _ in range(2)]
        ev_read = [torch.cuda.Event() for _ in range(2)]
        for ev in ev_scanned + ev_read:
            ev.record(stream)

        def e2e_step(j):
            dj, yj, fj, y_h, f_h = sets[j & 1]
            s_in.wait_event(ev_scanned[j & 1])     # step j - 2's scans read these inputs
            with torch.cuda.stream(s_in):
                for k in shared:
                    dj[k].copy_(host[k], non_blocking=True)
                for i in range(nch):
                    b0, b1 = cuts[i], cuts[i + 1]
                    for k in per_batch:
                        dj[k][b0:b1].copy_(host[k][b0:b1], non_blocking=True)
                    ev_in[i].record(s_in)
            s_run.wait_event(ev_read[j & 1])       # step j - 2's downloads read these outputs
            with torch.cuda.stream(s_run):
                for i in range(nch):
                    b0, b1 = cuts[i], cuts[i + 1]
                    s_run.wait_event(ev_in[i])
                    ssd.chunked_fwd(dj["x"][b0:b1], dj["dt"][b0:b1], dj["A"], dj["B"][b0:b1],
                                    dj["C"][b0:b1], dj["D"],
                                    None if dj["initial_states"] is None
                                    else dj["initial_states"][b0:b1],
                                    w.chunk_size, w.ngroups, y=yj[b0:b1],
                                    final_states=fj[b0:b1], workspace=ws_e2e)
                    ev_run[i].record(s_run)
                ev_scanned[j & 1].record(s_run)
            with torch.cuda.stream(s_out):
                for i in range(nch):
                    b0, b1 = cuts[i], cuts[i + 1]
                    s_out.wait_event(ev_run[i])
                    y_h[b0:b1].copy_(yj[b0:b1], non_blocking=True)
                    f_h[b0:b1].copy_(fj[b0:b1], non_blocking=True)
                ev_read[j & 1].record(s_out)

        def e2e_run(nsteps):
            for sd in (s_in, s_run, s_out):
                sd.wait_stream(stream)
            for j in range(nsteps):
                e2e_step(j)
            stream.wait_stream(s_out)   # the downloads wait on every scan, the scans on every upload

        k_e2e = max(10, min(args.steps, 200))
        e2e_run(3)
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_run(k_e2e)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ems = max_over_ranks(e0.elapsed_time(e1) / k_e2e, world)
        e2e = {"value": world * tokens / (ems / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k_e2e,
               "ms_per_step": ems,
               "pipelining": f"{nch} batch chunks through upload, scan and download streams; "
                             "two buffer sets, so a step's uploads overlap the previous "
                             "step's downloads"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp_cpu)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded; see state_space_model_gb300/inputs.py)",
            "config": {"workload": w.name, "batch": B, "seqlen": L, "nheads": H, "headdim": P,
                       "dstate": N, "ngroups": w.ngroups, "chunk_size": w.chunk_size,
                       "initial_states": w.init_states, "parallelism": f"replicas{world}",
                       **({"gate": "y * silu(z), a second pass after the fused kernel"}
                          if args.gate else {}),
                       "l2": (f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > "
                              f"{L2_BYTES / 1e6:.0f} MB), no flush")
                       if flush is None else
                       (f"inputs {in_bytes / 1e6:.1f} MB fit in L2: a {2 * L2_BYTES / 1e6:.0f} "
                        f"MB write before each timed step, steps timed one by one")},
            "roofline": roofline, "path_roofline": path_roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (launches + (1 if args.gate else 0)) * args.steps,
            "step_ms": step_stats,
            "plan": plan, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
