#!/usr/bin/env python
"""MoE-layer forward throughput on B300 (tokens/s), with roofline fractions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload clip] [--impl ours|reference]

One step = one forward pass of the whole layer (routing, sorting, both expert
GEMMs, combine) over one batch of synthetic tokens resident in HBM: one call
of libmoe's moe_forward (C ABI).  The stage breakdown comes from the same
sequence run as separate calls with CUDA events between the stages.  The default workload is the full 10 s preview clip
(T=107520 tokens, d=4096, E=128 experts, inter=1024, top-6, 12x256 latent
routing, Zipf(1.2)-skewed router bias).  For N > 1 (torchrun) every rank
runs its own clip on its own GPU with no exchange (token sharding needs
none): weak scaling, value = tokens over all ranks / max-over-ranks time.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on
a bounded token sample per step (rank 0 only).
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
import tempfile
import time
from dataclasses import replace
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import moe_inputs as mi  # noqa: E402

METRIC = "MoE-layer tokens/sec on 1 B300; grouped-GEMM % bf16 TC peak; permute GB/s"
KERNELS_PER_STEP = 8  # 2 router GEMMs, 3 sorting kernels, 2 expert GEMMs, combine
GEMM_SOURCES = ["gemm_tc.cuh", "epilogues.cuh", "ptx.cuh", "gemm_launch.cu"]
WARMUP_S = 1.0                 # at least this much untimed layer work before the timed region
NOMINAL_BF16_TFLOPS = 2250.0   # B300 dense bf16 at its maximum SM clock
NOMINAL_SM_MHZ = 2032.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="clip", choices=mi.CONFIG_ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=512, help="tokens in the CPU-oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--variant", choices=["headlocal", "ext"], default=None,
                    help="time one widened variant alone (its JSON entry only; for profiling)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def rank_workload(cfg, rank: int):
    """Token sharding: rank r runs its own batch of the workload (seed + r for
    x, shared weights), so per-GPU work is fixed as N grows."""
    return replace(cfg, seed=cfg.seed + rank)


def max_over_ranks(v: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity when world == 1)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def throughput(tokens_per_rank: int, world: int, steps: int, max_elapsed_s: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank * steps / max_elapsed_s


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        j = json.loads(p.read_text())
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


def workload_str(cfg) -> str:
    extra = {"zipf": f", Zipf({cfg.zipf_s}) router bias"}.get(cfg.bias, "")
    if cfg.router_init == "uniform":
        extra += ", uniform router init"
    if cfg.modality_split:
        extra += ", video|text|audio x scales " + "/".join(str(s) for _, s in cfg.modality_split)
    return (f"{cfg.name}: T={cfg.T}, d={cfg.d}, E={cfg.E}, inter={cfg.inter}, top-{cfg.top_k}, "
            f"{cfg.n_heads}x{cfg.head_dim} latent routing{extra}")


def algorithmic(cfg) -> dict:
    """Algorithmic flops and bytes per step (routed rows only, no tile padding)."""
    T, d, E, I, k, L = cfg.T, cfg.d, cfg.E, cfg.inter, cfg.top_k, cfg.L
    Tk = T * k
    return dict(
        router_flops=2 * T * d * L + 2 * T * (2 * L) * E,     # latent GEMM + hi/lo score GEMM
        gemm1_flops=2 * Tk * d * 2 * I,
        gemm2_flops=2 * Tk * I * d,
        permute_bytes=T * d * 2 + Tk * d * 2,                 # read x once, write x_perm
        combine_bytes=Tk * d * 2 + Tk * 8 + T * d * 2,        # read y rows + idx/gates, write out
    )


class Clocks:
    """nvidia-smi sampler for the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.f.flush()
        rows = [ln.split(",") for ln in Path(self.f.name).read_text().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(pw) if pw else None}


def gemm_src_hash() -> str:
    """Hash of the GEMM engine's code (comments and blank lines left out), so
    that a traffic capture stays attached to the kernel it measured."""
    h = hashlib.sha256()
    for n in GEMM_SOURCES:
        for line in (ROOT / "fine_grained_moe_02_b300" / "csrc" / n).read_text().splitlines():
            code = line.split("//", 1)[0].rstrip() if not line.lstrip().startswith("#include") else line.rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """Per-launch DRAM bytes of expert GEMM-1 from the committed ncu summary, if
    the kernel sources still match the ones it was captured from."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None, "no ncu capture"
    j = json.loads(p.read_text())
    ent = j.get(workload)
    if not ent:
        return None, "no ncu capture for this workload"
    if ent.get("src_hash") != gemm_src_hash():
        return None, "kernel changed since the ncu capture"
    return ent["dram_bytes_per_launch"], ent.get("note", "")


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------

def oracle_step(inp, tokens, widened):
    from oracle import moe_oracle as O
    cfg = inp["cfg"]
    x = O.widen_bf16(inp["x"][tokens])
    if widened is not None:
        return O.forward(x, widened["w_lat"], widened["w_head"], inp["bias"], widened["w_gate"],
                         widened["w_up"], widened["w_down"], cfg.n_heads, cfg.head_dim, cfg.top_k)
    return O.forward(x, O.widen_bf16(inp["w_lat"]), O.widen_bf16(inp["w_head"]), inp["bias"], inp["w_gate"],
                     inp["w_up"], inp["w_down"], cfg.n_heads, cfg.head_dim, cfg.top_k,
                     widen_experts=O.widen_bf16)


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else os.cpu_count()
    except Exception:  # noqa: BLE001
        return os.cpu_count()


def cpu_baseline(inp, n_tokens: int) -> dict:
    """The oracle as it stands on a bounded token sample (full weights)."""
    cfg = inp["cfg"]
    tokens = mi.sample_tokens(cfg.T, n_tokens, seed=7)
    t0 = time.perf_counter()
    oracle_step(inp, tokens, None)
    dt = time.perf_counter() - t0
    return {"value": len(tokens) / dt, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{len(tokens)} seeded tokens of the {cfg.name} workload, full weights, one fp64 "
                      f"forward incl. per-expert bf16->fp64 widening ({dt:.1f} s)"}


def host_available_bytes() -> int:
    """Host memory available to this process, from /proc/meminfo (MemAvailable),
    else free pages from sysconf; 0 if neither can be read (the oracle then
    widens the weights per step instead of once)."""
    try:
        for line in Path("/proc/meminfo").read_text().splitlines():
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    try:
        return os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


def run_reference(args, rank, world):
    if rank != 0:
        return
    from oracle import moe_oracle as O
    cfg = mi.CONFIGS[args.workload]
    inp = mi.make_inputs(cfg)
    weight_bytes_f64 = 8 * (inp["w_gate"].size + inp["w_up"].size + inp["w_down"].size)
    widened = None
    if host_available_bytes() > 2.5 * weight_bytes_f64:
        widened = {k: O.widen_bf16(inp[k]) for k in ("w_lat", "w_head", "w_gate", "w_up", "w_down")}
    per_step = max(16, min(256, 4096 // max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        oracle_step(inp, mi.sample_tokens(cfg.T, per_step, seed=1000 + i), widened)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(inp, mi.sample_tokens(cfg.T, per_step, seed=i), widened)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    sample = (f"{per_step} seeded tokens of the {cfg.name} workload per step, full weights"
              + (" (pre-widened to fp64 once, untimed)" if widened is not None else ", widened per step"))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_str(cfg)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def measure_headlocal_variant(torch, moe, steps: int, name: str = "headlocal") -> dict:
    """moe_forward_headlocal on a head-local workload (default: 12 x 256 head
    slices, 256 experts per head, top-6 per head)."""
    cfg = mi.CONFIGS[name]
    inp = mi.make_inputs(cfg)

    def up(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()

    dims = moe.moe_dims.make(cfg.T, cfg.d, cfg.E, cfg.inter, cfg.top_k, cfg.n_heads, cfg.head_dim)
    x, w_router, w_down = up(inp["x"]), up(inp["w_router"]), up(inp["w_down"])
    w13 = torch.empty((cfg.n_heads, cfg.E, 2 * cfg.inter, cfg.head_dim), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_weights_headlocal(dims, up(inp["w_gate"]), up(inp["w_up"]), w13)
    ws = moe.alloc_workspace(moe.moe_workspace_size_headlocal(dims))
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        moe.moe_forward_headlocal(dims, x, w_router, None, w13, w_down, out, None, None, ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        moe.moe_forward_headlocal(dims, x, w_router, None, w13, w_down, out, None, None, ws)
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status set by moe_forward_headlocal")
    ms = e0.elapsed_time(e1) / steps
    flops = cfg.T * cfg.n_heads * (2 * cfg.head_dim * cfg.E + 6 * cfg.top_k * cfg.head_dim * cfg.inter)
    # every head-local expert's weights are streamed once for few rows each;
    # the fused expert kernel gathers x's head slices on chip and keeps act
    # there, so of the intermediates only y_perm goes out and back
    H, Dh, E, I, T = cfg.n_heads, cfg.head_dim, cfg.E, cfg.inter, cfg.T
    Tk = T * cfg.top_k
    alg_bytes = (2 * T * cfg.d * 2 + H * E * Dh * 2          # x (router, expert gather), router weights
                 + H * Tk * 8                                 # indices + gates
                 + H * E * (2 * I * Dh + Dh * I) * 2          # expert weights
                 + 2 * H * Tk * Dh * 2 + T * cfg.d * 2)       # y_perm written and read, out
    # the method's own bytes: x read once, router and expert weights, out written
    essential = T * cfg.d * 2 + H * E * Dh * 2 + H * E * (2 * I * Dh + Dh * I) * 2 + T * cfg.d * 2
    hbm = peaks()["hbm"]
    return {"workload": cfg.note, "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "layer_tflops": flops / (ms * 1e-3) / 1e12,
            "essential_bytes": essential, "essential_gbs": essential / (ms * 1e-3) / 1e9,
            "frac_hbm": essential / (ms * 1e-3) / 1e9 / hbm,
            "frac_hbm_note": "essential bytes (x, router and expert weights, out) over the layer time",
            "traffic_bytes": alg_bytes, "traffic_gbs": alg_bytes / (ms * 1e-3) / 1e9,
            "traffic_frac": alg_bytes / (ms * 1e-3) / 1e9 / hbm,
            "traffic_note": "bytes of this implementation incl. its y_perm round trip",
            "path": "moe_forward_headlocal: all heads' routers + top-k as one batched GEMM, one sort over "
                    "(head, token), one fused expert kernel over all heads' experts (x head slices gathered "
                    "on chip, gate/up -> SwiGLU -> down with act on chip), one combine into each head's columns"}


def measure_ext_variant(torch, moe, steps: int) -> dict:
    """moe_forward_ext on the chunk_mm workload (video|text|audio stream with
    modality-specific routed experts and one shared expert)."""
    cfg = mi.CONFIGS["chunk_mm"]
    inp = mi.make_inputs(cfg)

    def up(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()

    n_exp = cfg.E + cfg.n_shared
    dims = moe.moe_dims.make(cfg.T, cfg.d, cfg.E, cfg.inter, cfg.top_k, cfg.n_heads, cfg.head_dim)
    dims_w = moe.moe_dims.make(cfg.T, cfg.d, n_exp, cfg.inter, cfg.top_k, cfg.n_heads, cfg.head_dim)
    x, w_lat, w_head, w_down = up(inp["x"]), up(inp["w_lat"]), up(inp["w_head"]), up(inp["w_down"])
    w13 = torch.empty((n_exp, 2 * cfg.inter, cfg.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_weights(dims_w, up(inp["w_gate"]), up(inp["w_up"]), w13)
    modality = torch.from_numpy(inp["modality"]).cuda()
    ext = moe.moe_ext.make(cfg.n_shared, cfg.modality_experts, modality)
    ws = moe.alloc_workspace(moe.moe_workspace_size_ext(dims, ext))
    out = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        moe.moe_forward_ext(dims, ext, x, w_lat, w_head, None, w13, w_down, out, ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        moe.moe_forward_ext(dims, ext, x, w_lat, w_head, None, w13, w_down, out, ws)
    e1.record()
    torch.cuda.synchronize()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status set by moe_forward_ext")
    ms = e0.elapsed_time(e1) / steps
    Tk = cfg.T * (cfg.top_k + cfg.n_shared)
    flops = 2 * cfg.T * cfg.d * cfg.L + 4 * cfg.T * cfg.L * cfg.E + 6 * Tk * cfg.d * cfg.inter
    return {"workload": workload_str(cfg) + f", experts per modality {list(cfg.modality_experts)}, "
                                            f"{cfg.n_shared} shared expert",
            "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "layer_tflops": flops / (ms * 1e-3) / 1e12,
            "path": "moe_forward_ext: modality-specific routing + shared expert (extra fixed slot per token)"}


def main():
    args = parse()
    rank, local, world = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch
    import torch.distributed as dist
    import fine_grained_moe_02_b300 as moe

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    if args.variant is not None:  # one variant alone, on this rank's GPU
        if args.variant == "headlocal":  # the head-local workload, or a head-local --workload given
            name = args.workload if mi.CONFIGS[args.workload].head_local else "headlocal"
            line = measure_headlocal_variant(torch, moe, max(3, args.steps), name)
        else:
            line = measure_ext_variant(torch, moe, max(3, args.steps))
        if rank == 0:
            print(json.dumps(line), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    cfg = mi.CONFIGS[args.workload]
    inp = mi.make_weights(cfg)
    inp["x"] = mi.make_x(rank_workload(cfg, rank))   # each rank its own tokens
    inp["cfg"] = cfg
    T, d, E, I, k = cfg.T, cfg.d, cfg.E, cfg.inter, cfg.top_k
    dims = moe.moe_dims.make(T, d, E, I, k, cfg.n_heads, cfg.head_dim)

    def up(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).cuda()

    x = up(inp["x"])
    w_lat, w_head, w_down = up(inp["w_lat"]), up(inp["w_head"]), up(inp["w_down"])
    bias = None if inp["bias"] is None else torch.from_numpy(inp["bias"]).cuda()
    w13 = torch.empty((E, 2 * I, d), dtype=torch.bfloat16, device="cuda")
    wg, wu = up(inp["w_gate"]), up(inp["w_up"])
    moe.moe_prepare_weights(dims, wg, wu, w13)
    del wg, wu
    ws = moe.alloc_workspace(moe.moe_workspace_size(dims))
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), dtype=torch.float32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_of = torch.empty((T, k), dtype=torch.int32, device="cuda")
    src = torch.empty(T * k, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device="cuda")
    act = torch.empty((T * k, I), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    y_perm = x_perm   # y_perm reuses x_perm's memory, as in moe_forward

    def step(ev=None):
        # exactly moe_forward's sequence, with an event between stages
        moe.moe_clear_device_status(ws)
        if ev: ev[0].record(stream)
        moe.moe_route(dims, x, w_lat, w_head, bias, idx, gate, None, ws)
        if ev: ev[1].record(stream)
        moe.moe_dispatch(dims, x, idx, offsets, row_of, src, x_perm, ws)
        if ev: ev[2].record(stream)
        moe.moe_expert_gemm1(dims, x_perm, offsets, w13, act, ws)
        if ev: ev[3].record(stream)
        moe.moe_expert_gemm2(dims, act, offsets, w_down, y_perm, ws)
        if ev: ev[4].record(stream)
        moe.moe_combine(dims, y_perm, row_of, gate, out)
        if ev: ev[5].record(stream)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step()
        moe.moe_forward(dims, x, w_lat, w_head, bias, w13, w_down, out, ws)
    # then untimed moe_forward calls until at least WARMUP_S of layer work has
    # run: on this power-capped part the clocks settle over the first few
    # hundred ms of sustained load, and the timed region should see the
    # steady state, not the transient
    def settle(seconds):
        """Untimed moe_forward calls until `seconds` of layer work have run; returns the call count."""
        n = 0
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record(stream)
        while True:
            for _ in range(5):
                moe.moe_forward(dims, x, w_lat, w_head, bias, w13, w_down, out, ws)
            n += 5
            w1.record(stream)
            w1.synchronize()
            if w0.elapsed_time(w1) >= 1000.0 * seconds or n >= 2000:
                return n

    extra_warm = settle(WARMUP_S)
    status = moe.moe_get_device_status(ws)
    if status != 0:
        raise SystemExit(f"device status {status:#x} after warm-up")
    counts = np.diff(offsets.cpu().numpy())

    # timed region: K calls of moe_forward, the whole layer in one C call (no
    # events or host work between its kernels)
    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = Clocks(vis[local] if local < len(vis) else local)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    clocks.start()
    t_start.record(stream)
    for _ in range(args.steps):
        moe.moe_forward(dims, x, w_lat, w_head, bias, w13, w_down, out, ws)
    t_end.record(stream)
    barrier()
    # stage breakdown: the same sequence as separate calls with an event
    # between stages, K steps started right after the timed loop (no idle
    # gap beyond one launch: an idle GPU drops its clocks, or recovers power
    # budget, within a few hundred ms), the clock sampler still running
    s0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    s1.record(stream)
    barrier()
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, "cuda")
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status set during the timed region")
    staged_ms = s0.elapsed_time(s1) / args.steps
    stage_names = ["route", "dispatch", "gemm1", "gemm2", "combine"]
    stage_ms = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, n in enumerate(stage_names)}
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status set during the stage loop")

    # the variants below are compared in the same sustained state (the clock
    # sampler's stop left the GPU idle for a moment)
    settle(0.5)

    # the folded-router variant of the layer (moe_forward_folded), same workload
    w_router = torch.empty((E, 2 * d), dtype=torch.bfloat16, device="cuda")
    moe.moe_prepare_router(dims, w_lat, w_head, w_router)
    for _ in range(3):
        moe.moe_forward_folded(dims, x, w_router, bias, w13, w_down, out, ws)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_fold = max(3, args.steps // 2)
    barrier()
    f0.record(stream)
    for _ in range(n_fold):
        moe.moe_forward_folded(dims, x, w_router, bias, w13, w_down, out, ws)
    f1.record(stream)
    barrier()
    fold_ms = max_over_ranks(f0.elapsed_time(f1) / n_fold, world, "cuda")
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    for _ in range(n_fold):
        moe.moe_route_folded(dims, x, w_router, bias, idx, gate, None, ws)
    r1.record(stream)
    barrier()
    fold_route_ms = r0.elapsed_time(r1) / n_fold
    # the two routers of the latent path, interleaved (one call each per round)
    rt = {"two_stage": [], "on_chip": []}
    for _ in range(2):
        moe.moe_route_two_stage(dims, x, w_lat, w_head, bias, idx, gate, None, ws)
        moe.moe_route_fused(dims, x, w_lat, w_head, bias, idx, gate, None, ws)
    barrier()
    for _ in range(n_fold):
        for name, fn in (("two_stage", moe.moe_route_two_stage), ("on_chip", moe.moe_route_fused)):
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            e[0].record(stream)
            fn(dims, x, w_lat, w_head, bias, idx, gate, None, ws)
            e[1].record(stream)
            rt[name].append(e)
    barrier()
    fused_route_ms = statistics.mean(a.elapsed_time(b) for a, b in rt["on_chip"])
    two_stage_route_ms = statistics.mean(a.elapsed_time(b) for a, b in rt["two_stage"])
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status set by a router variant")

    # moe_forward_fused: the gather inside expert GEMM-1, the gate inside expert
    # GEMM-2's epilogue, and both, timed in rounds that interleave them with the
    # plain moe_forward (one call each per round), so clock drift under the
    # power cap does not favour whichever ran first
    calls = {"plain": 0, "gather_in_gemm1": 1, "gate_in_gemm2": 2, "gather_and_gate": 3}
    for fuse in calls.values():
        moe.moe_forward_fused(dims, x, w_lat, w_head, bias, w13, w_down, out, fuse, ws)
    evs_f = {n: [] for n in calls}
    barrier()
    for _ in range(max(3, args.steps // 4)):
        for name, fuse in calls.items():
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            e[0].record(stream)
            moe.moe_forward_fused(dims, x, w_lat, w_head, bias, w13, w_down, out, fuse, ws)
            e[1].record(stream)
            evs_f[name].append(e)
    barrier()
    if moe.moe_get_device_status(ws) != 0:
        raise SystemExit("device status set by moe_forward_fused")
    fused = {}
    for name in calls:
        f_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in evs_f[name]), world, "cuda")
        fused[name] = {"value": throughput(T, world, 1, f_ms / 1e3), "unit": "tokens/s", "ms_per_step": f_ms}
    # the gate fold stage by stage: expert GEMM-2 + combine against the gated
    # GEMM-2 + row combine, alternating, on the routing of the last step
    moe.moe_route(dims, x, w_lat, w_head, bias, idx, gate, None, ws)
    moe.moe_dispatch(dims, x, idx, offsets, row_of, src, x_perm, ws)
    moe.moe_expert_gemm1(dims, x_perm, offsets, w13, act, ws)
    pair = {"plain": [], "gated": []}
    for i in range(2 * max(3, args.steps // 5)):
        kind = "plain" if i % 2 == 0 else "gated"
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        if kind == "plain":
            moe.moe_expert_gemm2(dims, act, offsets, w_down, y_perm, ws)
            ev[1].record(stream)
            moe.moe_combine(dims, y_perm, row_of, gate, out)
        else:
            moe.moe_expert_gemm2_gated(dims, act, offsets, w_down, src, row_of, gate, y_perm, ws)
            ev[1].record(stream)
            moe.moe_combine_rows(dims, y_perm, row_of, out)
        ev[2].record(stream)
        pair[kind].append(ev)
    barrier()
    gate_fold = {k: {"gemm2_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in v),
                     "combine_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in v)} for k, v in pair.items()}
    fused["gate_fold_stages"] = gate_fold

    ext_variant = measure_ext_variant(torch, moe, max(3, args.steps // 2)) if cfg.name == "clip" else None
    hl_variant = measure_headlocal_variant(torch, moe, max(3, args.steps // 2)) if cfg.name == "clip" else None

    # end to end through the public host-buffer entry point
    e2e = None
    if not args.no_e2e:
        ws_h = moe.alloc_workspace(moe.moe_workspace_size_host(dims))
        xh = x.cpu().pin_memory()
        oh = torch.empty_like(xh).pin_memory()
        for _ in range(2):
            moe.moe_forward_host(dims, xh, w_lat, w_head, bias, w13, w_down, oh, ws_h)
        n_e2e = max(3, args.steps // 5)
        barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            moe.moe_forward_host(dims, xh, w_lat, w_head, bias, w13, w_down, oh, ws_h)
        barrier()
        dt = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, "cuda")
        e2e = {"value": world * T / dt, "unit": "tokens/s", "h2d_bytes_per_step": world * T * d * 2,
               "d2h_bytes_per_step": world * T * d * 2, "ms_per_step": 1000 * dt,
               "path": "moe_forward_host (pinned host x and out, copies + layer + stream sync per step)"}
        del ws_h

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    pk = peaks()
    alg = algorithmic(cfg)
    ms_step = elapsed_ms / args.steps
    value = throughput(T, world, args.steps, elapsed_ms / 1e3)
    g1_tf = alg["gemm1_flops"] / (stage_ms["gemm1"] * 1e-3) / 1e12
    g2_tf = alg["gemm2_flops"] / (stage_ms["gemm2"] * 1e-3) / 1e12
    gg_tf = (alg["gemm1_flops"] + alg["gemm2_flops"]) / ((stage_ms["gemm1"] + stage_ms["gemm2"]) * 1e-3) / 1e12
    perm_gbs = alg["permute_bytes"] / (stage_ms["dispatch"] * 1e-3) / 1e9
    comb_gbs = alg["combine_bytes"] / (stage_ms["combine"] * 1e-3) / 1e9
    traffic, traffic_note = measured_traffic(cfg.name)
    tag = "of measured" if pk["source"] == "measured" else "of fallback"
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_str(cfg), "tokens_per_step_per_gpu": T,
                   "parallelism": f"token-sharded replicas x{world}, no collective",
                   "l2": "no flush: inputs larger than L2 (x 0.88 GB, expert weights 3.2 GB > 126 MB)"
                   if cfg.name == "clip" else "no flush",
                   "expert_rows_min_max": [int(counts.min()), int(counts.max())],
                   "warmup_note": f"{max(3, args.warmup)} warm-up steps, then {extra_warm} untimed moe_forward "
                                  f"calls (>= {WARMUP_S:.1f} s of layer work) so the clocks reach their sustained "
                                  f"state before the timed region"},
        "stages_ms": stage_ms,
        "stages_note": "CUDA events between the stages of the same sequence run as separate calls, K steps queued "
                       "right behind the timed moe_forward loop (where the host issues calls slower than the GPU "
                       "runs them, as on the smallest workloads, stage times include the host's gaps)",
        "staged_step_ms": staged_ms,
        "grouped_gemm_tflops": gg_tf,
        "grouped_gemm_frac_bf16_peak": gg_tf / pk["bf16_sus"],
        "gemm1_tflops": g1_tf, "gemm2_tflops": g2_tf,
        "router_tflops": alg["router_flops"] / (stage_ms["route"] * 1e-3) / 1e12,
        "permute_gbs": perm_gbs, "permute_frac_hbm": perm_gbs / pk["hbm"],
        "permute_note": "dispatch stage (histogram, rank assignment with the in-block scan, row gather)",
        "combine_gbs": comb_gbs, "combine_frac_hbm": comb_gbs / pk["hbm"],
        "roofline": {"kernel": "expert GEMM-1 + SwiGLU (gemm_tc_kernel<256, EpiSwiGLU>)", "bound": "tensor",
                     "achieved": g1_tf, "peak": pk["bf16_sus"], "unit": "TFLOP/s", "frac": g1_tf / pk["bf16_sus"],
                     "peak_kind": f"bf16 dense sustained ({tag}; kernel timed inside a long step)",
                     "traffic": traffic, "traffic_note": traffic_note,
                     "algorithmic_flops_per_launch": alg["gemm1_flops"],
                     "frac_burst": g1_tf / pk["bf16"],
                     "tflops_per_sm_mhz": g1_tf / clk["sm_mhz"] if clk.get("sm_mhz") else None,
                     "frac_nominal_at_sampled_clock": (g1_tf / (NOMINAL_BF16_TFLOPS * clk["sm_mhz"] / NOMINAL_SM_MHZ)
                                                       if clk.get("sm_mhz") else None)},
        "variants": {"folded_router": {
            "value": throughput(T, world, 1, fold_ms / 1e3), "unit": "tokens/s", "ms_per_step": fold_ms,
            "route_ms": fold_route_ms,
            "router_tflops": 2 * T * (2 * d) * E / (fold_route_ms * 1e-3) / 1e12,
            "path": "moe_forward_folded: router folded to s = x (W_head W_lat)^T + b, one bf16 hi/lo GEMM "
                    "(same outputs and tolerances; h never formed)"},
            "fused_forward": fused,
            "modality_shared_experts": ext_variant,
            "head_local_moe": hl_variant,
            "on_chip_router": {
                "route_ms": fused_route_ms,
                "router_tflops": alg["router_flops"] / (fused_route_ms * 1e-3) / 1e12,
                "two_stage_route_ms": two_stage_route_ms,
                "path": "moe_route_fused: latent h kept in tensor memory, head-group partial scores only; "
                        "timed in rounds interleaved with moe_route_two_stage"}},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "gpu_launches_note": "libmoe kernels launched inside the timed loop of moe_forward calls (route 2, sort 3, "
                             "expert GEMMs 2, combine 1 per call)",
        "clocks": clk,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_sample)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
