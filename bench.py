"""Benchmark of the MoE expert layer on GB300 (prints one JSON line).

A step is one pass of the whole hot path over one batch: router top-k,
dispatch, grouped gate/up GEMM + SwiGLU, grouped down GEMM, combine, and the
backward of all of them (dX, dW_gate, dW_up, dW_down, d router W), at the
Qwen3-30B-A3B-shaped workload T=8192 tokens, hidden 2048, intermediate 768,
128 experts, top-8 (seeded synthetic inputs, random weights).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain single-threaded C
restatement used by the tests) on a bounded sample of the same workload;
it is a deliberately slow baseline, not a tuned competitor.

With N > 1 (torchrun, one rank per GPU) every rank runs an independent
replica of the step (the layer has no data-path exchange on one node's
replicas), ranks are barrier-synchronised around the timed region, and the
slowest rank's time is used.
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
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "MoE layer tokens/s fwd & fwd+bwd on 1 GB300; grouped-GEMM TFLOP/s vs bf16 peak"
WORKLOAD = "qwen3_30b_fwd_bwd"
FWD_WORKLOAD = "qwen3_30b_fwd"


def peaks():
    try:
        return json.loads((ROOT / "MEASURED_PEAKS.json").read_text()), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def layer_flops(T, H, I, E, k):
    """Algorithmic flops (2 per multiply-add) of one layer pass."""
    R = T * k
    fwd = {"router": 2.0 * T * H * E, "gate_up": 2.0 * R * H * 2 * I, "down": 2.0 * R * I * H}
    bwd = {"down_bwd": 2 * fwd["down"], "gate_up_bwd": 2 * fwd["gate_up"], "router_bwd": 2 * fwd["router"]}
    return fwd, bwd


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.flush()
        rows = []
        for line in Path(self.f.name).read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        try:
            os.unlink(self.f.name)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1])]
        mx = [num(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------ ncu traffic

# DRAM traffic per launch recorded from one-pass ncu captures, per entry-point
# call, each valid only while the GEMM sources hash as recorded.
TRAFFIC_PROFILES = {"gate_up": "traffic_gate_up_fwd_T8192.md", "gate_up_bwd_dw": "traffic_dw_gate_up_T8192.md"}


def recorded_traffic(call="gate_up"):
    """DRAM bytes (read + write) per launch of `call`'s kernel as recorded
    from ncu under profiles/, or None when there is no record or the
    kernel's sources no longer hash to the values recorded there."""
    import hashlib
    name = TRAFFIC_PROFILES.get(call)
    prof = ROOT / "profiles" / name if name else None
    if prof is None or not prof.exists():
        return None
    value, hashes = None, {}
    for line in prof.read_text().splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            value = int(line.split(":")[1])
        elif line.startswith("source_sha256 "):
            name, digest = line[len("source_sha256 "):].split(":")
            hashes[name.strip()] = digest.strip()
    csrc = ROOT / "moe_expert_layer_topk_gb300" / "csrc"
    if value is None or not hashes:
        return None
    for name, digest in hashes.items():
        f = csrc / name
        if not f.exists() or hashlib.sha256(f.read_bytes()).hexdigest() != digest:
            return None
    return value


# --------------------------------------------------------- algorithmic costs

def call_costs(T, H, I, E, k):
    """Algorithmic flops (2 per multiply-add) and DRAM bytes of each call of
    the training step: every operand read once, every result written once.
    Weight gradients are fp32, activations bf16, indices and weights 4 bytes."""
    R = T * k
    W = E * I * H  # elements of one expert weight tensor (Wg, Wu or Wd)
    idx = T * k * 4
    return {
        "route": {"flops": 2.0 * T * H * E, "bytes": T * H * 2 + H * E * 4 + 2 * idx, "pipe": "fma"},
        "dispatch": {"flops": 0.0, "bytes": T * H * 2 + R * H * 2 + 3 * idx},
        "gate_up": {"flops": 2.0 * R * H * 2 * I, "bytes": R * H * 2 + 2 * W * 2 + R * I * 2 + R * 2 * I * 2},
        "down": {"flops": 2.0 * R * I * H, "bytes": R * I * 2 + W * 2 + R * H * 2},
        "combine": {"flops": 0.0, "bytes": R * H * 2 + T * H * 2 + 2 * idx},
        "combine_bwd": {"flops": 0.0, "bytes": T * H * 2 + 2 * R * H * 2 + 3 * idx},
        "down_bwd_dx": {"flops": 2.0 * R * H * I, "bytes": R * H * 2 + W * 2 + 2 * R * 2 * I * 2},
        "down_bwd_dw": {"flops": 2.0 * R * H * I, "bytes": R * H * 2 + R * I * 2 + W * 4},
        "gate_up_bwd_dx": {"flops": 2.0 * R * 2 * I * H, "bytes": R * 2 * I * 2 + 2 * W * 2 + R * H * 2},
        "gate_up_bwd_dw": {"flops": 2.0 * R * 2 * I * H, "bytes": R * 2 * I * 2 + R * H * 2 + 2 * W * 4},
        "dispatch_bwd": {"flops": 0.0, "bytes": R * H * 2 + T * H * 4 + idx},
        "route_bwd": {"flops": 2.0 * 2 * T * H * E, "bytes": T * H * 2 + T * H * 4 + T * H * 2 + H * E * 8 + 3 * idx},
    }


# the calls that launch one kernel (the weight-gradient halves also launch the
# segment-map kernel of a few microseconds before their GEMM)
SINGLE_KERNEL = {"gate_up": "grouped_gemm gate/up + SwiGLU (forward)", "down": "grouped_gemm down (forward)",
                 "combine": "combine (weighted unpermute)", "combine_bwd": "combine backward",
                 "down_bwd_dx": "grouped_gemm down backward dX + SwiGLU backward",
                 "down_bwd_dw": "grouped_gemm dW_down (fp32)",
                 "gate_up_bwd_dx": "grouped_gemm gate/up backward dX",
                 "gate_up_bwd_dw": "grouped_gemm dW_gate/up (fp32)", "dispatch_bwd": "dispatch backward"}


def rooflines(per_call, costs, pk, fma_tfma):
    """Roofline of every call: time at the bound (the larger of the tensor,
    FMA and HBM times) over the measured time.  Tensor-bound calls use the
    sustained bf16 peak (they run inside a step of a second or more)."""
    out = {}
    for n, ms in per_call.items():
        c = costs.get(n)
        if c is None or ms <= 0:
            continue
        t = ms * 1e-3
        t_mem = c["bytes"] / (pk["hbm_gbs"] * 1e9)
        if c.get("pipe") == "fma":
            t_cmp = c["flops"] / 2 / (fma_tfma * 1e12) if fma_tfma else 0.0
            cmp_peak, cmp_unit, cmp_bound = fma_tfma, "TFMA/s", "alu"
            achieved_cmp = c["flops"] / 2 / t / 1e12
        else:
            t_cmp = c["flops"] / (pk["bf16_tflops_sustained"] * 1e12)
            cmp_peak, cmp_unit, cmp_bound = pk["bf16_tflops_sustained"], "TFLOP/s", "tensor"
            achieved_cmp = c["flops"] / t / 1e12
        gbs = c["bytes"] / t / 1e9
        if t_cmp >= t_mem and c["flops"] > 0:
            r = {"bound": cmp_bound, "achieved": achieved_cmp, "peak": cmp_peak, "unit": cmp_unit}
        else:
            r = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s"}
        r["frac"] = max(t_cmp, t_mem) / t
        r["us"] = ms * 1e3
        r["gbs"] = gbs
        if c["flops"] > 0 and c.get("pipe") != "fma":
            r["tflops"] = c["flops"] / t / 1e12
            r["tensor_frac_of_burst"] = c["flops"] / t / 1e12 / pk["bf16_tflops"]
        out[n] = r
    return out


def host_cpu():
    """Host CPU threads and model name (lscpu, else the platform module)."""
    import platform
    model = None
    try:
        txt = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in txt.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"nproc": os.cpu_count(), "model": model or platform.processor() or platform.machine()}


# --------------------------------------------------------------- multi-rank

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
        return dist, dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return None, 0, 1, 0


def max_over_ranks(value: float, dist, device=None) -> float:
    """Largest `value` over all ranks (the slowest replica defines the time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# -------------------------------------------------------------- CPU oracle

def oracle_sample_step(inp, T_s):
    """Oracle forward+backward over the first T_s tokens of the workload."""
    import numpy as np

    import oracle
    from moe_expert_layer_topk_gb300.synth import bf16_bits
    x = bf16_bits(inp["x"][:T_s])
    Wr = inp["Wr"].numpy()
    Wg, Wu, Wd = (bf16_bits(inp[n]) for n in ("Wg", "Wu", "Wd"))
    k, E = inp["k"], inp["E"]
    rt = oracle.route_topk(x, Wr, None, k, inp["ep_size"])
    dp = oracle.dispatch(x, rt["topk_idx"], rt["offsets"], E)
    xp = oracle.widen_bf16(dp["x_perm"])
    h, gu = oracle.grouped_gemm_swiglu(xp, Wg, Wu, rt["offsets"], save_gu=True)
    yp = oracle.grouped_gemm_down(h, Wd, rt["offsets"])
    oracle.combine(yp, rt["topk_w"], dp["row_of_slot"])
    dy = oracle.widen_bf16(bf16_bits(inp["dy"][:T_s]))
    dyp, dw = oracle.combine_bwd(dy, yp, rt["topk_w"], dp["row_of_slot"])
    dgu, _ = oracle.grouped_gemm_down_bwd(dyp, h, gu, Wd, rt["offsets"])
    dxp, _, _ = oracle.grouped_gemm_swiglu_bwd(dgu, xp, Wg, Wu, rt["offsets"])
    dxa = oracle.dispatch_bwd(dxp, dp["row_of_slot"])
    oracle.route_topk_bwd(dw, rt["topk_w"], rt["topk_idx"], x, Wr, dxa)
    return np.int64(T_s)


def cpu_cores_used():
    return 1  # the oracle is single-threaded C


def run_reference(args, shape, inp):
    dist, rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    T_s = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample_step(inp, T_s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(inp, T_s)
    dt = time.perf_counter() - t0
    value = T_s * args.steps / dt
    sample = f"first {T_s} tokens of {WORKLOAD} (T={shape.T}) per step, forward+backward, full weights"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded normal inputs, random-init weights)",
            "config": {"workload": WORKLOAD, "T": shape.T, "H": shape.H, "I": shape.I, "E": shape.E,
                       "k": shape.k, "sample_tokens_per_step": T_s},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores_used(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

MIN_TIMED_S = 1.0  # the timed region covers whole blocks of K steps, at least this long


def run_ours(args, shape, inp):
    import torch

    import moe_expert_layer_topk_gb300 as m
    dist, rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    g = {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
    layer = m.MoELayer(T, H, I, E, k, shape.ep_size, device=dev)
    stream = torch.cuda.current_stream(dev)
    ws_dw2 = torch.empty_like(layer.ws_gemm_bwd)

    # per-call events: (name, start, end) recorded on the launching stream;
    # the backward GEMM calls run as their dX and weight-gradient halves
    names = ["route", "dispatch", "gate_up", "down", "combine", "combine_bwd", "down_bwd_dx", "down_bwd_dw",
             "gate_up_bwd_dx", "gate_up_bwd_dw", "dispatch_bwd", "route_bwd"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        R = layer.R
        mark(0)
        layer.route(g["x"], g["Wr"], g["bias"]); mark(1)
        layer.dispatch(g["x"]); mark(2)
        m.moe_grouped_gemm_swiglu(layer.x_perm, g["Wg"], g["Wu"], E, layer.offsets, None, R, H, I, E,
                                  layer.h, layer.gu); mark(3)
        m.moe_grouped_gemm_down(layer.h, g["Wd"], E, layer.offsets, None, R, H, I, E, layer.y_perm); mark(4)
        layer.combine(); mark(5)
        m.moe_combine_bwd(g["dy"], layer.y_perm, layer.topk_w, layer.row_of_slot, T, H, k, layer.dy_perm,
                          layer.d_w); mark(6)
        m.moe_grouped_gemm_down_bwd_dx(layer.dy_perm, layer.gu, g["Wd"], E, layer.offsets, None, R, H, I, E,
                                       layer.dgu); mark(7)
        m.moe_grouped_gemm_down_bwd_dw(layer.dy_perm, layer.h, E, layer.offsets, None, R, H, I, E, layer.dWd, 0,
                                       layer.ws_gemm_bwd); mark(8)
        m.moe_grouped_gemm_swiglu_bwd_dx(layer.dgu, g["Wg"], g["Wu"], E, layer.offsets, None, R, H, I, E,
                                         layer.dx_perm); mark(9)
        m.moe_grouped_gemm_swiglu_bwd_dw(layer.dgu, layer.x_perm, E, layer.offsets, None, R, H, I, E, layer.dWg,
                                         layer.dWu, 0, ws_dw2); mark(10)
        m.moe_dispatch_bwd(layer.dx_perm, layer.row_of_slot, T, H, k, layer.dx_acc); mark(11)
        m.moe_route_topk_bwd(layer.d_w, layer.topk_w, layer.topk_idx, g["x"], g["Wr"], layer.dx_acc, T, H,
                             E, k, layer.dWr, layer.dx, 0, layer.ws_route_bwd); mark(12)

    def layer_step():
        # the step as the layer runs it: the dispatch and router backward on a
        # side stream beside the gate/up weight gradient
        layer.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"])
        layer.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])

    for _ in range(args.warmup):
        layer_step()
        step()
    torch.cuda.synchronize(dev)
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during warm-up")
    # one untimed block of K steps sizes the timed region: whole blocks of K
    # steps, at least MIN_TIMED_S long, so that the clock samples see the load
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    for _ in range(args.steps):
        layer_step()
    p1.record(stream)
    torch.cuda.synchronize(dev)
    block_s = max(p0.elapsed_time(p1) * 1e-3, 1e-6)
    reps = max(1, min(200, int(-(-MIN_TIMED_S // block_s))))
    reps = int(max_over_ranks(float(reps), dist, dev))
    n_timed = reps * args.steps

    nev = len(names) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(n_timed)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c_start, c_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for i in range(n_timed):
            layer_step()
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        # the same steps with every call on one stream, bracketed by events of
        # its own: the per-call times and rooflines
        c_start.record(stream)
        for i in range(n_timed):
            step(evs[i])
        c_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms_local = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms_local, dist, dev)
    seq_ms = c_start.elapsed_time(c_end) / n_timed
    per_call = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n_timed))
                for j, n in enumerate(names)}
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during the timed region")
    del evs

    fma_tfma = measure_fma_rate(m, dev, stream)

    # forward-only throughput at T=4096 (the forward workload)
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_layer_inputs
    fshape = CONFIGS[FWD_WORKLOAD]
    fin = make_layer_inputs(fshape, 0)
    fg = {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in fin.items()}
    flayer = m.MoELayer(fshape.T, fshape.H, fshape.I, fshape.E, fshape.k, fshape.ep_size,
                        training=False, fused_dispatch=True, device=dev)
    for _ in range(args.warmup):
        flayer.forward(fg["x"], fg["Wr"], fg["bias"], fg["Wg"], fg["Wu"], fg["Wd"])
    fs, fe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    fs.record(stream)
    for _ in range(args.steps):
        flayer.forward(fg["x"], fg["Wr"], fg["bias"], fg["Wg"], fg["Wu"], fg["Wd"])
    fe.record(stream)
    torch.cuda.synchronize(dev)
    fwd_ms = fs.elapsed_time(fe) / args.steps
    del flayer
    # the same forward with the down GEMM and the combine fused (no y_perm)
    flayer = m.MoELayer(fshape.T, fshape.H, fshape.I, fshape.E, fshape.k, fshape.ep_size,
                        training=False, fused_dispatch=True, fused_combine=True, device=dev)
    for _ in range(args.warmup):
        flayer.forward(fg["x"], fg["Wr"], fg["bias"], fg["Wg"], fg["Wu"], fg["Wd"])
    torch.cuda.synchronize(dev)
    fs.record(stream)
    for _ in range(args.steps):
        flayer.forward(fg["x"], fg["Wr"], fg["bias"], fg["Wg"], fg["Wu"], fg["Wd"])
    fe.record(stream)
    torch.cuda.synchronize(dev)
    fused_combine_ms = fs.elapsed_time(fe) / args.steps
    del flayer
    fp8 = run_fp8_forward(m, fg, fshape, dev, stream, args)
    del fg
    pk, pk_kind = peaks()
    extra = {"zipf_fwd": run_fwd_workload(m, "qwen3_30b_zipf_fwd", dev, stream, args, pk),
             "ep_rank_local": run_ep_rank_local(m, dev, stream, args, pk),
             "tiny_fwd": run_fwd_workload(m, "tiny_fwd", dev, stream, args, pk)}

    # end to end through the public API with host buffers: every step copies
    # its x and dY from pinned host memory and reads its y and dX back.  The
    # copies run on their own streams, pipelined over two slots: the
    # host-to-device copy of step i+1 and the device-to-host read of step i-1
    # overlap step i's compute, which writes its y and dX straight into the
    # slot's output tensors (a slot is reused two steps later, after its
    # read has finished).
    hx = inp["x"].pin_memory()
    hdy = inp["dy"].pin_memory()
    hy = torch.empty_like(inp["x"]).pin_memory()
    hdx = torch.empty_like(inp["x"]).pin_memory()
    x_in = [torch.empty_like(g["x"]) for _ in range(2)]
    dy_in = [torch.empty_like(g["dy"]) for _ in range(2)]
    y_st = [torch.empty_like(g["x"]) for _ in range(2)]
    dx_st = [torch.empty_like(g["x"]) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    issued_out = [False, False]

    def e2e_step(i):
        s = i & 1
        with torch.cuda.stream(h2d):
            if issued_out[s]:
                h2d.wait_event(ev_out[s])  # step i-2 has left this slot
            x_in[s].copy_(hx, non_blocking=True)
            dy_in[s].copy_(hdy, non_blocking=True)
            ev_in[s].record(h2d)
        stream.wait_event(ev_in[s])
        layer.forward(x_in[s], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"], y=y_st[s])
        layer.backward(dy_in[s], x_in[s], g["Wr"], g["Wg"], g["Wu"], g["Wd"], dx=dx_st[s])
        ev_done[s].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[s])
            hy.copy_(y_st[s], non_blocking=True)
            hdx.copy_(dx_st[s], non_blocking=True)
            ev_out[s].record(d2h)
        issued_out[s] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    issued_out[0] = issued_out[1] = False
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    es.record(h2d)
    # as many steps as the device-timed region, so that both see the same
    # clocks under the power cap
    for i in range(n_timed):
        e2e_step(i)
    ee.record(d2h)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(es.elapsed_time(ee), dist, dev) / n_timed
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during the end-to-end steps")

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    costs = call_costs(T, H, I, E, k)
    roof = rooflines(per_call, costs, pk, fma_tfma)
    gemm_calls = ["gate_up", "down", "down_bwd_dx", "down_bwd_dw", "gate_up_bwd_dx", "gate_up_bwd_dw"]
    gemm_ms = sum(per_call[n] for n in gemm_calls)
    gemm_tflops = sum(costs[n]["flops"] for n in gemm_calls) / (gemm_ms * 1e-3) / 1e12
    # dominant kernel: the single-kernel call with the largest measured time
    dom = max(SINGLE_KERNEL, key=lambda n: per_call[n])
    dr = roof[dom]
    step_ms = ms / n_timed
    value = world * T / (step_ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal inputs, random-init weights)",
        "config": {"workload": WORKLOAD, "T": T, "H": H, "I": I, "E": E, "k": k,
                   "step": "forward+backward (router, dispatch, gate/up+SwiGLU, down, combine and their backward)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1.2 GB of expert weights per step)",
                   "timed": f"{reps} back-to-back blocks of {args.steps} steps ({n_timed} steps, "
                            f"{ms_local * 1e-3:.2f} s) between one pair of events",
                   "schedule": f"MoELayer.forward + backward; the dispatch and router backward on a side "
                               f"stream beside the gate/up weight gradient, which leaves "
                               f"{layer.TAIL_SMS} SMs to them"},
        "timed_steps": n_timed,
        "per_call_pass": {"ms_per_step": seq_ms,
                          "how": "the same steps again, every call on one stream with CUDA events of its "
                                 "own around it (per_call_ms and the rooflines come from this pass)"},
        "fwd_tokens_per_s": fshape.T / (fwd_ms * 1e-3),
        "fwd_ms": fwd_ms, "fwd_config": {"workload": FWD_WORKLOAD, "T": fshape.T,
                       "path": "fused dispatch: rows gathered from x by the gate/up GEMM"},
        "fused_combine_fwd": {"workload": FWD_WORKLOAD, "T": fshape.T,
                              "tokens_per_s": fshape.T / (fused_combine_ms * 1e-3), "ms": fused_combine_ms,
                              "path": "fused dispatch and fused combine (the down GEMM adds its weighted rows "
                                      "into the tokens' fp32 rows; no y_perm; not the headline path)"},
        "fp8_fwd": fp8,
        **extra,
        "grouped_gemm_tflops": gemm_tflops,
        "grouped_gemm_frac_of_sustained": gemm_tflops / pk["bf16_tflops_sustained"],
        "per_call_ms": per_call,
        "roofline": {"bound": dr["bound"], "kernel": SINGLE_KERNEL[dom], "call": dom,
                     "achieved": dr["achieved"], "peak": dr["peak"], "unit": dr["unit"], "frac": dr["frac"],
                     "peak_source": (f"{pk_kind} HBM copy" if dr["bound"] == "hbm" else
                                     f"{pk_kind} bf16 sustained"),
                     "algorithmic_bytes": costs[dom]["bytes"], "algorithmic_flops": costs[dom]["flops"],
                     "traffic": recorded_traffic(dom),
                     "traffic_source": "one-pass ncu capture recorded under profiles/ (valid while the GEMM "
                                       "sources hash as recorded there; else null)"},
        "rooflines": roof,
        "fma_peak_tfma_s": fma_tfma,
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s", "steps": n_timed,
                "h2d_bytes_per_step": int(hx.numel() * 2 + hdy.numel() * 2),
                "d2h_bytes_per_step": int(hy.numel() * 2 + hdx.numel() * 2),
                "copies": "pinned host x, dY in and y, dX out every step, on two copy streams; "
                          "step i+1's inputs and step i-1's outputs move during step i"},
        "gpu_launches": KERNELS_PER_STEP * n_timed,
        "clocks": clk.summary(),
    }
    if args.cpu_baseline:
        t0 = time.perf_counter()
        oracle_sample_step(inp, args.cpu_tokens)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": args.cpu_tokens / dt, "unit": "tokens/s", "cores": cpu_cores_used(),
                                "host": host_cpu(), "kind": "oracle",
                                "sample": f"first {args.cpu_tokens} tokens of {WORKLOAD}, forward+backward, "
                                          f"single-threaded C oracle, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def measure_fma_rate(m, dev, stream):
    """fp32 FMA rate of this GPU (TFMA/s) from the library's FMA-chain probe:
    the best of a few launches, scalar and packed two-lane FMAs, timed with
    events."""
    import torch
    out = torch.zeros(1, dtype=torch.float32, device=dev)
    best = 0.0
    for packed in (0, 1, 0, 1, 0, 1):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        n = m.moe_probe_fma(packed, 4, 256, out)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        best = max(best, n / (s0.elapsed_time(s1) * 1e-3) / 1e12)
    return best


def _timed_calls(calls, steps, warmup, stream, dev):
    """Mean per-call and per-step milliseconds of `calls` (name -> fn) run in
    order, `steps` times after `warmup` untimed passes, events on `stream`."""
    import torch
    for _ in range(warmup):
        for f in calls.values():
            f()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(steps)]
    torch.cuda.synchronize(dev)
    for i in range(steps):
        evs[i][0].record(stream)
        for j, f in enumerate(calls.values()):
            f()
            evs[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps))
           for j, n in enumerate(calls)}
    step_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][-1]) for i in range(steps))
    return per, step_ms


def run_fwd_workload(m, name, dev, stream, args, pk):
    """Forward of a routed workload (route, dispatch, gate/up, down, combine)
    on the permuted-row path, each call bracketed by events."""
    import torch
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_layer_inputs
    shape = CONFIGS[name]
    fin = make_layer_inputs(shape, 0)
    g = {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in fin.items()}
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    L = m.MoELayer(T, H, I, E, k, shape.ep_size, training=False, device=dev)
    R = L.R
    calls = {"route": lambda: L.route(g["x"], g["Wr"], g["bias"]),
             "dispatch": lambda: L.dispatch(g["x"]),
             "gate_up": lambda: m.moe_grouped_gemm_swiglu(L.x_perm, g["Wg"], g["Wu"], E, L.offsets, None, R, H, I,
                                                          E, L.h, None),
             "down": lambda: m.moe_grouped_gemm_down(L.h, g["Wd"], E, L.offsets, None, R, H, I, E, L.y_perm),
             "combine": lambda: L.combine()}
    per, step_ms = _timed_calls(calls, args.steps, args.warmup, stream, dev)
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError(f"device status word set during {name}")
    counts = L.counts.cpu()
    fl_gu, fl_dn = 2.0 * R * H * 2 * I, 2.0 * R * I * H
    gemm_tf = (fl_gu + fl_dn) / ((per["gate_up"] + per["down"]) * 1e-3) / 1e12
    out = {"workload": name, "T": T, "H": H, "I": I, "E": E, "k": k, "tokens_per_s": T / (step_ms * 1e-3),
           "ms": step_ms, "per_call_ms": per, "path": "permuted rows (dispatch writes x_perm)",
           "gate_up_tflops": fl_gu / (per["gate_up"] * 1e-3) / 1e12,
           "down_tflops": fl_dn / (per["down"] * 1e-3) / 1e12, "grouped_gemm_tflops": gemm_tf,
           "grouped_gemm_frac_of_burst": gemm_tf / pk["bf16_tflops"],
           "empty_experts": int((counts == 0).sum()), "max_expert_rows": int(counts.max())}
    if shape.bias == "zipf":
        out["routing"] = "Zipf(1.2) expert popularity from a router bias, 4 experts forced empty"
    if name == "tiny_fwd":
        # the same forward replayed as one CUDA graph (launch-bound batch)
        graph = L.capture_forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"])
        for _ in range(args.warmup):
            graph.replay()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        g0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        if m.moe_read_device_status(reset=True) != 0:
            raise RuntimeError("device status word set during the graphed tiny forward")
        gms = g0.elapsed_time(g1) / args.steps
        out["graph"] = {"tokens_per_s": T / (gms * 1e-3), "ms": gms,
                        "path": "MoELayer.forward captured once as a CUDA graph, replayed"}
    return out


def run_ep_rank_local(m, dev, stream, args, pk):
    """One EP rank's local expert compute: 32768 received rows in 8 source-rank
    blocks x 16 local experts (128 segments), gate/up + SwiGLU and down."""
    import torch
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_segment_inputs
    shape = CONFIGS["ep_rank_local"]
    s = make_segment_inputs(shape, 0)
    g = {n: (v.to(dev) if isinstance(v, torch.Tensor) else v) for n, v in s.items()}
    R, H, I, E, S = s["R"], s["H"], s["I"], s["E"], s["num_seg"]
    h = torch.empty(R, I, dtype=torch.bfloat16, device=dev)
    y = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    so, se = g["seg_offsets"], g["seg_expert"]
    calls = {"gate_up": lambda: m.moe_grouped_gemm_swiglu(g["x_perm"], g["Wg"], g["Wu"], S, so, se, R, H, I, E, h,
                                                          None),
             "down": lambda: m.moe_grouped_gemm_down(h, g["Wd"], S, so, se, R, H, I, E, y)}
    per, step_ms = _timed_calls(calls, args.steps, args.warmup, stream, dev)
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during ep_rank_local")
    fl_gu, fl_dn = 2.0 * R * H * 2 * I, 2.0 * R * I * H
    gemm_tf = (fl_gu + fl_dn) / (step_ms * 1e-3) / 1e12
    return {"workload": "ep_rank_local", "rows": R, "H": H, "I": I, "local_experts": E, "segments": S,
            "rows_per_s": R / (step_ms * 1e-3), "ms": step_ms, "per_call_ms": per,
            "gate_up_tflops": fl_gu / (per["gate_up"] * 1e-3) / 1e12,
            "down_tflops": fl_dn / (per["down"] * 1e-3) / 1e12, "grouped_gemm_tflops": gemm_tf,
            "grouped_gemm_frac_of_burst": gemm_tf / pk["bf16_tflops"],
            "weights_bytes": 3 * E * I * H * 2}


def run_fp8_forward(m, fg, fshape, dev, stream, args):
    """Forward of the T=4096 workload on e4m3 GEMMs (MoELayer(fp8=True)).

    The expert weights are quantised once, before the timed region (they do
    not change between forward passes); every step quantises x (inside the
    dispatch) and h.  Each call is bracketed by events on the launching
    stream."""
    import torch
    T, H, I, E, k = fshape.T, fshape.H, fshape.I, fshape.E, fshape.k
    L = m.MoELayer(T, H, I, E, k, fshape.ep_size, training=False, fp8=True, device=dev)
    w8 = L.quantize_weights(fg["Wg"], fg["Wu"], fg["Wd"])
    R = L.R
    names = ["route", "dispatch_e4m3", "gate_up_fp8", "quantize_h", "down_fp8", "combine"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        L.route(fg["x"], fg["Wr"], fg["bias"]); mark(1)
        L.dispatch(fg["x"]); mark(2)  # permuted rows written as e4m3 codes
        m.moe_grouped_gemm_swiglu_fp8(L.x_q, L.x_scale, None, 0, w8["Wg"], w8["Wg_scale"], w8["Wu"],
                                      w8["Wu_scale"], E, L.offsets, None, R, H, I, E, L.h); mark(3)
        m.moe_quantize_rows_e4m3(L.h, R, I, L.h_q, L.h_scale); mark(4)
        m.moe_grouped_gemm_down_fp8(L.h_q, L.h_scale, w8["Wd"], w8["Wd_scale"], E, L.offsets, None, R, H, I, E,
                                    L.y_perm); mark(5)
        L.combine(); mark(6)

    for _ in range(args.warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(args.steps)]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    s0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    s1.record(stream)
    torch.cuda.synchronize(dev)
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during the fp8 forward")
    ms = s0.elapsed_time(s1) / args.steps
    per_call = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                for j, n in enumerate(names)}
    fwd_fl, _ = layer_flops(T, H, I, E, k)
    pk, pk_kind = peaks()
    # e4m3 dense peak: the measured bf16 burst times the nominal fp8/bf16 ratio (4.5 / 2.25 PFLOP/s)
    fp8_peak = 2.0 * pk["bf16_tflops"]
    gu_tf = fwd_fl["gate_up"] / (per_call["gate_up_fp8"] * 1e-3) / 1e12
    dn_tf = fwd_fl["down"] / (per_call["down_fp8"] * 1e-3) / 1e12
    # weight bytes dominate at T=4096: e4m3 codes + one fp32 scale per output channel
    gu_bytes = R * H + R * 4 + 2 * E * I * H + 2 * E * I * 4 + R * I * 2
    return {"workload": FWD_WORKLOAD, "T": T, "tokens_per_s": T / (ms * 1e-3), "ms": ms,
            "path": "dispatch writes the permuted rows as e4m3 codes (one scale per token), h quantised "
                    "per row; weights quantised once outside the timed region",
            "per_call_ms": per_call, "gate_up_tflops": gu_tf, "down_tflops": dn_tf,
            "gate_up_frac_of_fp8_peak": gu_tf / fp8_peak,
            "fp8_peak_tflops": fp8_peak, "fp8_peak_source": f"2 x {pk_kind} bf16 burst (nominal fp8/bf16 ratio)",
            "gate_up_gbs": gu_bytes / (per_call["gate_up_fp8"] * 1e-3) / 1e9,
            "hbm_peak_gbs": pk["hbm_gbs"]}


# kernels launched per step by the calls in run_ours.step() (and by
# MoELayer.forward + backward, the same calls):
# route 4 (partial logits, top-k with per-chunk counts, chunk scan, offsets),
# dispatch 1 (rows from the route's chunk prefixes),
# gate/up 1, down 1, combine 1, combine_bwd 1, the dX halves 1 each and the
# weight-gradient halves 2 each (segment maps, dW GEMM), dispatch_bwd 1,
# route_bwd 7
KERNELS_PER_STEP = 4 + 1 + 1 + 1 + 1 + 1 + 3 + 3 + 1 + 7


def run_profile_router(args):
    """Untimed router passes (moe_route_topk only) of T tokens (for ncu captures)."""
    import torch

    import moe_expert_layer_topk_gb300 as m
    from moe_expert_layer_topk_gb300.synth import LayerShape, make_layer_inputs
    T, H, E, k = (int(v) for v in args.profile_router.split(","))
    g = torch.Generator().manual_seed(0)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16).cuda()
    Wr = (torch.randn(H, E, generator=g) * 0.02).cuda()
    layer = m.MoELayer(T, H, 64, E, k, 1, training=False)
    for _ in range(args.steps):
        layer.route(x, Wr, None)
    torch.cuda.synchronize()
    print(json.dumps({"profile_router": [T, H, E, k], "passes": args.steps,
                      "device_status": m.moe_read_device_status(reset=True)}))


def run_profile_case(args):
    """Untimed forward+backward passes of one layer shape (for ncu captures),
    the backward on one stream."""
    import torch

    import moe_expert_layer_topk_gb300 as m
    from moe_expert_layer_topk_gb300.synth import LayerShape, make_layer_inputs
    T, H, I, E, k = (int(v) for v in args.profile_case.split(","))
    shape = LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=1)
    inp = make_layer_inputs(shape, 0, with_dy=True)
    g = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
    layer = m.MoELayer(T, H, I, E, k, 1)
    for _ in range(args.steps):
        layer.forward(g["x"], g["Wr"], None, g["Wg"], g["Wu"], g["Wd"])
        # one stream, every GEMM on all SMs: the kernels as the per-call pass times them
        layer.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], overlap=False)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": [T, H, I, E, k], "passes": args.steps,
                      "device_status": m.moe_read_device_status(reset=True)}))


def run_profile_fp8(args):
    """Untimed fp8 forward passes of one layer shape (for ncu captures)."""
    import torch

    import moe_expert_layer_topk_gb300 as m
    from moe_expert_layer_topk_gb300.synth import LayerShape, make_layer_inputs
    T, H, I, E, k = (int(v) for v in args.profile_fp8.split(","))
    shape = LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=1)
    inp = make_layer_inputs(shape, 0, with_dy=False)
    g = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
    layer = m.MoELayer(T, H, I, E, k, 1, training=False, fp8=True)
    w8 = layer.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    for _ in range(args.steps):
        layer.forward(g["x"], g["Wr"], None, w8, None, None)
    torch.cuda.synchronize()
    print(json.dumps({"profile_fp8": [T, H, I, E, k], "passes": args.steps,
                      "device_status": m.moe_read_device_status(reset=True)}))


def run_profile_fwd(args):
    """Untimed bf16 forward passes of one layer shape, fused dispatch, with
    or without the fused combine (for ncu captures)."""
    import torch

    import moe_expert_layer_topk_gb300 as m
    from moe_expert_layer_topk_gb300.synth import LayerShape, make_layer_inputs
    spec, _, mode = args.profile_fwd.partition(":")
    T, H, I, E, k = (int(v) for v in spec.split(","))
    shape = LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=1)
    inp = make_layer_inputs(shape, 0, with_dy=False)
    g = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
    layer = m.MoELayer(T, H, I, E, k, 1, training=False, fused_dispatch=True,
                       fused_combine=(mode == "fused_combine"))
    for _ in range(args.steps):
        layer.forward(g["x"], g["Wr"], None, g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    print(json.dumps({"profile_fwd": [T, H, I, E, k], "fused_combine": mode == "fused_combine",
                      "passes": args.steps, "device_status": m.moe_read_device_status(reset=True)}))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-tokens", type=int, default=8, help="oracle tokens per reference step")
    ap.add_argument("--cpu-tokens", type=int, default=48, help="oracle tokens for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--profile-case", default=None, metavar="T,H,I,E,k",
                    help="run --steps untimed forward+backward passes of this shape and exit")
    ap.add_argument("--profile-router", default=None, metavar="T,H,E,k",
                    help="run --steps untimed router passes and exit")
    ap.add_argument("--profile-fwd", default=None, metavar="T,H,I,E,k[:fused_combine]",
                    help="run --steps untimed bf16 forward passes (fused dispatch) of this shape and exit")
    ap.add_argument("--profile-fp8", default=None, metavar="T,H,I,E,k",
                    help="run --steps untimed fp8 forward passes of this shape and exit")
    args = ap.parse_args(argv)
    if args.profile_router:
        return run_profile_router(args)
    if args.profile_case:
        return run_profile_case(args)
    if args.profile_fp8:
        return run_profile_fp8(args)
    if args.profile_fwd:
        return run_profile_fwd(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_layer_inputs
    shape = CONFIGS[WORKLOAD]
    inp = make_layer_inputs(shape, 0)
    if args.impl == "reference":
        run_reference(args, shape, inp)
    else:
        run_ours(args, shape, inp)


if __name__ == "__main__":
    main()
