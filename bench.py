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

def recorded_traffic():
    """DRAM bytes per launch of the forward gate/up GEMM as recorded from ncu
    in profiles/traffic_gate_up_fwd_T8192.md, or None once the kernel's
    sources no longer hash to the values recorded there."""
    import hashlib
    prof = ROOT / "profiles" / "traffic_gate_up_fwd_T8192.md"
    if not prof.exists():
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

    # per-call events: (name, start, end) recorded on the launching stream
    names = ["route", "dispatch", "gate_up", "down", "combine", "combine_bwd", "down_bwd",
             "gate_up_bwd", "dispatch_bwd", "route_bwd"]

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
        m.moe_grouped_gemm_down_bwd(layer.dy_perm, layer.h, layer.gu, g["Wd"], E, layer.offsets, None, R, H,
                                    I, E, layer.dgu, layer.dWd, 0, layer.ws_gemm_bwd); mark(7)
        m.moe_grouped_gemm_swiglu_bwd(layer.dgu, layer.x_perm, g["Wg"], g["Wu"], E, layer.offsets, None, R,
                                      H, I, E, layer.dx_perm, layer.dWg, layer.dWu, 0,
                                      layer.ws_gemm_bwd); mark(8)
        m.moe_dispatch_bwd(layer.dx_perm, layer.row_of_slot, T, H, k, layer.dx_acc); mark(9)
        m.moe_route_topk_bwd(layer.d_w, layer.topk_w, layer.topk_idx, g["x"], g["Wr"], layer.dx_acc, T, H,
                             E, k, layer.dWr, layer.dx, 0, layer.ws_route_bwd); mark(10)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(11)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        time.sleep(0.1)
        t_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms_local = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms_local, dist, dev)
    per_call = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                for j, n in enumerate(names)}

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
    fp8 = run_fp8_forward(m, fg, fshape, dev, stream, args)
    del fg

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
    for i in range(args.steps):
        e2e_step(i)
    ee.record(d2h)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(es.elapsed_time(ee), dist, dev) / args.steps
    if m.moe_read_device_status(reset=True) != 0:
        raise RuntimeError("device status word set during the timed region")

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    pk, pk_kind = peaks()
    fwd_fl, bwd_fl = layer_flops(T, H, I, E, k)
    gemm_fl = {"gate_up": fwd_fl["gate_up"], "down": fwd_fl["down"], "down_bwd": bwd_fl["down_bwd"],
               "gate_up_bwd": bwd_fl["gate_up_bwd"]}
    gemm_ms = sum(per_call[n] for n in gemm_fl)
    gemm_tflops = sum(gemm_fl.values()) / (gemm_ms * 1e-3) / 1e12
    # dominant single-kernel call: the forward gate/up GEMM is one launch
    dom = "gate_up"
    dom_tflops = gemm_fl[dom] / (per_call[dom] * 1e-3) / 1e12
    step_ms = ms / args.steps
    value = world * T / (step_ms * 1e-3)
    traffic = recorded_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal inputs, random-init weights)",
        "config": {"workload": WORKLOAD, "T": T, "H": H, "I": I, "E": E, "k": k,
                   "step": "forward+backward (router, dispatch, gate/up+SwiGLU, down, combine and their backward)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (1.2 GB of expert weights per step)"},
        "fwd_tokens_per_s": fshape.T / (fwd_ms * 1e-3),
        "fwd_ms": fwd_ms, "fwd_config": {"workload": FWD_WORKLOAD, "T": fshape.T,
                       "path": "fused dispatch: rows gathered from x by the gate/up GEMM"},
        "fp8_fwd": fp8,
        "grouped_gemm_tflops": gemm_tflops,
        "per_call_ms": per_call,
        "roofline": {"bound": "tensor", "kernel": "grouped_gemm gate/up + SwiGLU (forward)",
                     "achieved": dom_tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": dom_tflops / pk["bf16_tflops"], "peak_source": f"{pk_kind} bf16 burst",
                     "traffic": traffic},
        "e2e": {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": int(hx.numel() * 2 + hdy.numel() * 2),
                "d2h_bytes_per_step": int(hy.numel() * 2 + hdx.numel() * 2),
                "copies": "pinned host x, dY in and y, dX out every step, on two copy streams; "
                          "step i+1's inputs and step i-1's outputs move during step i"},
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clk.summary(),
    }
    if args.cpu_baseline:
        t0 = time.perf_counter()
        oracle_sample_step(inp, args.cpu_tokens)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": args.cpu_tokens / dt, "unit": "tokens/s", "cores": cpu_cores_used(),
                                "kind": "oracle",
                                "sample": f"first {args.cpu_tokens} tokens of {WORKLOAD}, forward+backward, "
                                          f"single-threaded C oracle, {dt:.1f} s"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


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


# kernels launched per step by the calls in run_ours.step():
# route 4 (zero counters, partial logits, top-k, offsets), dispatch 3,
# gate/up 1, down 1, combine 1, combine_bwd 1, down_bwd 3 and gate/up bwd 3
# (dX GEMM, segment maps, dW GEMM), dispatch_bwd 1, route_bwd 7
KERNELS_PER_STEP = 4 + 3 + 1 + 1 + 1 + 1 + 3 + 3 + 1 + 7


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
    """Untimed forward+backward passes of one layer shape (for ncu captures)."""
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
        layer.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
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
    ap.add_argument("--profile-fp8", default=None, metavar="T,H,I,E,k",
                    help="run --steps untimed fp8 forward passes of this shape and exit")
    args = ap.parse_args(argv)
    if args.profile_router:
        return run_profile_router(args)
    if args.profile_case:
        return run_profile_case(args)
    if args.profile_fp8:
        return run_profile_fp8(args)
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
