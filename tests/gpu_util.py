"""Helpers shared by the GPU parity tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_expert_layer_topk_gb300.synth import LayerShape, bf16_bits, make_layer_inputs

# Acceptance for floating-point outputs and gradients (bf16 storage):
MAX_ABS_FRAC = 2e-2     # max |err| <= 2e-2 * max |ref|
REL_L2 = 5e-3           # ||err||_2 / ||ref||_2 <= 5e-3


def assert_close(got, ref, what, max_frac=MAX_ABS_FRAC, rel=REL_L2):
    if isinstance(got, torch.Tensor):
        got = got.detach().float().cpu().numpy()
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    nrm = np.linalg.norm(ref)
    r = np.linalg.norm(got - ref) / (nrm if nrm > 0 else 1.0)
    if scale == 0:
        assert err.max() == 0, f"{what}: expected exact zeros, max err {err.max()}"
        return
    assert err.max() <= max_frac * scale, f"{what}: max err {err.max():.3e} > {max_frac} * {scale:.3e}"
    assert r <= rel, f"{what}: rel L2 {r:.3e} > {rel}"


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> uint16 bit patterns on the host."""
    return bf16_bits(t.detach().cpu())


def f32(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 tensor (any device) -> fp32 numpy (exact widening)."""
    return t.detach().float().cpu().numpy()


def shape(T, H, I, E, k, ep=1):
    return LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=ep)


def inputs(T, H, I, E, k, seed=0, ep=1, bias=None, with_dy=True, router_std=0.02):
    inp = make_layer_inputs(shape(T, H, I, E, k, ep), seed, with_dy=with_dy, bias=bias,
                            router_std=router_std)
    return inp


def to_dev(inp, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def oracle_chain(inp, save_gu=True):
    """Oracle forward chain on the host copies of `inp` (fp32 intermediates)."""
    x = bits(inp["x"])
    Wr = inp["Wr"].numpy()
    bias = None if inp.get("bias") is None else inp["bias"].numpy()
    rt = oracle.route_topk(x, Wr, bias, inp["k"], inp.get("ep_size", 1))
    dp = oracle.dispatch(x, rt["topk_idx"], rt["offsets"], inp["E"])
    xp = oracle.widen_bf16(dp["x_perm"])
    h, gu = oracle.grouped_gemm_swiglu(xp, bits(inp["Wg"]), bits(inp["Wu"]), rt["offsets"], save_gu=True)
    yp = oracle.grouped_gemm_down(h, bits(inp["Wd"]), rt["offsets"])
    y = oracle.combine(yp, rt["topk_w"], dp["row_of_slot"])
    return dict(rt=rt, dp=dp, x=x, Wr=Wr, x_perm=xp, h=h, gu=gu, y_perm=yp, y=y)


def oracle_backward(inp, f):
    dy = oracle.widen_bf16(bits(inp["dy"]))
    dyp, dw = oracle.combine_bwd(dy, f["y_perm"], f["rt"]["topk_w"], f["dp"]["row_of_slot"])
    dgu, dWd = oracle.grouped_gemm_down_bwd(dyp, f["h"], f["gu"], bits(inp["Wd"]), f["rt"]["offsets"])
    dxp, dWg, dWu = oracle.grouped_gemm_swiglu_bwd(dgu, f["x_perm"], bits(inp["Wg"]), bits(inp["Wu"]),
                                                   f["rt"]["offsets"])
    dxa = oracle.dispatch_bwd(dxp, f["dp"]["row_of_slot"])
    dWr, dx = oracle.route_topk_bwd(dw, f["rt"]["topk_w"], f["rt"]["topk_idx"], f["x"], f["Wr"], dxa)
    return dict(dy_perm=dyp, d_w=dw, dgu=dgu, dWd=dWd, dx_perm=dxp, dWg=dWg, dWu=dWu, dx_acc=dxa,
                dWr=dWr, dx=dx)


def dispatch_ws(T, E, k):
    """A workspace for moe_dispatch / moe_dispatch_e4m3 (the layer itself
    dispatches from the route's chunk prefixes and keeps none)."""
    import moe_expert_layer_topk_gb300 as m
    return torch.empty(max(256, m.moe_dispatch_workspace_size(T, E, k)), dtype=torch.uint8, device="cuda")
