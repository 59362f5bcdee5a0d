"""moe_grouped_gemm_swiglu_gather: the gate/up GEMM reading its permuted rows
straight from x by token id (no x_perm in memory).  It must reproduce
moe_dispatch + moe_grouped_gemm_swiglu bit for bit, and through them the
oracle; dispatch with x_perm = NULL must rank exactly as with the copy."""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import assert_close, bits, inputs, oracle_chain, to_dev, dispatch_ws
from moe_expert_layer_topk_gb300.synth import CONFIGS, make_layer_inputs

pytestmark = pytest.mark.gpu

CASES = {
    # T,   H,   I,   E,  k, ep, bias
    "tiny": (256, 128, 64, 8, 2, 2, None),
    "odd_tiles": (300, 192, 192, 6, 2, 3, None),
    "zipf_empty_experts": (500, 128, 128, 16, 4, 4, "zipf"),
    "wide": (600, 256, 256, 8, 3, 4, None),
}


def _route(L, g):
    L.route(g["x"], g["Wr"], g["bias"])


@pytest.mark.parametrize("case", sorted(CASES))
def test_gather_matches_permuted_path_and_oracle(case):
    T, H, I, E, k, ep, bias = CASES[case]
    inp = inputs(T, H, I, E, k, seed=7, ep=ep, bias=bias, router_std=0.02 if bias is None else 0.3)
    g = to_dev(inp)
    L = m.MoELayer(T, H, I, E, k, ep)
    _route(L, g)
    L.dispatch(g["x"])
    R = L.R
    h_ref = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    gu_ref = torch.empty(R, 2 * I, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_swiglu(L.x_perm, g["Wg"], g["Wu"], E, L.offsets, None, R, H, I, E, h_ref, gu_ref)
    # ranking only: must give the same rows
    rows = L.row_of_slot.clone()
    tok = L.token_of_row.clone()
    m.moe_dispatch(g["x"], L.topk_idx, L.offsets, T, H, E, k, None, L.row_of_slot, L.token_of_row,
                   dispatch_ws(T, E, k))
    h = torch.empty_like(h_ref)
    gu = torch.empty_like(gu_ref)
    m.moe_grouped_gemm_swiglu_gather(g["x"], L.token_of_row, T, g["Wg"], g["Wu"], E, L.offsets, None, R, H,
                                     I, E, h, gu)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(L.row_of_slot, rows) and torch.equal(L.token_of_row, tok)
    assert torch.equal(h, h_ref), "gathered rows must give the permuted path's h bit for bit"
    assert torch.equal(gu, gu_ref)
    f = oracle_chain(inp)
    assert_close(h, f["h"], "h")


def test_gather_full_size_bit_exact():
    shape = CONFIGS["qwen3_30b_fwd"]
    inp = make_layer_inputs(shape, 0)
    g = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in inp.items()}
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    L = m.MoELayer(T, H, I, E, k, shape.ep_size, training=False)
    L.route(g["x"], g["Wr"], g["bias"])
    L.dispatch(g["x"])
    R = L.R
    h_ref = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_swiglu(L.x_perm, g["Wg"], g["Wu"], E, L.offsets, None, R, H, I, E, h_ref, None)
    h = torch.empty_like(h_ref)
    m.moe_grouped_gemm_swiglu_gather(g["x"], L.token_of_row, T, g["Wg"], g["Wu"], E, L.offsets, None, R, H, I,
                                     E, h, None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(h, h_ref)


def test_gather_segments_and_arbitrary_rows():
    # rows taken from x in any order, over (source rank x expert) segments
    T, H, I, E = 96, 128, 64, 4
    gen = torch.Generator().manual_seed(3)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16).cuda()
    Wg = (torch.randn(E, I, H, generator=gen) * 0.02).to(torch.bfloat16).cuda()
    Wu = (torch.randn(E, I, H, generator=gen) * 0.02).to(torch.bfloat16).cuda()
    R = 300
    tor = torch.randint(0, T, (R,), generator=gen, dtype=torch.int32).cuda()
    so = torch.tensor([0, 40, 40, 170, 200, 299, 300], dtype=torch.int32).cuda()  # one empty segment
    se = torch.tensor([2, 0, 1, 3, 0, 2], dtype=torch.int32).cuda()
    xp = x[tor.long()].contiguous()
    h_ref = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_swiglu(xp, Wg, Wu, 6, so, se, R, H, I, E, h_ref, None)
    h = torch.empty_like(h_ref)
    m.moe_grouped_gemm_swiglu_gather(x, tor, T, Wg, Wu, 6, so, se, R, H, I, E, h, None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(h, h_ref)
    x_host = x.cpu()[tor.cpu().long()]  # the seeded rows, gathered on the host
    href = oracle.grouped_gemm_swiglu(oracle.widen_bf16(bits(x_host)), bits(Wg.cpu()), bits(Wu.cpu()),
                                      so.cpu().numpy(), se.cpu().numpy())
    assert_close(h, href, "h")


def test_gather_bad_token_id_sets_status():
    T, H, I, E = 32, 128, 64, 2
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros(E, I, H, dtype=torch.bfloat16, device="cuda")
    Wu = torch.zeros_like(Wg)
    tor = torch.zeros(64, dtype=torch.int32, device="cuda")
    tor[5] = T + 7
    so = torch.tensor([0, 32, 64], dtype=torch.int32, device="cuda")
    h = torch.empty(64, I, dtype=torch.bfloat16, device="cuda")
    m.moe_read_device_status(reset=True)
    m.moe_grouped_gemm_swiglu_gather(x, tor, T, Wg, Wu, 2, so, None, 64, H, I, E, h, None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) & 1  # MOE_STATUS_BAD_INDEX


def test_layer_fused_dispatch_forward_matches():
    T, H, I, E, k, ep = 400, 256, 128, 16, 4, 4
    inp = inputs(T, H, I, E, k, seed=11, ep=ep)
    g = to_dev(inp)
    ref = m.MoELayer(T, H, I, E, k, ep, training=False)
    fused = m.MoELayer(T, H, I, E, k, ep, training=False, fused_dispatch=True)
    assert fused.x_perm is None
    y_ref = ref.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"]).clone()
    y = fused.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(y, y_ref)
    with pytest.raises(ValueError):
        m.MoELayer(T, H, I, E, k, ep, training=True, fused_dispatch=True)
