"""The fused down projection + combine (moe_grouped_gemm_down_combine) against
the oracle: y = sum over a token's slots of w * (h . Wd[e]^T), added in fp32
in no fixed order, rounded to bf16 once.  Compared with the oracle's own fp32
chain (the same bars as every float output), and with the unfused
down + combine path of the library."""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import assert_close, bits, inputs, oracle_chain, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    # T,   H,   I,  E, k  (rows per expert: single-CTA tiles below 384, pairs above)
    "small": (256, 128, 64, 8, 2),
    "odd": (300, 192, 192, 6, 3),
    "pairs": (1024, 256, 128, 4, 2),
    "many_experts": (160, 512, 256, 40, 5),
}


def _layers(T, H, I, E, k, fused_dispatch):
    a = m.MoELayer(T, H, I, E, k, 1, training=False, fused_dispatch=fused_dispatch, fused_combine=True)
    b = m.MoELayer(T, H, I, E, k, 1, training=False)
    return a, b


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("fused_dispatch", [False, True])
def test_fused_combine_matches_oracle(name, fused_dispatch):
    T, H, I, E, k = CASES[name]
    inp = inputs(T, H, I, E, k, seed=40 + sorted(CASES).index(name), with_dy=False)
    g = to_dev(inp)
    fused, plain = _layers(T, H, I, E, k, fused_dispatch)
    assert fused.y_perm is None  # the permuted output rows are never materialised
    y = fused.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"]).clone()
    y_plain = plain.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"]).clone()
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    f = oracle_chain(inp)
    assert np.array_equal(fused.row_of_slot.cpu().numpy(), f["dp"]["row_of_slot"])
    assert_close(y, f["y"], "y (fused combine)")
    assert_close(y_plain, f["y"], "y (down, then combine)")
    # the fused path skips the bf16 rounding of y_perm: it is at least as
    # close to the oracle's fp32 chain as the unfused one, up to the last bf16 ulp
    ref = f["y"].astype(np.float64)
    e_fused = np.linalg.norm(y.float().cpu().numpy() - ref)
    e_plain = np.linalg.norm(y_plain.float().cpu().numpy() - ref)
    assert e_fused <= 1.05 * e_plain + 1e-6, (e_fused, e_plain)


def test_fused_combine_skips_unmatched_slots():
    """A slot whose row_of_slot entry is -1 contributes nothing (its row's
    token no longer points back to it); a token left with no slot gets y = 0."""
    T, H, I, E, k = 64, 128, 64, 4, 2
    inp = inputs(T, H, I, E, k, seed=47, with_dy=False)
    g = to_dev(inp)
    L = m.MoELayer(T, H, I, E, k, 1, training=False)
    L.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    ros = L.row_of_slot.clone()
    ros[5, 1] = -1
    ros[9, 0] = -1
    ros[9, 1] = -1  # token 9: no slot left
    y_acc = torch.empty(T, H, dtype=torch.float32, device="cuda")
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_down_combine(L.h, g["Wd"], E, L.offsets, None, L.R, H, I, E, L.token_of_row, ros,
                                    L.topk_w, T, k, y_acc, y)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    # expected: the oracle's down projection of the layer's own h (bf16),
    # combined over the slots that remain
    yp = oracle.grouped_gemm_down(oracle.widen_bf16(bits(L.h)), bits(inp["Wd"]), L.offsets.cpu().numpy())
    w = L.topk_w.cpu().numpy().copy()
    r = ros.cpu().numpy().copy()
    w[r < 0] = 0.0
    r[r < 0] = 0
    ref = oracle.combine(yp, w, r)
    assert np.all(ref[9] == 0)
    assert torch.all(y[9] == 0)
    assert_close(y, ref, "y with skipped slots")


def test_fused_combine_full_size_against_unfused():
    """T=4096 at the Qwen3-30B-A3B shapes (pairs of 256-row tiles are not
    taken at ~256 rows per expert; the 'pairs' case covers them): the fused
    and unfused forwards agree within the bf16 bars."""
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_layer_inputs
    shape = CONFIGS["qwen3_30b_fwd"]
    inp = make_layer_inputs(shape, 0, with_dy=False)
    g = to_dev(inp)
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    fused, plain = _layers(T, H, I, E, k, True)
    y = fused.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"]).clone()
    y_plain = plain.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"]).clone()
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(fused.topk_idx, plain.topk_idx)
    assert_close(y, y_plain.float().cpu().numpy(), "y fused vs unfused (T=4096)")
