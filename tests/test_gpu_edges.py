"""Edge cases of the CUDA path against the CPU oracle: one token, one expert
(a plain SwiGLU MLP), logit ties, k = E, the largest E and k (1024, 32), empty
experts, every token on one expert,
segmented (source-rank x expert) row layouts, gradient accumulation, and the
device status word for bad index data (kernels skip the bad entries)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import assert_close, inputs, oracle_backward, oracle_chain, to_dev, dispatch_ws
from moe_expert_layer_topk_gb300.synth import LayerShape, bf16_bits, make_segment_inputs

pytestmark = pytest.mark.gpu


def run_layer(inp, bias=None):
    g = to_dev(inp)
    L = m.MoELayer(inp["T"], inp["H"], inp["I"], inp["E"], inp["k"], inp["ep_size"])
    L.forward(g["x"], g["Wr"], g["bias"] if bias is None else bias, g["Wg"], g["Wu"], g["Wd"])
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    return L, g


def check_all(L, inp):
    f = oracle_chain(inp)
    b = oracle_backward(inp, f)
    assert np.array_equal(L.topk_idx.cpu().numpy(), f["rt"]["topk_idx"])
    assert np.array_equal(L.offsets.cpu().numpy(), f["rt"]["offsets"])
    assert np.array_equal(L.row_of_slot.cpu().numpy(), f["dp"]["row_of_slot"])
    assert_close(L.y, f["y"], "y")
    for name in ("dx", "dWg", "dWu", "dWd", "dWr"):
        assert_close(getattr(L, name), b[name], name)
    return f, b


def test_single_token():
    inp = inputs(1, 128, 64, 8, 2, seed=11, ep=2)
    L, _ = run_layer(inp)
    check_all(L, inp)


def test_one_expert_is_a_dense_swiglu_mlp():
    inp = inputs(300, 256, 128, 1, 1, seed=12)
    L, g = run_layer(inp)
    check_all(L, inp)
    assert torch.all(L.topk_w == 1.0)
    # independent fp32 torch reference of the dense MLP
    x = g["x"].float()
    ref = (F.silu(x @ g["Wg"][0].float().T) * (x @ g["Wu"][0].float().T)) @ g["Wd"][0].float().T
    assert_close(L.y, ref.cpu().numpy(), "y vs torch fp32 MLP")


def test_router_ties():
    """Equal logits go to the lower expert id: duplicated router columns
    (experts 5 = 2 and 6 = 1), zeroed columns (experts 0, 3, 7: logit 0 for
    every token) and all-zero tokens (every logit 0, so experts 0..k-1 in
    order, with equal weights)."""
    inp = inputs(160, 256, 64, 8, 3, seed=21, ep=2, router_std=0.05)
    Wr = inp["Wr"].clone()
    Wr[:, 5] = Wr[:, 2]
    Wr[:, 6] = Wr[:, 1]
    Wr[:, [0, 3, 7]] = 0.0
    inp["Wr"] = Wr
    x = inp["x"].clone()
    x[[4, 77, 159]] = 0.0
    inp["x"] = x
    L, _ = run_layer(inp)
    f, _ = check_all(L, inp)
    idx = L.topk_idx.cpu().numpy()
    for t in (4, 77, 159):
        assert idx[t].tolist() == [0, 1, 2]
        assert torch.all(L.topk_w[t] == L.topk_w[t, 0])
    # a tie inside the selection picks the lower id first
    ties = (idx[:, :, None] == np.array([2, 5])).any(1).all(1)
    for t in np.nonzero(ties)[0]:
        row = idx[t].tolist()
        assert row.index(2) < row.index(5)


def test_k_equals_E():
    inp = inputs(200, 128, 64, 4, 4, seed=13, router_std=0.3)
    L, _ = run_layer(inp)
    check_all(L, inp)
    w = L.topk_w.cpu().double()
    assert torch.allclose(w.sum(1), torch.ones(200, dtype=torch.float64), atol=1e-6)


def test_empty_experts_and_accumulate():
    inp = inputs(400, 128, 128, 8, 2, seed=14, router_std=0.3)
    bias = torch.zeros(8)
    bias[[1, 5, 6]] = -1.0e4
    inp["bias"] = bias
    L, g = run_layer(inp)
    counts = L.counts.cpu().numpy()
    assert counts[1] == counts[5] == counts[6] == 0
    check_all(L, inp)
    for name in ("dWg", "dWu", "dWd"):
        t = getattr(L, name)
        assert torch.count_nonzero(t[[1, 5, 6]]) == 0, name
    keep = {n: getattr(L, n).clone() for n in ("dWg", "dWu", "dWd", "dWr")}
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], accumulate=True)
    torch.cuda.synchronize()
    for n, v in keep.items():
        assert torch.equal(getattr(L, n), v + v), n   # prev + identical fresh sum


def test_every_token_on_one_expert():
    inp = inputs(1000, 256, 128, 8, 1, seed=15)
    bias = torch.zeros(8)
    bias[3] = 1.0e4
    inp["bias"] = bias
    L, _ = run_layer(inp)
    assert L.counts.cpu().tolist() == [0, 0, 0, 1000, 0, 0, 0, 0]
    check_all(L, inp)


def test_maximum_experts_and_topk():
    """The ABI's largest expert count and top-k together: E = 1024, k = 32,
    EP over 8 ranks.  3072 slots over 1024 experts leave most experts with
    a few rows and many with none; forward and backward against the oracle."""
    inp = inputs(96, 128, 64, 1024, 32, seed=21, ep=8, router_std=0.3)
    L, _ = run_layer(inp)
    f, _ = check_all(L, inp)
    counts = L.counts.cpu().numpy()
    assert counts.sum() == 96 * 32 and (counts == 0).any()
    assert np.array_equal(L.rank_offsets.cpu().numpy(), f["rt"]["rank_offsets"])
    assert np.array_equal(f["rt"]["rank_offsets"], f["rt"]["offsets"][::128])


def test_zero_tokens():
    L = m.MoELayer(0, 128, 64, 8, 2, 2)
    x = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    Wr = torch.randn(128, 8, device="cuda")
    m.moe_route_topk(x, Wr, None, 0, 128, 8, 2, 2, L.topk_idx, L.topk_w, L.counts, L.offsets,
                     L.rank_offsets, L.ws_route)
    torch.cuda.synchronize()
    assert L.counts.cpu().tolist() == [0] * 8
    assert L.offsets.cpu().tolist() == [0] * 9
    assert L.rank_offsets.cpu().tolist() == [0, 0, 0]


@pytest.mark.parametrize("R,H,I,E,S", [(1500, 256, 128, 4, 3), (700, 128, 192, 6, 2)])
def test_segmented_rows(R, H, I, E, S):
    """Receive-side layout: (source rank x local expert) segments, some empty;
    the weight gradient of an expert sums over all its segments."""
    shape = LayerShape(T=R, H=H, I=I, E=E, k=1, ep_size=1, segments=True, src_ranks=S)
    s = make_segment_inputs(shape, seed=16)
    so = s["seg_offsets"].clone()
    so[3] = so[2]              # segment 2 empty
    so[4:] = torch.maximum(so[4:], so[3])
    se = s["seg_expert"]
    dev = "cuda"
    xp, Wg, Wu, Wd = (s[n].to(dev) for n in ("x_perm", "Wg", "Wu", "Wd"))
    so_d, se_d = so.to(dev), se.to(dev)
    nseg = len(so) - 1
    h = torch.zeros(R, I, dtype=torch.bfloat16, device=dev)
    gu = torch.zeros(R, 2 * I, dtype=torch.bfloat16, device=dev)
    y = torch.zeros(R, H, dtype=torch.bfloat16, device=dev)
    m.moe_grouped_gemm_swiglu(xp, Wg, Wu, nseg, so_d, se_d, R, H, I, E, h, gu)
    m.moe_grouped_gemm_down(h, Wd, nseg, so_d, se_d, R, H, I, E, y)
    dy_host = torch.randn(R, H, generator=torch.Generator().manual_seed(29)).to(torch.bfloat16)
    dy = dy_host.to(dev)
    dgu = torch.zeros(R, 2 * I, dtype=torch.bfloat16, device=dev)
    dWd = torch.empty(E, H, I, device=dev)
    dx = torch.zeros(R, H, dtype=torch.bfloat16, device=dev)
    dWg = torch.empty(E, I, H, device=dev)
    dWu = torch.empty(E, I, H, device=dev)
    ws = torch.empty(m.moe_grouped_gemm_bwd_workspace_size(nseg), dtype=torch.uint8, device=dev)
    m.moe_grouped_gemm_down_bwd(dy, h, gu, Wd, nseg, so_d, se_d, R, H, I, E, dgu, dWd, 0, ws)
    m.moe_grouped_gemm_swiglu_bwd(dgu, xp, Wg, Wu, nseg, so_d, se_d, R, H, I, E, dx, dWg, dWu, 0, ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    son, sen = so.numpy(), se.numpy()
    xo = oracle.widen_bf16(bf16_bits(s["x_perm"]))
    h_ref, gu_ref = oracle.grouped_gemm_swiglu(xo, bf16_bits(s["Wg"]), bf16_bits(s["Wu"]), son, sen,
                                               save_gu=True)
    covered = slice(int(son[0]), int(son[-1]))
    assert_close(h[covered], h_ref[covered], "h")
    # the oracle's own chain from here on (its fp32 h, g|u and dgu)
    y_ref = oracle.grouped_gemm_down(h_ref, bf16_bits(s["Wd"]), son, sen)
    assert_close(y[covered], y_ref[covered], "y_perm")
    dy_ref = oracle.widen_bf16(bf16_bits(dy_host))
    dgu_ref, dWd_ref = oracle.grouped_gemm_down_bwd(dy_ref, h_ref, gu_ref, bf16_bits(s["Wd"]), son, sen)
    assert_close(dgu[covered], dgu_ref[covered], "dgu")
    assert_close(dWd, dWd_ref, "dWd")
    dx_ref, dWg_ref, dWu_ref = oracle.grouped_gemm_swiglu_bwd(dgu_ref, xo, bf16_bits(s["Wg"]),
                                                              bf16_bits(s["Wu"]), son, sen)
    assert_close(dx[covered], dx_ref[covered], "dx_perm")
    assert_close(dWg, dWg_ref, "dWg")
    assert_close(dWu, dWu_ref, "dWu")


def test_identity_table_with_fewer_segments_than_experts():
    """A null seg_expert with num_seg < E: segment s holds expert s's rows and
    the experts past the last segment have none, so their weight gradients
    are zeros, or stay as they were when accumulating."""
    R, H, I, E = 400, 128, 128, 6
    shape = LayerShape(T=R, H=H, I=I, E=E, k=1, ep_size=1, segments=True, src_ranks=1)
    s = make_segment_inputs(shape, seed=23)
    so = torch.tensor([0, 100, 100, 250, 400], dtype=torch.int32)  # segment 1 empty
    dev = "cuda"
    xp, Wg, Wu, Wd = (s[n].to(dev) for n in ("x_perm", "Wg", "Wu", "Wd"))
    so_d = so.to(dev)
    nseg = len(so) - 1
    h = torch.zeros(R, I, dtype=torch.bfloat16, device=dev)
    gu = torch.zeros(R, 2 * I, dtype=torch.bfloat16, device=dev)
    m.moe_grouped_gemm_swiglu(xp, Wg, Wu, nseg, so_d, None, R, H, I, E, h, gu)
    dy_host = torch.randn(R, H, generator=torch.Generator().manual_seed(31)).to(torch.bfloat16)
    dy = dy_host.to(dev)
    dgu = torch.zeros(R, 2 * I, dtype=torch.bfloat16, device=dev)
    dx = torch.zeros(R, H, dtype=torch.bfloat16, device=dev)
    dWd = torch.full((E, H, I), float("nan"), device=dev)
    dWg = torch.full((E, I, H), float("nan"), device=dev)
    dWu = torch.full((E, I, H), float("nan"), device=dev)
    ws = torch.empty(m.moe_grouped_gemm_bwd_workspace_size(nseg), dtype=torch.uint8, device=dev)
    m.moe_grouped_gemm_down_bwd(dy, h, gu, Wd, nseg, so_d, None, R, H, I, E, dgu, dWd, 0, ws)
    m.moe_grouped_gemm_swiglu_bwd(dgu, xp, Wg, Wu, nseg, so_d, None, R, H, I, E, dx, dWg, dWu, 0, ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    son = so.numpy()
    xo = oracle.widen_bf16(bf16_bits(s["x_perm"]))
    h_ref, gu_ref = oracle.grouped_gemm_swiglu(xo, bf16_bits(s["Wg"]), bf16_bits(s["Wu"]), son,
                                               save_gu=True)
    dy_ref = oracle.widen_bf16(bf16_bits(dy_host))
    dgu_ref, dWd_ref = oracle.grouped_gemm_down_bwd(dy_ref, h_ref, gu_ref, bf16_bits(s["Wd"]), son)
    dx_ref, dWg_ref, dWu_ref = oracle.grouped_gemm_swiglu_bwd(dgu_ref, xo, bf16_bits(s["Wg"]),
                                                              bf16_bits(s["Wu"]), son)
    for ref in (dWd_ref, dWg_ref, dWu_ref):
        assert np.all(ref[nseg:] == 0) and np.all(ref[1] == 0)
    assert_close(dgu, dgu_ref, "dgu")
    assert_close(dWd, dWd_ref, "dWd")
    assert_close(dx, dx_ref, "dx_perm")
    assert_close(dWg, dWg_ref, "dWg")
    assert_close(dWu, dWu_ref, "dWu")
    # accumulating: experts without rows keep their values bit for bit
    before = [t.clone() for t in (dWd, dWg, dWu)]
    m.moe_grouped_gemm_down_bwd(dy, h, gu, Wd, nseg, so_d, None, R, H, I, E, dgu, dWd, 1, ws)
    m.moe_grouped_gemm_swiglu_bwd(dgu, xp, Wg, Wu, nseg, so_d, None, R, H, I, E, dx, dWg, dWu, 1, ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    for t, b in zip((dWd, dWg, dWu), before):
        assert torch.equal(t[nseg:], b[nseg:]) and torch.equal(t[1], b[1])
        assert torch.equal(t[[0, 2, 3]], 2 * b[[0, 2, 3]])

def test_bad_index_data_sets_status_without_fault():
    """Out-of-range expert ids and offsets that disagree with them are skipped
    by the kernels and reported through the device status word."""
    inp = inputs(64, 128, 64, 8, 2, seed=17)
    g = to_dev(inp)
    L = m.MoELayer(64, 128, 64, 8, 2, 2)
    L.route(g["x"], g["Wr"], None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    bad = L.topk_idx.clone()
    bad[5, 1] = 8          # expert id == E
    bad[9, 0] = -3
    m.moe_dispatch(g["x"], bad, L.offsets, 64, 128, 8, 2, L.x_perm, L.row_of_slot, L.token_of_row,
                   dispatch_ws(64, 8, 2))
    torch.cuda.synchronize()
    st = m.moe_read_device_status(reset=True)
    assert st & 1, st  # MOE_STATUS_BAD_INDEX
    assert L.row_of_slot[5, 1].item() == -1 and L.row_of_slot[9, 0].item() == -1
    # segment table running past R
    so = L.offsets.clone()
    so[-1] = 64 * 2 + 500
    m.moe_grouped_gemm_swiglu(L.x_perm, g["Wg"], g["Wu"], 8, so, None, 128, 128, 64, 8, L.h, None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) & 2  # MOE_STATUS_BAD_SEGMENTS
