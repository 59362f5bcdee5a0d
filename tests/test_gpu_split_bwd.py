"""The backward GEMM calls issued as separate dX and weight-gradient halves
give bit for bit what the combined calls give: on the dispatch layout, on a
(source rank x expert) segment layout with accumulation, and with the two
halves running concurrently on two streams."""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
from gpu_util import assert_close, inputs, oracle_backward, oracle_chain, to_dev
from moe_expert_layer_topk_gb300.synth import LayerShape, make_segment_inputs

pytestmark = pytest.mark.gpu


def _aligned_ws(num_seg):
    raw = torch.empty(m.moe_grouped_gemm_bwd_workspace_size(num_seg) + 256, dtype=torch.uint8, device="cuda")
    off = (-raw.data_ptr()) % 128
    return raw[off:off + m.moe_grouped_gemm_bwd_workspace_size(num_seg)]


def test_split_halves_equal_combined_calls_dispatch_layout():
    inp = inputs(600, 256, 192, 12, 3, seed=81)
    g = to_dev(inp)
    T, H, I, E, k = 600, 256, 192, 12, 3
    L = m.MoELayer(T, H, I, E, k, 1)
    L.forward(g["x"], g["Wr"], None, g["Wg"], g["Wu"], g["Wd"])
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    R = L.R
    ws = _aligned_ws(E)
    dgu = torch.empty_like(L.dgu)
    dWd = torch.empty_like(L.dWd)
    m.moe_grouped_gemm_down_bwd_dx(L.dy_perm, L.gu, g["Wd"], E, L.offsets, None, R, H, I, E, dgu)
    m.moe_grouped_gemm_down_bwd_dw(L.dy_perm, L.h, E, L.offsets, None, R, H, I, E, dWd, 0, ws)
    dx_perm = torch.empty_like(L.dx_perm)
    dWg, dWu = torch.empty_like(L.dWg), torch.empty_like(L.dWu)
    m.moe_grouped_gemm_swiglu_bwd_dx(dgu, g["Wg"], g["Wu"], E, L.offsets, None, R, H, I, E, dx_perm)
    m.moe_grouped_gemm_swiglu_bwd_dw(dgu, L.x_perm, E, L.offsets, None, R, H, I, E, dWg, dWu, 0, ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    for name, got in (("dgu", dgu), ("dWd", dWd), ("dx_perm", dx_perm), ("dWg", dWg), ("dWu", dWu)):
        assert torch.equal(got, getattr(L, name)), name
    # and the layer's chain is the oracle's
    b = oracle_backward(inp, oracle_chain(inp))
    for name in ("dWd", "dWg", "dWu"):
        assert_close(getattr(L, name), b[name], name)


def test_split_halves_segments_accumulate_two_streams():
    shape = LayerShape(T=1500, H=256, I=128, E=6, k=1, ep_size=1, segments=True, src_ranks=4)
    s = make_segment_inputs(shape, seed=82)
    R, H, I, E, S = 1500, 256, 128, 6, 24
    g = {n: (v.cuda() if isinstance(v, torch.Tensor) else v) for n, v in s.items()}
    gen = torch.Generator(device="cuda").manual_seed(3)
    rnd = lambda *sh: torch.randn(*sh, device="cuda", generator=gen).to(torch.bfloat16)
    dy_perm, h, gu = rnd(R, H), rnd(R, I), rnd(R, 2 * I)
    so, se = g["seg_offsets"], g["seg_expert"]
    prev = [torch.randn(E, H, I, device="cuda", generator=gen), torch.randn(E, I, H, device="cuda", generator=gen),
            torch.randn(E, I, H, device="cuda", generator=gen)]
    ws = _aligned_ws(S)
    # combined calls, accumulating into copies of prev
    dgu_c = torch.empty(R, 2 * I, dtype=torch.bfloat16, device="cuda")
    dx_c = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    dWd_c, dWg_c, dWu_c = (p.clone() for p in prev)
    m.moe_grouped_gemm_down_bwd(dy_perm, h, gu, g["Wd"], S, so, se, R, H, I, E, dgu_c, dWd_c, 1, ws)
    m.moe_grouped_gemm_swiglu_bwd(dgu_c, g["x_perm"], g["Wg"], g["Wu"], S, so, se, R, H, I, E, dx_c, dWg_c,
                                  dWu_c, 1, ws)
    torch.cuda.synchronize()
    # halves: the dX half of each call on a second stream, beside the dW half
    ws2 = _aligned_ws(S)
    dgu = torch.empty_like(dgu_c)
    dx = torch.empty_like(dx_c)
    dWd, dWg, dWu = (p.clone() for p in prev)
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    m.moe_grouped_gemm_down_bwd_dx(dy_perm, gu, g["Wd"], S, so, se, R, H, I, E, dgu)
    ev = torch.cuda.Event()
    ev.record(main)
    side.wait_event(ev)
    m.moe_grouped_gemm_swiglu_bwd_dx(dgu, g["Wg"], g["Wu"], S, so, se, R, H, I, E, dx, stream=side)
    m.moe_grouped_gemm_down_bwd_dw(dy_perm, h, S, so, se, R, H, I, E, dWd, 1, ws)
    m.moe_grouped_gemm_swiglu_bwd_dw(dgu, g["x_perm"], S, so, se, R, H, I, E, dWg, dWu, 1, ws2)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    covered = slice(int(s["seg_offsets"][0]), int(s["seg_offsets"][-1]))
    assert torch.equal(dgu[covered], dgu_c[covered])
    assert torch.equal(dx[covered], dx_c[covered])
    for name, got, ref in (("dWd", dWd, dWd_c), ("dWg", dWg, dWg_c), ("dWu", dWu, dWu_c)):
        assert torch.equal(got, ref), name
    assert not torch.equal(dWd, prev[0])



def test_sm_limit_changes_no_result():
    """A limit on the GEMMs' persistent grid (here 20 SMs, and 1) changes
    nothing in the results; the previous limit comes back."""
    inp = inputs(700, 256, 128, 10, 3, seed=83)
    g = to_dev(inp)
    T, H, I, E, k = 700, 256, 128, 10, 3
    L = m.MoELayer(T, H, I, E, k, 1)
    L.forward(g["x"], g["Wr"], None, g["Wg"], g["Wu"], g["Wd"])
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], overlap=False)
    torch.cuda.synchronize()
    ref = {n: getattr(L, n).clone() for n in ("y", "dgu", "dx_perm", "dWg", "dWu", "dWd", "dWr", "dx")}
    for limit in (20, 1):
        assert m.moe_set_gemm_sm_limit(limit) == 0
        try:
            L.forward(g["x"], g["Wr"], None, g["Wg"], g["Wu"], g["Wd"])
            L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], overlap=False)
        finally:
            assert m.moe_set_gemm_sm_limit(0) == limit
        torch.cuda.synchronize()
        assert m.moe_read_device_status(reset=True) == 0
        for n, v in ref.items():
            assert torch.equal(getattr(L, n), v), (limit, n)


def test_layer_backward_overlap_matches_one_stream():
    """The backward with its dispatch and router tail on a side stream gives
    the one-stream results bit for bit, also on a caller's own stream and
    with accumulation into the weight gradients."""
    inp = inputs(900, 256, 128, 16, 4, seed=84, ep=2)
    g = to_dev(inp)
    T, H, I, E, k = 900, 256, 128, 16, 4
    L = m.MoELayer(T, H, I, E, k, 2)
    L.forward(g["x"], g["Wr"], None, g["Wg"], g["Wu"], g["Wd"])
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], overlap=False)
    torch.cuda.synchronize()
    names = ("dgu", "dx_perm", "dx_acc", "dWg", "dWu", "dWd", "dWr", "dx")
    ref = {n: getattr(L, n).clone() for n in names}
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for n in names:
            getattr(L, n).fill_(7.0)
        L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], stream=s)
    s.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    for n in names:
        assert torch.equal(getattr(L, n), ref[n]), n
    # accumulate: a second overlapped pass adds the same gradients again
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], accumulate=True)
    torch.cuda.synchronize()
    for n in ("dWg", "dWu", "dWd", "dWr"):
        assert torch.equal(getattr(L, n), ref[n] + ref[n]), n
