"""Full-size workloads (Qwen3-30B-A3B expert shapes: hidden 2048, intermediate
768, 128 experts, top-8), run the way bench.py runs them (MoELayer over the
C ABI).  Routing, counts, offsets and the permutation are compared bit for
bit over every token; floating-point outputs are compared on samples the
oracle can afford: whole per-token chains for sampled tokens (a token's
routing, rows, output and dX depend on that token alone), and whole weight
gradients of sampled experts with the GPU's stored bf16 operands fed to the
oracle."""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import assert_close, bits, f32, oracle_backward, oracle_chain, to_dev
from moe_expert_layer_topk_gb300.synth import CONFIGS, bf16_bits, make_layer_inputs, make_segment_inputs

pytestmark = pytest.mark.gpu


def subset(inp, toks):
    sub = dict(inp)
    sub["x"] = inp["x"][toks].contiguous()
    sub["dy"] = None if inp.get("dy") is None else inp["dy"][toks].contiguous()
    sub["T"] = len(toks)
    return sub


def rows_check(L, inp, rows, experts):
    """h and y_perm of chosen rows: the GPU's stored operands through the oracle."""
    so = np.arange(len(rows) + 1, dtype=np.int32)
    se = np.asarray(experts, np.int32)
    xp = f32(L.x_perm[rows])
    h = oracle.grouped_gemm_swiglu(xp, bits(inp["Wg"]), bits(inp["Wu"]), so, se)
    assert_close(L.h[rows], h, "h (sampled rows)")
    y = oracle.grouped_gemm_down(f32(L.h[rows]), bits(inp["Wd"]), so, se)
    assert_close(L.y_perm[rows], y, "y_perm (sampled rows)")


def run_fwd(name, with_bwd=False):
    shape = CONFIGS[name]
    inp = make_layer_inputs(shape, 0, with_dy=with_bwd)
    g = to_dev(inp)
    L = m.MoELayer(shape.T, shape.H, shape.I, shape.E, shape.k, shape.ep_size, training=with_bwd)
    L.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"])
    if with_bwd:
        L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    return shape, inp, g, L


def check_routing_and_dispatch(L, inp):
    x = bits(inp["x"])
    bias = None if inp.get("bias") is None else inp["bias"].numpy()
    rt = oracle.route_topk(x, inp["Wr"].numpy(), bias, inp["k"], inp["ep_size"])
    assert np.array_equal(L.topk_idx.cpu().numpy(), rt["topk_idx"])
    assert np.array_equal(L.counts.cpu().numpy(), rt["counts"])
    assert np.array_equal(L.offsets.cpu().numpy(), rt["offsets"])
    assert np.array_equal(L.rank_offsets.cpu().numpy(), rt["rank_offsets"])
    assert_close(L.topk_w, rt["topk_w"], "topk_w", max_frac=1e-5, rel=1e-6)
    dp = oracle.dispatch(None, rt["topk_idx"], rt["offsets"], inp["E"], copy_rows=False)
    ros = L.row_of_slot.cpu().numpy()
    assert np.array_equal(ros, dp["row_of_slot"])
    assert np.array_equal(L.token_of_row.cpu().numpy(), dp["token_of_row"])
    # x_perm is a pure copy: every row equals its token's x row
    xp = L.x_perm.view(torch.int16)
    xg = inp["x"].view(torch.int16).to(xp.device)
    assert torch.equal(xp, xg[L.token_of_row.long()])
    return rt


def sample_rows(offsets, rng, n):
    E = len(offsets) - 1
    nonempty = [e for e in range(E) if offsets[e + 1] > offsets[e]]
    es = rng.choice(nonempty, size=min(n, len(nonempty)), replace=False)
    rows, experts = [], []
    for e in es:
        a, b = int(offsets[e]), int(offsets[e + 1])
        for r in {a, b - 1, int(rng.integers(a, b))}:
            rows.append(r)
            experts.append(int(e))
    return rows, experts


def test_qwen3_fwd_T4096():
    shape, inp, g, L = run_fwd("qwen3_30b_fwd")
    rt = check_routing_and_dispatch(L, inp)
    rng = np.random.default_rng(0)
    rows, experts = sample_rows(rt["offsets"], rng, 12)
    rows_check(L, inp, rows, experts)
    toks = sorted(rng.choice(shape.T, 6, replace=False).tolist())
    f = oracle_chain(subset(inp, toks))
    assert_close(L.y[toks], f["y"], "y (sampled tokens, oracle chain)")


def test_qwen3_zipf_T16384_empty_experts():
    shape, inp, g, L = run_fwd("qwen3_30b_zipf_fwd")
    rt = check_routing_and_dispatch(L, inp)
    counts = rt["counts"]
    assert (counts == 0).sum() >= 4, counts   # the forced-empty tail at least
    assert counts.max() > 4 * counts.mean()   # skewed
    rng = np.random.default_rng(1)
    rows, experts = sample_rows(rt["offsets"], rng, 8)
    top = int(np.argmax(counts))
    rows += [int(rt["offsets"][top]) + 129, int(rt["offsets"][top + 1]) - 1]
    experts += [top, top]
    rows_check(L, inp, rows, experts)
    toks = sorted(rng.choice(shape.T, 4, replace=False).tolist())
    f = oracle_chain(subset(inp, toks))
    assert_close(L.y[toks], f["y"], "y (sampled tokens, oracle chain)")


def test_ep_rank_local_segments():
    shape = CONFIGS["ep_rank_local"]
    s = make_segment_inputs(shape, 0)
    R, H, I, E = s["R"], s["H"], s["I"], s["E"]
    dev = "cuda"
    xp, Wg, Wu, Wd = (s[n].to(dev) for n in ("x_perm", "Wg", "Wu", "Wd"))
    so, se = s["seg_offsets"].to(dev), s["seg_expert"].to(dev)
    h = torch.empty(R, I, dtype=torch.bfloat16, device=dev)
    y = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    m.moe_grouped_gemm_swiglu(xp, Wg, Wu, s["num_seg"], so, se, R, H, I, E, h, None)
    m.moe_grouped_gemm_down(h, Wd, s["num_seg"], so, se, R, H, I, E, y)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    son, sen = s["seg_offsets"].numpy(), s["seg_expert"].numpy()
    rng = np.random.default_rng(2)
    segs = rng.choice(s["num_seg"], 10, replace=False)
    rows, experts = [], []
    for q in segs:
        a, b = int(son[q]), int(son[q + 1])
        if b > a:
            for r in {a, b - 1}:
                rows.append(r)
                experts.append(int(sen[q]))
    so2 = np.arange(len(rows) + 1, dtype=np.int32)
    se2 = np.asarray(experts, np.int32)
    href = oracle.grouped_gemm_swiglu(oracle.widen_bf16(bf16_bits(s["x_perm"][rows])), bf16_bits(s["Wg"]),
                                      bf16_bits(s["Wu"]), so2, se2)
    assert_close(h[rows], href, "h (sampled rows)")
    yref = oracle.grouped_gemm_down(f32(h[rows]), bf16_bits(s["Wd"]), so2, se2)
    assert_close(y[rows], yref, "y_perm (sampled rows)")


def test_qwen3_fwd_bwd_T8192():
    shape, inp, g, L = run_fwd("qwen3_30b_fwd_bwd", with_bwd=True)
    rt = check_routing_and_dispatch(L, inp)
    offs = rt["offsets"]
    rng = np.random.default_rng(3)
    # whole weight gradients of two experts, GPU bf16 operands through the oracle
    for e in rng.choice(shape.E, 2, replace=False):
        a, b = int(offs[e]), int(offs[e + 1])
        so = np.array([0, b - a], np.int32)
        _, dWd = oracle.grouped_gemm_down_bwd(f32(L.dy_perm[a:b]), f32(L.h[a:b]), f32(L.gu[a:b]),
                                              bits(inp["Wd"][e:e + 1]), so)
        assert_close(L.dWd[e], dWd[0], f"dWd[{e}]")
        _, dWg, dWu = oracle.grouped_gemm_swiglu_bwd(f32(L.dgu[a:b]), f32(L.x_perm[a:b]),
                                                     bits(inp["Wg"][e:e + 1]), bits(inp["Wu"][e:e + 1]), so)
        assert_close(L.dWg[e], dWg[0], f"dWg[{e}]")
        assert_close(L.dWu[e], dWu[0], f"dWu[{e}]")
    # router weight gradient over all tokens from the GPU's d_w and dx_acc
    dWr, _ = oracle.route_topk_bwd(f32(L.d_w), f32(L.topk_w), rt["topk_idx"], bits(inp["x"]),
                                   inp["Wr"].numpy(), np.zeros((shape.T, shape.H), np.float32))
    assert_close(L.dWr, dWr, "dWr", max_frac=1e-3, rel=1e-4)
    # whole chains (forward and backward) of sampled tokens
    toks = sorted(rng.choice(shape.T, 4, replace=False).tolist())
    sub = subset(inp, toks)
    f = oracle_chain(sub)
    b = oracle_backward(sub, f)
    assert_close(L.y[toks], f["y"], "y (sampled tokens)")
    assert_close(L.dx[toks], b["dx"], "dx (sampled tokens)")
    assert_close(L.d_w[toks], b["d_w"], "d_w (sampled tokens)")
