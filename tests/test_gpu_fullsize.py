"""Full-size workloads (Qwen3-30B-A3B expert shapes: hidden 2048, intermediate
768, 128 experts, top-8), run the way bench.py runs them (MoELayer over the
C ABI).  Routing, counts, offsets and the permutation are compared bit for
bit over every token; floating-point outputs are compared on samples the
oracle can afford, always computed by the oracle from the seeded inputs
alone (no value the GPU computed is fed to it): whole per-token chains for
sampled tokens (a token's routing, rows, output and dX depend on that token
alone), sampled permuted rows, the whole backward of sampled experts (the
oracle recomputes every row routed to the expert), and the router weight
gradient over the whole matrix from a second backward pass whose dY is zero
outside a token sample (so every contribution comes from tokens the oracle
evaluates)."""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import assert_close, bits, oracle_backward, oracle_chain, to_dev
from moe_expert_layer_topk_gb300.synth import CONFIGS, bf16_bits, make_layer_inputs, make_segment_inputs

pytestmark = pytest.mark.gpu


def subset(inp, toks):
    sub = dict(inp)
    sub["x"] = inp["x"][toks].contiguous()
    sub["dy"] = None if inp.get("dy") is None else inp["dy"][toks].contiguous()
    sub["T"] = len(toks)
    return sub


def rows_check(L, inp, token_of_row, rows, experts):
    """h and y_perm of chosen permuted rows, the oracle chained on its own h."""
    so = np.arange(len(rows) + 1, dtype=np.int32)
    se = np.asarray(experts, np.int32)
    xp = oracle.widen_bf16(bits(inp["x"][token_of_row[rows]]))
    h = oracle.grouped_gemm_swiglu(xp, bits(inp["Wg"]), bits(inp["Wu"]), so, se)
    assert_close(L.h[rows], h, "h (sampled rows)")
    y = oracle.grouped_gemm_down(h, bits(inp["Wd"]), so, se)
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
    rt["token_of_row"] = dp["token_of_row"]
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
    rows_check(L, inp, rt["token_of_row"], rows, experts)
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
    rows_check(L, inp, rt["token_of_row"], rows, experts)
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
    yref = oracle.grouped_gemm_down(href, bf16_bits(s["Wd"]), so2, se2)
    assert_close(y[rows], yref, "y_perm (sampled rows)")


def expert_backward_oracle(inp, rt, e):
    """The oracle's forward and backward over every row routed to expert e,
    from the seeded inputs: returns its rows [a, b) and h, dgu, dx_perm,
    dW_down, dW_gate, dW_up of that expert."""
    a, b = int(rt["offsets"][e]), int(rt["offsets"][e + 1])
    tok = rt["token_of_row"][a:b]
    slot = np.argmax(rt["topk_idx"][tok] == e, axis=1)
    n = b - a
    so = np.array([0, n], np.int32)
    xe = oracle.widen_bf16(bits(inp["x"][tok]))
    Wg, Wu, Wd = (bits(inp[w][e:e + 1]) for w in ("Wg", "Wu", "Wd"))
    h, gu = oracle.grouped_gemm_swiglu(xe, Wg, Wu, so, save_gu=True)
    # dy_perm[row] = topk_w[t, j] * dy[t]: combine backward with one slot per row
    dye = oracle.widen_bf16(bits(inp["dy"][tok]))
    w = rt["topk_w"][tok, slot][:, None]
    dyp, _ = oracle.combine_bwd(dye, np.zeros((n, dye.shape[1]), np.float32), w,
                                np.arange(n, dtype=np.int32)[:, None])
    dgu, dWd = oracle.grouped_gemm_down_bwd(dyp, h, gu, Wd, so)
    dxp, dWg, dWu = oracle.grouped_gemm_swiglu_bwd(dgu, xe, Wg, Wu, so)
    return a, b, dict(h=h, dgu=dgu, dx_perm=dxp, dWd=dWd[0], dWg=dWg[0], dWu=dWu[0])


def test_qwen3_fwd_bwd_T8192():
    shape, inp, g, L = run_fwd("qwen3_30b_fwd_bwd", with_bwd=True)
    rt = check_routing_and_dispatch(L, inp)
    rng = np.random.default_rng(3)
    # the whole backward of two experts (every row routed to them)
    for e in rng.choice(shape.E, 2, replace=False):
        a, b, ref = expert_backward_oracle(inp, rt, int(e))
        assert_close(L.h[a:b], ref["h"], f"h rows of expert {e}")
        assert_close(L.dgu[a:b], ref["dgu"], f"dgu rows of expert {e}")
        assert_close(L.dx_perm[a:b], ref["dx_perm"], f"dx_perm rows of expert {e}")
        for n in ("dWd", "dWg", "dWu"):
            assert_close(getattr(L, n)[e], ref[n], f"{n}[{e}]")
    # whole chains (forward and backward) of sampled tokens
    toks = sorted(rng.choice(shape.T, 4, replace=False).tolist())
    sub = subset(inp, toks)
    f = oracle_chain(sub)
    bw = oracle_backward(sub, f)
    assert_close(L.y[toks], f["y"], "y (sampled tokens)")
    assert_close(L.dx[toks], bw["dx"], "dx (sampled tokens)")
    assert_close(L.d_w[toks], bw["d_w"], "d_w (sampled tokens)")
    # second backward, dY zero outside the sample: dWr over the whole
    # matrix, and every weight gradient, come from the sampled tokens alone
    dy_sparse = torch.zeros_like(g["dy"])
    dy_sparse[toks] = g["dy"][toks]
    L.backward(dy_sparse, g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert_close(L.dWr, bw["dWr"], "dWr (sparse dY)")
    assert_close(L.dx[toks], bw["dx"], "dx (sparse dY)")
    touched = sorted(set(f["rt"]["topk_idx"].reshape(-1).tolist()))
    for n in ("dWd", "dWg", "dWu"):
        assert_close(getattr(L, n)[touched], bw[n][touched], f"{n} of the sampled tokens' experts (sparse dY)")
    others = torch.ones(shape.E, dtype=torch.bool, device=L.dWd.device)
    others[touched] = False
    for n in ("dWd", "dWg", "dWu"):
        assert getattr(L, n)[others].abs().max().item() == 0.0, n
