"""FP8 (e4m3) forward path: per-row quantisation, the e4m3 gate/up + SwiGLU
and down GEMMs (tcgen05 kind::f8f6f4), the row-gathering variant and the
fp8 MoELayer forward, each against the oracle.

Parity here:
  - quantisation: codes and scales bit-exact (a pure function of the bits);
  - GEMMs: the oracle's codes and scales go to both sides, outputs within
    the bf16 acceptance (max |err| <= 2e-2 max |ref|, rel L2 <= 5e-3) -- the
    products of two e4m3 values are exact, so the GPU differs only by its
    fp32 summation order and the bf16 rounding of the output;
  - the gathering kernel: bit-identical to the permuted-row kernel;
  - layer: the fp8 layer against the oracle's fp8 chain (same acceptance),
    and, as a format check, against the bf16 oracle chain within the e4m3
    error: four e4m3 roundings lie on y's longest chain (x, Wg/Wu, h, Wd),
    each of relative error at most 2^-4 and RMS at most 2^-4/sqrt(3), so
    rel L2 <= sqrt(4) * 2^-4 / sqrt(3) ~= 0.072 for independent errors;
    asserted <= 0.1.
"""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import assert_close, bits, inputs, oracle_chain, to_dev, dispatch_ws

pytestmark = pytest.mark.gpu


def rne_bf16(a):
    """fp32 -> bf16 (round to nearest even) -> fp32, as the GPU stores h and y_perm."""
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return r.view(np.float32)


def _bf16_matrix(gen, rows, cols, spread=6.0):
    """Seeded bf16 rows with per-row magnitudes over e^-spread..e^spread, one
    all-zero row and one row whose small entries fall in e4m3's subnormals."""
    a = torch.randn(rows, cols, generator=gen) * torch.exp(torch.empty(rows, 1).uniform_(-spread, spread,
                                                                                          generator=gen))
    if rows > 2:
        a[1] = 0.0
        a[2, ::2] *= 1e-5
    return a.to(torch.bfloat16)


def _quant_gpu(a_bf16):
    rows, cols = a_bf16.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    m.moe_quantize_rows_e4m3(a_bf16, rows, cols, q, s)
    return q, s


@pytest.mark.parametrize("rows,cols", [(37, 64), (130, 2048), (9, 2600), (1000, 768), (3, 8)])
def test_quantize_rows_bit_exact(rows, cols):
    gen = torch.Generator().manual_seed(rows * 7 + cols)
    a = _bf16_matrix(gen, rows, cols)
    q, s = _quant_gpu(a.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(a)))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def _hard_quantize_rows(gen):
    """Rows that stress the quotient a / s: (i) power-of-two scales with
    entries on e4m3 midpoints (exact ties, rounded to even), (ii) rows of
    bf16-subnormal and near-subnormal magnitudes, whose scale is so small
    that 1 / s overflows fp32, (iii) many rows of widely spread magnitudes,
    so that some quotients fall within a few fp32 ulps of a midpoint."""
    codes = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8)).astype(np.float64)
    vals = np.sort(codes)
    mids = (vals[1:] + vals[:-1]) / 2                     # 125 midpoints, 448 is the largest code
    ties = []
    for k in (-20, -3, 0, 5):
        row = np.concatenate([mids, -mids, vals, [448.0]]) * 2.0 ** k
        row = np.resize(row, 384)
        row[0] = 448.0 * 2.0 ** k                          # amax: s = 2^k exactly
        ties.append(row)
    ties = torch.tensor(np.array(ties), dtype=torch.float32)
    tiny = torch.cat([torch.randn(6, 384, generator=gen) * 2.0 ** e for e in (-133, -130, -127, -125, -122, -118)])
    wide = torch.randn(2048, 384, generator=gen) * torch.exp(torch.empty(2048, 1).uniform_(-30, 30, generator=gen))
    return torch.cat([ties, tiny, wide]).to(torch.bfloat16)


def test_quantize_rows_bit_exact_hard_cases():
    gen = torch.Generator().manual_seed(4242)
    a = _hard_quantize_rows(gen)
    rows, cols = a.shape
    q, s = _quant_gpu(a.cuda())
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(a)))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantize_rejects_bad_args():
    a = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(4, 12, dtype=torch.uint8, device="cuda")
    s = torch.empty(4, dtype=torch.float32, device="cuda")
    with pytest.raises(m.MoEError):
        m.moe_quantize_rows_e4m3(a, 4, 12, q, s)   # cols % 8 != 0
    m.moe_quantize_rows_e4m3(a, 0, 16, q, s)       # no rows: no-op


def _seeded_fp8_operands(seed, R, H, I, E):
    """Oracle codes and scales of seeded bf16 activations and weights."""
    gen = torch.Generator().manual_seed(seed)
    a = torch.randn(R, H, generator=gen).to(torch.bfloat16)
    Wg = (torch.randn(E, I, H, generator=gen) * 0.02).to(torch.bfloat16)
    Wu = (torch.randn(E, I, H, generator=gen) * 0.02).to(torch.bfloat16)
    Wd = (torch.randn(E, H, I, generator=gen) * 0.02).to(torch.bfloat16)
    hb = (torch.randn(R, I, generator=gen) * 0.3).to(torch.bfloat16)
    q = lambda t: oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(t)))  # noqa: E731
    return dict(a=q(a), Wg=q(Wg), Wu=q(Wu), Wd=q(Wd), h=q(hb))


def _dev(x, dt=None):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.cuda() if dt is None else t.to(dt).cuda()


GEMM_CASES = {
    # R,   H,   I,  E, seg_offsets, seg_expert
    "one_tile": (128, 128, 128, 1, [0, 128], None),
    "ragged_empty": (300, 256, 128, 4, [0, 0, 77, 77, 300], None),
    "three_n_tiles_uncovered_tail": (520, 256, 384, 3, [0, 129, 390, 500], None),
    "segments": (400, 384, 256, 4, [0, 40, 40, 170, 200, 399, 400], [2, 0, 1, 3, 0, 2]),
    # two long segments whose last 128-row tiles hold 1 and 75 rows
    "long_segments": (1100, 256, 256, 2, [0, 513, 1100], None),
}


@pytest.mark.parametrize("case", sorted(GEMM_CASES))
def test_fp8_gemms_match_oracle(case):
    R, H, I, E, so, se = GEMM_CASES[case]
    ops = _seeded_fp8_operands(17, R, H, I, E)
    so_np = np.array(so, np.int32)
    se_np = None if se is None else np.array(se, np.int32)
    n = len(so) - 1
    so_d, se_d = _dev(so_np), (None if se is None else _dev(se_np))
    (aq, as_), (gq, gs), (uq, us), (dq, ds), (hq, hs) = (ops[k] for k in ("a", "Wg", "Wu", "Wd", "h"))
    h = torch.full((R, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_swiglu_fp8(_dev(aq), _dev(as_), None, 0, _dev(gq), _dev(gs.reshape(-1)), _dev(uq),
                                  _dev(us.reshape(-1)), n, so_d, se_d, R, H, I, E, h)
    y = torch.full((R, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_down_fp8(_dev(hq), _dev(hs), _dev(dq), _dev(ds.reshape(-1)), n, so_d, se_d, R, H, I, E,
                                y)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    h_ref = oracle.grouped_gemm_swiglu_fp8(aq, as_, gq, gs, uq, us, so_np, se_np)
    y_ref = oracle.grouped_gemm_down_fp8(hq, hs, dq, ds, so_np, se_np)
    covered = np.zeros(R, bool)
    for s in range(n):
        covered[so[s]:so[s + 1]] = True
    assert_close(h[torch.from_numpy(covered).cuda()], h_ref[covered], "h (fp8)")
    assert_close(y[torch.from_numpy(covered).cuda()], y_ref[covered], "y_perm (fp8)")
    # rows outside every segment are left untouched
    assert torch.isnan(h[torch.from_numpy(~covered).cuda()].float()).all()


def test_fp8_gather_matches_permuted_rows():
    T, H, I, E, R = 96, 256, 128, 4, 300
    gen = torch.Generator().manual_seed(3)
    x = torch.randn(T, H, generator=gen).to(torch.bfloat16)
    xq, xs = _quant_gpu(x.cuda())
    ops = _seeded_fp8_operands(4, 8, H, I, E)
    (gq, gs), (uq, us) = ops["Wg"], ops["Wu"]
    tor = torch.randint(0, T, (R,), generator=gen, dtype=torch.int32)
    so = torch.tensor([0, 40, 40, 170, 200, 299, 300], dtype=torch.int32).cuda()
    se = torch.tensor([2, 0, 1, 3, 0, 2], dtype=torch.int32).cuda()
    tor_d = tor.cuda()
    xq_perm, xs_perm = xq[tor_d.long()].contiguous(), xs[tor_d.long()].contiguous()
    args = (_dev(gq), _dev(gs.reshape(-1)), _dev(uq), _dev(us.reshape(-1)), 6, so, se, R, H, I, E)
    h_ref = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_swiglu_fp8(xq_perm, xs_perm, None, 0, *args, h_ref)
    h = torch.empty_like(h_ref)
    m.moe_grouped_gemm_swiglu_fp8(xq, xs, tor_d, T, *args, h)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(h, h_ref), "gathered e4m3 rows must give the permuted path's h bit for bit"
    xq_o, xs_o = oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(x)))
    t = tor.numpy()
    href = oracle.grouped_gemm_swiglu_fp8(xq_o[t], xs_o[t], gq, gs, uq, us, so.cpu().numpy(), se.cpu().numpy())
    assert_close(h, href, "h (fp8, gathered)")


def test_fp8_gather_bad_token_id_sets_status():
    T, H, I, E = 32, 128, 128, 2
    xq = torch.zeros(T, H, dtype=torch.uint8, device="cuda")
    xs = torch.ones(T, dtype=torch.float32, device="cuda")
    W = torch.zeros(E, I, H, dtype=torch.uint8, device="cuda")
    Ws = torch.ones(E * I, dtype=torch.float32, device="cuda")
    tor = torch.zeros(64, dtype=torch.int32, device="cuda")
    tor[5] = T + 7
    so = torch.tensor([0, 32, 64], dtype=torch.int32, device="cuda")
    h = torch.empty(64, I, dtype=torch.bfloat16, device="cuda")
    m.moe_read_device_status(reset=True)
    m.moe_grouped_gemm_swiglu_fp8(xq, xs, tor, T, W, Ws, W, Ws, 2, so, None, 64, H, I, E, h)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) & 1  # MOE_STATUS_BAD_INDEX
    assert torch.equal(h, torch.zeros_like(h))


def test_fp8_rejects_unsupported_shapes():
    z = torch.zeros(256, dtype=torch.uint8, device="cuda")
    f = torch.ones(256, dtype=torch.float32, device="cuda")
    so = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    h = torch.empty(256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoEError):  # I = 64 is not a multiple of 128
        m.moe_grouped_gemm_swiglu_fp8(z, f, None, 0, z, f, z, f, 1, so, None, 1, 128, 64, 1, h)
    with pytest.raises(m.MoEError):  # H = 192
        m.moe_grouped_gemm_down_fp8(z, f, z, f, 1, so, None, 1, 192, 128, 1, h)


def _oracle_fp8_chain(inp, f):
    """The oracle's fp8 forward on the seeded inputs: x and the weights
    quantised per row, rows gathered by token, h and y_perm rounded to bf16
    where the layer stores them."""
    xq, xs = oracle.quantize_rows_e4m3(oracle.widen_bf16(f["x"]))
    W = {n: oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(inp[n]))) for n in ("Wg", "Wu", "Wd")}
    tor = f["dp"]["token_of_row"]
    off = f["rt"]["offsets"]
    h = oracle.grouped_gemm_swiglu_fp8(xq[tor], xs[tor], W["Wg"][0], W["Wg"][1], W["Wu"][0], W["Wu"][1], off)
    hq, hs = oracle.quantize_rows_e4m3(rne_bf16(h))
    yp = oracle.grouped_gemm_down_fp8(hq, hs, W["Wd"][0], W["Wd"][1], off)
    return oracle.combine(rne_bf16(yp), f["rt"]["topk_w"], f["dp"]["row_of_slot"]), W


@pytest.mark.parametrize("T,H,I,E,k,ep", [(256, 256, 128, 8, 2, 2), (300, 256, 256, 12, 3, 4),
                                         (1024, 256, 128, 4, 2, 2)])  # the last: ~512 rows per expert
def test_fp8_layer_forward(T, H, I, E, k, ep):
    inp = inputs(T, H, I, E, k, seed=5, ep=ep)
    g = to_dev(inp)
    L = m.MoELayer(T, H, I, E, k, ep, training=False, fp8=True)
    w8 = L.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    y = L.forward(g["x"], g["Wr"], g["bias"], w8, None, None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    f = oracle_chain(inp)
    y8_ref, W = _oracle_fp8_chain(inp, f)
    for n in ("Wg", "Wu", "Wd"):
        assert np.array_equal(w8[n].cpu().numpy(), W[n][0])
        assert np.array_equal(w8[n + "_scale"].cpu().numpy(), W[n][1].reshape(-1))
    assert_close(y, y8_ref, "y (fp8 layer vs fp8 oracle)")
    # format check: the e4m3 forward stays within e4m3's error of the bf16 layer
    assert_close(y, f["y"], "y (fp8 layer vs bf16 oracle)", max_frac=0.25, rel=0.1)
    # deterministic: a second forward gives the same bits
    y1 = y.clone()
    y2 = L.forward(g["x"], g["Wr"], g["bias"], w8, None, None)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("workload", ["qwen3_30b_fwd", "qwen3_30b_zipf_fwd"])
def test_fp8_layer_full_size_sampled_tokens(workload):
    """The fp8 forward at full size (Qwen3-30B-A3B shapes; T=4096 as bench.py
    times it, and the Zipf-skewed T=16384 workload with empty experts):
    routing bit for bit over every token, the weight codes and scales of the
    experts the sampled tokens use bit for bit, and those tokens' outputs
    against the oracle's fp8 chain (x and h quantised per row, weights per
    output channel, h and y_perm rounded to bf16 where the layer stores them)."""
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_layer_inputs
    shape = CONFIGS[workload]
    inp = make_layer_inputs(shape, 0, with_dy=False)
    g = to_dev(inp)
    L = m.MoELayer(shape.T, shape.H, shape.I, shape.E, shape.k, shape.ep_size, training=False, fp8=True)
    w8 = L.quantize_weights(g["Wg"], g["Wu"], g["Wd"])
    y = L.forward(g["x"], g["Wr"], g["bias"], w8, None, None)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    bias = None if inp.get("bias") is None else inp["bias"].numpy()
    rt = oracle.route_topk(bits(inp["x"]), inp["Wr"].numpy(), bias, shape.k, shape.ep_size)
    assert np.array_equal(L.topk_idx.cpu().numpy(), rt["topk_idx"])
    assert np.array_equal(L.offsets.cpu().numpy(), rt["offsets"])
    if workload == "qwen3_30b_zipf_fwd":
        assert (rt["counts"] == 0).sum() >= 4  # empty experts in the gathering e4m3 GEMM
    rng = np.random.default_rng(8)
    toks = sorted(rng.choice(shape.T, 4, replace=False).tolist())
    sub = dict(inp)
    sub["x"] = inp["x"][toks].contiguous()
    sub["T"] = len(toks)
    f = oracle_chain(sub)
    # the oracle's fp8 chain over the experts these tokens use only
    used = sorted(set(f["rt"]["topk_idx"].reshape(-1).tolist()))
    remap = np.zeros(shape.E, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    W = {n: oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(inp[n][used]))) for n in ("Wg", "Wu", "Wd")}
    for n in ("Wg", "Wu", "Wd"):
        assert np.array_equal(w8[n][used].cpu().numpy(), W[n][0])
        assert np.array_equal(w8[n + "_scale"].view(shape.E, -1)[used].cpu().numpy(), W[n][1])
    xq, xs = oracle.quantize_rows_e4m3(oracle.widen_bf16(f["x"]))
    tor, off = f["dp"]["token_of_row"], f["rt"]["offsets"]
    h = oracle.grouped_gemm_swiglu_fp8(xq[tor], xs[tor], W["Wg"][0], W["Wg"][1], W["Wu"][0], W["Wu"][1], off,
                                       remap)
    hq, hs = oracle.quantize_rows_e4m3(rne_bf16(h))
    yp = oracle.grouped_gemm_down_fp8(hq, hs, W["Wd"][0], W["Wd"][1], off, remap)
    y_ref = oracle.combine(rne_bf16(yp), f["rt"]["topk_w"], f["dp"]["row_of_slot"])
    assert_close(y[toks], y_ref, "y (fp8, sampled tokens)")


def test_fp8_ep_rank_local_segments_full_size():
    """One EP rank's local expert compute in e4m3 at full size (32768 received
    rows, 16 local experts, 128 source-rank x expert segments): the received
    rows and the weights quantised on the GPU, both GEMMs over the segment
    table, sampled rows against the oracle's fp8 chain on the same seeded
    data (its own codes, its h rounded to bf16 and quantised)."""
    from moe_expert_layer_topk_gb300.synth import CONFIGS, make_segment_inputs
    shape = CONFIGS["ep_rank_local"]
    s = make_segment_inputs(shape, 0)
    R, H, I, E, nseg = s["R"], s["H"], s["I"], s["E"], s["num_seg"]
    xp = s["x_perm"].cuda()
    xq, xs = _quant_gpu(xp)
    L = m.MoELayer(1, H, I, E, 1, 1, training=False, fp8=True)
    w8 = L.quantize_weights(s["Wg"].cuda(), s["Wu"].cuda(), s["Wd"].cuda())
    so, se = s["seg_offsets"].cuda(), s["seg_expert"].cuda()
    h = torch.empty(R, I, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_swiglu_fp8(xq, xs, None, 0, w8["Wg"], w8["Wg_scale"], w8["Wu"], w8["Wu_scale"], nseg,
                                  so, se, R, H, I, E, h)
    hq, hs = _quant_gpu(h)
    y = torch.empty(R, H, dtype=torch.bfloat16, device="cuda")
    m.moe_grouped_gemm_down_fp8(hq, hs, w8["Wd"], w8["Wd_scale"], nseg, so, se, R, H, I, E, y)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    son, sen = s["seg_offsets"].numpy(), s["seg_expert"].numpy()
    rng = np.random.default_rng(9)
    rows, experts = [], []
    for q in rng.choice(nseg, 10, replace=False):
        a, b = int(son[q]), int(son[q + 1])
        for r in sorted({a, b - 1} if b > a else set()):
            rows.append(r)
            experts.append(int(sen[q]))
    so2 = np.arange(len(rows) + 1, dtype=np.int32)
    se2 = np.asarray(experts, np.int32)
    aq, as_ = oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(s["x_perm"][rows])))
    W = {n: oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(s[n]))) for n in ("Wg", "Wu", "Wd")}
    href = oracle.grouped_gemm_swiglu_fp8(aq, as_, W["Wg"][0], W["Wg"][1], W["Wu"][0], W["Wu"][1], so2, se2)
    assert_close(h[rows], href, "h (fp8, sampled rows)")
    hq_o, hs_o = oracle.quantize_rows_e4m3(rne_bf16(href))
    yref = oracle.grouped_gemm_down_fp8(hq_o, hs_o, W["Wd"][0], W["Wd"][1], so2, se2)
    assert_close(y[rows], yref, "y_perm (fp8, sampled rows)")


@pytest.mark.parametrize("T,H,E,k,bias", [(300, 256, 8, 2, None), (517, 2560, 16, 4, "zipf"), (64, 128, 130, 8, None)])
def test_dispatch_e4m3_bit_exact(T, H, E, k, bias):
    """moe_dispatch_e4m3: each permuted row holds its token's e4m3 codes and
    scale bit for bit as the oracle quantises x per token, with the rows,
    row_of_slot and token_of_row of moe_dispatch (H = 2560 takes the second
    pass over rows longer than the 256 vectors held in registers; the Zipf
    bias leaves experts empty)."""
    inp = inputs(T, H, 64, E, k, seed=T + H, bias=bias, router_std=0.02 if bias is None else 0.3)
    g = to_dev(inp)
    L = m.MoELayer(T, H, 64, E, k, 1, training=False)
    L.route(g["x"], g["Wr"], g["bias"])
    L.dispatch(g["x"])
    R = T * k
    xq = torch.full((R, H), 0x5A, dtype=torch.uint8, device="cuda")
    xs = torch.full((R,), float("nan"), dtype=torch.float32, device="cuda")
    ros = torch.empty_like(L.row_of_slot)
    tor = torch.empty_like(L.token_of_row)
    m.moe_dispatch_e4m3(g["x"], L.topk_idx, L.offsets, T, H, E, k, xq, xs, ros, tor, dispatch_ws(T, E, k))
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(ros, L.row_of_slot) and torch.equal(tor, L.token_of_row)
    q_ref, s_ref = oracle.quantize_rows_e4m3(oracle.widen_bf16(bits(inp["x"])))
    t = tor.cpu().numpy()
    assert np.array_equal(xq.cpu().numpy(), q_ref[t])
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), s_ref[t].view(np.uint32))
