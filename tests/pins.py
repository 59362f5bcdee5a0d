"""Checks that pin the CPU oracle to facts other than itself.

Each `pin_*` function raises AssertionError when the oracle (whichever build
`oracle.use()` points at) disagrees with: a hand-derived closed form, a brute
force over tiny inputs, a library routine the definition reduces to (fp64
torch matmul / softmax / silu / autograd), or an invariant.  The mutation
tests run all of them against deliberately broken oracle builds and require
every mutant to fail at least one.

Source of the definitions: "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP
Design", section 3 (permute -> grouped matmul -> unpermute, empty experts
allowed); "Qwen3-MoE-30B-A3B模型EP+FSDP2并行方案", model section (expert
tensor shapes) and "完整并行流程" (contiguous dim-0 expert blocks per EP rank).
"""
from __future__ import annotations

import itertools
import json
from pathlib import Path

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from moe_expert_layer_topk_gb300.synth import LayerShape, bf16_bits, make_layer_inputs, make_segment_inputs

GOLDEN = Path(__file__).resolve().parent / "golden"
U = 2.0 ** -24  # fp32 unit roundoff


# ------------------------------------------------------------------ helpers

def tiny(T=64, H=128, I=64, E=8, k=2, seed=0, bias=None, with_dy=False, router_std=0.02):
    shape = LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=1 if E % 2 else 2)
    return make_layer_inputs(shape, seed, router_std=router_std, with_dy=with_dy,
                             bias=bias if bias is not None else None)


def np_inputs(inp):
    out = dict(inp)
    for key in ("x", "Wg", "Wu", "Wd", "dy"):
        if inp.get(key) is not None:
            out[key] = bf16_bits(inp[key])
    out["Wr"] = inp["Wr"].numpy()
    out["bias"] = None if inp.get("bias") is None else inp["bias"].numpy()
    return out


def rel_l2(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def oracle_forward(d, save_gu=False):
    """Oracle chain A1..A6 on numpy inputs `d`."""
    k = d["k"]; E = d["E"]
    rt = oracle.route_topk(d["x"], d["Wr"], d["bias"], k, d.get("ep_size", 1))
    dp = oracle.dispatch(d["x"], rt["topk_idx"], rt["offsets"], E)
    xp = oracle.widen_bf16(dp["x_perm"])
    res = oracle.grouped_gemm_swiglu(xp, d["Wg"], d["Wu"], rt["offsets"], None, save_gu=save_gu)
    h, gu = res if save_gu else (res, None)
    y_perm = oracle.grouped_gemm_down(h, d["Wd"], rt["offsets"])
    y = oracle.combine(y_perm, rt["topk_w"], dp["row_of_slot"])
    return dict(rt=rt, dp=dp, x_perm=xp, h=h, gu=gu, y_perm=y_perm, y=y)


def dense_forward_fp64(d, topk_idx, leaf=False):
    """Per-token dense evaluation in fp64 with torch, no permutation.

    y[t] = sum_j softmax(sel logits)_j * FFN_{e_j}(x[t]),
    FFN_e(v) = (silu(v Wg[e]^T) * (v Wu[e]^T)) Wd[e]^T, routing held fixed.
    """
    x = torch.from_numpy(oracle.widen_bf16(d["x"]).astype(np.float64))
    Wr = torch.from_numpy(d["Wr"].astype(np.float64))
    Wg = torch.from_numpy(oracle.widen_bf16(d["Wg"]).astype(np.float64))
    Wu = torch.from_numpy(oracle.widen_bf16(d["Wu"]).astype(np.float64))
    Wd = torch.from_numpy(oracle.widen_bf16(d["Wd"]).astype(np.float64))
    leaves = [x, Wr, Wg, Wu, Wd]
    if leaf:
        for p in leaves:
            p.requires_grad_(True)
    logits = x @ Wr
    if d.get("bias") is not None:
        logits = logits + torch.from_numpy(d["bias"].astype(np.float64))
    idx = torch.from_numpy(topk_idx.astype(np.int64))
    w = torch.softmax(logits.gather(1, idx), dim=1)
    y = torch.zeros(x.shape[0], Wd.shape[1], dtype=torch.float64)
    for j in range(idx.shape[1]):
        for e in torch.unique(idx[:, j]).tolist():
            m = idx[:, j] == e
            v = x[m]
            out = (F.silu(v @ Wg[e].T) * (v @ Wu[e].T)) @ Wd[e].T
            y = y.index_add(0, torch.nonzero(m).flatten(), w[m, j:j + 1] * out)
    return y, w, leaves


# ------------------------------------------------------------- A1 router

def pin_logit_block_order():
    """Hand-derived logits that only the blocked summation order produces."""
    cases = json.loads((GOLDEN / "router_logit_blocks.json").read_text())["cases"]
    for c in cases:
        H = c["H"]
        x = np.full((1, H), 0x3F80, np.uint16)            # bf16 1.0
        Wr = np.ones((H, 2), np.float32)
        Wr[0, :] = 2.0 ** 24
        bias = None if c["bias"] is None else np.full(2, c["bias"], np.float32)
        got = oracle.router_logits(x, Wr, bias)
        assert got[0, 0] == np.float32(c["logit"]), (H, got[0, 0], c["logit"])
        assert got[0, 1] == np.float32(c["logit"])


def pin_logits_error_bound():
    """fp32 logits within the recursive-summation bound of the exact fp64 dot."""
    for E, H in ((8, 128), (5, 320), (1, 64)):
        d = np_inputs(tiny(T=32, H=H, E=E, k=1, seed=E + H))
        got = oracle.router_logits(d["x"], d["Wr"], None).astype(np.float64)
        xv = oracle.widen_bf16(d["x"]).astype(np.float64)
        ref = xv @ d["Wr"].astype(np.float64)
        bound = 2.0 * (H + 2) * U * (np.abs(xv) @ np.abs(d["Wr"].astype(np.float64)))
        assert np.all(np.abs(got - ref) <= bound + 1e-30), np.max(np.abs(got - ref) - bound)


def _best_subset(L, k):
    best, best_key = None, None
    for sub in itertools.combinations(range(len(L)), k):
        s = float(np.sum(np.asarray(L, np.float64)[list(sub)]))
        key = (s, tuple(-i for i in sub))
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return set(best)


def _check_topk_against_bruteforce(L, idx, k):
    for t in range(L.shape[0]):
        assert set(idx[t].tolist()) == _best_subset(L[t], k), (t, idx[t], L[t])
        for j in range(k - 1):
            a, b = idx[t, j], idx[t, j + 1]
            assert L[t, a] > L[t, b] or (L[t, a] == L[t, b] and a < b), (t, idx[t])


def pin_topk_bruteforce():
    """Selected set = the k-subset maximising the logit sum (lower ids on ties);
    slots in descending logit order, equal logits to the lower id."""
    d = np_inputs(tiny(T=64, E=8, k=2, seed=1))
    rt = oracle.route_topk(d["x"], d["Wr"], None, 2)
    L = oracle.router_logits(d["x"], d["Wr"], None)
    _check_topk_against_bruteforce(L, rt["topk_idx"], 2)
    d = np_inputs(tiny(T=16, E=7, k=3, seed=2))
    rt = oracle.route_topk(d["x"], d["Wr"], None, 3)
    L = oracle.router_logits(d["x"], d["Wr"], None)
    _check_topk_against_bruteforce(L, rt["topk_idx"], 3)


def pin_topk_ties():
    """Hand-built ties: duplicated router columns and all-zero tokens."""
    d = np_inputs(tiny(T=16, E=8, k=3, seed=3))
    Wr = d["Wr"].copy()
    Wr[:, 5] = Wr[:, 2]
    Wr[:, 6] = Wr[:, 2]
    Wr[:, 2] += 0.0                # columns 2, 5, 6 identical
    x = d["x"].copy()
    x[0] = 0                       # token 0: every logit is +0
    # make column 2 the largest for token 1: x[1] = sign pattern of Wr[:, 2]
    x[1] = np.where(Wr[:, 2] >= 0, 0x3F80, 0xBF80).astype(np.uint16)
    rt = oracle.route_topk(x, Wr, None, 3)
    idx = rt["topk_idx"]
    assert idx[0].tolist() == [0, 1, 2], idx[0]
    assert idx[1].tolist() == [2, 5, 6], idx[1]
    assert np.allclose(rt["topk_w"][0], 1.0 / 3, rtol=0, atol=1e-7)
    L = oracle.router_logits(x, Wr, None)
    _check_topk_against_bruteforce(L, idx, 3)


def pin_weights_closed_form():
    """w_j = p_{e_j} / sum_sel p with p the full softmax; k = E gives the full
    softmax; E = 1 gives w = 1; a hand-computable case gives 3/4, 1/4."""
    for bias in (None, "zipf"):
        d = np_inputs(tiny(T=64, E=8, k=3, seed=4, bias=bias, router_std=0.2))
        rt = oracle.route_topk(d["x"], d["Wr"], d["bias"], 3)
        L = oracle.router_logits(d["x"], d["Wr"], d["bias"]).astype(np.float64)
        p = torch.softmax(torch.from_numpy(L), dim=1).numpy()
        sel = np.take_along_axis(p, rt["topk_idx"].astype(np.int64), 1)
        ref = sel / sel.sum(1, keepdims=True)
        assert np.max(np.abs(rt["topk_w"] - ref)) < 2e-6
        assert np.max(np.abs(rt["topk_w"].astype(np.float64).sum(1) - 1)) < 2e-6
    d = np_inputs(tiny(T=16, E=6, k=6, seed=5, router_std=0.3))
    rt = oracle.route_topk(d["x"], d["Wr"], None, 6)
    L = oracle.router_logits(d["x"], d["Wr"], None).astype(np.float64)
    full = torch.softmax(torch.from_numpy(L), dim=1).numpy()
    got = np.zeros_like(full)
    np.put_along_axis(got, rt["topk_idx"].astype(np.int64), rt["topk_w"].astype(np.float64), 1)
    assert np.max(np.abs(got - full)) < 2e-6
    d = np_inputs(tiny(T=16, E=1, k=1, seed=6))
    rt = oracle.route_topk(d["x"], d["Wr"], None, 1)
    assert np.all(rt["topk_idx"] == 0) and np.all(rt["topk_w"] == 1.0)
    # logits ln3 and 0: weights 3/4 and 1/4 (to fp32 rounding of ln 3)
    x = np.full((1, 64), 0x3F80, np.uint16)
    Wr = np.zeros((64, 2), np.float32)
    Wr[0, 0] = np.float32(np.log(3.0))
    rt = oracle.route_topk(x, Wr, None, 2)
    assert rt["topk_idx"][0].tolist() == [0, 1]
    assert np.allclose(rt["topk_w"][0], [0.75, 0.25], rtol=0, atol=1e-7)


# ---------------------------------------------------------- A2 histogram

def pin_counts_offsets():
    for E, k, ep in ((8, 2, 2), (16, 4, 4), (12, 3, 3)):
        d = np_inputs(tiny(T=100, E=E, k=k, seed=E + k, router_std=0.3))
        rt = oracle.route_topk(d["x"], d["Wr"], None, k, ep)
        idx = rt["topk_idx"]
        assert rt["counts"].tolist() == np.bincount(idx.ravel(), minlength=E).tolist()
        assert int(rt["counts"].sum()) == 100 * k
        assert rt["offsets"].tolist() == [0] + np.cumsum(rt["counts"]).tolist()
        assert rt["offsets"][-1] == 100 * k
        per = E // ep
        assert rt["rank_offsets"].tolist() == [int(rt["offsets"][r * per]) for r in range(ep + 1)]
        assert np.all((rt["counts"] >= 0) & (rt["counts"] <= 100))


# ----------------------------------------------------------- A3 dispatch

def pin_permutation():
    for E, k in ((8, 2), (16, 4)):
        T = 96
        d = np_inputs(tiny(T=T, E=E, k=k, seed=10 + E, router_std=0.5))
        rt = oracle.route_topk(d["x"], d["Wr"], None, k)
        dp = oracle.dispatch(d["x"], rt["topk_idx"], rt["offsets"], E)
        ros, tor = dp["row_of_slot"], dp["token_of_row"]
        R = T * k
        assert sorted(ros.ravel().tolist()) == list(range(R))
        order = np.argsort(rt["topk_idx"].ravel(), kind="stable")   # slots sorted by expert, stable
        rows = np.empty(R, np.int64)
        rows[order] = np.arange(R)
        assert np.array_equal(rows.reshape(T, k), ros)
        assert np.array_equal(tor[ros], np.repeat(np.arange(T), k).reshape(T, k))
        for j in range(k):
            assert np.array_equal(dp["x_perm"][ros[:, j]], d["x"])     # unpermute(permute(x)) == x
        for e in range(E):
            rows_e = ros[rt["topk_idx"] == e]
            assert np.all((rows_e >= rt["offsets"][e]) & (rows_e < rt["offsets"][e + 1]))


# ---------------------------------------------------- A4..A6 the forward

def pin_forward_dense_fp64():
    for E, k, bias in ((8, 2, None), (8, 3, "zipf")):
        d = np_inputs(tiny(T=64, E=E, k=k, seed=20 + k, bias=bias, router_std=0.3))
        f = oracle_forward(d)
        ref, _, _ = dense_forward_fp64(d, f["rt"]["topk_idx"])
        ref = ref.numpy()
        assert rel_l2(f["y"], ref) < 1e-5, rel_l2(f["y"], ref)
        assert np.max(np.abs(f["y"] - ref)) < 1e-4 * np.max(np.abs(ref))


def pin_dense_mlp_special_case():
    """E = 1, k = 1: the layer is a plain SwiGLU MLP (torch fp64)."""
    d = np_inputs(tiny(T=32, H=64, I=64, E=1, k=1, seed=30))
    f = oracle_forward(d)
    x = torch.from_numpy(oracle.widen_bf16(d["x"]).astype(np.float64))
    Wg = torch.from_numpy(oracle.widen_bf16(d["Wg"][0]).astype(np.float64))
    Wu = torch.from_numpy(oracle.widen_bf16(d["Wu"][0]).astype(np.float64))
    Wd = torch.from_numpy(oracle.widen_bf16(d["Wd"][0]).astype(np.float64))
    ref = (F.silu(F.linear(x, Wg)) * F.linear(x, Wu)) @ Wd.T
    assert rel_l2(f["y"], ref.numpy()) < 1e-5


def pin_identity_experts():
    """Identity experts (y_perm = x_perm): combine returns x * sum_j w_j = x."""
    d = np_inputs(tiny(T=64, E=8, k=3, seed=40, router_std=0.5))
    rt = oracle.route_topk(d["x"], d["Wr"], None, 3)
    dp = oracle.dispatch(d["x"], rt["topk_idx"], rt["offsets"], 8)
    y = oracle.combine(oracle.widen_bf16(dp["x_perm"]), rt["topk_w"], dp["row_of_slot"])
    xv = oracle.widen_bf16(d["x"]).astype(np.float64)
    sw = rt["topk_w"].astype(np.float64).sum(1, keepdims=True)
    assert np.max(np.abs(y - xv * sw)) <= 8 * U * np.max(np.abs(xv))
    assert np.max(np.abs(y - xv)) <= 1e-5 * np.max(np.abs(xv))


def pin_segments_dense():
    """Segmented receive-side layout (source-rank blocks x experts, some
    segments empty) equals per-row dense fp64 evaluation."""
    shape = LayerShape(T=200, H=128, I=64, E=4, k=1, ep_size=2, segments=True, src_ranks=3)
    s = make_segment_inputs(shape, seed=50)
    xp = oracle.widen_bf16(bf16_bits(s["x_perm"]))
    Wg, Wu, Wd = (bf16_bits(s[n]) for n in ("Wg", "Wu", "Wd"))
    so = s["seg_offsets"].numpy().copy(); se = s["seg_expert"].numpy()
    so[5:7] = so[4]                      # force empty segments 4 and 5
    so[7:] = np.maximum(so[7:], so[4])
    h = oracle.grouped_gemm_swiglu(xp, Wg, Wu, so, se)
    y = oracle.grouped_gemm_down(h, Wd, so, se)
    xv = torch.from_numpy(xp.astype(np.float64))
    ref = torch.zeros(xv.shape[0], 128, dtype=torch.float64)
    for q in range(len(so) - 1):
        e = int(se[q]); a, b = int(so[q]), int(so[q + 1])
        if b == a:
            continue
        g = xv[a:b] @ torch.from_numpy(oracle.widen_bf16(Wg[e]).astype(np.float64)).T
        u = xv[a:b] @ torch.from_numpy(oracle.widen_bf16(Wu[e]).astype(np.float64)).T
        ref[a:b] = (F.silu(g) * u) @ torch.from_numpy(oracle.widen_bf16(Wd[e]).astype(np.float64)).T
    covered = np.zeros(xv.shape[0], bool)
    covered[so[0]:so[-1]] = True
    assert rel_l2(y[covered], ref.numpy()[covered]) < 1e-5


# ------------------------------------------------------------ B1..B5

def oracle_backward(d, f, dy):
    dy_perm, d_w = oracle.combine_bwd(dy, f["y_perm"], f["rt"]["topk_w"], f["dp"]["row_of_slot"])
    offs = f["rt"]["offsets"]
    dgu, dWd = oracle.grouped_gemm_down_bwd(dy_perm, f["h"], f["gu"], d["Wd"], offs)
    dx_perm, dWg, dWu = oracle.grouped_gemm_swiglu_bwd(dgu, f["x_perm"], d["Wg"], d["Wu"], offs)
    dx_acc = oracle.dispatch_bwd(dx_perm, f["dp"]["row_of_slot"])
    dWr, dx = oracle.route_topk_bwd(d_w, f["rt"]["topk_w"], f["rt"]["topk_idx"], d["x"], d["Wr"], dx_acc)
    return dict(dy_perm=dy_perm, d_w=d_w, dgu=dgu, dWd=dWd, dx_perm=dx_perm, dWg=dWg, dWu=dWu,
                dx_acc=dx_acc, dWr=dWr, dx=dx)


def pin_backward_autograd():
    """Oracle gradients = torch fp64 autograd of the dense forward (routing
    fixed), which is itself checked by central finite differences."""
    for E, k, H, I in ((4, 2, 16, 8), (8, 3, 64, 64)):
        d = np_inputs(tiny(T=8 if E == 4 else 24, H=H, I=I, E=E, k=k, seed=60 + E, with_dy=True,
                           router_std=0.5))
        f = oracle_forward(d, save_gu=True)
        dyv = oracle.widen_bf16(d["dy"])
        b = oracle_backward(d, f, dyv)
        y, _, leaves = dense_forward_fp64(d, f["rt"]["topk_idx"], leaf=True)
        dyt = torch.from_numpy(dyv.astype(np.float64))
        (y * dyt).sum().backward()
        x, Wr, Wg, Wu, Wd = leaves
        for name, got, ref in (("dx", b["dx"], x.grad), ("dWr", b["dWr"], Wr.grad),
                               ("dWg", b["dWg"], Wg.grad), ("dWu", b["dWu"], Wu.grad),
                               ("dWd", b["dWd"], Wd.grad)):
            err = rel_l2(got, ref.numpy())
            assert err < 2e-5, (name, err)
        # the dWr columns sum to zero: sum_j dlogit_j = 0 for every token
        colsum = b["dWr"].astype(np.float64).sum(1)
        assert np.max(np.abs(colsum)) <= 1e-5 * np.max(np.abs(b["dWr"])) * E
        if E == 4:
            _finite_difference_check(d, f["rt"]["topk_idx"], dyt, leaves)


def _finite_difference_check(d, idx, dyt, leaves, eps=1e-6):
    x, Wr, Wg, Wu, Wd = leaves
    rng = np.random.default_rng(0)

    def loss():
        with torch.no_grad():
            xx, WWr, WWg, WWu, WWd = (p.detach() for p in leaves)
            logits = xx @ WWr
            w = torch.softmax(logits.gather(1, torch.from_numpy(idx.astype(np.int64))), 1)
            y = torch.zeros(xx.shape[0], WWd.shape[1], dtype=torch.float64)
            for t in range(xx.shape[0]):
                for j in range(idx.shape[1]):
                    e = int(idx[t, j])
                    v = xx[t]
                    y[t] += w[t, j] * ((F.silu(WWg[e] @ v) * (WWu[e] @ v)) @ WWd[e].T)
            return float((y * dyt).sum())

    for p in (x, Wr, Wg, Wu, Wd):
        flat = p.data.view(-1)
        for q in rng.choice(flat.numel(), 3, replace=False):
            old = float(flat[q])
            flat[q] = old + eps; lp = loss()
            flat[q] = old - eps; lm = loss()
            flat[q] = old
            fd = (lp - lm) / (2 * eps)
            g = float(p.grad.view(-1)[q])
            assert abs(fd - g) <= 1e-6 + 1e-5 * abs(g), (fd, g)


def _bf16_of(rng, shape, std):
    v = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    return bf16_bits(v.to(torch.bfloat16))


def pin_segments_backward():
    """Backward over a receive-side segment table: several segments per
    expert in an order that is neither sorted nor identity, empty segments,
    an expert that owns no segment, and rows before the first and after the
    last segment.  dgu, dx_perm, dWd, dWg and dWu equal fp64 torch autograd
    of the per-segment dense forward; accumulate adds the fresh sum to the
    buffer exactly; the segment-less expert's gradients are exactly zero
    (overwrite) or untouched (accumulate); uncovered rows stay zero.

    The layout is the one an EP rank receives ("Qwen3-MoE-30B-A3B模型EP+FSDP2
    并行方案", "完整并行流程" and "Expert Parallelism Details": rows arrive per
    source rank, the expert compute runs on local tensors); empty groups:
    "FSDPTurbo EP/EFSDP and LlamaFactory FSDP2/CP Design", section 3.
    """
    rng = np.random.default_rng(75)
    H, I, E = 64, 64, 5
    lens = [10, 0, 15, 12, 7, 20, 0, 9, 14, 11, 25, 19]
    se = np.array([2, 0, 3, 1, 0, 2, 1, 3, 3, 1, 0, 2], np.int32)  # expert 4 owns no segment
    lead, tail = 8, 10
    so = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32) + lead
    R = int(so[-1]) + tail
    xb = _bf16_of(rng, (R, H), 1.0)
    Wg, Wu = _bf16_of(rng, (E, I, H), 0.2), _bf16_of(rng, (E, I, H), 0.2)
    Wd = _bf16_of(rng, (E, H, I), 0.2)
    dy = oracle.widen_bf16(_bf16_of(rng, (R, H), 1.0))
    xp = oracle.widen_bf16(xb)

    h, gu = oracle.grouped_gemm_swiglu(xp, Wg, Wu, so, se, save_gu=True)
    dgu, dWd = oracle.grouped_gemm_down_bwd(dy, h, gu, Wd, so, se)
    dx_perm, dWg, dWu = oracle.grouped_gemm_swiglu_bwd(dgu, xp, Wg, Wu, so, se)

    f64 = lambda a: torch.from_numpy(oracle.widen_bf16(a).astype(np.float64))
    x = torch.from_numpy(xp.astype(np.float64)).requires_grad_(True)
    tWg, tWu, tWd = (f64(a).requires_grad_(True) for a in (Wg, Wu, Wd))
    dyt = torch.from_numpy(dy.astype(np.float64))
    loss = torch.zeros((), dtype=torch.float64)
    parts = []
    for q in range(len(se)):
        a, b, e = int(so[q]), int(so[q + 1]), int(se[q])
        if b == a:
            continue
        g = x[a:b] @ tWg[e].T
        u = x[a:b] @ tWu[e].T
        g.retain_grad(); u.retain_grad()
        y = (F.silu(g) * u) @ tWd[e].T
        loss = loss + (y * dyt[a:b]).sum()
        parts.append((a, b, g, u))
    loss.backward()
    dgu_ref = np.zeros((R, 2 * I))
    for a, b, g, u in parts:
        dgu_ref[a:b, :I] = g.grad.numpy()
        dgu_ref[a:b, I:] = u.grad.numpy()
    cov = slice(int(so[0]), int(so[-1]))
    for name, got, ref in (("dgu", dgu[cov], dgu_ref[cov]), ("dx_perm", dx_perm[cov], x.grad.numpy()[cov]),
                           ("dWd", dWd, tWd.grad.numpy()), ("dWg", dWg, tWg.grad.numpy()),
                           ("dWu", dWu, tWu.grad.numpy())):
        err = rel_l2(got, ref)
        assert err < 2e-5, (name, err)
    for name, got in (("dgu", dgu), ("dx_perm", dx_perm)):
        assert not np.any(got[:lead]) and not np.any(got[R - tail:]), name
    for name, got in (("dWd", dWd), ("dWg", dWg), ("dWu", dWu)):
        assert np.all(got[4] == 0), name
    # every expert's gradient is the sum over all of its segments: dropping
    # any one non-empty segment changes it by a visible amount
    for e in range(4):
        own = [q for q in range(len(se)) if se[q] == e and so[q + 1] > so[q]]
        assert len(own) >= 2, e

    prev = [rng.standard_normal(a.shape).astype(np.float32) for a in (dWd, dWg, dWu)]
    _, acc_d = oracle.grouped_gemm_down_bwd(dy, h, gu, Wd, so, se, dWd=prev[0])
    _, acc_g, acc_u = oracle.grouped_gemm_swiglu_bwd(dgu, xp, Wg, Wu, so, se, dWg=prev[1], dWu=prev[2])
    for name, acc, p0, fresh, ref in (("dWd", acc_d, prev[0], dWd, tWd.grad.numpy()),
                                      ("dWg", acc_g, prev[1], dWg, tWg.grad.numpy()),
                                      ("dWu", acc_u, prev[2], dWu, tWu.grad.numpy())):
        assert np.array_equal(acc, p0 + fresh), name
        assert np.array_equal(acc[4], p0[4]), name
        assert rel_l2(acc - p0, ref) < 2e-5, name


def pin_accumulate_and_empty():
    """accumulate=1 adds the fresh sum to the buffer; an expert with no rows
    gets an exactly-zero weight gradient in overwrite mode."""
    d = np_inputs(tiny(T=16, H=64, I=64, E=8, k=1, seed=70, with_dy=True))
    d["bias"] = np.zeros(8, np.float32)
    d["bias"][[5, 7]] = -1.0e4     # experts 5 and 7 receive no token
    f = oracle_forward(d, save_gu=True)
    assert f["rt"]["counts"][5] == 0 and f["rt"]["counts"][7] == 0
    b = oracle_backward(d, f, oracle.widen_bf16(d["dy"]))
    for name in ("dWd", "dWg", "dWu"):
        assert np.all(b[name][5] == 0) and np.all(b[name][7] == 0), name
    prev = np.random.default_rng(1).standard_normal(b["dWd"].shape).astype(np.float32)
    offs = f["rt"]["offsets"]
    _, acc = oracle.grouped_gemm_down_bwd(b["dy_perm"], f["h"], f["gu"], d["Wd"], offs, dWd=prev)
    assert np.array_equal(acc, prev + b["dWd"])
    prev_r = np.random.default_rng(2).standard_normal(b["dWr"].shape).astype(np.float32)
    accr, _ = oracle.route_topk_bwd(b["d_w"], f["rt"]["topk_w"], f["rt"]["topk_idx"], d["x"], d["Wr"],
                                    b["dx_acc"], dWr=prev_r)
    assert np.array_equal(accr, prev_r + b["dWr"])


# ------------------------------------------------------------ FP8 (e4m3)
#
# Format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
# infinities, 0x7F/0xFF NaN, largest finite 448 (torch.float8_e4m3fn is the
# same format).  Scaling reading: one fp32 scale per stored row (token row,
# permuted row, expert output channel), s = amax / 448.


def _torch_e4m3_codes(v):
    return torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _finite_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


def pin_e4m3_decode():
    """Every finite code decodes as torch's float8_e4m3fn does; closed forms."""
    c = _finite_codes()
    dec = oracle.e4m3_decode(c)
    ref = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(dec.view(np.uint32), ref.view(np.uint32))
    closed = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
              0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    got = oracle.e4m3_decode(np.array(list(closed), np.uint8))
    assert np.array_equal(got, np.array(list(closed.values()), np.float32))


def pin_e4m3_encode():
    """Round to nearest even: every midpoint between neighbouring codes, one
    fp32 ulp either side of it, and seeded values over eight decades give
    torch's conversion; magnitudes at or above 448 saturate to 448."""
    c = _finite_codes()
    pos = np.sort(oracle.e4m3_decode(c[c < 0x80]).astype(np.float64))
    mids = ((pos[1:] + pos[:-1]) / 2).astype(np.float32)
    probes = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf)),
                             pos.astype(np.float32)])
    rng = np.random.default_rng(60)
    seeded = np.concatenate([(rng.standard_normal(20000) * sc).astype(np.float32)
                             for sc in (1e-4, 1e-3, 1e-2, 0.1, 1.0, 10.0, 100.0)])
    v = np.concatenate([probes, -probes, seeded, np.array([0.0, -0.0], np.float32)])
    v = v[np.abs(v) < 464]
    assert np.array_equal(oracle.e4m3_encode(v), _torch_e4m3_codes(v))
    big = np.array([448, 463.9, 464, 500, 1e30, -448, -1e10], np.float32)
    assert np.array_equal(oracle.e4m3_encode(big), np.array([0x7E] * 5 + [0xFE] * 2, np.uint8))


def pin_quantize_rows():
    """Per-row scaling: the largest magnitude of each row maps to code 448,
    dequantised values are within half a quantum (2^-4 relative, 2^-10 * s
    absolute in the subnormal range), signs are kept, an all-zero row gets
    scale 1 and zero codes."""
    rng = np.random.default_rng(61)
    a = (rng.standard_normal((40, 96)) * np.exp(rng.uniform(-8, 8, (40, 1)))).astype(np.float32)
    a[3] = 0.0
    a[5, :] = 0.0
    a[5, 17] = -3.5
    a[7, ::2] *= 1e-6                     # many values in the subnormal range of that row
    q, s = oracle.quantize_rows_e4m3(a)
    dec = oracle.e4m3_decode(q).astype(np.float64)
    for r in range(a.shape[0]):
        amax = np.abs(a[r]).max()
        if amax == 0:
            assert s[r] == 1.0 and not (q[r] & 0x7F).any()
            continue
        assert np.abs(dec[r]).max() == 448.0
        assert abs(s[r] * 448.0 - amax) <= 2 * U * amax
        err = np.abs(dec[r] * s[r] - a[r].astype(np.float64))
        assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(a[r]), 2.0 ** -10 * s[r]) * (1 + 4 * U) + 1e-45)
        nz = dec[r] != 0
        assert np.array_equal(np.sign(dec[r][nz]), np.sign(a[r][nz]))
    assert np.abs(dec[5]).max() == 448.0 and q[5, 17] == 0xFE


def pin_quantize_rows_power_of_two_scale():
    """A row whose largest magnitude is 448 * 2^j has the scale 2^j exactly,
    so every quotient a / s is exact and the codes must be torch's
    conversion of a * 2^-j: midpoints between codes (ties to even), one
    ulp either side of them and every code value, at scales from the fp32
    subnormal 2^-130 up to 2^7."""
    c = _finite_codes()
    pos = np.sort(oracle.e4m3_decode(c[c < 0x80]).astype(np.float32))
    mids = (pos[1:] + pos[:-1]) / np.float32(2)           # 5 significant bits: exact
    near = np.concatenate([np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf))])
    rows, expect = [], []
    for j in (-130, -20, 0, 7):
        # fp32 ulp neighbours only where 2^j keeps them normal; at 2^-130 they
        # would lose bits as subnormals, the midpoints and codes do not
        base = np.concatenate([mids, pos] + ([near] if j > -100 else [])).astype(np.float64)
        row = np.concatenate([[448.0], base, -base]) * 2.0 ** j
        row32 = row.astype(np.float32)
        assert np.array_equal(row32.astype(np.float64), row)
        rows.append(row32)
        expect.append(_torch_e4m3_codes((row / 2.0 ** j).astype(np.float32)))
    width = max(len(r) for r in rows)                      # pad with zeros (code 0)
    rows = [np.pad(r, (0, width - len(r))) for r in rows]
    expect = [np.pad(e, (0, width - len(e))) for e in expect]
    q, s = oracle.quantize_rows_e4m3(np.stack(rows))
    assert np.array_equal(s.astype(np.float64), np.array([2.0 ** j for j in (-130, -20, 0, 7)]))
    assert np.array_equal(q, np.stack(expect))


def _int_codes(rng, shape, lo=-8, hi=8):
    """e4m3 codes of random small integers (exactly representable)."""
    v = rng.integers(lo, hi + 1, shape).astype(np.float32)
    return oracle.e4m3_encode(v), v.astype(np.int64)


def pin_fp8_gemms_integer_case():
    """Integer-valued codes and power-of-two scales: g, u and y_perm are
    exact (integer matmul in numpy, per segment, with empty and reordered
    segments); h = silu(g) * u against torch fp64."""
    rng = np.random.default_rng(62)
    R, H, I, E = 70, 64, 32, 4
    aq, av = _int_codes(rng, (R, H))
    Wgq, wg = _int_codes(rng, (E, I, H)); Wuq, wu = _int_codes(rng, (E, I, H))
    Wdq, wd = _int_codes(rng, (E, H, I))
    sa = (2.0 ** rng.integers(-6, 4, R)).astype(np.float32)
    sg = (2.0 ** rng.integers(-6, 4, (E, I))).astype(np.float32)
    su = (2.0 ** rng.integers(-6, 4, (E, I))).astype(np.float32)
    sd = (2.0 ** rng.integers(-6, 4, (E, H))).astype(np.float32)
    so = np.array([0, 20, 20, 45, 70], np.int32); se = np.array([2, 0, 3, 1], np.int32)
    h = oracle.grouped_gemm_swiglu_fp8(aq, sa, Wgq, sg, Wuq, su, so, se)
    hq, _ = _int_codes(rng, (R, I))
    hs = (2.0 ** rng.integers(-6, 4, R)).astype(np.float32)
    y = oracle.grouped_gemm_down_fp8(hq, hs, Wdq, sd, so, se)
    for q in range(4):
        a, b, e = so[q], so[q + 1], se[q]
        if a == b:
            continue
        g = (av[a:b] @ wg[e].T).astype(np.float64) * sa[a:b, None] * sg[e][None, :]
        u = (av[a:b] @ wu[e].T).astype(np.float64) * sa[a:b, None] * su[e][None, :]
        ref_h = (F.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
        assert np.allclose(h[a:b], ref_h, rtol=1e-6, atol=1e-30)
        ref_y = (_decode_int(hq[a:b]) @ wd[e].T).astype(np.float64) * hs[a:b, None] * sd[e][None, :]
        assert np.array_equal(y[a:b], ref_y.astype(np.float32))


def _decode_int(q):
    return oracle.e4m3_decode(q).astype(np.int64)


def pin_fp8_reduces_to_bf16_oracle():
    """Scale 1 and e4m3-representable inputs (every e4m3 value is a bf16
    value): the FP8 GEMMs equal the pinned bf16 oracle GEMMs up to the
    latter's fp32 summation error."""
    rng = np.random.default_rng(63)
    R, H, I, E = 48, 128, 64, 3
    codes = lambda shape: oracle.e4m3_encode(rng.standard_normal(shape).astype(np.float32))
    aq, Wgq, Wuq, Wdq = codes((R, H)), codes((E, I, H)), codes((E, I, H)), codes((E, H, I))
    as_bf16 = lambda q: (oracle.e4m3_decode(q).view(np.uint32) >> 16).astype(np.uint16)
    so = np.array([0, 10, 30, 48], np.int32)
    one = lambda n: np.ones(n, np.float32)
    h8 = oracle.grouped_gemm_swiglu_fp8(aq, one(R), Wgq, one((E, I)), Wuq, one((E, I)), so)
    h16 = oracle.grouped_gemm_swiglu(oracle.e4m3_decode(aq), as_bf16(Wgq), as_bf16(Wuq), so)
    assert rel_l2(h8, h16) < 1e-6
    hq = codes((R, I))
    y8 = oracle.grouped_gemm_down_fp8(hq, one(R), Wdq, one((E, H)), so)
    y16 = oracle.grouped_gemm_down(oracle.e4m3_decode(hq), as_bf16(Wdq), so)
    assert rel_l2(y8, y16) < 1e-6


FP8_PINS = [pin_e4m3_decode, pin_e4m3_encode, pin_quantize_rows, pin_quantize_rows_power_of_two_scale,
            pin_fp8_gemms_integer_case, pin_fp8_reduces_to_bf16_oracle]

ALL_PINS = [pin_logit_block_order, pin_logits_error_bound, pin_topk_bruteforce, pin_topk_ties,
            pin_weights_closed_form, pin_counts_offsets, pin_permutation, pin_forward_dense_fp64,
            pin_dense_mlp_special_case, pin_identity_experts, pin_segments_dense,
            pin_backward_autograd, pin_segments_backward, pin_accumulate_and_empty] + FP8_PINS
