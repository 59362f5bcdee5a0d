"""Seeded random layer shapes, forward and backward, every stored tensor
against the oracle's own fp32 chain: shapes no hand-picked case covers
(any T, H and I multiples of 64 up to 512, 1 to 48 experts, k up to 8, EP
ranks dividing E, with and without a router bias).  Routing, counts,
offsets and the permutation bit for bit; floats within the acceptance bars.
The shapes come from a fixed seed, so a failure names a reproducible case."""
import random

import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
from gpu_util import assert_close, bits, inputs, oracle_backward, oracle_chain, to_dev

pytestmark = pytest.mark.gpu


def _shapes(n, seed=2024):
    rnd = random.Random(seed)
    out = []
    for _ in range(n):
        E = rnd.randint(1, 48)
        k = rnd.randint(1, min(E, 8))
        eps = [d for d in range(1, E + 1) if E % d == 0 and d <= 8]
        out.append(dict(T=rnd.randint(1, 700), H=64 * rnd.randint(1, 8), I=64 * rnd.randint(1, 6), E=E, k=k,
                        ep=rnd.choice(eps), bias=rnd.choice([None, "zipf"])))
    return out


SHAPES = _shapes(8)


@pytest.mark.parametrize("s", SHAPES, ids=[f"T{s['T']}_H{s['H']}_I{s['I']}_E{s['E']}_k{s['k']}" for s in SHAPES])
def test_random_shape_layer(s):
    T, H, I, E, k, ep = s["T"], s["H"], s["I"], s["E"], s["k"], s["ep"]
    inp = inputs(T, H, I, E, k, seed=T + 7 * E, ep=ep, bias=s["bias"],
                 router_std=0.02 if s["bias"] is None else 0.3)
    g = to_dev(inp)
    L = m.MoELayer(T, H, I, E, k, ep)
    L.forward(g["x"], g["Wr"], g["bias"], g["Wg"], g["Wu"], g["Wd"])
    L.backward(g["dy"], g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    f = oracle_chain(inp)
    b = oracle_backward(inp, f)
    assert np.array_equal(L.topk_idx.cpu().numpy(), f["rt"]["topk_idx"])
    assert np.array_equal(L.counts.cpu().numpy(), f["rt"]["counts"])
    assert np.array_equal(L.offsets.cpu().numpy(), f["rt"]["offsets"])
    assert np.array_equal(L.rank_offsets.cpu().numpy(), f["rt"]["rank_offsets"])
    assert np.array_equal(L.row_of_slot.cpu().numpy(), f["dp"]["row_of_slot"])
    assert np.array_equal(L.token_of_row.cpu().numpy(), f["dp"]["token_of_row"])
    assert np.array_equal(bits(L.x_perm), f["dp"]["x_perm"])
    assert_close(L.topk_w, f["rt"]["topk_w"], "topk_w", max_frac=1e-5, rel=1e-6)
    for name, ref in (("h", f["h"]), ("gu", f["gu"]), ("y_perm", f["y_perm"]), ("y", f["y"])):
        assert_close(getattr(L, name), ref, name)
    for name in ("dy_perm", "d_w", "dgu", "dWd", "dx_perm", "dWg", "dWu", "dx_acc", "dWr", "dx"):
        assert_close(getattr(L, name), b[name], name)
