"""The seeded input generators that feed both the CUDA path and the oracle:
same seed, same bytes; the documented draw order; bf16 values rounded from
the fp32 draws; the receive-side segment tables of one EP rank; the Zipf
router bias.  CPU only, small sizes."""
import math

import numpy as np
import torch

from moe_expert_layer_topk_gb300.synth import (CONFIGS, bf16_bits, make_layer_inputs,
                                               make_segment_inputs, zipf_router_bias)


def _same(a, b):
    return a.dtype == b.dtype and a.shape == b.shape and torch.equal(a, b)


def test_layer_inputs_deterministic_and_shaped():
    a = make_layer_inputs("tiny_fwd", 0, with_dy=True)
    b = make_layer_inputs("tiny_fwd", 0, with_dy=True)
    c = make_layer_inputs("tiny_fwd", 1, with_dy=True)
    sh = CONFIGS["tiny_fwd"]
    for name in ("x", "Wr", "Wg", "Wu", "Wd", "dy"):
        assert _same(a[name], b[name]), name
        assert not torch.equal(a[name].float(), c[name].float()), name
    assert a["x"].shape == (sh.T, sh.H) and a["x"].dtype == torch.bfloat16
    assert a["Wr"].shape == (sh.H, sh.E) and a["Wr"].dtype == torch.float32
    assert a["Wg"].shape == (sh.E, sh.I, sh.H) and a["Wu"].shape == (sh.E, sh.I, sh.H)
    assert a["Wd"].shape == (sh.E, sh.H, sh.I) and a["dy"].shape == (sh.T, sh.H)
    assert a["bias"] is None


def test_draw_order_and_bf16_rounding():
    """x is the first draw: N(0,1) fp32 rounded to nearest even bf16; Wr the
    second, N(0,1) * 0.02 in fp32."""
    T, H, E = 64, 128, 8
    d = make_layer_inputs("tiny_fwd", 3, T=T)
    g = torch.Generator().manual_seed(3)
    x32 = torch.randn(T * H, generator=g, dtype=torch.float32)
    wr = torch.randn(H, E, generator=g, dtype=torch.float32).mul_(0.02)
    b = x32.numpy().view(np.uint32).astype(np.uint64)
    rne = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)   # no NaN among normal draws
    assert np.array_equal(bf16_bits(d["x"]).reshape(-1), rne)
    assert torch.equal(d["Wr"], wr)


def test_segment_inputs_tables():
    s = make_segment_inputs("ep_rank_local", 5, R=3000)
    E, S = CONFIGS["ep_rank_local"].E, CONFIGS["ep_rank_local"].src_ranks
    so, se = s["seg_offsets"].numpy(), s["seg_expert"].numpy()
    assert s["num_seg"] == S * E and len(so) == S * E + 1 and so[0] == 0 and so[-1] == 3000
    assert np.all(np.diff(so) >= 0)
    assert np.array_equal(se, np.arange(S * E) % E)
    per_expert = np.diff(so).reshape(S, E).sum(0)        # source-rank-major, then expert
    assert np.array_equal(per_expert, s["counts_e"].numpy())
    assert s["x_perm"].shape == (3000, s["H"])
    again = make_segment_inputs("ep_rank_local", 5, R=3000)
    assert torch.equal(again["seg_offsets"], s["seg_offsets"])


def test_zipf_router_bias():
    E = 128
    bias = zipf_router_bias(torch.Generator().manual_seed(0), E).double().numpy()
    empty = bias == -1.0e4
    assert empty.sum() == 4
    live = np.sort(bias[~empty])[::-1]                   # ranks 1 .. E-4 in popularity order
    expect = np.array([-2.0 * 1.2 * math.log(r) for r in range(1, E - 3)])
    assert np.allclose(live, expect, rtol=0, atol=1e-5)
