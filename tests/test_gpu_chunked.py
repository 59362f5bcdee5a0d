"""The route's chunk prefixes and the one-kernel dispatch built on them.

moe_route_topk_chunks gives the same routing as moe_route_topk, plus per
(expert, 16-token chunk) the number of that expert's slots in earlier
chunks, checked here against a count on the host.  moe_dispatch_chunked and
moe_dispatch_e4m3_chunked give bit for bit what moe_dispatch and
moe_dispatch_e4m3 give (and the oracle's permutation), on ragged token
counts, E = 1024 with k = 32, skewed routing with empty experts, a single
token and no token; inconsistent prefixes are skipped and reported."""
import numpy as np
import pytest
import torch

import moe_expert_layer_topk_gb300 as m
import oracle
from gpu_util import bits, dispatch_ws, inputs, to_dev

pytestmark = pytest.mark.gpu

CASES = [(1000, 128, 64, 128, 8, None), (77, 128, 64, 1024, 32, None), (1, 128, 64, 8, 2, None),
         (4096, 256, 64, 64, 6, "zipf"), (333, 192, 64, 12, 3, None)]


def _route(inp, chunks):
    g = to_dev(inp)
    T, H, E, k = inp["T"], inp["H"], inp["E"], inp["k"]
    i32 = dict(dtype=torch.int32, device="cuda")
    out = {"topk_idx": torch.empty(T, k, **i32), "topk_w": torch.empty(T, k, dtype=torch.float32, device="cuda"),
           "counts": torch.empty(E, **i32), "offsets": torch.empty(E + 1, **i32),
           "rank_offsets": torch.empty(inp["ep_size"] + 1, **i32)}
    if chunks:
        out["chunk_prefix"] = torch.full((E, (T + 15) // 16), -7, **i32)
        ws = torch.empty(m.moe_route_topk_chunks_workspace_size(T, H, E), dtype=torch.uint8, device="cuda")
        m.moe_route_topk_chunks(g["x"], g["Wr"], g["bias"], T, H, E, k, inp["ep_size"], out["topk_idx"],
                                out["topk_w"], out["counts"], out["offsets"], out["rank_offsets"],
                                out["chunk_prefix"], ws)
    else:
        ws = torch.empty(m.moe_route_topk_workspace_size(T, H, E), dtype=torch.uint8, device="cuda")
        m.moe_route_topk(g["x"], g["Wr"], g["bias"], T, H, E, k, inp["ep_size"], out["topk_idx"], out["topk_w"],
                         out["counts"], out["offsets"], out["rank_offsets"], ws)
    return g, out


def _host_prefix(topk_idx, E):
    T, k = topk_idx.shape
    nc = (T + 15) // 16
    ref = np.zeros((E, nc), np.int64)
    for c in range(1, nc):
        ref[:, c] = ref[:, c - 1] + np.bincount(topk_idx[16 * (c - 1):16 * c].ravel(), minlength=E)
    return ref


@pytest.mark.parametrize("T,H,I,E,k,bias", CASES)
def test_chunked_route_and_dispatch(T, H, I, E, k, bias):
    ep = 2 if E % 2 == 0 else 1
    inp = inputs(T, H, I, E, k, seed=90 + T, ep=ep, bias=bias, with_dy=False, router_std=0.3)
    g, a = _route(inp, chunks=False)
    _, c = _route(inp, chunks=True)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    for name in ("topk_idx", "topk_w", "counts", "offsets", "rank_offsets"):
        assert torch.equal(a[name], c[name]), name
    idx = c["topk_idx"].cpu().numpy()
    assert np.array_equal(c["chunk_prefix"].cpu().numpy(), _host_prefix(idx, E))
    if bias == "zipf":
        assert (c["counts"] == 0).sum().item() >= 4

    R = T * k
    bf = dict(dtype=torch.bfloat16, device="cuda")
    i32 = dict(dtype=torch.int32, device="cuda")
    xp_a, xp_c = torch.zeros(R, H, **bf), torch.full((R, H), 3.0, **bf)
    ros_a, ros_c = torch.empty(T, k, **i32), torch.full((T, k), -5, **i32)
    tor_a, tor_c = torch.empty(R, **i32), torch.full((R,), -5, **i32)
    m.moe_dispatch(g["x"], a["topk_idx"], a["offsets"], T, H, E, k, xp_a, ros_a, tor_a, dispatch_ws(T, E, k))
    m.moe_dispatch_chunked(g["x"], c["topk_idx"], c["offsets"], c["chunk_prefix"], T, H, E, k, xp_c, ros_c, tor_c)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    assert torch.equal(ros_a, ros_c) and torch.equal(tor_a, tor_c) and torch.equal(xp_a, xp_c)
    # the oracle's permutation of the same routing
    od = oracle.dispatch(bits(inp["x"]), idx, c["offsets"].cpu().numpy(), E)
    assert np.array_equal(ros_c.cpu().numpy(), od["row_of_slot"])
    assert np.array_equal(bits(xp_c), od["x_perm"])
    # indices only
    ros_n, tor_n = torch.full((T, k), -5, **i32), torch.full((R,), -5, **i32)
    m.moe_dispatch_chunked(None, c["topk_idx"], c["offsets"], c["chunk_prefix"], T, H, E, k, None, ros_n, tor_n)
    torch.cuda.synchronize()
    assert torch.equal(ros_n, ros_a) and torch.equal(tor_n, tor_a)

    if H % 128 == 0:
        u8 = dict(dtype=torch.uint8, device="cuda")
        q_a, q_c = torch.zeros(R, H, **u8), torch.full((R, H), 0x5A, **u8)
        s_a, s_c = torch.zeros(R, dtype=torch.float32, device="cuda"), torch.full((R,), -1.0, device="cuda")
        m.moe_dispatch_e4m3(g["x"], a["topk_idx"], a["offsets"], T, H, E, k, q_a, s_a, ros_a, tor_a,
                            dispatch_ws(T, E, k))
        m.moe_dispatch_e4m3_chunked(g["x"], c["topk_idx"], c["offsets"], c["chunk_prefix"], T, H, E, k, q_c, s_c,
                                    ros_c, tor_c)
        torch.cuda.synchronize()
        assert m.moe_read_device_status(reset=True) == 0
        assert torch.equal(q_a, q_c) and torch.equal(s_a, s_c) and torch.equal(ros_a, ros_c)


def test_chunked_no_token():
    inp = inputs(0, 128, 64, 8, 2, seed=3, with_dy=False)
    _, c = _route(inp, chunks=True)
    torch.cuda.synchronize()
    assert torch.all(c["counts"] == 0) and torch.all(c["offsets"] == 0)
    i32 = dict(dtype=torch.int32, device="cuda")
    m.moe_dispatch_chunked(None, c["topk_idx"], c["offsets"], c["chunk_prefix"], 0, 128, 8, 2, None,
                           torch.empty(0, 2, **i32), torch.empty(0, **i32))
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0


def test_chunked_dispatch_skips_inconsistent_prefixes():
    """A prefix that points past the last row is skipped and reported (the
    kernel bounds every row it writes), the other slots still land."""
    inp = inputs(64, 128, 64, 8, 2, seed=4, with_dy=False)
    g, c = _route(inp, chunks=True)
    idx = c["topk_idx"].cpu().numpy()
    e = int(idx[16, 0])  # an expert that chunk 1 (tokens 16..31) uses
    bad = c["chunk_prefix"].clone()
    bad[e, 1] = 1 << 20
    R, i32 = 128, dict(dtype=torch.int32, device="cuda")
    ros, tor = torch.full((64, 2), -5, **i32), torch.full((R,), -5, **i32)
    xp = torch.zeros(R, 128, dtype=torch.bfloat16, device="cuda")
    m.moe_dispatch_chunked(g["x"], c["topk_idx"], c["offsets"], bad, 64, 128, 8, 2, xp, ros, tor)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) & 1  # MOE_STATUS_BAD_INDEX
    hit = np.zeros_like(idx, bool)
    hit[16:32] = idx[16:32] == e
    assert np.all(ros.cpu().numpy()[hit] == -1) and np.all(ros.cpu().numpy()[~hit] >= 0)
