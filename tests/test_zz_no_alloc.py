"""moe_dispatch_no_alloc (dispatch without a workspace) against moe_dispatch.

Some callers cannot allocate device memory for a workspace (a fixed memory
plan made at start-up, or a plain C caller without a device allocator); this
entry point keeps its scratch in an array built into the library.  The test
calls it through the C ABI twice in a row and requires results identical to
the workspace entry point (dispatch is integer and copy work, so identical
means bit for bit), and checks that sizes beyond the built-in scratch are
refused on the host.  A larger call with other routing runs first, so the
checked calls find the shared scratch holding another call's values.  It
runs last so that a failure here leaves every other test already run, and it
builds its own inputs so it also passes alone.
"""
import ctypes

import pytest
import torch

import moe_expert_layer_topk_gb300 as m
from moe_expert_layer_topk_gb300.synth import LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


def _routed(T, H, I, E, k, seed):
    inp = make_layer_inputs(LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=4), seed=seed, router_std=0.3)
    x = inp["x"].cuda()
    layer = m.MoELayer(T, H, I, E, k, 4, training=False)
    layer.route(x, inp["Wr"].cuda(), None)
    return x, layer


def _no_alloc(L, x, layer, stream):
    x_perm = torch.full_like(layer.x_perm, float("nan"))
    ros = torch.full_like(layer.row_of_slot, -7)
    tor = torch.full_like(layer.token_of_row, -7)
    rc = L.moe_dispatch_no_alloc(x.data_ptr(), layer.topk_idx.data_ptr(), layer.offsets.data_ptr(),
                                 layer.T, layer.H, layer.E, layer.k, x_perm.data_ptr(), ros.data_ptr(),
                                 tor.data_ptr(), ctypes.c_void_p(stream))
    assert rc == 0, L.moe_last_error_string()
    return x_perm, ros, tor


def test_no_alloc_dispatch_matches_workspace_dispatch():
    L = m.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # a larger call with other routing first, so that the shared scratch
    # holds another call's values when the checked calls start
    x_big, big = _routed(2600, 256, 64, 48, 6, seed=8)
    _no_alloc(L, x_big, big, stream)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0

    T, H, I, E, k = 1000, 256, 64, 16, 4
    x, layer = _routed(T, H, I, E, k, seed=7)
    ws = torch.empty(m.moe_dispatch_workspace_size(T, E, k), dtype=torch.uint8, device="cuda")
    ref = (torch.empty_like(layer.x_perm), torch.empty_like(layer.row_of_slot), torch.empty_like(layer.token_of_row))
    m.moe_dispatch(x, layer.topk_idx, layer.offsets, T, H, E, k, ref[0], ref[1], ref[2], ws)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    for call in range(2):
        x_perm, ros, tor = _no_alloc(L, x, layer, stream)
        torch.cuda.synchronize()
        assert m.moe_read_device_status(reset=True) == 0
        assert torch.equal(x_perm.view(torch.int16), ref[0].view(torch.int16)), call
        assert torch.equal(ros, ref[1]), call
        assert torch.equal(tor, ref[2]), call


def test_no_alloc_dispatch_refuses_sizes_beyond_its_scratch():
    L = m.lib()
    cap = L.moe_dispatch_no_alloc_max_scratch()
    E = 1024
    T = (cap // E + 1) * 16          # one chunk more than fits
    P = 0x10000                      # never dereferenced: refused before any launch
    assert L.moe_dispatch_no_alloc(P, P, P, T, 128, E, 2, P, P, P, None) == -4
    assert "scratch" in L.moe_last_error_string().decode()
