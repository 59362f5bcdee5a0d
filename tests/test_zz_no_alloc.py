"""moe_dispatch_no_alloc (dispatch without a workspace) against moe_dispatch.

Some callers cannot allocate device memory for a workspace (a fixed memory
plan made at start-up, or a plain C caller without a device allocator); this
entry point keeps its scratch in an array built into the library.  The test
calls it through the C ABI twice in a row and requires results identical to
the workspace entry point (dispatch is integer and copy work, so identical
means bit for bit), and checks that sizes beyond the built-in scratch are
refused on the host.  It runs last so that a failure here leaves every other
test already run, and it builds its own inputs so it also passes alone.
"""
import ctypes

import pytest
import torch

import moe_expert_layer_topk_gb300 as m
from moe_expert_layer_topk_gb300.synth import LayerShape, make_layer_inputs

pytestmark = pytest.mark.gpu


def test_no_alloc_dispatch_matches_workspace_dispatch():
    L = m.lib()
    T, H, I, E, k = 1000, 256, 64, 16, 4
    inp = make_layer_inputs(LayerShape(T=T, H=H, I=I, E=E, k=k, ep_size=4), seed=7, router_std=0.3)
    x = inp["x"].cuda()
    layer = m.MoELayer(T, H, I, E, k, 4, training=False)
    layer.route(x, inp["Wr"].cuda(), None)
    layer.dispatch(x)
    torch.cuda.synchronize()
    assert m.moe_read_device_status(reset=True) == 0
    ref = (layer.x_perm.clone(), layer.row_of_slot.clone(), layer.token_of_row.clone())
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        x_perm = torch.full_like(layer.x_perm, float("nan"))
        ros = torch.full_like(layer.row_of_slot, -7)
        tor = torch.full_like(layer.token_of_row, -7)
        rc = L.moe_dispatch_no_alloc(x.data_ptr(), layer.topk_idx.data_ptr(), layer.offsets.data_ptr(),
                                     T, H, E, k, x_perm.data_ptr(), ros.data_ptr(), tor.data_ptr(),
                                     ctypes.c_void_p(stream))
        assert rc == 0, L.moe_last_error_string()
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
