"""The C-ABI library loads and exports what include/moe_topk.h declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import re
from pathlib import Path

import pytest

import moe_expert_layer_topk_gb300 as m
from moe_expert_layer_topk_gb300 import build as b

HEADER = Path(__file__).resolve().parents[1] / "include" / "moe_topk.h"
DECL = re.compile(r"^(?:int|size_t|const char\*)\s+(moe_\w+)\s*\(([^;]*)\);", re.M | re.S)

OK, INVALID, SHAPE, ALIGN, WS = 0, -1, -2, -3, -4


@pytest.fixture(scope="module")
def L():
    b.build()
    return m.lib()


def header_decls():
    return {name: args for name, args in DECL.findall(HEADER.read_text())}


def test_abi_version(L):
    assert L.moe_abi_version() == 103  # 1.03: the fused down + combine call


def test_header_symbols_exported(L):
    decls = header_decls()
    assert len(decls) >= 16
    for name in decls:
        assert hasattr(L, name), name


def test_binding_matches_header(L):
    decls = header_decls()
    assert set(decls) == set(m.ENTRY_POINTS), set(decls) ^ set(m.ENTRY_POINTS)
    for name, args in decls.items():
        n = 0 if args.strip() in ("", "void") else args.count(",") + 1
        assert len(m.ENTRY_POINTS[name][0]) == n, name


def test_workspace_queries(L):
    assert m.moe_route_topk_workspace_size(4096, 2048, 128) >= 4096 * 128 * 4
    assert m.moe_dispatch_workspace_size(4096, 128, 8) >= (4096 // 32) * 128 * 4
    assert m.moe_route_topk_bwd_workspace_size(8192, 2048, 128) > 0
    assert m.moe_route_topk_workspace_size(-1, 2048, 128) == 0


def _err(L):
    return L.moe_last_error_string().decode()


FAKE = 0x10000  # never dereferenced: every call below fails host validation first


def test_route_rejects_bad_shapes(L):
    P = FAKE
    assert L.moe_route_topk(P, P, None, 16, 128, 8, 9, 1, P, P, P, P, P, P, 1 << 20, None) == SHAPE
    assert "k<=" in _err(L)
    assert L.moe_route_topk(P, P, None, 16, 100, 8, 2, 1, P, P, P, P, P, P, 1 << 20, None) == SHAPE
    assert L.moe_route_topk(P, P, None, 16, 128, 8, 2, 3, P, P, P, P, P, P, 1 << 20, None) == INVALID
    assert L.moe_route_topk(P, None, None, 16, 128, 8, 2, 1, P, P, P, P, P, P, 1 << 20, None) == INVALID
    assert L.moe_route_topk(P + 2, P, None, 16, 128, 8, 2, 1, P, P, P, P, P, P, 1 << 20, None) == ALIGN
    assert L.moe_route_topk(P, P, None, 4096, 128, 8, 2, 1, P, P, P, P, P, P, 64, None) == WS
    assert "workspace" in _err(L)


def test_grouped_gemm_rejects_bad_shapes(L):
    P = FAKE
    assert L.moe_grouped_gemm_swiglu(P, P, P, 8, P, None, 64, 100, 64, 8, P, None, None, 0, None) == SHAPE
    assert L.moe_grouped_gemm_swiglu(P, P, P, 2000, P, None, 64, 128, 64, 8, P, None, None, 0, None) == SHAPE
    assert L.moe_grouped_gemm_swiglu(P, P, P, 8, None, None, 64, 128, 64, 8, P, None, None, 0, None) == INVALID
    assert L.moe_grouped_gemm_down(P, P + 8, 8, P, None, 64, 128, 64, 8, P, None, 0, None) == ALIGN
    assert L.moe_grouped_gemm_down_bwd(P, P, None, P, 8, P, None, 64, 128, 64, 8, P, P, 0, None, 0,
                                       None) == INVALID
    assert L.moe_grouped_gemm_swiglu_bwd(P, P, P, P, 8, P, None, 64, 128, 96, 8, P, P, P, 0, None, 0,
                                         None) == SHAPE
    # the gathering gate/up GEMM: needs x and token ids when there is work
    assert L.moe_grouped_gemm_swiglu_gather(None, None, 16, P, P, 8, P, None, 64, 128, 64, 8, P, None,
                                            None) == INVALID
    assert L.moe_grouped_gemm_swiglu_gather(P, P, 16, P, P, 8, P, None, 64, 100, 64, 8, P, None, None) == SHAPE
    assert L.moe_grouped_gemm_swiglu_gather(P + 8, P, 16, P, P, 8, P, None, 64, 128, 64, 8, P, None,
                                            None) == ALIGN
    # the backward GEMMs' dX and weight-gradient halves check like the combined calls
    assert L.moe_grouped_gemm_down_bwd_dx(P, None, P, 8, P, None, 64, 128, 64, 8, P, None) == INVALID
    assert L.moe_grouped_gemm_down_bwd_dw(P, P, 8, P, None, 64, 128, 64, 8, P, 0, None, 0, None) == WS
    assert L.moe_grouped_gemm_swiglu_bwd_dx(P, P, P, 8, P, None, 64, 100, 64, 8, P, None) == SHAPE
    assert L.moe_grouped_gemm_swiglu_bwd_dw(P, P + 8, 8, P, None, 64, 128, 64, 8, P, P, 0, P, 1 << 20,
                                            None) == ALIGN
    # the backward GEMMs need 256 bytes of 128-byte aligned workspace per segment
    assert L.moe_grouped_gemm_bwd_workspace_size(8) == 8 * 256
    assert L.moe_grouped_gemm_bwd_workspace_size(0) == 0
    assert L.moe_grouped_gemm_down_bwd(P, P, P, P, 8, P, None, 64, 128, 64, 8, P, P, 0, None, 0,
                                       None) == WS
    assert "workspace" in _err(L)
    assert L.moe_grouped_gemm_swiglu_bwd(P, P, P, P, 8, P, None, 64, 128, 64, 8, P, P, P, 0, P, 2047,
                                         None) == WS
    assert L.moe_grouped_gemm_down_bwd(P, P, P, P, 8, P, None, 64, 128, 64, 8, P, P, 0, P + 64, 4096,
                                       None) == ALIGN


def test_fused_combine_rejects_bad_args(L):
    # moe_grouped_gemm_down_combine(h, Wd, num_seg, seg_offsets, seg_expert, R, H, I, E,
    #                               token_of_row, row_of_slot, topk_w, T, k, y_acc, y, stream)
    P = FAKE
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 64, 100, 64, 8, P, P, P, 32, 2, P, P, None) == SHAPE
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 64, 128, 64, 8, P, P, P, 32, 0, P, P, None) == INVALID
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 64, 128, 64, 8, P, P, P, 32, 33, P, P, None) == INVALID
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 64, 128, 64, 8, None, P, P, 32, 2, P, P,
                                           None) == INVALID
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 64, 128, 64, 8, P, P, P, 32, 2, None, P,
                                           None) == INVALID
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 64, 128, 64, 8, P, P, P, 32, 2, P + 8, P,
                                           None) == ALIGN
    assert "moe_grouped_gemm_down_combine" in _err(L)
    # no tokens: nothing to write, no launch
    assert L.moe_grouped_gemm_down_combine(P, P, 8, P, None, 0, 128, 64, 8, P, P, P, 0, 2, None, None,
                                           None) == OK


def test_rows_ops_reject_bad_args(L):
    P = FAKE
    assert L.moe_combine(P, P, P, 16, 128, 33, P, None) == SHAPE
    assert L.moe_combine(P, P, P, 16, 128, 2, None, None) == INVALID
    assert L.moe_dispatch(P, P, P, 16, 128, 8, 2, P, P, P, P, 0, None) == WS
    assert L.moe_dispatch_bwd(P + 4, P, 16, 128, 2, P, None) == ALIGN
    assert L.moe_combine_bwd(P, P, P, P, -1, 128, 2, P, P, None) == INVALID
    assert L.moe_route_topk_bwd(P, P, P, P, P, P, 16, 128, 8, 2, P, P, 0, P, 16, None) == WS


def test_zero_tokens_is_a_no_op(L):
    # T == 0: nothing to do, no launch, OK
    P = FAKE
    assert L.moe_combine(P, P, P, 0, 128, 2, P, None) == OK
    assert L.moe_dispatch_bwd(P, P, 0, 128, 2, P, None) == OK
    assert L.moe_grouped_gemm_swiglu(P, P, P, 8, P, None, 0, 128, 64, 8, P, None, None, 0, None) == OK
    assert L.moe_grouped_gemm_down(P, P, 0, None, None, 64, 128, 64, 8, P, None, 0, None) == OK


def test_fp8_entry_points_reject_bad_args(L):
    P = FAKE
    # per-row quantiser: cols must be a positive multiple of 8; no rows is a no-op
    assert L.moe_quantize_rows_e4m3(P, 16, 12, P, P, None) == INVALID
    assert L.moe_quantize_rows_e4m3(P, 0, 16, P, P, None) == OK
    assert L.moe_quantize_rows_e4m3(P, 16, 16, None, P, None) == INVALID
    assert L.moe_quantize_rows_e4m3(P + 8, 16, 16, P, P, None) == ALIGN
    assert L.moe_quantize_rows_e4m3(P, 16, 16, P + 4, P, None) == ALIGN
    # e4m3 GEMMs: H and I multiples of 128
    assert L.moe_grouped_gemm_swiglu_fp8(P, P, None, 0, P, P, P, P, 8, P, None, 64, 128, 64, 8, P, None) == SHAPE
    assert "128" in _err(L)
    assert L.moe_grouped_gemm_down_fp8(P, P, P, P, 8, P, None, 64, 192, 128, 8, P, None) == SHAPE
    assert L.moe_grouped_gemm_swiglu_fp8(P, None, None, 0, P, P, P, P, 8, P, None, 64, 128, 128, 8, P,
                                         None) == INVALID
    assert L.moe_grouped_gemm_swiglu_fp8(P, P, P, 0, P, P, P, P, 8, P, None, 64, 128, 128, 8, P,
                                         None) == INVALID  # gathering needs T > 0
    assert L.moe_grouped_gemm_down_fp8(P, P, P, P + 4, 8, P, None, 64, 128, 128, 8, P, None) == ALIGN
    # no rows: nothing to do
    assert L.moe_grouped_gemm_swiglu_fp8(P, P, None, 0, P, P, P, P, 8, P, None, 0, 128, 128, 8, P, None) == OK
    assert L.moe_grouped_gemm_down_fp8(P, P, P, P, 8, P, None, 0, 128, 128, 8, P, None) == OK


def test_gemm_sm_limit_is_host_state(L):
    """The GEMM grid limit is a per-thread host setting: set, read back as
    the previous value, and rejected when negative (no device needed)."""
    prev = ctypes.c_int(-1)
    assert L.moe_set_gemm_sm_limit(5, ctypes.byref(prev)) == OK and prev.value == 0
    assert L.moe_set_gemm_sm_limit(0, ctypes.byref(prev)) == OK and prev.value == 5
    assert L.moe_set_gemm_sm_limit(-1, None) == INVALID
    assert m.moe_set_gemm_sm_limit(0) == 0


def test_fma_probe_rejects_bad_arguments(L):
    n = ctypes.c_longlong(0)
    assert L.moe_probe_fma(0, 0, 16, FAKE, ctypes.byref(n), None) == INVALID     # per_sm < 1
    assert L.moe_probe_fma(1, 4, 0, FAKE, ctypes.byref(n), None) == INVALID     # iters < 1
    assert L.moe_probe_fma(0, 4, 16, None, ctypes.byref(n), None) == INVALID    # no out
