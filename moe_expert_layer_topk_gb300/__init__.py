"""GB300 (sm_103a) MoE expert layer: router top-k -> dispatch -> grouped
gate/up GEMM + SwiGLU -> grouped down GEMM -> weighted combine, forward and
backward, as a C-ABI CUDA library (include/moe_topk.h).

This module is the thin Python binding: it loads libmoe_topk.so and exposes
every C entry point under the same name, taking torch tensors (device
memory) and passing their pointers, sizes and the current CUDA stream.  All
arithmetic runs in the library's kernels; nothing here computes the layer,
and there is no fallback -- calls fail loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from . import build as _build_mod

__all__ = ["lib", "MoEError", "LIB_PATH", "ENTRY_POINTS",
           "moe_route_topk", "moe_route_topk_chunks", "moe_route_topk_chunks_workspace_size",
           "moe_dispatch", "moe_dispatch_chunked", "moe_dispatch_e4m3_chunked", "moe_dispatch_no_alloc",
           "moe_grouped_gemm_swiglu",
           "moe_grouped_gemm_swiglu_gather", "moe_grouped_gemm_down", "moe_grouped_gemm_down_combine",
           "moe_quantize_rows_e4m3", "moe_dispatch_e4m3", "moe_grouped_gemm_swiglu_fp8",
           "moe_grouped_gemm_down_fp8",
           "moe_combine", "moe_combine_bwd", "moe_grouped_gemm_down_bwd",
           "moe_grouped_gemm_swiglu_bwd", "moe_grouped_gemm_down_bwd_dx", "moe_grouped_gemm_down_bwd_dw",
           "moe_grouped_gemm_swiglu_bwd_dx", "moe_grouped_gemm_swiglu_bwd_dw",
           "moe_dispatch_bwd", "moe_route_topk_bwd",
           "moe_route_topk_workspace_size", "moe_dispatch_workspace_size",
           "moe_route_topk_bwd_workspace_size", "moe_grouped_gemm_bwd_workspace_size",
           "moe_read_device_status", "moe_abi_version", "moe_probe_fma", "moe_set_gemm_sm_limit", "sm_count"]

LIB_PATH: Path = _build_mod.LIB

_P, _I, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

# name -> (argtypes, restype); mirrors include/moe_topk.h
# the ABI version of include/moe_topk.h these signatures follow
ABI_VERSION = 103

ENTRY_POINTS = {
    "moe_abi_version": ([], _I),
    "moe_last_error_string": ([], ctypes.c_char_p),
    "moe_read_device_status": ([_P, _I, _P], _I),
    "moe_route_topk_workspace_size": ([_I, _I, _I], _Z),
    "moe_route_topk": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_route_topk_chunks_workspace_size": ([_I, _I, _I], _Z),
    "moe_route_topk_chunks": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_dispatch_workspace_size": ([_I, _I, _I], _Z),
    "moe_dispatch_chunked": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_dispatch_e4m3_chunked": ([_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_dispatch": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P], _I),
    "moe_dispatch_no_alloc_max_scratch": ([], _Z),
    "moe_dispatch_no_alloc": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_swiglu": ([_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _Z, _P], _I),
    "moe_grouped_gemm_swiglu_gather": ([_P, _P, _I, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_down": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _Z, _P], _I),
    "moe_grouped_gemm_down_combine": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _I, _P, _P, _P], _I),
    "moe_quantize_rows_e4m3": ([_P, _I, _I, _P, _P, _P], _I),
    "moe_dispatch_e4m3": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_grouped_gemm_swiglu_fp8": ([_P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_grouped_gemm_down_fp8": ([_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_combine": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_combine_bwd": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_bwd_workspace_size": ([_I], _Z),
    "moe_grouped_gemm_down_bwd": ([_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _Z, _P], _I),
    "moe_grouped_gemm_swiglu_bwd": ([_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _Z, _P],
                                    _I),
    "moe_grouped_gemm_down_bwd_dx": ([_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_grouped_gemm_down_bwd_dw": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _I, _P, _Z, _P], _I),
    "moe_grouped_gemm_swiglu_bwd_dx": ([_P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "moe_grouped_gemm_swiglu_bwd_dw": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _Z, _P], _I),
    "moe_dispatch_bwd": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "moe_route_topk_bwd_workspace_size": ([_I, _I, _I], _Z),
    "moe_route_topk_bwd": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _Z, _P], _I),
    "moe_probe_fma": ([_I, _I, _I, _P, ctypes.POINTER(ctypes.c_longlong), _P], _I),
    "moe_set_gemm_sm_limit": ([_I, ctypes.POINTER(ctypes.c_int)], _I),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, name: str, code: int, msg: str):
        super().__init__(f"{name} failed with code {code}: {msg}")
        self.code = code


def lib(path: Path | str | None = None) -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built."""
    global _lib
    if _lib is None or path is not None:
        p = Path(path) if path is not None else LIB_PATH
        if not p.exists():
            raise RuntimeError(f"CUDA library {p} is not built: run "
                               f"`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(str(p))
        for name, (args, res) in ENTRY_POINTS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        if L.moe_abi_version() != ABI_VERSION:
            raise RuntimeError(f"CUDA library {p} has ABI version {L.moe_abi_version()}, this binding "
                               f"expects {ABI_VERSION}: rebuild it")
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor arguments must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return t.data_ptr()


# the raw handle of the current stream without building a Stream object
# (torch.cuda.current_stream() costs about 3 us a call, a third of a small
# kernel call's host time)
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise MoEError(name, rc, lib().moe_last_error_string().decode(errors="replace"))


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


# ------------------------------------------------- entry points (same names)

def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_route_topk_workspace_size(T, H, E) -> int:
    return lib().moe_route_topk_workspace_size(T, H, E)


def moe_route_topk_chunks_workspace_size(T, H, E) -> int:
    return lib().moe_route_topk_chunks_workspace_size(T, H, E)


def moe_dispatch_workspace_size(T, E, k) -> int:
    return lib().moe_dispatch_workspace_size(T, E, k)


def moe_route_topk_bwd_workspace_size(T, H, E) -> int:
    return lib().moe_route_topk_bwd_workspace_size(T, H, E)


def moe_grouped_gemm_bwd_workspace_size(num_seg) -> int:
    return lib().moe_grouped_gemm_bwd_workspace_size(num_seg)


def moe_read_device_status(reset: bool = True, stream=None) -> int:
    v = ctypes.c_int(0)
    _call("moe_read_device_status", ctypes.addressof(v), int(reset), _stream(stream))
    return v.value


def moe_route_topk(x, Wr, bias, T, H, E, k, ep_size, topk_idx, topk_w, counts, offsets,
                   rank_offsets, ws, stream=None):
    _call("moe_route_topk", _ptr(x), _ptr(Wr), _ptr(bias), T, H, E, k, ep_size, _ptr(topk_idx),
          _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(rank_offsets), _ptr(ws), _nbytes(ws),
          _stream(stream))


def moe_route_topk_chunks(x, Wr, bias, T, H, E, k, ep_size, topk_idx, topk_w, counts, offsets,
                          rank_offsets, chunk_prefix, ws, stream=None):
    _call("moe_route_topk_chunks", _ptr(x), _ptr(Wr), _ptr(bias), T, H, E, k, ep_size, _ptr(topk_idx),
          _ptr(topk_w), _ptr(counts), _ptr(offsets), _ptr(rank_offsets), _ptr(chunk_prefix), _ptr(ws),
          _nbytes(ws), _stream(stream))


def moe_dispatch_chunked(x, topk_idx, offsets, chunk_prefix, T, H, E, k, x_perm, row_of_slot, token_of_row,
                         stream=None):
    _call("moe_dispatch_chunked", _ptr(x), _ptr(topk_idx), _ptr(offsets), _ptr(chunk_prefix), T, H, E, k,
          _ptr(x_perm), _ptr(row_of_slot), _ptr(token_of_row), _stream(stream))


def moe_dispatch_e4m3_chunked(x, topk_idx, offsets, chunk_prefix, T, H, E, k, xq_perm, xs_perm, row_of_slot,
                              token_of_row, stream=None):
    _call("moe_dispatch_e4m3_chunked", _ptr(x), _ptr(topk_idx), _ptr(offsets), _ptr(chunk_prefix), T, H, E, k,
          _ptr(xq_perm), _ptr(xs_perm), _ptr(row_of_slot), _ptr(token_of_row), _stream(stream))


def moe_dispatch(x, topk_idx, offsets, T, H, E, k, x_perm, row_of_slot, token_of_row, ws,
                 stream=None):
    _call("moe_dispatch", _ptr(x), _ptr(topk_idx), _ptr(offsets), T, H, E, k, _ptr(x_perm),
          _ptr(row_of_slot), _ptr(token_of_row), _ptr(ws), _nbytes(ws), _stream(stream))


def moe_dispatch_no_alloc(x, topk_idx, offsets, T, H, E, k, x_perm, row_of_slot, token_of_row,
                          stream=None):
    """moe_dispatch with the library's built-in scratch instead of a workspace."""
    _call("moe_dispatch_no_alloc", _ptr(x), _ptr(topk_idx), _ptr(offsets), T, H, E, k, _ptr(x_perm),
          _ptr(row_of_slot), _ptr(token_of_row), _stream(stream))


def moe_grouped_gemm_swiglu(x_perm, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E, h,
                            gu_save=None, ws=None, stream=None):
    _call("moe_grouped_gemm_swiglu", _ptr(x_perm), _ptr(Wg), _ptr(Wu), num_seg, _ptr(seg_offsets),
          _ptr(seg_expert), R, H, I, E, _ptr(h), _ptr(gu_save), _ptr(ws), _nbytes(ws),
          _stream(stream))


def moe_grouped_gemm_swiglu_gather(x, token_of_row, T, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H,
                                   I, E, h, gu_save=None, stream=None):
    _call("moe_grouped_gemm_swiglu_gather", _ptr(x), _ptr(token_of_row), T, _ptr(Wg), _ptr(Wu), num_seg,
          _ptr(seg_offsets), _ptr(seg_expert), R, H, I, E, _ptr(h), _ptr(gu_save), _stream(stream))


def moe_grouped_gemm_down(h, Wd, num_seg, seg_offsets, seg_expert, R, H, I, E, y_perm, ws=None,
                          stream=None):
    _call("moe_grouped_gemm_down", _ptr(h), _ptr(Wd), num_seg, _ptr(seg_offsets),
          _ptr(seg_expert), R, H, I, E, _ptr(y_perm), _ptr(ws), _nbytes(ws), _stream(stream))


def moe_grouped_gemm_down_combine(h, Wd, num_seg, seg_offsets, seg_expert, R, H, I, E, token_of_row,
                                  row_of_slot, topk_w, T, k, y_acc, y, stream=None):
    _call("moe_grouped_gemm_down_combine", _ptr(h), _ptr(Wd), num_seg, _ptr(seg_offsets),
          _ptr(seg_expert), R, H, I, E, _ptr(token_of_row), _ptr(row_of_slot), _ptr(topk_w), T, k,
          _ptr(y_acc), _ptr(y), _stream(stream))


def moe_quantize_rows_e4m3(a, rows, cols, q, scale, stream=None):
    _call("moe_quantize_rows_e4m3", _ptr(a), rows, cols, _ptr(q), _ptr(scale), _stream(stream))


def moe_dispatch_e4m3(x, topk_idx, offsets, T, H, E, k, xq_perm, xs_perm, row_of_slot, token_of_row, ws,
                      stream=None):
    _call("moe_dispatch_e4m3", _ptr(x), _ptr(topk_idx), _ptr(offsets), T, H, E, k, _ptr(xq_perm), _ptr(xs_perm),
          _ptr(row_of_slot), _ptr(token_of_row), _ptr(ws), _nbytes(ws), _stream(stream))


def moe_grouped_gemm_swiglu_fp8(a, a_scale, token_of_row, T, Wg, Wg_scale, Wu, Wu_scale, num_seg,
                                seg_offsets, seg_expert, R, H, I, E, h, stream=None):
    _call("moe_grouped_gemm_swiglu_fp8", _ptr(a), _ptr(a_scale), _ptr(token_of_row), T, _ptr(Wg),
          _ptr(Wg_scale), _ptr(Wu), _ptr(Wu_scale), num_seg, _ptr(seg_offsets), _ptr(seg_expert), R, H,
          I, E, _ptr(h), _stream(stream))


def moe_grouped_gemm_down_fp8(h, h_scale, Wd, Wd_scale, num_seg, seg_offsets, seg_expert, R, H, I, E,
                              y_perm, stream=None):
    _call("moe_grouped_gemm_down_fp8", _ptr(h), _ptr(h_scale), _ptr(Wd), _ptr(Wd_scale), num_seg,
          _ptr(seg_offsets), _ptr(seg_expert), R, H, I, E, _ptr(y_perm), _stream(stream))


def moe_combine(y_perm, topk_w, row_of_slot, T, H, k, y, stream=None):
    _call("moe_combine", _ptr(y_perm), _ptr(topk_w), _ptr(row_of_slot), T, H, k, _ptr(y),
          _stream(stream))


def moe_combine_bwd(dy, y_perm, topk_w, row_of_slot, T, H, k, dy_perm, d_w, stream=None):
    _call("moe_combine_bwd", _ptr(dy), _ptr(y_perm), _ptr(topk_w), _ptr(row_of_slot), T, H, k,
          _ptr(dy_perm), _ptr(d_w), _stream(stream))


def moe_grouped_gemm_down_bwd(dy_perm, h, gu_save, Wd, num_seg, seg_offsets, seg_expert, R, H, I,
                              E, dgu, dWd, accumulate=0, ws=None, stream=None):
    _call("moe_grouped_gemm_down_bwd", _ptr(dy_perm), _ptr(h), _ptr(gu_save), _ptr(Wd), num_seg,
          _ptr(seg_offsets), _ptr(seg_expert), R, H, I, E, _ptr(dgu), _ptr(dWd), int(accumulate),
          _ptr(ws), _nbytes(ws), _stream(stream))


def moe_grouped_gemm_swiglu_bwd(dgu, x_perm, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E,
                                dx_perm, dWg, dWu, accumulate=0, ws=None, stream=None):
    _call("moe_grouped_gemm_swiglu_bwd", _ptr(dgu), _ptr(x_perm), _ptr(Wg), _ptr(Wu), num_seg,
          _ptr(seg_offsets), _ptr(seg_expert), R, H, I, E, _ptr(dx_perm), _ptr(dWg), _ptr(dWu),
          int(accumulate), _ptr(ws), _nbytes(ws), _stream(stream))


def moe_grouped_gemm_down_bwd_dx(dy_perm, gu_save, Wd, num_seg, seg_offsets, seg_expert, R, H, I, E, dgu,
                                 stream=None):
    _call("moe_grouped_gemm_down_bwd_dx", _ptr(dy_perm), _ptr(gu_save), _ptr(Wd), num_seg, _ptr(seg_offsets),
          _ptr(seg_expert), R, H, I, E, _ptr(dgu), _stream(stream))


def moe_grouped_gemm_down_bwd_dw(dy_perm, h, num_seg, seg_offsets, seg_expert, R, H, I, E, dWd, accumulate=0,
                                 ws=None, stream=None):
    _call("moe_grouped_gemm_down_bwd_dw", _ptr(dy_perm), _ptr(h), num_seg, _ptr(seg_offsets), _ptr(seg_expert),
          R, H, I, E, _ptr(dWd), int(accumulate), _ptr(ws), _nbytes(ws), _stream(stream))


def moe_grouped_gemm_swiglu_bwd_dx(dgu, Wg, Wu, num_seg, seg_offsets, seg_expert, R, H, I, E, dx_perm,
                                   stream=None):
    _call("moe_grouped_gemm_swiglu_bwd_dx", _ptr(dgu), _ptr(Wg), _ptr(Wu), num_seg, _ptr(seg_offsets),
          _ptr(seg_expert), R, H, I, E, _ptr(dx_perm), _stream(stream))


def moe_grouped_gemm_swiglu_bwd_dw(dgu, x_perm, num_seg, seg_offsets, seg_expert, R, H, I, E, dWg, dWu,
                                   accumulate=0, ws=None, stream=None):
    _call("moe_grouped_gemm_swiglu_bwd_dw", _ptr(dgu), _ptr(x_perm), num_seg, _ptr(seg_offsets),
          _ptr(seg_expert), R, H, I, E, _ptr(dWg), _ptr(dWu), int(accumulate), _ptr(ws), _nbytes(ws),
          _stream(stream))


def moe_dispatch_bwd(dx_perm, row_of_slot, T, H, k, dx_acc, stream=None):
    _call("moe_dispatch_bwd", _ptr(dx_perm), _ptr(row_of_slot), T, H, k, _ptr(dx_acc),
          _stream(stream))


def moe_route_topk_bwd(d_w, topk_w, topk_idx, x, Wr, dx_acc, T, H, E, k, dWr, dx, accumulate=0,
                       ws=None, stream=None):
    _call("moe_route_topk_bwd", _ptr(d_w), _ptr(topk_w), _ptr(topk_idx), _ptr(x), _ptr(Wr),
          _ptr(dx_acc), T, H, E, k, _ptr(dWr), _ptr(dx), int(accumulate), _ptr(ws), _nbytes(ws),
          _stream(stream))


def moe_set_gemm_sm_limit(max_sms: int) -> int:
    """Limit the grouped GEMMs issued from this thread to max_sms SMs (0 = all);
    returns the previous limit."""
    prev = ctypes.c_int(0)
    _call("moe_set_gemm_sm_limit", int(max_sms), ctypes.byref(prev))
    return prev.value


def sm_count(device=None) -> int:
    return torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device()) \
        .multi_processor_count


from .layer import MoELayer  # noqa: E402  (buffers + call sequence over the entry points)

__all__.append("MoELayer")


def moe_probe_fma(packed, per_sm, iters, out, stream=None) -> int:
    """Launch the FMA-rate probe; returns the number of FMAs it performs."""
    n = ctypes.c_longlong(0)
    _call("moe_probe_fma", int(packed), int(per_sm), int(iters), _ptr(out), ctypes.byref(n), _stream(stream))
    return int(n.value)

