"""CPU oracle for the MoE expert layer -- TEST INFRASTRUCTURE ONLY.

Loads the single-threaded fp32 C oracle (moe_oracle.c) with ctypes and wraps
each entry point with numpy arrays.  Only the test suite, the smoke check and
the benchmark's CPU-baseline / reference leg may import this package; the
product path never does.

`build()` compiles moe_oracle.c with gcc into liboracle.so next to it (plain
-O2, no fast-math, no floating-point contraction, so that only the explicit
fmaf calls of the router are fused).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_DIR = Path(__file__).resolve().parent
_SRC = _DIR / "moe_oracle.c"
_LIB = _DIR / "liboracle.so"

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

def build(force: bool = False, src_dir: Path | None = None, out: Path | None = None) -> Path:
    """Compile the oracle (or a copy of its sources in `src_dir`) into a shared library."""
    src_dir = _DIR if src_dir is None else Path(src_dir)
    out = (_LIB if src_dir == _DIR else src_dir / "liboracle.so") if out is None else Path(out)
    srcs = [src_dir / "moe_oracle.c", src_dir / "moe_oracle.h"]
    if not force and out.exists() and all(out.stat().st_mtime >= s.stat().st_mtime for s in srcs):
        return out
    tmp = out.with_suffix(f".so.{os.getpid()}")
    subprocess.run(["gcc", *GCC_FLAGS, "-o", str(tmp), str(srcs[0]), "-lm"], check=True)
    os.replace(tmp, out)
    return out


class _Ptr:
    """ctypes argtype accepting a numpy array of the right dtype or None."""

    def __init__(self, dtype):
        self.dtype = np.dtype(dtype)

    def from_param(self, a):
        if a is None:
            return ctypes.c_void_p(0)
        if not isinstance(a, np.ndarray) or a.dtype != self.dtype or not a.flags.c_contiguous:
            raise TypeError(f"expected C-contiguous {self.dtype} array, got "
                            f"{type(a).__name__} {getattr(a, 'dtype', '')}")
        return ctypes.c_void_p(a.ctypes.data)


U8, U16, I32, F32 = _Ptr(np.uint8), _Ptr(np.uint16), _Ptr(np.int32), _Ptr(np.float32)
C_INT = ctypes.c_int

_SIGS = {
    "oracle_route_topk": [U16, F32, F32, C_INT, C_INT, C_INT, C_INT, C_INT, I32, F32, I32, I32, I32],
    "oracle_router_logits": [U16, F32, F32, C_INT, C_INT, C_INT, F32],
    "oracle_dispatch": [U16, I32, I32, C_INT, C_INT, C_INT, C_INT, U16, I32, I32],
    "oracle_grouped_gemm_swiglu": [F32, U16, U16, C_INT, I32, I32, C_INT, C_INT, C_INT, C_INT, F32, F32],
    "oracle_grouped_gemm_down": [F32, U16, C_INT, I32, I32, C_INT, C_INT, C_INT, C_INT, F32],
    "oracle_combine": [F32, F32, I32, C_INT, C_INT, C_INT, F32],
    "oracle_combine_bwd": [F32, F32, F32, I32, C_INT, C_INT, C_INT, F32, F32],
    "oracle_grouped_gemm_down_bwd": [F32, F32, F32, U16, C_INT, I32, I32, C_INT, C_INT, C_INT, C_INT,
                                     F32, F32, C_INT],
    "oracle_grouped_gemm_swiglu_bwd": [F32, F32, U16, U16, C_INT, I32, I32, C_INT, C_INT, C_INT, C_INT,
                                       F32, F32, F32, C_INT],
    "oracle_dispatch_bwd": [F32, I32, C_INT, C_INT, C_INT, F32],
    "oracle_route_topk_bwd": [F32, F32, I32, U16, F32, F32, C_INT, C_INT, C_INT, C_INT, F32, F32, C_INT],
    "oracle_e4m3_decode": [U8, C_INT, F32],
    "oracle_e4m3_encode": [F32, C_INT, U8],
    "oracle_quantize_rows_e4m3": [F32, C_INT, C_INT, U8, F32],
    "oracle_grouped_gemm_swiglu_fp8": [U8, F32, U8, F32, U8, F32, C_INT, I32, I32, C_INT, C_INT, C_INT,
                                       C_INT, F32],
    "oracle_grouped_gemm_down_fp8": [U8, F32, U8, F32, C_INT, I32, I32, C_INT, C_INT, C_INT, C_INT, F32],
}

def load(path) -> ctypes.CDLL:
    """Load an oracle shared library and declare its signatures."""
    L = ctypes.CDLL(str(path))
    for name, args in _SIGS.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    return L


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def use(L):
    """Point the wrappers below at another oracle build (used by mutation tests)."""
    global _lib
    prev, _lib = _lib, L
    return prev


def _ok(rc: int, name: str):
    if rc != 0:
        raise RuntimeError(f"{name} returned {rc}")


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> fp32 widening of uint16 bit patterns."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- wrappers


def route_topk(x, Wr, bias, k, ep_size=1):
    x = _c(x, np.uint16); Wr = _c(Wr, np.float32); bias = _c(bias, np.float32)
    T, H = x.shape
    E = Wr.shape[1]
    idx = np.empty((T, k), np.int32); w = np.empty((T, k), np.float32)
    counts = np.empty(E, np.int32); offsets = np.empty(E + 1, np.int32)
    rank_offsets = np.empty(ep_size + 1, np.int32)
    _ok(lib().oracle_route_topk(x, Wr, bias, T, H, E, k, ep_size, idx, w, counts, offsets,
                                rank_offsets), "oracle_route_topk")
    return dict(topk_idx=idx, topk_w=w, counts=counts, offsets=offsets, rank_offsets=rank_offsets)


def router_logits(x, Wr, bias=None):
    x = _c(x, np.uint16); Wr = _c(Wr, np.float32); bias = _c(bias, np.float32)
    T, H = x.shape
    E = Wr.shape[1]
    out = np.empty((T, E), np.float32)
    _ok(lib().oracle_router_logits(x, Wr, bias, T, H, E, out), "oracle_router_logits")
    return out


def dispatch(x, topk_idx, offsets, E, copy_rows=True):
    topk_idx = _c(topk_idx, np.int32); offsets = _c(offsets, np.int32)
    T, k = topk_idx.shape
    if x is not None:
        x = _c(x, np.uint16)
        H = x.shape[1]
    else:
        H = 1
    R = T * k
    x_perm = np.empty((R, H), np.uint16) if (copy_rows and x is not None) else None
    ros = np.empty((T, k), np.int32); tor = np.empty(R, np.int32)
    _ok(lib().oracle_dispatch(x if copy_rows else None, topk_idx, offsets, T, H, E, k, x_perm, ros,
                              tor), "oracle_dispatch")
    return dict(x_perm=x_perm, row_of_slot=ros, token_of_row=tor)


def _segs(num_seg, seg_offsets, seg_expert):
    return _c(seg_offsets, np.int32), _c(seg_expert, np.int32)


def grouped_gemm_swiglu(x_perm, Wg, Wu, seg_offsets, seg_expert=None, save_gu=False):
    x_perm = _c(x_perm, np.float32); Wg = _c(Wg, np.uint16); Wu = _c(Wu, np.uint16)
    so, se = _segs(None, seg_offsets, seg_expert)
    R, H = x_perm.shape
    E, I, _ = Wg.shape
    num_seg = len(so) - 1
    h = np.zeros((R, I), np.float32)
    gu = np.zeros((R, 2 * I), np.float32) if save_gu else None
    _ok(lib().oracle_grouped_gemm_swiglu(x_perm, Wg, Wu, num_seg, so, se, R, H, I, E, h, gu),
        "oracle_grouped_gemm_swiglu")
    return (h, gu) if save_gu else h


def grouped_gemm_down(h, Wd, seg_offsets, seg_expert=None):
    h = _c(h, np.float32); Wd = _c(Wd, np.uint16)
    so, se = _segs(None, seg_offsets, seg_expert)
    R, I = h.shape
    E, H, _ = Wd.shape
    y = np.zeros((R, H), np.float32)
    _ok(lib().oracle_grouped_gemm_down(h, Wd, len(so) - 1, so, se, R, H, I, E, y),
        "oracle_grouped_gemm_down")
    return y


def combine(y_perm, topk_w, row_of_slot):
    y_perm = _c(y_perm, np.float32); topk_w = _c(topk_w, np.float32)
    row_of_slot = _c(row_of_slot, np.int32)
    T, k = topk_w.shape
    H = y_perm.shape[1]
    y = np.empty((T, H), np.float32)
    _ok(lib().oracle_combine(y_perm, topk_w, row_of_slot, T, H, k, y), "oracle_combine")
    return y


def combine_bwd(dy, y_perm, topk_w, row_of_slot, R=None):
    dy = _c(dy, np.float32); y_perm = _c(y_perm, np.float32); topk_w = _c(topk_w, np.float32)
    row_of_slot = _c(row_of_slot, np.int32)
    T, k = topk_w.shape
    H = dy.shape[1]
    R = y_perm.shape[0] if R is None else R
    dy_perm = np.zeros((R, H), np.float32); d_w = np.empty((T, k), np.float32)
    _ok(lib().oracle_combine_bwd(dy, y_perm, topk_w, row_of_slot, T, H, k, dy_perm, d_w),
        "oracle_combine_bwd")
    return dy_perm, d_w


def grouped_gemm_down_bwd(dy_perm, h, gu, Wd, seg_offsets, seg_expert=None, dWd=None):
    dy_perm = _c(dy_perm, np.float32); h = _c(h, np.float32); gu = _c(gu, np.float32)
    Wd = _c(Wd, np.uint16)
    so, se = _segs(None, seg_offsets, seg_expert)
    R, H = dy_perm.shape
    E, _, I = Wd.shape
    dgu = np.zeros((R, 2 * I), np.float32)
    acc = dWd is not None
    out = np.ascontiguousarray(dWd, np.float32).copy() if acc else np.empty((E, H, I), np.float32)
    _ok(lib().oracle_grouped_gemm_down_bwd(dy_perm, h, gu, Wd, len(so) - 1, so, se, R, H, I, E, dgu,
                                           out, int(acc)), "oracle_grouped_gemm_down_bwd")
    return dgu, out


def grouped_gemm_swiglu_bwd(dgu, x_perm, Wg, Wu, seg_offsets, seg_expert=None, dWg=None, dWu=None):
    dgu = _c(dgu, np.float32); x_perm = _c(x_perm, np.float32)
    Wg = _c(Wg, np.uint16); Wu = _c(Wu, np.uint16)
    so, se = _segs(None, seg_offsets, seg_expert)
    R, H = x_perm.shape
    E, I, _ = Wg.shape
    dx_perm = np.zeros((R, H), np.float32)
    acc = dWg is not None
    og = np.ascontiguousarray(dWg, np.float32).copy() if acc else np.empty((E, I, H), np.float32)
    ou = np.ascontiguousarray(dWu, np.float32).copy() if acc else np.empty((E, I, H), np.float32)
    _ok(lib().oracle_grouped_gemm_swiglu_bwd(dgu, x_perm, Wg, Wu, len(so) - 1, so, se, R, H, I, E,
                                             dx_perm, og, ou, int(acc)),
        "oracle_grouped_gemm_swiglu_bwd")
    return dx_perm, og, ou


def dispatch_bwd(dx_perm, row_of_slot):
    dx_perm = _c(dx_perm, np.float32); row_of_slot = _c(row_of_slot, np.int32)
    T, k = row_of_slot.shape
    H = dx_perm.shape[1]
    out = np.empty((T, H), np.float32)
    _ok(lib().oracle_dispatch_bwd(dx_perm, row_of_slot, T, H, k, out), "oracle_dispatch_bwd")
    return out


def route_topk_bwd(d_w, topk_w, topk_idx, x, Wr, dx_acc, dWr=None):
    d_w = _c(d_w, np.float32); topk_w = _c(topk_w, np.float32); topk_idx = _c(topk_idx, np.int32)
    x = _c(x, np.uint16); Wr = _c(Wr, np.float32); dx_acc = _c(dx_acc, np.float32)
    T, k = topk_idx.shape
    H, E = Wr.shape
    acc = dWr is not None
    out = np.ascontiguousarray(dWr, np.float32).copy() if acc else np.empty((H, E), np.float32)
    dx = np.empty((T, H), np.float32)
    _ok(lib().oracle_route_topk_bwd(d_w, topk_w, topk_idx, x, Wr, dx_acc, T, H, E, k, out, dx,
                                    int(acc)), "oracle_route_topk_bwd")
    return out, dx


# ------------------------------------------------------------ FP8 (e4m3)


def e4m3_decode(q):
    q = _c(q, np.uint8)
    out = np.empty(q.shape, np.float32)
    _ok(lib().oracle_e4m3_decode(q.reshape(-1), q.size, out.reshape(-1)), "oracle_e4m3_decode")
    return out


def e4m3_encode(v):
    v = _c(v, np.float32)
    q = np.empty(v.shape, np.uint8)
    _ok(lib().oracle_e4m3_encode(v.reshape(-1), v.size, q.reshape(-1)), "oracle_e4m3_encode")
    return q


def quantize_rows_e4m3(a):
    """Per-row e4m3 codes and fp32 scales of a 2-D fp32 array (or [..., cols])."""
    a = _c(a, np.float32)
    cols = a.shape[-1]
    rows = a.size // cols
    q = np.empty(a.shape, np.uint8)
    s = np.empty(a.shape[:-1], np.float32)
    _ok(lib().oracle_quantize_rows_e4m3(a.reshape(rows, cols), rows, cols, q.reshape(rows, cols),
                                        s.reshape(rows)), "oracle_quantize_rows_e4m3")
    return q, s


def grouped_gemm_swiglu_fp8(aq, a_scale, Wgq, Wg_scale, Wuq, Wu_scale, seg_offsets, seg_expert=None):
    aq = _c(aq, np.uint8); a_scale = _c(a_scale, np.float32)
    Wgq = _c(Wgq, np.uint8); Wuq = _c(Wuq, np.uint8)
    Wg_scale = _c(Wg_scale, np.float32); Wu_scale = _c(Wu_scale, np.float32)
    so, se = _segs(None, seg_offsets, seg_expert)
    R, H = aq.shape
    E, I, _ = Wgq.shape
    h = np.zeros((R, I), np.float32)
    _ok(lib().oracle_grouped_gemm_swiglu_fp8(aq, a_scale, Wgq, Wg_scale, Wuq, Wu_scale, len(so) - 1, so,
                                             se, R, H, I, E, h), "oracle_grouped_gemm_swiglu_fp8")
    return h


def grouped_gemm_down_fp8(hq, h_scale, Wdq, Wd_scale, seg_offsets, seg_expert=None):
    hq = _c(hq, np.uint8); h_scale = _c(h_scale, np.float32)
    Wdq = _c(Wdq, np.uint8); Wd_scale = _c(Wd_scale, np.float32)
    so, se = _segs(None, seg_offsets, seg_expert)
    R, I = hq.shape
    E, H, _ = Wdq.shape
    y = np.zeros((R, H), np.float32)
    _ok(lib().oracle_grouped_gemm_down_fp8(hq, h_scale, Wdq, Wd_scale, len(so) - 1, so, se, R, H, I, E,
                                           y), "oracle_grouped_gemm_down_fp8")
    return y
