"""Buffers and call order of one MoE expert layer over the C entry points.

`MoELayer` owns the device tensors one layer needs for a fixed token count
(outputs, activations kept for the backward pass, gradients, workspaces),
allocated once through torch, and issues the library calls in order on one
stream.  It adds no arithmetic of its own.
"""
from __future__ import annotations

import torch

from . import (moe_combine, moe_combine_bwd, moe_dispatch_bwd, moe_dispatch_chunked,
               moe_dispatch_e4m3_chunked, moe_grouped_gemm_bwd_workspace_size,
               moe_grouped_gemm_down, moe_grouped_gemm_down_bwd, moe_grouped_gemm_down_combine,
               moe_grouped_gemm_down_fp8,
               moe_grouped_gemm_swiglu, moe_grouped_gemm_swiglu_bwd_dw, moe_grouped_gemm_swiglu_bwd_dx,
               moe_grouped_gemm_swiglu_fp8, moe_set_gemm_sm_limit, sm_count,
               moe_grouped_gemm_swiglu_gather, moe_quantize_rows_e4m3, moe_route_topk_bwd,
               moe_route_topk_bwd_workspace_size, moe_route_topk_chunks,
               moe_route_topk_chunks_workspace_size)


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device)


class MoELayer:
    """One layer's buffers for T tokens of hidden size H, E experts of size I, top-k.

    fused_dispatch (forward only): dispatch only ranks the slots and the
    gate/up GEMM reads its rows straight from x by token id, so x_perm is
    never written (moe_grouped_gemm_swiglu_gather).

    fp8 (forward only): dispatch writes the permuted rows as e4m3 codes with
    one scale per token (moe_dispatch_e4m3), h is quantised per row, and
    both GEMMs run on e4m3 weights prepared once by `quantize_weights` (one
    scale per output channel).

    fused_combine (forward only, bf16): the down GEMM adds each weighted row
    into its token's fp32 row and y is rounded from those
    (moe_grouped_gemm_down_combine), so y_perm is never written; the order
    of those fp32 additions is not fixed from run to run.  It saves the
    [T*k, H] y_perm buffer but measured slower than down + combine."""

    def __init__(self, T: int, H: int, I: int, E: int, k: int, ep_size: int = 1, *,
                 training: bool = True, fused_dispatch: bool = False, fp8: bool = False,
                 fused_combine: bool = False, device: str | torch.device = "cuda"):
        if fp8 and training:
            raise ValueError("the e4m3 path is forward only")
        if fused_combine and (training or fp8):
            raise ValueError("fused_combine is a bf16 forward-only path (the combine backward needs y_perm)")
        if fused_dispatch and training:
            raise ValueError("fused_dispatch keeps no x_perm, which the backward pass needs")
        self.T, self.H, self.I, self.E, self.k, self.ep_size = T, H, I, E, k, ep_size
        self.R = R = T * k
        self.training = training
        self.fused_dispatch = fused_dispatch
        self.fused_combine = fused_combine
        self.fp8 = fp8
        self._x = None
        self._side = None  # side stream of the backward's tail (created on first use)
        dev = torch.device(device)
        i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
        e = lambda *s, dt: torch.empty(*s, dtype=dt, device=dev)  # noqa: E731
        self.topk_idx = e(T, k, dt=i32)
        self.topk_w = e(T, k, dt=f32)
        self.counts = e(E, dt=i32)
        self.offsets = e(E + 1, dt=i32)
        self.rank_offsets = e(ep_size + 1, dt=i32)
        self.ws_route = _ws(moe_route_topk_chunks_workspace_size(T, H, E), dev)
        # where each 16-token chunk starts in each expert's rows (from the route, for the dispatch)
        self.chunk_prefix = e(E, (T + 15) // 16, dt=i32)
        self.x_perm = None if (fused_dispatch or fp8) else e(R, H, dt=bf)
        self.row_of_slot = e(T, k, dt=i32)
        self.token_of_row = e(R, dt=i32)
        self.h = e(R, I, dt=bf)
        self.gu = e(R, 2 * I, dt=bf) if training else None
        self.y_perm = None if fused_combine else e(R, H, dt=bf)
        self.y_acc = e(T, H, dt=f32) if fused_combine else None
        self.y = e(T, H, dt=bf)
        if fp8:
            u8 = torch.uint8
            self.x_q, self.x_scale = e(R, H, dt=u8), e(R, dt=f32)  # permuted rows, their tokens' scales
            self.h_q, self.h_scale = e(R, I, dt=u8), e(R, dt=f32)
        if training:
            self.dy_perm = e(R, H, dt=bf)
            self.d_w = e(T, k, dt=f32)
            self.dgu = e(R, 2 * I, dt=bf)
            self.dx_perm = e(R, H, dt=bf)
            self.dx_acc = e(T, H, dt=f32)
            self.dx = e(T, H, dt=bf)
            self.dWg = e(E, I, H, dt=f32)
            self.dWu = e(E, I, H, dt=f32)
            self.dWd = e(E, H, I, dt=f32)
            self.dWr = e(H, E, dt=f32)
            self.ws_route_bwd = _ws(moe_route_topk_bwd_workspace_size(T, H, E), dev)
            self.ws_gemm_bwd = _ws(moe_grouped_gemm_bwd_workspace_size(E), dev)

    # ---------------------------------------------------------------- forward
    def quantize_weights(self, Wg, Wu, Wd, stream=None):
        """e4m3 codes and per-output-channel scales of the expert weights."""
        E, H, I = self.E, self.H, self.I
        out = {}
        for name, W, rows, cols in (("Wg", Wg, E * I, H), ("Wu", Wu, E * I, H), ("Wd", Wd, E * H, I)):
            q = torch.empty(W.shape, dtype=torch.uint8, device=W.device)
            sc = torch.empty(rows, dtype=torch.float32, device=W.device)
            moe_quantize_rows_e4m3(W, rows, cols, q, sc, stream)
            out[name], out[name + "_scale"] = q, sc
        return out

    def route(self, x, Wr, bias=None, stream=None):
        moe_route_topk_chunks(x, Wr, bias, self.T, self.H, self.E, self.k, self.ep_size, self.topk_idx,
                              self.topk_w, self.counts, self.offsets, self.rank_offsets, self.chunk_prefix,
                              self.ws_route, stream)

    def dispatch(self, x, stream=None):
        self._x = x  # the fused gate/up GEMM reads the rows from here
        if self.fp8:
            moe_dispatch_e4m3_chunked(x, self.topk_idx, self.offsets, self.chunk_prefix, self.T, self.H, self.E,
                                      self.k, self.x_q, self.x_scale, self.row_of_slot, self.token_of_row, stream)
            return
        moe_dispatch_chunked(x, self.topk_idx, self.offsets, self.chunk_prefix, self.T, self.H, self.E, self.k,
                             self.x_perm, self.row_of_slot, self.token_of_row, stream)

    def experts(self, Wg, Wu, Wd, stream=None, y=None):
        """Wg, Wu, Wd: bf16 expert weights, or (fp8 layers) the dict that
        `quantize_weights` returns, passed as Wg (Wu and Wd unused).
        y: the output of a fused_combine layer (default: the layer's own)."""
        if self.fp8:
            w = Wg
            T, H, I, E, R = self.T, self.H, self.I, self.E, self.R
            moe_grouped_gemm_swiglu_fp8(self.x_q, self.x_scale, None, 0, w["Wg"], w["Wg_scale"], w["Wu"],
                                        w["Wu_scale"], E, self.offsets, None, R, H, I, E, self.h, stream)
            moe_quantize_rows_e4m3(self.h, R, I, self.h_q, self.h_scale, stream)
            moe_grouped_gemm_down_fp8(self.h_q, self.h_scale, w["Wd"], w["Wd_scale"], E, self.offsets,
                                      None, R, H, I, E, self.y_perm, stream)
            return
        if self.fused_dispatch:
            moe_grouped_gemm_swiglu_gather(self._x, self.token_of_row, self.T, Wg, Wu, self.E,
                                           self.offsets, None, self.R, self.H, self.I, self.E, self.h,
                                           None, stream)
        else:
            moe_grouped_gemm_swiglu(self.x_perm, Wg, Wu, self.E, self.offsets, None, self.R, self.H,
                                    self.I, self.E, self.h, self.gu, None, stream)
        if self.fused_combine:
            moe_grouped_gemm_down_combine(self.h, Wd, self.E, self.offsets, None, self.R, self.H, self.I,
                                          self.E, self.token_of_row, self.row_of_slot, self.topk_w, self.T,
                                          self.k, self.y_acc, self.y if y is None else y, stream)
            return
        moe_grouped_gemm_down(self.h, Wd, self.E, self.offsets, None, self.R, self.H, self.I,
                              self.E, self.y_perm, None, stream)

    def combine(self, stream=None, y=None):
        moe_combine(self.y_perm, self.topk_w, self.row_of_slot, self.T, self.H, self.k,
                    self.y if y is None else y, stream)

    def forward(self, x, Wr, bias, Wg, Wu, Wd, stream=None, y=None):
        """y: optional bf16 [T,H] output tensor (default: the layer's own)."""
        self.route(x, Wr, bias, stream)
        self.dispatch(x, stream)
        self.experts(Wg, Wu, Wd, stream, y)
        if not self.fused_combine:
            self.combine(stream, y)
        return self.y if y is None else y

    def capture_forward(self, x, Wr, bias, Wg, Wu, Wd) -> "torch.cuda.CUDAGraph":
        """Record forward() on these tensors as a CUDA graph and return it.

        `graph.replay()` then re-runs the whole forward (all its kernels,
        one launch from the host) on whatever the same tensors hold, into
        the layer's own y: for small batches, whose forward is bound by the
        host issuing one call per kernel.  One forward runs first, outside
        the capture, so that each call's first-use set-up (kernel
        attributes, the device status word) is done before it."""
        self.forward(x, Wr, bias, Wg, Wu, Wd)
        torch.cuda.synchronize(self.y.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self.forward(x, Wr, bias, Wg, Wu, Wd)
        return graph

    # --------------------------------------------------------------- backward
    # SMs left free for the backward's tail (dispatch and router backward, on
    # a side stream) while the gate/up weight-gradient GEMM runs: measured at
    # T=8192 on GB300, the two together took 514 us this way against 558 us
    # one after the other (525 us on two streams with no limit).
    TAIL_SMS = 16

    def backward(self, dy, x, Wr, Wg, Wu, Wd, accumulate: bool = False, stream=None, dx=None,
                 overlap: bool = True):
        """dx: optional bf16 [T,H] output tensor (default: the layer's own).

        overlap: run the dispatch and router backward on a side stream beside
        the gate/up weight gradient (which then leaves TAIL_SMS SMs free);
        the results are the same either way, and the call returns with the
        work of both streams ordered before anything later on `stream`."""
        assert self.training, "layer was built without backward buffers"
        dx = self.dx if dx is None else dx
        T, H, I, E, k, R = self.T, self.H, self.I, self.E, self.k, self.R
        moe_combine_bwd(dy, self.y_perm, self.topk_w, self.row_of_slot, T, H, k, self.dy_perm,
                        self.d_w, stream)
        moe_grouped_gemm_down_bwd(self.dy_perm, self.h, self.gu, Wd, E, self.offsets, None, R, H, I,
                                  E, self.dgu, self.dWd, accumulate, self.ws_gemm_bwd, stream)
        moe_grouped_gemm_swiglu_bwd_dx(self.dgu, Wg, Wu, E, self.offsets, None, R, H, I, E, self.dx_perm,
                                       stream)
        tail = stream
        if overlap:
            main = stream if stream is not None else torch.cuda.current_stream(self.dx_perm.device)
            if self._side is None:
                self._side = torch.cuda.Stream(self.dx_perm.device)
                self._ev_fork, self._ev_join = torch.cuda.Event(), torch.cuda.Event()
            self._ev_fork.record(main)
            self._side.wait_event(self._ev_fork)
            tail = self._side
            prev = moe_set_gemm_sm_limit(max(1, sm_count(self.dx_perm.device) - self.TAIL_SMS))
            try:
                moe_grouped_gemm_swiglu_bwd_dw(self.dgu, self.x_perm, E, self.offsets, None, R, H, I, E, self.dWg,
                                               self.dWu, accumulate, self.ws_gemm_bwd, main)
            finally:
                moe_set_gemm_sm_limit(prev)
        else:
            moe_grouped_gemm_swiglu_bwd_dw(self.dgu, self.x_perm, E, self.offsets, None, R, H, I, E, self.dWg,
                                           self.dWu, accumulate, self.ws_gemm_bwd, stream)
        moe_dispatch_bwd(self.dx_perm, self.row_of_slot, T, H, k, self.dx_acc, tail)
        moe_route_topk_bwd(self.d_w, self.topk_w, self.topk_idx, x, Wr, self.dx_acc, T, H, E, k,
                           self.dWr, dx, accumulate, self.ws_route_bwd, tail)
        if overlap:
            self._ev_join.record(self._side)
            main.wait_event(self._ev_join)
        return dx
