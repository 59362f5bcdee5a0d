"""Seeded synthetic inputs for the MoE expert layer.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic (no routing, no matmul, no activation).  Both the CUDA path
and the CPU oracle are fed from the bytes it returns, so a comparison between
them always starts from identical inputs.

Workloads (shapes from "Qwen3-MoE-30B-A3B EP+FSDP2", section on the model's
expert tensors: 128 experts, hidden 2048, expert intermediate 768; the EP
split of 128 experts over 8 ranks from the same page's 16-GPU example):

  tiny_fwd            T=256,   H=128,  I=64,  E=8,   top-2
  qwen3_30b_fwd       T=4096,  H=2048, I=768, E=128, top-8
  qwen3_30b_zipf_fwd  T=16384, same shapes, per-expert router bias giving a
                      Zipf(1.2)-like popularity with 4 experts forced empty
  ep_rank_local       32768 received rows, 16 local experts, 8 source-rank
                      blocks x 16 experts = 128 segments (no routing step)
  qwen3_30b_fwd_bwd   T=8192, same shapes, plus upstream gradient dY

Draw order (one torch CPU Generator, manual_seed(seed)):
  x, Wr, Wg, Wu, Wd, bias | segment counts, dY.
Values are fp32 N(0,1)*std, rounded to bf16 (round-to-nearest-even) where the
tensor is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["LayerShape", "CONFIGS", "make_layer_inputs", "make_segment_inputs",
           "bf16_bits", "zipf_router_bias"]


@dataclass(frozen=True)
class LayerShape:
    T: int          # tokens (for ep_rank_local: received rows R)
    H: int          # hidden size
    I: int          # expert intermediate size
    E: int          # experts (local experts for ep_rank_local)
    k: int          # experts per token
    ep_size: int = 1
    bias: str | None = None      # None | "zipf"
    backward: bool = False
    segments: bool = False       # ep_rank_local: rows arrive as (source rank x expert) blocks
    src_ranks: int = 1
    note: str = ""

    @property
    def R(self) -> int:
        return self.T if self.segments else self.T * self.k


CONFIGS: dict[str, LayerShape] = {
    "tiny_fwd": LayerShape(T=256, H=128, I=64, E=8, k=2, note="tiny MoE layer forward"),
    "qwen3_30b_fwd": LayerShape(T=4096, H=2048, I=768, E=128, k=8, ep_size=8,
                                note="Qwen3-30B-A3B-shaped MoE layer forward, T=4096"),
    "qwen3_30b_zipf_fwd": LayerShape(T=16384, H=2048, I=768, E=128, k=8, ep_size=8, bias="zipf",
                                     note="same shapes, T=16384, Zipf-skewed routing, empty experts"),
    "ep_rank_local": LayerShape(T=32768, H=2048, I=768, E=16, k=1, ep_size=8, segments=True,
                                src_ranks=8, note="one EP rank's local experts (16 of 128), 32768 rows, "
                                                  "8 source-rank blocks x 16 experts"),
    "qwen3_30b_fwd_bwd": LayerShape(T=8192, H=2048, I=768, E=128, k=8, ep_size=8, backward=True,
                                    note="Qwen3-30B-A3B-shaped MoE layer forward+backward, T=8192"),
}


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (no copy of values)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def _randn_bf16(g: torch.Generator, shape, std: float) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16)
    flat = out.view(-1)
    n = flat.numel()
    step = 1 << 26  # draw in slices to bound the fp32 temporary
    for s in range(0, n, step):
        e = min(n, s + step)
        v = torch.randn(e - s, generator=g, dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        flat[s:e] = v.to(torch.bfloat16)
    return out


def zipf_router_bias(g: torch.Generator, E: int, alpha: float = 1.2, scale: float = 2.0,
                     n_forced_empty: int = 4) -> torch.Tensor:
    """Per-expert router bias giving a Zipf-like expert popularity.

    A seeded permutation gives every expert a popularity rank r in 1..E; the
    bias is -scale*alpha*ln(r), and the n_forced_empty least popular experts
    get -1e4 so that some groups are guaranteed to receive no token.
    """
    perm = torch.randperm(E, generator=g)
    rank = (perm + 1).to(torch.float64)
    bias = -scale * alpha * torch.log(rank)
    bias[rank > E - n_forced_empty] = -1.0e4
    return bias.to(torch.float32)


def make_layer_inputs(shape: LayerShape | str, seed: int = 0, *, T: int | None = None,
                      router_std: float = 0.02, w_std: float = 0.02, with_dy: bool | None = None,
                      bias: str | None | bool = False) -> dict:
    """Inputs for a routed layer: x, Wr, Wg, Wu, Wd, optional bias, optional dY.

    All tensors live on the CPU.  `T` overrides the token count (the weights and
    their draw order do not change, so a smaller T gives a prefix-consistent x
    only when drawn separately; callers compare like with like).
    """
    if isinstance(shape, str):
        shape = CONFIGS[shape]
    assert not shape.segments, "use make_segment_inputs for segmented workloads"
    T = shape.T if T is None else T
    H, I, E, k = shape.H, shape.I, shape.E, shape.k
    if with_dy is None:
        with_dy = shape.backward
    if bias is False:
        bias = shape.bias
    g = torch.Generator().manual_seed(seed)
    out = {"T": T, "H": H, "I": I, "E": E, "k": k, "ep_size": shape.ep_size}
    out["x"] = _randn_bf16(g, (T, H), 1.0)
    out["Wr"] = torch.randn(H, E, generator=g, dtype=torch.float32).mul_(router_std)
    out["Wg"] = _randn_bf16(g, (E, I, H), w_std)
    out["Wu"] = _randn_bf16(g, (E, I, H), w_std)
    out["Wd"] = _randn_bf16(g, (E, H, I), w_std)
    out["bias"] = zipf_router_bias(g, E) if bias == "zipf" else None
    out["dy"] = _randn_bf16(g, (T, H), 1.0) if with_dy else None
    return out


def make_segment_inputs(shape: LayerShape | str = "ep_rank_local", seed: int = 0, *,
                        R: int | None = None, w_std: float = 0.02) -> dict:
    """Receive-side inputs of one EP rank: rows already grouped by (source rank, expert).

    counts_e ~ Multinomial(R, uniform over E local experts); each expert's rows
    are then split over the source ranks by Multinomial(counts_e, uniform).
    Buffer order is source-rank-major, then expert, so segment s*E+e holds the
    rows source rank s sent to local expert e, and seg_expert[s*E+e] = e.
    """
    if isinstance(shape, str):
        shape = CONFIGS[shape]
    R = shape.T if R is None else R
    H, I, E, S = shape.H, shape.I, shape.E, shape.src_ranks
    g = torch.Generator().manual_seed(seed)
    x_perm = _randn_bf16(g, (R, H), 1.0)
    Wg = _randn_bf16(g, (E, I, H), w_std)
    Wu = _randn_bf16(g, (E, I, H), w_std)
    Wd = _randn_bf16(g, (E, H, I), w_std)
    pick = torch.multinomial(torch.full((E,), 1.0 / E, dtype=torch.float64), R, replacement=True,
                             generator=g)
    counts_e = torch.bincount(pick, minlength=E)
    c = torch.zeros(S, E, dtype=torch.int64)
    for e in range(E):
        n = int(counts_e[e])
        if n:
            src = torch.multinomial(torch.full((S,), 1.0 / S, dtype=torch.float64), n,
                                    replacement=True, generator=g)
            c[:, e] = torch.bincount(src, minlength=S)
    seg_len = c.reshape(-1)                       # s-major, then e
    seg_offsets = torch.zeros(S * E + 1, dtype=torch.int32)
    seg_offsets[1:] = torch.cumsum(seg_len, 0).to(torch.int32)
    seg_expert = torch.arange(S * E, dtype=torch.int32) % E
    return {"R": R, "H": H, "I": I, "E": E, "num_seg": S * E, "x_perm": x_perm, "Wg": Wg,
            "Wu": Wu, "Wd": Wd, "seg_offsets": seg_offsets, "seg_expert": seg_expert,
            "counts_e": counts_e.to(torch.int32)}

