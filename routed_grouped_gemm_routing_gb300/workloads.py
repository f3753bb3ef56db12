"""Seeded synthetic workloads for the routed MoE expert layer.

This module only draws inputs; it holds none of the layer's arithmetic.  The
tests, the benchmark and the smoke check use it to feed the same values to
the CUDA library and to the CPU oracle.

Shapes follow the DeepSeek-style layers the pages benchmark (Primus-Turbo
"Mega MoE" README, "Performance / Test Configuration": hidden 7168,
intermediate 2048, 256 experts, top-k 8, 8192 tokens; the DeepGEMM Mega-MoE
article's usage example: 384 experts, top-k 6, hidden 7168, intermediate
3072, 4096 tokens).  No dataset or trained weights exist for them, so every
tensor is drawn from a seeded generator:

  x  ~ N(0, 1)            [T, H]      bfloat16
  W1 ~ N(0, 1/H)          [E, H, 2I]  bfloat16   (columns [0,I) gate, [I,2I) up)
  W2 ~ N(0, 1/I)          [E, I, H]   bfloat16
  dY ~ N(0, 1)            [T, H]      bfloat16
  logits ~ N(0, 1)        [T, E]      float32, plus an optional per-expert bias
  topk_idx = the k largest logits per token (ties to the lower expert id)
  topk_w   = softmax over the k selected logits (float32)

The skewed workload adds bias_e = -c * 1.2 * ln(e + 1) (c = 0.5) to every
token's logits, so expert popularity falls off as a power law over the
expert id.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    skew_c: float = 0.0

    @property
    def slots(self) -> int:
        return self.T * self.k

    def flops_forward(self) -> float:
        """Useful multiply-add FLOPs of the forward pass (padding excluded):
        L1 is 2*H*2I per slot, L2 is 2*I*H per slot."""
        return 6.0 * self.H * self.I * self.slots

    def flops_backward(self) -> float:
        """Useful FLOPs of the backward pass: L2 dgrad 2HI, dW2 2HI,
        dW1 4HI, L1 dgrad 4HI per slot."""
        return 12.0 * self.H * self.I * self.slots


CONFIGS = {
    "tiny": LayerShape("tiny", T=64, H=128, I=64, E=8, k=2),
    "v2lite": LayerShape("v2lite", T=4096, H=2048, I=1408, E=64, k=6),
    "v3": LayerShape("v3", T=8192, H=7168, I=2048, E=256, k=8),
    "wide": LayerShape("wide", T=4096, H=7168, I=3072, E=384, k=6),
    "skew": LayerShape("skew", T=8192, H=7168, I=2048, E=256, k=8, skew_c=0.5),
    # twice as sharp: the top expert takes nearly every token and many
    # experts get no slot at all (a correctness case for empty experts)
    "skew_c1": LayerShape("skew_c1", T=8192, H=7168, I=2048, E=256, k=8, skew_c=1.0),
    # V3 expert shapes with 16 experts and 512 tokens: the same ~256 routed
    # rows per expert as the V3 layer in ~3 GB of device memory (kernel
    # profiling captures must stay small).
    "v3_slice": LayerShape("v3_slice", T=512, H=7168, I=2048, E=16, k=8),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_routing(T: int, E: int, k: int, seed: int = 0, skew_c: float = 0.0, device="cpu"):
    """(topk_idx int32 [T,k], topk_w float32 [T,k]) from Gaussian logits."""
    g = _gen(device, seed * 7919 + 11)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if skew_c:
        bias = -skew_c * 1.2 * torch.log(torch.arange(1, E + 1, device=device, dtype=torch.float32))
        logits = logits + bias
    order = torch.sort(logits, dim=1, descending=True, stable=True).indices[:, :k]
    sel = torch.gather(logits, 1, order)
    w = torch.softmax(sel, dim=1)
    return order.to(torch.int32).contiguous(), w.to(torch.float32).contiguous()


def _normal_bf16(shape, std: float, g: torch.Generator, device) -> torch.Tensor:
    """N(0, std^2) in bfloat16, drawn in slabs along dim 0 to bound the FP32
    temporary for multi-GB weights."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    rows = shape[0]
    per_row = out[0].numel()
    step = max(1, (1 << 27) // max(per_row, 1))
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        tmp = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device, dtype=torch.float32)
        out[r0:r1] = (tmp * std).to(torch.bfloat16)
    return out


def make_layer_inputs(shape: LayerShape, seed: int = 0, device="cpu", with_grad_out: bool = True):
    """Dict with x, W1, W2, dY (bfloat16), topk_idx (int32), topk_w (float32)."""
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    idx, w = make_routing(T, E, k, seed=seed, skew_c=shape.skew_c, device=device)
    out = dict(
        x=_normal_bf16((T, H), 1.0, _gen(device, seed * 7919 + 1), device),
        W1=_normal_bf16((E, H, 2 * I), 1.0 / math.sqrt(H), _gen(device, seed * 7919 + 2), device),
        W2=_normal_bf16((E, I, H), 1.0 / math.sqrt(I), _gen(device, seed * 7919 + 3), device),
        topk_idx=idx,
        topk_w=w,
    )
    if with_grad_out:
        out["dY"] = _normal_bf16((T, H), 1.0, _gen(device, seed * 7919 + 4), device)
    return out


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a bfloat16 tensor's bit patterns."""
    import numpy as np

    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
