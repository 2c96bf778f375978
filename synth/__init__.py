"""Seeded synthetic inputs for the fused MoE layer forward.

This module only draws random numbers and lays them out in the shapes of the
layer's inputs. It holds none of the layer's arithmetic (no routing, no
permute, no expert MLP, no finalize), so both the CPU oracle's tests and the
CUDA path's tests/benchmark can take their inputs from it without sharing any
of the method.

The one piece of number formatting here is the MXFP4 *quantiser* used to make
the DeepSeek-V3-shaped routed weights: the layer consumes e2m1 codes with an
E8M0 scale per 32 values (flashinfer_moe_ep.py, the MXFP4 recipe comments and
``_dequant_fp4_ue8m0_gran32``), and the pages never say how such a checkpoint
was produced. The quantiser follows the OCP Microscaling (MX) v1.0 rule:
shared exponent ``floor(log2(amax)) - 2`` (2 = e2m1's largest exponent),
values divided by ``2**shared_exp`` and rounded to the nearest e2m1 grid
point (ties to the even code), saturating at +-6; an all-zero block gets scale
byte 127. Parity never depends on it: the oracle and the kernels consume the
same bytes.

Every generator takes a ``torch.Generator`` seed and a device. Values drawn
on the CPU and on a GPU differ (different generators); a test always feeds
the *same* bytes to both sides.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = [
    "MoEConfig", "CONFIGS", "LayerInputs", "make_layer", "make_tokens",
    "quantize_mxfp4", "masked_expert_map",
]


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """Shape and distribution recipe of one synthetic MoE layer.

    K = hidden size, N = expert intermediate size (the gate and the up
    projection each have N rows, so W1 has 2N rows), E = routed experts,
    top_k = experts per token.
    """
    name: str
    K: int
    N: int
    E: int
    top_k: int
    route: str                      # "softmax" | "sigmoid_grouped"
    w1_std: float                   # std of W1 entries (bf16 or pre-quantisation)
    w2_std: float
    logit_bias_std: float = 0.0     # per-expert bias baked into the logits (skewed load)
    n_group: int = 1
    topk_group: int = 1
    routed_scaling_factor: float = 1.0
    score_bias_std: float = 0.0     # selection-only bias of the sigmoid router
    weight_format: str = "bf16"     # "bf16" | "mxfp4"
    shared_N: int = 0               # shared expert intermediate size (0 = none)
    shared_std: float = 0.02
    m_sweep: tuple = ()
    seed: int = 0


# Shapes and distributions of the workloads the layer is measured on.
CONFIGS = {
    # K=128, N=256, E=8, k=2; W ~ N(0, 1/sqrt(fan_in)) (second parameter read
    # as the standard deviation); softmax, top-k, renormalise; seed 0.
    "tiny": MoEConfig("tiny", K=128, N=256, E=8, top_k=2, route="softmax",
                      w1_std=1.0 / math.sqrt(128), w2_std=1.0 / math.sqrt(256),
                      m_sweep=(16,), seed=0),
    # Mixtral-8x7B-shaped: near-uniform load from N(0,1) logits.
    "mixtral": MoEConfig("mixtral", K=4096, N=14336, E=8, top_k=2, route="softmax",
                         w1_std=0.02, w2_std=0.02,
                         m_sweep=(1, 8, 64, 512, 4096, 8192), seed=1),
    # Qwen3-30B-A3B-shaped: logits N(0,1) plus a per-expert N(0,1.5) bias, so
    # the expert load is heavy-tailed and some experts get no tokens.
    "qwen3": MoEConfig("qwen3", K=2048, N=768, E=128, top_k=8, route="softmax",
                       w1_std=0.02, w2_std=0.02, logit_bias_std=1.5,
                       m_sweep=(1, 32, 256, 2048, 8192), seed=2),
    # DeepSeek-V3-shaped: sigmoid scores + N(0,0.1) selection bias, 8 groups of
    # 32, 4 groups kept, top-8, scale 2.5 folded into the weights; MXFP4 routed
    # weights quantised from N(0,0.02); one bf16 shared expert with N=2048.
    "deepseek": MoEConfig("deepseek", K=7168, N=2048, E=256, top_k=8,
                          route="sigmoid_grouped", w1_std=0.02, w2_std=0.02,
                          n_group=8, topk_group=4, routed_scaling_factor=2.5,
                          score_bias_std=0.1, weight_format="mxfp4",
                          shared_N=2048, shared_std=0.02,
                          m_sweep=(1, 64, 1024, 8192), seed=3),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, std, g, device, dtype=torch.bfloat16, chunk_rows=None):
    """N(0, std^2) drawn in fp32 then cast (RNE) to ``dtype``."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1, shape[-1])
    rows = flat.shape[0]
    step = chunk_rows or rows
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        flat[r0:r1] = (torch.randn(r1 - r0, shape[-1], generator=g, device=device,
                                   dtype=torch.float32) * std).to(dtype)
    return out


# e2m1 magnitudes in code order 0..7 (sign is bit 3).
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_mxfp4(w: torch.Tensor):
    """OCP-MX quantiser: float [rows, C] -> (packed u8 [rows, C/2], scale u8 [rows, C/32]).

    Element 2j goes to the low nibble of byte j and element 2j+1 to the high
    nibble, the layout ``_dequant_fp4_ue8m0_gran32`` in flashinfer_moe_ep.py
    reads back.
    """
    rows, C = w.shape
    assert C % 32 == 0
    x = w.to(torch.float32).view(rows, C // 32, 32)
    amax = x.abs().amax(dim=-1, keepdim=True)
    zero_block = amax == 0
    e = torch.floor(torch.log2(torch.where(zero_block, torch.ones_like(amax), amax))) - 2.0
    e = torch.where(zero_block, torch.zeros_like(e), e).clamp(-126.0, 127.0)
    q = x / torch.exp2(e)
    mag = q.abs()
    # nearest grid point; at an exact midpoint take the even code.
    bounds = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], device=w.device)
    code = torch.bucketize(mag, bounds, right=False)        # ties -> lower code
    tie_up = torch.zeros_like(mag, dtype=torch.bool)
    for b in (0.75, 1.75, 3.5):     # midpoints whose lower neighbour has an odd code
        tie_up |= mag == b
    code = code + tie_up.to(code.dtype)
    code = code.clamp(max=7)
    sign = (q < 0) & (code > 0)
    code = (code | (sign.to(code.dtype) << 3)).to(torch.uint8).view(rows, C)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    scale = (e.view(rows, C // 32) + 127.0).to(torch.uint8).contiguous()
    return packed, scale


@dataclasses.dataclass
class LayerInputs:
    """Weights of one MoE layer (all experts; device tensors)."""
    cfg: MoEConfig
    w1: torch.Tensor                 # bf16 [E, 2N, K] or u8 [E, 2N, K/2]
    w2: torch.Tensor                 # bf16 [E, K, N]  or u8 [E, K, N/2]
    w1_scale: Optional[torch.Tensor] = None   # u8 [E, 2N, K/32]
    w2_scale: Optional[torch.Tensor] = None   # u8 [E, K, N/32]
    score_bias: Optional[torch.Tensor] = None # f32 [E] (sigmoid router)
    logit_bias: Optional[torch.Tensor] = None # f32 [E] (baked into logits)
    ws1: Optional[torch.Tensor] = None        # bf16 [2Ns, K] shared expert
    ws2: Optional[torch.Tensor] = None        # bf16 [K, Ns]


def make_layer(cfg: MoEConfig, device="cpu", experts=None) -> LayerInputs:
    """Seeded weights of ``cfg``; ``experts`` restricts generation to a subset
    of expert indices (the others are left as zeros), for cheap CPU use."""
    g = _gen(device, cfg.seed * 1000 + 1)
    E, K, N = cfg.E, cfg.K, cfg.N
    li = LayerInputs(cfg=cfg, w1=None, w2=None)
    if cfg.logit_bias_std:
        li.logit_bias = torch.randn(E, generator=g, device=device) * cfg.logit_bias_std
    if cfg.score_bias_std:
        li.score_bias = torch.randn(E, generator=g, device=device) * cfg.score_bias_std
    sel = range(E) if experts is None else experts
    if cfg.weight_format == "bf16":
        li.w1 = torch.zeros(E, 2 * N, K, dtype=torch.bfloat16, device=device)
        li.w2 = torch.zeros(E, K, N, dtype=torch.bfloat16, device=device)
        for e in sel:
            ge = _gen(device, cfg.seed * 1000 + 7 + e)
            li.w1[e] = _randn((2 * N, K), cfg.w1_std, ge, device, chunk_rows=4096)
            li.w2[e] = _randn((K, N), cfg.w2_std, ge, device, chunk_rows=4096)
    else:
        li.w1 = torch.zeros(E, 2 * N, K // 2, dtype=torch.uint8, device=device)
        li.w2 = torch.zeros(E, K, N // 2, dtype=torch.uint8, device=device)
        li.w1_scale = torch.full((E, 2 * N, K // 32), 127, dtype=torch.uint8, device=device)
        li.w2_scale = torch.full((E, K, N // 32), 127, dtype=torch.uint8, device=device)
        for e in sel:
            ge = _gen(device, cfg.seed * 1000 + 7 + e)
            p, s = quantize_mxfp4(_randn((2 * N, K), cfg.w1_std, ge, device, chunk_rows=4096))
            li.w1[e], li.w1_scale[e] = p, s
            p, s = quantize_mxfp4(_randn((K, N), cfg.w2_std, ge, device, chunk_rows=4096))
            li.w2[e], li.w2_scale[e] = p, s
    if cfg.shared_N:
        gs = _gen(device, cfg.seed * 1000 + 3)
        li.ws1 = _randn((2 * cfg.shared_N, K), cfg.shared_std, gs, device, chunk_rows=4096)
        li.ws2 = _randn((K, cfg.shared_N), cfg.shared_std, gs, device, chunk_rows=4096)
    return li


def make_tokens(cfg: MoEConfig, M: int, device="cpu", layer: Optional[LayerInputs] = None,
                seed_offset: int = 0):
    """Seeded activations x bf16 [M, K] and router logits f32 [M, E].

    Logits are N(0,1); for a skewed config the layer's per-expert bias is
    added (baked in), which makes the expert load heavy-tailed.
    """
    g = _gen(device, cfg.seed * 1000 + 500 + M + 7919 * seed_offset)
    x = _randn((M, cfg.K), 1.0, g, device, chunk_rows=8192)
    logits = torch.randn(M, cfg.E, generator=g, device=device, dtype=torch.float32)
    if layer is not None and layer.logit_bias is not None:
        logits = logits + layer.logit_bias.to(device)[None, :]
    return x, logits.contiguous()


def masked_expert_map(E: int, seed: int, device="cpu"):
    """expert_map [E] int32 marking a seeded random half of the experts
    non-local (-1); local ids ascend with the global ids."""
    g = _gen("cpu", seed * 1000 + 11)
    perm = torch.randperm(E, generator=g)
    local = torch.zeros(E, dtype=torch.bool)
    local[perm[: E // 2]] = True
    emap = torch.full((E,), -1, dtype=torch.int32)
    emap[local] = torch.arange(int(local.sum()), dtype=torch.int32)
    return emap.to(device), int(local.sum())
