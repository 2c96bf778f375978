"""CPU oracle of the fused MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference arm may import or run anything in this package. The product path
(the CUDA library and its binding) never imports it, and this module imports
nothing from the product.

What it computes, and where the pages define it
-----------------------------------------------
The layer is the pipeline ``[Router] -> [Quantize-Dispatch] ->
[Permute-Experts-Unpermute] -> [Combine]`` (modular_kernel.py, module header
comment). Each step below is written plainly in numpy, in float64 unless a
page fixes the precision:

* route_softmax_topk / route_sigmoid_grouped -- the [Router] step. The pages
  name it and pass its outputs (``topk_ids``, ``topk_weights``;
  modular_kernel.py ``FusedMoEModularKernel.forward``) but never give its
  math. The readings used here: softmax -> top-k -> renormalise (the top_k
  largest logits, ties to the lower id), and DeepSeek-V3's published rule,
  sigmoid + bias -> grouped top-k -> renormalise x scale (a group scores the
  sum of its two largest biased scores).
  Where floating point decides an integer (the sigmoid router's selection),
  the decision is taken in float32 with the written ``sigmoid_f32_spec``,
  the same spec the CUDA router implements independently.
* permute -- groups routes by local expert; ``expanded_idx_to_permuted_idx``
  with -1 for a non-local expert (moe_output.py ``UnfinalizedMoEOutput``,
  field comments; ``expert_map`` in modular_kernel.py
  ``FusedMoEPrepareAndFinalize.prepare``).
* expert_mlp / experts -- GEMM1, ``silu_and_mul``, GEMM2; unweighted and
  unreduced (modular_kernel.py header comment on
  ``FusedMoEPermuteExpertsUnpermute`` and its ``activation`` method).
* finalize -- applies the routing weights and reduces over top_k
  (modular_kernel.py ``FusedMoEPrepareAndFinalize.finalize``), then the
  routed scale and the shared-expert add (moe_output.py ``MoEOutput`` field
  comments).
* expert_mlp's activation: ``silu_and_mul`` or ``gelu_and_mul`` (the two
  activations of modular_kernel.py ``FusedMoEPermuteExpertsUnpermute
  .activation``), GELU in its exact erf form; and the optional
  ``activation_clamp`` of flashinfer_moe_ep.py ``build_fi_mega_config``,
  which the pages pass through without defining (reading: the gate is
  clamped from above and the up projection to [-c, c] before the activation).
* experts_batched -- the same experts on the BatchedExperts activation format
  (modular_kernel.py ``FusedMoEActivationFormat``: [experts, max tokens per
  expert, hidden], with per-expert token counts).
* add_rmsnorm / finalize_add_rmsnorm -- the consumer moe_output.py
  ``MoEOutput`` names for an open reduction, the next layer's RMSNorm, with
  the top-k reduction folded in: residual += out; y = residual /
  sqrt(mean(residual^2) + eps) * gamma (RMSNorm as published by Zhang and
  Sennrich, 2019, in its fused residual-add form).
* mxfp8_quantize / experts_mxfp8 -- the experts with quantised activations,
  the ``quantize_input`` step that flashinfer_moe_ep.py ``build_fi_mega_config``
  enables beside e2m1 + ue8m0-per-32 weights (``FI_MOE_EP_BACKEND_SPECS``,
  the deep_gemm entry). The pages name the step but not its format; the
  reading used here is the MX recipe of the weights applied to the
  activations: FP8 E4M3 elements with one E8M0 scale per 32 consecutive
  values along each GEMM's reduction axis (OCP Microscaling Formats v1.0:
  scale 2^(floor(log2 amax) - 8), elements rounded to nearest-even and
  saturated at the largest finite E4M3 value). The E4M3 codec is written
  from the format's definition (sign, 4 exponent bits with bias 7, 3
  mantissa bits, subnormals at exponent 0, no infinities).
* e2m1 / E8M0 decode (flashinfer_moe_ep.py ``_E2M1_LUT`` and
  ``_dequant_fp4_ue8m0_gran32``): here the page fixes the arithmetic --
  an fp32 product of the table value and the scale, returned as bf16 -- and
  the oracle follows it.

Parity pins: every function here is pinned by tests in ``tests/`` against
values the pages print (the e2m1 table), closed forms, brute force over every
subset / every expert, and invariants the pages state. None is unpinned.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

__all__ = [
    "E2M1_TABLE", "e2m1_value", "ue8m0_scale", "dequant_mxfp4",
    "sigmoid_f32_spec", "route_softmax_topk", "route_sigmoid_grouped",
    "permute", "expert_mlp", "experts", "finalize", "shared_expert",
    "moe_forward", "bf16_round", "gelu_erf", "experts_batched", "add_rmsnorm",
    "finalize_add_rmsnorm", "E4M3_MAX", "e4m3_value", "e4m3_round", "mxfp8_scale_byte",
    "mxfp8_quantize", "mxfp8_dequantize", "mxfp8_qdq", "experts_mxfp8", "experts_chunked",
    "e4m3_split_scale_byte", "e4m3_split", "e4m3_split_value",
]

# --------------------------------------------------------------------------
# MXFP4 decode (flashinfer_moe_ep.py: ``_E2M1_LUT``, ``_dequant_fp4_ue8m0_gran32``,
# ``_dequant_expert_weights_to_bf16``)
# --------------------------------------------------------------------------

#: The 16 e2m1 code values in code order. Codes 0-7 are the non-negative
#: magnitudes; codes 8-15 repeat them with the sign bit (bit 3) set. The table
#: is an interface both sides must agree on, so it is kept value for value.
E2M1_TABLE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0)


def e2m1_value(code: int) -> float:
    """Value of one 4-bit e2m1 code (``_E2M1_LUT``)."""
    return E2M1_TABLE[int(code) & 0xF]


def ue8m0_scale(s) -> np.ndarray:
    """E8M0 scale byte -> float32: the byte becomes the fp32 exponent field,
    i.e. the float whose bits are ``s << 23`` (``_dequant_fp4_ue8m0_gran32``).
    Byte 0 therefore decodes to 0.0 and byte 255 to +inf, as the bit rule says.
    """
    s = np.asarray(s, dtype=np.uint32)
    return (s << np.uint32(23)).astype(np.uint32).view(np.float32)


def bf16_round(x) -> np.ndarray:
    """float -> nearest bfloat16 (ties to even), returned as float32 values.

    Works on the float32 bit pattern: add 0x7FFF plus the lowest kept bit,
    then clear the low 16 bits (for finite inputs and infinities this cannot
    overflow 32 bits); NaN stays NaN."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    r += u
    r += np.uint32(0x7FFF)
    r &= np.uint32(0xFFFF0000)
    out = r.view(np.float32)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = np.float32(np.nan)
    return out


def dequant_mxfp4(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Packed e2m1 [rows, C/2] + E8M0 scales [rows, C/32] -> values [rows, C].

    Byte j of a row holds element 2j in its low nibble and element 2j+1 in its
    high nibble; scale byte b covers elements 32b..32b+31. The product is taken
    in float32 and rounded to bf16, as ``_dequant_fp4_ue8m0_gran32`` does; for
    scale bytes 1..254 every product is exactly representable, so the bf16
    rounding changes nothing there. Returned as float64.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    rows, half = packed.shape
    C = 2 * half
    assert scales.shape == (rows, C // 32)
    table = np.array(E2M1_TABLE, dtype=np.float32)
    vals = np.empty((rows, C), dtype=np.float32)
    vals[:, 0::2] = table[packed & 0x0F]
    vals[:, 1::2] = table[packed >> 4]
    sf = ue8m0_scale(scales)                              # [rows, C/32], one scale per 32 values
    with np.errstate(over="ignore", invalid="ignore"):
        prod = (vals.reshape(rows, C // 32, 32) * sf[:, :, None]).reshape(rows, C)
    return bf16_round(prod).astype(np.float64)


# --------------------------------------------------------------------------
# MXFP8 activations: FP8 E4M3 elements, one E8M0 scale per 32 values
# --------------------------------------------------------------------------

#: The largest finite E4M3 value, 1.75 * 2^8 (code 0x7E); E4M3 has no infinities.
E4M3_MAX = 448.0


def e4m3_value(code) -> np.ndarray:
    """E4M3 code(s) -> value(s), float64. Bit 7 is the sign, bits 6..3 the
    exponent (bias 7), bits 2..0 the mantissa. Exponent field 0 holds the
    subnormals m/8 * 2^-6; every other field the normals (1 + m/8) * 2^(e-7),
    except S.1111.111, which is NaN."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


def e4m3_round(v) -> np.ndarray:
    """Value(s) -> nearest E4M3 code(s), ties to the even code, magnitudes
    above 448 saturated to 448 (NaN -> 0x7F). The quantum of a magnitude a is
    2^(max(floor(log2 a), -6) - 3): the normals' binade spacing, and the
    subnormals' fixed 2^-9 below 2^-6. a / quantum is exact in float64, so
    numpy's half-to-even round is the rounding rule itself."""
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v)
    a = np.minimum(np.abs(v), E4M3_MAX)
    with np.errstate(divide="ignore", invalid="ignore"):
        ex = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    ex = np.maximum(ex, -6.0)
    q = np.exp2(ex - 3.0)
    r = np.round(a / q) * q                       # rounded magnitude, still <= 448
    # encode r: a carry into the next binade is a normal with mantissa 0
    with np.errstate(divide="ignore", invalid="ignore"):
        er = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    normal = r >= 2.0 ** -6
    e_field = np.where(normal, er + 7.0, 0.0)
    m_field = np.where(normal, np.round((r / np.exp2(er) - 1.0) * 8.0), np.round(r / 2.0 ** -9))
    code = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    code = np.where(sign, code | 0x80, code)
    code = np.where(np.isnan(v), 0x7F, code)
    return code.astype(np.uint8)


def mxfp8_scale_byte(amax) -> np.ndarray:
    """E8M0 scale byte of blocks with largest magnitude ``amax`` (float32):
    the scale is 2^(floor(log2 amax) - 8), 8 being E4M3's largest exponent,
    so that amax / scale lies in [256, 512). On the float32 bit pattern,
    floor(log2 amax) + 127 is the exponent field, hence byte = field - 8. The
    byte is kept in 1..254, where every E8M0 decode gives 2^(byte - 127) (an
    all-zero block gets byte 1 and codes 0)."""
    a = np.abs(np.asarray(amax, dtype=np.float32))
    field = (a.reshape(-1).view(np.uint32) >> np.uint32(23)).astype(np.int64) & 0xFF
    return np.clip(field - 8, 1, 254).astype(np.uint8).reshape(a.shape)


def mxfp8_quantize(x):
    """x [..., C] (C a multiple of 32), taken as float32 -> (codes uint8
    [..., C], scale bytes uint8 [..., C/32]): blocks of 32 consecutive
    values along the last axis share one scale; each value becomes
    e4m3_round(value / scale) (value / scale is an exact power-of-two
    division)."""
    x = np.asarray(x, dtype=np.float32)
    C = x.shape[-1]
    assert C % 32 == 0
    blocks = x.reshape(x.shape[:-1] + (C // 32, 32)).astype(np.float64)
    amax = np.abs(blocks).max(axis=-1).astype(np.float32)
    sb = mxfp8_scale_byte(amax)
    scale = np.exp2(sb.astype(np.float64) - 127.0)
    codes = e4m3_round(blocks / scale[..., None])
    return codes.reshape(x.shape), sb


def mxfp8_dequantize(codes, scales) -> np.ndarray:
    """(codes [..., C], scale bytes [..., C/32]) -> values [..., C], float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    C = codes.shape[-1]
    vals = e4m3_value(codes).reshape(codes.shape[:-1] + (C // 32, 32))
    scale = np.exp2(np.asarray(scales, dtype=np.float64) - 127.0)
    return (vals * scale[..., None]).reshape(codes.shape)


def e4m3_split_scale_byte(amax) -> np.ndarray:
    """Scale byte of a block of the two-term split: the smallest b with
    amax <= 448 * 2^(b - 127) (no code of the block saturates), kept in
    1..254 (an all-zero block gets 1). With amax = m * 2^e, m in [1, 2),
    the candidates are e + 119 and e + 120."""
    a = np.abs(np.asarray(amax, dtype=np.float64))
    m, ex = np.frexp(np.where(a > 0, a, 1.0))          # a = m * 2^ex, m in [0.5, 1)
    b = (ex - 1) + 119
    b = np.where(a > 448.0 * np.exp2(b - 127.0), b + 1, b)
    b = np.where(a > 0, b, 1)
    return np.clip(b, 1, 254).astype(np.uint8)


def e4m3_split(x):
    """bf16 activations as two E4M3 terms (the MXFP4_A16 path): along the last
    axis, every block of 32 values (float32) gets
        hi = e4m3_round(x / s1),          s1 = 2^(b1 - 127), b1 from max |x|,
        r  = x - e4m3_value(hi) * s1      (exact),
        lo = e4m3_round(r / s2),          s2 = 2^(b2 - 127), b2 from max |r|,
    with the scale bytes of e4m3_split_scale_byte. Returns (hi codes, hi scale
    bytes, lo codes, lo scale bytes): codes [..., C], bytes [..., C/32]."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    C = x.shape[-1]
    assert C % 32 == 0
    blk = x.reshape(x.shape[:-1] + (C // 32, 32))
    b1 = e4m3_split_scale_byte(np.abs(blk).max(axis=-1))
    s1 = np.exp2(b1.astype(np.float64) - 127.0)[..., None]
    hi = e4m3_round(blk / s1)
    r = blk - e4m3_value(hi) * s1
    b2 = e4m3_split_scale_byte(np.abs(r).max(axis=-1))
    s2 = np.exp2(b2.astype(np.float64) - 127.0)[..., None]
    lo = e4m3_round(r / s2)
    return hi.reshape(x.shape), b1, lo.reshape(x.shape), b2


def e4m3_split_value(hi, b1, lo, b2) -> np.ndarray:
    """The value a two-term split stands for: hi * s1 + lo * s2, float64."""
    return mxfp8_dequantize(hi, b1) + mxfp8_dequantize(lo, b2)


def mxfp8_qdq(x) -> np.ndarray:
    """x as the GEMM consuming its MXFP8 form sees it: dequantize(quantize(x))."""
    return mxfp8_dequantize(*mxfp8_quantize(x))


# --------------------------------------------------------------------------
# Router
# --------------------------------------------------------------------------

def _topk_desc(keys: np.ndarray, k: int, allowed=None) -> list:
    """Indices of the k largest keys, ordered by key descending; equal keys
    go to the lower index. ``allowed`` masks candidates (None = all)."""
    idx = [i for i in range(len(keys)) if allowed is None or allowed[i]]
    idx.sort(key=lambda i: (-float(keys[i]), i))
    return idx[:k]


def route_softmax_topk(logits: np.ndarray, top_k: int, routed_scaling_factor: float = 1.0):
    """Softmax router: probabilities over all E experts, the top_k largest
    kept and renormalised to sum to one, times the routed scale.

    Selection is made on the float32 logits themselves (softmax is strictly
    increasing, so the top_k probabilities are the top_k logits), ordered by
    logit descending, ties to the lower expert id. Weights: float64 softmax
    over all experts, restricted to the selected ones, divided by their sum.
    Returns (ids int32 [M, k], weights float64 [M, k]).
    """
    logits = np.asarray(logits, dtype=np.float32)
    M, E = logits.shape
    ids = np.zeros((M, top_k), dtype=np.int32)
    w = np.zeros((M, top_k), dtype=np.float64)
    for t in range(M):
        sel = _topk_desc(logits[t], top_k)
        l64 = logits[t].astype(np.float64)
        p = np.exp(l64 - l64.max())
        p = p / p.sum()
        ps = p[sel]
        ids[t] = sel
        w[t] = ps / ps.sum() * routed_scaling_factor
    return ids, w


# Constants of the written float32 exp spec (Cody & Waite argument reduction,
# Taylor polynomial). LN2_HI is ln 2 cut to 16 significant bits so that
# n * LN2_HI is exact for |n| <= 256; LN2_LO is the float32 remainder.
_LOG2E = np.float32(1.4426950408889634)
_LN2_HI = np.float32(0.693145751953125)
_LN2_LO = np.float32(1.4286068203094173e-06)
_INV_FACT = [np.float32(1.0 / math.factorial(i)) for i in range(8)]   # 1/0! .. 1/7!


def _exp_f32_spec(t) -> np.ndarray:
    """exp(t) in float32 by the written spec, elementwise: every step one IEEE
    float32 operation rounded to nearest (no fused multiply-add).

      t > 88      -> +inf            t < -80 -> 0
      n = rint(t * LOG2E)            (float32 product, round half to even)
      r = (t - n*LN2_HI) - n*LN2_LO
      p = ((((((c7 r + c6) r + c5) r + c4) r + c3) r + c2) r + c1) r + c0,  c_i = fl32(1/i!)
      exp = p * 2^n                  (exact: 2^n is built from its bits)
    """
    t = np.asarray(t, dtype=np.float32)
    inner = (t <= np.float32(88.0)) & (t >= np.float32(-80.0))
    ti = np.where(inner, t, np.float32(0.0)).astype(np.float32)
    n = np.rint((ti * _LOG2E).astype(np.float32)).astype(np.float32)
    r = (ti - (n * _LN2_HI).astype(np.float32)).astype(np.float32)
    r = (r - (n * _LN2_LO).astype(np.float32)).astype(np.float32)
    p = np.full_like(r, _INV_FACT[7])
    for c in reversed(_INV_FACT[:7]):
        p = ((p * r).astype(np.float32) + c).astype(np.float32)
    two_n = ((n.astype(np.int32) + 127) << 23).astype(np.uint32).view(np.float32)
    e = (p * two_n).astype(np.float32)
    e = np.where(t > np.float32(88.0), np.float32(np.inf), e)
    e = np.where(t < np.float32(-80.0), np.float32(0.0), e)
    return np.where(np.isnan(t), t, e).astype(np.float32)


def sigmoid_f32_spec(x) -> np.ndarray:
    """sigma(x) = 1 / (1 + exp(-x)) in float32 with the written exp spec; one
    rounded float32 add and one rounded float32 divide (elementwise)."""
    x = np.asarray(x, dtype=np.float32)
    e = _exp_f32_spec(-x)
    one = np.float32(1.0)
    with np.errstate(over="ignore"):
        return (one / (one + e).astype(np.float32)).astype(np.float32)


def route_sigmoid_grouped(logits: np.ndarray, score_bias: np.ndarray, top_k: int,
                          n_group: int, topk_group: int,
                          routed_scaling_factor: float = 1.0):
    """Sigmoid + bias router with grouped top-k (DeepSeek-V3's published rule).

    s_e = sigmoid(l_e); b_e = s_e + bias_e (float32; the bias steers selection
    only). The E experts form n_group contiguous groups; a group's score is
    the float32 sum of its two largest b. The topk_group best groups are kept
    (ties to the lower group id); among their experts the top_k largest b are
    selected, ordered by b descending, ties to the lower expert id. The
    weights are the unbiased s of the selected experts divided by their sum,
    times the routed scale -- which is folded into the weights here, so the
    caller's later routed scale is 1.0 (moe_output.py, ``MoEOutput``
    ``routed_scaling_factor`` comment).
    Returns (ids int32 [M, k], weights float64 [M, k]).
    """
    logits = np.asarray(logits, dtype=np.float32)
    bias = np.asarray(score_bias, dtype=np.float32)
    M, E = logits.shape
    assert E % n_group == 0
    G = E // n_group
    s32 = sigmoid_f32_spec(logits)
    b32 = (s32 + bias[None, :]).astype(np.float32)
    ids = np.zeros((M, top_k), dtype=np.int32)
    w = np.zeros((M, top_k), dtype=np.float64)
    for t in range(M):
        gscore = np.zeros(n_group, dtype=np.float32)
        for g in range(n_group):
            top2 = sorted(b32[t, g * G:(g + 1) * G].tolist(), reverse=True)[:2]
            gscore[g] = np.float32(np.float32(top2[0]) + np.float32(top2[1]))
        groups = _topk_desc(gscore, topk_group)
        allowed = np.zeros(E, dtype=bool)
        for g in groups:
            allowed[g * G:(g + 1) * G] = True
        sel = _topk_desc(b32[t], top_k, allowed)
        s64 = 1.0 / (1.0 + np.exp(-logits[t].astype(np.float64)))
        ids[t] = sel
        w[t] = s64[sel] / s64[sel].sum() * routed_scaling_factor
    return ids, w


# --------------------------------------------------------------------------
# Permute (the permute map of moe_output.py ``UnfinalizedMoEOutput``)
# --------------------------------------------------------------------------

def permute(topk_ids: np.ndarray, E: int, expert_map=None):
    """Group the M*k routes by local expert.

    ``expert_map[e]`` gives the local id of global expert e, -1 if it is not
    local; without a map every expert is local with its own id. Routes are
    ordered expert-major and, within an expert, by expanded index t*k + j.
    Returns (offsets int32 [E_local+1], map int32 [M, k] with -1 for masked
    routes, inverse int32 [R] giving the expanded index of each permuted row,
    E_local).
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, k = ids.shape
    if expert_map is None:
        emap = np.arange(E, dtype=np.int64)
        E_local = E
    else:
        emap = np.asarray(expert_map, dtype=np.int64)
        E_local = int(emap.max()) + 1 if (emap >= 0).any() else 0
    local = emap[ids.reshape(-1)]                  # [M*k]
    routes = [(int(local[i]), i) for i in range(M * k) if local[i] >= 0]
    routes.sort()                                  # expert-major, then expanded index
    counts = np.zeros(E_local, dtype=np.int64)
    for le, _ in routes:
        counts[le] += 1
    offsets = np.zeros(E_local + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    pmap = np.full(M * k, -1, dtype=np.int32)
    inverse = np.zeros(len(routes), dtype=np.int32)
    for p, (_, i) in enumerate(routes):
        pmap[i] = p
        inverse[p] = i
    return offsets, pmap.reshape(M, k), inverse, E_local


# --------------------------------------------------------------------------
# Experts (GEMM1 -> silu_and_mul -> GEMM2), unweighted and unreduced
# --------------------------------------------------------------------------

def gelu_erf(z) -> np.ndarray:
    """GELU in its exact form, z * Phi(z) = z/2 * (1 + erf(z / sqrt 2)), with
    Phi the standard normal CDF (erf from scipy.special)."""
    from scipy.special import erf
    z = np.asarray(z, dtype=np.float64)
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def expert_mlp(x: np.ndarray, w1: np.ndarray, w2: np.ndarray, activation: str = "silu",
               clamp=None, qdq=None) -> np.ndarray:
    """One expert on token rows x [T, K]: h = x W1^T [T, 2N]; the first N
    columns are the gate, the last N the up projection (the ``*_and_mul``
    activations: output width half the input width). With ``clamp`` = c the
    gate is clamped to at most c and up to [-c, c] first. Then
    a = act(gate) * up, with silu(z) = z / (1 + e^-z) or gelu = gelu_erf;
    y = a W2^T [T, K]. Float64.

    ``qdq`` (quantised activations): applied to x before GEMM1 and to a,
    rounded to float32, before GEMM2 -- each GEMM then reads its activation
    operand as its quantised form dequantised."""
    if qdq is not None:
        x = qdq(x)
    x = np.asarray(x, dtype=np.float64)
    w1 = np.asarray(w1, dtype=np.float64)
    w2 = np.asarray(w2, dtype=np.float64)
    N = w1.shape[0] // 2
    h = x @ w1.T
    gate, up = h[:, :N], h[:, N:]
    if clamp is not None:
        gate = np.minimum(gate, clamp)
        up = np.clip(up, -clamp, clamp)
    if activation == "silu":
        with np.errstate(over="ignore"):
            a = gate / (1.0 + np.exp(-gate)) * up
    elif activation == "gelu":
        a = gelu_erf(gate) * up
    else:
        raise ValueError(activation)
    if qdq is not None:
        a = qdq(np.asarray(a, dtype=np.float32))
    return a @ w2.T


def experts(x: np.ndarray, w1: np.ndarray, w2: np.ndarray, offsets: np.ndarray,
            inverse: np.ndarray, top_k: int, activation: str = "silu", clamp=None,
            qdq=None) -> np.ndarray:
    """``gemm2_permuted`` [R, K]: row p is the output of expert le (the p-th
    row falls in [offsets[le], offsets[le+1])) on token inverse[p] // top_k.
    ``w1``/``w2`` are the local experts' weights as float arrays; ``qdq`` as
    in expert_mlp."""
    x = np.asarray(x, dtype=np.float64)
    R = int(offsets[-1])
    out = np.zeros((R, w2.shape[1]), dtype=np.float64)
    for le in range(len(offsets) - 1):
        r0, r1 = int(offsets[le]), int(offsets[le + 1])
        if r1 > r0:
            toks = np.asarray(inverse[r0:r1], dtype=np.int64) // top_k
            out[r0:r1] = expert_mlp(x[toks], w1[le], w2[le], activation, clamp, qdq)
    return out


def experts_chunked(x: np.ndarray, topk_ids: np.ndarray, w1, w2, E: int, chunk_tokens: int,
                    expert_map=None, activation: str = "silu", clamp=None):
    """Activation chunking (modular_kernel.py, FusedMoEModularKernel.forward:
    M is split into chunks of CHUNK_SIZE tokens and the experts' apply() runs
    on each chunk's activations and topk_ids, writing that chunk's slice of
    the output). Chunk c holds tokens [t0, t1), t0 = c * chunk_tokens; its
    routes are permuted on their own (the canonical order of ``permute``),
    its expert outputs fill rows [t0 * k, t0 * k + R_c) of a [M * k, K]
    gemm2_permuted, and its map entries are offset by t0 * k to point there.
    Returns (map int32 [M, k] with -1 for masked routes, gemm2_permuted
    float64 [M * k, K] with NaN in rows no map entry points to)."""
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, k = ids.shape
    x = np.asarray(x, dtype=np.float64)
    pmap = np.full((M, k), -1, dtype=np.int32)
    g2 = np.full((M * k, w2.shape[1]), np.nan)
    for t0 in range(0, M, chunk_tokens):
        t1 = min(M, t0 + chunk_tokens)
        offsets, m, inverse, _ = permute(ids[t0:t1], E, expert_map)
        R = int(offsets[-1])
        g2[t0 * k:t0 * k + R] = experts(x[t0:t1], w1, w2, offsets, inverse, k, activation, clamp)
        pmap[t0:t1] = np.where(m >= 0, m + t0 * k, -1)
    return pmap, g2


def experts_mxfp8(x: np.ndarray, w1: np.ndarray, w2: np.ndarray, offsets: np.ndarray,
                  inverse: np.ndarray, top_k: int, activation: str = "silu", clamp=None) -> np.ndarray:
    """``experts`` with MXFP8 activations: every token row quantised per 32
    along K before GEMM1, the activation output (float32) per 32 along N
    before GEMM2; the weights as given (MXFP4 weights: their exact dequantised
    values)."""
    return experts(x, w1, w2, offsets, inverse, top_k, activation, clamp, qdq=mxfp8_qdq)


def experts_batched(xb: np.ndarray, counts: np.ndarray, w1: np.ndarray, w2: np.ndarray,
                    activation: str = "silu", clamp=None) -> np.ndarray:
    """The experts on the BatchedExperts format: xb [E, T_max, K], expert e's
    tokens are rows 0 .. counts[e]-1 of xb[e]. Returns y [E, T_max, K] with
    y[e, r] = the expert's output for r < counts[e], and 0 beyond."""
    xb = np.asarray(xb, dtype=np.float64)
    E, T, _ = xb.shape
    y = np.zeros((E, T, w2.shape[1]), dtype=np.float64)
    for e in range(E):
        c = int(counts[e])
        if c > 0:
            y[e, :c] = expert_mlp(xb[e, :c], w1[e], w2[e], activation, clamp)
    return y


def shared_expert(x: np.ndarray, ws1: np.ndarray, ws2: np.ndarray) -> np.ndarray:
    """The shared expert: the same gated MLP applied to every token."""
    return expert_mlp(x, ws1, ws2)


# --------------------------------------------------------------------------
# Finalize (modular_kernel.py ``FusedMoEPrepareAndFinalize.finalize``;
# moe_output.py ``MoEOutput``)
# --------------------------------------------------------------------------

def finalize(gemm2_permuted: np.ndarray, expert_weights: np.ndarray, pmap: np.ndarray,
             shared=None, routed_scaling_factor: float = 1.0) -> np.ndarray:
    """out[t] = rsf * sum_j w[t,j] * gemm2_permuted[map[t,j]] + shared[t], the
    sum over the routes with map != -1 (a -1 route contributes nothing), in
    j order; the shared output is added after the routed scale."""
    g = np.asarray(gemm2_permuted, dtype=np.float64)
    w = np.asarray(expert_weights, dtype=np.float64)
    pmap = np.asarray(pmap)
    M, k = pmap.shape
    out = np.zeros((M, g.shape[1] if g.ndim == 2 else 0), dtype=np.float64)
    for t in range(M):
        acc = np.zeros(out.shape[1], dtype=np.float64)
        for j in range(k):
            p = int(pmap[t, j])
            if p >= 0:
                acc += w[t, j] * g[p]
        out[t] = routed_scaling_factor * acc
        if shared is not None:
            out[t] += np.asarray(shared[t], dtype=np.float64)
    return out


def add_rmsnorm(x: np.ndarray, residual: np.ndarray, gamma: np.ndarray, eps: float):
    """RMSNorm with the residual add in front: r = residual + x;
    y = r / sqrt(mean over the hidden dim of r^2 + eps) * gamma.
    Returns (r, y), float64."""
    r = np.asarray(residual, dtype=np.float64) + np.asarray(x, dtype=np.float64)
    ms = np.mean(r * r, axis=-1, keepdims=True)
    y = r / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)
    return r, y


def finalize_add_rmsnorm(gemm2_permuted, expert_weights, pmap, residual, gamma, eps, shared=None,
                         routed_scaling_factor: float = 1.0):
    """finalize, then add_rmsnorm on its output: the next layer's RMSNorm
    with the MoE's top-k reduction folded in. Returns (residual', y)."""
    out = finalize(gemm2_permuted, expert_weights, pmap, shared, routed_scaling_factor)
    return add_rmsnorm(out, residual, gamma, eps)


def moe_forward(x, logits, w1, w2, top_k, route="softmax", score_bias=None,
                n_group=1, topk_group=1, routed_scaling_factor=1.0,
                expert_map=None, ws1=None, ws2=None):
    """The whole layer: route -> permute -> experts -> finalize (+ shared).

    ``w1``/``w2`` are float arrays of the local experts only ([E_local, 2N, K],
    [E_local, K, N]). The routed scale of the sigmoid router is folded into
    its weights, so finalize then uses 1.0. Returns a dict of every
    intermediate (ids, weights, offsets, map, inverse, gemm2_permuted,
    shared, out).
    """
    x = np.asarray(x, dtype=np.float64)
    logits = np.asarray(logits, dtype=np.float32)
    E = logits.shape[1]
    if route == "softmax":
        ids, w = route_softmax_topk(logits, top_k, routed_scaling_factor)
    else:
        ids, w = route_sigmoid_grouped(logits, score_bias, top_k, n_group, topk_group,
                                       routed_scaling_factor)
    offsets, pmap, inverse, _ = permute(ids, E, expert_map)
    g2 = experts(x, w1, w2, offsets, inverse, top_k)
    shared = shared_expert(x, ws1, ws2) if ws1 is not None else None
    out = finalize(g2, w, pmap, shared, 1.0)
    return dict(ids=ids, weights=w, offsets=offsets, map=pmap, inverse=inverse,
                gemm2_permuted=g2, shared=shared, out=out)
