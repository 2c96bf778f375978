"""GPU parity of the MXFP4-weight x MXFP8-activation experts (block-scaled
tensor-core MMAs): the MXFP8 quantiser bit for bit against the oracle's, the
rearranged weight scales byte for byte, and the experts (gemm2_permuted, the
finalize, the finalize folded into GEMM2, the whole DeepSeek-shaped layer)
against the oracle's experts_mxfp8 on the same bytes.

Tolerance of the experts: both sides quantise x identically (bit-exact), so
what differs is the fp32 accumulation of GEMM1 and GEMM2 (the products of
e2m1, E4M3 and power-of-two scales are exact; the sums agree to ~1e-7) and,
through GEMM1's sum, the E4M3 rounding of an activation value lying within
that ~1e-7 of a rounding boundary: there the GPU's code and the oracle's are
both correct roundings of the values each side holds, one quantum apart (a
few per million values). So every value must lie within 1e-2 * RMS(ref) (the
bf16 path's bar) plus the largest change one such flip can make on it (the
largest quantum of its row's activations times the largest |W2| entry of
its output), and at most 0.5 % of the rows (at least 2) may use that
allowance.
"""
import numpy as np
import pytest
import torch

import oracle as O
from _helpers import lib, max_err, tol
from test_gpu_parity import _check_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    m = lib()
    assert m.moe_device_check() == 0, "needs a compute capability 10.3 device"
    return m


def _check_no_error(moe):
    st = moe.moe_get_error()
    assert st == 0, moe.status_string(st)


# ------------------------------------------------------------------ quantiser

@pytest.mark.parametrize("rows,C", [(1, 128), (37, 384), (300, 1024), (9, 7168)])
def test_mxfp8_quantize_bitexact(moe, rows, C):
    """Codes and scale bytes equal the oracle's on rows spanning 2^-20 .. 2^20
    in magnitude, with special rows: all zero, one huge value swamping its
    block, bf16 subnormals, and values that saturate."""
    g = torch.Generator().manual_seed(rows * 31 + C)
    x = torch.randn(rows, C, generator=g) * torch.exp(torch.empty(rows, 1).uniform_(-14, 14, generator=g))
    if rows >= 9:
        x[1] = 0.0
        x[2, 5] = 3.0e38
        x[3] = torch.randn(C, generator=g) * 1e-39          # bf16 subnormals
        x[4, ::7] = -2.0 ** 120
        x[5, :32] = torch.tensor([448.0 * 2 ** 3, 463.0 * 2 ** 3] + [1.0] * 30)
        x[6, 32:64] = 2.0 ** -126                           # a block at the smallest normal
    xb = x.to(torch.bfloat16)
    codes = torch.full((rows, C), 0x55, dtype=torch.uint8, device=DEV)
    scales = torch.full((rows, C // 32), 0x55, dtype=torch.uint8, device=DEV)
    moe.moe_mxfp8_quantize(xb.to(DEV), rows, C, codes, scales)
    torch.cuda.synchronize()
    rc, rs = O.mxfp8_quantize(xb.float().numpy())
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_mxfp8_quantize_argument_checks(moe):
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device=DEV)
    c = torch.empty(4, 128, dtype=torch.uint8, device=DEV)
    s = torch.empty(4, 4, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_mxfp8_quantize(x, 4, 96, c, s)
    assert e.value.status == moe.MOE_ERR_ALIGNMENT
    moe.moe_mxfp8_quantize(x, 0, 128, c, s)                 # empty: no-op


# ------------------------------------------------------------------ weight-scale layout

def test_mx_prepare_scales_layout(moe):
    """Every byte lands where the atom layout puts it: row r of tile r // 128,
    k-block kb, chunk j at byte (r % 32) * 16 + ((r % 128) // 32) * 4 + j of
    atom (r // 128, kb)."""
    E, rows, cols = 3, 256, 384
    g = torch.Generator().manual_seed(5)
    sc = torch.randint(0, 256, (E, rows, cols // 32), generator=g, dtype=torch.uint8)
    n = moe.moe_mx_prepared_scales_size(E, rows, cols)
    assert n == E * rows // 128 * cols // 128 * 512
    out = torch.zeros(n, dtype=torch.uint8, device=DEV)
    moe.moe_mx_prepare_scales(sc.to(DEV), E, rows, cols, out)
    torch.cuda.synchronize()
    flat = sc.reshape(E * rows, cols // 32).numpy()
    want = np.zeros((E * rows // 128, cols // 128, 512), np.uint8)
    for R in range(E * rows):
        r = R % 128
        for kb in range(cols // 128):
            for j in range(4):
                want[R // 128, kb, (r % 32) * 16 + (r // 32) * 4 + j] = flat[R, kb * 4 + j]
    assert np.array_equal(out.cpu().numpy().reshape(want.shape), want)
    assert moe.moe_mx_prepared_scales_size(E, 100, cols) == 0


# ------------------------------------------------------------------ experts

def _oracle_a8(x, w1, w2, offs, inv, k, activation="silu", clamp=None):
    """The oracle's experts_mxfp8 rows, and per row and output the largest
    change one activation rounded to the neighbouring E4M3 code would make:
    max over the row's activations of the E4M3 quantum at the value (times
    its block scale), times max |W2[e][j, :]|. The activations are the ones
    the oracle quantises, taken through its quantisation hook."""
    calls = []

    def spy(a):
        calls.append(np.asarray(a))
        return O.mxfp8_qdq(a)
    ref = O.experts(x, w1, w2, offs, inv, k, activation, clamp, qdq=spy)
    assert np.array_equal(ref, O.experts_mxfp8(x, w1, w2, offs, inv, k, activation, clamp))
    acts = calls[1::2]                                    # per expert call: x first, then the activation
    R, K = ref.shape
    allow = np.zeros((R, K))
    i = 0
    for e in range(len(offs) - 1):
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 == r0:
            continue
        a = acts[i].astype(np.float64)
        i += 1
        _, sb = O.mxfp8_quantize(acts[i - 1])
        X = np.repeat(np.exp2(sb.astype(np.float64) - 127.0), 32, axis=1)
        mag = np.abs(a) / X
        quantum = np.exp2(np.maximum(np.floor(np.log2(np.maximum(mag, 1e-300))), -6.0) - 3.0) * X
        allow[r0:r1] = quantum.max(axis=1)[:, None] * np.abs(w2[e]).max(axis=1)[None, :]
    return ref, allow


def _assert_a8_close(got, ref, allow, rows_min=2):
    """Within 1e-2 * RMS everywhere but on a few rows, and within that plus
    the one-flip allowance on those."""
    err = np.abs(np.asarray(got, np.float64) - ref)
    tight = tol(ref, 1e-2, 0.0)
    over = err > tight
    assert np.all(err <= tight + allow), float(np.max(err - tight - allow))
    n_rows = int(np.sum(np.any(over, axis=1)))
    assert n_rows <= max(rows_min, 0.005 * ref.shape[0]), (n_rows, ref.shape[0])


def _random_mx_problem(E, K, N, M, k, seed, scale_lo=(112, 110)):
    """Random e2m1 codes (all 16 values) under a spread of scale bytes, bf16
    tokens, distinct random experts per token; permuted on the host by the
    oracle."""
    g = torch.Generator().manual_seed(seed)
    p1 = torch.randint(0, 256, (E, 2 * N, K // 2), generator=g, dtype=torch.uint8)
    s1 = torch.randint(scale_lo[0], scale_lo[0] + 15, (E, 2 * N, K // 32), generator=g, dtype=torch.uint8)
    p2 = torch.randint(0, 256, (E, K, N // 2), generator=g, dtype=torch.uint8)
    s2 = torch.randint(scale_lo[1], scale_lo[1] + 15, (E, K, N // 32), generator=g, dtype=torch.uint8)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    ids = np.stack([np.random.default_rng(seed * 1000 + t).permutation(E)[:k] for t in range(M)]).astype(np.int32)
    return p1, s1, p2, s2, x, ids


def _a8_weights(moe, p1, s1, p2, s2, E, K, N, activation=0, clamp=None):
    d = dict(p1=p1.to(DEV), p2=p2.to(DEV))
    d["a1"] = torch.empty(moe.moe_mx_prepared_scales_size(E, 2 * N, K), dtype=torch.uint8, device=DEV)
    d["a2"] = torch.empty(moe.moe_mx_prepared_scales_size(E, K, N), dtype=torch.uint8, device=DEV)
    moe.moe_mx_prepare_scales(s1.to(DEV), E, 2 * N, K, d["a1"])
    moe.moe_mx_prepare_scales(s2.to(DEV), E, K, N, d["a2"])
    cw = moe.make_weights(moe.MOE_WEIGHTS_MXFP4_A8, E, K, N, d["p1"], d["p2"], d["a1"], d["a2"], activation, clamp)
    return cw, d


@pytest.mark.parametrize("E,K,N,M,k,bt,splits", [
    (4, 256, 128, 1, 1, 0, (0, 0)),           # one route
    (8, 512, 256, 37, 2, 0, (0, 0)),          # ragged tiles
    (8, 512, 384, 300, 2, 0, (0, 0)),         # three GEMM1 weight tiles
    (16, 1024, 256, 1000, 4, 0, (0, 0)),      # 128-row token tiles
    (8, 512, 256, 200, 2, 16, (3, 2)),        # 16-row tiles, split-K on both GEMMs
    (8, 512, 256, 200, 2, 32, (0, 0)),
    (8, 512, 256, 200, 2, 64, (2, 1)),
    (8, 768, 256, 90, 3, 128, (1, 3)),
])
def test_experts_a8_parity(moe, E, K, N, M, k, bt, splits):
    """gemm2_permuted (f32) of moe_experts with MXFP4_A8 weights against the
    oracle's experts_mxfp8 on the same codes and scales, every row; then the
    finalize of the same call (do_finalize = 1) and the finalize folded into
    GEMM2 (moe_experts_fused_finalize), every token."""
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=E * 7 + M)
    offs, pmap, inv, _ = O.permute(ids, E)
    R = int(offs[-1])
    xp = x[torch.from_numpy(inv.astype(np.int64) // k)]
    w = np.random.default_rng(M).uniform(0.1, 1.0, (M, k)).astype(np.float32)
    moe.moe_set_plan_override(bt, splits[0], splits[1], 0, 0)
    try:
        cw, keep = _a8_weights(moe, p1, s1, p2, s2, E, K, N)
        ws_n = moe.moe_experts_workspace_size(cw, M, k)
        ws = torch.zeros(ws_n, dtype=torch.uint8, device=DEV)
        g2 = torch.full((M * k, K), float("nan"), dtype=torch.float32, device=DEV)
        out = torch.empty(M, K, dtype=torch.float32, device=DEV)
        offs_d = torch.from_numpy(offs).to(DEV)
        pmap_d = torch.from_numpy(pmap.astype(np.int32)).to(DEV)
        inv_d = torch.from_numpy(inv.astype(np.int32)).to(DEV)
        w_d = torch.from_numpy(w).to(DEV)
        moe.moe_experts(cw, xp.to(DEV), offs_d, M, k, g2, moe.MOE_DTYPE_F32, 1, w_d, moe.MOE_DTYPE_F32, pmap_d,
                        None, 0, 1.0, out, moe.MOE_DTYPE_F32, ws, ws_n)
        fused = torch.empty(M, K, dtype=torch.float32, device=DEV)
        moe.moe_experts_fused_finalize(cw, xp.to(DEV), offs_d, M, k, w_d, moe.MOE_DTYPE_F32, inv_d, None, 0, 1.0,
                                       fused, ws, ws_n)
        # the same with a shared-expert output and a routed scale (the shared output is added after the scale)
        shared = torch.randn(M, K, generator=torch.Generator().manual_seed(M)).to(DEV)
        fused_sh = torch.empty(M, K, dtype=torch.float32, device=DEV)
        moe.moe_experts_fused_finalize(cw, xp.to(DEV), offs_d, M, k, w_d, moe.MOE_DTYPE_F32, inv_d, shared,
                                       moe.MOE_DTYPE_F32, 2.5, fused_sh, ws, ws_n)
        torch.cuda.synchronize()
        _check_no_error(moe)
    finally:
        moe.moe_set_plan_override(0, 0, 0, 0, 0)
    w1 = np.stack([O.dequant_mxfp4(p1[e].numpy(), s1[e].numpy()) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e].numpy(), s2[e].numpy()) for e in range(E)])
    ref, allow = _oracle_a8(x.double().numpy(), w1, w2, offs, inv, k)
    _assert_a8_close(g2[:R].double().cpu().numpy(), ref, allow)
    ref_out = O.finalize(ref, w.astype(np.float64), pmap)
    allow_out = O.finalize(allow, np.abs(w.astype(np.float64)), pmap)     # sum_j |w| * allowance
    _assert_a8_close(out.double().cpu().numpy(), ref_out, allow_out)
    _assert_a8_close(fused.double().cpu().numpy(), ref_out, allow_out)
    sh = shared.double().cpu().numpy()
    ref_sh = O.finalize(ref, w.astype(np.float64), pmap, sh, 2.5)
    _assert_a8_close(fused_sh.double().cpu().numpy() - sh, ref_sh - sh, 2.5 * allow_out)
    # the quantised path is not the unquantised one: its distance to the
    # W4A16 oracle is of the order of the E4M3 rounding (a few percent)
    ref16 = O.experts(x.double().numpy(), w1, w2, offs, inv, k)
    assert max_err(ref, ref16) > 1e-3 * tol(ref16, 1.0, 0.0)


def test_experts_a8_gelu_clamp(moe):
    """gelu_and_mul with the activation clamp in the quantising epilogue."""
    E, K, N, M, k = 8, 512, 256, 64, 2
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=91, scale_lo=(100, 110))
    offs, pmap, inv, _ = O.permute(ids, E)
    R = int(offs[-1])
    xp = x[torch.from_numpy(inv.astype(np.int64) // k)]
    cw, keep = _a8_weights(moe, p1, s1, p2, s2, E, K, N, activation=moe.MOE_ACT_GELU, clamp=3.0)
    ws_n = moe.moe_experts_workspace_size(cw, M, k)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device=DEV)
    g2 = torch.empty(M * k, K, dtype=torch.float32, device=DEV)
    moe.moe_experts(cw, xp.to(DEV), torch.from_numpy(offs).to(DEV), M, k, g2, moe.MOE_DTYPE_F32, 0, None, 0,
                    None, None, 0, 1.0, None, 0, ws, ws_n)
    torch.cuda.synchronize()
    _check_no_error(moe)
    w1 = np.stack([O.dequant_mxfp4(p1[e].numpy(), s1[e].numpy()) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e].numpy(), s2[e].numpy()) for e in range(E)])
    ref, allow = _oracle_a8(x.double().numpy(), w1, w2, offs, inv, k, activation="gelu", clamp=3.0)
    _assert_a8_close(g2[:R].double().cpu().numpy(), ref, allow)


def test_experts_a8_argument_checks(moe):
    E, K, N = 2, 128, 128                                   # K % 256 != 0
    p1, s1, p2, s2, _, _ = _random_mx_problem(E, 256, N, 1, 1, seed=3)
    cw, keep = _a8_weights(moe, p1, s1, p2, s2, E, 256, N)
    cw.K = K
    assert moe.moe_experts_workspace_size(cw, 4, 1) == 0
    cw.K = 256
    assert moe.moe_experts_workspace_size(cw, 4, 1) > 0
    assert moe.moe_experts_launches(cw, 4, 1, True) == 3     # quantiser, GEMM1 (+ output start), GEMM2
    assert moe.moe_experts_launches(cw, 4, 1, False) == 3
    ws = torch.zeros(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_experts_batched(cw, torch.zeros(E, 4, 256, dtype=torch.bfloat16, device=DEV),
                                torch.zeros(E, dtype=torch.int32, device=DEV), 4,
                                torch.zeros(E, 4, 256, dtype=torch.float32, device=DEV), moe.MOE_DTYPE_F32, ws, 16)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


# ------------------------------------------------------------------ the DeepSeek-shaped layer

@pytest.mark.parametrize("M", [1, 64, 1024])
def test_layer_deepseek_a8(moe, M):
    """The DeepSeek-V3-shaped layer with its MXFP4 routed experts on MXFP8
    activations: routing and map bit-exact over all tokens, outputs on a
    token sample against the oracle with the same activation quantisation."""
    _check_layer(moe, "deepseek", M, sample=8, a8=True, few_experts=True)


def test_experts_a8_offsets_not_starting_at_zero(moe):
    """Caller-built offsets whose first group starts past row 0: the grouped
    rows match the oracle's experts on those rows, and the rows outside every
    group (before the first, after the last) are left untouched."""
    E, K, N, k = 2, 256, 128, 1
    p1, s1, p2, s2, _, _ = _random_mx_problem(E, K, N, 1, 1, seed=17)
    rows = 10
    g = torch.Generator().manual_seed(18)
    xp = torch.randn(rows, K, generator=g).to(torch.bfloat16)
    offs = np.array([2, 5, 9], np.int32)
    cw, keep = _a8_weights(moe, p1, s1, p2, s2, E, K, N)
    ws_n = moe.moe_experts_workspace_size(cw, rows, k)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device=DEV)
    g2 = torch.full((rows, K), float("nan"), dtype=torch.float32, device=DEV)
    moe.moe_experts(cw, xp.to(DEV), torch.from_numpy(offs).to(DEV), rows, k, g2, moe.MOE_DTYPE_F32, 0, None, 0,
                    None, None, 0, 1.0, None, 0, ws, ws_n)
    torch.cuda.synchronize()
    _check_no_error(moe)
    got = g2.double().cpu().numpy()
    w1 = np.stack([O.dequant_mxfp4(p1[e].numpy(), s1[e].numpy()) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e].numpy(), s2[e].numpy()) for e in range(E)])
    # the same problem with its rows moved to start at 0: rows 2..8, identity inverse
    x = xp.double().numpy()[2:9]
    ref, allow = _oracle_a8(x, w1, w2, offs - 2, np.arange(7), 1)
    _assert_a8_close(got[2:9], ref, allow)
    assert np.isnan(got[:2]).all() and np.isnan(got[9:]).all()
