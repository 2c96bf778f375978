"""GPU parity of the MXFP4-weight experts with bf16 activations on the
block-scaled tensor cores (MOE_WEIGHTS_MXFP4_A16): every bf16 activation is
split into two E4M3 terms whose sum is the bf16 value, so the path computes
the W4A16 contraction of MOE_WEIGHTS_MXFP4 (flashinfer_moe_ep.py,
_dequant_fp4_ue8m0_gran32: e2m1 x 2^(s-127) weights; bf16 activations).

Bars: the split itself bit for bit against the oracle's e4m3_split; the
experts at the MXFP4 path's 3e-2 * RMS against the oracle on the same bytes;
and, since both formats compute the same products with float32 sums and round
the activation output to bf16 alike, an error against the oracle no larger
than the bf16-decode path's (MOE_WEIGHTS_MXFP4) on the same inputs, up to
1.5x + 5e-4 * RMS for the different float32 summation order inside the
tensor cores -- a lost lo term (about 2^-5 of each value) or a wrong scale
would be an order of magnitude above it.
"""
import numpy as np
import pytest
import torch

import oracle as O
from _helpers import lib, max_err, tol
from test_gpu_mx8 import _random_mx_problem
from test_gpu_parity import _check_layer, layer_inputs, make_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32 = 1


@pytest.fixture(scope="module")
def moe():
    m = lib()
    assert m.moe_device_check() == 0, "needs a compute capability 10.3 device"
    return m


def _check_no_error(moe):
    st = moe.moe_get_error()
    assert st == 0, moe.status_string(st)


def _as_accurate(got, decode, ref):
    """got's error against the oracle is that of the bf16-decode path's, up to
    1.5x + 5e-4 * RMS(ref)."""
    e_got, e_dec = max_err(got, ref), max_err(decode, ref)
    assert e_got <= 1.5 * e_dec + tol(ref, 5e-4, 0.0), (e_got, e_dec)


@pytest.mark.parametrize("rows,C", [(1, 128), (37, 384), (300, 1024), (9, 7168)])
def test_e4m3_split_bitexact(moe, rows, C):
    """moe_e4m3_split: hi and lo codes and their scale bytes equal the
    oracle's e4m3_split on rows spanning 2^-30 .. 2^30, with an all-zero row,
    a value swamping its block, bf16 subnormals and a block whose largest
    value would saturate under the plain MX scale."""
    g = torch.Generator().manual_seed(rows * 17 + C)
    x = torch.randn(rows, C, generator=g) * torch.exp(torch.empty(rows, 1).uniform_(-20, 20, generator=g))
    if rows >= 9:
        x[1] = 0.0
        x[2, 5] = 3.0e30
        x[3] = torch.randn(C, generator=g) * 1e-39
        x[4, :32] = torch.randn(32, generator=g)
        x[4, 7] = 1.875
    xb = x.to(torch.bfloat16)
    codes = torch.full((2 * rows, C), 0x55, dtype=torch.uint8, device=DEV)
    scales = torch.full((2 * rows, C // 32), 0x55, dtype=torch.uint8, device=DEV)
    moe.moe_e4m3_split(xb.to(DEV), rows, C, codes, scales)
    torch.cuda.synchronize()
    _check_no_error(moe)
    hi, b1, lo, b2 = O.e4m3_split(xb.float().numpy())
    c, sc = codes.cpu().numpy(), scales.cpu().numpy()
    assert np.array_equal(c[0::2], hi) and np.array_equal(c[1::2], lo)
    assert np.array_equal(sc[0::2], b1) and np.array_equal(sc[1::2], b2)


def _weights(moe, fmt, p1, s1, p2, s2, E, K, N, activation=0, clamp=None):
    d = dict(p1=p1.to(DEV), p2=p2.to(DEV))
    if fmt == moe.MOE_WEIGHTS_MXFP4:
        d["a1"], d["a2"] = s1.to(DEV), s2.to(DEV)
    else:
        d["a1"] = torch.empty(moe.moe_mx_prepared_scales_size(E, 2 * N, K), dtype=torch.uint8, device=DEV)
        d["a2"] = torch.empty(moe.moe_mx_prepared_scales_size(E, K, N), dtype=torch.uint8, device=DEV)
        moe.moe_mx_prepare_scales(s1.to(DEV), E, 2 * N, K, d["a1"])
        moe.moe_mx_prepare_scales(s2.to(DEV), E, K, N, d["a2"])
    return moe.make_weights(fmt, E, K, N, d["p1"], d["p2"], d["a1"], d["a2"], activation, clamp), d


def _run(moe, fmt, p1, s1, p2, s2, E, K, N, M, k, xp, offs, pmap, inv, w, activation=0, clamp=None):
    cw, keep = _weights(moe, fmt, p1, s1, p2, s2, E, K, N, activation, clamp)
    ws_n = moe.moe_experts_workspace_size(cw, M, k)
    ws = torch.zeros(ws_n, dtype=torch.uint8, device=DEV)
    g2 = torch.full((M * k, K), float("nan"), dtype=torch.float32, device=DEV)
    out = torch.empty(M, K, dtype=torch.float32, device=DEV)
    offs_d = torch.from_numpy(offs).to(DEV)
    pmap_d = torch.from_numpy(pmap.astype(np.int32)).to(DEV)
    inv_d = torch.from_numpy(inv.astype(np.int32)).to(DEV)
    w_d = torch.from_numpy(w).to(DEV)
    moe.moe_experts(cw, xp.to(DEV), offs_d, M, k, g2, F32, 1, w_d, F32, pmap_d, None, 0, 1.0, out, F32, ws, ws_n)
    fused = torch.empty(M, K, dtype=torch.float32, device=DEV)
    moe.moe_experts_fused_finalize(cw, xp.to(DEV), offs_d, M, k, w_d, F32, inv_d, None, 0, 1.0, fused, ws, ws_n)
    torch.cuda.synchronize()
    _check_no_error(moe)
    return g2, out, fused


@pytest.mark.parametrize("E,K,N,M,k,bt,splits", [
    (4, 512, 512, 1, 1, 0, (0, 0)),           # one route
    (8, 512, 512, 37, 2, 0, (0, 0)),          # ragged tiles
    (8, 1024, 512, 300, 2, 0, (0, 0)),        # several GEMM2 weight tiles
    (16, 1024, 512, 1000, 4, 0, (0, 0)),      # 64-token (128-row) tiles
    (8, 512, 512, 200, 2, 16, (3, 2)),        # 16-token tiles, split-K on both GEMMs
    (8, 512, 512, 200, 2, 32, (0, 0)),
    (8, 512, 512, 200, 2, 64, (2, 1)),
])
def test_experts_a16_parity(moe, E, K, N, M, k, bt, splits):
    """gemm2_permuted (f32), the finalize (do_finalize = 1) and the finalize
    folded into GEMM2: against the W4A16 oracle on the same codes and scales,
    and against the bf16-decode path on the same inputs."""
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=E * 11 + M)
    offs, pmap, inv, _ = O.permute(ids, E)
    R = int(offs[-1])
    xp = x[torch.from_numpy(inv.astype(np.int64) // k)]
    w = np.random.default_rng(M).uniform(0.1, 1.0, (M, k)).astype(np.float32)
    moe.moe_set_plan_override(bt, splits[0], splits[1], 0, 0)
    try:
        g2, out, fused = _run(moe, moe.MOE_WEIGHTS_MXFP4_A16, p1, s1, p2, s2, E, K, N, M, k, xp, offs, pmap, inv, w)
    finally:
        moe.moe_set_plan_override(0, 0, 0, 0, 0)
    g2d, outd, _ = _run(moe, moe.MOE_WEIGHTS_MXFP4, p1, s1, p2, s2, E, K, N, M, k, xp, offs, pmap, inv, w)
    w1 = np.stack([O.dequant_mxfp4(p1[e].numpy(), s1[e].numpy()) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e].numpy(), s2[e].numpy()) for e in range(E)])
    ref = O.experts(x.double().numpy(), w1, w2, offs, inv, k)
    got = g2[:R].double().cpu().numpy()
    assert max_err(got, ref) <= tol(ref, 3e-2, 0.0)
    _as_accurate(got, g2d[:R].double().cpu().numpy(), ref)
    ref_out = O.finalize(ref, w.astype(np.float64), pmap)
    for o in (out, fused):
        assert max_err(o.double().cpu().numpy(), ref_out) <= tol(ref_out, 3e-2, 0.0)
        _as_accurate(o.double().cpu().numpy(), outd.double().cpu().numpy(), ref_out)


def test_experts_a16_gelu_clamp(moe):
    """gelu_and_mul with the activation clamp in the splitting epilogue."""
    E, K, N, M, k = 8, 512, 512, 64, 2
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=93, scale_lo=(100, 110))
    offs, pmap, inv, _ = O.permute(ids, E)
    R = int(offs[-1])
    xp = x[torch.from_numpy(inv.astype(np.int64) // k)]
    w = np.ones((M, k), np.float32)
    g2, _, _ = _run(moe, moe.MOE_WEIGHTS_MXFP4_A16, p1, s1, p2, s2, E, K, N, M, k, xp, offs, pmap, inv, w,
                    activation=moe.MOE_ACT_GELU, clamp=3.0)
    w1 = np.stack([O.dequant_mxfp4(p1[e].numpy(), s1[e].numpy()) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e].numpy(), s2[e].numpy()) for e in range(E)])
    ref = O.experts(x.double().numpy(), w1, w2, offs, inv, k, activation="gelu", clamp=3.0)
    assert max_err(g2[:R].double().cpu().numpy(), ref) <= tol(ref, 3e-2, 0.0)


def test_experts_a16_tiny_and_huge_activations(moe):
    """Rows spanning 2^-30 .. 2^30 in magnitude, a block holding one value
    2^20 times its neighbours, and all-zero rows: the two-term split keeps
    every row at the decode path's result (within 5e-3 of each row's own
    RMS; exactly zero for the zero row)."""
    E, K, N, M, k = 4, 512, 512, 24, 1
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=5)
    xf = x.float() * torch.exp2(torch.linspace(-30, 30, M))[:, None]
    xf[3] = 0.0
    xf[5, 7] = 2.0 ** 20
    xb = xf.to(torch.bfloat16)
    offs, pmap, inv, _ = O.permute(ids, E)
    xp = xb[torch.from_numpy(inv.astype(np.int64) // k)]
    w = np.ones((M, k), np.float32)
    g2, _, _ = _run(moe, moe.MOE_WEIGHTS_MXFP4_A16, p1, s1, p2, s2, E, K, N, M, k, xp, offs, pmap, inv, w)
    g2d, _, _ = _run(moe, moe.MOE_WEIGHTS_MXFP4, p1, s1, p2, s2, E, K, N, M, k, xp, offs, pmap, inv, w)
    a, b = g2[:M].double().cpu().numpy(), g2d[:M].double().cpu().numpy()
    for r in range(M):
        rms = float(np.sqrt(np.mean(b[r] ** 2)))
        assert np.all(np.abs(a[r] - b[r]) <= 5e-3 * rms + 1e-30), r


@pytest.mark.parametrize("M", [1, 64, 1024, 8192])
def test_layer_deepseek_a16(moe, M):
    """The DeepSeek-V3-shaped layer with its MXFP4 routed experts on bf16
    activations through the block-scaled MMAs: routing and map bit-exact over
    all tokens, outputs on a sample reaching every touched expert against the
    W4A16 oracle (3e-2 * RMS)."""
    _check_layer(moe, "deepseek", M, a16=True)


@pytest.mark.parametrize("M", [64, 1024])
def test_layer_deepseek_a16_equals_decode_path(moe, M):
    """The same layer forward with MXFP4_A16 and with the bf16-decode MXFP4
    format: every output value of every token within 5e-3 * RMS. The two
    compute the same products and round the activation output to bf16 alike;
    what differs is the float32 summation order inside the tensor cores (and
    the rare bf16 rounding flip of an activation it causes), far below the
    ~2 % a lost lo term or a wrong block scale would cause."""
    import synth
    cfg = synth.CONFIGS["deepseek"]
    li = layer_inputs("deepseek")
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    outs = []
    for fmt in (moe.MOE_WEIGHTS_MXFP4_A16, moe.MOE_WEIGHTS_MXFP4):
        lay = make_layer(moe, "deepseek", li, fmt=fmt, fused_finalize=True)
        outs.append(lay.forward(x, logits).out.double().clone())
        del lay
    torch.cuda.synchronize()
    _check_no_error(moe)
    a, b = outs[0].cpu().numpy(), outs[1].cpu().numpy()
    assert max_err(a, b) <= 5e-3 * float(np.sqrt(np.mean(b ** 2)))


_X_PLANS = {
    # automatic plan
    "auto": (None, 96),
    # two one-CTA launches, GEMM1 split in two along K (several token tiles
    # per expert and ragged tails)
    "two_split": ((0, 2, 1, 0, 2), 700),
    # the same with 16-token tiles
    "two_t16": ((16, 1, 1, 0, 2), 300),
    # CTA pairs (bf16)
    "pairs": ((128, 0, 0, 0, 3), 700),
}


@pytest.mark.parametrize("plan", list(_X_PLANS))
@pytest.mark.parametrize("fmt_name", ["MOE_WEIGHTS_MXFP4_A16", "MOE_WEIGHTS_MXFP4_A8", "MOE_WEIGHTS_MXFP4",
                                      "MOE_WEIGHTS_BF16"])
def test_fused_finalize_x_gathers_rows(moe, fmt_name, plan):
    """moe_experts_fused_finalize_x (x in token order, rows gathered through
    permuted_to_expanded inside the experts) equals moe_experts_fused_finalize
    on x_perm under the same launch plan up to the order of the folded
    finalize's float32 additions (1e-4 * RMS), on every weight format; an
    out-of-range inverse entry is reported as MOE_ERR_DEVICE_INDEX and leaves
    the output finite."""
    fmt = getattr(moe, fmt_name)
    override, M = _X_PLANS[plan]
    if plan != "auto" and fmt in (moe.MOE_WEIGHTS_MXFP4_A16, moe.MOE_WEIGHTS_MXFP4_A8):
        pytest.skip("the block-scaled formats have one launch plan")
    if plan == "pairs" and fmt != moe.MOE_WEIGHTS_BF16:
        pytest.skip("CTA pairs run bf16 weights")
    if override is not None:
        moe.moe_set_plan_override(*override)
    try:
        _fused_finalize_x_case(moe, fmt, M)
    finally:
        moe.moe_set_plan_override(0, 0, 0, 0, 0)


def _fused_finalize_x_case(moe, fmt, M):
    E, K, N, k = 8, 512, 512, 2
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=77)
    if fmt == moe.MOE_WEIGHTS_BF16:
        g = torch.Generator().manual_seed(78)
        p1 = (torch.randn(E, 2 * N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
        p2 = (torch.randn(E, K, N, generator=g) / N ** 0.5).to(torch.bfloat16)
    offs, pmap, inv, _ = O.permute(ids, E)
    xp = x[torch.from_numpy(inv.astype(np.int64) // k)]
    w = np.random.default_rng(9).uniform(0.1, 1.0, (M, k)).astype(np.float32)
    if fmt == moe.MOE_WEIGHTS_BF16:
        d = dict(p1=p1.to(DEV), p2=p2.to(DEV))
        cw = moe.make_weights(fmt, E, K, N, d["p1"], d["p2"])
    else:
        cw, d = _weights(moe, fmt, p1, s1, p2, s2, E, K, N)
    n = max(moe.moe_experts_workspace_size(cw, M, k), moe.moe_experts_x_workspace_size(cw, M, k))
    assert moe.moe_experts_x_workspace_size(cw, M, k) >= moe.moe_experts_workspace_size(cw, M, k)
    ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
    offs_d = torch.from_numpy(offs).to(DEV)
    inv_d = torch.from_numpy(inv.astype(np.int32)).to(DEV)
    w_d = torch.from_numpy(w).to(DEV)
    xd = x.to(DEV)
    ref = torch.empty(M, K, dtype=torch.float32, device=DEV)
    moe.moe_experts_fused_finalize(cw, xp.to(DEV), offs_d, M, k, w_d, F32, inv_d, None, F32, 1.0, ref, ws, n)
    got = torch.empty(M, K, dtype=torch.float32, device=DEV)
    moe.moe_experts_fused_finalize_x(cw, xd, offs_d, M, k, w_d, F32, inv_d, None, F32, 1.0, got, ws, n)
    torch.cuda.synchronize()
    _check_no_error(moe)
    rms = float(ref.pow(2).mean().sqrt())
    assert float((got - ref).abs().max()) <= 1e-4 * rms
    bad = inv_d.clone()
    bad[3] = 10 ** 7
    moe.moe_experts_fused_finalize_x(cw, xd, offs_d, M, k, w_d, F32, bad, None, F32, 1.0, got, ws, n)
    torch.cuda.synchronize()
    assert moe.moe_get_error() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_error() == 0
    assert torch.isfinite(got).all()


_AFTER_PLANS = {"auto": None, "two": (0, 0, 0, 0, 2), "pairs": (128, 0, 0, 0, 3), "fused": (0, 0, 0, 0, 1)}


@pytest.mark.parametrize("plan", list(_AFTER_PLANS))
@pytest.mark.parametrize("x_order", [0, 1])
@pytest.mark.parametrize("fmt_name", ["MOE_WEIGHTS_MXFP4_A16", "MOE_WEIGHTS_MXFP4_A8", "MOE_WEIGHTS_MXFP4",
                                      "MOE_WEIGHTS_BF16"])
def test_fused_finalize_after_adds_into_a_preset_start(moe, fmt_name, x_order, plan):
    """moe_experts_fused_finalize_after: out holds a start written on a
    second stream after a long wait there (the event is what orders it),
    and the routed sum is added into it. Equal to moe_experts_fused_finalize
    with shared_out = the start (f32) up to the order of the f32 additions
    (1e-5 * RMS), for x_perm (x_order 0) and token order (1), on every weight
    format and, for bf16, on each plan (one fused launch, two launches, CTA
    pairs: the wait sits before a different launch in each). A NULL event
    with the start written on the same stream gives the same."""
    fmt = getattr(moe, fmt_name)
    override = _AFTER_PLANS[plan]
    if plan != "auto" and fmt != moe.MOE_WEIGHTS_BF16:
        pytest.skip("plan overrides are exercised on bf16 weights")
    E, K, N, M, k = 8, 512, 512, 300, 2
    p1, s1, p2, s2, x, ids = _random_mx_problem(E, K, N, M, k, seed=91)
    if fmt == moe.MOE_WEIGHTS_BF16:
        g = torch.Generator().manual_seed(92)
        p1 = (torch.randn(E, 2 * N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
        p2 = (torch.randn(E, K, N, generator=g) / N ** 0.5).to(torch.bfloat16)
        d = dict(p1=p1.to(DEV), p2=p2.to(DEV))
        cw = moe.make_weights(fmt, E, K, N, d["p1"], d["p2"])
    else:
        cw, d = _weights(moe, fmt, p1, s1, p2, s2, E, K, N)
    offs, pmap, inv, _ = O.permute(ids, E)
    xp = x[torch.from_numpy(inv.astype(np.int64) // k)]
    w = np.random.default_rng(93).uniform(0.1, 1.0, (M, k)).astype(np.float32)
    start = (torch.randn(M, K, generator=torch.Generator().manual_seed(94)) * 0.7).to(DEV)
    offs_d = torch.from_numpy(offs).to(DEV)
    inv_d = torch.from_numpy(inv.astype(np.int32)).to(DEV)
    w_d = torch.from_numpy(w).to(DEV)
    xin = (x if x_order else xp).to(DEV)
    if override is not None:
        moe.moe_set_plan_override(*override)
    try:
        n = max(moe.moe_experts_workspace_size(cw, M, k), moe.moe_experts_x_workspace_size(cw, M, k))
        ws = torch.zeros(n, dtype=torch.uint8, device=DEV)
        ref = torch.empty(M, K, dtype=torch.float32, device=DEV)
        moe.moe_experts_fused_finalize(cw, xp.to(DEV), offs_d, M, k, w_d, F32, inv_d, start, F32, 1.5, ref, ws, n)
        torch.cuda.synchronize()
        # the start, written on a second stream after a long wait there
        got = torch.full((M, K), float("nan"), device=DEV)
        side, ev = torch.cuda.Stream(), torch.cuda.Event()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            torch.cuda._sleep(20_000_000)
            got.copy_(start)
        ev.record(side)
        moe.moe_experts_fused_finalize_after(cw, xin, x_order, offs_d, M, k, w_d, F32, inv_d, 1.5, got, ev, ws, n)
        # the start on the same stream, no event
        got2 = start.clone()
        moe.moe_experts_fused_finalize_after(cw, xin, x_order, offs_d, M, k, w_d, F32, inv_d, 1.5, got2, None,
                                             ws, n)
        torch.cuda.synchronize()
        _check_no_error(moe)
    finally:
        moe.moe_set_plan_override(0, 0, 0, 0, 0)
    rms = float(ref.pow(2).mean().sqrt())
    assert float((got - ref).abs().max()) <= 1e-5 * rms
    assert float((got2 - ref).abs().max()) <= 1e-5 * rms


@pytest.mark.parametrize("M", [1, 64, 1024])
def test_layer_shared_expert_overlap_equals_serial(moe, M):
    """The DeepSeek-shaped layer (A16 routed experts, bf16 shared expert)
    with the shared expert on a second stream writing the output start
    (MoELayer's default with the folded finalize) equals the same layer with
    the shared expert first on the one stream, up to the order of the f32
    additions (1e-5 * RMS); routing and map are the same bits."""
    import synth
    cfg = synth.CONFIGS["deepseek"]
    li = layer_inputs("deepseek")
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    res = []
    for ov in (True, False):
        lay = make_layer(moe, "deepseek", li, fmt=moe.MOE_WEIGHTS_MXFP4_A16, fused_finalize=True,
                         overlap_shared=ov)
        assert lay.overlap_shared == ov
        b = lay.forward(x, logits)
        res.append((b.out.clone(), b.topk_ids.clone(), b.pmap.clone()))
        del lay
    torch.cuda.synchronize()
    _check_no_error(moe)
    (o1, i1, p1), (o2, i2, p2) = res
    assert torch.equal(i1, i2) and torch.equal(p1, p2)
    rms = float(o2.pow(2).mean().sqrt())
    assert float((o1 - o2).abs().max()) <= 1e-5 * rms
