"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer results (routing ids, permute map, offsets, inverse map, the gathered
rows) must match bit for bit; values must satisfy
    max |gpu - oracle| <= 1e-2 * RMS(oracle) + 1e-3
with routing weights, gemm2_permuted and the output stored as float32 (the
bf16-activation pipeline: bf16 x, weights and act, fp32 accumulation). With
the pages' bf16 storage of those three tensors the bar is the same plus the
rounding bound of each stored bf16 value (unit roundoff 2^-8): that of the
output, and that of the two bf16 factors of every weighted route the
finalize adds (the stored dtype's own rounding is not an error of the
computation).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from _helpers import (ExpertsF64, lib, max_err, oracle_tokens, oracle_tokens_mxfp4, sample_tokens,
                      sample_tokens_covering, sample_tokens_few_experts, tol)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    m = lib()
    assert m.moe_device_check() == 0, "needs a compute capability 10.3 device"
    return m


_LAYERS = {}


def layer_inputs(name):
    if name not in _LAYERS:
        _LAYERS.clear()
        torch.cuda.empty_cache()
        _LAYERS[name] = synth.make_layer(synth.CONFIGS[name], DEV)
    return _LAYERS[name]


def make_layer(moe, name, li, **kw):
    cfg = li.cfg
    args = dict(K=cfg.K, N=cfg.N, E=cfg.E, top_k=cfg.top_k, w1=li.w1, w2=li.w2,
                w1_scale=li.w1_scale, w2_scale=li.w2_scale,
                fmt=moe.MOE_WEIGHTS_MXFP4 if cfg.weight_format == "mxfp4" else moe.MOE_WEIGHTS_BF16,
                route="softmax" if cfg.route == "softmax" else "sigmoid",
                score_bias=li.score_bias, n_group=cfg.n_group, topk_group=cfg.topk_group,
                routed_scaling_factor=cfg.routed_scaling_factor, ws1=li.ws1, ws2=li.ws2)
    args.update(kw)
    return moe.MoELayer(**args)


def check_no_device_error(moe):
    st = moe.moe_get_error()
    assert st == 0, moe.status_string(st)


# ------------------------------------------------------------------ sigmoid spec

def test_sigmoid_spec_bitexact(moe):
    x = np.concatenate([np.linspace(-100, 100, 200001),
                        np.random.default_rng(0).standard_normal(100000) * 4,
                        [0.0, -0.0, 88.0, -88.0, 80.0, -80.0, 87.99, -79.99]]).astype(np.float32)
    xd = torch.from_numpy(x).to(DEV)
    y = torch.empty_like(xd)
    moe.moe_debug_sigmoid(xd, y, x.size)
    got = y.cpu().numpy()
    want = O.sigmoid_f32_spec(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("name,M", [("tiny", 16), ("mixtral", 8192), ("qwen3", 8192), ("qwen3", 1),
                                    ("mixtral", 3)])
def test_router_softmax(moe, name, M):
    cfg = synth.CONFIGS[name]
    li = synth.make_layer(cfg, "cpu", experts=[]) if cfg.logit_bias_std else None
    _, logits = synth.make_tokens(cfg, M, DEV, li)
    ids = torch.empty(M, cfg.top_k, dtype=torch.int32, device=DEV)
    for wdt, tdt in ((moe.MOE_DTYPE_F32, torch.float32), (moe.MOE_DTYPE_BF16, torch.bfloat16)):
        w = torch.empty(M, cfg.top_k, dtype=tdt, device=DEV)
        moe.moe_route(logits, M, cfg.E, cfg.top_k, moe.MOE_ROUTE_SOFTMAX_TOPK, None, 1, 1, 1.0, ids, w, wdt)
        rid, rw = O.route_softmax_topk(logits.cpu().numpy(), cfg.top_k)
        assert np.array_equal(ids.cpu().numpy(), rid)
        got = w.float().cpu().numpy()
        if wdt == moe.MOE_DTYPE_F32:
            np.testing.assert_allclose(got, rw, rtol=2e-6, atol=1e-7)
        else:
            np.testing.assert_allclose(got, O.bf16_round(rw), rtol=2 ** -8, atol=0)
    check_no_device_error(moe)


@pytest.mark.parametrize("M", [1, 64, 8192])
def test_router_sigmoid_grouped(moe, M):
    cfg = synth.CONFIGS["deepseek"]
    li = synth.make_layer(cfg, "cpu", experts=[])
    _, logits = synth.make_tokens(cfg, M, DEV)
    bias = li.score_bias.to(DEV)
    ids = torch.empty(M, cfg.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(M, cfg.top_k, dtype=torch.float32, device=DEV)
    moe.moe_route(logits, M, cfg.E, cfg.top_k, moe.MOE_ROUTE_SIGMOID_GROUPED_TOPK, bias, cfg.n_group,
                  cfg.topk_group, cfg.routed_scaling_factor, ids, w, moe.MOE_DTYPE_F32)
    rid, rw = O.route_sigmoid_grouped(logits.cpu().numpy(), li.score_bias.numpy(), cfg.top_k, cfg.n_group,
                                      cfg.topk_group, cfg.routed_scaling_factor)
    assert np.array_equal(ids.cpu().numpy(), rid)
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=5e-6, atol=1e-7)
    check_no_device_error(moe)


def test_router_ties_lower_id_first(moe):
    logits = torch.tensor([[0.5, 1.0, 1.0, -2.0, 1.0, 0.0, 1.0, -0.0]] * 3, device=DEV)
    ids = torch.empty(3, 3, dtype=torch.int32, device=DEV)
    w = torch.empty(3, 3, dtype=torch.float32, device=DEV)
    moe.moe_route(logits, 3, 8, 3, moe.MOE_ROUTE_SOFTMAX_TOPK, None, 1, 1, 1.0, ids, w, moe.MOE_DTYPE_F32)
    assert ids.cpu().tolist() == [[1, 2, 4]] * 3


# ------------------------------------------------------------------ permute

def _permute(moe, ids_np, E, K, emap=None, E_l=None, x=None):
    M, k = ids_np.shape
    E_l = E if E_l is None else E_l
    ids = torch.from_numpy(ids_np).to(DEV)
    if x is None:
        x = torch.randn(M, K, device=DEV).to(torch.bfloat16)
    offs = torch.empty(E_l + 1, dtype=torch.int32, device=DEV)
    pmap = torch.empty(M, k, dtype=torch.int32, device=DEV)
    inv = torch.full((max(M * k, 1),), -7, dtype=torch.int32, device=DEV)
    xp = torch.zeros(max(M * k, 1), K, dtype=torch.bfloat16, device=DEV)
    wsb = moe.moe_permute_workspace_size(M, k, E_l)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    em = None if emap is None else torch.from_numpy(np.asarray(emap, np.int32)).to(DEV)
    moe.moe_permute(ids, M, k, E, em, E_l, x, K, offs, pmap, inv, xp, ws, ws.numel())
    return x, offs.cpu().numpy(), pmap.cpu().numpy(), inv.cpu().numpy(), xp


@pytest.mark.parametrize("name,M,masked", [("tiny", 16, False), ("mixtral", 1, False), ("mixtral", 8192, False),
                                           ("qwen3", 8192, False), ("qwen3", 4096, True), ("qwen3", 33, True),
                                           ("deepseek", 1024, False)])
def test_permute_bitexact(moe, name, M, masked):
    cfg = synth.CONFIGS[name]
    rng = np.random.default_rng(M)
    ids = np.stack([rng.permutation(cfg.E)[:cfg.top_k] for _ in range(M)]).astype(np.int32)
    if name == "qwen3":    # heavy-tailed load: route with the skewed logits
        li = synth.make_layer(cfg, "cpu", experts=[])
        _, logits = synth.make_tokens(cfg, M, "cpu", li)
        ids, _ = O.route_softmax_topk(logits.numpy(), cfg.top_k)
    emap, E_l = (None, cfg.E)
    if masked:
        em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
        emap = em.numpy()
    K = min(cfg.K, 1024)
    x, offs, pmap, inv, xp = _permute(moe, ids, cfg.E, K, emap, E_l)
    r_offs, r_map, r_inv, _ = O.permute(ids, cfg.E, emap)
    assert np.array_equal(offs, r_offs)
    assert np.array_equal(pmap, r_map)
    R = int(r_offs[-1])
    assert np.array_equal(inv[:R], r_inv)
    tok = torch.from_numpy(r_inv.astype(np.int64) // cfg.top_k).to(DEV)
    assert torch.equal(xp[:R], x[tok])                         # gathered rows, bitwise
    check_no_device_error(moe)


def test_permute_empty_and_all_masked(moe):
    offs = torch.full((9,), 5, dtype=torch.int32, device=DEV)
    moe.moe_permute(None, 0, 2, 8, None, 8, None, 128, offs, None, None, None, None, 0)
    assert offs.cpu().tolist() == [0] * 9
    ids = np.array([[0, 1], [1, 0]], np.int32)
    x, offs, pmap, inv, xp = _permute(moe, ids, 4, 128, emap=np.array([-1, -1, 0, 1], np.int32), E_l=2)
    assert offs.tolist() == [0, 0, 0] and (pmap == -1).all()


def test_permute_bad_ids_set_device_error(moe):
    ids = np.array([[0, 1], [9, 2], [3, -1]], np.int32)        # 9 and -1 are out of range for E = 8
    _, offs, pmap, inv, _ = _permute(moe, ids, 8, 128)
    assert moe.moe_get_error() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_error() == 0                            # cleared by the read
    assert pmap[1, 0] == -1 and pmap[2, 1] == -1               # skipped like non-local routes
    assert offs[-1] == 4


# ------------------------------------------------------------------ route + permute

def _route_permute(moe, cfg, li, logits, x, M, emap, E_l, wdt, fused):
    k, K = cfg.top_k, x.shape[1]
    sig = cfg.route != "softmax"
    method = moe.MOE_ROUTE_SIGMOID_GROUPED_TOPK if sig else moe.MOE_ROUTE_SOFTMAX_TOPK
    bias = li.score_bias.to(DEV) if sig else None
    rsf = cfg.routed_scaling_factor if sig else 1.0
    tdt = torch.float32 if wdt == moe.MOE_DTYPE_F32 else torch.bfloat16
    fill = 3 if fused else 5
    ids = torch.full((M, k), fill, dtype=torch.int32, device=DEV)
    w = torch.full((M, k), float(fill), dtype=tdt, device=DEV)
    offs = torch.full((E_l + 1,), fill, dtype=torch.int32, device=DEV)
    pmap = torch.full((M, k), fill, dtype=torch.int32, device=DEV)
    inv = torch.full((max(M * k, 1),), fill, dtype=torch.int32, device=DEV)
    xp = torch.full((max(M * k, 1), K), float(fill), dtype=torch.bfloat16, device=DEV)
    wsb = moe.moe_permute_workspace_size(M, k, E_l)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    em = None if emap is None else torch.from_numpy(np.asarray(emap, np.int32)).to(DEV)
    if fused:
        moe.moe_route_permute(logits, M, cfg.E, k, method, bias, cfg.n_group, cfg.topk_group, rsf, ids, w, wdt,
                              em, E_l, x, K, offs, pmap, inv, xp, ws, ws.numel())
    else:
        moe.moe_route(logits, M, cfg.E, k, method, bias, cfg.n_group, cfg.topk_group, rsf, ids, w, wdt)
        moe.moe_permute(ids, M, k, cfg.E, em, E_l, x, K, offs, pmap, inv, xp, ws, ws.numel())
    R = int(offs[-1])
    return ids, w, offs, pmap, inv[:R], xp[:R]


@pytest.mark.parametrize("name,M,masked", [("tiny", 16, False), ("mixtral", 1, False), ("mixtral", 8, False),
                                           ("mixtral", 64, False), ("qwen3", 1, False), ("qwen3", 32, True),
                                           ("qwen3", 64, False), ("deepseek", 1, False), ("deepseek", 64, True),
                                           ("mixtral", 65, False), ("qwen3", 4096, True), ("deepseek", 512, False)])
def test_route_permute_matches_two_calls(moe, name, M, masked):
    """moe_route_permute (one kernel for M <= 64, else the two launches) gives
    the results of moe_route followed by moe_permute, bit for bit."""
    cfg = synth.CONFIGS[name]
    li = synth.make_layer(cfg, "cpu", experts=[])
    x, logits = synth.make_tokens(cfg, M, DEV, li if cfg.logit_bias_std else None)
    x = x[:, :1024].contiguous()
    emap, E_l = None, cfg.E
    if masked:
        em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
        emap = em.numpy()
    for wdt in (moe.MOE_DTYPE_F32, moe.MOE_DTYPE_BF16):
        a = _route_permute(moe, cfg, li, logits, x, M, emap, E_l, wdt, fused=False)
        b = _route_permute(moe, cfg, li, logits, x, M, emap, E_l, wdt, fused=True)
        for u, v in zip(a, b):
            assert u.shape == v.shape and torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u,
                                                      v.view(torch.int16) if v.dtype == torch.bfloat16 else v)
    # and the ids are the oracle's
    if cfg.route == "softmax":
        rid, _ = O.route_softmax_topk(logits.cpu().numpy(), cfg.top_k)
    else:
        rid, _ = O.route_sigmoid_grouped(logits.cpu().numpy(), li.score_bias.numpy(), cfg.top_k, cfg.n_group,
                                         cfg.topk_group, cfg.routed_scaling_factor)
    assert np.array_equal(b[0].cpu().numpy(), rid)
    r_offs, r_map, _, _ = O.permute(rid, cfg.E, emap)
    assert np.array_equal(b[2].cpu().numpy(), r_offs) and np.array_equal(b[3].cpu().numpy(), r_map)
    check_no_device_error(moe)


# ------------------------------------------------------------------ failure detection

def test_bounded_wait_gives_up_and_reports(moe):
    """A wait on a flag that nothing sets runs out after its limit: the kernel
    returns, the error word reads MOE_ERR_DEVICE_TIMEOUT, and the context stays
    usable (the next calls run and report no error)."""
    import time
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_debug_bounded_wait(flag, 1, 50_000_000)                  # 50 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert moe.moe_get_error() == moe.MOE_ERR_DEVICE_TIMEOUT
    assert moe.moe_get_error() == 0                                 # cleared by the read
    assert 0.04 <= dt < 5.0
    flag.fill_(1)                                                   # satisfied: returns at once
    moe.moe_debug_bounded_wait(flag, 1, 50_000_000)
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    with pytest.raises(moe.MoEError):
        moe.moe_debug_bounded_wait(flag, 1, 0)
    x = torch.linspace(-5, 5, 101, device=DEV)
    y = torch.empty_like(x)
    moe.moe_debug_sigmoid(x, y, x.numel())
    torch.cuda.synchronize()
    assert torch.isfinite(y).all() and moe.moe_get_error() == 0


# ------------------------------------------------------------------ whole layer

def _check_layer(moe, name, M, sample=None, masked=False, bf16_storage=False, seed_offset=0, fused_finalize=False,
                 activation="silu", clamp=None, a8=False, few_experts=False, a16=False):
    cfg = synth.CONFIGS[name]
    li = layer_inputs(name)
    x, logits = synth.make_tokens(cfg, M, DEV, li, seed_offset=seed_offset)
    kw = {}
    emap_np = None
    if masked:
        em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
        emap_np = em.numpy()
        keep = torch.from_numpy(np.nonzero(emap_np >= 0)[0]).to(DEV)
        kw = dict(expert_map=em.to(DEV), E_local=E_l, w1=li.w1[keep].contiguous(), w2=li.w2[keep].contiguous())
        if li.w1_scale is not None:
            kw.update(w1_scale=li.w1_scale[keep].contiguous(), w2_scale=li.w2_scale[keep].contiguous())
    if bf16_storage:
        kw.update(weights_dtype=moe.MOE_DTYPE_BF16, gemm2_dtype=moe.MOE_DTYPE_BF16, out_dtype=moe.MOE_DTYPE_BF16)
    if fused_finalize:
        kw.update(fused_finalize=True)
    if activation != "silu" or clamp is not None:
        kw.update(activation=activation, activation_clamp=clamp)
    if a8:                        # MXFP4 weights x MXFP8 activations (block-scaled MMAs)
        kw.update(fmt=moe.MOE_WEIGHTS_MXFP4_A8)
    if a16:                       # MXFP4 weights x bf16 activations as two E4M3 terms (block-scaled MMAs)
        kw.update(fmt=moe.MOE_WEIGHTS_MXFP4_A16)
    layer = make_layer(moe, name, li, **kw)
    b = layer.forward(x, logits)
    torch.cuda.synchronize()
    check_no_device_error(moe)

    # routing and permute: bit-exact over all M tokens
    lg = logits.cpu().numpy()
    if cfg.route == "softmax":
        rid, rw = O.route_softmax_topk(lg, cfg.top_k)
    else:
        rid, rw = O.route_sigmoid_grouped(lg, li.score_bias.cpu().numpy(), cfg.top_k, cfg.n_group,
                                          cfg.topk_group, cfg.routed_scaling_factor)
    assert np.array_equal(b.topk_ids.cpu().numpy(), rid)
    r_offs, r_map, r_inv, _ = O.permute(rid, cfg.E, emap_np)
    assert np.array_equal(b.offsets.cpu().numpy(), r_offs)
    assert np.array_equal(b.pmap.cpu().numpy(), r_map)

    # values on a token sample (all tokens when M <= sample size). MXFP4
    # experts: the sample covers every expert that any of the M tokens routes
    # to, with at least `sample` (default 256) tokens; the oracle dequantises
    # each of those experts once, in a pool of CPU workers.
    cover = cfg.weight_format == "mxfp4" and not few_experts
    if cover:
        toks = sample_tokens_covering(rid, sample or 256, emap_np, seed=M)
    elif cfg.weight_format == "mxfp4":
        toks = sample_tokens_few_experts(rid, sample or 16, budget=48, seed=M)
    else:
        toks = sample_tokens(M, sample or 256)
    xs = x.to(torch.float64).cpu().numpy()
    shared = None
    if li.ws1 is not None:
        shared = np.zeros((M, cfg.K))
        shared[toks] = O.shared_expert(xs[toks], li.ws1.double().cpu().numpy(), li.ws2.double().cpu().numpy())
    # the oracle dequantises the row-major scale bytes (the A8 layer keeps its
    # rearranged copy to itself)
    if cover:
        ref, ys = oracle_tokens_mxfp4(xs, rid, rw, kw.get("w1", li.w1), kw.get("w1_scale", li.w1_scale),
                                      kw.get("w2", li.w2), kw.get("w2_scale", li.w2_scale), toks, emap_np, shared,
                                      activation=activation, clamp=clamp, mxfp8=a8)
        if emap_np is None:       # every touched expert was evaluated
            assert len({int(e) for e in rid[toks].reshape(-1)}) == len(np.unique(rid))
    else:
        w1 = ExpertsF64(kw.get("w1", li.w1), kw.get("w1_scale", li.w1_scale))
        w2 = ExpertsF64(kw.get("w2", li.w2), kw.get("w2_scale", li.w2_scale))
        ref, ys = oracle_tokens(xs, rid, rw, w1, w2, toks, emap_np, shared, activation=activation, clamp=clamp,
                                qdq=O.mxfp8_qdq if a8 else None)
    got = b.out.double().cpu().numpy()[toks]
    g2 = b.gemm2.double().cpu().numpy()
    rel = 3e-2 if (cfg.weight_format == "mxfp4" and not a8) else 1e-2
    abs_ = 0.0 if cfg.weight_format == "mxfp4" else 1e-3
    if bf16_storage:
        # The stored bf16 tensors each round once (unit roundoff u = 2^-8):
        # out itself (u |out|), and every product w * y of the finalize from a
        # bf16 weight and a bf16 gemm2_permuted row (2u |w y| + u^2). The bar
        # is the stated one for the computation plus those rounding bounds.
        u = 2.0 ** -8
        wy = np.zeros_like(ref)
        for a, t_ in enumerate(toks):
            for j in range(cfg.top_k):
                if (t_, j) in ys:
                    wy[a] += abs(rw[t_, j]) * np.abs(ys[(t_, j)])
        if shared is not None:    # the shared expert's output is stored in bf16 too
            wy += np.abs(shared[toks]) / 2
        bound = tol(ref, rel, abs_) + u * np.abs(ref) * (1 + 2 * u) + (2 * u + u * u) * wy
        assert np.all(np.abs(got - ref) <= bound), float(np.max(np.abs(got - ref) - bound))
    else:
        t = tol(ref, rel, abs_)
        err = max_err(got, ref)
        assert err <= t, f"max|gpu-oracle| = {err:.4g} > {t:.4g}"
        if fused_finalize:        # gemm2_permuted is not produced on this path
            return layer, b, x, logits
        # each gathered expert output row (gemm2_permuted), same bar
        ty = tol(np.stack(list(ys.values())), rel, abs_)
        pm = b.pmap.cpu().numpy()
        worst = max(max_err(g2[pm[t_, j]], y) for (t_, j), y in ys.items())
        assert worst <= ty, f"gemm2_permuted row error {worst:.4g} > {ty:.4g}"
    return layer, b, x, logits


# ------------------------------------------------------------------ finalize folded into GEMM2

@pytest.mark.parametrize("name,M,masked", [("tiny", 16, False), ("tiny", 300, True), ("mixtral", 1, False),
                                           ("mixtral", 64, False), ("mixtral", 1024, False),
                                           ("qwen3", 32, False), ("qwen3", 2048, True),
                                           ("deepseek", 64, False)])
def test_fused_finalize_layer(moe, name, M, masked):
    """moe_experts_fused_finalize: out within the oracle's bar, and equal to the
    two-pass result (moe_experts + moe_finalize) up to the order of its f32
    additions."""
    layer, b, x, logits = _check_layer(moe, name, M, masked=masked, fused_finalize=True)
    fused = b.out.clone()
    layer.fused_finalize = False
    b2 = layer.forward(x, logits)
    torch.cuda.synchronize()
    check_no_device_error(moe)
    two_pass = b2.out.double().cpu().numpy()
    rms = float(np.sqrt(np.mean(two_pass ** 2)))
    diff = float((fused.double().cpu() - b2.out.double().cpu()).abs().max())
    assert diff <= 1e-4 * rms + 1e-6, f"fused vs two-pass finalize differ by {diff:.3g} (rms {rms:.3g})"


@pytest.mark.parametrize("name,M,bt,masked,fused", [("qwen3", 2048, 128, False, True), ("qwen3", 2048, 256, False, False),
                                                   ("qwen3", 4096, 256, True, True), ("mixtral", 512, 256, False, True),
                                                   ("mixtral", 512, 128, False, False)])
def test_cta_pair_gemms(moe, name, M, bt, masked, fused):
    """GEMM1 and GEMM2 on CTA pairs (forced by the plan override): the oracle's
    bar, with the finalize folded into GEMM2 or as its own pass."""
    moe.moe_set_plan_override(bt, 0, 0, 0, 3)
    try:
        _check_layer(moe, name, M, masked=masked, fused_finalize=fused)
    finally:
        moe.moe_set_plan_override(0, 0, 0, 0, 0)


def test_fused_finalize_bad_inverse_sets_device_error(moe):
    """An out-of-range permuted_to_expanded entry is reported and skipped."""
    cfg = synth.CONFIGS["tiny"]
    li = layer_inputs("tiny")
    M = 16
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    layer = make_layer(moe, "tiny", li, fused_finalize=True)
    b = layer.forward(x, logits)
    torch.cuda.synchronize()
    good = b.out.clone()
    R = int(b.offsets[-1])
    b.inverse[R - 1] = 10 ** 6                                # out of [0, M*top_k)
    L = moe
    rsf = layer.rsf
    L.moe_experts_fused_finalize(layer.cw, b.x_perm, b.offsets, M, cfg.top_k, b.topk_weights, L.MOE_DTYPE_F32,
                                 b.inverse, None, L.MOE_DTYPE_F32, rsf, b.out, b.exp_ws, b.exp_ws.numel())
    torch.cuda.synchronize()
    assert moe.moe_get_error() == moe.MOE_ERR_DEVICE_INDEX
    assert moe.moe_get_error() == 0
    assert torch.isfinite(b.out).all()
    # only the token of the corrupted row changed (beyond the f32 reordering
    # the unordered additions allow)
    t_bad = int(b.pmap.flatten().tolist().index(R - 1)) // cfg.top_k
    d = (b.out - good).abs().max(dim=1).values
    rms = float(good.pow(2).mean().sqrt())
    others = torch.cat([d[:t_bad], d[t_bad + 1:]])
    assert float(others.max()) <= 1e-5 * rms
    assert float(d[t_bad]) > 1e-3 * rms


@pytest.mark.parametrize("M", [16, 1, 5, 300])
def test_layer_tiny(moe, M):
    _check_layer(moe, "tiny", M)


def test_layer_tiny_bf16_storage(moe):
    _check_layer(moe, "tiny", 16, bf16_storage=True)


@pytest.mark.parametrize("M", [1, 32, 256, 2048, 8192])
def test_layer_qwen3(moe, M):
    _check_layer(moe, "qwen3", M, sample=256)


@pytest.mark.parametrize("M", [1, 8, 64, 512, 4096, 8192])
def test_layer_mixtral(moe, M):
    _check_layer(moe, "mixtral", M)


# the pages' storage dtype: bf16 routing weights, gemm2_permuted and output
# (moe_output.py, UnfinalizedMoEOutput), against the oracle rounded to bf16
@pytest.mark.parametrize("name,M", [("mixtral", 1), ("mixtral", 512), ("mixtral", 8192), ("qwen3", 32),
                                    ("qwen3", 8192), ("deepseek", 64), ("deepseek", 1024)])
def test_layer_bf16_storage(moe, name, M):
    _check_layer(moe, name, M, bf16_storage=True)


@pytest.mark.parametrize("M", [1, 64, 1024, 8192])
def test_layer_deepseek_mxfp4(moe, M):
    """DeepSeek-V3-shaped layer: sigmoid grouped router, MXFP4 routed experts,
    bf16 shared expert; 3e-2 * RMS against the oracle on the same bytes, on a
    sample of at least 256 tokens (all of them at M <= 256) that reaches every
    expert any token routes to."""
    _check_layer(moe, "deepseek", M)


def test_mxfp4_decode_all_codes(moe):
    """Random e2m1 codes (all 16 values, uniformly) under a spread of scale
    bytes, compared over the whole output with the MXFP4 path's bar
    (3e-2 * RMS) against the oracle on the same bytes. A decode error (nibble
    order, sign, scale exponent) would be of the order of the values."""
    g = torch.Generator(device="cpu").manual_seed(21)
    E, K, N, M, k = 4, 512, 512, 48, 2
    p1 = torch.randint(0, 256, (E, 2 * N, K // 2), generator=g, dtype=torch.uint8)
    s1 = torch.randint(112, 127, (E, 2 * N, K // 32), generator=g, dtype=torch.uint8)
    p2 = torch.randint(0, 256, (E, K, N // 2), generator=g, dtype=torch.uint8)
    s2 = torch.randint(110, 125, (E, K, N // 32), generator=g, dtype=torch.uint8)
    x = torch.randn(M, K, generator=g).to(torch.bfloat16)
    logits = torch.randn(M, E, generator=g)
    lay = moe.MoELayer(K=K, N=N, E=E, top_k=k, w1=p1.to(DEV), w2=p2.to(DEV), w1_scale=s1.to(DEV),
                       w2_scale=s2.to(DEV), fmt=moe.MOE_WEIGHTS_MXFP4)
    b = lay.forward(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    check_no_device_error(moe)
    w1 = np.stack([O.dequant_mxfp4(p1[e].numpy(), s1[e].numpy()) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e].numpy(), s2[e].numpy()) for e in range(E)])
    r = O.moe_forward(x.double().numpy(), logits.numpy(), w1, w2, k)
    assert np.array_equal(b.pmap.cpu().numpy(), r["map"])
    got = b.out.double().cpu().numpy()
    assert max_err(got, r["out"]) <= tol(r["out"], 3e-2, 0.0)
    R = int(r["offsets"][-1])
    assert max_err(b.gemm2[:R].double().cpu().numpy(), r["gemm2_permuted"]) <= tol(r["gemm2_permuted"], 3e-2, 0.0)


def test_masked_stress_deferred_finalize(moe):
    """Qwen3-shaped layer at M = 4096, half the experts non-local: the deferred
    output (gemm2_permuted + weights + map) finalized by a separate call equals
    the fused finalize bit for bit, and both match the oracle."""
    layer, b, x, logits = _check_layer(moe, "qwen3", 4096, sample=128, masked=True)
    fused = b.out.clone()
    g2_before = b.gemm2.clone()
    b2 = layer.forward(x, logits, do_finalize=False)
    b2.out.fill_(float("nan"))
    layer.finalize(b2)
    torch.cuda.synchronize()
    R = int(b2.offsets[-1])
    assert torch.equal(b2.gemm2[:R], g2_before[:R])                 # deterministic experts
    assert torch.equal(b2.out, fused)                               # deferred == fused, bitwise
    check_no_device_error(moe)

    # The deferred triple consumed by a separate finalize + shared-expert add
    # (moe_output.py, MoEOutput: whoever finalizes folds the shared output in,
    # after the routed scale).
    cfg = synth.CONFIGS["qwen3"]
    M, k, K = 4096, cfg.top_k, cfg.K
    F = moe.MOE_DTYPE_F32
    g = torch.Generator(device=DEV).manual_seed(77)
    shared = torch.randn(M, K, generator=g, device=DEV)
    out_d = torch.full((M, K), float("nan"), device=DEV)
    moe.moe_finalize(b2.gemm2, F, b2.gemm2.shape[0], b2.topk_weights, F, b2.pmap, M, k, K, shared, F, 1.0,
                     out_d, F)
    # the same finalize run by moe_experts(do_finalize = 1), bit for bit
    out_f = torch.full((M, K), float("nan"), device=DEV)
    g2_f = torch.empty_like(b2.gemm2)
    moe.moe_experts(layer.cw, b2.x_perm, b2.offsets, M, k, g2_f, F, 1, b2.topk_weights, F, b2.pmap, shared, F,
                    1.0, out_f, F, b2.exp_ws, b2.exp_ws.numel())
    torch.cuda.synchronize()
    check_no_device_error(moe)
    assert torch.equal(out_d, out_f)
    # the shared output is added once, after the routed sum
    scale = float((b2.out.abs() + shared.abs()).max())
    assert float((out_d - (b2.out + shared)).abs().max()) <= 2 ** -22 * scale
    # and against the oracle on a token sample
    li = layer_inputs("qwen3")
    em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
    emap_np = em.numpy()
    keep = torch.from_numpy(np.nonzero(emap_np >= 0)[0]).to(DEV)
    rid, rw = O.route_softmax_topk(logits.cpu().numpy(), k)
    toks = sample_tokens(M, 128, seed=5)
    xs = x.to(torch.float64).cpu().numpy()
    sh = np.zeros((M, K))
    sh[toks] = shared.double().cpu().numpy()[toks]
    ref, _ = oracle_tokens(xs, rid, rw, ExpertsF64(li.w1[keep].contiguous()), ExpertsF64(li.w2[keep].contiguous()),
                           toks, emap_np, sh)
    got = out_d.double().cpu().numpy()[toks]
    assert max_err(got, ref) <= tol(ref), (max_err(got, ref), tol(ref))


def test_complement_mask_additivity(moe):
    """out(map A) + out(map not A) = out(no map), with the routing fixed."""
    cfg = synth.CONFIGS["qwen3"]
    li = layer_inputs("qwen3")
    M = 512
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    full = make_layer(moe, "qwen3", li)
    out_full = full.forward(x, logits).out.clone()
    ids, w = full.buffers(M).topk_ids.clone(), full.buffers(M).topk_weights.clone()
    em, E_l = synth.masked_expert_map(cfg.E, seed=5)
    sel = em.numpy() >= 0
    outs = []
    for keep in (sel, ~sel):
        emap = np.full(cfg.E, -1, np.int32)
        emap[keep] = np.arange(keep.sum())
        kidx = torch.from_numpy(np.nonzero(keep)[0]).to(DEV)
        lay = make_layer(moe, "qwen3", li, expert_map=torch.from_numpy(emap).to(DEV), E_local=int(keep.sum()),
                         w1=li.w1[kidx].contiguous(), w2=li.w2[kidx].contiguous())
        outs.append(lay.forward(x, logits, topk_ids=ids, topk_weights=w).out.double().clone())
    torch.cuda.synchronize()
    s = (outs[0] + outs[1]).cpu().numpy()
    ref = out_full.double().cpu().numpy()
    assert max_err(s, ref) <= 1e-5 * float(np.sqrt((ref ** 2).mean())) + 1e-6
    check_no_device_error(moe)


def test_masked_routes_and_padding_do_not_leak(moe):
    """NaN in the weights of -1 routes and in never-referenced gemm2 rows
    must not reach the output."""
    cfg = synth.CONFIGS["qwen3"]
    li = layer_inputs("qwen3")
    M = 64
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
    keep = torch.from_numpy(np.nonzero(em.numpy() >= 0)[0]).to(DEV)
    lay = make_layer(moe, "qwen3", li, expert_map=em.to(DEV), E_local=E_l,
                     w1=li.w1[keep].contiguous(), w2=li.w2[keep].contiguous())
    b = lay.forward(x, logits, do_finalize=False)
    lay.finalize(b)
    torch.cuda.synchronize()
    clean = b.out.clone()
    R = int(b.offsets[-1])
    b.gemm2[R:] = float("nan")
    b.topk_weights[b.pmap < 0] = float("nan")
    lay.finalize(b)
    torch.cuda.synchronize()
    assert torch.isfinite(b.out).all()
    assert torch.equal(b.out, clean)


def test_shared_expert(moe):
    cfg = synth.CONFIGS["deepseek"]
    g = torch.Generator(device=DEV).manual_seed(3)
    M, K, Ns = 64, cfg.K, cfg.shared_N
    ws1 = (torch.randn(2 * Ns, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    ws2 = (torch.randn(K, Ns, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    x = torch.randn(M, K, generator=g, device=DEV).to(torch.bfloat16)
    out = torch.empty(M, K, dtype=torch.float32, device=DEV)
    wsb = moe.moe_shared_expert_workspace_size(M, K, Ns)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    moe.moe_shared_expert(ws1, ws2, K, Ns, x, M, out, moe.MOE_DTYPE_F32, ws, wsb)
    torch.cuda.synchronize()
    ref = O.shared_expert(x.double().cpu().numpy(), ws1.double().cpu().numpy(), ws2.double().cpu().numpy())
    assert max_err(out.cpu().numpy(), ref) <= tol(ref)
    check_no_device_error(moe)
