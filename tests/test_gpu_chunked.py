"""Activation chunking (modular_kernel.py, FusedMoEModularKernel.forward: M
split into chunks of VLLM_FUSED_MOE_CHUNK_SIZE tokens, each run through the
experts with a workspace sized for one chunk): moe_experts_chunked against
the oracle's experts_chunked, and against the unchunked path."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from _helpers import ExpertsF64, lib, max_err, sample_tokens, tol

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32 = 1


@pytest.fixture(scope="module")
def moe():
    m = lib()
    assert m.moe_device_check() == 0, "needs a compute capability 10.3 device"
    return m


_LI = {}


def _layer_inputs(name):
    if name not in _LI:
        _LI.clear()
        torch.cuda.empty_cache()
        _LI[name] = synth.make_layer(synth.CONFIGS[name], DEV)
    return _LI[name]


def _setup(moe, name, M, masked):
    cfg = synth.CONFIGS[name]
    li = _layer_inputs(name)
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    rid, rw = O.route_softmax_topk(logits.cpu().numpy(), cfg.top_k)
    emap = None
    E_l = cfg.E
    w1, w2 = li.w1, li.w2
    if masked:
        em, E_l = synth.masked_expert_map(cfg.E, seed=cfg.seed)
        emap = em.numpy()
        keep = torch.from_numpy(np.nonzero(emap >= 0)[0]).to(DEV)
        w1, w2 = li.w1[keep].contiguous(), li.w2[keep].contiguous()
    w = moe.make_weights(moe.MOE_WEIGHTS_BF16, E_l, cfg.K, cfg.N, w1, w2)
    ids = torch.from_numpy(rid).to(DEV)
    wts = torch.from_numpy(rw.astype(np.float32)).to(DEV)
    return cfg, x, ids, wts, rid, rw, emap, E_l, w, w1, w2


def _chunked(moe, cfg, w, x, ids, wts, M, emap, chunk, do_finalize=1, gemm2_dtype=F32):
    k, K = cfg.top_k, cfg.K
    em = None if emap is None else torch.from_numpy(emap).to(DEV)
    pmap = torch.full((M, k), -7, dtype=torch.int32, device=DEV)
    tdt = torch.float32 if gemm2_dtype == F32 else torch.bfloat16
    g2 = torch.full((M * k, K), float("nan"), dtype=tdt, device=DEV)
    out = torch.full((M, K), float("nan"), device=DEV) if do_finalize else None
    wsb = moe.moe_experts_chunked_workspace_size(w, M, k, chunk)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    moe.moe_experts_chunked(w, x, ids, M, k, cfg.E, em, chunk, pmap, g2, gemm2_dtype, do_finalize,
                            wts if do_finalize else None, F32, None, F32, 1.0, out, F32, ws, wsb)
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    return pmap, g2, out


def _unchunked(moe, cfg, w, x, ids, wts, M, emap, E_l, fused=False):
    k, K = cfg.top_k, cfg.K
    em = None if emap is None else torch.from_numpy(emap).to(DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    offs, pmap, inv = torch.empty(E_l + 1, **i32), torch.empty(M, k, **i32), torch.empty(M * k, **i32)
    xp = torch.empty(M * k, K, dtype=torch.bfloat16, device=DEV)
    pws = torch.empty(max(moe.moe_permute_workspace_size(M, k, E_l), 16), dtype=torch.uint8, device=DEV)
    moe.moe_permute(ids, M, k, cfg.E, em, E_l, x, K, offs, pmap, inv, xp, pws, pws.numel())
    ews = torch.zeros(max(moe.moe_experts_workspace_size(w, M, k), 16), dtype=torch.uint8, device=DEV)
    g2 = torch.full((M * k, K), float("nan"), device=DEV)
    out = torch.full((M, K), float("nan"), device=DEV)
    if fused:
        out.zero_()
        moe.moe_experts_fused_finalize(w, xp, offs, M, k, wts, F32, inv, None, F32, 1.0, out, ews, ews.numel())
    else:
        moe.moe_experts(w, xp, offs, M, k, g2, F32, 1, wts, F32, pmap, None, F32, 1.0, out, F32, ews, ews.numel())
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    return pmap, g2, out


@pytest.mark.parametrize("name,M,chunk,masked", [("tiny", 5, 1, False), ("tiny", 300, 64, True),
                                                 ("qwen3", 300, 64, False), ("qwen3", 1000, 256, True),
                                                 ("qwen3", 8192, 2048, False), ("mixtral", 600, 256, False)])
def test_chunked_matches_oracle(moe, name, M, chunk, masked):
    """Map bit-exact against the oracle's per-chunk permute; every route's
    gemm2_permuted row and the finalized output within the bar."""
    cfg, x, ids, wts, rid, rw, emap, E_l, w, w1, w2 = _setup(moe, name, M, masked)
    pmap, g2, out = _chunked(moe, cfg, w, x, ids, wts, M, emap, chunk)
    r_map = np.full((M, cfg.top_k), -1, np.int32)
    for t0 in range(0, M, chunk):
        _, m, _, _ = O.permute(rid[t0:t0 + chunk], cfg.E, emap)
        r_map[t0:t0 + chunk] = np.where(m >= 0, m + t0 * cfg.top_k, -1)
    pm = pmap.cpu().numpy()
    assert np.array_equal(pm, r_map)
    toks = sample_tokens(M, 96, seed=M)
    xs = x.double().cpu().numpy()
    W1, W2 = ExpertsF64(w1), ExpertsF64(w2)
    r_map_s, r_g2 = O.experts_chunked(xs[toks], rid[toks], W1, W2, cfg.E, len(toks), emap)
    ref_out = O.finalize(r_g2, rw[toks], r_map_s, None, 1.0)
    assert max_err(out.double().cpu().numpy()[toks], ref_out) <= tol(ref_out)
    g2h = g2.double().cpu().numpy()
    got_rows = np.stack([g2h[pm[t, j]] for t in toks for j in range(cfg.top_k) if pm[t, j] >= 0])
    ref_rows = np.stack([r_g2[r_map_s[a, j]] for a in range(len(toks)) for j in range(cfg.top_k)
                         if r_map_s[a, j] >= 0])
    assert max_err(got_rows, ref_rows) <= tol(ref_rows)


@pytest.mark.parametrize("name,M,chunk,masked", [("qwen3", 2048, 300, False), ("qwen3", 4096, 1024, True),
                                                 ("mixtral", 1024, 384, False)])
def test_chunked_equals_unchunked(moe, name, M, chunk, masked):
    """With one launch plan for every call (token tile, no split-K, two
    one-CTA launches), the chunked experts give every route the same
    gemm2_permuted row as the unchunked path, and the same output, bit for
    bit. With the automatic plans, the chunked output is within 1e-4 * RMS of
    the unchunked output with the finalize folded into GEMM2."""
    cfg, x, ids, wts, rid, rw, emap, E_l, w, w1, w2 = _setup(moe, name, M, masked)
    moe.moe_set_plan_override(64, 1, 1, 2, 2)
    try:
        cmap, cg2, cout = _chunked(moe, cfg, w, x, ids, wts, M, emap, chunk)
        umap, ug2, uout = _unchunked(moe, cfg, w, x, ids, wts, M, emap, E_l)
    finally:
        moe.moe_set_plan_override(0, 0, 0, 0, 0)
    cm, um = cmap.cpu().numpy().reshape(-1), umap.cpu().numpy().reshape(-1)
    assert np.array_equal(cm < 0, um < 0)
    v = np.nonzero(cm >= 0)[0]
    assert torch.equal(cg2[torch.from_numpy(cm[v]).to(DEV).long()], ug2[torch.from_numpy(um[v]).to(DEV).long()])
    assert torch.equal(cout, uout)
    # automatic plans: chunked two-pass vs unchunked folded finalize
    _, _, cout2 = _chunked(moe, cfg, w, x, ids, wts, M, emap, chunk)
    _, _, fout = _unchunked(moe, cfg, w, x, ids, wts, M, emap, E_l, fused=True)
    rms = float(fout.pow(2).mean().sqrt())
    assert float((cout2 - fout).abs().max()) <= 1e-4 * rms + 1e-6


def test_chunked_deferred_and_edges(moe):
    """do_finalize = 0 leaves the deferred triple, which moe_finalize turns into
    the do_finalize = 1 output bit for bit; a chunk of at least M tokens is the
    plain permute + experts; bf16 gemm2_permuted; M = 0 is a no-op; a
    workspace below the query is rejected."""
    cfg, x, ids, wts, rid, rw, emap, E_l, w, w1, w2 = _setup(moe, "qwen3", 777, False)
    M, k, K = 777, cfg.top_k, cfg.K
    pmap, g2, _ = _chunked(moe, cfg, w, x, ids, wts, M, emap, 100, do_finalize=0)
    out = torch.full((M, K), float("nan"), device=DEV)
    moe.moe_finalize(g2, F32, M * k, wts, F32, pmap, M, k, K, None, F32, 1.0, out, F32)
    _, _, out1 = _chunked(moe, cfg, w, x, ids, wts, M, emap, 100)
    torch.cuda.synchronize()
    assert torch.equal(out, out1)
    # one chunk: the map is moe_permute's
    pm1, _, _ = _chunked(moe, cfg, w, x, ids, wts, M, emap, 10 ** 6)
    _, r_map, _, _ = O.permute(rid, cfg.E)
    assert np.array_equal(pm1.cpu().numpy(), r_map)
    # bf16 gemm2_permuted: the rows are the f32 rows rounded once
    pmb, g2b, _ = _chunked(moe, cfg, w, x, ids, wts, M, emap, 100, do_finalize=0, gemm2_dtype=0)
    assert torch.equal(pmb, pmap)
    v = pmap.reshape(-1)[pmap.reshape(-1) >= 0].long()
    assert torch.equal(g2b[v], g2[v].to(torch.bfloat16))
    # M = 0, and a workspace that is too small
    moe.moe_experts_chunked(w, x, ids, 0, k, cfg.E, None, 64, pmap, g2, F32, 0, None, F32, None, F32, 1.0, None,
                            F32, None, 0)
    wsb = moe.moe_experts_chunked_workspace_size(w, M, k, 100)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_experts_chunked(w, x, ids, M, k, cfg.E, None, 100, pmap, g2, F32, 0, None, F32, None, F32, 1.0,
                                None, F32, ws, wsb - 256)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
