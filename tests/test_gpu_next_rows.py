"""GPU parity of the rows built beyond the core path: the finalize folded into
the next layer's residual add + RMSNorm; gelu_and_mul and activation_clamp in
GEMM1's epilogue. Each is checked against the CPU oracle on the same seeded
inputs."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from _helpers import lib, max_err, oracle_tokens, sample_tokens, tol
from test_gpu_parity import _check_layer

pytestmark = pytest.mark.gpu

DEV = "cuda"
TD = {0: torch.bfloat16, 1: torch.float32}


@pytest.fixture(scope="module")
def moe():
    m = lib()
    assert m.moe_device_check() == 0, "needs a compute capability 10.3 device"
    return m


def _dt(moe, torch_dtype):
    return moe.MOE_DTYPE_F32 if torch_dtype == torch.float32 else moe.MOE_DTYPE_BF16


def _bound(ref, got_dtype, rel):
    """f32 results: rel * RMS(ref) + tiny; bf16 results: that plus one bf16
    ulp of the reference value (the result is rounded once to bf16)."""
    b = rel * float(np.sqrt(np.mean(ref ** 2))) + 1e-6
    if got_dtype == torch.bfloat16:
        return b + 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
    return b


# ------------------------------------------------------------------ finalize + residual add + RMSNorm

@pytest.mark.parametrize("M,K,k,g2t,rt,yt,gt,with_shared", [
    (16, 128, 2, torch.float32, torch.float32, torch.float32, torch.float32, False),
    (33, 4096, 2, torch.float32, torch.bfloat16, torch.bfloat16, torch.bfloat16, True),
    (64, 7168, 8, torch.bfloat16, torch.float32, torch.float32, torch.float32, True),
    (5, 16384, 8, torch.float32, torch.float32, torch.bfloat16, torch.float32, False),
])
def test_finalize_add_rmsnorm_kernel(moe, M, K, k, g2t, rt, yt, gt, with_shared):
    """The kernel alone on seeded inputs (masked routes included) against the
    oracle's finalize_add_rmsnorm: new residual and y."""
    g = torch.Generator().manual_seed(M * 7 + K)
    R = M * k
    g2 = torch.randn(R, K, generator=g).to(g2t)
    w = torch.rand(M, k, generator=g, dtype=torch.float32) + 0.1
    pmap = torch.randperm(R, generator=g)[:M * k].reshape(M, k).to(torch.int32)
    mask = torch.rand(M, k, generator=g) < 0.2
    pmap[mask] = -1
    w[mask] = float("nan")                                          # must not leak through a -1 route
    shared = torch.randn(M, K, generator=g).to(g2t) if with_shared else None
    res = (3.0 * torch.randn(M, K, generator=g)).to(rt)
    gamma = (torch.rand(K, generator=g) + 0.5).to(gt)
    eps, rsf = 1e-6, 1.5
    ref_r, ref_y = O.finalize_add_rmsnorm(g2.double().numpy(), w.double().numpy(), pmap.numpy(),
                                          res.double().numpy(), gamma.double().numpy(), eps,
                                          None if shared is None else shared.double().numpy(), rsf)
    d = lambda t: None if t is None else t.to(DEV)
    res_d, y_d = res.to(DEV), torch.full((M, K), float("nan"), dtype=yt, device=DEV)
    moe.moe_finalize_add_rmsnorm(d(g2), _dt(moe, g2t), R, d(w), moe.MOE_DTYPE_F32, d(pmap), M, k, K, d(shared),
                                 _dt(moe, g2t), rsf, res_d, _dt(moe, rt), d(gamma), _dt(moe, gt), eps, y_d,
                                 _dt(moe, yt))
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    got_r, got_y = res_d.double().cpu().numpy(), y_d.double().cpu().numpy()
    assert np.isfinite(got_y).all()
    assert np.all(np.abs(got_r - ref_r) <= _bound(ref_r, rt, 2e-6))
    assert np.all(np.abs(got_y - ref_y) <= _bound(ref_y, yt, 2e-6))


def test_finalize_add_rmsnorm_rejects_bad_arguments(moe):
    K, M, k = 64, 4, 2
    f = lambda *a, **kw: torch.zeros(*a, device=DEV, **kw)
    g2, w, pmap = f(M * k, K), f(M, k), torch.zeros(M, k, dtype=torch.int32, device=DEV)
    res, gamma, y = f(M, K), f(K), f(M, K)
    F = moe.MOE_DTYPE_F32
    with pytest.raises(moe.MoEError) as e:                            # K not a multiple of 8
        moe.moe_finalize_add_rmsnorm(g2, F, M * k, w, F, pmap, M, k, 60, None, F, 1.0, res, F, gamma, F, 1e-6, y, F)
    assert e.value.status == moe.MOE_ERR_ALIGNMENT
    with pytest.raises(moe.MoEError) as e:                            # y aliases the residual
        moe.moe_finalize_add_rmsnorm(g2, F, M * k, w, F, pmap, M, k, K, None, F, 1.0, res, F, gamma, F, 1e-6, res, F)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG
    with pytest.raises(moe.MoEError) as e:                            # negative eps
        moe.moe_finalize_add_rmsnorm(g2, F, M * k, w, F, pmap, M, k, K, None, F, 1.0, res, F, gamma, F, -1.0, y, F)
    assert e.value.status == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("name,M", [("mixtral", 64), ("qwen3", 256)])
def test_layer_deferred_output_into_add_rmsnorm(moe, name, M):
    """The whole chain: the layer's deferred output (do_finalize = 0) consumed
    by moe_finalize_add_rmsnorm, against the full oracle (experts, finalize,
    residual add, RMSNorm) on a token sample, at the layer's bar."""
    cfg = synth.CONFIGS[name]
    li = synth.make_layer(cfg, DEV)
    x, logits = synth.make_tokens(cfg, M, DEV, li)
    layer = moe.MoELayer(K=cfg.K, N=cfg.N, E=cfg.E, top_k=cfg.top_k, w1=li.w1, w2=li.w2)
    b = layer.forward(x, logits, do_finalize=False)
    g = torch.Generator().manual_seed(M)
    res = torch.randn(M, cfg.K, generator=g).to(DEV)
    res0 = res.double().cpu().numpy()
    gamma = (torch.rand(cfg.K, generator=g) + 0.5).to(DEV)
    y = torch.empty(M, cfg.K, device=DEV)
    eps = 1e-5
    moe.moe_finalize_add_rmsnorm(b.gemm2, layer.gemm2_dtype, b.gemm2.shape[0], b.topk_weights, layer.weights_dtype,
                                 b.pmap, M, cfg.top_k, cfg.K, None, moe.MOE_DTYPE_F32, 1.0, res, moe.MOE_DTYPE_F32,
                                 gamma, moe.MOE_DTYPE_F32, eps, y, moe.MOE_DTYPE_F32)
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    rid, rw = O.route_softmax_topk(logits.cpu().numpy(), cfg.top_k)
    toks = sample_tokens(M, 32)
    xs = x.double().cpu().numpy()
    w1 = [li.w1[e].double().cpu().numpy() for e in range(cfg.E)]
    w2 = [li.w2[e].double().cpu().numpy() for e in range(cfg.E)]
    out_ref, _ = oracle_tokens(xs, rid, rw, w1, w2, toks)
    r_ref, y_ref = O.add_rmsnorm(out_ref, res0[toks], gamma.double().cpu().numpy(), eps)
    got_y = y.double().cpu().numpy()[toks]
    assert max_err(got_y, y_ref) <= tol(y_ref)
    assert max_err(res.double().cpu().numpy()[toks], r_ref) <= tol(r_ref)


# ------------------------------------------------------------------ gelu_and_mul, activation_clamp

@pytest.mark.parametrize("name,M,act,clamp,fused", [("tiny", 16, "gelu", None, False), ("tiny", 300, "silu", 1.0, True),
                                                    ("tiny", 300, "gelu", 1.0, False),
                                                    ("qwen3", 32, "gelu", 1.0, True),
                                                    ("mixtral", 64, "gelu", None, True),
                                                    ("qwen3", 8192, "gelu", 1.0, True)])
def test_layer_activation(moe, name, M, act, clamp, fused):
    """The layer with gelu_and_mul and/or the activation clamp, one-CTA and
    CTA-pair GEMMs (Qwen3-shaped at M = 8192 runs on pairs), against the
    oracle's expert_mlp with the same activation, at the layer's bar."""
    _check_layer(moe, name, M, activation=act, clamp=clamp, fused_finalize=fused, sample=64 if M > 1000 else None)


# ------------------------------------------------------------------ BatchedExperts format

@pytest.mark.parametrize("name,T,act,rows_per_expert", [("tiny", 40, "silu", None), ("tiny", 300, "gelu", None),
                                                        ("mixtral", 96, "silu", 6)])
def test_experts_batched(moe, name, T, act, rows_per_expert):
    """moe_experts_batched on [E, max_tokens, K] with ragged counts (0 and
    max_tokens included) against the oracle's experts_batched; rows past each
    count are left as they were."""
    cfg = synth.CONFIGS[name]
    li = synth.make_layer(cfg, DEV)
    E, K = cfg.E, cfg.K
    g = torch.Generator().manual_seed(T)
    counts = torch.randint(0, T + 1, (E,), generator=g, dtype=torch.int32)
    counts[0], counts[-1] = 0, T
    xb = torch.randn(E, T, K, generator=g).to(torch.bfloat16)
    w = moe.make_weights(moe.MOE_WEIGHTS_BF16, E, K, cfg.N, li.w1, li.w2,
                         activation=moe.MOE_ACT_GELU if act == "gelu" else moe.MOE_ACT_SILU)
    ws = torch.zeros(max(moe.moe_experts_batched_workspace_size(w, T), 16), dtype=torch.uint8, device=DEV)
    y = torch.full((E, T, K), float("nan"), device=DEV)
    for _ in range(2):                                                # twice: counters left at zero
        moe.moe_experts_batched(w, xb.to(DEV), counts.to(DEV), T, y, moe.MOE_DTYPE_F32, ws, ws.numel())
    torch.cuda.synchronize()
    assert moe.moe_get_error() == 0
    got = y.double().cpu().numpy()
    w1 = [li.w1[e].double().cpu().numpy() for e in range(E)]
    w2 = [li.w2[e].double().cpu().numpy() for e in range(E)]
    xs = xb.double().numpy()
    refs, gots = [], []
    for e in range(E):
        c = int(counts[e])
        assert np.isnan(got[e, c:]).all()                             # untouched past the count
        rows = list(range(c)) if rows_per_expert is None else sorted(set(np.linspace(0, c - 1, rows_per_expert,
                                                                                   dtype=int).tolist()))
        if c and rows:
            if rows_per_expert is None:
                ref = O.experts_batched(xs[e:e + 1], counts[e:e + 1].numpy(), np.stack([w1[e]]), np.stack([w2[e]]),
                                        act)[0, :c]
            else:
                ref = O.expert_mlp(xs[e, rows], w1[e], w2[e], act)
            refs.append(ref)
            gots.append(got[e, rows])
    ref, gv = np.concatenate(refs), np.concatenate(gots)
    assert max_err(gv, ref) <= tol(ref)
