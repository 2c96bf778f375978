"""Pins of the CPU oracle against facts fixed outside the oracle itself:
the e2m1 table printed on the page, closed forms, brute force over every
subset / every expert, library routines for special cases, and invariants
the pages state. CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_from_bits(code: int) -> float:
    """e2m1 by its bit fields (OCP MX v1.0): sign bit 3, exponent bits 2-1
    (bias 1), mantissa bit 0; exponent 0 is subnormal (m * 0.5)."""
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return -mag if s else mag


# ---------------------------------------------------------------- MXFP4 decode

def test_e2m1_table_matches_page():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_table.txt"))
            if l.strip() and not l.startswith("#")]
    page = {int(c): float(v) for c, v in rows}
    assert len(page) == 16
    for code in range(16):
        got = O.e2m1_value(code)
        assert got == page[code]
        assert math.copysign(1.0, got) == math.copysign(1.0, page[code])


def test_e2m1_table_matches_bitfield_definition():
    for code in range(16):
        got, want = O.e2m1_value(code), _e2m1_from_bits(code)
        assert got == want and math.copysign(1, got) == math.copysign(1, want)


def test_ue8m0_closed_form():
    s = np.arange(256)
    got = O.ue8m0_scale(s)
    assert got[0] == 0.0 and np.isinf(got[255])
    for v in range(1, 255):
        assert got[v] == math.ldexp(1.0, v - 127)


def test_dequant_exhaustive_bytes_and_scales():
    # every packed byte value, under every finite scale byte
    packed = np.tile(np.arange(256, dtype=np.uint8), (254, 1))      # [254 rows, 256 bytes] -> C = 512
    scales = np.repeat(np.arange(1, 255, dtype=np.uint8)[:, None], 16, axis=1)  # [254, 512/32]
    got = O.dequant_mxfp4(packed, scales)

    def f32(v):   # the page multiplies in float32: beyond its range the product is inf
        return v if abs(v) <= 3.4028234663852886e38 else math.copysign(math.inf, v)

    for r in range(254):
        sc = math.ldexp(1.0, (r + 1) - 127)
        for j in range(256):
            assert got[r, 2 * j] == f32(_e2m1_from_bits(j & 0xF) * sc)
            assert got[r, 2 * j + 1] == f32(_e2m1_from_bits(j >> 4) * sc)


def test_dequant_scale_granularity_is_32():
    rng = np.random.default_rng(5)
    packed = rng.integers(0, 256, size=(3, 64), dtype=np.uint8)          # C = 128
    scales = rng.integers(100, 140, size=(3, 4), dtype=np.uint8)
    got = O.dequant_mxfp4(packed, scales)
    for r in range(3):
        for c in range(128):
            byte = packed[r, c // 2]
            code = (byte & 0xF) if c % 2 == 0 else (byte >> 4)
            assert got[r, c] == _e2m1_from_bits(int(code)) * 2.0 ** (int(scales[r, c // 32]) - 127)


def test_bf16_round_matches_torch():
    x = np.random.default_rng(1).standard_normal(10000).astype(np.float32) * 37
    x[:4] = [0.0, -0.0, 1e-40, 3.0e38]
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(O.bf16_round(x), want)


# ---------------------------------------------------------------- sigmoid spec

def test_sigmoid_spec_close_to_exact():
    x = np.concatenate([np.linspace(-30, 30, 20001), np.linspace(-90, 90, 2001)]).astype(np.float32)
    got = O.sigmoid_f32_spec(x).astype(np.float64)
    exact = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    ulp = np.spacing(exact.astype(np.float32)).astype(np.float64)
    normal = x > -88.0
    assert np.all(np.abs(got - exact)[normal] <= 2 * ulp[normal])
    # below -88 the true value is a float32 subnormal; the spec returns 0 there
    assert np.all(got[~normal] == 0.0) and np.all(exact[~normal] < 2.0 ** -126)
    assert O.sigmoid_f32_spec(np.float32(0.0)) == np.float32(0.5)
    assert O.sigmoid_f32_spec(np.float32(100.0)) == 1.0
    assert O.sigmoid_f32_spec(np.float32(-100.0)) == 0.0


def test_sigmoid_spec_monotone():
    x = np.sort(np.random.default_rng(2).standard_normal(20000).astype(np.float32) * 6)
    y = O.sigmoid_f32_spec(x)
    assert np.all(np.diff(y) >= 0)


def test_exp_spec_constants():
    # LN2_HI has at most 16 significant bits, and HI + LO is ln 2 to float64 rounding
    hi = float(O.moe_oracle._LN2_HI)
    m, e = math.frexp(hi)
    assert (m * 2 ** 16) == int(m * 2 ** 16)
    assert abs(hi + float(O.moe_oracle._LN2_LO) - math.log(2.0)) < 1e-13


# ---------------------------------------------------------------- routers

def _brute_best_subset(keys, k, allowed=None):
    cand = [i for i in range(len(keys)) if allowed is None or allowed[i]]
    best, best_s = None, None
    for sub in itertools.combinations(cand, k):
        s = sum(float(keys[i]) for i in sub)
        if best_s is None or s > best_s:
            best, best_s = set(sub), s
    return best


@pytest.mark.parametrize("E,k", [(8, 2), (9, 3), (12, 4)])
def test_softmax_router_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    logits = rng.standard_normal((40, E)).astype(np.float32)
    ids, w = O.route_softmax_topk(logits, k, 1.0)
    for t in range(40):
        p = torch.softmax(torch.from_numpy(logits[t]).double(), 0).numpy()
        assert set(ids[t].tolist()) == _brute_best_subset(p, k)
        assert all(p[ids[t][i]] >= p[ids[t][i + 1]] for i in range(k - 1))
        assert abs(w[t].sum() - 1.0) < 1e-12
        # renormalised softmax: every ratio is exp of the logit difference
        for a in range(k):
            for b in range(k):
                r = w[t, a] / w[t, b]
                assert abs(r - math.exp(float(logits[t, ids[t, a]]) - float(logits[t, ids[t, b]]))) < 1e-9 * max(1, r)


def test_softmax_router_ties_and_scale():
    logits = np.array([[0.5, 1.0, 1.0, -2.0, 1.0, 0.0]], dtype=np.float32)
    ids, w = O.route_softmax_topk(logits, 3, 2.5)
    assert ids.tolist() == [[1, 2, 4]]
    np.testing.assert_allclose(w, [[2.5 / 3] * 3], rtol=1e-12)
    # -0.0 and +0.0 compare equal: lower id first
    ids, _ = O.route_softmax_topk(np.array([[-0.0, 0.0, -1.0]], dtype=np.float32), 2)
    assert ids.tolist() == [[0, 1]]


def test_sigmoid_grouped_router_brute_force():
    rng = np.random.default_rng(7)
    E, n_group, topk_group, k = 16, 4, 2, 3
    logits = rng.standard_normal((60, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    ids, w = O.route_sigmoid_grouped(logits, bias, k, n_group, topk_group, 2.5)
    G = E // n_group
    for t in range(60):
        s = 1.0 / (1.0 + np.exp(-logits[t].astype(np.float64)))
        b = s + bias.astype(np.float64)
        gs = [sum(sorted(b[g * G:(g + 1) * G], reverse=True)[:2]) for g in range(n_group)]
        best_groups = _brute_best_subset(np.array(gs), topk_group)
        allowed = np.zeros(E, bool)
        for g in best_groups:
            allowed[g * G:(g + 1) * G] = True
        assert set(ids[t].tolist()) == _brute_best_subset(b, k, allowed)
        assert all(allowed[i] for i in ids[t])
        assert all(b[ids[t][i]] >= b[ids[t][i + 1]] for i in range(k - 1))
        np.testing.assert_allclose(w[t], s[ids[t]] / s[ids[t]].sum() * 2.5, rtol=1e-12)
        assert abs(w[t].sum() - 2.5) < 1e-12


def test_sigmoid_grouped_single_group_is_plain_topk():
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((20, 10)).astype(np.float32)
    bias = np.zeros(10, np.float32)
    ids, _ = O.route_sigmoid_grouped(logits, bias, 3, 1, 1)
    ids2, _ = O.route_softmax_topk(logits, 3)        # sigmoid is increasing
    assert (ids == ids2).all()


def _exact_grouped_selection(logits, bias, top_k, n_group, topk_group):
    """DeepSeek-V3's grouped selection on float64 keys with the exact sigma
    (no float32 spec): returns the ids and, per token, the margins at the two
    places where a near-tie could change the result -- the kept/dropped group
    boundary and the order of the top_k + 1 best allowed keys."""
    b = 1.0 / (1.0 + np.exp(-logits.astype(np.float64))) + bias.astype(np.float64)[None, :]
    M, E = b.shape
    G = E // n_group
    gscore = -np.sort(-b.reshape(M, n_group, G), axis=2)[:, :, :2].sum(axis=2)
    gorder = np.argsort(-gscore, axis=1, kind="stable")
    allowed = np.zeros((M, n_group), bool)
    np.put_along_axis(allowed, gorder[:, :topk_group], True, axis=1)
    key = np.where(np.repeat(allowed, G, axis=1), b, -np.inf)
    order = np.argsort(-key, axis=1, kind="stable")
    gs = np.take_along_axis(gscore, gorder, axis=1)
    ks = np.take_along_axis(key, order[:, :top_k + 1], axis=1)
    g_margin = (gs[:, topk_group - 1] - gs[:, topk_group]) / np.spacing(gs[:, 0].astype(np.float32))
    k_margin = np.min(ks[:, :-1] - ks[:, 1:], axis=1) / np.spacing(ks[:, 0].astype(np.float32))
    return order[:, :top_k].astype(np.int32), g_margin, k_margin


def test_sigmoid_grouped_selection_spec_equals_exact_sigma():
    """The router's selection is taken on float32 keys built with the written
    sigmoid spec (so that the oracle and the kernel decide near-ties alike).
    Away from ties that approximation must not change what is selected:
    over 10^5 tokens of the DeepSeek-V3-shaped router (E = 256, 8 groups, 4
    kept, top-8; logits N(0, 1), selection bias N(0, 0.1)), the oracle's ids
    equal the ids of an exact float64 selection on every token whose float64
    keys are more than 4 float32 ulp from a tie at a decision boundary."""
    rng = np.random.default_rng(20251)
    M, E, k, ng, tg = 100_000, 256, 8, 8, 4
    logits = rng.standard_normal((M, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    ids, _ = O.route_sigmoid_grouped(logits, bias, k, ng, tg, 2.5)
    exact, g_margin, k_margin = _exact_grouped_selection(logits, bias, k, ng, tg)
    tie_free = (g_margin > 4) & (k_margin > 4)
    assert tie_free.mean() > 0.99                         # near-ties are rare at these sizes
    assert np.array_equal(ids[tie_free], exact[tie_free])
    # and a near-tie token still gets a valid selection of distinct experts
    for t in np.nonzero(~tie_free)[0][:50]:
        assert len(set(ids[t].tolist())) == k


# ---------------------------------------------------------------- permute

def _check_permute(ids, E, emap=None):
    offsets, pmap, inv, E_l = O.permute(ids, E, emap)
    M, k = ids.shape
    em = np.arange(E) if emap is None else np.asarray(emap)
    local = em[ids.reshape(-1)]
    masked = int((local < 0).sum())
    R = int(offsets[-1])
    assert R == M * k - masked                                   # counts sum
    assert np.all(np.diff(offsets) >= 0) and offsets[0] == 0      # monotone offsets
    flat = pmap.reshape(-1)
    assert np.all((flat == -1) == (local < 0))                   # -1 exactly on masked routes
    assert sorted(flat[flat >= 0].tolist()) == list(range(R))    # bijection onto [0, R)
    for p in range(R):
        assert flat[inv[p]] == p
    # second formulation: stable argsort of the local ids
    keep = np.nonzero(local >= 0)[0]
    order = keep[np.argsort(local[keep], kind="stable")]
    assert (inv == order).all()
    for le in range(E_l):
        assert offsets[le + 1] - offsets[le] == (local == le).sum()
    return offsets, pmap, inv


def test_permute_invariants():
    rng = np.random.default_rng(3)
    for E, k, M in [(8, 2, 16), (16, 4, 33), (5, 5, 7), (128, 8, 50)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
        _check_permute(ids, E)
        emap = np.full(E, -1, np.int32)
        keep = np.sort(rng.permutation(E)[: E // 2])
        emap[keep] = np.arange(len(keep))
        _check_permute(ids, E, emap)


def test_permute_empty_and_all_masked():
    offsets, pmap, inv, _ = O.permute(np.zeros((0, 2), np.int32), 4)
    assert offsets.tolist() == [0, 0, 0, 0, 0] and pmap.shape == (0, 2) and len(inv) == 0
    emap = np.array([-1, -1, 0, 1], np.int32)
    offsets, pmap, inv, _ = O.permute(np.array([[0, 1]], np.int32), 4, emap)
    assert offsets.tolist() == [0, 0, 0] and pmap.tolist() == [[-1, -1]]


# ---------------------------------------------------------------- experts and finalize

def _tiny_weights(rng, E, K, N):
    w1 = rng.standard_normal((E, 2 * N, K)) / math.sqrt(K)
    w2 = rng.standard_normal((E, K, N)) / math.sqrt(N)
    return w1, w2


def test_expert_mlp_matches_torch_swiglu():
    rng = np.random.default_rng(4)
    K, N = 24, 40
    x = rng.standard_normal((9, K))
    w1, w2 = _tiny_weights(rng, 1, K, N)
    xt = torch.from_numpy(x)
    g = xt @ torch.from_numpy(w1[0][:N]).T
    u = xt @ torch.from_numpy(w1[0][N:]).T
    want = (torch.nn.functional.silu(g) * u) @ torch.from_numpy(w2[0]).T
    np.testing.assert_allclose(O.expert_mlp(x, w1[0], w2[0]), want.numpy(), rtol=1e-12, atol=1e-12)


def test_top1_weight1_is_dense_mlp():
    """top_k = 1 with weight 1 reproduces the single expert's dense MLP."""
    rng = np.random.default_rng(6)
    M, K, N, E = 12, 16, 32, 3
    x = rng.standard_normal((M, K))
    w1, w2 = _tiny_weights(rng, E, K, N)
    ids = rng.integers(0, E, size=(M, 1)).astype(np.int32)
    offsets, pmap, inv, _ = O.permute(ids, E)
    g2 = O.experts(x, w1, w2, offsets, inv, 1)
    out = O.finalize(g2, np.ones((M, 1)), pmap)
    for t in range(M):
        e = ids[t, 0]
        xt = torch.from_numpy(x[t:t + 1])
        h = xt @ torch.from_numpy(w1[e]).T
        want = (torch.nn.functional.silu(h[:, :N]) * h[:, N:]) @ torch.from_numpy(w2[e]).T
        np.testing.assert_allclose(out[t], want.numpy()[0], rtol=1e-12, atol=1e-12)


def test_routed_equals_dense_brute_force():
    """Every token through every expert, weighted by a dense [M, E] gate that
    is zero off-route, equals the routed permute/experts/finalize result."""
    rng = np.random.default_rng(9)
    M, K, N, E, k = 10, 16, 24, 6, 3
    x = rng.standard_normal((M, K))
    w1, w2 = _tiny_weights(rng, E, K, N)
    logits = rng.standard_normal((M, E)).astype(np.float32)
    r = O.moe_forward(x, logits, w1, w2, k)
    dense_gate = np.zeros((M, E))
    for t in range(M):
        dense_gate[t, r["ids"][t]] = r["weights"][t]
    want = np.zeros((M, K))
    for e in range(E):
        xt = torch.from_numpy(x)
        h = xt @ torch.from_numpy(w1[e]).T
        ye = ((torch.nn.functional.silu(h[:, :N]) * h[:, N:]) @ torch.from_numpy(w2[e]).T).numpy()
        want += dense_gate[:, e:e + 1] * ye
    np.testing.assert_allclose(r["out"], want, rtol=1e-11, atol=1e-11)


def test_masked_routes_contribute_zero_and_nan_does_not_leak():
    rng = np.random.default_rng(10)
    M, K, N, E, k = 8, 16, 16, 4, 2
    x = rng.standard_normal((M, K))
    w1, w2 = _tiny_weights(rng, E, K, N)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    emap = np.array([0, -1, 1, -1], np.int32)
    offsets, pmap, inv, E_l = O.permute(ids, E, emap)
    g2 = O.experts(x, w1[[0, 2]], w2[[0, 2]], offsets, inv, k)
    w = rng.random((M, k))
    w_poison = w.copy()
    w_poison[pmap < 0] = np.nan
    g2_pad = np.vstack([g2, np.full((M * k - len(g2), K), np.nan)])   # padded rows never referenced
    a = O.finalize(g2, w, pmap)
    b = O.finalize(g2_pad, w_poison, pmap)
    assert np.isfinite(b).all()
    np.testing.assert_array_equal(a, b)


def test_complement_mask_additivity():
    """out(map A) + out(map complement of A) = out(no map)."""
    rng = np.random.default_rng(11)
    M, K, N, E, k = 9, 16, 16, 6, 2
    x = rng.standard_normal((M, K))
    w1, w2 = _tiny_weights(rng, E, K, N)
    logits = rng.standard_normal((M, E)).astype(np.float32)
    full = O.moe_forward(x, logits, w1, w2, k)["out"]
    sel = np.array([1, 0, 1, 1, 0, 0], bool)
    emap_a = np.full(E, -1, np.int32); emap_a[sel] = np.arange(sel.sum())
    emap_b = np.full(E, -1, np.int32); emap_b[~sel] = np.arange((~sel).sum())
    out_a = O.moe_forward(x, logits, w1[sel], w2[sel], k, expert_map=emap_a)["out"]
    out_b = O.moe_forward(x, logits, w1[~sel], w2[~sel], k, expert_map=emap_b)["out"]
    np.testing.assert_allclose(out_a + out_b, full, rtol=1e-12, atol=1e-12)


def test_finalize_scale_before_shared_add():
    g2 = np.array([[1.0, 2.0], [3.0, 4.0]])
    pmap = np.array([[0, 1]])
    w = np.array([[0.25, 0.5]])
    shared = np.array([[10.0, 20.0]])
    out = O.finalize(g2, w, pmap, shared, routed_scaling_factor=2.0)
    np.testing.assert_array_equal(out, [[2.0 * (0.25 + 1.5) + 10.0, 2.0 * (0.5 + 2.0) + 20.0]])


def test_shared_expert_is_top1_mlp():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((5, 16))
    w1, w2 = _tiny_weights(rng, 1, 16, 8)
    np.testing.assert_array_equal(O.shared_expert(x, w1[0], w2[0]), O.expert_mlp(x, w1[0], w2[0]))


def test_mxfp4_layer_equals_bf16_layer_on_dequantised_weights():
    """The MXFP4 path is the bf16 path on the dequantised weights: dequantise,
    then run the plain layer; compare with a layer whose weights are the
    bit-field decode of the same bytes."""
    rng = np.random.default_rng(13)
    E, K, N, M, k = 3, 64, 64, 6, 2
    p1 = rng.integers(0, 256, size=(E, 2 * N, K // 2), dtype=np.uint8)
    s1 = rng.integers(118, 124, size=(E, 2 * N, K // 32), dtype=np.uint8)
    p2 = rng.integers(0, 256, size=(E, K, N // 2), dtype=np.uint8)
    s2 = rng.integers(118, 124, size=(E, K, N // 32), dtype=np.uint8)
    w1 = np.stack([O.dequant_mxfp4(p1[e], s1[e]) for e in range(E)])
    w2 = np.stack([O.dequant_mxfp4(p2[e], s2[e]) for e in range(E)])
    lut = np.array([_e2m1_from_bits(c) for c in range(16)])
    def bitdec(p, s):
        v = np.empty(p.shape[:-1] + (p.shape[-1] * 2,))
        v[..., 0::2] = lut[p & 15]; v[..., 1::2] = lut[p >> 4]
        return v * np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=-1)
    np.testing.assert_array_equal(w1, bitdec(p1, s1))
    np.testing.assert_array_equal(w2, bitdec(p2, s2))
    x = rng.standard_normal((M, K))
    logits = rng.standard_normal((M, E)).astype(np.float32)
    r = O.moe_forward(x, logits, w1, w2, k)
    assert np.isfinite(r["out"]).all()


# ---------------------------------------------------------------- gelu_and_mul, activation_clamp

def test_gelu_erf_values_and_odd_identity():
    """GELU(1) = Phi(1) (the standard normal CDF at 1, 0.8413447460685429);
    GELU(0) = 0; GELU(z) - GELU(-z) = z for every z (erf is odd); and the
    values agree with Python's math.erf, a second implementation of erf."""
    assert O.gelu_erf(1.0) == pytest.approx(0.8413447460685429, abs=1e-15)
    assert O.gelu_erf(0.0) == 0.0
    z = np.linspace(-8, 8, 1601)
    np.testing.assert_allclose(O.gelu_erf(z) - O.gelu_erf(-z), z, rtol=0, atol=1e-13)
    ref = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in z])
    np.testing.assert_allclose(O.gelu_erf(z), ref, rtol=1e-14, atol=1e-15)


def test_gelu_and_mul_expert_matches_torch():
    """expert_mlp with the gelu activation against torch's exact GELU."""
    rng = np.random.default_rng(41)
    K, N = 24, 40
    x = rng.standard_normal((9, K))
    w1, w2 = _tiny_weights(rng, 1, K, N)
    xt = torch.from_numpy(x)
    g = xt @ torch.from_numpy(w1[0][:N]).T
    u = xt @ torch.from_numpy(w1[0][N:]).T
    want = (torch.nn.functional.gelu(g, approximate="none") * u) @ torch.from_numpy(w2[0]).T
    np.testing.assert_allclose(O.expert_mlp(x, w1[0], w2[0], "gelu"), want.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["silu", "gelu"])
def test_activation_clamp(act):
    """The clamp bounds the gate from above and up to [-c, c] (torch.clamp as
    the second implementation); a clamp above every value changes nothing."""
    rng = np.random.default_rng(43)
    K, N, c = 16, 24, 0.75
    x = 3.0 * rng.standard_normal((11, K))
    w1, w2 = _tiny_weights(rng, 1, K, N)
    xt = torch.from_numpy(x)
    g = torch.clamp(xt @ torch.from_numpy(w1[0][:N]).T, max=c)
    u = torch.clamp(xt @ torch.from_numpy(w1[0][N:]).T, min=-c, max=c)
    f = torch.nn.functional.silu if act == "silu" else (lambda v: torch.nn.functional.gelu(v, approximate="none"))
    want = (f(g) * u) @ torch.from_numpy(w2[0]).T
    got = O.expert_mlp(x, w1[0], w2[0], act, clamp=c)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)
    assert np.abs(got - O.expert_mlp(x, w1[0], w2[0], act)).max() > 1e-3       # the clamp is active here
    np.testing.assert_array_equal(O.expert_mlp(x, w1[0], w2[0], act, clamp=1e9),
                                  O.expert_mlp(x, w1[0], w2[0], act))


# ---------------------------------------------------------------- BatchedExperts format

def test_experts_batched_equals_grouped():
    """The batched layout computes, row for row, what the grouped experts()
    computes on the same tokens in the permuted (expert-major) layout; rows
    past each expert's count are zero."""
    rng = np.random.default_rng(47)
    E, T, K, N = 5, 7, 16, 24
    counts = np.array([3, 0, 7, 1, 5])
    w1, w2 = _tiny_weights(rng, E, K, N)
    xb = rng.standard_normal((E, T, K))
    yb = O.experts_batched(xb, counts, w1, w2, "gelu", clamp=2.0)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = np.concatenate([xb[e, :counts[e]] for e in range(E)])
    inverse = np.arange(rows.shape[0], dtype=np.int32)               # top_k = 1: token p is row p
    g = O.experts(rows, w1, w2, offsets, inverse, 1, "gelu", clamp=2.0)
    for e in range(E):
        np.testing.assert_array_equal(yb[e, :counts[e]], g[offsets[e]:offsets[e + 1]])
        assert not yb[e, counts[e]:].any()


# ---------------------------------------------------------------- residual add + RMSNorm

def test_rmsnorm_worked_example():
    """x = [1, 2, 3, 4], no residual, gamma = 1, eps = 0: the RMS is
    sqrt(30/4) = sqrt(7.5), so y = x / 2.7386127875258306."""
    r, y = O.add_rmsnorm(np.array([[1.0, 2.0, 3.0, 4.0]]), np.zeros((1, 4)), np.ones(4), 0.0)
    np.testing.assert_array_equal(r, [[1.0, 2.0, 3.0, 4.0]])
    np.testing.assert_allclose(y, [[0.3651483716701107, 0.7302967433402214, 1.0954451150103321,
                                    1.4605934866804429]], rtol=1e-15)


def test_rmsnorm_invariants():
    """With gamma = 1 and eps = 0 every row of y has mean square 1; y does not
    change when x and the residual are scaled by the same c > 0; gamma scales
    y column by column; eps > 0 only shrinks the row norm."""
    rng = np.random.default_rng(53)
    x, res = rng.standard_normal((6, 32)), rng.standard_normal((6, 32))
    gamma = rng.uniform(0.5, 2.0, 32)
    r, y = O.add_rmsnorm(x, res, np.ones(32), 0.0)
    np.testing.assert_allclose(r, x + res, rtol=0, atol=0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.add_rmsnorm(3.5 * x, 3.5 * res, np.ones(32), 0.0)[1], y, rtol=1e-13)
    np.testing.assert_allclose(O.add_rmsnorm(x, res, gamma, 0.0)[1], y * gamma, rtol=1e-14)
    assert np.all(np.mean(O.add_rmsnorm(x, res, np.ones(32), 1e-2)[1] ** 2, axis=1) < 1.0)


def test_finalize_add_rmsnorm_composition():
    """finalize_add_rmsnorm = add_rmsnorm(finalize(...)): masked routes add
    nothing (a NaN behind them does not leak), the shared output is added after
    the routed scale, and the normalised rows have unit mean square."""
    rng = np.random.default_rng(59)
    M, k, K, R = 5, 2, 16, 10
    g2 = rng.standard_normal((R, K))
    w = rng.uniform(0.1, 1.0, (M, k))
    pmap = rng.permutation(R)[:M * k].reshape(M, k).astype(np.int32)
    pmap[1, 1] = -1
    w[1, 1] = np.nan
    shared, res = rng.standard_normal((M, K)), rng.standard_normal((M, K))
    r, y = O.finalize_add_rmsnorm(g2, w, pmap, res, np.ones(K), 0.0, shared, 2.5)
    assert np.isfinite(r).all() and np.isfinite(y).all()
    for t in range(M):
        want = shared[t] + res[t] + 2.5 * sum(w[t, j] * g2[pmap[t, j]] for j in range(k) if pmap[t, j] >= 0)
        np.testing.assert_allclose(r[t], want, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- MXFP8 activations

def test_e4m3_decode_matches_library_and_closed_forms():
    """All 256 codes against torch's float8_e4m3fn decode (a library routine),
    and the format's landmarks: 1.0, the largest finite value, the smallest
    normal and subnormal, the NaN codes."""
    codes = np.arange(256)
    ours = O.e4m3_value(codes)
    lib = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    fin = ~np.isnan(ours)
    assert np.array_equal(ours[fin], lib[fin].astype(np.float64))
    assert O.e4m3_value(0x38) == 1.0 and O.e4m3_value(0x7E) == O.E4M3_MAX == 448.0
    assert O.e4m3_value(0x08) == 2.0 ** -6 and O.e4m3_value(0x01) == 2.0 ** -9
    assert O.e4m3_value(0xB8) == -1.0
    assert np.isnan(O.e4m3_value(0x7F)) and np.isnan(O.e4m3_value(0xFF))
    assert np.isnan(ours).sum() == 2


def test_e4m3_round_matches_library_including_ties():
    """Every representable value, every midpoint between neighbours (the
    ties), points just off the midpoints, and random values, against torch's
    round-to-nearest-even float8_e4m3fn cast; saturation at 448 by its own
    closed form (torch does not saturate)."""
    vals = np.unique(O.e4m3_value(np.arange(256))[~np.isnan(O.e4m3_value(np.arange(256)))])
    pos = vals[vals >= 0]
    mids = (pos[1:] + pos[:-1]) / 2
    probe = np.concatenate([vals, mids, -mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20),
                            np.random.default_rng(61).uniform(-448, 448, 20000)]).astype(np.float32)
    ours = O.e4m3_round(probe)
    lib = torch.from_numpy(probe).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    # a tie goes to the even mantissa: 1 + 1/16 lies between 1.0 (m=0) and 1.125 (m=1)
    assert O.e4m3_round(np.float32(1.0625)) == 0x38
    assert O.e4m3_round(np.float32(1.1875)) == 0x3A          # between m=1 and m=2 -> m=2
    for big, code in ((448.0, 0x7E), (463.9, 0x7E), (500.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE)):
        assert O.e4m3_round(np.float32(big)) == code
    assert O.e4m3_round(np.float32(2.0 ** -10)) == 0x00         # half the smallest subnormal: tie to 0
    assert O.e4m3_round(np.float32(-0.0)) == 0x80


@pytest.mark.parametrize("j", [-100, -7, 0, 3, 20, 100])
def test_mxfp8_scale_rule_closed_form(j):
    """For amax in [2^j, 2^(j+1)) the scale is 2^(j-8): amax / scale lies in
    [256, 512); the byte is j + 119. Clamped to 1..254 at the ends."""
    for f in (1.0, 1.3, 1.75, 1.999):
        amax = np.float32(f * 2.0 ** j)
        b = int(O.mxfp8_scale_byte(amax))
        assert b == j + 119
        assert 256 <= float(amax) / 2.0 ** (b - 127) < 512
    assert int(O.mxfp8_scale_byte(np.float32(0.0))) == 1
    assert int(O.mxfp8_scale_byte(np.float32(2.0 ** -130))) == 1
    assert int(O.mxfp8_scale_byte(np.float32(3e38))) == 246          # exponent field 254


def test_mxfp8_qdq_identity_on_representable_blocks():
    """A block whose values are E4M3 values times 2^s, with its largest
    magnitude in [256, 448] * 2^s, is its own quantisation: the scale rule
    picks 2^s and every element is already on the grid."""
    rng = np.random.default_rng(67)
    grid = O.e4m3_value(np.arange(256))
    grid = grid[~np.isnan(grid)]
    rows = []
    for s in (-20, -3, 0, 5):
        for _ in range(8):
            v = rng.choice(grid, 32)
            v[rng.integers(32)] = rng.choice(grid[(np.abs(grid) >= 256)])
            rows.append(v * 2.0 ** s)
    x = np.array(rows).reshape(8, 4 * 32)
    codes, sb = O.mxfp8_quantize(x)
    assert np.array_equal(O.mxfp8_dequantize(codes, sb), x)


def test_mxfp8_qdq_error_bound_and_block_axis():
    """Each value's error is at most half a quantum of its binade: 2^-4 of its
    magnitude for normals, 2^-10 * scale below 2^-6 * scale, and saturation
    only within [448, 512) * scale. Blocks run along the last axis in groups
    of 32: a huge value in one block leaves the next block's precision
    alone, and transposing the input changes the result."""
    rng = np.random.default_rng(71)
    x = (rng.standard_normal((32, 256)) * np.exp(rng.uniform(-8, 8, (32, 1)))).astype(np.float32)
    codes, sb = O.mxfp8_quantize(x)
    q = O.mxfp8_dequantize(codes, sb)
    scale = np.repeat(np.exp2(sb.astype(np.float64) - 127), 32, axis=1)
    a = np.abs(x.astype(np.float64))
    bound = np.where(a / scale >= 2.0 ** -6, 2.0 ** -4 * a, 2.0 ** -10 * scale)
    bound = np.where(a / scale > 448, a - 448 * scale, bound)
    assert np.all(np.abs(q - x) <= bound * (1 + 1e-12))
    y = np.ones((1, 64), np.float32)
    y[0, 0] = 1e6
    y[0, 32:] = np.linspace(1, 2, 32, dtype=np.float32)
    qy = O.mxfp8_qdq(y)
    assert np.all(qy[0, 1:32] == 0.0)                     # swamped by 1e6 in their block
    assert np.all(np.abs(qy[0, 32:] - y[0, 32:]) <= 2.0 ** -4 * y[0, 32:])
    xt = np.ascontiguousarray(x[:, :32].T)
    assert not np.array_equal(O.mxfp8_qdq(xt).T, q[:, :32])


def test_experts_mxfp8_quantises_both_gemm_inputs():
    """experts_mxfp8 = experts with MXFP8 quantisation of x [T, K] before GEMM1
    and of the float32 activation output [T, N] before GEMM2, nothing else:
    with an identity quantiser the result is experts' own (up to the float32
    rounding of the activation), a recording
    quantiser sees exactly those two operands, and the quantised result sits
    within the first-order error bound of the exact one."""
    rng = np.random.default_rng(73)
    E, K, N, M, k = 3, 64, 96, 7, 2
    w1 = rng.standard_normal((E, 2 * N, K)) / np.sqrt(K)
    w2 = rng.standard_normal((E, K, N)) / np.sqrt(N)
    x = O.bf16_round(rng.standard_normal((M, K))).astype(np.float64)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    offs, pmap, inv, _ = O.permute(ids, E)
    exact = O.experts(x, w1, w2, offs, inv, k)
    # identity quantiser: only the activation's float32 rounding remains
    ident = O.experts(x, w1, w2, offs, inv, k, qdq=lambda a: np.asarray(a, np.float64))
    np.testing.assert_allclose(ident, exact, rtol=1e-5, atol=1e-6 * np.abs(exact).max())
    seen = []

    def spy(a):
        seen.append((np.asarray(a).shape, np.asarray(a).dtype))
        return O.mxfp8_qdq(a)
    spied = O.experts(x, w1, w2, offs, inv, k, qdq=spy)
    got = O.experts_mxfp8(x, w1, w2, offs, inv, k)
    assert np.array_equal(spied, got)
    shapes = sorted({s for s, _ in seen})
    assert all(s[1] in (K, N) for s in shapes) and {s[1] for s in shapes} == {K, N}
    assert all(d == np.float32 for s, d in seen if s[1] == N)
    # first-order bound: |dy| <= |W2| (|da|), |da| <= 2^-4 |a| + |d act / dh| |W1| |dx| (loose, x4)
    rel = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert 1e-4 < rel < 0.1


# ---------------------------------------------------------------- activation chunking

@pytest.mark.parametrize("chunk,masked", [(1, False), (3, True), (7, False), (16, True), (40, False)])
def test_experts_chunked(chunk, masked):
    """Chunked experts (one permute + experts per chunk of tokens): each
    chunk's map entries are a bijection onto its own rows [t0*k, t0*k + R_c);
    every route's row holds the same expert output as without chunking; the
    finalize of the chunked triple equals the unchunked one; a chunk of at
    least M tokens is the plain permute."""
    rng = np.random.default_rng(31 + chunk)
    M, K, N, E, k = 23, 32, 48, 6, 2
    x = rng.standard_normal((M, K))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    w = rng.random((M, k))
    emap = None
    E_l = E
    if masked:
        emap = np.array([0, -1, 1, 2, -1, 3], np.int32)
        E_l = 4
    w1 = rng.standard_normal((E_l, 2 * N, K)) / np.sqrt(K)
    w2 = rng.standard_normal((E_l, K, N)) / np.sqrt(N)
    offs, pmap, inv, _ = O.permute(ids, E, emap)
    g2 = O.experts(x, w1, w2, offs, inv, k)
    cmap, cg2 = O.experts_chunked(x, ids, w1, w2, E, chunk, emap)
    assert cmap.shape == (M, k) and cg2.shape == (M * k, K)
    assert np.array_equal(cmap < 0, pmap < 0)                       # -1 exactly on masked routes
    for t0 in range(0, M, chunk):
        t1 = min(M, t0 + chunk)
        part = cmap[t0:t1].reshape(-1)
        valid = part[part >= 0]
        assert sorted(valid.tolist()) == list(range(t0 * k, t0 * k + valid.size))
    for t in range(M):
        for j in range(k):
            if pmap[t, j] >= 0:
                np.testing.assert_allclose(cg2[cmap[t, j]], g2[pmap[t, j]], rtol=1e-12, atol=1e-14)
    out = O.finalize(g2, w, pmap, None, 1.0)
    cout = O.finalize(cg2, w, cmap, None, 1.0)
    assert np.all(np.isfinite(cout))                                # unused (NaN) rows never read
    np.testing.assert_allclose(cout, out, rtol=1e-12, atol=1e-14)
    whole_map, whole_g2 = O.experts_chunked(x, ids, w1, w2, E, M, emap)
    assert np.array_equal(whole_map, pmap)
    R = int(offs[-1])
    np.testing.assert_allclose(whole_g2[:R], g2, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- two-term E4M3 split (MXFP4_A16)

def test_e4m3_split_scale_rule_closed_form():
    """The split's scale is the smallest power of two s with amax <= 448 s:
    then amax / s lies in (224, 448]; an all-zero block gets byte 1."""
    amax = np.concatenate([np.exp2(np.arange(-100, 100)), np.exp2(np.arange(-100, 100)) * 1.75,
                           np.exp2(np.arange(-100, 100)) * np.nextafter(1.75, 2),
                           np.random.default_rng(3).uniform(1e-20, 1e20, 5000)]).astype(np.float32)
    b = O.e4m3_split_scale_byte(amax).astype(np.float64)
    s = np.exp2(b - 127.0)
    a = amax.astype(np.float64)
    assert np.all(a <= 448.0 * s) and np.all(a > 224.0 * s)
    assert O.e4m3_split_scale_byte(np.float32(448.0)) == 127          # 448 = 448 * 2^0: no step up
    assert O.e4m3_split_scale_byte(np.float32(449.0)) == 128
    assert O.e4m3_split_scale_byte(np.float32(0.0)) == 1


def test_e4m3_split_is_exact_on_bf16():
    """hi + lo equals the bf16 value exactly for every element within 2^14 of
    its block's largest magnitude, and within 2^-22 of that magnitude
    otherwise; no code saturates (every |code value| <= 448, no NaN code). Rows
    span 2^-40 .. 2^40, with an all-zero row, a block whose largest value sits
    in (448, 512) times a power of two (the plain MX scale would saturate it),
    a value 2^20 times its neighbours, and bf16 subnormals."""
    rng = np.random.default_rng(41)
    R, C = 96, 512
    x = rng.standard_normal((R, C)) * np.exp2(rng.uniform(-40, 40, (R, 1)))
    x[1] = 0.0
    x[2, :32] = rng.standard_normal(32)
    x[2, 5] = 1.875                                   # 480 * 2^-8
    x[3, 64:96] = rng.standard_normal(32) * 1e-3
    x[3, 70] = 2.0 ** 10
    x[4] = rng.standard_normal(C) * 2.0 ** -130       # bf16 subnormals
    xb = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
    hi, b1, lo, b2 = O.e4m3_split(xb)
    v = O.e4m3_split_value(hi, b1, lo, b2)
    amax = np.repeat(np.abs(xb.reshape(R, C // 32, 32)).max(axis=-1), 32, axis=1)
    near = np.abs(xb) >= amax * 2.0 ** -14
    assert np.array_equal(v[near], xb[near].astype(np.float64))
    assert np.all(np.abs(v - xb) <= amax * 2.0 ** -22)
    for c in (hi, lo):
        assert np.all(np.abs(O.e4m3_value(c)) <= 448.0) and not np.any((c & 0x7F) == 0x7F)
    # hi is the MX-style rounding of x to E4M3 at the split scale
    s1 = np.repeat(np.exp2(b1.astype(np.float64) - 127.0), 32, axis=1)
    assert np.array_equal(hi, O.e4m3_round(xb / s1))
    # the plain MX rule would saturate row 2's first block: the split rule keeps it exact
    sb = O.mxfp8_scale_byte(np.float32(1.875))
    assert 1.875 / 2.0 ** (int(sb) - 127) > 448.0
    assert v[2, 5] == 1.875
