"""Test helpers: build/import the library, per-expert float64 views of device
weights for the oracle, and the oracle's output on a sample of tokens."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O


def lib():
    from mixture_experts_layer_15_gb300 import build
    build.build()
    import mixture_experts_layer_15_gb300 as m
    return m


def tol(ref, rel=1e-2, abs_=1e-3):
    """The value bar: max |gpu - ref| <= rel * RMS(ref) + abs."""
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
    return rel * rms + abs_


def max_err(got, ref):
    return float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))


_DEQ_CACHE = {}


class ExpertsF64:
    """``[e]`` -> float64 numpy weights of local expert e, converted lazily
    (bf16 tensors, or MXFP4 bytes dequantised by the oracle; the latter kept
    in a bounded cache, since dequantising one expert takes seconds)."""

    def __init__(self, w, scale=None, cache=64):
        self.w, self.scale, self.cache = w, scale, cache

    def __len__(self):
        return self.w.shape[0]

    def __getitem__(self, e):
        if self.scale is None:
            return self.w[e].to(torch.float64).cpu().numpy()
        key = (self.w.data_ptr(), tuple(self.w.shape), int(e))
        if key not in _DEQ_CACHE:
            if len(_DEQ_CACHE) >= self.cache:
                _DEQ_CACHE.pop(next(iter(_DEQ_CACHE)))
            _DEQ_CACHE[key] = O.dequant_mxfp4(self.w[e].cpu().numpy(),
                                              self.scale[e].cpu().numpy()).astype(np.float32)
        return _DEQ_CACHE[key].astype(np.float64)

    @property
    def shape(self):
        s = tuple(self.w.shape)
        return s if self.scale is None else s[:-1] + (s[-1] * 2,)


def oracle_tokens(x, ids, weights, w1, w2, tokens, expert_map=None, shared=None, rsf=1.0, activation="silu",
                  clamp=None, qdq=None):
    """Oracle output rows for ``tokens`` (and the expert output y of each of
    their routes): the experts and finalize of the oracle applied to the
    sub-problem made of those tokens' routes.

    x: float64 [M, K]; ids int [M, k]; weights float64 [M, k]; w1/w2 indexable
    per local expert; shared: float64 [M, K] or None; qdq: the activations'
    quantisation (oracle.expert_mlp), or None.
    Returns (out [T, K], y dict {(t, j): [K]}).
    """
    tokens = list(tokens)
    k = ids.shape[1]
    emap = None if expert_map is None else np.asarray(expert_map)
    sub_ids = ids[tokens]
    local = sub_ids if emap is None else emap[sub_ids]
    by_expert = {}
    for a, t in enumerate(tokens):
        for j in range(k):
            le = int(local[a, j])
            if le >= 0:
                by_expert.setdefault(le, []).append((a, j))
    ys = {}
    for le, routes in by_expert.items():
        xt = x[[tokens[a] for a, _ in routes]]
        y = O.expert_mlp(xt, w1[le], w2[le], activation, clamp, qdq)
        for r, (a, j) in enumerate(routes):
            ys[(a, j)] = y[r]
    # sub-problem gemm2 rows and map, then the oracle's finalize
    rows, pmap = [], np.full((len(tokens), k), -1, np.int32)
    for (a, j), y in ys.items():
        pmap[a, j] = len(rows)
        rows.append(y)
    K = x.shape[1]
    g2 = np.stack(rows) if rows else np.zeros((0, K))
    sh = None if shared is None else shared[tokens]
    out = O.finalize(g2, weights[tokens], pmap, sh, rsf)
    return out, {(tokens[a], j): y for (a, j), y in ys.items()}


def sample_tokens_few_experts(ids, n, budget, seed=0):
    """Up to n tokens whose routes together touch at most ``budget`` experts
    (the first and last token always considered), for oracles whose cost is
    per expert."""
    M = ids.shape[0]
    order = [0, M - 1] + np.random.default_rng(seed).permutation(M).tolist()
    seen, toks = set(), []
    for t in order:
        if t in toks:
            continue
        new = set(int(e) for e in ids[t]) - seen
        if len(seen) + len(new) <= budget:
            seen |= new
            toks.append(int(t))
        if len(toks) >= n:
            break
    return sorted(toks)


def sample_tokens(M, n=256, seed=0):
    if M <= n:
        return list(range(M))
    rng = np.random.default_rng(seed)
    s = set(rng.choice(M, size=n - 2, replace=False).tolist()) | {0, M - 1}
    return sorted(s)


# ------------------------------------------------------------------ oracle on many MXFP4 experts

def _expert_job(args):
    """Pool worker: the oracle's expert MLP of one local expert on its rows,
    from the packed MXFP4 bytes (dequantised here, by the oracle) or from
    float64 weights. Runs in a spawned CPU process."""
    import oracle as Oc
    x, w1, s1, w2, s2, activation, clamp, mxfp8 = args
    if s1 is not None:
        w1 = Oc.dequant_mxfp4(w1, s1)
        w2 = Oc.dequant_mxfp4(w2, s2)
    return Oc.expert_mlp(x, w1, w2, activation, clamp, Oc.mxfp8_qdq if mxfp8 else None)


_POOL = None


def oracle_pool():
    """A process pool for the oracle, started with ``spawn`` (a pool forked
    from a process that already holds a CUDA context can hang)."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        import os
        n = max(1, min(16, (os.cpu_count() or 2) - 1))
        _POOL = mp.get_context("spawn").Pool(n)
    return _POOL


def oracle_tokens_mxfp4(x, ids, weights, w1, s1, w2, s2, tokens, expert_map=None, shared=None, rsf=1.0,
                        activation="silu", clamp=None, mxfp8=False):
    """oracle_tokens for MXFP4 experts given as packed bytes (torch tensors
    [E_local, rows, cols/2] and scales [E_local, rows, cols/32], any device):
    each local expert touched by the sampled tokens is dequantised once, in a
    worker of the spawned oracle pool, and evaluated on all its sampled
    routes; ``mxfp8`` quantises both GEMM inputs as the MXFP8-activation
    format does (oracle.mxfp8_qdq). Returns (out [T, K], y dict {(t, j): [K]})."""
    tokens = list(tokens)
    k = ids.shape[1]
    emap = None if expert_map is None else np.asarray(expert_map)
    local = ids[tokens] if emap is None else emap[ids[tokens]]
    by_expert = {}
    for a in range(len(tokens)):
        for j in range(k):
            le = int(local[a, j])
            if le >= 0:
                by_expert.setdefault(le, []).append((a, j))
    experts = sorted(by_expert)
    jobs = [(x[[tokens[a] for a, _ in by_expert[le]]], w1[le].cpu().numpy(), s1[le].cpu().numpy(),
             w2[le].cpu().numpy(), s2[le].cpu().numpy(), activation, clamp, mxfp8) for le in experts]
    results = oracle_pool().map(_expert_job, jobs, chunksize=1)
    ys = {}
    for le, y in zip(experts, results):
        for r, (a, j) in enumerate(by_expert[le]):
            ys[(a, j)] = y[r]
    rows, pmap = [], np.full((len(tokens), k), -1, np.int32)
    for (a, j), y in ys.items():
        pmap[a, j] = len(rows)
        rows.append(y)
    K = x.shape[1]
    g2 = np.stack(rows) if rows else np.zeros((0, K))
    sh = None if shared is None else shared[tokens]
    out = O.finalize(g2, weights[tokens], pmap, sh, rsf)
    return out, {(tokens[a], j): y for (a, j), y in ys.items()}


def sample_tokens_covering(ids, n, expert_map=None, seed=0):
    """A token sample of at least min(n, M) tokens in which every expert that
    any token routes to (every local one, with a map) appears at least once:
    the first and last token, then tokens in a seeded random order, taking
    first every token that brings an expert not yet covered, then filling up
    to n."""
    M = ids.shape[0]
    emap = None if expert_map is None else np.asarray(expert_map)
    loc = ids if emap is None else emap[ids]
    want = set(int(e) for e in np.unique(loc) if e >= 0)
    order = [0, M - 1] + np.random.default_rng(seed).permutation(M).tolist()
    seen, toks = set(), []
    for t in order:
        if t in toks:
            continue
        new = set(int(e) for e in loc[t] if e >= 0) - seen
        if new or len(toks) < 2:
            seen |= new
            toks.append(int(t))
        if seen == want:
            break
    for t in order:
        if len(toks) >= min(n, M):
            break
        if t not in toks:
            toks.append(int(t))
    return sorted(toks)
