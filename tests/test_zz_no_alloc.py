"""moe_permute_noalloc -- the permute for callers that cannot allocate device
memory (graph capture into a fixed pool, runtimes that reserve the
allocator, paths that must never call cudaMalloc) -- must give exactly what
moe_permute gives with a caller-provided workspace.

The scratch of the no-alloc variant is a fixed array inside the library that
all calls share, so the test runs two different problems back to back and
checks both. The problems span many 1024-route chunks, so the scratch is
really used. Integer results are compared bit for bit, the gathered rows
bitwise: the same bar as the permute's parity tests.

This file is collected last and must pass alone in a fresh process as well
as after the other tests.
"""
import numpy as np
import pytest
import torch

import synth
from _helpers import lib

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def moe():
    m = lib()
    assert m.moe_device_check() == 0, "needs a compute capability 10.3 device"
    return m


def _outputs(M, k, E_l, K):
    i32 = dict(dtype=torch.int32, device=DEV)
    return (torch.full((E_l + 1,), -5, **i32), torch.full((M, k), -5, **i32),
            torch.full((M * k,), -5, **i32), torch.zeros(M * k, K, dtype=torch.bfloat16, device=DEV))


def _problem(seed, M, cfg, masked):
    g = torch.Generator(device="cpu").manual_seed(seed)
    logits = torch.randn(M, cfg.E, generator=g) + torch.randn(cfg.E, generator=g) * 1.5
    ids = torch.topk(logits, cfg.top_k, dim=1).indices.to(torch.int32)
    x = torch.randn(M, 256, generator=g).to(torch.bfloat16)
    emap, E_l = None, cfg.E
    if masked:
        em, E_l = synth.masked_expert_map(cfg.E, seed=seed)
        emap = em.to(DEV)
    return ids.to(DEV), x.to(DEV), emap, E_l


@pytest.mark.parametrize("masked", [False, True])
def test_noalloc_matches_workspace_permute_on_consecutive_calls(moe, masked):
    cfg = synth.CONFIGS["qwen3"]
    K = 256
    for call, (seed, M) in enumerate([(11, 8192), (12, 3000)]):
        ids, x, emap, E_l = _problem(seed, M, cfg, masked)
        k = cfg.top_k
        assert moe.moe_permute_workspace_size(M, k, E_l) > 0          # several chunks: scratch in use
        ref = _outputs(M, k, E_l, K)
        wsb = moe.moe_permute_workspace_size(M, k, E_l)
        ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
        moe.moe_permute(ids, M, k, cfg.E, emap, E_l, x, K, *ref, ws, wsb)
        got = _outputs(M, k, E_l, K)
        moe.moe_permute_noalloc(ids, M, k, cfg.E, emap, E_l, x, K, *got)
        torch.cuda.synchronize()
        assert moe.moe_get_error() == 0
        R = int(ref[0][-1].item())
        assert torch.equal(got[0], ref[0]), f"offsets differ on call {call}"
        assert torch.equal(got[1], ref[1]), f"permute map differs on call {call}"
        assert torch.equal(got[2][:R], ref[2][:R]), f"inverse map differs on call {call}"
        assert torch.equal(got[3][:R], ref[3][:R]), f"gathered rows differ on call {call}"


def test_noalloc_rejects_problems_beyond_its_scratch(moe):
    # 2^21 + 1024 routes at 128 local experts need more than the 1 MiB scratch
    M, k, E = (1 << 18) + 128, 8, 128
    assert moe.moe_permute_workspace_size(M, k, E) > (1 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_permute_noalloc(dummy, M, k, E, None, E, None, 0, dummy, dummy, dummy, None)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
