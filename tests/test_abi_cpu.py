"""The C-ABI library builds, loads, exports every declared symbol, and its
host-side validation rejects bad arguments before touching a device. CPU only:
no call here reaches a kernel launch."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_15_gb300 import build
    build.build()
    import mixture_experts_layer_15_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("moe_route", "moe_permute", "moe_experts", "moe_finalize"):
        assert required in names


def test_every_declared_symbol_is_exported(moe):
    names = _declared()
    assert set(names) == set(moe.EXPORTS)
    for n in names:
        assert hasattr(moe.lib, n), n


def test_status_strings(moe):
    for code in range(9):
        assert moe.status_string(code)
    assert moe.status_string(0) == "ok"
    assert moe.status_string(123) == "unknown status"


def _status(fn, *a):
    import mixture_experts_layer_15_gb300 as m
    try:
        fn(*a)
        return 0
    except m.MoEError as e:
        return e.status


def test_route_validation(moe):
    P = 0x1000  # never dereferenced: validation fails first
    S = moe.MOE_ROUTE_SOFTMAX_TOPK
    # num_tokens must be non-negative, top_k positive (convert_flashinfer_moe_output)
    assert _status(moe.moe_route, P, -1, 8, 2, S, None, 1, 1, 1.0, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 8, 0, S, None, 1, 1, 1.0, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 8, 9, S, None, 1, 1, 1.0, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 8, 2, S, P, 1, 1, 1.0, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 8, 2, S, None, 1, 1, 1.0, P, P, 7, 0) == moe.MOE_ERR_INVALID_ARG
    G = moe.MOE_ROUTE_SIGMOID_GROUPED_TOPK
    assert _status(moe.moe_route, P, 4, 256, 8, G, None, 8, 4, 2.5, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 256, 8, G, P, 7, 4, 2.5, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 256, 8, G, P, 8, 9, 2.5, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_route, P, 4, 16, 9, G, P, 8, 4, 2.5, P, P, 1, 0) == moe.MOE_ERR_INVALID_ARG
    # M = 0 is a valid no-op that needs no device
    assert _status(moe.moe_route, None, 0, 8, 2, S, None, 1, 1, 1.0, None, None, 1, 0) == 0


def _weights(moe, K=256, N=256, E=8, fmt=0, scales=False):
    P = 0x1000
    return moe.make_weights(fmt, E, K, N, P, P, P if scales else None, P if scales else None)


def test_experts_validation(moe):
    P = 0x1000
    w = _weights(moe)
    B, F = moe.MOE_DTYPE_BF16, moe.MOE_DTYPE_F32
    call = lambda w, M, k, fin, out, **kw: _status(
        moe.moe_experts, w, P, P, M, k, P, F, fin, P, F, P, None, F, 1.0, out, F, P, 1 << 30, 0)
    # a deferred output cannot have a destination (convert_flashinfer_moe_output)
    O = P + 4096
    assert call(w, 4, 2, 0, O) == moe.MOE_ERR_INVALID_ARG
    assert call(w, -1, 2, 1, O) == moe.MOE_ERR_INVALID_ARG
    assert call(w, 4, 0, 1, O) == moe.MOE_ERR_INVALID_ARG
    assert call(w, 4, 2, 2, O) == moe.MOE_ERR_INVALID_ARG
    assert call(_weights(moe, K=200), 4, 2, 1, O) == moe.MOE_ERR_ALIGNMENT
    assert call(_weights(moe, N=192), 4, 2, 1, O) == moe.MOE_ERR_ALIGNMENT
    assert call(_weights(moe, E=0), 4, 2, 1, O) == moe.MOE_ERR_INVALID_ARG
    assert call(_weights(moe, fmt=1), 4, 2, 1, O) == moe.MOE_ERR_INVALID_ARG      # MXFP4 needs scales
    assert call(_weights(moe, scales=True), 4, 2, 1, O) == moe.MOE_ERR_INVALID_ARG  # bf16 takes none
    # finalized output to its own destination only: out may not alias gemm2
    assert _status(moe.moe_experts, w, P, P, 4, 2, P, F, 1, P + 64, F, P + 128, None, F, 1.0, P, F,
                   P, 1 << 30, 0) == moe.MOE_ERR_INVALID_ARG
    # M = 0: nothing arrives, nothing to do
    assert call(w, 0, 2, 1, P + 4096) == 0
    assert call(w, 0, 2, 0, None) == 0


def test_finalize_and_permute_validation(moe):
    P = 0x1000
    F = moe.MOE_DTYPE_F32
    fin = lambda M, k, K, out, g2=P: _status(moe.moe_finalize, g2, F, 8, P, F, P, M, k, K, None, F, 1.0,
                                            out, F, 0)
    assert fin(-1, 2, 128, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert fin(4, 0, 128, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert fin(4, 2, 100, P + 4096) == moe.MOE_ERR_ALIGNMENT
    assert fin(4, 2, 128, None) == moe.MOE_ERR_INVALID_ARG
    assert fin(4, 2, 128, P) == moe.MOE_ERR_INVALID_ARG          # out aliases gemm2_permuted
    assert fin(0, 2, 128, None) == 0
    perm = lambda M, k, E, emap, El: _status(moe.moe_permute, P, M, k, E, emap, El, P, 128, P, P, P, P,
                                             P, 1 << 20, 0)
    assert perm(-1, 2, 8, None, 8) == moe.MOE_ERR_INVALID_ARG
    assert perm(4, 0, 8, None, 8) == moe.MOE_ERR_INVALID_ARG
    assert perm(4, 2, 8, None, 4) == moe.MOE_ERR_INVALID_ARG     # no map: E_local must be E
    assert perm(4, 9, 8, None, 8) == moe.MOE_ERR_INVALID_ARG


def test_workspace_sizes_are_host_computable(moe):
    w = moe.make_weights(0, 8, 4096, 14336, 0x1000, 0x1000)
    small = moe.moe_experts_workspace_size(w, 1, 2)
    big = moe.moe_experts_workspace_size(w, 8192, 2)
    assert small > 0 and big > 8192 * 2 * 14336 * 2      # holds the bf16 activations
    assert moe.moe_permute_workspace_size(16, 2, 8) == 0     # one chunk: no scratch
    assert moe.moe_permute_workspace_size(8192, 8, 128) > 0
    assert moe.moe_shared_expert_workspace_size(64, 7168, 2048) > 64 * 2048 * 2


def test_mxfp8_entries_validate_on_the_host(moe):
    """The MXFP4-weight x MXFP8-activation format and its helpers: argument
    rules that fail before any device is touched, and the host-computed
    sizes (the scale atoms, the workspace with codes and atoms)."""
    P = 0x1000                                               # 32-byte aligned, never dereferenced
    A8 = moe.MOE_WEIGHTS_MXFP4_A8
    # prepared scales: 512-byte atoms per 128 rows x 128 columns per expert
    assert moe.moe_mx_prepared_scales_size(256, 4096, 7168) == 256 * 32 * 56 * 512
    assert moe.moe_mx_prepared_scales_size(2, 100, 256) == 0
    assert moe.moe_mx_prepared_scales_size(0, 128, 128) == 0
    assert _status(moe.moe_mx_prepare_scales, P, 2, 100, 256, P) == moe.MOE_ERR_ALIGNMENT
    assert _status(moe.moe_mx_prepare_scales, P + 2, 2, 128, 256, P) == moe.MOE_ERR_ALIGNMENT
    assert _status(moe.moe_mx_prepare_scales, None, 2, 128, 256, P) == moe.MOE_ERR_INVALID_ARG
    # the quantiser: C a multiple of 128, 16-byte aligned rows; rows = 0 is a no-op
    assert _status(moe.moe_mxfp8_quantize, P, 4, 96, P, P) == moe.MOE_ERR_ALIGNMENT
    assert _status(moe.moe_mxfp8_quantize, P + 8, 4, 128, P, P) == moe.MOE_ERR_ALIGNMENT
    assert _status(moe.moe_mxfp8_quantize, P, -1, 128, P, P) == moe.MOE_ERR_INVALID_ARG
    assert _status(moe.moe_mxfp8_quantize, P, 0, 128, None, None) == 0
    # the weight format: prepared scales required, codes 32-byte aligned, K % 256 == 0
    w = moe.make_weights(A8, 8, 7168, 2048, P, P, P, P)
    assert moe.moe_experts_workspace_size(w, 64, 8) > 64 * 8 * (7168 + 2048)   # x and act codes
    assert moe.moe_experts_workspace_size(moe.make_weights(A8, 8, 7168, 2048, P, P), 64, 8) == 0
    assert moe.moe_experts_workspace_size(moe.make_weights(A8, 8, 7168, 2048, P + 16, P, P, P), 64, 8) == 0
    assert moe.moe_experts_workspace_size(moe.make_weights(A8, 8, 384, 2048, P, P, P, P), 64, 8) == 0
    F = moe.MOE_DTYPE_F32
    # the BatchedExperts entry does not take the format
    assert _status(moe.moe_experts_batched, w, P, P, 4, P + 4096, F, P, 1 << 30) == moe.MOE_ERR_UNSUPPORTED


def test_permute_noalloc_validates_like_moe_permute(moe):
    """The no-alloc permute shares moe_permute's host checks: the same bad
    arguments give the same status, before any device is touched, plus its
    own limit (a problem whose histograms exceed the fixed 1 MiB scratch)."""
    P = 0x1000                                               # never dereferenced
    na = lambda M, k, E, emap, El, ids=P, offs=P, pmap=P, inv=P, x=P, xp=P, K=128: _status(
        moe.moe_permute_noalloc, ids, M, k, E, emap, El, x, K, offs, pmap, inv, xp)
    wp = lambda M, k, E, emap, El, ids=P, offs=P, pmap=P, inv=P, x=P, xp=P, K=128: _status(
        moe.moe_permute, ids, M, k, E, emap, El, x, K, offs, pmap, inv, xp, P, 1 << 30)
    cases = [
        dict(M=-1, k=2, E=8, emap=None, El=8),                      # num_tokens >= 0
        dict(M=4, k=0, E=8, emap=None, El=8),                       # top_k > 0
        dict(M=4, k=9, E=8, emap=None, El=8),                       # top_k <= E
        dict(M=4, k=2, E=2048, emap=P, El=1025),                    # E_local <= 1024
        dict(M=4, k=2, E=8, emap=None, El=4),                       # no map: E_local == E
        dict(M=1 << 27, k=8, E=128, emap=None, El=128),             # M * top_k < 2^30
        dict(M=4, k=2, E=8, emap=None, El=8, ids=None),             # required pointers
        dict(M=4, k=2, E=8, emap=None, El=8, offs=None),
        dict(M=4, k=2, E=8, emap=None, El=8, pmap=None),
        dict(M=4, k=2, E=8, emap=None, El=8, inv=None),
        dict(M=4, k=2, E=8, emap=None, El=8, x=None),               # x needed for x_perm
        dict(M=4, k=2, E=8, emap=None, El=8, K=100),                # 16-byte row gather
        dict(M=4, k=2, E=8, emap=None, El=8, x=P + 8),
    ]
    want = [moe.MOE_ERR_INVALID_ARG] * 5 + [moe.MOE_ERR_UNSUPPORTED] + [moe.MOE_ERR_INVALID_ARG] * 5 + \
        [moe.MOE_ERR_ALIGNMENT] * 2
    for c, w in zip(cases, want):
        assert na(**c) == w, c
        assert wp(**c) == w, c
    # beyond the fixed scratch: 2^21 + 1024 routes at 128 local experts
    M = (1 << 18) + 128
    assert moe.moe_permute_workspace_size(M, 8, 128) > (1 << 20)
    assert na(M, 8, 128, None, 128) == moe.MOE_ERR_WORKSPACE


def test_chunked_workspace_is_sized_by_the_chunk(moe):
    """Activation chunking caps the scratch: the chunked workspace depends on
    M only through the ragged tail, so it is the same for every multiple of
    the chunk, and far below the unchunked permute + experts workspaces."""
    w = moe.make_weights(0, 128, 2048, 768, 0x1000, 0x1000)
    a = moe.moe_experts_chunked_workspace_size(w, 8192, 8, 1024)
    b = moe.moe_experts_chunked_workspace_size(w, 4096, 8, 1024)
    c = moe.moe_experts_chunked_workspace_size(w, 65536, 8, 1024)
    assert a == b == c > 0
    whole = moe.moe_experts_workspace_size(w, 65536, 8) + 65536 * 8 * 2048 * 2
    assert c * 8 < whole
    assert moe.moe_experts_chunked_workspace_size(w, 8192, 8, 0) == 0
    P = 0x1000
    F = moe.MOE_DTYPE_F32
    call = lambda M, k, E, chunk, fin, out: _status(moe.moe_experts_chunked, w, P, P, M, k, E, None, chunk, P, P,
                                                    F, fin, P, F, None, F, 1.0, out, F, P, 1 << 30)
    assert call(64, 8, 128, 0, 1, P + 4096) == moe.MOE_ERR_INVALID_ARG       # chunk_tokens >= 1
    assert call(64, 8, 128, 16, 0, P + 4096) == moe.MOE_ERR_INVALID_ARG      # deferred: no destination
    assert call(64, 8, 64, 16, 1, P + 4096) == moe.MOE_ERR_INVALID_ARG       # no map: E_local must be E
    assert call(-1, 8, 128, 16, 1, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert call(0, 8, 128, 16, 0, None) == 0                                  # nothing to do


def test_fused_finalize_x_validates_on_the_host(moe):
    """The token-order experts entry: its workspace holds the gathered rows
    only for formats that read x_perm by TMA, and its argument rules fail
    before any device is touched."""
    P = 0x1000
    F = moe.MOE_DTYPE_F32
    bf = moe.make_weights(0, 8, 4096, 1024, P, P)
    a16 = moe.make_weights(moe.MOE_WEIGHTS_MXFP4_A16, 8, 4096, 1024, P, P, P, P)
    M, k = 512, 2
    assert moe.moe_experts_x_workspace_size(bf, M, k) >= moe.moe_experts_workspace_size(bf, M, k) + M * k * 4096 * 2
    assert moe.moe_experts_x_workspace_size(a16, M, k) == moe.moe_experts_workspace_size(a16, M, k)
    call = lambda w, x, M, k, out: _status(moe.moe_experts_fused_finalize_x, w, x, P, M, k, P, F, P, None, F, 1.0,
                                           out, P, 1 << 30)
    assert call(bf, P, -1, k, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert call(bf, P, M, 0, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert call(bf, None, M, k, P + 4096) == moe.MOE_ERR_INVALID_ARG            # x required
    assert call(bf, P + 8, M, k, P + 4096) == moe.MOE_ERR_ALIGNMENT
    assert call(bf, P, M, k, P) == moe.MOE_ERR_INVALID_ARG                      # out may not alias x
    assert call(bf, P, 0, k, P + 4096) == 0                                     # nothing to do


def test_fused_finalize_after_validates_on_the_host(moe):
    """The preset-start experts entry: x_order picks x_perm (0) or token
    order (1); its argument rules fail before any device is touched, and an
    empty batch is a no-op whatever the event."""
    P = 0x1000
    F = moe.MOE_DTYPE_F32
    bf = moe.make_weights(0, 8, 4096, 1024, P, P)
    M, k = 512, 2
    call = lambda x, order, M, k, wts, out: _status(moe.moe_experts_fused_finalize_after, bf, x, order, P, M, k,
                                                    wts, F, P, 1.0, out, None, P, 1 << 30)
    assert call(P, 2, M, k, P, P + 4096) == moe.MOE_ERR_INVALID_ARG             # x_order 0 or 1
    assert call(P, -1, M, k, P, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert call(P, 0, -1, k, P, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert call(P, 1, M, 0, P, P + 4096) == moe.MOE_ERR_INVALID_ARG
    assert call(P, 0, M, k, None, P + 4096) == moe.MOE_ERR_INVALID_ARG          # routing weights required
    assert call(P, 0, M, k, P, None) == moe.MOE_ERR_INVALID_ARG                 # out required
    assert call(P, 1, M, k, P, P + 8) == moe.MOE_ERR_ALIGNMENT
    assert call(P, 0, M, k, P, P) == moe.MOE_ERR_INVALID_ARG                    # out may not alias x
    assert call(None, 1, M, k, P, P + 4096) == moe.MOE_ERR_INVALID_ARG          # x required
    assert call(P + 8, 1, M, k, P, P + 4096) == moe.MOE_ERR_ALIGNMENT
    assert call(P, 0, 0, k, P, P + 4096) == 0                                   # nothing to do
