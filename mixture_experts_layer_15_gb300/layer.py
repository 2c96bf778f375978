"""The whole MoE layer forward as a sequence of C-ABI calls.

``MoELayer`` holds device weights and reusable device buffers (allocated with
torch, which is only the allocator and stream provider here) and runs
moe_route -> moe_permute -> [moe_shared_expert] -> moe_experts(+finalize), the
order of vllm/model_executor/layers/fused_moe/modular_kernel.py,
FusedMoEModularKernel.forward with the dispatch/combine being no-ops on one
GPU. Every arithmetic step runs in the CUDA library.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import _lib as L

_TORCH = {L.MOE_DTYPE_BF16: torch.bfloat16, L.MOE_DTYPE_F32: torch.float32}


@dataclasses.dataclass
class Buffers:
    M: int
    topk_ids: torch.Tensor
    topk_weights: torch.Tensor
    offsets: torch.Tensor
    pmap: torch.Tensor
    inverse: torch.Tensor
    x_perm: torch.Tensor
    gemm2: torch.Tensor
    out: torch.Tensor
    shared: Optional[torch.Tensor]
    perm_ws: torch.Tensor
    exp_ws: torch.Tensor
    shared_ws: Optional[torch.Tensor]


def _as_stream(stream):
    """The torch stream for a stream argument of the binding (None: current)."""
    if stream is None:
        return torch.cuda.current_stream()
    if isinstance(stream, int):
        return torch.cuda.ExternalStream(stream)
    return stream


class MoELayer:
    """One MoE layer on the current CUDA device.

    w1/w2 (and scales) hold the E_local local experts; ``expert_map`` (int32
    [E]) maps global expert ids to local ids (-1 = not local). Routing weights,
    gemm2_permuted and the output are stored in the given dtypes (float32 by
    default: see the precision notes of the C ABI). ``fused_finalize`` (f32
    output only) folds the finalize into GEMM2 (moe_experts_fused_finalize):
    no gemm2_permuted round trip, the top-k reduction order is not fixed.
    With ``fmt`` = MOE_WEIGHTS_MXFP4_A8 the MXFP4 weights are given as for
    MOE_WEIGHTS_MXFP4 (codes + row-major E8M0 scales); the layer rearranges
    the scales once (moe_mx_prepare_scales) and the experts run with MXFP8
    activations on the block-scaled tensor cores. MOE_WEIGHTS_MXFP4_A16 takes
    the same weights and keeps bf16 activations (W4A16), each split into two
    E4M3 terms for the block-scaled tensor cores. With a shared expert and
    ``fused_finalize``, ``overlap_shared`` (the default then) runs the shared
    expert on a second stream, writing its output straight into ``out`` as the
    start that the routed experts add into (moe_experts_fused_finalize_after);
    the buffers' ``shared`` tensor is then not written.
    """

    def __init__(self, *, K, N, E, top_k, w1, w2, w1_scale=None, w2_scale=None,
                 fmt=L.MOE_WEIGHTS_BF16, route="softmax", score_bias=None, n_group=1, topk_group=1,
                 routed_scaling_factor=1.0, expert_map=None, E_local=None, ws1=None, ws2=None,
                 weights_dtype=L.MOE_DTYPE_F32, gemm2_dtype=L.MOE_DTYPE_F32,
                 out_dtype=L.MOE_DTYPE_F32, fused_finalize=False, activation="silu", activation_clamp=None,
                 gather_in_experts=None, overlap_shared=None):
        self.K, self.N, self.E, self.top_k = K, N, E, top_k
        self.E_local = E if E_local is None else E_local
        self.w1, self.w2, self.w1_scale, self.w2_scale = w1, w2, w1_scale, w2_scale
        self.fmt = fmt
        self.method = (L.MOE_ROUTE_SOFTMAX_TOPK if route == "softmax"
                       else L.MOE_ROUTE_SIGMOID_GROUPED_TOPK)
        self.score_bias = score_bias
        self.n_group, self.topk_group = n_group, topk_group
        self.rsf = float(routed_scaling_factor)
        self.expert_map = expert_map
        self.ws1, self.ws2 = ws1, ws2
        self.Ns = 0 if ws1 is None else ws1.shape[0] // 2
        self.weights_dtype, self.gemm2_dtype, self.out_dtype = weights_dtype, gemm2_dtype, out_dtype
        if fused_finalize and out_dtype != L.MOE_DTYPE_F32:
            raise ValueError("fused_finalize accumulates into an f32 output")
        self.fused_finalize = bool(fused_finalize)
        # the folded finalize can read x in token order and gather its rows in
        # the experts (moe_experts_fused_finalize_x); None: on the block-scaled
        # formats, whose quantiser then reads x directly, for batches past the
        # one-kernel route + permute (M > 64), which copies its rows cheaply
        self.gather_in_experts = gather_in_experts
        # with the folded finalize the shared expert runs on a second stream
        # beside the router, the permute and the routed experts' first
        # launches, writing the output start into out itself
        # (moe_experts_fused_finalize_after); None: whenever there is one
        self.overlap_shared = (ws1 is not None and self.fused_finalize) if overlap_shared is None \
            else bool(overlap_shared) and ws1 is not None and self.fused_finalize
        self._side = None
        act = {"silu": L.MOE_ACT_SILU, "gelu": L.MOE_ACT_GELU}[activation]
        if fmt in (L.MOE_WEIGHTS_MXFP4_A8, L.MOE_WEIGHTS_MXFP4_A16):
            w1_scale = self._prepare_scales(w1_scale, 2 * N, K)
            w2_scale = self._prepare_scales(w2_scale, K, N)
            self.w1_scale, self.w2_scale = w1_scale, w2_scale
        self.cw = L.make_weights(fmt, self.E_local, K, N, w1, w2, w1_scale, w2_scale, act, activation_clamp)
        self._bufs = {}

    def gathers_in_experts(self, M: int) -> bool:
        """Whether a folded-finalize forward of M tokens gathers the rows in the
        experts (moe_experts_fused_finalize_x) instead of in the permute."""
        if self.gather_in_experts is not None:
            return bool(self.gather_in_experts)
        return self.fmt in (L.MOE_WEIGHTS_MXFP4_A8, L.MOE_WEIGHTS_MXFP4_A16) and M > 64

    def _prepare_scales(self, scales, rows, cols):
        out = torch.empty(L.moe_mx_prepared_scales_size(self.E_local, rows, cols), dtype=torch.uint8,
                          device=scales.device)
        L.moe_mx_prepare_scales(scales, self.E_local, rows, cols, out)
        return out

    def buffers(self, M: int) -> Buffers:
        b = self._bufs.get(M)
        if b is not None:
            return b
        dev = self.w1.device
        R = max(M * self.top_k, 1)
        i32 = dict(dtype=torch.int32, device=dev)
        pws = L.moe_permute_workspace_size(M, self.top_k, self.E_local)
        ews = max(L.moe_experts_workspace_size(self.cw, M, self.top_k),
                  L.moe_experts_x_workspace_size(self.cw, M, self.top_k))
        shared = shared_ws = None
        if self.ws1 is not None:
            shared = torch.empty(M, self.K, dtype=_TORCH[self.gemm2_dtype], device=dev)
            sws = L.moe_shared_expert_workspace_size(M, self.K, self.Ns)
            shared_ws = torch.zeros(max(sws, 16), dtype=torch.uint8, device=dev)
        b = Buffers(
            M=M,
            topk_ids=torch.empty(M, self.top_k, **i32),
            topk_weights=torch.empty(M, self.top_k, dtype=_TORCH[self.weights_dtype], device=dev),
            offsets=torch.empty(self.E_local + 1, **i32),
            pmap=torch.empty(M, self.top_k, **i32),
            inverse=torch.empty(R, **i32),
            x_perm=torch.empty(R, self.K, dtype=torch.bfloat16, device=dev),
            gemm2=torch.empty(R, self.K, dtype=_TORCH[self.gemm2_dtype], device=dev),
            out=torch.empty(M, self.K, dtype=_TORCH[self.out_dtype], device=dev),
            shared=shared,
            perm_ws=torch.empty(max(pws, 16), dtype=torch.uint8, device=dev),
            # zero-filled once: the split-K counters in it start at zero
            exp_ws=torch.zeros(max(ews, 16), dtype=torch.uint8, device=dev),
            shared_ws=shared_ws,
        )
        self._bufs[M] = b
        return b

    def route(self, logits, b: Buffers, stream=None):
        M = logits.shape[0]
        L.moe_route(logits, M, self.E, self.top_k, self.method, self.score_bias, self.n_group,
                    self.topk_group, self.rsf if self.method == L.MOE_ROUTE_SIGMOID_GROUPED_TOPK else 1.0,
                    b.topk_ids, b.topk_weights, self.weights_dtype, stream)

    def forward(self, x, logits, do_finalize=True, stream=None, topk_ids=None, topk_weights=None) -> Buffers:
        """Run the layer on x bf16 [M, K] and logits f32 [M, E]; returns the
        buffers (out, gemm2_permuted, map, ...). ``topk_ids``/``topk_weights``
        skip the router and use the given routing instead."""
        M = x.shape[0]
        b = self.buffers(M)
        # with the row gather folded into the experts the permute copies no rows
        gx = do_finalize and self.fused_finalize and self.gathers_in_experts(M)
        xp = None if gx else b.x_perm
        side = do_finalize and self.overlap_shared
        if side:
            main = _as_stream(stream)
            if self._side is None:
                self._side = (torch.cuda.Stream(device=x.device), torch.cuda.Event(), torch.cuda.Event())
            sstream, ev_in, ev_sh = self._side
            # the shared expert writes out's start (f32) on the second stream
            ev_in.record(main)
            sstream.wait_event(ev_in)
            L.moe_shared_expert(self.ws1, self.ws2, self.K, self.Ns, x, M, b.out, L.MOE_DTYPE_F32,
                                b.shared_ws, b.shared_ws.numel(), sstream)
            ev_sh.record(sstream)
        if topk_ids is None:
            # route and permute (one kernel for small batches)
            rsf = self.rsf if self.method == L.MOE_ROUTE_SIGMOID_GROUPED_TOPK else 1.0
            L.moe_route_permute(logits, M, self.E, self.top_k, self.method, self.score_bias, self.n_group,
                                self.topk_group, rsf, b.topk_ids, b.topk_weights, self.weights_dtype,
                                self.expert_map, self.E_local, x, self.K, b.offsets, b.pmap, b.inverse, xp,
                                b.perm_ws, b.perm_ws.numel(), stream)
            ids, wts = b.topk_ids, b.topk_weights
        else:
            ids, wts = topk_ids, topk_weights
            L.moe_permute(ids, M, self.top_k, self.E, self.expert_map, self.E_local, x, self.K, b.offsets,
                          b.pmap, b.inverse, xp, b.perm_ws, b.perm_ws.numel(), stream)
        if self.ws1 is not None and not side:
            L.moe_shared_expert(self.ws1, self.ws2, self.K, self.Ns, x, M, b.shared, self.gemm2_dtype,
                                b.shared_ws, b.shared_ws.numel(), stream)
        # the sigmoid router folds the routed scale into its weights
        rsf = 1.0 if self.method == L.MOE_ROUTE_SIGMOID_GROUPED_TOPK else self.rsf
        wdt = L.MOE_DTYPE_F32 if wts.dtype == torch.float32 else L.MOE_DTYPE_BF16
        if side:
            # routed contributions added into the start, once the second stream
            # has written it (waited for before the first launch that adds)
            L.moe_experts_fused_finalize_after(self.cw, x if gx else b.x_perm, 1 if gx else 0, b.offsets, M,
                                               self.top_k, wts, wdt, b.inverse, rsf, b.out, ev_sh, b.exp_ws,
                                               b.exp_ws.numel(), main)
            return b
        if do_finalize and self.fused_finalize:
            if gx:
                L.moe_experts_fused_finalize_x(self.cw, x, b.offsets, M, self.top_k, wts, wdt, b.inverse, b.shared,
                                               self.gemm2_dtype, rsf, b.out, b.exp_ws, b.exp_ws.numel(), stream)
            else:
                L.moe_experts_fused_finalize(self.cw, b.x_perm, b.offsets, M, self.top_k, wts, wdt, b.inverse,
                                             b.shared, self.gemm2_dtype, rsf, b.out, b.exp_ws, b.exp_ws.numel(),
                                             stream)
            return b
        L.moe_experts(self.cw, b.x_perm, b.offsets, M, self.top_k, b.gemm2, self.gemm2_dtype,
                      1 if do_finalize else 0,
                      wts if do_finalize else None, wdt, b.pmap if do_finalize else None,
                      b.shared if do_finalize else None, self.gemm2_dtype, rsf,
                      b.out if do_finalize else None, self.out_dtype,
                      b.exp_ws, b.exp_ws.numel(), stream)
        return b

    def finalize(self, b: Buffers, stream=None):
        """The deferred finalize: moe_finalize on the buffers of a forward
        that ran with do_finalize=False."""
        rsf = 1.0 if self.method == L.MOE_ROUTE_SIGMOID_GROUPED_TOPK else self.rsf
        wdt = L.MOE_DTYPE_F32 if b.topk_weights.dtype == torch.float32 else L.MOE_DTYPE_BF16
        L.moe_finalize(b.gemm2, self.gemm2_dtype, b.gemm2.shape[0], b.topk_weights, wdt, b.pmap, b.M,
                       self.top_k, self.K, b.shared, self.gemm2_dtype, rsf, b.out, self.out_dtype, stream)
