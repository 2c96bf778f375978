"""ctypes binding of ``libmoe_gb300.so`` (the C ABI declared in include/moe.h).

Argument marshalling only: every function has the C name and argument order;
tensors are passed as device pointers (``data_ptr()``), ``None`` as NULL, and
a missing stream means torch's current stream. A non-OK status raises
``MoEError`` (its ``status`` attribute holds the code). There is no fallback:
if the library is not built, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_ALIGNMENT = 2
MOE_ERR_UNSUPPORTED = 3
MOE_ERR_UNSUPPORTED_ARCH = 4
MOE_ERR_WORKSPACE = 5
MOE_ERR_CUDA = 6
MOE_ERR_DEVICE_INDEX = 7
MOE_ERR_DEVICE_TIMEOUT = 8

MOE_DTYPE_BF16 = 0
MOE_DTYPE_F32 = 1
MOE_ROUTE_SOFTMAX_TOPK = 0
MOE_ROUTE_SIGMOID_GROUPED_TOPK = 1
MOE_WEIGHTS_BF16 = 0
MOE_WEIGHTS_MXFP4 = 1
MOE_WEIGHTS_MXFP4_A8 = 2
MOE_WEIGHTS_MXFP4_A16 = 3
MOE_ACT_SILU = 0
MOE_ACT_GELU = 1

#: every function the header declares (checked against include/moe.h by the tests)
EXPORTS = (
    "moe_route", "moe_permute_workspace_size", "moe_permute", "moe_route_permute", "moe_permute_noalloc",
    "moe_experts_workspace_size",
    "moe_experts", "moe_experts_fused_finalize", "moe_experts_launches", "moe_finalize",
    "moe_experts_chunked_workspace_size", "moe_experts_chunked", "moe_experts_x_workspace_size",
    "moe_experts_fused_finalize_x",
    "moe_experts_fused_finalize_after",
    "moe_finalize_add_rmsnorm", "moe_experts_batched_workspace_size", "moe_experts_batched", "moe_shared_expert_workspace_size",
    "moe_shared_expert",
    "moe_status_string", "moe_get_error", "moe_device_check", "moe_set_plan_override",
    "moe_debug_sigmoid", "moe_debug_bounded_wait",
    "moe_mxfp8_quantize", "moe_mx_prepared_scales_size", "moe_mx_prepare_scales", "moe_e4m3_split",
)


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = int(status)
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


class moe_weights(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int),
        ("E_local", ctypes.c_int),
        ("K", ctypes.c_int),
        ("N", ctypes.c_int),
        ("w1", ctypes.c_void_p),
        ("w1_scale", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p),
        ("activation", ctypes.c_int),
        ("activation_clamp", ctypes.c_float),
    ]


if not os.path.exists(LIB_PATH):
    raise ImportError(f"the MoE CUDA library is not built ({LIB_PATH}); run "
                      "mixture_experts_layer_15_gb300.build.build() first")
lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

_SIGS = {
    "moe_route": ([_P, _I, _I, _I, _I, _P, _I, _I, _F, _P, _P, _I, _P], _I),
    "moe_permute_workspace_size": ([_I, _I, _I], _Z),
    "moe_permute": ([_P, _I, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P, _P, _Z, _P], _I),
    "moe_route_permute": ([_P, _I, _I, _I, _I, _P, _I, _I, _F, _P, _P, _I, _P, _I, _P, _I, _P, _P, _P, _P, _P, _Z,
                           _P], _I),
    "moe_permute_noalloc": ([_P, _I, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P, _P], _I),
    "moe_experts_workspace_size": ([ctypes.POINTER(moe_weights), _I, _I], _Z),
    "moe_experts": ([ctypes.POINTER(moe_weights), _P, _P, _I, _I, _P, _I, _I, _P, _I, _P, _P, _I, _F,
                     _P, _I, _P, _Z, _P], _I),
    "moe_experts_fused_finalize": ([ctypes.POINTER(moe_weights), _P, _P, _I, _I, _P, _I, _P, _P, _I, _F, _P,
                                    _P, _Z, _P], _I),
    "moe_experts_launches": ([ctypes.POINTER(moe_weights), _I, _I, _I], _I),
    "moe_experts_x_workspace_size": ([ctypes.POINTER(moe_weights), _I, _I], _Z),
    "moe_experts_fused_finalize_x": ([ctypes.POINTER(moe_weights), _P, _P, _I, _I, _P, _I, _P, _P, _I, _F, _P,
                                      _P, _Z, _P], _I),
    "moe_experts_fused_finalize_after": ([ctypes.POINTER(moe_weights), _P, _I, _P, _I, _I, _P, _I, _P, _F, _P,
                                          _P, _P, _Z, _P], _I),
    "moe_experts_chunked_workspace_size": ([ctypes.POINTER(moe_weights), _I, _I, _I], _Z),
    "moe_experts_chunked": ([ctypes.POINTER(moe_weights), _P, _P, _I, _I, _I, _P, _I, _P, _P, _I, _I, _P, _I, _P,
                             _I, _F, _P, _I, _P, _Z, _P], _I),
    "moe_experts_batched_workspace_size": ([ctypes.POINTER(moe_weights), _I], _Z),
    "moe_experts_batched": ([ctypes.POINTER(moe_weights), _P, _P, _I, _P, _I, _P, _Z, _P], _I),
    "moe_finalize": ([_P, _I, _I, _P, _I, _P, _I, _I, _I, _P, _I, _F, _P, _I, _P], _I),
    "moe_finalize_add_rmsnorm": ([_P, _I, _I, _P, _I, _P, _I, _I, _I, _P, _I, _F, _P, _I, _P, _I, _F, _P, _I, _P],
                                 _I),
    "moe_shared_expert_workspace_size": ([_I, _I, _I], _Z),
    "moe_shared_expert": ([_P, _P, _I, _I, _P, _I, _P, _I, _P, _Z, _P], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_get_error": ([_P], _I),
    "moe_device_check": ([], _I),
    "moe_set_plan_override": ([_I, _I, _I, _I, _I], _I),
    "moe_debug_sigmoid": ([_P, _P, _I, _P], _I),
    "moe_debug_bounded_wait": ([_P, _I, ctypes.c_ulonglong, _P], _I),
    "moe_mxfp8_quantize": ([_P, _I, _I, _P, _P, _P], _I),
    "moe_e4m3_split": ([_P, _I, _I, _P, _P, _P], _I),
    "moe_mx_prepared_scales_size": ([_I, _I, _I], _Z),
    "moe_mx_prepare_scales": ([_P, _I, _I, _I, _P, _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.argtypes = _args
    _f.restype = _res


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("MoE buffers must be contiguous")
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x)} as a device pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn, st):
    if st != MOE_OK:
        raise MoEError(fn, st)


def status_string(status: int) -> str:
    return lib.moe_status_string(int(status)).decode()


def make_weights(fmt, E_local, K, N, w1, w2, w1_scale=None, w2_scale=None, activation=0,
                 activation_clamp=None) -> moe_weights:
    return moe_weights(int(fmt), int(E_local), int(K), int(N), _ptr(w1), _ptr(w1_scale), _ptr(w2),
                       _ptr(w2_scale), int(activation), float(activation_clamp or 0.0))


def moe_route(logits, M, E, top_k, method, score_bias, n_group, topk_group, routed_scaling_factor,
              topk_ids, topk_weights, weights_dtype, stream=None):
    _check("moe_route", lib.moe_route(_ptr(logits), M, E, top_k, method, _ptr(score_bias), n_group,
                                      topk_group, routed_scaling_factor, _ptr(topk_ids),
                                      _ptr(topk_weights), weights_dtype, _stream(stream)))


def moe_permute_workspace_size(M, top_k, E_local) -> int:
    return int(lib.moe_permute_workspace_size(M, top_k, E_local))


def moe_permute(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm, workspace, workspace_bytes,
                stream=None):
    _check("moe_permute", lib.moe_permute(_ptr(topk_ids), M, top_k, E, _ptr(expert_map), E_local,
                                          _ptr(x), K, _ptr(expert_offsets),
                                          _ptr(expanded_idx_to_permuted_idx), _ptr(permuted_to_expanded),
                                          _ptr(x_perm), _ptr(workspace), int(workspace_bytes),
                                          _stream(stream)))


def moe_route_permute(logits, M, E, top_k, method, score_bias, n_group, topk_group, routed_scaling_factor,
                      topk_ids, topk_weights, weights_dtype, expert_map, E_local, x, K, expert_offsets,
                      expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm, workspace, workspace_bytes,
                      stream=None):
    _check("moe_route_permute", lib.moe_route_permute(
        _ptr(logits), M, E, top_k, method, _ptr(score_bias), n_group, topk_group, routed_scaling_factor,
        _ptr(topk_ids), _ptr(topk_weights), weights_dtype, _ptr(expert_map), E_local, _ptr(x), K,
        _ptr(expert_offsets), _ptr(expanded_idx_to_permuted_idx), _ptr(permuted_to_expanded), _ptr(x_perm),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def moe_permute_noalloc(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                        expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm, stream=None):
    """moe_permute without a workspace: its scratch is a fixed array in the library."""
    _check("moe_permute_noalloc", lib.moe_permute_noalloc(_ptr(topk_ids), M, top_k, E, _ptr(expert_map),
                                                          E_local, _ptr(x), K, _ptr(expert_offsets),
                                                          _ptr(expanded_idx_to_permuted_idx),
                                                          _ptr(permuted_to_expanded), _ptr(x_perm),
                                                          _stream(stream)))


def moe_experts_workspace_size(weights: moe_weights, M, top_k) -> int:
    return int(lib.moe_experts_workspace_size(ctypes.byref(weights), M, top_k))


def moe_experts(weights: moe_weights, x_perm, expert_offsets, M, top_k, gemm2_permuted, gemm2_dtype,
                do_finalize, expert_weights, weights_dtype, expanded_idx_to_permuted_idx, shared_out,
                shared_dtype, routed_scaling_factor, out, out_dtype, workspace, workspace_bytes,
                stream=None):
    _check("moe_experts", lib.moe_experts(ctypes.byref(weights), _ptr(x_perm), _ptr(expert_offsets), M,
                                          top_k, _ptr(gemm2_permuted), gemm2_dtype, int(do_finalize),
                                          _ptr(expert_weights), weights_dtype,
                                          _ptr(expanded_idx_to_permuted_idx), _ptr(shared_out),
                                          shared_dtype, routed_scaling_factor, _ptr(out), out_dtype,
                                          _ptr(workspace), int(workspace_bytes), _stream(stream)))


def moe_experts_chunked_workspace_size(weights: moe_weights, M, top_k, chunk_tokens) -> int:
    return int(lib.moe_experts_chunked_workspace_size(ctypes.byref(weights), M, top_k, chunk_tokens))


def moe_experts_chunked(weights: moe_weights, x, topk_ids, M, top_k, E, expert_map, chunk_tokens,
                        expanded_idx_to_permuted_idx, gemm2_permuted, gemm2_dtype, do_finalize, expert_weights,
                        weights_dtype, shared_out, shared_dtype, routed_scaling_factor, out, out_dtype, workspace,
                        workspace_bytes, stream=None):
    _check("moe_experts_chunked", lib.moe_experts_chunked(
        ctypes.byref(weights), _ptr(x), _ptr(topk_ids), M, top_k, E, _ptr(expert_map), chunk_tokens,
        _ptr(expanded_idx_to_permuted_idx), _ptr(gemm2_permuted), gemm2_dtype, int(do_finalize),
        _ptr(expert_weights), weights_dtype, _ptr(shared_out), shared_dtype, routed_scaling_factor, _ptr(out),
        out_dtype, _ptr(workspace), int(workspace_bytes), _stream(stream)))


def moe_experts_x_workspace_size(weights: moe_weights, M, top_k) -> int:
    return int(lib.moe_experts_x_workspace_size(ctypes.byref(weights), M, top_k))


def moe_experts_fused_finalize_x(weights: moe_weights, x, expert_offsets, M, top_k, expert_weights, weights_dtype,
                                 permuted_to_expanded, shared_out, shared_dtype, routed_scaling_factor, out, workspace,
                                 workspace_bytes, stream=None):
    _check("moe_experts_fused_finalize_x", lib.moe_experts_fused_finalize_x(
        ctypes.byref(weights), _ptr(x), _ptr(expert_offsets), M, top_k, _ptr(expert_weights), weights_dtype,
        _ptr(permuted_to_expanded), _ptr(shared_out), shared_dtype, routed_scaling_factor, _ptr(out),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def _event(e):
    """A torch.cuda.Event (recorded), a raw cudaEvent_t as int, or None."""
    if e is None or isinstance(e, int):
        return e
    return e.cuda_event


def moe_experts_fused_finalize_after(weights: moe_weights, x, x_order, expert_offsets, M, top_k, expert_weights,
                                     weights_dtype, permuted_to_expanded, routed_scaling_factor, out, out_ready,
                                     workspace, workspace_bytes, stream=None):
    _check("moe_experts_fused_finalize_after", lib.moe_experts_fused_finalize_after(
        ctypes.byref(weights), _ptr(x), int(x_order), _ptr(expert_offsets), M, top_k, _ptr(expert_weights),
        weights_dtype, _ptr(permuted_to_expanded), routed_scaling_factor, _ptr(out), _event(out_ready),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def moe_experts_fused_finalize(weights: moe_weights, x_perm, expert_offsets, M, top_k, expert_weights,
                               weights_dtype, permuted_to_expanded, shared_out, shared_dtype,
                               routed_scaling_factor, out, workspace, workspace_bytes, stream=None):
    _check("moe_experts_fused_finalize", lib.moe_experts_fused_finalize(
        ctypes.byref(weights), _ptr(x_perm), _ptr(expert_offsets), M, top_k, _ptr(expert_weights), weights_dtype,
        _ptr(permuted_to_expanded), _ptr(shared_out), shared_dtype, routed_scaling_factor, _ptr(out),
        _ptr(workspace), int(workspace_bytes), _stream(stream)))


def moe_finalize_add_rmsnorm(gemm2_permuted, gemm2_dtype, num_permuted_rows, expert_weights, weights_dtype,
                             expanded_idx_to_permuted_idx, M, top_k, K, shared_out, shared_dtype,
                             routed_scaling_factor, residual, residual_dtype, gamma, gamma_dtype, eps, y, y_dtype,
                             stream=None):
    _check("moe_finalize_add_rmsnorm", lib.moe_finalize_add_rmsnorm(
        _ptr(gemm2_permuted), gemm2_dtype, num_permuted_rows, _ptr(expert_weights), weights_dtype,
        _ptr(expanded_idx_to_permuted_idx), M, top_k, K, _ptr(shared_out), shared_dtype, routed_scaling_factor,
        _ptr(residual), residual_dtype, _ptr(gamma), gamma_dtype, eps, _ptr(y), y_dtype, _stream(stream)))


def moe_experts_batched_workspace_size(weights: moe_weights, max_tokens) -> int:
    return int(lib.moe_experts_batched_workspace_size(ctypes.byref(weights), max_tokens))


def moe_experts_batched(weights: moe_weights, x, expert_num_tokens, max_tokens, y, y_dtype, workspace,
                        workspace_bytes, stream=None):
    _check("moe_experts_batched", lib.moe_experts_batched(
        ctypes.byref(weights), _ptr(x), _ptr(expert_num_tokens), max_tokens, _ptr(y), y_dtype, _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def moe_experts_launches(weights: moe_weights, M, top_k, fused_finalize) -> int:
    return int(lib.moe_experts_launches(ctypes.byref(weights), M, top_k, 1 if fused_finalize else 0))


def moe_finalize(gemm2_permuted, gemm2_dtype, num_permuted_rows, expert_weights, weights_dtype,
                 expanded_idx_to_permuted_idx, M, top_k, K, shared_out, shared_dtype,
                 routed_scaling_factor, out, out_dtype, stream=None):
    _check("moe_finalize", lib.moe_finalize(_ptr(gemm2_permuted), gemm2_dtype, num_permuted_rows,
                                            _ptr(expert_weights), weights_dtype,
                                            _ptr(expanded_idx_to_permuted_idx), M, top_k, K,
                                            _ptr(shared_out), shared_dtype, routed_scaling_factor,
                                            _ptr(out), out_dtype, _stream(stream)))


def moe_shared_expert_workspace_size(M, K, Ns) -> int:
    return int(lib.moe_shared_expert_workspace_size(M, K, Ns))


def moe_shared_expert(ws1, ws2, K, Ns, x, M, shared_out, shared_dtype, workspace, workspace_bytes,
                      stream=None):
    _check("moe_shared_expert", lib.moe_shared_expert(_ptr(ws1), _ptr(ws2), K, Ns, _ptr(x), M,
                                                      _ptr(shared_out), shared_dtype, _ptr(workspace),
                                                      int(workspace_bytes), _stream(stream)))


def moe_get_error(stream=None) -> int:
    """Synchronizes the stream; returns (does not raise) the device error status."""
    return int(lib.moe_get_error(_stream(stream)))


def moe_device_check() -> int:
    return int(lib.moe_device_check())


def moe_set_plan_override(token_tile=0, splits_gemm1=0, splits_gemm2=0, gemm2_tiles=0, fuse=0):
    _check("moe_set_plan_override", lib.moe_set_plan_override(token_tile, splits_gemm1, splits_gemm2,
                                                              gemm2_tiles, fuse))


def moe_debug_bounded_wait(flag, target, limit_ns, stream=None):
    _check("moe_debug_bounded_wait", lib.moe_debug_bounded_wait(_ptr(flag), int(target), int(limit_ns),
                                                                 _stream(stream)))


def moe_debug_sigmoid(x, y, n, stream=None):
    _check("moe_debug_sigmoid", lib.moe_debug_sigmoid(_ptr(x), _ptr(y), n, _stream(stream)))


def moe_mxfp8_quantize(x, rows, C, codes, scales, stream=None):
    _check("moe_mxfp8_quantize", lib.moe_mxfp8_quantize(_ptr(x), rows, C, _ptr(codes), _ptr(scales),
                                                         _stream(stream)))


def moe_e4m3_split(x, rows, C, codes, scales, stream=None):
    _check("moe_e4m3_split", lib.moe_e4m3_split(_ptr(x), rows, C, _ptr(codes), _ptr(scales), _stream(stream)))


def moe_mx_prepared_scales_size(E_local, rows, cols):
    return lib.moe_mx_prepared_scales_size(E_local, rows, cols)


def moe_mx_prepare_scales(scales, E_local, rows, cols, out, stream=None):
    _check("moe_mx_prepare_scales", lib.moe_mx_prepare_scales(_ptr(scales), E_local, rows, cols, _ptr(out),
                                                               _stream(stream)))
