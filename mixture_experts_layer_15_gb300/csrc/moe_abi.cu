// C ABI of the MoE layer forward (declared in include/moe.h): argument
// validation on the host, then the launchers of the kernel translation units.
//
// Validation mirrors the checks of vllm/model_executor/layers/fused_moe/
// moe_output.py, convert_flashinfer_moe_output (num_tokens >= 0, top_k > 0,
// a finalized result goes to the given destination, a deferred result has
// none, the permute map is int32, contiguous buffers) and the arch allowlist
// of vllm/utils/flashinfer_moe_ep.py, validate_fi_moe_ep_config. Every check
// runs before anything is enqueued; no call allocates or synchronizes (except
// moe_get_error, which is documented to).
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "moe_internal.h"
#include <math.h>

namespace moe {

namespace {
__device__ int g_error_word;     // first device-detected error since the last moe_get_error
__device__ int g_error_taken;    // the value the last moe_get_error took out of g_error_word

// One device's cached properties and symbol addresses. Only a complete,
// successful set-up is cached: a lookup that failed (no device yet, a query
// error) is retried by the next call.
constexpr int kMaxDevices = 64;
struct DevSlot {
    std::mutex mu;
    std::atomic<bool> ok{false};
    DeviceInfo info;
    int* err = nullptr;
    int* taken = nullptr;
};
DevSlot g_dev[kMaxDevices];

// A CUDA runtime error that this code's own call returned is cleared here (it
// is reported as a status); errors of other calls are left for their owner.
inline bool cuda_ok(cudaError_t e) {
    if (e == cudaSuccess) return true;
    cudaGetLastError();
    return false;
}

DevSlot* current_slot() {
    int d = -1;
    if (!cuda_ok(cudaGetDevice(&d)) || d < 0 || d >= kMaxDevices) return nullptr;
    DevSlot* s = &g_dev[d];
    if (s->ok.load(std::memory_order_acquire)) return s;
    std::lock_guard<std::mutex> lock(s->mu);
    if (s->ok.load(std::memory_order_relaxed)) return s;
    DeviceInfo i;
    void* e = nullptr;
    void* t = nullptr;
    if (!cuda_ok(cudaDeviceGetAttribute(&i.sm_count, cudaDevAttrMultiProcessorCount, d)) ||
        !cuda_ok(cudaDeviceGetAttribute(&i.cc_major, cudaDevAttrComputeCapabilityMajor, d)) ||
        !cuda_ok(cudaDeviceGetAttribute(&i.cc_minor, cudaDevAttrComputeCapabilityMinor, d)) ||
        !cuda_ok(cudaDeviceGetAttribute(&i.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d)) ||
        !cuda_ok(cudaGetSymbolAddress(&e, g_error_word)) || !cuda_ok(cudaGetSymbolAddress(&t, g_error_taken)))
        return nullptr;
    s->info = i;
    s->err = static_cast<int*>(e);
    s->taken = static_cast<int*>(t);
    s->ok.store(true, std::memory_order_release);
    return s;
}

// Reads and clears the error word in one atomic step, so no error that a
// kernel on another stream records at the same time can be lost.
__global__ void take_error_kernel(int* err, int* taken) { *taken = atomicExch(err, 0); }
}  // namespace

bool current_device_info(DeviceInfo* info) {
    DevSlot* s = current_slot();
    if (!s) return false;
    *info = s->info;
    return true;
}

int* device_error_word() {
    DevSlot* s = current_slot();
    return s ? s->err : nullptr;
}

// moe_get_error's device part: enqueue the read-and-clear on `stream`, copy the
// taken value back, wait for it.
cudaError_t take_device_error(cudaStream_t stream, int* value) {
    DevSlot* s = current_slot();
    if (!s) return cudaErrorNoDevice;
    void* args[] = {&s->err, &s->taken};
    cudaError_t e = cudaLaunchKernel(reinterpret_cast<const void*>(take_error_kernel), dim3(1), dim3(1), args, 0,
                                     stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(value, s->taken, sizeof(int), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

}  // namespace moe

using moe::DeviceInfo;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_dtype(int d) { return d == MOE_DTYPE_BF16 || d == MOE_DTYPE_F32; }

// Device gate: a cc 10.3 device must be current.
moe_status device_gate(DeviceInfo* info, int** err) {
    if (!moe::current_device_info(info)) return MOE_ERR_CUDA;
    if (info->cc_major != 10 || info->cc_minor != 3) return MOE_ERR_UNSUPPORTED_ARCH;
    *err = moe::device_error_word();
    return MOE_OK;
}

inline moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_weights(const moe_weights* w) {
    if (w == nullptr || w->w1 == nullptr || w->w2 == nullptr) return MOE_ERR_INVALID_ARG;
    if (w->E_local < 1 || w->E_local > 1024 || w->K <= 0 || w->N <= 0) return MOE_ERR_INVALID_ARG;
    if (w->format != MOE_WEIGHTS_BF16 && w->format != MOE_WEIGHTS_MXFP4 && w->format != MOE_WEIGHTS_MXFP4_A8 &&
        w->format != MOE_WEIGHTS_MXFP4_A16)
        return MOE_ERR_INVALID_ARG;
    if (w->activation != MOE_ACT_SILU && w->activation != MOE_ACT_GELU) return MOE_ERR_INVALID_ARG;
    if (!(w->activation_clamp == w->activation_clamp) || w->activation_clamp == INFINITY) return MOE_ERR_INVALID_ARG;
    if (w->K % 128 != 0 || w->N % 128 != 0) return MOE_ERR_ALIGNMENT;
    if (!aligned16(w->w1) || !aligned16(w->w2)) return MOE_ERR_ALIGNMENT;
    if (w->format == MOE_WEIGHTS_MXFP4_A8 || w->format == MOE_WEIGHTS_MXFP4_A16) {
        // codes by 16U4 TMA (32-byte aligned); prepared scale atoms by bulk copies
        if (w->w1_scale == nullptr || w->w2_scale == nullptr) return MOE_ERR_INVALID_ARG;
        if (!aligned16(w->w1_scale) || !aligned16(w->w2_scale)) return MOE_ERR_ALIGNMENT;
        if ((reinterpret_cast<uintptr_t>(w->w1) & 31) != 0 || (reinterpret_cast<uintptr_t>(w->w2) & 31) != 0)
            return MOE_ERR_ALIGNMENT;
        if (w->K % 256 != 0) return MOE_ERR_ALIGNMENT;
    } else if (w->format == MOE_WEIGHTS_MXFP4) {
        if (w->w1_scale == nullptr || w->w2_scale == nullptr) return MOE_ERR_INVALID_ARG;
        if (!aligned16(w->w1_scale) || !aligned16(w->w2_scale)) return MOE_ERR_ALIGNMENT;
        // scale rows of K/32 and N/32 bytes must be 16-byte multiples for the TMA
        if (w->K % 512 != 0 || w->N % 512 != 0) return MOE_ERR_ALIGNMENT;
    } else if (w->w1_scale != nullptr || w->w2_scale != nullptr) {
        return MOE_ERR_INVALID_ARG;
    }
    // the largest row index a TMA coordinate can address is 2^31 - 1
    if (static_cast<long long>(w->E_local) * 2 * w->N >= (1LL << 31) ||
        static_cast<long long>(w->E_local) * w->K >= (1LL << 31))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Shared checks of the finalize arguments (moe_finalize and moe_experts with
// do_finalize = 1).
moe_status check_finalize_args(const void* weights, int wdtype, const int32_t* map, const void* shared,
                               int sdtype, void* out, int odtype) {
    if (weights == nullptr || map == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
    if (!valid_dtype(wdtype) || !valid_dtype(odtype)) return MOE_ERR_INVALID_ARG;
    if (shared != nullptr && !valid_dtype(sdtype)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(out) || (shared != nullptr && !aligned16(shared))) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

// Workspace of moe_experts_chunked for chunks of C tokens (the last chunk
// holds the ragged tail of M): the permute scratch, the chunk's expert
// offsets, its inverse map, its x_perm rows, then the experts workspace --
// each sized for the larger of the two chunk shapes, 256-byte aligned.
struct ChunkLayout {
    size_t off_offs, off_inv, off_xp, off_exp, exp_bytes, total;
};

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

ChunkLayout chunk_layout(const moe_weights* w, int M, int top_k, int C, const DeviceInfo& info) {
    const int first = C < M ? C : M;
    const int tail = M % first;
    size_t perm = moe::permute_workspace_bytes(first, top_k, w->E_local);
    size_t exp = moe::experts_workspace_bytes(w, first * top_k, first, info);
    if (tail > 0) {
        const size_t p2 = moe::permute_workspace_bytes(tail, top_k, w->E_local);
        const size_t e2 = moe::experts_workspace_bytes(w, tail * top_k, tail, info);
        perm = p2 > perm ? p2 : perm;
        exp = e2 > exp ? e2 : exp;
    }
    const size_t rows = static_cast<size_t>(first) * top_k;
    ChunkLayout L;
    L.off_offs = align256(perm);
    L.off_inv = align256(L.off_offs + sizeof(int32_t) * (w->E_local + 1));
    L.off_xp = align256(L.off_inv + sizeof(int32_t) * rows);
    L.off_exp = align256(L.off_xp + rows * w->K * 2);
    L.exp_bytes = exp;
    L.total = align256(L.off_exp + exp);
    return L;
}

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_ALIGNMENT: return "size or pointer alignment";
        case MOE_ERR_UNSUPPORTED: return "unsupported combination";
        case MOE_ERR_UNSUPPORTED_ARCH: return "device is not compute capability 10.3";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_INDEX: return "device: expert id or map entry out of range";
        case MOE_ERR_DEVICE_TIMEOUT: return "device: pipeline wait exceeded its limit";
        default: return "unknown status";
    }
}

moe_status moe_device_check(void) {
    DeviceInfo info;
    int* err = nullptr;
    return device_gate(&info, &err);
}

moe_status moe_get_error(cudaStream_t stream) {
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    // everything enqueued on `stream` so far completes before the read
    int v = 0;
    if (moe::take_device_error(stream, &v) != cudaSuccess) return MOE_ERR_CUDA;
    return static_cast<moe_status>(v);
}

moe_status moe_set_plan_override(int token_tile, int splits_gemm1, int splits_gemm2, int gemm2_tiles, int fuse) {
    if (token_tile != 0 && token_tile != 16 && token_tile != 32 && token_tile != 64 && token_tile != 128 &&
        token_tile != 256)
        return MOE_ERR_INVALID_ARG;
    if (splits_gemm1 < 0 || splits_gemm1 > 64 || splits_gemm2 < 0 || splits_gemm2 > 64) return MOE_ERR_INVALID_ARG;
    if (gemm2_tiles < 0 || gemm2_tiles > 2 || fuse < 0 || fuse > 3) return MOE_ERR_INVALID_ARG;
    moe::set_plan_override(token_tile, splits_gemm1, splits_gemm2, gemm2_tiles, fuse);
    return MOE_OK;
}

moe_status moe_mxfp8_quantize(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales,
                              cudaStream_t stream) {
    if (rows < 0 || C <= 0) return MOE_ERR_INVALID_ARG;
    if (C % 128 != 0) return MOE_ERR_ALIGNMENT;
    if (static_cast<long long>(rows) * C >= (1LL << 40)) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_mxfp8_quantize(x, rows, C, codes, scales, err, info, stream));
}

moe_status moe_e4m3_split(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
    if (rows < 0 || C <= 0) return MOE_ERR_INVALID_ARG;
    if (C % 128 != 0) return MOE_ERR_ALIGNMENT;
    if (static_cast<long long>(rows) * C >= (1LL << 39)) return MOE_ERR_UNSUPPORTED;
    if (rows == 0) return MOE_OK;
    if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(codes)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_e4m3_split(x, rows, C, codes, scales, err, info, stream));
}

size_t moe_mx_prepared_scales_size(int E_local, int rows, int cols) {
    if (E_local < 1 || rows <= 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0) return 0;
    return static_cast<size_t>(E_local) * (rows / 128) * (cols / 128) * 512;
}

moe_status moe_mx_prepare_scales(const uint8_t* scales, int E_local, int rows, int cols, uint8_t* out,
                                 cudaStream_t stream) {
    if (E_local < 1 || rows <= 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (rows % 128 != 0 || cols % 128 != 0) return MOE_ERR_ALIGNMENT;
    if (scales == nullptr || out == nullptr) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(scales) & 3) != 0 || !aligned16(out)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_mx_prepare_scales(scales, static_cast<long long>(E_local) * rows, cols, out, info,
                                                   stream));
}

moe_status moe_debug_sigmoid(const float* x, float* y, int n, cudaStream_t stream) {
    if (n < 0 || (n > 0 && (x == nullptr || y == nullptr))) return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_debug_sigmoid(x, y, n, stream));
}

moe_status moe_debug_bounded_wait(const int* flag, int target, unsigned long long limit_ns, cudaStream_t stream) {
    if (flag == nullptr || limit_ns == 0 || limit_ns > 2000000000ull) return MOE_ERR_INVALID_ARG;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_debug_bounded_wait(flag, target, limit_ns, err, stream));
}

moe_status moe_route(const float* logits, int M, int E, int top_k, moe_route_method method,
                     const float* score_bias, int n_group, int topk_group, float routed_scaling_factor,
                     int32_t* topk_ids, void* topk_weights, moe_dtype weights_dtype, cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;                               // num_tokens >= 0
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;                          // top_k > 0
    if (E < 1 || E > 1024 || top_k > E || top_k > 32) return MOE_ERR_INVALID_ARG;
    if (!valid_dtype(weights_dtype)) return MOE_ERR_INVALID_ARG;
    if (method == MOE_ROUTE_SOFTMAX_TOPK) {
        if (score_bias != nullptr) return MOE_ERR_INVALID_ARG;
    } else if (method == MOE_ROUTE_SIGMOID_GROUPED_TOPK) {
        if (score_bias == nullptr) return MOE_ERR_INVALID_ARG;
        if (n_group < 1 || n_group > 32 || E % n_group != 0 || E / n_group < 2) return MOE_ERR_INVALID_ARG;
        if (topk_group < 1 || topk_group > n_group) return MOE_ERR_INVALID_ARG;
        if (top_k > topk_group * (E / n_group)) return MOE_ERR_INVALID_ARG;
    } else {
        return MOE_ERR_INVALID_ARG;
    }
    if (M == 0) return MOE_OK;
    if (logits == nullptr || topk_ids == nullptr || topk_weights == nullptr) return MOE_ERR_INVALID_ARG;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_route(logits, M, E, top_k, method, score_bias, n_group, topk_group,
                                       routed_scaling_factor, topk_ids, topk_weights, weights_dtype, err,
                                       stream));
}

size_t moe_permute_workspace_size(int M, int top_k, int E_local) {
    if (M <= 0 || top_k <= 0 || E_local <= 0) return 0;
    return moe::permute_workspace_bytes(M, top_k, E_local);
}

moe_status moe_permute(const int32_t* topk_ids, int M, int top_k, int E, const int32_t* expert_map,
                       int E_local, const void* x, int K, int32_t* expert_offsets,
                       int32_t* expanded_idx_to_permuted_idx, int32_t* permuted_to_expanded, void* x_perm,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    const moe_status a = moe::check_permute_args(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                                 expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm);
    if (a != MOE_OK) return a;
    const size_t need = moe::permute_workspace_bytes(M > 0 ? M : 1, top_k, E_local);
    if (M > 0 && need > 0 && (workspace == nullptr || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    if (M == 0) {
        // no routes: every expert is empty
        return from_cuda(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E_local + 1), stream));
    }
    return from_cuda(moe::launch_permute(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                         expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm,
                                         workspace, err, info, stream));
}

moe_status moe_route_permute(const float* logits, int M, int E, int top_k, moe_route_method method,
                             const float* score_bias, int n_group, int topk_group, float routed_scaling_factor,
                             int32_t* topk_ids, void* topk_weights, moe_dtype weights_dtype,
                             const int32_t* expert_map, int E_local, const void* x, int K,
                             int32_t* expert_offsets, int32_t* expanded_idx_to_permuted_idx,
                             int32_t* permuted_to_expanded, void* x_perm, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    // the checks of moe_route ...
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    if (E < 1 || E > 1024 || top_k > E || top_k > 32) return MOE_ERR_INVALID_ARG;
    if (!valid_dtype(weights_dtype)) return MOE_ERR_INVALID_ARG;
    if (method == MOE_ROUTE_SOFTMAX_TOPK) {
        if (score_bias != nullptr) return MOE_ERR_INVALID_ARG;
    } else if (method == MOE_ROUTE_SIGMOID_GROUPED_TOPK) {
        if (score_bias == nullptr) return MOE_ERR_INVALID_ARG;
        if (n_group < 1 || n_group > 32 || E % n_group != 0 || E / n_group < 2) return MOE_ERR_INVALID_ARG;
        if (topk_group < 1 || topk_group > n_group) return MOE_ERR_INVALID_ARG;
        if (top_k > topk_group * (E / n_group)) return MOE_ERR_INVALID_ARG;
    } else {
        return MOE_ERR_INVALID_ARG;
    }
    // ... and of moe_permute
    const moe_status a = moe::check_permute_args(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                                 expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm);
    if (a != MOE_OK) return a;
    if (M > 0 && (logits == nullptr || topk_weights == nullptr)) return MOE_ERR_INVALID_ARG;
    const bool fused = M > 0 && moe::route_permute_fusible(M, top_k, E, E_local, method);
    const size_t need = moe::permute_workspace_bytes(M > 0 ? M : 1, top_k, E_local);
    if (M > 0 && !fused && need > 0 && (workspace == nullptr || workspace_bytes < need)) return MOE_ERR_WORKSPACE;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    if (M == 0) return from_cuda(cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E_local + 1), stream));
    if (fused)
        return from_cuda(moe::launch_route_permute(logits, M, E, top_k, method, score_bias, n_group, topk_group,
                                                   routed_scaling_factor, topk_ids, topk_weights, weights_dtype,
                                                   expert_map, E_local, x, K, expert_offsets,
                                                   expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm,
                                                   err, info, stream));
    const cudaError_t e = moe::launch_route(logits, M, E, top_k, method, score_bias, n_group, topk_group,
                                            routed_scaling_factor, topk_ids, topk_weights, weights_dtype, err,
                                            stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return from_cuda(moe::launch_permute(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                         expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm, workspace,
                                         err, info, stream));
}

size_t moe_experts_workspace_size(const moe_weights* w, int M, int top_k) {
    if (check_weights(w) != MOE_OK || M < 0 || top_k <= 0) return 0;
    DeviceInfo info;
    if (!moe::current_device_info(&info)) info.sm_count = 152;
    const int rows = M * top_k > 0 ? M * top_k : 1;
    return moe::experts_workspace_bytes(w, rows, M > 0 ? M : 1, info);
}

moe_status moe_finalize(const void* gemm2_permuted, moe_dtype gemm2_dtype, int num_permuted_rows,
                        const void* expert_weights, moe_dtype weights_dtype,
                        const int32_t* expanded_idx_to_permuted_idx, int M, int top_k, int K,
                        const void* shared_out, moe_dtype shared_dtype, float routed_scaling_factor, void* out,
                        moe_dtype out_dtype, cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    if (K <= 0 || num_permuted_rows < 0 || !valid_dtype(gemm2_dtype)) return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (K % 8 != 0) return MOE_ERR_ALIGNMENT;
    const moe_status a = check_finalize_args(expert_weights, weights_dtype, expanded_idx_to_permuted_idx,
                                             shared_out, shared_dtype, out, out_dtype);
    if (a != MOE_OK) return a;
    if (num_permuted_rows > 0 && gemm2_permuted == nullptr) return MOE_ERR_INVALID_ARG;
    if (gemm2_permuted != nullptr && !aligned16(gemm2_permuted)) return MOE_ERR_ALIGNMENT;
    if (out == gemm2_permuted || out == shared_out || out == expert_weights) return MOE_ERR_INVALID_ARG;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_finalize(gemm2_permuted, gemm2_dtype, num_permuted_rows, expert_weights,
                                          weights_dtype, expanded_idx_to_permuted_idx, M, top_k, K, shared_out,
                                          shared_dtype, routed_scaling_factor, out, out_dtype, err, stream));
}

moe_status moe_finalize_add_rmsnorm(const void* gemm2_permuted, moe_dtype gemm2_dtype, int num_permuted_rows,
                                    const void* expert_weights, moe_dtype weights_dtype,
                                    const int32_t* expanded_idx_to_permuted_idx, int M, int top_k, int K,
                                    const void* shared_out, moe_dtype shared_dtype, float routed_scaling_factor,
                                    void* residual, moe_dtype residual_dtype, const void* gamma,
                                    moe_dtype gamma_dtype, float eps, void* y, moe_dtype y_dtype,
                                    cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    if (K <= 0 || num_permuted_rows < 0 || !valid_dtype(gemm2_dtype)) return MOE_ERR_INVALID_ARG;
    if (!valid_dtype(residual_dtype) || !valid_dtype(gamma_dtype) || !valid_dtype(y_dtype)) return MOE_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps == INFINITY) return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (K % 8 != 0) return MOE_ERR_ALIGNMENT;
    if (K > 16384) return MOE_ERR_UNSUPPORTED;
    const moe_status a = check_finalize_args(expert_weights, weights_dtype, expanded_idx_to_permuted_idx,
                                             shared_out, shared_dtype, y, y_dtype);
    if (a != MOE_OK) return a;
    if (residual == nullptr || gamma == nullptr) return MOE_ERR_INVALID_ARG;
    if (num_permuted_rows > 0 && gemm2_permuted == nullptr) return MOE_ERR_INVALID_ARG;
    if ((gemm2_permuted != nullptr && !aligned16(gemm2_permuted)) || !aligned16(residual) || !aligned16(gamma))
        return MOE_ERR_ALIGNMENT;
    // y and the residual are written; neither may alias an input or each other
    const void* ins[4] = {gemm2_permuted, shared_out, expert_weights, gamma};
    for (const void* q : ins)
        if (q != nullptr && (q == y || q == residual)) return MOE_ERR_INVALID_ARG;
    if (y == residual) return MOE_ERR_INVALID_ARG;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_finalize_rmsnorm(gemm2_permuted, gemm2_dtype, num_permuted_rows, expert_weights,
                                                  weights_dtype, expanded_idx_to_permuted_idx, M, top_k, K,
                                                  shared_out, shared_dtype, routed_scaling_factor, residual,
                                                  residual_dtype, gamma, gamma_dtype, eps, y, y_dtype, err, stream));
}

moe_status moe_experts(const moe_weights* w, const void* x_perm, const int32_t* expert_offsets, int M,
                       int top_k, void* gemm2_permuted, moe_dtype gemm2_dtype, int do_finalize,
                       const void* expert_weights, moe_dtype weights_dtype,
                       const int32_t* expanded_idx_to_permuted_idx, const void* shared_out,
                       moe_dtype shared_dtype, float routed_scaling_factor, void* out, moe_dtype out_dtype,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    const moe_status ws_ok = check_weights(w);
    if (ws_ok != MOE_OK) return ws_ok;
    if (do_finalize != 0 && do_finalize != 1) return MOE_ERR_INVALID_ARG;
    if (!do_finalize && out != nullptr) return MOE_ERR_INVALID_ARG;     // a deferred output has no destination
    if (!valid_dtype(gemm2_dtype)) return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    if (do_finalize) {
        const moe_status a = check_finalize_args(expert_weights, weights_dtype, expanded_idx_to_permuted_idx,
                                                 shared_out, shared_dtype, out, out_dtype);
        if (a != MOE_OK) return a;
        if (out == gemm2_permuted || out == shared_out || out == expert_weights) return MOE_ERR_INVALID_ARG;
    }
    if (M == 0) return MOE_OK;                                          // nothing arrives: empty output
    if (x_perm == nullptr || expert_offsets == nullptr || gemm2_permuted == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(gemm2_permuted)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    const int rows = M * top_k;
    const size_t need = moe::experts_workspace_bytes(w, rows, M, info);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    moe::ExpertsProblem p;
    p.w = w;
    p.x = x_perm;
    p.rows_alloc = rows;
    p.M = M;
    p.offsets = expert_offsets;
    p.single_rows = 0;
    p.y = gemm2_permuted;
    p.y_dtype = gemm2_dtype;
    cudaError_t e = moe::launch_experts(p, workspace, workspace_bytes, err, info, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (!do_finalize) return MOE_OK;
    return from_cuda(moe::launch_finalize(gemm2_permuted, gemm2_dtype, rows, expert_weights, weights_dtype,
                                          expanded_idx_to_permuted_idx, M, top_k, w->K, shared_out,
                                          shared_dtype, routed_scaling_factor, out, out_dtype, err, stream));
}

size_t moe_experts_chunked_workspace_size(const moe_weights* w, int M, int top_k, int chunk_tokens) {
    if (check_weights(w) != MOE_OK || M <= 0 || top_k <= 0 || chunk_tokens <= 0) return 0;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return 0;
    DeviceInfo info;
    if (!moe::current_device_info(&info)) info.sm_count = 152;
    return chunk_layout(w, M, top_k, chunk_tokens, info).total;
}

moe_status moe_experts_chunked(const moe_weights* w, const void* x, const int32_t* topk_ids, int M, int top_k,
                               int E, const int32_t* expert_map, int chunk_tokens,
                               int32_t* expanded_idx_to_permuted_idx, void* gemm2_permuted, moe_dtype gemm2_dtype,
                               int do_finalize, const void* expert_weights, moe_dtype weights_dtype,
                               const void* shared_out, moe_dtype shared_dtype, float routed_scaling_factor,
                               void* out, moe_dtype out_dtype, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    if (M < 0 || top_k <= 0 || chunk_tokens <= 0) return MOE_ERR_INVALID_ARG;
    const moe_status ws_ok = check_weights(w);
    if (ws_ok != MOE_OK) return ws_ok;
    if (do_finalize != 0 && do_finalize != 1) return MOE_ERR_INVALID_ARG;
    if (!do_finalize && out != nullptr) return MOE_ERR_INVALID_ARG;     // a deferred output has no destination
    if (!valid_dtype(gemm2_dtype)) return MOE_ERR_INVALID_ARG;
    // the permute's rules (moe_permute), for the caller's buffers
    if (E < 1 || top_k > E) return MOE_ERR_INVALID_ARG;
    if (expert_map == nullptr && w->E_local != E) return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    if (M > 0 && (topk_ids == nullptr || expanded_idx_to_permuted_idx == nullptr)) return MOE_ERR_INVALID_ARG;
    if (do_finalize) {
        const moe_status a = check_finalize_args(expert_weights, weights_dtype, expanded_idx_to_permuted_idx,
                                                 shared_out, shared_dtype, out, out_dtype);
        if (a != MOE_OK) return a;
        if (out == gemm2_permuted || out == shared_out || out == expert_weights || out == x)
            return MOE_ERR_INVALID_ARG;
    }
    if (M == 0) return MOE_OK;
    if (x == nullptr || gemm2_permuted == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(gemm2_permuted)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    const ChunkLayout L = chunk_layout(w, M, top_k, chunk_tokens, info);
    if (workspace == nullptr || workspace_bytes < L.total || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* offs = reinterpret_cast<int32_t*>(ws + L.off_offs);
    int32_t* inv = reinterpret_cast<int32_t*>(ws + L.off_inv);
    void* xp = ws + L.off_xp;
    const int K = w->K;
    const size_t g2_row = static_cast<size_t>(K) * (gemm2_dtype == MOE_DTYPE_F32 ? 4 : 2);
    const int C = chunk_tokens < M ? chunk_tokens : M;
    for (int t0 = 0; t0 < M; t0 += C) {
        const int Mc = M - t0 < C ? M - t0 : C;
        const size_t r0 = static_cast<size_t>(t0) * top_k;     // first expanded index of the chunk
        // the chunk's routes in canonical order; its map entries point at its
        // rows of gemm2_permuted, [t0 * top_k, t0 * top_k + R_chunk)
        cudaError_t e = moe::launch_permute(topk_ids + r0, Mc, top_k, E, expert_map, w->E_local,
                                            static_cast<const uint8_t*>(x) + static_cast<size_t>(t0) * K * 2, K,
                                            offs, expanded_idx_to_permuted_idx + r0, inv, xp, ws, err, info,
                                            stream, static_cast<int>(r0));
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        moe::ExpertsProblem p;
        p.w = w;
        p.x = xp;
        p.rows_alloc = Mc * top_k;
        p.M = Mc;
        p.offsets = offs;
        p.single_rows = 0;
        p.y = static_cast<uint8_t*>(gemm2_permuted) + r0 * g2_row;
        p.y_dtype = gemm2_dtype;
        e = moe::launch_experts(p, ws + L.off_exp, L.exp_bytes, err, info, stream);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (!do_finalize) return MOE_OK;
    return from_cuda(moe::launch_finalize(gemm2_permuted, gemm2_dtype, M * top_k, expert_weights, weights_dtype,
                                          expanded_idx_to_permuted_idx, M, top_k, K, shared_out, shared_dtype,
                                          routed_scaling_factor, out, out_dtype, err, stream));
}

moe_status moe_experts_fused_finalize(const moe_weights* w, const void* x_perm, const int32_t* expert_offsets,
                                      int M, int top_k, const void* expert_weights, moe_dtype weights_dtype,
                                      const int32_t* permuted_to_expanded, const void* shared_out,
                                      moe_dtype shared_dtype, float routed_scaling_factor, float* out,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    const moe_status ws_ok = check_weights(w);
    if (ws_ok != MOE_OK) return ws_ok;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    const moe_status a = check_finalize_args(expert_weights, weights_dtype, permuted_to_expanded, shared_out,
                                             shared_dtype, out, MOE_DTYPE_F32);
    if (a != MOE_OK) return a;
    if (static_cast<const void*>(out) == shared_out || static_cast<const void*>(out) == expert_weights ||
        static_cast<const void*>(out) == x_perm)
        return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (x_perm == nullptr || expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    const int rows = M * top_k;
    const size_t need = moe::experts_workspace_bytes(w, rows, M, info);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    moe::ExpertsProblem p;
    p.w = w;
    p.x = x_perm;
    p.rows_alloc = rows;
    p.M = M;
    p.offsets = expert_offsets;
    p.single_rows = 0;
    p.y = nullptr;
    p.y_dtype = MOE_DTYPE_F32;
    p.fin_out = out;
    p.inverse = permuted_to_expanded;
    p.fin_weights = expert_weights;
    p.fin_weights_dtype = weights_dtype;
    p.fin_shared = shared_out;
    p.fin_shared_dtype = shared_dtype;
    p.top_k = top_k;
    p.rsf = routed_scaling_factor;
    return from_cuda(moe::launch_experts(p, workspace, workspace_bytes, err, info, stream));
}

size_t moe_experts_x_workspace_size(const moe_weights* w, int M, int top_k) {
    if (check_weights(w) != MOE_OK || M < 0 || top_k <= 0) return 0;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return 0;
    DeviceInfo info;
    if (!moe::current_device_info(&info)) info.sm_count = 152;
    const int rows = M * top_k > 0 ? M * top_k : 1;
    return moe::experts_workspace_bytes(w, rows, M > 0 ? M : 1, info, false, true);
}

moe_status moe_experts_fused_finalize_x(const moe_weights* w, const void* x, const int32_t* expert_offsets, int M,
                                        int top_k, const void* expert_weights, moe_dtype weights_dtype,
                                        const int32_t* permuted_to_expanded, const void* shared_out,
                                        moe_dtype shared_dtype, float routed_scaling_factor, float* out,
                                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    const moe_status ws_ok = check_weights(w);
    if (ws_ok != MOE_OK) return ws_ok;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    const moe_status a = check_finalize_args(expert_weights, weights_dtype, permuted_to_expanded, shared_out,
                                             shared_dtype, out, MOE_DTYPE_F32);
    if (a != MOE_OK) return a;
    if (static_cast<const void*>(out) == shared_out || static_cast<const void*>(out) == expert_weights ||
        static_cast<const void*>(out) == x)
        return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (x == nullptr || expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    const int rows = M * top_k;
    const size_t need = moe::experts_workspace_bytes(w, rows, M, info, false, true);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    moe::ExpertsProblem p;
    p.w = w;
    p.x = x;
    p.x_tokens = true;
    p.rows_alloc = rows;
    p.M = M;
    p.offsets = expert_offsets;
    p.single_rows = 0;
    p.y = nullptr;
    p.y_dtype = MOE_DTYPE_F32;
    p.fin_out = out;
    p.inverse = permuted_to_expanded;
    p.fin_weights = expert_weights;
    p.fin_weights_dtype = weights_dtype;
    p.fin_shared = shared_out;
    p.fin_shared_dtype = shared_dtype;
    p.top_k = top_k;
    p.rsf = routed_scaling_factor;
    return from_cuda(moe::launch_experts(p, workspace, workspace_bytes, err, info, stream));
}

moe_status moe_experts_fused_finalize_after(const moe_weights* w, const void* x, int x_order,
                                            const int32_t* expert_offsets, int M, int top_k,
                                            const void* expert_weights, moe_dtype weights_dtype,
                                            const int32_t* permuted_to_expanded, float routed_scaling_factor,
                                            float* out, cudaEvent_t out_ready, void* workspace,
                                            size_t workspace_bytes, cudaStream_t stream) {
    if (M < 0) return MOE_ERR_INVALID_ARG;
    if (top_k <= 0) return MOE_ERR_INVALID_ARG;
    if (x_order != 0 && x_order != 1) return MOE_ERR_INVALID_ARG;
    const moe_status ws_ok = check_weights(w);
    if (ws_ok != MOE_OK) return ws_ok;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    const moe_status a = check_finalize_args(expert_weights, weights_dtype, permuted_to_expanded, nullptr,
                                             MOE_DTYPE_F32, out, MOE_DTYPE_F32);
    if (a != MOE_OK) return a;
    if (static_cast<const void*>(out) == expert_weights || static_cast<const void*>(out) == x)
        return MOE_ERR_INVALID_ARG;
    if (M == 0) return MOE_OK;
    if (x == nullptr || expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    const int rows = M * top_k;
    const size_t need = moe::experts_workspace_bytes(w, rows, M, info, false, x_order == 1);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    moe::ExpertsProblem p;
    p.w = w;
    p.x = x;
    p.x_tokens = x_order == 1;
    p.rows_alloc = rows;
    p.M = M;
    p.offsets = expert_offsets;
    p.single_rows = 0;
    p.y = nullptr;
    p.y_dtype = MOE_DTYPE_F32;
    p.fin_out = out;
    p.inverse = permuted_to_expanded;
    p.fin_weights = expert_weights;
    p.fin_weights_dtype = weights_dtype;
    p.top_k = top_k;
    p.rsf = routed_scaling_factor;
    p.out_preset = true;
    p.out_ready = out_ready;
    return from_cuda(moe::launch_experts(p, workspace, workspace_bytes, err, info, stream));
}

int moe_experts_launches(const moe_weights* w, int M, int top_k, int fused_finalize) {
    if (M <= 0 || top_k <= 0 || check_weights(w) != MOE_OK) return 0;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return 0;
    DeviceInfo info;
    if (!moe::current_device_info(&info)) return 0;
    return moe::experts_launches(w, M * top_k, M, fused_finalize != 0, info);
}

size_t moe_experts_batched_workspace_size(const moe_weights* w, int max_tokens) {
    if (max_tokens <= 0 || check_weights(w) != MOE_OK) return 0;
    const long long rows = static_cast<long long>(w->E_local) * max_tokens;
    if (rows >= (1LL << 30)) return 0;
    DeviceInfo info;
    if (!moe::current_device_info(&info)) info.sm_count = 152;
    return moe::experts_workspace_bytes(w, static_cast<int>(rows), max_tokens, info, true);
}

moe_status moe_experts_batched(const moe_weights* w, const void* x, const int32_t* expert_num_tokens,
                               int max_tokens, void* y, moe_dtype y_dtype, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    if (max_tokens < 0) return MOE_ERR_INVALID_ARG;
    const moe_status ws_ok = check_weights(w);
    if (ws_ok != MOE_OK) return ws_ok;
    if (w->format == MOE_WEIGHTS_MXFP4_A8 || w->format == MOE_WEIGHTS_MXFP4_A16) return MOE_ERR_UNSUPPORTED;
    if (!valid_dtype(y_dtype)) return MOE_ERR_INVALID_ARG;
    const long long rows = static_cast<long long>(w->E_local) * max_tokens;
    if (rows >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    if (max_tokens == 0) return MOE_OK;
    if (x == nullptr || expert_num_tokens == nullptr || y == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return MOE_ERR_ALIGNMENT;
    if (x == y) return MOE_ERR_INVALID_ARG;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    const size_t need = moe::experts_workspace_bytes(w, static_cast<int>(rows), max_tokens, info, true);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    moe::ExpertsProblem p;
    p.w = w;
    p.x = x;
    p.rows_alloc = static_cast<int>(rows);
    p.M = max_tokens;
    p.offsets = nullptr;
    p.single_rows = 0;
    p.y = y;
    p.y_dtype = y_dtype;
    p.counts = expert_num_tokens;
    p.batch_stride = max_tokens;
    return from_cuda(moe::launch_experts(p, workspace, workspace_bytes, err, info, stream));
}

size_t moe_shared_expert_workspace_size(int M, int K, int Ns) {
    if (M <= 0 || K <= 0 || Ns <= 0 || K % 128 != 0 || Ns % 128 != 0) return 0;
    moe_weights w{};
    w.format = MOE_WEIGHTS_BF16;
    w.E_local = 1;
    w.K = K;
    w.N = Ns;
    DeviceInfo info;
    if (!moe::current_device_info(&info)) info.sm_count = 152;
    return moe::experts_workspace_bytes(&w, M, M, info);
}

moe_status moe_shared_expert(const void* ws1, const void* ws2, int K, int Ns, const void* x, int M,
                             void* shared_out, moe_dtype shared_dtype, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
    if (M < 0 || K <= 0 || Ns <= 0 || !valid_dtype(shared_dtype)) return MOE_ERR_INVALID_ARG;
    if (K % 128 != 0 || Ns % 128 != 0) return MOE_ERR_ALIGNMENT;
    if (M == 0) return MOE_OK;
    if (ws1 == nullptr || ws2 == nullptr || x == nullptr || shared_out == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ws1) || !aligned16(ws2) || !aligned16(x) || !aligned16(shared_out)) return MOE_ERR_ALIGNMENT;
    DeviceInfo info;
    int* err = nullptr;
    const moe_status st = device_gate(&info, &err);
    if (st != MOE_OK) return st;
    moe_weights w{};
    w.format = MOE_WEIGHTS_BF16;
    w.E_local = 1;
    w.K = K;
    w.N = Ns;
    w.w1 = ws1;
    w.w2 = ws2;
    const size_t need = moe::experts_workspace_bytes(&w, M, M, info);
    if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)) return MOE_ERR_WORKSPACE;
    moe::ExpertsProblem p;
    p.w = &w;
    p.x = x;
    p.rows_alloc = M;
    p.M = M;
    p.offsets = nullptr;
    p.single_rows = M;
    p.y = shared_out;
    p.y_dtype = shared_dtype;
    return from_cuda(moe::launch_experts(p, workspace, workspace_bytes, err, info, stream));
}

}  // extern "C"
