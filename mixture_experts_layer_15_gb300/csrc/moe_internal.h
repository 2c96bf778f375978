// Internal host-side interfaces between the C ABI (moe_abi.cu) and the kernel
// translation units. Arguments are validated by the ABI layer before any of
// these is called; launchers only configure and enqueue.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

struct DeviceInfo {
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;
};

// Cached properties of the current device; returns false if there is none.
bool current_device_info(DeviceInfo* info);

// Address (device pointer) of the current device's error word.
int* device_error_word();

inline bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host checks of the permute's arguments, shared by moe_permute,
// moe_permute_noalloc and the permute half of moe_route_permute: sizes and
// ranges, required pointers, the row gather's alignment.
inline moe_status check_permute_args(const int32_t* topk_ids, int M, int top_k, int E, const int32_t* expert_map,
                                     int E_local, const void* x, int K, const int32_t* expert_offsets,
                                     const int32_t* map, const int32_t* inverse, const void* x_perm) {
    if (M < 0 || top_k <= 0 || E < 1 || E_local < 1 || E_local > 1024 || top_k > E) return MOE_ERR_INVALID_ARG;
    if (expert_map == nullptr && E_local != E) return MOE_ERR_INVALID_ARG;
    if (static_cast<long long>(M) * top_k >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    if (x_perm != nullptr) {
        if (x == nullptr || K <= 0) return MOE_ERR_INVALID_ARG;
        if (K % 8 != 0 || !is_aligned16(x) || !is_aligned16(x_perm)) return MOE_ERR_ALIGNMENT;
    }
    if (expert_offsets == nullptr) return MOE_ERR_INVALID_ARG;
    if (M > 0 && (topk_ids == nullptr || map == nullptr || inverse == nullptr)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// ---- router (router.cu) --------------------------------------------------------
cudaError_t launch_route(const float* logits, int M, int E, int top_k, int method,
                         const float* score_bias, int n_group, int topk_group, float rsf,
                         int32_t* topk_ids, void* topk_weights, int weights_dtype,
                         int* err, cudaStream_t stream);
cudaError_t launch_debug_sigmoid(const float* x, float* y, int n, cudaStream_t stream);
cudaError_t launch_debug_bounded_wait(const int* flag, int target, unsigned long long limit_ns, int* err,
                                      cudaStream_t stream);

// ---- permute (permute.cu) ------------------------------------------------------
size_t permute_workspace_bytes(int M, int top_k, int E_local);
cudaError_t launch_permute(const int32_t* topk_ids, int M, int top_k, int E,
                           const int32_t* expert_map, int E_local, const void* x, int K,
                           int32_t* expert_offsets, int32_t* map, int32_t* inverse,
                           void* x_perm, void* workspace, int* err, const DeviceInfo& dev,
                           cudaStream_t stream, int map_base = 0);

// Router + single-chunk permute in one kernel (small batches); same results as
// launch_route followed by launch_permute.
bool route_permute_fusible(int M, int top_k, int E, int E_local, int method);
cudaError_t launch_route_permute(const float* logits, int M, int E, int top_k, int method,
                                 const float* score_bias, int n_group, int topk_group, float rsf,
                                 int32_t* topk_ids, void* topk_weights, int weights_dtype,
                                 const int32_t* expert_map, int E_local, const void* x, int K,
                                 int32_t* expert_offsets, int32_t* map, int32_t* inverse, void* x_perm,
                                 int* err, const DeviceInfo& dev, cudaStream_t stream);

// ---- finalize (finalize.cu) ----------------------------------------------------
cudaError_t launch_finalize(const void* gemm2, int gemm2_dtype, int num_rows,
                            const void* weights, int weights_dtype, const int32_t* map,
                            int M, int top_k, int K, const void* shared, int shared_dtype,
                            float rsf, void* out, int out_dtype, int* err, cudaStream_t stream);
// Finalize + residual add + RMSNorm (finalize_rmsnorm.cu); K % 8 == 0, K <= 16384.
cudaError_t launch_finalize_rmsnorm(const void* gemm2, int gemm2_dtype, int num_rows, const void* weights,
                                    int weights_dtype, const int32_t* map, int M, int top_k, int K,
                                    const void* shared, int shared_dtype, float rsf, void* residual,
                                    int residual_dtype, const void* gamma, int gamma_dtype, float eps, void* y,
                                    int y_dtype, int* err, cudaStream_t stream);
// ---- grouped expert GEMMs (gemm.cu) --------------------------------------------
// One grouped "gated MLP" problem: E groups of rows of `x` (bf16 [rows_alloc, K]),
// group g = rows [offsets[g], offsets[g+1]) (or one group of `single_rows`
// rows when offsets == nullptr), weights per group W1 [2N, K], W2 [K, N].
struct ExpertsProblem {
    const moe_weights* w;
    const void* x;
    int rows_alloc;              // rows allocated in x / act / y (M * top_k)
    int M;                       // tokens (bounds the rows one group can have)
    const int32_t* offsets;      // [E+1] device, or nullptr
    int single_rows;             // rows of the single group when offsets == nullptr
    void* y;                     // [rows_alloc, K] output (bf16 or f32); unused when fin_out is set
    int y_dtype;
    // Finalize in the GEMM2 epilogue (fin_out != nullptr): fin_out [M, K] f32
    // = fin_shared + rsf * sum over routes of w * y, f32 reductions.
    float* fin_out = nullptr;
    const int32_t* inverse = nullptr;     // permuted_to_expanded [rows_alloc]
    const void* fin_weights = nullptr;    // [M * top_k], expanded order
    int fin_weights_dtype = 0;
    const void* fin_shared = nullptr;     // [M, K] or nullptr
    int fin_shared_dtype = 0;
    int top_k = 1;
    float rsf = 1.0f;
    // BatchedExperts layout: group g's rows are g*batch_stride .. + counts[g]-1
    // (counts on the device); offsets is then unused.
    const int32_t* counts = nullptr;
    int batch_stride = 0;
    // x given in token order (M rows): permuted row p is x[inverse[p] / top_k]
    // (the block-scaled formats read it so; the others gather into the workspace)
    bool x_tokens = false;
    // fin_out already holds the output start (nothing is copied into it); the
    // first launch that adds into it waits for out_ready (if not null) first
    bool out_preset = false;
    cudaEvent_t out_ready = nullptr;
};

// ---- MXFP8 activations (mx8_quant.cu) ----------------------------------------------
// x bf16 [rows, C] -> E4M3 codes [rows, C] + E8M0 scales [rows, C/32] (C % 128 == 0).
cudaError_t launch_mxfp8_quantize(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales, int* err,
                                  const DeviceInfo& dev, cudaStream_t stream);
// x bf16 [rows, C] -> two E4M3 terms per value: codes [2 * rows, C] and E8M0
// scales [2 * rows, C/32] (rows 2p hi, 2p + 1 lo; C % 128 == 0).
cudaError_t launch_e4m3_split(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales, int* err,
                              const DeviceInfo& dev, cudaStream_t stream);
// The same for the grouped rows of x_perm, scales into the token-tile atoms
// of the block-scaled GEMM (tiles of bt rows per group, at most max_tiles).
// hl: split each value into two E4M3 terms (hi, lo) that sum to it: codes
// [2 * rows_alloc, C] (row 2p hi, 2p + 1 lo), B rows 2n and 2n + 1 of a tile's
// atoms for its token n (bt tokens per tile). gather_inv (or NULL): x is in
// token order and row p reads token gather_inv[p] / gather_topk.
cudaError_t launch_mxfp8_quantize_tiles(const void* x, int rows_alloc, int C, const int32_t* offsets, int groups,
                                        int bt, int max_tiles, uint8_t* codes, uint8_t* atoms, int* err,
                                        const DeviceInfo& dev, cudaStream_t stream, bool hl = false,
                                        const int32_t* gather_inv = nullptr, int gather_topk = 1);
// x_perm[p] = x[inverse[p] / top_k] for p < offsets[E_l] (the permute's row
// gather on its own; permute.cu).
cudaError_t launch_gather_rows(const int32_t* offsets, int E_l, const int32_t* inverse, int top_k, int rows_alloc,
                               const void* x, int K, void* x_perm, const DeviceInfo& dev, cudaStream_t stream);
// Weight scales [rows_total, cols/32] -> atoms [rows_total/128][cols/128][512].
cudaError_t launch_mx_prepare_scales(const uint8_t* scales, long long rows_total, int cols, uint8_t* out,
                                     const DeviceInfo& dev, cudaStream_t stream);

void set_plan_override(int token_tile, int splits_gemm1, int splits_gemm2, int gemm2_tiles, int fuse);
// x_tokens: x is given in token order (ExpertsProblem::x_tokens).
size_t experts_workspace_bytes(const moe_weights* w, int rows_alloc, int M, const DeviceInfo& dev,
                               bool batched = false, bool x_tokens = false);
// Kernels one experts call launches (fin: the finalize folded into GEMM2,
// counting its out initialisation).
int experts_launches(const moe_weights* w, int rows_alloc, int M, bool fin, const DeviceInfo& dev);
cudaError_t launch_experts(const ExpertsProblem& p, void* workspace, size_t workspace_bytes,
                           int* err, const DeviceInfo& dev, cudaStream_t stream);

}  // namespace moe
