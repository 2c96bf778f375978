/*
 * moe.h -- C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer forward.
 *
 * The layer is the pipeline [Router] -> [Quantize-Dispatch] ->
 * [Permute-Experts-Unpermute] -> [Combine] laid out in the module header of
 * vllm/model_executor/layers/fused_moe/modular_kernel.py. On one GPU with all
 * experts local the dispatch and combine are no-ops, so the calls are:
 *
 *   moe_route     logits -> topk_ids, topk_weights                  [Router]
 *   moe_permute   topk_ids -> expert_offsets, expanded_idx_to_permuted_idx,
 *                 permuted_to_expanded, x_perm                        (permute)
 *   moe_experts   x_perm -> gemm2_permuted (GEMM1, silu_and_mul, GEMM2;
 *                 unweighted, unreduced), optionally finalized   (experts)
 *   moe_finalize  gemm2_permuted, weights, map, shared -> out    (unpermute+reduce)
 *
 * Conventions that hold for every call:
 *  - Every pointer argument is a DEVICE pointer to a dense row-major
 *    (contiguous) array, unless it is documented as a host pointer. The
 *    deferred-finalize contract requires contiguous buffers
 *    (moe_output.py, convert_flashinfer_moe_output).
 *  - The caller owns and allocates every buffer. The library never
 *    allocates device memory, never synchronizes, and enqueues all work on
 *    `stream` (asynchronous).
 *  - Every call returns a moe_status. Nothing throws across the ABI.
 *    Argument validation runs on the host before anything is enqueued; a
 *    call that fails validation enqueues nothing.
 *  - Problems found on the device (an expert id or a map entry out of range,
 *    a pipeline wait that ran out) do not trap: the offending route is
 *    skipped and a device error word is set, which moe_get_error() returns.
 *  - The device must have compute capability 10.3 (GB300); other devices get
 *    MOE_ERR_UNSUPPORTED_ARCH (flashinfer_moe_ep.py,
 *    validate_fi_moe_ep_config: the mega MoE kernels are Blackwell-only and
 *    fail loudly elsewhere).
 *  - bf16 means IEEE bfloat16 stored as 16-bit words; f32 is IEEE binary32.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* a size, range, NULL or dtype rule is broken   */
    MOE_ERR_ALIGNMENT = 2,         /* K or N not a multiple of 128; a pointer not 16-byte aligned */
    MOE_ERR_UNSUPPORTED = 3,       /* a combination this library does not implement */
    MOE_ERR_UNSUPPORTED_ARCH = 4,  /* the current device is not compute capability 10.3 */
    MOE_ERR_WORKSPACE = 5,         /* workspace NULL or smaller than the *_workspace_size() */
    MOE_ERR_CUDA = 6,              /* a CUDA runtime call (launch, attribute, no device) failed */
    MOE_ERR_DEVICE_INDEX = 7,      /* device-detected: an expert id or map entry out of range */
    MOE_ERR_DEVICE_TIMEOUT = 8     /* device-detected: a pipeline wait exceeded its limit */
} moe_status;

typedef enum moe_dtype {
    MOE_DTYPE_BF16 = 0,
    MOE_DTYPE_F32 = 1
} moe_dtype;

typedef enum moe_route_method {
    /* softmax over the E logits, top_k largest, renormalised to sum 1, x scale */
    MOE_ROUTE_SOFTMAX_TOPK = 0,
    /* sigmoid scores + selection bias, grouped top-k, renormalised, x scale */
    MOE_ROUTE_SIGMOID_GROUPED_TOPK = 1
} moe_route_method;

typedef enum moe_weight_format {
    MOE_WEIGHTS_BF16 = 0,          /* bf16 weights                                     */
    MOE_WEIGHTS_MXFP4 = 1,         /* e2m1 codes, two per byte, + one E8M0 byte per 32 */
    MOE_WEIGHTS_MXFP4_A8 = 2,      /* MXFP4 weights, scales as moe_mx_prepare_scales
                                      writes them; activations quantised to MXFP8   */
    MOE_WEIGHTS_MXFP4_A16 = 3      /* MXFP4 weights, scales as moe_mx_prepare_scales
                                      writes them; bf16 activations (W4A16) on the
                                      block-scaled tensor cores                      */
} moe_weight_format;

/*
 * Expert weights of the E_local local experts (modular_kernel.py,
 * _moe_problem_size: w1 is [E, 2N, .], w2 is [., K, .]; for packed formats the
 * trailing dimension is halved, so K and N are given explicitly here).
 *
 *   BF16:  w1 bf16 [E_local, 2N, K]; rows 0..N-1 of each expert are the gate
 *          projection, rows N..2N-1 the up projection (silu_and_mul multiplies
 *          silu(first half) by the second half).
 *          w2 bf16 [E_local, K, N].
 *   MXFP4: w1 u8 [E_local, 2N, K/2] and w1_scale u8 [E_local, 2N, K/32];
 *          w2 u8 [E_local, K, N/2] and w2_scale u8 [E_local, K, N/32].
 *          Byte j of a row holds element 2j in its low nibble and element
 *          2j+1 in its high nibble; scale byte b of a row scales elements
 *          32b..32b+31 by the float whose bits are (b << 23), i.e. 2^(b-127)
 *          (flashinfer_moe_ep.py, _E2M1_LUT and _dequant_fp4_ue8m0_gran32).
 *          Scale bytes must lie in 1..254 and every decoded value must be a
 *          normal bf16 or zero (the kernels decode to bf16 before the MMA).
 *   MXFP4_A8: the MXFP4 codes as above (w1, w2; 32-byte aligned); w1_scale
 *          and w2_scale hold the same scales rearranged by
 *          moe_mx_prepare_scales (w1: rows 2N, cols K; w2: rows K, cols N).
 *          The experts then run with MXFP8 activations -- the quantize_input
 *          step of flashinfer_moe_ep.py build_fi_mega_config, read as the
 *          weights' MX recipe: every 32 consecutive values along a GEMM's
 *          reduction axis share an E8M0 scale 2^(floor(log2 amax) - 8) (byte
 *          kept in 1..254) and are rounded to E4M3 (nearest, ties to even,
 *          saturated at 448) -- x_perm before GEMM1 and the activation output
 *          before GEMM2; block-scaled tensor-core MMAs apply both scales.
 *          Outputs therefore differ from the MXFP4 format's by the
 *          activations' quantisation error. K % 256 == 0, N % 128 == 0;
 *          moe_experts and moe_experts_fused_finalize only.
 *   MXFP4_A16: weights as for MXFP4_A8 (codes, prepared scales), bf16
 *          activations: the W4A16 computation of MOE_WEIGHTS_MXFP4 -- the
 *          same bf16 x and the same bf16 rounding of the activation output --
 *          run on the block-scaled tensor cores instead of a decode to bf16.
 *          Each bf16 value v of a 32-element block is written as two E4M3
 *          terms, hi = e4m3(v / s1) * s1 and lo = e4m3((v - hi) / s2) * s2,
 *          s1, s2 the smallest powers of two that keep the block's codes
 *          within 448 (no saturation); hi + lo == v exactly for every v within
 *          2^14 of its block's largest magnitude (the error of the others is
 *          below 2^-21 of that magnitude). The MMAs take the two terms as two
 *          B rows per token and the epilogues add their accumulators. Same
 *          limits as MXFP4_A8.
 *
 * K and N must be multiples of 128 (of 512 for MXFP4). All pointers 16-byte
 * aligned.
 */
typedef struct moe_weights {
    moe_weight_format format;
    int E_local;
    int K;                 /* hidden size                 */
    int N;                 /* expert intermediate size    */
    const void* w1;
    const uint8_t* w1_scale;   /* MXFP4 only, else NULL */
    const void* w2;
    const uint8_t* w2_scale;   /* MXFP4 only, else NULL */
    /* GEMM1's activation (FusedMoEPermuteExpertsUnpermute.activation):
     * MOE_ACT_SILU (0, silu_and_mul) or MOE_ACT_GELU (1, gelu_and_mul, exact
     * erf GELU), on the gate (rows 0..N-1 of W1) times the up projection. */
    int activation;
    /* activation_clamp (flashinfer_moe_ep.py, build_fi_mega_config): c > 0
     * clamps the gate to at most c and the up projection to [-c, c] before
     * the activation; 0 (or less) means no clamp. */
    float activation_clamp;
} moe_weights;

enum { MOE_ACT_SILU = 0, MOE_ACT_GELU = 1 };

/* ------------------------------------------------------------------------
 * moe_route -- the [Router] step (modular_kernel.py module header; its
 * outputs are FusedMoEModularKernel.forward's topk_ids / topk_weights).
 *
 *   logits        f32 [M, E] router logits.
 *   method        MOE_ROUTE_SOFTMAX_TOPK: select the top_k largest logits,
 *                 ordered by logit descending, equal logits to the lower
 *                 expert id; weight_j = exp(l_j - l_max) / sum over the
 *                 selected of exp(l_i - l_max), times routed_scaling_factor.
 *                 MOE_ROUTE_SIGMOID_GROUPED_TOPK: s_e = sigmoid(l_e) computed
 *                 by a fixed float32 spec (see moe_debug_sigmoid),
 *                 b_e = s_e + score_bias[e]; the experts form n_group
 *                 contiguous groups of E/n_group; a group's score is the
 *                 float32 sum of its two largest b; the topk_group best groups
 *                 are kept (ties to the lower group); the top_k largest b
 *                 among their experts are selected, ordered by b descending
 *                 (ties to the lower id); weight_j = s_j / sum_selected s,
 *                 times routed_scaling_factor (the scale is then folded:
 *                 moe_output.py, UnfinalizedMoEOutput expert_weights comment).
 *   score_bias    f32 [E]; required for the sigmoid method, must be NULL for softmax.
 *   n_group, topk_group   sigmoid method only (E % n_group == 0,
 *                 E/n_group >= 2, 1 <= topk_group <= n_group,
 *                 top_k <= topk_group * E/n_group); pass 1, 1 for softmax.
 *   topk_ids      out, i32 [M, top_k], global expert ids.
 *   topk_weights  out, [M, top_k] in weights_dtype (bf16 or f32).
 * Limits: 1 <= E <= 1024, 1 <= top_k <= min(E, 32), M >= 0 (M = 0: no work).
 * Logits must be finite (NaN gives an unspecified but in-range selection).
 * ---------------------------------------------------------------------- */
moe_status moe_route(const float* logits, int M, int E, int top_k,
                     moe_route_method method, const float* score_bias,
                     int n_group, int topk_group, float routed_scaling_factor,
                     int32_t* topk_ids, void* topk_weights, moe_dtype weights_dtype,
                     cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute -- group the M*top_k routes by local expert (the permute half
 * of [Permute-Experts-Unpermute]; the map is UnfinalizedMoEOutput's
 * expanded_idx_to_permuted_idx, moe_output.py).
 *
 *   topk_ids      i32 [M, top_k] global expert ids in [0, E).
 *   expert_map    i32 [E] or NULL. expert_map[e] is the local id of global
 *                 expert e, or -1 when e is not local (modular_kernel.py,
 *                 prepare/apply expert_map). Local ids must be < E_local and
 *                 no two global experts may share one. NULL = identity
 *                 (then E_local must equal E).
 *   x             bf16 [M, K] token activations; may be NULL iff x_perm is NULL.
 *
 * Outputs. Routes are ordered expert-major, and within an expert by their
 * expanded index t*top_k + j (a canonical order that does not depend on any
 * tiling). R = number of routes to local experts.
 *   expert_offsets               i32 [E_local+1]: rows of local expert le are
 *                                [offsets[le], offsets[le+1]); offsets[E_local] = R.
 *   expanded_idx_to_permuted_idx i32 [M, top_k]: permuted row of route (t, j),
 *                                -1 for a route to a non-local expert.
 *   permuted_to_expanded         i32 [M*top_k]: entries [0, R) give the expanded
 *                                index of each permuted row; the rest are not written.
 *   x_perm                       bf16 [M*top_k, K] or NULL: row p = x[inverse[p] / top_k]
 *                                for p < R; rows >= R are not written.
 *   workspace                    device scratch of moe_permute_workspace_size() bytes
 *                                (contents on entry do not matter).
 * Out-of-range ids or map entries set MOE_ERR_DEVICE_INDEX and the route is
 * treated as non-local.
 * ---------------------------------------------------------------------- */
size_t moe_permute_workspace_size(int M, int top_k, int E_local);

moe_status moe_permute(const int32_t* topk_ids, int M, int top_k, int E,
                       const int32_t* expert_map, int E_local,
                       const void* x, int K,
                       int32_t* expert_offsets, int32_t* expanded_idx_to_permuted_idx,
                       int32_t* permuted_to_expanded, void* x_perm,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_route_permute -- moe_route followed by moe_permute, with the arguments
 * of both, giving the same results bit for bit. For small batches (M <= 64
 * and M*top_k routes within one permute chunk) one kernel routes every token
 * and permutes the routes, one launch fewer on the latency-bound path; the
 * workspace is then not used (it may be NULL). Otherwise it runs the two
 * steps and needs moe_permute_workspace_size() bytes of workspace.
 * ---------------------------------------------------------------------- */
moe_status moe_route_permute(const float* logits, int M, int E, int top_k,
                             moe_route_method method, const float* score_bias,
                             int n_group, int topk_group, float routed_scaling_factor,
                             int32_t* topk_ids, void* topk_weights, moe_dtype weights_dtype,
                             const int32_t* expert_map, int E_local, const void* x, int K,
                             int32_t* expert_offsets, int32_t* expanded_idx_to_permuted_idx,
                             int32_t* permuted_to_expanded, void* x_perm,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute_noalloc -- moe_permute for callers that cannot allocate device
 * memory. The paper has no counterpart: it exists for this library's users.
 * Some callers may neither call cudaMalloc nor hand the library a workspace:
 * an inference engine that carves all device memory out of one arena at
 * start-up and gives the libraries it hosts no allocator, a plugin loaded
 * into a process whose allocator belongs to the host application, or a
 * latency-critical path that must never reach cudaMalloc (which can
 * synchronise the device). This entry point takes the same arguments as
 * moe_permute minus the workspace and gives the same results bit for bit.
 * Its scratch (the per-chunk expert histograms) is a fixed 1 MiB array inside
 * the library, which every GPU that loads the library holds until the
 * process exits.
 *  - Limit: moe_permute_workspace_size(M, top_k, E_local) must be at most
 *    1 MiB (for example M*top_k up to 2^21 routes at E_local = 128); larger
 *    problems return MOE_ERR_WORKSPACE and enqueue nothing.
 *  - The first call on each device does the set-up: with that device current
 *    it looks up the array's device address (cudaGetSymbolAddress) and caches
 *    it. Make that first call before any stream capture. A lookup that fails
 *    returns MOE_ERR_CUDA and is tried again by the next call. The cached
 *    address belongs to the device's primary context: cudaDeviceReset, or a
 *    context of the caller's own, is not supported while the library is loaded.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 *  - All calls on one device share the array. Nothing in it needs clearing
 *    between calls (every entry read is written first by the same call), but
 *    calls whose kernels overlap on the GPU race on it and give wrong maps:
 *    order them (one stream, or explicit events).
 *  - Argument checks and status codes are those of moe_permute.
 * ---------------------------------------------------------------------- */
moe_status moe_permute_noalloc(const int32_t* topk_ids, int M, int top_k, int E,
                               const int32_t* expert_map, int E_local,
                               const void* x, int K,
                               int32_t* expert_offsets, int32_t* expanded_idx_to_permuted_idx,
                               int32_t* permuted_to_expanded, void* x_perm, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_finalize_add_rmsnorm -- moe_finalize folded into its consumer, the next
 * layer's residual add + RMSNorm (moe_output.py, MoEOutput: the consumer of an
 * open reduction, typically the next layer's RMSNorm, can take the top-k
 * reduction of an unfinalized routed output into the same kernel):
 *
 *   r[t]        = rsf * sum_j w[t,j] * gemm2_permuted[map[t,j]] + shared[t] + residual[t]
 *   residual[t] <- r[t]
 *   y[t]        = r[t] / sqrt(mean over K of r[t]^2 + eps) * gamma
 *
 *   gemm2_permuted .. routed_scaling_factor: as in moe_finalize.
 *   residual   [M, K] in residual_dtype, read and overwritten with r (the
 *              accumulation is f32; y is computed from the unrounded r).
 *   gamma      [K] in gamma_dtype; eps >= 0 (MOE_ERR_INVALID_ARG otherwise).
 *   y          [M, K] in y_dtype.
 * K must be a multiple of 8 (MOE_ERR_ALIGNMENT) and at most 16384
 * (MOE_ERR_UNSUPPORTED). y and residual may not alias each other or an input.
 * ---------------------------------------------------------------------- */
moe_status moe_finalize_add_rmsnorm(const void* gemm2_permuted, moe_dtype gemm2_dtype, int num_permuted_rows,
                                    const void* expert_weights, moe_dtype weights_dtype,
                                    const int32_t* expanded_idx_to_permuted_idx, int M, int top_k, int K,
                                    const void* shared_out, moe_dtype shared_dtype, float routed_scaling_factor,
                                    void* residual, moe_dtype residual_dtype, const void* gamma,
                                    moe_dtype gamma_dtype, float eps, void* y, moe_dtype y_dtype,
                                    cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_experts -- the experts: GEMM1, silu_and_mul, GEMM2, per local expert on
 * its rows of x_perm (modular_kernel.py, FusedMoEPermuteExpertsUnpermute.apply
 * and .activation). The result is unweighted and unreduced.
 *
 *   x_perm           bf16 [M*top_k, K] (rows [0, R) valid, from moe_permute).
 *   expert_offsets   i32 [E_local+1] (from moe_permute); read on the device, so
 *                    the host never learns R.
 *   gemm2_permuted   out, [M*top_k, K] in gemm2_dtype (bf16 or f32): row p is
 *                    W2[le] . (silu(W1g[le] x) * (W1u[le] x)) for the token of
 *                    permuted row p, densely packed at K; rows >= R are not
 *                    written (UnfinalizedMoEOutput: indexed by row, padded row
 *                    count never referenced).
 *   do_finalize      0: stop after GEMM2 (the deferred output is gemm2_permuted,
 *                    expert_weights and expanded_idx_to_permuted_idx); `out`
 *                    must be NULL -- a deferred output has no destination
 *                    (convert_flashinfer_moe_output).
 *                    1: also run moe_finalize into `out`, with the same
 *                    result bit for bit as a separate moe_finalize call.
 *   expert_weights, weights_dtype, expanded_idx_to_permuted_idx, shared_out,
 *   shared_dtype, routed_scaling_factor, out, out_dtype:
 *                    as in moe_finalize (ignored when do_finalize = 0; pass NULL).
 *   workspace        device scratch of at least moe_experts_workspace_size()
 *                    bytes, ZERO-FILLED BEFORE ITS FIRST USE. Every completed
 *                    call leaves its synchronisation counters at zero again, so
 *                    a workspace is zeroed once, and again only after a call
 *                    that reported MOE_ERR_DEVICE_TIMEOUT. Calls that share a
 *                    workspace must not overlap on the GPU.
 * ---------------------------------------------------------------------- */
size_t moe_experts_workspace_size(const moe_weights* w, int M, int top_k);

moe_status moe_experts(const moe_weights* w,
                       const void* x_perm, const int32_t* expert_offsets,
                       int M, int top_k,
                       void* gemm2_permuted, moe_dtype gemm2_dtype,
                       int do_finalize,
                       const void* expert_weights, moe_dtype weights_dtype,
                       const int32_t* expanded_idx_to_permuted_idx,
                       const void* shared_out, moe_dtype shared_dtype,
                       float routed_scaling_factor,
                       void* out, moe_dtype out_dtype,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_experts_chunked -- the permute and the experts run chunk by chunk over
 * the tokens, so that the scratch they need is sized by the chunk, not by M:
 * activation chunking (modular_kernel.py, FusedMoEModularKernel.forward
 * splits M into chunks of VLLM_FUSED_MOE_CHUNK_SIZE tokens when the experts
 * object supports chunking, sizes workspace13 and workspace2 for one chunk
 * -- FusedMoEPermuteExpertsUnpermute.workspace_shapes, whose first dimension
 * must be the number of tokens -- and runs apply() on each chunk's
 * activations and topk_ids, writing the chunk's rows of the output).
 *
 * For chunk c of tokens [t0, t1), t0 = c * chunk_tokens (the last chunk holds
 * the ragged tail): the chunk's routes are permuted in the canonical order of
 * moe_permute (expert-major, then expanded index), its experts run on its
 * rows, and its unweighted GEMM2 rows land in gemm2_permuted rows
 * [t0 * top_k, t0 * top_k + R_c). expanded_idx_to_permuted_idx[t, j] (t in
 * the chunk) is t0 * top_k + the route's row within the chunk, or -1 for a
 * non-local expert. With do_finalize = 1, moe_finalize then runs over all M
 * tokens with that map into `out`.
 *
 *   x                 bf16 [M, K] token activations (not permuted).
 *   topk_ids          i32 [M, top_k] global expert ids in [0, E).
 *   expert_map, E     as in moe_permute (E_local = w->E_local).
 *   chunk_tokens      >= 1 tokens per chunk; >= M gives one chunk (then the
 *                     result is moe_permute + moe_experts, bit for bit).
 *   expanded_idx_to_permuted_idx  out, i32 [M, top_k] (above).
 *   gemm2_permuted    out, [M * top_k, K] in gemm2_dtype; rows that no map
 *                     entry points to are not written.
 *   do_finalize .. out_dtype: as in moe_experts.
 *   workspace         moe_experts_chunked_workspace_size() bytes, zero-filled
 *                     before first use (it holds the experts' counters: the
 *                     moe_experts rule applies). Its size depends on M only
 *                     through the tail chunk: at most that of chunk_tokens
 *                     and M mod chunk_tokens tokens.
 * Errors: those of moe_permute and moe_experts; chunk_tokens <= 0 ->
 * MOE_ERR_INVALID_ARG. Per-route results equal those of the unchunked
 * moe_permute + moe_experts up to the launch plan's split-K choice, which
 * depends on the number of routes in a call (without split-K in both, bit for
 * bit).
 * ---------------------------------------------------------------------- */
size_t moe_experts_chunked_workspace_size(const moe_weights* w, int M, int top_k, int chunk_tokens);

moe_status moe_experts_chunked(const moe_weights* w, const void* x, const int32_t* topk_ids, int M, int top_k,
                               int E, const int32_t* expert_map, int chunk_tokens,
                               int32_t* expanded_idx_to_permuted_idx, void* gemm2_permuted, moe_dtype gemm2_dtype,
                               int do_finalize, const void* expert_weights, moe_dtype weights_dtype,
                               const void* shared_out, moe_dtype shared_dtype, float routed_scaling_factor,
                               void* out, moe_dtype out_dtype, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_experts_fused_finalize -- the experts with the finalize folded into
 * GEMM2 (moe_output.py, UnfinalizedMoEOutput: when the routed output is left
 * unfinalized, the top-k reduction can fold into the consumer that runs
 * next; here the consumer is GEMM2's own epilogue). Computes
 *
 *   out[t] = shared_out[t] + rsf * sum_{routes (t, j) with a local expert} w[t,j] * y[t,j]
 *
 * with y the unweighted GEMM2 row of the route, as moe_experts followed by
 * moe_finalize does, without writing gemm2_permuted: every GEMM2 accumulator
 * value goes straight from the tensor memory into out with an f32 reduction.
 * This removes the [R, K] f32 round trip through HBM and the finalize launch.
 *
 *   x_perm, expert_offsets, M, top_k, workspace: as in moe_experts (same
 *                    workspace size query, same zero-once rule).
 *   expert_weights   [M, top_k] in weights_dtype (expanded order t*top_k+j).
 *   permuted_to_expanded  i32 [M*top_k] from moe_permute: entry p < R is the
 *                    expanded index of permuted row p (the inverse of
 *                    expanded_idx_to_permuted_idx). Entries outside
 *                    [0, M*top_k) set MOE_ERR_DEVICE_INDEX and are skipped.
 *   shared_out       [M, K] in shared_dtype, or NULL (then out starts at 0).
 *   out              f32 [M, K] (f32 only: the reductions accumulate in it).
 *
 * Differences from moe_experts + moe_finalize: the order in which the top_k
 * routes (and the split-K parts of one route) are added is not fixed, so the
 * result can differ between runs by f32 rounding (a few ulp of out); it is
 * within the same tolerance of the exact result. gemm2_permuted is neither
 * read nor written. Returns MOE_ERR_INVALID_ARG if out aliases an input.
 * ---------------------------------------------------------------------- */
moe_status moe_experts_fused_finalize(const moe_weights* w,
                                      const void* x_perm, const int32_t* expert_offsets,
                                      int M, int top_k,
                                      const void* expert_weights, moe_dtype weights_dtype,
                                      const int32_t* permuted_to_expanded,
                                      const void* shared_out, moe_dtype shared_dtype,
                                      float routed_scaling_factor, float* out,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_experts_fused_finalize_x -- moe_experts_fused_finalize with the
 * permute's row gather folded in: it reads the token activations x in token
 * order, and permuted row p is x[permuted_to_expanded[p] / top_k] (the row
 * that moe_permute would have copied to x_perm[p]; pair it with moe_permute
 * or moe_route_permute called with x_perm = NULL). The block-scaled formats
 * (MOE_WEIGHTS_MXFP4_A8, MOE_WEIGHTS_MXFP4_A16) quantise the gathered rows
 * straight from x, so the [M*top_k, K] x_perm is never written or read; the
 * other formats gather x_perm into the workspace first. Results equal
 * moe_experts_fused_finalize's on the gathered rows.
 *
 *   x                bf16 [M, K] (16-byte aligned).
 *   permuted_to_expanded  i32 [M*top_k]: entries [0, R) as moe_permute writes
 *                    them; an entry outside [0, M*top_k) sets
 *                    MOE_ERR_DEVICE_INDEX and its row reads as zeros (block-
 *                    scaled formats) or is skipped.
 *   workspace        moe_experts_x_workspace_size() bytes, zero-filled before
 *                    first use (the moe_experts rule).
 *   the rest         as in moe_experts_fused_finalize.
 * ---------------------------------------------------------------------- */
size_t moe_experts_x_workspace_size(const moe_weights* w, int M, int top_k);

moe_status moe_experts_fused_finalize_x(const moe_weights* w, const void* x, const int32_t* expert_offsets, int M,
                                        int top_k, const void* expert_weights, moe_dtype weights_dtype,
                                        const int32_t* permuted_to_expanded, const void* shared_out,
                                        moe_dtype shared_dtype, float routed_scaling_factor, float* out,
                                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_experts_fused_finalize_after -- the routed experts with the finalize
 * folded in, added into an output that already holds its start.
 * (moe_output.py, MoEOutput: the shared-expert output plus the routed sum;
 * modular_kernel.py, FusedMoEModularKernel.forward: the shared experts run
 * beside the routed ones.) The shared expert can then run on another stream
 * at the same time as the router, the permute and the routed experts' first
 * launches: moe_shared_expert with shared_out = out (shared_dtype F32) writes
 * the start, an event recorded after it is out_ready, and this call waits for
 * that event only before its first launch that adds into out.
 *
 *   x, x_order       x_order = 0: x is x_perm [M*top_k, K], as in
 *                    moe_experts_fused_finalize (workspace:
 *                    moe_experts_workspace_size); x_order = 1: x is in token
 *                    order [M, K], as in moe_experts_fused_finalize_x
 *                    (workspace: moe_experts_x_workspace_size).
 *   out              f32 [M, K]: holds the output start when the wait ends;
 *                    out[t] += rsf * sum over t's routes of w * y.
 *   out_ready        an event (recorded on the stream that writes the start),
 *                    or NULL when the start is already ordered before this
 *                    call on `stream`. It is waited for on `stream`, as with
 *                    cudaStreamWaitEvent; the event itself is not changed.
 *   the rest         as in moe_experts_fused_finalize (no shared_out: the
 *                    start is out's own content).
 *
 * Results equal moe_experts_fused_finalize's with shared_out = the start (f32),
 * up to the order of the f32 additions. The launches before the wait (the
 * activation quantiser and GEMM1 where the plan has them) neither read nor
 * write out. Returns MOE_ERR_INVALID_ARG for x_order outside {0, 1} or when
 * out aliases x or expert_weights.
 * ---------------------------------------------------------------------- */
moe_status moe_experts_fused_finalize_after(const moe_weights* w, const void* x, int x_order,
                                            const int32_t* expert_offsets, int M, int top_k,
                                            const void* expert_weights, moe_dtype weights_dtype,
                                            const int32_t* permuted_to_expanded, float routed_scaling_factor,
                                            float* out, cudaEvent_t out_ready, void* workspace,
                                            size_t workspace_bytes, cudaStream_t stream);

/* The number of kernels that moe_experts_fused_finalize (fused_finalize = 1,
 * counting the initialisation of out) or moe_experts with do_finalize = 0
 * (fused_finalize = 0) launches for this batch size, from the same launch plan
 * the calls use; 0 for invalid arguments or without a device. Host-only. */
int moe_experts_launches(const moe_weights* w, int M, int top_k, int fused_finalize);

/* ------------------------------------------------------------------------
 * moe_experts_batched -- the experts on the BatchedExperts activation format
 * (modular_kernel.py, FusedMoEActivationFormat: [num experts, max tokens per
 * expert, hidden], with expert_num_tokens, the per-expert counts that
 * FusedMoEPermuteExpertsUnpermute.apply receives in that format). The
 * fixed-shape layout suits graph capture and batched dispatchers.
 *
 *   x                  bf16 [E_local, max_tokens, K]; expert e's tokens are
 *                      rows 0 .. expert_num_tokens[e]-1 of block e.
 *   expert_num_tokens  i32 [E_local] on the device; a count outside
 *                      [0, max_tokens] sets MOE_ERR_DEVICE_INDEX and is
 *                      clamped.
 *   y                  [E_local, max_tokens, K] in y_dtype: row r of block e is
 *                      W2[e] . act(W1[e] x[e, r]) for r < count_e (unweighted);
 *                      rows past the count are not written.
 *   workspace          at least moe_experts_batched_workspace_size() bytes,
 *                      zero-filled before first use (as for moe_experts).
 * The activation and clamp of `w` apply. GEMM1 and GEMM2 run as two launches.
 * ---------------------------------------------------------------------- */
size_t moe_experts_batched_workspace_size(const moe_weights* w, int max_tokens);

moe_status moe_experts_batched(const moe_weights* w, const void* x, const int32_t* expert_num_tokens,
                               int max_tokens, void* y, moe_dtype y_dtype, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_finalize -- apply the routing weights and reduce over top_k
 * (modular_kernel.py, FusedMoEPrepareAndFinalize.finalize), then the routed
 * scale and the shared-expert add (moe_output.py, MoEOutput: the shared
 * output is folded in by whoever finalizes; the routed scale is applied to
 * the routed sum before the shared add and is 1.0 when folded):
 *
 *   out[t] = routed_scaling_factor * sum_{j : map[t,j] != -1}
 *                 expert_weights[t,j] * gemm2_permuted[map[t,j]]
 *            + shared_out[t]
 *
 * accumulated in float32 in j order, then rounded once to out_dtype.
 *   gemm2_permuted     [num_permuted_rows, K] in gemm2_dtype.
 *   num_permuted_rows  rows allocated in gemm2_permuted (for the device bounds
 *                      check only; map entries >= it set MOE_ERR_DEVICE_INDEX
 *                      and are skipped).
 *   expert_weights     [M, top_k] in weights_dtype.
 *   expanded_idx_to_permuted_idx  i32 [M, top_k].
 *   shared_out         [M, K] in shared_dtype, or NULL.
 *   out                out, [M, K] in out_dtype; may not alias any input.
 * ---------------------------------------------------------------------- */
moe_status moe_finalize(const void* gemm2_permuted, moe_dtype gemm2_dtype, int num_permuted_rows,
                        const void* expert_weights, moe_dtype weights_dtype,
                        const int32_t* expanded_idx_to_permuted_idx, int M, int top_k, int K,
                        const void* shared_out, moe_dtype shared_dtype,
                        float routed_scaling_factor,
                        void* out, moe_dtype out_dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * moe_shared_expert -- the shared expert: the same gated MLP on every token
 * (its output is MoEOutput.shared_output, moe_output.py), run by the same
 * grouped GEMM kernels with one group of M rows.
 *   ws1 bf16 [2*Ns, K] (gate rows then up rows), ws2 bf16 [K, Ns], x bf16 [M, K],
 *   shared_out out [M, K] in shared_dtype. K, Ns multiples of 128.
 *   workspace: moe_shared_expert_workspace_size() bytes, zero-filled before
 *   first use (same rule as moe_experts).
 * ---------------------------------------------------------------------- */
size_t moe_shared_expert_workspace_size(int M, int K, int Ns);

moe_status moe_shared_expert(const void* ws1, const void* ws2, int K, int Ns,
                             const void* x, int M,
                             void* shared_out, moe_dtype shared_dtype,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Diagnostics.
 * ---------------------------------------------------------------------- */
/* Static text for a status code (never NULL). */
/* ------------------------------------------------------------------------
 * MXFP8 quantisation and the block-scaled weight layout
 * ------------------------------------------------------------------------
 * moe_mxfp8_quantize: x bf16 [rows, C] -> codes u8 [rows, C] (E4M3) and
 * scales u8 [rows, C/32] (E8M0): the MXFP8 rule of MOE_WEIGHTS_MXFP4_A8
 * (blocks of 32 consecutive values of a row; scale byte = clamp(exponent
 * field of the block's largest magnitude - 8, 1, 254); code = E4M3 nearest to
 * value * 2^(127 - byte), ties to even, saturated at 448). C % 128 == 0
 * (MOE_ERR_ALIGNMENT); x and codes 16-byte aligned. rows == 0 is a no-op.
 *
 * moe_mx_prepared_scales_size / moe_mx_prepare_scales: the E8M0 scales of
 * an MXFP4 matrix, u8 [E_local, rows, cols/32] row-major, rearranged for the
 * block-scaled MMA: for each 128-row tile and 128-column block of a 512-byte
 * atom, row r's four scale bytes at byte (r % 32) * 16 + ((r % 128) / 32) * 4.
 * rows and cols multiples of 128 (MOE_ERR_ALIGNMENT); scales 4-byte aligned,
 * out 16-byte aligned, of moe_mx_prepared_scales_size() bytes (0 for invalid
 * sizes). A one-time weight preparation; asynchronous on `stream`.
 * ---------------------------------------------------------------------- */
moe_status moe_mxfp8_quantize(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales,
                              cudaStream_t stream);

/* moe_e4m3_split: the activation format of MOE_WEIGHTS_MXFP4_A16 on its own.
 * x bf16 [rows, C] -> codes u8 [2 * rows, C] and E8M0 scale bytes u8
 * [2 * rows, C/32]; rows 2p and 2p + 1 hold the hi and lo terms of row p: for
 * every block of 32 consecutive values, hi = e4m3(v / s1) and
 * lo = e4m3((v - hi * s1) / s2) (nearest, ties to even), s1 and s2 the
 * smallest powers of two 2^(b - 127) with the block's largest |v| (|v - hi s1|
 * for s2) at most 448 * s (b kept in 1..254). hi * s1 + lo * s2 == v for every v
 * within 2^14 of its block's largest magnitude. C % 128 == 0
 * (MOE_ERR_ALIGNMENT); x and codes 16-byte aligned. rows == 0 is a no-op. */
moe_status moe_e4m3_split(const void* x, int rows, int C, uint8_t* codes, uint8_t* scales, cudaStream_t stream);
size_t moe_mx_prepared_scales_size(int E_local, int rows, int cols);
moe_status moe_mx_prepare_scales(const uint8_t* scales, int E_local, int rows, int cols, uint8_t* out,
                                 cudaStream_t stream);

const char* moe_status_string(int status);

/* Returns and clears the device error word of the current device: MOE_OK,
 * MOE_ERR_DEVICE_INDEX or MOE_ERR_DEVICE_TIMEOUT (MOE_ERR_CUDA if a CUDA call
 * failed). The read and the clear are one atomic exchange on the device,
 * enqueued on `stream` after everything enqueued there before; the call then
 * waits for it (it synchronizes `stream`). Not for the hot path, and not to be
 * called from several host threads at once for one device (they share the
 * slot the exchanged value is copied through). */
moe_status moe_get_error(cudaStream_t stream);

/* MOE_OK if the current device has compute capability 10.3. */
moe_status moe_device_check(void);

/* Launch-plan override for moe_experts and moe_shared_expert (tuning and
 * tests): token tile width (16, 32, 64, 128 or 256), the split-K factor of
 * GEMM1 and GEMM2 (clamped so every split keeps at least one K-block), and
 * the number of 128-row weight tiles per GEMM2 work unit (1 or 2; 2 needs
 * K % 256 == 0), and how GEMM1 and GEMM2 run: one fused launch (1), two
 * launches (2), or two launches on CTA pairs (3: bf16 weights, 128- or
 * 256-token tiles, no split-K; otherwise as 2). 0 restores the automatic
 * choice. It applies to every later
 * call in the process, including the *_workspace_size() queries, so query the
 * workspace size after setting it. Not synchronised with concurrent calls. */
moe_status moe_set_plan_override(int token_tile, int splits_gemm1, int splits_gemm2, int gemm2_tiles,
                                 int fuse);

/* The float32 sigmoid spec the sigmoid router selects with, applied to
 * x f32 [n] -> y f32 [n] (a test hook: the CPU oracle implements the same
 * written spec independently, and the two must agree bit for bit). */
moe_status moe_debug_sigmoid(const float* x, float* y, int n, cudaStream_t stream);

/* The kernels' bounded wait on a device counter, alone (a test hook for the
 * failure path): one thread waits until flag[0] >= target for at most
 * limit_ns nanoseconds (1 .. 2e9, else MOE_ERR_INVALID_ARG). If the wait runs
 * out, the device error word gets MOE_ERR_DEVICE_TIMEOUT (read with
 * moe_get_error) and the kernel returns; nothing traps. */
moe_status moe_debug_bounded_wait(const int* flag, int target, unsigned long long limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
