// Host side of the experts step: TMA descriptors, the launch plan (token-tile
// width, split-K), the workspace layout, and the GEMM1 -> GEMM2 launches.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_kernel.cuh"
#include "gemm_mx8_kernel.cuh"
#include "gemm_pair_kernel.cuh"

namespace moe {
namespace {

using gemm::GemmArgs;
using gemm::kBK;
using gemm::kBM;
using gemm::kMaxSplitTiles;

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D row-major tensor [outer, inner] of 1- or 2-byte elements, box {box_inner, box_outer}.
bool encode_2d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * esize};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 operand tile: 64 elements (128 bytes) x box_outer rows, 128-byte swizzle.
bool encode_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    return encode_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, kBK, box_outer,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// Packed e2m1 codes [outer, inner codes] (inner / 2 bytes per row) for the
// block-scaled MMA: 128 codes x 128 rows per box, landing as 128-byte padded
// rows under the 128-byte swizzle (16U4_ALIGN16B).
bool encode_fp4(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner / 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(gemm::kMxBK), static_cast<cuuint32_t>(kBM)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- plan: token-tile width, split-K and workspace layout --------------------------
struct PlanOverride {
    int token_tile = 0;          // 0 = automatic
    int splits[2] = {0, 0};      // GEMM1, GEMM2; 0 = automatic
    int gemm2_na = 0;            // 128-row A tiles per GEMM2 unit (1 or 2); 0 = automatic
    int fuse = 0;                // 0 = automatic, 1 = one fused launch, 2 = two launches, 3 = CTA pairs
};
PlanOverride g_override;

// Token tile: about twice the average rows per group, four times with 64 or
// more groups (a group never holds more than M rows: a token routes to an
// expert once), at least 32. With many experts the load per expert is
// heavy-tailed, and a busy expert cut into several tiles streams its weights
// once per tile. 256-row tiles fill all 512 TMEM columns, which leaves the
// epilogue unoverlapped; they pay off only when work units are long (both
// reductions >= 4096) or when each decoded MXFP4 weight tile should serve as
// many tokens as possible.
int pick_bt(int M, int rows_alloc, int groups, int K, int N, bool mx) {
    const int avg = (rows_alloc + groups - 1) / (groups > 0 ? groups : 1);
    const int mult = groups >= 64 ? 4 : 2;
    const int want = avg * mult < M ? avg * mult : M;
    const int cap = (mx || (K >= 4096 && N >= 4096)) ? 256 : 128;
    int bt = 32;
    while (bt < want && bt < cap) bt <<= 1;
    return bt;
}

struct GemmPlan {
    int na, n_wtiles, splits, max_tiles;
    size_t partial_bytes;
};

// direct: the splits reduce into the output themselves (the finalizing GEMM2):
// no partial tiles, and an extra split costs one more tile of reductions.
GemmPlan plan_gemm(int gemm_index, int bt, int na, int n_wtiles, int kr, int rows_alloc, int groups,
                   int sm_count, bool direct = false) {
    GemmPlan p;
    p.na = na;
    p.n_wtiles = n_wtiles;
    const int nonempty = groups < rows_alloc ? groups : rows_alloc;
    p.max_tiles = n_wtiles * (rows_alloc / bt + nonempty + 1);
    const int tt = (rows_alloc + bt - 1) / bt > nonempty ? (rows_alloc + bt - 1) / bt : nonempty;
    const long long est = static_cast<long long>(n_wtiles) * (tt > 0 ? tt : 1);   // expected tiles
    const int nkb = kr / kBK;
    int s = 1;
    if (est < 2LL * sm_count && p.max_tiles <= kMaxSplitTiles) {
        // time ~ waves x (k-blocks per unit + the split epilogue's extra
        // traffic: writing and reading back the fp32 partial tile, counted in
        // k-blocks of operand traffic)
        const double part = (direct ? 1.0 : 2.0) * na * kBM * bt * 4.0;
        const double kblock = na * kBM * kBK * 2.0 + bt * kBK * 2.0;
        const double ovh = part / kblock;
        const int cap = nkb / 4 > 1 ? (nkb / 4 < 16 ? nkb / 4 : 16) : 1;
        double best = 1e30;
        for (int c = 1; c <= cap; ++c) {
            const long long units = est * c;
            const long long waves = (units + sm_count - 1) / sm_count;
            const double t = static_cast<double>(waves) * (static_cast<double>(nkb) / c + (c > 1 ? ovh : 0.0));
            if (t < best - 1e-9) { best = t; s = c; }
        }
    }
    if (g_override.splits[gemm_index] > 0 && p.max_tiles <= kMaxSplitTiles) s = g_override.splits[gemm_index];
    if (s > nkb) s = nkb;
    p.splits = s;
    p.partial_bytes = (s > 1 && !direct) ? static_cast<size_t>(p.max_tiles) * s * na * kBM * bt * sizeof(float) : 0;
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Counters at the start of the workspace, kept zero between calls: four
// regions of kMaxSplitTiles (split-K arrivals of GEMM1 and GEMM2, token-tile
// ready and consumed counts), then the output-start counters of a fused
// finalizing launch (KernelArgs::init_done).
constexpr size_t kCounterBytes = (4 * static_cast<size_t>(kMaxSplitTiles) + 64) * sizeof(int);

// A finalizing call's output start, written by its GEMM1 launch: out = the
// shared expert's output, or 0.
void set_out_init(GemmArgs& a, const ExpertsProblem& p) {
    if (p.out_preset) return;                          // the caller wrote the start
    a.init_out = p.fin_out;
    a.init_src = p.fin_shared;
    a.init_src_dtype = p.fin_shared_dtype;
    a.init_n = static_cast<long long>(p.M) * p.w->K;
}

// Before the first launch that adds into a preset output start: wait for
// the event after which the start is written (another stream's work).
cudaError_t wait_out_ready(const ExpertsProblem& p, cudaStream_t s) {
    return (p.fin_out != nullptr && p.out_ready != nullptr) ? cudaStreamWaitEvent(s, p.out_ready, 0) : cudaSuccess;
}

struct Layout {
    int bt;
    bool fused;
    bool pair;
    int max_token_tiles;
    GemmPlan g1, g2;
    size_t off_act, off_p1, off_p2, total;
    // MXFP8 activations (MOE_WEIGHTS_MXFP4_A8): x codes and atoms, act codes and atoms
    size_t off_xq = 0, off_xs = 0, off_aq = 0, off_as = 0;
    // x in token order on a format that reads x_perm by TMA: the gathered rows
    size_t off_xg = 0;
};

// MXFP4 weights on the block-scaled MMAs: three launches (quantise x, GEMM1
// with the quantising epilogue, GEMM2), token tiles of at most 128 B rows (one
// scale atom per tile and k-block). MXFP8 activations (A8): one B row per
// token. bf16 activations as two E4M3 terms (A16): two B rows per token, so
// tiles of at most 64 tokens and twice the code buffers. L.bt counts tokens.
// Plans count k-blocks of 128 elements.
Layout make_layout_a8(const moe_weights* w, int rows_alloc, int M, int groups, int sm_count, bool fin) {
    Layout L;
    const int K = w->K, N = w->N;
    const int rb = w->format == MOE_WEIGHTS_MXFP4_A16 ? 2 : 1;       // B rows per token
    L.bt = g_override.token_tile > 0 ? g_override.token_tile : pick_bt(M, rows_alloc, groups, K, N, false);
    if (L.bt > 128 / rb) L.bt = 128 / rb;
    // bf16 activations (two B rows per token): 56-token tiles rather than 64,
    // so that the 112-column accumulators leave TMEM room for two buffers
    // (2 x 2 x 112 + the ring's scale columns = 512) and the epilogue of one
    // unit overlaps the next unit's MMAs
    if (rb == 2 && L.bt == 64 && g_override.token_tile == 0) L.bt = 56;
    L.g1 = plan_gemm(0, L.bt, 2, N / kBM, K / 2, rows_alloc, groups, sm_count);
    L.g2 = plan_gemm(1, L.bt, 2, K / (2 * kBM), N / 2, rows_alloc, groups, sm_count, fin);
    // a split's fp32 partial tile holds every B row of the token tile: rb rows per token
    L.g1.partial_bytes *= rb;
    L.g2.partial_bytes *= rb;
    L.fused = false;
    L.pair = false;
    L.max_token_tiles = rows_alloc / L.bt + (groups < rows_alloc ? groups : rows_alloc) + 1;
    const size_t tiles = static_cast<size_t>(L.max_token_tiles);
    size_t off = kCounterBytes;
    L.off_act = 0;
    L.off_xq = off;
    off = align256(off + static_cast<size_t>(rb) * rows_alloc * K);
    L.off_xs = off;
    off = align256(off + tiles * (K / gemm::kMxBK) * gemm::kAtom);
    L.off_aq = off;
    off = align256(off + static_cast<size_t>(rb) * rows_alloc * N);
    L.off_as = off;
    off = align256(off + tiles * (N / gemm::kMxBK) * gemm::kAtom);
    L.off_p1 = off;
    off = align256(off + L.g1.partial_bytes);
    L.off_p2 = off;
    off = align256(off + L.g2.partial_bytes);
    L.total = off;
    return L;
}

// fin: GEMM2 finalizes in its epilogue (needs no more workspace than without)
// batched: the BatchedExperts layout, which runs as two one-CTA launches
Layout make_layout(const moe_weights* w, int rows_alloc, int M, int groups, int sm_count, bool fin = false,
                   bool batched = false) {
    if (w->format == MOE_WEIGHTS_MXFP4_A8 || w->format == MOE_WEIGHTS_MXFP4_A16)
        return make_layout_a8(w, rows_alloc, M, groups, sm_count, fin);
    Layout L;
    const int K = w->K, N = w->N;
    L.bt = g_override.token_tile > 0 ? g_override.token_tile
                                     : pick_bt(M, rows_alloc, groups, K, N, w->format == MOE_WEIGHTS_MXFP4);
    L.g1 = plan_gemm(0, L.bt, 2, N / kBM, K, rows_alloc, groups, sm_count);
    int na2 = (K % 256 == 0) ? 2 : 1;
    if (g_override.gemm2_na == 1 || (g_override.gemm2_na == 2 && K % 256 == 0)) na2 = g_override.gemm2_na;
    L.g2 = plan_gemm(1, L.bt, na2, K / (na2 * kBM), N, rows_alloc, groups, sm_count, fin);
    // GEMM1 and GEMM2 in one launch when GEMM2 units take two A tiles and the
    // token-tile counters fit their region
    L.max_token_tiles = rows_alloc / L.bt + (groups < rows_alloc ? groups : rows_alloc) + 1;
    // With many experts that each hold long runs of rows (16 or more groups,
    // at least 256 rows on average) the two GEMMs run as two launches: a
    // same-box sweep of the Qwen3-shaped layer at M = 8192 measured 518 us
    // against 531 us for the one fused launch (which still wins at M = 2048,
    // 212 us against 217 us).
    const bool long_runs = g_override.fuse == 0 && groups >= 16 && rows_alloc / groups >= 256;
    L.fused = L.g2.na == 2 && L.max_token_tiles <= kMaxSplitTiles && g_override.fuse != 2 &&
              g_override.fuse != 3 && !batched && !long_runs;
    // GEMM1 and GEMM2 on CTA pairs (two launches): bf16 weights, 128- or
    // 256-token tiles, every unit whole (no split-K), 256-row GEMM2 units.
    // Forced by the override (fuse = 3, with its tile width); chosen
    // automatically with 256-token tiles when the experts average at least
    // 256 rows, so that most tiles are full and the units fill the grid, and
    // the intermediate size is at least 2048: a same-box sweep measured pairs
    // ahead at Mixtral M = 4096 (1.67 ms against 1.90 on one CTA) and for the
    // DeepSeek shared expert at M = 8192 (413 us against 467), and behind at
    // Qwen3 M = 8192 (N = 768: 546 us against 518). The choice does not
    // depend on `fin`, so the workspace query and the launch agree on the
    // layout.
    const bool pair_ok = w->format == MOE_WEIGHTS_BF16 && K % 256 == 0 && N % kBM == 0 &&
                         g_override.gemm2_na != 1 && !batched;
    L.pair = false;
    if (pair_ok && g_override.fuse == 3 && (L.bt == 128 || L.bt == 256) && L.g1.splits == 1 && L.g2.na == 2 &&
        plan_gemm(1, L.bt, 2, K / (2 * kBM), N, rows_alloc, groups, sm_count).splits == 1) {
        L.pair = true;
    } else if (pair_ok && g_override.fuse == 0 && g_override.token_tile == 0 && groups > 0 &&
               rows_alloc / groups >= 256 && N >= 2048) {
        const GemmPlan p1 = plan_gemm(0, 256, 2, N / kBM, K, rows_alloc, groups, sm_count);
        const GemmPlan p2 = plan_gemm(1, 256, 2, K / (2 * kBM), N, rows_alloc, groups, sm_count);
        if (p1.splits == 1 && p2.splits == 1) {
            L.pair = true;
            L.bt = 256;
            L.g1 = p1;
            L.g2 = p2;
        }
    }
    if (L.pair) {
        L.fused = false;
        L.g1.splits = L.g2.splits = 1;                   // pair units are whole
        L.g1.partial_bytes = L.g2.partial_bytes = 0;
    }
    // four counter regions, kept zero between calls: split-K arrivals of
    // GEMM1 and GEMM2, token-tile ready and consumed counts
    size_t off = kCounterBytes;
    L.off_act = off;
    off = align256(off + static_cast<size_t>(rows_alloc) * N * 2);
    L.off_p1 = off;
    off = align256(off + L.g1.partial_bytes);
    L.off_p2 = off;
    off = align256(off + L.g2.partial_bytes);
    L.total = off;
    return L;
}

// A-operand descriptors of one weight matrix [E*rows, kr] (bf16) or its packed
// codes [E*rows, kr/2] + scales [E*rows, kr/32] (MXFP4).
bool encode_weights(CUtensorMap* tmA, CUtensorMap* tmS, bool mx, const void* w, const uint8_t* sc,
                    uint64_t kr, uint64_t rows) {
    if (!mx) {
        if (!encode_bf16(tmA, w, kr, rows, kBM)) return false;
        *tmS = *tmA;                                        // unused
        return true;
    }
    return encode_2d(tmA, w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kr / 2, rows, kBK / 2, kBM,
                     CU_TENSOR_MAP_SWIZZLE_NONE) &&
           encode_2d(tmS, sc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kr / 32, rows, 16, kBM,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
}

// The experts with MXFP8 activations: x_perm -> codes + atoms, GEMM1 (act
// codes + atoms), GEMM2 (y, or the finalize into the f32 out).
cudaError_t launch_experts_a8(const ExpertsProblem& p, const Layout& L, uint8_t* ws, int* err, const DeviceInfo& dev,
                              cudaStream_t s) {
    const moe_weights* w = p.w;
    const int K = w->K, N = w->N;
    const uint64_t E = static_cast<uint64_t>(w->E_local);
    const bool fin = p.fin_out != nullptr;
    const bool hl = w->format == MOE_WEIGHTS_MXFP4_A16;
    const int rb = hl ? 2 : 1;                                   // B rows per token
    const uint64_t brows = static_cast<uint64_t>(rb) * p.rows_alloc;
    uint8_t* xq = ws + L.off_xq;
    uint8_t* xs = ws + L.off_xs;
    uint8_t* aq = ws + L.off_aq;
    uint8_t* as = ws + L.off_as;
    int* counters = reinterpret_cast<int*>(ws);
    CUtensorMap tA1, tB1, tA2, tB2;
    if (!encode_fp4(&tA1, w->w1, K, E * 2 * N) || !encode_fp4(&tA2, w->w2, N, E * K) ||
        !encode_2d(&tB1, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, brows, gemm::kMxBK, rb * L.bt,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tB2, aq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, brows, gemm::kMxBK, rb * L.bt,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    gemm::Mx8Args m1{};
    GemmArgs& a1 = m1.g;
    a1.offsets = p.offsets;
    a1.groups = w->E_local;
    a1.rows_alloc = p.rows_alloc;
    a1.kr = K;
    a1.rows_per_group = 2 * N;
    a1.n_wtiles = L.g1.n_wtiles;
    a1.wtile_rows = kBM;
    a1.a1_offset = N;
    a1.splits = L.g1.splits;
    a1.out_ld = N;
    a1.out = aq;
    a1.partials = reinterpret_cast<float*>(ws + L.off_p1);
    a1.counters = counters;
    a1.max_tiles = L.g1.max_tiles;
    a1.err = err;
    a1.act = w->activation;
    a1.clamp = w->activation_clamp;
    m1.sfa = w->w1_scale;
    m1.sfb = xs;
    m1.sfb_out = as;
    m1.max_token_tiles = L.max_token_tiles;
    gemm::Mx8Args m2 = m1;
    GemmArgs& a2 = m2.g;
    a2.init_out = nullptr;
    a2.kr = N;
    a2.rows_per_group = K;
    a2.n_wtiles = L.g2.n_wtiles;
    a2.wtile_rows = 2 * kBM;
    a2.a1_offset = kBM;
    a2.splits = L.g2.splits;
    a2.out_ld = K;
    a2.out = fin ? static_cast<void*>(p.fin_out) : p.y;
    a2.inverse = p.inverse;
    a2.fw = p.fin_weights;
    a2.fw_dtype = p.fin_weights_dtype;
    a2.top_k = p.top_k;
    a2.rsf = p.rsf;
    a2.partials = reinterpret_cast<float*>(ws + L.off_p2);
    a2.counters = counters + kMaxSplitTiles;
    a2.max_tiles = L.g2.max_tiles;
    m2.sfa = w->w2_scale;
    m2.sfb = as;
    m2.sfb_out = nullptr;
    const int grid = dev.sm_count;
    if (fin) set_out_init(a1, p);                       // GEMM1 writes the output start
    cudaError_t e = launch_mxfp8_quantize_tiles(p.x, p.rows_alloc, K, p.offsets, w->E_local, L.bt, L.max_token_tiles,
                                                xq, xs, err, dev, s, hl, p.x_tokens ? p.inverse : nullptr, p.top_k);
    if (e != cudaSuccess) return e;
    auto gemm_launch = hl ? gemm::launch_gemm_mx8_hl : gemm::launch_gemm_mx8;
    e = gemm_launch(gemm::MODE_SWIGLU, rb * L.bt, MOE_DTYPE_BF16, tA1, tB1, m1, grid, s);
    if (e != cudaSuccess) return e;
    if ((e = wait_out_ready(p, s)) != cudaSuccess) return e;
    return gemm_launch(fin ? gemm::MODE_FINAL : gemm::MODE_PLAIN, rb * L.bt, p.y_dtype, tA2, tB2, m2, grid, s);
}

cudaError_t launch_one(bool mx, int fused, int mode, int bt, int na, int out_dtype, const gemm::Maps& m,
                       const gemm::KernelArgs& ka, int grid, cudaStream_t s) {
    return mx ? gemm::launch_gemm_mxfp4(fused, mode, bt, na, out_dtype, m, ka, grid, s)
              : gemm::launch_gemm_bf16(fused, mode, bt, na, out_dtype, m, ka, grid, s);
}

}  // namespace

void set_plan_override(int token_tile, int splits1, int splits2, int gemm2_na, int fuse) {
    g_override.token_tile = token_tile;
    g_override.splits[0] = splits1;
    g_override.splits[1] = splits2;
    g_override.gemm2_na = gemm2_na;
    g_override.fuse = fuse;
}

namespace {
// The block-scaled formats quantise x row by row and can read it in token
// order; the others load x_perm by TMA and need it gathered first.
bool reads_x_tokens(const moe_weights* w) {
    return w->format == MOE_WEIGHTS_MXFP4_A8 || w->format == MOE_WEIGHTS_MXFP4_A16;
}

// With x in token order on a format that needs x_perm, the gathered rows
// [rows_alloc, K] bf16 go after the rest of the workspace (whose layout does
// not change).
Layout make_layout_x(const moe_weights* w, int rows_alloc, int M, int groups, int sm_count, bool fin, bool batched,
                     bool x_tokens) {
    Layout L = make_layout(w, rows_alloc, M, groups, sm_count, fin, batched);
    if (x_tokens && !reads_x_tokens(w)) {
        L.off_xg = L.total;
        L.total = align256(L.total + static_cast<size_t>(rows_alloc) * w->K * 2);
    }
    return L;
}
}  // namespace

size_t experts_workspace_bytes(const moe_weights* w, int rows_alloc, int M, const DeviceInfo& dev, bool batched,
                               bool x_tokens) {
    return make_layout_x(w, rows_alloc, M, w->E_local, dev.sm_count, false, batched, x_tokens).total;
}

namespace {
// The kernels' bounded counter wait, alone (a test hook for the give-up path):
// wait until *flag >= target for at most limit_ns; on expiry the error word
// gets MOE_ERR_DEVICE_TIMEOUT and the kernel returns.
__global__ void bounded_wait_kernel(const int* flag, int target, unsigned long long limit_ns, int* err) {
    __shared__ int abort_flag;
    abort_flag = 0;
    gemm::wait_counter(flag, target, &abort_flag, err, limit_ns);
}
}  // namespace

cudaError_t launch_debug_bounded_wait(const int* flag, int target, unsigned long long limit_ns, int* err,
                                      cudaStream_t s) {
    return launch_plain(bounded_wait_kernel, dim3(1), dim3(1), 0, s, flag, target, limit_ns, err);
}

int experts_launches(const moe_weights* w, int rows_alloc, int M, bool fin, const DeviceInfo& dev) {
    if (w->format == MOE_WEIGHTS_MXFP4_A8 || w->format == MOE_WEIGHTS_MXFP4_A16) return 3;
    const Layout L = make_layout(w, rows_alloc, M, w->E_local, dev.sm_count, fin);
    return (L.pair || !L.fused) ? 2 : 1;
}

cudaError_t launch_experts(const ExpertsProblem& p_in, void* workspace, size_t /*workspace_bytes*/, int* err,
                           const DeviceInfo& dev, cudaStream_t s) {
    // x in token order: the block-scaled formats read it so (their quantiser
    // gathers the rows); the others get x_perm gathered into the workspace
    // first and then run on it
    ExpertsProblem pg;
    const ExpertsProblem* pp = &p_in;
    if (p_in.x_tokens && !reads_x_tokens(p_in.w)) {
        const Layout Lx = make_layout_x(p_in.w, p_in.rows_alloc, p_in.M, p_in.w->E_local, dev.sm_count,
                                        p_in.fin_out != nullptr, false, true);
        uint8_t* xg = static_cast<uint8_t*>(workspace) + Lx.off_xg;
        const cudaError_t eg = launch_gather_rows(p_in.offsets, p_in.w->E_local, p_in.inverse, p_in.top_k,
                                                  p_in.rows_alloc, p_in.x, p_in.w->K, xg, dev, s);
        if (eg != cudaSuccess) return eg;
        pg = p_in;
        pg.x = xg;
        pg.x_tokens = false;
        pp = &pg;
    }
    const ExpertsProblem& p = *pp;
    const moe_weights* w = p.w;
    const int K = w->K, N = w->N;
    const bool mx = w->format == MOE_WEIGHTS_MXFP4;
    const int groups = (p.offsets != nullptr || p.counts != nullptr) ? w->E_local : 1;
    const bool fin = p.fin_out != nullptr;
    const bool batched = p.counts != nullptr;
    const Layout L = make_layout(w, p.rows_alloc, p.M, groups, dev.sm_count, fin, batched);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* counters = reinterpret_cast<int*>(ws);
    void* act = ws + L.off_act;

    const uint64_t E = static_cast<uint64_t>(w->E_local);
    if (w->format == MOE_WEIGHTS_MXFP4_A8 || w->format == MOE_WEIGHTS_MXFP4_A16)
        return launch_experts_a8(p, L, ws, err, dev, s);

    gemm::Maps m;
    if (!encode_weights(&m.A[0], &m.S[0], mx, w->w1, w->w1_scale, K, E * 2 * N) ||
        !encode_weights(&m.A[1], &m.S[1], mx, w->w2, w->w2_scale, N, E * K) ||
        !encode_bf16(&m.B[0], p.x, K, p.rows_alloc, L.bt) || !encode_bf16(&m.B[1], act, N, p.rows_alloc, L.bt))
        return cudaErrorInvalidValue;

    gemm::KernelArgs ka{};
    GemmArgs& a1 = ka.g[0];
    a1.offsets = p.offsets;
    a1.single_rows = p.single_rows;
    a1.groups = groups;
    a1.rows_alloc = p.rows_alloc;
    a1.kr = K;
    a1.rows_per_group = 2 * N;
    a1.n_wtiles = L.g1.n_wtiles;
    a1.wtile_rows = kBM;
    a1.a1_offset = N;
    a1.splits = L.g1.splits;
    a1.out_ld = N;
    a1.out = act;
    a1.partials = reinterpret_cast<float*>(ws + L.off_p1);
    a1.counters = counters;
    a1.max_tiles = L.g1.max_tiles;
    a1.err = err;
    a1.act = w->activation;
    a1.clamp = w->activation_clamp;
    a1.counts = p.counts;
    a1.batch_stride = p.batch_stride;
    GemmArgs& a2 = ka.g[1];
    a2 = a1;
    a2.init_out = nullptr;
    a2.kr = N;
    a2.rows_per_group = K;
    a2.n_wtiles = L.g2.n_wtiles;
    a2.wtile_rows = L.g2.na * kBM;
    a2.a1_offset = kBM;
    a2.splits = L.g2.splits;
    a2.out_ld = K;
    a2.out = fin ? static_cast<void*>(p.fin_out) : p.y;
    a2.inverse = p.inverse;
    a2.fw = p.fin_weights;
    a2.fw_dtype = p.fin_weights_dtype;
    a2.top_k = p.top_k;
    a2.rsf = p.rsf;
    a2.partials = reinterpret_cast<float*>(ws + L.off_p2);
    a2.counters = counters + kMaxSplitTiles;
    a2.max_tiles = L.g2.max_tiles;
    ka.ready = counters + 2 * kMaxSplitTiles;
    ka.consumed = counters + 3 * kMaxSplitTiles;
    ka.max_token_tiles = L.max_token_tiles;

    const int grid = dev.sm_count;
    if (fin) {
        // out = shared (or 0), written by GEMM1's launch before GEMM2's
        // epilogues add every route into it
        set_out_init(a1, p);
        ka.init_done = counters + 4 * kMaxSplitTiles;
    }
    if (L.pair) {
        // the same units as the one-CTA plan; each CTA of a pair holds half of
        // a unit's weight rows (64-row boxes for GEMM1's gate and up halves)
        // and half of its token rows
        CUtensorMap pa1, pa2, pb1, pb2;
        if (!encode_bf16(&pa1, w->w1, K, E * 2 * N, 64) || !encode_bf16(&pa2, w->w2, N, E * K, kBM) ||
            !encode_bf16(&pb1, p.x, K, p.rows_alloc, L.bt / 2) || !encode_bf16(&pb2, act, N, p.rows_alloc, L.bt / 2))
            return cudaErrorInvalidValue;
        const int pairs = dev.sm_count / 2;
        cudaError_t e = gemm::launch_gemm_pair_bf16(gemm::MODE_SWIGLU, L.bt, MOE_DTYPE_BF16, pa1, pb1, a1, pairs, s);
        if (e != cudaSuccess) return e;
        if ((e = wait_out_ready(p, s)) != cudaSuccess) return e;
        return gemm::launch_gemm_pair_bf16(fin ? gemm::MODE_FINAL : gemm::MODE_PLAIN, L.bt, p.y_dtype, pa2, pb2, a2,
                                           pairs, s);
    }
    if (L.fused) {
        ka.nphase = 2;
        const cudaError_t ew = wait_out_ready(p, s);
        if (ew != cudaSuccess) return ew;
        if (fin) return mx ? gemm::launch_gemm_final_mxfp4(1, L.bt, 2, m, ka, grid, s)
                           : gemm::launch_gemm_final_bf16(1, L.bt, 2, m, ka, grid, s);
        return launch_one(mx, 1, gemm::MODE_PLAIN, L.bt, 2, p.y_dtype, m, ka, grid, s);
    }
    ka.nphase = 1;
    gemm::Maps m1 = m;                                   // phase-0 maps of each launch
    cudaError_t e = launch_one(mx, 0, gemm::MODE_SWIGLU, L.bt, 2, MOE_DTYPE_BF16, m1, ka, grid, s);
    if (e != cudaSuccess) return e;
    gemm::KernelArgs k2 = ka;
    k2.g[0] = a2;
    gemm::Maps m2 = m;
    m2.A[0] = m.A[1];
    m2.S[0] = m.S[1];
    m2.B[0] = m.B[1];
    if ((e = wait_out_ready(p, s)) != cudaSuccess) return e;
    if (fin) return mx ? gemm::launch_gemm_final_mxfp4(0, L.bt, L.g2.na, m2, k2, grid, s)
                       : gemm::launch_gemm_final_bf16(0, L.bt, L.g2.na, m2, k2, grid, s);
    return launch_one(mx, 0, gemm::MODE_PLAIN, L.bt, L.g2.na, p.y_dtype, m2, k2, grid, s);
}

}  // namespace moe
