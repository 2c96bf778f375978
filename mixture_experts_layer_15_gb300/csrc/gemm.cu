// Grouped expert GEMMs of the MoE layer on the sm_103a tensor cores.
//
// The experts step (vllm/model_executor/layers/fused_moe/modular_kernel.py,
// FusedMoEPermuteExpertsUnpermute.apply and .activation) is, per local expert
// g and each of its rows r of x_perm:
//     GEMM1 + silu_and_mul:  act[r]  = silu(W1g[g] x[r]) * (W1u[g] x[r])     (N outputs)
//     GEMM2:                 y[r]    = W2[g] act[r]                           (K outputs)
// unweighted and unreduced. Both are dense contractions over bf16 operands
// with fp32 accumulation and run on tcgen05 MMAs with TMEM accumulators.
//
// Tile shape ("weights as the MMA's M side"): the MMA M dimension (128) runs
// over weight rows and its N dimension (BT = 16..256) over token rows. Decode
// batches (a few tokens per expert) then stream the weights at full MMA width
// instead of padding tokens up to 128. A work unit is
//     (group g, weight tile wt, token tile tt, k-split s)
// and covers two 128-row A tiles (GEMM1: the gate rows n0..n0+127 and the
// matching up rows N+n0..; GEMM2: output rows k0..k0+255) against one
// BT-row token tile, i.e. two accumulators of 128 x BT fp32 in TMEM; the
// GEMM1 epilogue therefore sees gate and up of the same output column in the
// same thread and applies silu(gate)*up with no second pass.
//
// CTA = 6 warps, persistent (one CTA per SM):
//   warp 0     TMA producer: A0, A1, B tiles of 64 reduction elements into a
//              STAGES-deep shared-memory ring (full/empty mbarriers);
//   warp 1     TMEM allocator and MMA issuer (one thread), commits free ring
//              slots and signals finished accumulators;
//   warps 2-5  epilogue: tcgen05.ld of the accumulators (warp w reads TMEM
//              lanes 32*(w%4)..), activation, masked stores by row.
// Accumulators are double-buffered in TMEM when 2 x (2 x BT) <= 512 columns,
// so the epilogue of one unit overlaps the mainloop of the next.
//
// The unit list is built on the device from the group offsets: every CTA
// scans ceil(count_g / BT) * weight tiles * splits over the groups in shared
// memory and strides through units blockIdx.x, +gridDim.x, ... The host never
// learns the routed row count.
//
// Split-K (few units, e.g. decode): each split writes its fp32 partial tile
// to the workspace; a per-tile arrival counter elects the last split, which
// sums the partials in split order (deterministic) and runs the epilogue,
// then resets the counter to zero.
//
// Every mbarrier wait is bounded (~2 s of %globaltimer); on expiry the
// kernel records MOE_ERR_DEVICE_TIMEOUT, raises a shared abort flag that
// releases the other roles, lets its in-flight TMA loads and MMAs land,
// frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int kBM = 128;                  // weight rows per A tile (MMA M)
constexpr int kBK = 64;                   // reduction elements per ring stage (128 B of bf16)
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kMaxGroups = 1024;
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxSplitTiles = 16384;     // capacity of one counter region
constexpr uint64_t kWaitLimitNs = 2000000000ull;

enum { MODE_SWIGLU = 0, MODE_PLAIN = 1 };

struct GemmArgs {
    const int32_t* offsets;   // [groups+1] or nullptr
    int single_rows;          // rows of the single group when offsets == nullptr
    int groups;
    int rows_alloc;           // rows allocated in the B operand and the output
    int kr;                   // reduction length
    int rows_per_group;       // A rows per group
    int n_wtiles;             // weight tiles per group
    int wtile_rows;           // A-row distance between weight tiles
    int a1_offset;            // A-row distance from the first to the second A tile
    int splits;
    int out_ld;               // output row stride (elements)
    void* out;
    float* partials;
    int* counters;
    int max_tiles;
    int* err;
};

template <int BT, int NA>
struct Cfg {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BT * kBK * 2;
    static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
    static constexpr int STAGES_FIT = (kSmemBudget - 12 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int ACC_COLS = NA * BT;
    static constexpr int NBUF = (2 * ACC_COLS <= 512) ? 2 : 1;
    static constexpr int TMEM_NEED = NBUF * ACC_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                   : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    // shared memory layout (offsets from the 1024-aligned base)
    static constexpr int OFF_BAR = STAGES * STAGE_BYTES;          // full[S], empty[S], tfull[2], tempty[2], drain
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;       // tmem base, abort, last flag
    static constexpr int OFF_PREFIX = OFF_MISC + 16;              // [kMaxGroups+1]
    static constexpr int OFF_OFFS = OFF_PREFIX + (kMaxGroups + 1) * 4;   // [kMaxGroups+1]
    static constexpr int OFF_TMP = OFF_OFFS + (kMaxGroups + 1) * 4;      // [33]
    static constexpr int SMEM_BYTES = OFF_TMP + 33 * 4 + 1024;   // + alignment slack
    static_assert(STAGES >= 2, "ring too shallow");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(BT % 16 == 0 && BT >= 16 && BT <= 256, "MMA N");
};

struct Unit {
    int g, wt, s, row0, row_end, kb0, kb1, tile;
};

__device__ __forceinline__ Unit decode_unit(int u, const int* prefix, const int* offs, int BT,
                                            const GemmArgs& a) {
    int lo = 0, hi = a.groups;                 // prefix[lo] <= u < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid;
    }
    Unit un;
    un.g = lo;
    int local = u - prefix[lo];
    un.s = local % a.splits;
    local /= a.splits;
    const int beg = offs[lo], end = offs[lo + 1];
    const int ntt = (end - beg + BT - 1) / BT;
    const int tt = local % ntt;
    un.wt = local / ntt;
    un.row0 = beg + tt * BT;
    un.row_end = min(end, a.rows_alloc);
    const int nkb = a.kr / kBK;
    un.kb0 = un.s * nkb / a.splits;
    un.kb1 = (un.s + 1) * nkb / a.splits;
    un.tile = u / a.splits;
    return un;
}

// Bounded wait on an mbarrier phase. Returns false when the wait was given up
// (this thread timed out, or another role raised the abort flag).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 127u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                set_error(err, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

template <typename OutT>
__device__ __forceinline__ void store_out(OutT* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// Epilogue of 16 token columns [c0, c0+16) for this thread's weight row.
template <int NA, int MODE, typename OutT>
__device__ __forceinline__ void emit16(const Unit& un, const GemmArgs& a, int row_in_tile, int c0,
                                       const float (&v0)[16], const float (&v1)[16]) {
    OutT* out = static_cast<OutT*>(a.out);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int r = un.row0 + c0 + i;
        if (r < un.row_end) {
            const size_t rb = static_cast<size_t>(r) * a.out_ld;
            if (MODE == MODE_SWIGLU) {
                store_out<OutT>(out + rb + un.wt * kBM + row_in_tile, silu_mul(v0[i], v1[i]));
            } else {
                const int col = un.wt * a.wtile_rows + row_in_tile;
                store_out<OutT>(out + rb + col, v0[i]);
                if (NA == 2) store_out<OutT>(out + rb + col + kBM, v1[i]);
            }
        }
    }
}

template <int BT, int NA, int MODE, typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmArgs a) {
    using C = Cfg<BT, NA>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2 + b); };
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    int* offs = reinterpret_cast<int*>(smem + C::OFF_OFFS);
    int* tmp = reinterpret_cast<int*>(smem + C::OFF_TMP);

    // ---- prologue: barriers, TMEM, unit schedule ----
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kEpiThreads);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    // group offsets (validated: non-decreasing, within the allocation)
    for (int g = tid; g <= a.groups; g += kThreads) {
        int v = a.offsets != nullptr ? __ldg(a.offsets + g) : (g == 0 ? 0 : a.single_rows);
        if (v < 0 || v > a.rows_alloc) { set_error(a.err, MOE_ERR_DEVICE_INDEX); v = v < 0 ? 0 : a.rows_alloc; }
        offs[g] = v;
    }
    __syncthreads();
    for (int g = tid; g < a.groups; g += kThreads) {
        int cnt = offs[g + 1] - offs[g];
        if (cnt < 0) { set_error(a.err, MOE_ERR_DEVICE_INDEX); cnt = 0; }
        prefix[g] = ((cnt + BT - 1) / BT) * a.n_wtiles * a.splits;
    }
    __syncthreads();
    const int total_units = block_exclusive_scan(prefix, a.groups, tmp);
    if (tid == 0) prefix[a.groups] = total_units;
    // make the TMEM address written by tcgen05.alloc visible to all threads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_phase = 0;       // per-stage: load in flight / its phase
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
                const Unit un = decode_unit(u, prefix, offs, BT, a);
                const int a0 = un.g * a.rows_per_group + un.wt * a.wtile_rows;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
                    const uint32_t sA = sbase + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), C::STAGE_BYTES);
                    tma_load_2d(sA, &tmA, kb * kBK, a0, full_bar(stage));
                    if (NA == 2) tma_load_2d(sA + C::A_BYTES, &tmA, kb * kBK, a0 + a.a1_offset, full_bar(stage));
                    tma_load_2d(sA + NA * C::A_BYTES, &tmB, kb * kBK, un.row0, full_bar(stage));
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                // let the loads already issued land before the CTA goes away
                for (int s = 0; s < C::STAGES; ++s) {
                    if (!((issued >> s) & 1u)) continue;
                    const uint32_t p = (issued_phase >> s) & 1u;
                    const uint64_t t0 = globaltimer();
                    while (!mbar_try_wait(full_bar(s), p) && globaltimer() - t0 < kWaitLimitNs) {}
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BT);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++it) {
                const Unit un = decode_unit(u, prefix, offs, BT, a);
                const int buf = C::NBUF == 2 ? (it & 1) : 0;
                const uint32_t use = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
                if (!wait_bar(tempty_bar(buf), use ^ 1u, abort_flag, a.err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + buf * C::ACC_COLS;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(full_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA0 = sbase + stage * C::STAGE_BYTES;
                    const uint32_t sB = sA0 + NA * C::A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t bdesc = sw128_kmajor_desc(sB + kk * 32);
                        const uint32_t acc = (kb > un.kb0 || kk > 0) ? 1u : 0u;
                        mma_f16(d, sw128_kmajor_desc(sA0 + kk * 32), bdesc, idesc, acc);
                        if (NA == 2)
                            mma_f16(d + BT, sw128_kmajor_desc(sA0 + C::A_BYTES + kk * 32), bdesc, idesc, acc);
                    }
                    mma_commit(empty_bar(stage));            // ring slot free once these MMAs finish
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(tfull_bar(buf));                  // accumulator ready for the epilogue
            }
            // all MMAs of this CTA complete before TMEM is released
            mma_commit(drain_bar);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {}
        }
        __syncwarp();
    } else {
        // ================= epilogue (warps 2..5) =================
        const int q = warp & 3;                              // TMEM lanes 32q..32q+31
        const int row_in_tile = q * 32 + lane;
        const int etid = tid - 64;
        int it = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++it) {
            const Unit un = decode_unit(u, prefix, offs, BT, a);
            const int buf = C::NBUF == 2 ? (it & 1) : 0;
            const uint32_t use = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
            wait_bar(tfull_bar(buf), use, abort_flag, a.err);
            named_bar_sync(1, kEpiThreads);                  // all threads decide together
            if (*abort_flag) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_COLS;
            if (a.splits == 1) {
#pragma unroll 1
                for (int c0 = 0; c0 < BT; c0 += 16) {
                    float v0[16], v1[16];
                    if (NA == 2) tmem_ld16x2(tb + c0, tb + BT + c0, v0, v1);
                    else tmem_ld16(tb + c0, v0);
                    emit16<NA, MODE, OutT>(un, a, row_in_tile, c0, v0, v1);
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(buf));
            } else {
                const size_t slot = static_cast<size_t>(NA) * kBM * BT;
                const bool tile_ok = un.tile < a.max_tiles;
                float* part = a.partials + (static_cast<size_t>(un.tile) * a.splits + un.s) * slot;
#pragma unroll 1
                for (int c0 = 0; c0 < BT; c0 += 16) {
                    float v0[16], v1[16];
                    if (NA == 2) tmem_ld16x2(tb + c0, tb + BT + c0, v0, v1);
                    else tmem_ld16(tb + c0, v0);
                    if (tile_ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            part[static_cast<size_t>(c0 + i) * kBM + row_in_tile] = v0[i];
                            if (NA == 2) part[static_cast<size_t>(BT + c0 + i) * kBM + row_in_tile] = v1[i];
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(buf));
                __threadfence();
                named_bar_sync(1, kEpiThreads);
                if (etid == 0) {
                    int last = 0;
                    if (tile_ok) {
                        const int old = atomicAdd(a.counters + un.tile, 1);
                        last = (old == a.splits - 1);
                        if (last) a.counters[un.tile] = 0;   // left at zero for the next call
                    } else {
                        set_error(a.err, MOE_ERR_DEVICE_INDEX);
                    }
                    *last_flag = last;
                }
                named_bar_sync(1, kEpiThreads);
                const int last = *last_flag;
                if (last) {
                    __threadfence();
                    const float* p0 = a.partials + static_cast<size_t>(un.tile) * a.splits * slot;
#pragma unroll 1
                    for (int c0 = 0; c0 < BT; c0 += 16) {
                        float v0[16], v1[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) { v0[i] = 0.0f; v1[i] = 0.0f; }
                        for (int s = 0; s < a.splits; ++s) {
                            const float* ps = p0 + s * slot;
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                v0[i] += __ldcg(ps + static_cast<size_t>(c0 + i) * kBM + row_in_tile);
                                if (NA == 2) v1[i] += __ldcg(ps + static_cast<size_t>(BT + c0 + i) * kBM + row_in_tile);
                            }
                        }
                        emit16<NA, MODE, OutT>(un, a, row_in_tile, c0, v0, v1);
                    }
                }
                named_bar_sync(1, kEpiThreads);              // last_flag is reused by the next unit
            }
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------

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

// bf16 2D tensor [outer, inner] (row-major) with a (box_outer x 64) box, 128B swizzle.
bool encode_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BT, int NA, int MODE, typename OutT>
cudaError_t launch_kernel(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                          cudaStream_t s) {
    using C = Cfg<BT, NA>;
    auto kern = grouped_gemm_kernel<BT, NA, MODE, OutT>;
    static std::atomic<uint64_t> configured{0};      // bit per device ordinal
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    kern<<<grid, kThreads, C::SMEM_BYTES, s>>>(tmA, tmB, a);
    return cudaGetLastError();
}

template <int NA, int MODE, typename OutT>
cudaError_t launch_bt(int bt, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                      cudaStream_t s) {
    switch (bt) {
        case 16: return launch_kernel<16, NA, MODE, OutT>(tmA, tmB, a, grid, s);
        case 32: return launch_kernel<32, NA, MODE, OutT>(tmA, tmB, a, grid, s);
        case 64: return launch_kernel<64, NA, MODE, OutT>(tmA, tmB, a, grid, s);
        case 128: return launch_kernel<128, NA, MODE, OutT>(tmA, tmB, a, grid, s);
        default: return launch_kernel<256, NA, MODE, OutT>(tmA, tmB, a, grid, s);
    }
}

// ---- plan: token-tile width, split-K and workspace layout --------------------------
int pick_bt(int M, int rows_alloc, int groups) {
    // a group never holds more than M rows (a token routes to an expert once)
    const int avg = (rows_alloc + groups - 1) / (groups > 0 ? groups : 1);
    int want = avg * 2 < M ? avg * 2 : M;
    int bt = 16;
    while (bt < want && bt < 256) bt <<= 1;
    return bt;
}

struct GemmPlan {
    int na, n_wtiles, splits, max_tiles;
    size_t partial_bytes;
};

GemmPlan plan_gemm(int bt, int na, int n_wtiles, int kr, int rows_alloc, int groups, int sm_count) {
    GemmPlan p;
    p.na = na;
    p.n_wtiles = n_wtiles;
    const int nonempty = groups < rows_alloc ? groups : rows_alloc;
    p.max_tiles = n_wtiles * (rows_alloc / bt + nonempty + 1);
    const int est_tt = (rows_alloc + bt - 1) / bt > nonempty ? (rows_alloc + bt - 1) / bt : nonempty;
    const long long est = static_cast<long long>(n_wtiles) * (est_tt > 0 ? est_tt : 1);
    const int nkb = kr / kBK;
    int s = 1;
    if (est < 2LL * sm_count && p.max_tiles <= kMaxSplitTiles) {
        s = static_cast<int>((2LL * sm_count + est - 1) / est);
        int cap = nkb / 4 > 1 ? nkb / 4 : 1;
        if (s > cap) s = cap;
        if (s > 16) s = 16;
        if (s < 1) s = 1;
    }
    p.splits = s;
    p.partial_bytes = s > 1 ? static_cast<size_t>(p.max_tiles) * s * na * kBM * bt * sizeof(float) : 0;
    return p;
}

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct Layout {
    int bt;
    GemmPlan g1, g2;
    size_t off_act, off_p1, off_p2, total;
};

Layout make_layout(const moe_weights* w, int rows_alloc, int M, int groups, int sm_count) {
    Layout L;
    const int K = w->K, N = w->N;
    L.bt = pick_bt(M, rows_alloc, groups);
    L.g1 = plan_gemm(L.bt, 2, N / kBM, K, rows_alloc, groups, sm_count);
    const int na2 = (K % 256 == 0) ? 2 : 1;
    L.g2 = plan_gemm(L.bt, na2, K / (na2 * kBM), N, rows_alloc, groups, sm_count);
    size_t off = 2 * kMaxSplitTiles * sizeof(int);           // two counter regions, kept zero
    L.off_act = off;
    off = align256(off + static_cast<size_t>(rows_alloc) * N * 2);
    L.off_p1 = off;
    off = align256(off + L.g1.partial_bytes);
    L.off_p2 = off;
    off = align256(off + L.g2.partial_bytes);
    L.total = off;
    return L;
}

}  // namespace

size_t experts_workspace_bytes(const moe_weights* w, int rows_alloc, int M, const DeviceInfo& dev) {
    return make_layout(w, rows_alloc, M, w->E_local, dev.sm_count).total;
}

cudaError_t launch_experts(const ExpertsProblem& p, void* workspace, size_t /*workspace_bytes*/, int* err,
                           const DeviceInfo& dev, cudaStream_t s) {
    const moe_weights* w = p.w;
    const int K = w->K, N = w->N;
    const int groups = p.offsets != nullptr ? w->E_local : 1;
    const Layout L = make_layout(w, p.rows_alloc, p.M, groups, dev.sm_count);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int* counters1 = reinterpret_cast<int*>(ws);
    int* counters2 = counters1 + kMaxSplitTiles;
    void* act = ws + L.off_act;

    if (w->format != MOE_WEIGHTS_BF16) return cudaErrorNotSupported;

    CUtensorMap tmW1, tmX, tmW2, tmAct;
    const uint64_t E = static_cast<uint64_t>(w->E_local);
    if (!encode_bf16_2d(&tmW1, w->w1, K, E * 2 * N, kBM) ||
        !encode_bf16_2d(&tmX, p.x, K, p.rows_alloc, L.bt) ||
        !encode_bf16_2d(&tmW2, w->w2, N, E * K, kBM) ||
        !encode_bf16_2d(&tmAct, act, N, p.rows_alloc, L.bt))
        return cudaErrorInvalidValue;

    const int grid = dev.sm_count;
    GemmArgs a1{};
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
    a1.counters = counters1;
    a1.max_tiles = L.g1.max_tiles;
    a1.err = err;
    cudaError_t e = launch_bt<2, MODE_SWIGLU, __nv_bfloat16>(L.bt, tmW1, tmX, a1, grid, s);
    if (e != cudaSuccess) return e;

    GemmArgs a2 = a1;
    a2.kr = N;
    a2.rows_per_group = K;
    a2.n_wtiles = L.g2.n_wtiles;
    a2.wtile_rows = L.g2.na * kBM;
    a2.a1_offset = kBM;
    a2.splits = L.g2.splits;
    a2.out_ld = K;
    a2.out = p.y;
    a2.partials = reinterpret_cast<float*>(ws + L.off_p2);
    a2.counters = counters2;
    a2.max_tiles = L.g2.max_tiles;
    if (L.g2.na == 2) {
        if (p.y_dtype == MOE_DTYPE_F32) return launch_bt<2, MODE_PLAIN, float>(L.bt, tmW2, tmAct, a2, grid, s);
        return launch_bt<2, MODE_PLAIN, __nv_bfloat16>(L.bt, tmW2, tmAct, a2, grid, s);
    }
    if (p.y_dtype == MOE_DTYPE_F32) return launch_bt<1, MODE_PLAIN, float>(L.bt, tmW2, tmAct, a2, grid, s);
    return launch_bt<1, MODE_PLAIN, __nv_bfloat16>(L.bt, tmW2, tmAct, a2, grid, s);
}

}  // namespace moe
