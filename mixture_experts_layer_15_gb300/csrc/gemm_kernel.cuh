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
// over weight rows and its N dimension (up to BT = 16..256) over token rows.
// Decode batches (a few tokens per expert) then stream the weights at full MMA
// width instead of padding tokens up to 128; the MMA N of each tile is cut to
// the tile's row count rounded up to 16, so a partial token tile does not pay
// for the rows it does not have. A work unit is
//     (group g, weight tile wt, token tile tt, k-split s)
// and covers two 128-row A tiles (GEMM1: the gate rows n0..n0+127 and the
// matching up rows N+n0..; GEMM2: output rows k0..k0+255) against one token
// tile, i.e. two accumulators of 128 x BT fp32 in TMEM; the GEMM1 epilogue
// therefore sees gate and up of the same output column in the same thread and
// applies silu(gate)*up with no second pass.
//
// CTA warps, persistent (one CTA per SM):
//   warp 0     TMA producer: A, B tiles of 64 reduction elements into a
//              shared-memory ring (full/empty mbarriers);
//   warps 1..NA TMEM allocation (warp 1) and the MMA issuers, one thread per
//              A tile of the unit, each committing free ring slots and
//              finished accumulators (the barriers count every issuer);
//   epilogue   8 warps (bf16 weights) or 4 (MXFP4): tcgen05.ld of the
//              accumulators (warp w reads TMEM lanes 32*(w%4)..; with 8 warps
//              the two warps of a lane quarter take alternate 16-column
//              chunks), activation, masked stores by row;
//   converters 8 warps (MXFP4 weights only): decode the packed e2m1 codes
//              and their E8M0 scales (flashinfer_moe_ep.py, _E2M1_LUT and
//              _dequant_fp4_ue8m0_gran32) to bf16 in the 128-byte-swizzled
//              layout the MMA reads, two threads per weight row.
// Accumulators are double-buffered in TMEM when 2 x (2 x BT) <= 512 columns,
// so the epilogue of one unit overlaps the mainloop of the next.
//
// MXFP4: the TMA ring carries the packed A tiles (128 rows x 32 bytes per 64
// elements), the matching scale tiles (128 rows x 16 bytes = 8 k-blocks of
// scales, re-read per k-block from L2) and the B tile; a second, shallower
// ring holds the decoded bf16 A tiles. Decoding: two byte-permute lookups turn
// four 3-bit magnitudes into the bf16 bit patterns of {0, .5, 1, 1.5, 2, 3, 4,
// 6}, the sign bits are moved into place, and one bf16x2 multiply by the
// power-of-two scale applies 2^(s-127) (exact for normal results).
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
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace gemm {

using namespace ptx;

constexpr int kBM = 128;                  // weight rows per A tile (MMA M)
constexpr int kBK = 64;                   // reduction elements per ring stage (128 B of bf16)
// Warp budget per CTA: bf16 weights use 8 epilogue warps; MXFP4 weights use
// 4 epilogue warps and 8 converter warps (the decode is the heavier job).
template <bool MX> struct Warps {
    static constexpr int EPI = MX ? 4 : 8;
    static constexpr int EPI_THREADS = 32 * EPI;
    static constexpr int CONV_THREADS = MX ? 256 : 0;
};
constexpr int kMaxGroups = 1024;
constexpr int kSmemBudget = 220 * 1024;
constexpr int kMaxSplitTiles = 16384;     // capacity of one counter region
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// MODE_FINAL: GEMM2 with the finalize folded into its epilogue: every
// accumulator value y of permuted row p is added as rsf * w[e] * y into
// out[e / top_k] (e = permuted_to_expanded[p]) with f32 reductions; nothing
// else is stored, and a split-K split reduces its own partial directly.
enum { MODE_SWIGLU = 0, MODE_PLAIN = 1, MODE_FINAL = 2 };

struct GemmArgs {
    const int32_t* offsets;   // [groups+1] or nullptr
    // BatchedExperts layout (non-fused one-CTA launches): group g's rows are
    // g*batch_stride .. + counts[g] - 1 (counts on the device), instead of offsets
    const int32_t* counts;
    int batch_stride;
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
    // MODE_SWIGLU: the activation (MOE_ACT_SILU / MOE_ACT_GELU) and the clamp
    // (<= 0: none) applied to the gate and up values
    int act;
    float clamp;
    // MODE_FINAL only
    const int32_t* inverse;   // permuted_to_expanded [rows]
    const void* fw;           // routing weights [rows] (expanded order)
    int fw_dtype;
    int top_k;
    float rsf;
    // The start of a folded finalize's f32 output, written by this launch
    // (GEMM1 of a finalizing experts call): init_out[i] = init_src[i]
    // (init_src_dtype; the shared expert's output) or 0, for i < init_n (a
    // multiple of 4). Each CTA's epilogue threads write an even share of it
    // before their first accumulator, so it overlaps the mainloop. nullptr:
    // nothing to write.
    float* init_out;
    const void* init_src;
    int init_src_dtype;
    long long init_n;
};

// Arguments of one launch: a single GEMM (nphase = 1), or GEMM1 followed by
// GEMM2 in the same persistent grid (nphase = 2). In the fused form a GEMM2
// unit may only read the act rows of its token tile once every GEMM1 weight
// tile of that token tile has been written: ready[t] counts those tiles,
// consumed[t] counts the GEMM2 units that have loaded the tile; the last one
// returns both to zero, so the counters are zero between calls.
struct KernelArgs {
    GemmArgs g[2];
    int nphase;
    int* ready;                  // [token tiles]
    int* consumed;               // [token tiles]
    int max_token_tiles;
    // fused launches that write a finalize's output start (g[0].init_out):
    // init_done[0] counts the CTAs whose share is written (GEMM2's reductions
    // wait for all of them); init_done[1] counts the CTAs that have finished,
    // and the last one returns both to zero
    int* init_done;
};

template <int BT, int NA, bool MX>
struct Cfg {
    // warp 0 producer, warps 1..NA one MMA issuer per A tile, then the epilogue
    // (and converter) warps
    static constexpr int ISSUERS = NA;
    static constexpr int EPI_WARP0 = 1 + NA;
    static constexpr int THREADS = 32 * EPI_WARP0 + Warps<MX>::EPI_THREADS + Warps<MX>::CONV_THREADS;
    static constexpr int A_BYTES = kBM * kBK * 2;                 // bf16 A tile (TMA'd or decoded)
    static constexpr int RAW_BYTES = kBM * kBK / 2;               // packed e2m1 A tile
    static constexpr int SC_BYTES = kBM * 16;                     // scale tile: 8 k-blocks of scales
    static constexpr int B_BYTES = BT * kBK * 2;
    // ring stage: [A x NA | B] (bf16) or [raw x NA | scales x NA | B] (MXFP4)
    static constexpr int B_OFF = MX ? NA * (RAW_BYTES + SC_BYTES) : NA * A_BYTES;
    static constexpr int STAGE_BYTES = B_OFF + B_BYTES;
    static constexpr int DSTAGES = MX ? (BT >= 128 ? 2 : 3) : 0;  // decoded-A ring (MXFP4)
    static constexpr int DSTAGE_BYTES = NA * A_BYTES;
    static constexpr int STAGES_FIT = (kSmemBudget - 20 * 1024 - DSTAGES * DSTAGE_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int ACC_COLS = NA * BT;
    static constexpr int NBUF = (2 * ACC_COLS <= 512) ? 2 : 1;
    static constexpr int TMEM_NEED = NBUF * ACC_COLS;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64
                                   : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
    // shared memory layout (offsets from the 1024-aligned base)
    static constexpr int OFF_DEC = STAGES * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_DEC + DSTAGES * DSTAGE_BYTES;
    // full[S], empty[S], dfull[DS], dempty[DS], tfull[2], tempty[2], drain
    static constexpr int NUM_BARS = 2 * STAGES + 2 * DSTAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;       // tmem base, abort, last flag
    static constexpr int OFF_PREFIX = OFF_MISC + 16;              // [2][kMaxGroups+1] units per phase
    static constexpr int OFF_TTP = OFF_PREFIX + 2 * (kMaxGroups + 1) * 4;  // [kMaxGroups+1] token tiles
    static constexpr int OFF_OFFS = OFF_TTP + (kMaxGroups + 1) * 4;      // [kMaxGroups+1]
    static constexpr int OFF_TMP = OFF_OFFS + (kMaxGroups + 1) * 4;      // [33]
    static constexpr int OFF_ROUTE = OFF_TMP + 36 * 4;                   // MODE_FINAL: [BT] token, [BT] scale
    static constexpr int SMEM_BYTES = OFF_ROUTE + 2 * BT * 4 + 1024;    // + alignment slack
    static_assert(STAGES >= 2, "ring too shallow");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(BT % 16 == 0 && BT >= 16 && BT <= 256, "MMA N");
    static_assert(B_OFF % 1024 == 0 && STAGE_BYTES % 1024 == 0, "128B-swizzled tiles need 1024-byte alignment");
};

struct Unit {
    int g, wt, s, row0, row_end, kb0, kb1, tile, ncols;
};

// Group g's rows are [offs[g], ends[g]) (ends = offs + 1 for packed groups).
__device__ __forceinline__ Unit decode_unit(int u, const int* prefix, const int* offs, const int* ends, int BT,
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
    const int beg = offs[lo], end = ends[lo];
    const int ntt = (end - beg + BT - 1) / BT;
    const int tt = local % ntt;
    un.wt = local / ntt;
    un.row0 = beg + tt * BT;
    un.row_end = min(end, a.rows_alloc);
    const int rows = min(BT, un.row_end - un.row0);
    un.ncols = (rows + 15) & ~15;              // MMA N of this tile: its rows rounded up to 16
    if (un.ncols < 16) un.ncols = 16;
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

// Bounded wait until *p >= target (acquire, gpu scope). Same give-up rules as
// wait_bar (limit_ns: the time limit).
__device__ __forceinline__ bool wait_counter(const int* p, int target, volatile int* abort_flag, int* err,
                                             uint64_t limit_ns = kWaitLimitNs) {
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 0;; ++i) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if ((i & 15u) == 15u) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > limit_ns) {
                set_error(err, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// GEMM1's activation on a (gate, up) pair: silu_and_mul or gelu_and_mul (exact
// GELU, g/2 * (1 + erf(g / sqrt 2))), after the optional clamp: the gate to at
// most c, up to [-c, c]. Callers branch on act_is_plain() outside their
// unrolled loops, so that the plain SiLU loop holds no erf (a branch inside
// the loop is turned into selects that evaluate both activations).
__device__ __forceinline__ bool act_is_plain(int act, float clamp) { return act == MOE_ACT_SILU && !(clamp > 0.0f); }
__device__ __forceinline__ float act_mul(float g, float u, int act, float clamp) {
    if (clamp > 0.0f) {
        g = fminf(g, clamp);
        u = fminf(fmaxf(u, -clamp), clamp);
    }
    if (act == MOE_ACT_GELU) return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f)) * u;
    return silu_mul(g, u);
}

template <typename OutT>
__device__ __forceinline__ void store_out(OutT* p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16>(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
}

// This CTA's share of a folded finalize's output start (GemmArgs::init_out):
// 16-byte vectors, thread t of nthreads.
__device__ __forceinline__ void init_out_share(const GemmArgs& a, int cta, int nctas, int t, int nthreads) {
    const long long n4 = a.init_n >> 2;
    const long long per = (n4 + nctas - 1) / nctas;
    const long long b = per * cta;
    const long long e = b + per < n4 ? b + per : n4;
    float4* o = reinterpret_cast<float4*>(a.init_out);
    for (long long i = b + t; i < e; i += nthreads) {
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (a.init_src != nullptr) {
            if (a.init_src_dtype == MOE_DTYPE_F32) {
                v = __ldg(reinterpret_cast<const float4*>(a.init_src) + i);
            } else {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(a.init_src) + i);
                const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
                const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
                v = make_float4(lo.x, lo.y, hi.x, hi.y);
            }
        }
        o[i] = v;
    }
}

// Epilogue of 16 token columns [c0, c0+16) for this thread's weight row.
template <int NA, int MODE, typename OutT>
__device__ __forceinline__ void emit16(const Unit& un, const GemmArgs& a, int row_in_tile, int c0,
                                       const float (&v0)[16], const float (&v1)[16]) {
    OutT* out = static_cast<OutT*>(a.out);
    if (MODE == MODE_SWIGLU && !act_is_plain(a.act, a.clamp)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = un.row0 + c0 + i;
            if (r < un.row_end)
                store_out<OutT>(out + static_cast<size_t>(r) * a.out_ld + un.wt * kBM + row_in_tile,
                                act_mul(v0[i], v1[i], a.act, a.clamp));
        }
        return;
    }
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

// The routing of a unit's token columns, loaded into shared memory by the
// epilogue threads before they wait for the accumulator (so the loads overlap
// the unit's mainloop): tok[c] = token of column c (-1: none), scl[c] =
// rsf * routing weight.
__device__ __forceinline__ void load_route_table(const Unit& un, const GemmArgs& a, int etid, int nthreads,
                                                 int* tok, float* scl) {
    for (int c = etid; c < un.ncols; c += nthreads) {
        const int r = un.row0 + c;
        int t = -1;
        float sc = 0.0f;
        if (r < un.row_end) {
            const int e = __ldg(a.inverse + r);
            if (e < 0 || e >= a.rows_alloc) {
                set_error(a.err, MOE_ERR_DEVICE_INDEX);
            } else {
                t = e / a.top_k;
                sc = a.rsf * load_as_f32(a.fw, static_cast<size_t>(e), a.fw_dtype);
            }
        }
        tok[c] = t;
        scl[c] = sc;
    }
}

// MODE_FINAL epilogue of 16 token columns [c0, c0+16): every lane adds its
// weight row's values, times the column's scaled weight, into the tokens'
// output rows. The 32 lanes of a warp hold 32 consecutive weight rows, so
// each reduction instruction covers 128 contiguous bytes of one output row.
template <int NA>
__device__ __forceinline__ void emit16_final(const Unit& un, const GemmArgs& a, int row_in_tile, int c0,
                                             const int* tok, const float* scl,
                                             const float (&v0)[16], const float (&v1)[16]) {
    float* out = static_cast<float*>(a.out);
    const int col = un.wt * a.wtile_rows + row_in_tile;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int t = tok[c0 + i];                   // same address in every lane: a broadcast
        if (t >= 0) {
            const float si = scl[c0 + i];
            float* o = out + static_cast<size_t>(t) * a.out_ld + col;
            atomicAdd(o, si * v0[i]);
            if (NA == 2) atomicAdd(o + kBM, si * v1[i]);
        }
    }
}

// ---- MXFP4 decode -------------------------------------------------------------------
// Eight e2m1 codes (one 32-bit word, element 2j in the low nibble of byte j)
// -> eight bf16 values times 2^(scale-127), as four bf16x2 words.
// Byte tables indexed by the 3-bit magnitude code: high and low bytes of the
// bf16 encodings of 0, 0.5, 1, 1.5, 2, 3, 4, 6.
constexpr uint32_t kE2m1HiLo = 0x3F3F3F00u, kE2m1HiHi = 0x40404040u;
constexpr uint32_t kE2m1LoLo = 0xC0800000u, kE2m1LoHi = 0xC0804000u;

__device__ __forceinline__ void decode8(uint32_t w, uint32_t scale2, uint32_t (&o)[4]) {
    const uint32_t sel_a = w & 0x7777u;                 // magnitudes of elements 0..3
    const uint32_t sel_b = (w >> 16) & 0x7777u;         // magnitudes of elements 4..7
    const uint32_t hi_a = __byte_perm(kE2m1HiLo, kE2m1HiHi, sel_a);
    const uint32_t lo_a = __byte_perm(kE2m1LoLo, kE2m1LoHi, sel_a);
    const uint32_t hi_b = __byte_perm(kE2m1HiLo, kE2m1HiHi, sel_b);
    const uint32_t lo_b = __byte_perm(kE2m1LoLo, kE2m1LoHi, sel_b);
    // Signs: byte j of w holds elements 2j (low nibble, sign bit 3) and 2j+1
    // (high nibble, sign bit 7); in w4 = w << 4 byte j's top bit is element
    // 2j's sign. A byte permute in sign-replicate mode (selector bit 3) copies
    // a byte's top bit over the whole output byte: bytes 1 and 3 of sgn_j get
    // the signs of elements 2j and 2j+1, which the mask 0x80008000 keeps as
    // bits 15 and 31 of the bf16 pair.
    const uint32_t w4 = w << 4;
    uint32_t mag[4];
    mag[0] = __byte_perm(lo_a, hi_a, 0x5140);
    mag[1] = __byte_perm(lo_a, hi_a, 0x7362);
    mag[2] = __byte_perm(lo_b, hi_b, 0x5140);
    mag[3] = __byte_perm(lo_b, hi_b, 0x7362);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // output byte 1 <- replicate(top bit of w4.byte j), byte 3 <- replicate(top bit of w.byte j)
        uint32_t sgn;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(sgn) : "r"(w), "r"(w4), "r"(((0x8u | j) << 12) | ((0x8u | (4 + j)) << 4)));
        o[j] = mag[j] | (sgn & 0x80008000u);
    }
    const __nv_bfloat162 s = *reinterpret_cast<const __nv_bfloat162*>(&scale2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&o[i]);
        v = __hmul2(v, s);
        o[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

// Half a weight row of one k-block: 16 packed bytes (32 codes) + their scale
// byte -> 32 bf16, written into the 128-byte-swizzled K-major tile (row r,
// 16-byte chunk c at chunk position c ^ (r & 7); the tile base is 1024-byte
// aligned). Half h covers chunks 4h .. 4h+3.
__device__ __forceinline__ void decode_half(const uint8_t* raw, uint32_t sc, uint8_t* dec_tile, int r, int h) {
    const uint4 p = *reinterpret_cast<const uint4*>(raw);
    const uint32_t words[4] = {p.x, p.y, p.z, p.w};
    // bf16 2^(s-127) has exponent field s and a zero mantissa: bits s << 7
    const uint32_t s2 = (sc << 7) | (sc << 23);
    uint8_t* row = dec_tile + r * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = 4 * h + j;
        uint32_t o[4];
        decode8(words[j], s2, o);
        *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// MODE/OutT describe phase 0 of a single-GEMM launch. A fused launch
// (FUSED = true, NA = 2) runs GEMM1 (silu_and_mul, bf16 act) as phase 0 and
// GEMM2 (plain, OutT) as phase 1.
template <int BT, int NA, int MODE, typename OutT, bool MX, bool FUSED>
__global__ void __launch_bounds__(Cfg<BT, NA, MX>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmS0,
                    const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmS1, const __grid_constant__ CUtensorMap tmB1,
                    const KernelArgs ka) {
    using C = Cfg<BT, NA, MX>;
    static_assert(!FUSED || NA == 2, "fused launches use two A tiles per unit");
    constexpr int kEpiWarps = Warps<MX>::EPI;
    constexpr int kEpiThreads = Warps<MX>::EPI_THREADS;
    constexpr int kConvThreads = Warps<MX>::CONV_THREADS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
    auto dfull_bar = [&](int d) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + d); };
    auto dempty_bar = [&](int d) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + C::DSTAGES + d); };
    auto tfull_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2 * C::DSTAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2 * C::DSTAGES + 2 + b); };
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2 * C::DSTAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
    int* prefix0 = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    int* prefix1 = prefix0 + (kMaxGroups + 1);
    int* ttp = reinterpret_cast<int*>(smem + C::OFF_TTP);
    int* offs = reinterpret_cast<int*>(smem + C::OFF_OFFS);
    int* tmp = reinterpret_cast<int*>(smem + C::OFF_TMP);
    int* route_tok = reinterpret_cast<int*>(smem + C::OFF_ROUTE);
    float* route_scl = reinterpret_cast<float*>(smem + C::OFF_ROUTE + 4 * BT);
    const GemmArgs& a0 = ka.g[0];
    const int groups = a0.groups;

    // ---- prologue: barriers, TMEM, unit schedule ----
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            // MXFP4: the converters release the packed tile, the MMA the B tile
            // MXFP4: one arrival per converter warp frees the packed tile, the MMA the B tile
            mbar_init(empty_bar(s), MX ? C::ISSUERS + kConvThreads / 32 : C::ISSUERS);
        }
        for (int d = 0; d < C::DSTAGES; ++d) {
            mbar_init(dfull_bar(d), kConvThreads / 32);
            mbar_init(dempty_bar(d), C::ISSUERS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), C::ISSUERS);
            mbar_init(tempty_bar(b), kEpiThreads);
        }
        mbar_init(drain_bar, C::ISSUERS);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA0);
        if (MX) prefetch_tensormap(&tmS0);
        prefetch_tensormap(&tmB0);
        if (FUSED) {
            prefetch_tensormap(&tmA1);
            if (MX) prefetch_tensormap(&tmS1);
            prefetch_tensormap(&tmB1);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    // everything above is CTA-local; from here on the kernel reads what the
    // previous kernels of the stream wrote
    pdl_wait();
    pdl_trigger();
    // group offsets (validated: non-decreasing, within the allocation)
    const bool batched = !FUSED && a0.counts != nullptr;
    for (int g = tid; g <= groups; g += C::THREADS) {
        int v = batched ? g * a0.batch_stride
                        : (a0.offsets != nullptr ? __ldg(a0.offsets + g) : (g == 0 ? 0 : a0.single_rows));
        if (v < 0 || v > a0.rows_alloc) { set_error(a0.err, MOE_ERR_DEVICE_INDEX); v = v < 0 ? 0 : a0.rows_alloc; }
        offs[g] = v;
    }
    __syncthreads();
    for (int g = tid; g < groups; g += C::THREADS) {
        int cnt;
        if (batched) {
            // batched rows: the group's count, at most its block (ttp holds the ends)
            cnt = __ldg(a0.counts + g);
            if (cnt < 0 || cnt > a0.batch_stride) {
                set_error(a0.err, MOE_ERR_DEVICE_INDEX);
                cnt = cnt < 0 ? 0 : a0.batch_stride;
            }
            ttp[g] = offs[g] + cnt;
        } else {
            cnt = offs[g + 1] - offs[g];
        }
        if (cnt < 0) { set_error(a0.err, MOE_ERR_DEVICE_INDEX); cnt = 0; }
        const int ntt = (cnt + BT - 1) / BT;
        prefix0[g] = ntt * a0.n_wtiles * a0.splits;
        if (FUSED) {
            prefix1[g] = ntt * ka.g[1].n_wtiles * ka.g[1].splits;
            ttp[g] = ntt;
        }
    }
    __syncthreads();
    const int units0 = block_exclusive_scan(prefix0, groups, tmp);
    int units1 = 0;
    if (FUSED) {
        units1 = block_exclusive_scan(prefix1, groups, tmp);
        const int ntiles = block_exclusive_scan(ttp, groups, tmp);
        if (ntiles > ka.max_token_tiles) {               // cannot happen with the host's sizing
            if (tid == 0) set_error(a0.err, MOE_ERR_DEVICE_INDEX);
            units1 = 0;
        }
    }
    if (tid == 0) { prefix0[groups] = units0; if (FUSED) prefix1[groups] = units1; }
    const int total_units = units0 + units1;
    // make the TMEM address written by tcgen05.alloc visible to all threads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // unit u -> (phase, decoded unit)
    const int* ends = batched ? ttp : offs + 1;
    auto unit_at = [&](int u, int& ph) -> Unit {
        ph = (FUSED && u >= units0) ? 1 : 0;
        return ph ? decode_unit(u - units0, prefix1, offs, ends, BT, ka.g[1])
                  : decode_unit(u, prefix0, offs, ends, BT, a0);
    };
    // global index of a unit's token tile (fused launches)
    auto tile_index = [&](const Unit& un) { return ttp[un.g] + (un.row0 - offs[un.g]) / BT; };

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issued_phase = 0;       // per-stage: load in flight / its phase
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
                int ph;
                const Unit un = unit_at(u, ph);
                const GemmArgs& a = ka.g[ph];
                const CUtensorMap* tA = ph ? &tmA1 : &tmA0;
                const CUtensorMap* tS = ph ? &tmS1 : &tmS0;
                const CUtensorMap* tB = ph ? &tmB1 : &tmB0;
                const int a_row = un.g * a.rows_per_group + un.wt * a.wtile_rows;
                // the weight-side loads of k-block kb into ring slot `stage` (the
                // slot's full barrier is armed for the whole stage, act included)
                auto load_a = [&](int kb) {
                    const uint32_t st = sbase + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), C::STAGE_BYTES);
                    if (MX) {
                        tma_load_2d(st, tA, kb * (kBK / 2), a_row, full_bar(stage));
                        tma_load_2d(st + NA * C::RAW_BYTES, tS, (kb >> 3) * 16, a_row, full_bar(stage));
                        if (NA == 2) {
                            tma_load_2d(st + C::RAW_BYTES, tA, kb * (kBK / 2), a_row + a.a1_offset, full_bar(stage));
                            tma_load_2d(st + NA * C::RAW_BYTES + C::SC_BYTES, tS, (kb >> 3) * 16,
                                        a_row + a.a1_offset, full_bar(stage));
                        }
                    } else {
                        tma_load_2d(st, tA, kb * kBK, a_row, full_bar(stage));
                        if (NA == 2) tma_load_2d(st + C::A_BYTES, tA, kb * kBK, a_row + a.a1_offset, full_bar(stage));
                    }
                };
                int kb_start = un.kb0;
                if (FUSED && ph == 1) {
                    // The act rows of this token tile must be complete before they
                    // are loaded, but the weight tiles do not depend on them: while
                    // the tile is not ready, the weight loads of a long unit's first
                    // k-blocks go out first (up to a ring's worth). Short units are
                    // not started early: fetched whole, they would compete with the
                    // GEMM1 tail that the act is waiting for.
                    const int* rp = ka.ready + tile_index(un);
                    int v;
                    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(rp) : "memory");
                    const int first_stage = stage;
                    int pre = 0;
                    if (v < ka.g[0].n_wtiles && un.kb1 - un.kb0 >= 4 * C::STAGES) {
                        for (int kb = un.kb0; kb < un.kb1 && pre < C::STAGES; ++kb) {
                            if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, a0.err)) { ok = false; break; }
                            load_a(kb);
                            issued |= 1u << stage;
                            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                            if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                            ++pre;
                        }
                    }
                    const bool got = ok && wait_counter(rp, ka.g[0].n_wtiles, abort_flag, a0.err);
                    fence_proxy_async_global();
                    // the act loads of those k-blocks; issued also when the wait gave up,
                    // so that every armed barrier completes before the CTA leaves
                    for (int i = 0, s2 = first_stage; i < pre; ++i) {
                        tma_load_2d(sbase + s2 * C::STAGE_BYTES + C::B_OFF, tB, (un.kb0 + i) * kBK, un.row0,
                                    full_bar(s2));
                        if (++s2 == C::STAGES) s2 = 0;
                    }
                    if (!got) { ok = false; break; }
                    kb_start = un.kb0 + pre;
                }
                for (int kb = kb_start; kb < un.kb1; ++kb) {
                    if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, a0.err)) { ok = false; break; }
                    const uint32_t st = sbase + stage * C::STAGE_BYTES;
                    // packed codes (MXFP4): 32 bytes per row per k-block; scales: the
                    // 16-byte group of 8 k-blocks that holds this one
                    load_a(kb);
                    tma_load_2d(st + C::B_OFF, tB, kb * kBK, un.row0, full_bar(stage));
                    issued |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (FUSED && ph == 1 && ok) {
                    // the last unit to have read this token tile clears its counters
                    const int t = tile_index(un);
                    const int done = atomicAdd(ka.consumed + t, 1) + 1;
                    if (done == ka.g[1].n_wtiles * ka.g[1].splits) {
                        ka.ready[t] = 0;
                        ka.consumed[t] = 0;
                    }
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
    } else if (warp <= C::ISSUERS) {
        // ================= MMA issuers: warp 1 + h issues A tile h's MMAs =================
        // (one thread issuing every MMA of a k-block set the pace at mid-size
        // tiles; each issuer commits to the ring, decoded-ring, accumulator and
        // drain barriers, which count every issuer)
        const int h = warp - 1;
        if (lane == 0) {
            int stage = 0, dstage = 0;
            uint32_t phase = 0, dphase = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x, ++it) {
                int ph;
                const Unit un = unit_at(u, ph);
                const uint32_t idesc = idesc_bf16_f32(kBM, un.ncols);
                const int buf = C::NBUF == 2 ? (it & 1) : 0;
                const uint32_t use = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
                if (!wait_bar(tempty_bar(buf), use ^ 1u, abort_flag, a0.err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + buf * C::ACC_COLS + h * BT;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(full_bar(stage), phase, abort_flag, a0.err)) { ok = false; break; }
                    if (MX && !wait_bar(dfull_bar(dstage), dphase, abort_flag, a0.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t st = sbase + stage * C::STAGE_BYTES;
                    const uint32_t sA0 = MX ? sbase + C::OFF_DEC + dstage * C::DSTAGE_BYTES : st;
                    const uint32_t sB = st + C::B_OFF;
                    // step kk starts 32 bytes further into each 128-byte row: +2 in the
                    // descriptors' 16-byte address field (tiles are 1024-byte aligned)
                    const uint64_t dA = sw128_kmajor_desc(sA0 + h * C::A_BYTES), dB = sw128_kmajor_desc(sB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t acc = (kb > un.kb0 || kk > 0) ? 1u : 0u;
                        mma_f16(d, dA + 2 * kk, dB + 2 * kk, idesc, acc);
                    }
                    mma_commit(empty_bar(stage));            // ring slot free once these MMAs finish
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                    if (MX) {
                        mma_commit(dempty_bar(dstage));      // decoded tile free likewise
                        if (++dstage == C::DSTAGES) { dstage = 0; dphase ^= 1u; }
                    }
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
    } else if (warp < C::EPI_WARP0 + kEpiWarps) {
        // ================= epilogue (the warps after the issuers) =================
        const int q = warp & 3;                              // TMEM lanes 32q..32q+31
        const int row_in_tile = q * 32 + lane;
        const int etid = tid - 32 * C::EPI_WARP0;
        const int c_first = 16 * ((warp - C::EPI_WARP0) >> 2);   // this warp's first 16-column chunk
        constexpr int c_step = 16 * (kEpiWarps / 4);
        // one unit's outputs from the accumulator values v0/v1 of columns [c0, c0+16)
        auto emit = [&](int ph, const Unit& un, const GemmArgs& a, int c0, const float (&v0)[16],
                        const float (&v1)[16]) {
            if (FUSED && ph == 0) {
                emit16<2, MODE_SWIGLU, __nv_bfloat16>(un, a, row_in_tile, c0, v0, v1);
            } else if (MODE == MODE_FINAL) {
                emit16_final<NA>(un, a, row_in_tile, c0, route_tok, route_scl, v0, v1);
            } else {
                emit16<NA, (FUSED ? MODE_PLAIN : MODE), OutT>(un, a, row_in_tile, c0, v0, v1);
            }
        };
        // fused launches: after the stores of a finished GEMM1 tile, count it
        auto signal_ready = [&](int ph, const Unit& un) {
            if (!FUSED || ph != 0) return;
            fence_proxy_async_global();                      // act stores -> later TMA reads
            __threadfence();
            named_bar_sync(1, kEpiThreads);
            if (etid == 0) atomicAdd(ka.ready + tile_index(un), 1);
        };
        // a finalizing call's output start (GEMM1's launch writes it): this
        // CTA's share first; in a fused launch GEMM2's reductions may only
        // start once every CTA's share is written
        const bool init = a0.init_out != nullptr;
        if (init) {
            init_out_share(a0, blockIdx.x, gridDim.x, etid, kEpiThreads);
            if (FUSED) {
                __threadfence();
                named_bar_sync(1, kEpiThreads);
                if (etid == 0) atomicAdd(ka.init_done, 1);
            }
        }
        bool init_seen = !(FUSED && MODE == MODE_FINAL && init);
        int it = 0;
        for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++it) {
            int ph;
            const Unit un = unit_at(u, ph);
            const GemmArgs& a = ka.g[ph];
            const int buf = C::NBUF == 2 ? (it & 1) : 0;
            const uint32_t use = C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1);
            if (MODE == MODE_FINAL && (!FUSED || ph == 1)) {
                named_bar_sync(1, kEpiThreads);              // the previous unit is done with the table
                if (!init_seen) {
                    // every other thread passes the barrier after the accumulator
                    // wait below only once this wait is over
                    if (etid == 0) wait_counter(ka.init_done, static_cast<int>(gridDim.x), abort_flag, a0.err);
                    init_seen = true;
                }
                load_route_table(un, a, etid, kEpiThreads, route_tok, route_scl);
            }
            wait_bar(tfull_bar(buf), use, abort_flag, a0.err);
            // all threads decide together (and the route table is visible)
            if (named_bar_or(1, kEpiThreads, *abort_flag != 0)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_COLS;
            // a finalizing phase reduces every split's partial into out directly
            const bool direct = a.splits == 1 || (MODE == MODE_FINAL && (!FUSED || ph == 1));
            if (direct) {
#pragma unroll 1
                for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
                    float v0[16], v1[16];
                    if (NA == 2) tmem_ld16x2(tb + c0, tb + BT + c0, v0, v1);
                    else tmem_ld16(tb + c0, v0);
                    emit(ph, un, a, c0, v0, v1);
                }
                tc_fence_before();
                mbar_arrive(tempty_bar(buf));
                signal_ready(ph, un);
            } else {
                const size_t slot = static_cast<size_t>(NA) * kBM * BT;
                const bool tile_ok = un.tile < a.max_tiles;
                float* part = a.partials + (static_cast<size_t>(un.tile) * a.splits + un.s) * slot;
#pragma unroll 1
                for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
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
                        set_error(a0.err, MOE_ERR_DEVICE_INDEX);
                    }
                    *last_flag = last;
                }
                named_bar_sync(1, kEpiThreads);
                const int last = *last_flag;
                if (last) {
                    __threadfence();
                    const float* p0 = a.partials + static_cast<size_t>(un.tile) * a.splits * slot;
#pragma unroll 1
                    for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
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
                        emit(ph, un, a, c0, v0, v1);
                    }
                    signal_ready(ph, un);
                }
                named_bar_sync(1, kEpiThreads);              // last_flag is reused by the next unit
            }
        }
    } else if (MX) {
        // ================= converters (MXFP4 only: the warps after the epilogue) =================
        // two threads per weight row: h = 0 decodes elements 0..31 of the
        // k-block, h = 1 elements 32..63, each with its own scale byte
        const int ct = tid - 32 * C::EPI_WARP0 - kEpiThreads;
        const int r = ct >> 1, h = ct & 1;
        int stage = 0, dstage = 0;
        uint32_t phase = 0, dphase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            int ph;
            const Unit un = unit_at(u, ph);
            for (int kb = un.kb0; kb < un.kb1; ++kb) {
                if (!wait_bar(full_bar(stage), phase, abort_flag, a0.err)) { ok = false; break; }
                if (!wait_bar(dempty_bar(dstage), dphase ^ 1u, abort_flag, a0.err)) { ok = false; break; }
                const uint8_t* st = smem + stage * C::STAGE_BYTES;
                uint8_t* dec = smem + C::OFF_DEC + dstage * C::DSTAGE_BYTES;
                const int sb = 2 * (kb & 7) + h;             // this half's scale byte
#pragma unroll
                for (int t = 0; t < NA; ++t) {
                    const uint8_t sc = st[NA * C::RAW_BYTES + t * C::SC_BYTES + r * 16 + sb];
                    decode_half(st + t * C::RAW_BYTES + r * 32 + h * 16, sc, dec + t * C::A_BYTES, r, h);
                }
                // generic-proxy shared-memory writes -> visible to the MMA (async
                // proxy); then one arrival per warp, after all its lanes' writes
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if ((tid & 31) == 0) {
                    mbar_arrive(empty_bar(stage));
                    mbar_arrive(dfull_bar(dstage));
                }
                if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                if (++dstage == C::DSTAGES) { dstage = 0; dphase ^= 1u; }
            }
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
    if (FUSED && tid == 0 && a0.init_out != nullptr) {
        // the last CTA to finish returns the output-start counters to zero
        if (atomicAdd(ka.init_done + 1, 1) == static_cast<int>(gridDim.x) - 1) {
            ka.init_done[0] = 0;
            ka.init_done[1] = 0;
        }
    }
}

// ---- launching one instantiation ------------------------------------------------------
struct Maps {
    CUtensorMap A[2], S[2], B[2];
};

template <int BT, int NA, int MODE, typename OutT, bool MX, bool FUSED>
cudaError_t launch_kernel(const Maps& m, const KernelArgs& ka, int grid, cudaStream_t s) {
    using C = Cfg<BT, NA, MX>;
    auto kern = grouped_gemm_kernel<BT, NA, MODE, OutT, MX, FUSED>;
    static std::atomic<uint64_t> configured{0};      // bit per device ordinal
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    if (!FUSED)
        return launch_pdl(kern, dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, s, m.A[0], m.S[0], m.B[0], m.A[0],
                          m.S[0], m.B[0], ka);
    // the CTAs of a fused launch wait on one another: all of them must be
    // resident at once, which a cooperative launch guarantees
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, m.A[0], m.S[0], m.B[0], m.A[1], m.S[1], m.B[1], ka);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cfg.numAttrs = 1;                            // cooperative only
        e = cudaLaunchKernelEx(&cfg, kern, m.A[0], m.S[0], m.B[0], m.A[1], m.S[1], m.B[1], ka);
    }
    return e;
}

template <int NA, int MODE, typename OutT, bool MX, bool FUSED>
cudaError_t launch_bt(int bt, const Maps& m, const KernelArgs& ka, int grid, cudaStream_t s) {
    switch (bt) {
        case 16: return launch_kernel<16, NA, MODE, OutT, MX, FUSED>(m, ka, grid, s);
        case 32: return launch_kernel<32, NA, MODE, OutT, MX, FUSED>(m, ka, grid, s);
        case 64: return launch_kernel<64, NA, MODE, OutT, MX, FUSED>(m, ka, grid, s);
        case 128: return launch_kernel<128, NA, MODE, OutT, MX, FUSED>(m, ka, grid, s);
        default: return launch_kernel<256, NA, MODE, OutT, MX, FUSED>(m, ka, grid, s);
    }
}

// A single GEMM (fused = 0; mode 0 = GEMM1, 1 = GEMM2 with na tiles per unit)
// or GEMM1 -> GEMM2 fused (fused = 1), of one weight format.
// GEMM2 with the finalize in its epilogue (MODE_FINAL, f32 out): alone with
// na tiles per unit, or as phase 1 of a fused launch (fused = 1, na = 2).
template <bool MX>
cudaError_t launch_gemm_final(int fused, int bt, int na, const Maps& m, const KernelArgs& ka, int grid,
                              cudaStream_t s) {
    if (fused) return launch_bt<2, MODE_FINAL, float, MX, true>(bt, m, ka, grid, s);
    if (na == 2) return launch_bt<2, MODE_FINAL, float, MX, false>(bt, m, ka, grid, s);
    return launch_bt<1, MODE_FINAL, float, MX, false>(bt, m, ka, grid, s);
}

template <bool MX>
cudaError_t launch_gemm(int fused, int mode, int bt, int na, int out_dtype, const Maps& m, const KernelArgs& ka,
                        int grid, cudaStream_t s) {
    if (fused) {
        if (out_dtype == MOE_DTYPE_F32) return launch_bt<2, MODE_PLAIN, float, MX, true>(bt, m, ka, grid, s);
        return launch_bt<2, MODE_PLAIN, __nv_bfloat16, MX, true>(bt, m, ka, grid, s);
    }
    if (mode == MODE_SWIGLU) return launch_bt<2, MODE_SWIGLU, __nv_bfloat16, MX, false>(bt, m, ka, grid, s);
    if (na == 2) {
        if (out_dtype == MOE_DTYPE_F32) return launch_bt<2, MODE_PLAIN, float, MX, false>(bt, m, ka, grid, s);
        return launch_bt<2, MODE_PLAIN, __nv_bfloat16, MX, false>(bt, m, ka, grid, s);
    }
    if (out_dtype == MOE_DTYPE_F32) return launch_bt<1, MODE_PLAIN, float, MX, false>(bt, m, ka, grid, s);
    return launch_bt<1, MODE_PLAIN, __nv_bfloat16, MX, false>(bt, m, ka, grid, s);
}

// Defined in gemm_bf16.cu and gemm_mxfp4.cu (one translation unit per weight format).
cudaError_t launch_gemm_bf16(int fused, int mode, int bt, int na, int out_dtype, const Maps& m,
                             const KernelArgs& ka, int grid, cudaStream_t s);
cudaError_t launch_gemm_mxfp4(int fused, int mode, int bt, int na, int out_dtype, const Maps& m,
                              const KernelArgs& ka, int grid, cudaStream_t s);
// Defined in gemm_final_bf16.cu and gemm_final_mxfp4.cu.
cudaError_t launch_gemm_final_bf16(int fused, int bt, int na, const Maps& m, const KernelArgs& ka, int grid,
                                   cudaStream_t s);
cudaError_t launch_gemm_final_mxfp4(int fused, int bt, int na, const Maps& m, const KernelArgs& ka, int grid,
                                    cudaStream_t s);

}  // namespace gemm
}  // namespace moe
