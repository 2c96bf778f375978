// Grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2), bf16 weights.
//
// Same math and unit list as gemm_kernel.cuh (one launch per GEMM here), with
// the MMA spread over the two SMs of a cluster: M = 256 weight rows, 128 from
// each CTA's shared memory, against up to BT = 256 tokens, whose rows are
// split in halves between the two CTAs. One thread of the even CTA issues
// the MMAs; each CTA's TMEM receives its own 128 rows for all token columns.
//
// Why: with one CTA, a 128-row MMA re-reads its whole token tile from shared
// memory for every A tile, and the TMA writes of both operands come on top;
// the shared-memory traffic per FLOP then caps the tensor pipe (measured ~74 %
// busy at 256-token tiles, ~44 % at 128). On a pair each SM reads its own A
// rows and half of B per MMA, and loads half of B, which halves the traffic
// per FLOP, and one accumulator per unit (BT columns) leaves TMEM
// double-buffered even at BT = 256.
//
// A rows per CTA (rank r of the pair):
//   GEMM1 (SwiGLU): gate rows n0 + 64r .. +63 then up rows N + n0 + 64r .. +63
//                   (two 64-row TMA boxes), so a CTA holds gate and up of the
//                   same 64 act columns: TMEM lanes 0..63 gate, 64..127 up;
//   GEMM2:          output rows k0 + 128r .. +127.
// B rows per CTA: token rows row0 + r * ncols/2 .. (the MMA reads ncols/2).
//
// Pipeline: each CTA's producer loads its own halves into its own ring slot
// and signals the EVEN CTA's full barrier (cta_group::2 TMA); only the even
// CTA expects the transaction bytes (both halves). The MMA commit arrives on
// the empty barriers (and accumulator-full barriers) of both CTAs at once
// (multicast). Each CTA's epilogue drains its own TMEM and then arrives on the
// even CTA's accumulator-empty barrier. All waits are bounded as in the
// one-CTA kernel; both CTAs allocate and free TMEM together (one warp each).
//
// SwiGLU epilogue: a TMEM lane quarter is readable only by warps w with
// w % 4 == quarter, so the up values (lanes 64..127) reach the gate warps
// (lanes 0..63) through a small shared-memory exchange per 16 columns.
#pragma once

#include "gemm_kernel.cuh"

namespace moe {
namespace gemm {

template <int BT>
struct PairCfg {
    static constexpr int EPI_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int A_BYTES = kBM * kBK * 2;                  // this CTA's 128 A rows
    static constexpr int B_BYTES = (BT / 2) * kBK * 2;             // this CTA's half of the token tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int XCHG_BYTES = 2 * 16 * 64 * 4;             // two column groups x [16][64] floats
    static constexpr int STAGES_FIT = (kSmemBudget - 20 * 1024 - XCHG_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int ACC_COLS = BT;
    static constexpr int TMEM_COLS = 2 * BT;                       // double-buffered accumulator
    static constexpr int OFF_XCHG = STAGES * STAGE_BYTES;
    static constexpr int OFF_BAR = OFF_XCHG + XCHG_BYTES;
    // full[S], empty[S], tfull[2], tempty[2], drain
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_PREFIX = OFF_MISC + 16;
    static constexpr int OFF_OFFS = OFF_PREFIX + (kMaxGroups + 1) * 4;
    static constexpr int OFF_TMP = OFF_OFFS + (kMaxGroups + 1) * 4;
    static constexpr int OFF_ROUTE = OFF_TMP + 36 * 4;
    static constexpr int SMEM_BYTES = OFF_ROUTE + 2 * BT * 4 + 1024;
    static_assert(BT == 128 || BT == 256, "pair tiles are 128 or 256 tokens");
    static_assert(STAGES >= 3, "ring too shallow");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
    static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "128B-swizzled tiles need 1024-byte alignment");
    static_assert(TMEM_COLS <= 512, "TMEM");
};

// MMA N of a pair unit: the tile's rows rounded up to 16, at least 32, so each
// CTA's half is a whole number of 8-row swizzle atoms.
__device__ __forceinline__ int pair_cols(const Unit& un, int BT) {
    int rows = un.row_end - un.row0;
    if (rows > BT) rows = BT;
    int n = (rows + 15) & ~15;
    return n < 32 ? 32 : n;
}

template <int BT, int MODE, typename OutT>
__global__ void __launch_bounds__(PairCfg<BT>::THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const GemmArgs a) {
    using C = PairCfg<BT>;
    constexpr int kEpiThreads = 32 * C::EPI_WARPS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    // the same offset in both CTAs: the pair MMA reads both at the same address
    uint8_t* smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool even = rank == 0;
    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + b); };
    auto tempty_bar = [&](int b) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2 + b); };
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
    int* prefix = reinterpret_cast<int*>(smem + C::OFF_PREFIX);
    int* offs = reinterpret_cast<int*>(smem + C::OFF_OFFS);
    int* tmp = reinterpret_cast<int*>(smem + C::OFF_TMP);
    int* route_tok = reinterpret_cast<int*>(smem + C::OFF_ROUTE);
    float* route_scl = reinterpret_cast<float*>(smem + C::OFF_ROUTE + 4 * BT);
    float* xchg = reinterpret_cast<float*>(smem + C::OFF_XCHG);
    const int groups = a.groups;

    // ---- prologue: barriers (visible to the peer before any remote signal), TMEM ----
    if (tid == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);          // the even CTA's expect_tx arrival (+ both CTAs' bytes)
            mbar_init(empty_bar(s), 1);         // the pair MMA's multicast commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);         // multicast commit
            mbar_init(tempty_bar(b), 2);        // one arrival from each CTA's epilogue
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    __syncwarp();
    cluster_sync_all();
    pdl_wait();
    pdl_trigger();
    for (int g = tid; g <= groups; g += C::THREADS) {
        int v = a.offsets != nullptr ? __ldg(a.offsets + g) : (g == 0 ? 0 : a.single_rows);
        if (v < 0 || v > a.rows_alloc) { set_error(a.err, MOE_ERR_DEVICE_INDEX); v = v < 0 ? 0 : a.rows_alloc; }
        offs[g] = v;
    }
    __syncthreads();
    for (int g = tid; g < groups; g += C::THREADS) {
        int cnt = offs[g + 1] - offs[g];
        if (cnt < 0) { set_error(a.err, MOE_ERR_DEVICE_INDEX); cnt = 0; }
        prefix[g] = ((cnt + BT - 1) / BT) * a.n_wtiles;           // splits == 1 on pairs
    }
    __syncthreads();
    const int total_units = block_exclusive_scan(prefix, groups, tmp);
    if (tid == 0) prefix[groups] = total_units;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    auto unit_at = [&](int u) {
        Unit un = decode_unit(u, prefix, offs, offs + 1, BT, a);
        un.ncols = pair_cols(un, BT);
        return un;
    };

    if (warp == 0) {
        // ================= TMA producer (both CTAs) =================
        if (lane == 0) {
            const uint32_t full_even0 = mapa_shared(full_bar(0), 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, issued_any = false;
            for (int u = pair; u < total_units && ok; u += npairs) {
                const Unit un = unit_at(u);
                const int brow = un.row0 + static_cast<int>(rank) * (un.ncols / 2);
                const int arow = un.g * a.rows_per_group + un.wt * a.wtile_rows +
                                 static_cast<int>(rank) * (MODE == MODE_SWIGLU ? 64 : kBM);
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(empty_bar(stage), phase ^ 1u, abort_flag, a.err)) { ok = false; break; }
                    const uint32_t st = sbase + stage * C::STAGE_BYTES;
                    if (even) mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
                    const uint32_t fb = full_even0 + 8u * stage;
                    if (MODE == MODE_SWIGLU) {
                        tma_load_2d_pair(st, &tmA, kb * kBK, arow, fb);                       // gate
                        tma_load_2d_pair(st + C::A_BYTES / 2, &tmA, kb * kBK, arow + a.a1_offset, fb);  // up
                    } else {
                        tma_load_2d_pair(st, &tmA, kb * kBK, arow, fb);
                    }
                    tma_load_2d_pair(st + C::A_BYTES, &tmB, kb * kBK, brow, fb);
                    issued_any = true;
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok && issued_any) {
                // the loads signal the even CTA's barriers: give the ones in
                // flight a bounded moment to land before this CTA can go away
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {}
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================= MMA issuer (even CTA) =================
        if (lane == 0 && even) {
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = pair; u < total_units && ok; u += npairs, ++it) {
                const Unit un = unit_at(u);
                const uint32_t idesc = idesc_bf16_f32(2 * kBM, un.ncols);
                const int buf = it & 1;
                const uint32_t use = (it >> 1) & 1;
                if (!wait_bar(tempty_bar(buf), use ^ 1u, abort_flag, a.err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + buf * C::ACC_COLS;
                for (int kb = un.kb0; kb < un.kb1; ++kb) {
                    if (!wait_bar(full_bar(stage), phase, abort_flag, a.err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA = sbase + stage * C::STAGE_BYTES;
                    const uint32_t sB = sA + C::A_BYTES;
                    // step kk: +32 bytes, +2 in the descriptors' 16-byte address field
                    const uint64_t dA = sw128_kmajor_desc(sA), dB = sw128_kmajor_desc(sB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t acc = (kb > un.kb0 || kk > 0) ? 1u : 0u;
                        mma_f16_pair(d, dA + 2 * kk, dB + 2 * kk, idesc, acc);
                    }
                    mma_commit_pair(empty_bar(stage), 0x3);   // both CTAs' ring slots free
                    if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair(tfull_bar(buf), 0x3);         // both CTAs' accumulators ready
            }
            mma_commit_pair(drain_bar, 0x3);                  // every pair MMA done, in both CTAs
        }
        // both CTAs: the even CTA's MMAs write this CTA's TMEM; wait for them
        if (lane == 0) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < kWaitLimitNs) {}
        }
        __syncwarp();
    } else {
        // ================= epilogue (both CTAs, 8 warps) =================
        const int q = warp & 3;                               // TMEM lanes 32q .. 32q+31
        const int etid = tid - 64;
        const int grp = (warp - 2) >> 2;                      // column group: chunks 16*grp, +32, ...
        const int c_first = 16 * grp;
        constexpr int c_step = 32;
        float* xg = xchg + grp * 16 * 64;                     // [16][64]: up values of this group's chunk
        const int l64 = (q & 1) * 32 + lane;                  // lane within the 64 gate (or up) rows
        const uint32_t tempty_even = mapa_shared(tempty_bar(0), 0);
        // a finalizing call's output start (written by its GEMM1 launch)
        if (a.init_out != nullptr) init_out_share(a, blockIdx.x, gridDim.x, etid, kEpiThreads);
        int it = 0;
        for (int u = pair; u < total_units; u += npairs, ++it) {
            const Unit un = unit_at(u);
            const int buf = it & 1;
            const uint32_t use = (it >> 1) & 1;
            if (MODE == MODE_FINAL) {
                named_bar_sync(1, kEpiThreads);               // the previous unit is done with the table
                load_route_table(un, a, etid, kEpiThreads, route_tok, route_scl);
            }
            wait_bar(tfull_bar(buf), use, abort_flag, a.err);
            if (named_bar_or(1, kEpiThreads, *abort_flag != 0)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_COLS;
#pragma unroll 1
            for (int c0 = c_first; c0 < un.ncols; c0 += c_step) {
                float v[16];
                tmem_ld16(tb + c0, v);
                if (MODE == MODE_SWIGLU) {
                    if (q >= 2) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) xg[i * 64 + l64] = v[i];
                    }
                    named_bar_sync(2 + grp, 128);
                    if (q < 2) {
                        __nv_bfloat16* act = static_cast<__nv_bfloat16*>(a.out);
                        const int col = un.wt * a.wtile_rows + static_cast<int>(rank) * 64 + l64;
                        if (act_is_plain(a.act, a.clamp)) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int r = un.row0 + c0 + i;
                                if (r < un.row_end)
                                    act[static_cast<size_t>(r) * a.out_ld + col] =
                                        __float2bfloat16_rn(silu_mul(v[i], xg[i * 64 + l64]));
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int r = un.row0 + c0 + i;
                                if (r < un.row_end)
                                    act[static_cast<size_t>(r) * a.out_ld + col] =
                                        __float2bfloat16_rn(act_mul(v[i], xg[i * 64 + l64], a.act, a.clamp));
                            }
                        }
                    }
                    named_bar_sync(2 + grp, 128);             // the exchange buffer is free again
                } else if (MODE == MODE_FINAL) {
                    emit16_final<1>(un, a, static_cast<int>(rank) * kBM + q * 32 + lane, c0, route_tok, route_scl,
                                    v, v);
                } else {
                    emit16<1, MODE_PLAIN, OutT>(un, a, static_cast<int>(rank) * kBM + q * 32 + lane, c0, v, v);
                }
            }
            tc_fence_before();
            named_bar_sync(1, kEpiThreads);
            if (etid == 0) {
                if (even) mbar_arrive(tempty_bar(buf));
                else mbar_arrive_cluster(tempty_even + 8u * buf);
            }
        }
    }

    // ---- teardown: both CTAs done before TMEM is freed together ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();
    if (warp == 1) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
}

template <int BT, int MODE, typename OutT>
cudaError_t launch_pair_kernel(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int pairs,
                               cudaStream_t s) {
    using C = PairCfg<BT>;
    auto kern = grouped_gemm_pair_kernel<BT, MODE, OutT>;
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    return launch_pdl_cluster(kern, dim3(2 * pairs), dim3(C::THREADS), C::SMEM_BYTES, 2, s, tmA, tmB, a);
}

// One GEMM on CTA pairs: mode SWIGLU (GEMM1, bf16 act), PLAIN (GEMM2 into an
// f32 or bf16 output) or FINAL (GEMM2 reduced into an f32 out); bt 128 or 256.
inline cudaError_t launch_gemm_pair(int mode, int bt, int out_dtype, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                    const GemmArgs& a, int pairs, cudaStream_t s) {
    if (bt == 256) {
        if (mode == MODE_SWIGLU) return launch_pair_kernel<256, MODE_SWIGLU, __nv_bfloat16>(tmA, tmB, a, pairs, s);
        if (mode == MODE_FINAL) return launch_pair_kernel<256, MODE_FINAL, float>(tmA, tmB, a, pairs, s);
        if (out_dtype == MOE_DTYPE_F32) return launch_pair_kernel<256, MODE_PLAIN, float>(tmA, tmB, a, pairs, s);
        return launch_pair_kernel<256, MODE_PLAIN, __nv_bfloat16>(tmA, tmB, a, pairs, s);
    }
    if (mode == MODE_SWIGLU) return launch_pair_kernel<128, MODE_SWIGLU, __nv_bfloat16>(tmA, tmB, a, pairs, s);
    if (mode == MODE_FINAL) return launch_pair_kernel<128, MODE_FINAL, float>(tmA, tmB, a, pairs, s);
    if (out_dtype == MOE_DTYPE_F32) return launch_pair_kernel<128, MODE_PLAIN, float>(tmA, tmB, a, pairs, s);
    return launch_pair_kernel<128, MODE_PLAIN, __nv_bfloat16>(tmA, tmB, a, pairs, s);
}

// Defined in gemm_pair.cu.
cudaError_t launch_gemm_pair_bf16(int mode, int bt, int out_dtype, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const GemmArgs& a, int pairs, cudaStream_t s);

}  // namespace gemm
}  // namespace moe
