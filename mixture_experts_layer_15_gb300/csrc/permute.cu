// Permute: group the M*top_k routes by local expert and build the permute map
// expanded_idx_to_permuted_idx (-1 = expert not local) of
// vllm/model_executor/layers/fused_moe/moe_output.py, UnfinalizedMoEOutput,
// plus the per-expert offsets (the "expert_num_tokens" of modular_kernel.py,
// FusedMoEPrepareAndFinalize.prepare), the inverse map and the row gather
// x_perm[p] = x[token of row p].
//
// The order is canonical: expert-major, then expanded index t*top_k + j. It is
// a stable counting sort. Routes are cut into chunks of 32*W (one route per
// thread, warp w owns 32 consecutive routes). Inside a warp, __match_any_sync
// gives each route its rank among the warp's routes to the same expert; a
// per-warp histogram and an exclusive scan over warps give the rank inside
// the chunk; an exclusive scan over chunks (per expert) and over experts
// gives the global row. No atomics decide an order, so the result is
// deterministic.
//
// One chunk (M*top_k <= 32*W): a single kernel; every CTA recomputes the tiny
// sort in shared memory and copies its share of the rows.
// Several chunks: count -> scan -> scatter -> gather (4 launches).
//
// map_base (0 for moe_permute) is added to every non-negative map entry: the
// chunked experts permute each chunk of tokens on its own and point its map
// entries at the chunk's rows of the caller's gemm2_permuted. The offsets,
// the inverse map and x_perm stay relative to the chunk.
#include "router_device.cuh"

namespace moe {
namespace {

// Warps per chunk: per-warp histograms are W x E_local ints in shared memory;
// keep them within 32 KB.
__host__ __device__ inline int warps_per_chunk(int E_local) {
    int w = 8192 / (E_local > 0 ? E_local : 1);
    return w < 1 ? 1 : (w > 32 ? 32 : w);
}

__device__ __forceinline__ int local_expert(const int32_t* __restrict__ ids,
                                            const int32_t* __restrict__ emap,
                                            int i, int n, int E, int E_l, int* err) {
    if (i >= n) return -2;                 // padding lane: in no group
    const int id = ids[i];                 // global or shared memory
    if (id < 0 || id >= E) { set_error(err, MOE_ERR_DEVICE_INDEX); return -1; }
    if (emap == nullptr) return id;
    const int le = __ldg(emap + id);
    if (le < -1 || le >= E_l) { set_error(err, MOE_ERR_DEVICE_INDEX); return -1; }
    return le;
}

// Per-warp histograms of one chunk -> exclusive scan over warps, in place.
// hist is [W][E_l]; on return hist[w][le] = routes to le in warps < w, and
// chunk_total[le] = routes to le in the whole chunk. Also returns, per
// thread, the route's local expert and its rank within its warp.
__device__ void chunk_ranks(const int32_t* ids, const int32_t* emap, int chunk_base, int n,
                            int E, int E_l, int* hist, int* chunk_total, int* err,
                            int& le, int& rank) {
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, W = blockDim.x >> 5;
    for (int i = tid; i < W * E_l; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    le = local_expert(ids, emap, chunk_base + tid, n, E, E_l, err);
    const unsigned peers = __match_any_sync(0xffffffffu, le);
    rank = __popc(peers & ((1u << lane) - 1u));
    if (rank == 0 && le >= 0) hist[warp * E_l + le] = __popc(peers);
    __syncthreads();
    for (int e = tid; e < E_l; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < W; ++w) {
            const int c = hist[w * E_l + e];
            hist[w * E_l + e] = run;
            run += c;
        }
        chunk_total[e] = run;
    }
    __syncthreads();
}

__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         int n16, int lane) {
    int c = lane;
    for (; c + 96 < n16; c += 128) {
        const uint4 a = __ldg(src + c), b = __ldg(src + c + 32);
        const uint4 d = __ldg(src + c + 64), e = __ldg(src + c + 96);
        dst[c] = a; dst[c + 32] = b; dst[c + 64] = d; dst[c + 96] = e;
    }
    for (; c < n16; c += 32) dst[c] = __ldg(src + c);
}

// Segments of a row copy: 128 16-byte vectors (2 KB; four per lane, loaded
// before any is stored), so that a few long rows still spread over many warps.
constexpr int kSegVec = 128;
__host__ __device__ inline int row_segments(int K) { return (K / 8 + kSegVec - 1) / kSegVec; }

__device__ __forceinline__ void copy_segment(const uint4* __restrict__ src, uint4* __restrict__ dst, int n16, int seg,
                                             int lane) {
    const int b = seg * kSegVec + lane;
    const int e = (seg + 1) * kSegVec < n16 ? (seg + 1) * kSegVec : n16;
    uint4 v[kSegVec / 32];
#pragma unroll
    for (int j = 0; j < kSegVec / 32; ++j)
        if (b + 32 * j < e) v[j] = __ldg(src + b + 32 * j);
#pragma unroll
    for (int j = 0; j < kSegVec / 32; ++j)
        if (b + 32 * j < e) dst[b + 32 * j] = v[j];
}

// ---- single chunk: one kernel ------------------------------------------------
// The whole permute of at most blockDim.x routes (ids in global or shared
// memory): every CTA sorts them in shared memory; CTA 0 writes the offsets and
// maps; every CTA copies its share of the rows.
__device__ __forceinline__ void permute_single_chunk(const int32_t* ids, int n, int top_k, int E,
                                                     const int32_t* __restrict__ emap, int E_l,
                                                     const __nv_bfloat16* __restrict__ x, int K,
                                                     int32_t* __restrict__ offsets, int32_t* __restrict__ map,
                                                     int32_t* __restrict__ inverse,
                                                     __nv_bfloat16* __restrict__ x_perm, int* err, int* sm,
                                                     int map_base = 0) {
    const int W = blockDim.x >> 5;
    int* hist = sm;                          // [W][E_l]
    int* total = hist + W * E_l;             // [E_l + 1]
    int* pos = total + E_l + 1;              // [32 W] permuted row of each route
    int* tmp = pos + blockDim.x;             // [33]
    int le, rank;
    // Only CTA 0 reports device errors (all CTAs see the same ids).
    chunk_ranks(ids, emap, 0, n, E, E_l, hist, total, blockIdx.x == 0 ? err : nullptr, le, rank);
    const int R = block_exclusive_scan(total, E_l, tmp);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int p = le >= 0 ? total[le] + hist[warp * E_l + le] + rank : -1;
    pos[tid] = p;
    if (blockIdx.x == 0) {
        for (int e = tid; e < E_l; e += blockDim.x) offsets[e] = total[e];
        if (tid == 0) offsets[E_l] = R;
        if (tid < n) {
            map[tid] = p >= 0 ? p + map_base : -1;
            if (p >= 0) inverse[p] = tid;
        }
    }
    if (x_perm == nullptr) return;
    __syncthreads();
    // rows: segment s of route i's row (i < n, local) is copied by global warp
    // (i * segs + s) % (grid * W)
    const int gw = blockIdx.x * W + warp, nw = gridDim.x * W, n16 = K / 8, segs = row_segments(K);
    for (int it = gw; it < n * segs; it += nw) {
        const int i = it / segs;
        const int pi = pos[i];
        if (pi < 0) continue;
        copy_segment(reinterpret_cast<const uint4*>(x + static_cast<size_t>(i / top_k) * K),
                     reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(pi) * K), n16, it % segs, tid & 31);
    }
}

__global__ void permute_fused_kernel(const int32_t* __restrict__ ids, int n, int top_k, int E,
                                     const int32_t* __restrict__ emap, int E_l,
                                     const __nv_bfloat16* __restrict__ x, int K,
                                     int32_t* __restrict__ offsets, int32_t* __restrict__ map,
                                     int32_t* __restrict__ inverse, __nv_bfloat16* __restrict__ x_perm,
                                     int* err, int map_base) {
    extern __shared__ int sm[];
    permute_single_chunk(ids, n, top_k, E, emap, E_l, x, K, offsets, map, inverse, x_perm, err, sm, map_base);
}

// Router and single-chunk permute in one kernel (small batches), launched in
// clusters of G CTAs. The CTAs of a cluster split the tokens (one warp per
// token, the router's own per-token code) and keep the routed ids in their
// shared memory; after a cluster barrier every CTA reads the whole id list
// through distributed shared memory, and after a second one (no CTA reads
// another's shared memory past it) every CTA runs the same single-chunk
// permute and copies its share of the rows. Clusters beyond the first redo
// the routing (cheap at these sizes) and only add row-copy bandwidth; the
// first cluster writes the ids and weights.
template <int SLOTS, bool SIGMOID>
__global__ void route_permute_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int M,
                                     int E, int top_k, int n_group, int topk_group, float rsf,
                                     int32_t* __restrict__ ids_out, void* __restrict__ w_out, int wdtype,
                                     const int32_t* __restrict__ emap, int E_l,
                                     const __nv_bfloat16* __restrict__ x, int K,
                                     int32_t* __restrict__ offsets, int32_t* __restrict__ map,
                                     int32_t* __restrict__ inverse, __nv_bfloat16* __restrict__ x_perm,
                                     int G, int* err) {
    extern __shared__ int sm[];
    const int W = blockDim.x >> 5, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = M * top_k;
    const int rank = static_cast<int>(cluster_ctarank());
    const bool first_cluster = static_cast<int>(blockIdx.x) < G;
    int* ids_own = sm;                                           // [blockDim] routes this CTA routed
    int* ids_all = ids_own + blockDim.x;                         // [blockDim] every route
    float* bsc = reinterpret_cast<float*>(ids_all + blockDim.x); // [W][E] sigmoid router scratch
    int* rest = reinterpret_cast<int*>(bsc + (SIGMOID ? W * E : 0));
    pdl_wait();
    pdl_trigger();
    const int GW = G * W;
    for (int t = rank * W + warp; t < M; t += GW) {
        int id;
        float w;
        if (SIGMOID)
            route::route_token_sigmoid<SLOTS>(logits + static_cast<size_t>(t) * E, bias, E, top_k, n_group,
                                              topk_group, rsf, lane, bsc + warp * E, id, w);
        else
            route::route_token_softmax<SLOTS>(logits + static_cast<size_t>(t) * E, E, top_k, rsf, lane, id, w);
        if (lane < top_k) {
            const int o = t * top_k + lane;
            ids_own[o] = id;
            if (first_cluster) {
                ids_out[o] = id;
                store_from_f32(w_out, o, w, wdtype);
            }
        }
    }
    __syncwarp();
    cluster_sync_all();                                          // routed ids visible cluster-wide
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int owner = ((i / top_k) % GW) / W;                // the CTA whose warp routed token i / top_k
        ids_all[i] = owner == rank ? ids_own[i] : ld_cluster_i32(ids_own + i, static_cast<uint32_t>(owner));
    }
    __syncwarp();
    cluster_sync_all();                                          // remote reads done; ids_all visible
    permute_single_chunk(ids_all, n, top_k, E, emap, E_l, x, K, offsets, map, inverse, x_perm, err, rest);
}

template <int SLOTS, bool SIGMOID>
cudaError_t launch_route_permute_t(int clusters, int G, dim3 block, size_t smem, cudaStream_t s,
                                   const float* logits, const float* bias, int M, int E, int top_k, int n_group,
                                   int topk_group, float rsf, int32_t* ids, void* w, int wdtype,
                                   const int32_t* emap, int E_l, const __nv_bfloat16* x, int K, int32_t* offsets,
                                   int32_t* map, int32_t* inverse, __nv_bfloat16* xp, int* err) {
    return launch_pdl_cluster(route_permute_kernel<SLOTS, SIGMOID>, dim3(clusters * G), block, smem, G, s, logits,
                              bias, M, E, top_k, n_group, topk_group, rsf, ids, w, wdtype, emap, E_l, x, K, offsets,
                              map, inverse, xp, G, err);
}

// Launch shape of the fused kernel: W warps per CTA (one thread per route for
// the permute, and enough warps that a cluster of G <= 8 CTAs routes every
// token with one warp), and its shared memory.
struct RoutePermuteShape {
    int W, G;
    size_t smem;
};
RoutePermuteShape route_permute_shape(int M, int top_k, int E, int E_l, int method) {
    RoutePermuteShape r;
    const int n = M * top_k;
    int W = (n + 31) / 32;
    const int per_cluster = (M + 7) / 8;                         // warps per CTA so 8 CTAs cover M tokens
    if (W < per_cluster) W = per_cluster;
    if (W < 1) W = 1;
    r.W = W;
    r.G = (M + W - 1) / W;
    if (r.G > 8) r.G = 8;
    if (r.G < 1) r.G = 1;
    const bool sig = method == MOE_ROUTE_SIGMOID_GROUPED_TOPK;
    r.smem = sizeof(int) * (2 * 32 * W + W * E_l + E_l + 1 + 32 * W + 33) + (sig ? sizeof(float) * W * E : 0);
    return r;
}

// ---- several chunks ------------------------------------------------------------
__global__ void permute_count_kernel(const int32_t* __restrict__ ids, int n, int E,
                                     const int32_t* __restrict__ emap, int E_l,
                                     int32_t* __restrict__ chunk_counts, int* err) {
    extern __shared__ int sm[];
    const int W = blockDim.x >> 5;
    int* hist = sm;
    int* total = hist + W * E_l;
    int le, rank;
    chunk_ranks(ids, emap, blockIdx.x * blockDim.x, n, E, E_l, hist, total, err, le, rank);
    for (int e = threadIdx.x; e < E_l; e += blockDim.x)
        chunk_counts[static_cast<size_t>(blockIdx.x) * E_l + e] = total[e];
}

// chunk_counts[c][e] -> global first row of (chunk c, expert e); offsets.
__global__ void permute_scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E_l,
                                    int32_t* __restrict__ offsets) {
    extern __shared__ int sm[];
    int* total = sm;                         // [E_l]
    int* tmp = total + E_l;                  // [33]
    pdl_wait();
    pdl_trigger();
    for (int e = threadIdx.x; e < E_l; e += blockDim.x) {
        // the counts of 8 chunks are loaded before any is used, so the loads
        // overlap instead of forming one long dependent chain
        int run = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 8) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = c0 + i < nchunks ? chunk_counts[static_cast<size_t>(c0 + i) * E_l + e] : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (c0 + i < nchunks) chunk_counts[static_cast<size_t>(c0 + i) * E_l + e] = run;
                run += v[i];
            }
        }
        total[e] = run;
    }
    __syncthreads();
    const int R = block_exclusive_scan(total, E_l, tmp);
    for (int e = threadIdx.x; e < E_l; e += blockDim.x) {
        const int base = total[e];
        offsets[e] = base;
        for (int c0 = 0; c0 < nchunks; c0 += 8) {
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = c0 + i < nchunks ? chunk_counts[static_cast<size_t>(c0 + i) * E_l + e] : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (c0 + i < nchunks) chunk_counts[static_cast<size_t>(c0 + i) * E_l + e] = v[i] + base;
        }
    }
    if (threadIdx.x == 0) offsets[E_l] = R;
}

__global__ void permute_scatter_kernel(const int32_t* __restrict__ ids, int n, int E,
                                       const int32_t* __restrict__ emap, int E_l,
                                       const int32_t* __restrict__ chunk_base,
                                       int32_t* __restrict__ map, int32_t* __restrict__ inverse, int map_base) {
    extern __shared__ int sm[];
    const int W = blockDim.x >> 5;
    int* hist = sm;
    int* total = hist + W * E_l;
    int le, rank;
    const int base = blockIdx.x * blockDim.x;
    chunk_ranks(ids, emap, base, n, E, E_l, hist, total, nullptr, le, rank);
    const int i = base + threadIdx.x;
    if (i >= n) return;
    int p = -1;
    if (le >= 0)
        p = chunk_base[static_cast<size_t>(blockIdx.x) * E_l + le] + hist[(threadIdx.x >> 5) * E_l + le] + rank;
    map[i] = p >= 0 ? p + map_base : -1;
    if (p >= 0) inverse[p] = i;
}

// x_perm[p] = x[inverse[p] / top_k] for p < offsets[E_l]; one warp per row.
// R and the inverse entries are checked against rows_alloc (when they come
// from a caller, not from this permute): an out-of-range one sets
// MOE_ERR_DEVICE_INDEX and its row is skipped.
__global__ void permute_gather_kernel(const int32_t* __restrict__ offsets, int E_l,
                                      const int32_t* __restrict__ inverse, int top_k,
                                      const __nv_bfloat16* __restrict__ x, int K,
                                      __nv_bfloat16* __restrict__ x_perm, int rows_alloc, int* err) {
    pdl_wait();
    pdl_trigger();
    int R = __ldg(offsets + E_l);
    if (R < 0 || R > rows_alloc) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, MOE_ERR_DEVICE_INDEX);
        R = R < 0 ? 0 : rows_alloc;
    }
    const int warps = blockDim.x >> 5;
    const int n16 = K / 8;
    for (int p = blockIdx.x * warps + (threadIdx.x >> 5); p < R; p += gridDim.x * warps) {
        const int e = __ldg(inverse + p);
        if (e < 0 || e >= rows_alloc) {
            if ((threadIdx.x & 31) == 0) set_error(err, MOE_ERR_DEVICE_INDEX);
            continue;
        }
        copy_row(reinterpret_cast<const uint4*>(x + static_cast<size_t>(e / top_k) * K),
                 reinterpret_cast<uint4*>(x_perm + static_cast<size_t>(p) * K), n16, threadIdx.x & 31);
    }
}

}  // namespace

bool route_permute_fusible(int M, int top_k, int E, int E_l, int method) {
    const int n = M * top_k;
    if (M > 64 || n > 32 * warps_per_chunk(E_l)) return false;
    const RoutePermuteShape r = route_permute_shape(M, top_k, E, E_l, method);
    return r.W <= warps_per_chunk(E_l) && r.smem <= 48 * 1024;
}

cudaError_t launch_route_permute(const float* logits, int M, int E, int top_k, int method, const float* bias,
                                 int n_group, int topk_group, float rsf, int32_t* ids, void* w, int wdtype,
                                 const int32_t* emap, int E_l, const void* x, int K, int32_t* offsets,
                                 int32_t* map, int32_t* inverse, void* x_perm, int* err, const DeviceInfo& dev,
                                 cudaStream_t s) {
    const int n = M * top_k;
    const RoutePermuteShape r = route_permute_shape(M, top_k, E, E_l, method);
    const bool sig = method == MOE_ROUTE_SIGMOID_GROUPED_TOPK;
    // clusters: one is enough to route; more add row-copy bandwidth (one warp per row)
    int clusters = 1;
    if (x_perm != nullptr) {
        clusters = ceil_div(n * row_segments(K), r.G * r.W);
        const int cap = (2 * dev.sm_count) / r.G;
        if (clusters > cap) clusters = cap;
        if (clusters < 1) clusters = 1;
    }
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    __nv_bfloat16* xp = static_cast<__nv_bfloat16*>(x_perm);
    const dim3 block(32 * r.W);
    const int slots = ceil_div(E, 32);
#define MOE_RP(S)                                                                                            \
    return sig ? launch_route_permute_t<S, true>(clusters, r.G, block, r.smem, s, logits, bias, M, E, top_k,   \
                                                 n_group, topk_group, rsf, ids, w, wdtype, emap, E_l, xb, K,   \
                                                 offsets, map, inverse, xp, err)                              \
               : launch_route_permute_t<S, false>(clusters, r.G, block, r.smem, s, logits, bias, M, E, top_k, \
                                                  n_group, topk_group, rsf, ids, w, wdtype, emap, E_l, xb, K,  \
                                                  offsets, map, inverse, xp, err)
    if (slots <= 1) MOE_RP(1);
    if (slots <= 2) MOE_RP(2);
    if (slots <= 4) MOE_RP(4);
    if (slots <= 8) MOE_RP(8);
    if (slots <= 16) MOE_RP(16);
    MOE_RP(32);
#undef MOE_RP
}

size_t permute_workspace_bytes(int M, int top_k, int E_local) {
    const long long n = static_cast<long long>(M) * top_k;
    const int chunk = 32 * warps_per_chunk(E_local);
    const long long nchunks = (n + chunk - 1) / chunk;
    if (nchunks <= 1) return 0;
    return static_cast<size_t>(nchunks) * E_local * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* ids, int M, int top_k, int E, const int32_t* emap,
                           int E_l, const void* x, int K, int32_t* offsets, int32_t* map,
                           int32_t* inverse, void* x_perm, void* ws, int* err,
                           const DeviceInfo& dev, cudaStream_t s, int map_base) {
    const int n = M * top_k;
    const int W = warps_per_chunk(E_l);
    const int threads = 32 * W;
    const int nchunks = ceil_div(n, threads);
    // a single chunk uses only as many warps as it has routes
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    __nv_bfloat16* xp = static_cast<__nv_bfloat16*>(x_perm);
    if (nchunks <= 1) {
        const int w1 = ceil_div(n, 32) < 1 ? 1 : ceil_div(n, 32);
        const int t1 = 32 * w1;
        const size_t smem = sizeof(int) * (w1 * E_l + E_l + 1 + t1 + 33);
        int grid = 1;
        if (x_perm != nullptr) {
            // one warp per 2 KB segment of a gathered row (at most 2 CTAs per SM)
            grid = ceil_div(n * row_segments(K), w1);
            grid = grid < 1 ? 1 : (grid > 2 * dev.sm_count ? 2 * dev.sm_count : grid);
        }
        return launch_pdl(permute_fused_kernel, dim3(grid), dim3(t1), smem, s, ids, n, top_k, E, emap, E_l,
                          xb, K, offsets, map, inverse, xp, err, map_base);
    }
    int32_t* chunk = static_cast<int32_t*>(ws);
    const size_t smem_h = sizeof(int) * (W * E_l + E_l);
    cudaError_t e = launch_pdl(permute_count_kernel, dim3(nchunks), dim3(threads), smem_h, s, ids, n, E, emap,
                               E_l, chunk, err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), sizeof(int) * (E_l + 33), s, chunk, nchunks, E_l,
                   offsets);
    if (e != cudaSuccess) return e;
    e = launch_pdl(permute_scatter_kernel, dim3(nchunks), dim3(threads), smem_h, s, ids, n, E, emap, E_l,
                   static_cast<const int32_t*>(chunk), map, inverse, map_base);
    if (e != cudaSuccess || x_perm == nullptr) return e;
    const int rows_per_block = 8;   // 256 threads, one warp per row
    int grid = ceil_div(n, rows_per_block);
    if (grid > 8 * dev.sm_count) grid = 8 * dev.sm_count;
    return launch_pdl(permute_gather_kernel, dim3(grid), dim3(32 * rows_per_block), 0, s,
                      static_cast<const int32_t*>(offsets), E_l, static_cast<const int32_t*>(inverse), top_k, xb,
                      K, xp, n, err);
}

cudaError_t launch_gather_rows(const int32_t* offsets, int E_l, const int32_t* inverse, int top_k, int rows_alloc,
                               const void* x, int K, void* x_perm, const DeviceInfo& dev, cudaStream_t s) {
    const int rows_per_block = 8;
    int grid = ceil_div(rows_alloc, rows_per_block);
    if (grid > 8 * dev.sm_count) grid = 8 * dev.sm_count;
    if (grid < 1) grid = 1;
    return launch_pdl(permute_gather_kernel, dim3(grid), dim3(32 * rows_per_block), 0, s, offsets, E_l, inverse,
                      top_k, static_cast<const __nv_bfloat16*>(x), K, static_cast<__nv_bfloat16*>(x_perm),
                      rows_alloc, device_error_word());
}

}  // namespace moe
