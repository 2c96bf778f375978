// moe_permute_noalloc: the permute for callers that cannot allocate device
// memory. Examples are an inference engine that carves all device memory out
// of one arena at start-up and gives the libraries it hosts no allocator, a
// plugin loaded into a process whose allocator belongs to the host
// application, and a latency-critical path that must never reach cudaMalloc
// (it can synchronise the device and has no bounded cost). It computes exactly
// what moe_permute computes. The per-chunk expert histograms that moe_permute
// keeps in the caller's workspace live in a fixed array inside this library
// instead.
//
// The array is a file-scope static __device__ buffer of
// kNoAllocScratchInts ints (1 MiB). Every GPU that loads the library holds
// one copy of it until the process exits. Host code never passes the array's
// name to a kernel: in host code that name stands for a host-side shadow, not
// a device address. On the first call on a device, with that device current,
// cudaGetSymbolAddress gives the device pointer. A successful lookup is
// cached per device and passed to the kernels; a failed one is reported as
// MOE_ERR_CUDA and tried again by the next call. The cache assumes the
// device's primary context (the runtime API's default) for the life of the
// process.
//
// The permute writes every scratch entry it later reads (the count kernel
// fills the histograms before the scan reads them), so nothing has to be
// cleared between calls. All calls on a device share the one array: two
// calls whose kernels overlap on the GPU (for example on two streams with no
// ordering between them) race on it and give wrong maps.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kNoAllocScratchInts = 262144;   // 1 MiB

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    std::mutex mu;
    std::atomic<int32_t*> ptr{nullptr};
};
ScratchSlot g_scratch[kMaxDevices];

// Device pointer of the current device's scratch array, or nullptr if the
// lookup failed (then nothing is cached and the next call tries again).
int32_t* scratch_for_current_device() {
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) {
        cudaGetLastError();                      // this call's own error, reported as a status
        return nullptr;
    }
    if (d < 0 || d >= kMaxDevices) return nullptr;
    ScratchSlot* s = &g_scratch[d];
    int32_t* p = s->ptr.load(std::memory_order_acquire);
    if (p != nullptr) return p;
    std::lock_guard<std::mutex> lock(s->mu);
    p = s->ptr.load(std::memory_order_relaxed);
    if (p != nullptr) return p;
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_permute_scratch) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    p = static_cast<int32_t*>(addr);
    s->ptr.store(p, std::memory_order_release);
    return p;
}

}  // namespace

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_ids, int M, int top_k, int E,
                                          const int32_t* expert_map, int E_local, const void* x, int K,
                                          int32_t* expert_offsets, int32_t* expanded_idx_to_permuted_idx,
                                          int32_t* permuted_to_expanded, void* x_perm, cudaStream_t stream) {
    const moe_status a = moe::check_permute_args(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                                 expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm);
    if (a != MOE_OK) return a;
    // the fixed scratch bounds the problem size
    if (M > 0 && moe::permute_workspace_bytes(M, top_k, E_local) > kNoAllocScratchInts * sizeof(int32_t))
        return MOE_ERR_WORKSPACE;
    moe::DeviceInfo info;
    if (!moe::current_device_info(&info)) return MOE_ERR_CUDA;
    if (info.cc_major != 10 || info.cc_minor != 3) return MOE_ERR_UNSUPPORTED_ARCH;
    int32_t* scratch = scratch_for_current_device();
    if (scratch == nullptr) return MOE_ERR_CUDA;
    if (M == 0) {
        return cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E_local + 1), stream) == cudaSuccess
                   ? MOE_OK : MOE_ERR_CUDA;
    }
    const cudaError_t e = moe::launch_permute(topk_ids, M, top_k, E, expert_map, E_local, x, K, expert_offsets,
                                              expanded_idx_to_permuted_idx, permuted_to_expanded, x_perm, scratch,
                                              moe::device_error_word(), info, stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
