// dispatch_noalloc.cu -- moe_dispatch for callers that cannot allocate.
//
// moe_dispatch needs a small caller-provided scratch buffer (the per-chunk,
// per-expert histograms of its first pass). Some callers cannot hand one
// over: their device memory is owned by a pool that allows no allocation
// after start-up (a serving engine that reserves all of HBM up front, or a
// plugin whose host framework gives it no scratch space in its enqueue
// step), or they cannot afford the device-wide synchronisation that
// cudaMalloc / cudaFree imply on a latency-critical path. This entry point
// takes the same inputs and outputs as moe_dispatch and keeps that scratch in
// a fixed array that the library itself owns on every device.
#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// The built-in scratch: 256 KiB of per-chunk histogram counters (the size
// moe_dispatch_workspace_size reports must not exceed it). Every GPU on
// which the library is loaded holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 256u * 1024u;
static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

// In host code g_dispatch_scratch names a host-side stand-in, not device
// memory, so the device address is looked up once per device (with that
// device current) and cached; device ordinals past the cache are looked up
// on every call.
void *scratch_device_address(cudaError_t *err)
{
    static std::atomic<void *> cache[kCachedDevices];
    static std::mutex mu;
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    void *p = nullptr;
    if (dev < 0 || dev >= kCachedDevices) {
        *err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        return *err == cudaSuccess ? p : nullptr;
    }
    p = cache[dev].load();
    if (p != nullptr) return p;
    std::lock_guard<std::mutex> lock(mu);
    p = cache[dev].load();
    if (p != nullptr) return p;
    *err = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (*err != cudaSuccess) return nullptr;
    cache[dev].store(p);
    return p;
}

}  // namespace
}  // namespace moe

extern "C" int moe_dispatch_noalloc(const uint32_t *expert_indices, int64_t T, int top_k,
                                    int64_t E, const void *x, int x_dtype, int64_t H,
                                    int32_t *counts, int32_t *offsets, int32_t *row_of,
                                    int32_t *src_of, void *x_disp, void *stream)
{
    // the argument checks of moe_dispatch first, so a call fails with the
    // status moe_dispatch would give it
    const int rc = moe::check_dispatch_args(expert_indices, T, top_k, E, 0, x, x_dtype, H,
                                            counts, offsets, row_of, src_of, x_disp);
    if (rc != MOE_OK || T == 0) return rc;
    // then sizes beyond the built-in array, before anything is enqueued
    const size_t need = moe_dispatch_workspace_size(T, top_k, E);
    if (need > moe::kNoAllocScratchBytes)
        return moe::report_error(MOE_ERR_WORKSPACE,
                                 "moe_dispatch_noalloc: this T*top_k and E need more than the "
                                 "256 KiB built-in scratch (moe_dispatch_workspace_size); use "
                                 "moe_dispatch with a workspace");
    cudaError_t err = cudaSuccess;
    void *scratch = moe::scratch_device_address(&err);
    if (scratch == nullptr)
        return moe::report_error(MOE_ERR_CUDA,
                                 "moe_dispatch_noalloc: cannot resolve the scratch address");
    return moe_dispatch(expert_indices, T, top_k, E, x, x_dtype, H, counts, offsets, row_of,
                        src_of, x_disp, scratch, moe::kNoAllocScratchBytes, stream);
}
