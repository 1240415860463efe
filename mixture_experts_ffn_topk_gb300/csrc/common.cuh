// common.cuh -- device helpers shared by the kernels of the GB300 MoE path.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

enum : int { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };

// Index element types of the training calls (moe_index_dtype in moe.h).
enum : int { IDX_U32 = 0, IDX_I32 = 1, IDX_I64 = 2 };

// Bits of the per-device status word (see moe_device_status in moe.h).
enum : unsigned { ST_BAD_INDEX = 1u, ST_TIMEOUT = 2u, ST_BOUNDS = 4u };

// Checks of the bounds-checking build (MOE_DEBUG_BOUNDS=1 at compile time):
// MOE_BOUNDS_OK(cond, status) is true when cond holds; when it does not, it
// records ST_BOUNDS in the status word and is false, so the caller skips the
// access. In the normal build it is `true` and costs nothing.
#ifndef MOE_DEBUG_BOUNDS
#define MOE_DEBUG_BOUNDS 0
#endif
#if MOE_DEBUG_BOUNDS
#define MOE_BOUNDS_OK(cond, status) ((cond) ? true : (atomicOr((status), ST_BOUNDS), false))
#else
#define MOE_BOUNDS_OK(cond, status) true
#endif

// Element access by dtype code. 16-bit types are loaded as raw words.
template <int DT> struct Elem;

template <> struct Elem<DT_F32> {
    using T = float;
    static __device__ __forceinline__ float to_f(T v) { return v; }
    static __device__ __forceinline__ T from_f(float v) { return v; }
};
template <> struct Elem<DT_BF16> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float to_f(T v) { return __bfloat162float(v); }
    static __device__ __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
};
template <> struct Elem<DT_F16> {
    using T = __half;
    static __device__ __forceinline__ float to_f(T v) { return __half2float(v); }
    static __device__ __forceinline__ T from_f(float v) { return __float2half_rn(v); }
};

// Load element i of a buffer whose dtype is only known at run time.
__device__ __forceinline__ float load_as_float(const void *p, int dt, int64_t i)
{
    if (dt == DT_F32) return static_cast<const float *>(p)[i];
    if (dt == DT_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    return __half2float(static_cast<const __half *>(p)[i]);
}

__device__ __forceinline__ void store_from_float(void *p, int dt, int64_t i, float v)
{
    if (dt == DT_F32) static_cast<float *>(p)[i] = v;
    else if (dt == DT_BF16) static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
    else static_cast<__half *>(p)[i] = __float2half_rn(v);
}

// Eight 16-bit elements (or four floats) travel as one 16-byte vector; the
// 16-bit pairs are reinterpreted from the 32-bit words w[].
union Vec16 {
    uint4 u;
    float f[4];
    uint32_t w[4];
};

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w)
{
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}
__device__ __forceinline__ uint32_t float2_to_bf16x2(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t float2_to_f16x2(float a, float b)
{
    const __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialisation allowed, so it may start while the
// previous kernel on the stream drains; it calls pdl_wait() before its first
// global-memory access (which returns once the previous grid has completed and
// its writes are visible) and pdl_launch_dependents() to let the next kernel
// start early in turn -- at entry for short kernels, after the main loop for
// bandwidth-heavy ones whose occupancy the next kernel's resident CTAs would
// cut. Launched without the attribute, both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host-side per-device caches (SM counts, symbol addresses, attribute
// opt-ins) cover device ordinals below this bound; higher ordinals skip the
// cache and look the value up on every call.
constexpr int kCachedDevices = 64;

// Every spin-wait in this library gives up after a bounded time (2 s unless
// moe_set_wait_limit_ns() chose another), sets ST_TIMEOUT in the status word
// and lets the kernel wind down. Kernels receive the limit as an argument,
// taken from wait_limit_ns() at launch.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

}  // namespace moe
