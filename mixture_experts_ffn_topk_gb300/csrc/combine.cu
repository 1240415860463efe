// combine.cu -- weighted combine back to token order, optionally fused with
// the residual Add + RMSNorm epilogue.
//
// ruDNN user guide, sections 3 and 6 (DispatchedTokens::combine restores token
// order and sums expert outputs times routing weights);
// aclnnMoeDistributeCombineAddRmsNormV2, "Function" formula:
//   x = combineOut + residualX,  y = x / sqrt(mean(x^2) + eps) * gamma,
// with rstdOut = 1 / sqrt(mean(x^2) + eps) in FP32; ruDNN user guide section 7
// (FP32 statistics, output in the input dtype).
//
// One CTA per token (grid-stride). Each thread owns V 16-byte vectors of the
// row; for every slot j it issues V independent 16-byte loads of expert output
// row row_of[t*k+j], so a CTA keeps k*V loads in flight. The sum runs in FP32
// in slot order. With the norm, x is rounded to the output dtype first and the
// statistics are taken on the rounded x (so y == RMSNorm(x_out)); x stays in
// registers between the two passes. HBM-bound.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

template <int DT> struct VecTraits;
template <> struct VecTraits<DT_F32> { static constexpr int N = 4; };
template <> struct VecTraits<DT_BF16> { static constexpr int N = 8; };
template <> struct VecTraits<DT_F16> { static constexpr int N = 8; };

template <int DT>
__device__ __forceinline__ void unpack(const Vec16 &v, float (&f)[VecTraits<DT>::N])
{
    if constexpr (DT == DT_F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = v.f[i];
    } else if constexpr (DT == DT_BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = bf16x2_to_float2(v.w[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = f16x2_to_float2(v.w[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
}

template <int DT>
__device__ __forceinline__ Vec16 pack(const float (&f)[VecTraits<DT>::N])
{
    Vec16 v;
    if constexpr (DT == DT_F32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v.f[i] = f[i];
    } else if constexpr (DT == DT_BF16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v.w[i] = float2_to_bf16x2(f[2 * i], f[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v.w[i] = float2_to_f16x2(f[2 * i], f[2 * i + 1]);
    }
    return v;
}

template <int DT, int V, bool NORM>
__global__ void __launch_bounds__(256)
combine_kernel(const uint4 *__restrict__ out_disp, const void *__restrict__ w,
               int wdt, const int32_t *__restrict__ row_of,
               const uint4 *__restrict__ residual, const void *__restrict__ gamma,
               int gdt, float eps, int64_t T, int top_k, int64_t H,
               uint4 *__restrict__ y, uint4 *__restrict__ x_out,
               float *__restrict__ rstd)
{
    constexpr int N = VecTraits<DT>::N;
    const int64_t nvec = H / N;
    __shared__ float red[8];
    __shared__ float s_rstd;

    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        // rows handled in passes of V * blockDim vectors (one pass when NORM)
        for (int64_t base = 0; base < nvec; base += (int64_t)V * blockDim.x) {
            float acc[V][N];
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int i = 0; i < N; ++i) acc[v][i] = 0.0f;
            bool nan_row = false;
#pragma unroll 2
            for (int j = 0; j < top_k; ++j) {
                const int32_t r = row_of[t * top_k + j];
                const float wj = load_as_float(w, wdt, t * top_k + j);
                if (r < 0) { nan_row = true; continue; }
                const uint4 *src = out_disp + (int64_t)r * nvec;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                    if (c < nvec) {
                        Vec16 q;
                        q.u = __ldg(src + c);
                        float f[N];
                        unpack<DT>(q, f);
#pragma unroll
                        for (int i = 0; i < N; ++i) acc[v][i] = fmaf(wj, f[i], acc[v][i]);
                    }
                }
            }
            if (nan_row) {
#pragma unroll
                for (int v = 0; v < V; ++v)
#pragma unroll
                    for (int i = 0; i < N; ++i) acc[v][i] = __int_as_float(0x7fc00000);
            }
            if constexpr (!NORM) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                    if (c < nvec) y[t * nvec + c] = pack<DT>(acc[v]).u;
                }
            } else {
                // x = acc + residual, rounded to dtype; sum of squares of it
                float ss = 0.0f;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                    if (c < nvec) {
                        Vec16 q;
                        q.u = __ldg(residual + t * nvec + c);
                        float f[N];
                        unpack<DT>(q, f);
#pragma unroll
                        for (int i = 0; i < N; ++i) acc[v][i] += f[i];
                        const Vec16 xr = pack<DT>(acc[v]);
                        x_out[t * nvec + c] = xr.u;
                        unpack<DT>(xr, acc[v]);
#pragma unroll
                        for (int i = 0; i < N; ++i) ss = fmaf(acc[v][i], acc[v][i], ss);
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (lane_id() == 0) red[threadIdx.x / 32] = ss;
                __syncthreads();
                if (threadIdx.x == 0) {
                    float tot = 0.0f;
                    for (int i = 0; i < (int)(blockDim.x / 32); ++i) tot += red[i];
                    const float r = 1.0f / sqrtf(tot / (float)H + eps);
                    s_rstd = r;
                    rstd[t] = r;
                }
                __syncthreads();
                const float r = s_rstd;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                    if (c < nvec) {
                        float f[N];
#pragma unroll
                        for (int i = 0; i < N; ++i)
                            f[i] = acc[v][i] * r * load_as_float(gamma, gdt, c * N + i);
                        y[t * nvec + c] = pack<DT>(f).u;
                    }
                }
            }
        }
    }
}

template <int DT, bool NORM>
cudaError_t launch_combine_dt(const void *out_disp, const void *w, int wdt,
                              const int32_t *row_of, const void *residual,
                              const void *gamma, int gdt, float eps, int64_t T,
                              int top_k, int64_t H, void *y, void *x_out,
                              float *rstd, cudaStream_t s)
{
    constexpr int N = VecTraits<DT>::N;
    const int64_t nvec = H / N;
    int V = 1;
    while (V < 8 && nvec > (int64_t)V * 256) V *= 2;
    int64_t threads = (nvec + V - 1) / V;
    threads = (threads + 31) / 32 * 32;
    if (threads > 256) threads = 256;
    if (threads < 32) threads = 32;
    int64_t blocks = T;
    const int64_t cap = (int64_t)device_sm_count() * 32;
    if (blocks > cap) blocks = cap;
    const uint4 *od = static_cast<const uint4 *>(out_disp);
    const uint4 *res = static_cast<const uint4 *>(residual);
    uint4 *yv = static_cast<uint4 *>(y);
    uint4 *xv = static_cast<uint4 *>(x_out);
#define MOE_COMBINE_LAUNCH(VV)                                                  \
    combine_kernel<DT, VV, NORM><<<(unsigned)blocks, (unsigned)threads, 0, s>>>( \
        od, w, wdt, row_of, res, gamma, gdt, eps, T, top_k, H, yv, xv, rstd)
    switch (V) {
    case 1: MOE_COMBINE_LAUNCH(1); break;
    case 2: MOE_COMBINE_LAUNCH(2); break;
    case 4: MOE_COMBINE_LAUNCH(4); break;
    default: MOE_COMBINE_LAUNCH(8); break;
    }
#undef MOE_COMBINE_LAUNCH
    return cudaGetLastError();
}

template <bool NORM>
cudaError_t launch_combine_norm(int dt, const void *out_disp, const void *w,
                                int wdt, const int32_t *row_of,
                                const void *residual, const void *gamma,
                                int gdt, float eps, int64_t T, int top_k,
                                int64_t H, void *y, void *x_out, float *rstd,
                                cudaStream_t s)
{
    switch (dt) {
    case DT_F32:
        return launch_combine_dt<DT_F32, NORM>(out_disp, w, wdt, row_of, residual, gamma, gdt, eps, T, top_k, H, y, x_out, rstd, s);
    case DT_BF16:
        return launch_combine_dt<DT_BF16, NORM>(out_disp, w, wdt, row_of, residual, gamma, gdt, eps, T, top_k, H, y, x_out, rstd, s);
    default:
        return launch_combine_dt<DT_F16, NORM>(out_disp, w, wdt, row_of, residual, gamma, gdt, eps, T, top_k, H, y, x_out, rstd, s);
    }
}

}  // namespace

// With the norm the whole row must fit one pass: 8 vectors x 256 threads.
int combine_max_h(int dt, bool norm)
{
    if (!norm) return 1 << 30;
    return 8 * 256 * (dt == DT_F32 ? 4 : 8);
}

cudaError_t launch_combine(const void *out_disp, int dt, const void *w, int wdt,
                           const int32_t *row_of, const void *residual,
                           const void *gamma, int gdt, float eps, int64_t T,
                           int top_k, int64_t H, void *y, void *x_out,
                           float *rstd, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    if (residual != nullptr)
        return launch_combine_norm<true>(dt, out_disp, w, wdt, row_of, residual, gamma, gdt, eps, T, top_k, H, y, x_out, rstd, s);
    return launch_combine_norm<false>(dt, out_disp, w, wdt, row_of, residual, gamma, gdt, eps, T, top_k, H, y, x_out, rstd, s);
}

}  // namespace moe
