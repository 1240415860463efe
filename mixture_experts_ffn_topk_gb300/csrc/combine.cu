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
// One CTA per token (grid-stride). A row is moved in groups of 8 elements (one
// 16-byte vector of a 16-bit type, two of FP32). Each thread owns V groups; for
// every slot j it issues V independent loads of expert-output row
// row_of[t*k+j], so a CTA keeps k*V loads in flight. The sum runs in FP32 in
// slot order. Expert outputs may be FP32 (the one-call forward keeps them
// unrounded) or the activation dtype. With the norm, x is rounded to the
// activation dtype first and the statistics are taken on the rounded x (so
// y == RMSNorm(x_out)); x stays in registers between the two passes.
// HBM-bound.
//
// With extras (aclnnMoeDistributeCombineAddRmsNormV2, formula and parameter
// list): a slot the active mask drops contributes nothing; an expert id
// past the E routed experts names a special expert -- zero (contributes 0),
// copy (the token's original row oriX) or const (alpha1[c] * oriX + alpha2[c]
// * V[c]); and a shared-expert row is added once per kept slot, scaled like
// it, i.e. (sum of the kept weights) * sharedX.
//
// rmsnorm_kernel is the standalone RMSNorm of ruDNN user guide section 7:
// y = x / sqrt(mean(x^2) + eps) * gamma per row, FP32 statistics, output in
// the input dtype.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kMaxV = 8;          // groups per thread
constexpr int kMaxThreads = 256;

template <int DT>
__device__ __forceinline__ void load8(const void *base, int64_t g, float (&f)[8])
{
    if constexpr (DT == DT_F32) {
        const uint4 *p = static_cast<const uint4 *>(base) + 2 * g;
        Vec16 a, b;
        a.u = __ldg(p);
        b.u = __ldg(p + 1);
#pragma unroll
        for (int i = 0; i < 4; ++i) { f[i] = a.f[i]; f[4 + i] = b.f[i]; }
    } else {
        Vec16 a;
        a.u = __ldg(static_cast<const uint4 *>(base) + g);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 p = DT == DT_BF16 ? bf16x2_to_float2(a.w[i]) : f16x2_to_float2(a.w[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
}

// Round to DT; f is replaced by the rounded values.
template <int DT>
__device__ __forceinline__ void store8(void *base, int64_t g, float (&f)[8])
{
    if constexpr (DT == DT_F32) {
        uint4 *p = static_cast<uint4 *>(base) + 2 * g;
        p[0] = make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
        p[1] = make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                          __float_as_uint(f[7]));
    } else {
        Vec16 a;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a.w[i] = DT == DT_BF16 ? float2_to_bf16x2(f[2 * i], f[2 * i + 1])
                                   : float2_to_f16x2(f[2 * i], f[2 * i + 1]);
            const float2 p = DT == DT_BF16 ? bf16x2_to_float2(a.w[i]) : f16x2_to_float2(a.w[i]);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
        static_cast<uint4 *>(base)[g] = a.u;
    }
}

__device__ __forceinline__ void load8_rt(const void *base, int dt, int64_t g, float (&f)[8])
{
    if (dt == DT_F32) load8<DT_F32>(base, g, f);
    else if (dt == DT_BF16) load8<DT_BF16>(base, g, f);
    else load8<DT_F16>(base, g, f);
}

// Sources of a slot other than a dispatched expert row (see the header).
enum SlotKind : int { kRouted = 0, kZero = 1, kCopy = 2, kConst = 3, kBad = 4, kSkip = 5 };

template <int ODT, int YDT, int V, bool NORM, bool EXTRAS>
__global__ void __launch_bounds__(kMaxThreads)
combine_kernel(const void *__restrict__ out_disp, const void *__restrict__ w, int wdt,
               const int32_t *__restrict__ row_of, const void *__restrict__ residual,
               const void *__restrict__ gamma, int gdt, float eps, int64_t T, int top_k,
               int64_t H, void *__restrict__ y, void *__restrict__ x_out,
               float *__restrict__ rstd, CombineExtras ex)
{
    const int64_t ng = H / 8;
    __shared__ float red[kMaxThreads / 32];
    __shared__ float s_rstd;
    // EXTRAS: one chunk of classified slots (kind, weight, row offset or const index)
    __shared__ int s_kind[EXTRAS ? kMaxThreads : 1];
    __shared__ float s_w[EXTRAS ? kMaxThreads : 1];
    __shared__ int64_t s_off[EXTRAS ? kMaxThreads : 1];
    const int64_t elem_o = ODT == DT_F32 ? 4 : 2;
    pdl_wait();
    pdl_launch_dependents();

    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        // groups handled in passes of V * blockDim (a single pass with NORM)
        for (int64_t base = 0; base < ng; base += (int64_t)V * blockDim.x) {
            float acc[V][8];
#pragma unroll
            for (int v = 0; v < V; ++v)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[v][i] = 0.0f;
            bool nan_row = false;
            float wkept = 0.0f;                 // sum of the kept slots' weights (shared term)
            if constexpr (!EXTRAS) {
                // unrolled by 8 so up to eight slots' rows are requested
                // before the first is summed (top_k = 8: 2 -> 8 took the
                // combine + Add + RMSNorm workload from 71 % to 81 % of HBM)
#pragma unroll 8
                for (int j = 0; j < top_k; ++j) {
                    const int64_t a = t * top_k + j;
                    const float wj = load_as_float(w, wdt, a);
                    const int32_t r = row_of[a];
                    if (r < 0 || (int64_t)r >= T * top_k) { nan_row = true; continue; }
                    const void *src = static_cast<const uint8_t *>(out_disp) + (int64_t)r * H * elem_o;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                        if (c < ng) {
                            float f[8];
                            load8<ODT>(src, c, f);
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[v][i] = fmaf(wj, f[i], acc[v][i]);
                        }
                    }
                }
            } else {
                // slots in chunks of blockDim: one thread per slot classifies it
                // (mask bit, id, weight, row) into shared memory, then every thread
                // walks the chunk with only its data loads left to wait for
                for (int j0 = 0; j0 < top_k; j0 += blockDim.x) {
                    const int nj = top_k - j0 < (int)blockDim.x ? top_k - j0 : (int)blockDim.x;
                    __syncthreads();                    // the previous chunk's readers are done
                    if ((int)threadIdx.x < nj) {
                        const int64_t a = t * top_k + j0 + threadIdx.x;
                        int k2 = kRouted;
                        int64_t off = 0;
                        float wv = 0.0f;
                        if ((ex.mask_dims == 1 && !ex.mask[t]) || (ex.mask_dims == 2 && !ex.mask[a])) {
                            k2 = kSkip;
                        } else {
                            if (ex.ids != nullptr) {
                                const int64_t id = ex.ids[a];
                                if (id >= ex.E) {
                                    const int64_t sp = id - ex.E;
                                    k2 = sp < ex.zero_n ? kZero
                                       : sp < ex.zero_n + ex.copy_n ? kCopy
                                       : sp < ex.zero_n + ex.copy_n + ex.const_n ? kConst : kBad;
                                    off = sp - ex.zero_n - ex.copy_n;
                                }
                            }
                            wv = load_as_float(w, wdt, a);
                            if (k2 == kRouted) {
                                const int32_t r = row_of[a];
                                if (r < 0 || (int64_t)r >= T * top_k) k2 = kBad;
                                else off = (int64_t)r * H * elem_o;
                            }
                        }
                        s_kind[threadIdx.x] = k2;
                        s_w[threadIdx.x] = wv;
                        s_off[threadIdx.x] = off;
                    }
                    __syncthreads();
                    // routed slots first, in the same tight loop as the plain combine
                    // (the loads of two slots in flight together)
#pragma unroll 2
                    for (int jj = 0; jj < nj; ++jj) {
                        if (s_kind[jj] != kRouted) continue;
                        const float wj = s_w[jj];
                        wkept += wj;
                        const void *src = static_cast<const uint8_t *>(out_disp) + s_off[jj];
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                            if (c < ng) {
                                float f[8];
                                load8<ODT>(src, c, f);
#pragma unroll
                                for (int i = 0; i < 8; ++i) acc[v][i] = fmaf(wj, f[i], acc[v][i]);
                            }
                        }
                    }
                    // then the rest: dropped, bad, zero, copy and const slots
                    for (int jj = 0; jj < nj; ++jj) {
                        const int k2 = s_kind[jj];
                        if (k2 == kRouted || k2 == kSkip) continue;
                        if (k2 == kBad) { nan_row = true; continue; }
                        const float wj = s_w[jj];
                        wkept += wj;
                        if (k2 == kZero) continue;
                        const int64_t off = s_off[jj];
                        float a1 = 0.0f, a2 = 0.0f;
                        if (k2 == kConst) {
                            a1 = load_as_float(ex.alpha1, YDT, off);
                            a2 = load_as_float(ex.alpha2, YDT, off);
                        }
#pragma unroll
                        for (int v = 0; v < V; ++v) {
                            const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                            if (c < ng) {
                                float f[8];
                                load8<YDT>(ex.ori_x, t * ng + c, f);
                                if (k2 == kConst) {
                                    float cv[8];
                                    load8<YDT>(ex.const_v, off * ng + c, cv);
#pragma unroll
                                    for (int i = 0; i < 8; ++i) f[i] = a1 * f[i] + a2 * cv[i];
                                }
#pragma unroll
                                for (int i = 0; i < 8; ++i) acc[v][i] = fmaf(wj, f[i], acc[v][i]);
                            }
                        }
                    }
                }
            }
            if constexpr (EXTRAS) {
                if (ex.shared_x != nullptr && !nan_row) {
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                        if (c < ng) {
                            float f[8];
                            load8<YDT>(ex.shared_x, t * ng + c, f);
#pragma unroll
                            for (int i = 0; i < 8; ++i) acc[v][i] = fmaf(wkept, f[i], acc[v][i]);
                        }
                    }
                }
            }
            if (nan_row) {
#pragma unroll
                for (int v = 0; v < V; ++v)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[v][i] = __int_as_float(0x7fc00000);
            }
            if constexpr (!NORM) {
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                    if (c < ng) store8<YDT>(y, t * ng + c, acc[v]);
                }
            } else {
                // x = acc + residual, rounded to the activation dtype; sum of
                // squares of the rounded x
                float ss = 0.0f;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int64_t c = base + threadIdx.x + (int64_t)v * blockDim.x;
                    if (c < ng) {
                        float f[8];
                        load8<YDT>(residual, t * ng + c, f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[v][i] += f[i];
                        store8<YDT>(x_out, t * ng + c, acc[v]);
#pragma unroll
                        for (int i = 0; i < 8; ++i) ss = fmaf(acc[v][i], acc[v][i], ss);
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
                    if (c < ng) {
                        float gm[8];
                        load8_rt(gamma, gdt, c, gm);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[v][i] = acc[v][i] * r * gm[i];
                        store8<YDT>(y, t * ng + c, acc[v]);
                    }
                }
            }
        }
    }
}

template <int ODT, int YDT, bool NORM, bool EXTRAS>
cudaError_t launch_typed(const void *out_disp, const void *w, int wdt, const int32_t *row_of,
                         const void *residual, const void *gamma, int gdt, float eps,
                         int64_t T, int top_k, int64_t H, void *y, void *x_out, float *rstd,
                         const CombineExtras &ex, cudaStream_t s)
{
    const int64_t ng = H / 8;
    int V = 1;
    while (V < kMaxV && ng > (int64_t)V * kMaxThreads) V *= 2;
    int64_t threads = (ng + V - 1) / V;
    threads = (threads + 31) / 32 * 32;
    if (threads > kMaxThreads) threads = kMaxThreads;
    if (threads < 32) threads = 32;
    int64_t blocks = T;
    const int64_t cap = (int64_t)device_sm_count() * 32;
    if (blocks > cap) blocks = cap;
#define MOE_COMBINE_LAUNCH(VV)                                                             \
    return launch_pdl(combine_kernel<ODT, YDT, VV, NORM, EXTRAS>, dim3((unsigned)blocks),   \
                      dim3((unsigned)threads), 0, s, out_disp, w, wdt, row_of, residual,    \
                      gamma, gdt, eps, T, top_k, H, y, x_out, rstd, ex)
    switch (V) {
    case 1: MOE_COMBINE_LAUNCH(1);
    case 2: MOE_COMBINE_LAUNCH(2);
    case 4: MOE_COMBINE_LAUNCH(4);
    default: MOE_COMBINE_LAUNCH(8);
    }
#undef MOE_COMBINE_LAUNCH
}

template <bool NORM, bool EXTRAS>
cudaError_t launch_norm(const void *out_disp, int odt, const void *w, int wdt,
                        const int32_t *row_of, const void *residual, const void *gamma,
                        int gdt, float eps, int64_t T, int top_k, int64_t H, void *y, int ydt,
                        void *x_out, float *rstd, const CombineExtras &ex, cudaStream_t s)
{
#define MOE_TYPED(O, Y)                                                                     \
    return launch_typed<O, Y, NORM, EXTRAS>(out_disp, w, wdt, row_of, residual, gamma, gdt, \
                                            eps, T, top_k, H, y, x_out, rstd, ex, s)
    if (ydt == DT_F32) MOE_TYPED(DT_F32, DT_F32);
    if (ydt == DT_BF16) {
        if (odt == DT_F32) MOE_TYPED(DT_F32, DT_BF16);
        MOE_TYPED(DT_BF16, DT_BF16);
    }
    if (odt == DT_F32) MOE_TYPED(DT_F32, DT_F16);
    MOE_TYPED(DT_F16, DT_F16);
#undef MOE_TYPED
}

// Standalone RMSNorm: one CTA per row (grid-stride), the row in registers.
template <int XDT, int V>
__global__ void __launch_bounds__(kMaxThreads)
rmsnorm_kernel(const void *__restrict__ x, const void *__restrict__ gamma, int gdt, float eps,
               int64_t rows, int64_t H, void *__restrict__ y, float *__restrict__ rstd)
{
    const int64_t ng = H / 8;
    __shared__ float red[kMaxThreads / 32];
    __shared__ float s_rstd;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = blockIdx.x; t < rows; t += gridDim.x) {
        float f[V][8];
        float ss = 0.0f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int64_t c = threadIdx.x + (int64_t)v * blockDim.x;
            if (c < ng) {
                load8<XDT>(x, t * ng + c, f[v]);
#pragma unroll
                for (int i = 0; i < 8; ++i) ss = fmaf(f[v][i], f[v][i], ss);
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
            if (rstd != nullptr) rstd[t] = r;
        }
        __syncthreads();
        const float r = s_rstd;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int64_t c = threadIdx.x + (int64_t)v * blockDim.x;
            if (c < ng) {
                float gm[8];
                load8_rt(gamma, gdt, c, gm);
#pragma unroll
                for (int i = 0; i < 8; ++i) f[v][i] = f[v][i] * r * gm[i];
                store8<XDT>(y, t * ng + c, f[v]);
            }
        }
        __syncthreads();     // red / s_rstd are reused by the next row
    }
}

template <int XDT>
cudaError_t launch_rmsnorm_dt(const void *x, const void *gamma, int gdt, float eps, int64_t rows,
                              int64_t H, void *y, float *rstd, cudaStream_t s)
{
    const int64_t ng = H / 8;
    int V = 1;
    while (V < kMaxV && ng > (int64_t)V * kMaxThreads) V *= 2;
    int64_t threads = (ng + V - 1) / V;
    threads = (threads + 31) / 32 * 32;
    if (threads > kMaxThreads) threads = kMaxThreads;
    if (threads < 32) threads = 32;
    int64_t blocks = rows;
    const int64_t cap = (int64_t)device_sm_count() * 32;
    if (blocks > cap) blocks = cap;
#define MOE_RMS(VV)                                                                        \
    return launch_pdl(rmsnorm_kernel<XDT, VV>, dim3((unsigned)blocks), dim3((unsigned)threads), \
                      0, s, x, gamma, gdt, eps, rows, H, y, rstd)
    switch (V) {
    case 1: MOE_RMS(1);
    case 2: MOE_RMS(2);
    case 4: MOE_RMS(4);
    default: MOE_RMS(8);
    }
#undef MOE_RMS
}

// y = y_acc (FP32) rounded to YDT, 8 elements per thread and step.
template <int YDT>
__global__ void __launch_bounds__(256)
finalize_kernel(const float *__restrict__ y_acc, int64_t groups, void *__restrict__ y)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < groups; g += stride) {
        float f[8];
        load8<DT_F32>(y_acc, g, f);
        store8<YDT>(y, g, f);
    }
}

}  // namespace

cudaError_t launch_finalize(const float *y_acc, int64_t T, int64_t H, void *y, int ydt,
                            cudaStream_t s)
{
    const int64_t groups = T * H / 8;
    if (groups == 0) return cudaSuccess;
    int64_t blocks = (groups + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (ydt == DT_BF16)
        return launch_pdl(finalize_kernel<DT_BF16>, dim3((unsigned)blocks), dim3(256), 0, s,
                          y_acc, groups, y);
    if (ydt == DT_F16)
        return launch_pdl(finalize_kernel<DT_F16>, dim3((unsigned)blocks), dim3(256), 0, s,
                          y_acc, groups, y);
    return launch_pdl(finalize_kernel<DT_F32>, dim3((unsigned)blocks), dim3(256), 0, s, y_acc,
                      groups, y);
}

// With the norm the whole row must fit one pass: 8 groups x 256 threads.
int combine_max_h(bool norm)
{
    if (!norm) return 1 << 30;
    return kMaxV * kMaxThreads * 8;
}

cudaError_t launch_combine(const void *out_disp, int odt, const void *w, int wdt,
                           const int32_t *row_of, const void *residual,
                           const void *gamma, int gdt, float eps, int64_t T,
                           int top_k, int64_t H, void *y, int ydt, void *x_out,
                           float *rstd, cudaStream_t s, const CombineExtras *ex)
{
    if (T == 0) return cudaSuccess;
    const CombineExtras none{};
    if (ex != nullptr) {
        if (residual != nullptr)
            return launch_norm<true, true>(out_disp, odt, w, wdt, row_of, residual, gamma, gdt,
                                           eps, T, top_k, H, y, ydt, x_out, rstd, *ex, s);
        return launch_norm<false, true>(out_disp, odt, w, wdt, row_of, residual, gamma, gdt, eps,
                                        T, top_k, H, y, ydt, x_out, rstd, *ex, s);
    }
    if (residual != nullptr)
        return launch_norm<true, false>(out_disp, odt, w, wdt, row_of, residual, gamma, gdt, eps,
                                        T, top_k, H, y, ydt, x_out, rstd, none, s);
    return launch_norm<false, false>(out_disp, odt, w, wdt, row_of, residual, gamma, gdt, eps, T,
                                     top_k, H, y, ydt, x_out, rstd, none, s);
}

cudaError_t launch_rmsnorm(const void *x, int xdt, const void *gamma, int gdt, float eps,
                           int64_t rows, int64_t H, void *y, float *rstd, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    if (xdt == DT_BF16) return launch_rmsnorm_dt<DT_BF16>(x, gamma, gdt, eps, rows, H, y, rstd, s);
    if (xdt == DT_F16) return launch_rmsnorm_dt<DT_F16>(x, gamma, gdt, eps, rows, H, y, rstd, s);
    return launch_rmsnorm_dt<DT_F32>(x, gamma, gdt, eps, rows, H, y, rstd, s);
}

}  // namespace moe
