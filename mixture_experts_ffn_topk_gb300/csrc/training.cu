// training.cu -- the memory-bound steps of first-order MoE training.
//
// ruDNN user guide, section 12 "MoE first-order training":
//   * router weights of a fixed selection (selected_router_weights) and their
//     logits gradient (selected_router_backward): softmax or sigmoid scoring,
//     optional renormalisation of the selected weights, a finite positive
//     scale; repeated ids act as a gather; an id outside [0, E) makes the
//     whole row NaN without reading out of bounds; no derivative through the
//     selection itself;
//   * combine backward: the expert-output gradient (the routing weight times
//     the output gradient) and the FP32 routing-weight gradient (a dot product
//     of the output gradient with the expert's output row);
//   * dispatch backward: every token sums the gradient rows of its k
//     dispatched copies, without the routing weight (the combine backward has
//     applied it already).
// All three are warp-per-unit kernels on 16-byte vectors; arithmetic in FP32.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kMaxSlots = 64;              // top_k limit of the training calls

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Slot index as a signed 64-bit id: U32 zero-extends, I32 sign-extends.
__device__ __forceinline__ int64_t load_index(const void *p, int idt, int64_t i)
{
    if (idt == IDX_U32) return (int64_t) static_cast<const uint32_t *>(p)[i];
    if (idt == IDX_I32) return (int64_t) static_cast<const int32_t *>(p)[i];
    return static_cast<const int64_t *>(p)[i];
}

// One warp per token. Lane l holds the logits of experts l, l+32, ... (EPL
// of them) and slots l and l+32 of the selection. BWD = false writes the
// FP32 weights; BWD = true writes the logits gradient for the upstream
// weight gradient gw.
template <int LDT, int EPL, bool BWD>
__global__ void __launch_bounds__(32 * kWarpsPerCta)
router_train_kernel(const void *__restrict__ logits, int64_t T, int E,
                    const void *__restrict__ idx, int idt, int k, int sigmoid, int renorm,
                    float scale, const float *__restrict__ gw, float *__restrict__ w_out,
                    void *__restrict__ dl_out, unsigned *status)
{
    using L = Elem<LDT>;
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    for (int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); t < T; t += nwarps) {
        const typename L::T *lrow = static_cast<const typename L::T *>(logits) + t * E;
        float l[EPL];
        bool bad = false, all_ninf = true;
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            l[i] = e < E ? L::to_f(lrow[e]) : -INFINITY;
            if (e < E) {
                bad |= isnan(l[i]) || l[i] == INFINITY;
                all_ninf &= l[i] == -INFINITY;
                m = fmaxf(m, l[i]);
            }
        }
        m = warp_max(m);
        float ssum = 0.0f;
        if (!sigmoid) {
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if (lane + 32 * i < E) ssum += expf(l[i] - m);
            ssum = warp_sum(ssum);
        }
        // the two slots of this lane
        int64_t ej[2] = {0, 0};
        bool live[2] = {lane < k, lane + 32 < k};
        bool id_bad = false;
#pragma unroll
        for (int s = 0; s < 2; ++s)
            if (live[s]) {
                ej[s] = load_index(idx, idt, t * k + lane + 32 * s);
                id_bad |= ej[s] < 0 || ej[s] >= E;
            }
        id_bad = __any_sync(0xffffffffu, id_bad);
        const bool row_bad = id_bad || (!sigmoid && __any_sync(0xffffffffu, bad)) ||
                             (!sigmoid && __all_sync(0xffffffffu, all_ninf));
        if (id_bad && lane == 0) atomicOr(status, ST_BAD_INDEX);
        if (row_bad) {
            if constexpr (!BWD) {
#pragma unroll
                for (int s = 0; s < 2; ++s)
                    if (live[s]) w_out[t * k + lane + 32 * s] = __int_as_float(0x7fc00000);
            } else {
                typename L::T *drow = static_cast<typename L::T *>(dl_out) + t * E;
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (lane + 32 * i < E) drow[lane + 32 * i] = L::from_f(__int_as_float(0x7fc00000));
            }
            continue;
        }
        // scores of this lane's slots (the selected logit is re-read; the row
        // was just loaded, so it comes from L1)
        float sc[2] = {0.0f, 0.0f};
#pragma unroll
        for (int s = 0; s < 2; ++s)
            if (live[s]) {
                const float x = L::to_f(lrow[ej[s]]);
                sc[s] = sigmoid ? 1.0f / (1.0f + expf(-x)) : expf(x - m) / ssum;
            }
        const float z = warp_sum(sc[0] + sc[1]);
        if constexpr (!BWD) {
#pragma unroll
            for (int s = 0; s < 2; ++s)
                if (live[s]) w_out[t * k + lane + 32 * s] = (renorm ? sc[s] / z : sc[s]) * scale;
        } else {
            float g[2] = {0.0f, 0.0f};
#pragma unroll
            for (int s = 0; s < 2; ++s)
                if (live[s]) g[s] = gw[t * k + lane + 32 * s];
            float ds[2];
            if (renorm) {
                const float gbar = warp_sum(g[0] * sc[0] + g[1] * sc[1]) / z;
#pragma unroll
                for (int s = 0; s < 2; ++s) ds[s] = scale * (g[s] - gbar) / z;
            } else {
#pragma unroll
                for (int s = 0; s < 2; ++s) ds[s] = scale * g[s];
            }
            // G[e]: the slot gradients summed per expert (the gather's adjoint)
            float G[EPL];
            unsigned selmask = 0u;
#pragma unroll
            for (int i = 0; i < EPL; ++i) G[i] = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int src = j & 31, s = j >> 5;
                const int e = __shfl_sync(0xffffffffu, (int)(s ? ej[1] : ej[0]), src);
                const float d = __shfl_sync(0xffffffffu, s ? ds[1] : ds[0], src);
                if ((e & 31) == lane) {
#pragma unroll
                    for (int i = 0; i < EPL; ++i)
                        if (i == (e >> 5)) { G[i] += d; selmask |= 1u << i; }
                }
            }
            typename L::T *drow = static_cast<typename L::T *>(dl_out) + t * E;
            if (!sigmoid) {
                // c = sum_e p_e G_e = sum over slots of score * slot gradient
                const float c = warp_sum((live[0] ? sc[0] * ds[0] : 0.0f) +
                                         (live[1] ? sc[1] * ds[1] : 0.0f));
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (lane + 32 * i < E) {
                        const float p = expf(l[i] - m) / ssum;
                        drow[lane + 32 * i] = L::from_f(p * (G[i] - c));
                    }
            } else {
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (lane + 32 * i < E) {
                        float v = 0.0f;
                        if (selmask >> i & 1u) {
                            const float sg = 1.0f / (1.0f + expf(-l[i]));
                            v = G[i] * sg * (1.0f - sg);
                        }
                        drow[lane + 32 * i] = L::from_f(v);
                    }
            }
        }
    }
}

template <int LDT, bool BWD>
cudaError_t launch_router_ldt(const void *logits, int64_t T, int E, const void *idx, int idt,
                              int k, int sigmoid, int renorm, float scale, const float *gw,
                              float *w_out, void *dl_out, unsigned *status, cudaStream_t s)
{
    const int64_t ctas_needed = (T + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    const dim3 grid((unsigned)(ctas_needed < cap ? ctas_needed : cap)), block(32 * kWarpsPerCta);
    const int epl = (E + 31) / 32;
#define MOE_ROUTER_EPL(N)                                                                      \
    if (epl <= N)                                                                             \
        return launch_pdl(router_train_kernel<LDT, N, BWD>, grid, block, 0, s, logits, T, E, \
                          idx, idt, k, sigmoid, renorm, scale, gw, w_out, dl_out, status);
    MOE_ROUTER_EPL(1)
    MOE_ROUTER_EPL(2)
    MOE_ROUTER_EPL(4)
    MOE_ROUTER_EPL(8)
    MOE_ROUTER_EPL(16)
    MOE_ROUTER_EPL(32)
#undef MOE_ROUTER_EPL
    return cudaErrorInvalidValue;
}

template <bool BWD>
cudaError_t launch_router(const void *logits, int ldt, int64_t T, int E, const void *idx,
                          int idt, int k, int sigmoid, int renorm, float scale, const float *gw,
                          float *w_out, void *dl_out, unsigned *status, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    if (ldt == DT_F32)
        return launch_router_ldt<DT_F32, BWD>(logits, T, E, idx, idt, k, sigmoid, renorm, scale,
                                              gw, w_out, dl_out, status, s);
    if (ldt == DT_BF16)
        return launch_router_ldt<DT_BF16, BWD>(logits, T, E, idx, idt, k, sigmoid, renorm,
                                               scale, gw, w_out, dl_out, status, s);
    return launch_router_ldt<DT_F16, BWD>(logits, T, E, idx, idt, k, sigmoid, renorm, scale, gw,
                                          w_out, dl_out, status, s);
}

// Eight consecutive elements of a row as floats / back to the row's dtype.
template <int DT>
__device__ __forceinline__ void load8(const void *row, int64_t col, float (&v)[8])
{
    if constexpr (DT == DT_F32) {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(row) + col);
        const float4 a = p[0], b = p[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        Vec16 q;
        q.u = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(row) + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = DT == DT_BF16 ? bf16x2_to_float2(q.w[i]) : f16x2_to_float2(q.w[i]);
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

template <int DT>
__device__ __forceinline__ void store8(void *row, int64_t col, const float (&v)[8])
{
    if constexpr (DT == DT_F32) {
        float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(row) + col);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        Vec16 q;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            q.w[i] = DT == DT_BF16 ? float2_to_bf16x2(v[2 * i], v[2 * i + 1])
                                   : float2_to_f16x2(v[2 * i], v[2 * i + 1]);
        *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(row) + col) = q.u;
    }
}

// One warp per assignment a = t*k + j:
//   dexp[row_of[a]] = w[a] * gy[t]   (dtype DT),   dw[a] = <gy[t], out[row_of[a]]>.
// A slot with no row writes no dexp row and gets dw = NaN.
template <int DT, int ODT>
__global__ void __launch_bounds__(32 * kWarpsPerCta)
combine_backward_kernel(const void *__restrict__ out_disp, const void *__restrict__ w, int wdt,
                        const int32_t *__restrict__ row_of, const void *__restrict__ gy,
                        int64_t A, int k, int64_t H, void *__restrict__ dexp,
                        float *__restrict__ dw)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    const int64_t ob = ODT == DT_F32 ? 4 : 2, eb = DT == DT_F32 ? 4 : 2;
    for (int64_t a = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); a < A; a += nwarps) {
        const int64_t r = row_of[a];
        if (r < 0 || r >= A) {             // no row (or none inside out_disp)
            if (lane == 0) dw[a] = __int_as_float(0x7fc00000);
            continue;
        }
        const float wa = load_as_float(w, wdt, a);
        const int64_t t = a / k;
        const uint8_t *grow = static_cast<const uint8_t *>(gy) + t * H * eb;
        const uint8_t *orow = static_cast<const uint8_t *>(out_disp) + r * H * ob;
        uint8_t *drow = static_cast<uint8_t *>(dexp) + r * H * eb;
        float acc = 0.0f;
        for (int64_t c = (int64_t)lane * 8; c < H; c += 256) {
            float g[8], o[8], d[8];
            load8<DT>(grow, c, g);
            load8<ODT>(orow, c, o);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc = fmaf(g[i], o[i], acc);
                d[i] = wa * g[i];
            }
            store8<DT>(drow, c, d);
        }
        acc = warp_sum(acc);
        if (lane == 0) dw[a] = acc;
    }
    pdl_launch_dependents();
}

// One warp per token: dx[t] = sum over slots j of d[row_of[t*k + j]] (FP32
// sum in slot order, rounded once); slots with no row add nothing.
template <int DT>
__global__ void __launch_bounds__(32 * kWarpsPerCta)
dispatch_backward_kernel(const void *__restrict__ d, const int32_t *__restrict__ row_of,
                         int64_t T, int k, int64_t H, void *__restrict__ dx)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerCta;
    const int64_t eb = DT == DT_F32 ? 4 : 2;
    for (int64_t t = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5); t < T; t += nwarps) {
        uint8_t *xrow = static_cast<uint8_t *>(dx) + t * H * eb;
        // every lane runs every round (the shuffles need the whole warp);
        // lanes past the row's end only skip the loads and the store
        for (int64_t c0 = 0; c0 < H; c0 += 256) {
            const int64_t c = c0 + (int64_t)lane * 8;
            const bool on = c < H;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j0 = 0; j0 < k; j0 += 32) {
                const int rj = j0 + lane < k ? row_of[t * k + j0 + lane] : -1;
                const int n = k - j0 < 32 ? k - j0 : 32;
                for (int j = 0; j < n; ++j) {
                    const int64_t r = __shfl_sync(0xffffffffu, rj, j);
                    if (r < 0 || r >= T * k || !on) continue;
                    float v[8];
                    load8<DT>(static_cast<const uint8_t *>(d) + r * H * eb, c, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] += v[i];
                }
            }
            if (on) store8<DT>(xrow, c, acc);
        }
    }
    pdl_launch_dependents();
}

dim3 warp_grid(int64_t units)
{
    const int64_t ctas = (units + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    return dim3((unsigned)(ctas < cap ? ctas : cap));
}

}  // namespace

int router_train_max_top_k() { return kMaxSlots; }

cudaError_t launch_router_weights(const void *logits, int ldt, int64_t T, int E, const void *idx,
                                  int idt, int k, int sigmoid, int renorm, float scale,
                                  float *w_out, unsigned *status, cudaStream_t s)
{
    return launch_router<false>(logits, ldt, T, E, idx, idt, k, sigmoid, renorm, scale, nullptr,
                                w_out, nullptr, status, s);
}

cudaError_t launch_router_backward(const void *logits, int ldt, int64_t T, int E,
                                   const void *idx, int idt, int k, const float *gw,
                                   int sigmoid, int renorm, float scale, void *dl_out,
                                   unsigned *status, cudaStream_t s)
{
    return launch_router<true>(logits, ldt, T, E, idx, idt, k, sigmoid, renorm, scale, gw,
                               nullptr, dl_out, status, s);
}

cudaError_t launch_combine_backward(const void *out_disp, int odt, const void *w, int wdt,
                                    const int32_t *row_of, const void *gy, int dt, int64_t T,
                                    int k, int64_t H, void *dexp, float *dw, cudaStream_t s)
{
    const int64_t A = T * k;
    if (A == 0) return cudaSuccess;
    const dim3 grid = warp_grid(A), block(32 * kWarpsPerCta);
#define MOE_CB(D, O)                                                                        \
    if (dt == D && odt == O)                                                                \
        return launch_pdl(combine_backward_kernel<D, O>, grid, block, 0, s, out_disp, w, wdt, \
                          row_of, gy, A, k, H, dexp, dw);
    MOE_CB(DT_F32, DT_F32)
    MOE_CB(DT_BF16, DT_BF16)
    MOE_CB(DT_BF16, DT_F32)
    MOE_CB(DT_F16, DT_F16)
    MOE_CB(DT_F16, DT_F32)
#undef MOE_CB
    return cudaErrorInvalidValue;
}

cudaError_t launch_dispatch_backward(const void *d, int dt, const int32_t *row_of, int64_t T,
                                     int k, int64_t H, void *dx, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const dim3 grid = warp_grid(T), block(32 * kWarpsPerCta);
    if (dt == DT_F32)
        return launch_pdl(dispatch_backward_kernel<DT_F32>, grid, block, 0, s, d, row_of, T, k, H, dx);
    if (dt == DT_BF16)
        return launch_pdl(dispatch_backward_kernel<DT_BF16>, grid, block, 0, s, d, row_of, T, k, H, dx);
    return launch_pdl(dispatch_backward_kernel<DT_F16>, grid, block, 0, s, d, row_of, T, k, H, dx);
}

}  // namespace moe
