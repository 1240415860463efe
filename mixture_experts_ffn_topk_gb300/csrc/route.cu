// route.cu -- softmax top-k routing, one warp per token.
//
// ruDNN user guide, section 4 "Routing contract": FP32 softmax over all E
// experts before top-k; ties favour the lower expert id; optional
// renormalisation, then a cast to the logits dtype; rows holding NaN, +inf or
// only -inf keep NaN weights.
//
// Each lane keeps EPL = ceil(E/32) logits in registers (expert e lives in lane
// e % 32, slot e / 32). The softmax max and sum are warp reductions. The k
// selections are k rounds of a warp-wide argmax over (logit desc, id asc):
// ranking by the FP32 logit is ranking by the exact softmax, and it makes the
// chosen ids independent of exp rounding. Weights are summed in slot order.
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRouteThreads = 256;

// true if candidate (la, ea) ranks before (lb, eb); ea/eb == INT_MAX is "none".
__device__ __forceinline__ bool ranks_before(float la, int ea, float lb, int eb)
{
    if (ea == INT_MAX) return false;
    if (eb == INT_MAX) return true;
    return la > lb || (la == lb && ea < eb);
}

template <int EPL, int LDT>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const void *__restrict__ logits, int64_t T, int E, int top_k,
             int renormalize, uint32_t *__restrict__ idx_out,
             void *__restrict__ w_out)
{
    using ET = typename Elem<LDT>::T;
    const ET *L = static_cast<const ET *>(logits);
    ET *W = static_cast<ET *>(w_out);
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    pdl_wait();
    pdl_launch_dependents();

    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
         t < T; t += warps) {
        float l[EPL];
        unsigned avail = 0;  // bit i: expert lane + 32 i exists, not yet taken
        bool bad = false, all_ninf = true;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane + 32 * i;
            l[i] = -INFINITY;
            if (e < E) {
                l[i] = Elem<LDT>::to_f(L[t * E + e]);
                avail |= 1u << i;
                bad |= isnan(l[i]) || l[i] == INFINITY;
                all_ninf &= (l[i] == -INFINITY);
            }
        }
        bad = __any_sync(kFull, bad);
        all_ninf = __all_sync(kFull, all_ninf);
        if (bad || all_ninf) {
            for (int j = lane; j < top_k; j += 32) {
                idx_out[t * top_k + j] = (uint32_t)j;
                W[t * top_k + j] = Elem<LDT>::from_f(__int_as_float(0x7fc00000));
            }
            continue;
        }

        // FP32 softmax statistics over all E experts.
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (avail >> i & 1u) m = fmaxf(m, l[i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (avail >> i & 1u) s += expf(l[i] - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);

        // k rounds of warp argmax. Slot j of the output lives in lane j % 32,
        // register j / 32.
        int sel_e[EPL];
        float sel_p[EPL];
#pragma unroll
        for (int i = 0; i < EPL; ++i) { sel_e[i] = 0; sel_p[i] = 0.0f; }
        float z = 0.0f;
        for (int j = 0; j < top_k; ++j) {
            float bl = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if ((avail >> i & 1u) && (be == INT_MAX || l[i] > bl)) {
                    bl = l[i];
                    be = lane + 32 * i;
                }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ol = __shfl_xor_sync(kFull, bl, o);
                const int oe = __shfl_xor_sync(kFull, be, o);
                if (ranks_before(ol, oe, bl, be)) { bl = ol; be = oe; }
            }
            const int owner = be & 31, slot = be >> 5;
            float mine = 0.0f;
            if (lane == owner) {
                avail &= ~(1u << slot);
                mine = expf(bl - m) / s;
            }
            const float p = __shfl_sync(kFull, mine, owner);
            z += p;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if ((j >> 5) == i && (j & 31) == lane) { sel_e[i] = be; sel_p[i] = p; }
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int j = lane + 32 * i;
            if (j < top_k) {
                idx_out[t * top_k + j] = (uint32_t)sel_e[i];
                const float w = renormalize ? sel_p[i] / z : sel_p[i];
                W[t * top_k + j] = Elem<LDT>::from_f(w);
            }
        }
    }
}

template <int LDT>
cudaError_t launch_route_dt(const void *logits, int64_t T, int E, int top_k,
                            int renorm, uint32_t *idx, void *w, cudaStream_t s)
{
    const int warps_per_block = kRouteThreads / 32;
    int64_t blocks = (T + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid((unsigned)blocks), block(kRouteThreads);
    const int epl = (E + 31) / 32;
    if (epl <= 1) return launch_pdl(route_kernel<1, LDT>, grid, block, 0, s, logits, T, E, top_k, renorm, idx, w);
    else if (epl <= 2) return launch_pdl(route_kernel<2, LDT>, grid, block, 0, s, logits, T, E, top_k, renorm, idx, w);
    else if (epl <= 4) return launch_pdl(route_kernel<4, LDT>, grid, block, 0, s, logits, T, E, top_k, renorm, idx, w);
    else if (epl <= 8) return launch_pdl(route_kernel<8, LDT>, grid, block, 0, s, logits, T, E, top_k, renorm, idx, w);
    else if (epl <= 16) return launch_pdl(route_kernel<16, LDT>, grid, block, 0, s, logits, T, E, top_k, renorm, idx, w);
    return launch_pdl(route_kernel<32, LDT>, grid, block, 0, s, logits, T, E, top_k, renorm, idx, w);
}

}  // namespace

cudaError_t launch_route(const void *logits, int ldt, int64_t T, int E,
                         int top_k, int renormalize, uint32_t *idx, void *w,
                         cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    switch (ldt) {
    case DT_F32: return launch_route_dt<DT_F32>(logits, T, E, top_k, renormalize, idx, w, s);
    case DT_BF16: return launch_route_dt<DT_BF16>(logits, T, E, top_k, renormalize, idx, w, s);
    default: return launch_route_dt<DT_F16>(logits, T, E, top_k, renormalize, idx, w, s);
    }
}

}  // namespace moe
