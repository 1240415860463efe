// route.cu -- softmax top-k routing, one warp per token.
//
// ruDNN user guide, section 4 "Routing contract": FP32 softmax over all E
// experts before top-k; ties favour the lower expert id; optional
// renormalisation, then a cast to the logits dtype; rows holding NaN, +inf or
// only -inf keep NaN weights.
//
// Two kernels. At large T (E <= 64, top_k <= 8) one thread routes one token:
// the E logits sit in its registers, each of the k selections is a scan for
// the first maximum (so among equal logits the lower id wins), and the k
// weights stay in registers until their slot-order sum is known -- no
// communication between lanes, the fewest instructions per token. Below that
// T, too few threads would be in flight, and a group of lanes shares a token:
//
// A group of G lanes (G = 1..32, a power of two) routes one token, so a warp
// routes 32/G tokens at once; lane r of a group holds logits r*EPL ..
// r*EPL+EPL-1 in registers (G*EPL >= E, EPL <= 32), so a group reads one
// contiguous row. The softmax max and sum are shuffle reductions inside the
// group. The k selections are k rounds of a group-wide argmax over
// (logit desc, id asc): ranking by the FP32 logit is ranking by the exact
// softmax, and it makes the chosen ids independent of exp rounding. Weights are
// summed in slot order. G is picked so that EPL <= 8 where E allows it.
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

// OR / AND / max / sum over the G lanes of a group (xor offsets < G stay in it).
template <int G>
__device__ __forceinline__ int group_or(int v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v |= __shfl_xor_sync(kFull, v, o);
    return v;
}
template <int G>
__device__ __forceinline__ int group_and(int v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v &= __shfl_xor_sync(kFull, v, o);
    return v;
}

template <int G, int EPL, int LDT>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const void *__restrict__ logits, int64_t T, int E, int top_k,
             int renormalize, uint32_t *__restrict__ idx_out,
             void *__restrict__ w_out)
{
    using ET = typename Elem<LDT>::T;
    const ET *L = static_cast<const ET *>(logits);
    ET *W = static_cast<ET *>(w_out);
    constexpr int TPW = 32 / G;                          // tokens per warp
    // per warp: TPW tokens x (G*EPL >= top_k) selected probabilities
    __shared__ float sp[kRouteThreads / 32][32 * EPL];
    const int lane = (int)lane_id();
    const int r = lane % G, gbase = lane - r;            // lane in group, group's first lane
    const int64_t slots = (int64_t)gridDim.x * (blockDim.x / 32) * TPW;
    pdl_wait();
    pdl_launch_dependents();

    // the loop is uniform across the warp: groups past T work on a clamped
    // token and store nothing, so every shuffle sees the full warp
    for (int64_t t0 = ((int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * TPW;
         t0 < T; t0 += slots) {
        const int64_t t_raw = t0 + lane / G;
        const bool live = t_raw < T;
        const int64_t t = live ? t_raw : T - 1;
        float l[EPL];
        unsigned avail = 0;  // bit i: expert r*EPL + i exists, not yet taken
        int bad = 0, all_ninf = 1;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = r * EPL + i;
            l[i] = -INFINITY;
            if (e < E) {
                l[i] = Elem<LDT>::to_f(L[t * E + e]);
                avail |= 1u << i;
                bad |= isnan(l[i]) || l[i] == INFINITY;
                all_ninf &= (l[i] == -INFINITY);
            }
        }
        // both group votes run on every lane: a short-circuit here would let
        // part of the warp skip a full-mask shuffle
        const int any_bad = group_or<G>(bad);
        const int every_ninf = group_and<G>(all_ninf);
        const bool invalid = any_bad || every_ninf;

        // FP32 softmax over all E experts: exp(l - max) once per expert (as
        // exp2 of the scaled difference), kept for the selected ones
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (avail >> i & 1u) m = fmaxf(m, l[i]);
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        constexpr float kLog2e = 1.4426950408889634f;
        float ex[EPL];
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            ex[i] = (avail >> i & 1u) ? exp2f((l[i] - m) * kLog2e) : 0.0f;
            s += ex[i];
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        const float inv_s = 1.0f / s;

        // k rounds of a group argmax; ids go straight to the output, the
        // selected probabilities wait in shared memory for their sum
        float *pw = sp[threadIdx.x / 32] + (lane / G) * (G * EPL);
        float z = 0.0f;
        for (int j = 0; j < top_k; ++j) {
            float bl = -INFINITY;
            int be = INT_MAX;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if ((avail >> i & 1u) && (be == INT_MAX || l[i] > bl)) {
                    bl = l[i];
                    be = r * EPL + i;
                }
#pragma unroll
            for (int o = G / 2; o > 0; o >>= 1) {
                const float ol = __shfl_xor_sync(kFull, bl, o);
                const int oe = __shfl_xor_sync(kFull, be, o);
                if (ranks_before(ol, oe, bl, be)) { bl = ol; be = oe; }
            }
            // an invalid row may have no candidate left; its results are
            // replaced below, so any in-range owner will do
            const int eb = be == INT_MAX ? 0 : be;
            const int owner = eb / EPL, slot = eb % EPL;
            float mine = 0.0f;
            if (r == owner) {
                avail &= ~(1u << slot);
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (i == slot) mine = ex[i] * inv_s;
            }
            const float p = __shfl_sync(kFull, mine, gbase + owner);
            z += p;
            if (r == j % G) {
                pw[j] = p;
                if (live && !invalid) idx_out[t * top_k + j] = (uint32_t)eb;
            }
        }
        __syncwarp();
        if (live) {
            for (int j = r; j < top_k; j += G) {
                if (invalid) {
                    idx_out[t * top_k + j] = (uint32_t)j;
                    W[t * top_k + j] = Elem<LDT>::from_f(__int_as_float(0x7fc00000));
                } else {
                    const float w = renormalize ? pw[j] / z : pw[j];
                    W[t * top_k + j] = Elem<LDT>::from_f(w);
                }
            }
        }
        __syncwarp();   // pw is reused by the next token of this group
    }
}

// ---- one thread per token ----------------------------------------------------

constexpr int kMaxThreadTopK = 8;

template <int EPL, int LDT>
__global__ void __launch_bounds__(kRouteThreads)
route_thread_kernel(const void *__restrict__ logits, int64_t T, int E, int top_k,
                    int renormalize, int vec_rows, uint32_t *__restrict__ idx_out,
                    void *__restrict__ w_out)
{
    using ET = typename Elem<LDT>::T;
    constexpr int VEC = 16 / (int)sizeof(ET);          // elements per 16-byte load
    static_assert(EPL % VEC == 0, "rows are read in 16-byte pieces");
    const ET *L = static_cast<const ET *>(logits);
    ET *W = static_cast<ET *>(w_out);
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x) {
        float l[EPL];
        const ET *row = L + t * E;
        if (vec_rows) {
            // E * sizeof(ET) is a multiple of 16 and the buffer 16-byte aligned
#pragma unroll
            for (int c = 0; c < EPL; c += VEC) {
                if (c < E) {
                    Vec16 v;
                    v.u = *reinterpret_cast<const uint4 *>(row + c);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        if constexpr (LDT == DT_F32) l[c + i] = v.f[i];
                        else {
                            const float2 f = LDT == DT_BF16 ? bf16x2_to_float2(v.w[i / 2])
                                                            : f16x2_to_float2(v.w[i / 2]);
                            l[c + i] = (i & 1) ? f.y : f.x;
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VEC; ++i) l[c + i] = -INFINITY;
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < EPL; ++i) l[i] = i < E ? Elem<LDT>::to_f(row[i]) : -INFINITY;
        }
        int bad = 0, all_ninf = 1;
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i < E) {
                bad |= isnan(l[i]) || l[i] == INFINITY;
                all_ninf &= (l[i] == -INFINITY);
                m = fmaxf(m, l[i]);
            }
        const bool invalid = bad || all_ninf;

        // FP32 softmax over all E experts, exp(l - max) as exp2 of the scaled
        // difference; the selected ones are recomputed below (same value)
        constexpr float kLog2e = 1.4426950408889634f;
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < EPL; ++i)
            if (i < E) s += exp2f((l[i] - m) * kLog2e);
        const float inv_s = 1.0f / s;

        uint64_t avail = E >= 64 ? ~0ull : ((1ull << E) - 1ull);
        float p[kMaxThreadTopK];
        int id[kMaxThreadTopK];
        float z = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxThreadTopK; ++j) {
            p[j] = 0.0f;
            id[j] = j;
            if (j < top_k) {
                float bl = -INFINITY;
                int be = -1;
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if ((avail >> i & 1ull) && (be < 0 || l[i] > bl)) {
                        bl = l[i];
                        be = i;
                    }
                if (be >= 0) {
                    avail &= ~(1ull << be);
                    id[j] = be;
                    p[j] = exp2f((bl - m) * kLog2e) * inv_s;
                    z += p[j];
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kMaxThreadTopK; ++j) {
            if (j < top_k) {
                if (invalid) {
                    idx_out[t * top_k + j] = (uint32_t)j;
                    W[t * top_k + j] = Elem<LDT>::from_f(__int_as_float(0x7fc00000));
                } else {
                    idx_out[t * top_k + j] = (uint32_t)id[j];
                    W[t * top_k + j] = Elem<LDT>::from_f(renormalize ? p[j] / z : p[j]);
                }
            }
        }
    }
}

template <int EPL, int LDT>
cudaError_t launch_route_thread(const void *logits, int64_t T, int E, int top_k, int renorm,
                                uint32_t *idx, void *w, cudaStream_t s)
{
    using ET = typename Elem<LDT>::T;
    const int vec_rows = ((int64_t)E * (int64_t)sizeof(ET)) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(logits) % 16 == 0;
    int64_t blocks = (T + kRouteThreads - 1) / kRouteThreads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(route_thread_kernel<EPL, LDT>, dim3((unsigned)blocks), dim3(kRouteThreads),
                      0, s, logits, T, E, top_k, renorm, vec_rows, idx, w);
}

// One thread per token once there are at least two warps of tokens per SM.
bool thread_route_fits(int64_t T, int E, int top_k)
{
    return E <= 64 && top_k <= kMaxThreadTopK && T >= (int64_t)device_sm_count() * 64;
}

template <int G, int EPL, int LDT>
cudaError_t launch_route_cfg(const void *logits, int64_t T, int E, int top_k, int renorm,
                             uint32_t *idx, void *w, cudaStream_t s)
{
    const int64_t tokens_per_block = (kRouteThreads / 32) * (32 / G);
    int64_t blocks = (T + tokens_per_block - 1) / tokens_per_block;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(route_kernel<G, EPL, LDT>, dim3((unsigned)blocks), dim3(kRouteThreads), 0,
                      s, logits, T, E, top_k, renorm, idx, w);
}

template <int LDT>
cudaError_t launch_route_dt(const void *logits, int64_t T, int E, int top_k,
                            int renorm, uint32_t *idx, void *w, cudaStream_t s)
{
    if (thread_route_fits(T, E, top_k)) {
        if (E <= 8) return launch_route_thread<8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
        if (E <= 16) return launch_route_thread<16, LDT>(logits, T, E, top_k, renorm, idx, w, s);
        if (E <= 32) return launch_route_thread<32, LDT>(logits, T, E, top_k, renorm, idx, w, s);
        return launch_route_thread<64, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    }
    if (E <= 8) return launch_route_cfg<1, 8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    if (E <= 16) return launch_route_cfg<2, 8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    if (E <= 32) return launch_route_cfg<4, 8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    if (E <= 64) return launch_route_cfg<8, 8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    if (E <= 128) return launch_route_cfg<16, 8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    if (E <= 256) return launch_route_cfg<32, 8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    if (E <= 512) return launch_route_cfg<32, 16, LDT>(logits, T, E, top_k, renorm, idx, w, s);
    return launch_route_cfg<32, 32, LDT>(logits, T, E, top_k, renorm, idx, w, s);
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
