// route_sigmoid.cu -- group-limited sigmoid routing, one warp per token.
//
// ruDNN user guide, section 10 "Group-limited sigmoid MoE routing": per token
// the scores are s_e = sigmoid(l_e); an optional FP32 correction bias gives
// the selection scores c_e = s_e + bias_e (the bias steers the selection
// only); the E experts form `groups` groups of E/groups consecutive experts,
// each scored by its best c (or the sum of its two best with group_top_two);
// the `selected_groups` best groups are kept and top_k experts are picked by
// c inside them; equal scores favour the lower id (groups and experts alike);
// the weights are the raw scores s of the picks, divided by their sum in
// slot order when renormalize is set, times `scale`, cast to the logits
// dtype. A row whose corrected scores hold a NaN gets ids 0..k-1 and NaN
// weights, as in the softmax contract.
//
// Scores are FP32, each the sigmoid evaluated in double and rounded once to
// FP32: 1 / (1 + exp(-l)) with l widened exactly. The double result lies
// within a few double ulps of the exact sigmoid, so its one rounding to FP32
// gives the correctly rounded score except when the exact value sits within
// that distance of an FP32 rounding boundary (about 2^-28 of inputs); every
// selection decision therefore compares the same FP32 values as any other
// implementation that rounds the sigmoid once. T * E double evaluations per
// call are a negligible load at GB300's FP64 rate for the routing shapes.
//
// Lane r holds experts r*EPL .. r*EPL+EPL-1 in registers and their corrected
// scores in a per-warp shared-memory row, from which lanes score the groups
// (lane g takes groups g, g+32, g+64, g+96). Group and expert picks are
// rounds of a warp argmax on (score desc, id asc).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kSgWarps = 8;            // tokens (warps) per block
constexpr int kSgMaxTopK = 64;
constexpr int kSgMaxGroups = 128;

// true if (a, ia) ranks before (b, ib); an id < 0 is "none"
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib)
{
    if (ia < 0) return false;
    if (ib < 0) return true;
    return a > b || (a == b && ia < ib);
}

__device__ __forceinline__ void warp_argmax(float &v, int &i)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, v, o);
        const int oi = __shfl_xor_sync(kFull, i, o);
        if (ranks_before(ov, oi, v, i)) { v = ov; i = oi; }
    }
}

template <int EPL, int LDT>
__global__ void __launch_bounds__(kSgWarps * 32)
route_sigmoid_grouped_kernel(const void *__restrict__ logits, int64_t T, int E,
                             const float *__restrict__ bias, int top_k, int groups,
                             int selected_groups, int group_top_two, int renormalize,
                             float scale, uint32_t *__restrict__ idx_out,
                             void *__restrict__ w_out)
{
    using ET = typename Elem<LDT>::T;
    const ET *L = static_cast<const ET *>(logits);
    ET *W = static_cast<ET *>(w_out);
    extern __shared__ float sg_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *cs = sg_smem + (size_t)warp * (E + kSgMaxTopK);   // corrected scores [E]
    float *pw = cs + E;                                       // picked scores [top_k]
    const int gs = E / groups;
    const bool all_groups = selected_groups == groups;
    pdl_wait();
    pdl_launch_dependents();

    float b[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
        const int e = lane * EPL + i;
        b[i] = (bias != nullptr && e < E) ? bias[e] : 0.0f;
    }

    for (int64_t t = (int64_t)blockIdx.x * kSgWarps + warp; t < T;
         t += (int64_t)gridDim.x * kSgWarps) {
        float s[EPL], c[EPL];
        int nan = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane * EPL + i;
            s[i] = 0.0f;
            c[i] = -INFINITY;
            if (e < E) {
                const float l = Elem<LDT>::to_f(L[t * E + e]);
                s[i] = (float)(1.0 / (1.0 + exp(-(double)l)));
                c[i] = s[i] + b[i];
                nan |= isnan(c[i]);
                cs[e] = c[i];
            }
        }
        const bool invalid = __any_sync(kFull, nan);
        __syncwarp();

        // kept groups as a 128-bit mask, the same in every lane
        uint32_t keep[4] = {~0u, ~0u, ~0u, ~0u};
        if (!all_groups) {
            float gv[4];
            int gid[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int g = lane + 32 * m;
                gid[m] = -1;
                gv[m] = -INFINITY;
                if (g < groups) {
                    float first = -INFINITY, second = -INFINITY;
                    for (int e = g * gs; e < (g + 1) * gs; ++e) {
                        const float v = cs[e];
                        if (v > first) { second = first; first = v; }
                        else if (v > second) second = v;
                    }
                    gv[m] = group_top_two ? first + second : first;
                    gid[m] = g;
                }
            }
            keep[0] = keep[1] = keep[2] = keep[3] = 0u;
            for (int n = 0; n < selected_groups; ++n) {
                float bv = -INFINITY;
                int bi = -1;
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (ranks_before(gv[m], gid[m], bv, bi)) { bv = gv[m]; bi = gid[m]; }
                warp_argmax(bv, bi);
                if (bi < 0) break;                 // cannot happen for valid limits
                keep[bi >> 5] |= 1u << (bi & 31);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (gid[m] == bi) gid[m] = -1;  // taken
            }
        }

        uint32_t avail = 0;                        // bit i: expert lane*EPL+i is a candidate
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
            const int e = lane * EPL + i;
            if (e < E) {
                const int g = e / gs;
                if (keep[g >> 5] >> (g & 31) & 1u) avail |= 1u << i;
            }
        }

        float z = 0.0f;
        for (int j = 0; j < top_k; ++j) {
            float bv = -INFINITY;
            int bi = -1;
#pragma unroll
            for (int i = 0; i < EPL; ++i)
                if ((avail >> i & 1u) && ranks_before(c[i], lane * EPL + i, bv, bi)) {
                    bv = c[i];
                    bi = lane * EPL + i;
                }
            warp_argmax(bv, bi);
            const int win = bi < 0 ? 0 : bi;       // invalid rows are replaced below
            const int owner = win / EPL, slot = win % EPL;
            float mine = 0.0f;
            if (lane == owner) {
                avail &= ~(1u << slot);
#pragma unroll
                for (int i = 0; i < EPL; ++i)
                    if (i == slot) mine = s[i];
            }
            const float p = __shfl_sync(kFull, mine, owner);
            z += p;
            if (lane == (j & 31)) {
                pw[j] = p;
                if (!invalid) idx_out[t * top_k + j] = (uint32_t)win;
            }
        }
        __syncwarp();
        for (int j = lane; j < top_k; j += 32) {
            if (invalid) {
                idx_out[t * top_k + j] = (uint32_t)j;
                W[t * top_k + j] = Elem<LDT>::from_f(__int_as_float(0x7fc00000));
            } else {
                const float w = renormalize ? pw[j] / z : pw[j];
                W[t * top_k + j] = Elem<LDT>::from_f(w * scale);
            }
        }
        __syncwarp();                              // cs and pw are reused by the next token
    }
}

template <int EPL, int LDT>
cudaError_t launch_sg_cfg(const void *logits, int64_t T, int E, const float *bias, int top_k,
                          int groups, int selected, int top_two, int renorm, float scale,
                          uint32_t *idx, void *w, cudaStream_t s)
{
    int64_t blocks = (T + kSgWarps - 1) / kSgWarps;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    const size_t smem = (size_t)kSgWarps * (E + kSgMaxTopK) * sizeof(float);
    return launch_pdl(route_sigmoid_grouped_kernel<EPL, LDT>, dim3((unsigned)blocks),
                      dim3(kSgWarps * 32), smem, s, logits, T, E, bias, top_k, groups, selected,
                      top_two, renorm, scale, idx, w);
}

template <int LDT>
cudaError_t launch_sg_dt(const void *logits, int64_t T, int E, const float *bias, int top_k,
                         int groups, int selected, int top_two, int renorm, float scale,
                         uint32_t *idx, void *w, cudaStream_t s)
{
#define MOE_SG(EPL)                                                                            \
    return launch_sg_cfg<EPL, LDT>(logits, T, E, bias, top_k, groups, selected, top_two,      \
                                   renorm, scale, idx, w, s)
    if (E <= 32) MOE_SG(1);
    if (E <= 64) MOE_SG(2);
    if (E <= 128) MOE_SG(4);
    if (E <= 256) MOE_SG(8);
    if (E <= 512) MOE_SG(16);
    MOE_SG(32);
#undef MOE_SG
}

}  // namespace

int sigmoid_route_max_top_k() { return kSgMaxTopK; }
int sigmoid_route_max_groups() { return kSgMaxGroups; }

cudaError_t launch_route_sigmoid_grouped(const void *logits, int ldt, int64_t T, int E,
                                         const float *bias, int top_k, int groups,
                                         int selected_groups, int group_top_two,
                                         int renormalize, float scale, uint32_t *idx, void *w,
                                         cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    switch (ldt) {
    case DT_F32:
        return launch_sg_dt<DT_F32>(logits, T, E, bias, top_k, groups, selected_groups,
                                    group_top_two, renormalize, scale, idx, w, s);
    case DT_BF16:
        return launch_sg_dt<DT_BF16>(logits, T, E, bias, top_k, groups, selected_groups,
                                     group_top_two, renormalize, scale, idx, w, s);
    default:
        return launch_sg_dt<DT_F16>(logits, T, E, bias, top_k, groups, selected_groups,
                                    group_top_two, renormalize, scale, idx, w, s);
    }
}

}  // namespace moe
