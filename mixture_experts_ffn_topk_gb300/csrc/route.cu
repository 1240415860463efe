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

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kRouteThreads = 256;
// fused kernel: enough warps for one pass over a chunk's tokens (its
// per-warp probability rows stay within 32 KiB of static shared memory)
template <int EPL>
__host__ __device__ constexpr int route_count_threads() { return EPL >= 32 ? 256 : 512; }

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

// Routes tokens t0 .. t0 + 32/G - 1 (one per group of G lanes; those past T
// work on a clamped token and store nothing). Called by the whole warp, so
// every shuffle sees the full mask. sp: this warp's 32 * EPL floats.
template <int G, int EPL, int LDT>
__device__ __forceinline__ void route_group_tokens(const typename Elem<LDT>::T *__restrict__ L,
                                                   typename Elem<LDT>::T *__restrict__ W,
                                                   int64_t T, int E, int top_k, int renormalize,
                                                   uint32_t *__restrict__ idx_out, int64_t t0,
                                                   float *sp)
{
    using ET = typename Elem<LDT>::T;
    (void)sizeof(ET);
    const int lane = (int)lane_id();
    const int r = lane % G, gbase = lane - r;            // lane in group, group's first lane
    {
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
        float *pw = sp + (lane / G) * (G * EPL);
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
    const int64_t slots = (int64_t)gridDim.x * (blockDim.x / 32) * TPW;
    pdl_wait();
    pdl_launch_dependents();

    // the loop is uniform across the warp: groups past T work on a clamped
    // token and store nothing, so every shuffle sees the full warp
    for (int64_t t0 = ((int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * TPW;
         t0 < T; t0 += slots)
        route_group_tokens<G, EPL, LDT>(L, W, T, E, top_k, renormalize, idx_out, t0,
                                        sp[threadIdx.x / 32]);
}

// ---- one thread per token ----------------------------------------------------

constexpr int kMaxThreadTopK = 8;
// one thread per token: 128 threads, so each thread's column of EPL keys
// stays within 32 KiB of shared memory per block; a compile-time column
// stride keeps the key addresses immediate offsets
constexpr int kThreadRouteThreads = 128;

template <int EPL, int LDT>
__global__ void __launch_bounds__(kThreadRouteThreads)
route_thread_kernel(const void *__restrict__ logits, int64_t T, int E, int top_k,
                    int renormalize, int vec_rows, uint32_t *__restrict__ idx_out,
                    void *__restrict__ w_out)
{
    using ET = typename Elem<LDT>::T;
    constexpr int VEC = 16 / (int)sizeof(ET);          // elements per 16-byte load
    static_assert(EPL % VEC == 0, "rows are read in 16-byte pieces");
    const ET *L = static_cast<const ET *>(logits);
    ET *W = static_cast<ET *>(w_out);
    extern __shared__ uint32_t keys[];               // [EPL][kThreadRouteThreads]
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

        // Selection on order-preserving integer keys of the logits (a larger
        // key is a larger logit; -inf is 0x007fffff, so 0 marks a taken or
        // absent expert; NaN and +inf rows are invalid and never reach here).
        // The keys sit in this thread's column of shared memory, the best key
        // of each group of 8 experts in registers: a round compares the group
        // bests, takes the winner, and rescans only the winner's group. Every
        // scan runs in ascending id with a strict '>', so among equal logits
        // the lower id wins.
        constexpr int NG = EPL / 8;
        uint32_t *col = keys + threadIdx.x;          // key i at col[i * kThreadRouteThreads]
        uint32_t gk[NG];
        int gi[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            gk[g] = 0u;
            gi[g] = g * 8;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = g * 8 + q;
                uint32_t key = 0u;
                if (i < E) {
                    // -0 and +0 are equal logits: one key, so the lower id wins
                    const uint32_t b = l[i] == 0.0f ? 0u : __float_as_uint(l[i]);
                    key = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
                }
                col[i * kThreadRouteThreads] = key;
                if (key > gk[g]) { gk[g] = key; gi[g] = i; }
            }
        }
        float p[kMaxThreadTopK];
        int id[kMaxThreadTopK];
        float z = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxThreadTopK; ++j) {
            p[j] = 0.0f;
            id[j] = j;
            if (j < top_k && !invalid) {
                uint32_t bk = gk[0];
                int bi = gi[0], bg = 0;
#pragma unroll
                for (int g = 1; g < NG; ++g)
                    if (gk[g] > bk) { bk = gk[g]; bi = gi[g]; bg = g; }
                id[j] = bi;
                const uint32_t lb = (bk & 0x80000000u) ? (bk & 0x7fffffffu) : ~bk;
                p[j] = exp2f((__uint_as_float(lb) - m) * kLog2e) * inv_s;
                z += p[j];
                // take it, and rescan its group
                col[bi * kThreadRouteThreads] = 0u;
                uint32_t nk = 0u;
                int ni = bg * 8;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t key = col[(bg * 8 + q) * kThreadRouteThreads];
                    if (key > nk) { nk = key; ni = bg * 8 + q; }
                }
#pragma unroll
                for (int g = 0; g < NG; ++g)
                    if (g == bg) { gk[g] = nk; gi[g] = ni; }
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

// ---- one thread per token, 16-bit logits on packed pairs ----------------------
//
// BF16 / F16 logits whose rows are whole 16-byte vectors (E % 8 == 0): the
// thread keeps its row as E/2 packed 32-bit words and works on pairs where it
// can, which cuts the instructions per token about fourfold:
//   * the row maximum is a NaN-propagating packed max, so one look at it
//     tells an invalid row (a NaN, a +inf, or every logit -inf);
//   * each logit becomes a 32-bit selection key: its order-preserving 16-bit
//     code in the high half (-0 and +0 share one code, so they tie) and
//     63 - id in the low half, so one integer max compares the logits and
//     breaks ties toward the lower id; shared memory keeps only the codes
//     (the id is the position), a group of 8 experts in one 16-byte word,
//     and a round's rescan rebuilds that group's keys from one 16-byte read
//     (half the bytes of stored keys, so more threads fit an SM);
//   * the softmax sum takes one FFMA and one ex2 per logit.
// The selected probabilities are recomputed from their keys' codes (the same
// FP32 operations as in the sum).

// Order-preserving codes of the two 16-bit floats in w (IEEE sign-magnitude,
// BF16 or F16): a positive value h maps to h + 0x8000, a negative one to
// 0x8000 - |h|, so -0 and +0 share 0x8000, larger values get larger codes and
// no code is 0. Per 16-bit lane with no carry or borrow across lanes.
__device__ __forceinline__ uint32_t order_codes2(uint32_t w)
{
    const uint32_t sgn = (w >> 15) & 0x00010001u;     // 1 in each negative lane
    const uint32_t neg = sgn * 0xffffu;               // 0xffff in each negative lane
    const uint32_t mag = w & 0x7fff7fffu;
    return 0x80008000u + (mag & ~neg) - (mag & neg);
}

// The 16-bit float bits of a code (the inverse of order_codes2; -0 comes
// back as +0).
__device__ __forceinline__ uint32_t code_to_bits16(uint32_t code)
{
    return code >= 0x8000u ? code - 0x8000u : (0x8000u | (0x8000u - code));
}

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int LDT>
__device__ __forceinline__ float half_lo(uint32_t w)
{
    if constexpr (LDT == DT_BF16) return __uint_as_float(w << 16);
    else return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
}
template <int LDT>
__device__ __forceinline__ float half_hi(uint32_t w)
{
    if constexpr (LDT == DT_BF16) return __uint_as_float(w & 0xffff0000u);
    else return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}
template <int LDT>
__device__ __forceinline__ uint32_t max2_nan(uint32_t a, uint32_t b)
{
    if constexpr (LDT == DT_BF16) {
        const __nv_bfloat162 r = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162 *>(&a),
                                             *reinterpret_cast<const __nv_bfloat162 *>(&b));
        return *reinterpret_cast<const uint32_t *>(&r);
    } else {
        const __half2 r = __hmax2_nan(*reinterpret_cast<const __half2 *>(&a),
                                      *reinterpret_cast<const __half2 *>(&b));
        return *reinterpret_cast<const uint32_t *>(&r);
    }
}

constexpr int kKeyPad = 4;                 // words after each thread's code row (bank spread)

template <int EPL, int LDT>
__global__ void __launch_bounds__(kThreadRouteThreads)
route_thread16_kernel(const void *__restrict__ logits, int64_t T, int E, int top_k,
                      int renormalize, uint32_t *__restrict__ idx_out,
                      void *__restrict__ w_out)
{
    static_assert(EPL % 8 == 0 && EPL <= 64, "rows of whole 16-byte vectors, ids below 64");
    constexpr int NW = EPL / 2;                       // packed words per row
    constexpr int NG = EPL / 8;                       // groups of 8 experts
    constexpr int ROW = EPL / 2 + kKeyPad;            // code words per thread
    constexpr uint32_t kNegInf2 = LDT == DT_BF16 ? 0xff80ff80u : 0xfc00fc00u;
    using ET = typename Elem<LDT>::T;
    const uint4 *L = static_cast<const uint4 *>(logits);
    ET *W = static_cast<ET *>(w_out);
    extern __shared__ uint4 key_smem[];               // [threads][ROW] words
    uint32_t *kr = reinterpret_cast<uint32_t *>(key_smem) + threadIdx.x * ROW;
    const int vecs = E / 8;                           // 16-byte vectors per row
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x) {
        uint32_t w[NW];
        const uint4 *row = L + t * vecs;
#pragma unroll
        for (int c = 0; c < EPL / 8; ++c) {
            uint4 v = make_uint4(kNegInf2, kNegInf2, kNegInf2, kNegInf2);
            if (c < vecs) v = row[c];
            w[4 * c] = v.x;
            w[4 * c + 1] = v.y;
            w[4 * c + 2] = v.z;
            w[4 * c + 3] = v.w;
        }
        // row maximum, NaN-propagating: NaN if any logit is NaN
        uint32_t mp = w[0];
#pragma unroll
        for (int i = 1; i < NW; ++i) mp = max2_nan<LDT>(mp, w[i]);
        const float ma = half_lo<LDT>(mp), mb = half_hi<LDT>(mp);
        const float m = (isnan(ma) || isnan(mb)) ? __int_as_float(0x7fc00000) : fmaxf(ma, mb);
        const bool invalid = !(fabsf(m) < INFINITY);  // NaN, +inf, or every logit -inf

        // FP32 softmax sum, exp(l - m) = 2^(l log2e - m log2e) with one FFMA
        // per logit; where m log2e would overflow FP32 (|m| near the format's
        // largest values), 2^((l - m) log2e) instead
        constexpr float kLog2e = 1.4426950408889634f;
        const bool big = !(fabsf(m) < 1.0e30f);
        const float mb2 = big ? 0.0f : -m * kLog2e;
        auto arg = [&](float l) { return big ? (l - m) * kLog2e : fmaf(l, kLog2e, mb2); };
        float s = 0.0f;
        if (!invalid) {
            if (!big) {
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    s += ex2_approx(fmaf(half_lo<LDT>(w[i]), kLog2e, mb2));
                    s += ex2_approx(fmaf(half_hi<LDT>(w[i]), kLog2e, mb2));
                }
            } else {
#pragma unroll
                for (int i = 0; i < NW; ++i) {
                    s += ex2_approx((half_lo<LDT>(w[i]) - m) * kLog2e);
                    s += ex2_approx((half_hi<LDT>(w[i]) - m) * kLog2e);
                }
            }
        }
        const float inv_s = 1.0f / s;

        // keys (code << 16 | 63 - id), stored per group of 8; group bests kept
        uint32_t gk[NG];
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            uint32_t k8[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t code = order_codes2(w[4 * g + q]);
                const int id = 8 * g + 2 * q;
                k8[2 * q] = (code << 16) | (uint32_t)(63 - id);
                k8[2 * q + 1] = (code & 0xffff0000u) | (uint32_t)(62 - id);
            }
            reinterpret_cast<uint4 *>(kr + 4 * g)[0] =
                make_uint4(order_codes2(w[4 * g]), order_codes2(w[4 * g + 1]),
                           order_codes2(w[4 * g + 2]), order_codes2(w[4 * g + 3]));
            uint32_t b = k8[0];
#pragma unroll
            for (int q = 1; q < 8; ++q) b = max(b, k8[q]);
            gk[g] = b;
        }

        float p[kMaxThreadTopK];
        int id[kMaxThreadTopK];
        float z = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxThreadTopK; ++j) {
            p[j] = 0.0f;
            id[j] = j;
            if (j < top_k && !invalid) {
                uint32_t best = gk[0];
#pragma unroll
                for (int g = 1; g < NG; ++g) best = max(best, gk[g]);
                const int e = 63 - (int)(best & 0xffffu);
                id[j] = e;
                const uint32_t bits = code_to_bits16(best >> 16);
                const float l = LDT == DT_BF16 ? __uint_as_float(bits << 16)
                                               : __half2float(__ushort_as_half((unsigned short)bits));
                p[j] = ex2_approx(arg(l)) * inv_s;
                z += p[j];
                // take it (code 0: its rebuilt key, 63 - id, is below every
                // untaken key), then rescan its group's codes
                const int g0 = e & ~7;
                reinterpret_cast<unsigned short *>(kr)[e] = 0;
                const uint4 a = reinterpret_cast<const uint4 *>(kr + g0 / 2)[0];
                const uint32_t cw[4] = {a.x, a.y, a.z, a.w};
                uint32_t nk = 0u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int id0 = g0 + 2 * q;
                    nk = max(nk, (cw[q] << 16) | (uint32_t)(63 - id0));
                    nk = max(nk, (cw[q] & 0xffff0000u) | (uint32_t)(62 - id0));
                }
#pragma unroll
                for (int g = 0; g < NG; ++g)
                    if (gk[g] == best) gk[g] = nk;
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
cudaError_t launch_route_thread16(const void *logits, int64_t T, int E, int top_k, int renorm,
                                  uint32_t *idx, void *w, cudaStream_t s)
{
    constexpr int kThreads = kThreadRouteThreads;
    const size_t smem = (size_t)kThreads * (EPL / 2 + kKeyPad) * sizeof(uint32_t);
    static std::atomic<uint64_t> opted{0};       // the > 48 KiB opt-in, per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev >= 0 && dev < kCachedDevices ? 1ull << dev : 0ull;
    if (smem > 48 * 1024 && (bit == 0 || !(opted.load() & bit))) {
        err = cudaFuncSetAttribute(route_thread16_kernel<EPL, LDT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        opted.fetch_or(bit);
    }
    int64_t blocks = (T + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(route_thread16_kernel<EPL, LDT>, dim3((unsigned)blocks), dim3(kThreads),
                      smem, s, logits, T, E, top_k, renorm, idx, w);
}

template <int EPL, int LDT>
cudaError_t launch_route_thread(const void *logits, int64_t T, int E, int top_k, int renorm,
                                uint32_t *idx, void *w, cudaStream_t s)
{
    using ET = typename Elem<LDT>::T;
    const int vec_rows = ((int64_t)E * (int64_t)sizeof(ET)) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(logits) % 16 == 0;
    constexpr int kThreads = kThreadRouteThreads;
    int64_t blocks = (T + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(route_thread_kernel<EPL, LDT>, dim3((unsigned)blocks), dim3(kThreads),
                      (size_t)EPL * kThreads * sizeof(uint32_t), s, logits, T, E, top_k, renorm,
                      vec_rows, idx, w);
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
        if (LDT != DT_F32 && E % 8 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0) {
            if (E <= 8) return launch_route_thread16<8, LDT>(logits, T, E, top_k, renorm, idx, w, s);
            if (E <= 16) return launch_route_thread16<16, LDT>(logits, T, E, top_k, renorm, idx, w, s);
            if (E <= 32) return launch_route_thread16<32, LDT>(logits, T, E, top_k, renorm, idx, w, s);
            return launch_route_thread16<64, LDT>(logits, T, E, top_k, renorm, idx, w, s);
        }
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

// ---- routing fused with the dispatch counts ----------------------------------

// CTA c routes the tokens of assignment chunk c ([c * chunk, (c + 1) * chunk)
// of the A = T * top_k assignments; a token on a chunk edge is routed by both
// neighbours, with identical results), counts the chunk's assignments per
// expert in shared memory and stores the counts in chunk_counts[E][nchunks]
// (each expert's counts contiguous, as the dispatch passes keep them). The
// last CTA to finish (a completion counter it resets afterwards) turns every
// expert's column of counts into the first row each chunk may use inside the
// expert and writes the expert totals: what the rank/scatter kernel reads.
template <int G, int EPL, int LDT>
__global__ void __launch_bounds__(route_count_threads<EPL>())
route_count_kernel(const void *__restrict__ logits, int64_t T, int E, int top_k,
                   int renormalize, uint32_t *__restrict__ idx_out, void *__restrict__ w_out,
                   int64_t chunk, int64_t nchunks, int *__restrict__ chunk_counts,
                   int32_t *__restrict__ counts, unsigned *__restrict__ done)
{
    using ET = typename Elem<LDT>::T;
    const ET *L = static_cast<const ET *>(logits);
    ET *W = static_cast<ET *>(w_out);
    constexpr int TPW = 32 / G;
    constexpr int NT = route_count_threads<EPL>();
    constexpr int WARPS = NT / 32;
    __shared__ float sp[WARPS][32 * EPL];
    __shared__ int is_last;
    extern __shared__ int hist[];                        // [E]
    pdl_wait();
    pdl_launch_dependents();
    const int64_t A = T * top_k;
    const int64_t c = blockIdx.x;
    const int64_t a0 = c * chunk, a1 = a0 + chunk < A ? a0 + chunk : A;
    const int64_t t_lo = a0 / top_k, t_hi = (a1 - 1) / top_k;
    const int warp = threadIdx.x / 32;
    for (int e = threadIdx.x; e < E; e += NT) hist[e] = 0;
    for (int64_t t0 = t_lo + (int64_t)warp * TPW; t0 <= t_hi; t0 += (int64_t)WARPS * TPW)
        route_group_tokens<G, EPL, LDT>(L, W, T, E, top_k, renormalize, idx_out, t0, sp[warp]);
    __syncthreads();         // this CTA's ids (all its chunk's tokens) are written
    for (int64_t a = a0 + threadIdx.x; a < a1; a += NT) {
        const uint32_t e = idx_out[a];
        if (e < (uint32_t)E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NT) chunk_counts[(int64_t)e * nchunks + c] = hist[e];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(done, 1u) == (unsigned)(nchunks - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // every CTA's counts into shared memory with all threads' loads in flight
    // (a column walk in global memory would wait for each load in turn), then
    // one thread per expert scans its column there
    int *cc = hist + E;                                // [E][nchunks]
    const int n = (int)(nchunks * E);
    for (int i = threadIdx.x; i < n; i += NT) cc[i] = __ldcg(chunk_counts + i);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NT) {
        int run = 0;
        for (int k = 0; k < (int)nchunks; ++k) {
            const int v = cc[e * (int)nchunks + k];
            chunk_counts[(int64_t)e * nchunks + k] = run;
            run += v;
        }
        counts[e] = run;
    }
    if (threadIdx.x == 0) *done = 0u;                  // ready for the next launch
}

// Largest nchunks x E the last CTA scans in shared memory (with hist: 56 KiB).
constexpr int64_t kFusedMaxCounts = 14 * 1024;

template <int G, int EPL, int LDT>
cudaError_t launch_route_count(const void *logits, int64_t T, int E, int top_k, int renorm,
                               uint32_t *idx, void *w, int64_t chunk, int64_t nchunks,
                               int *chunk_counts, int32_t *counts, unsigned *done, cudaStream_t s)
{
    const size_t smem = ((size_t)E + (size_t)nchunks * E) * sizeof(int);
    static std::atomic<uint64_t> opted{0};       // the > 48 KiB opt-in, per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev >= 0 && dev < kCachedDevices ? 1ull << dev : 0ull;
    if (bit == 0 || !(opted.load() & bit)) {
        err = cudaFuncSetAttribute(route_count_kernel<G, EPL, LDT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)((1024 + kFusedMaxCounts) * sizeof(int)));
        if (err != cudaSuccess) return err;
        opted.fetch_or(bit);
    }
    return launch_pdl(route_count_kernel<G, EPL, LDT>, dim3((unsigned)nchunks),
                      dim3(route_count_threads<EPL>()), smem, s, logits, T, E, top_k, renorm, idx, w, chunk,
                      nchunks, chunk_counts, counts, done);
}

template <int LDT>
cudaError_t launch_route_count_dt(const void *logits, int64_t T, int E, int top_k, int renorm,
                                  uint32_t *idx, void *w, int64_t chunk, int64_t nchunks,
                                  int *cc, int32_t *counts, unsigned *done, cudaStream_t s)
{
    if (E <= 8) return launch_route_count<1, 8, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    if (E <= 16) return launch_route_count<2, 8, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    if (E <= 32) return launch_route_count<4, 8, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    if (E <= 64) return launch_route_count<8, 8, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    if (E <= 128) return launch_route_count<16, 8, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    if (E <= 256) return launch_route_count<32, 8, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    if (E <= 512) return launch_route_count<32, 16, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
    return launch_route_count<32, 32, LDT>(logits, T, E, top_k, renorm, idx, w, chunk, nchunks, cc, counts, done, s);
}

}  // namespace

cudaError_t launch_route_dispatch(const void *logits, int ldt, int64_t T, int E, int top_k,
                                  int renormalize, uint32_t *idx, void *w, const void *x,
                                  int xdt, int64_t H, int32_t *counts, int32_t *offsets,
                                  int32_t *row_of, int32_t *src_of, void *x_disp, void *ws,
                                  unsigned *zeroed_counter, unsigned *status, cudaStream_t s)
{
    const int64_t A = T * top_k;
    if (A == 0) return cudaSuccess;
    const int64_t chunk = dispatch_chunk_len(A);
    const int64_t nchunks = (A + chunk - 1) / chunk;
    if (thread_route_fits(T, E, top_k) || nchunks * E > kFusedMaxCounts || E > 1024) {
        cudaError_t err = launch_route(logits, ldt, T, E, top_k, renormalize, idx, w, s);
        if (err != cudaSuccess) return err;
        return launch_dispatch(idx, T, top_k, E, 0, x, xdt, H, counts, offsets, row_of, src_of,
                               x_disp, ws, status, s);
    }
    unsigned *done = zeroed_counter;
    cudaError_t err = cudaSuccess;
    if (done == nullptr) {
        done = dispatch_done_counter(ws, A, E);
        err = cudaMemsetAsync(done, 0, sizeof(unsigned), s);
        if (err != cudaSuccess) return err;
    }
    int *cc = static_cast<int *>(ws);
    switch (ldt) {
    case DT_F32: err = launch_route_count_dt<DT_F32>(logits, T, E, top_k, renormalize, idx, w, chunk, nchunks, cc, counts, done, s); break;
    case DT_BF16: err = launch_route_count_dt<DT_BF16>(logits, T, E, top_k, renormalize, idx, w, chunk, nchunks, cc, counts, done, s); break;
    default: err = launch_route_count_dt<DT_F16>(logits, T, E, top_k, renormalize, idx, w, chunk, nchunks, cc, counts, done, s); break;
    }
    if (err != cudaSuccess) return err;
    return launch_dispatch_rank_gather(idx, T, top_k, E, x, xdt, H, counts, offsets, row_of,
                                       src_of, x_disp, ws, status, s);
}

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
