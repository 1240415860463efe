// experts_simt_train.cu -- FP32 SwiGLU expert backward on CUDA cores.
//
// ruDNN user guide, section 12 "MoE first-order training" (cache.backward of
// SwiGluExperts::forward_dispatched_training): for every dispatched row r of
// expert e, with the forward's g = Wg[e] x_r, u = Wu[e] x_r, h = SiLU(g) * u
// and the output gradient do_r,
//   dh  = Wd[e]^T do_r,  s = sigmoid(g),
//   dg  = dh * u * s * (1 + g * (1 - s)),   du = dh * g * s,
//   dx_r = Wg[e]^T dg + Wu[e]^T du,
//   dWd[e] += do_r h^T,  dWg[e] += dg x_r^T,  dWu[e] += du x_r^T.
// True FP32 FFMA throughout (the FP32 tolerance rules out TF32).
//
// Three launches of one 64 x 64-tile kernel (256 threads, 4 x 4 outputs each,
// K step 16), differing in how a tile's operands are addressed:
//   DH  rows x I,  K = H:   A = do rows, B = Wd[e] read across its rows;
//                           epilogue forms dg and du into dgu [rows, 2I];
//   DX  rows x H,  K = 2I:  A = dgu rows, B = Wg[e] then Wu[e];
//   WG  per expert, M x N, K = the expert's rows: A and B are columns of two
//       row-major activations (do and h for dWd; dg or du and x for dWg,
//       dWu); experts without rows write zero tiles.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int TBM = 64, TBN = 64, TBK = 16, TTHREADS = 256, TMAX_E = 1024;

enum : int { kDH = 0, kDX = 1, kWG = 2 };

struct BwdArgs {
    const float *x_disp, *gate, *up, *down, *cache, *dout;
    const int32_t *offsets;
    float *dgu, *dx;
    // WG: P [rows, ldp] columns m, Q [rows, ldq] columns n, W [E, M, N]
    const float *P, *Q;
    float *W;
    int ldp, ldq, M, N;
    int E, H, I;
    int64_t rows;
};

// Block-wide prefix of the experts' M-tile counts times n_tiles (DH, DX).
__device__ void tile_prefix(const int32_t *offsets, int E, int n_tiles, int *prefix, int *wsum)
{
    const int per = (E + TTHREADS - 1) / TTHREADS;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int e = e0; e < e0 + per && e < E; ++e)
        local += (offsets[e + 1] - offsets[e] + TBM - 1) / TBM * n_tiles;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int wbase = 0;
    for (int i = 0; i < w; ++i) wbase += wsum[i];
    int run = wbase + incl - local;
    for (int e = e0; e < e0 + per && e < E; ++e) {
        prefix[e] = run;
        run += (offsets[e + 1] - offsets[e] + TBM - 1) / TBM * n_tiles;
    }
    if (threadIdx.x == TTHREADS - 1) prefix[E] = wbase + incl;
    __syncthreads();
}

// acc[i][j] += sum_k A(m0 + tr*4 + i, k) * B(n0 + tc*4 + j, k) for k < K.
// ld_a(r, k) / ld_b(c, k) return an operand element (0 outside the tile's
// valid range); A_K / B_K say whether k is the contiguous index of that
// operand in memory (chooses the thread-to-element map of the loads).
template <bool A_K, bool B_K, class LA, class LB>
__device__ __forceinline__ void tile_product(float (&acc)[4][4], int K, LA ld_a, LB ld_b,
                                             float (*As)[TBM + 4], float (*Bs)[TBN + 4])
{
    const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;
    for (int k0 = 0; k0 < K; k0 += TBK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int li = threadIdx.x + q * TTHREADS;
            const int ra = A_K ? li / TBK : li % TBM, ka = A_K ? li % TBK : li / TBM;
            As[ka][ra] = k0 + ka < K ? ld_a(ra, k0 + ka) : 0.0f;
            const int rb = B_K ? li / TBK : li % TBN, kb = B_K ? li % TBK : li / TBN;
            Bs[kb][rb] = k0 + kb < K ? ld_b(rb, k0 + kb) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TBK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tc * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
}

template <int MODE>
__global__ void __launch_bounds__(TTHREADS) experts_simt_bwd_kernel(BwdArgs p)
{
    __shared__ int prefix[TMAX_E + 1];
    __shared__ int wsum[TTHREADS / 32];
    __shared__ float As[TBK][TBM + 4];
    __shared__ float Bs[TBK][TBN + 4];
    pdl_wait();
    pdl_launch_dependents();
    const int E = p.E, H = p.H, I = p.I;
    const int N = MODE == kDH ? I : MODE == kDX ? H : p.N;
    const int n_tiles = (N + TBN - 1) / TBN;
    int total;
    if constexpr (MODE == kWG) {
        total = E * ((p.M + TBM - 1) / TBM) * n_tiles;
    } else {
        tile_prefix(p.offsets, E, n_tiles, prefix, wsum);
        total = prefix[E];
    }
    const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;
    const float *hc = p.cache, *gc = p.cache + p.rows * I, *uc = p.cache + 2 * p.rows * I;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
        if constexpr (MODE == kWG) {
            const int mt = (p.M + TBM - 1) / TBM, per_e = mt * n_tiles;
            const int e = tile / per_e, loc = tile % per_e;
            const int m0 = (loc / n_tiles) * TBM, n0 = (loc % n_tiles) * TBN;
            const int seg0 = p.offsets[e], seg1 = p.offsets[e + 1];
            const int M = p.M;
            tile_product<false, false>(
                acc, seg1 - seg0,
                [&](int r, int k) { return m0 + r < M ? p.P[(int64_t)(seg0 + k) * p.ldp + m0 + r] : 0.0f; },
                [&](int c, int k) { return n0 + c < N ? p.Q[(int64_t)(seg0 + k) * p.ldq + n0 + c] : 0.0f; },
                As, Bs);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = m0 + tr * 4 + i;
                if (m >= M) continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = n0 + tc * 4 + j;
                    if (n < N) p.W[((int64_t)e * M + m) * N + n] = acc[i][j];
                }
            }
        } else {
            int lo = 0, hi = E - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
            }
            const int e = lo;
            const int seg0 = p.offsets[e], seg1 = p.offsets[e + 1];
            const int mt = (seg1 - seg0 + TBM - 1) / TBM;
            const int loc = tile - prefix[e];
            const int row0 = seg0 + (loc % mt) * TBM, n0 = (loc / mt) * TBN;
            if constexpr (MODE == kDH) {
                const float *wd = p.down + (int64_t)e * H * I;
                tile_product<true, false>(
                    acc, H,
                    [&](int r, int k) { return row0 + r < seg1 ? p.dout[(int64_t)(row0 + r) * H + k] : 0.0f; },
                    [&](int c, int k) { return n0 + c < I ? wd[(int64_t)k * I + n0 + c] : 0.0f; },
                    As, Bs);
            } else {
                const float *wg = p.gate + (int64_t)e * I * H, *wu = p.up + (int64_t)e * I * H;
                tile_product<true, false>(
                    acc, 2 * I,
                    [&](int r, int k) { return row0 + r < seg1 ? p.dgu[(int64_t)(row0 + r) * 2 * I + k] : 0.0f; },
                    [&](int c, int k) {
                        if (n0 + c >= H) return 0.0f;
                        return k < I ? wg[(int64_t)k * H + n0 + c] : wu[(int64_t)(k - I) * H + n0 + c];
                    },
                    As, Bs);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = row0 + tr * 4 + i;
                if (r >= seg1) continue;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = n0 + tc * 4 + j;
                    if (n >= N) continue;
                    if constexpr (MODE == kDH) {
                        const float g = gc[(int64_t)r * I + n], u = uc[(int64_t)r * I + n];
                        const float s = 1.0f / (1.0f + expf(-g));
                        const float dh = acc[i][j];
                        p.dgu[(int64_t)r * 2 * I + n] = dh * u * s * (1.0f + g * (1.0f - s));
                        p.dgu[(int64_t)r * 2 * I + I + n] = dh * g * s;
                    } else {
                        p.dx[(int64_t)r * H + n] = acc[i][j];
                    }
                }
            }
            (void)hc;
        }
    }
}

unsigned grid_for(int64_t tiles)
{
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (tiles < 1) tiles = 1;
    return (unsigned)(tiles < cap ? tiles : cap);
}

}  // namespace

cudaError_t launch_experts_simt_backward(const float *x_disp, const int32_t *offsets,
                                         int64_t rows, const float *gate, const float *up,
                                         const float *down, int E, int64_t H, int64_t I,
                                         const float *cache, const float *dout, float *dgu,
                                         float *dx, float *dgate, float *dup, float *ddown,
                                         cudaStream_t s)
{
    BwdArgs a{};
    a.x_disp = x_disp; a.gate = gate; a.up = up; a.down = down; a.cache = cache; a.dout = dout;
    a.offsets = offsets; a.dgu = dgu; a.dx = dx;
    a.E = E; a.H = (int)H; a.I = (int)I; a.rows = rows;
    const dim3 block(TTHREADS);
    cudaError_t err;
    if (rows > 0) {
        const int64_t mt = rows / TBM + (rows < E ? rows : E);
        err = launch_pdl(experts_simt_bwd_kernel<kDH>, dim3(grid_for(mt * ((I + TBN - 1) / TBN))),
                         block, 0, s, a);
        if (err != cudaSuccess) return err;
        err = launch_pdl(experts_simt_bwd_kernel<kDX>, dim3(grid_for(mt * ((H + TBN - 1) / TBN))),
                         block, 0, s, a);
        if (err != cudaSuccess) return err;
    }
    // weight gradients (every expert, rows or not)
    struct { const float *P, *Q; float *W; int ldp, ldq, M, N; } wg[3] = {
        {dout, cache, ddown, (int)H, (int)I, (int)H, (int)I},          // dWd = do^T h
        {dgu, x_disp, dgate, (int)(2 * I), (int)H, (int)I, (int)H},    // dWg = dg^T x
        {dgu ? dgu + I : nullptr, x_disp, dup, (int)(2 * I), (int)H, (int)I, (int)H},  // dWu
    };
    for (const auto &w : wg) {
        a.P = w.P; a.Q = w.Q; a.W = w.W; a.ldp = w.ldp; a.ldq = w.ldq; a.M = w.M; a.N = w.N;
        const int64_t tiles = (int64_t)E * ((w.M + TBM - 1) / TBM) * ((w.N + TBN - 1) / TBN);
        err = launch_pdl(experts_simt_bwd_kernel<kWG>, dim3(grid_for(tiles)), block, 0, s, a);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace moe
