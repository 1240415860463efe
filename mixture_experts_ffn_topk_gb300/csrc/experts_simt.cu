// experts_simt.cu -- FP32 bias-free SwiGLU experts on CUDA cores.
//
// ruDNN user guide, sections 3 and 5: per dispatched row r of expert e,
// h = SiLU(x_r Wg[e]^T) * (x_r Wu[e]^T), out_r = h Wd[e]^T, with gate/up
// [E,I,H] and down [E,H,I]. FP32 data stays FP32 end to end (plain FFMA, no
// TF32), which the 1e-4 relative tolerance of FP32 outputs requires.
//
// Grouped tiling: every expert segment [offsets[e], offsets[e+1]) is cut into
// 64-row M-tiles; each CTA maps its linear tile id to (expert, n-tile, m-tile)
// through a per-CTA prefix over the experts' tile counts, computed from the
// device-side offsets (no host synchronisation). 64x64 output tiles, K step
// 16, 256 threads with 4x4 outputs each (two accumulators for gate and up).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int SBM = 64, SBN = 64, SBK = 16, STHREADS = 256, SMAX_E = 1024;

// SWIGLU: C = SiLU(A B0^T) * (A B1^T); with pre-activation outputs g_out /
// u_out (training) the two products are stored there too. Otherwise C = A B0^T.
template <bool SWIGLU>
__global__ void __launch_bounds__(STHREADS)
experts_simt_kernel(const float *__restrict__ A, const int32_t *__restrict__ offsets,
                    int E, const float *__restrict__ B0,
                    const float *__restrict__ B1, int N, int K, int n_tiles,
                    float *__restrict__ C, float *__restrict__ g_out = nullptr,
                    float *__restrict__ u_out = nullptr)
{
    __shared__ int prefix[SMAX_E + 1];
    __shared__ int warp_sum[STHREADS / 32];
    __shared__ float As[SBK][SBM + 4];
    __shared__ float Bs[SBK][SBN + 4];
    __shared__ float Us[SWIGLU ? SBK : 1][SWIGLU ? SBN + 4 : 1];
    pdl_wait();
    pdl_launch_dependents();

    // prefix[e] = number of tiles of experts < e (block scan over experts)
    const int per = (E + STHREADS - 1) / STHREADS;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) {
        const int cnt = offsets[e + 1] - offsets[e];
        local += (cnt + SBM - 1) / SBM * n_tiles;
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    int wbase = 0;
    for (int i = 0; i < w; ++i) wbase += warp_sum[i];
    int run = wbase + incl - local;
    for (int e = e0; e < e0 + per && e < E; ++e) {
        prefix[e] = run;
        const int cnt = offsets[e + 1] - offsets[e];
        run += (cnt + SBM - 1) / SBM * n_tiles;
    }
    if (threadIdx.x == STHREADS - 1) prefix[E] = wbase + incl;
    __syncthreads();

    const int total = prefix[E];
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        int lo = 0, hi = E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        const int e = lo;
        const int seg0 = offsets[e], seg1 = offsets[e + 1];
        const int mt = (seg1 - seg0 + SBM - 1) / SBM;
        const int loc = tile - prefix[e];
        const int n = loc / mt, m = loc % mt;
        const int row0 = seg0 + m * SBM, col0 = n * SBN;
        const float *Be = B0 + (int64_t)e * N * K;
        const float *Ue = SWIGLU ? B1 + (int64_t)e * N * K : nullptr;

        const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;  // 16 x 16 threads
        float accg[4][4], accu[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) { accg[i][j] = 0.0f; accu[i][j] = 0.0f; }

        for (int k0 = 0; k0 < K; k0 += SBK) {
            // 64 x 16 tile of A and of each B: 1024 elements, 4 per thread
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int li = threadIdx.x + q * STHREADS;
                const int r = li / SBK, kk = li % SBK;
                const int gr = row0 + r, gk = k0 + kk;
                As[kk][r] = (gr < seg1 && gk < K) ? A[(int64_t)gr * K + gk] : 0.0f;
                const int gn = col0 + r;
                Bs[kk][r] = (gn < N && gk < K) ? Be[(int64_t)gn * K + gk] : 0.0f;
                if (SWIGLU) Us[kk][r] = (gn < N && gk < K) ? Ue[(int64_t)gn * K + gk] : 0.0f;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < SBK; ++kk) {
                float a[4], b[4], u[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kk][tr * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    b[j] = Bs[kk][tc * 4 + j];
                    if (SWIGLU) u[j] = Us[kk][tc * 4 + j];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        accg[i][j] = fmaf(a[i], b[j], accg[i][j]);
                        if (SWIGLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
                    }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gr = row0 + tr * 4 + i;
            if (gr >= seg1) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int gn = col0 + tc * 4 + j;
                if (gn >= N) continue;
                float v = accg[i][j];
                if (SWIGLU) {
                    if (g_out != nullptr) {
                        g_out[(int64_t)gr * N + gn] = v;
                        u_out[(int64_t)gr * N + gn] = accu[i][j];
                    }
                    v = v / (1.0f + expf(-v)) * accu[i][j];
                }
                C[(int64_t)gr * N + gn] = v;
            }
        }
    }
}

int64_t tile_upper_bound(int64_t rows, int E, int64_t n_tiles)
{
    const int64_t mt = rows / SBM + (rows < E ? rows : E);
    return mt * n_tiles;
}

}  // namespace

cudaError_t launch_experts_simt(const float *x_disp, const int32_t *offsets,
                                int64_t rows, const float *gate,
                                const float *up, const float *down, int E,
                                int64_t H, int64_t I, float *h_ws,
                                float *out_disp, cudaStream_t s, float *g_out, float *u_out)
{
    if (rows == 0) return cudaSuccess;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    const int nt1 = (int)((I + SBN - 1) / SBN);
    int64_t g1 = tile_upper_bound(rows, E, nt1);
    if (g1 > cap) g1 = cap;
    cudaError_t err = launch_pdl(experts_simt_kernel<true>, dim3((unsigned)g1), dim3(STHREADS), 0,
                                 s, x_disp, offsets, E, gate, up, (int)I, (int)H, nt1, h_ws,
                                 g_out, u_out);
    if (err != cudaSuccess) return err;
    const int nt2 = (int)((H + SBN - 1) / SBN);
    int64_t g2 = tile_upper_bound(rows, E, nt2);
    if (g2 > cap) g2 = cap;
    return launch_pdl(experts_simt_kernel<false>, dim3((unsigned)g2), dim3(STHREADS), 0, s,
                      (const float *)h_ws, offsets, E, down, (const float *)nullptr, (int)H,
                      (int)I, nt2, out_disp, (float *)nullptr, (float *)nullptr);
}

}  // namespace moe
