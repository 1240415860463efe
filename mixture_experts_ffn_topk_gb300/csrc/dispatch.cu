// dispatch.cu -- compact, no-drop dispatch with a saved map.
//
// ruDNN user guide, section 5 "Expert weights and dispatch": no token is
// dropped to enforce a capacity; order inside an expert is unspecified; a
// saved map restores token order.
//
// The A = T*top_k assignments are cut into nchunks <= 128 contiguous chunks,
// one warp each:
//   1. count:   per-chunk, per-expert histograms (shared-memory atomics);
//   2. scan:    one CTA turns them into counts[E], offsets[E+1] and, per chunk
//               and expert, the first row that chunk may use;
//   3. rank:    each warp walks its chunk in order, 32 assignments at a time,
//               and ranks equal experts with __match_any_sync, so rows inside
//               an expert follow the assignment order (deterministic);
//   4. gather:  x_disp[row] = x[src_of[row] / top_k], 16-byte vectors, one
//               warp per row (HBM-bound copy).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kChunkWarps = 4;          // warps (chunks) per CTA in count/rank
constexpr int kMaxChunks = 128;

struct ChunkPlan {
    int64_t A;
    int64_t chunk;    // assignments per chunk (multiple of 32)
    int nchunks;
};

ChunkPlan plan_chunks(int64_t A)
{
    ChunkPlan p;
    p.A = A;
    int64_t c = (A + kMaxChunks - 1) / kMaxChunks;
    c = (c + 31) / 32 * 32;
    if (c < 256) c = 256;
    p.chunk = c;
    p.nchunks = (int)((A + c - 1) / c);
    return p;
}

__global__ void __launch_bounds__(kChunkWarps * 32)
dispatch_count_kernel(const uint32_t *__restrict__ idx, int64_t A, int E,
                      int64_t chunk, int nchunks, int *__restrict__ chunk_counts,
                      unsigned *status)
{
    extern __shared__ int hist[];
    pdl_wait();
    pdl_launch_dependents();
    const int w = threadIdx.x / 32, lane = (int)lane_id();
    const int c = blockIdx.x * kChunkWarps + w;
    int *h = hist + (size_t)w * E;
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    if (c >= nchunks) return;
    const int64_t a0 = (int64_t)c * chunk;
    const int64_t a1 = a0 + chunk < A ? a0 + chunk : A;
    bool saw_bad = false;
    for (int64_t a = a0 + lane; a < a1; a += 32) {
        const uint32_t e = idx[a];
        if (e < (uint32_t)E) atomicAdd(&h[e], 1);
        else saw_bad = true;
    }
    if (__any_sync(kFull, saw_bad) && lane == 0) atomicOr(status, ST_BAD_INDEX);
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_counts[(size_t)c * E + e] = h[e];
}

// One CTA of 1024 threads; thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(int *__restrict__ chunk_counts, int nchunks, int E,
                     int64_t A, int32_t *__restrict__ counts,
                     int32_t *__restrict__ offsets, int32_t *__restrict__ src_of)
{
    __shared__ int warp_tot[32];
    __shared__ int total_rows;
    pdl_wait();
    pdl_launch_dependents();
    const int e = threadIdx.x, lane = e & 31, w = e >> 5;
    int total = 0;
    if (e < E) {
#pragma unroll 8
        for (int c = 0; c < nchunks; ++c) total += chunk_counts[(size_t)c * E + e];
    }
    int incl = total;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(kFull, v, o);
            if (lane >= o) v += u;
        }
        warp_tot[lane] = v;   // inclusive over warps
        if (lane == 31) total_rows = v;
    }
    __syncthreads();
    const int excl = incl - total + (w > 0 ? warp_tot[w - 1] : 0);
    if (e < E) {
        counts[e] = total;
        offsets[e] = excl;
        if (e == E - 1) offsets[E] = excl + total;
        int run = excl;
        for (int c = 0; c < nchunks; ++c) {
            const int v = chunk_counts[(size_t)c * E + e];
            chunk_counts[(size_t)c * E + e] = run;
            run += v;
        }
    }
    // rows past the last one (only when some index was >= E) map to nothing
    for (int64_t r = (int64_t)total_rows + threadIdx.x; r < A; r += blockDim.x) src_of[r] = -1;
}

__global__ void __launch_bounds__(kChunkWarps * 32)
dispatch_rank_kernel(const uint32_t *__restrict__ idx, int64_t A, int E,
                     int64_t chunk, int nchunks,
                     const int *__restrict__ chunk_base,
                     int32_t *__restrict__ row_of, int32_t *__restrict__ src_of)
{
    extern __shared__ int base[];
    pdl_wait();
    pdl_launch_dependents();
    const int w = threadIdx.x / 32, lane = (int)lane_id();
    const int c = blockIdx.x * kChunkWarps + w;
    if (c >= nchunks) return;
    int *b = base + (size_t)w * E;
    for (int e = lane; e < E; e += 32) b[e] = chunk_base[(size_t)c * E + e];
    __syncwarp();
    const int64_t a0 = (int64_t)c * chunk;
    const int64_t a1 = a0 + chunk < A ? a0 + chunk : A;
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t s = a0; s < a1; s += 32) {
        const int64_t a = s + lane;
        const bool act = a < a1;
        const uint32_t e = act ? idx[a] : 0xffffffffu;
        const bool ok = act && e < (uint32_t)E;
        const uint32_t key = ok ? e : 0xffffffffu;
        const unsigned peers = __match_any_sync(kFull, key);
        int row = -1;
        if (ok) {
            row = b[e] + __popc(peers & lt);
            src_of[row] = (int32_t)a;
        }
        if (act) row_of[a] = row;
        __syncwarp();
        if (ok && lane == __ffs(peers) - 1) b[e] += __popc(peers);
        __syncwarp();
    }
}

// One warp per dispatched row; 16-byte vectors when rows are 16-byte multiples.
template <bool VEC>
__global__ void __launch_bounds__(256)
dispatch_gather_kernel(const uint8_t *__restrict__ x, int64_t rows,
                       int64_t row_bytes, int top_k,
                       const int32_t *__restrict__ src_of,
                       uint8_t *__restrict__ x_disp)
{
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
         r < rows; r += warps) {
        const int32_t a = src_of[r];
        if (a < 0) continue;
        const int64_t t = a / top_k;
        if (VEC) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + t * row_bytes);
            uint4 *dst = reinterpret_cast<uint4 *>(x_disp + r * row_bytes);
            const int64_t nv = row_bytes / 16;
#pragma unroll 4
            for (int64_t v = lane; v < nv; v += 32) dst[v] = __ldg(src + v);
        } else {
            const uint8_t *src = x + t * row_bytes;
            uint8_t *dst = x_disp + r * row_bytes;
            for (int64_t v = lane; v < row_bytes; v += 32) dst[v] = src[v];
        }
    }
}

}  // namespace

size_t dispatch_workspace_bytes(int64_t A, int E)
{
    if (A <= 0) return 0;
    const ChunkPlan p = plan_chunks(A);
    return (size_t)p.nchunks * (size_t)E * sizeof(int);
}

cudaError_t launch_dispatch(const uint32_t *idx, int64_t T, int top_k, int E,
                            const void *x, int xdt, int64_t H, int32_t *counts,
                            int32_t *offsets, int32_t *row_of, int32_t *src_of,
                            void *x_disp, void *ws, unsigned *status,
                            cudaStream_t s)
{
    const int64_t A = T * top_k;
    if (A == 0) return cudaSuccess;
    const ChunkPlan p = plan_chunks(A);
    int *chunk = static_cast<int *>(ws);
    const int blocks = (p.nchunks + kChunkWarps - 1) / kChunkWarps;
    const size_t hist_bytes = (size_t)kChunkWarps * E * sizeof(int);
    cudaError_t err = launch_pdl(dispatch_count_kernel, dim3(blocks), dim3(kChunkWarps * 32),
                                 hist_bytes, s, idx, A, E, p.chunk, p.nchunks, chunk, status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(dispatch_scan_kernel, dim3(1), dim3(1024), 0, s, chunk, p.nchunks, E, A,
                     counts, offsets, src_of);
    if (err != cudaSuccess) return err;
    err = launch_pdl(dispatch_rank_kernel, dim3(blocks), dim3(kChunkWarps * 32), hist_bytes, s,
                     idx, A, E, p.chunk, p.nchunks, (const int *)chunk, row_of, src_of);
    if (err != cudaSuccess) return err;
    const int64_t row_bytes = H * (xdt == DT_F32 ? 4 : 2);
    int64_t gblocks = (A + 7) / 8;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (gblocks > cap) gblocks = cap;
    const bool vec = (row_bytes % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(x_disp) % 16 == 0);
    const uint8_t *xb = static_cast<const uint8_t *>(x);
    uint8_t *xd = static_cast<uint8_t *>(x_disp);
    if (vec)
        err = launch_pdl(dispatch_gather_kernel<true>, dim3((unsigned)gblocks), dim3(256), 0, s,
                         xb, A, row_bytes, top_k, (const int32_t *)src_of, xd);
    else
        err = launch_pdl(dispatch_gather_kernel<false>, dim3((unsigned)gblocks), dim3(256), 0, s,
                         xb, A, row_bytes, top_k, (const int32_t *)src_of, xd);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe
