// dispatch.cu -- compact, no-drop dispatch with a saved map.
//
// ruDNN user guide, section 5 "Expert weights and dispatch": no token is
// dropped to enforce a capacity; order inside an expert is unspecified; a
// saved map restores token order.
//
// The A = T*top_k assignments are cut into chunks of 256..2048 (sized so every
// SM gets several), one warp each:
//   1. count:   per-chunk, per-expert histograms in shared memory (equal
//               experts of a 32-assignment batch aggregated with
//               __match_any_sync, one atomic per distinct expert);
//   2. scan:    one CTA per 32 experts turns their columns of chunk counts
//               into the first row each chunk may use inside the expert, and
//               the counts (coalesced: lanes on consecutive experts);
//   3. rank:    each CTA scans the E counts into offsets[] (CTA 0 writes them),
//               then each warp walks its chunk in order, 32 assignments at a
//               time, ranking equal experts with __match_any_sync, so rows
//               inside an expert follow the assignment order (deterministic);
//   4. gather:  x_disp[row] = x[src_of[row] / top_k] in 16-byte vectors, a
//               warp per wide row or a thread per vector of narrow rows
//               (HBM-bound copy).
// Every pass is parallel over chunks or experts, so the work scales with T.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kChunkWarps = 4;          // warps (chunks) per CTA in count/rank
constexpr int64_t kMinChunk = 256, kMaxChunk = 2048;   // assignments per chunk
constexpr int kBatch = 8;               // 32-assignment batches whose indices load together
constexpr int kScanThreads = 1024;
constexpr int kRankThreads = kChunkWarps * 32;

// Enough chunks to give every SM several warps, each chunk a multiple of
// kBatch * 32 assignments.
int64_t chunk_size(int64_t A)
{
    const int64_t want = A / ((int64_t)device_sm_count() * 8);
    int64_t c = kMinChunk;
    while (c < kMaxChunk && c < want) c *= 2;
    return c;
}
int64_t num_chunks(int64_t A) { return (A + chunk_size(A) - 1) / chunk_size(A); }

__global__ void __launch_bounds__(kChunkWarps * 32)
dispatch_count_kernel(const uint32_t *__restrict__ idx, int64_t A, int E, int64_t special,
                      int64_t chunk, int64_t nchunks, int *__restrict__ chunk_counts,
                      unsigned *status)
{
    extern __shared__ int hist[];
    pdl_wait();
    pdl_launch_dependents();
    const int w = threadIdx.x / 32, lane = (int)lane_id();
    const int64_t c = (int64_t)blockIdx.x * kChunkWarps + w;
    int *h = hist + (size_t)w * E;
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    if (c >= nchunks) return;
    const int64_t a0 = c * chunk;
    const int64_t a1 = a0 + chunk < A ? a0 + chunk : A;
    bool saw_bad = false;
    for (int64_t s0 = a0; s0 < a1; s0 += 32 * kBatch) {
        uint32_t ev[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {          // independent loads in flight
            const int64_t a = s0 + 32 * b + lane;
            ev[b] = a < a1 ? idx[a] : 0xffffffffu;
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const bool act = s0 + 32 * b + lane < a1;
            const bool ok = act && ev[b] < (uint32_t)E;
            // ids in [E, E + special) name special experts: no row, not bad
            saw_bad |= act && !ok && (uint64_t)ev[b] >= (uint64_t)E + (uint64_t)special;
            const unsigned peers = __match_any_sync(kFull, ok ? ev[b] : 0xffffffffu);
            if (ok && lane == __ffs(peers) - 1) atomicAdd(&h[ev[b]], __popc(peers));
        }
    }
    if (__any_sync(kFull, saw_bad) && lane == 0) atomicOr(status, ST_BAD_INDEX);
    __syncwarp();
    for (int e = lane; e < E; e += 32) chunk_counts[c * E + e] = h[e];
}

// CTA b covers experts 32b..32b+31 (one per lane) over all chunks: warp w
// sums a contiguous range of chunks (each load a coalesced 128-byte row
// piece), the 32 warps' sums are scanned through shared memory, and a second
// pass replaces every count by the first row its chunk may use inside the
// expert. Lane sums of warp 31 plus its prefix give the expert's total.
__global__ void __launch_bounds__(kScanThreads)
dispatch_scan_kernel(int *__restrict__ chunk_counts, int64_t nchunks, int E,
                     int32_t *__restrict__ counts)
{
    __shared__ int part[kScanThreads / 32][32];
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int W = kScanThreads / 32;
    const int e = blockIdx.x * 32 + lane;
    const bool live = e < E;
    const int64_t per = (nchunks + W - 1) / W;
    const int64_t c0 = (int64_t)w * per;
    const int64_t c1 = c0 + per < nchunks ? c0 + per : nchunks;
    int local = 0;
    if (live) {
#pragma unroll 8
        for (int64_t c = c0; c < c1; ++c) local += chunk_counts[c * E + e];
    }
    part[w][lane] = local;
    __syncthreads();
    int run = 0, total = 0;
    for (int i = 0; i < W; ++i) {
        if (i < w) run += part[i][lane];
        total += part[i][lane];
    }
    if (live) {
        for (int64_t c = c0; c < c1; ++c) {
            const int v = chunk_counts[c * E + e];
            chunk_counts[c * E + e] = run;
            run += v;
        }
        if (w == 0) counts[e] = total;
    }
}

__global__ void __launch_bounds__(kRankThreads)
dispatch_rank_kernel(const uint32_t *__restrict__ idx, int64_t A, int E, int64_t chunk,
                     int64_t nchunks,
                     const int *__restrict__ chunk_base, const int32_t *__restrict__ counts,
                     int32_t *__restrict__ offsets, int32_t *__restrict__ row_of,
                     int32_t *__restrict__ src_of)
{
    extern __shared__ int smem[];
    int *off = smem;                        // [E + 1] expert offsets
    int *bases = smem + E + 1;              // [kChunkWarps][E] next free row per expert
    __shared__ int warp_tot[kChunkWarps];
    pdl_wait();
    pdl_launch_dependents();
    const int w = threadIdx.x / 32, lane = (int)lane_id();

    // offsets = exclusive scan of counts (each thread owns a run of experts)
    const int per = (E + kRankThreads - 1) / kRankThreads;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) local += counts[e];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[w] = incl;
    __syncthreads();
    int before = 0, total_rows = 0;
    for (int i = 0; i < kChunkWarps; ++i) {
        if (i < w) before += warp_tot[i];
        total_rows += warp_tot[i];
    }
    int run = before + incl - local;
    for (int e = e0; e < e0 + per && e < E; ++e) {
        off[e] = run;
        run += counts[e];
    }
    if (threadIdx.x == 0) off[E] = total_rows;
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += kRankThreads) offsets[e] = off[e];
        // rows past the last one (only when some index was >= E) map to nothing
        for (int64_t r = (int64_t)total_rows + threadIdx.x; r < A; r += kRankThreads) src_of[r] = -1;
    }

    const int64_t c = (int64_t)blockIdx.x * kChunkWarps + w;
    if (c >= nchunks) return;
    int *b = bases + (size_t)w * E;
    for (int e = lane; e < E; e += 32) b[e] = off[e] + chunk_base[c * E + e];
    __syncwarp();
    const int64_t a0 = c * chunk;
    const int64_t a1 = a0 + chunk < A ? a0 + chunk : A;
    const unsigned lt = (1u << lane) - 1u;
    for (int64_t s0 = a0; s0 < a1; s0 += 32 * kBatch) {
        uint32_t ev[kBatch];
#pragma unroll
        for (int bb = 0; bb < kBatch; ++bb) {        // independent loads in flight
            const int64_t a = s0 + 32 * bb + lane;
            ev[bb] = a < a1 ? idx[a] : 0xffffffffu;
        }
#pragma unroll
        for (int bb = 0; bb < kBatch; ++bb) {        // batches in assignment order
            const int64_t a = s0 + 32 * bb + lane;
            const bool act = a < a1;
            const uint32_t e = ev[bb];
            const bool ok = act && e < (uint32_t)E;
            const unsigned peers = __match_any_sync(kFull, ok ? e : 0xffffffffu);
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
}

// x_disp[row] = x[src_of[row] / top_k]. Rows of 32 or more 16-byte vectors:
// one warp per row (lanes on consecutive vectors). Narrower rows: one thread
// per vector of the whole output, so every lane stays busy; per byte when
// rows are not 16-byte multiples.
__global__ void __launch_bounds__(256)
dispatch_gather_rows_kernel(const uint4 *__restrict__ x, int64_t rows, int64_t per_row,
                            int top_k, const int32_t *__restrict__ src_of,
                            uint4 *__restrict__ x_disp)
{
    // the next kernel (the first expert GEMM) is not let in before this
    // copy ends: its resident CTAs would take registers from the copy
    pdl_wait();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < rows;
         r += warps) {
        const int32_t a = src_of[r];
        if (a < 0) continue;
        const uint4 *src = x + (int64_t)(a / top_k) * per_row;
        uint4 *dst = x_disp + r * per_row;
#pragma unroll 4
        for (int64_t v = lane; v < per_row; v += 32) dst[v] = __ldg(src + v);
    }
    pdl_launch_dependents();
}

template <bool VEC>
__global__ void __launch_bounds__(256)
dispatch_gather_kernel(const uint8_t *__restrict__ x, int64_t rows,
                       int64_t row_bytes, int top_k,
                       const int32_t *__restrict__ src_of,
                       uint8_t *__restrict__ x_disp)
{
    pdl_wait();
    const int64_t unit = VEC ? 16 : 1;
    const int64_t per_row = row_bytes / unit;
    const int64_t n = rows * per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t r = i / per_row, v = i - r * per_row;
        const int32_t a = src_of[r];
        if (a < 0) continue;
        const int64_t t = a / top_k;
        if (VEC)
            reinterpret_cast<uint4 *>(x_disp + r * row_bytes)[v] =
                __ldg(reinterpret_cast<const uint4 *>(x + t * row_bytes) + v);
        else
            x_disp[r * row_bytes + v] = x[t * row_bytes + v];
    }
    pdl_launch_dependents();
}

}  // namespace

// Workspace: the per-chunk counts [nchunks][E]. The fused routing-and-count
// path of the one-call forward adds (256-byte aligned) its completion counter.
size_t dispatch_workspace_bytes(int64_t A, int E)
{
    if (A <= 0) return 0;
    return (size_t)num_chunks(A) * (size_t)E * sizeof(int);
}

size_t route_dispatch_workspace_bytes(int64_t A, int E)
{
    if (A <= 0) return 0;
    return (dispatch_workspace_bytes(A, E) + 255) / 256 * 256 + 256;
}

int64_t dispatch_chunk_len(int64_t A) { return chunk_size(A); }

unsigned *dispatch_done_counter(void *ws, int64_t A, int E)
{
    const size_t counts = (size_t)num_chunks(A) * (size_t)E * sizeof(int);
    return reinterpret_cast<unsigned *>(static_cast<uint8_t *>(ws) + (counts + 255) / 256 * 256);
}

cudaError_t launch_dispatch(const uint32_t *idx, int64_t T, int top_k, int E, int64_t special,
                            const void *x, int xdt, int64_t H, int32_t *counts,
                            int32_t *offsets, int32_t *row_of, int32_t *src_of,
                            void *x_disp, void *ws, unsigned *status,
                            cudaStream_t s)
{
    const int64_t A = T * top_k;
    if (A == 0) return cudaSuccess;
    const int64_t chunk_len = chunk_size(A);
    const int64_t nchunks = (A + chunk_len - 1) / chunk_len;
    int *chunk = static_cast<int *>(ws);
    const unsigned blocks = (unsigned)((nchunks + kChunkWarps - 1) / kChunkWarps);
    const size_t hist_bytes = (size_t)kChunkWarps * E * sizeof(int);
    cudaError_t err = launch_pdl(dispatch_count_kernel, dim3(blocks), dim3(kChunkWarps * 32),
                                 hist_bytes, s, idx, A, E, special, chunk_len, nchunks, chunk,
                                 status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(dispatch_scan_kernel, dim3((unsigned)((E + 31) / 32)), dim3(kScanThreads),
                     0, s, chunk, nchunks, E, counts);
    if (err != cudaSuccess) return err;
    return launch_dispatch_rank_gather(idx, T, top_k, E, x, xdt, H, counts, offsets, row_of,
                                       src_of, x_disp, ws, s);
}

cudaError_t launch_dispatch_rank_gather(const uint32_t *idx, int64_t T, int top_k, int E,
                                        const void *x, int xdt, int64_t H, const int32_t *counts,
                                        int32_t *offsets, int32_t *row_of, int32_t *src_of,
                                        void *x_disp, void *ws, cudaStream_t s)
{
    const int64_t A = T * top_k;
    if (A == 0) return cudaSuccess;
    const int64_t chunk_len = chunk_size(A);
    const int64_t nchunks = (A + chunk_len - 1) / chunk_len;
    int *chunk = static_cast<int *>(ws);
    const unsigned blocks = (unsigned)((nchunks + kChunkWarps - 1) / kChunkWarps);
    cudaError_t err = cudaSuccess;
    const size_t rank_bytes = ((size_t)E + 1 + (size_t)kChunkWarps * E) * sizeof(int);
    err = launch_pdl(dispatch_rank_kernel, dim3(blocks), dim3(kRankThreads), rank_bytes, s, idx,
                     A, E, chunk_len, nchunks, (const int *)chunk, (const int32_t *)counts,
                     offsets, row_of,
                     src_of);
    if (err != cudaSuccess) return err;
    const int64_t row_bytes = H * (xdt == DT_F32 ? 4 : 2);
    const bool vec = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(x_disp) % 16 == 0;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    const uint8_t *xb = static_cast<const uint8_t *>(x);
    uint8_t *xd = static_cast<uint8_t *>(x_disp);
    if (vec && row_bytes / 16 >= 32) {
        int64_t gblocks = (A + 7) / 8;
        if (gblocks > cap) gblocks = cap;
        err = launch_pdl(dispatch_gather_rows_kernel, dim3((unsigned)gblocks), dim3(256), 0, s,
                         reinterpret_cast<const uint4 *>(xb), A, row_bytes / 16, top_k,
                         (const int32_t *)src_of, reinterpret_cast<uint4 *>(xd));
    } else {
        const int64_t units = A * (vec ? row_bytes / 16 : row_bytes);
        int64_t gblocks = (units + 255) / 256;
        if (gblocks > cap) gblocks = cap;
        if (vec)
            err = launch_pdl(dispatch_gather_kernel<true>, dim3((unsigned)gblocks), dim3(256), 0,
                             s, xb, A, row_bytes, top_k, (const int32_t *)src_of, xd);
        else
            err = launch_pdl(dispatch_gather_kernel<false>, dim3((unsigned)gblocks), dim3(256),
                             0, s, xb, A, row_bytes, top_k, (const int32_t *)src_of, xd);
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe
