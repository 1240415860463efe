// dispatch.cu -- compact, no-drop dispatch with a saved map.
//
// ruDNN user guide, section 5 "Expert weights and dispatch": no token is
// dropped to enforce a capacity; order inside an expert is unspecified; a
// saved map restores token order.
//
// The A = T*top_k assignments are cut into chunks of 256..8192 (a power of
// two, sized so every SM gets about four), one CTA each with one warp per
// 512 assignments of the chunk:
//   1. count:   per-chunk, per-expert histograms in shared memory (each
//               thread loads four ids per 16-byte read and adds them with
//               shared-memory atomics);
//   2. scan:    one CTA per expert turns its chunk counts (kept contiguous
//               per expert) into the first row each chunk may use inside the
//               expert, and the expert's total;
//   3. rank:    each CTA scans the E counts into offsets[] (CTA 0 writes them);
//               each warp loads its run of up to 512 assignments of the chunk
//               into registers and counts it per expert; the warps' counts
//               are scanned into each warp's first row per expert; then each
//               warp walks its run in order, 32 assignments at a time,
//               ranking equal experts by lane (a peer mask from one ballot
//               per bit of the expert id), so rows inside an expert follow
//               the assignment order (deterministic);
//   4. gather:  x_disp[row] = x[src_of[row] / top_k] in 16-byte vectors, a
//               warp per wide row, a thread per narrow row (at most eight
//               vectors), else a thread per vector (HBM-bound copy).
// Every pass is parallel over chunks or experts, so the work scales with T.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int64_t kMinChunk = 256, kMaxChunk = 8192;   // assignments per chunk
constexpr int kRunBatches = 16;         // 32-assignment batches per warp in the rank pass
constexpr int kRun = 32 * kRunBatches;  // assignments per warp in the rank pass
constexpr int kMaxChunkWarps = (int)(kMaxChunk / kRun);
constexpr int kCountThreads = 512;
constexpr int kCountIds = 16;           // ids per count thread per step (four 16-byte reads)
constexpr int kScanThreads = 256;
#ifndef MOE_TOKEN_GATHER_MIN_BYTES
#define MOE_TOKEN_GATHER_MIN_BYTES (32ll << 20)
#endif
// Rows of at least 512 bytes are gathered in token order once x passes this
// size (a fair share of L2); below it the row-order gather's reads of x hit L2.
constexpr int64_t kTokenGatherMinBytes = MOE_TOKEN_GATHER_MIN_BYTES;

// About four chunks per SM, a power of two of at least 256 assignments (so
// every chunk starts on a 16-byte boundary of the ids).
int64_t chunk_size(int64_t A)
{
    const int64_t want = A / ((int64_t)device_sm_count() * 4);
    int64_t c = kMinChunk;
    while (c < kMaxChunk && c < want) c *= 2;
    return c;
}
int64_t num_chunks(int64_t A) { return (A + chunk_size(A) - 1) / chunk_size(A); }
// warps of the rank pass: one per run of kRun assignments of the chunk
int chunk_warps(int64_t chunk) { return (int)((chunk + kRun - 1) / kRun); }

// CTA c counts chunk c's assignments per expert.
__global__ void __launch_bounds__(kCountThreads)
dispatch_count_kernel(const uint32_t *__restrict__ idx, int64_t A, int E, int64_t special,
                      int64_t chunk, int64_t nchunks, int *__restrict__ chunk_counts,
                      unsigned *status)
{
    extern __shared__ int hist[];                     // [E]
    pdl_wait();
    pdl_launch_dependents();
    const int64_t c = blockIdx.x;
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t a0 = c * chunk;
    const int64_t a1 = a0 + chunk < A ? a0 + chunk : A;
    int bad = 0;
    for (int64_t s0 = a0 + (int64_t)threadIdx.x * 4; s0 < a1;
         s0 += (int64_t)blockDim.x * kCountIds) {
        uint32_t ev[kCountIds];
#pragma unroll
        for (int v = 0; v < kCountIds / 4; ++v) {      // independent loads in flight
            const int64_t a = s0 + (int64_t)v * blockDim.x * 4;
            if (a + 4 <= a1) {
                const uint4 q = *reinterpret_cast<const uint4 *>(idx + a);
                ev[4 * v] = q.x;
                ev[4 * v + 1] = q.y;
                ev[4 * v + 2] = q.z;
                ev[4 * v + 3] = q.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) ev[4 * v + i] = a + i < a1 ? idx[a + i] : (uint32_t)E;
            }
        }
#pragma unroll
        for (int v = 0; v < kCountIds / 4; ++v) {
            const int64_t a = s0 + (int64_t)v * blockDim.x * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t e = ev[4 * v + i];
                if (a + i >= a1) continue;
                if (e < (uint32_t)E) atomicAdd(&hist[e], 1);
                // ids in [E, E + special) name special experts: no row, not bad
                else bad |= (uint64_t)e >= (uint64_t)E + (uint64_t)special;
            }
        }
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, ST_BAD_INDEX);
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(int64_t)e * nchunks + c] = hist[e];
}

// CTA e scans expert e's chunk counts (contiguous: chunk_counts[e][c]) in
// place into the first row each chunk may use inside the expert, and writes
// the expert's total: tiles of kScanThreads * 4 counts, each thread four
// consecutive ones, a block-wide scan of the thread sums per tile.
__global__ void __launch_bounds__(kScanThreads)
dispatch_scan_kernel(int *__restrict__ chunk_counts, int64_t nchunks, int E,
                     int32_t *__restrict__ counts)
{
    __shared__ int wsum[kScanThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    constexpr int W = kScanThreads / 32;
    const int e = blockIdx.x;
    int *col = chunk_counts + (int64_t)e * nchunks;
    int carry = 0;
    for (int64_t t0 = 0; t0 < nchunks; t0 += (int64_t)kScanThreads * 4) {
        const int64_t i0 = t0 + (int64_t)threadIdx.x * 4;
        int v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = i0 + i < nchunks ? col[i0 + i] : 0;
        const int local = v[0] + v[1] + v[2] + v[3];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        if (lane == 31) wsum[w] = incl;
        __syncthreads();
        int before = 0, tile = 0;
        for (int i = 0; i < W; ++i) {
            if (i < w) before += wsum[i];
            tile += wsum[i];
        }
        int run = carry + before + incl - local;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i0 + i < nchunks) col[i0 + i] = run;
            run += v[i];
        }
        carry += tile;
        __syncthreads();                   // wsum is reused by the next tile
    }
    if (threadIdx.x == 0) counts[e] = carry;
}

// Lanes of the warp whose key equals this lane's: the AND over the key's
// nbits bits of the ballot of that bit (or of its complement). Ballots run
// on the integer pipes; __match_any_sync, which computes the same mask, runs
// on the address-divergence unit and was what held this pass back.
template <int NBITS>
__device__ __forceinline__ unsigned peers_of(uint32_t key)
{
    unsigned peers = kFull;
#pragma unroll
    for (int b = 0; b < NBITS; ++b) {
        const bool bit = (key >> b) & 1u;
        const unsigned on = __ballot_sync(kFull, bit);
        peers &= bit ? on : ~on;
    }
    return peers;
}

// Bits of the rank keys: expert ids 0..E-1 and the key 2^NBITS - 1 of ids
// that get no row, above every expert.
int rank_key_bits(int E)
{
    int nbits = 1;
    while ((1 << nbits) <= E) ++nbits;
    return nbits;
}

// CTA c ranks chunk c: warp w owns assignments [a0 + w * kRun, ...) of it.
template <int NBITS>
__global__ void __launch_bounds__(kMaxChunkWarps * 32)
dispatch_rank_kernel(const uint32_t *__restrict__ idx, int64_t A, int E, int64_t chunk,
                     int64_t nchunks,
                     const int *__restrict__ chunk_base, const int32_t *__restrict__ counts,
                     int32_t *__restrict__ offsets, int32_t *__restrict__ row_of,
                     int32_t *__restrict__ src_of, unsigned *status)
{
    (void)status;
    extern __shared__ int smem[];
    const int nw = (int)(blockDim.x / 32);
    int *off = smem;                        // [E + 1] expert offsets
    int *wb = off + E + 1;                  // [warps][E] per-warp counts, then next free row
    __shared__ int warp_tot[kMaxChunkWarps];
    pdl_wait();
    pdl_launch_dependents();
    const int w = threadIdx.x / 32, lane = (int)lane_id();
    const int nthreads = (int)blockDim.x;
    const int64_t c = blockIdx.x;
    const int64_t a0 = c * chunk;
    const int64_t a1 = a0 + chunk < A ? a0 + chunk : A;
    const int64_t r0 = a0 + (int64_t)w * kRun;        // this warp's run
    const int64_t r1 = r0 + kRun < a1 ? r0 + kRun : a1;

    // this warp's ids into registers first (their loads overlap the scan)
    uint32_t ev[kRunBatches];
#pragma unroll
    for (int b = 0; b < kRunBatches; ++b) {
        const int64_t a = r0 + 32 * b + lane;
        ev[b] = a < r1 ? idx[a] : 0xffffffffu;
    }
    for (int i = threadIdx.x; i < nw * E; i += nthreads) wb[i] = 0;

    // offsets = exclusive scan of counts (each thread owns a run of experts)
    const int per = (E + nthreads - 1) / nthreads;
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
    for (int i = 0; i < nw; ++i) {
        if (i < w) before += warp_tot[i];
        total_rows += warp_tot[i];
    }
    int run = before + incl - local;
    for (int e = e0; e < e0 + per && e < E; ++e) {
        off[e] = run;
        run += counts[e];
    }
    if (threadIdx.x == 0) off[E] = total_rows;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += nthreads) offsets[e] = off[e];
        if (threadIdx.x == 0) offsets[E] = total_rows;
        // rows past the last one (only when some index was >= E) map to nothing
        for (int64_t r = (int64_t)total_rows + threadIdx.x; r < A; r += nthreads) src_of[r] = -1;
    }

    // this warp's counts per expert
    int *mine = wb + (size_t)w * E;
#pragma unroll
    for (int b = 0; b < kRunBatches; ++b)
        if (ev[b] < (uint32_t)E) atomicAdd(&mine[ev[b]], 1);
    __syncthreads();
    // each warp's first row per expert: the expert's offset, the rows of the
    // earlier chunks, then those of the earlier warps of this chunk
    for (int e = threadIdx.x; e < E; e += nthreads) {
        int r = off[e] + chunk_base[(int64_t)e * nchunks + c];
        for (int i = 0; i < nw; ++i) {
            const int v = wb[(size_t)i * E + e];
            wb[(size_t)i * E + e] = r;
            r += v;
        }
    }
    __syncthreads();

    // walk the run in order, 32 assignments at a time: equal experts of a
    // batch take consecutive rows in lane order, so rows inside an expert
    // follow the assignment order (deterministic); ids that get no row share
    // the key 2^NBITS - 1, above every expert
    const uint32_t none = (1u << NBITS) - 1u;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int b = 0; b < kRunBatches; ++b) {
        if (r0 + 32 * b >= r1) break;               // uniform across the warp
        const int64_t a = r0 + 32 * b + lane;
        const bool act = a < r1;
        const uint32_t e = ev[b];
        const bool ok = act && e < (uint32_t)E;
        const unsigned peers = peers_of<NBITS>(ok ? e : none);
        int row = -1;
        if (ok) {
            row = mine[e] + __popc(peers & lt);
            // bounds-checking build: the row lies inside the expert's segment
            if (MOE_BOUNDS_OK(row >= off[e] && row < off[e + 1], status)) src_of[row] = (int32_t)a;
            else row = -1;
        }
        if (act) row_of[a] = row;
        __syncwarp();
        if (ok && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
}

// x_disp[row] = x[src_of[row] / top_k]. Rows of 32 or more 16-byte vectors:
// one warp per row (lanes on consecutive vectors). Narrower rows: one thread
// per vector of the whole output, so every lane stays busy; per byte when
// rows are not 16-byte multiples.
__global__ void __launch_bounds__(256)
dispatch_gather_rows_kernel(const uint4 *__restrict__ x, int64_t rows, int64_t per_row,
                            int top_k, const int32_t *__restrict__ src_of,
                            uint4 *__restrict__ x_disp, unsigned *status)
{
    (void)status;
    // the next kernel (the first expert GEMM) is not let in before this
    // copy ends: its resident CTAs would take registers from the copy
    pdl_wait();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < rows;
         r += warps) {
        const int32_t a = src_of[r];
        if (a < 0) continue;
        if (!MOE_BOUNDS_OK((int64_t)a < rows, status)) continue;
        const uint4 *src = x + (int64_t)(a / top_k) * per_row;
        uint4 *dst = x_disp + r * per_row;
#pragma unroll 4
        for (int64_t v = lane; v < per_row; v += 32) dst[v] = __ldg(src + v);
    }
    pdl_launch_dependents();
}

// Rows of PER <= 8 16-byte vectors: one thread per row, four of a thread's
// rows (a grid stride apart) with their map entries and vectors in flight.
template <int PER>
__global__ void __launch_bounds__(256)
dispatch_gather_narrow_kernel(const uint4 *__restrict__ x, int64_t rows, int top_k,
                              const int32_t *__restrict__ src_of, uint4 *__restrict__ x_disp,
                              unsigned *status)
{
    (void)status;
    constexpr int U = 4;
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r0 < rows;
         r0 += U * stride) {
        int32_t a[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t r = r0 + u * stride;
            a[u] = r < rows ? src_of[r] : -1;
            if (a[u] >= 0 && !MOE_BOUNDS_OK((int64_t)a[u] < rows, status)) a[u] = -1;
        }
        uint4 v[U][PER];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (a[u] >= 0) {
                const uint4 *src = x + (int64_t)(a[u] / top_k) * PER;
#pragma unroll
                for (int i = 0; i < PER; ++i) v[u][i] = __ldg(src + i);
            }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (a[u] >= 0) {
                uint4 *dst = x_disp + (r0 + u * stride) * PER;
#pragma unroll
                for (int i = 0; i < PER; ++i) dst[i] = v[u][i];
            }
    }
    pdl_launch_dependents();
}

// Token order: x_disp[row_of[t * top_k + j]] = x[t] for every slot j. A warp
// per token reads its row once, in chunks of 32 lanes x V 16-byte vectors,
// and writes each chunk to the token's dispatched rows; x is then read from
// DRAM once even where it outgrows L2 (the row-order gather reads a token's
// row once per slot). Slots without a row (row_of < 0) are skipped.
template <int V>
__global__ void __launch_bounds__(256)
dispatch_gather_tokens_kernel(const uint4 *__restrict__ x, int64_t T, int64_t per_row,
                              int top_k, int64_t rows, const int32_t *__restrict__ row_of,
                              uint4 *__restrict__ x_disp, unsigned *status)
{
    (void)status;
    (void)rows;
    pdl_wait();
    const int lane = (int)lane_id();
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; t < T;
         t += warps) {
        const uint4 *src = x + t * per_row;
        const int32_t *slots = row_of + t * top_k;
        // the rows of the first 32 slots, one per lane (most top_k fit)
        const int32_t first = lane < top_k ? slots[lane] : -1;
        for (int64_t c0 = 0; c0 < per_row; c0 += 32 * V) {
            uint4 buf[V];
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int64_t c = c0 + lane + 32 * v;
                if (c < per_row) buf[v] = __ldg(src + c);
            }
            for (int j0 = 0; j0 < top_k; j0 += 32) {
                const int jn = top_k - j0 < 32 ? top_k - j0 : 32;
                const int32_t mine = j0 == 0 ? first : (lane < jn ? slots[j0 + lane] : -1);
                for (int j = 0; j < jn; ++j) {
                    const int32_t r = __shfl_sync(kFull, mine, j);
                    if (r < 0 || !MOE_BOUNDS_OK((int64_t)r < rows, status)) continue;
                    uint4 *dst = x_disp + (int64_t)r * per_row;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int64_t c = c0 + lane + 32 * v;
                        if (c < per_row) dst[c] = buf[v];
                    }
                }
            }
        }
    }
    pdl_launch_dependents();
}

template <int PER>
cudaError_t launch_gather_narrow(const uint4 *x, int64_t rows, int top_k, const int32_t *src_of,
                                 uint4 *x_disp, unsigned *status, cudaStream_t s)
{
    int64_t blocks = (rows + 1023) / 1024;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(dispatch_gather_narrow_kernel<PER>, dim3((unsigned)blocks), dim3(256), 0, s,
                      x, rows, top_k, src_of, x_disp, status);
}

template <bool VEC>
__global__ void __launch_bounds__(256)
dispatch_gather_kernel(const uint8_t *__restrict__ x, int64_t rows,
                       int64_t row_bytes, int top_k,
                       const int32_t *__restrict__ src_of,
                       uint8_t *__restrict__ x_disp, unsigned *status)
{
    (void)status;
    pdl_wait();
    const int64_t unit = VEC ? 16 : 1;
    const int64_t per_row = row_bytes / unit;
    const int64_t n = rows * per_row;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t r = i / per_row, v = i - r * per_row;
        const int32_t a = src_of[r];
        if (a < 0) continue;
        if (!MOE_BOUNDS_OK((int64_t)a < rows, status)) continue;
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
    // a thread per kCountIds ids of the chunk (at least a warp, at most 512)
    int64_t cthreads = chunk_len / kCountIds;
    cthreads = cthreads < 32 ? 32 : (cthreads > kCountThreads ? kCountThreads : cthreads);
    cudaError_t err = launch_pdl(dispatch_count_kernel, dim3((unsigned)nchunks),
                                 dim3((unsigned)cthreads), (size_t)E * sizeof(int), s, idx, A,
                                 E, special, chunk_len, nchunks, chunk, status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(dispatch_scan_kernel, dim3((unsigned)E), dim3(kScanThreads), 0, s, chunk,
                     nchunks, E, counts);
    if (err != cudaSuccess) return err;
    return launch_dispatch_rank_gather(idx, T, top_k, E, x, xdt, H, counts, offsets, row_of,
                                       src_of, x_disp, ws, status, s);
}

namespace {

template <int NB>
cudaError_t launch_rank(const uint32_t *idx, int64_t A, int E, int64_t chunk_len,
                        int64_t nchunks, const int *chunk, const int32_t *counts,
                        int32_t *offsets, int32_t *row_of, int32_t *src_of, int nw,
                        size_t rank_bytes, unsigned *status, cudaStream_t s)
{
    if (rank_bytes > 48 * 1024) {
        // up to 16 warps x 1024 experts of counts: past the default 48 KiB
        static std::atomic<uint64_t> opted{0};
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        const uint64_t bit = dev >= 0 && dev < kCachedDevices ? 1ull << dev : 0ull;
        if (bit == 0 || !(opted.load() & bit)) {
            err = cudaFuncSetAttribute(dispatch_rank_kernel<NB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(((size_t)1025 + (size_t)kMaxChunkWarps * 1024) *
                                             sizeof(int)));
            if (err != cudaSuccess) return err;
            opted.fetch_or(bit);
        }
    }
    return launch_pdl(dispatch_rank_kernel<NB>, dim3((unsigned)nchunks), dim3(nw * 32),
                      rank_bytes, s, idx, A, E, chunk_len, nchunks, chunk, counts, offsets,
                      row_of, src_of, status);
}

}  // namespace

cudaError_t launch_dispatch_rank_gather(const uint32_t *idx, int64_t T, int top_k, int E,
                                        const void *x, int xdt, int64_t H, const int32_t *counts,
                                        int32_t *offsets, int32_t *row_of, int32_t *src_of,
                                        void *x_disp, void *ws, unsigned *status, cudaStream_t s)
{
    const int64_t A = T * top_k;
    if (A == 0) return cudaSuccess;
    const int64_t chunk_len = chunk_size(A);
    const int64_t nchunks = (A + chunk_len - 1) / chunk_len;
    int *chunk = static_cast<int *>(ws);
    const int nw = chunk_warps(chunk_len);
    cudaError_t err = cudaSuccess;
    // offsets and the per-warp rows of every expert
    const size_t rank_bytes = ((size_t)E + 1 + (size_t)nw * E) * sizeof(int);
    switch (rank_key_bits(E)) {
#define MOE_RANK(NB)                                                                          \
    case NB: err = launch_rank<NB>(idx, A, E, chunk_len, nchunks, chunk, counts, offsets,     \
                                   row_of, src_of, nw, rank_bytes, status, s); break;
    MOE_RANK(1) MOE_RANK(2) MOE_RANK(3) MOE_RANK(4) MOE_RANK(5) MOE_RANK(6)
    MOE_RANK(7) MOE_RANK(8) MOE_RANK(9) MOE_RANK(10)
#undef MOE_RANK
    default: err = launch_rank<11>(idx, A, E, chunk_len, nchunks, chunk, counts, offsets, row_of,
                                   src_of, nw, rank_bytes, status, s); break;
    }
    if (err != cudaSuccess) return err;
    const int64_t row_bytes = H * (xdt == DT_F32 ? 4 : 2);
    const bool vec = row_bytes % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(x_disp) % 16 == 0;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    const uint8_t *xb = static_cast<const uint8_t *>(x);
    uint8_t *xd = static_cast<uint8_t *>(x_disp);
    const int64_t vpr = row_bytes / 16;
    const uint4 *xv = reinterpret_cast<const uint4 *>(xb);
    uint4 *xdv = reinterpret_cast<uint4 *>(xd);
    const int32_t *so = src_of;
    if (vec && vpr <= 8) {
        switch (vpr) {
        case 1: err = launch_gather_narrow<1>(xv, A, top_k, so, xdv, status, s); break;
        case 2: err = launch_gather_narrow<2>(xv, A, top_k, so, xdv, status, s); break;
        case 3: err = launch_gather_narrow<3>(xv, A, top_k, so, xdv, status, s); break;
        case 4: err = launch_gather_narrow<4>(xv, A, top_k, so, xdv, status, s); break;
        case 5: err = launch_gather_narrow<5>(xv, A, top_k, so, xdv, status, s); break;
        case 6: err = launch_gather_narrow<6>(xv, A, top_k, so, xdv, status, s); break;
        case 7: err = launch_gather_narrow<7>(xv, A, top_k, so, xdv, status, s); break;
        default: err = launch_gather_narrow<8>(xv, A, top_k, so, xdv, status, s); break;
        }
    } else if (vec && row_bytes / 16 >= 32 && T * row_bytes > kTokenGatherMinBytes) {
        int64_t gblocks = (T + 7) / 8;
        if (gblocks > cap) gblocks = cap;
        err = launch_pdl(dispatch_gather_tokens_kernel<8>, dim3((unsigned)gblocks), dim3(256), 0,
                         s, reinterpret_cast<const uint4 *>(xb), T, row_bytes / 16, top_k, A,
                         (const int32_t *)row_of, reinterpret_cast<uint4 *>(xd), status);
    } else if (vec && row_bytes / 16 >= 32) {
        int64_t gblocks = (A + 7) / 8;
        if (gblocks > cap) gblocks = cap;
        err = launch_pdl(dispatch_gather_rows_kernel, dim3((unsigned)gblocks), dim3(256), 0, s,
                         reinterpret_cast<const uint4 *>(xb), A, row_bytes / 16, top_k,
                         (const int32_t *)src_of, reinterpret_cast<uint4 *>(xd), status);
    } else {
        const int64_t units = A * (vec ? row_bytes / 16 : row_bytes);
        int64_t gblocks = (units + 255) / 256;
        if (gblocks > cap) gblocks = cap;
        if (vec)
            err = launch_pdl(dispatch_gather_kernel<true>, dim3((unsigned)gblocks), dim3(256), 0,
                             s, xb, A, row_bytes, top_k, (const int32_t *)src_of, xd, status);
        else
            err = launch_pdl(dispatch_gather_kernel<false>, dim3((unsigned)gblocks), dim3(256),
                             0, s, xb, A, row_bytes, top_k, (const int32_t *)src_of, xd, status);
    }
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace moe
