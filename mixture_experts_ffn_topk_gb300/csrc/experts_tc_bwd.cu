// experts_tc_bwd.cu -- BF16/F16 SwiGLU expert backward on tcgen05 tensor cores.
//
// ruDNN user guide, section 12 "MoE first-order training" (cache.backward of
// SwiGluExperts::forward_dispatched_training). Per dispatched row r of
// expert e, with the forward's cached g = x Wg[e]^T, u = x Wu[e]^T and
// h = SiLU(g) * u, and the expert-output gradient do:
//   DH  dh = do Wd[e]        [rows x I], K = H; the epilogue reads the cached
//                             FP32 g and u and forms
//                             dg = dh * u * s * (1 + g (1 - s)) and
//                             du = dh * g * s (s = sigmoid(g)) into
//                             dgu [rows, 2I] (dg | du) in the input dtype;
//   DX  dx = dg Wg[e] + du Wu[e]   [rows x H], K = 2I;
//   WG  dWd[e] = do^T h  [H x I],  dWg[e] = dg^T x, dWu[e] = du^T x  [I x H],
//       K = the expert's rows; FP32 outputs, zeros for experts without rows.
// Inputs BF16 or F16, FP32 accumulation in tensor memory.
//
// One persistent, warp-specialised kernel per step (one CTA per SM):
//   warp 0     TMA producer, stages of 48 KiB (A 128 x 64, B 256 x 64);
//   warp 1     tcgen05.mma issuer, M=128 N=256 K=16, two TMEM accumulators;
//   warps 2-5  epilogue (tcgen05.ld, math, swizzled staging, line stores).
// Where experts average thousands of rows the same kernel runs on CTA pairs
// (tcgen05 cta_group::2): M = 256 over the two CTAs' 128 rows each, each CTA
// loading its A rows and half of B into 32 KiB stages, so a CTA holds six
// stages (dh five) instead of four (three) and more of the copies' latency
// is covered; the leader issues the MMAs and owns the stage barriers.
// DH's epilogue reads 256 KiB of cached FP32 g / u per tile, one row per lane;
// with four warps those loads, not the MMA, set its pace, so DH runs eight
// epilogue warps (two per TMEM lane quadrant, 128 columns each, 16 columns
// per step to stay within the register file) and three stages to make room
// for their staging buffers; DX and WG keep four stages and four warps.
// Operand layouts: the activation rows of DH and DX are K-major (rows of the
// dispatched matrices, as in the forward). The weights read across their rows
// (Wd as [H][I] for dh, Wg/Wu as [I][H] for dx) and both WG operands (columns
// of row-major activations, reduced over rows) are MN-major: TMA boxes of
// 64 M/N elements (128 bytes) by 64 k-rows with 128-byte swizzle, described
// to the MMA with MN-major shared-memory descriptors (64-element groups 8 KiB
// apart) and the transpose bits of the instruction descriptor.
// WG reduces over an expert's row segment, which starts and ends anywhere, so
// a 64-row block of the whole matrix would mix experts. Instead every expert
// gets its own tensor maps: a small kernel copies each operand's map into the
// workspace once per expert and rewrites its base address (the segment's first
// row) and row count (the segment's length) with tensormap.replace; the TMA
// then zero-fills the rows past the segment by itself, and a NaN row of
// another expert never enters a sum.
//
// Every wait is bounded (p.wait_ns); on expiry the kernel sets ST_TIMEOUT,
// stops issuing work, drains its own copies and MMAs, frees TMEM and exits.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;                  // UMMA M: rows (DH, DX) or weight rows (WG)
constexpr int BN = 256;                  // UMMA N
constexpr int BK = 64;                   // k per stage
constexpr int UK = 16;                   // k per tcgen05.mma kind::f16
constexpr int BOX = 64;                  // MN-major box: 64 elements x 64 k-rows
constexpr int BOX_BYTES = BOX * BK * 2;  // 8 KiB
constexpr int A_BYTES = BM * BK * 2;     // 16 KiB
constexpr int B_BYTES = BN * BK * 2;     // 32 KiB
// a stage: this CTA's A tile and its share of B (all of it, or half on a pair)
template <int CG>
__host__ __device__ constexpr int stage_bytes() { return A_BYTES + B_BYTES / CG; }
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int MAX_E = 1024;
constexpr int EPI_ROW_BYTES = 128;
constexpr int MAP_BYTES = 128;            // one CUtensorMap
constexpr uint64_t kDrainLimitNs = 100000000ull;

enum Mode : int { kDH = 0, kDX = 1, kWG = 2 };

template <int MODE, int CG>
__host__ __device__ constexpr int stages_of()
{
    return CG == 2 ? (MODE == kDH ? 5 : 6) : (MODE == kDH ? 3 : 4);
}
template <int MODE>
__host__ __device__ constexpr int epi_warps_of() { return MODE == kDH ? 8 : 4; }
template <int MODE>
__host__ __device__ constexpr int threads_of() { return 32 * (2 + epi_warps_of<MODE>()); }

template <int MODE, int CG>
struct __align__(1024) BwdSmem {
    static constexpr int STAGES = stages_of<MODE, CG>();
    uint8_t stage[STAGES][stage_bytes<CG>()];
    uint8_t epi[epi_warps_of<MODE>()][32 * EPI_ROW_BYTES];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int prefix[MAX_E + 1];
    int offs[MAX_E + 1];
};
template <int MODE, int CG>
constexpr size_t kBwdSmemBytes = sizeof(BwdSmem<MODE, CG>) + 1024;

struct BwdParams {
    const int32_t *offsets;
    int E;
    int n_tiles;      // N tiles of 256
    int num_k;        // DH: H; DX: I (each half); WG: unused
    int N;            // output columns (DH: I, DX: H, WG: weight columns)
    int M;            // WG: weight rows
    int nprob;        // WG: problems in this launch (1: dWd; 2: dWg, dWu)
    const float *g_plane, *u_plane;     // DH: the cached FP32 g and u [rows, I]
    uint8_t *out0, *out1;               // DH: dgu; DX: dx; WG: W of problem 0 / 1
    int64_t out_row_bytes;              // bytes per output row
    int64_t du_col_bytes;               // DH: byte offset of du inside a dgu row
    const uint8_t *emaps;               // WG: per-expert tensor maps, maps_per_expert each
    int maps_per_expert;                // WG: nprob A maps, then the B map
    unsigned *status;
    uint64_t wait_ns;                   // limit of every bounded wait
};

// Unit id -> (expert, m, n, problem). An m-unit is BM * CG rows (a pair
// computes M = 256, 128 rows per CTA). DH / DX: m-units of an expert's rows,
// m fastest (weight tiles shared through L2). WG: expert slowest, then
// weight-row unit m, then column tile n.
template <int MODE, int CG>
__device__ __forceinline__ void decode(const BwdSmem<MODE, CG> &S, const BwdParams &p, int tile,
                                       int &e, int &m, int &n, int &prob)
{
    if constexpr (MODE == kWG) {
        const int mt = (p.M + BM * CG - 1) / (BM * CG), per = mt * p.n_tiles;
        prob = tile / (p.E * per);
        const int rem = tile - prob * p.E * per;
        e = rem / per;
        const int loc = rem - e * per;
        m = loc / p.n_tiles;
        n = loc - m * p.n_tiles;
    } else {
        int lo = 0, hi = p.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (S.prefix[mid] <= tile) lo = mid; else hi = mid - 1;
        }
        e = lo;
        const int mu = (S.offs[e + 1] - S.offs[e] + BM * CG - 1) / (BM * CG);
        const int local = tile - S.prefix[e];
        n = local / mu;
        m = local - n * mu;
        prob = 0;
    }
}

template <int MODE, int CG>
__device__ __forceinline__ int k_blocks(const BwdSmem<MODE, CG> &S, const BwdParams &p, int e)
{
    if constexpr (MODE == kDH) return (p.num_k + BK - 1) / BK;
    else if constexpr (MODE == kDX) return 2 * ((p.num_k + BK - 1) / BK);
    else return (S.offs[e + 1] - S.offs[e] + BK - 1) / BK;
}

// Writes 32 rows x 128 bytes (this lane's row in v[]) through the warp's
// swizzled staging buffer so that each store instruction covers four whole
// 128-byte row segments. Row rr goes to base + rr * row_bytes + col_byte when
// rr < rows_valid and the column is below col_limit (bytes).
__device__ __forceinline__ void emit_rows(uint8_t *stg, const uint32_t (&v)[32], uint8_t *base,
                                          int64_t row_bytes, int64_t col_byte,
                                          int64_t col_limit, int rows_valid)
{
    const int lane = threadIdx.x & 31, cch = lane & 7;
#pragma unroll
    for (int p = 0; p < 8; ++p)
        *reinterpret_cast<uint4 *>(stg + lane * EPI_ROW_BYTES + ((p ^ (lane & 7)) << 4)) =
            make_uint4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
    __syncwarp();
    const int64_t cb = col_byte + cch * 16;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int rr = 4 * j + (lane >> 3);
        const uint4 q = *reinterpret_cast<const uint4 *>(stg + rr * EPI_ROW_BYTES +
                                                         ((cch ^ (rr & 7)) << 4));
        if (rr < rows_valid && cb < col_limit)
            *reinterpret_cast<uint4 *>(base + rr * row_bytes + cb) = q;
    }
    __syncwarp();
}

// Orders this thread's later TMA copies through a tensor map in global
// memory after the tensormap.replace writes that produced it.
__device__ __forceinline__ void tensormap_acquire(const void *map)
{
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

// Per-expert tensor maps for the weight-gradient GEMMs: for expert e and map
// j, a copy of base[j] whose base address is the expert's first row and whose
// row count is the expert's (at least 1), at out + (e * nmaps + j) * 128.
// One warp per expert builds its maps in shared memory (lanes 8j..8j+7 copy
// map j, lane j rewrites its address and row count there), then the warp
// publishes each whole 128-byte map with one tensormap.cp_fenceproxy copy,
// which releases it to the tensormap proxy that the consumers' TMA copies
// read it through (after their acquire fence): no map is ever visible in
// global memory half old and half new.
__global__ void __launch_bounds__(32)
expert_maps_kernel(const __grid_constant__ CUtensorMap base0, const __grid_constant__ CUtensorMap base1,
                   const __grid_constant__ CUtensorMap base2, uint64_t addr0, uint64_t addr1,
                   uint64_t addr2, int64_t stride0, int64_t stride1, int64_t stride2, int nmaps,
                   const int32_t *__restrict__ offsets, uint8_t *__restrict__ out)
{
    __shared__ __align__(128) uint8_t sm[3 * MAP_BYTES];
    pdl_wait();
    const int e = blockIdx.x, lane = threadIdx.x;
    const int r0 = offsets[e], rows = offsets[e + 1] - r0;
    uint8_t *slot = out + (size_t)e * nmaps * MAP_BYTES;
    if (lane < 8 * nmaps) {
        const int j = lane >> 3, c = lane & 7;
        const CUtensorMap *src = j == 0 ? &base0 : j == 1 ? &base1 : &base2;
        reinterpret_cast<uint4 *>(sm + j * MAP_BYTES)[c] = reinterpret_cast<const uint4 *>(src)[c];
    }
    __syncwarp();
    if (lane < nmaps) {
        const uint64_t a = lane == 0 ? addr0 : lane == 1 ? addr1 : addr2;
        const int64_t st = lane == 0 ? stride0 : lane == 1 ? stride1 : stride2;
        const uint32_t map = smem_u32(sm + lane * MAP_BYTES);
        const uint64_t first = a + (uint64_t)((int64_t)r0 * st);
        const uint32_t n = (uint32_t)(rows > 0 ? rows : 1);
        asm volatile("tensormap.replace.tile.global_address.shared::cta.b1024.b64 [%0], %1;"
                     ::"r"(map), "l"(first) : "memory");
        asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], 1, %1;"
                     ::"r"(map), "r"(n) : "memory");
    }
    __syncwarp();
    for (int j = 0; j < nmaps; ++j)
        asm volatile("tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu"
                     ".sync.aligned [%0], [%1], 128;"
                     ::"l"(slot + j * MAP_BYTES), "r"(smem_u32(sm + j * MAP_BYTES)) : "memory");
    pdl_launch_dependents();
}

template <int DT, int MODE, int CG>
__global__ void __launch_bounds__(threads_of<MODE>(), 1)
bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                const BwdParams p)
{
    constexpr int STAGES = stages_of<MODE, CG>();
    constexpr int STAGE_BYTES = stage_bytes<CG>();
    constexpr int B_BOXES = BN / BOX / CG;          // MN-major B boxes this CTA loads per stage
    constexpr int EPI_WARPS = epi_warps_of<MODE>();
    constexpr int THREADS = threads_of<MODE>();
    constexpr int MU = BM * CG;                     // rows of an m-unit
    extern __shared__ uint8_t smem_raw[];
    BwdSmem<MODE, CG> &S = *reinterpret_cast<BwdSmem<MODE, CG> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned *status = p.status;
    // CTA pair: rank 0 issues the MMAs (M = 256 over both CTAs' A rows and
    // B halves) and owns the stage barriers both CTAs' copies complete on
    const int rank = CG == 2 ? (int)cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / CG, unit_step = (int)gridDim.x / CG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&S.full[s], 1); mbar_init(&S.empty[s], 1); }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&S.acc_full[a], 1);
            mbar_init(&S.acc_empty[a], EPI_WARPS * CG);
        }
        mbar_init(&S.drain, 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc<CG>(&S.tmem_base, TMEM_COLS);
        tmem_relinquish<CG>();
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int i = threadIdx.x; i <= p.E; i += THREADS) S.offs[i] = p.offsets[i];
    __syncthreads();
    if (MODE != kWG && warp == 0) {
        // prefix[e] = units of experts < e (lane l owns a contiguous run)
        const int per = (p.E + 31) / 32, e0 = lane * per;
        int local = 0;
        for (int e = e0; e < e0 + per && e < p.E; ++e)
            local += (S.offs[e + 1] - S.offs[e] + MU - 1) / MU * p.n_tiles;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int e = e0; e < e0 + per && e < p.E; ++e) {
            S.prefix[e] = run;
            run += (S.offs[e + 1] - S.offs[e] + MU - 1) / MU * p.n_tiles;
        }
        if (lane == 31) S.prefix[p.E] = incl;
    }
    tc_fence_before();
    // a pair also makes each CTA's barrier initialisation visible to the
    // other before any copy or arrival targets it
    if constexpr (CG == 2) cluster_sync();
    else __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = S.tmem_base;
    const int total_tiles = MODE == kWG ? p.nprob * p.E * ((p.M + MU - 1) / MU) * p.n_tiles
                                        : S.prefix[p.E];
    volatile int *abort_flag = &S.abort;
    uint32_t filled_mask = 0, filled_parity = 0;       // producer: stages in flight

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = unit0; tile < total_tiles && ok; tile += unit_step) {
            int e, m, n, prob;
            decode<MODE, CG>(S, p, tile, e, m, n, prob);
            const int nkb = k_blocks<MODE, CG>(S, p, e);
            const int seg0 = S.offs[e];
            const int a_row = m * MU + rank * BM;               // this CTA's first A row / M element
            const int b_col = n * BN + rank * (BN / CG);        // this CTA's first B column
            const CUtensorMap *wa = nullptr, *wb = nullptr;
            if constexpr (MODE == kWG) {
                const uint8_t *maps = p.emaps + (size_t)e * p.maps_per_expert * MAP_BYTES;
                wa = reinterpret_cast<const CUtensorMap *>(maps + prob * MAP_BYTES);
                wb = reinterpret_cast<const CUtensorMap *>(maps + (p.maps_per_expert - 1) * MAP_BYTES);
                if (nkb > 0) {
                    tensormap_acquire(wa);
                    tensormap_acquire(wb);
                }
            }
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait<CG>(&S.empty[stage], phase ^ 1u, abort_flag, status, p.wait_ns)) { ok = false; break; }
                uint8_t *sa = S.stage[stage];
                uint8_t *sb = sa + A_BYTES;
                // both CTAs' copies complete on the leader's barrier, which
                // expects both; a peer's copy may land before the leader arms
                // it (the phase cannot complete while the leader's arrival is
                // pending)
                if (leader) mbar_arrive_expect_tx(&S.full[stage], CG * STAGE_BYTES);
                const uint32_t bar = CG == 2 ? mapa_shared(smem_u32(&S.full[stage]), 0)
                                             : smem_u32(&S.full[stage]);
                auto load2 = [&](void *dst, const CUtensorMap *map, int c0, int c1) {
                    if constexpr (CG == 2) tma_load_2d_pair(dst, map, bar, c0, c1);
                    else tma_load_2d(dst, map, &S.full[stage], c0, c1);
                };
                auto load3 = [&](void *dst, const CUtensorMap *map, int c0, int c1, int c2) {
                    if constexpr (CG == 2) tma_load_3d_pair(dst, map, bar, c0, c1, c2);
                    else tma_load_3d(dst, map, &S.full[stage], c0, c1, c2);
                };
                if constexpr (MODE == kDH) {
                    load2(sa, &tmA0, kb * BK, seg0 + a_row);
#pragma unroll
                    for (int j = 0; j < B_BOXES; ++j)
                        load3(sb + j * BOX_BYTES, &tmB0, b_col + j * BOX, kb * BK, e);
                } else if constexpr (MODE == kDX) {
                    const int half = (p.num_k + BK - 1) / BK;
                    const bool second = kb >= half;
                    const int kk = (second ? kb - half : kb) * BK;
                    load2(sa, second ? &tmA1 : &tmA0, kk, seg0 + a_row);
#pragma unroll
                    for (int j = 0; j < B_BOXES; ++j)
                        load3(sb + j * BOX_BYTES, second ? &tmB1 : &tmB0, b_col + j * BOX, kk, e);
                } else {
                    // rows relative to the expert's own maps: past its last row
                    // the TMA fills zeros
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        load2(sa + j * BOX_BYTES, wa, a_row + j * BOX, kb * BK);
#pragma unroll
                    for (int j = 0; j < B_BOXES; ++j)
                        load2(sb + j * BOX_BYTES, wb, b_col + j * BOX, kb * BK);
                }
                filled_mask |= 1u << stage;
                filled_parity = (filled_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_f16_major<DT>(BM * CG, BN, MODE == kWG, true);
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        for (int tile = unit0; tile < total_tiles && ok; tile += unit_step, ++it) {
            int e, m, n, prob;
            decode<MODE, CG>(S, p, tile, e, m, n, prob);
            const int nkb = k_blocks<MODE, CG>(S, p, e);
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait<CG>(&S.acc_empty[acc], acc_phase ^ 1u, abort_flag, status, p.wait_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(acc * ACC_COLS);
            for (int kb = 0; kb < nkb; ++kb) {
                if (!mbar_wait<CG>(&S.full[stage], phase, abort_flag, status, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(S.stage[stage]);
                const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
                for (int k = 0; k < BK / UK; ++k) {
                    const uint64_t ad = MODE == kWG ? sdesc_mn_sw128(a0 + k * UK * 128, BOX_BYTES)
                                                    : sdesc_k_sw128(a0 + k * UK * 2);
                    const uint64_t bd = sdesc_mn_sw128(b0 + k * UK * 128, BOX_BYTES);
                    umma_f16<CG>(d, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                }
                if constexpr (CG == 2) umma_commit_pair(&S.empty[stage]);
                else umma_commit<1>(&S.empty[stage]);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            // (an expert without rows commits with no MMA: its epilogue writes zeros)
            if (ok) {
                if constexpr (CG == 2) umma_commit_pair(&S.acc_full[acc]);
                else umma_commit<1>(&S.acc_full[acc]);
            }
        }
        if (*abort_flag) {
            // every MMA issued so far must finish before TMEM is released
            umma_commit<CG>(&S.drain);
            mbar_wait(&S.drain, 0, nullptr, status, kDrainLimitNs);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------ epilogue
        const int q = warp & 3;                    // TMEM lane quadrant (fixed by the warp id)
        static_assert(MODE == kDH || EPI_WARPS == 4, "only DH splits columns over two warps");
        uint8_t *stg = S.epi[warp - 2];
        int it = 0;
        for (int tile = unit0; tile < total_tiles; tile += unit_step, ++it) {
            int e, m, n, prob;
            decode<MODE, CG>(S, p, tile, e, m, n, prob);
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            const bool ready = mbar_wait<CG>(&S.acc_full[acc], acc_phase, abort_flag, status, p.wait_ns);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            if constexpr (MODE == kWG) {
                // rows: weight rows m*MU + rank*128 + q*32 + r; FP32, 32 columns
                // per round; the next round's tensor-memory load is in flight
                // while the current one is stored
                const int row0 = m * MU + rank * BM + q * 32;
                const int rows_valid = p.M - row0;
                const bool empty_expert = S.offs[e + 1] == S.offs[e];
                uint8_t *W = (prob ? p.out1 : p.out0) + ((int64_t)e * p.M + row0) * p.out_row_bytes;
                constexpr int CHUNKS = BN / 32;
                uint32_t v[32];
                if (empty_expert) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0u;
                } else {
                    tmem_ld32(tbase, v);
                    tmem_ld_wait(v);
                }
#pragma unroll 2
                for (int rd = 0; rd < CHUNKS; ++rd) {
                    uint32_t vn[32];
                    const bool more = rd + 1 < CHUNKS && !empty_expert;
                    if (more) tmem_ld32(tbase + (rd + 1) * 32, vn);
                    emit_rows(stg, v, W, p.out_row_bytes, (int64_t)(n * BN + rd * 32) * 4,
                              p.out_row_bytes, rows_valid);
                    if (more) {
                        tmem_ld_wait(vn);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = vn[i];
                    }
                }
            } else {
                const int seg_rows = S.offs[e + 1] - S.offs[e];
                const int r_seg = m * MU + rank * BM + q * 32;          // warp's first row in the segment
                const int rows_valid = seg_rows - r_seg;
                const int64_t grow0 = (int64_t)S.offs[e] + r_seg;       // its dispatched row
                uint8_t *ob = p.out0 + grow0 * p.out_row_bytes;
                const int64_t col_limit = (int64_t)p.N * 2;
#pragma unroll 1
                for (int rd = 0; rd < BN / 64; ++rd) {
                    uint32_t v0[32];
                    if constexpr (MODE == kDX) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t d[32];
                            tmem_ld32(tbase + (rd * 2 + half) * 32, d);
                            tmem_ld_wait(d);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                v0[half * 16 + i] = pack2<DT>(__uint_as_float(d[2 * i]),
                                                              __uint_as_float(d[2 * i + 1]));
                        }
                        emit_rows(stg, v0, ob, p.out_row_bytes, (int64_t)(n * BN + rd * 64) * 2,
                                  col_limit, rows_valid);
                    } else {
                        // this warp: 128 of the tile's 256 columns, 64 per round, 16 per step
                        const int col_half = (warp - 2) >> 2;
                        if (rd >= 2) break;
                        const int cbase = col_half * 128 + rd * 64;        // column in the tile
                        uint32_t v1[32];
                        const bool row_ok = lane < rows_valid;
                        const int64_t grow = grow0 + lane;
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd) {
                            const int col0 = n * BN + cbase + qd * 16;
                            uint32_t d[16];
                            tmem_ld16(tbase + cbase + qd * 16, d);
                            // the cached FP32 g and u of these 16 columns of this lane's row
                            float4 gv[4], uv[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                if (row_ok && col0 + 4 * c < p.N) {
                                    const int64_t off = grow * p.N + col0 + 4 * c;
                                    gv[c] = *reinterpret_cast<const float4 *>(p.g_plane + off);
                                    uv[c] = *reinterpret_cast<const float4 *>(p.u_plane + off);
                                } else {
                                    gv[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                                    uv[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                                }
                            }
                            tmem_ld_wait16(d);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 g4 = gv[i / 2], u4 = uv[i / 2];
                                const float2 g = (i & 1) ? make_float2(g4.z, g4.w) : make_float2(g4.x, g4.y);
                                const float2 u = (i & 1) ? make_float2(u4.z, u4.w) : make_float2(u4.x, u4.y);
                                const float dh0 = __uint_as_float(d[2 * i]);
                                const float dh1 = __uint_as_float(d[2 * i + 1]);
                                const float s0 = 1.0f / (1.0f + __expf(-g.x));
                                const float s1 = 1.0f / (1.0f + __expf(-g.y));
                                v0[qd * 8 + i] = pack2<DT>(dh0 * u.x * s0 * (1.0f + g.x * (1.0f - s0)),
                                                           dh1 * u.y * s1 * (1.0f + g.y * (1.0f - s1)));
                                v1[qd * 8 + i] = pack2<DT>(dh0 * g.x * s0, dh1 * g.y * s1);
                            }
                        }
                        const int64_t cb = (int64_t)(n * BN + cbase) * 2;
                        emit_rows(stg, v0, ob, p.out_row_bytes, cb, col_limit, rows_valid);
                        emit_rows(stg, v1, ob + p.du_col_bytes, p.out_row_bytes, cb, col_limit,
                                  rows_valid);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (CG == 2 && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&S.acc_empty[acc]), 0));
                else mbar_arrive(&S.acc_empty[acc]);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        if (CG == 1 || leader) {
            // let the outstanding TMA copies land before shared memory goes
            for (int s = 0; s < STAGES; ++s)
                if (filled_mask >> s & 1u)
                    mbar_wait(&S.full[s], filled_parity >> s & 1u, nullptr, status, kDrainLimitNs);
        } else {
            // a peer's copies complete on the leader's barriers, which it
            // cannot wait on: give them the same bounded time to land
            const uint64_t t0 = global_timer_ns();
            while (global_timer_ns() - t0 < kDrainLimitNs) { }
        }
    }
    // a pair keeps both CTAs (their shared memory is read by the leader's
    // MMAs and signalled by its commits) until both are done
    if constexpr (CG == 2) cluster_sync();
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
    }
}

// ---- host side ---------------------------------------------------------------

// Experts averaging at least this many rows run the backward GEMMs on CTA
// pairs: a CTA then holds 32 KiB stages instead of 48, so six fit (five
// beside dh's eight staging buffers), and more of the copies' latency is
// covered. With a few hundred rows per expert (weight gradients reducing over
// K = 384) the pairs measured slower.
#ifndef MOE_BWD_PAIR_MIN_ROWS
#define MOE_BWD_PAIR_MIN_ROWS 2048
#endif
// Which launches may pair (bit 0: dh, bit 1: dx, bit 2: weight gradients).
#ifndef MOE_BWD_PAIR_MODES
#define MOE_BWD_PAIR_MODES 7
#endif

template <int DT, int MODE, int CG>
cudaError_t launch_step_cg(int64_t units, const CUtensorMap &a0, const CUtensorMap &a1,
                           const CUtensorMap &b0, const CUtensorMap &b1, const BwdParams &p,
                           cudaStream_t s)
{
    static std::atomic<uint64_t> done_mask{0};
    static std::atomic<int> pairs_cached[kCachedDevices];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const bool use_cache = dev >= 0 && dev < kCachedDevices;
    const uint64_t bit = use_cache ? 1ull << dev : 0ull;
    if (bit == 0 || !(done_mask.load() & bit)) {
        err = cudaFuncSetAttribute(bwd_gemm_kernel<DT, MODE, CG>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kBwdSmemBytes<MODE, CG>);
        if (err != cudaSuccess) return err;
        done_mask.fetch_or(bit);
    }
    const int64_t sms = device_sm_count();
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(threads_of<MODE>());
    cfg.dynamicSmemBytes = kBwdSmemBytes<MODE, CG>;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CG;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    int grid = 0;
    if constexpr (CG == 1) {
        grid = (int)(units < sms ? (units < 1 ? 1 : units) : sms);
        cfg.numAttrs = 1;
    } else {
        // one wave of pairs: as many as the GPU holds at once (cluster
        // placement can leave SMs unpaired)
        int pairs = use_cache ? pairs_cached[dev].load() : 0;
        if (pairs == 0) {
            cudaLaunchConfig_t q = cfg;
            q.gridDim = dim3((unsigned)(sms & ~int64_t(1)));
            q.attrs = &attr[1];
            q.numAttrs = 1;
            err = cudaOccupancyMaxActiveClusters(&pairs, bwd_gemm_kernel<DT, MODE, CG>, &q);
            if (err != cudaSuccess) return err;
            if (pairs < 1) return cudaErrorInvalidConfiguration;
            if (use_cache) pairs_cached[dev].store(pairs);
        }
        grid = 2 * (int)(units < pairs ? (units < 1 ? 1 : units) : pairs);
        cfg.numAttrs = 2;
    }
    cfg.gridDim = dim3((unsigned)grid);
    return cudaLaunchKernelEx(&cfg, bwd_gemm_kernel<DT, MODE, CG>, a0, a1, b0, b1, p);
}

// units1 / units2: upper bounds on the launch's work units with m-units of
// 128 rows (single CTAs) and of 256 (pairs)
template <int DT, int MODE>
cudaError_t launch_step(bool pair, int64_t units1, int64_t units2, const CUtensorMap &a0,
                        const CUtensorMap &a1, const CUtensorMap &b0, const CUtensorMap &b1,
                        const BwdParams &p, cudaStream_t s)
{
    if (pair && (MOE_BWD_PAIR_MODES >> MODE & 1))
        return launch_step_cg<DT, MODE, 2>(units2, a0, a1, b0, b1, p, s);
    return launch_step_cg<DT, MODE, 1>(units1, a0, a1, b0, b1, p, s);
}

template <int DT>
cudaError_t launch_backward(const void *x_disp, const int32_t *offsets, int64_t rows,
                            const void *gate, const void *up, const void *down, int E, int64_t H,
                            int64_t I, const void *cache, const void *dout, void *dgu, void *dx,
                            float *dgate, float *dup, float *ddown, void *maps_ws,
                            unsigned *status, cudaStream_t s)
{
    const CUtensorMapDataType tdt =
        DT == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t R = (uint64_t)(rows > 0 ? rows : 1);
    if (rows == 0) {
        // no activation rows: only the zero weight gradients are written and no
        // activation tensor map below is ever read; gate stands in for the
        // absent pointers
        dout = cache = x_disp = gate;
        dgu = const_cast<void *>(gate);
    }
    const uint8_t *cb = static_cast<const uint8_t *>(cache);
    const float *g_plane = reinterpret_cast<const float *>(cb + rows * I * 2);
    const uint8_t *dgu_b = static_cast<const uint8_t *>(dgu);
    // DH: dout rows (K-major) x Wd[e] read as [H][I] (MN-major)
    // DX: dg / du column views of dgu (K-major) x Wg[e], Wu[e] read as [I][H]
    // WG: columns of do / dg / du (MN-major) x columns of h / x (MN-major),
    //     per expert (the maps below are the templates the expert maps copy)
    CUtensorMap dh_a, dh_b, dx_a0, dx_a1, dx_b0, dx_b1, wd_a, wd_b, wgu_a0, wgu_a1, wgu_b;
    if (!encode_2d(&dh_a, tdt, dout, (uint64_t)H, R, BK, BM) ||
        !encode_3d(&dh_b, tdt, down, (uint64_t)I, (uint64_t)H, (uint64_t)E, BOX, BK) ||
        !encode_2d_strided(&dx_a0, tdt, dgu_b, (uint64_t)I, R, (uint64_t)(4 * I), BK, BM) ||
        !encode_2d_strided(&dx_a1, tdt, dgu_b + 2 * I, (uint64_t)I, R, (uint64_t)(4 * I), BK, BM) ||
        !encode_3d(&dx_b0, tdt, gate, (uint64_t)H, (uint64_t)I, (uint64_t)E, BOX, BK) ||
        !encode_3d(&dx_b1, tdt, up, (uint64_t)H, (uint64_t)I, (uint64_t)E, BOX, BK) ||
        !encode_2d(&wd_a, tdt, dout, (uint64_t)H, R, BOX, BK) ||
        !encode_2d(&wd_b, tdt, cb, (uint64_t)I, R, BOX, BK) ||
        !encode_2d_strided(&wgu_a0, tdt, dgu_b, (uint64_t)I, R, (uint64_t)(4 * I), BOX, BK) ||
        !encode_2d_strided(&wgu_a1, tdt, dgu_b + 2 * I, (uint64_t)I, R, (uint64_t)(4 * I), BOX, BK) ||
        !encode_2d(&wgu_b, tdt, x_disp, (uint64_t)H, R, BOX, BK))
        return cudaErrorInvalidValue;

    // per-expert maps: [E][2] for dWd (do, h), then [E][3] for dWg / dWu (dg, du, x)
    uint8_t *maps_d = static_cast<uint8_t *>(maps_ws);
    uint8_t *maps_gu = maps_d + (size_t)E * 2 * MAP_BYTES;
    const uint64_t a_dout = reinterpret_cast<uint64_t>(dout), a_h = reinterpret_cast<uint64_t>(cb);
    const uint64_t a_dg = reinterpret_cast<uint64_t>(dgu_b), a_du = a_dg + 2 * I;
    const uint64_t a_x = reinterpret_cast<uint64_t>(x_disp);
    cudaError_t err = launch_pdl(expert_maps_kernel, dim3((unsigned)E), dim3(32), 0, s, wd_a, wd_b,
                                 wd_b, a_dout, a_h, a_h, (int64_t)(2 * H), (int64_t)(2 * I),
                                 (int64_t)(2 * I), 2, offsets, maps_d);
    if (err != cudaSuccess) return err;
    err = launch_pdl(expert_maps_kernel, dim3((unsigned)E), dim3(32), 0, s, wgu_a0, wgu_a1, wgu_b,
                     a_dg, a_du, a_x, (int64_t)(4 * I), (int64_t)(4 * I), (int64_t)(2 * H), 3,
                     offsets, maps_gu);
    if (err != cudaSuccess) return err;

    const bool pair = rows >= (int64_t)MOE_BWD_PAIR_MIN_ROWS * E;
    BwdParams p{};
    p.offsets = offsets;
    p.E = E;
    p.status = status;
    p.wait_ns = wait_limit_ns();
    if (rows > 0) {
        const int64_t mt = rows / BM + (rows < E ? rows : E);     // M-tiles, upper bound
        const int64_t mt2 = rows / (2 * BM) + (rows < E ? rows : E);   // pair m-units
        // DH: dh, then dg / du into dgu
        p.n_tiles = (int)((I + BN - 1) / BN);
        p.num_k = (int)H;
        p.N = (int)I;
        p.g_plane = g_plane;
        p.u_plane = g_plane + rows * I;
        p.out0 = static_cast<uint8_t *>(dgu);
        p.out_row_bytes = 4 * I;
        p.du_col_bytes = 2 * I;
        err = launch_step<DT, kDH>(pair, mt * p.n_tiles, mt2 * p.n_tiles, dh_a, dh_a, dh_b, dh_b, p, s);
        if (err != cudaSuccess) return err;
        // DX
        p.n_tiles = (int)((H + BN - 1) / BN);
        p.num_k = (int)I;
        p.N = (int)H;
        p.out0 = static_cast<uint8_t *>(dx);
        p.out_row_bytes = 2 * H;
        err = launch_step<DT, kDX>(pair, mt * p.n_tiles, mt2 * p.n_tiles, dx_a0, dx_a1, dx_b0, dx_b1, p, s);
        if (err != cudaSuccess) return err;
    }
    // WG: dWd (M = H rows of Wd, N = I)
    p.M = (int)H;
    p.N = (int)I;
    p.n_tiles = (int)((I + BN - 1) / BN);
    p.nprob = 1;
    p.out0 = reinterpret_cast<uint8_t *>(ddown);
    p.out1 = nullptr;
    p.out_row_bytes = 4 * I;
    p.emaps = maps_d;
    p.maps_per_expert = 2;
    err = launch_step<DT, kWG>(pair, (int64_t)E * ((H + BM - 1) / BM) * p.n_tiles,
                               (int64_t)E * ((H + 2 * BM - 1) / (2 * BM)) * p.n_tiles, wd_a, wd_a,
                               wd_b, wd_b, p, s);
    if (err != cudaSuccess) return err;
    // WG: dWg, dWu (M = I rows, N = H)
    p.M = (int)I;
    p.N = (int)H;
    p.n_tiles = (int)((H + BN - 1) / BN);
    p.nprob = 2;
    p.out0 = reinterpret_cast<uint8_t *>(dgate);
    p.out1 = reinterpret_cast<uint8_t *>(dup);
    p.out_row_bytes = 4 * H;
    p.emaps = maps_gu;
    p.maps_per_expert = 3;
    return launch_step<DT, kWG>(pair, 2 * (int64_t)E * ((I + BM - 1) / BM) * p.n_tiles,
                                2 * (int64_t)E * ((I + 2 * BM - 1) / (2 * BM)) * p.n_tiles, wgu_a0,
                                wgu_a1, wgu_b, wgu_b, p, s);
}

}  // namespace

size_t experts_tc_backward_maps_bytes(int E) { return (size_t)E * 5 * MAP_BYTES; }

cudaError_t launch_experts_tc_backward(int dt, const void *x_disp, const int32_t *offsets,
                                       int64_t rows, const void *gate, const void *up,
                                       const void *down, int E, int64_t H, int64_t I,
                                       const void *cache, const void *dout, void *dgu_ws,
                                       void *maps_ws, void *dx, float *dgate, float *dup,
                                       float *ddown, unsigned *status, cudaStream_t s)
{
    if (dt == DT_BF16)
        return launch_backward<DT_BF16>(x_disp, offsets, rows, gate, up, down, E, H, I, cache,
                                        dout, dgu_ws, dx, dgate, dup, ddown, maps_ws, status, s);
    return launch_backward<DT_F16>(x_disp, offsets, rows, gate, up, down, E, H, I, cache, dout,
                                   dgu_ws, dx, dgate, dup, ddown, maps_ws, status, s);
}

}  // namespace moe
