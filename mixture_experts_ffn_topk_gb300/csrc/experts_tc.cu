// experts_tc.cu -- BF16/F16 bias-free SwiGLU experts on tcgen05 tensor cores.
//
// ruDNN user guide, sections 3 and 5: per dispatched row r of expert e,
//   h_r = SiLU(x_r Wg[e]^T) * (x_r Wu[e]^T),   out_r = h_r Wd[e]^T,
// gate/up [E,I,H], down [E,H,I] (aclnnFFN "Formula" with no bias and a SwiGLU
// activation). Inputs BF16 or F16, FP32 accumulation in tensor memory, h
// rounded to the input dtype between the two GEMMs.
//
// Two launches of one persistent, warp-specialised grouped GEMM:
//   GEMM1 (SWIGLU):  B tile = 128 gate rows stacked on 128 up rows of the
//                    same output columns; one 128x256x16 MMA computes both;
//                    the epilogue forms SiLU(g)*u for 128 columns of h.
//   GEMM2:           B tile = 256 rows of down; the epilogue writes FP32 or
//                    rounds to dtype (the caller's choice of output type), or,
//                    in the one-call forward, multiplies each row by its
//                    routing weight and reduces it in FP32 into its token's
//                    row of y_acc [T, H] (red.global.add.v4.f32; the combine).
// Per CTA (one per SM, 192 threads):
//   warp 0  TMA producer: x tile [128 rows x 64 k] and weight tile
//           [256 rows x 64 k] per stage, 128-byte swizzle, 4 stages;
//   warp 1  MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M=128 N=256 K=16,
//           accumulators double-buffered in TMEM (2 x 256 columns);
//   warps 2-5  epilogue: tcgen05.ld 32 lanes x 32 columns, math, then a
//           swizzled shared-memory hop so every store writes whole lines.
// Paired form (CG = 2, a cluster of two CTAs on two SMs): the pair computes
// a 256 x 256 tile with tcgen05.mma.cta_group::2 (M=256): each CTA holds its
// own 128 x rows and HALF of the 256 weight rows (the MMA reads the other
// half from the peer's shared memory), so a stage is 32 KiB per CTA instead
// of 48 and six stages fit: the load pipeline covers 2.5x more MMA time,
// which the load-latency-bound prefill GEMMs need. For experts with many
// rows (long, L2-fed, MMA-bound units) the pair runs the same shared memory
// as three stages of two k-blocks, each operand's two k-blocks fetched by
// one TMA box of a [K / 64][rows][64] view. The even CTA issues the
// MMAs and commits them to both CTAs' barriers; both CTAs' TMA copies
// complete on the even CTA's stage barrier; both CTAs' epilogues read their
// own TMEM and release the accumulator on the even CTA's barrier.
// Tiles: each expert's row segment [offsets[e], offsets[e+1]) is cut into
// 128-row M-tiles (256-row units on a pair); linear unit ids run over
// (expert, n-tile, m-unit) with the m-unit fastest, so CTAs working at the
// same time share weight tiles in L2. A pair's last unit of an expert with at
// most 128 rows left runs as an M = 128 pair MMA: each CTA loads 64 rows of A
// (and, for SwiGLU, 64 gate rows over the same 64 up rows), and TMEM lanes
// 0-63 / 64-127 of each CTA hold its rows against the two halves of the
// tile's N. The schedule is computed per CTA from the device-side offsets: no
// host synchronisation. Rows of a tile past the segment end belong to the
// next expert (or are TMA zero-fill past the last row); they are computed and
// not stored. TMA zero-fills the K and N edges.
//
// In the one-call forward GEMM2 does not wait for GEMM1 as a whole: GEMM1's
// epilogue warps count each stored tile of h in a per-expert counter (after a
// memory fence), and GEMM2's producers wait, before their first load of an
// expert, until its counter covers all of the expert's tiles (acquire, then a
// generic-to-async proxy fence for the TMA reads). GEMM2's CTAs take the SMs
// that GEMM1's persistent CTAs leave, so they work on finished experts during
// GEMM1's last, partly filled round of units.
//
// Every wait is bounded (wait_ns); on expiry the kernel sets ST_TIMEOUT,
// stops issuing work, drains its own TMA copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128;                      // rows per tile (UMMA M)
constexpr int BK = 64;                       // K per stage: 128 bytes of 16-bit
constexpr int UK = 16;                       // K per tcgen05.mma kind::f16
constexpr int BN = 256;                      // B rows per tile (UMMA N)
constexpr int A_BYTES = BM * BK * 2;         // 16 KiB

// Per-CTA pipeline shape for one CTA per tile (CG = 1) or a CTA pair (CG = 2).
// A pair may run its ring as three stages of two k-blocks each (kps = 2):
// half as many barrier round trips and commits per unit, for the long,
// L2-fed units of experts with many rows; short units fed from DRAM keep
// six single-k-block stages (the finer ring hides more load latency).
template <int CG>
struct Pipe {
    static constexpr int B_ROWS = BN / CG;                     // weight rows this CTA loads
    static constexpr int B_BYTES = B_ROWS * BK * 2;            // per k-block: 32 / 16 KiB
    static constexpr int SLOT_BYTES = A_BYTES + B_BYTES;       // 48 / 32 KiB
    static constexpr int SLOTS = CG == 2 ? 6 : 4;              // single-k-block stages
};
constexpr int ACC_COLS = 256;                // fp32 columns per accumulator
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int THREADS = 192;
constexpr int MAX_E = 1024;
constexpr uint64_t kDrainLimitNs = 100000000ull;   // 100 ms per teardown drain
// Bytes of A rows one m-block of an expert may cover (see decode_unit): well
// inside the 129 MB L2, which also carries the streamed weights and the
// outputs.
constexpr int64_t kMBlockBytes = 48ll << 20;

constexpr int EPI_ROW_BYTES = 128;           // epilogue staging: 32 rows x 128 B per warp

// What the epilogue does with the accumulator tile.
enum OutMode : int {
    kOutDtype = 0,     // rows in the input dtype (h of GEMM1, or expert outputs)
    kOutF32 = 1,       // rows in FP32 (unrounded expert outputs)
    kOutCombine = 2,   // routing weight x row, reduced in FP32 into y_acc [T, N]
    kOutSaveGU = 3,    // GEMM1 for training: h, and the gate / up products g, u
                       // kept in FP32 (g_out, u_out: [rows, I])
};

// kOutCombine: dispatched row r belongs to assignment a = src_of[r], token
// a / top_k, weight w[a] (dtype wdt). kOutSaveGU: g_out / u_out receive the
// FP32 gate and up products of the training cache.
struct CombineInto {
    const int32_t *src_of;
    const void *w;
    int wdt;
    int top_k;
    float *g_out, *u_out;
    // Per-expert readiness of h (nullptr: off). GEMM1's epilogue warps add 1
    // to ready[e] after storing each tile of expert e; GEMM2 does not wait
    // for GEMM1 as a whole but, before its first load of expert e, until
    // ready[e] counts all of that expert's tiles (nt1 n-tiles per m-unit,
    // 4 warps per CTA): it starts on finished experts during GEMM1's tail.
    unsigned *ready;
    int nt1;
};

template <int CG>
struct __align__(1024) SharedStorage {
    // the stage ring: stage i of a kps-k-block ring starts at slot i * kps
    // and holds the A tiles of its k-blocks, then their B tiles
    uint8_t slot[Pipe<CG>::SLOTS][Pipe<CG>::SLOT_BYTES];      // each 1024-byte aligned
    uint8_t epi[4][32 * EPI_ROW_BYTES];      // per epilogue warp, 16-byte chunks swizzled
    uint64_t full[Pipe<CG>::SLOTS];
    uint64_t empty[Pipe<CG>::SLOTS];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int prefix[MAX_E + 1];
    int offs[MAX_E + 1];
};

template <int CG>
constexpr size_t kSmemBytes = sizeof(SharedStorage<CG>) + 1024;  // + alignment slack


// M-tile units of one expert: 128-row tiles, or pairs of them (CG = 2).
template <int CG>
__device__ __forceinline__ int m_units(int seg_rows)
{
    return (seg_rows + BM * CG - 1) / (BM * CG);
}

// Unit id -> (expert, n-tile, m-unit j). With CG = 2 unit j covers rows
// [256 j, 256 j + 256) of the expert's segment; when at most 128 of them
// remain (`half`), the pair computes an M = 128 tile instead (64 rows per
// CTA), so no CTA works on rows past the segment for nothing.
// An expert's units run in m-blocks of up to `mblock` m-units: all n-tiles
// of one m-block, the m-unit fastest, then the next m-block. The A rows of an
// m-block (mblock x rows x K) are sized to stay in L2 while the block's
// n-tiles stream the weights past them; without the blocks, an expert whose
// A rows outgrow L2 (thousands of rows at K in the thousands) has them
// re-read from DRAM for every round of n-tiles.
template <int CG, typename SS>
__device__ __forceinline__ void decode_unit(const SS &S, int E, int tile, int n_tiles,
                                            int mblock, int &e, int &n, int &j, bool &half)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S.prefix[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int seg = S.offs[e + 1] - S.offs[e];
    const int mu = m_units<CG>(seg);
    const int local = tile - S.prefix[e];
    const int span = mblock * n_tiles;            // units of one full m-block
    const int b = local / span;
    const int mb = mu - b * mblock < mblock ? mu - b * mblock : mblock;
    const int rem = local - b * span;
    n = rem / mb;
    j = b * mblock + rem % mb;
    half = CG == 2 && seg - j * (BM * CG) <= BM;
}

// First row (within the expert's segment) of this CTA's A rows in unit j.
template <int CG>
__device__ __forceinline__ int unit_row0(int j, int rank, bool half)
{
    return j * (BM * CG) + rank * (half ? BM / 2 : BM);
}


// load_as_float through L2 (see the offsets load in the kernel's prologue)
__device__ __forceinline__ float load_as_float_cg(const void *p, int dt, int64_t i)
{
    if (dt == DT_F32) return __ldcg(static_cast<const float *>(p) + i);
    const unsigned short b = __ldcg(static_cast<const unsigned short *>(p) + i);
    return dt == DT_BF16 ? __uint_as_float((uint32_t)b << 16)
                         : __half2float(__ushort_as_half(b));
}

// Bounded wait until *c >= need (acquire at GPU scope); false on abort or
// timeout (which sets ST_TIMEOUT and raises the abort flag).
__device__ __forceinline__ bool wait_counter(const unsigned *c, unsigned need,
                                             volatile int *abort_flag, unsigned *status,
                                             uint64_t limit_ns)
{
    auto load = [&] {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(c) : "memory");
        return v;
    };
    if (load() >= need) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (load() >= need) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(status, ST_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
        __nanosleep(100);
    }
}


// ---- the kernel -------------------------------------------------------------

template <int DT, bool SWIGLU, int OUT, int CG, int KPS>
__global__ void __launch_bounds__(THREADS, 1)
grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmAh,
                       const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmB1,
                       const __grid_constant__ CUtensorMap tmB0h,
                       const __grid_constant__ CUtensorMap tmB1h,
                       const int32_t *__restrict__ offsets, int E, int N, int K,
                       int n_tiles, int mblock, void *__restrict__ out, unsigned *status,
                       CombineInto comb, uint64_t wait_ns, int kbox)
{
    // KPS: k-blocks per pipeline stage (1, or 2 on a pair); kbox: the A and
    // B maps (not the M = 128 SwiGLU weight maps) give boxes of KPS
    // k-blocks (else one box per k-block)
    static_assert(KPS == 1 || (KPS == 2 && CG == 2), "two k-blocks per stage on pairs only");
    using P = Pipe<CG>;
    constexpr int kps = KPS;
    constexpr int n_stages = P::SLOTS / KPS;
    if (CG == 1) (void)kbox;
    extern __shared__ uint8_t smem_raw[];
    SharedStorage<CG> &S = *reinterpret_cast<SharedStorage<CG> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int N_OUT = SWIGLU ? BN / 2 : BN;      // output columns per tile
    const int num_kb = (K + BK - 1) / BK;
    const int num_ks = (num_kb + kps - 1) / kps;    // pipeline stages per unit
    // CTA pair: rank 0 issues the MMAs and owns the stage and accumulator
    // barriers that both CTAs' copies and epilogues signal
    const int rank = CG == 2 ? (int)cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / CG, unit_step = (int)gridDim.x / CG;

    if (threadIdx.x == 0) {
        for (int s = 0; s < n_stages; ++s) { mbar_init(&S.full[s], 1); mbar_init(&S.empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&S.acc_full[a], 1); mbar_init(&S.acc_empty[a], 4 * CG); }
        mbar_init(&S.drain, 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc<CG>(&S.tmem_base, TMEM_COLS);
        tmem_relinquish<CG>();
    }
    // everything above is CTA-local; the offsets and operands come from the
    // previous kernels on the stream
    // GEMM2 with per-expert readiness waits per expert instead (below);
    // everything else it reads was complete before GEMM1 let it launch
    if (SWIGLU || comb.ready == nullptr) pdl_wait();
    pdl_launch_dependents();
    // read through L2 (GEMM2 with per-expert readiness runs without the
    // grid-level wait, so no line may come from a stale L1)
    for (int i = threadIdx.x; i <= E; i += THREADS) S.offs[i] = __ldcg(offsets + i);
    __syncthreads();
#if MOE_DEBUG_BOUNDS
    // bounds-checking build: the caller's offsets start at 0 and never fall;
    // otherwise the launch records ST_BOUNDS and computes nothing
    {
        int bad = 0;
        for (int i = threadIdx.x; i < E; i += THREADS) bad |= S.offs[i + 1] < S.offs[i];
        bad |= S.offs[0] != 0;
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) atomicOr(status, ST_BOUNDS);
            for (int i = threadIdx.x; i <= E; i += THREADS) S.offs[i] = 0;
            __syncthreads();
        }
    }
#endif
    if (warp == 0) {
        // prefix[e] = tiles of experts < e; lane l owns a contiguous run of experts
        const int per = (E + 31) / 32, e0 = lane * per;
        int local = 0;
        for (int e = e0; e < e0 + per && e < E; ++e)
            local += m_units<CG>(S.offs[e + 1] - S.offs[e]) * n_tiles;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int e = e0; e < e0 + per && e < E; ++e) {
            S.prefix[e] = run;
            run += m_units<CG>(S.offs[e + 1] - S.offs[e]) * n_tiles;
        }
        if (lane == 31) S.prefix[E] = incl;
    }
    tc_fence_before();
    // a pair also makes each CTA's barrier initialisation visible to the
    // other before any copy or arrival targets it
    if constexpr (CG == 2) cluster_sync();
    else __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = S.tmem_base;
    const int total_tiles = S.prefix[E];
    volatile int *abort_flag = &S.abort;

    // producer bookkeeping for a safe drain on abort
    uint32_t filled_mask = 0, filled_parity = 0;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0;
        int ready_e = -1;                        // last expert found ready
        for (int tile = unit0; tile < total_tiles; tile += unit_step) {
            int e, n, j;
            bool half;
            decode_unit<CG>(S, E, tile, n_tiles, mblock, e, n, j, half);
            const int row0 = S.offs[e] + unit_row0<CG>(j, rank, half);
            bool ok = true;
            if (!SWIGLU && comb.ready != nullptr && e != ready_e) {
                const unsigned need = (unsigned)(m_units<CG>(S.offs[e + 1] - S.offs[e]) * comb.nt1 * 4 * CG);
                if (!wait_counter(comb.ready + e, need, abort_flag, status, wait_ns)) break;
                // the h tiles were written through the generic proxy; the TMA
                // reads below go through the async proxy
                asm volatile("fence.proxy.async.global;" ::: "memory");
                ready_e = e;
            }
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait<CG>(&S.empty[stage], phase ^ 1u, abort_flag, status, wait_ns)) { ok = false; break; }
                uint8_t *sa = S.slot[stage * kps];
                uint8_t *sb = sa + kps * A_BYTES;
                const int kb0 = ks * kps;
                // k-blocks of this stage inside K (the last stage of an odd count
                // with kps = 2 has one)
                const int nkb = num_kb - kb0 < kps ? num_kb - kb0 : kps;
                if constexpr (CG == 2) {
                    const int a_kb = half ? A_BYTES / 2 : A_BYTES;      // A bytes per k-block
                    // a box of kps k-blocks always lands whole (zero fill past
                    // K); one-k-block boxes are issued inside K only
                    const int a_bytes = (kbox ? kps : nkb) * a_kb;
                    const int b_bytes = ((half && SWIGLU) || !kbox ? nkb : kps) * P::B_BYTES;
                    // the leader's barrier expects both CTAs' bytes; a peer's
                    // copy may land before the leader arms it (the phase
                    // cannot complete while the leader's arrival is pending)
                    if (leader) mbar_arrive_expect_tx(&S.full[stage], 2 * (a_bytes + b_bytes));
                    const uint32_t bar = mapa_shared(smem_u32(&S.full[stage]), 0);
                    const CUtensorMap *ma = half ? &tmAh : &tmA;
                    if (kbox) {
                        tma_load_3d_pair(sa, ma, bar, 0, row0, kb0);
                    } else {
                        for (int q = 0; q < nkb; ++q)
                            tma_load_2d_pair(sa + q * a_kb, ma, bar, (kb0 + q) * BK, row0);
                    }
                    if (half && SWIGLU) {
                        // 64 rows of A per CTA; each CTA holds 64 gate rows over
                        // the same 64 up rows, so each TMEM lane half of the
                        // M = 128 tile sees both factors of 64 h columns
                        const int c1 = n * (BN / 2) + rank * (BN / 4);
                        for (int q = 0; q < nkb; ++q) {
                            uint8_t *dq = sb + q * P::B_BYTES;
                            tma_load_3d_pair(dq, &tmB0h, bar, (kb0 + q) * BK, c1, e);
                            tma_load_3d_pair(dq + P::B_BYTES / 2, &tmB1h, bar, (kb0 + q) * BK, c1, e);
                        }
                    } else {
                        // SwiGLU: CTA 0 holds the gate rows, CTA 1 the up rows
                        const CUtensorMap *mb = SWIGLU && rank == 1 ? &tmB1 : &tmB0;
                        const int nrow = SWIGLU ? n * (BN / 2) : n * BN + rank * (BN / 2);
                        if (kbox) {
                            tma_load_4d_pair(sb, mb, bar, 0, nrow, kb0, e);
                        } else {
                            for (int q = 0; q < nkb; ++q)
                                tma_load_3d_pair(sb + q * P::B_BYTES, mb, bar, (kb0 + q) * BK, nrow, e);
                        }
                    }
                } else {
                    (void)half; (void)nkb;
                    mbar_arrive_expect_tx(&S.full[stage], P::SLOT_BYTES);
                    tma_load_2d(sa, &tmA, &S.full[stage], kb0 * BK, row0);
                    if (SWIGLU) {
                        tma_load_3d(sb, &tmB0, &S.full[stage], kb0 * BK, n * (BN / 2), e);
                        tma_load_3d(sb + P::B_BYTES / 2, &tmB1, &S.full[stage], kb0 * BK, n * (BN / 2), e);
                    } else {
                        tma_load_3d(sb, &tmB0, &S.full[stage], kb0 * BK, n * BN, e);
                    }
                }
                filled_mask |= 1u << stage;
                filled_parity = (filled_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == n_stages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_full = idesc_f16<DT>(BM * CG, BN);
        constexpr uint32_t idesc_half = idesc_f16<DT>(BM, BN);    // CG = 2 only
        int stage = 0;
        uint32_t phase = 0;
        int it = 0;
        bool ok = true;
        for (int tile = unit0; tile < total_tiles && ok; tile += unit_step, ++it) {
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            int e, n, j;
            bool half;
            decode_unit<CG>(S, E, tile, n_tiles, mblock, e, n, j, half);
            const uint32_t idesc = half ? idesc_half : idesc_full;
            if (!mbar_wait<CG>(&S.acc_empty[acc], acc_phase ^ 1u, abort_flag, status, wait_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(acc * ACC_COLS);
            const uint32_t a_kb = half ? A_BYTES / 2 : A_BYTES;     // A bytes per k-block
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait<CG>(&S.full[stage], phase, abort_flag, status, wait_ns)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(S.slot[stage * kps]);
                const uint32_t b0 = a0 + (uint32_t)(kps * A_BYTES);
                const int nkb = num_kb - ks * kps < kps ? num_kb - ks * kps : kps;
#pragma unroll
                for (int q = 0; q < KPS; ++q) {
                    if (q < nkb) {
#pragma unroll
                        for (int k = 0; k < BK / UK; ++k)
                            umma_f16<CG>(d, sdesc_k_sw128(a0 + q * a_kb + k * UK * 2),
                                         sdesc_k_sw128(b0 + q * P::B_BYTES + k * UK * 2),
                                         idesc, (ks | q | k) != 0 ? 1u : 0u);
                    }
                }
                if constexpr (CG == 2) umma_commit_pair(&S.empty[stage]);
                else umma_commit<CG>(&S.empty[stage]);
                if (++stage == n_stages) { stage = 0; phase ^= 1u; }
            }
            if (ok) {
                if constexpr (CG == 2) umma_commit_pair(&S.acc_full[acc]);
                else umma_commit<CG>(&S.acc_full[acc]);
            }
        }
        if (*abort_flag) {
            // every MMA issued so far must finish before TMEM is released
            umma_commit<CG>(&S.drain);
            mbar_wait(&S.drain, 0, nullptr, status, kDrainLimitNs);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------ epilogue
        // Each warp owns 32 accumulator rows (its TMEM lane quadrant). Per
        // round it turns 128 output bytes of each row into its staging rows
        // (thread = row; 16-byte chunk p stored at p ^ (row & 7) so the 32
        // writes of one instruction spread over all banks), then copies the
        // 32 x 128 bytes out with each store instruction writing four whole
        // rows' 128-byte lines, masked to the expert's rows and to N.
        const int q = warp & 3;            // TMEM lane quadrant of this warp
        uint8_t *stg = S.epi[warp - 2];
        constexpr bool F32ACC = !SWIGLU && OUT != kOutDtype;   // FP32 values leave the tile
        constexpr int ESZ = F32ACC ? 4 : 2;                     // output element bytes
        constexpr int RCOLS = EPI_ROW_BYTES / ESZ;              // columns per round
        constexpr int ROUNDS = N_OUT / RCOLS;
        const int64_t out_row_bytes = (int64_t)N * ESZ;
        const int cch = lane & 7;                               // chunk this lane copies out
        int it = 0;
        for (int tile = unit0; tile < total_tiles; tile += unit_step, ++it) {
            int e, n, j;
            bool half;
            decode_unit<CG>(S, E, tile, n_tiles, mblock, e, n, j, half);
            const int seg_rows = S.offs[e + 1] - S.offs[e];
            // this warp's first row in the segment and first output column of
            // the tile: an M = 128 pair tile keeps a CTA's 64 rows in lanes
            // 0-63 against the first half of the tile's N and in lanes 64-127
            // against the second half, each in TMEM columns [0, N / 2)
            const int r_base = unit_row0<CG>(j, rank, half) + (half ? (q & 1) : q) * 32;
            const int cblk = half ? (q >> 1) * (N_OUT / 2) : 0;
            const int rounds = half ? ROUNDS / 2 : ROUNDS;
            const int u_col = half ? BN / 4 : BN / 2;        // TMEM column of u (SwiGLU)
            uint8_t *out_base = static_cast<uint8_t *>(out) + ((int64_t)S.offs[e] + r_base) * out_row_bytes;
            // kOutCombine: token and routing weight of this lane's row
            int row_tok = -1;
            float row_w = 0.0f;
            if constexpr (OUT == kOutCombine) {
                if (r_base + lane < seg_rows) {
                    const int a = __ldcg(comb.src_of + S.offs[e] + r_base + lane);
                    row_tok = a / comb.top_k;
                    row_w = load_as_float_cg(comb.w, comb.wdt, a);
                }
            }
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            // every lane waits; the warp leaves together if any lane gave up,
            // since tcgen05.ld below needs the whole warp converged
            const bool ready = mbar_wait<CG>(&S.acc_full[acc], acc_phase, abort_flag, status, wait_ns);
            if (!__all_sync(0xffffffffu, ready)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * ACC_COLS);
            // 32 rows x 128 bytes (this lane's row in v) to row0 + rr * row_bytes
            // + col_byte through the staging buffer, masked to the expert's
            // rows and to col_limit bytes
            auto emit_lines = [&](const uint32_t (&v)[32], uint8_t *row0, int64_t row_bytes,
                                  int64_t col_byte, int64_t col_limit) {
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    *reinterpret_cast<uint4 *>(stg + lane * EPI_ROW_BYTES + ((p ^ (lane & 7)) << 4)) =
                        make_uint4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3]);
                __syncwarp();
                const int64_t cb = col_byte + cch * 16;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int rr = 4 * j + (lane >> 3);
                    const uint4 q = *reinterpret_cast<const uint4 *>(
                        stg + rr * EPI_ROW_BYTES + ((cch ^ (rr & 7)) << 4));
                    if (r_base + rr < seg_rows && cb < col_limit)
                        *reinterpret_cast<uint4 *>(row0 + rr * row_bytes + cb) = q;
                }
                __syncwarp();
            };
            (void)emit_lines;
#pragma unroll 1
            for (int rd = 0; rd < rounds; ++rd) {
                uint32_t w[32];                                 // this row's 128 output bytes
                if constexpr (F32ACC) {
                    tmem_ld32(tbase + rd * 32, w);
                    tmem_ld_wait(w);
                    if constexpr (OUT == kOutCombine) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            w[i] = __float_as_uint(__uint_as_float(w[i]) * row_w);
                    }
                } else {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int c = rd * 2 + hf;              // 32-column TMEM chunk
                        uint32_t g[32];
                        tmem_ld32(tbase + c * 32, g);
                        if constexpr (SWIGLU) {
                            uint32_t u[32];
                            tmem_ld32(tbase + u_col + c * 32, u);
                            tmem_ld_wait(g);
                            tmem_ld_wait(u);
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                                const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
                                const float h0 = g0 / (1.0f + __expf(-g0)) * u0;
                                const float h1 = g1 / (1.0f + __expf(-g1)) * u1;
                                w[hf * 16 + i] = pack2<DT>(h0, h1);
                            }
                            if constexpr (OUT == kOutSaveGU) {
                                // the FP32 g and u of these 32 columns, as they are
                                const int64_t gu_row = (int64_t)N * 4;
                                const int64_t cb = (int64_t)(n * N_OUT + cblk + rd * RCOLS + hf * 32) * 4;
                                const int64_t r0 = (int64_t)S.offs[e] + r_base;
                                emit_lines(g, reinterpret_cast<uint8_t *>(comb.g_out) + r0 * gu_row,
                                           gu_row, cb, gu_row);
                                emit_lines(u, reinterpret_cast<uint8_t *>(comb.u_out) + r0 * gu_row,
                                           gu_row, cb, gu_row);
                            }
                        } else {
                            tmem_ld_wait(g);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                w[hf * 16 + i] = pack2<DT>(__uint_as_float(g[2 * i]),
                                                             __uint_as_float(g[2 * i + 1]));
                        }
                    }
                }
                const int64_t col_byte = (int64_t)(n * N_OUT + cblk + rd * RCOLS) * ESZ + cch * 16;
#pragma unroll
                for (int p = 0; p < 8; ++p)
                    *reinterpret_cast<uint4 *>(stg + lane * EPI_ROW_BYTES + ((p ^ (lane & 7)) << 4)) =
                        make_uint4(w[4 * p], w[4 * p + 1], w[4 * p + 2], w[4 * p + 3]);
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int rr = 4 * j + (lane >> 3);
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        stg + rr * EPI_ROW_BYTES + ((cch ^ (rr & 7)) << 4));
                    if constexpr (OUT == kOutCombine) {
                        const int tk = __shfl_sync(0xffffffffu, row_tok, rr);
                        if (tk >= 0 && col_byte < out_row_bytes) {
                            float *dst = reinterpret_cast<float *>(
                                static_cast<uint8_t *>(out) + (int64_t)tk * out_row_bytes + col_byte);
                            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst),
                                         "f"(__uint_as_float(v.x)), "f"(__uint_as_float(v.y)),
                                         "f"(__uint_as_float(v.z)), "f"(__uint_as_float(v.w))
                                         : "memory");
                        }
                    } else {
                        if (r_base + rr < seg_rows && col_byte < out_row_bytes)
                            *reinterpret_cast<uint4 *>(out_base + rr * out_row_bytes + col_byte) = v;
                    }
                }
                __syncwarp();
            }
            if (SWIGLU && comb.ready != nullptr) {
                // this warp's h rows of the tile are stored: publish them
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(comb.ready + e, 1u);
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
    // GEMM2 with per-expert readiness skipped the grid-level wait at entry;
    // waiting here, once its own work is done, restores the usual guarantee
    // for whatever the stream runs next: when GEMM2 has completed, GEMM1 has
    // too (its h, counters and every other write are done and visible)
    if (!SWIGLU && comb.ready != nullptr) pdl_wait();
    if (*abort_flag && warp == 0 && lane == 0) {
        if (CG == 1 || leader) {
            // let the outstanding TMA copies land before shared memory goes
            for (int s = 0; s < n_stages; ++s)
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


// The dynamic shared-memory opt-in is per device and per kernel instance.
template <int DT, bool SWIGLU, int OUT, int CG, int KPS>
cudaError_t ensure_smem_attr()
{
    static std::atomic<uint64_t> done_mask{0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = dev >= 0 && dev < kCachedDevices ? 1ull << dev : 0ull;
    if (bit != 0 && (done_mask.load() & bit)) return cudaSuccess;
    err = cudaFuncSetAttribute(grouped_gemm_tc_kernel<DT, SWIGLU, OUT, CG, KPS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes<CG>);
    if (err == cudaSuccess) done_mask.fetch_or(bit);
    return err;
}

// Upper bound on the tile units of a grouped GEMM: every expert adds at most
// one partial unit.
int64_t tc_unit_upper_bound(int64_t rows, int E, int64_t n_tiles, int cg)
{
    const int64_t per = (int64_t)BM * cg;
    const int64_t mu = rows / per + (rows < E ? rows : E);
    return mu * n_tiles;
}

// CTAs to launch: one per SM for CG = 1; for CG = 2 twice the number of
// pairs the GPU holds at once (cluster placement can leave SMs unpaired), so
// the persistent grid is always a single wave.
template <int DT, bool SWIGLU, int OUT, int CG, int KPS>
cudaError_t grid_size(int64_t units, int *grid)
{
    const int64_t sms = device_sm_count();
    if constexpr (CG == 1) {
        *grid = (int)(units < sms ? units : sms);
        return cudaSuccess;
    } else {
        static std::atomic<int> cached[kCachedDevices];
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        const bool use_cache = dev >= 0 && dev < kCachedDevices;
        int pairs = use_cache ? cached[dev].load() : 0;
        if (pairs == 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(sms & ~int64_t(1)));
            cfg.blockDim = dim3(THREADS);
            cfg.dynamicSmemBytes = kSmemBytes<CG>;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            err = cudaOccupancyMaxActiveClusters(&pairs, grouped_gemm_tc_kernel<DT, SWIGLU, OUT, CG, KPS>,
                                                 &cfg);
            if (err != cudaSuccess) return err;
            if (pairs < 1) return cudaErrorInvalidConfiguration;
            if (use_cache) cached[dev].store(pairs);
        }
        *grid = 2 * (int)(units < pairs ? units : pairs);
        return cudaSuccess;
    }
}

// Programmatic dependent launch (unless pdl is false: plain stream order),
// in clusters of CG CTAs.
template <int DT, bool SWIGLU, int OUT, int CG, int KPS>
cudaError_t launch_gemm(int64_t units, cudaStream_t s, const CUtensorMap &ta, const CUtensorMap &tah,
                        const CUtensorMap &tb0, const CUtensorMap &tb1, const CUtensorMap &tb0h,
                        const CUtensorMap &tb1h, const int32_t *offsets, int E, int N, int K,
                        int n_tiles, void *out, unsigned *status, const CombineInto &comb,
                        int kbox = 0, bool pdl = true)
{
    cudaError_t err = ensure_smem_attr<DT, SWIGLU, OUT, CG, KPS>();
    if (err != cudaSuccess) return err;
    int grid = 0;
    err = grid_size<DT, SWIGLU, OUT, CG, KPS>(units, &grid);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = kSmemBytes<CG>;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CG;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CG == 2 ? 2 : 1;
    // m-blocks whose A rows take at most kMBlockBytes (see decode_unit)
    int64_t mblock = kMBlockBytes / ((int64_t)BM * CG * K * 2);
    mblock = mblock < 1 ? 1 : (mblock > (1 << 20) ? (1 << 20) : mblock);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_tc_kernel<DT, SWIGLU, OUT, CG, KPS>, ta, tah, tb0, tb1,
                              tb0h, tb1h, offsets, E, N, K, n_tiles, (int)mblock, out, status,
                              comb, wait_limit_ns(), kbox);
}

// CTA pairs pay when experts average at least two M-tiles: a pair's second
// M-tile past an expert's rows is computed for nothing.
constexpr int64_t kPairMinRowsPerExpert = 2 * BM;
// Two k-blocks per stage pay when experts average at least 2048 rows (each
// weight tile then serves eight or more pair units from L2, and the
// launches are bound by the MMAs, not by load latency): on the coarse
// prefill shapes (4096 rows per expert) GEMM1 4.43 -> 4.23 ms; with 384
// rows per expert (weights streamed from DRAM) both GEMMs were 3-4 % slower.
constexpr int64_t kTwoKbMinRowsPerExpert = 2048;

// Tensor maps of both GEMMs (x / h rows, gate / up / down weights, the
// M = 128 pair tile's boxes) and whether their A / B maps give two-k-block
// boxes.
struct TcMaps {
    CUtensorMap mx, mxh, mg, mu, mgh, muh, mh, mhh, md;
    int kbox1, kbox2;
};

// GEMM1 (SwiGLU into h_ws) then GEMM2 (out_mode) with KPS k-blocks per stage.
template <int DT, int CG, int KPS>
cudaError_t launch_gemm_pair(const TcMaps &m, const int32_t *offsets, int64_t rows, int E,
                             int64_t H, int64_t I, void *h_ws, void *out, int out_mode,
                             const CombineInto &comb, unsigned *status, cudaStream_t s)
{
    const int nt1 = (int)((I + BN / 2 - 1) / (BN / 2));
    const int nt2 = (int)((H + BN - 1) / BN);
    const int64_t u1 = tc_unit_upper_bound(rows, E, nt1, CG);
    const int64_t u2 = tc_unit_upper_bound(rows, E, nt2, CG);
    cudaError_t err =
        comb.g_out != nullptr
            ? launch_gemm<DT, true, kOutSaveGU, CG, KPS>(u1, s, m.mx, m.mxh, m.mg, m.mu, m.mgh,
                                                        m.muh, offsets, E, (int)I, (int)H, nt1,
                                                        h_ws, status, comb, m.kbox1)
            : launch_gemm<DT, true, kOutDtype, CG, KPS>(u1, s, m.mx, m.mxh, m.mg, m.mu, m.mgh,
                                                       m.muh, offsets, E, (int)I, (int)H, nt1,
                                                       h_ws, status, comb, m.kbox1);
    if (err != cudaSuccess) return err;
    if (out_mode == kOutF32)
        return launch_gemm<DT, false, kOutF32, CG, KPS>(u2, s, m.mh, m.mhh, m.md, m.md, m.md,
                                                        m.md, offsets, E, (int)H, (int)I, nt2,
                                                        out, status, comb, m.kbox2);
    if (out_mode == kOutCombine)
        return launch_gemm<DT, false, kOutCombine, CG, KPS>(u2, s, m.mh, m.mhh, m.md, m.md, m.md,
                                                            m.md, offsets, E, (int)H, (int)I, nt2,
                                                            out, status, comb, m.kbox2);
    return launch_gemm<DT, false, kOutDtype, CG, KPS>(u2, s, m.mh, m.mhh, m.md, m.md, m.md, m.md,
                                                      offsets, E, (int)H, (int)I, nt2, out,
                                                      status, comb, m.kbox2);
}

template <int DT, int CG>
cudaError_t launch_tc_cg(const void *x_disp, const int32_t *offsets, int64_t rows,
                         const void *gate, const void *up, const void *down, int E,
                         int64_t H, int64_t I, void *h_ws, void *out, int out_mode,
                         const CombineInto &comb, unsigned *status, cudaStream_t s)
{
    const CUtensorMapDataType tdt =
        DT == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap mx, mg, mu, mh, md;
    if (!encode_2d(&mx, tdt, x_disp, (uint64_t)H, (uint64_t)rows, BK, BM) ||
        !encode_3d(&mg, tdt, gate, (uint64_t)H, (uint64_t)I, (uint64_t)E, BK, BN / 2) ||
        !encode_3d(&mu, tdt, up, (uint64_t)H, (uint64_t)I, (uint64_t)E, BK, BN / 2) ||
        !encode_2d(&mh, tdt, h_ws, (uint64_t)I, (uint64_t)rows, BK, BM) ||
        !encode_3d(&md, tdt, down, (uint64_t)I, (uint64_t)H, (uint64_t)E, BK, BN / CG))
        return cudaErrorInvalidValue;
    // M = 128 pair tiles: 64-row boxes of x / h, and of gate / up
    CUtensorMap mxh = mx, mhh = mh, mgh = mg, muh = mu;
    if (CG == 2 &&
        (!encode_2d(&mxh, tdt, x_disp, (uint64_t)H, (uint64_t)rows, BK, BM / 2) ||
         !encode_2d(&mhh, tdt, h_ws, (uint64_t)I, (uint64_t)rows, BK, BM / 2) ||
         !encode_3d(&mgh, tdt, gate, (uint64_t)H, (uint64_t)I, (uint64_t)E, BK, BN / 4) ||
         !encode_3d(&muh, tdt, up, (uint64_t)H, (uint64_t)I, (uint64_t)E, BK, BN / 4)))
        return cudaErrorInvalidValue;
    // Experts with many rows: two k-blocks per stage, in boxes of two
    // k-blocks where K is a whole number of them
    const int kps = CG == 2 && rows >= kTwoKbMinRowsPerExpert * E ? 2 : 1;
    int kbox1 = 0, kbox2 = 0;
    if (kps == 2) {
        CUtensorMap t0, t1, t2, t3;
        if (encode_kblocks(&t0, tdt, x_disp, (uint64_t)H, (uint64_t)rows, BM, 2) &&
            encode_kblocks(&t1, tdt, x_disp, (uint64_t)H, (uint64_t)rows, BM / 2, 2) &&
            encode_kblocks_e(&t2, tdt, gate, (uint64_t)H, (uint64_t)I, (uint64_t)E, BN / 2, 2) &&
            encode_kblocks_e(&t3, tdt, up, (uint64_t)H, (uint64_t)I, (uint64_t)E, BN / 2, 2)) {
            mx = t0; mxh = t1; mg = t2; mu = t3; kbox1 = 1;
        }
        if (encode_kblocks(&t0, tdt, h_ws, (uint64_t)I, (uint64_t)rows, BM, 2) &&
            encode_kblocks(&t1, tdt, h_ws, (uint64_t)I, (uint64_t)rows, BM / 2, 2) &&
            encode_kblocks_e(&t2, tdt, down, (uint64_t)I, (uint64_t)H, (uint64_t)E, BN / CG, 2)) {
            mh = t0; mhh = t1; md = t2; kbox2 = 1;
        }
    }
    const TcMaps m{mx, mxh, mg, mu, mgh, muh, mh, mhh, md, kbox1, kbox2};
    if constexpr (CG == 2) {
        if (kps == 2)
            return launch_gemm_pair<DT, CG, 2>(m, offsets, rows, E, H, I, h_ws, out, out_mode,
                                               comb, status, s);
    }
    return launch_gemm_pair<DT, CG, 1>(m, offsets, rows, E, H, I, h_ws, out, out_mode, comb,
                                       status, s);
}

// GEMM2 of the one-call forward on its own: h [rows, I] times down, each row
// weighted and reduced into y_acc, starting on expert e once ready[e] counts
// all of its h tiles (as GEMM1 would publish them).
template <int DT, int CG>
cudaError_t launch_down_combine_cg(const int32_t *offsets, int64_t rows, const void *down, int E,
                                   int64_t H, int64_t I, const void *h, const CombineInto &comb,
                                   float *y_acc, unsigned *status, cudaStream_t s)
{
    const CUtensorMapDataType tdt =
        DT == DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap mh, md;
    if (!encode_2d(&mh, tdt, h, (uint64_t)I, (uint64_t)rows, BK, BM) ||
        !encode_3d(&md, tdt, down, (uint64_t)I, (uint64_t)H, (uint64_t)E, BK, BN / CG))
        return cudaErrorInvalidValue;
    CUtensorMap mhh = mh;
    if (CG == 2 && !encode_2d(&mhh, tdt, h, (uint64_t)I, (uint64_t)rows, BK, BM / 2))
        return cudaErrorInvalidValue;
    const int nt2 = (int)((H + BN - 1) / BN);
    // plain stream order: this GEMM reads the offsets before any grid-level
    // wait, so they must be complete when it starts
    return launch_gemm<DT, false, kOutCombine, CG, 1>(tc_unit_upper_bound(rows, E, nt2, CG), s, mh,
                                                   mhh, md, md, md, md, offsets, E, (int)H,
                                                   (int)I, nt2, y_acc, status, comb, 0, false);
}

// offsets[e] = e * rows_per_expert (e <= E), src_of[r] = r: the dispatch map
// of one token per row and top_k = 1
__global__ void selftest_map_kernel(int32_t *offsets, int32_t *src_of, int E, int rows_per_expert)
{
    const int rows = E * rows_per_expert;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= rows; i += gridDim.x * blockDim.x) {
        if (i <= E) offsets[i] = i * rows_per_expert;
        if (i < rows) src_of[i] = i;
    }
}

template <int DT>
cudaError_t launch_tc_dt(const void *x_disp, const int32_t *offsets, int64_t rows,
                         const void *gate, const void *up, const void *down, int E,
                         int64_t H, int64_t I, void *h_ws, void *out, int out_mode,
                         const CombineInto &comb, unsigned *status, cudaStream_t s)
{
    if (rows >= kPairMinRowsPerExpert * E)
        return launch_tc_cg<DT, 2>(x_disp, offsets, rows, gate, up, down, E, H, I, h_ws, out,
                                   out_mode, comb, status, s);
    return launch_tc_cg<DT, 1>(x_disp, offsets, rows, gate, up, down, E, H, I, h_ws, out,
                               out_mode, comb, status, s);
}

}  // namespace

cudaError_t launch_experts_tc(int dt, const void *x_disp, const int32_t *offsets,
                              int64_t rows, const void *gate, const void *up,
                              const void *down, int E, int64_t H, int64_t I,
                              void *h_ws, void *out_disp, bool out_f32, unsigned *status,
                              cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    const CombineInto none{nullptr, nullptr, DT_F32, 1, nullptr, nullptr, nullptr, 0};
    const int mode = out_f32 ? kOutF32 : kOutDtype;
    if (dt == DT_BF16)
        return launch_tc_dt<DT_BF16>(x_disp, offsets, rows, gate, up, down, E, H, I, h_ws,
                                     out_disp, mode, none, status, s);
    return launch_tc_dt<DT_F16>(x_disp, offsets, rows, gate, up, down, E, H, I, h_ws, out_disp,
                                mode, none, status, s);
}

size_t selftest_wait_workspace_bytes(int E, int rows_per_expert, int64_t H, int64_t I)
{
    const size_t rows = (size_t)E * (size_t)rows_per_expert;
    auto r = [](size_t v) { return (v + 255) / 256 * 256; };
    return r((size_t)(E + 1) * 4) + r(rows * 4) + r(rows * 4) + r((size_t)E * 4) +
           r(rows * (size_t)I * 2) + r((size_t)E * (size_t)H * (size_t)I * 2);
}

cudaError_t launch_selftest_wait_expiry(int E, int rows_per_expert, int64_t H, int64_t I,
                                        void *ws, float *y_acc, unsigned *status, cudaStream_t s)
{
    const int64_t rows = (int64_t)E * rows_per_expert;
    auto r = [](size_t v) { return (v + 255) / 256 * 256; };
    uint8_t *p = static_cast<uint8_t *>(ws);
    int32_t *offsets = reinterpret_cast<int32_t *>(p);
    p += r((size_t)(E + 1) * 4);
    int32_t *src_of = reinterpret_cast<int32_t *>(p);
    p += r((size_t)rows * 4);
    float *w = reinterpret_cast<float *>(p);
    p += r((size_t)rows * 4);
    unsigned *ready = reinterpret_cast<unsigned *>(p);
    p += r((size_t)E * 4);
    void *h = p;
    p += r((size_t)rows * (size_t)I * 2);
    void *down = p;
    // zero h, the weights, the routing weights and the readiness counters
    cudaError_t err = cudaMemsetAsync(ws, 0, selftest_wait_workspace_bytes(E, rows_per_expert, H, I), s);
    if (err != cudaSuccess) return err;
    selftest_map_kernel<<<(unsigned)((rows + 256) / 256), 256, 0, s>>>(offsets, src_of, E,
                                                                          rows_per_expert);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const CombineInto comb{src_of, w, DT_F32, 1, nullptr, nullptr, ready,
                           (int)((I + BN / 2 - 1) / (BN / 2))};
    if (rows >= kPairMinRowsPerExpert * E)
        return launch_down_combine_cg<DT_BF16, 2>(offsets, rows, down, E, H, I, h, comb, y_acc,
                                                  status, s);
    return launch_down_combine_cg<DT_BF16, 1>(offsets, rows, down, E, H, I, h, comb, y_acc,
                                              status, s);
}

cudaError_t launch_experts_tc_training(int dt, const void *x_disp, const int32_t *offsets,
                                       int64_t rows, const void *gate, const void *up,
                                       const void *down, int E, int64_t H, int64_t I,
                                       void *cache, void *out_disp, bool out_f32,
                                       unsigned *status, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    // cache: h [rows, I] in dt, then g and u [rows, I] in FP32
    uint8_t *c = static_cast<uint8_t *>(cache);
    float *g = reinterpret_cast<float *>(c + rows * I * 2);
    const CombineInto save{nullptr, nullptr, DT_F32, 1, g, g + rows * I, nullptr, 0};
    const int mode = out_f32 ? kOutF32 : kOutDtype;
    if (dt == DT_BF16)
        return launch_tc_dt<DT_BF16>(x_disp, offsets, rows, gate, up, down, E, H, I, cache,
                                     out_disp, mode, save, status, s);
    return launch_tc_dt<DT_F16>(x_disp, offsets, rows, gate, up, down, E, H, I, cache, out_disp,
                                mode, save, status, s);
}

cudaError_t launch_experts_tc_combine(int dt, const void *x_disp, const int32_t *offsets,
                                      int64_t rows, const void *gate, const void *up,
                                      const void *down, int E, int64_t H, int64_t I,
                                      void *h_ws, const int32_t *src_of, const void *w,
                                      int wdt, int top_k, float *y_acc, unsigned *ready,
                                      unsigned *status, cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    const CombineInto comb{src_of, w, wdt, top_k, nullptr, nullptr, ready,
                           (int)((I + BN / 2 - 1) / (BN / 2))};
    if (dt == DT_BF16)
        return launch_tc_dt<DT_BF16>(x_disp, offsets, rows, gate, up, down, E, H, I, h_ws,
                                     y_acc, kOutCombine, comb, status, s);
    return launch_tc_dt<DT_F16>(x_disp, offsets, rows, gate, up, down, E, H, I, h_ws, y_acc,
                                kOutCombine, comb, status, s);
}

}  // namespace moe
