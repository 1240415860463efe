// moe_abi.cu -- the extern "C" boundary declared in include/moe.h: host-side
// argument validation, workspace carving and kernel launches. Nothing here
// allocates device memory; nothing here synchronises except
// moe_device_status().
#include <math.h>

#include <cmath>
#include <stdio.h>

#include <atomic>
#include <initializer_list>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {

// Per-device status word (ST_* bits); see moe_device_status().
__device__ unsigned g_moe_status = 0u;

int device_sm_count()
{
    static std::atomic<int> cache[kCachedDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const bool cached = dev >= 0 && dev < kCachedDevices;
    int v = cached ? cache[dev].load() : 0;
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 1;
    if (cached) cache[dev].store(v);
    return v;
}

namespace {
std::atomic<uint64_t> g_wait_limit_ns{kWaitLimitNs};
}

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

namespace {

// An NVTX range around each compute entry point, so a profiler's timeline
// shows which library call enqueued which kernels (header-only NVTX: without
// an attached tool each push / pop is a check of a null function pointer).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

thread_local char g_detail[256] = "";

int fail(int code, const char *what)
{
    snprintf(g_detail, sizeof g_detail, "%s", what);
    return code;
}

int cuda_fail(cudaError_t err, const char *where)
{
    snprintf(g_detail, sizeof g_detail, "%s: %s", where, cudaGetErrorString(err));
    return MOE_ERR_CUDA;
}

unsigned *status_ptr()
{
    static std::atomic<unsigned *> cache[kCachedDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    const bool cached = dev >= 0 && dev < kCachedDevices;
    unsigned *p = cached ? cache[dev].load() : nullptr;
    if (p != nullptr) return p;
    void *q = nullptr;
    if (cudaGetSymbolAddress(&q, g_moe_status) != cudaSuccess) return nullptr;
    if (cached) cache[dev].store(static_cast<unsigned *>(q));
    return static_cast<unsigned *>(q);
}

bool valid_dtype(int dt) { return dt == MOE_F32 || dt == MOE_BF16 || dt == MOE_F16; }
size_t elem_bytes(int dt) { return dt == MOE_F32 ? 4 : 2; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int64_t kMaxE = 1024;
constexpr uint64_t kMaxWaitLimitNs = 60ull * 1000000000ull;   // moe_set_wait_limit_ns bound
constexpr int64_t kMaxRows = 0x7fffffff;   // dispatched rows are int32

// Vector width rule shared by the experts and combine kernels: rows are moved
// in 16-byte vectors and TMA strides are 16-byte multiples.
bool vec_dim_ok(int64_t n, int dt) { return n >= 1 && (n * (int64_t)elem_bytes(dt)) % 16 == 0; }

int check_route_args(const void *logits, int ldt, int64_t T, int64_t E, int top_k,
                     const uint32_t *idx, const void *w)
{
    if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype must be F32, BF16 or F16");
    if (T < 0 || E < 1 || E > kMaxE) return fail(MOE_ERR_SHAPE, "need T >= 0 and 1 <= E <= 1024");
    if (top_k < 1 || top_k > E) return fail(MOE_ERR_SHAPE, "need 1 <= top_k <= E");
    if (T * top_k > kMaxRows) return fail(MOE_ERR_SHAPE, "T * top_k exceeds 2^31 - 1");
    if (T == 0) return MOE_OK;
    if (!logits || !idx || !w) return fail(MOE_ERR_NULL, "moe_route: NULL tensor");
    if (!aligned16(logits) || !aligned16(idx) || !aligned16(w))
        return fail(MOE_ERR_ALIGN, "moe_route: tensors must be 16-byte aligned");
    return MOE_OK;
}

// Limits of ruDNN section 10 on top of the shared routing checks.
int check_sigmoid_grouped_args(int64_t E, const float *bias, int top_k, int groups,
                               int selected_groups, int group_top_two, float scale)
{
    if (groups < 1 || groups > sigmoid_route_max_groups() || E % groups != 0)
        return fail(MOE_ERR_SHAPE, "need 1 <= groups <= 128 dividing E");
    if (selected_groups < 1 || selected_groups > groups)
        return fail(MOE_ERR_SHAPE, "need 1 <= selected_groups <= groups");
    if (top_k > sigmoid_route_max_top_k() || (int64_t)top_k > (int64_t)selected_groups * (E / groups))
        return fail(MOE_ERR_SHAPE, "need top_k <= 64 and top_k <= selected_groups * E / groups");
    if (group_top_two && E / groups < 2)
        return fail(MOE_ERR_SHAPE, "group_top_two needs at least two experts per group");
    if (!std::isfinite(scale) || !(scale > 0.0f))
        return fail(MOE_ERR_VALUE, "scale must be finite and > 0");
    if (bias != nullptr && !aligned16(bias)) return fail(MOE_ERR_ALIGN, "bias must be 16-byte aligned");
    return MOE_OK;
}

int check_experts_args(int64_t rows, int64_t E, int64_t H, int64_t I, int dt)
{
    if (!valid_dtype(dt)) return fail(MOE_ERR_DTYPE, "expert dtype must be F32, BF16 or F16");
    if (rows < 0 || rows > kMaxRows || E < 1 || E > kMaxE)
        return fail(MOE_ERR_SHAPE, "need 0 <= rows < 2^31 and 1 <= E <= 1024");
    if (!vec_dim_ok(H, dt) || !vec_dim_ok(I, dt))
        return fail(MOE_ERR_SHAPE, "H and I must be >= 1 with H*elem and I*elem multiples of 16 bytes");
    if (H > 0x7fffffff || I > 0x7fffffff) return fail(MOE_ERR_SHAPE, "H and I must fit int32");
    return MOE_OK;
}

int check_combine_args(int odt, int wdt, int dt, int64_t T, int top_k, int64_t H, bool norm)
{
    if (!valid_dtype(odt) || !valid_dtype(wdt) || !valid_dtype(dt))
        return fail(MOE_ERR_DTYPE, "dtype must be F32, BF16 or F16");
    if (odt != dt && odt != MOE_F32)
        return fail(MOE_ERR_DTYPE, "expert outputs must be in the activation dtype or F32");
    if (T < 0 || top_k < 1 || T * top_k > kMaxRows) return fail(MOE_ERR_SHAPE, "need T >= 0, top_k >= 1, T*top_k < 2^31");
    if (H < 1 || H % 8 != 0) return fail(MOE_ERR_SHAPE, "H must be a positive multiple of 8");
    if (H > combine_max_h(norm)) return fail(MOE_ERR_SHAPE, "H too large for the fused norm (one pass per row)");
    return MOE_OK;
}

// The one-call forward folds the combine into the second expert GEMM (FP32
// reductions into y_acc [T, H]) when y_acc stays well inside the 129 MB L2;
// a larger y_acc would turn every reduction into an HBM read-modify-write, so
// then the expert outputs go to HBM in FP32 and the combine kernel sums them.
constexpr size_t kFoldCombineMaxBytes = 64u << 20;

bool fold_combine(int64_t T, int64_t H, int dt)
{
    return dt != MOE_F32 && (size_t)T * (size_t)H * 4 <= kFoldCombineMaxBytes;
}

// y_acc's bytes, rounded so the word after it stays aligned
size_t fold_acc_bytes(int64_t T, int64_t H) { return round_up((size_t)T * (size_t)H * 4, 256); }

struct ForwardLayout {
    size_t idx, w, counts, offsets, row_of, src_of, disp_ws, x_disp, h, out_disp, total;
};

// The one-call forward folds the combine into GEMM2 unless the caller asked
// for the deterministic (slot-order) combine.
bool forward_folds(int64_t T, int64_t H, int dt, unsigned flags)
{
    return (flags & MOE_FORWARD_DETERMINISTIC) == 0 && fold_combine(T, H, dt);
}

ForwardLayout forward_layout(int64_t T, int64_t H, int64_t I, int64_t E, int top_k,
                             int dt, int ldt, unsigned flags)
{
    const size_t A = (size_t)(T * top_k), eb = elem_bytes(dt);
    ForwardLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t at = off; off = round_up(off + bytes, 256); return at; };
    L.idx = take(A * 4);
    L.w = take(A * elem_bytes(ldt));
    L.counts = take((size_t)E * 4);
    L.offsets = take((size_t)(E + 1) * 4);
    L.row_of = take(A * 4);
    L.src_of = take(A * 4);
    L.disp_ws = take(route_dispatch_workspace_bytes((int64_t)A, (int)E));
    L.x_disp = take(A * (size_t)H * eb);
    L.h = take(A * (size_t)I * eb);
    // FP32 expert outputs [A, H] for the combine kernel, or y_acc [T, H]
    // when the combine is folded into the second GEMM
    // (folded: y_acc, then 256 bytes whose first word counts the CTAs of the
    // fused routing kernel, then the experts' h-readiness counters [E]; one
    // memset clears them all)
    L.out_disp = take(forward_folds(T, H, dt, flags)
                          ? fold_acc_bytes(T, H) + 256 + round_up((size_t)E * 4, 256)
                          : A * (size_t)H * 4);
    L.total = off;
    return L;
}

int run_experts(const void *x_disp, const int32_t *offsets, int64_t rows, const void *gate,
                const void *up, const void *down, int64_t E, int64_t H, int64_t I, int dt,
                void *h_ws, void *out_disp, int odt, cudaStream_t s)
{
    cudaError_t err;
    if (dt == MOE_F32) {
        err = launch_experts_simt(static_cast<const float *>(x_disp), offsets, rows,
                                  static_cast<const float *>(gate), static_cast<const float *>(up),
                                  static_cast<const float *>(down), (int)E, H, I,
                                  static_cast<float *>(h_ws), static_cast<float *>(out_disp), s);
    } else {
        unsigned *st = status_ptr();
        if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
        err = launch_experts_tc(dt, x_disp, offsets, rows, gate, up, down, (int)E, H, I, h_ws,
                                out_disp, odt == MOE_F32, st, s);
        if (err == cudaErrorInvalidValue)
            return fail(MOE_ERR_ALIGN, "TMA descriptor rejected (pointer alignment or shape)");
    }
    if (err != cudaSuccess) return cuda_fail(err, "experts launch");
    return MOE_OK;
}

// Where the one-call forward's routing and dispatch write.
struct DispatchOut {
    int32_t *counts, *offsets, *row_of, *src_of;
    void *x_disp, *ws;
    unsigned *zeroed;        // a word already cleared on the stream, or nullptr
    unsigned *status;
};

// The one-call forward: route_dispatch(idx, w, d, stream) enqueues the routing
// into the workspace's idx / w and the dispatch into d; then the experts and
// the combine.
template <typename RouteFn>
int forward_impl(const char *name, const void *x, int dtype, const void *logits,
                 int logits_dtype, const void *gate, const void *up, const void *down,
                 int64_t T, int64_t H, int64_t I, int64_t E, int top_k, void *y,
                 void *workspace, size_t workspace_bytes, const moe_forward_options *opt,
                 void *stream, RouteFn route)
{
    const unsigned flags = opt != nullptr ? opt->flags : 0u;
    if (flags & ~(unsigned)MOE_FORWARD_DETERMINISTIC)
        return fail(MOE_ERR_VALUE, "unknown moe_forward_options flag");
    if (!valid_dtype(logits_dtype)) return fail(MOE_ERR_DTYPE, "logits dtype must be F32, BF16 or F16");
    int rc = check_experts_args(T * (int64_t)(top_k > 0 ? top_k : 1), E, H, I, dtype);
    if (rc != MOE_OK) return rc;
    if (T < 0 || top_k < 1 || top_k > E || T * top_k > kMaxRows)
        return fail(MOE_ERR_SHAPE, "need T >= 0 and 1 <= top_k <= E");
    if (H % 8 != 0) return fail(MOE_ERR_SHAPE, "H must be a multiple of 8");
    if (T == 0) return MOE_OK;
    if (!x || !logits || !gate || !up || !down || !y) return fail(MOE_ERR_NULL, name);
    if (!aligned16(x) || !aligned16(logits) || !aligned16(gate) || !aligned16(up) ||
        !aligned16(down) || !aligned16(y))
        return fail(MOE_ERR_ALIGN, "tensors must be 16-byte aligned");
    const ForwardLayout L = forward_layout(T, H, I, E, top_k, dtype, logits_dtype, flags);
    if (workspace_bytes < L.total || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "workspace too small or not 256-byte aligned");
    unsigned *st = status_ptr();
    if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint32_t *idx = reinterpret_cast<uint32_t *>(ws + L.idx);
    void *w = ws + L.w;
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *row_of = reinterpret_cast<int32_t *>(ws + L.row_of);
    int32_t *src_of = reinterpret_cast<int32_t *>(ws + L.src_of);
    void *x_disp = ws + L.x_disp, *h = ws + L.h, *out_disp = ws + L.out_disp;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t A = T * top_k;

    const bool fused_combine = forward_folds(T, H, dtype, flags);
    cudaEvent_t ev_begin = opt != nullptr ? static_cast<cudaEvent_t>(opt->experts_begin_event) : nullptr;
    cudaEvent_t ev_end = opt != nullptr ? static_cast<cudaEvent_t>(opt->experts_end_event) : nullptr;
    cudaError_t err = cudaSuccess;
    unsigned *zeroed = nullptr, *ready = nullptr;
    if (fused_combine) {
        uint8_t *tail = static_cast<uint8_t *>(out_disp) + fold_acc_bytes(T, H);
        zeroed = reinterpret_cast<unsigned *>(tail);
        ready = reinterpret_cast<unsigned *>(tail + 256);
        err = cudaMemsetAsync(out_disp, 0, fold_acc_bytes(T, H) + 256 + round_up((size_t)E * 4, 256), s);
        if (err != cudaSuccess) return cuda_fail(err, "forward/zero");
    }
    const DispatchOut d{counts, offsets, row_of, src_of, x_disp, ws + L.disp_ws, zeroed, st};
    err = route(idx, w, d, s);
    if (err != cudaSuccess) return cuda_fail(err, "forward/route+dispatch");
    if (ev_begin != nullptr && (err = cudaEventRecord(ev_begin, s)) != cudaSuccess)
        return cuda_fail(err, "forward/experts_begin_event");
    if (fused_combine) {
        err = launch_experts_tc_combine(dtype, x_disp, offsets, A, gate, up, down, (int)E, H, I,
                                        h, src_of, w, logits_dtype, top_k,
                                        static_cast<float *>(out_disp), ready, st, s);
        if (err == cudaErrorInvalidValue)
            return fail(MOE_ERR_ALIGN, "TMA descriptor rejected (pointer alignment or shape)");
        if (err != cudaSuccess) return cuda_fail(err, "forward/experts");
        if (ev_end != nullptr && (err = cudaEventRecord(ev_end, s)) != cudaSuccess)
            return cuda_fail(err, "forward/experts_end_event");
        err = launch_finalize(static_cast<const float *>(out_disp), T, H, y, dtype, s);
        return err == cudaSuccess ? MOE_OK : cuda_fail(err, "forward/finalize");
    }
    rc = run_experts(x_disp, offsets, A, gate, up, down, E, H, I, dtype, h, out_disp, MOE_F32, s);
    if (rc != MOE_OK) return rc;
    if (ev_end != nullptr && (err = cudaEventRecord(ev_end, s)) != cudaSuccess)
        return cuda_fail(err, "forward/experts_end_event");
    err = launch_combine(out_disp, MOE_F32, w, logits_dtype, row_of, nullptr, nullptr, MOE_F32,
                         1.0f, T, top_k, H, y, dtype, nullptr, nullptr, s);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "forward/combine");
}

}  // namespace

int report_error(int code, const char *what) { return fail(code, what); }

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "a required pointer is NULL";
    case MOE_ERR_SHAPE: return "a size is out of range or inconsistent";
    case MOE_ERR_DTYPE: return "unsupported dtype or dtype combination";
    case MOE_ERR_VALUE: return "invalid scalar argument";
    case MOE_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device wait gave up";
    case MOE_ERR_BAD_INDEX: return "an expert index >= E reached dispatch";
    case MOE_ERR_BOUNDS: return "a device-side bounds check failed (bounds-checking build)";
    default: return "unknown status";
    }
}

int moe_abi_version(void) { return 101; }

const char *moe_last_error_detail(void) { return g_detail; }

int moe_route(const void *logits, int logits_dtype, int64_t T, int64_t E, int top_k,
              int renormalize, uint32_t *expert_indices, void *weights, void *stream)
{
    const NvtxRange nvtx("moe_route");
    int rc = check_route_args(logits, logits_dtype, T, E, top_k, expert_indices, weights);
    if (rc != MOE_OK || T == 0) return rc;
    cudaError_t err = launch_route(logits, logits_dtype, T, (int)E, top_k, renormalize,
                                   expert_indices, weights, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_route");
}

int moe_route_sigmoid_grouped(const void *logits, int logits_dtype, int64_t T, int64_t E,
                              const float *bias, int top_k, int groups, int selected_groups,
                              int group_top_two, int renormalize, float scale,
                              uint32_t *expert_indices, void *weights, void *stream)
{
    const NvtxRange nvtx("moe_route_sigmoid_grouped");
    int rc = check_route_args(logits, logits_dtype, T, E, top_k, expert_indices, weights);
    if (rc != MOE_OK) return rc;
    rc = check_sigmoid_grouped_args(E, bias, top_k, groups, selected_groups, group_top_two, scale);
    if (rc != MOE_OK || T == 0) return rc;
    cudaError_t err = launch_route_sigmoid_grouped(logits, logits_dtype, T, (int)E, bias, top_k,
                                                   groups, selected_groups, group_top_two,
                                                   renormalize, scale, expert_indices, weights,
                                                   static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_route_sigmoid_grouped");
}

size_t moe_dispatch_workspace_size(int64_t T, int top_k, int64_t E)
{
    if (T <= 0 || top_k < 1 || E < 1 || E > kMaxE) return 0;
    return round_up(dispatch_workspace_bytes(T * top_k, (int)E), 256);
}

}  // extern "C"

namespace moe {

int check_dispatch_args(const uint32_t *expert_indices, int64_t T, int top_k, int64_t E,
                        int64_t special_experts, const void *x, int x_dtype, int64_t H,
                        const int32_t *counts, const int32_t *offsets, const int32_t *row_of,
                        const int32_t *src_of, const void *x_disp)
{
    if (!valid_dtype(x_dtype)) return fail(MOE_ERR_DTYPE, "x dtype must be F32, BF16 or F16");
    if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || H < 1 || T * top_k > kMaxRows)
        return fail(MOE_ERR_SHAPE, "need T >= 0, 1 <= E <= 1024, top_k >= 1, H >= 1");
    if (special_experts < 0 || special_experts > 0x7fffffff - E)
        return fail(MOE_ERR_SHAPE, "need 0 <= special_experts and E + special_experts < 2^31");
    if (T == 0) return MOE_OK;
    if (!expert_indices || !x || !counts || !offsets || !row_of || !src_of || !x_disp)
        return fail(MOE_ERR_NULL, "moe_dispatch: NULL tensor");
    if (!aligned16(expert_indices) || !aligned16(x) || !aligned16(counts) || !aligned16(offsets) ||
        !aligned16(row_of) || !aligned16(src_of) || !aligned16(x_disp))
        return fail(MOE_ERR_ALIGN, "moe_dispatch: tensors must be 16-byte aligned");
    return MOE_OK;
}

}  // namespace moe

extern "C" {

int moe_dispatch_special(const uint32_t *expert_indices, int64_t T, int top_k, int64_t E,
                         int64_t special_experts,
                 const void *x, int x_dtype, int64_t H, int32_t *counts, int32_t *offsets,
                 int32_t *row_of, int32_t *src_of, void *x_disp, void *workspace,
                 size_t workspace_bytes, void *stream)
{
    const NvtxRange nvtx("moe_dispatch");
    const int rc = check_dispatch_args(expert_indices, T, top_k, E, special_experts, x, x_dtype,
                                       H, counts, offsets, row_of, src_of, x_disp);
    if (rc != MOE_OK || T == 0) return rc;
    const size_t need = moe_dispatch_workspace_size(T, top_k, E);
    if (workspace_bytes < need || (need && !workspace) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_dispatch: workspace too small or not 256-byte aligned");
    unsigned *st = status_ptr();
    if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
    cudaError_t err = launch_dispatch(expert_indices, T, top_k, (int)E, special_experts, x, x_dtype, H, counts,
                                      offsets, row_of, src_of, x_disp, workspace, st,
                                      static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_dispatch");
}

int moe_dispatch(const uint32_t *expert_indices, int64_t T, int top_k, int64_t E,
                 const void *x, int x_dtype, int64_t H, int32_t *counts, int32_t *offsets,
                 int32_t *row_of, int32_t *src_of, void *x_disp, void *workspace,
                 size_t workspace_bytes, void *stream)
{
    return moe_dispatch_special(expert_indices, T, top_k, E, 0, x, x_dtype, H, counts, offsets,
                                row_of, src_of, x_disp, workspace, workspace_bytes, stream);
}

size_t moe_experts_workspace_size(int64_t rows, int64_t E, int64_t H, int64_t I, int dtype)
{
    (void)E;
    (void)H;
    if (rows <= 0 || I <= 0 || !valid_dtype(dtype)) return 0;
    return round_up((size_t)rows * (size_t)I * elem_bytes(dtype), 256);
}

int moe_experts_forward(const void *x_disp, const int32_t *offsets, int64_t rows,
                        const void *gate, const void *up, const void *down, int64_t E,
                        int64_t H, int64_t I, int dtype, void *out_disp, int out_dtype,
                        void *workspace, size_t workspace_bytes, void *stream)
{
    const NvtxRange nvtx("moe_experts_forward");
    int rc = check_experts_args(rows, E, H, I, dtype);
    if (rc != MOE_OK) return rc;
    if (out_dtype != dtype && out_dtype != MOE_F32)
        return fail(MOE_ERR_DTYPE, "out_dtype must be the expert dtype or F32");
    if (rows == 0) return MOE_OK;
    if (!x_disp || !offsets || !gate || !up || !down || !out_disp)
        return fail(MOE_ERR_NULL, "moe_experts_forward: NULL tensor");
    if (!aligned16(x_disp) || !aligned16(offsets) || !aligned16(gate) || !aligned16(up) ||
        !aligned16(down) || !aligned16(out_disp))
        return fail(MOE_ERR_ALIGN, "moe_experts_forward: tensors must be 16-byte aligned");
    const size_t need = moe_experts_workspace_size(rows, E, H, I, dtype);
    if (workspace_bytes < need || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_experts_forward: workspace too small or not 256-byte aligned");
    return run_experts(x_disp, offsets, rows, gate, up, down, E, H, I, dtype, workspace,
                       out_disp, out_dtype, static_cast<cudaStream_t>(stream));
}

int moe_combine(const void *out_disp, int out_dtype, const void *weights, int weights_dtype,
                const int32_t *row_of, int64_t T, int top_k, int64_t H, void *y, int dtype,
                void *stream)
{
    const NvtxRange nvtx("moe_combine");
    int rc = check_combine_args(out_dtype, weights_dtype, dtype, T, top_k, H, false);
    if (rc != MOE_OK || T == 0) return rc;
    if (!out_disp || !weights || !row_of || !y) return fail(MOE_ERR_NULL, "moe_combine: NULL tensor");
    if (!aligned16(out_disp) || !aligned16(weights) || !aligned16(row_of) || !aligned16(y))
        return fail(MOE_ERR_ALIGN, "moe_combine: tensors must be 16-byte aligned");
    cudaError_t err = launch_combine(out_disp, out_dtype, weights, weights_dtype, row_of, nullptr,
                                     nullptr, MOE_F32, 1.0f, T, top_k, H, y, dtype, nullptr,
                                     nullptr, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_combine");
}

int moe_combine_add_rmsnorm(const void *out_disp, int out_dtype, const void *weights,
                            int weights_dtype, const int32_t *row_of, const void *residual,
                            int dtype, const void *gamma, int gamma_dtype, float eps, int64_t T,
                            int top_k, int64_t H, void *y, void *x_out, float *rstd,
                            void *stream)
{
    const NvtxRange nvtx("moe_combine_add_rmsnorm");
    int rc = check_combine_args(out_dtype, weights_dtype, dtype, T, top_k, H, true);
    if (rc != MOE_OK) return rc;
    if (!valid_dtype(gamma_dtype)) return fail(MOE_ERR_DTYPE, "gamma dtype must be F32, BF16 or F16");
    if (!(isfinite(eps) && eps > 0.0f)) return fail(MOE_ERR_VALUE, "eps must be finite and > 0");
    if (T == 0) return MOE_OK;
    if (!out_disp || !weights || !row_of || !residual || !gamma || !y || !x_out || !rstd)
        return fail(MOE_ERR_NULL, "moe_combine_add_rmsnorm: NULL tensor");
    if (!aligned16(out_disp) || !aligned16(weights) || !aligned16(row_of) || !aligned16(residual) ||
        !aligned16(gamma) || !aligned16(y) || !aligned16(x_out) || !aligned16(rstd))
        return fail(MOE_ERR_ALIGN, "moe_combine_add_rmsnorm: tensors must be 16-byte aligned");
    cudaError_t err = launch_combine(out_disp, out_dtype, weights, weights_dtype, row_of, residual,
                                     gamma, gamma_dtype, eps, T, top_k, H, y, dtype, x_out, rstd,
                                     static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_combine_add_rmsnorm");
}

int moe_combine_v2(const void *out_disp, int out_dtype, const void *weights, int weights_dtype,
                   const int32_t *row_of, const moe_combine_extras *extras,
                   const void *residual, const void *gamma, int gamma_dtype, float eps,
                   int64_t T, int top_k, int64_t H, void *y, int dtype, void *x_out,
                   float *rstd, void *stream)
{
    const NvtxRange nvtx("moe_combine_v2");
    const bool norm = residual != nullptr;
    int rc = check_combine_args(out_dtype, weights_dtype, dtype, T, top_k, H, norm);
    if (rc != MOE_OK) return rc;
    if (norm) {
        if (!valid_dtype(gamma_dtype)) return fail(MOE_ERR_DTYPE, "gamma dtype must be F32, BF16 or F16");
        if (!(isfinite(eps) && eps > 0.0f)) return fail(MOE_ERR_VALUE, "eps must be finite and > 0");
    }
    CombineExtras ex{};
    if (extras != nullptr) {
        const moe_combine_extras &e = *extras;
        const int64_t special = e.zero_experts + e.copy_experts + e.const_experts;
        if (e.num_experts < 1 || e.zero_experts < 0 || e.copy_experts < 0 || e.const_experts < 0 ||
            special > 0x7fffffff - e.num_experts)
            return fail(MOE_ERR_SHAPE, "moe_combine_v2: need num_experts >= 1 and special expert counts >= 0");
        if (e.active_mask_dims < 0 || e.active_mask_dims > 2)
            return fail(MOE_ERR_SHAPE, "moe_combine_v2: active_mask_dims must be 0, 1 or 2");
        if (T > 0) {
            if ((special > 0 && !e.expert_indices) ||
                ((e.copy_experts > 0 || e.const_experts > 0) && !e.ori_x) ||
                (e.const_experts > 0 && (!e.const_alpha1 || !e.const_alpha2 || !e.const_v)) ||
                (e.active_mask_dims > 0 && !e.active_mask))
                return fail(MOE_ERR_NULL, "moe_combine_v2: an input its configured experts or mask need is NULL");
            if ((e.ori_x && !aligned16(e.ori_x)) || (e.const_v && !aligned16(e.const_v)) ||
                (e.shared_expert_x && !aligned16(e.shared_expert_x)))
                return fail(MOE_ERR_ALIGN, "moe_combine_v2: ori_x, const_v and shared_expert_x must be 16-byte aligned");
        }
        ex.ids = e.expert_indices;
        ex.E = e.num_experts;
        ex.zero_n = e.zero_experts;
        ex.copy_n = e.copy_experts;
        ex.const_n = e.const_experts;
        ex.ori_x = e.ori_x;
        ex.alpha1 = e.const_alpha1;
        ex.alpha2 = e.const_alpha2;
        ex.const_v = e.const_v;
        ex.shared_x = e.shared_expert_x;
        ex.mask = e.active_mask;
        ex.mask_dims = e.active_mask_dims;
    }
    if (T == 0) return MOE_OK;
    if (!out_disp || !weights || !row_of || !y || (norm && (!gamma || !x_out || !rstd)))
        return fail(MOE_ERR_NULL, "moe_combine_v2: NULL tensor");
    if (!aligned16(out_disp) || !aligned16(weights) || !aligned16(row_of) || !aligned16(y) ||
        (norm && (!aligned16(residual) || !aligned16(gamma) || !aligned16(x_out) || !aligned16(rstd))))
        return fail(MOE_ERR_ALIGN, "moe_combine_v2: tensors must be 16-byte aligned");
    cudaError_t err = launch_combine(out_disp, out_dtype, weights, weights_dtype, row_of, residual,
                                     gamma, gamma_dtype, eps, T, top_k, H, y, dtype, x_out, rstd,
                                     static_cast<cudaStream_t>(stream),
                                     extras != nullptr ? &ex : nullptr);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_combine_v2");
}

int moe_rmsnorm(const void *x, int dtype, const void *gamma, int gamma_dtype, float eps,
                int64_t rows, int64_t H, void *y, float *rstd, void *stream)
{
    const NvtxRange nvtx("moe_rmsnorm");
    if (!valid_dtype(dtype)) return fail(MOE_ERR_DTYPE, "x dtype must be F32, BF16 or F16");
    if (gamma_dtype != MOE_F32 && gamma_dtype != dtype)
        return fail(MOE_ERR_DTYPE, "gamma dtype must be F32 or the input dtype");
    if (rows < 0 || H < 1 || H % 8 != 0 || H > combine_max_h(true))
        return fail(MOE_ERR_SHAPE, "need rows >= 0 and H a multiple of 8 in [8, 16384]");
    if (!(isfinite(eps) && eps > 0.0f)) return fail(MOE_ERR_VALUE, "eps must be finite and > 0");
    if (rows == 0) return MOE_OK;
    if (!x || !gamma || !y) return fail(MOE_ERR_NULL, "moe_rmsnorm: NULL tensor");
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(y) || (rstd && !aligned16(rstd)))
        return fail(MOE_ERR_ALIGN, "moe_rmsnorm: tensors must be 16-byte aligned");
    cudaError_t err = launch_rmsnorm(x, dtype, gamma, gamma_dtype, eps, rows, H, y, rstd,
                                     static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_rmsnorm");
}

size_t moe_forward_workspace_size_ex(int64_t T, int64_t H, int64_t I, int64_t E, int top_k,
                                     int dtype, int logits_dtype, unsigned flags)
{
    if (T <= 0 || H < 1 || I < 1 || E < 1 || E > kMaxE || top_k < 1 || top_k > E ||
        !valid_dtype(dtype) || !valid_dtype(logits_dtype) ||
        (flags & ~(unsigned)MOE_FORWARD_DETERMINISTIC))
        return 0;
    return forward_layout(T, H, I, E, top_k, dtype, logits_dtype, flags).total;
}

size_t moe_forward_workspace_size(int64_t T, int64_t H, int64_t I, int64_t E, int top_k,
                                  int dtype, int logits_dtype)
{
    return moe_forward_workspace_size_ex(T, H, I, E, top_k, dtype, logits_dtype, 0u);
}

int moe_forward_workspace_layout(int64_t T, int64_t H, int64_t I, int64_t E, int top_k,
                                 int dtype, int logits_dtype, unsigned flags,
                                 moe_forward_layout *layout)
{
    if (layout == nullptr) return fail(MOE_ERR_NULL, "moe_forward_workspace_layout: NULL layout");
    if (!valid_dtype(dtype) || !valid_dtype(logits_dtype))
        return fail(MOE_ERR_DTYPE, "dtype must be F32, BF16 or F16");
    if (flags & ~(unsigned)MOE_FORWARD_DETERMINISTIC)
        return fail(MOE_ERR_VALUE, "unknown moe_forward_options flag");
    if (T <= 0 || H < 1 || I < 1 || E < 1 || E > kMaxE || top_k < 1 || top_k > E ||
        T * top_k > kMaxRows)
        return fail(MOE_ERR_SHAPE, "need T >= 1, H, I >= 1, 1 <= E <= 1024, 1 <= top_k <= E");
    const ForwardLayout L = forward_layout(T, H, I, E, top_k, dtype, logits_dtype, flags);
    layout->expert_indices = L.idx;
    layout->weights = L.w;
    layout->counts = L.counts;
    layout->offsets = L.offsets;
    layout->row_of = L.row_of;
    layout->src_of = L.src_of;
    layout->x_disp = L.x_disp;
    layout->total = L.total;
    return MOE_OK;
}

int moe_forward_ex(const void *x, int dtype, const void *logits, int logits_dtype,
                   const void *gate, const void *up, const void *down, int64_t T, int64_t H,
                   int64_t I, int64_t E, int top_k, int renormalize, void *y, void *workspace,
                   size_t workspace_bytes, const moe_forward_options *options, void *stream)
{
    const NvtxRange nvtx("moe_forward_ex");
    const moe_sigmoid_grouped_routing *sg = options != nullptr ? options->sigmoid_grouped : nullptr;
    if (sg == nullptr)
        return forward_impl("moe_forward: NULL tensor", x, dtype, logits, logits_dtype, gate, up,
                            down, T, H, I, E, top_k, y, workspace, workspace_bytes, options,
                            stream,
                            [&](uint32_t *idx, void *w, const DispatchOut &d, cudaStream_t s) {
                                return launch_route_dispatch(
                                    logits, logits_dtype, T, (int)E, top_k, renormalize, idx, w,
                                    x, dtype, H, d.counts, d.offsets, d.row_of, d.src_of,
                                    d.x_disp, d.ws, d.zeroed, d.status, s);
                            });
    if (E >= 1 && E <= kMaxE && top_k >= 1) {
        const int rc = check_sigmoid_grouped_args(E, sg->bias, top_k, sg->groups,
                                                  sg->selected_groups, sg->group_top_two,
                                                  sg->scale);
        if (rc != MOE_OK) return rc;
    }
    return forward_impl("moe_forward_sigmoid_grouped: NULL tensor", x, dtype, logits,
                        logits_dtype, gate, up, down, T, H, I, E, top_k, y, workspace,
                        workspace_bytes, options, stream,
                        [&](uint32_t *idx, void *w, const DispatchOut &d, cudaStream_t s) {
                            cudaError_t err = launch_route_sigmoid_grouped(
                                logits, logits_dtype, T, (int)E, sg->bias, top_k, sg->groups,
                                sg->selected_groups, sg->group_top_two, renormalize, sg->scale,
                                idx, w, s);
                            if (err != cudaSuccess) return err;
                            return launch_dispatch(idx, T, top_k, (int)E, 0, x, dtype, H,
                                                   d.counts, d.offsets, d.row_of, d.src_of,
                                                   d.x_disp, d.ws, d.status, s);
                        });
}

int moe_forward(const void *x, int dtype, const void *logits, int logits_dtype, const void *gate,
                const void *up, const void *down, int64_t T, int64_t H, int64_t I, int64_t E,
                int top_k, int renormalize, void *y, void *workspace, size_t workspace_bytes,
                void *stream)
{
    return moe_forward_ex(x, dtype, logits, logits_dtype, gate, up, down, T, H, I, E, top_k,
                          renormalize, y, workspace, workspace_bytes, nullptr, stream);
}

int moe_forward_sigmoid_grouped(const void *x, int dtype, const void *logits, int logits_dtype,
                                const float *bias, const void *gate, const void *up,
                                const void *down, int64_t T, int64_t H, int64_t I, int64_t E,
                                int top_k, int groups, int selected_groups, int group_top_two,
                                int renormalize, float scale, void *y, void *workspace,
                                size_t workspace_bytes, void *stream)
{
    const moe_sigmoid_grouped_routing sg{bias, groups, selected_groups, group_top_two, scale};
    moe_forward_options opt{};
    opt.sigmoid_grouped = &sg;
    return moe_forward_ex(x, dtype, logits, logits_dtype, gate, up, down, T, H, I, E, top_k,
                          renormalize, y, workspace, workspace_bytes, &opt, stream);
}

int moe_set_wait_limit_ns(uint64_t limit_ns)
{
    if (limit_ns > kMaxWaitLimitNs)
        return fail(MOE_ERR_VALUE, "moe_set_wait_limit_ns: the limit must be at most 60 s");
    g_wait_limit_ns.store(limit_ns == 0 ? kWaitLimitNs : limit_ns);
    return MOE_OK;
}

uint64_t moe_wait_limit_ns(void) { return wait_limit_ns(); }

size_t moe_selftest_wait_expiry_workspace_size(int64_t E, int64_t rows_per_expert, int64_t H,
                                               int64_t I)
{
    if (E < 1 || E > kMaxE || rows_per_expert < 1 || rows_per_expert > 4096 || H < 8 ||
        H > 8192 || H % 8 != 0 || I < 8 || I > 8192 || I % 8 != 0)
        return 0;
    return selftest_wait_workspace_bytes((int)E, (int)rows_per_expert, H, I);
}

int moe_selftest_wait_expiry(int64_t E, int64_t rows_per_expert, int64_t H, int64_t I,
                             float *y_acc, void *workspace, size_t workspace_bytes, void *stream)
{
    const NvtxRange nvtx("moe_selftest_wait_expiry");
    const size_t need = moe_selftest_wait_expiry_workspace_size(E, rows_per_expert, H, I);
    if (need == 0)
        return fail(MOE_ERR_SHAPE, "moe_selftest_wait_expiry: need 1 <= E <= 1024, "
                                   "1 <= rows_per_expert <= 4096, H and I multiples of 8 in [8, 8192]");
    if (y_acc == nullptr || workspace == nullptr)
        return fail(MOE_ERR_NULL, "moe_selftest_wait_expiry: NULL y_acc or workspace");
    if (!aligned16(y_acc)) return fail(MOE_ERR_ALIGN, "moe_selftest_wait_expiry: y_acc must be 16-byte aligned");
    if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_selftest_wait_expiry: workspace too small or not 256-byte aligned");
    unsigned *st = status_ptr();
    if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
    cudaError_t err = launch_selftest_wait_expiry((int)E, (int)rows_per_expert, H, I, workspace,
                                                  y_acc, st, static_cast<cudaStream_t>(stream));
    if (err == cudaErrorInvalidValue)
        return fail(MOE_ERR_ALIGN, "TMA descriptor rejected (pointer alignment or shape)");
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_selftest_wait_expiry");
}

// ---- first-order training (ruDNN user guide, section 12) ------------------

namespace {

int check_router_train_args(const void *logits, int ldt, int64_t T, int64_t E, const void *idx,
                            int idt, int top_k, int scoring, float scale, const void *in2,
                            const void *out)
{
    if (!valid_dtype(ldt)) return fail(MOE_ERR_DTYPE, "logits dtype must be F32, BF16 or F16");
    if (idt != MOE_INDEX_U32 && idt != MOE_INDEX_I32 && idt != MOE_INDEX_I64)
        return fail(MOE_ERR_DTYPE, "index dtype must be U32, I32 or I64");
    if (scoring != MOE_SCORING_SOFTMAX && scoring != MOE_SCORING_SIGMOID)
        return fail(MOE_ERR_DTYPE, "scoring must be softmax or sigmoid");
    if (T < 0 || E < 1 || E > kMaxE) return fail(MOE_ERR_SHAPE, "need T >= 0 and 1 <= E <= 1024");
    if (top_k < 1 || top_k > E || top_k > router_train_max_top_k())
        return fail(MOE_ERR_SHAPE, "need 1 <= top_k <= min(E, 64)");
    if (T * top_k > kMaxRows) return fail(MOE_ERR_SHAPE, "T * top_k exceeds 2^31 - 1");
    if (!std::isfinite(scale) || !(scale > 0.0f)) return fail(MOE_ERR_VALUE, "scale must be finite and > 0");
    if (T == 0) return MOE_OK;
    if (!logits || !idx || !in2 || !out) return fail(MOE_ERR_NULL, "router training: NULL tensor");
    if (!aligned16(logits) || !aligned16(idx) || !aligned16(in2) || !aligned16(out))
        return fail(MOE_ERR_ALIGN, "router training: tensors must be 16-byte aligned");
    return MOE_OK;
}

// Training cache: h [rows, I] in the expert dtype, then g and u [rows, I] in FP32.
size_t cache_bytes_for(int64_t rows, int64_t I, int dt)
{
    return round_up((size_t)rows * (size_t)I * (elem_bytes(dt) + 8), 256);
}

int check_experts_ptrs(const char *name, std::initializer_list<const void *> ptrs)
{
    for (const void *q : ptrs)
        if (!q) return fail(MOE_ERR_NULL, name);
    for (const void *q : ptrs)
        if (!aligned16(q)) return fail(MOE_ERR_ALIGN, name);
    return MOE_OK;
}

}  // namespace

int moe_router_weights(const void *logits, int logits_dtype, int64_t T, int64_t E,
                       const void *indices, int index_dtype, int top_k, int scoring,
                       int renormalize, float scale, float *weights, void *stream)
{
    const NvtxRange nvtx("moe_router_weights");
    int rc = check_router_train_args(logits, logits_dtype, T, E, indices, index_dtype, top_k,
                                     scoring, scale, weights, weights);
    if (rc != MOE_OK || T == 0) return rc;
    unsigned *st = status_ptr();
    if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
    cudaError_t err = launch_router_weights(logits, logits_dtype, T, (int)E, indices, index_dtype,
                                            top_k, scoring == MOE_SCORING_SIGMOID, renormalize != 0,
                                            scale, weights, st, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_router_weights");
}

int moe_router_backward(const void *logits, int logits_dtype, int64_t T, int64_t E,
                        const void *indices, int index_dtype, int top_k,
                        const float *grad_weights, int scoring, int renormalize, float scale,
                        void *grad_logits, void *stream)
{
    const NvtxRange nvtx("moe_router_backward");
    int rc = check_router_train_args(logits, logits_dtype, T, E, indices, index_dtype, top_k,
                                     scoring, scale, grad_weights, grad_logits);
    if (rc != MOE_OK || T == 0) return rc;
    unsigned *st = status_ptr();
    if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
    cudaError_t err = launch_router_backward(logits, logits_dtype, T, (int)E, indices,
                                             index_dtype, top_k, grad_weights,
                                             scoring == MOE_SCORING_SIGMOID, renormalize != 0,
                                             scale, grad_logits, st,
                                             static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_router_backward");
}

int moe_combine_backward(const void *out_disp, int out_dtype, const void *weights,
                         int weights_dtype, const int32_t *row_of, const void *grad_y,
                         int64_t T, int top_k, int64_t H, int dtype, void *grad_out_disp,
                         float *grad_weights, void *stream)
{
    const NvtxRange nvtx("moe_combine_backward");
    if (!valid_dtype(out_dtype) || !valid_dtype(weights_dtype) || !valid_dtype(dtype))
        return fail(MOE_ERR_DTYPE, "dtype must be F32, BF16 or F16");
    if (out_dtype != dtype && out_dtype != MOE_F32)
        return fail(MOE_ERR_DTYPE, "expert outputs must be in the activation dtype or F32");
    if (T < 0 || top_k < 1 || T * top_k > kMaxRows)
        return fail(MOE_ERR_SHAPE, "need T >= 0, top_k >= 1, T*top_k < 2^31");
    if (H < 1 || H % 8 != 0) return fail(MOE_ERR_SHAPE, "H must be a positive multiple of 8");
    if (T == 0) return MOE_OK;
    int rc = check_experts_ptrs("moe_combine_backward: tensors must be non-NULL and 16-byte aligned",
                                {out_disp, weights, row_of, grad_y, grad_out_disp, grad_weights});
    if (rc != MOE_OK) return rc;
    cudaError_t err = launch_combine_backward(out_disp, out_dtype, weights, weights_dtype, row_of,
                                              grad_y, dtype, T, top_k, H, grad_out_disp,
                                              grad_weights, static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_combine_backward");
}

int moe_dispatch_backward(const void *grad_x_disp, int dtype, const int32_t *row_of,
                          int64_t T, int top_k, int64_t H, void *grad_x, void *stream)
{
    const NvtxRange nvtx("moe_dispatch_backward");
    if (!valid_dtype(dtype)) return fail(MOE_ERR_DTYPE, "dtype must be F32, BF16 or F16");
    if (T < 0 || top_k < 1 || T * top_k > kMaxRows)
        return fail(MOE_ERR_SHAPE, "need T >= 0, top_k >= 1, T*top_k < 2^31");
    if (H < 1 || H % 8 != 0) return fail(MOE_ERR_SHAPE, "H must be a positive multiple of 8");
    if (T == 0) return MOE_OK;
    int rc = check_experts_ptrs("moe_dispatch_backward: tensors must be non-NULL and 16-byte aligned",
                                {grad_x_disp, row_of, grad_x});
    if (rc != MOE_OK) return rc;
    cudaError_t err = launch_dispatch_backward(grad_x_disp, dtype, row_of, T, top_k, H, grad_x,
                                               static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_dispatch_backward");
}

size_t moe_experts_training_cache_size(int64_t rows, int64_t I, int dtype)
{
    if (rows <= 0 || I <= 0 || !valid_dtype(dtype)) return 0;
    return cache_bytes_for(rows, I, dtype);
}

int moe_experts_forward_training(const void *x_disp, const int32_t *offsets, int64_t rows,
                                 const void *gate, const void *up, const void *down, int64_t E,
                                 int64_t H, int64_t I, int dtype, void *out_disp, int out_dtype,
                                 void *cache, size_t cache_bytes, void *stream)
{
    const NvtxRange nvtx("moe_experts_forward_training");
    int rc = check_experts_args(rows, E, H, I, dtype);
    if (rc != MOE_OK) return rc;
    if (out_dtype != dtype && out_dtype != MOE_F32)
        return fail(MOE_ERR_DTYPE, "out_dtype must be the expert dtype or F32");
    if (rows == 0) return MOE_OK;
    rc = check_experts_ptrs("moe_experts_forward_training: tensors must be non-NULL and 16-byte aligned",
                            {x_disp, offsets, gate, up, down, out_disp});
    if (rc != MOE_OK) return rc;
    if (cache_bytes < cache_bytes_for(rows, I, dtype) || !cache ||
        (reinterpret_cast<uintptr_t>(cache) & 255u))
        return fail(MOE_ERR_WORKSPACE, "moe_experts_forward_training: cache too small or not 256-byte aligned");
    uint8_t *h = static_cast<uint8_t *>(cache);
    uint8_t *g = h + (size_t)rows * (size_t)I * elem_bytes(dtype);
    uint8_t *u = g + (size_t)rows * (size_t)I * 4;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (dtype == MOE_F32) {
        err = launch_experts_simt(static_cast<const float *>(x_disp), offsets, rows,
                                  static_cast<const float *>(gate), static_cast<const float *>(up),
                                  static_cast<const float *>(down), (int)E, H, I,
                                  reinterpret_cast<float *>(h), static_cast<float *>(out_disp), s,
                                  reinterpret_cast<float *>(g), reinterpret_cast<float *>(u));
    } else {
        unsigned *st = status_ptr();
        if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
        err = launch_experts_tc_training(dtype, x_disp, offsets, rows, gate, up, down, (int)E, H,
                                         I, cache, out_disp, out_dtype == MOE_F32, st, s);
        if (err == cudaErrorInvalidValue)
            return fail(MOE_ERR_ALIGN, "TMA descriptor rejected (pointer alignment or shape)");
    }
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_experts_forward_training");
}

// Expert backward workspace: dgu [rows, 2I] in the expert dtype, then (BF16 /
// F16) the per-expert tensor maps of the weight-gradient GEMMs.
size_t backward_dgu_bytes(int64_t rows, int64_t I, int dtype)
{
    return round_up(2 * (size_t)(rows > 0 ? rows : 0) * (size_t)I * elem_bytes(dtype), 256);
}

size_t moe_experts_backward_workspace_size(int64_t rows, int64_t E, int64_t H, int64_t I,
                                           int dtype)
{
    (void)H;
    if (rows < 0 || I <= 0 || E < 1 || E > kMaxE || !valid_dtype(dtype)) return 0;
    size_t n = backward_dgu_bytes(rows, I, dtype);
    if (dtype != MOE_F32) n += round_up(experts_tc_backward_maps_bytes((int)E), 256);
    return n;
}

int moe_experts_backward(const void *x_disp, const int32_t *offsets, int64_t rows,
                         const void *gate, const void *up, const void *down, int64_t E,
                         int64_t H, int64_t I, int dtype, const void *cache,
                         const void *grad_out, void *grad_x_disp, float *grad_gate,
                         float *grad_up, float *grad_down, void *workspace,
                         size_t workspace_bytes, void *stream)
{
    const NvtxRange nvtx("moe_experts_backward");
    int rc = check_experts_args(rows, E, H, I, dtype);
    if (rc != MOE_OK) return rc;
    rc = check_experts_ptrs("moe_experts_backward: tensors must be non-NULL and 16-byte aligned",
                            {offsets, gate, up, down, grad_gate, grad_up, grad_down});
    if (rc != MOE_OK) return rc;
    if (rows > 0) {
        rc = check_experts_ptrs("moe_experts_backward: tensors must be non-NULL and 16-byte aligned",
                                {x_disp, cache, grad_out, grad_x_disp});
        if (rc != MOE_OK) return rc;
        if ((reinterpret_cast<uintptr_t>(cache) & 255u))
            return fail(MOE_ERR_WORKSPACE, "moe_experts_backward: cache not 256-byte aligned");
    }
    const size_t need = moe_experts_backward_workspace_size(rows, E, H, I, dtype);
    if (need > 0 && (workspace_bytes < need || !workspace ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(MOE_ERR_WORKSPACE, "moe_experts_backward: workspace too small or not 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t err;
    if (dtype == MOE_F32) {
        err = launch_experts_simt_backward(
            static_cast<const float *>(x_disp), offsets, rows, static_cast<const float *>(gate),
            static_cast<const float *>(up), static_cast<const float *>(down), (int)E, H, I,
            static_cast<const float *>(cache), static_cast<const float *>(grad_out),
            static_cast<float *>(workspace), static_cast<float *>(grad_x_disp), grad_gate, grad_up,
            grad_down, s);
    } else {
        unsigned *st = status_ptr();
        if (!st) return fail(MOE_ERR_CUDA, "cannot resolve the device status word");
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        err = launch_experts_tc_backward(dtype, x_disp, offsets, rows, gate, up, down, (int)E, H, I,
                                         cache, grad_out, rows > 0 ? ws : nullptr,
                                         ws + backward_dgu_bytes(rows, I, dtype), grad_x_disp,
                                         grad_gate, grad_up, grad_down, st, s);
        if (err == cudaErrorInvalidValue)
            return fail(MOE_ERR_ALIGN, "TMA descriptor rejected (pointer alignment or shape)");
    }
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_experts_backward");
}

int moe_device_status(void *stream, int clear)
{
    cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (err != cudaSuccess) return cuda_fail(err, "moe_device_status/sync");
    unsigned v = 0;
    err = cudaMemcpyFromSymbol(&v, g_moe_status, sizeof v);
    if (err != cudaSuccess) return cuda_fail(err, "moe_device_status/read");
    if (clear) {
        const unsigned zero = 0;
        err = cudaMemcpyToSymbol(g_moe_status, &zero, sizeof zero);
        if (err != cudaSuccess) return cuda_fail(err, "moe_device_status/clear");
    }
    if (v & ST_TIMEOUT) return MOE_ERR_DEVICE_TIMEOUT;
    if (v & ST_BOUNDS) return MOE_ERR_BOUNDS;
    if (v & ST_BAD_INDEX) return MOE_ERR_BAD_INDEX;
    return MOE_OK;
}

}  // extern "C"
