// kernels.h -- host-side launchers of the GB300 MoE kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Records `what` as the text moe_last_error_detail() returns on this thread
// and returns `code`.
int report_error(int code, const char *what);

// Softmax top-k routing, warp per token. E <= 1024.
cudaError_t launch_route(const void *logits, int ldt, int64_t T, int E,
                         int top_k, int renormalize, uint32_t *idx, void *w,
                         cudaStream_t s);

// Group-limited sigmoid routing (one warp per token); the limits are the
// caller's to check. Largest top_k and group count the kernel supports.
cudaError_t launch_route_sigmoid_grouped(const void *logits, int ldt, int64_t T, int E,
                                         const float *bias, int top_k, int groups,
                                         int selected_groups, int group_top_two,
                                         int renormalize, float scale, uint32_t *idx, void *w,
                                         cudaStream_t s);
int sigmoid_route_max_top_k();
int sigmoid_route_max_groups();

// Dispatch: per-chunk histograms, a scan, a stable rank/scatter, a row gather.
size_t dispatch_workspace_bytes(int64_t A, int E);
// Expert ids in [E, E + special) are special experts (see CombineExtras):
// they get no row and are not reported as bad indices.
cudaError_t launch_dispatch(const uint32_t *idx, int64_t T, int top_k, int E, int64_t special,
                            const void *x, int xdt, int64_t H, int32_t *counts,
                            int32_t *offsets, int32_t *row_of, int32_t *src_of,
                            void *x_disp, void *ws, unsigned *status,
                            cudaStream_t s);

// Weighted combine, optionally followed by residual Add + RMSNorm.
// out_disp in odt; y, residual and x_out in ydt; H % 8 == 0.
int combine_max_h(bool norm);
// Special experts, shared expert and active mask of the combine (all zero /
// NULL: none). ori_x, alpha1/2, const_v and shared_x are in the activation
// dtype; ids may be NULL when no special experts are configured.
struct CombineExtras {
    const uint32_t *ids;
    int64_t E, zero_n, copy_n, const_n;
    const void *ori_x, *alpha1, *alpha2, *const_v, *shared_x;
    const uint8_t *mask;
    int mask_dims;                // 0, 1 ([T]) or 2 ([T, top_k])
};

cudaError_t launch_combine(const void *out_disp, int odt, const void *w, int wdt,
                           const int32_t *row_of, const void *residual,
                           const void *gamma, int gdt, float eps, int64_t T,
                           int top_k, int64_t H, void *y, int ydt, void *x_out,
                           float *rstd, cudaStream_t s,
                           const CombineExtras *extras = nullptr);

// Standalone RMSNorm of rows x [rows, H] (H % 8 == 0, H <= combine_max_h(true)).
cudaError_t launch_rmsnorm(const void *x, int xdt, const void *gamma, int gdt, float eps,
                           int64_t rows, int64_t H, void *y, float *rstd, cudaStream_t s);

// FP32 SwiGLU experts on CUDA cores. h_ws holds [rows, I] floats.
cudaError_t launch_experts_simt(const float *x_disp, const int32_t *offsets,
                                int64_t rows, const float *gate,
                                const float *up, const float *down, int E,
                                int64_t H, int64_t I, float *h_ws,
                                float *out_disp, cudaStream_t s);

// BF16/F16 SwiGLU experts on tcgen05 tensor cores (TMA + TMEM).
// h_ws holds [rows, I] elements of dt; out_disp is FP32 when out_f32, else dt.
// Returns cudaErrorInvalidValue when a TMA descriptor cannot be encoded for
// the given shapes/pointers.
cudaError_t launch_experts_tc(int dt, const void *x_disp,
                              const int32_t *offsets, int64_t rows,
                              const void *gate, const void *up,
                              const void *down, int E, int64_t H, int64_t I,
                              void *h_ws, void *out_disp, bool out_f32,
                              unsigned *status, cudaStream_t s);

// Same GEMMs, with the weighted combine folded into GEMM2: every dispatched
// row r adds w[src_of[r]] * out_r into y_acc[src_of[r] / top_k] (FP32 [T, H],
// zeroed by the caller), in an order that varies from run to run.
cudaError_t launch_experts_tc_combine(int dt, const void *x_disp,
                                      const int32_t *offsets, int64_t rows,
                                      const void *gate, const void *up,
                                      const void *down, int E, int64_t H, int64_t I,
                                      void *h_ws, const int32_t *src_of,
                                      const void *w, int wdt, int top_k,
                                      float *y_acc, unsigned *status, cudaStream_t s);

// y = y_acc rounded to ydt ([T, H], H % 8 == 0).
cudaError_t launch_finalize(const float *y_acc, int64_t T, int64_t H, void *y, int ydt,
                            cudaStream_t s);

}  // namespace moe
