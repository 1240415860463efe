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

// Host-side argument checks of moe_dispatch_special (moe_dispatch with
// special_experts = 0) short of the workspace: MOE_OK or the status the call
// returns, with the detail recorded.
int check_dispatch_args(const uint32_t *expert_indices, int64_t T, int top_k, int64_t E,
                        int64_t special_experts, const void *x, int x_dtype, int64_t H,
                        const int32_t *counts, const int32_t *offsets, const int32_t *row_of,
                        const int32_t *src_of, const void *x_disp);

// Limit of every bounded device wait, passed to the kernels at launch
// (kWaitLimitNs unless moe_set_wait_limit_ns() set another).
uint64_t wait_limit_ns();

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
// Assignments per dispatch chunk; the workspace of launch_route_dispatch
// (the dispatch workspace and the fused kernel's completion counter after
// it) and where that counter sits.
int64_t dispatch_chunk_len(int64_t A);
size_t route_dispatch_workspace_bytes(int64_t A, int E);
unsigned *dispatch_done_counter(void *ws, int64_t A, int E);
// The rank/scatter and the row gather alone, once the workspace holds each
// chunk's first row inside every expert and counts[] the expert totals.
cudaError_t launch_dispatch_rank_gather(const uint32_t *idx, int64_t T, int top_k, int E,
                                        const void *x, int xdt, int64_t H, const int32_t *counts,
                                        int32_t *offsets, int32_t *row_of, int32_t *src_of,
                                        void *x_disp, void *ws, unsigned *status, cudaStream_t s);
// Routing fused with the dispatch's chunk counts and their scan (one kernel:
// each CTA routes the tokens of one assignment chunk and counts them; the
// last CTA to finish scans the counts), then the rank/scatter and the gather:
// three launches instead of five. Falls back to launch_route + launch_dispatch
// where the fused kernel does not apply (one thread per token pays, E > 1024,
// or more chunk counts than the last CTA scans in shared memory).
// zeroed_counter: a zero word the caller has cleared on the stream for the
// kernel's completion count (nullptr: one in ws, cleared here).
cudaError_t launch_route_dispatch(const void *logits, int ldt, int64_t T, int E, int top_k,
                                  int renormalize, uint32_t *idx, void *w, const void *x,
                                  int xdt, int64_t H, int32_t *counts, int32_t *offsets,
                                  int32_t *row_of, int32_t *src_of, void *x_disp, void *ws,
                                  unsigned *zeroed_counter, unsigned *status, cudaStream_t s);
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

// FP32 SwiGLU experts on CUDA cores. h_ws holds [rows, I] floats. With
// g_out / u_out (training) the gate and up products [rows, I] are kept too.
cudaError_t launch_experts_simt(const float *x_disp, const int32_t *offsets,
                                int64_t rows, const float *gate,
                                const float *up, const float *down, int E,
                                int64_t H, int64_t I, float *h_ws,
                                float *out_disp, cudaStream_t s, float *g_out = nullptr,
                                float *u_out = nullptr);

// FP32 SwiGLU expert backward on CUDA cores, in three steps:
//   dgu [rows, 2I]: per row, dg = dh * u * s * (1 + g (1 - s)) in columns
//                   [0, I) and du = dh * g * s in [I, 2I), dh = dout Wd[e]
//                   (s = sigmoid(g); g, u from the forward's cache);
//   dx  [rows, H] = dg Wg[e] + du Wu[e];
//   dgate/dup [E, I, H] and ddown [E, H, I] (FP32): sums over each expert's
//   rows of dg x^T, du x^T and dout h^T; experts without rows get zeros.
// cache holds h, g, u as three [rows, I] arrays.
cudaError_t launch_experts_simt_backward(const float *x_disp, const int32_t *offsets,
                                         int64_t rows, const float *gate, const float *up,
                                         const float *down, int E, int64_t H, int64_t I,
                                         const float *cache, const float *dout, float *dgu,
                                         float *dx, float *dgate, float *dup, float *ddown,
                                         cudaStream_t s);

// ---- first-order training (ruDNN user guide, section 12) ----
int router_train_max_top_k();
// FP32 weights [T, k] of a fixed selection (idt: IDX_*); sigmoid selects the
// scoring; ids outside [0, E) NaN the row and set ST_BAD_INDEX.
cudaError_t launch_router_weights(const void *logits, int ldt, int64_t T, int E, const void *idx,
                                  int idt, int k, int sigmoid, int renorm, float scale,
                                  float *w_out, unsigned *status, cudaStream_t s);
// Logits gradient [T, E] in ldt for the FP32 weight gradient gw [T, k].
cudaError_t launch_router_backward(const void *logits, int ldt, int64_t T, int E,
                                   const void *idx, int idt, int k, const float *gw,
                                   int sigmoid, int renorm, float scale, void *dl_out,
                                   unsigned *status, cudaStream_t s);
// dexp[row_of[a]] = w[a] * gy[a / k] (dtype dt), dw[a] = <gy, out_disp row>
// (FP32); out_disp in odt (dt or F32); H % 8 == 0.
cudaError_t launch_combine_backward(const void *out_disp, int odt, const void *w, int wdt,
                                    const int32_t *row_of, const void *gy, int dt, int64_t T,
                                    int k, int64_t H, void *dexp, float *dw, cudaStream_t s);
// dx[t] = sum_j d[row_of[t*k + j]] (rows with row_of < 0 skipped); H % 8 == 0.
cudaError_t launch_dispatch_backward(const void *d, int dt, const int32_t *row_of, int64_t T,
                                     int k, int64_t H, void *dx, cudaStream_t s);

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
// zeroed by the caller), in an order that varies from run to run. ready: E
// zeroed per-expert counters through which GEMM2 starts on each expert as
// soon as GEMM1 has stored its h rows (nullptr: GEMM2 waits for all of GEMM1).
cudaError_t launch_experts_tc_combine(int dt, const void *x_disp,
                                      const int32_t *offsets, int64_t rows,
                                      const void *gate, const void *up,
                                      const void *down, int E, int64_t H, int64_t I,
                                      void *h_ws, const int32_t *src_of,
                                      const void *w, int wdt, int top_k,
                                      float *y_acc, unsigned *ready, unsigned *status,
                                      cudaStream_t s);

// Training forward: launch_experts_tc with g and u kept. cache holds h, g, u
// as three [rows, I] arrays of dt (h feeds the second GEMM).
cudaError_t launch_experts_tc_training(int dt, const void *x_disp, const int32_t *offsets,
                                       int64_t rows, const void *gate, const void *up,
                                       const void *down, int E, int64_t H, int64_t I,
                                       void *cache, void *out_disp, bool out_f32,
                                       unsigned *status, cudaStream_t s);

// Expert backward on tcgen05 (see launch_experts_simt_backward for the
// math); dgu_ws holds [rows, 2I] of dt, maps_ws the per-expert tensor maps of
// the weight-gradient GEMMs (experts_tc_backward_maps_bytes(E), 128-byte
// aligned).
size_t experts_tc_backward_maps_bytes(int E);
cudaError_t launch_experts_tc_backward(int dt, const void *x_disp, const int32_t *offsets,
                                       int64_t rows, const void *gate, const void *up,
                                       const void *down, int E, int64_t H, int64_t I,
                                       const void *cache, const void *dout, void *dgu_ws,
                                       void *maps_ws, void *dx, float *dgate, float *dup,
                                       float *ddown, unsigned *status, cudaStream_t s);

// The library's test of its bounded waits: GEMM2 of the one-call forward
// (BF16, combine folded into y_acc [E * rows_per_expert, H] FP32, top_k 1,
// per-expert readiness) launched on its own over zeroed data, with readiness
// counters that nothing raises; ws holds selftest_wait_workspace_bytes(...)
// (offsets, map, routing weights, counters, h, down).
size_t selftest_wait_workspace_bytes(int E, int rows_per_expert, int64_t H, int64_t I);
cudaError_t launch_selftest_wait_expiry(int E, int rows_per_expert, int64_t H, int64_t I,
                                        void *ws, float *y_acc, unsigned *status, cudaStream_t s);

// y = y_acc rounded to ydt ([T, H], H % 8 == 0).
cudaError_t launch_finalize(const float *y_acc, int64_t T, int64_t H, void *y, int ydt,
                            cudaStream_t s);

}  // namespace moe
