// fcm_internal.h -- host-side internals shared by the C ABI, the planner and the launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/fcm.h"

// An NVTX range over the scope of one entry point (a profiler's timeline shows each call; with
// no tool attached a push or pop costs one indirect call).
struct FcmNvtxRange {
    explicit FcmNvtxRange(const char *name) { nvtxRangePushA(name); }
    ~FcmNvtxRange() { nvtxRangePop(); }
    FcmNvtxRange(const FcmNvtxRange &) = delete;
    FcmNvtxRange &operator=(const FcmNvtxRange &) = delete;
};

// Bytes of one element of a storage type.
inline int fcm_dtype_bytes(int dtype) { return dtype == FCM_F32 ? 4 : dtype == FCM_I8 ? 1 : 2; }

// Device error word bits, written by kernels with atomicOr and read by fcm_check.
enum : unsigned {
    FCM_DEVERR_TIMEOUT = 1u,   // a bounded mbarrier wait gave up
    FCM_DEVERR_CHECK = 2u,     // a kernel-side consistency check failed
};

// Planner-chosen configuration of the tensor-core kernels.
struct TcPlan {
    int tile_h = 0, tile_w = 0;   // output tile (tile_h * tile_w <= 128 = MMA M)
    int in_rows = 0, in_cols = 0; // input halo box
    int chunk_c = 0;              // channels per input stage
    int nchunks = 0;              // C / chunk_c
    int stages = 0;               // input ring depth
    int dw_warps = 0;             // warps running the DW stencil
    int tiles_w = 0, tiles_h = 0; // tiles per image along W and H
    long long num_tiles = 0;
    int smem_bytes = 0;
    int threads = 0;
    int ctas = 0;
    int tmem_cols = 0;
    int out_bufs = 1;             // DW->PW output staging tiles (2: stores overlap the next tile)
    int dw_per_chunk = 0;         // >0: each DW warp serves one channel chunk (taps in registers)
    // Fused DW->PW kernel variant: 0 = dwpw_kernel (dedicated producer/MMA/epilogue/stencil
    // warps), 1 = dwpw_fused_kernel (worker warps that run the stencil and the epilogue)
    int variant = 0;
    int qw = 0, qh = 0, nqx = 0;  // variant 1: pixels of a TMEM lane quadrant (qw x qh), quadrants across
    int nw = 0;                   // variant 1: worker warps
    int abufs = 0;                // variant 1: A tiles (2: the stencil of tile t+1 overlaps the MMA of t)
    int sbufs = 0;                // variant 1: output staging buffers (2: stores overlap the next tile)
    int cp = 0;                   // variant 1: channels padded to a multiple of 64
    int ngroups = 0;              // variant 1: 4-pixel DW units per tile row
};

struct fcm_handle {
    fcm_desc d{};
    fcm_plan_info plan{};
    TcPlan tc{};
    TcPlan tc2{};             // PWDW: plan of the layer-by-layer depthwise stage;
                              // INT8: plan of the PW-only stage (identity stencil, k = 1)
    TcPlan tc_lbl{};          // DW->PW handles whose fused plan is variant 1: the plan of the
                              // layer-by-layer modes (DW-only, PW-only) on dwpw_kernel;
                              // INT8 PWDW: the plan of its first layer alone (identity stencil)
    int device = -1;
    int ho = 0, wo = 0, cm = 0;
    int esize = 0;
    size_t x_elems = 0, m_elems = 0, y_elems = 0;
    int num_sms = 0, smem_optin = 0;

    // weights in the layouts the kernels read (all owned, device memory)
    float *w1t = nullptr;     // DW: [k*k][C] fp32; dense: [k*k*C][Cm] fp32   (SIMT)
    float *wpt = nullptr;     // [Cm][K] fp32                                  (SIMT)
    void *w1_raw = nullptr;   // storage dtype, the caller's layout
    void *wp_img = nullptr;   // tcgen05 B-operand image of wp (128B-swizzled, K-major)
    size_t wp_img_bytes = 0;
    void *w1_img = nullptr;   // tcgen05 B-operand images of dense conv1, one per tap
    size_t w1_img_bytes = 0;
    void *w1dw_img = nullptr; // DW taps for the tcgen05 DW stage: [k*k][C], storage dtype (f16 for INT8)
    void *w1dw_pad = nullptr; // the same taps as [k*k][Cp], Cp = C rounded up to 64, zero-padded
                              // (dwpw_fused_kernel); INT8 PW-only views point it at i8_idtap
    float *s1 = nullptr, *b1 = nullptr, *s2 = nullptr, *b2 = nullptr;
    // host copy of the second layer's biases (K <= 128), valid for the device array b2_host_of
    // points to; the DW->PW role kernel passes them as kernel parameters
    float b2_host[128] = {};
    const float *b2_host_of = nullptr;
    float b1_host[128] = {};          // the same for the first layer's biases (Cm <= 128)
    const float *b1_host_of = nullptr;
    // INT8: 1152 * (sum of each channel's taps), and the identity stencil (one f16 tap of 1,
    // scale 1, bias 0, offset 1152) through which the PW-only mode runs on the fused kernel
    float *q1 = nullptr;
    float *i8_one = nullptr, *i8_zero = nullptr, *i8_idq = nullptr;
    void *i8_idtap = nullptr;
    unsigned *d_err = nullptr;

    void *mid_buf = nullptr;  // FCM_MODE_UNFUSED intermediate (lazily allocated)
    size_t mid_bytes = 0;
    void *stage_in = nullptr, *stage_out = nullptr;  // fcm_run_host staging
    size_t stage_in_bytes = 0, stage_out_bytes = 0;
    // fcm_run_host pipelining: copy streams and per-chunk events (created on first use)
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    cudaStream_t compute = nullptr;   // fcm_run_host_async's kernels
    cudaEvent_t ev_start = nullptr;
    cudaEvent_t ev_in[8] = {}, ev_run[8] = {}, ev_out[8] = {};
    // the previous host call: chunks (0 = none, 1 = unsplit, on the caller's stream), mode and
    // output buffer, which order fcm_run_host_async's copies after it
    int host_prev_nch = 0, host_prev_mode = -1;
    const void *host_prev_out = nullptr;
    size_t host_prev_out_bytes = 0;
};

// thread-local last-error message (fcm_api.cu)
fcm_status fcm_fail(fcm_status st, const char *fmt, ...);

// Unique id of the calling thread's current CUDA context (never reused within a process), or
// 0 when there is none or the driver cannot say (fcm_api.cu).  Per-context caches compare it
// so that they are rebuilt after a device reset or on another device.
unsigned long long fcm_current_ctx_id();

// planner.cu
fcm_status fcm_validate_desc(const fcm_desc *d, int *ho, int *wo, int *cm);
fcm_status fcm_make_plan(const fcm_desc *d, int num_sms, int smem_per_block, fcm_plan_info *info,
                         TcPlan *tc);
int fcm_tc_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why);
fcm_status fcm_tc_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_per_block,
                       TcPlan *tc);
// tc_dwpw.cu: the depthwise -> pointwise plan on dwpw_kernel alone (variant 0), which also
// serves the layer-by-layer modes
fcm_status fcm_tc_plan_dwpw_roles(const fcm_desc *d, int ho, int wo, int cm, int num_sms,
                                  int smem_per_block, TcPlan *tc);
// tc_dwpw_fused.cu: the depthwise -> pointwise plan on dwpw_fused_kernel (variant 1), or an
// error status when that kernel does not take the shape or no tile fits
fcm_status fcm_fused_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_per_block,
                          TcPlan *tc);
cudaError_t launch_tc_fused(const fcm_handle *h, const void *x, void *y, cudaStream_t st);

// tc_b2b.cu: dense k x k -> 1x1 on tcgen05
int fcm_b2b_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why);
fcm_status fcm_b2b_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_per_block,
                        TcPlan *tc);
fcm_status fcm_b2b_prepare(fcm_handle *h, const void *w1_host, const void *wp_host);

// tc_dwpw.cu: INT8 parts of a handle (stencil offsets of a depthwise w1_host, or none when
// w1_host is NULL; the identity stencil and plan of the PW-only mode)
fcm_status fcm_i8_prepare(fcm_handle *h, const void *w1_host);
fcm_status fcm_i8_constants(fcm_handle *h, const void *taps_host, int n_id);
fcm_desc fcm_i8_pw_desc(const fcm_handle *h);

// tc_pwdw.cu: 1x1 -> depthwise (PWDW) on tcgen05 + CUDA cores
int fcm_pwdw_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why);
fcm_status fcm_pwdw_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_per_block,
                         TcPlan *tc);
fcm_status fcm_pwdw_prepare(fcm_handle *h, const void *w1_host, const void *wp_host);
cudaError_t launch_tc_pwdw(const fcm_handle *h, const void *x, void *y, cudaStream_t st);
cudaError_t launch_tc_pwdw_first(const fcm_handle *h, const void *x, void *m, cudaStream_t st);
cudaError_t launch_tc_pwdw_second(const fcm_handle *h, const void *m, void *y, cudaStream_t st);

// simt_kernels.cu
cudaError_t launch_pwdw_fused_simt(const fcm_handle *h, const void *x, void *y, cudaStream_t st);
cudaError_t launch_pwdw_first_simt(const fcm_handle *h, const void *x, void *m, cudaStream_t st);
cudaError_t launch_pwdw_second_simt(const fcm_handle *h, const void *m, void *y, cudaStream_t st);
cudaError_t launch_conv1_simt(const fcm_handle *h, const void *x, void *m, cudaStream_t st);
cudaError_t launch_pw_simt(const fcm_handle *h, const void *m, void *y, cudaStream_t st);
cudaError_t launch_fused_simt(const fcm_handle *h, const void *x, void *y, cudaStream_t st);

// tc_dwpw.cu (depthwise -> pointwise on tcgen05) and tc_b2b.cu (dense 3x3 -> 1x1)
cudaError_t launch_tc_dwpw(const fcm_handle *h, int mode, const void *in, void *out,
                           cudaStream_t st);
cudaError_t launch_tc_b2b(const fcm_handle *h, int mode, const void *in, void *out,
                          cudaStream_t st);
cudaError_t launch_tc_pw(const fcm_handle *h, const void *m, void *y, cudaStream_t st);
// Build the tcgen05 operand images of the weights (host copies in the caller's layouts).
fcm_status fcm_tc_prepare(fcm_handle *h, const void *w1_host, const void *wp_host);
