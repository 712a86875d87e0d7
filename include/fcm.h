/*
 * fcm.h -- C ABI of the fused convolutional module (FCM) library for GB300 (sm_103a).
 *
 * One call runs a block-resident fused pair of convolutions on NHWC activations:
 *
 *     m = act1(s1 * conv1(x) + b1)          conv1: depthwise k x k, or dense k x k
 *     y = act2(s2 * (m . wp^T) + b2)        1x1 pointwise convolution
 *
 * or, for the PWDW module (FCM_CONV1_POINTWISE, an inverted residual's expansion and
 * depthwise layers; the paper's PWDW_R, section II-D, Figure 3(b)):
 *
 *     m = act1(s1 * (x . w1^T) + b1)        1x1 pointwise convolution C -> Cm
 *     y = act2(s2 * dw(m) + b2)             depthwise k x k over m (m zero-padded)
 *
 * where the intermediate m never leaves the thread block (shared memory / tensor memory);
 * in the PWDW case every tile recomputes the intermediate under its depthwise halo.
 * Definitions: "Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs",
 * section II-B (DW and PW convolutions), section II-D (the DWPW tile must hold all channels),
 * section III (FCMs: up to six fused layers -- two convolutions, each followed by its
 * normalization and activation -- with the intermediate kept in a shared "commBuffer"), and
 * section IV (FusePlanner cost models, Equations 1-4).  The dense case follows "Fusing two
 * back-to-back convolutions" (CUTLASS discussion #208): the second convolution must be 1x1 so
 * that a block never needs another block's intermediate.
 *
 * Conventions for every entry point:
 *  - A handle may be used from one host thread at a time (fcm_run_host and the first
 *    FCM_MODE_UNFUSED run keep per-handle buffers and streams); different handles are
 *    independent.
 *  - Status codes only: no exception, abort or exit crosses the ABI.  A human-readable
 *    message for the last failure on the calling thread is returned by fcm_last_error().
 *  - Activations are NHWC, contiguous, of the handle's dtype, 16-byte aligned, in device
 *    memory owned by the caller (except fcm_run_host, which takes host memory).
 *  - Scales and biases are float32.  Weights are of the handle's dtype.
 *  - Arithmetic: products and sums in fp32 (fp16/bf16 storage widened exactly); the
 *    intermediate is rounded to the storage dtype (round to nearest even) before the second
 *    convolution consumes it; the output is rounded to the storage dtype.  INT8: exact
 *    integer sums, then the requantization described at fcm_dtype.
 *  - Zero padding, cross-correlation (no filter flip):
 *    Ho = (H + 2*pad - ksize) / stride + 1, likewise Wo.
 */
#ifndef FCM_H
#define FCM_H

#include <stddef.h>

#if defined(__GNUC__)
#define FCM_API __attribute__((visibility("default")))
#else
#define FCM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fcm_status {
    FCM_OK = 0,
    FCM_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, bad enum value */
    FCM_ERR_UNSUPPORTED = 2,   /* valid request this library does not implement */
    FCM_ERR_ALIGNMENT = 3,     /* activation pointer not 16-byte aligned */
    FCM_ERR_SMEM_BUDGET = 4,   /* no tile fits in shared memory */
    FCM_ERR_CUDA = 5,          /* a CUDA runtime call failed (message has the CUDA error) */
    FCM_ERR_TIMEOUT = 6,       /* a kernel's bounded wait ran out (reported by fcm_check) */
    FCM_ERR_DEVICE_FAULT = 7,  /* a kernel's own consistency check failed (fcm_check) */
    FCM_ERR_NO_DEVICE = 8      /* no CUDA device, or not a compute capability 10.3 device */
} fcm_status;

/* Storage types.  FCM_I8 is the INT8 module of the paper's section III-B (int8 feature maps
 * and weights, 32-bit integer accumulation, int8 intermediate): every activation, weight and
 * the intermediate are int8; scales and biases stay float32 and requantize each accumulator,
 *     q = clamp(rint(act(fmaf(s, (float)acc, b))), -128, 127)      (rint: ties to even),
 * the fma and the rounding in fp32 (|acc| < 2^24 for every supported shape, so acc converts
 * exactly).  INT8 runs on the tensor-core kernels: the depthwise module (FCM_CONV1_DEPTHWISE;
 * C <= 256 and K multiples of 16, K <= 256, ksize 1/3/5/7) and the PWPW module
 * (FCM_CONV1_DENSE with ksize 1, pad 0: two 1x1 convolutions; C a multiple of 64, mid + k_out
 * <= 256, and the tile's int8 and f16 input rings must fit in shared memory next to the
 * weights, which holds up to C = 128); other INT8 requests return FCM_ERR_UNSUPPORTED.  The results are exact: the same integers on every run and in every
 * mode. */
typedef enum fcm_dtype { FCM_F32 = 0, FCM_F16 = 1, FCM_BF16 = 2, FCM_I8 = 3 } fcm_dtype;
typedef enum fcm_act { FCM_ACT_NONE = 0, FCM_ACT_RELU = 1, FCM_ACT_RELU6 = 2 } fcm_act;
/* The module's layer pair.  DEPTHWISE and DENSE: a k x k first convolution, then 1x1.
 * POINTWISE (PWDW): a 1x1 first convolution C -> Cm (Cm = mid, or C when mid is 0), then a
 * depthwise k x k convolution over the Cm channels; k_out must equal Cm. */
typedef enum fcm_conv1_kind {
    FCM_CONV1_DEPTHWISE = 0,
    FCM_CONV1_DENSE = 1,
    FCM_CONV1_POINTWISE = 2
} fcm_conv1_kind;

/* What fcm_run computes.  The three non-fused modes are the layer-by-layer (LBL) baselines of
 * the paper's section V-C, built from the same building blocks as the fused kernels.  For
 * FCM_CONV1_POINTWISE, "CONV1" is the 1x1 convolution (m is [N,H,W,Cm], the input's extent)
 * and "PW_ONLY" runs the second convolution, the depthwise one, on m. */
typedef enum fcm_mode {
    FCM_MODE_FUSED = 0,       /* in = x [N,H,W,C]    -> out = y [N,Ho,Wo,K]                 */
    FCM_MODE_CONV1_ONLY = 1,  /* in = x [N,H,W,C]    -> out = m [N,Ho,Wo,Cm] (storage dtype) */
    FCM_MODE_PW_ONLY = 2,     /* in = m [N,Ho,Wo,Cm] -> out = y [N,Ho,Wo,K]                 */
    FCM_MODE_UNFUSED = 3      /* CONV1_ONLY then PW_ONLY through an intermediate buffer the
                                 handle allocates on first use and owns                     */
} fcm_mode;

/* Kernel family request.  AUTO picks the tensor-core (tcgen05) kernels whenever the shape
 * is supported by them, else the CUDA-core (SIMT) kernels.  fp32 always runs SIMT.
 * The depthwise module has two tensor-core kernels for its fused mode: one with dedicated warp
 * roles (loader, MMA issuer, epilogue warps, stencil warps) and one whose worker warps each run
 * the stencil and a share of the 1x1's epilogue.  TC and AUTO take the worker-warp kernel for
 * 5x5 and 7x7 filters when the shape fits it (C <= 256, 16 <= K <= 256), where it measured
 * faster, else the role kernel; TC_ROLES and TC_WORKERS ask for one of them (TC_WORKERS fails
 * with FCM_ERR_UNSUPPORTED where the worker kernel does not take the shape).  Other module
 * kinds treat both as TC. */
typedef enum fcm_kernel_pref {
    FCM_KERNEL_AUTO = 0,
    FCM_KERNEL_SIMT = 1,
    FCM_KERNEL_TC = 2,
    FCM_KERNEL_TC_ROLES = 3,
    FCM_KERNEL_TC_WORKERS = 4
} fcm_kernel_pref;

typedef struct fcm_desc {
    int n, h, w, c;        /* input feature maps, NHWC                                     */
    int k_out;             /* 1x1 convolution output channels K                             */
    int mid;               /* first convolution's output channels Cm (0 = C); 0 or C for DW */
    int ksize, stride, pad;/* the k x k convolution's filter size, stride, zero padding     */
    int conv1;             /* fcm_conv1_kind                                                */
    int dtype;             /* fcm_dtype of activations and weights                          */
    int act1, act2;        /* fcm_act after conv1 and after the 1x1 convolution             */
    int tile_h, tile_w;    /* output tile override (0 = the planner chooses)                */
    int kernel;            /* fcm_kernel_pref                                               */
} fcm_desc;

/* What the tile planner chose, and the byte counts it compared (section IV). */
typedef struct fcm_plan_info {
    int ho, wo, cm;
    int kernel;                  /* 1 = SIMT kernels, 2 = tcgen05 kernels                     */
    int tile_h, tile_w;          /* output tile (pixels), all channels (section II-D rule)    */
    int chunk_c;                 /* conv1 channels per pipeline stage                         */
    int stages;                  /* input pipeline depth                                      */
    int ctas;                    /* persistent grid size                                      */
    int threads;                 /* threads per CTA                                           */
    int smem_bytes;              /* dynamic shared memory per CTA                             */
    long long num_tiles;         /* output tiles over the whole batch                         */
    long long bytes_fused_min;   /* input + weights + scale/bias + output, each once          */
    long long bytes_unfused_min; /* the above + one write and one read of the intermediate    */
    long long gma_fused_model;   /* DWPW estimator built from Eq. 1-3 (PWDW: Eq. 4), bytes,
                                    whole batch                                               */
    long long gma_lbl_model;     /* Eq. 3 (DW) + Eq. 2 (PW), bytes, whole batch               */
    long long overlap_elems;     /* Eq. 1 for the chosen tile, elements per channel per image */
    int tc_variant;              /* depthwise module on tcgen05: 1 = worker-warp kernel (each
                                    warp runs the stencil and its share of the 1x1's epilogue;
                                    channels in chunks of 64, the last one zero-padded),
                                    2 = dedicated warp roles; 0 otherwise                     */
} fcm_plan_info;

typedef struct fcm_handle fcm_handle;

/* Create a module.  w1: DW filters [C][k][k] or dense filters [Cm][k][k][C]; wp: 1x1 filters
 * [K][Cm]; s1,b1: [Cm]; s2,b2: [K].  PWDW (FCM_CONV1_POINTWISE): w1 is the 1x1 filters
 * [Cm][C] and wp the depthwise filters [Cm][k][k]; s2,b2: [Cm].  Each pointer may be host or device memory (unified
 * addressing decides); the handle copies and repacks everything into device memory it owns,
 * so the caller may free its copies on return.  Rejects (FCM_ERR_UNSUPPORTED) a second
 * convolution that is not 1x1 by construction: there is no parameter for it.  Uses the
 * current CUDA device; every later call on the handle must run with that device current.
 * On failure *out is set to NULL. */
FCM_API fcm_status fcm_create(const fcm_desc *desc, const void *w1, const void *wp,
                      const float *s1, const float *b1, const float *s2, const float *b2,
                      fcm_handle **out);

/* Enqueue one evaluation on `stream` (a cudaStream_t; NULL = legacy default stream).
 * `in`/`out` are caller-owned device pointers as described by fcm_mode; they must not
 * overlap.  Asynchronous: returns after the launch; launch errors are reported here, errors
 * found by the kernel itself are reported by fcm_check.
 * The tensor-core kernels are launched with programmatic stream serialization allowed: one may
 * start while the previous kernel on the stream is finishing, so that its set-up overlaps that
 * kernel's tail, but it reads `in` and writes `out` only once that kernel has completed and its
 * writes are visible -- stream order holds as for any launch.  Once its set-up is done it lets
 * the next kernel on the stream start launching (griddepcontrol.launch_dependents); a kernel of
 * the caller's that is launched with programmatic serialization allowed must therefore wait
 * (cudaGridDependencySynchronize) before it reads `out`, as programmatic dependent launch requires of any dependent. */
FCM_API fcm_status fcm_run(fcm_handle *h, int mode, const void *in, void *out, void *stream);

/* End-to-end variant of fcm_run on HOST buffers: copies `host_in` to a device staging buffer
 * owned by the handle (allocated on first use), runs `mode`, copies the result to `host_out`
 * and synchronizes `stream` before returning.  For batches of two or more images (all modes
 * but FCM_MODE_UNFUSED) the batch is split into up to 6 chunks whose input copies, kernels (on
 * `stream`) and output copies overlap, using two copy streams the handle creates on first
 * use.  Pinned host memory makes the copies faster and lets them overlap; pageable memory
 * also works. */
FCM_API fcm_status fcm_run_host(fcm_handle *h, int mode, const void *host_in, void *host_out,
                        void *stream);

/* fcm_run_host without the wait: enqueues the same copies and kernels and returns.  The result
 * is in `host_out` once `stream` has completed the work enqueued so far (cudaStreamSynchronize,
 * or an event recorded on `stream` after the call).  Until then `host_in` must not change and
 * `host_out` must not be read.  The input copies are ordered after this handle's previous host
 * calls (chunk by chunk when the batch is split the same way, so that one call's output copies
 * overlap the next call's input copies, and after all of the previous call's output copies when
 * `host_in` overlaps its `host_out`), but not after other work on `stream`: the caller orders
 * the producers of `host_in` itself.  Consecutive calls on one handle may therefore be in
 * flight together; they must come from one host thread.  Pinned host memory is required for
 * the copies to overlap.  The batch is split into two chunks (not six): calls in flight
 * together overlap their copies anyway, and fewer copies cost less host time per call. */
FCM_API fcm_status fcm_run_host_async(fcm_handle *h, int mode, const void *host_in,
                                      void *host_out, void *stream);

/* Layer-by-layer evaluation that allocates nothing: the same result as fcm_run with
 * FCM_MODE_UNFUSED, but the intermediate is kept in a fixed 16 MiB device array compiled into
 * the library instead of a buffer the handle allocates on first use.  The paper has no
 * counterpart; it exists for callers that cannot call cudaMalloc while they run -- a serving
 * loop whose memory is budgeted up front, a host thread that must not take the allocator's
 * locks or trigger its implicit synchronisation, a process whose device memory belongs to
 * another allocator.  `in`/`out` as for FCM_MODE_UNFUSED (caller-owned device memory).
 *  - Rejects (FCM_ERR_UNSUPPORTED) an intermediate N*Ho*Wo*Cm*element-size above 16 MiB.
 *  - The array exists once per device that loads the library and is kept until exit.
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress),
 *    and so does the first call after the device's context changed (cudaDeviceReset);
 *    make those calls before any stream capture.  The current device must be the handle's
 *    device.
 *  - Every call uses the same array and leaves its intermediate there; each call rewrites all
 *    of it before reading it.  Calls that overlap on the GPU (other streams, other handles,
 *    other threads) race on it: serialise them. */
FCM_API fcm_status fcm_run_unfused_static(fcm_handle *h, const void *in, void *out, void *stream);

/* Synchronize `stream`, then read and clear the handle's device error word.  Returns
 * FCM_ERR_TIMEOUT if a bounded wait in a kernel ran out, FCM_ERR_DEVICE_FAULT if a kernel's
 * own check failed, FCM_OK otherwise. */
FCM_API fcm_status fcm_check(fcm_handle *h, void *stream);

/* Self-test of the kernels' failure detection on the current device: one kernel waits, through
 * the bounded wait every tensor-core kernel uses, on an mbarrier phase that nothing completes.
 * After `limit_ns` (in (0, 10 s]) the wait gives up, sets a device error word and the kernel
 * returns, leaving the context usable.  Returns FCM_ERR_TIMEOUT when that happened as designed
 * (the expected result), FCM_ERR_DEVICE_FAULT if the wait did not report it, FCM_ERR_CUDA on a
 * CUDA failure, FCM_ERR_INVALID_ARG for a limit out of range.  Synchronizes the device. */
FCM_API fcm_status fcm_selftest_wait_timeout(unsigned long long limit_ns);

/* The plan of an existing handle. */
FCM_API fcm_status fcm_plan(const fcm_handle *h, fcm_plan_info *info);

/* Run the tile planner for a descriptor without a GPU: `num_sms` and `smem_per_block` (bytes
 * of opt-in dynamic shared memory per CTA) describe the target (152 and 232448 on GB300). */
FCM_API fcm_status fcm_plan_desc(const fcm_desc *desc, int num_sms, int smem_per_block,
                         fcm_plan_info *info);

/* Size in bytes of each tensor of a descriptor: x, m (intermediate), y. */
FCM_API fcm_status fcm_tensor_bytes(const fcm_desc *desc, size_t *x_bytes, size_t *m_bytes,
                            size_t *y_bytes);

/* Free the handle and everything it owns.  NULL is ignored.  The caller must first make sure
 * that the work it enqueued with the handle has finished (synchronize the streams it passed to
 * fcm_run / fcm_run_unfused_static): fcm_destroy waits only for the handle's own copy streams
 * (fcm_run_host), not for the device, so that other streams of the process are not stalled. */
FCM_API void fcm_destroy(fcm_handle *h);

/* Message of the last failing call on this thread ("" if none).  Valid until the next call. */
FCM_API const char *fcm_last_error(void);

/* ---- FusePlanner cost models, section IV (element counts per image; exported for tests). */
/* Eq. 1: halo elements per channel re-read across tiles.  A filter narrower than the stride
 * (windows that do not overlap) counts 0 halo columns/rows, not a negative number.  Returns -1
 * for a tile extent <= 0. */
FCM_API long long fcm_model_overlap(long long channel_w, long long channel_h, long long tile_w,
                            long long tile_h, long long filter_w, long long filter_h,
                            long long strides);
/* Eq. 2: PW layer-by-layer global memory accesses. */
FCM_API long long fcm_model_pw_gma(long long weights_sz, long long weights_tile_sz, long long ifms_sz,
                           long long ofms_sz, long long ofms_tile_sz);
/* Eq. 3: DW layer-by-layer global memory accesses. */
FCM_API long long fcm_model_dw_gma(long long ifms_d, long long overlap, long long ifms_sz,
                           long long ofms_sz, long long ofms_hw, long long ofms_tile_hw,
                           long long weights_sz);
/* DWPW FCM estimator, built from Eq. 2 and 3 the way section IV-B builds Eq. 4:
 * (2*C*Overlap + DwIFMsSz) * ceil(PwWeightsSz/PwWeightsTileSz) + PwOFMsSz
 *   + ceil(OFMsHW/OFMsTileHW) * (DwWeightsSz + PwWeightsSz). */
FCM_API long long fcm_model_dwpw_gma(long long c, long long overlap, long long dw_ifms_sz,
                             long long pw_weights_sz, long long pw_weights_tile_sz,
                             long long pw_ofms_sz, long long ofms_hw, long long ofms_tile_hw,
                             long long dw_weights_sz);

/* Eq. 4: PWDW FCM global memory accesses, as printed. */
FCM_API long long fcm_model_pwdw_gma(long long pw_ifms_d, long long dw_overlap, long long pw_ifms_sz,
                             long long pw_weights_sz, long long pw_weights_tile_sz,
                             long long dw_weights_sz, long long dw_weights_tile_sz,
                             long long dw_ofms_sz, long long dw_ofms_tile_sz, long long dw_ofms_hw,
                             long long dw_ofms_tile_hw);
/* PWPW FCM estimator, built from Eq. 2 the way section IV-B builds Eq. 4 (the first layer's
 * input is re-read once per weight tile of the second layer, which recomputes the
 * intermediate; the second layer's output is written once; both layers' weights are read once
 * per spatial tile):
 * Pw1IFMsSz * ceil(Pw2WeightsSz/Pw2WeightsTileSz) + Pw2OFMsSz
 *   + ceil(OFMsHW/OFMsTileHW) * (Pw1WeightsSz + Pw2WeightsSz). */
FCM_API long long fcm_model_pwpw_gma(long long pw1_ifms_sz, long long pw1_weights_sz,
                             long long pw2_weights_sz, long long pw2_weights_tile_sz,
                             long long pw2_ofms_sz, long long ofms_hw, long long ofms_tile_hw);

/* ---- FusePlanner over a chain of layers, section IV ("FusePlanner overview", IV-A, IV-B).
 * The i-th layer's input is the (i-1)-th layer's output (H, W, C checked).  Each layer's
 * minimum layer-by-layer estimate (Eq. 3 for DW, Eq. 2 for PW) and each adjacent pair's
 * minimum FCM estimate (DWPW: fcm_model_dwpw_gma; PWDW: Eq. 4; PWPW: fcm_model_pwpw_gma) are
 * searched over the tiles that fit in L1 (three tiles for a layer, five for an FCM) and give
 * at least `num_sms` output tiles over a batch of `batch` images, tile sizes being multiples of
 * the warp size (pixels per tile, channels per tile; a dimension below 32 is taken whole).
 * When no such tile reaches `num_sms` output tiles, those with the most tiles are taken and
 * `tiles_ok` / `fcm_tiles_ok` say so.  A pair is fused when its
 * FCM estimate is below the sum of its layers' estimates; where candidate pairs share a layer
 * the decomposition with the smallest chain total is chosen.  No counterpart for DW -> DW. */
typedef enum { FCM_LAYER_DW = 0, FCM_LAYER_PW = 1 } fcm_layer_kind;
typedef enum {
    FCM_MODULE_LBL_DW = 0,       /* this layer runs alone (depthwise) */
    FCM_MODULE_LBL_PW = 1,       /* this layer runs alone (pointwise) */
    FCM_MODULE_DWPW = 2,         /* this layer and the next form a DWPW FCM */
    FCM_MODULE_PWDW = 3,         /* ... a PWDW FCM */
    FCM_MODULE_PWPW = 4,         /* ... a PWPW FCM */
    FCM_MODULE_FUSED_SECOND = 5  /* second layer of the FCM chosen for the previous layer */
} fcm_module_kind;
typedef struct {
    int kind;           /* fcm_layer_kind */
    int h, w, c;        /* input extent and channels */
    int k_out;          /* PW: filters; DW: 0 or c */
    int ksize, stride, pad;   /* DW only (a PW layer is 1x1, stride 1, no padding) */
} fcm_layer;
typedef struct {
    int fuse_with_next; /* 1: this layer and the next run as one FCM */
    int module;         /* fcm_module_kind chosen for this layer */
    int fcm_module;     /* FCM kind this layer would form with the next (-1: none exists) */
    int tile_h, tile_w, tile_c;              /* best layer-by-layer OFM tile (pixels, channels) */
    int fcm_tile_h, fcm_tile_w, fcm_tile_c;  /* best FCM OFM tile with the next layer */
    int tiles_ok;       /* 1: the layer-by-layer tile gives >= num_sms output tiles */
    int fcm_tiles_ok;   /* same for the FCM tile */
    long long gma_lbl;  /* minimum layer-by-layer estimate, elements per image */
    long long gma_fcm;  /* minimum FCM estimate of this layer and the next, -1 if none */
} fcm_layer_plan;
/* `layers[n_layers]` (host memory, read only); `out[n_layers]` (host memory, written);
 * `total_gma` (optional) receives the chain total of the chosen decomposition.  `l1_bytes` is
 * the on-chip capacity the tiles must fit in, `elem_bytes` the element size.  Errors:
 * FCM_ERR_INVALID_ARG for bad or mismatched shapes, FCM_ERR_SMEM_BUDGET when a layer has no
 * admissible tile.  Host only, no GPU needed. */
FCM_API fcm_status fcm_fuse_plan(const fcm_layer *layers, int n_layers, int batch,
                                 int num_sms, long long l1_bytes, int elem_bytes,
                                 fcm_layer_plan *out, long long *total_gma);

#ifdef __cplusplus
}
#endif
#endif /* FCM_H */
