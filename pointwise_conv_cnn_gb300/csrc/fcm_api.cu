// fcm_api.cu -- the C ABI: argument checks, handle lifetime, weight repacking, dispatch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include <mutex>
#include <vector>

#include "fcm_internal.h"

static thread_local char g_last_error[512] = "";

fcm_status fcm_fail(fcm_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

unsigned long long fcm_current_ctx_id() {
    typedef CUresult (*GetCurrentFn)(CUcontext *);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

static fcm_status cuda_fail(cudaError_t e, const char *what) {
    return fcm_fail(FCM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define FCM_CUDA(call)                                              \
    do {                                                            \
        cudaError_t e__ = (call);                                   \
        if (e__ != cudaSuccess) return cuda_fail(e__, #call);       \
    } while (0)

// storage -> float on the host (CUDA's own host-side conversions)
static float host_to_f(const void *base, size_t i, int dtype) {
    switch (dtype) {
    case FCM_F32: return static_cast<const float *>(base)[i];
    case FCM_F16: return __half2float(static_cast<const __half *>(base)[i]);
    case FCM_I8: return (float)static_cast<const signed char *>(base)[i];
    default: return __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]);
    }
}

template <typename T>
static fcm_status upload(T **dst, const T *src, size_t count) {
    FCM_CUDA(cudaMalloc(reinterpret_cast<void **>(dst), count * sizeof(T)));
    FCM_CUDA(cudaMemcpy(*dst, src, count * sizeof(T), cudaMemcpyHostToDevice));
    return FCM_OK;
}

static fcm_status fetch(std::vector<unsigned char> &dst, const void *src, size_t bytes,
                        const char *name) {
    if (!src) return fcm_fail(FCM_ERR_INVALID_ARG, "%s is NULL", name);
    dst.resize(bytes);
    cudaError_t e = cudaMemcpy(dst.data(), src, bytes, cudaMemcpyDefault);
    if (e != cudaSuccess) return cuda_fail(e, name);
    return FCM_OK;
}

static void free_handle(fcm_handle *h) {
    if (!h) return;
    for (int i = 0; i < 8; i++) {
        if (h->ev_in[i]) cudaEventDestroy(h->ev_in[i]);
        if (h->ev_run[i]) cudaEventDestroy(h->ev_run[i]);
        if (h->ev_out[i]) cudaEventDestroy(h->ev_out[i]);
    }
    if (h->ev_start) cudaEventDestroy(h->ev_start);
    if (h->copy_in) cudaStreamDestroy(h->copy_in);
    if (h->copy_out) cudaStreamDestroy(h->copy_out);
    if (h->compute) cudaStreamDestroy(h->compute);
    void *ptrs[] = {h->w1t, h->wpt, h->w1_raw, h->wp_img, h->w1_img, h->w1dw_img, h->w1dw_pad, h->s1, h->b1,
                    h->s2, h->b2, h->q1, h->i8_one, h->i8_zero, h->i8_idq, h->i8_idtap,
                    h->d_err, h->mid_buf, h->stage_in, h->stage_out};
    for (void *p : ptrs)
        if (p) cudaFree(p);
    delete h;
}

extern "C" {

const char *fcm_last_error(void) { return g_last_error; }

fcm_status fcm_tensor_bytes(const fcm_desc *desc, size_t *x_bytes, size_t *m_bytes,
                            size_t *y_bytes) {
    int ho, wo, cm;
    fcm_status st = fcm_validate_desc(desc, &ho, &wo, &cm);
    if (st != FCM_OK) return st;
    size_t e = (size_t)fcm_dtype_bytes(desc->dtype);
    if (x_bytes) *x_bytes = (size_t)desc->n * desc->h * desc->w * desc->c * e;
    const bool pwdw = desc->conv1 == FCM_CONV1_POINTWISE;   // m keeps the input's extent
    if (m_bytes) *m_bytes = (size_t)desc->n * (pwdw ? desc->h : ho) * (pwdw ? desc->w : wo) * cm * e;
    if (y_bytes) *y_bytes = (size_t)desc->n * ho * wo * desc->k_out * e;
    return FCM_OK;
}

fcm_status fcm_plan_desc(const fcm_desc *desc, int num_sms, int smem_per_block,
                         fcm_plan_info *info) {
    return fcm_make_plan(desc, num_sms, smem_per_block, info, nullptr);
}

fcm_status fcm_plan(const fcm_handle *h, fcm_plan_info *info) {
    if (!h || !info) return fcm_fail(FCM_ERR_INVALID_ARG, "handle or info is NULL");
    *info = h->plan;
    return FCM_OK;
}

fcm_status fcm_create(const fcm_desc *desc, const void *w1, const void *wp, const float *s1,
                      const float *b1, const float *s2, const float *b2, fcm_handle **out) {
    FcmNvtxRange nvtx("fcm_create");
    if (!out) return fcm_fail(FCM_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    int ho, wo, cm;
    fcm_status st = fcm_validate_desc(desc, &ho, &wo, &cm);
    if (st != FCM_OK) return st;

    int dev = 0, ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
        cudaGetLastError();
        return fcm_fail(FCM_ERR_NO_DEVICE, "no CUDA device");
    }
    FCM_CUDA(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    FCM_CUDA(cudaGetDeviceProperties(&prop, dev));
    if (prop.major != 10 || prop.minor != 3)
        return fcm_fail(FCM_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a",
                        dev, prop.major, prop.minor);

    fcm_handle *h = new fcm_handle();
    h->d = *desc;
    h->device = dev;
    h->ho = ho;
    h->wo = wo;
    h->cm = cm;
    h->esize = fcm_dtype_bytes(desc->dtype);
    h->num_sms = prop.multiProcessorCount;
    h->smem_optin = (int)prop.sharedMemPerBlockOptin;
    h->x_elems = (size_t)desc->n * desc->h * desc->w * desc->c;
    const bool pwdw = desc->conv1 == FCM_CONV1_POINTWISE;
    h->m_elems = pwdw ? (size_t)desc->n * desc->h * desc->w * cm : (size_t)desc->n * ho * wo * cm;
    h->y_elems = (size_t)desc->n * ho * wo * desc->k_out;

    st = fcm_make_plan(desc, h->num_sms, h->smem_optin, &h->plan, &h->tc);
    if (st != FCM_OK) {
        free_handle(h);
        return st;
    }

    const int C = desc->c, K = desc->k_out, k = desc->ksize, dt = desc->dtype;
    const bool dense = desc->conv1 == FCM_CONV1_DENSE;
    const size_t n_w1 = dense ? (size_t)cm * k * k * C : pwdw ? (size_t)cm * C : (size_t)C * k * k;
    const size_t n_wp = pwdw ? (size_t)cm * k * k : (size_t)K * cm;
    std::vector<unsigned char> hw1, hwp, hs1, hb1, hs2, hb2;
    if ((st = fetch(hw1, w1, n_w1 * h->esize, "w1")) != FCM_OK ||
        (st = fetch(hwp, wp, n_wp * h->esize, "wp")) != FCM_OK ||
        (st = fetch(hs1, s1, cm * 4, "s1")) != FCM_OK ||
        (st = fetch(hb1, b1, cm * 4, "b1")) != FCM_OK ||
        (st = fetch(hs2, s2, K * 4, "s2")) != FCM_OK ||
        (st = fetch(hb2, b2, K * 4, "b2")) != FCM_OK) {
        free_handle(h);
        return st;
    }

    // SIMT layouts: conv1 taps major ([k*k][C] for DW, [k*k*C][Cm] for dense), wp as [Cm][K];
    // PWDW: the 1x1 filters as [C][Cm] (the 1x1 kernel's layout), the depthwise taps [k*k][Cm]
    std::vector<float> w1t(n_w1), wpt(n_wp);
    if (pwdw) {
        for (int j = 0; j < cm; j++)
            for (int c = 0; c < C; c++)
                w1t[(size_t)c * cm + j] = host_to_f(hw1.data(), (size_t)j * C + c, dt);
        for (int j = 0; j < cm; j++)
            for (int t = 0; t < k * k; t++)
                wpt[(size_t)t * cm + j] = host_to_f(hwp.data(), (size_t)j * k * k + t, dt);
    } else if (dense) {
        for (int j = 0; j < cm; j++)
            for (int t = 0; t < k * k; t++)
                for (int c = 0; c < C; c++)
                    w1t[((size_t)t * C + c) * cm + j] = host_to_f(hw1.data(), ((size_t)j * k * k + t) * C + c, dt);
    } else {
        for (int c = 0; c < C; c++)
            for (int t = 0; t < k * k; t++)
                w1t[(size_t)t * C + c] = host_to_f(hw1.data(), (size_t)c * k * k + t, dt);
    }
    if (!pwdw)
        for (int kk = 0; kk < K; kk++)
            for (int c = 0; c < cm; c++)
                wpt[(size_t)c * K + kk] = host_to_f(hwp.data(), (size_t)kk * cm + c, dt);

    if ((st = upload(&h->w1t, w1t.data(), w1t.size())) != FCM_OK ||
        (st = upload(&h->wpt, wpt.data(), wpt.size())) != FCM_OK ||
        (st = upload(reinterpret_cast<unsigned char **>(&h->w1_raw), hw1.data(), hw1.size())) != FCM_OK ||
        (st = upload(&h->s1, reinterpret_cast<const float *>(hs1.data()), cm)) != FCM_OK ||
        (st = upload(&h->b1, reinterpret_cast<const float *>(hb1.data()), cm)) != FCM_OK ||
        (st = upload(&h->s2, reinterpret_cast<const float *>(hs2.data()), K)) != FCM_OK ||
        (st = upload(&h->b2, reinterpret_cast<const float *>(hb2.data()), K)) != FCM_OK) {
        free_handle(h);
        return st;
    }
    if (K <= 128) {
        memcpy(h->b2_host, hb2.data(), sizeof(float) * (size_t)K);
        h->b2_host_of = h->b2;
    }
    if (cm <= 128) {
        memcpy(h->b1_host, hb1.data(), sizeof(float) * (size_t)cm);
        h->b1_host_of = h->b1;
    }
    if (h->plan.kernel == FCM_KERNEL_TC) {
        st = fcm_tc_prepare(h, hw1.data(), hwp.data());
        if (st != FCM_OK) {
            free_handle(h);
            return st;
        }
    }
    // error word: [0] flags, [1] the first failed index check of a debug build
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&h->d_err), 2 * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, 2 * sizeof(unsigned));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "fcm_create");
    }
    *out = h;
    return FCM_OK;
}

static fcm_status check_ptr(const void *p, const char *name) {
    if (!p) return fcm_fail(FCM_ERR_INVALID_ARG, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
        return fcm_fail(FCM_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
    return FCM_OK;
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

static fcm_status run_one(fcm_handle *h, int mode, const void *in, void *out, cudaStream_t st) {
    const bool tc = h->plan.kernel == FCM_KERNEL_TC;
    const bool dense = h->d.conv1 == FCM_CONV1_DENSE;
    cudaError_t e = cudaSuccess;
    if (h->d.conv1 == FCM_CONV1_POINTWISE) {
        switch (mode) {
        case FCM_MODE_FUSED:
            e = tc ? launch_tc_pwdw(h, in, out, st) : launch_pwdw_fused_simt(h, in, out, st);
            break;
        case FCM_MODE_CONV1_ONLY:
            e = tc ? launch_tc_pwdw_first(h, in, out, st) : launch_pwdw_first_simt(h, in, out, st);
            break;
        case FCM_MODE_PW_ONLY:
            e = tc ? launch_tc_pwdw_second(h, in, out, st) : launch_pwdw_second_simt(h, in, out, st);
            break;
        default: return fcm_fail(FCM_ERR_INVALID_ARG, "mode %d", mode);
        }
        if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
        return FCM_OK;
    }
    switch (mode) {
    case FCM_MODE_FUSED:
        e = tc ? (dense ? launch_tc_b2b(h, mode, in, out, st) : launch_tc_dwpw(h, mode, in, out, st))
               : launch_fused_simt(h, in, out, st);
        break;
    case FCM_MODE_CONV1_ONLY:
        e = tc ? (dense ? launch_tc_b2b(h, mode, in, out, st) : launch_tc_dwpw(h, mode, in, out, st))
               : launch_conv1_simt(h, in, out, st);
        break;
    case FCM_MODE_PW_ONLY:
        e = tc ? launch_tc_pw(h, in, out, st) : launch_pw_simt(h, in, out, st);
        break;
    default: return fcm_fail(FCM_ERR_INVALID_ARG, "mode %d", mode);
    }
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return FCM_OK;
}

fcm_status fcm_run(fcm_handle *h, int mode, const void *in, void *out, void *stream) {
    FcmNvtxRange nvtx("fcm_run");
    if (!h) return fcm_fail(FCM_ERR_INVALID_ARG, "handle is NULL");
    fcm_status st;
    if ((st = check_ptr(in, "in")) != FCM_OK || (st = check_ptr(out, "out")) != FCM_OK) return st;
    if (mode < FCM_MODE_FUSED || mode > FCM_MODE_UNFUSED)
        return fcm_fail(FCM_ERR_INVALID_ARG, "mode %d", mode);
    size_t e = h->esize;
    size_t in_b = (mode == FCM_MODE_PW_ONLY ? h->m_elems : h->x_elems) * e;
    size_t out_b = (mode == FCM_MODE_CONV1_ONLY ? h->m_elems : h->y_elems) * e;
    if (overlaps(in, in_b, out, out_b))
        return fcm_fail(FCM_ERR_INVALID_ARG, "in and out overlap");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == FCM_MODE_UNFUSED) {
        if (!h->mid_buf) {
            cudaError_t ce = cudaMalloc(&h->mid_buf, h->m_elems * e);
            if (ce != cudaSuccess) {
                h->mid_buf = nullptr;
                return cuda_fail(ce, "intermediate buffer");
            }
            h->mid_bytes = h->m_elems * e;
        }
        if ((st = run_one(h, FCM_MODE_CONV1_ONLY, in, h->mid_buf, s)) != FCM_OK) return st;
        return run_one(h, FCM_MODE_PW_ONLY, h->mid_buf, out, s);
    }
    return run_one(h, mode, in, out, s);
}

// A handle restricted to images [n0, n0 + nc) of the batch: the same weights and plan, with the
// batch size and the tile counts of the sub-batch (callers offset the activation pointers).
static fcm_handle batch_view(const fcm_handle *h, int nc) {
    fcm_handle v = *h;
    const int n = h->d.n;
    v.d.n = nc;
    v.x_elems = h->x_elems / n * nc;
    v.m_elems = h->m_elems / n * nc;
    v.y_elems = h->y_elems / n * nc;
    for (TcPlan *p : {&v.tc, &v.tc2, &v.tc_lbl}) {
        if (p->num_tiles <= 0) continue;
        p->num_tiles = p->num_tiles / n * nc;
        p->ctas = (int)(p->num_tiles < h->num_sms ? p->num_tiles : h->num_sms);
    }
    v.plan.num_tiles = h->plan.num_tiles / n * nc;
    v.mid_buf = nullptr;
    return v;
}

// Chunks of a synchronous host call (as even as possible).  Each chunk costs host time (copies, events, a launch);
// fewer chunks lengthen the pipeline's fill and drain.  Measured per call: MobileNet layer
// 420 / 416 / 412 / 428 us and stride-2 layer 1365 / 1201 / 1237 / 1274 us with 8 / 6 / 4 / 3
// chunks.
static int host_chunks(const fcm_handle *h, int mode) {
    if (mode == FCM_MODE_UNFUSED || h->d.n < 2) return 1;
    return h->d.n < 6 ? h->d.n : 6;
}

// fcm_run_host and fcm_run_host_async.  `wait` = the synchronous entry point: the copies start
// after the work already queued on `stream`, and the call returns once it has completed.
// Otherwise the input copies are ordered only after this handle's previous host calls -- chunk
// by chunk when the previous call split the batch the same way, so that its output copies
// overlap this call's input copies -- and the call returns once the work is enqueued.
static fcm_status run_host_impl(fcm_handle *h, int mode, const void *host_in, void *host_out,
                                void *stream, bool wait) {
    if (!h) return fcm_fail(FCM_ERR_INVALID_ARG, "handle is NULL");
    if (!host_in || !host_out) return fcm_fail(FCM_ERR_INVALID_ARG, "host buffer is NULL");
    if (mode < FCM_MODE_FUSED || mode > FCM_MODE_UNFUSED)
        return fcm_fail(FCM_ERR_INVALID_ARG, "mode %d", mode);
    size_t e = h->esize;
    size_t in_b = (mode == FCM_MODE_PW_ONLY ? h->m_elems : h->x_elems) * e;
    size_t out_b = (mode == FCM_MODE_CONV1_ONLY ? h->m_elems : h->y_elems) * e;
    // (cudaFree waits for the device, so a staging buffer is never freed under a copy in flight)
    if (h->stage_in_bytes < in_b) {
        if (h->stage_in) cudaFree(h->stage_in);
        h->stage_in = nullptr;
        h->stage_in_bytes = 0;
        h->host_prev_nch = 0;
        FCM_CUDA(cudaMalloc(&h->stage_in, in_b));
        h->stage_in_bytes = in_b;
    }
    if (h->stage_out_bytes < out_b) {
        if (h->stage_out) cudaFree(h->stage_out);
        h->stage_out = nullptr;
        h->stage_out_bytes = 0;
        h->host_prev_nch = 0;
        FCM_CUDA(cudaMalloc(&h->stage_out, out_b));
        h->stage_out_bytes = out_b;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The asynchronous call splits the batch in two: consecutive calls overlap their copies
    // anyway, and fewer, larger copies cost less host time per call (MobileNet layer, calls
    // back to back: 0.374 / 0.337 / 0.320 ms a call with 8 / 4 / 2 chunks).
    const int nch = wait ? host_chunks(h, mode) : std::min(host_chunks(h, mode), 2);
    if (nch == 1) {
        // everything on `stream`; a previous chunked call ended with `stream` waiting for its
        // last output copy, so stream order covers the staging buffers
        FCM_CUDA(cudaMemcpyAsync(h->stage_in, host_in, in_b, cudaMemcpyHostToDevice, s));
        fcm_status st = fcm_run(h, mode, h->stage_in, h->stage_out, stream);
        if (st != FCM_OK) return st;
        FCM_CUDA(cudaMemcpyAsync(host_out, h->stage_out, out_b, cudaMemcpyDeviceToHost, s));
        h->host_prev_nch = 1;
        if (wait) FCM_CUDA(cudaStreamSynchronize(s));
        return FCM_OK;
    }
    // Pipelined over chunks of the batch: the input copy of chunk i+1 (copy_in stream), the
    // kernel of chunk i (the caller's stream) and the output copy of chunk i-1 (copy_out
    // stream) overlap; events order each chunk's copy -> kernel -> copy.
    if (!h->copy_in) {
        FCM_CUDA(cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking));
        FCM_CUDA(cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking));
        FCM_CUDA(cudaStreamCreateWithFlags(&h->compute, cudaStreamNonBlocking));
        FCM_CUDA(cudaEventCreateWithFlags(&h->ev_start, cudaEventDisableTiming));
        for (int i = 0; i < 8; i++) {
            FCM_CUDA(cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming));
            FCM_CUDA(cudaEventCreateWithFlags(&h->ev_run[i], cudaEventDisableTiming));
            FCM_CUDA(cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming));
        }
    }
    const int prev = h->host_prev_nch;
    const bool same_split = prev == nch && h->host_prev_mode == mode;
    // the previous call's output copies may still be writing host memory this call reads
    const char *prev_lo = static_cast<const char *>(h->host_prev_out);
    const char *in_lo = static_cast<const char *>(host_in);
    const bool in_overlaps_prev_out = prev > 1 && prev_lo && in_lo < prev_lo + h->host_prev_out_bytes &&
                                      prev_lo < in_lo + in_b;
    // The synchronous call runs its kernels on the caller's stream, after the work queued there.
    // The asynchronous call runs them on the handle's compute stream, ordered chunk by chunk
    // after the previous call's kernels and copies, so that the caller's stream only waits for
    // the end of this call's copies out and the next call is not held up by it.
    cudaStream_t ks = wait ? s : h->compute;
    if (wait || prev == 1) {
        // after the work already queued on the caller's stream (for the asynchronous call: the
        // previous call ran its staging copies there)
        FCM_CUDA(cudaEventRecord(h->ev_start, s));
        FCM_CUDA(cudaStreamWaitEvent(h->copy_in, h->ev_start, 0));
        if (!wait) FCM_CUDA(cudaStreamWaitEvent(ks, h->ev_start, 0));
    } else if (prev > 1 && !same_split) {
        FCM_CUDA(cudaStreamWaitEvent(h->copy_in, h->ev_run[prev - 1], 0));   // all its kernels
        FCM_CUDA(cudaStreamWaitEvent(ks, h->ev_out[prev - 1], 0));           // all its copies out
    }
    if (!wait && in_overlaps_prev_out)
        FCM_CUDA(cudaStreamWaitEvent(h->copy_in, h->ev_out[prev - 1], 0));   // all its copies out
    const int n = h->d.n;
    const size_t in_img = in_b / n, out_img = out_b / n;
    int n0 = 0;
    for (int i = 0; i < nch; i++) {
        const int nc = n / nch + (i < n % nch ? 1 : 0);
        const char *hin = static_cast<const char *>(host_in) + (size_t)n0 * in_img;
        char *hout = static_cast<char *>(host_out) + (size_t)n0 * out_img;
        char *din = static_cast<char *>(h->stage_in) + (size_t)n0 * in_img;
        char *dout = static_cast<char *>(h->stage_out) + (size_t)n0 * out_img;
        if (!wait && same_split) {
            // staging chunk i: its input is free once the previous call's kernel i has read it,
            // its output once the previous call's copy out i is done (both waits are issued
            // before this call records those events again)
            FCM_CUDA(cudaStreamWaitEvent(h->copy_in, h->ev_run[i], 0));
            FCM_CUDA(cudaStreamWaitEvent(ks, h->ev_out[i], 0));
        }
        FCM_CUDA(cudaMemcpyAsync(din, hin, (size_t)nc * in_img, cudaMemcpyHostToDevice, h->copy_in));
        FCM_CUDA(cudaEventRecord(h->ev_in[i], h->copy_in));
        FCM_CUDA(cudaStreamWaitEvent(ks, h->ev_in[i], 0));
        fcm_handle v = batch_view(h, nc);
        fcm_status st = run_one(&v, mode, din, dout, ks);
        if (st != FCM_OK) return st;
        FCM_CUDA(cudaEventRecord(h->ev_run[i], ks));
        FCM_CUDA(cudaStreamWaitEvent(h->copy_out, h->ev_run[i], 0));
        FCM_CUDA(cudaMemcpyAsync(hout, dout, (size_t)nc * out_img, cudaMemcpyDeviceToHost, h->copy_out));
        FCM_CUDA(cudaEventRecord(h->ev_out[i], h->copy_out));
        n0 += nc;
    }
    // `stream` completes after the last output copy (copy_out runs its copies in order, each
    // after its chunk's kernel)
    FCM_CUDA(cudaStreamWaitEvent(s, h->ev_out[nch - 1], 0));
    h->host_prev_nch = nch;
    h->host_prev_mode = mode;
    h->host_prev_out = host_out;
    h->host_prev_out_bytes = out_b;
    if (wait) FCM_CUDA(cudaStreamSynchronize(s));
    return FCM_OK;
}

fcm_status fcm_run_host(fcm_handle *h, int mode, const void *host_in, void *host_out,
                        void *stream) {
    FcmNvtxRange nvtx("fcm_run_host");
    return run_host_impl(h, mode, host_in, host_out, stream, true);
}

fcm_status fcm_run_host_async(fcm_handle *h, int mode, const void *host_in, void *host_out,
                              void *stream) {
    FcmNvtxRange nvtx("fcm_run_host_async");
    return run_host_impl(h, mode, host_in, host_out, stream, false);
}

fcm_status fcm_check(fcm_handle *h, void *stream) {
    FcmNvtxRange nvtx("fcm_check");
    if (!h) return fcm_fail(FCM_ERR_INVALID_ARG, "handle is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FCM_CUDA(cudaStreamSynchronize(s));
    unsigned words[2] = {0, 0};
    FCM_CUDA(cudaMemcpy(words, h->d_err, sizeof(words), cudaMemcpyDeviceToHost));
    const unsigned word = words[0];
    if (word) FCM_CUDA(cudaMemset(h->d_err, 0, sizeof(words)));
    if (word & FCM_DEVERR_TIMEOUT)
        return fcm_fail(FCM_ERR_TIMEOUT, "a kernel's bounded wait ran out (error word 0x%x)", word);
    if (word)
        return fcm_fail(FCM_ERR_DEVICE_FAULT,
                        "a kernel's consistency check failed (error word 0x%x; first index check "
                        "%u at index %u)",
                        word, words[1] >> 24, words[1] & 0xFFFFFFu);
    return FCM_OK;
}

void fcm_destroy(fcm_handle *h) {
    if (!h) return;
    // the handle's own streams (fcm_run_host's copies); the caller's streams are the caller's
    if (h->copy_in) cudaStreamSynchronize(h->copy_in);
    if (h->copy_out) cudaStreamSynchronize(h->copy_out);
    if (h->compute) cudaStreamSynchronize(h->compute);
    free_handle(h);
}

}  // extern "C"
