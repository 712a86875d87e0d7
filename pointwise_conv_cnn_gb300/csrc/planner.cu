// planner.cu -- descriptor validation and the tile planner (host only).
//
// The planner follows FusePlanner's idea ("Fusing Depthwise and Pointwise Convolutions for
// Efficient Inference on GPUs", section IV): enumerate the tile shapes that satisfy the
// constraints (the tiles fit on chip; at least as many output tiles as SMs, section IV-A),
// count the global-memory accesses of each with the cost models of Equations 1-3 and the DWPW
// estimator built like Equation 4 (section IV-B), and keep the cheapest.  On GB300 the halo
// re-reads of Eq. 1 are largely served by the 126 MB L2, so the planner reports both the
// paper's estimate and the DRAM floor (every tensor once) next to each other.
#include <limits.h>
#include <string.h>

#include "fcm_internal.h"

extern "C" {

static long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

long long fcm_model_overlap(long long channel_w, long long channel_h, long long tile_w,
                            long long tile_h, long long filter_w, long long filter_h,
                            long long strides) {
    if (tile_w <= 0 || tile_h <= 0) return -1;
    // a filter narrower than the stride leaves gaps between neighbouring windows: no element
    // is read twice, so the halo width is clamped at zero rather than going negative
    long long halo_w = filter_w > strides ? filter_w - strides : 0;
    long long halo_h = filter_h > strides ? filter_h - strides : 0;
    return (ceil_div_ll(channel_w, tile_w) - 1) * halo_w * channel_h +
           (ceil_div_ll(channel_h, tile_h) - 1) * halo_h * channel_w;
}

long long fcm_model_pw_gma(long long weights_sz, long long weights_tile_sz, long long ifms_sz,
                           long long ofms_sz, long long ofms_tile_sz) {
    if (weights_tile_sz <= 0 || ofms_tile_sz <= 0) return -1;
    return ceil_div_ll(weights_sz, weights_tile_sz) * ifms_sz + ofms_sz +
           ceil_div_ll(ofms_sz, ofms_tile_sz) * weights_sz;
}

long long fcm_model_dw_gma(long long ifms_d, long long overlap, long long ifms_sz,
                           long long ofms_sz, long long ofms_hw, long long ofms_tile_hw,
                           long long weights_sz) {
    if (ofms_tile_hw <= 0) return -1;
    return 2 * ifms_d * overlap + ifms_sz + ofms_sz + ceil_div_ll(ofms_hw, ofms_tile_hw) * weights_sz;
}

long long fcm_model_dwpw_gma(long long c, long long overlap, long long dw_ifms_sz,
                             long long pw_weights_sz, long long pw_weights_tile_sz,
                             long long pw_ofms_sz, long long ofms_hw, long long ofms_tile_hw,
                             long long dw_weights_sz) {
    if (pw_weights_tile_sz <= 0 || ofms_tile_hw <= 0) return -1;
    return (2 * c * overlap + dw_ifms_sz) * ceil_div_ll(pw_weights_sz, pw_weights_tile_sz) +
           pw_ofms_sz + ceil_div_ll(ofms_hw, ofms_tile_hw) * (dw_weights_sz + pw_weights_sz);
}

}  // extern "C"

static int out_extent(int in, int k, int s, int p) {
    if (k < 1 || s < 1 || p < 0 || in + 2 * p < k) return -1;
    return (in + 2 * p - k) / s + 1;
}

fcm_status fcm_validate_desc(const fcm_desc *d, int *ho, int *wo, int *cm) {
    if (!d) return fcm_fail(FCM_ERR_INVALID_ARG, "desc is NULL");
    if (d->n < 1 || d->h < 1 || d->w < 1 || d->c < 1 || d->k_out < 1)
        return fcm_fail(FCM_ERR_INVALID_ARG, "n, h, w, c and k_out must be >= 1");
    if (d->ksize < 1 || d->ksize > 7)
        return fcm_fail(FCM_ERR_UNSUPPORTED, "ksize %d outside 1..7", d->ksize);
    if (d->stride < 1 || d->stride > 2)
        return fcm_fail(FCM_ERR_UNSUPPORTED, "stride %d outside 1..2", d->stride);
    if (d->pad < 0 || d->pad >= d->ksize)
        return fcm_fail(FCM_ERR_INVALID_ARG, "pad %d must be in [0, ksize)", d->pad);
    if (d->conv1 != FCM_CONV1_DEPTHWISE && d->conv1 != FCM_CONV1_DENSE &&
        d->conv1 != FCM_CONV1_POINTWISE)
        return fcm_fail(FCM_ERR_INVALID_ARG, "conv1 kind %d", d->conv1);
    if (d->dtype < FCM_F32 || d->dtype > FCM_I8)
        return fcm_fail(FCM_ERR_INVALID_ARG, "dtype %d", d->dtype);
    if (d->act1 < FCM_ACT_NONE || d->act1 > FCM_ACT_RELU6 || d->act2 < FCM_ACT_NONE ||
        d->act2 > FCM_ACT_RELU6)
        return fcm_fail(FCM_ERR_INVALID_ARG, "activation code out of range");
    if (d->kernel < FCM_KERNEL_AUTO || d->kernel > FCM_KERNEL_TC_WORKERS)
        return fcm_fail(FCM_ERR_INVALID_ARG, "kernel preference %d", d->kernel);
    if (d->tile_h < 0 || d->tile_w < 0)
        return fcm_fail(FCM_ERR_INVALID_ARG, "negative tile override");
    int m = d->mid == 0 ? d->c : d->mid;
    if (d->conv1 == FCM_CONV1_DEPTHWISE && m != d->c)
        return fcm_fail(FCM_ERR_INVALID_ARG, "depthwise conv1 keeps the channel count (mid %d != c %d)",
                        d->mid, d->c);
    if (m < 1) return fcm_fail(FCM_ERR_INVALID_ARG, "mid channels %d", m);
    if (d->conv1 == FCM_CONV1_POINTWISE && d->k_out != m)
        return fcm_fail(FCM_ERR_INVALID_ARG,
                        "PWDW: the depthwise layer keeps the channel count (k_out %d != mid %d)",
                        d->k_out, m);
    int h_o = out_extent(d->h, d->ksize, d->stride, d->pad);
    int w_o = out_extent(d->w, d->ksize, d->stride, d->pad);
    if (h_o < 1 || w_o < 1) return fcm_fail(FCM_ERR_INVALID_ARG, "empty output");
    // every NHWC row must start on a 16-byte boundary for the vector paths
    int esize = fcm_dtype_bytes(d->dtype);
    if (((long long)d->c * esize) % 16 != 0 || ((long long)m * esize) % 16 != 0 ||
        ((long long)d->k_out * esize) % 16 != 0)
        return fcm_fail(FCM_ERR_ALIGNMENT,
                        "c, mid and k_out times the element size must be multiples of 16 bytes");
    // simple size guards (32-bit indices inside tiles, 64-bit across the batch)
    if ((long long)d->n * d->h * d->w * d->c > (1LL << 40))
        return fcm_fail(FCM_ERR_UNSUPPORTED, "input larger than 2^40 elements");
    if (m > 2048 || d->k_out > 4096)
        return fcm_fail(FCM_ERR_UNSUPPORTED, "mid channels <= 2048 and k_out <= 4096 supported");
    if (ho) *ho = h_o;
    if (wo) *wo = w_o;
    if (cm) *cm = m;
    return FCM_OK;
}

// Byte counts and the section IV cost models for an output tile of th x tw pixels.
static void fill_bytes(const fcm_desc *d, int ho, int wo, int cm, int th, int tw,
                       fcm_plan_info *info) {
    long long e = fcm_dtype_bytes(d->dtype);
    long long N = d->n, H = d->h, W = d->w, C = d->c, K = d->k_out, k = d->ksize;
    const bool pwdw = d->conv1 == FCM_CONV1_POINTWISE;
    long long x = N * H * W * C, y = N * ho * wo * K;
    long long mid = pwdw ? N * H * W * cm : N * ho * wo * cm;
    long long w1 = d->conv1 == FCM_CONV1_DENSE ? (long long)cm * k * k * C
                   : pwdw                      ? (long long)cm * C
                                               : C * k * k;
    long long wp = pwdw ? (long long)cm * k * k : K * cm;
    long long sb = 4 * (2LL * cm + 2LL * K);
    info->bytes_fused_min = (x + y + w1 + wp) * e + sb;
    info->bytes_unfused_min = info->bytes_fused_min + 2 * mid * e;
    long long s = d->stride;
    long long ov = fcm_model_overlap(W, H, (long long)tw * s, (long long)th * s, k, k, s);
    info->overlap_elems = ov;
    if (pwdw) {
        // PW (C -> Cm over H x W) then DW (Cm, k x k): Eq. 2 + Eq. 3 layer by layer, Eq. 4 fused
        // (the tile holds all Cm channels: weight tiles are whole)
        long long hw = H * W, ohw = (long long)ho * wo, thw = (long long)th * tw;
        long long lbl_pw = fcm_model_pw_gma(w1, w1, hw * C, hw * cm, thw * cm);
        long long lbl_dw = fcm_model_dw_gma(cm, ov, hw * cm, ohw * cm, ohw, thw, wp);
        long long fused = fcm_model_pwdw_gma(C, ov, hw * C, w1, w1, wp, wp, ohw * cm, thw * cm,
                                             ohw, thw);
        info->gma_lbl_model = (lbl_pw + lbl_dw) * N * e;
        info->gma_fused_model = fused * N * e;
        return;
    }
    long long ifm = H * W * C, ofm1 = (long long)ho * wo * cm, ofm = (long long)ho * wo * K;
    long long lbl_dw = fcm_model_dw_gma(C, ov, ifm, ofm1, (long long)ho * wo, (long long)th * tw, w1);
    long long lbl_pw = fcm_model_pw_gma(wp, wp, ofm1, ofm, (long long)th * tw * K);
    long long fused = fcm_model_dwpw_gma(C, ov, ifm, wp, wp, ofm, (long long)ho * wo,
                                         (long long)th * tw, w1);
    info->gma_lbl_model = (lbl_dw + lbl_pw) * N * e;
    info->gma_fused_model = fused * N * e;
}

fcm_status fcm_make_plan(const fcm_desc *d, int num_sms, int smem_per_block, fcm_plan_info *info,
                         TcPlan *tc) {
    int ho, wo, cm;
    fcm_status st = fcm_validate_desc(d, &ho, &wo, &cm);
    if (st != FCM_OK) return st;
    if (!info) return fcm_fail(FCM_ERR_INVALID_ARG, "info is NULL");
    if (num_sms < 1 || smem_per_block < 1024)
        return fcm_fail(FCM_ERR_INVALID_ARG, "num_sms / smem_per_block");
    memset(info, 0, sizeof(*info));
    info->ho = ho;
    info->wo = wo;
    info->cm = cm;
    TcPlan local;
    TcPlan *t = tc ? tc : &local;
    *t = TcPlan();

    const char *why = nullptr;
    bool want_tc = d->kernel != FCM_KERNEL_SIMT && d->dtype != FCM_F32;
    bool tc_ok = want_tc && fcm_tc_supported(d, ho, wo, cm, &why) &&
                 fcm_tc_plan(d, ho, wo, cm, num_sms, smem_per_block, t) == FCM_OK;
    if (d->kernel >= FCM_KERNEL_TC && !tc_ok)
        return fcm_fail(FCM_ERR_UNSUPPORTED, "tensor-core kernels requested but unavailable: %s",
                        why ? why : (d->dtype == FCM_F32 ? "fp32 runs on CUDA cores" : "no tile fits"));
    if (d->dtype == FCM_I8 && !tc_ok)   // INT8 has no CUDA-core kernels
        return fcm_fail(FCM_ERR_UNSUPPORTED, "INT8 needs the tensor-core kernels: %s",
                        why ? why : (d->kernel == FCM_KERNEL_SIMT ? "SIMT requested" : "no tile fits"));
    if (tc_ok) {
        info->kernel = FCM_KERNEL_TC;
        info->tile_h = t->tile_h;
        // the worker-warp kernel's tile pitch may exceed the image: report the pixels it covers
        info->tile_w = t->variant == 1 ? (t->tile_w < wo ? t->tile_w : wo) : t->tile_w;
        info->chunk_c = t->chunk_c;
        info->stages = t->stages;
        info->ctas = t->ctas;
        info->threads = t->threads;
        info->smem_bytes = t->smem_bytes;
        info->num_tiles = t->num_tiles;
        if (d->conv1 == FCM_CONV1_DEPTHWISE) info->tc_variant = t->variant == 1 ? 1 : 2;
    } else {
        // SIMT kernels: flattened tiles of 32 output pixels, all channels
        const int px = 32;
        long long P = (long long)d->n * ho * wo;
        long long smem = d->conv1 == FCM_CONV1_POINTWISE ? 0 : 4LL * px * cm;
        if (smem > smem_per_block)
            return fcm_fail(FCM_ERR_SMEM_BUDGET, "commBuffer of %lld bytes exceeds %d", smem,
                            smem_per_block);
        info->kernel = FCM_KERNEL_SIMT;
        info->tile_h = 1;
        info->tile_w = px < wo ? px : wo;
        info->chunk_c = cm;
        info->stages = 1;
        info->num_tiles = (P + px - 1) / px;
        info->ctas = (int)(info->num_tiles < (long long)num_sms * 8 ? info->num_tiles
                                                                     : (long long)num_sms * 8);
        info->threads = 256;
        info->smem_bytes = (int)smem;
    }
    fill_bytes(d, ho, wo, cm, info->tile_h, info->tile_w, info);
    return FCM_OK;
}
