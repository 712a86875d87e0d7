// tc_dwpw.cu -- host side of the tensor-core depthwise -> pointwise kernels: the tile planner,
// the weight images and the launches.  The kernels themselves are in tc_dwpw_kernel.cuh,
// instantiated by tc_dwpw_inst_*.cu (several translation units, compiled in parallel).
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "tc_dwpw.cuh"

namespace fcm {
namespace tc {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

uint32_t pow2_cols(int k2) {
    uint32_t c = 32;
    while ((int)c < k2) c <<= 1;
    return c;
}

// Shared-memory layout of one mode for a plan.  Returns total bytes (incl. alignment slack).
struct Layout {
    uint32_t off_b, off_a, off_out, off_in, in_stage_bytes, in_stage_stride, off_wdw, off_sb,
        off_bar, total;
    int stages;
};

Layout make_layout(const fcm_desc *d, const TcPlan &p, int cm, int mode, int smem_cap,
                   int out_bufs) {
    Layout L{};
    const int C = cm, K = d->k_out, nkb = (C + 63) / 64;
    const int es = fcm_dtype_bytes(d->dtype);
    const bool i8 = d->dtype == FCM_I8;
    // the B image and the A tile are 16-bit for every storage type (INT8 as exact f16)
    const uint32_t b_bytes = mode == DWONLY ? 0u : (uint32_t)nkb * K * 128;
    const uint32_t a_bytes = mode == FUSED ? (uint32_t)nkb * kTileM * 128 : 0u;
    const uint32_t out_bytes =
        mode == DWONLY ? 0u : (uint32_t)(out_bufs * ((K + 63) / 64)) * (uint32_t)out_block_bytes(es);
    L.off_b = 0;
    L.off_a = align_up(b_bytes, 1024);
    L.off_out = align_up(L.off_a + a_bytes, 1024);
    L.off_in = align_up(L.off_out + out_bytes, 1024);
    if (mode == PWONLY)
        L.in_stage_bytes = (uint32_t)nkb * kTileM * 128;
    else
        L.in_stage_bytes = (uint32_t)p.in_rows * p.in_cols * p.chunk_c * es;
    L.in_stage_stride = align_up(L.in_stage_bytes, 1024);
    const uint32_t wdw = mode == PWONLY ? 0u : (uint32_t)C * d->ksize * d->ksize * 2;
    const uint32_t sb = (uint32_t)(2 * C + 2 * K + (i8 ? C : 0)) * 4;
    const uint32_t tail = align_up(wdw, 16) + align_up(sb, 16) + kBarBytes + 16 + 1024;
    int stages = mode == PWONLY ? 4 : p.stages;
    for (; stages >= 1; stages--) {
        uint32_t total = L.off_in + (uint32_t)stages * L.in_stage_stride + tail;
        if ((int)total <= smem_cap) break;
    }
    if (stages > kMaxStages) stages = kMaxStages;
    L.stages = stages;
    L.off_wdw = L.off_in + (uint32_t)std::max(stages, 0) * L.in_stage_stride;
    L.off_sb = L.off_wdw + align_up(wdw, 16);
    L.off_bar = L.off_sb + align_up(sb, 16);
    L.total = L.off_bar + kBarBytes + 16 + 1024;
    return L;
}

}  // namespace tc
}  // namespace fcm

using namespace fcm::tc;

extern "C" long long fcm_model_overlap(long long, long long, long long, long long, long long,
                                       long long, long long);
extern "C" long long fcm_model_dwpw_gma(long long, long long, long long, long long, long long,
                                        long long, long long, long long, long long);

int fcm_tc_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why) {
    auto no = [&](const char *w) {
        if (why) *why = w;
        return 0;
    };
    if (d->dtype == FCM_F32) return no("fp32 runs on CUDA cores");
    if (d->conv1 == FCM_CONV1_POINTWISE) return fcm_pwdw_supported(d, ho, wo, cm, why);
    if (d->conv1 != FCM_CONV1_DEPTHWISE) return fcm_b2b_supported(d, ho, wo, cm, why);
    if (cm % 16 != 0) return no("channels must be a multiple of 16");
    // INT8: the 1x1's fp32 partial sums stay below 256 * 128 * 128 = 2^22, exact on the tensor core
    if (d->dtype == FCM_I8 && cm > 256) return no("INT8 takes at most 256 channels");
    if (d->k_out % 16 != 0 || d->k_out < 16 || d->k_out > 256)
        return no("k_out must be a multiple of 16 in [16, 256]");
    if (d->ksize != 1 && d->ksize != 3 && d->ksize != 5 && d->ksize != 7)
        return no("ksize must be 1, 3, 5 or 7");
    (void)ho;
    (void)wo;
    return 1;
}

fcm_status fcm_tc_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_cap,
                       TcPlan *p) {
    if (d->conv1 == FCM_CONV1_DENSE) return fcm_b2b_plan(d, ho, wo, cm, num_sms, smem_cap, p);
    if (d->conv1 == FCM_CONV1_POINTWISE) return fcm_pwdw_plan(d, ho, wo, cm, num_sms, smem_cap, p);
    // the worker-warp kernel where it measured faster (5x5 and 7x7 filters: a long stencil per
    // unit), or on request; the role kernel otherwise
    if (d->kernel == FCM_KERNEL_TC_WORKERS)
        return fcm_fused_plan(d, ho, wo, cm, num_sms, smem_cap, p);
    if (d->kernel != FCM_KERNEL_TC_ROLES && d->ksize >= 5 &&
        fcm_fused_plan(d, ho, wo, cm, num_sms, smem_cap, p) == FCM_OK)
        return FCM_OK;
    return fcm_tc_plan_dwpw_roles(d, ho, wo, cm, num_sms, smem_cap, p);
}

// Tile search of dwpw_kernel, after FusePlanner (section IV): every candidate tile (rows x the
// width split evenly into tiles of at most 128 pixels) with a channel chunk that fits shared
// memory is scored by its work efficiency (useful output pixels over the MMA rows its tiles
// occupy); tiles within 3% of the best are admissible, and among them the planner takes the
// smallest global-memory-access estimate of the DWPW module (the Eq. 1-4 form the plan
// reports), then the best pipeline score (thread use of the DW warps, halo share, stages).
fcm_status fcm_tc_plan_dwpw_roles(const fcm_desc *d, int ho, int wo, int cm, int num_sms,
                                  int smem_cap, TcPlan *p) {
    const int S = d->stride, KS = d->ksize, C = cm;
    struct Cand {
        TcPlan t;
        double eff, score;
        long long gma;
    };
    std::vector<Cand> cands;
    double max_eff = 0.0;
    int tw_choices[2] = {0, 0};
    int ncol_tiles = (wo + kTileM - 1) / kTileM;
    tw_choices[0] = (wo + ncol_tiles - 1) / ncol_tiles;
    if (d->tile_w > 0) tw_choices[0] = std::min(d->tile_w, kTileM);
    for (int tw : tw_choices) {
        if (tw <= 0) continue;
        int ngroups = (tw + kR - 1) / kR;
        int in_cols = (ngroups * kR - 1) * S + KS;
        if (in_cols > 256) continue;
        int th_max = std::max(1, std::min(kTileM / tw, ho));
        for (int th = th_max; th >= 1; th--) {
            if (d->tile_h > 0 && th != d->tile_h) continue;
            int in_rows = (th - 1) * S + KS;
            if (in_rows > 256) continue;
            for (int chunk = std::min(C, 256); chunk >= 16; chunk -= 16) {
                if (C % chunk != 0 || C / chunk > kMaxChunks) continue;
                TcPlan t;
                t.tile_h = th;
                t.tile_w = tw;
                t.in_rows = in_rows;
                t.in_cols = in_cols;
                t.chunk_c = chunk;
                t.nchunks = C / chunk;
                t.stages = kMaxStages;
                // two output staging tiles when that still leaves three input stages
                Layout L = make_layout(d, t, cm, FUSED, smem_cap, 2);
                t.out_bufs = 2;
                if (L.stages < 3) {
                    L = make_layout(d, t, cm, FUSED, smem_cap, 1);
                    t.out_bufs = 1;
                }
                if (L.stages < 2) continue;
                t.stages = L.stages;
                t.smem_bytes = (int)L.total;
                t.tiles_w = (wo + tw - 1) / tw;
                t.tiles_h = (ho + th - 1) / th;
                t.num_tiles = (long long)d->n * t.tiles_w * t.tiles_h;
                // DW warps: best use of threads for this chunk's work units
                int units = th * ngroups * (chunk / 8);
                int best_w = 4;
                double best_eff = 0.0;
                for (int w = 4; w <= kMaxDwWarps; w++) {
                    int thr = 32 * w;
                    double eff = (double)units / ((double)((units + thr - 1) / thr) * thr);
                    if (eff > best_eff + 1e-9 || (eff > best_eff - 1e-9 && w > best_w)) {
                        best_eff = eff;
                        best_w = w;
                    }
                }
                t.threads = 32 * (kFirstDwWarp + best_w);
                t.dw_warps = best_w;
                t.dw_per_chunk = 0;
                // chunk-bound DW warps (taps in registers) when the taps fit (k <= 3), one unit
                // per thread, and at most kMaxDwWarpsBound warps
                const int wpc = (units + 31) / 32;
                if (KS <= 3 && wpc * t.nchunks <= kMaxDwWarpsBound) {
                    t.dw_per_chunk = wpc;
                    t.dw_warps = wpc * t.nchunks;
                    t.threads = 32 * (kFirstDwWarp + t.dw_warps);
                    best_eff = (double)units / (32.0 * wpc);
                }
                t.ctas = (int)std::min<long long>(t.num_tiles, num_sms);
                t.tmem_cols = (int)pow2_cols(2 * d->k_out);
                // pipeline score: thread efficiency x halo share x pipeline depth x occupancy
                double halo = (double)(th * tw * S * S) / (double)(in_rows * in_cols);
                double score = best_eff * (0.5 + 0.5 * halo) * (t.stages >= 3 ? 1.0 : 0.9) *
                               (t.num_tiles >= num_sms ? 1.0 : 0.5);
                const double eff = (double)ho * wo / ((double)t.tiles_w * t.tiles_h * kTileM);
                const long long ov = fcm_model_overlap(d->w, d->h, (long long)tw * S,
                                                       (long long)th * S, KS, KS, S);
                const long long gma = fcm_model_dwpw_gma(
                    C, ov, (long long)d->h * d->w * C, (long long)d->k_out * C,
                    (long long)d->k_out * C, (long long)ho * wo * d->k_out, (long long)ho * wo,
                    (long long)th * tw, (long long)C * KS * KS);
                cands.push_back(Cand{t, eff, score, gma});
                max_eff = std::max(max_eff, eff);
            }
        }
    }
    const Cand *pick = nullptr;
    for (const Cand &c : cands) {
        if (c.eff < 0.97 * max_eff) continue;
        if (!pick || c.gma < pick->gma || (c.gma == pick->gma && c.score > pick->score + 1e-12))
            pick = &c;
    }
    if (!pick) return FCM_ERR_SMEM_BUDGET;
    *p = pick->t;
    return FCM_OK;
}

// The PW-only mode of an INT8 handle: the fused DW->PW kernel with an identity stencil over the
// intermediate m [N, Ho, Wo, Cm].
fcm_desc fcm_i8_pw_desc(const fcm_handle *h) {
    fcm_desc v = h->d;
    v.conv1 = FCM_CONV1_DEPTHWISE;   // the identity stencil (also for the PWPW module's 2nd layer)
    v.h = h->ho;
    v.w = h->wo;
    v.c = h->cm;
    v.mid = 0;
    v.ksize = 1;
    v.stride = 1;
    v.pad = 0;
    v.act1 = FCM_ACT_NONE;
    v.tile_h = 0;
    v.tile_w = 0;
    return v;
}

// INT8 constants of a handle: the per-channel stencil offsets 1152 * sum(taps) of the h->cm
// channels of a depthwise layer (taps_host [cm][k][k], or none), and the identity stencil
// (one f16 tap of 1, scale 1, bias 0, offset 1152) over n_id channels, through which the fused
// DW->PW kernel runs a lone 1x1 convolution.
fcm_status fcm_i8_constants(fcm_handle *h, const void *taps_host, int n_id) {
    const int C = h->cm, KS = h->d.ksize;
    const int ni = std::max(n_id, C);
    std::vector<float> q1(C, 0.0f), one(ni, 1.0f), zero(ni, 0.0f), idq(ni, I8::kBias);
    const void *w1_host = taps_host;
    if (w1_host) {
        const signed char *w8 = static_cast<const signed char *>(w1_host);
        for (int c = 0; c < C; c++) {
            int sum = 0;
            for (int t = 0; t < KS * KS; t++) sum += w8[(size_t)c * KS * KS + t];
            q1[c] = I8::kBias * (float)sum;   // |sum| <= 49 * 128: exact
        }
    }
    const __half h1 = __float2half_rn(1.0f);
    // the identity taps, zero-padded to a multiple of 64 channels (the worker-warp kernel
    // reads [k*k][Cp] taps)
    const int cp = (ni + 63) / 64 * 64;
    std::vector<__half> idtap(cp, __float2half_rn(0.0f));
    for (int c = 0; c < ni; c++) idtap[c] = h1;
    const size_t fb = (size_t)C * sizeof(float), fbi = (size_t)ni * sizeof(float);
    if (cudaMalloc(&h->q1, fb) != cudaSuccess ||
        cudaMemcpy(h->q1, q1.data(), fb, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->i8_one, fbi) != cudaSuccess ||
        cudaMemcpy(h->i8_one, one.data(), fbi, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->i8_zero, fbi) != cudaSuccess ||
        cudaMemcpy(h->i8_zero, zero.data(), fbi, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->i8_idq, fbi) != cudaSuccess ||
        cudaMemcpy(h->i8_idq, idq.data(), fbi, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->i8_idtap, (size_t)cp * 2) != cudaSuccess ||
        cudaMemcpy(h->i8_idtap, idtap.data(), (size_t)cp * 2, cudaMemcpyHostToDevice) != cudaSuccess)
        return fcm_fail(FCM_ERR_CUDA, "INT8 stencil constants: %s",
                        cudaGetErrorString(cudaGetLastError()));
    return FCM_OK;
}

// INT8 handle parts of the depthwise and PWPW modules: the constants above (w1_host = the
// depthwise taps, or none) and the plan of the PW-only mode (the fused DW->PW kernel with
// k = 1 over the intermediate).
fcm_status fcm_i8_prepare(fcm_handle *h, const void *w1_host) {
    fcm_status st = fcm_i8_constants(h, w1_host, h->cm);
    if (st != FCM_OK) return st;
    const int C = h->cm;
    const fcm_desc v = fcm_i8_pw_desc(h);
    if (fcm_tc_plan(&v, h->ho, h->wo, C, h->num_sms, h->smem_optin, &h->tc2) != FCM_OK)
        return fcm_fail(FCM_ERR_SMEM_BUDGET, "INT8 PW-only stage: no tile fits");
    return FCM_OK;
}

fcm_status fcm_tc_prepare(fcm_handle *h, const void *w1_host, const void *wp_host) {
    if (h->d.conv1 == FCM_CONV1_DENSE) return fcm_b2b_prepare(h, w1_host, wp_host);
    if (h->d.conv1 == FCM_CONV1_POINTWISE) return fcm_pwdw_prepare(h, w1_host, wp_host);
    const fcm_desc &d = h->d;
    const int C = h->cm, K = d.k_out, KS = d.ksize, nkb = (C + 63) / 64;
    const bool i8 = d.dtype == FCM_I8;
    // 16-bit pattern of weight i: the storage value itself, or for INT8 the f16 of the int8
    // value (exact)
    auto w16 = [&](const void *base, size_t i) -> uint16_t {
        if (i8) {
            __half hv = __float2half_rn((float)static_cast<const signed char *>(base)[i]);
            uint16_t b;
            memcpy(&b, &hv, 2);
            return b;
        }
        return static_cast<const uint16_t *>(base)[i];
    };
    // B operand image: row n = output channel, K-dim = input channel, 128B swizzle
    h->wp_img_bytes = (size_t)nkb * K * 128;
    std::vector<uint8_t> img(h->wp_img_bytes, 0);
    for (int n = 0; n < K; n++)
        for (int c = 0; c < C; c++) {
            uint32_t off = sw128_offset(n, c, K, 2);
            const uint16_t b = w16(wp_host, (size_t)n * C + c);
            memcpy(&img[off], &b, 2);
        }
    // DW taps in the storage dtype (f16 for INT8), tap-major: [k*k][C] (lane v of a warp reads
    // channels 8v..8v+7 of one tap as one 16-byte vector, consecutive lanes consecutive vectors)
    std::vector<uint16_t> wdw((size_t)C * KS * KS);
    for (int c = 0; c < C; c++)
        for (int t = 0; t < KS * KS; t++) wdw[(size_t)t * C + c] = w16(w1_host, (size_t)c * KS * KS + t);
    if (i8) {
        fcm_status st = fcm_i8_prepare(h, w1_host);
        if (st != FCM_OK) return st;
    }
    // the same taps with the channel stride padded to a multiple of 64 (worker-warp kernel)
    const int cp = nkb * 64;
    std::vector<uint16_t> wdwp((size_t)cp * KS * KS, 0);
    for (int t = 0; t < KS * KS; t++)
        for (int c = 0; c < C; c++) wdwp[(size_t)t * cp + c] = wdw[(size_t)t * C + c];
    if (cudaMalloc(&h->wp_img, h->wp_img_bytes) != cudaSuccess ||
        cudaMemcpy(h->wp_img, img.data(), h->wp_img_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->w1dw_img, wdw.size() * 2) != cudaSuccess ||
        cudaMemcpy(h->w1dw_img, wdw.data(), wdw.size() * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->w1dw_pad, wdwp.size() * 2) != cudaSuccess ||
        cudaMemcpy(h->w1dw_pad, wdwp.data(), wdwp.size() * 2, cudaMemcpyHostToDevice) != cudaSuccess)
        return fcm_fail(FCM_ERR_CUDA, "tensor-core weight images: %s",
                        cudaGetErrorString(cudaGetLastError()));
    // the layer-by-layer modes run on dwpw_kernel: their own plan when the fused mode runs on
    // the worker-warp kernel
    if (h->tc.variant == 1 &&
        fcm_tc_plan_dwpw_roles(&h->d, h->ho, h->wo, C, h->num_sms, h->smem_optin, &h->tc_lbl) != FCM_OK)
        return fcm_fail(FCM_ERR_SMEM_BUDGET, "layer-by-layer DW->PW stages: no tile fits");
    return FCM_OK;
}

namespace {

template <typename T, int KS, int S, int MODE>
cudaError_t launch_t(const Args &a, int ctas, int threads, uint32_t smem, cudaStream_t st) {
    if constexpr (KS <= 3 && MODE != PWONLY) {
        if (a.dw_per_chunk > 0 && KS == 3 && MODE != PWONLY && threads <= kMaxThreadsBound2)
            return launch_k<T, KS, S, MODE, 2>(a, ctas, threads, smem, st);
        if (a.dw_per_chunk > 0) return launch_k<T, KS, S, MODE, 1>(a, ctas, threads, smem, st);
    }
    return launch_k<T, KS, S, MODE, 0>(a, ctas, threads, smem, st);
}

template <typename T, int MODE>
cudaError_t dispatch_ks(const Args &a, int ks, int s, int ctas, int threads, uint32_t smem,
                        cudaStream_t st) {
    if (MODE == PWONLY) return launch_t<T, 1, 1, MODE>(a, ctas, threads, smem, st);
#define FCM_CASE(KSV, SV) \
    if (ks == KSV && s == SV) return launch_t<T, KSV, SV, MODE>(a, ctas, threads, smem, st);
    FCM_CASE(1, 1) FCM_CASE(1, 2) FCM_CASE(3, 1) FCM_CASE(3, 2)
    FCM_CASE(5, 1) FCM_CASE(5, 2) FCM_CASE(7, 1) FCM_CASE(7, 2)
#undef FCM_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_mode(const fcm_handle *h, int mode, const void *in, void *out, cudaStream_t st) {
    if (mode == FUSED && h->tc.variant == 1) return launch_tc_fused(h, in, out, st);
    const fcm_desc &d = h->d;
    const TcPlan &p = h->tc.variant == 1 ? h->tc_lbl : h->tc;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int out_bufs = mode == FUSED ? p.out_bufs : 1;
    Layout L = make_layout(&d, p, h->cm, mode, h->smem_optin, out_bufs);
    if (L.stages < 1) return cudaErrorInvalidConfiguration;
    Args a;
    memset(&a, 0, sizeof(a));
    const bool i8 = d.dtype == FCM_I8;
    if (i8 && mode == PWONLY) return cudaErrorInvalidValue;   // runs as FUSED (launch_tc_pw)
    const CUtensorMapDataType dt = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : d.dtype == FCM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t es = (cuuint64_t)fcm_dtype_bytes(d.dtype);
    CUresult cr;
    if (mode == PWONLY) {
        long long P = (long long)d.n * h->ho * h->wo;
        cuuint64_t gdim[2] = {(cuuint64_t)h->cm, (cuuint64_t)P};
        cuuint64_t gstride[1] = {(cuuint64_t)h->cm * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kTileM};
        cuuint32_t estr[2] = {1, 1};
        cr = enc(&a.tmap, dt, 2, const_cast<void *>(in), gdim, gstride, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        a.P = P;
        if (P > (long long)INT_MAX - kTileM) return cudaErrorInvalidValue;   // 32-bit TMA coordinates
        a.num_tiles = (int)((P + kTileM - 1) / kTileM);
    } else {
        cuuint64_t gdim[4] = {(cuuint64_t)d.c, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)d.c * es, (cuuint64_t)d.w * d.c * es,
                                 (cuuint64_t)d.h * d.w * d.c * es};
        cuuint32_t box[4] = {(cuuint32_t)p.chunk_c, (cuuint32_t)p.in_cols, (cuuint32_t)p.in_rows, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        cr = enc(&a.tmap, dt, 4, const_cast<void *>(in), gdim, gstride, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (p.num_tiles > INT_MAX) return cudaErrorInvalidValue;
        a.num_tiles = (int)p.num_tiles;
    }
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (mode == PWONLY) {
        cuuint64_t gdim[2] = {(cuuint64_t)d.k_out, (cuuint64_t)a.P};
        cuuint64_t gstride[1] = {(cuuint64_t)d.k_out * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)kTileM};
        cuuint32_t estr[2] = {1, 1};
        cr = enc(&a.tmap_out, dt, 2, out, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (mode == FUSED) {
        cuuint64_t gdim[4] = {(cuuint64_t)d.k_out, (cuuint64_t)h->wo, (cuuint64_t)h->ho,
                              (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)d.k_out * es, (cuuint64_t)h->wo * d.k_out * es,
                                 (cuuint64_t)h->ho * h->wo * d.k_out * es};
        cuuint32_t box[4] = {64, (cuuint32_t)p.tile_w, (cuuint32_t)p.tile_h, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        // staging rows of 64 elements: 128 bytes (16-bit) or 64 bytes (int8), swizzled to match
        cr = enc(&a.tmap_out, dt, 4, out, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 i8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    a.out = out;
    a.wp_img = static_cast<const uint8_t *>(h->wp_img);
    a.wdw = static_cast<const uint4 *>(h->w1dw_img);
    a.s1 = h->s1;
    a.b1 = h->b1;
    a.s2 = h->s2;
    a.b2 = h->b2;
    if (h->b2 && h->b2 == h->b2_host_of && (d.k_out == 64 || d.k_out == 128) &&
        d.k_out <= kMaxBiasParams) {
        memcpy(a.b2c, h->b2_host, sizeof(float) * (size_t)d.k_out);
        a.b2c_n = d.k_out;
    }
    a.q1 = h->q1;
    a.err = h->d_err;
    a.wait_limit_ns = kWaitLimitNs;
    a.N = d.n; a.H = d.h; a.W = d.w; a.C = h->cm; a.K = d.k_out; a.Ho = h->ho; a.Wo = h->wo;
    a.pad = d.pad;
    a.tile_h = p.tile_h;
    a.tile_w = p.tile_w;
    a.tiles_w = p.tiles_w;
    a.tiles_per_img = p.tiles_w * p.tiles_h;
    a.ngroups = (p.tile_w + kR - 1) / kR;
    a.in_rows = p.in_rows;
    a.in_cols = p.in_cols;
    a.chunk_c = p.chunk_c;
    a.nchunks = p.nchunks;
    a.stages = L.stages;
    a.n_dw_warps = mode == PWONLY ? 0 : p.dw_warps;
    a.dw_per_chunk = mode == PWONLY ? 0 : p.dw_per_chunk;
    a.act1 = d.act1;
    a.act2 = d.act2;
    a.tmem_cols = (uint32_t)p.tmem_cols;
    a.idesc = idesc_f16(d.dtype == FCM_BF16, kTileM, d.k_out);   // INT8: f16 operands
    a.wp_img_bytes = (uint32_t)h->wp_img_bytes;
    a.in_stage_bytes = L.in_stage_bytes;
    a.in_stage_stride = L.in_stage_stride;
    a.off_b = L.off_b;
    a.off_a = L.off_a;
    a.off_out = L.off_out;
    a.out_bufs = out_bufs;
    a.out_buf_bytes = (uint32_t)((d.k_out + 63) / 64) * (uint32_t)out_block_bytes((int)es);
    a.off_in = L.off_in;
    a.off_wdw = L.off_wdw;
    a.off_sb = L.off_sb;
    a.off_bar = L.off_bar;
    const int threads = mode == PWONLY ? 32 * kFirstDwWarp : p.threads;
    const int ctas = (int)std::min<long long>(a.num_tiles, h->num_sms);
    if (i8) {
        if (mode == FUSED) return dispatch_ks<int8_t, FUSED>(a, d.ksize, d.stride, ctas, threads, L.total, st);
        return dispatch_ks<int8_t, DWONLY>(a, d.ksize, d.stride, ctas, threads, L.total, st);
    }
    if (d.dtype == FCM_F16) {
        if (mode == FUSED) return dispatch_ks<__half, FUSED>(a, d.ksize, d.stride, ctas, threads, L.total, st);
        if (mode == DWONLY) return dispatch_ks<__half, DWONLY>(a, d.ksize, d.stride, ctas, threads, L.total, st);
        return dispatch_ks<__half, PWONLY>(a, 1, 1, ctas, threads, L.total, st);
    }
    if (mode == FUSED) return dispatch_ks<__nv_bfloat16, FUSED>(a, d.ksize, d.stride, ctas, threads, L.total, st);
    if (mode == DWONLY) return dispatch_ks<__nv_bfloat16, DWONLY>(a, d.ksize, d.stride, ctas, threads, L.total, st);
    return dispatch_ks<__nv_bfloat16, PWONLY>(a, 1, 1, ctas, threads, L.total, st);
}

}  // namespace

cudaError_t launch_tc_dwpw(const fcm_handle *h, int mode, const void *in, void *out,
                           cudaStream_t st) {
    return launch_mode(h, mode == FCM_MODE_FUSED ? FUSED : DWONLY, in, out, st);
}

cudaError_t launch_tc_pw(const fcm_handle *h, const void *m, void *y, cudaStream_t st) {
    if (h->d.dtype == FCM_I8) {
        // INT8: the fused kernel over m with the identity stencil (k = 1, tap 1, scale 1,
        // bias 0, no activation), which hands each int8 value of m to the tensor core as f16
        fcm_handle v = *h;
        v.d = fcm_i8_pw_desc(h);
        v.tc = h->tc2;
        v.s1 = h->i8_one;
        v.b1 = h->i8_zero;
        v.q1 = h->i8_idq;
        v.w1dw_img = h->i8_idtap;
        v.w1dw_pad = h->i8_idtap;
        return launch_mode(&v, FUSED, m, y, st);
    }
    return launch_mode(h, PWONLY, m, y, st);
}
