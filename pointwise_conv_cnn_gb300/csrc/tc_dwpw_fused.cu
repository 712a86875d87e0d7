// tc_dwpw_fused.cu -- host side of dwpw_fused_kernel (tc_dwpw_fused.cuh): its tile planner,
// shared-memory layout, tensor maps and launch.
//
// Planner.  Every output tile is 128 GEMM rows: four TMEM lane quadrants of qw x qh output
// pixels (qw in {32, 16, 8}), nqx quadrants across and 4 / nqx down.  Candidate tiles are
// ranked in two steps, after FusePlanner ("Fusing Depthwise and Pointwise Convolutions for
// Efficient Inference on GPUs", section IV): the kernel is bound by the issue of its CUDA-core
// work, so a tile is admissible only if it wastes at most 3% more of the tensor-core rows and
// stencil lanes than the best tile does (efficiency = useful / MMA rows x useful / stencil
// pixels); among admissible tiles the planner takes the smallest global-memory-access estimate
// of the DWPW module (Eq. 1 overlap in the section IV-B form, built like Eq. 4), then the
// deeper input ring, then the larger tile count.  The pipeline depth (input stages, one or two
// A tiles) is the deepest that fits 227 KB of shared memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <string.h>

#include <algorithm>

#include "tc_dwpw_fused.cuh"

namespace fcm {
namespace tc {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();   // tc_dwpw.cu

namespace {

uint32_t al(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

struct FLayout {
    uint32_t off_b, off_a, a_buf_bytes, off_out, off_in, in_stage_bytes, in_stage_stride, off_wdw,
        off_sb, off_bar, total;
    int stages;
};

// 128-byte output staging blocks per pixel row (64 channels of 16-bit, 128 of int8)
int f_nblk(int k_out, int esize) { return (k_out * esize + 127) / 128; }

// Shared memory of a plan with `abufs` A tiles, `sbufs` output staging buffers and as many
// input stages as fit (<= kFMaxStages).
FLayout f_layout(int cp, int k_out, int ks, int esize, int in_rows, int in_cols, int abufs,
                 int sbufs, int smem_cap) {
    FLayout L{};
    const int nch = cp / 64;
    const uint32_t b_bytes = (uint32_t)nch * (uint32_t)k_out * 128u;
    L.a_buf_bytes = (uint32_t)nch * (uint32_t)kTileM * 128u;
    L.off_b = 0;
    L.off_a = al(b_bytes, 1024);
    L.off_out = al(L.off_a + (uint32_t)abufs * L.a_buf_bytes, 1024);
    const uint32_t out_bytes = (uint32_t)sbufs * 4u * (uint32_t)f_nblk(k_out, esize) * 4096u;
    L.off_in = al(L.off_out + out_bytes, 1024);
    L.in_stage_bytes = (uint32_t)in_rows * (uint32_t)in_cols * 64u * (uint32_t)esize;
    L.in_stage_stride = al(L.in_stage_bytes, 1024);
    const uint32_t wdw = (uint32_t)(ks * ks * cp * 2);
    const uint32_t sb = (uint32_t)(3 * cp + 2 * k_out) * 4u;
    const uint32_t tail = al(wdw, 16) + al(sb, 16) + kFBarBytes + 16 + 1024;
    const int cap = std::min(smem_cap, kFSmemMax);
    int stages = kFMaxStages;
    for (; stages >= 1; stages--)
        if ((long long)L.off_in + (long long)stages * L.in_stage_stride + tail <= cap) break;
    L.stages = stages;
    L.off_wdw = L.off_in + (uint32_t)std::max(stages, 0) * L.in_stage_stride;
    L.off_sb = L.off_wdw + al(wdw, 16);
    L.off_bar = L.off_sb + al(sb, 16);
    L.total = L.off_bar + kFBarBytes + 16 + 1024;
    return L;
}

int ilog2(int v) {
    int l = 0;
    while ((1 << (l + 1)) <= v) l++;
    return l;
}

// ceil(2^32 / d) for 2 <= d < 2^16 (the kernel's multiply-high division), 0 for d = 1
uint32_t recip16(int d) {
    if (d <= 1) return 0u;
    return (uint32_t)(((1ull << 32) + (unsigned long long)d - 1) / (unsigned long long)d);
}

int pow2_at_least(int v) {
    int c = 32;
    while (c < v) c <<= 1;
    return c;
}

}  // namespace
}  // namespace tc
}  // namespace fcm

using namespace fcm::tc;

extern "C" long long fcm_model_overlap(long long, long long, long long, long long, long long,
                                       long long, long long);
extern "C" long long fcm_model_dwpw_gma(long long, long long, long long, long long, long long,
                                        long long, long long, long long, long long);

fcm_status fcm_fused_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_cap,
                          TcPlan *out) {
    if (d->conv1 != FCM_CONV1_DEPTHWISE || d->dtype == FCM_F32) return FCM_ERR_UNSUPPORTED;
    const int C = cm, K = d->k_out, KS = d->ksize, S = d->stride;
    const int es = fcm_dtype_bytes(d->dtype);
    const int cp = (C + 63) / 64 * 64, nch = cp / 64;
    if (nch > kFMaxChunks || C % 8 != 0) return FCM_ERR_UNSUPPORTED;
    if (K % 16 != 0 || K < 16 || K > 256) return FCM_ERR_UNSUPPORTED;
    if (KS != 1 && KS != 3 && KS != 5 && KS != 7) return FCM_ERR_UNSUPPORTED;
    if (d->dtype == FCM_I8 && C > 256) return FCM_ERR_UNSUPPORTED;   // exact f16 1x1 sums
    // 14 workers: warps 2..15, so TMEM lane quadrants 2 and 3 have four workers each and
    // quadrants 0 and 1 three
    const int nw = kFMaxWorkers;
    struct Cand {
        TcPlan p;
        double eff;
        long long gma;
    };
    Cand cands[9];
    int ncand = 0;
    double best_eff = 0.0;
    for (int qw : {32, 16, 8}) {
        const int qh = 32 / qw;
        for (int nqx : {1, 2, 4}) {
            const int tw = qw * nqx, th = qh * (4 / nqx);
            if (d->tile_h > 0 && th != d->tile_h) continue;
            if (d->tile_w > 0 && tw != d->tile_w) continue;
            const int twv = std::min(tw, wo);
            const int ngroups = (twv + kFUnitPx - 1) / kFUnitPx;
            const int in_cols = (ngroups * kFUnitPx - 1) * S + KS;
            const int in_rows = (th - 1) * S + KS;
            if (in_cols > 256 || in_rows > 256) continue;
            const long long tiles_w = (wo + tw - 1) / tw, tiles_h = (ho + th - 1) / th;
            const long long num_tiles = (long long)d->n * tiles_w * tiles_h;
            if (num_tiles > INT_MAX) continue;
            TcPlan t;
            t.variant = 1;
            t.tile_h = th;
            t.tile_w = tw;
            t.qw = qw;
            t.qh = qh;
            t.nqx = nqx;
            t.in_rows = in_rows;
            t.in_cols = in_cols;
            t.chunk_c = 64;
            t.nchunks = nch;
            t.cp = cp;
            t.ngroups = ngroups;
            t.nw = nw;
            t.dw_warps = nw;
            // pipeline depth: the first of (A tiles, staging buffers) = (2, 2), (1, 2), (2, 1),
            // (1, 1) that leaves three input stages, else the first that leaves two
            FLayout L{};
            bool found = false;
            for (int need = 3; need >= 2 && !found; need--)
                for (int combo = 0; combo < 4 && !found; combo++) {
                    const int ab = combo == 0 || combo == 2 ? 2 : 1, sbf = combo < 2 ? 2 : 1;
                    L = f_layout(cp, K, KS, es, in_rows, in_cols, ab, sbf, smem_cap);
                    if (L.stages >= need) {
                        found = true;
                        t.abufs = ab;
                        t.sbufs = sbf;
                    }
                }
            if (!found) continue;
            t.stages = L.stages;
            t.smem_bytes = (int)L.total;
            t.tiles_w = (int)tiles_w;
            t.tiles_h = (int)tiles_h;
            t.num_tiles = num_tiles;
            t.threads = 32 * (2 + nw);
            t.ctas = (int)std::min<long long>(num_tiles, num_sms);
            t.tmem_cols = pow2_at_least(2 * K);
            const double useful = (double)ho * wo;
            const double mma_rows = (double)tiles_w * tiles_h * kTileM;
            const double stencil_px = (double)tiles_w * tiles_h * th * ngroups * kFUnitPx;
            const double eff = (useful / mma_rows) * (useful / stencil_px);
            // section IV-B estimate of the module's global-memory accesses with this tile
            const long long ov = fcm_model_overlap(d->w, d->h, (long long)twv * S, (long long)th * S,
                                                   KS, KS, S);
            const long long gma = fcm_model_dwpw_gma(C, ov, (long long)d->h * d->w * C,
                                                     (long long)K * C, (long long)K * C,
                                                     (long long)ho * wo * K, (long long)ho * wo,
                                                     (long long)th * twv, (long long)C * KS * KS);
            cands[ncand++] = Cand{t, eff, gma};
            best_eff = std::max(best_eff, eff);
        }
    }
    const Cand *pick = nullptr;
    for (int i = 0; i < ncand; i++) {
        const Cand &c = cands[i];
        if (c.eff < 0.97 * best_eff) continue;
        if (!pick || c.gma < pick->gma ||
            (c.gma == pick->gma && (c.p.stages > pick->p.stages ||
                                    (c.p.stages == pick->p.stages && c.p.num_tiles > pick->p.num_tiles))))
            pick = &c;
    }
    if (!pick) return FCM_ERR_SMEM_BUDGET;
    *out = pick->p;
    return FCM_OK;
}

cudaError_t launch_tc_fused(const fcm_handle *h, const void *x, void *y, cudaStream_t st) {
    const fcm_desc &d = h->d;
    const TcPlan &p = h->tc;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (p.variant != 1 || !h->w1dw_pad) return cudaErrorInvalidConfiguration;
    const int es = fcm_dtype_bytes(d.dtype);
    const FLayout L = f_layout(p.cp, d.k_out, d.ksize, es, p.in_rows, p.in_cols, p.abufs, p.sbufs,
                               h->smem_optin);
    if (L.stages != p.stages) return cudaErrorInvalidConfiguration;
    FArgs a;
    memset(&a, 0, sizeof(a));
    const bool i8 = d.dtype == FCM_I8;
    const CUtensorMapDataType dt = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : d.dtype == FCM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t e = (cuuint64_t)es;
    {
        cuuint64_t gdim[4] = {(cuuint64_t)d.c, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)d.c * e, (cuuint64_t)d.w * d.c * e,
                                 (cuuint64_t)d.h * d.w * d.c * e};
        cuuint32_t box[4] = {64, (cuuint32_t)p.in_cols, (cuuint32_t)p.in_rows, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&a.tmap_x, dt, 4, const_cast<void *>(x), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // one store per 128-byte staging block of a lane quadrant: 128 / esize channels of qw x qh
        // pixels (channels past K are clipped)
        cuuint64_t gdim[4] = {(cuuint64_t)d.k_out, (cuuint64_t)h->wo, (cuuint64_t)h->ho,
                              (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)d.k_out * e, (cuuint64_t)h->wo * d.k_out * e,
                                 (cuuint64_t)h->ho * h->wo * d.k_out * e};
        // a quadrant of one pixel row stores only the columns inside the image (its first
        // min(qw, Wo) staging rows); taller quadrants store their full qw x qh box, clipped
        const int bw = p.qh == 1 ? std::min(p.qw, h->wo) : p.qw;
        cuuint32_t box[4] = {(cuuint32_t)(128 / es), (cuuint32_t)bw, (cuuint32_t)p.qh, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&a.tmap_y, dt, 4, y, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (p.num_tiles > INT_MAX) return cudaErrorInvalidValue;
    a.wp_img = static_cast<const uint8_t *>(h->wp_img);
    a.wdw = static_cast<const uint4 *>(h->w1dw_pad);
    a.s1 = h->s1;
    a.b1 = h->b1;
    a.s2 = h->s2;
    a.b2 = h->b2;
    a.q1 = h->q1;
    a.err = h->d_err;
    a.wait_limit_ns = kWaitLimitNs;
    a.num_tiles = (int)p.num_tiles;
    a.C = h->cm;
    a.Cp = p.cp;
    a.K = d.k_out;
    a.Ho = h->ho;
    a.Wo = h->wo;
    a.pad = d.pad;
    a.tiles_w = p.tiles_w;
    a.tiles_per_img = p.tiles_w * p.tiles_h;
    a.th = p.tile_h;
    a.tw = p.tile_w;
    a.qw = p.qw;
    a.qh = p.qh;
    a.nqx = p.nqx;
    a.ngroups = p.ngroups;
    a.in_rows = p.in_rows;
    a.in_cols = p.in_cols;
    a.nchunks = p.nchunks;
    a.stages = L.stages;
    a.nw = p.nw;
    a.abufs = p.abufs;
    a.sbufs = p.sbufs;
    a.nblk = f_nblk(d.k_out, es);
    a.lg_qw = ilog2(p.qw);
    a.lg_qh = ilog2(p.qh);
    const int npg4 = (p.tile_h * p.ngroups + 3) & ~3;
    a.mg_ngroups = recip16(p.ngroups);
    a.mg_uc = recip16(8 * npg4);
    if (p.nchunks * 8 * npg4 >= 65536) return cudaErrorInvalidValue;   // fdiv's range
    a.act1 = d.act1;
    a.act2 = d.act2;
    a.tmem_cols = (uint32_t)p.tmem_cols;
    a.idesc = idesc_f16(d.dtype == FCM_BF16, kTileM, d.k_out);   // INT8: f16 operands
    a.wp_img_bytes = (uint32_t)h->wp_img_bytes;
    a.in_stage_bytes = L.in_stage_bytes;
    a.in_stage_stride = L.in_stage_stride;
    a.off_b = L.off_b;
    a.off_a = L.off_a;
    a.a_buf_bytes = L.a_buf_bytes;
    a.off_out = L.off_out;
    a.off_in = L.off_in;
    a.off_wdw = L.off_wdw;
    a.off_sb = L.off_sb;
    a.off_bar = L.off_bar;
    const int threads = 32 * (2 + p.nw);
    const int ctas = (int)std::min<long long>(p.num_tiles, h->num_sms);
    // the grid size in (images, tile rows, tile columns), for the kernel's tile iterators
    const int tpi = p.tiles_w * p.tiles_h;
    a.step_n = ctas / tpi;
    a.step_ty = (ctas % tpi) / p.tiles_w;
    a.step_tx = (ctas % tpi) % p.tiles_w;
    a.tiles_h = p.tiles_h;
    const int ks = d.ksize, s = d.stride;
#define FCM_CASE(T, KSV, SV) \
    if (ks == KSV && s == SV) return launch_fused<T, KSV, SV>(a, ctas, threads, L.total, st);
#define FCM_CASES(T)                                                                    \
    FCM_CASE(T, 1, 1) FCM_CASE(T, 1, 2) FCM_CASE(T, 3, 1) FCM_CASE(T, 3, 2) FCM_CASE(T, 5, 1) \
    FCM_CASE(T, 5, 2) FCM_CASE(T, 7, 1) FCM_CASE(T, 7, 2)
    if (i8) {
        FCM_CASES(int8_t)
    } else if (d.dtype == FCM_F16) {
        FCM_CASES(__half)
    } else {
        FCM_CASES(__nv_bfloat16)
    }
#undef FCM_CASES
#undef FCM_CASE
    return cudaErrorInvalidValue;
}
