// tc_pwdw.cu -- the PWDW module (1x1 convolution, then a depthwise k x k convolution of its
// output) for sm_103a: the expansion and depthwise layers of an inverted residual.
//
// "Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs": the PWDW_R
// FCM of section II-D (Figure 3(b)) and section III-A.  A tile of the depthwise output needs
// the intermediate over the tile's halo, which the neighbouring tiles also need: the values
// there do not exist before the kernel starts, so every tile recomputes them (the "_R").  On
// Blackwell the recomputation is cheap -- it is part of a tensor-core GEMM -- and the
// intermediate never leaves the SM:
//
//   producer   TMA: the input halo box of a tile (R = (TH-1)s+k rows x Q columns, all C input
//              channels, 128-byte swizzled, zero-filled outside the image) -- the GEMM's A
//              operand, one row per halo pixel, in M blocks of 128 rows
//   MMA        1x1 convolution for one 64-channel chunk of the intermediate:
//              D[halo pixel, 64] = A x W1[chunk]^T into TMEM (double-buffered)
//   mid        8 warps: TMEM -> scale/bias/act1 -> 16-bit -> the commBuffer in shared memory
//              (one 128-byte row per halo pixel, 16-byte chunks swizzled by the pixel index);
//              halo pixels outside the image are written as zeros -- the depthwise layer pads
//              its own input, the intermediate
//   DW         CUDA-core stencil over the commBuffer (mixed-precision FMA, fp32 sums) ->
//              scale/bias/act2 -> 128-byte-swizzled output staging -> TMA tensor store
//
// Work items are (tile, 64-channel chunk); the input box of a tile is loaded once and serves
// all its chunks.  Every wait is bounded, as in the other kernels.
//
// INT8 (T = int8_t; the INT8 FCMs of section III-B: int8 input, weights, intermediate and
// output, exact integer sums): the producer warp loads the int8 halo box into a ring of its
// own and widens it exactly to the f16 A operand (int8 values are exact in f16; every partial
// sum of the 1x1 stays below 256 * 128 * 128 = 2^22, exact in the fp32 accumulator); the mid
// warps requantize the intermediate (fp32 fma, round to nearest even, saturate) and keep it as
// exact f16 values in the commBuffer (int8 zero outside the image); the stencil runs on f16 images
// of the int8 taps (sums below 2^24, exact) and the output is requantized to int8.
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "fcm_internal.h"
#include "tc_common.cuh"

namespace fcm {
namespace pwdw {

using namespace fcm::tc;

constexpr int kMidWarps = 8;     // two per TMEM lane quadrant: even and odd M blocks
constexpr int kFirstDwWarp = 2 + kMidWarps;
constexpr int kMaxDwWarps = 10;
constexpr int kMaxThreads = 32 * (kFirstDwWarp + kMaxDwWarps);
constexpr int kR = 4;           // output pixels per DW work unit (along W)
constexpr int kCt = 64;         // intermediate channels per work item
constexpr int kMaxBlk = 4;      // M blocks of 128 halo pixels
constexpr int kMaxStages = 4;
constexpr uint32_t kBlk = 128 * 128;   // one 128-row, 128-byte operand block
constexpr int kMaxStages8 = 3;          // INT8: stages of the producer's int8 ring

struct Args {
    CUtensorMap tmap_x;        // x: 4-D (C, W, H, N), box (64, Q, R, 1), 128B swizzle
                               // (INT8: no swizzle, into the int8 ring)
    CUtensorMap tmap_y;        // y: 4-D (Cm, Wo, Ho, N), box (64, Wo, TH, 1), 128B swizzle
                               // (INT8: 64-byte rows, 64B swizzle)
    const uint8_t *w1_img;     // B operand: C/64 blocks of [Cm rows x 128 B]
    const uint4 *wdw;          // depthwise taps [k*k][Cm], storage dtype
    const float *s1, *b1, *s2, *b2;
    unsigned *err;
    unsigned long long wait_limit_ns;
    int num_tiles, tiles_per_img, nchunks;
    int H, W, C, Cm, Ho, Wo, pad;
    int TH, R, Q, nblk, ngroups;
    int stages, n_dw_warps, act1, act2;
    uint32_t tmem_cols, idesc, w1_bytes, plane_bytes, x_stage_bytes, x_stage_stride, comm_bytes;
    uint32_t off_w1, off_x, off_comm, off_out, off_wdw, off_sb, off_bar;
    // INT8: the producer's ring of int8 halo boxes (nkb planes of R*Q pixels x 64 bytes)
    uint32_t off_x8, plane8_bytes, x8_stage_bytes, x8_stage_stride;
    int stages8;
};

struct Bars {
    uint32_t full, empty, accfull, accempty, commfull, commempty, wbar, drain, full8;
    __device__ Bars(uint32_t base) {
        full = base;
        empty = full + 8 * kMaxStages;
        accfull = empty + 8 * kMaxStages;
        accempty = accfull + 16;
        commfull = accempty + 16;
        commempty = commfull + 16;
        wbar = commempty + 16;
        drain = wbar + 8;
        full8 = drain + 8;   // INT8: [kMaxStages8]
    }
};
constexpr uint32_t kBarBytes = 8 * (2 * kMaxStages + 8 + 2 + kMaxStages8) + 16;

__device__ __forceinline__ void tile_coords(const Args &a, int t, int &n, int &ho0) {
    n = t / a.tiles_per_img;
    ho0 = (t - n * a.tiles_per_img) * a.TH;
}

// One DW work unit: kR consecutive output pixels of tile row r, 8 channels (v) of chunk j.
// The commBuffer row of halo pixel p holds its 64 channels with 16-byte chunk c at c ^ (p & 7).
// INT8: the commBuffer and the taps hold f16 images of int8 values; the output is requantized
// and staged as 64-byte rows (16-byte chunk c at c ^ ((row >> 1) & 3), the TMA's 64B swizzle).
template <typename T, int KS, int S, int ACT>
__device__ __forceinline__ void dw_unit(const Args &a, int r, int g, int v, int j,
                                        const uint8_t *comm, const uint8_t *wdw,
                                        const float *s2_s, const float *b2_s, uint32_t out_s) {
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    using TM = typename std::conditional<kI8, __half, T>::type;   // arithmetic type
    const int c_glob = j * kCt + v * 8;
    const uint8_t *wb = wdw + (uint32_t)c_glob * 2u;
    const uint32_t tap_bytes = (uint32_t)a.Cm * 2u;
    float acc[kR][8];
#pragma unroll
    for (int jj = 0; jj < kR; jj++)
#pragma unroll
        for (int c = 0; c < 8; c++) acc[jj][c] = 0.0f;
#pragma unroll
    for (int i = 0; i < KS; i++) {
        uint4 w[KS];
#pragma unroll
        for (int t = 0; t < KS; t++)
            w[t] = *reinterpret_cast<const uint4 *>(wb + (uint32_t)(i * KS + t) * tap_bytes);
        const int prow = (r * S + i) * a.Q + g * kR * S;   // halo pixel of this row's first tap
#pragma unroll
        for (int q = 0; q < (kR - 1) * S + KS; q++) {
            const uint32_t pix = (uint32_t)(prow + q);
            const uint4 x = *reinterpret_cast<const uint4 *>(
                comm + pix * 128u + ((((uint32_t)v) ^ (pix & 7u)) << 4));
#pragma unroll
            for (int jj = 0; jj < kR; jj++) {
                const int t = q - jj * S;
                if (t >= 0 && t < KS) {
                    Fma16<TM>::fma2(acc[jj][0], acc[jj][1], x.x, w[t].x);
                    Fma16<TM>::fma2(acc[jj][2], acc[jj][3], x.y, w[t].y);
                    Fma16<TM>::fma2(acc[jj][4], acc[jj][5], x.z, w[t].z);
                    Fma16<TM>::fma2(acc[jj][6], acc[jj][7], x.w, w[t].w);
                }
            }
        }
    }
    const float4 sc0 = *reinterpret_cast<const float4 *>(s2_s + c_glob);
    const float4 sc1 = *reinterpret_cast<const float4 *>(s2_s + c_glob + 4);
    const float4 bi0 = *reinterpret_cast<const float4 *>(b2_s + c_glob);
    const float4 bi1 = *reinterpret_cast<const float4 *>(b2_s + c_glob + 4);
    const float sc[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
    const float bi[8] = {bi0.x, bi0.y, bi0.z, bi0.w, bi1.x, bi1.y, bi1.z, bi1.w};
#pragma unroll
    for (int jj = 0; jj < kR; jj++) {
        const int oc = g * kR + jj;
        if (oc >= a.Wo) break;
        const uint32_t row = (uint32_t)(r * a.Wo + oc);
        if constexpr (kI8) {
            float y[8];
#pragma unroll
            for (int c = 0; c < 8; c++) y[c] = fmaf(sc[c], acc[jj][c], bi[c]);
            const uint32_t ch = (((uint32_t)v >> 1) ^ ((row >> 1) & 3u)) << 4;
            sts64(out_s + row * 64u + ch + ((uint32_t)v & 1u) * 8u, I8::bytes4<ACT>(y[0], y[1], y[2], y[3]),
                  I8::bytes4<ACT>(y[4], y[5], y[6], y[7]));
        } else {
            uint32_t pk[4];
#pragma unroll
            for (int c = 0; c < 4; c++)
                pk[c] = Pack2<T>::template run<ACT>(fmaf(sc[2 * c], acc[jj][2 * c], bi[2 * c]),
                                                    fmaf(sc[2 * c + 1], acc[jj][2 * c + 1], bi[2 * c + 1]));
            sts128(out_s + row * 128u + ((((uint32_t)v) ^ (row & 7u)) << 4), pk[0], pk[1], pk[2], pk[3]);
        }
    }
}

template <typename T, int KS, int S>
__global__ void __launch_bounds__(kMaxThreads, 1) pwdw_kernel(const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base_g = smem_raw + (base_s - raw_s);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool kI8 = std::is_same<T, int8_t>::value;

    uint4 *wdw_s = reinterpret_cast<uint4 *>(base_g + a.off_wdw);
    float *sb_s = reinterpret_cast<float *>(base_g + a.off_sb);
    float *s1_s = sb_s, *b1_s = sb_s + a.Cm, *s2_s = sb_s + 2 * a.Cm, *b2_s = sb_s + 3 * a.Cm;
    Bars bars(base_s + a.off_bar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_g + a.off_bar + kBarBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base_g + a.off_bar + kBarBytes + 4);

    {
        const int nw = a.Cm * KS * KS / 8;
        for (int i = threadIdx.x; i < nw; i += blockDim.x) wdw_s[i] = a.wdw[i];
        for (int i = threadIdx.x; i < a.Cm; i += blockDim.x) {
            s1_s[i] = a.s1[i];
            b1_s[i] = a.b1[i];
            s2_s[i] = a.s2[i];
            b2_s[i] = a.b2[i];
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; s++) {
            mbar_init(bars.full + 8 * s, 1);
            mbar_init(bars.empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bars.accfull + 8 * b, 1);
            mbar_init(bars.accempty + 8 * b, kMidWarps);
            mbar_init(bars.commfull + 8 * b, kMidWarps);
            mbar_init(bars.commempty + 8 * b, a.n_dw_warps);
        }
        mbar_init(bars.wbar, 1);
        mbar_init(bars.drain, 1);
        if (kI8)
            for (int s = 0; s < a.stages8; s++) mbar_init(bars.full8 + 8 * s, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const unsigned long long lim = a.wait_limit_ns;
    const int my_tiles = (a.num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int nkb = a.C / 64;
    const uint32_t buf_cols = (uint32_t)(a.nblk * kCt);

    if (warp == 0 && kI8) {
        // ===================================================== INT8 producer
        // Loads tile lt + stages8 - 1 into its int8 ring while it widens tile lt into the f16
        // A operand (stage lt % stages): it frees its own ring slots, so only the A stages wait.
        bool ok = true;
        int issued = 0;   // int8 boxes issued; box i went to ring slot i % stages8
        if (lane == 0) {
            mbar_arrive_expect_tx(bars.wbar, a.w1_bytes);
            bulk_load(base_s + a.off_w1, a.w1_img, a.w1_bytes, bars.wbar);
            tma_prefetch_desc(&a.tmap_x);
        }
        pdl_wait();
        auto load8 = [&](int lt) {
            const int t = (int)blockIdx.x + lt * (int)gridDim.x;
            int n, ho0;
            tile_coords(a, t, n, ho0);
            const int s8 = lt % a.stages8;
            if (lane == 0) {
                const uint32_t dst = base_s + a.off_x8 + (uint32_t)s8 * a.x8_stage_stride;
                mbar_arrive_expect_tx(bars.full8 + 8 * s8, a.x8_stage_bytes);
                for (int kb = 0; kb < nkb; kb++)
                    tma_load_4d(dst + (uint32_t)kb * a.plane8_bytes, &a.tmap_x, bars.full8 + 8 * s8,
                                kb * 64, -a.pad, ho0 * S - a.pad, n);
            }
            __syncwarp();
        };
        for (; issued < my_tiles && issued < a.stages8; issued++) load8(issued);
        const __half2 bias2 = __float2half2_rn(I8::kBias);
        const int RQ = a.R * a.Q;
        for (int lt = 0; lt < my_tiles; lt++) {
            const int s = lt % a.stages, s8 = lt % a.stages8;
            if (!mbar_wait(bars.full8 + 8 * s8, (uint32_t)(lt / a.stages8) & 1u, abort_flag, a.err, lim) ||
                !mbar_wait(bars.empty + 8 * s, ((uint32_t)(lt / a.stages) & 1u) ^ 1u, abort_flag, a.err,
                           lim)) {
                ok = false;
                break;
            }
            const uint8_t *src = base_g + a.off_x8 + (uint32_t)s8 * a.x8_stage_stride;
            const uint32_t dst = base_s + a.off_x + (uint32_t)s * a.x_stage_stride;
            for (int p = lane; p < RQ; p += 32) {
                const uint32_t swz = (uint32_t)p & 7u;
                for (int kb = 0; kb < nkb; kb++) {
                    const uint8_t *row8 = src + (uint32_t)kb * a.plane8_bytes + (uint32_t)p * 64u;
                    const uint32_t row_s = dst + (uint32_t)kb * a.plane_bytes + (uint32_t)p * 128u;
#pragma unroll
                    for (int hh = 0; hh < 4; hh++) {   // 16 channels -> two 16-byte chunks of f16
                        const uint4 v = *reinterpret_cast<const uint4 *>(row8 + (uint32_t)hh * 16u);
                        uint32_t w[8];
                        I8::widen4(v.x, w[0], w[1]);
                        I8::widen4(v.y, w[2], w[3]);
                        I8::widen4(v.z, w[4], w[5]);
                        I8::widen4(v.w, w[6], w[7]);
#pragma unroll
                        for (int i = 0; i < 8; i++) {   // (1152 + x) - 1152 = x, exact in f16
                            __half2 hv = *reinterpret_cast<__half2 *>(&w[i]);
                            hv = __hsub2(hv, bias2);
                            w[i] = *reinterpret_cast<uint32_t *>(&hv);
                        }
                        sts128(row_s + (((uint32_t)(2 * hh) ^ swz) << 4), w[0], w[1], w[2], w[3]);
                        sts128(row_s + (((uint32_t)(2 * hh + 1) ^ swz) << 4), w[4], w[5], w[6], w[7]);
                    }
                }
            }
            fence_proxy_async_smem();   // the f16 operand is read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.full + 8 * s);
            // ring slot s8 is read: load the next box into it
            if (issued < my_tiles) load8(issued++);
        }
        if (!ok) {
            // every box this warp issued lands before the CTA exits (box i went to slot
            // i % stages8)
            volatile int no_abort = 0;
            for (int q = 0; q < a.stages8 && q < issued; q++) {
                const int nq = (issued - 1 - q) / a.stages8 + 1;
                mbar_wait(bars.full8 + 8 * q, (uint32_t)(nq - 1) & 1u, &no_abort, a.err, lim);
            }
            mbar_wait(bars.wbar, 0, &no_abort, a.err, lim);
        }
    } else if (warp == 0) {
        // ===================================================== TMA producer
        bool ok = true;
        int issued = 0;   // tiles loaded so far; tile i goes to stage i % stages
        if (lane == 0) {
            mbar_arrive_expect_tx(bars.wbar, a.w1_bytes);
            bulk_load(base_s + a.off_w1, a.w1_img, a.w1_bytes, bars.wbar);
            tma_prefetch_desc(&a.tmap_x);
        }
        pdl_wait();
        for (int lt = 0; lt < my_tiles; lt++) {
            const int t = (int)blockIdx.x + lt * (int)gridDim.x;
            int n, ho0;
            tile_coords(a, t, n, ho0);
            const int s = lt % a.stages;
            const uint32_t ph = (uint32_t)(lt / a.stages) & 1u;
            if (!mbar_wait(bars.empty + 8 * s, ph ^ 1u, abort_flag, a.err, lim)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t dst = base_s + a.off_x + (uint32_t)s * a.x_stage_stride;
                mbar_arrive_expect_tx(bars.full + 8 * s, a.x_stage_bytes);
                for (int kb = 0; kb < nkb; kb++)
                    tma_load_4d(dst + (uint32_t)kb * a.plane_bytes, &a.tmap_x, bars.full + 8 * s,
                                kb * 64, -a.pad, ho0 * S - a.pad, n);
            }
            issued++;
            __syncwarp();
        }
        if (!ok) {
            volatile int no_abort = 0;
            for (int q = 0; q < a.stages && q < issued; q++) {
                const int nq = (issued - 1 - q) / a.stages + 1;
                mbar_wait(bars.full + 8 * q, (uint32_t)(nq - 1) & 1u, &no_abort, a.err, lim);
            }
            mbar_wait(bars.wbar, 0, &no_abort, a.err, lim);
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        bool ok = mbar_wait(bars.wbar, 0, abort_flag, a.err, lim);
        const uint64_t w_base = sw128_kmajor_desc(base_s + a.off_w1);
        const uint32_t w_kb = (uint32_t)a.Cm * 128u;   // one 64-wide K block of the weights
        for (int lt = 0; ok && lt < my_tiles; lt++) {
            const int s = lt % a.stages;
            if (!mbar_wait(bars.full + 8 * s, (uint32_t)(lt / a.stages) & 1u, abort_flag, a.err,
                           lim)) {
                ok = false;
                break;
            }
            const uint64_t x_base =
                sw128_kmajor_desc(base_s + a.off_x + (uint32_t)s * a.x_stage_stride);
            for (int j = 0; j < a.nchunks; j++) {
                const int li = lt * a.nchunks + j, b = li & 1;
                if (!mbar_wait(bars.accempty + 8 * b, ((uint32_t)(li >> 1) & 1u) ^ 1u, abort_flag,
                               a.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    for (int blk = 0; blk < a.nblk; blk++) {
                        const uint32_t d = tmem_base + (uint32_t)b * buf_cols + (uint32_t)blk * kCt;
                        for (int kb = 0; kb < nkb; kb++) {
                            const uint64_t ad =
                                desc_advance(x_base, (uint32_t)kb * a.plane_bytes + (uint32_t)blk * kBlk);
                            const uint64_t bd =
                                desc_advance(w_base, (uint32_t)kb * w_kb + (uint32_t)j * kCt * 128u);
#pragma unroll
                            for (int k16 = 0; k16 < 4; k16++)
                                mma_f16(d, desc_advance(ad, 32u * k16), desc_advance(bd, 32u * k16),
                                        a.idesc, (kb | k16) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(bars.accfull + 8 * b);
                    if (j == a.nchunks - 1) mma_commit(bars.empty + 8 * s);   // stage read
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            volatile int no_abort = 0;
            mma_commit(bars.drain);
            mbar_wait(bars.drain, 0, &no_abort, a.err, lim);
        }
        __syncwarp();
    } else if (warp < kFirstDwWarp) {
        // ===================================================== mid epilogue
        const int q = warp & 3;          // TMEM lane quadrant
        const int half = (warp - 2) >> 2; // this warp converts the M blocks of this parity
        const int RQ = a.R * a.Q;
        with_act(a.act1, [&](auto act_tag) {
            constexpr int ACT = decltype(act_tag)::value;
            for (int lt = 0; lt < my_tiles; lt++) {
                const int t = (int)blockIdx.x + lt * (int)gridDim.x;
                int n, ho0;
                tile_coords(a, t, n, ho0);
                (void)n;
                bool ok = true;
                for (int j = 0; j < a.nchunks; j++) {
                    const int li = lt * a.nchunks + j, b = li & 1;
                    const uint32_t use = (uint32_t)(li >> 1) & 1u;
                    if (!mbar_wait(bars.accfull + 8 * b, use, abort_flag, a.err, lim) ||
                        !mbar_wait(bars.commempty + 8 * b, use ^ 1u, abort_flag, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t comm_s = base_s + a.off_comm + (uint32_t)b * a.comm_bytes;
                    for (int blk = half; blk < a.nblk; blk += 2) {
                        const int pix = blk * 128 + q * 32 + lane;
                        const int r = pix / a.Q, c = pix - (pix / a.Q) * a.Q;
                        const int ih = ho0 * S - a.pad + r, iw = c - a.pad;
                        const bool inside = pix < RQ && ih >= 0 && ih < a.H && iw >= 0 && iw < a.W;
                        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                                               (uint32_t)b * buf_cols + (uint32_t)blk * kCt;
                        const uint32_t row_s = comm_s + (uint32_t)pix * 128u;
                        const uint32_t swz = (uint32_t)pix & 7u;
                        for (int c0 = 0; c0 < kCt; c0 += 32) {
                            uint32_t ra[16], rb[16];
                            tmem_ld16(taddr + (uint32_t)c0, ra);
                            tmem_ld16(taddr + (uint32_t)(c0 + 16), rb);
                            tmem_ld_wait(ra, rb);
                            if (pix < RQ) {
#pragma unroll
                                for (int h = 0; h < 2; h++) {
                                    const uint32_t *rr = h ? rb : ra;
                                    const int cc = c0 + 16 * h;
                                    const int cg = j * kCt + cc;
                                    uint32_t pk[8];
#pragma unroll
                                    for (int i4 = 0; i4 < 4; i4++) {
                                        const float4 sc = *reinterpret_cast<const float4 *>(s1_s + cg + 4 * i4);
                                        const float4 bi = *reinterpret_cast<const float4 *>(b1_s + cg + 4 * i4);
                                        const float v0 = fmaf(sc.x, __uint_as_float(rr[4 * i4]), bi.x);
                                        const float v1 = fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), bi.y);
                                        const float v2 = fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), bi.z);
                                        const float v3 = fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), bi.w);
                                        if constexpr (kI8) {
                                            pk[2 * i4] = inside ? I8::half2<ACT>(v0, v1) : 0u;
                                            pk[2 * i4 + 1] = inside ? I8::half2<ACT>(v2, v3) : 0u;
                                        } else {
                                            pk[2 * i4] = inside ? Pack2<T>::template run<ACT>(v0, v1) : 0u;
                                            pk[2 * i4 + 1] = inside ? Pack2<T>::template run<ACT>(v2, v3) : 0u;
                                        }
                                    }
                                    const uint32_t ch = (uint32_t)(cc >> 3);
                                    sts128(row_s + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                                    sts128(row_s + (((ch + 1) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(bars.accempty + 8 * b);
                        mbar_arrive(bars.commfull + 8 * b);
                    }
                }
                if (!ok) break;
            }
        });
    } else if (warp < kFirstDwWarp + a.n_dw_warps) {
        // ===================================================== DW warps (+ output stores)
        const int tid = (warp - kFirstDwWarp) * 32 + lane;
        const int nthr = a.n_dw_warps * 32;
        const int units = a.TH * a.ngroups * (kCt / 8);
        const bool issuer = tid == 0;
        const uint8_t *wdw_g = base_g + a.off_wdw;
        with_act(a.act2, [&](auto act_tag) {
            constexpr int ACT = decltype(act_tag)::value;
            for (int lt = 0; lt < my_tiles; lt++) {
                const int t = (int)blockIdx.x + lt * (int)gridDim.x;
                int n, ho0;
                tile_coords(a, t, n, ho0);
                bool ok = true;
                for (int j = 0; j < a.nchunks; j++) {
                    const int li = lt * a.nchunks + j, b = li & 1;
                    const bool got =
                        mbar_wait(bars.commfull + 8 * b, (uint32_t)(li >> 1) & 1u, abort_flag, a.err, lim);
                    // staging b is free once the store that last read it (item li - 2) is done
                    if (issuer) bulk_wait_group_read<1>();
                    if (named_barrier_or(2, nthr, !got)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *comm_g = base_g + a.off_comm + (uint32_t)b * a.comm_bytes;
                    const uint32_t out_s = base_s + a.off_out + (uint32_t)b * (kI8 ? kBlk / 2 : kBlk);
                    for (int u = tid; u < units; u += nthr) {
                        const int v = u & 7, rest = u >> 3;
                        const int g = rest % a.ngroups, r = rest / a.ngroups;
                        dw_unit<T, KS, S, ACT>(a, r, g, v, j, comm_g, wdw_g, s2_s, b2_s, out_s);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bars.commempty + 8 * b);   // commBuffer reusable
                    fence_proxy_async_smem();                              // staging -> TMA
                    named_barrier(2, nthr);
                    if (issuer) {
                        tma_store_4d(&a.tmap_y, out_s, j * kCt, 0, ho0, n);
                        bulk_commit_group();
                    }
                }
                if (!ok) break;
            }
        });
        if (issuer) bulk_wait_group<0>();
    }

    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, a.tmem_cols);
    }
}

// ================================================================================== host
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

uint32_t align_up(uint32_t v, uint32_t al) { return (v + al - 1) / al * al; }

struct Geometry {
    int TH, R, Q, nblk, ngroups, units, dw_warps;
};

Geometry geometry(const fcm_desc *d, int wo, int th) {
    Geometry g;
    g.TH = th;
    g.ngroups = (wo + kR - 1) / kR;
    g.R = (th - 1) * d->stride + d->ksize;
    g.Q = (g.ngroups * kR - 1) * d->stride + d->ksize;
    g.nblk = (g.R * g.Q + 127) / 128;
    g.units = th * g.ngroups * (kCt / 8);
    g.dw_warps = (g.units + 31) / 32;
    return g;
}

struct Layout {
    uint32_t off_w1, off_x, off_comm, off_out, off_wdw, off_sb, off_bar, w1_bytes, plane_bytes,
        x_stage_bytes, x_stage_stride, comm_bytes, total;
    uint32_t off_x8, plane8_bytes, x8_stage_bytes, x8_stage_stride;   // INT8 ring
    int stages, stages8;
};

Layout make_layout(const fcm_desc *d, int cm, const Geometry &g, int smem_cap) {
    Layout L{};
    const int nkb = d->c / 64;
    L.w1_bytes = (uint32_t)(nkb * cm) * 128u;
    L.plane_bytes = (uint32_t)g.nblk * kBlk;
    L.x_stage_bytes = (uint32_t)(nkb * g.R * g.Q) * 128u;   // what the TMA writes
    L.x_stage_stride = (uint32_t)nkb * L.plane_bytes;
    L.comm_bytes = align_up((uint32_t)(g.R * g.Q) * 128u, 1024);
    L.off_w1 = 0;
    L.off_comm = align_up(L.w1_bytes, 1024);
    L.off_out = L.off_comm + 2 * L.comm_bytes;
    const bool i8 = d->dtype == FCM_I8;
    // output staging (two chunks): 128-byte rows, or 64-byte rows of int8
    L.off_x8 = L.off_out + 2 * (i8 ? kBlk / 2 : kBlk);
    if (i8) {
        L.plane8_bytes = (uint32_t)(g.R * g.Q) * 64u;
        L.x8_stage_bytes = (uint32_t)nkb * L.plane8_bytes;
        L.x8_stage_stride = align_up(L.x8_stage_bytes, 1024);
        L.stages8 = 2;
    }
    L.off_x = L.off_x8 + (uint32_t)L.stages8 * L.x8_stage_stride;
    const uint32_t wdw = (uint32_t)(cm * d->ksize * d->ksize) * 2u;
    const uint32_t sb = (uint32_t)(4 * cm) * 4u;
    (void)i8;
    const uint32_t tail = align_up(wdw, 16) + align_up(sb, 16) + kBarBytes + 16 + 1024;
    int stages = kMaxStages;
    for (; stages >= 1; stages--)
        if ((int)(L.off_x + (uint32_t)stages * L.x_stage_stride + tail) <= smem_cap) break;
    L.stages = stages;
    L.off_wdw = L.off_x + (uint32_t)std::max(stages, 0) * L.x_stage_stride;
    L.off_sb = L.off_wdw + align_up(wdw, 16);
    L.off_bar = L.off_sb + align_up(sb, 16);
    L.total = L.off_bar + kBarBytes + 16 + 1024;
    return L;
}

uint32_t pow2_cols(int n) {
    uint32_t c = 32;
    while ((int)c < n) c <<= 1;
    return c;
}

}  // namespace pwdw
}  // namespace fcm

using namespace fcm::pwdw;

int fcm_pwdw_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why) {
    auto no = [&](const char *w) {
        if (why) *why = w;
        return 0;
    };
    (void)ho;
    if (d->dtype == FCM_F32) return no("fp32 runs on CUDA cores");
    // (INT8: the 1x1's fp32 partial sums stay below 256 * 128 * 128 = 2^22, exact)
    if (d->c % 64 != 0 || d->c > 256) return no("PWDW: input channels a multiple of 64, at most 256");
    if (cm % 64 != 0 || cm > 256)
        return no("PWDW: intermediate channels a multiple of 64, at most 256 (the 1x1 stage's N)");
    if (wo > 128) return no("PWDW: output width above 128");
    if (d->ksize != 1 && d->ksize != 3 && d->ksize != 5 && d->ksize != 7)
        return no("PWDW: ksize 1, 3, 5 or 7");
    const Geometry g = geometry(d, wo, 1);
    if (g.Q > 256 || g.nblk > kMaxBlk) return no("PWDW: the halo of one output row is too wide");
    return 1;
}

fcm_status fcm_pwdw_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_cap,
                         TcPlan *p) {
    // the tallest tile whose output fits the 128-row staging, whose halo fits kMaxBlk M blocks
    // and whose DW units fit the DW warps, with at least two input stages
    for (int th = std::min(ho, 128 / std::max(wo, 1)); th >= 1; th--) {
        if (d->tile_h > 0 && th != d->tile_h) continue;
        const Geometry g = geometry(d, wo, th);
        if (g.Q > 256 || g.nblk > kMaxBlk || g.dw_warps > kMaxDwWarps || th * wo > 128) continue;
        const Layout L = make_layout(d, cm, g, smem_cap);
        if (L.stages < 2) continue;
        TcPlan t;
        t.tile_h = th;
        t.tile_w = wo;
        t.in_rows = g.R;
        t.in_cols = g.Q;
        t.chunk_c = kCt;
        t.nchunks = cm / kCt;
        t.stages = L.stages;
        t.dw_warps = g.dw_warps;
        t.tiles_w = 1;
        t.tiles_h = (ho + th - 1) / th;
        t.num_tiles = (long long)d->n * t.tiles_h;
        if (t.num_tiles >= (1LL << 31)) return FCM_ERR_UNSUPPORTED;
        t.smem_bytes = (int)L.total;
        t.threads = 32 * (kFirstDwWarp + g.dw_warps);
        t.ctas = (int)std::min<long long>(t.num_tiles, num_sms);
        t.tmem_cols = (int)pow2_cols(2 * g.nblk * kCt);
        *p = t;
        return FCM_OK;
    }
    return FCM_ERR_SMEM_BUDGET;
}

// The 1x1 stage of a PWDW handle as a DW->PW handle's PW-only view: x [N,H,W,C] -> m
// [N,H,W,Cm] with the module's 1x1 weights, first norm and activation.
static fcm_handle pwdw_first_view(const fcm_handle *h) {
    fcm_handle v = *h;
    v.d.conv1 = FCM_CONV1_DEPTHWISE;
    v.d.k_out = h->cm;
    v.d.act2 = h->d.act1;
    v.cm = h->d.c;
    v.ho = h->d.h;
    v.wo = h->d.w;
    v.wp_img = h->w1_img;
    v.wp_img_bytes = h->w1_img_bytes;
    v.s2 = h->s1;
    v.b2 = h->b1;
    v.tc = TcPlan();
    v.tc.tmem_cols = (int)pow2_cols(2 * h->cm);
    v.tc2 = h->tc_lbl;   // INT8: the identity-stencil plan of this stage
    return v;
}

fcm_status fcm_pwdw_prepare(fcm_handle *h, const void *w1_host, const void *wp_host) {
    const fcm_desc &d = h->d;
    const int C = d.c, Cm = h->cm, KS = d.ksize, nkb = C / 64;
    const bool i8 = d.dtype == FCM_I8;
    // 16-bit pattern of weight i: the storage value, or for INT8 the f16 of the int8 value (exact)
    auto w16 = [&](const void *base, size_t i) -> uint16_t {
        if (i8) {
            __half hv = __float2half_rn((float)static_cast<const signed char *>(base)[i]);
            uint16_t b;
            memcpy(&b, &hv, 2);
            return b;
        }
        return static_cast<const uint16_t *>(base)[i];
    };
    // B operand of the 1x1 convolution: Cm rows (filters) over C input channels ([Cm][C])
    std::vector<uint8_t> w1((size_t)nkb * Cm * 128, 0);
    for (int j = 0; j < Cm; j++)
        for (int c = 0; c < C; c++) {
            const uint16_t b = w16(w1_host, (size_t)j * C + c);
            memcpy(&w1[fcm::tc::sw128_offset(j, c, Cm, 2)], &b, 2);
        }
    // depthwise taps ([Cm][k][k]), tap-major [k*k][Cm] (16-byte vectors of 8 channels)
    std::vector<uint16_t> wdw((size_t)KS * KS * Cm);
    for (int j = 0; j < Cm; j++)
        for (int t = 0; t < KS * KS; t++) wdw[(size_t)t * Cm + j] = w16(wp_host, (size_t)j * KS * KS + t);
    h->w1_img_bytes = w1.size();
    if (cudaMalloc(&h->w1_img, w1.size()) != cudaSuccess ||
        cudaMemcpy(h->w1_img, w1.data(), w1.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->w1dw_img, wdw.size() * 2) != cudaSuccess ||
        cudaMemcpy(h->w1dw_img, wdw.data(), wdw.size() * 2, cudaMemcpyHostToDevice) != cudaSuccess)
        return fcm_fail(FCM_ERR_CUDA, "PWDW weight images: %s", cudaGetErrorString(cudaGetLastError()));
    // the layer-by-layer depthwise stage runs the DW-only kernel over Cm channels: plan it as a
    // depthwise layer of that width
    fcm_desc dd = d;
    dd.conv1 = FCM_CONV1_DEPTHWISE;
    dd.c = Cm;
    dd.mid = 0;
    dd.k_out = 16;   // the DW-only mode has no 1x1 stage: plan with the smallest one
    dd.tile_h = dd.tile_w = 0;
    fcm_status st = fcm_tc_plan_dwpw_roles(&dd, h->ho, h->wo, Cm, h->num_sms, h->smem_optin, &h->tc2);
    if (st != FCM_OK) return fcm_fail(st, "PWDW: no tile for the layer-by-layer depthwise stage");
    if (i8) {
        // the depthwise stage's stencil offsets (its taps are wp), the identity stencil over
        // the C input channels, and the plan of the 1x1 stage alone (identity stencil, k = 1)
        if ((st = fcm_i8_constants(h, wp_host, C)) != FCM_OK) return st;
        const fcm_handle v = pwdw_first_view(h);
        const fcm_desc vd = fcm_i8_pw_desc(&v);
        if (fcm_tc_plan(&vd, d.h, d.w, C, h->num_sms, h->smem_optin, &h->tc_lbl) != FCM_OK)
            return fcm_fail(FCM_ERR_SMEM_BUDGET, "INT8 PWDW: no tile for the layer-by-layer 1x1 stage");
    }
    return FCM_OK;
}

namespace {

template <typename T, int KS, int S>
cudaError_t launch_t(const Args &a, int ctas, int threads, uint32_t smem, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_ctx{0};
    return launch_pdl(pwdw_kernel<T, KS, S>, attr_ctx, ctas, threads, smem, st, a);
}

template <typename T>
cudaError_t dispatch(const Args &a, int ks, int s, int ctas, int threads, uint32_t smem,
                     cudaStream_t st) {
#define FCM_CASE(KSV, SV) \
    if (ks == KSV && s == SV) return launch_t<T, KSV, SV>(a, ctas, threads, smem, st);
    FCM_CASE(1, 1) FCM_CASE(1, 2) FCM_CASE(3, 1) FCM_CASE(3, 2)
    FCM_CASE(5, 1) FCM_CASE(5, 2) FCM_CASE(7, 1) FCM_CASE(7, 2)
#undef FCM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_tc_pwdw(const fcm_handle *h, const void *x, void *y, cudaStream_t st) {
    const fcm_desc &d = h->d;
    const TcPlan &p = h->tc;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const Geometry g = geometry(&d, h->wo, p.tile_h);
    const Layout L = make_layout(&d, h->cm, g, h->smem_optin);
    if (L.stages < 2 || g.nblk > kMaxBlk) return cudaErrorInvalidConfiguration;
    Args a;
    memset(&a, 0, sizeof(a));
    const bool i8 = d.dtype == FCM_I8;
    const CUtensorMapDataType dt = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : d.dtype == FCM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t es = i8 ? 1 : 2;
    {
        // INT8: the box lands unswizzled in the producer's int8 ring
        cuuint64_t gdim[4] = {(cuuint64_t)d.c, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)d.c * es, (cuuint64_t)d.w * d.c * es,
                                 (cuuint64_t)d.h * d.w * d.c * es};
        cuuint32_t box[4] = {64, (cuuint32_t)g.Q, (cuuint32_t)g.R, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&a.tmap_x, dt, 4, const_cast<void *>(x), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, i8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // staging rows of 64 channels: 128 bytes (16-bit, 128B swizzle) or 64 (int8, 64B)
        cuuint64_t gdim[4] = {(cuuint64_t)h->cm, (cuuint64_t)h->wo, (cuuint64_t)h->ho,
                              (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)h->cm * es, (cuuint64_t)h->wo * h->cm * es,
                                 (cuuint64_t)h->ho * h->wo * h->cm * es};
        cuuint32_t box[4] = {64, (cuuint32_t)h->wo, (cuuint32_t)g.TH, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&a.tmap_y, dt, 4, y, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                i8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    a.w1_img = static_cast<const uint8_t *>(h->w1_img);
    a.wdw = static_cast<const uint4 *>(h->w1dw_img);
    a.s1 = h->s1;
    a.b1 = h->b1;
    a.s2 = h->s2;
    a.b2 = h->b2;
    a.err = h->d_err;
    a.wait_limit_ns = kWaitLimitNs;
    a.num_tiles = (int)p.num_tiles;
    a.tiles_per_img = p.tiles_h;
    a.nchunks = h->cm / kCt;
    a.H = d.h;
    a.W = d.w;
    a.C = d.c;
    a.Cm = h->cm;
    a.Ho = h->ho;
    a.Wo = h->wo;
    a.pad = d.pad;
    a.TH = g.TH;
    a.R = g.R;
    a.Q = g.Q;
    a.nblk = g.nblk;
    a.ngroups = g.ngroups;
    a.stages = L.stages;
    a.n_dw_warps = g.dw_warps;
    a.act1 = d.act1;
    a.act2 = d.act2;
    a.tmem_cols = (uint32_t)p.tmem_cols;
    a.idesc = idesc_f16(d.dtype == FCM_BF16, 128, kCt);   // INT8: f16 operands
    a.w1_bytes = L.w1_bytes;
    a.plane_bytes = L.plane_bytes;
    a.x_stage_bytes = L.x_stage_bytes;
    a.x_stage_stride = L.x_stage_stride;
    a.comm_bytes = L.comm_bytes;
    a.off_w1 = L.off_w1;
    a.off_x = L.off_x;
    a.off_comm = L.off_comm;
    a.off_out = L.off_out;
    a.off_wdw = L.off_wdw;
    a.off_sb = L.off_sb;
    a.off_bar = L.off_bar;
    a.off_x8 = L.off_x8;
    a.plane8_bytes = L.plane8_bytes;
    a.x8_stage_bytes = L.x8_stage_bytes;
    a.x8_stage_stride = L.x8_stage_stride;
    a.stages8 = L.stages8;
    const int threads = 32 * (kFirstDwWarp + g.dw_warps);
    const int ctas = std::min(a.num_tiles, h->num_sms);
    if (i8) return dispatch<int8_t>(a, d.ksize, d.stride, ctas, threads, L.total, st);
    if (d.dtype == FCM_F16) return dispatch<__half>(a, d.ksize, d.stride, ctas, threads, L.total, st);
    return dispatch<__nv_bfloat16>(a, d.ksize, d.stride, ctas, threads, L.total, st);
}

// Layer by layer on the DW->PW kernels: the 1x1 convolution x -> m [N,H,W,Cm] is their
// PW-only mode with this module's 1x1 weights, norm and activation; the depthwise one m -> y
// is their DW-only mode over Cm channels with the second norm and activation.
cudaError_t launch_tc_pwdw_first(const fcm_handle *h, const void *x, void *m, cudaStream_t st) {
    const fcm_handle v = pwdw_first_view(h);   // a view with the 1x1 layer's operands
    return launch_tc_pw(&v, x, m, st);
}

cudaError_t launch_tc_pwdw_second(const fcm_handle *h, const void *m, void *y, cudaStream_t st) {
    fcm_handle v = *h;   // a view with the depthwise layer's operands
    v.d.conv1 = FCM_CONV1_DEPTHWISE;
    v.d.c = h->cm;
    v.d.mid = 0;
    v.d.k_out = h->cm;
    v.d.act1 = h->d.act2;
    v.s1 = h->s2;
    v.b1 = h->b2;
    v.tc = h->tc2;
    return launch_tc_dwpw(&v, FCM_MODE_CONV1_ONLY, m, y, st);
}
