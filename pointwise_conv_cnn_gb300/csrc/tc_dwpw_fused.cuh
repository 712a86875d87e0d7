// tc_dwpw_fused.cuh -- the fused depthwise -> pointwise module on tcgen05 with worker warps
// that run both CUDA-core roles (the DW stencil and the 1x1's epilogue).
//
// The FCM of "Fusing Depthwise and Pointwise Convolutions for Efficient Inference on GPUs"
// (section III-B: weights prefetched once, the first layer's conv-norm-activation written to
// a shared commBuffer, the second layer reading it and writing the OFMs once; section II-D:
// a DWPW tile holds all channels of its pixels).  Here the commBuffer is the A operand of a
// tcgen05.mma 1x1 GEMM (128-byte swizzled, K-major), the accumulator lives in tensor memory,
// and the same warps that fill the commBuffer also drain the accumulator:
//
//   warp 0        TMA producer: per output tile and 64-channel chunk, the input halo box
//                 ((th-1)*s+k rows x (tw-1)*s+k columns x 64 channels, zero-filled outside
//                 the image, i.e. the zero padding) into a ring of stages
//   warp 1        TMEM owner and MMA issuer: per chunk, 4 x kind::f16 MMAs (M = 128, N = K,
//                 K = 16) as soon as the chunk of the A tile is complete
//   warps 2..     workers.  Iteration t: the DW stencil of tile t for the worker's channel
//                 chunk, written into the A tile (double-buffered when it fits), then the
//                 epilogue of tile t-1 for the worker's TMEM lane quadrant (warp % 4) and
//                 column range: tcgen05.ld -> scale/bias/act -> 16-bit (or int8) -> the
//                 worker's own swizzled staging block -> its own TMA tensor stores.
//
// Giving every worker both roles keeps the issue slots of all four schedulers busy with one
// mix of work; with dedicated epilogue warps (one per scheduler) the epilogue fell behind
// the stencil warps and stalled the pipeline.  The epilogue needs no barrier across warps:
// each worker stores exactly the pixels and channels it converted.
//
// Output tile: th rows x tw columns of output pixels, th * tw = 128 (the MMA M).  Each TMEM
// lane quadrant q holds a qh x qw rectangle of pixels (qw * qh = 32), quadrants laid
// out nqx across and 4 / nqx down, so that one quadrant's rows of the accumulator are one
// TMA box of the NHWC output.  GEMM row of pixel (r, c):
//     q = (r / qh) * nqx + c / qw,   row = 32 q + (r % qh) * qw + c % qw.
// Pixels beyond the image are computed from zero-filled input and clipped by the stores.
//
// Every mbarrier wait is bounded; a timeout sets the device error word, raises a CTA-wide
// abort flag, and the kernel drains its copies and MMAs before releasing TMEM.
//
// T is the storage type: __half, __nv_bfloat16, or int8_t (the INT8 FCM of section III-B,
// computed exactly on the 16-bit paths as in the other DW -> PW kernels).
#pragma once

#include <atomic>

#include "tc_dwpw.cuh"

namespace fcm {
namespace tc {

constexpr int kFMaxWorkers = 14;
constexpr int kFThreads = 32 * (2 + kFMaxWorkers);   // 576 threads: up to 112 registers each
constexpr int kFMaxStages = 6;
constexpr int kFMaxChunks = 4;                       // channels (padded) <= 256
constexpr int kFUnitPx = 4;                          // output pixels per DW work unit
constexpr int kFSmemMax = 227 * 1024;                // dynamic shared memory a block may use

struct FArgs {
    CUtensorMap tmap_x;      // x: 4-D (C, W, H, N), box (64, in_cols, in_rows, 1), no swizzle
    CUtensorMap tmap_y;      // y: 4-D (K, Wo, Ho, N), box (128 / esize, qw, qh, 1), 128-byte swizzle
    const uint8_t *wp_img;   // B operand: K rows x Cp (64-channel blocks of 128-byte swizzled rows)
    const uint4 *wdw;        // DW taps [k*k][Cp], 16-bit (f16 for INT8), zero beyond C
    const float *s1, *b1, *s2, *b2;
    const float *q1;         // INT8: 1152 * sum of each channel's taps
    unsigned *err;
    unsigned long long wait_limit_ns;
    int num_tiles;
    int C, Cp, K, Ho, Wo, pad;
    int tiles_w, tiles_per_img;
    int th, tw, qw, qh, nqx;
    int ngroups;             // DW units per tile row: ceil(min(tw, Wo) / 4)
    int in_rows, in_cols;
    int nchunks, stages, nw, abufs;
    int sbufs;               // output staging buffers (2: a quadrant's stores overlap the next tile)
    int nblk;                // 128-byte staging blocks per pixel row: ceil(K * esize / 128)
    int lg_qw, lg_qh;        // log2 of qw and qh (powers of two)
    uint32_t mg_ngroups, mg_uc;   // multiply-high reciprocals of ngroups and of the units per
                                  // chunk (fdiv below); 0 for a divisor of 1
    int step_n, step_ty, step_tx; // the grid size as (images, tile rows, tile columns)
    int tiles_h;
    int act1, act2;
    uint32_t tmem_cols, idesc, wp_img_bytes, in_stage_bytes, in_stage_stride;
    uint32_t off_b, off_a, a_buf_bytes, off_out, off_in, off_wdw, off_sb, off_bar;
};

struct FBars {
    uint32_t full, empty, afull, aempty, accfull, accempty, wbar, drain;
    __device__ FBars(uint32_t base) {
        full = base;
        empty = full + 8 * kFMaxStages;
        afull = empty + 8 * kFMaxStages;          // [2][kFMaxChunks]
        aempty = afull + 8 * 2 * kFMaxChunks;     // [2][kFMaxChunks]
        accfull = aempty + 8 * 2 * kFMaxChunks;   // [2]
        accempty = accfull + 16;                  // [2]
        wbar = accempty + 16;
        drain = wbar + 8;
    }
};
constexpr uint32_t kFBarBytes = 8 * (2 * kFMaxStages + 4 * kFMaxChunks + 4 + 2) + 16;

// Launch dwpw_fused_kernel<T, KS, S> (instantiated in tc_dwpw_fused_inst_*.cu).
template <typename T, int KS, int S>
cudaError_t launch_fused(const FArgs &a, int ctas, int threads, uint32_t smem, cudaStream_t st);

#ifdef FCM_FUSED_KERNEL_BODY

// x / d for 0 <= x < 2^16 and 1 <= d < 2^16 by a multiply-high with m = ceil(2^32 / d) (the
// error of the reciprocal stays below 1 / d over that range); m = 0 stands for d = 1.
__device__ __forceinline__ uint32_t fdiv(uint32_t x, uint32_t m) { return m ? __umulhi(x, m) : x; }

// A CTA's tiles t = blockIdx.x, blockIdx.x + gridDim.x, ... as (image, tile row, tile column),
// advanced by additions: the grid size is passed pre-split into the same three units.
struct TileIter {
    int n, ty, tx;
    __device__ __forceinline__ void init(const FArgs &a, int t) {
        n = t / a.tiles_per_img;
        const int rem = t - n * a.tiles_per_img;
        ty = rem / a.tiles_w;
        tx = rem - ty * a.tiles_w;
    }
    __device__ __forceinline__ void next(const FArgs &a) {
        tx += a.step_tx;
        if (tx >= a.tiles_w) {
            tx -= a.tiles_w;
            ty++;
        }
        ty += a.step_ty;
        if (ty >= a.tiles_h) {
            ty -= a.tiles_h;
            n++;
        }
        n += a.step_n;
    }
};

// Position (stage, phase parity) in the ring of input stages, kept as a running counter.
struct RingPos {
    int s;
    uint32_t ph;
    __device__ __forceinline__ void advance(int by, int stages) {
        s += by;
        while (s >= stages) {
            s -= stages;
            ph ^= 1u;
        }
    }
};


__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 ldsf4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

// Shared-memory addresses (32-bit) of the per-CTA constants.
struct FSmem {
    uint32_t wdw, s1, b1, q1, s2, b2;
    __device__ __forceinline__ FSmem(const FArgs &a, uint32_t base_s) {
        wdw = base_s + a.off_wdw;
        s1 = base_s + a.off_sb;
        b1 = s1 + 4u * (uint32_t)a.Cp;
        q1 = b1 + 4u * (uint32_t)a.Cp;
        s2 = q1 + 4u * (uint32_t)a.Cp;
        b2 = s2 + 4u * (uint32_t)a.K;
    }
};

// One DW work unit: 4 consecutive output pixels of tile row r (columns oc0 .. oc0+3) x 8
// channels (c_glob .. c_glob+7).  Products of 16-bit inputs and taps are exact and summed in
// fp32 (fma.rn.f32.{f16,bf16}); then scale/bias/act, rounding to the A operand's 16-bit type
// and one swizzled 16-byte store per pixel into the A tile (GEMM rows row0 .. row0+3).  The
// stage holds 64 channels per pixel, so every input vector sits at a compile-time offset from
// its row's start.  All addresses are 32-bit shared-memory addresses.
template <typename T, int KS, int S, int ACT>
__device__ __forceinline__ void fused_unit(uint32_t x_s, uint32_t row_bytes, uint32_t wdw_s,
                                           uint32_t tap_stride, const FSmem &sm, int c_glob,
                                           uint32_t a_chunk_s, uint32_t row0, uint32_t v,
                                           unsigned *a_err) {
    (void)a_err;
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    using TM = typename std::conditional<kI8, __half, T>::type;
    constexpr uint32_t kPx = 64u * (uint32_t)sizeof(T);   // bytes of one stage pixel

    float acc[kFUnitPx][8];
    if constexpr (kI8) {
        const float4 q0 = ldsf4(sm.q1 + 4u * (uint32_t)c_glob);
        const float4 q1 = ldsf4(sm.q1 + 4u * (uint32_t)c_glob + 16u);
        const float qq[8] = {-q0.x, -q0.y, -q0.z, -q0.w, -q1.x, -q1.y, -q1.z, -q1.w};
#pragma unroll
        for (int jj = 0; jj < kFUnitPx; jj++)
#pragma unroll
            for (int c = 0; c < 8; c++) acc[jj][c] = qq[c];
    } else {
#pragma unroll
        for (int jj = 0; jj < kFUnitPx; jj++)
#pragma unroll
            for (int c = 0; c < 8; c++) acc[jj][c] = 0.0f;
    }

#pragma unroll
    for (int i = 0; i < KS; i++) {
        uint4 w[KS];
#pragma unroll
        for (int t = 0; t < KS; t++) w[t] = lds128(wdw_s + (uint32_t)(i * KS + t) * tap_stride);
        const uint32_t xr = x_s + (uint32_t)i * row_bytes;
#pragma unroll
        for (int qq = 0; qq < (kFUnitPx - 1) * S + KS; qq++) {
            uint4 x;
            if constexpr (kI8) {
                const uint2 x8 = lds64(xr + (uint32_t)qq * kPx);
                I8::widen4(x8.x, x.x, x.y);
                I8::widen4(x8.y, x.z, x.w);
            } else {
                x = lds128(xr + (uint32_t)qq * kPx);
            }
#pragma unroll
            for (int jj = 0; jj < kFUnitPx; jj++) {
                const int t = qq - jj * S;
                if (t >= 0 && t < KS) {
                    Fma16<TM>::fma2(acc[jj][0], acc[jj][1], x.x, w[t].x);
                    Fma16<TM>::fma2(acc[jj][2], acc[jj][3], x.y, w[t].y);
                    Fma16<TM>::fma2(acc[jj][4], acc[jj][5], x.z, w[t].z);
                    Fma16<TM>::fma2(acc[jj][6], acc[jj][7], x.w, w[t].w);
                }
            }
        }
    }
    const float4 sc0 = ldsf4(sm.s1 + 4u * (uint32_t)c_glob);
    const float4 sc1 = ldsf4(sm.s1 + 4u * (uint32_t)c_glob + 16u);
    const float4 bi0 = ldsf4(sm.b1 + 4u * (uint32_t)c_glob);
    const float4 bi1 = ldsf4(sm.b1 + 4u * (uint32_t)c_glob + 16u);
    const float sc[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
    const float bi[8] = {bi0.x, bi0.y, bi0.z, bi0.w, bi1.x, bi1.y, bi1.z, bi1.w};
    FCM_DCHECK(row0 + kFUnitPx <= (uint32_t)kTileM, a_err, 11, row0);   // 11: A-tile rows
#pragma unroll
    for (int jj = 0; jj < kFUnitPx; jj++) {
        const uint32_t row = row0 + (uint32_t)jj;
        const uint32_t dst = a_chunk_s + row * 128u + ((v ^ (row & 7u)) << 4);
        if constexpr (kI8) {
            float y[8];
#pragma unroll
            for (int c = 0; c < 8; c++) y[c] = fmaf(sc[c], acc[jj][c], bi[c]);
            sts128(dst, I8::half2<ACT>(y[0], y[1]), I8::half2<ACT>(y[2], y[3]),
                   I8::half2<ACT>(y[4], y[5]), I8::half2<ACT>(y[6], y[7]));
        } else {
            uint32_t pk[4];
#pragma unroll
            for (int c = 0; c < 4; c++)
                pk[c] = Pack2<T>::template run<ACT>(fmaf(sc[2 * c], acc[jj][2 * c], bi[2 * c]),
                                                    fmaf(sc[2 * c + 1], acc[jj][2 * c + 1], bi[2 * c + 1]));
            sts128(dst, pk[0], pk[1], pk[2], pk[3]);
        }
    }
}

// Scale/bias/act of 16 accumulator columns (c0 .. c0+15 of the output channels) of this
// thread's pixel, packed into 16-bit pairs (8 words) or int8 quads (4 words).
template <typename T, int ACT>
__device__ __forceinline__ void fused_convert16(const uint32_t (&rr)[16], int c0, const FSmem &sm,
                                                uint32_t (&pk)[8]) {
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    using TS = typename std::conditional<kI8, __half, T>::type;
#pragma unroll
    for (int i4 = 0; i4 < 4; i4++) {
        const float4 sc = ldsf4(sm.s2 + 4u * (uint32_t)(c0 + 4 * i4));
        const float4 bi = ldsf4(sm.b2 + 4u * (uint32_t)(c0 + 4 * i4));
        const float y0 = fmaf(sc.x, __uint_as_float(rr[4 * i4]), bi.x);
        const float y1 = fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), bi.y);
        const float y2 = fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), bi.z);
        const float y3 = fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), bi.w);
        if constexpr (kI8) {
            pk[i4] = I8::bytes4<ACT>(y0, y1, y2, y3);
        } else {
            pk[2 * i4] = Pack2<TS>::template run<ACT>(y0, y1);
            pk[2 * i4 + 1] = Pack2<TS>::template run<ACT>(y2, y3);
        }
    }
}

template <typename T, int KS, int S>
__global__ void __launch_bounds__(kFThreads, 1) dwpw_fused_kernel(const __grid_constant__ FArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base_g = smem_raw + (base_s - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    constexpr uint32_t kEs = (uint32_t)sizeof(T);

    float *s1_g = reinterpret_cast<float *>(base_g + a.off_sb);
    float *b1_g = s1_g + a.Cp;
    float *q1_g = b1_g + a.Cp;
    float *s2_g = q1_g + a.Cp;
    float *b2_g = s2_g + a.K;
    FBars bars(base_s + a.off_bar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_g + a.off_bar + kFBarBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base_g + a.off_bar + kFBarBytes + 4);
    // the stencil's work units, chunk-major: chunk j holds uc units (8-channel vector x 4-pixel
    // group), padded to a multiple of 32 so that a warp's 32 consecutive units share a chunk
    const int npg = a.th * a.ngroups;
    const int npg4 = (npg + 3) & ~3;
    const int uc = 8 * npg4;
    const uint32_t rounds_per_chunk = (uint32_t)(uc / 32);   // warp-rounds that fill one chunk

    // ---- prologue: taps, scales and biases to shared memory (zero beyond the real channels),
    // the A tiles zeroed (rows no unit writes stay zero), barriers, TMEM
    {
        uint4 *wdw_s = reinterpret_cast<uint4 *>(base_g + a.off_wdw);
        const int nw16 = KS * KS * a.Cp / 8;
        for (int i = threadIdx.x; i < nw16; i += blockDim.x) wdw_s[i] = a.wdw[i];
        for (int i = threadIdx.x; i < a.Cp; i += blockDim.x) {
            const bool in = i < a.C;
            s1_g[i] = in ? a.s1[i] : 0.0f;
            b1_g[i] = in ? a.b1[i] : 0.0f;
            q1_g[i] = (kI8 && in) ? a.q1[i] : 0.0f;
        }
        for (int i = threadIdx.x; i < a.K; i += blockDim.x) {
            s2_g[i] = a.s2[i];
            b2_g[i] = a.b2[i];
        }
        uint4 *az = reinterpret_cast<uint4 *>(base_g + a.off_a);
        const int na = (int)(a.abufs * a.a_buf_bytes / 16u);
        for (int i = threadIdx.x; i < na; i += blockDim.x) az[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();   // the zeros are read by the tensor core
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; s++) {
            mbar_init(bars.full + 8 * s, 1);
            mbar_init(bars.empty + 8 * s, rounds_per_chunk);
        }
        for (int b = 0; b < 2; b++)
            for (int j = 0; j < a.nchunks; j++) {
                mbar_init(bars.afull + 8 * (b * kFMaxChunks + j), rounds_per_chunk);
                mbar_init(bars.aempty + 8 * (b * kFMaxChunks + j), 1);
            }
        // the accumulator is read by the workers that own output blocks: per lane quadrant
        // min(its workers, blocks)
        uint32_t readers = 0;
        for (int qq = 0; qq < 4; qq++) {
            const int first = qq >= 2 ? qq : qq + 4;
            const int wqq = (a.nw + 1 - first) / 4 + 1;
            readers += (uint32_t)(wqq < a.nblk ? wqq : a.nblk);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bars.accfull + 8 * b, 1);
            mbar_init(bars.accempty + 8 * b, readers);
        }
        mbar_init(bars.wbar, 1);
        mbar_init(bars.drain, 1);
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

    if (warp == 0) {
        // ===================================================== TMA producer
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(bars.wbar, a.wp_img_bytes);
            bulk_load(base_s + a.off_b, a.wp_img, a.wp_img_bytes, bars.wbar);
            tma_prefetch_desc(&a.tmap_x);
        }
        pdl_wait();
        int it = 0;
        RingPos rp{0, 0u};
        TileIter ti;
        ti.init(a, blockIdx.x);
        for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, ti.next(a)) {
            const int ho0 = ti.ty * a.th, wo0 = ti.tx * a.tw;
            for (int j = 0; j < a.nchunks; j++, it++, rp.advance(1, a.stages)) {
                if (!mbar_wait(bars.empty + 8 * rp.s, rp.ph ^ 1u, abort_flag, a.err, lim)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = base_s + a.off_in + (uint32_t)rp.s * a.in_stage_stride;
                    mbar_arrive_expect_tx(bars.full + 8 * rp.s, a.in_stage_bytes);
                    tma_load_4d(dst, &a.tmap_x, bars.full + 8 * rp.s, j * 64, wo0 * S - a.pad,
                                ho0 * S - a.pad, ti.n);
                }
                __syncwarp();
            }
        }
        if (!ok) {
            // every copy this warp issued lands before the CTA exits (load i went to stage
            // i % stages)
            volatile int no_abort = 0;
            for (int s = 0; s < a.stages && s < it; s++) {
                const int issued = (it - 1 - s) / a.stages + 1;
                mbar_wait(bars.full + 8 * s, (uint32_t)(issued - 1) & 1u, &no_abort, a.err, lim);
            }
            mbar_wait(bars.wbar, 0, &no_abort, a.err, lim);
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        bool ok = mbar_wait(bars.wbar, 0, abort_flag, a.err, lim);
        const uint32_t b_s = base_s + a.off_b;
        const uint64_t b_desc0 = sw128_kmajor_desc(b_s);
        int lt = 0;
        for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, lt++) {
            const int ab = lt & 1;
            const int buf = a.abufs == 2 ? (lt & 1) : 0;
            const uint32_t fill_par = (uint32_t)(a.abufs == 2 ? (lt >> 1) : lt) & 1u;
            if (!mbar_wait(bars.accempty + 8 * ab, ((uint32_t)(lt >> 1) & 1u) ^ 1u, abort_flag, a.err,
                           lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)ab * (a.tmem_cols >> 1);
            const uint64_t a_desc0 = sw128_kmajor_desc(base_s + a.off_a + (uint32_t)buf * a.a_buf_bytes);
            for (int j = 0; j < a.nchunks; j++) {
                const int bj = buf * kFMaxChunks + j;
                if (!mbar_wait(bars.afull + 8 * bj, fill_par, abort_flag, a.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) {
                        const int k16 = j * 4 + kk;
                        mma_f16(d_tmem, desc_advance(a_desc0, k16_offset(k16, kTileM)),
                                desc_advance(b_desc0, k16_offset(k16, a.K)), a.idesc,
                                k16 > 0 ? 1u : 0u);
                    }
                    mma_commit(bars.aempty + 8 * bj);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (lane == 0) mma_commit(bars.accfull + 8 * ab);
            __syncwarp();
        }
        if (!ok && lane == 0) {
            volatile int no_abort = 0;
            mma_commit(bars.drain);
            mbar_wait(bars.drain, 0, &no_abort, a.err, lim);
        }
        __syncwarp();
    } else {
        // ===================================================== workers
        const int w = warp - 2;
        const int total_u = a.nchunks * uc;
        const int stride_u = 32 * a.nw;
        const FSmem sm(a, base_s);
        const uint32_t row_bytes = (uint32_t)a.in_cols * 64u * kEs;   // one stage row
        const uint32_t tap_stride = 2u * (uint32_t)a.Cp;              // bytes between taps
        // epilogue role: TMEM lane quadrant q (the hardware ties warp w to lanes 32 (w % 4) ..).
        // The quadrant's output is cut into 128-byte blocks per pixel row (128 / esize
        // channels); its workers (warps first_q, first_q + 4, ...) own whole blocks, round
        // robin, and each converts its blocks into its own 128-byte-swizzled staging and issues
        // their TMA stores itself: no synchronisation between workers in the epilogue.
        const int q = warp & 3;
        const int first_q = q >= 2 ? q : q + 4;
        const int wq = (a.nw + 1 - first_q) / 4 + 1;
        const int wi = (warp - first_q) / 4;
        const bool reader = wi < a.nblk;   // owns at least one block
        constexpr int kLgCb = kI8 ? 7 : 6;                 // log2 of channels per staging block
        const uint32_t q_bytes = (uint32_t)a.nblk * 4096u;  // one quadrant's staging blocks
        const uint32_t swz = (uint32_t)lane & 7u;
        const uint32_t stage_q = base_s + a.off_out + (uint32_t)q * q_bytes + (uint32_t)lane * 128u;
        const uint32_t taddr_q = tmem_base + ((uint32_t)(q * 32) << 16);
        const int qx = q % a.nqx, qy = q / a.nqx;

        int lt = 0;
        RingPos rp0{0, 0u};   // ring position of chunk 0 of the current tile
        TileIter ti;          // the tile whose epilogue comes next
        ti.init(a, blockIdx.x);
        for (int t = blockIdx.x;; t += gridDim.x, lt++) {
            const bool have = t < a.num_tiles;
            if (have) {
                // ---------------- stencil of tile t -> A tile, in rounds of 32 units
                const int buf = a.abufs == 2 ? (lt & 1) : 0;
                const uint32_t fill_par = (uint32_t)(a.abufs == 2 ? (lt >> 1) : lt) & 1u;
                bool ok = true;
                for (int ub = 32 * w; ub < total_u; ub += stride_u) {
                    const int j = (int)fdiv((uint32_t)ub, a.mg_uc);   // the round's chunk (warp-uniform)
                    RingPos rp = rp0;
                    rp.advance(j, a.stages);
                    const int bj = buf * kFMaxChunks + j;
                    if (!mbar_wait(bars.full + 8 * rp.s, rp.ph, abort_flag, a.err, lim) ||
                        !mbar_wait(bars.aempty + 8 * bj, fill_par ^ 1u, abort_flag, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    const int s = rp.s;
                    const int ui = ub + lane - j * uc;   // unit within the chunk
                    const int v = ui & 7, pg = ui >> 3;
                    if (pg < npg) {
                        const int r = (int)fdiv((uint32_t)pg, a.mg_ngroups);
                        const int oc0 = (pg - r * a.ngroups) * kFUnitPx;
                        const int c_glob = j * 64 + v * 8;
                        // the unit's first input vector in the stage, its taps, its A-tile rows
                        const uint32_t x_s = base_s + a.off_in + (uint32_t)s * a.in_stage_stride +
                                             ((uint32_t)(r * S) * (uint32_t)a.in_cols + (uint32_t)(oc0 * S)) *
                                                 (64u * kEs) +
                                             (uint32_t)v * 8u * kEs;
                        const uint32_t a_chunk_s = base_s + a.off_a + (uint32_t)buf * a.a_buf_bytes +
                                                   (uint32_t)j * (kTileM * 128u);
                        const int qd = (r >> a.lg_qh) * a.nqx + (oc0 >> a.lg_qw);
                        const uint32_t row0 = (uint32_t)((qd << 5) + ((r & ((1 << a.lg_qh) - 1)) << a.lg_qw) +
                                                         (oc0 & ((1 << a.lg_qw) - 1)));
                        // 10: the unit's last input vector lies inside its stage
                        FCM_DCHECK((uint32_t)((r * S + KS - 1) * a.in_cols + oc0 * S + (kFUnitPx - 1) * S + KS) *
                                           (64u * kEs) <= a.in_stage_bytes,
                                   a.err, 10, pg);
                        with_act(a.act1, [&](auto act_tag) {
                            constexpr int ACT1 = decltype(act_tag)::value;
                            fused_unit<T, KS, S, ACT1>(x_s, row_bytes, sm.wdw + 2u * (uint32_t)c_glob,
                                                       tap_stride, sm, c_glob, a_chunk_s, row0,
                                                       (uint32_t)v, a.err);
                        });
                    }
                    fence_proxy_async_smem();   // A visible to the tensor core
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(bars.empty + 8 * s);
                        mbar_arrive(bars.afull + 8 * bj);
                    }
                }
                if (!ok) break;
                rp0.advance(a.nchunks, a.stages);
            }
            if (lt >= 1 && reader) {
                // ---------------- epilogue of the previous tile
                const int plt = lt - 1, ab = plt & 1;
                const int sb = a.sbufs == 2 ? (plt & 1) : 0;   // staging buffer of tile plt
                if (!mbar_wait(bars.accfull + 8 * ab, (uint32_t)(plt >> 1) & 1u, abort_flag, a.err,
                               lim))
                    break;
                tc_fence_after();
                // this warp's stores of tile plt - sbufs have read the staging buffer
                if (lane == 0) {
                    if (a.sbufs == 2)
                        bulk_wait_group_read<1>();
                    else
                        bulk_wait_group_read<0>();
                }
                __syncwarp();
                const uint32_t tcol = taddr_q + (uint32_t)ab * (a.tmem_cols >> 1);
                const uint32_t stage_b = stage_q + (uint32_t)sb * 4u * q_bytes;
                with_act(a.act2, [&](auto act_tag) {
                    constexpr int ACT2 = decltype(act_tag)::value;
                    // 16 accumulator columns from c0 -> their 16-byte chunks of the staging row
                    auto emit16 = [&](const uint32_t (&rr)[16], int c0) {
                        uint32_t pk[8];
                        FCM_DCHECK(c0 + 16 <= a.K && (c0 >> kLgCb) < a.nblk, a.err, 12, c0);   // 12
                        fused_convert16<T, ACT2>(rr, c0, sm, pk);
                        const uint32_t blk = stage_b + (uint32_t)(c0 >> kLgCb) * 4096u;
                        const uint32_t ch = ((uint32_t)(c0 & ((1 << kLgCb) - 1)) * kEs) >> 4;
                        sts128(blk + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                        if (!kI8) sts128(blk + (((ch + 1u) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
                    };
#pragma unroll 1
                    for (int b = wi; b < a.nblk; b += wq) {
                        const int c_end = min(a.K, (b + 1) << kLgCb);
                        // two TMEM loads per wait
#pragma unroll 1
                        for (int c0 = b << kLgCb; c0 < c_end; c0 += 32) {
                            uint32_t ra[16], rb2[16];
                            const bool two = c0 + 16 < c_end;
                            tmem_ld16(tcol + (uint32_t)c0, ra);
                            if (two) tmem_ld16(tcol + (uint32_t)(c0 + 16), rb2);
                            tmem_ld_wait(ra, rb2);
                            emit16(ra, c0);
                            if (two) emit16(rb2, c0 + 16);
                        }
                    }
                });
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.accempty + 8 * ab);   // TMEM buffer reusable
                fence_proxy_async_smem();                              // staging visible to TMA
                __syncwarp();
                if (lane == 0) {
                    const int ho0 = ti.ty * a.th + qy * a.qh, wo0 = ti.tx * a.tw + qx * a.qw;
                    for (int b = wi; b < a.nblk; b += wq)
                        tma_store_4d(&a.tmap_y, stage_b - (uint32_t)lane * 128u + (uint32_t)b * 4096u,
                                     b << kLgCb, wo0, ho0, ti.n);
                    bulk_commit_group();
                }
                __syncwarp();
                ti.next(a);
            }
            if (!have) break;
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, a.tmem_cols);
    }
}

template <typename T, int KS, int S>
cudaError_t launch_fused(const FArgs &a, int ctas, int threads, uint32_t smem, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_ctx{0};
    return launch_pdl(dwpw_fused_kernel<T, KS, S>, attr_ctx, ctas, threads, smem, st, a);
}

#endif  // FCM_FUSED_KERNEL_BODY

}  // namespace tc
}  // namespace fcm
