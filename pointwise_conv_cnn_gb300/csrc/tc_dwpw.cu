// tc_dwpw.cu -- the tensor-core (tcgen05) depthwise -> pointwise kernels for sm_103a.
//
// One persistent, warp-specialised kernel template serves three modes:
//   FUSED   halo tile (TMA) -> DW stencil on CUDA cores -> A tile in shared memory ->
//           1x1 conv as tcgen05.mma into TMEM -> epilogue (scale/bias/act) -> y, stored once
//   DWONLY  halo tile (TMA) -> DW stencil -> intermediate m in HBM (layer-by-layer baseline)
//   PWONLY  m tile (TMA, 128B-swizzled) -> tcgen05.mma -> epilogue -> y (layer-by-layer baseline)
//
// This is the FCM structure of "Fusing Depthwise and Pointwise Convolutions for Efficient
// Inference on GPUs" (section III-B: weights prefetched, the first layer's
// conv-norm-activation written to a shared commBuffer, the second layer reading it and
// writing the OFMs once), re-designed for Blackwell: the commBuffer IS the A operand of the
// tensor-core GEMM, written directly in the 128-byte-swizzled K-major layout tcgen05.mma
// reads (bank-conflict free for the writers, section III-B's concern), and the accumulator
// lives in tensor memory.  Each output tile covers all channels (section II-D's rule for
// DWPW), so no block ever needs another block's intermediate.
//
// Warp roles (persistent CTA, one per SM, static round-robin over output tiles):
//   warp 0      TMA producer: input halo tiles (channel chunks) into a ring of stages
//   warp 1      TMEM owner and MMA issuer (one lane issues)
//   warps 2-5   epilogue: TMEM -> registers -> scale/bias/act -> global (warp w reads TMEM
//               lanes 32*(w%4) .. +31)
//   warps 6..   DW warps: stencil over a stage, result into the A tile (or HBM in DWONLY)
// Synchronisation is by mbarriers only; every wait is bounded (about one second) and a
// timeout sets the device error word, raises a CTA-wide abort flag and drains in-flight
// copies and MMAs before TMEM is released.
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "fcm_internal.h"
#include "tc_common.cuh"

namespace fcm {
namespace tc {

constexpr int kEpiWarps = 4;
constexpr int kFirstDwWarp = 2 + kEpiWarps;
constexpr int kMaxDwWarps = 10;   // 16 warps in all: up to 128 registers a thread
constexpr int kMaxThreads = 32 * (kFirstDwWarp + kMaxDwWarps);
// Chunk-bound DW warps (each warp serves one channel chunk and keeps its taps in registers):
// up to 14 DW warps, 20 in all, 96 registers a thread.
constexpr int kMaxDwWarpsBound = 14;
constexpr int kMaxThreadsBound = 32 * (kFirstDwWarp + kMaxDwWarpsBound);
constexpr int kR = 4;          // output pixels per DW work unit (along W)
constexpr int kTileM = 128;    // MMA M: pixels per output tile (padded)
constexpr int kMaxStages = 8;
constexpr int kMaxChunks = 16;

enum Mode { FUSED = 0, DWONLY = 1, PWONLY = 2 };

struct Args {
    CUtensorMap tmap;          // x (FUSED/DWONLY: 4-D C,W,H,N) or m (PWONLY: 2-D C,P)
    CUtensorMap tmap_out;      // y: 4-D K,Wo,Ho,N box (64,tile_w,tile_h,1) or 2-D K,P box (64,128)
    void *out;                 // m for DWONLY (direct stores)
    const uint8_t *wp_img;     // B operand image (K rows, swizzled, K-major)
    const uint4 *wdw;          // DW taps, storage dtype, [k*k][C/8] x 8 channels
    const float *s1, *b1, *s2, *b2;
    unsigned *err;
    unsigned long long wait_limit_ns;
    int num_tiles;
    long long P;               // PWONLY: pixel count
    int N, H, W, C, K, Ho, Wo, pad;
    int tile_h, tile_w, tiles_w, tiles_per_img, ngroups;
    int in_rows, in_cols;
    int chunk_c, nchunks, stages, n_dw_warps;
    int dw_per_chunk;          // chunk-bound DW warps per chunk (0: every DW warp serves every chunk)
    int act1, act2;
    uint32_t tmem_cols, idesc, wp_img_bytes, in_stage_bytes;
    uint32_t off_b, off_a, off_in, in_stage_stride, off_out, off_wdw, off_sb, off_bar;
    int out_bufs;              // output staging tiles (2: a tile's stores overlap the next tile)
    uint32_t out_buf_bytes;
};

struct Bars {
    uint32_t full, empty, afull, aempty, accfull, accempty, wbar, drain;
    __device__ Bars(uint32_t base) {
        full = base;
        empty = full + 8 * kMaxStages;
        afull = empty + 8 * kMaxStages;
        aempty = afull + 8 * kMaxChunks;
        accfull = aempty + 8 * kMaxChunks;
        accempty = accfull + 16;
        wbar = accempty + 16;
        drain = wbar + 8;
    }
};
constexpr uint32_t kBarBytes = 8 * (2 * kMaxStages + 2 * kMaxChunks + 4 + 2) + 16;
constexpr int kOutBlock = kTileM * 128;   // bytes of one 64-channel block of the output stage

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Where one DW work unit (kR consecutive output pixels of one tile row, 8 channels) sits in a
// stage and in the A tile.  None of it depends on the tile or on the channel chunk, so each
// thread works it out once for the units it owns.
struct DwUnit {
    uint32_t x_off;   // byte offset of the unit's first input vector within a stage
    int m_row0;       // A-tile row of the unit's first output pixel (= pixel index in the tile)
    int cv;           // first of the unit's 8 channels within a chunk
    int nvalid;       // output pixels of the unit inside the tile (1..kR)
    int r, oc0;       // tile row and first tile column of the unit
};

template <int S>
__device__ __forceinline__ DwUnit dw_unit_geom(const Args &a, int u) {
    const int nv = a.chunk_c >> 3;
    const int v = u % nv;
    const int rest = u / nv;
    const int g = rest % a.ngroups;
    DwUnit d;
    d.r = rest / a.ngroups;
    d.oc0 = g * kR;
    d.cv = v * 8;
    d.x_off = (uint32_t)((d.r * S) * a.in_cols + d.oc0 * S) * (uint32_t)a.chunk_c * 2u + (uint32_t)v * 16u;
    d.m_row0 = d.r * a.tile_w + d.oc0;
    d.nvalid = min(kR, a.tile_w - d.oc0);
    return d;
}

// One DW work unit.  Products of 16-bit inputs and 16-bit taps are exact; sums are fp32
// (fma.rn.f32.{f16,bf16}).  `stage` and `wdw` are shared-memory pointers; the loads are plain
// C++ loads so that the compiler may schedule them early (they stay after the mbarrier waits,
// which clobber memory).
template <typename T, int KS, int S, int MODE, int ACT, bool RT>
__device__ __forceinline__ void dw_unit(const Args &a, const DwUnit &g, int chunk,
                                        const uint8_t *stage, const uint8_t *wdw,
                                        const uint4 (&wreg)[KS * KS], const float *s1_s,
                                        const float *b1_s, uint32_t a_saddr, int n, int ho0,
                                        int wo0) {
    const int c_glob = chunk * a.chunk_c + g.cv;
    const uint32_t px_bytes = (uint32_t)a.chunk_c * 2u;
    const uint32_t row_bytes = (uint32_t)a.in_cols * px_bytes;
    const uint32_t tap_bytes = (uint32_t)a.C * 2u;   // bytes between taps of the weight image
    const uint8_t *xb = stage + g.x_off;
    const uint8_t *wb = wdw + (uint32_t)c_glob * 2u;

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
            w[t] = RT ? wreg[i * KS + t]
                      : *reinterpret_cast<const uint4 *>(wb + (uint32_t)(i * KS + t) * tap_bytes);
        const uint8_t *xr = xb + (uint32_t)i * row_bytes;
#pragma unroll
        for (int q = 0; q < (kR - 1) * S + KS; q++) {
            const uint4 x = *reinterpret_cast<const uint4 *>(xr + (uint32_t)q * px_bytes);
#pragma unroll
            for (int jj = 0; jj < kR; jj++) {
                const int t = q - jj * S;
                if (t >= 0 && t < KS) {
                    Fma16<T>::fma2(acc[jj][0], acc[jj][1], x.x, w[t].x);
                    Fma16<T>::fma2(acc[jj][2], acc[jj][3], x.y, w[t].y);
                    Fma16<T>::fma2(acc[jj][4], acc[jj][5], x.z, w[t].z);
                    Fma16<T>::fma2(acc[jj][6], acc[jj][7], x.w, w[t].w);
                }
            }
        }
    }
    const float4 sc0 = *reinterpret_cast<const float4 *>(s1_s + c_glob);
    const float4 sc1 = *reinterpret_cast<const float4 *>(s1_s + c_glob + 4);
    const float4 bi0 = *reinterpret_cast<const float4 *>(b1_s + c_glob);
    const float4 bi1 = *reinterpret_cast<const float4 *>(b1_s + c_glob + 4);
    const float sc[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
    const float bi[8] = {bi0.x, bi0.y, bi0.z, bi0.w, bi1.x, bi1.y, bi1.z, bi1.w};
    // A-tile address of (row, c_glob): 64-channel block, 128-byte row, swizzled 16-byte chunk
    const uint32_t a_blk = a_saddr + (uint32_t)(c_glob >> 6) * (kTileM * 128u);
    const uint32_t a_chunk = (uint32_t)(c_glob >> 3) & 7u;
#pragma unroll
    for (int jj = 0; jj < kR; jj++) {
        if (jj >= g.nvalid) break;
        uint32_t pk[4];
#pragma unroll
        for (int c = 0; c < 4; c++)
            pk[c] = Pack2<T>::template run<ACT>(fmaf(sc[2 * c], acc[jj][2 * c], bi[2 * c]),
                                                fmaf(sc[2 * c + 1], acc[jj][2 * c + 1], bi[2 * c + 1]));
        if (MODE == FUSED) {
            const uint32_t m_row = (uint32_t)(g.m_row0 + jj);
            sts128(a_blk + m_row * 128u + ((a_chunk ^ (m_row & 7u)) << 4), pk[0], pk[1], pk[2], pk[3]);
        } else {
            const int ho = ho0 + g.r, wo = wo0 + g.oc0 + jj;
            if (ho < a.Ho && wo < a.Wo) {
                T *dst = static_cast<T *>(a.out) +
                         (((size_t)n * a.Ho + ho) * a.Wo + wo) * a.C + c_glob;
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
    }
}

// Byte offset of the 16-wide K step k16 in a K-major operand of `rows` rows stored as 64-wide
// K blocks of 128-byte swizzled rows.
__device__ __forceinline__ uint32_t k16_offset(int k16, int rows) {
    return (uint32_t)(k16 >> 2) * (uint32_t)rows * 128u + (uint32_t)(k16 & 3) * 32u;
}

__device__ __forceinline__ void tile_coords(const Args &a, int t, int &n, int &ho0, int &wo0) {
    n = t / a.tiles_per_img;
    const int rem = t - n * a.tiles_per_img;
    ho0 = (rem / a.tiles_w) * a.tile_h;
    wo0 = (rem % a.tiles_w) * a.tile_w;
}

// DWB: chunk-bound DW warps (Args::dw_per_chunk > 0), with their own register budget.
template <typename T, int KS, int S, int MODE, int DWB>
__global__ void __launch_bounds__(DWB ? kMaxThreadsBound : kMaxThreads, 1)
    dwpw_kernel(const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base_g = smem_raw + (base_s - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool has_mma = MODE != DWONLY;
    const bool has_dw = MODE != PWONLY;

    uint4 *wdw_s = reinterpret_cast<uint4 *>(base_g + a.off_wdw);   // filled in the prologue
    float *sb_s = reinterpret_cast<float *>(base_g + a.off_sb);
    float *s1_s = sb_s, *b1_s = sb_s + a.C, *s2_s = sb_s + 2 * a.C, *b2_s = sb_s + 2 * a.C + a.K;
    const uint32_t bar_base = base_s + a.off_bar;
    Bars bars(bar_base);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_g + a.off_bar + kBarBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base_g + a.off_bar + kBarBytes + 4);

    // ---- prologue: weights/scales to shared memory, barriers, TMEM
    if (has_dw) {
        const int nw = a.C * KS * KS / 8;
        for (int i = threadIdx.x; i < nw; i += blockDim.x) wdw_s[i] = a.wdw[i];
    }
    if (has_dw)
        for (int i = threadIdx.x; i < a.C; i += blockDim.x) {
            s1_s[i] = a.s1[i];
            b1_s[i] = a.b1[i];
        }
    for (int i = threadIdx.x; i < a.K; i += blockDim.x) {
        s2_s[i] = a.s2[i];
        b2_s[i] = a.b2[i];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; s++) {
            mbar_init(bars.full + 8 * s, 1);
            mbar_init(bars.empty + 8 * s, MODE == PWONLY ? 1 : DWB ? a.dw_per_chunk : a.n_dw_warps);
        }
        if (MODE == FUSED) {
            for (int j = 0; j < a.nchunks; j++) {
                mbar_init(bars.afull + 8 * j, DWB ? a.dw_per_chunk : a.n_dw_warps);
                mbar_init(bars.aempty + 8 * j, 1);
            }
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bars.accfull + 8 * b, 1);
            mbar_init(bars.accempty + 8 * b, kEpiWarps);
        }
        mbar_init(bars.wbar, 1);
        mbar_init(bars.drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (has_mma && warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = has_mma ? *tmem_slot : 0u;
    const unsigned long long lim = a.wait_limit_ns;

    if (warp == 0) {
        // ===================================================== TMA producer
        bool ok = true;
        if (has_mma && lane == 0) {
            mbar_arrive_expect_tx(bars.wbar, a.wp_img_bytes);
            bulk_load(base_s + a.off_b, a.wp_img, a.wp_img_bytes, bars.wbar);
        }
        if (lane == 0) tma_prefetch_desc(&a.tmap);
        int it = 0;
        for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x) {
            int n = 0, ho0 = 0, wo0 = 0;
            if (MODE != PWONLY) tile_coords(a, t, n, ho0, wo0);
            const int nloads = MODE == PWONLY ? 1 : a.nchunks;
            for (int j = 0; j < nloads; j++, it++) {
                const int s = it % a.stages;
                const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
                if (!mbar_wait(bars.empty + 8 * s, ph ^ 1u, abort_flag, a.err, lim)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t dst = base_s + a.off_in + (uint32_t)s * a.in_stage_stride;
                    mbar_arrive_expect_tx(bars.full + 8 * s, a.in_stage_bytes);
                    if (MODE == PWONLY) {
                        const int nkb = (a.C + 63) / 64;
                        for (int kb = 0; kb < nkb; kb++)
                            tma_load_2d(dst + (uint32_t)kb * kTileM * 128, &a.tmap, bars.full + 8 * s,
                                        kb * 64, (int)(t * kTileM));
                    } else {
                        tma_load_4d(dst, &a.tmap, bars.full + 8 * s, j * a.chunk_c,
                                    wo0 * S - a.pad, ho0 * S - a.pad, n);
                    }
                }
                __syncwarp();
            }
        }
        if (!ok) {
            // drain: every copy this warp issued lands before the CTA exits (`it` loads were
            // issued, load i into stage i % stages)
            volatile int no_abort = 0;
            for (int s = 0; s < a.stages && s < it; s++) {
                const int issued = (it - 1 - s) / a.stages + 1;
                mbar_wait(bars.full + 8 * s, (uint32_t)(issued - 1) & 1u, &no_abort, a.err, lim);
            }
            if (has_mma) mbar_wait(bars.wbar, 0, &no_abort, a.err, lim);
        }
    } else if (warp == 1 && has_mma) {
        // ===================================================== MMA issuer
        bool ok = mbar_wait(bars.wbar, 0, abort_flag, a.err, lim);
        const uint32_t b_s = base_s + a.off_b;
        const int kb_rows_b = a.K;   // rows of each 64-wide K block of B
        int lt = 0, it = 0;
        for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, lt++) {
            const int ab = lt & 1;
            if (!mbar_wait(bars.accempty + 8 * ab, ((uint32_t)(lt >> 1) & 1u) ^ 1u, abort_flag,
                           a.err, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)ab * (a.tmem_cols >> 1);
            if (MODE == PWONLY) {
                const int s = it % a.stages;
                const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
                it++;
                if (!mbar_wait(bars.full + 8 * s, ph, abort_flag, a.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a_s = base_s + a.off_in + (uint32_t)s * a.in_stage_stride;
                if (lane == 0) {
                    const uint64_t a0 = sw128_kmajor_desc(a_s), b0 = sw128_kmajor_desc(b_s);
                    for (int k16 = 0; k16 < a.C / 16; k16++)
                        mma_f16(d_tmem, desc_advance(a0, k16_offset(k16, kTileM)),
                                desc_advance(b0, k16_offset(k16, kb_rows_b)), a.idesc, k16 > 0 ? 1u : 0u);
                    mma_commit(bars.empty + 8 * s);
                    mma_commit(bars.accfull + 8 * ab);
                }
                __syncwarp();
            } else {
                // one A tile: chunk j of tile lt is its (lt+1)-th fill
                const uint32_t apar = (uint32_t)lt & 1u;
                const uint32_t a_s = base_s + a.off_a;
                const uint32_t afull_b = bars.afull, aempty_b = bars.aempty;
                const uint64_t a_desc0 = sw128_kmajor_desc(a_s), b_desc0 = sw128_kmajor_desc(b_s);
                const int k16_per_chunk = a.chunk_c / 16;
                for (int j = 0; j < a.nchunks; j++) {
                    if (!mbar_wait(afull_b + 8 * j, apar, abort_flag, a.err, lim)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        for (int kk = 0; kk < k16_per_chunk; kk++) {
                            const int k16 = j * k16_per_chunk + kk;
                            mma_f16(d_tmem, desc_advance(a_desc0, k16_offset(k16, kTileM)),
                                    desc_advance(b_desc0, k16_offset(k16, kb_rows_b)), a.idesc,
                                    k16 > 0 ? 1u : 0u);
                        }
                        mma_commit(aempty_b + 8 * j);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (lane == 0) mma_commit(bars.accfull + 8 * ab);
                __syncwarp();
            }
        }
        if (!ok && lane == 0) {
            volatile int no_abort = 0;
            mma_commit(bars.drain);
            mbar_wait(bars.drain, 0, &no_abort, a.err, lim);
        }
        __syncwarp();
    } else if (warp >= 2 && warp < 2 + kEpiWarps && has_mma) {
        // ===================================================== epilogue
        // TMEM -> registers -> scale/bias/act -> 16-bit -> 128B-swizzled staging tile in shared
        // memory -> one TMA tensor store per 64-channel block (full lines, clipped at the edges).
        // (Splitting the stores per block so that they overlap the next block's math measured
        // slower: more barriers and proxy fences per tile.)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const bool issuer = warp == 2 && lane == 0;
        const int nkb_out = (a.K + 63) / 64;
        const uint32_t swz = (uint32_t)(row & 7);
        uint32_t out_s = base_s + a.off_out, row_s = out_s + (uint32_t)row * 128;
        with_act(a.act2, [&](auto act_tag) {
            constexpr int ACT = decltype(act_tag)::value;
            // scale/bias/act on 16 accumulator columns starting at c0, rounded and written to the
            // swizzled staging row
            auto emit16 = [&](const uint32_t (&rr)[16], int c0) {
                uint32_t pk[8];
#pragma unroll
                for (int i4 = 0; i4 < 4; i4++) {
                    const float4 sc = *reinterpret_cast<const float4 *>(s2_s + c0 + 4 * i4);
                    const float4 bi = *reinterpret_cast<const float4 *>(b2_s + c0 + 4 * i4);
                    const float y0 = fmaf(sc.x, __uint_as_float(rr[4 * i4]), bi.x);
                    const float y1 = fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), bi.y);
                    const float y2 = fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), bi.z);
                    const float y3 = fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), bi.w);
                    pk[2 * i4] = Pack2<T>::template run<ACT>(y0, y1);
                    pk[2 * i4 + 1] = Pack2<T>::template run<ACT>(y2, y3);
                }
                const uint32_t blk = (uint32_t)(c0 >> 6) * kOutBlock;
                const uint32_t ch = (uint32_t)((c0 & 63) >> 3);
                sts128(row_s + blk + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                sts128(row_s + blk + (((ch + 1) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
            };
            int lt = 0;
            for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, lt++) {
                const int ab = lt & 1;
                const bool ok = mbar_wait(bars.accfull + 8 * ab, (uint32_t)(lt >> 1) & 1u,
                                          abort_flag, a.err, lim);
                // this tile's staging buffer is free once the stores that last read it are done
                // reading (with two buffers the previous tile's stores may still be running)
                if (issuer) {
                    if (a.out_bufs == 2)
                        bulk_wait_group_read<1>();
                    else
                        bulk_wait_group_read<0>();
                }
                if (named_barrier_or(1, 32 * kEpiWarps, !ok)) break;
                out_s = base_s + a.off_out + (uint32_t)(a.out_bufs == 2 ? (lt & 1) : 0) * a.out_buf_bytes;
                row_s = out_s + (uint32_t)row * 128;
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)ab * (a.tmem_cols >> 1);
                // two loads of 16 columns, one wait (K is a multiple of 16; keeping a load in
                // flight across the conversion measured slower)
                for (int c0 = 0; c0 < a.K; c0 += 32) {
                    uint32_t ra[16], rb[16];
                    const bool two = c0 + 16 < a.K;
                    tmem_ld16(taddr + (uint32_t)c0, ra);
                    if (two) tmem_ld16(taddr + (uint32_t)(c0 + 16), rb);
                    tmem_ld_wait();
                    emit16(ra, c0);
                    if (two) emit16(rb, c0 + 16);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bars.accempty + 8 * ab);   // TMEM buffer reusable
                fence_proxy_async_smem();                              // staging visible to TMA
                named_barrier(1, 32 * kEpiWarps);
                if (issuer) {
                    if (MODE == PWONLY) {
                        for (int kb = 0; kb < nkb_out; kb++)
                            tma_store_2d(&a.tmap_out, out_s + (uint32_t)kb * kOutBlock, kb * 64,
                                         t * kTileM);
                    } else {
                        int n, ho0, wo0;
                        tile_coords(a, t, n, ho0, wo0);
                        for (int kb = 0; kb < nkb_out; kb++)
                            tma_store_4d(&a.tmap_out, out_s + (uint32_t)kb * kOutBlock, kb * 64,
                                     wo0, ho0, n);
                    }
                    bulk_commit_group();
                }
            }
        });
        if (issuer) bulk_wait_group<0>();
    } else if (warp >= kFirstDwWarp && has_dw) {
        // ===================================================== DW warps
        const int units = a.tile_h * a.ngroups * (a.chunk_c >> 3);
        const uint8_t *wdw_g = base_g + a.off_wdw;
        const uint32_t a_s = base_s + a.off_a;
        if (DWB) {
            // Chunk-bound: warp w serves chunk w / dw_per_chunk of every tile, one unit per
            // thread (the planner guarantees units <= 32 * dw_per_chunk), with the unit's taps
            // held in registers for the whole kernel.
            const int dw_w = warp - kFirstDwWarp;
            const int jm = dw_w / a.dw_per_chunk;
            const int tid = (dw_w % a.dw_per_chunk) * 32 + lane;
            const bool has_unit = tid < units;
            const DwUnit g0 = dw_unit_geom<S>(a, has_unit ? tid : 0);
            uint4 wreg[KS * KS];
            {
                const uint8_t *wb = wdw_g + (uint32_t)(jm * a.chunk_c + g0.cv) * 2u;
#pragma unroll
                for (int t = 0; t < KS * KS; t++)
                    wreg[t] = *reinterpret_cast<const uint4 *>(wb + (uint32_t)t * (uint32_t)a.C * 2u);
            }
            with_act(a.act1, [&](auto act_tag) {
                constexpr int ACT = decltype(act_tag)::value;
                int lt = 0;
                for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x, lt++) {
                    int n, ho0, wo0;
                    tile_coords(a, t, n, ho0, wo0);
                    const int it = lt * a.nchunks + jm;   // the producer's load index of this chunk
                    const int s = it % a.stages;
                    const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
                    if (!mbar_wait(bars.full + 8 * s, ph, abort_flag, a.err, lim)) break;
                    if (MODE == FUSED && !mbar_wait(bars.aempty + 8 * jm, ((uint32_t)lt & 1u) ^ 1u,
                                                    abort_flag, a.err, lim))
                        break;
                    const uint8_t *stage_g = base_g + a.off_in + (uint32_t)s * a.in_stage_stride;
                    if (has_unit)
                        dw_unit<T, KS, S, MODE, ACT, true>(a, g0, jm, stage_g, wdw_g, wreg, s1_s,
                                                           b1_s, a_s, n, ho0, wo0);
                    if (MODE == FUSED) fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(bars.empty + 8 * s);
                        if (MODE == FUSED) mbar_arrive(bars.afull + 8 * jm);
                    }
                }
            });
        } else {
            // Every DW warp serves every chunk; taps are read from shared memory.
            const int tid = (warp - kFirstDwWarp) * 32 + lane;
            const int nthr = a.n_dw_warps * 32;
            const uint4 wnone[KS * KS] = {};
            // the thread's first unit (most plans give each thread at most one per chunk)
            const DwUnit g0 = dw_unit_geom<S>(a, tid < units ? tid : 0);
            with_act(a.act1, [&](auto act_tag) {
                constexpr int ACT = decltype(act_tag)::value;
                int lt = 0, it = 0;
                bool ok = true;
                for (int t = blockIdx.x; ok && t < a.num_tiles; t += gridDim.x, lt++) {
                    int n, ho0, wo0;
                    tile_coords(a, t, n, ho0, wo0);
                    for (int j = 0; j < a.nchunks; j++, it++) {
                        const int s = it % a.stages;
                        const uint32_t ph = (uint32_t)(it / a.stages) & 1u;
                        if (!mbar_wait(bars.full + 8 * s, ph, abort_flag, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        if (MODE == FUSED && !mbar_wait(bars.aempty + 8 * j, ((uint32_t)lt & 1u) ^ 1u,
                                                        abort_flag, a.err, lim)) {
                            ok = false;
                            break;
                        }
                        const uint8_t *stage_g = base_g + a.off_in + (uint32_t)s * a.in_stage_stride;
                        if (tid < units)
                            dw_unit<T, KS, S, MODE, ACT, false>(a, g0, j, stage_g, wdw_g, wnone, s1_s,
                                                                b1_s, a_s, n, ho0, wo0);
                        for (int u = tid + nthr; u < units; u += nthr)
                            dw_unit<T, KS, S, MODE, ACT, false>(a, dw_unit_geom<S>(a, u), j, stage_g,
                                                                wdw_g, wnone, s1_s, b1_s, a_s, n,
                                                                ho0, wo0);
                        if (MODE == FUSED) fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            mbar_arrive(bars.empty + 8 * s);
                            if (MODE == FUSED) mbar_arrive(bars.afull + 8 * j);
                        }
                    }
                }
            });
        }
    }

    __syncwarp();
    __syncthreads();
    if (has_mma && warp == 1) {
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
    const uint32_t b_bytes = mode == DWONLY ? 0u : (uint32_t)nkb * K * 128;
    const uint32_t a_bytes = mode == FUSED ? (uint32_t)nkb * kTileM * 128 : 0u;
    const uint32_t out_bytes =
        mode == DWONLY ? 0u : (uint32_t)(out_bufs * ((K + 63) / 64)) * kOutBlock;
    L.off_b = 0;
    L.off_a = align_up(b_bytes, 1024);
    L.off_out = align_up(L.off_a + a_bytes, 1024);
    L.off_in = align_up(L.off_out + out_bytes, 1024);
    if (mode == PWONLY)
        L.in_stage_bytes = (uint32_t)nkb * kTileM * 128;
    else
        L.in_stage_bytes = (uint32_t)p.in_rows * p.in_cols * p.chunk_c * 2;
    L.in_stage_stride = align_up(L.in_stage_bytes, 1024);
    const uint32_t wdw = mode == PWONLY ? 0u : (uint32_t)C * d->ksize * d->ksize * 2;
    const uint32_t sb = (uint32_t)(2 * C + 2 * K) * 4;
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

int fcm_tc_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why) {
    auto no = [&](const char *w) {
        if (why) *why = w;
        return 0;
    };
    if (d->dtype == FCM_F32) return no("fp32 runs on CUDA cores");
    if (d->conv1 == FCM_CONV1_POINTWISE) return fcm_pwdw_supported(d, ho, wo, cm, why);
    if (d->conv1 != FCM_CONV1_DEPTHWISE) return fcm_b2b_supported(d, ho, wo, cm, why);
    if (cm % 16 != 0) return no("channels must be a multiple of 16");
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
    const int S = d->stride, KS = d->ksize, C = cm;
    TcPlan best;
    double best_score = -1.0;
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
                // score: pixels per tile (MMA/halo efficiency) x thread efficiency x pipeline
                double halo = (double)(th * tw * S * S) / (double)(in_rows * in_cols);
                double score = (double)(th * tw) / kTileM * best_eff * (0.5 + 0.5 * halo) *
                               (t.stages >= 3 ? 1.0 : 0.9) *
                               (t.num_tiles >= num_sms ? 1.0 : 0.5);
                if (score > best_score + 1e-12) {
                    best_score = score;
                    best = t;
                }
            }
        }
    }
    if (best_score < 0) return FCM_ERR_SMEM_BUDGET;
    *p = best;
    return FCM_OK;
}

fcm_status fcm_tc_prepare(fcm_handle *h, const void *w1_host, const void *wp_host) {
    if (h->d.conv1 == FCM_CONV1_DENSE) return fcm_b2b_prepare(h, w1_host, wp_host);
    if (h->d.conv1 == FCM_CONV1_POINTWISE) return fcm_pwdw_prepare(h, w1_host, wp_host);
    const fcm_desc &d = h->d;
    const int C = h->cm, K = d.k_out, KS = d.ksize, nkb = (C + 63) / 64;
    // B operand image: row n = output channel, K-dim = input channel, 128B swizzle
    h->wp_img_bytes = (size_t)nkb * K * 128;
    std::vector<uint8_t> img(h->wp_img_bytes, 0);
    const uint16_t *wp16 = static_cast<const uint16_t *>(wp_host);
    for (int n = 0; n < K; n++)
        for (int c = 0; c < C; c++) {
            uint32_t off = sw128_offset(n, c, K, 2);
            memcpy(&img[off], &wp16[(size_t)n * C + c], 2);
        }
    // DW taps in the storage dtype, tap-major: [k*k][C] (lane v of a warp reads channels
    // 8v..8v+7 of one tap as one 16-byte vector, consecutive lanes consecutive vectors)
    std::vector<uint16_t> wdw((size_t)C * KS * KS);
    const uint16_t *w1b = static_cast<const uint16_t *>(w1_host);
    for (int c = 0; c < C; c++)
        for (int t = 0; t < KS * KS; t++) wdw[(size_t)t * C + c] = w1b[(size_t)c * KS * KS + t];
    if (cudaMalloc(&h->wp_img, h->wp_img_bytes) != cudaSuccess ||
        cudaMemcpy(h->wp_img, img.data(), h->wp_img_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->w1dw_img, wdw.size() * 2) != cudaSuccess ||
        cudaMemcpy(h->w1dw_img, wdw.data(), wdw.size() * 2, cudaMemcpyHostToDevice) != cudaSuccess)
        return fcm_fail(FCM_ERR_CUDA, "tensor-core weight images: %s",
                        cudaGetErrorString(cudaGetLastError()));
    return FCM_OK;
}

namespace {

template <typename T, int KS, int S, int MODE, int DWB>
cudaError_t launch_k(const Args &a, int ctas, int threads, uint32_t smem, cudaStream_t st) {
    auto k = dwpw_kernel<T, KS, S, MODE, DWB>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<ctas, threads, smem, st>>>(a);
    return cudaGetLastError();
}

template <typename T, int KS, int S, int MODE>
cudaError_t launch_t(const Args &a, int ctas, int threads, uint32_t smem, cudaStream_t st) {
    if constexpr (KS <= 3 && MODE != PWONLY) {
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
    const fcm_desc &d = h->d;
    const TcPlan &p = h->tc;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    const int out_bufs = mode == FUSED ? p.out_bufs : 1;
    Layout L = make_layout(&d, p, h->cm, mode, h->smem_optin, out_bufs);
    if (L.stages < 1) return cudaErrorInvalidConfiguration;
    Args a;
    memset(&a, 0, sizeof(a));
    const CUtensorMapDataType dt =
        d.dtype == FCM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
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
        cuuint64_t gstride[3] = {(cuuint64_t)d.c * 2, (cuuint64_t)d.w * d.c * 2,
                                 (cuuint64_t)d.h * d.w * d.c * 2};
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
        cuuint64_t gstride[3] = {(cuuint64_t)d.k_out * 2, (cuuint64_t)h->wo * d.k_out * 2,
                                 (cuuint64_t)h->ho * h->wo * d.k_out * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)p.tile_w, (cuuint32_t)p.tile_h, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        cr = enc(&a.tmap_out, dt, 4, out, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
    a.out = out;
    a.wp_img = static_cast<const uint8_t *>(h->wp_img);
    a.wdw = static_cast<const uint4 *>(h->w1dw_img);
    a.s1 = h->s1;
    a.b1 = h->b1;
    a.s2 = h->s2;
    a.b2 = h->b2;
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
    a.idesc = idesc_f16(d.dtype == FCM_BF16, kTileM, d.k_out);
    a.wp_img_bytes = (uint32_t)h->wp_img_bytes;
    a.in_stage_bytes = L.in_stage_bytes;
    a.in_stage_stride = L.in_stage_stride;
    a.off_b = L.off_b;
    a.off_a = L.off_a;
    a.off_out = L.off_out;
    a.out_bufs = out_bufs;
    a.out_buf_bytes = (uint32_t)((d.k_out + 63) / 64) * kOutBlock;
    a.off_in = L.off_in;
    a.off_wdw = L.off_wdw;
    a.off_sb = L.off_sb;
    a.off_bar = L.off_bar;
    const int threads = mode == PWONLY ? 32 * kFirstDwWarp : p.threads;
    const int ctas = (int)std::min<long long>(a.num_tiles, h->num_sms);
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
    return launch_mode(h, PWONLY, m, y, st);
}
