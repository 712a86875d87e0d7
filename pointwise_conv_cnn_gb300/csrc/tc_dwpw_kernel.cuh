// tc_dwpw_kernel.cuh -- device code of the tensor-core (tcgen05) depthwise -> pointwise
// kernels; included only by the translation units that instantiate them.
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
//   warps 2-9   epilogue: TMEM -> registers -> scale/bias/act -> swizzled staging -> TMA
//               stores (warp w reads TMEM lanes 32*(w%4) .. +31; the two warps of a lane
//               quadrant convert half of the columns each)
//   warps 10..  DW warps: stencil over a stage, result into the A tile (or HBM in DWONLY)
// Synchronisation is by mbarriers only; every wait is bounded (about one second) and a
// timeout sets the device error word, raises a CTA-wide abort flag and drains in-flight
// copies and MMAs before TMEM is released.
//
// T is the storage type: __half, __nv_bfloat16, or int8_t for the INT8 module (section III-B).
// INT8 computes on the f16 paths (int8 values are exact in f16): the stencil widens its inputs
// to f16 holding 1152 + x (I8::widen4) and starts its sums at minus the offset, the intermediate is
// requantized and handed to the tensor core as f16, the output is requantized to int8.
#pragma once

#include "tc_dwpw.cuh"

namespace fcm {
namespace tc {

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

template <typename T, int S>
__device__ __forceinline__ DwUnit dw_unit_geom(const Args &a, int u) {
    const int nv = a.chunk_c >> 3;
    const int v = u % nv;
    const int rest = u / nv;
    const int g = rest % a.ngroups;
    DwUnit d;
    d.r = rest / a.ngroups;
    d.oc0 = g * kR;
    d.cv = v * 8;
    d.x_off = ((uint32_t)((d.r * S) * a.in_cols + d.oc0 * S) * (uint32_t)a.chunk_c + (uint32_t)v * 8u) *
              (uint32_t)sizeof(T);
    d.m_row0 = d.r * a.tile_w + d.oc0;
    d.nvalid = min(kR, a.tile_w - d.oc0);
    return d;
}

// One DW work unit.  Products of 16-bit inputs and 16-bit taps are exact; sums are fp32
// (fma.rn.f32.{f16,bf16}).  `stage` and `wdw` are shared-memory pointers; the loads are plain
// C++ loads so that the compiler may schedule them early (they stay after the mbarrier waits,
// which clobber memory).  INT8: 8-byte input vectors widened to f16 (1152 + x), f16 taps, and
// the sums started at -1152 * sum(taps) of each channel (q1_s), which the offsets cancel.
// The first layer's scale and bias of a unit's 8 channels, held in registers by a chunk-bound
// stencil thread, whose channels never change.
struct DwNorm {
    float s[8], b[8];
};

template <typename T, int KS, int S, int MODE, int ACT, bool RT, bool NR>
__device__ __forceinline__ void dw_unit(const Args &a, const DwUnit &g, int chunk,
                                        const uint8_t *stage, const uint8_t *wdw,
                                        const uint4 (&wreg)[KS * KS], const DwNorm &nr,
                                        const float *s1_s, const float *b1_s, const float *q1_s,
                                        uint32_t a_saddr, int n, int ho0, int wo0) {
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    using TM = typename std::conditional<kI8, __half, T>::type;   // arithmetic type
    const int c_glob = chunk * a.chunk_c + g.cv;
    const uint32_t px_bytes = (uint32_t)a.chunk_c * (uint32_t)sizeof(T);
    const uint32_t row_bytes = (uint32_t)a.in_cols * px_bytes;
    const uint32_t tap_bytes = (uint32_t)a.C * 2u;   // bytes between taps of the weight image
    const uint8_t *xb = stage + g.x_off;
    const uint8_t *wb = wdw + (uint32_t)c_glob * 2u;
    // 1: the unit's last input vector lies inside the stage
    FCM_DCHECK(g.x_off + (uint32_t)(KS - 1) * row_bytes + (uint32_t)((kR - 1) * S + KS - 1) * px_bytes +
                       8u * (uint32_t)sizeof(T) <= (uint32_t)a.in_stage_bytes,
               a.err, 1, g.x_off);

    // INT8: the sums start at -1152 * sum(taps), the offset the widened inputs carry
    float acc[kR][8];
    if constexpr (kI8) {
        float qq[8];
        {
            const float4 q0 = *reinterpret_cast<const float4 *>(q1_s + c_glob);
            const float4 q1 = *reinterpret_cast<const float4 *>(q1_s + c_glob + 4);
            const float qv[8] = {-q0.x, -q0.y, -q0.z, -q0.w, -q1.x, -q1.y, -q1.z, -q1.w};
#pragma unroll
            for (int c = 0; c < 8; c++) qq[c] = qv[c];
        }
#pragma unroll
        for (int jj = 0; jj < kR; jj++)
#pragma unroll
            for (int c = 0; c < 8; c++) acc[jj][c] = qq[c];
    } else {
#pragma unroll
        for (int jj = 0; jj < kR; jj++)
#pragma unroll
            for (int c = 0; c < 8; c++) acc[jj][c] = 0.0f;
    }

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
            uint4 x;
            if constexpr (kI8) {
                const uint2 x8 = *reinterpret_cast<const uint2 *>(xr + (uint32_t)q * px_bytes);
                I8::widen4(x8.x, x.x, x.y);
                I8::widen4(x8.y, x.z, x.w);
            } else {
                x = *reinterpret_cast<const uint4 *>(xr + (uint32_t)q * px_bytes);
            }
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
    float sc[8], bi[8];
    if constexpr (NR) {
#pragma unroll
        for (int c = 0; c < 8; c++) {
            sc[c] = nr.s[c];
            bi[c] = nr.b[c];
        }
    } else {
        const float4 sc0 = *reinterpret_cast<const float4 *>(s1_s + c_glob);
        const float4 sc1 = *reinterpret_cast<const float4 *>(s1_s + c_glob + 4);
        const float4 bi0 = *reinterpret_cast<const float4 *>(b1_s + c_glob);
        const float4 bi1 = *reinterpret_cast<const float4 *>(b1_s + c_glob + 4);
        const float sv[8] = {sc0.x, sc0.y, sc0.z, sc0.w, sc1.x, sc1.y, sc1.z, sc1.w};
        const float bv[8] = {bi0.x, bi0.y, bi0.z, bi0.w, bi1.x, bi1.y, bi1.z, bi1.w};
#pragma unroll
        for (int c = 0; c < 8; c++) {
            sc[c] = sv[c];
            bi[c] = bv[c];
        }
    }
    // A-tile address of (row, c_glob): 64-channel block, 128-byte row, swizzled 16-byte chunk
    const uint32_t a_blk = a_saddr + (uint32_t)(c_glob >> 6) * (kTileM * 128u);
    const uint32_t a_chunk = (uint32_t)(c_glob >> 3) & 7u;
#pragma unroll
    for (int jj = 0; jj < kR; jj++) {
        if (jj >= g.nvalid) break;
        const uint32_t m_row = (uint32_t)(g.m_row0 + jj);
        const int ho = ho0 + g.r, wo = wo0 + g.oc0 + jj;
        FCM_DCHECK(m_row < (uint32_t)kTileM, a.err, 2, m_row);   // 2: A-tile row
        if constexpr (kI8) {
            float v[8];
#pragma unroll
            for (int c = 0; c < 8; c++) v[c] = fmaf(sc[c], acc[jj][c], bi[c]);
            if (MODE == FUSED) {
                sts128(a_blk + m_row * 128u + ((a_chunk ^ (m_row & 7u)) << 4),
                       I8::half2<ACT>(v[0], v[1]), I8::half2<ACT>(v[2], v[3]),
                       I8::half2<ACT>(v[4], v[5]), I8::half2<ACT>(v[6], v[7]));
            } else if (ho < a.Ho && wo < a.Wo) {
                T *dst = static_cast<T *>(a.out) +
                         (((size_t)n * a.Ho + ho) * a.Wo + wo) * a.C + c_glob;
                FCM_DCHECK(n < a.N && c_glob + 8 <= a.C, a.err, 3, c_glob);   // 3: intermediate store
                *reinterpret_cast<uint2 *>(dst) = make_uint2(I8::bytes4<ACT>(v[0], v[1], v[2], v[3]),
                                                             I8::bytes4<ACT>(v[4], v[5], v[6], v[7]));
            }
        } else {
            uint32_t pk[4];
#pragma unroll
            for (int c = 0; c < 4; c++)
                pk[c] = Pack2<T>::template run<ACT>(fmaf(sc[2 * c], acc[jj][2 * c], bi[2 * c]),
                                                    fmaf(sc[2 * c + 1], acc[jj][2 * c + 1], bi[2 * c + 1]));
            if (MODE == FUSED) {
                sts128(a_blk + m_row * 128u + ((a_chunk ^ (m_row & 7u)) << 4), pk[0], pk[1], pk[2], pk[3]);
            } else if (ho < a.Ho && wo < a.Wo) {
                T *dst = static_cast<T *>(a.out) +
                         (((size_t)n * a.Ho + ho) * a.Wo + wo) * a.C + c_glob;
                FCM_DCHECK(n < a.N && c_glob + 8 <= a.C, a.err, 3, c_glob);
                *reinterpret_cast<uint4 *>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        }
    }
}

__device__ __forceinline__ void tile_coords(const Args &a, int t, int &n, int &ho0, int &wo0) {
    n = t / a.tiles_per_img;
    const int rem = t - n * a.tiles_per_img;
    ho0 = (rem / a.tiles_w) * a.tile_h;
    wo0 = (rem % a.tiles_w) * a.tile_w;
}

// DWB: chunk-bound DW warps (Args::dw_per_chunk > 0), with their own register budget: 1 for
// up to kMaxThreadsBound threads, 2 for up to kMaxThreadsBound2.
template <typename T, int KS, int S, int MODE, int DWB>
__global__ void __launch_bounds__(DWB == 2 ? kMaxThreadsBound2 : DWB ? kMaxThreadsBound : kMaxThreads, 1)
    dwpw_kernel(const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base_g = smem_raw + (base_s - raw_s);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool has_mma = MODE != DWONLY;
    const bool has_dw = MODE != PWONLY;
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    static_assert(!(kI8 && MODE == PWONLY), "INT8 PW-only runs as FUSED with an identity stencil");
    // output staging: 64-channel blocks of kTileM rows; rows of 128 bytes (16-bit, 128-byte
    // swizzle) or 64 bytes (int8, 64-byte swizzle)
    constexpr uint32_t kRowBytes = 64u * (uint32_t)sizeof(T);
    constexpr uint32_t kBlockBytes = (uint32_t)kTileM * kRowBytes;
    using TS = typename std::conditional<kI8, __half, T>::type;   // 16-bit packing (non-INT8)

    uint4 *wdw_s = reinterpret_cast<uint4 *>(base_g + a.off_wdw);   // filled in the prologue
    float *sb_s = reinterpret_cast<float *>(base_g + a.off_sb);
    float *s1_s = sb_s, *b1_s = sb_s + a.C, *s2_s = sb_s + 2 * a.C, *b2_s = sb_s + 2 * a.C + a.K;
    float *q1_s = sb_s + 2 * a.C + 2 * a.K;   // INT8: 1152 * sum of each channel's taps
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
            if (kI8) q1_s[i] = a.q1[i];
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
    pdl_launch_dependents();
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
        pdl_wait();
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
        // kEpiWarps / 4 warps per TMEM lane quadrant split the columns in groups of 16
        const int ng = a.K / 16, part = (warp - 2) >> 2, nparts = kEpiWarps / 4;
        const int c_lo = (part * ng / nparts) * 16, c_hi = ((part + 1) * ng / nparts) * 16;
        const int nkb_out = (a.K + 63) / 64;
        const uint32_t swz = kI8 ? (uint32_t)((row >> 1) & 3) : (uint32_t)(row & 7);
        uint32_t out_s = base_s + a.off_out, row_s = out_s + (uint32_t)row * kRowBytes;
        with_act(a.act2, [&](auto act_tag) {
            constexpr int ACT = decltype(act_tag)::value;
            // scale/bias/act on 16 accumulator columns starting at c0, rounded and written to the
            // swizzled staging row
            auto emit16 = [&](const uint32_t (&rr)[16], int c0) {
                if constexpr (kI8) {
                    // 16 int8 outputs = one 16-byte chunk of the 64-byte row
                    uint32_t pk[4];
#pragma unroll
                    for (int i4 = 0; i4 < 4; i4++) {
                        const float4 sc = *reinterpret_cast<const float4 *>(s2_s + c0 + 4 * i4);
                        const float4 bi = *reinterpret_cast<const float4 *>(b2_s + c0 + 4 * i4);
                        pk[i4] = I8::bytes4<ACT>(fmaf(sc.x, __uint_as_float(rr[4 * i4]), bi.x),
                                                 fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), bi.y),
                                                 fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), bi.z),
                                                 fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), bi.w));
                    }
                    const uint32_t blk = (uint32_t)(c0 >> 6) * kBlockBytes;
                    const uint32_t ch = (uint32_t)((c0 & 63) >> 4);
                    sts128(row_s + blk + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                    return;
                }
                uint32_t pk[8];
#pragma unroll
                for (int i4 = 0; i4 < 4; i4++) {
                    const float4 sc = *reinterpret_cast<const float4 *>(s2_s + c0 + 4 * i4);
                    const float4 bi = *reinterpret_cast<const float4 *>(b2_s + c0 + 4 * i4);
                    const float y0 = fmaf(sc.x, __uint_as_float(rr[4 * i4]), bi.x);
                    const float y1 = fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), bi.y);
                    const float y2 = fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), bi.z);
                    const float y3 = fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), bi.w);
                    pk[2 * i4] = Pack2<TS>::template run<ACT>(y0, y1);
                    pk[2 * i4 + 1] = Pack2<TS>::template run<ACT>(y2, y3);
                }
                const uint32_t blk = (uint32_t)(c0 >> 6) * kBlockBytes;
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
                row_s = out_s + (uint32_t)row * kRowBytes;
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)ab * (a.tmem_cols >> 1);
                // two loads of 16 columns, one wait (K is a multiple of 16; keeping a load in
                // flight across the conversion measured slower)
                // The same on compile-time columns, with the biases from the kernel parameters
                // (used when K is 64 or 128: each warp's column range is then fixed at compile
                // time up to the choice of its half).
                auto emit16c = [&](const uint32_t (&rr)[16], auto c0t) {
                    constexpr int C0 = decltype(c0t)::value;
                    if constexpr (kI8) {
                        uint32_t pk[4];
#pragma unroll
                        for (int i4 = 0; i4 < 4; i4++) {
                            const float4 sc = *reinterpret_cast<const float4 *>(s2_s + C0 + 4 * i4);
                            pk[i4] = I8::bytes4<ACT>(
                                fmaf(sc.x, __uint_as_float(rr[4 * i4]), a.b2c[C0 + 4 * i4]),
                                fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), a.b2c[C0 + 4 * i4 + 1]),
                                fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), a.b2c[C0 + 4 * i4 + 2]),
                                fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), a.b2c[C0 + 4 * i4 + 3]));
                        }
                        constexpr uint32_t blk = (uint32_t)(C0 >> 6) * kBlockBytes;
                        constexpr uint32_t ch = (uint32_t)((C0 & 63) >> 4);
                        sts128(row_s + blk + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                    } else {
                        uint32_t pk[8];
#pragma unroll
                        for (int i4 = 0; i4 < 4; i4++) {
                            const float4 sc = *reinterpret_cast<const float4 *>(s2_s + C0 + 4 * i4);
                            const float y0 = fmaf(sc.x, __uint_as_float(rr[4 * i4]), a.b2c[C0 + 4 * i4]);
                            const float y1 = fmaf(sc.y, __uint_as_float(rr[4 * i4 + 1]), a.b2c[C0 + 4 * i4 + 1]);
                            const float y2 = fmaf(sc.z, __uint_as_float(rr[4 * i4 + 2]), a.b2c[C0 + 4 * i4 + 2]);
                            const float y3 = fmaf(sc.w, __uint_as_float(rr[4 * i4 + 3]), a.b2c[C0 + 4 * i4 + 3]);
                            pk[2 * i4] = Pack2<TS>::template run<ACT>(y0, y1);
                            pk[2 * i4 + 1] = Pack2<TS>::template run<ACT>(y2, y3);
                        }
                        constexpr uint32_t blk = (uint32_t)(C0 >> 6) * kBlockBytes;
                        constexpr uint32_t ch = (uint32_t)((C0 & 63) >> 3);
                        sts128(row_s + blk + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
                        sts128(row_s + blk + (((ch + 1) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
                    }
                };
                // 32 columns from compile-time column C0: two 16-column loads, one wait
                auto cols32 = [&](auto c0t) {
                    constexpr int C0 = decltype(c0t)::value;
                    uint32_t ra[16], rb[16];
                    tmem_ld16(taddr + (uint32_t)C0, ra);
                    tmem_ld16(taddr + (uint32_t)(C0 + 16), rb);
                    tmem_ld_wait(ra, rb);
                    emit16c(ra, std::integral_constant<int, C0>{});
                    emit16c(rb, std::integral_constant<int, C0 + 16>{});
                };
                static_assert(kEpiWarps == 8, "two epilogue warps per lane quadrant");
                if (a.b2c_n == 128 && a.K == 128) {
                    if (part == 0) {
                        cols32(std::integral_constant<int, 0>{});
                        cols32(std::integral_constant<int, 32>{});
                    } else {
                        cols32(std::integral_constant<int, 64>{});
                        cols32(std::integral_constant<int, 96>{});
                    }
                } else if (a.b2c_n == 64 && a.K == 64) {
                    if (part == 0)
                        cols32(std::integral_constant<int, 0>{});
                    else
                        cols32(std::integral_constant<int, 32>{});
                } else
                for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
                    uint32_t ra[16], rb[16];
                    const bool two = c0 + 16 < c_hi;
                    tmem_ld16(taddr + (uint32_t)c0, ra);
                    if (two) tmem_ld16(taddr + (uint32_t)(c0 + 16), rb);
                    tmem_ld_wait(ra, rb);
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
                            tma_store_2d(&a.tmap_out, out_s + (uint32_t)kb * kBlockBytes, kb * 64,
                                         t * kTileM);
                    } else {
                        int n, ho0, wo0;
                        tile_coords(a, t, n, ho0, wo0);
                        for (int kb = 0; kb < nkb_out; kb++)
                            tma_store_4d(&a.tmap_out, out_s + (uint32_t)kb * kBlockBytes, kb * 64,
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
            const DwUnit g0 = dw_unit_geom<T, S>(a, has_unit ? tid : 0);
            uint4 wreg[KS * KS] = {};
            if (kDwTapsInRegs) {
                const uint8_t *wb = wdw_g + (uint32_t)(jm * a.chunk_c + g0.cv) * 2u;
#pragma unroll
                for (int t = 0; t < KS * KS; t++)
                    wreg[t] = *reinterpret_cast<const uint4 *>(wb + (uint32_t)t * (uint32_t)a.C * 2u);
            }
            // (16-bit storage in the fused mode of the 768-thread tier: INT8, the 544-thread tier
            // and the depthwise-only mode spill far more with them and measured slower)
            constexpr bool kNormRegs = kDwNormInRegs && !kI8 && DWB == 1 && MODE == FUSED;
            DwNorm nreg;
            if (kNormRegs) {
                const int cg = jm * a.chunk_c + g0.cv;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    nreg.s[c] = s1_s[cg + c];
                    nreg.b[c] = b1_s[cg + c];
                }
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
                        dw_unit<T, KS, S, MODE, ACT, kDwTapsInRegs, kNormRegs>(a, g0, jm, stage_g, wdw_g, wreg, nreg, s1_s,
                                                           b1_s, q1_s, a_s, n, ho0, wo0);
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
            const DwNorm nnone{};
            // the thread's first unit (most plans give each thread at most one per chunk)
            const DwUnit g0 = dw_unit_geom<T, S>(a, tid < units ? tid : 0);
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
                            dw_unit<T, KS, S, MODE, ACT, false, false>(a, g0, j, stage_g, wdw_g, wnone, nnone, s1_s,
                                                                b1_s, q1_s, a_s, n, ho0, wo0);
                        for (int u = tid + nthr; u < units; u += nthr)
                            dw_unit<T, KS, S, MODE, ACT, false, false>(a, dw_unit_geom<T, S>(a, u), j, stage_g,
                                                                wdw_g, wnone, nnone, s1_s, b1_s, q1_s, a_s,
                                                                n, ho0, wo0);
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
template <typename T, int KS, int S, int MODE, int DWB>
cudaError_t launch_k(const Args &a, int ctas, int threads, uint32_t smem, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_ctx{0};
    return launch_pdl(dwpw_kernel<T, KS, S, MODE, DWB>, attr_ctx, ctas, threads, smem, st, a);
}

}  // namespace tc
}  // namespace fcm
