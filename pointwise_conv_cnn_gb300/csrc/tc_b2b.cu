// tc_b2b.cu -- back-to-back dense k x k -> 1x1 convolution on tcgen05 (sm_103a).
//
// The CONV1 -> CONV2 example of "Fusing two back-to-back convolutions" (CUTLASS discussion
// #208): a dense k x k convolution with scale/bias/activation whose output stays in the
// block and feeds a 1x1 convolution with scale/bias/activation; the second convolution is
// 1x1, so a block never needs another block's intermediate.  On Blackwell both convolutions
// run on the tensor cores with fp32 accumulators in tensor memory:
//
//   conv1  implicit GEMM.  The input tile (tile rows + k-1 halo rows, a pitch of P >= Wo+k-1
//          columns, 64-channel planes, 128-byte swizzled) is loaded by TMA; for filter tap
//          (r, t) the A operand is the same tile read from pixel offset r*P + t, so every
//          output pixel (row, col) is GEMM row row*P + col and the k*k taps are k*k
//          shifted shared-memory descriptors over one tile.  Columns col >= Wo are computed
//          and discarded.
//   mid    TMEM -> registers -> scale/bias/act -> 16-bit -> the A operand of conv2 in shared
//          memory (128-byte swizzled, K-major): the intermediate never leaves the SM.
//   conv2  1x1 GEMM into a second TMEM accumulator.
//   out    TMEM -> scale/bias/act -> 16-bit -> swizzled staging (two tiles) -> TMA tensor
//          stores, one per output row and 64-channel block, clipped at Wo.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2-5 mid epilogue,
// warps 6-9 output epilogue.  Accumulators are double-buffered so conv1 of tile t overlaps
// the epilogues of tile t-1.  In CONV1 mode (the layer-by-layer baseline) the mid warps store
// the intermediate to HBM instead.  Every wait is bounded, as in the DW->PW kernels.
//
// INT8 (T = int8_t, k = 1: the PWPW module of section III-B's INT8 FCMs): the TMA loads the
// int8 input tile into its own ring, warps 10-13 widen it exactly to the f16 A operand
// (128-byte swizzled, as the TMA would have written it), and both GEMMs run as kind::f16 on
// int8 values (exact: every partial sum stays below 2^22); the mid epilogue requantizes into the
// f16 A2 operand, the output epilogue to int8 (64-byte rows, 64-byte swizzle).
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "fcm_internal.h"
#include "tc_common.cuh"

namespace fcm {
namespace b2b {

using namespace fcm::tc;

constexpr int kTileM = 128;
constexpr int kMaxStages = 6;
constexpr int kMidWarps = 4;
constexpr int kOutWarps = 4;
constexpr int kThreads = 32 * (2 + kMidWarps + kOutWarps);
constexpr int kConvWarps = 4;                       // INT8: int8 -> f16 A operand
constexpr int kFirstConvWarp = 2 + kMidWarps + kOutWarps;
constexpr int kThreadsI8 = 32 * (kFirstConvWarp + kConvWarps);
constexpr uint32_t kBlk = kTileM * 128;   // one 64-channel block of a 128-row operand

enum Mode { FUSED = 0, CONV1 = 1 };

struct Args {
    CUtensorMap tmap_in;    // x: 4-D (C, W, H, N), box (64, P, in_rows, 1), 128B swizzle
    CUtensorMap tmap_out;   // y (FUSED) or m (CONV1): 4-D (K, Wo, Ho, N), box (64, P, 1, 1)
    const uint8_t *w1_img;  // conv1 B images: [tap][64-channel block][Cm rows x 128 B]
    const uint8_t *w2_img;  // conv2 B image: [64-channel block][K rows x 128 B]
    const float *s1, *b1, *s2, *b2;
    unsigned *err;
    unsigned long long wait_limit_ns;
    int num_tiles, tiles_per_img;
    int C, Cm, K, Ho, Wo, ks, pad;
    int P, TH, in_rows, nkb_in, nkb_mid;
    int stages, act1, act2;
    uint32_t tmem_cols, idesc1, idesc2;
    uint32_t w1_bytes, w2_bytes, plane_bytes, in_stage_bytes, in_stage_stride;
    uint32_t off_w1, off_w2, off_a2, off_out, off_in, off_sb, off_bar;
    uint32_t out_bytes;     // one output staging tile (FUSED keeps two)
    // INT8: the ring of int8 input tiles the TMA fills (planes of 64 channels x 64 bytes)
    uint32_t off_in8, in8_stage_bytes, in8_stage_stride, plane8_bytes;
    // The two layers' biases as kernel parameters (b1c_n = Cm, b2c_n = K when that is 64 or
    // 128, else 0): the epilogues' FMAs then read them as constant operands instead of loading
    // them from shared memory
    int b1c_n, b2c_n;
    float b1c[128], b2c[128];
};

struct Bars {
    // full/empty: the input stage (INT8: full = int8 tile landed, empty = f16 A operand free);
    // INT8 only: full1 = f16 A operand written, empty8 = int8 tile converted
    uint32_t full, empty, acc1full, acc1empty, a2full, a2empty, acc2full, acc2empty, wbar, drain,
        full1, empty8;
    __device__ Bars(uint32_t base) {
        full = base;
        empty = full + 8 * kMaxStages;
        acc1full = empty + 8 * kMaxStages;
        acc1empty = acc1full + 16;
        a2full = acc1empty + 16;
        a2empty = a2full + 16;
        acc2full = a2empty + 16;
        acc2empty = acc2full + 16;
        wbar = acc2empty + 16;
        drain = wbar + 8;
        full1 = drain + 8;
        empty8 = full1 + 8 * kMaxStages;
    }
};
constexpr uint32_t kBarBytes = 8 * (4 * kMaxStages + 12 + 2) + 16;

// 128B-swizzled K-major descriptor whose start may sit at any 128-byte row of a swizzle atom:
// the tensor core applies the swizzle to absolute shared-memory address bits, the same bits
// the TMA used when it wrote the tile, so a start shifted by t rows reads pixel i + t as row i
// with the base-offset field left at 0 (measured: setting it to the start's row phase breaks
// parity).
__device__ __forceinline__ uint64_t shifted_desc(uint32_t saddr) { return sw128_kmajor_desc(saddr); }

// TMEM accumulator (128 lanes x ncols fp32) -> scale/bias/act -> 16-bit -> a 128-row,
// 128B-swizzled K-major image in shared memory (64-channel blocks of kBlk bytes).
template <typename T, int ACT>
__device__ __forceinline__ void emit16(const uint32_t (&rr)[16], int cc, const float *sc_s,
                                       const float *bi_s, uint32_t dst_s, int row) {
    const uint32_t swz = (uint32_t)(row & 7);
    uint32_t pk[8];
#pragma unroll
    for (int i4 = 0; i4 < 4; i4++) {
        const float4 s = *reinterpret_cast<const float4 *>(sc_s + cc + 4 * i4);
        const float4 b = *reinterpret_cast<const float4 *>(bi_s + cc + 4 * i4);
        pk[2 * i4] = Pack2<T>::template run<ACT>(fmaf(s.x, __uint_as_float(rr[4 * i4]), b.x),
                                                 fmaf(s.y, __uint_as_float(rr[4 * i4 + 1]), b.y));
        pk[2 * i4 + 1] = Pack2<T>::template run<ACT>(fmaf(s.z, __uint_as_float(rr[4 * i4 + 2]), b.z),
                                                     fmaf(s.w, __uint_as_float(rr[4 * i4 + 3]), b.w));
    }
    const uint32_t base = dst_s + (uint32_t)(cc >> 6) * kBlk + (uint32_t)row * 128;
    const uint32_t ch = (uint32_t)((cc & 63) >> 3);
    sts128(base + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
    sts128(base + (((ch + 1) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
}

// INT8, requantized to f16 (the A2 operand): the same 128-row, 128B-swizzled image.
template <int ACT>
__device__ __forceinline__ void emit16_i8_half(const uint32_t (&rr)[16], int cc, const float *sc_s,
                                               const float *bi_s, uint32_t dst_s, int row) {
    const uint32_t swz = (uint32_t)(row & 7);
    uint32_t pk[8];
#pragma unroll
    for (int i4 = 0; i4 < 4; i4++) {
        const float4 s = *reinterpret_cast<const float4 *>(sc_s + cc + 4 * i4);
        const float4 b = *reinterpret_cast<const float4 *>(bi_s + cc + 4 * i4);
        pk[2 * i4] = I8::half2<ACT>(fmaf(s.x, __uint_as_float(rr[4 * i4]), b.x),
                                    fmaf(s.y, __uint_as_float(rr[4 * i4 + 1]), b.y));
        pk[2 * i4 + 1] = I8::half2<ACT>(fmaf(s.z, __uint_as_float(rr[4 * i4 + 2]), b.z),
                                        fmaf(s.w, __uint_as_float(rr[4 * i4 + 3]), b.w));
    }
    const uint32_t base = dst_s + (uint32_t)(cc >> 6) * kBlk + (uint32_t)row * 128;
    const uint32_t ch = (uint32_t)((cc & 63) >> 3);
    sts128(base + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
    sts128(base + (((ch + 1) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
}

// INT8, requantized to int8 bytes: a 128-row image of 64-byte rows (64-channel blocks of
// kTileM * 64 bytes), 64-byte swizzled (16-byte chunk c of row r at c ^ ((r >> 1) & 3)).
template <int ACT>
__device__ __forceinline__ void emit16_i8_bytes(const uint32_t (&rr)[16], int cc, const float *sc_s,
                                                const float *bi_s, uint32_t dst_s, int row) {
    uint32_t pk[4];
#pragma unroll
    for (int i4 = 0; i4 < 4; i4++) {
        const float4 s = *reinterpret_cast<const float4 *>(sc_s + cc + 4 * i4);
        const float4 b = *reinterpret_cast<const float4 *>(bi_s + cc + 4 * i4);
        pk[i4] = I8::bytes4<ACT>(fmaf(s.x, __uint_as_float(rr[4 * i4]), b.x),
                                 fmaf(s.y, __uint_as_float(rr[4 * i4 + 1]), b.y),
                                 fmaf(s.z, __uint_as_float(rr[4 * i4 + 2]), b.z),
                                 fmaf(s.w, __uint_as_float(rr[4 * i4 + 3]), b.w));
    }
    const uint32_t base = dst_s + (uint32_t)(cc >> 6) * (kTileM * 64u) + (uint32_t)row * 64u;
    const uint32_t ch = (uint32_t)((cc & 63) >> 4);
    sts128(base + ((ch ^ (uint32_t)((row >> 1) & 3)) << 4), pk[0], pk[1], pk[2], pk[3]);
}

// What an accumulator becomes: the storage dtype (16-bit, 128B swizzle), or for INT8 the f16
// A operand of the next GEMM or int8 bytes (64B swizzle).
enum OutKind { OUT_STORAGE = 0, OUT_I8_HALF = 1, OUT_I8_BYTES = 2 };

// TMEM accumulator (128 lanes x ncols fp32, ncols a multiple of 16) -> scale/bias/act -> the
// image of OutKind in shared memory.  Two loads of 16 columns, then one wait.
template <typename T, int KIND, int ACT>
__device__ __forceinline__ void acc_to_smem_act(uint32_t taddr_row, int ncols, const float *sc_s,
                                                const float *bi_s, uint32_t dst_s, int row) {
    auto emit = [&](const uint32_t (&rr)[16], int cc) {
        if constexpr (KIND == OUT_I8_HALF)
            emit16_i8_half<ACT>(rr, cc, sc_s, bi_s, dst_s, row);
        else if constexpr (KIND == OUT_I8_BYTES)
            emit16_i8_bytes<ACT>(rr, cc, sc_s, bi_s, dst_s, row);
        else
            emit16<T, ACT>(rr, cc, sc_s, bi_s, dst_s, row);
    };
    for (int c0 = 0; c0 < ncols; c0 += 32) {
        uint32_t ra[16], rb[16];
        const bool two = c0 + 16 < ncols;
        tmem_ld16(taddr_row + (uint32_t)c0, ra);
        if (two) tmem_ld16(taddr_row + (uint32_t)(c0 + 16), rb);
        tmem_ld_wait(ra, rb);
        emit(ra, c0);
        if (two) emit(rb, c0 + 16);
    }
}

// The same with NC compile-time columns and the biases from the kernel parameters (a.b1c
// for the first layer, MID, else a.b2c), read by the FMAs as constant operands.
template <typename T, int KIND, int ACT, int NC, bool MID>
__device__ __forceinline__ void acc_to_smem_ct(const Args &a, uint32_t taddr_row, const float *sc_s,
                                               uint32_t dst_s, int row) {
    auto bias = [&](int c) -> float { return MID ? a.b1c[c] : a.b2c[c]; };
    auto emit = [&](const uint32_t (&rr)[16], auto cct) {
        constexpr int cc = decltype(cct)::value;
        if constexpr (KIND == OUT_I8_BYTES) {
            uint32_t pk[4];
#pragma unroll
            for (int i4 = 0; i4 < 4; i4++) {
                const float4 sv = *reinterpret_cast<const float4 *>(sc_s + cc + 4 * i4);
                pk[i4] = I8::bytes4<ACT>(fmaf(sv.x, __uint_as_float(rr[4 * i4]), bias(cc + 4 * i4)),
                                         fmaf(sv.y, __uint_as_float(rr[4 * i4 + 1]), bias(cc + 4 * i4 + 1)),
                                         fmaf(sv.z, __uint_as_float(rr[4 * i4 + 2]), bias(cc + 4 * i4 + 2)),
                                         fmaf(sv.w, __uint_as_float(rr[4 * i4 + 3]), bias(cc + 4 * i4 + 3)));
            }
            const uint32_t base = dst_s + (uint32_t)(cc >> 6) * (kTileM * 64u) + (uint32_t)row * 64u;
            constexpr uint32_t ch = (uint32_t)((cc & 63) >> 4);
            sts128(base + ((ch ^ (uint32_t)((row >> 1) & 3)) << 4), pk[0], pk[1], pk[2], pk[3]);
        } else {
            const uint32_t swz = (uint32_t)(row & 7);
            uint32_t pk[8];
#pragma unroll
            for (int i4 = 0; i4 < 4; i4++) {
                const float4 sv = *reinterpret_cast<const float4 *>(sc_s + cc + 4 * i4);
                const float y0 = fmaf(sv.x, __uint_as_float(rr[4 * i4]), bias(cc + 4 * i4));
                const float y1 = fmaf(sv.y, __uint_as_float(rr[4 * i4 + 1]), bias(cc + 4 * i4 + 1));
                const float y2 = fmaf(sv.z, __uint_as_float(rr[4 * i4 + 2]), bias(cc + 4 * i4 + 2));
                const float y3 = fmaf(sv.w, __uint_as_float(rr[4 * i4 + 3]), bias(cc + 4 * i4 + 3));
                if constexpr (KIND == OUT_I8_HALF) {
                    pk[2 * i4] = I8::half2<ACT>(y0, y1);
                    pk[2 * i4 + 1] = I8::half2<ACT>(y2, y3);
                } else {
                    pk[2 * i4] = Pack2<T>::template run<ACT>(y0, y1);
                    pk[2 * i4 + 1] = Pack2<T>::template run<ACT>(y2, y3);
                }
            }
            const uint32_t base = dst_s + (uint32_t)(cc >> 6) * kBlk + (uint32_t)row * 128;
            constexpr uint32_t ch = (uint32_t)((cc & 63) >> 3);
            sts128(base + ((ch ^ swz) << 4), pk[0], pk[1], pk[2], pk[3]);
            sts128(base + (((ch + 1) ^ swz) << 4), pk[4], pk[5], pk[6], pk[7]);
        }
    };
    auto cols32 = [&](auto c0t) {
        constexpr int c0 = decltype(c0t)::value;
        uint32_t ra[16], rb[16];
        tmem_ld16(taddr_row + (uint32_t)c0, ra);
        tmem_ld16(taddr_row + (uint32_t)(c0 + 16), rb);
        tmem_ld_wait(ra, rb);
        emit(ra, std::integral_constant<int, c0>{});
        emit(rb, std::integral_constant<int, c0 + 16>{});
    };
    static_assert(NC == 64 || NC == 128, "64 or 128 columns");
    cols32(std::integral_constant<int, 0>{});
    cols32(std::integral_constant<int, 32>{});
    if constexpr (NC == 128) {
        cols32(std::integral_constant<int, 64>{});
        cols32(std::integral_constant<int, 96>{});
    }
}

template <typename T, int KIND, bool MID>
__device__ __forceinline__ void acc_to_smem(const Args &a, uint32_t taddr_row, int ncols,
                                            const float *sc_s, const float *bi_s, int act,
                                            uint32_t dst_s, int row) {
    // (16-bit storage only: the INT8 kernel measured slower with it, 28.0 against 25.7 us on
    // the INT8 PWPW layer, where the 16-bit one gains 3%)
    const int bc_n = std::is_same<T, int8_t>::value ? 0 : MID ? a.b1c_n : a.b2c_n;
    with_act(act, [&](auto act_tag) {
        constexpr int ACT = decltype(act_tag)::value;
        if (bc_n == ncols && ncols == 128)
            acc_to_smem_ct<T, KIND, ACT, 128, MID>(a, taddr_row, sc_s, dst_s, row);
        else if (bc_n == ncols && ncols == 64)
            acc_to_smem_ct<T, KIND, ACT, 64, MID>(a, taddr_row, sc_s, dst_s, row);
        else
            acc_to_smem_act<T, KIND, ACT>(taddr_row, ncols, sc_s, bi_s, dst_s, row);
    });
}

// Called by one thread after its warp group staged a tile: one TMA store per output row of
// the tile and 64-channel block; rows past Ho are skipped, columns past Wo are clipped by the
// tensor map.
// (Staging rows of 64 channels: row_bytes 128 for 16-bit storage, 64 for int8.)
__device__ __forceinline__ void store_tile(const Args &a, const CUtensorMap *map, uint32_t stage_s,
                                           int nch, int n, int ho0, uint32_t row_bytes) {
    const int nkb = (nch + 63) / 64;
    for (int r = 0; r < a.TH; r++) {
        if (ho0 + r >= a.Ho) break;
        for (int kb = 0; kb < nkb; kb++)
            tma_store_4d(map, stage_s + (uint32_t)kb * kTileM * row_bytes + (uint32_t)(r * a.P) * row_bytes,
                         kb * 64, 0, ho0 + r, n);
    }
    bulk_commit_group();
}

template <typename T, int KS, int MODE>
__global__ void __launch_bounds__(std::is_same<T, int8_t>::value ? kThreadsI8 : kThreads, 1)
    b2b_kernel(const __grid_constant__ Args a) {
    constexpr bool kI8 = std::is_same<T, int8_t>::value;
    static_assert(!kI8 || KS == 1, "INT8 back-to-back runs k = 1 (two 1x1 convolutions)");
    // what the epilogues write: the storage dtype, or for INT8 f16 A2 / int8 bytes
    constexpr int kMidKind = !kI8 ? OUT_STORAGE : MODE == FUSED ? OUT_I8_HALF : OUT_I8_BYTES;
    constexpr int kOutKind = kI8 ? OUT_I8_BYTES : OUT_STORAGE;
    constexpr uint32_t kRowB = 64u * (uint32_t)sizeof(T);   // staging row bytes of stored data
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    uint8_t *base_g = smem_raw + (base_s - raw_s);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    float *sb_s = reinterpret_cast<float *>(base_g + a.off_sb);
    float *s1_s = sb_s, *b1_s = sb_s + a.Cm, *s2_s = sb_s + 2 * a.Cm, *b2_s = sb_s + 2 * a.Cm + a.K;
    Bars bars(base_s + a.off_bar);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base_g + a.off_bar + kBarBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base_g + a.off_bar + kBarBytes + 4);

    for (int i = threadIdx.x; i < a.Cm; i += blockDim.x) {
        s1_s[i] = a.s1[i];
        b1_s[i] = a.b1[i];
    }
    if (MODE == FUSED)
        for (int i = threadIdx.x; i < a.K; i += blockDim.x) {
            s2_s[i] = a.s2[i];
            b2_s[i] = a.b2[i];
        }
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; s++) {
            mbar_init(bars.full + 8 * s, 1);
            mbar_init(bars.empty + 8 * s, 1);
            if (kI8) {
                mbar_init(bars.full1 + 8 * s, kConvWarps);
                mbar_init(bars.empty8 + 8 * s, kConvWarps);
            }
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(bars.acc1full + 8 * b, 1);
            mbar_init(bars.acc1empty + 8 * b, kMidWarps);
            mbar_init(bars.a2full + 8 * b, kMidWarps);
            mbar_init(bars.a2empty + 8 * b, 1);
            mbar_init(bars.acc2full + 8 * b, 1);
            mbar_init(bars.acc2empty + 8 * b, kOutWarps);
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
    const uint32_t acc1_col = 0, acc2_col = 2u * (uint32_t)a.Cm;
    const unsigned long long lim = a.wait_limit_ns;
    const int my_tiles = (a.num_tiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

    if (warp == 0) {
        // ===================================================== TMA producer
        int issued = 0;   // loads issued so far; load i goes to stage i % stages
        bool ok = true;
        if (lane == 0) {
            mbar_arrive_expect_tx(bars.wbar, a.w1_bytes + (MODE == FUSED ? a.w2_bytes : 0u));
            bulk_load(base_s + a.off_w1, a.w1_img, a.w1_bytes, bars.wbar);
            if (MODE == FUSED) bulk_load(base_s + a.off_w2, a.w2_img, a.w2_bytes, bars.wbar);
            tma_prefetch_desc(&a.tmap_in);
        }
        pdl_wait();
        int s = 0;
        uint32_t ph = 0;
        for (int lt = 0; ok && lt < my_tiles; lt++) {
            const int t = (int)blockIdx.x + lt * (int)gridDim.x;
            const int n = t / a.tiles_per_img;
            const int ho0 = (t - n * a.tiles_per_img) * a.TH;
            // INT8: the int8 tile ring is free once the converters have read it
            if (!mbar_wait((kI8 ? bars.empty8 : bars.empty) + 8 * s, ph ^ 1u, abort_flag, a.err, lim)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t dst = kI8 ? base_s + a.off_in8 + (uint32_t)s * a.in8_stage_stride
                                         : base_s + a.off_in + (uint32_t)s * a.in_stage_stride;
                const uint32_t plane = kI8 ? a.plane8_bytes : a.plane_bytes;
                mbar_arrive_expect_tx(bars.full + 8 * s, kI8 ? a.in8_stage_bytes : a.in_stage_bytes);
                for (int kb = 0; kb < a.nkb_in; kb++)
                    tma_load_4d(dst + (uint32_t)kb * plane, &a.tmap_in, bars.full + 8 * s,
                                kb * 64, -a.pad, ho0 - a.pad, n);
            }
            issued++;
            __syncwarp();
            if (++s == a.stages) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) {
            volatile int no_abort = 0;
            for (int q = 0; q < a.stages && q < issued; q++) {
                const int nq = (issued - 1 - q) / a.stages + 1;   // loads that went to stage q
                mbar_wait(bars.full + 8 * q, (uint32_t)(nq - 1) & 1u, &no_abort, a.err, lim);
            }
            mbar_wait(bars.wbar, 0, &no_abort, a.err, lim);
        }
    } else if (warp == 1) {
        // ===================================================== MMA issuer
        bool ok = mbar_wait(bars.wbar, 0, abort_flag, a.err, lim);
        const uint32_t w1_s = base_s + a.off_w1, w2_s = base_s + a.off_w2;
        int s = 0;
        uint32_t ph = 0;
        const int last = MODE == FUSED ? my_tiles : my_tiles - 1;
        for (int lt = 0; ok && lt <= last; lt++) {
            if (lt < my_tiles) {
                const int b = lt & 1;
                if (!mbar_wait((kI8 ? bars.full1 : bars.full) + 8 * s, ph, abort_flag, a.err, lim) ||
                    !mbar_wait(bars.acc1empty + 8 * b, ((uint32_t)(lt >> 1) & 1u) ^ 1u, abort_flag,
                               a.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    // descriptors are advanced from two bases; the tap loops unroll (KS is a
                    // template parameter), so each MMA costs a couple of integer adds to issue
                    const uint32_t in_s = base_s + a.off_in + (uint32_t)s * a.in_stage_stride;
                    const uint32_t d = tmem_base + acc1_col + (uint32_t)b * (uint32_t)a.Cm;
                    const uint64_t a_base = shifted_desc(in_s);
                    const uint64_t b_base = sw128_kmajor_desc(w1_s);
                    const uint32_t w_kb = (uint32_t)a.Cm * 128u;            // one 64-channel block of a tap
                    const uint32_t w_tap = (uint32_t)a.nkb_in * w_kb;       // one tap
#pragma unroll
                    for (int r = 0; r < KS; r++)
#pragma unroll
                        for (int tt = 0; tt < KS; tt++)
                            for (int kb = 0; kb < a.nkb_in; kb++) {
                                const uint64_t ad = desc_advance(
                                    a_base, (uint32_t)kb * a.plane_bytes + (uint32_t)(r * a.P + tt) * 128u);
                                const uint64_t bd = desc_advance(
                                    b_base, (uint32_t)(r * KS + tt) * w_tap + (uint32_t)kb * w_kb);
#pragma unroll
                                for (int k16 = 0; k16 < 4; k16++)
                                    mma_f16(d, desc_advance(ad, 32u * k16), desc_advance(bd, 32u * k16),
                                            a.idesc1, (r | tt | kb | k16) != 0 ? 1u : 0u);
                            }
                    mma_commit(bars.empty + 8 * s);
                    mma_commit(bars.acc1full + 8 * b);
                }
                __syncwarp();
                if (++s == a.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (MODE == FUSED && lt >= 1) {
                const int pl = lt - 1, b = pl & 1;
                const uint32_t use = (uint32_t)(pl >> 1) & 1u;
                if (!mbar_wait(bars.a2full + 8 * b, use, abort_flag, a.err, lim) ||
                    !mbar_wait(bars.acc2empty + 8 * b, use ^ 1u, abort_flag, a.err, lim)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a2_s = base_s + a.off_a2 + (uint32_t)b * (uint32_t)a.nkb_mid * kBlk;
                    const uint32_t d = tmem_base + acc2_col + (uint32_t)b * (uint32_t)a.K;
                    const uint64_t a_base = sw128_kmajor_desc(a2_s), b_base = sw128_kmajor_desc(w2_s);
                    for (int kb = 0; kb < a.nkb_mid; kb++) {
                        const uint64_t ad = desc_advance(a_base, (uint32_t)kb * kBlk);
                        const uint64_t bd = desc_advance(b_base, (uint32_t)kb * (uint32_t)a.K * 128u);
                        const int n16 = min(4, (a.Cm - 64 * kb) / 16);
                        for (int k16 = 0; k16 < n16; k16++)
                            mma_f16(d, desc_advance(ad, 32u * k16), desc_advance(bd, 32u * k16), a.idesc2,
                                    (kb | k16) != 0 ? 1u : 0u);
                    }
                    mma_commit(bars.a2empty + 8 * b);
                    mma_commit(bars.acc2full + 8 * b);
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
    } else if (warp >= 2 && warp < 2 + kMidWarps) {
        // ===================================================== mid epilogue (conv1 -> A2)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const bool issuer = warp == 2 && lane == 0;
        for (int lt = 0; lt < my_tiles; lt++) {
            const int b = lt & 1;
            const uint32_t use = (uint32_t)(lt >> 1) & 1u;
            bool ok = mbar_wait(bars.acc1full + 8 * b, use, abort_flag, a.err, lim);
            if (MODE == FUSED) {
                if (ok) ok = mbar_wait(bars.a2empty + 8 * b, use ^ 1u, abort_flag, a.err, lim);
                if (!ok) break;
            } else {
                if (issuer) bulk_wait_group_read<0>();
                if (named_barrier_or(1, 32 * kMidWarps, !ok)) break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc1_col + (uint32_t)b * (uint32_t)a.Cm;
            const uint32_t dst = MODE == FUSED
                                     ? base_s + a.off_a2 + (uint32_t)b * (uint32_t)a.nkb_mid * kBlk
                                     : base_s + a.off_out;
            acc_to_smem<T, kMidKind, true>(a, taddr, a.Cm, s1_s, b1_s, a.act1, dst, row);
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.acc1empty + 8 * b);
            if (MODE == FUSED) {
                if (lane == 0) mbar_arrive(bars.a2full + 8 * b);
            } else {
                named_barrier(1, 32 * kMidWarps);
                if (issuer) {
                    const int t = (int)blockIdx.x + lt * (int)gridDim.x;
                    const int n = t / a.tiles_per_img;
                    store_tile(a, &a.tmap_out, dst, a.Cm, n, (t - n * a.tiles_per_img) * a.TH, kRowB);
                }
            }
        }
        if (MODE == CONV1 && issuer) bulk_wait_group<0>();
    } else if (MODE == FUSED && warp >= 2 + kMidWarps && warp < 2 + kMidWarps + kOutWarps) {
        // ===================================================== output epilogue (conv2 -> y)
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const bool issuer = warp == 2 + kMidWarps && lane == 0;
        for (int lt = 0; lt < my_tiles; lt++) {
            const int b = lt & 1;
            const bool ok = mbar_wait(bars.acc2full + 8 * b, (uint32_t)(lt >> 1) & 1u, abort_flag,
                                      a.err, lim);
            // two staging tiles: this one is free once the stores of tile lt - 2 have read it
            if (issuer) bulk_wait_group_read<1>();
            if (named_barrier_or(2, 32 * kOutWarps, !ok)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc2_col + (uint32_t)b * (uint32_t)a.K;
            const uint32_t dst = base_s + a.off_out + (uint32_t)b * a.out_bytes;
            acc_to_smem<T, kOutKind, false>(a, taddr, a.K, s2_s, b2_s, a.act2, dst, row);
            tc_fence_before();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars.acc2empty + 8 * b);
            named_barrier(2, 32 * kOutWarps);
            if (issuer) {
                const int t = (int)blockIdx.x + lt * (int)gridDim.x;
                const int n = t / a.tiles_per_img;
                store_tile(a, &a.tmap_out, dst, a.K, n, (t - n * a.tiles_per_img) * a.TH, kRowB);
            }
        }
        if (issuer) bulk_wait_group<0>();
    } else if (kI8 && warp >= kFirstConvWarp && warp < kFirstConvWarp + kConvWarps) {
        // ===================================================== INT8: int8 tile -> f16 A operand
        // Thread p converts pixel row p of the tile (TH * P = 128 rows): per 64-channel plane,
        // 64 int8 bytes -> 64 exact f16 values = one 128-byte row, 128B-swizzled as the tensor
        // core reads it (16-byte chunk c at c ^ (p & 7)).
        const int p = (warp - kFirstConvWarp) * 32 + lane;
        const uint32_t swz = (uint32_t)(p & 7);
        const __half2 bias2 = __float2half2_rn(I8::kBias);
        int s = 0;
        uint32_t ph = 0;
        for (int lt = 0; lt < my_tiles; lt++) {
            // the int8 tile has landed, and the MMAs of this stage's previous tile are done
            if (!mbar_wait(bars.full + 8 * s, ph, abort_flag, a.err, lim) ||
                !mbar_wait(bars.empty + 8 * s, ph ^ 1u, abort_flag, a.err, lim))
                break;
            const uint8_t *src = base_g + a.off_in8 + (uint32_t)s * a.in8_stage_stride + (uint32_t)p * 64u;
            const uint32_t dst = base_s + a.off_in + (uint32_t)s * a.in_stage_stride + (uint32_t)p * 128u;
            for (int kb = 0; kb < a.nkb_in; kb++) {
#pragma unroll
                for (int h = 0; h < 4; h++) {   // 16 channels -> two 16-byte chunks of f16
                    const uint4 v = *reinterpret_cast<const uint4 *>(src + (uint32_t)kb * a.plane8_bytes +
                                                                     (uint32_t)h * 16u);
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
                    const uint32_t row_s = dst + (uint32_t)kb * a.plane_bytes;
                    sts128(row_s + (((uint32_t)(2 * h) ^ swz) << 4), w[0], w[1], w[2], w[3]);
                    sts128(row_s + (((uint32_t)(2 * h + 1) ^ swz) << 4), w[4], w[5], w[6], w[7]);
                }
            }
            fence_proxy_async_smem();   // the f16 tile is read by the tensor core (async proxy)
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bars.full1 + 8 * s);
                mbar_arrive(bars.empty8 + 8 * s);
            }
            if (++s == a.stages) {
                s = 0;
                ph ^= 1u;
            }
        }
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

struct Layout {
    uint32_t off_w1, off_w2, off_a2, off_out, off_in, off_sb, off_bar, out_bytes, plane_bytes,
        in_stage_bytes, in_stage_stride, w1_bytes, w2_bytes, total;
    uint32_t off_in8, plane8_bytes, in8_stage_bytes, in8_stage_stride;   // INT8 input ring
    int stages;
};

Layout make_layout(const fcm_desc *d, const TcPlan &p, int cm, int mode, int smem_cap) {
    Layout L{};
    const int C = d->c, K = d->k_out, ks = d->ksize;
    const int nkb_in = C / 64, nkb_mid = (cm + 63) / 64;
    L.w1_bytes = (uint32_t)(ks * ks * nkb_in * cm) * 128u;
    L.w2_bytes = mode == FUSED ? (uint32_t)(nkb_mid * K) * 128u : 0u;
    const uint32_t a2 = mode == FUSED ? 2u * (uint32_t)nkb_mid * kBlk : 0u;
    const bool i8 = d->dtype == FCM_I8;
    // output staging: 64-channel blocks of kTileM rows of 128 (16-bit) or 64 (int8) bytes
    L.out_bytes = (uint32_t)(((mode == FUSED ? K : cm) + 63) / 64) * (i8 ? kTileM * 64u : kBlk);
    const uint32_t out = (mode == FUSED ? 2u : 1u) * L.out_bytes;
    L.off_w1 = 0;
    L.off_w2 = align_up(L.w1_bytes, 1024);
    L.off_a2 = align_up(L.off_w2 + L.w2_bytes, 1024);
    L.off_out = align_up(L.off_a2 + a2, 1024);
    L.off_in = align_up(L.off_out + out, 1024);
    L.plane_bytes = (uint32_t)(p.in_rows * p.tile_w) * 128u;
    L.in_stage_bytes = (uint32_t)nkb_in * L.plane_bytes;
    L.in_stage_stride = align_up(L.in_stage_bytes + 1024u, 1024);   // slack: taps read past the tile
    if (i8) {
        L.plane8_bytes = (uint32_t)(p.in_rows * p.tile_w) * 64u;
        L.in8_stage_bytes = (uint32_t)nkb_in * L.plane8_bytes;
        L.in8_stage_stride = align_up(L.in8_stage_bytes, 1024);
    }
    const uint32_t slot = L.in_stage_stride + L.in8_stage_stride;   // per stage: f16 (+ int8) tile
    const uint32_t sb = (uint32_t)(2 * cm + 2 * K) * 4;
    const uint32_t tail = align_up(sb, 16) + kBarBytes + 16 + 1024;
    int stages = kMaxStages;
    for (; stages >= 1; stages--)
        if ((int)(L.off_in + (uint32_t)stages * slot + tail) <= smem_cap) break;
    L.stages = stages;
    L.off_in8 = L.off_in + (uint32_t)std::max(stages, 0) * L.in_stage_stride;
    L.off_sb = L.off_in + (uint32_t)std::max(stages, 0) * slot;
    L.off_bar = L.off_sb + align_up(sb, 16);
    L.total = L.off_bar + kBarBytes + 16 + 1024;
    return L;
}

uint32_t pow2_cols(int n) {
    uint32_t c = 32;
    while ((int)c < n) c <<= 1;
    return c;
}

}  // namespace b2b
}  // namespace fcm

using namespace fcm::b2b;

int fcm_b2b_supported(const fcm_desc *d, int ho, int wo, int cm, const char **why) {
    auto no = [&](const char *w) {
        if (why) *why = w;
        return 0;
    };
    (void)ho;
    if (d->dtype == FCM_F32) return no("fp32 runs on CUDA cores");
    if (d->stride != 1) return no("dense conv1 on tensor cores needs stride 1");
    // INT8: two 1x1 convolutions (PWPW); C, Cm <= 256 keep every partial sum below 2^22
    if (d->dtype == FCM_I8 && (d->ksize != 1 || d->pad != 0))
        return no("INT8 back-to-back takes k = 1 (the PWPW module)");
    if (d->ksize != 1 && d->ksize != 3 && d->ksize != 5) return no("dense conv1 ksize must be 1, 3 or 5");
    if (d->c % 64 != 0 || d->c > 256) return no("dense conv1 needs C a multiple of 64, at most 256");
    if (cm % 16 != 0 || d->k_out % 16 != 0) return no("mid and k_out must be multiples of 16");
    if (cm + d->k_out > 256) return no("mid + k_out above 256 TMEM columns per buffer");
    if (wo + d->ksize - 1 > 128) return no("output width + ksize - 1 above 128");
    return 1;
}

fcm_status fcm_b2b_plan(const fcm_desc *d, int ho, int wo, int cm, int num_sms, int smem_cap,
                        TcPlan *p) {
    TcPlan t;
    t.tile_w = wo + d->ksize - 1 <= 64 ? 64 : 128;   // pitch of the input tile
    t.tile_h = kTileM / t.tile_w;
    if (d->tile_h > 0) t.tile_h = std::min(t.tile_h, d->tile_h);
    t.in_rows = t.tile_h + d->ksize - 1;
    t.in_cols = t.tile_w;
    t.chunk_c = d->c;
    t.nchunks = 1;
    t.tiles_w = 1;
    t.tiles_h = (ho + t.tile_h - 1) / t.tile_h;
    t.num_tiles = (long long)d->n * t.tiles_h;
    if (t.num_tiles >= (1LL << 31)) return FCM_ERR_UNSUPPORTED;
    Layout L = make_layout(d, t, cm, FUSED, smem_cap);
    if (L.stages < 2) return FCM_ERR_SMEM_BUDGET;
    t.stages = L.stages;
    t.smem_bytes = (int)L.total;
    t.threads = kThreads;
    t.ctas = (int)std::min<long long>(t.num_tiles, num_sms);
    t.tmem_cols = (int)pow2_cols(2 * (cm + d->k_out));
    if (d->dtype == FCM_I8) t.threads = kThreadsI8;
    *p = t;
    return FCM_OK;
}

fcm_status fcm_b2b_prepare(fcm_handle *h, const void *w1_host, const void *wp_host) {
    const fcm_desc &d = h->d;
    const int C = d.c, Cm = h->cm, K = d.k_out, ks = d.ksize;
    const int nkb_in = C / 64, nkb_mid = (Cm + 63) / 64;
    const bool i8 = d.dtype == FCM_I8;
    // 16-bit pattern of weight i: the storage value, or for INT8 the f16 of the int8 (exact)
    auto w16 = [&](const void *base, size_t i) -> uint16_t {
        if (i8) {
            __half hv = __float2half_rn((float)static_cast<const signed char *>(base)[i]);
            uint16_t b;
            memcpy(&b, &hv, 2);
            return b;
        }
        return static_cast<const uint16_t *>(base)[i];
    };
    // conv1: for each tap, a B image with Cm rows (output channels) over the C input channels
    std::vector<uint8_t> w1((size_t)ks * ks * nkb_in * Cm * 128, 0);   // w1_host: [Cm][ks][ks][C]
    for (int j = 0; j < Cm; j++)
        for (int tap = 0; tap < ks * ks; tap++)
            for (int c = 0; c < C; c++) {
                const int kb = c / 64;
                const size_t blk = ((size_t)tap * nkb_in + kb) * Cm * 128;
                const uint32_t off = fcm::tc::sw128_offset(j, c % 64, Cm, 2);
                const uint16_t v = w16(w1_host, ((size_t)j * ks * ks + tap) * C + c);
                memcpy(&w1[blk + off], &v, 2);
            }
    // conv2: K rows over Cm channels (wp_host: [K][Cm])
    h->wp_img_bytes = (size_t)nkb_mid * K * 128;
    std::vector<uint8_t> w2(h->wp_img_bytes, 0);
    for (int n = 0; n < K; n++)
        for (int c = 0; c < Cm; c++) {
            const uint16_t v = w16(wp_host, (size_t)n * Cm + c);
            memcpy(&w2[fcm::tc::sw128_offset(n, c, K, 2)], &v, 2);
        }
    h->w1_img_bytes = w1.size();
    if (cudaMalloc(&h->w1_img, w1.size()) != cudaSuccess ||
        cudaMemcpy(h->w1_img, w1.data(), w1.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMalloc(&h->wp_img, w2.size()) != cudaSuccess ||
        cudaMemcpy(h->wp_img, w2.data(), w2.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return fcm_fail(FCM_ERR_CUDA, "back-to-back weight images: %s",
                        cudaGetErrorString(cudaGetLastError()));
    // INT8: the layer-by-layer second stage runs on the DW->PW kernel's identity stencil
    if (i8) return fcm_i8_prepare(h, nullptr);
    return FCM_OK;
}

namespace {

template <typename T, int KS, int MODE>
cudaError_t launch_t(const Args &a, int ctas, uint32_t smem, cudaStream_t st) {
    static std::atomic<unsigned long long> attr_ctx{0};
    return launch_pdl(b2b_kernel<T, KS, MODE>, attr_ctx, ctas,
                      std::is_same<T, int8_t>::value ? kThreadsI8 : kThreads, smem, st, a);
}

template <typename T, int KS>
cudaError_t dispatch_mode(const Args &a, int mode, int ctas, uint32_t smem, cudaStream_t st) {
    return mode == FUSED ? launch_t<T, KS, FUSED>(a, ctas, smem, st)
                         : launch_t<T, KS, CONV1>(a, ctas, smem, st);
}

template <typename T>
cudaError_t dispatch_ks(const Args &a, int ks, int mode, int ctas, uint32_t smem, cudaStream_t st) {
    if (ks == 1) return dispatch_mode<T, 1>(a, mode, ctas, smem, st);
    if (ks == 3) return dispatch_mode<T, 3>(a, mode, ctas, smem, st);
    if (ks == 5) return dispatch_mode<T, 5>(a, mode, ctas, smem, st);
    return cudaErrorInvalidValue;
}

cudaError_t dispatch_dtype(const Args &a, int dtype, int ks, int mode, int ctas, uint32_t smem,
                           cudaStream_t st) {
    if (dtype == FCM_I8)
        return ks == 1 ? dispatch_mode<int8_t, 1>(a, mode, ctas, smem, st) : cudaErrorInvalidValue;
    return dtype == FCM_F16 ? dispatch_ks<__half>(a, ks, mode, ctas, smem, st)
                            : dispatch_ks<__nv_bfloat16>(a, ks, mode, ctas, smem, st);
}

}  // namespace

cudaError_t launch_tc_b2b(const fcm_handle *h, int mode_in, const void *in, void *out,
                          cudaStream_t st) {
    const fcm_desc &d = h->d;
    const TcPlan &p = h->tc;
    const int mode = mode_in == FCM_MODE_FUSED ? FUSED : CONV1;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    Layout L = make_layout(&d, p, h->cm, mode, h->smem_optin);
    if (L.stages < 2) return cudaErrorInvalidConfiguration;
    Args a;
    memset(&a, 0, sizeof(a));
    const bool i8 = d.dtype == FCM_I8;
    const CUtensorMapDataType dt = i8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : d.dtype == FCM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t es = (cuuint64_t)fcm_dtype_bytes(d.dtype);
    {
        // 16-bit: straight into the 128B-swizzled A operand; INT8: into the int8 ring (64-byte
        // rows per 64-channel plane, unswizzled) that the converter warps read
        cuuint64_t gdim[4] = {(cuuint64_t)d.c, (cuuint64_t)d.w, (cuuint64_t)d.h, (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)d.c * es, (cuuint64_t)d.w * d.c * es,
                                 (cuuint64_t)d.h * d.w * d.c * es};
        cuuint32_t box[4] = {64, (cuuint32_t)p.tile_w, (cuuint32_t)p.in_rows, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&a.tmap_in, dt, 4, const_cast<void *>(in), gdim, gstride, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                i8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const int ch = mode == FUSED ? d.k_out : h->cm;
        cuuint64_t gdim[4] = {(cuuint64_t)ch, (cuuint64_t)h->wo, (cuuint64_t)h->ho, (cuuint64_t)d.n};
        cuuint64_t gstride[3] = {(cuuint64_t)ch * es, (cuuint64_t)h->wo * ch * es,
                                 (cuuint64_t)h->ho * h->wo * ch * es};
        cuuint32_t box[4] = {64, (cuuint32_t)p.tile_w, 1, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        if (enc(&a.tmap_out, dt, 4, out, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                i8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    a.w1_img = static_cast<const uint8_t *>(h->w1_img);
    a.w2_img = static_cast<const uint8_t *>(h->wp_img);
    a.s1 = h->s1;
    a.b1 = h->b1;
    a.s2 = h->s2;
    a.b2 = h->b2;
    if (h->b1 && h->b1 == h->b1_host_of && (h->cm == 64 || h->cm == 128)) {
        memcpy(a.b1c, h->b1_host, sizeof(float) * (size_t)h->cm);
        a.b1c_n = h->cm;
    }
    if (h->b2 && h->b2 == h->b2_host_of && (d.k_out == 64 || d.k_out == 128)) {
        memcpy(a.b2c, h->b2_host, sizeof(float) * (size_t)d.k_out);
        a.b2c_n = d.k_out;
    }
    a.err = h->d_err;
    a.wait_limit_ns = kWaitLimitNs;
    a.num_tiles = (int)p.num_tiles;
    a.tiles_per_img = p.tiles_h;
    a.C = d.c;
    a.Cm = h->cm;
    a.K = d.k_out;
    a.Ho = h->ho;
    a.Wo = h->wo;
    a.ks = d.ksize;
    a.pad = d.pad;
    a.P = p.tile_w;
    a.TH = p.tile_h;
    a.in_rows = p.in_rows;
    a.nkb_in = d.c / 64;
    a.nkb_mid = (h->cm + 63) / 64;
    a.stages = L.stages;
    a.act1 = d.act1;
    a.act2 = d.act2;
    a.tmem_cols = (uint32_t)p.tmem_cols;
    a.idesc1 = idesc_f16(d.dtype == FCM_BF16, kTileM, h->cm);   // INT8: f16 operands
    a.idesc2 = idesc_f16(d.dtype == FCM_BF16, kTileM, d.k_out);
    a.w1_bytes = L.w1_bytes;
    a.w2_bytes = (uint32_t)h->wp_img_bytes;
    a.plane_bytes = L.plane_bytes;
    a.in_stage_bytes = L.in_stage_bytes;
    a.in_stage_stride = L.in_stage_stride;
    a.off_w1 = L.off_w1;
    a.off_w2 = L.off_w2;
    a.off_a2 = L.off_a2;
    a.off_out = L.off_out;
    a.out_bytes = L.out_bytes;
    a.off_in = L.off_in;
    a.off_sb = L.off_sb;
    a.off_bar = L.off_bar;
    a.off_in8 = L.off_in8;
    a.plane8_bytes = L.plane8_bytes;
    a.in8_stage_bytes = L.in8_stage_bytes;
    a.in8_stage_stride = L.in8_stage_stride;
    const int ctas = std::min(a.num_tiles, h->num_sms);
    return dispatch_dtype(a, d.dtype, d.ksize, mode, ctas, L.total, st);
}
