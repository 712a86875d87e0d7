// tc_dwpw.cuh -- declarations shared by the DW->PW kernel's host code (tc_dwpw.cu) and the
// translation units that instantiate the kernel (tc_dwpw_inst_*.cu): constants, the kernel
// arguments, and the launcher template (defined in tc_dwpw_kernel.cuh).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fcm_internal.h"
#include "tc_common.cuh"

namespace fcm {
namespace tc {

// Two epilogue warps per TMEM lane quadrant, half the columns each (measured on the MobileNet
// layer: 39.1 us against 41.1 us with one per quadrant).  At 24 warps a thread gets 80 registers,
// so the chunk-bound DW warps read their taps from shared memory instead of holding them.
constexpr int kEpiWarps = 8;
constexpr bool kDwTapsInRegs = false;
// Chunk-bound DW warps (768-thread tier, 16-bit storage) hold their channels' scale and bias
// in registers instead of loading them for every unit (MobileNet layer: 29.8 us against 30.8 us
// a launch, back to back).
constexpr bool kDwNormInRegs = true;
constexpr int kFirstDwWarp = 2 + kEpiWarps;
constexpr int kMaxDwWarps = 10;   // 16 warps in all: up to 128 registers a thread
constexpr int kMaxThreads = 32 * (kFirstDwWarp + kMaxDwWarps);
// Chunk-bound DW warps (each warp serves one channel chunk and keeps its taps in registers):
// up to 14 DW warps, 20 in all, 96 registers a thread.
constexpr int kMaxDwWarpsBound = 14;
constexpr int kMaxThreadsBound = 32 * (kFirstDwWarp + kMaxDwWarpsBound);
// Chunk-bound plans of a single 64-channel chunk (7 stencil warps for a 112-pixel tile) launch
// at most this many threads; their instantiations (DWB = 2) are compiled for it, so a thread
// gets 120 registers instead of the 80 that 768 threads leave.
constexpr int kMaxDwWarpsBound2 = 7;
constexpr int kMaxThreadsBound2 = 32 * (kFirstDwWarp + kMaxDwWarpsBound2);
constexpr int kR = 4;          // output pixels per DW work unit (along W)
constexpr int kTileM = 128;    // MMA M: pixels per output tile (padded)
constexpr int kMaxStages = 8;
constexpr int kMaxChunks = 16;

enum Mode { FUSED = 0, DWONLY = 1, PWONLY = 2 };

constexpr int kMaxBiasParams = 128;   // biases passed as kernel parameters (Args::b2c)

struct Args {
    CUtensorMap tmap;          // x (FUSED/DWONLY: 4-D C,W,H,N) or m (PWONLY: 2-D C,P)
    CUtensorMap tmap_out;      // y: 4-D K,Wo,Ho,N box (64,tile_w,tile_h,1) or 2-D K,P box (64,128)
    void *out;                 // m for DWONLY (direct stores)
    const uint8_t *wp_img;     // B operand image (K rows, swizzled, K-major)
    const uint4 *wdw;          // DW taps, storage dtype, [k*k][C/8] x 8 channels
    const float *s1, *b1, *s2, *b2;
    const float *q1;           // INT8: 1152 * sum of each channel's taps (removed from the stencil)
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
    // The 1x1's biases as kernel parameters (b2c_n = K when K is 64 or 128, else 0): the
    // epilogue's FMAs then read them as constant operands instead of loading them from shared
    // memory (measured on the MobileNet layer: 30.6 us against 32.0 us a launch)
    int b2c_n;
    float b2c[kMaxBiasParams];
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
// bytes of one 64-channel block of the output stage (kTileM rows of 64 elements)
constexpr int out_block_bytes(int esize) { return kTileM * 64 * esize; }

// Launch dwpw_kernel<T, KS, S, MODE, DWB> (instantiated in tc_dwpw_inst_*.cu).
template <typename T, int KS, int S, int MODE, int DWB>
cudaError_t launch_k(const Args &a, int ctas, int threads, uint32_t smem, cudaStream_t st);

}  // namespace tc
}  // namespace fcm
