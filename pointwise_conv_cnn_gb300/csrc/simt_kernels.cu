// simt_kernels.cu -- CUDA-core (SIMT) kernels of the module: the fp32 path and the fallback
// for shapes the tensor-core kernels do not take.
//
//   k_conv1_dw   depthwise k x k + scale/bias/act      -> intermediate in HBM  (LBL DW)
//   k_conv1_dense dense k x k + scale/bias/act         -> intermediate in HBM  (LBL conv1)
//   k_pw         1x1 conv + scale/bias/act              (LBL PW)
//   k_fused      conv1 -> shared-memory commBuffer -> 1x1, one pass (FCM)
//
// The fused kernel follows the FCM structure of "Fusing Depthwise and Pointwise Convolutions
// for Efficient Inference on GPUs", section III-B: the first layer writes its tile of the
// intermediate, over all channels (section II-D), into a shared buffer, the block
// synchronizes, and the second layer reads it and writes the output once (output-stationary,
// section IV-A).  The per-element arithmetic (tap order, fmaf for the norm, rounding of the
// intermediate to the storage type) is the same in the fused and the layer-by-layer kernels,
// so fused == conv1-then-PW bit for bit.
#include <cuda_runtime.h>

#include <algorithm>

#include "fcm_device.cuh"
#include "fcm_internal.h"

namespace fcm {
namespace {

constexpr int kPwPixels = 32;      // pixels per CTA in the PW and fused kernels
constexpr int kThreads = 256;

// Depthwise value for VEC channels c0..c0+VEC-1 of output pixel (n, ho, wo), before the norm.
template <typename T, int VEC>
__device__ __forceinline__ void dw_point(const T *__restrict__ x, const float *__restrict__ wt,
                                         int n, int ho, int wo, int c0, int H, int W, int C,
                                         int k, int s, int p, float (&acc)[VEC]) {
#pragma unroll
    for (int v = 0; v < VEC; v++) acc[v] = 0.0f;
    for (int i = 0; i < k; i++) {
        int hi = ho * s - p + i;
        if (hi < 0 || hi >= H) continue;
        for (int j = 0; j < k; j++) {
            int wi = wo * s - p + j;
            if (wi < 0 || wi >= W) continue;
            float xv[VEC];
            load_vec<T, VEC>(x + (((size_t)n * H + hi) * W + wi) * C + c0, xv);
            const float *wr = wt + (size_t)(i * k + j) * C + c0;
#pragma unroll
            for (int v = 0; v < VEC; v++) acc[v] = fmaf(xv[v], __ldg(wr + v), acc[v]);
        }
    }
}

// Dense value for output channel j of pixel (n, ho, wo), before the norm; taps (r, u) then c.
template <typename T>
__device__ __forceinline__ float dense_point(const T *__restrict__ x, const float *__restrict__ wt,
                                             int n, int ho, int wo, int j, int H, int W, int C,
                                             int Cm, int k, int s, int p) {
    float acc = 0.0f;
    for (int r = 0; r < k; r++) {
        int hi = ho * s - p + r;
        if (hi < 0 || hi >= H) continue;
        for (int u = 0; u < k; u++) {
            int wi = wo * s - p + u;
            if (wi < 0 || wi >= W) continue;
            const T *xp = x + (((size_t)n * H + hi) * W + wi) * C;
            const float *wp = wt + (size_t)((r * k + u) * C) * Cm + j;
            for (int c = 0; c < C; c++)
                acc = fmaf(Storage<T>::to_f(xp[c]), __ldg(wp + (size_t)c * Cm), acc);
        }
    }
    return acc;
}

template <typename T, int VEC>
__global__ void __launch_bounds__(kThreads) k_conv1_dw(
    const T *__restrict__ x, const float *__restrict__ wt, const float *__restrict__ s1,
    const float *__restrict__ b1, T *__restrict__ m, int N, int H, int W, int C, int Ho, int Wo,
    int k, int s, int p, int act) {
    const int cv_per_px = C / VEC;
    const long long total = (long long)N * Ho * Wo * cv_per_px;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int cv = (int)(idx % cv_per_px);
        long long pix = idx / cv_per_px;
        int wo = (int)(pix % Wo);
        long long t = pix / Wo;
        int ho = (int)(t % Ho);
        int n = (int)(t / Ho);
        int c0 = cv * VEC;
        float acc[VEC];
        dw_point<T, VEC>(x, wt, n, ho, wo, c0, H, W, C, k, s, p, acc);
#pragma unroll
        for (int v = 0; v < VEC; v++)
            acc[v] = act_apply(fmaf(__ldg(s1 + c0 + v), acc[v], __ldg(b1 + c0 + v)), act);
        store_vec<T, VEC>(m + pix * C + c0, acc);
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_conv1_dense(
    const T *__restrict__ x, const float *__restrict__ wt, const float *__restrict__ s1,
    const float *__restrict__ b1, T *__restrict__ m, int N, int H, int W, int C, int Cm, int Ho,
    int Wo, int k, int s, int p, int act) {
    const long long total = (long long)N * Ho * Wo * Cm;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        int j = (int)(idx % Cm);
        long long pix = idx / Cm;
        int wo = (int)(pix % Wo);
        long long t = pix / Wo;
        int ho = (int)(t % Ho);
        int n = (int)(t / Ho);
        float acc = dense_point<T>(x, wt, n, ho, wo, j, H, W, C, Cm, k, s, p);
        m[idx] = Storage<T>::from_f(act_apply(fmaf(__ldg(s1 + j), acc, __ldg(b1 + j)), act));
    }
}

// 1x1 convolution of a tile of kPwPixels pixels held (as fp32) in shared memory `tile`
// [kPwPixels][Cm]; thread item = (group of 4 pixels, output channel).
template <typename T>
__device__ __forceinline__ void pw_tile(const float *tile, long long p0, long long P, int Cm,
                                        int K, const float *__restrict__ wpt,
                                        const float *__restrict__ s2,
                                        const float *__restrict__ b2, int act, T *__restrict__ y) {
    const int items = (kPwPixels / 4) * K;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
        int kk = it % K;
        int pg = it / K;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const float *t0 = tile + (size_t)(pg * 4) * Cm;
        for (int c = 0; c < Cm; c++) {
            float w = __ldg(wpt + (size_t)c * K + kk);
#pragma unroll
            for (int q = 0; q < 4; q++) acc[q] = fmaf(t0[(size_t)q * Cm + c], w, acc[q]);
        }
        float sc = __ldg(s2 + kk), bi = __ldg(b2 + kk);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            long long pix = p0 + pg * 4 + q;
            if (pix < P) y[pix * K + kk] = Storage<T>::from_f(act_apply(fmaf(sc, acc[q], bi), act));
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads) k_pw(
    const T *__restrict__ m, const float *__restrict__ wpt, const float *__restrict__ s2,
    const float *__restrict__ b2, T *__restrict__ y, long long P, int Cm, int K, int act) {
    extern __shared__ float tile[];   // [kPwPixels][Cm]
    for (long long blk = blockIdx.x; blk * kPwPixels < P; blk += gridDim.x) {
        long long p0 = blk * kPwPixels;
        __syncthreads();
        for (int e = threadIdx.x; e < kPwPixels * Cm; e += blockDim.x) {
            long long pix = p0 + e / Cm;
            tile[e] = pix < P ? Storage<T>::to_f(m[p0 * Cm + e]) : 0.0f;
        }
        __syncthreads();
        pw_tile<T>(tile, p0, P, Cm, K, wpt, s2, b2, act, y);
    }
}

// Fused conv1 -> commBuffer -> 1x1.  The commBuffer holds the intermediate of kPwPixels
// consecutive output pixels over all Cm channels, rounded to the storage type.  A depthwise
// conv1 works on VEC channels per thread item (16-byte vectors, as k_conv1_dw does), so a tile
// of a narrow layer is one item per thread; the per-channel arithmetic is the same either way.
template <typename T, bool DENSE, int VEC>
__global__ void __launch_bounds__(kThreads) k_fused(
    const T *__restrict__ x, const float *__restrict__ w1t, const float *__restrict__ s1,
    const float *__restrict__ b1, const float *__restrict__ wpt, const float *__restrict__ s2,
    const float *__restrict__ b2, T *__restrict__ y, int N, int H, int W, int C, int Cm, int K,
    int Ho, int Wo, int k, int s, int p, int act1, int act2) {
    extern __shared__ float comm[];   // [kPwPixels][Cm]
    const long long P = (long long)N * Ho * Wo;
    const int cv_per_px = Cm / VEC;
    for (long long blk = blockIdx.x; blk * kPwPixels < P; blk += gridDim.x) {
        long long p0 = blk * kPwPixels;
        __syncthreads();
        for (int e = threadIdx.x; e < kPwPixels * cv_per_px; e += blockDim.x) {
            long long pix = p0 + e / cv_per_px;
            const int j = (e % cv_per_px) * VEC;
            float v[VEC];
#pragma unroll
            for (int q = 0; q < VEC; q++) v[q] = 0.0f;
            if (pix < P) {
                int wo = (int)(pix % Wo);
                long long t = pix / Wo;
                int ho = (int)(t % Ho);
                int n = (int)(t / Ho);
                float acc[VEC];
                if constexpr (DENSE) {
                    acc[0] = dense_point<T>(x, w1t, n, ho, wo, j, H, W, C, Cm, k, s, p);
                } else {
                    dw_point<T, VEC>(x, w1t, n, ho, wo, j, H, W, C, k, s, p, acc);
                }
                // round to the storage type exactly as the layer-by-layer path stores it
#pragma unroll
                for (int q = 0; q < VEC; q++)
                    v[q] = Storage<T>::to_f(Storage<T>::from_f(
                        act_apply(fmaf(__ldg(s1 + j + q), acc[q], __ldg(b1 + j + q)), act1)));
            }
#pragma unroll
            for (int q = 0; q < VEC; q++) comm[(pix - p0) * Cm + j + q] = v[q];
        }
        __syncthreads();
        pw_tile<T>(comm, p0, P, Cm, K, wpt, s2, b2, act2, y);
    }
}

// PWDW in one pass: thread item = (output pixel, channel j).  The intermediate under each
// depthwise tap is the 1x1 convolution of the input pixel there, recomputed (PWDW_R), rounded
// to the storage type as the layer-by-layer path stores it; taps over the padding read zero.
// Same operation order as k_pw followed by k_conv1_dw, so fused == unfused bit for bit.
template <typename T>
__global__ void __launch_bounds__(kThreads) k_fused_pwdw(
    const T *__restrict__ x, const float *__restrict__ wq, const float *__restrict__ s1,
    const float *__restrict__ b1, const float *__restrict__ wd, const float *__restrict__ s2,
    const float *__restrict__ b2, T *__restrict__ y, int N, int H, int W, int C, int Cm, int Ho,
    int Wo, int k, int s, int p, int act1, int act2) {
    const long long total = (long long)N * Ho * Wo * Cm;
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(idx % Cm);
        const long long pix = idx / Cm;
        const int wo = (int)(pix % Wo);
        const long long t = pix / Wo;
        const int ho = (int)(t % Ho);
        const int n = (int)(t / Ho);
        float acc = 0.0f;
        for (int i = 0; i < k; i++) {
            const int hi = ho * s - p + i;
            if (hi < 0 || hi >= H) continue;
            for (int u = 0; u < k; u++) {
                const int wi = wo * s - p + u;
                if (wi < 0 || wi >= W) continue;
                const T *xp = x + (((size_t)n * H + hi) * W + wi) * C;
                float q = 0.0f;
                for (int c = 0; c < C; c++)
                    q = fmaf(Storage<T>::to_f(xp[c]), __ldg(wq + (size_t)c * Cm + j), q);
                const float mval = Storage<T>::to_f(Storage<T>::from_f(
                    act_apply(fmaf(__ldg(s1 + j), q, __ldg(b1 + j)), act1)));
                acc = fmaf(mval, __ldg(wd + (size_t)(i * k + u) * Cm + j), acc);
            }
        }
        y[idx] = Storage<T>::from_f(act_apply(fmaf(__ldg(s2 + j), acc, __ldg(b2 + j)), act2));
    }
}

// PWDW in one pass with the intermediate tiled in shared memory: a block takes TH output rows
// of one image over the full width and CC intermediate channels.  It first computes the
// intermediate over the rows and columns those outputs read (the 1x1 convolution of each input
// pixel there, rounded to the storage type, as the layer-by-layer path stores it; zero where the
// depthwise layer pads), then the depthwise layer from shared memory.  Each intermediate value
// is computed once per block instead of once per depthwise tap, and the per-element arithmetic
// is that of k_pw followed by k_conv1_dw, so fused == unfused bit for bit.
template <typename T>
__global__ void __launch_bounds__(kThreads) k_fused_pwdw_tiled(
    const T *__restrict__ x, const float *__restrict__ wq, const float *__restrict__ s1,
    const float *__restrict__ b1, const float *__restrict__ wd, const float *__restrict__ s2,
    const float *__restrict__ b2, T *__restrict__ y, int N, int H, int W, int C, int Cm, int Ho,
    int Wo, int k, int s, int p, int act1, int act2, int TH, int CC) {
    extern __shared__ float mt[];   // [R][Q][CC]: halo rows x halo columns x channels
    const int R = (TH - 1) * s + k, Q = (Wo - 1) * s + k;
    const int row_tiles = (Ho + TH - 1) / TH, ch_tiles = (Cm + CC - 1) / CC;
    const long long blocks = (long long)N * row_tiles * ch_tiles;
    for (long long b = blockIdx.x; b < blocks; b += gridDim.x) {
        const int ct = (int)(b % ch_tiles);
        const long long rest = b / ch_tiles;
        const int rt = (int)(rest % row_tiles);
        const int n = (int)(rest / row_tiles);
        const int ho0 = rt * TH, j0 = ct * CC;
        const int hi0 = ho0 * s - p, wi0 = -p;
        __syncthreads();
        for (int e = threadIdx.x; e < R * Q * CC; e += blockDim.x) {
            const int jj = e % CC;
            const int q = (e / CC) % Q;
            const int r = e / (CC * Q);
            const int hi = hi0 + r, wi = wi0 + q, j = j0 + jj;
            float v = 0.0f;
            if (hi >= 0 && hi < H && wi >= 0 && wi < W && j < Cm) {
                const T *xp = x + (((size_t)n * H + hi) * W + wi) * C;
                float acc = 0.0f;
                for (int c = 0; c < C; c++)
                    acc = fmaf(Storage<T>::to_f(xp[c]), __ldg(wq + (size_t)c * Cm + j), acc);
                v = Storage<T>::to_f(Storage<T>::from_f(
                    act_apply(fmaf(__ldg(s1 + j), acc, __ldg(b1 + j)), act1)));
            }
            mt[e] = v;
        }
        __syncthreads();
        const int rows = min(TH, Ho - ho0);
        for (int e = threadIdx.x; e < rows * Wo * CC; e += blockDim.x) {
            const int jj = e % CC;
            const int wo = (e / CC) % Wo;
            const int r = e / (CC * Wo);
            const int j = j0 + jj, ho = ho0 + r;
            if (j >= Cm) continue;
            float acc = 0.0f;
            for (int i = 0; i < k; i++) {
                const int hi = ho * s - p + i;
                if (hi < 0 || hi >= H) continue;
                for (int u = 0; u < k; u++) {
                    const int wi = wo * s - p + u;
                    if (wi < 0 || wi >= W) continue;
                    const float mv = mt[((r * s + i) * Q + wo * s + u) * CC + jj];
                    acc = fmaf(mv, __ldg(wd + (size_t)(i * k + u) * Cm + j), acc);
                }
            }
            y[(((size_t)n * Ho + ho) * Wo + wo) * Cm + j] =
                Storage<T>::from_f(act_apply(fmaf(__ldg(s2 + j), acc, __ldg(b2 + j)), act2));
        }
    }
}

int grid_for(long long work_items, int threads, int num_sms) {
    long long blocks = (work_items + threads - 1) / threads;
    long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (int)blocks;
}

template <typename T>
cudaError_t conv1_t(const fcm_handle *h, const void *xin, void *mout, cudaStream_t st) {
    const fcm_desc &d = h->d;
    const T *x = static_cast<const T *>(xin);
    T *m = static_cast<T *>(mout);
    if (d.conv1 == FCM_CONV1_DENSE) {
        long long items = (long long)d.n * h->ho * h->wo * h->cm;
        k_conv1_dense<T><<<grid_for(items, kThreads, h->num_sms), kThreads, 0, st>>>(
            x, h->w1t, h->s1, h->b1, m, d.n, d.h, d.w, d.c, h->cm, h->ho, h->wo, d.ksize,
            d.stride, d.pad, d.act1);
    } else {
        constexpr int V16 = 16 / (int)sizeof(T);
        if (d.c % V16 == 0) {
            long long items = (long long)d.n * h->ho * h->wo * (d.c / V16);
            k_conv1_dw<T, V16><<<grid_for(items, kThreads, h->num_sms), kThreads, 0, st>>>(
                x, h->w1t, h->s1, h->b1, m, d.n, d.h, d.w, d.c, h->ho, h->wo, d.ksize, d.stride,
                d.pad, d.act1);
        } else {
            long long items = (long long)d.n * h->ho * h->wo * d.c;
            k_conv1_dw<T, 1><<<grid_for(items, kThreads, h->num_sms), kThreads, 0, st>>>(
                x, h->w1t, h->s1, h->b1, m, d.n, d.h, d.w, d.c, h->ho, h->wo, d.ksize, d.stride,
                d.pad, d.act1);
        }
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t pw_t(const fcm_handle *h, const void *min, void *yout, cudaStream_t st) {
    long long P = (long long)h->d.n * h->ho * h->wo;
    size_t smem = sizeof(float) * kPwPixels * h->cm;
    cudaError_t e = cudaFuncSetAttribute(k_pw<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    long long blocks = (P + kPwPixels - 1) / kPwPixels;
    int grid = (int)(blocks < (long long)h->num_sms * 8 ? blocks : (long long)h->num_sms * 8);
    k_pw<T><<<grid, kThreads, smem, st>>>(static_cast<const T *>(min), h->wpt, h->s2, h->b2,
                                          static_cast<T *>(yout), P, h->cm, h->d.k_out,
                                          h->d.act2);
    return cudaGetLastError();
}

template <typename T>
cudaError_t fused_t(const fcm_handle *h, const void *xin, void *yout, cudaStream_t st) {
    const fcm_desc &d = h->d;
    long long P = (long long)d.n * h->ho * h->wo;
    size_t smem = sizeof(float) * kPwPixels * h->cm;
    long long blocks = (P + kPwPixels - 1) / kPwPixels;
    int grid = (int)(blocks < (long long)h->num_sms * 8 ? blocks : (long long)h->num_sms * 8);
    auto launch = [&](auto kernel) -> cudaError_t {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kernel<<<grid, kThreads, smem, st>>>(
            static_cast<const T *>(xin), h->w1t, h->s1, h->b1, h->wpt, h->s2, h->b2,
            static_cast<T *>(yout), d.n, d.h, d.w, d.c, h->cm, d.k_out, h->ho, h->wo, d.ksize,
            d.stride, d.pad, d.act1, d.act2);
        return cudaGetLastError();
    };
    constexpr int V16 = 16 / (int)sizeof(T);
    if (d.conv1 == FCM_CONV1_DENSE) return launch(k_fused<T, true, 1>);
    if (h->cm % V16 == 0) return launch(k_fused<T, false, V16>);
    return launch(k_fused<T, false, 1>);
}

// PWDW layer by layer: the 1x1 convolution x -> m [N,H,W,Cm] (k_pw with C inputs), then the
// depthwise convolution m -> y (k_conv1_dw over Cm channels).
template <typename T>
cudaError_t pwdw_first_t(const fcm_handle *h, const void *xin, void *mout, cudaStream_t st) {
    const fcm_desc &d = h->d;
    long long P = (long long)d.n * d.h * d.w;
    size_t smem = sizeof(float) * kPwPixels * d.c;
    cudaError_t e = cudaFuncSetAttribute(k_pw<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    long long blocks = (P + kPwPixels - 1) / kPwPixels;
    int grid = (int)(blocks < (long long)h->num_sms * 8 ? blocks : (long long)h->num_sms * 8);
    k_pw<T><<<grid, kThreads, smem, st>>>(static_cast<const T *>(xin), h->w1t, h->s1, h->b1,
                                          static_cast<T *>(mout), P, d.c, h->cm, d.act1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t pwdw_second_t(const fcm_handle *h, const void *min, void *yout, cudaStream_t st) {
    const fcm_desc &d = h->d;
    const T *m = static_cast<const T *>(min);
    T *y = static_cast<T *>(yout);
    constexpr int V16 = 16 / (int)sizeof(T);
    if (h->cm % V16 == 0) {
        long long items = (long long)d.n * h->ho * h->wo * (h->cm / V16);
        k_conv1_dw<T, V16><<<grid_for(items, kThreads, h->num_sms), kThreads, 0, st>>>(
            m, h->wpt, h->s2, h->b2, y, d.n, d.h, d.w, h->cm, h->ho, h->wo, d.ksize, d.stride,
            d.pad, d.act2);
    } else {
        long long items = (long long)d.n * h->ho * h->wo * h->cm;
        k_conv1_dw<T, 1><<<grid_for(items, kThreads, h->num_sms), kThreads, 0, st>>>(
            m, h->wpt, h->s2, h->b2, y, d.n, d.h, d.w, h->cm, h->ho, h->wo, d.ksize, d.stride,
            d.pad, d.act2);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t pwdw_fused_t(const fcm_handle *h, const void *xin, void *yout, cudaStream_t st) {
    const fcm_desc &d = h->d;
    // the tiled kernel with the largest channel slice whose intermediate tile fits 96 KB of
    // shared memory (four output rows a block, fewer for short images)
    const int TH = std::min(4, h->ho);
    const long long R = (long long)(TH - 1) * d.stride + d.ksize;
    const long long Q = (long long)(h->wo - 1) * d.stride + d.ksize;
    for (int CC = 32; CC >= 1; CC >>= 1) {
        const long long smem = R * Q * CC * (long long)sizeof(float);
        if (smem > 96 * 1024) continue;
        cudaError_t e = cudaFuncSetAttribute(k_fused_pwdw_tiled<T>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const long long blocks = (long long)d.n * ((h->ho + TH - 1) / TH) * ((h->cm + CC - 1) / CC);
        const int grid = (int)std::min<long long>(blocks, (long long)h->num_sms * 8);
        k_fused_pwdw_tiled<T><<<grid, kThreads, (size_t)smem, st>>>(
            static_cast<const T *>(xin), h->w1t, h->s1, h->b1, h->wpt, h->s2, h->b2,
            static_cast<T *>(yout), d.n, d.h, d.w, d.c, h->cm, h->ho, h->wo, d.ksize, d.stride,
            d.pad, d.act1, d.act2, TH, CC);
        return cudaGetLastError();
    }
    // a row of the halo does not fit even one channel: one thread per output element
    long long items = (long long)d.n * h->ho * h->wo * h->cm;
    k_fused_pwdw<T><<<grid_for(items, kThreads, h->num_sms), kThreads, 0, st>>>(
        static_cast<const T *>(xin), h->w1t, h->s1, h->b1, h->wpt, h->s2, h->b2,
        static_cast<T *>(yout), d.n, d.h, d.w, d.c, h->cm, h->ho, h->wo, d.ksize, d.stride,
        d.pad, d.act1, d.act2);
    return cudaGetLastError();
}

}  // namespace
}  // namespace fcm

#define FCM_BY_DTYPE(fn, ...)                                              \
    switch (h->d.dtype) {                                                   \
    case FCM_F32: return fcm::fn<float>(__VA_ARGS__);                       \
    case FCM_F16: return fcm::fn<__half>(__VA_ARGS__);                      \
    default: return fcm::fn<__nv_bfloat16>(__VA_ARGS__);                   \
    }

cudaError_t launch_pwdw_fused_simt(const fcm_handle *h, const void *x, void *y, cudaStream_t st) {
    FCM_BY_DTYPE(pwdw_fused_t, h, x, y, st)
}

cudaError_t launch_pwdw_first_simt(const fcm_handle *h, const void *x, void *m, cudaStream_t st) {
    FCM_BY_DTYPE(pwdw_first_t, h, x, m, st)
}

cudaError_t launch_pwdw_second_simt(const fcm_handle *h, const void *m, void *y, cudaStream_t st) {
    FCM_BY_DTYPE(pwdw_second_t, h, m, y, st)
}

cudaError_t launch_conv1_simt(const fcm_handle *h, const void *x, void *m, cudaStream_t st) {
    switch (h->d.dtype) {
    case FCM_F32: return fcm::conv1_t<float>(h, x, m, st);
    case FCM_F16: return fcm::conv1_t<__half>(h, x, m, st);
    default: return fcm::conv1_t<__nv_bfloat16>(h, x, m, st);
    }
}

cudaError_t launch_pw_simt(const fcm_handle *h, const void *m, void *y, cudaStream_t st) {
    switch (h->d.dtype) {
    case FCM_F32: return fcm::pw_t<float>(h, m, y, st);
    case FCM_F16: return fcm::pw_t<__half>(h, m, y, st);
    default: return fcm::pw_t<__nv_bfloat16>(h, m, y, st);
    }
}

cudaError_t launch_fused_simt(const fcm_handle *h, const void *x, void *y, cudaStream_t st) {
    switch (h->d.dtype) {
    case FCM_F32: return fcm::fused_t<float>(h, x, y, st);
    case FCM_F16: return fcm::fused_t<__half>(h, x, y, st);
    default: return fcm::fused_t<__nv_bfloat16>(h, x, y, st);
    }
}
