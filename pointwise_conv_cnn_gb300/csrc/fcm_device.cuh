// fcm_device.cuh -- device helpers shared by the CUDA kernels: storage conversions, the
// activation functions, vector loads/stores.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fcm {

// Storage <-> fp32.  Widening is exact; narrowing rounds to nearest even.
template <typename T> struct Storage;
template <> struct Storage<float> {
    static __device__ __forceinline__ float to_f(float v) { return v; }
    static __device__ __forceinline__ float from_f(float v) { return v; }
};
template <> struct Storage<__half> {
    static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
    static __device__ __forceinline__ __half from_f(float v) { return __float2half_rn(v); }
};
template <> struct Storage<__nv_bfloat16> {
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// Activation after the folded norm: 0 none, 1 ReLU, 2 ReLU6 (min(max(v,0),6)).
__device__ __forceinline__ float act_apply(float v, int act) {
    if (act == 1) return fmaxf(v, 0.0f);
    if (act == 2) return fminf(fmaxf(v, 0.0f), 6.0f);
    return v;
}

// Load VEC consecutive storage elements (VEC * sizeof(T) bytes, naturally aligned) as fp32.
template <typename T, int VEC>
__device__ __forceinline__ void load_vec(const T *__restrict__ p, float (&out)[VEC]) {
    constexpr int BYTES = VEC * (int)sizeof(T);
    if constexpr (BYTES == 16) {
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int i = 0; i < VEC; i++) out[i] = Storage<T>::to_f(e[i]);
    } else if constexpr (BYTES == 8) {
        uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        const T *e = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int i = 0; i < VEC; i++) out[i] = Storage<T>::to_f(e[i]);
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i++) out[i] = Storage<T>::to_f(p[i]);
    }
}

// Store VEC fp32 values as storage elements (rounded to nearest even).
template <typename T, int VEC>
__device__ __forceinline__ void store_vec(T *__restrict__ p, const float (&v)[VEC]) {
    constexpr int BYTES = VEC * (int)sizeof(T);
    if constexpr (BYTES == 16 || BYTES == 8) {
        T e[VEC];
#pragma unroll
        for (int i = 0; i < VEC; i++) e[i] = Storage<T>::from_f(v[i]);
        if constexpr (BYTES == 16)
            *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(e);
        else
            *reinterpret_cast<uint2 *>(p) = *reinterpret_cast<const uint2 *>(e);
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i++) p[i] = Storage<T>::from_f(v[i]);
    }
}

}  // namespace fcm
