// common.cuh -- shared device helpers of the DDPM core kernels (sm_103a).
//
// Problem geometry (README "lartpang/DynamicConvolutionOperator", section
// "CUDA 动态过滤"): taps channel o = (di*C + c)*K*K + ky*K + kx; tap (ky,kx) of
// dilation d reads x at (h + (ky - r)*d, w + (kx - r)*d), zero outside.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ddpm {

// Host-validated problem description passed by value to every kernel.
struct Dims {
    int B, C, H, W, K, r;   // r = K / 2
    int dil[3];
    int dtype;               // 0 = fp32, 1 = bf16
    unsigned flags;
    long long HW;            // H * W
    long long O;             // 3 * C * K * K

    __host__ __device__ int R() const {  // halo radius: largest dilation * (K / 2)
        int m = dil[0] > dil[1] ? dil[0] : dil[1];
        m = m > dil[2] ? m : dil[2];
        return m * r;
    }
};

// ---- element conversions -------------------------------------------------

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// The generator output as the filter consumes it: unchanged for fp32, rounded
// to bf16 (nearest, ties to even) for bf16 problems ("BF16 在写出动态 tap 前显式量化").
template <typename T> __device__ __forceinline__ float quantise_tap(float t);
template <> __device__ __forceinline__ float quantise_tap<float>(float t) { return t; }
template <> __device__ __forceinline__ float quantise_tap<__nv_bfloat16>(float t) {
    return __bfloat162float(__float2bfloat16_rn(t));
}

// d.dil[di] without a dynamic index into the kernel parameter block
__host__ __device__ __forceinline__ int dil_of(const Dims& d, int di) {
    return di == 0 ? d.dil[0] : (di == 1 ? d.dil[1] : d.dil[2]);
}

template <typename T> __device__ __forceinline__ float ldg_f(const T* p) { return to_f(__ldg(p)); }

// x[b, c, h, w] with zero padding outside the image
template <typename T>
__device__ __forceinline__ float x_at(const T* __restrict__ xplane, int H, int W, int h, int w) {
    return (h >= 0 && h < H && w >= 0 && w < W) ? ldg_f(xplane + (long long)h * W + w) : 0.0f;
}

}  // namespace ddpm
