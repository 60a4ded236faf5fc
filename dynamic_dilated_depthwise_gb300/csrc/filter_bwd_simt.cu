// filter_bwd_simt.cu -- backward of the dynamic filter with given taps.
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA 动态过滤": with
// the dynamic kernels already generated, the filter's backward forms dX and
// dK (the taps' gradient) directly, without building a patch matrix.  For
// L = <grad_out, out>, out = [x, d1, d3, d5]:
//
//   dtaps[b,o,h,w] = grad[b,(1+di)C+c,h,w] * x[b,c,h+(ky-r)d, w+(kx-r)d]   (0 outside)
//   dx[b,c,h,w]    = grad[b,c,h,w]
//                  + sum_{di,ky,kx} taps[b,o,h',w'] * grad[b,(1+di)C+c,h',w'],
//                    (h',w') = (h-(ky-r)d, w-(kx-r)d) inside the image,
//   o = (di*C + c)*K*K + ky*K + kx.
//
// Both are bound by HBM: dtaps writes O values per pixel, dx reads O tap values
// per pixel, each exactly once.  One thread per pixel of one channel: a warp
// covers 32 consecutive pixels of a row, so every tap-plane load or store is one
// coalesced 64- (bf16) or 128-byte (fp32) access; the grad and x values a thread
// reads at shifted positions are shared with its neighbours through L1.
// Products and sums are FP32; each output is rounded once to its dtype.
#include "common.cuh"
#include "launch.h"

namespace ddpm {
namespace {

constexpr int kFbThreads = 256;

template <typename T, int K>
__global__ void __launch_bounds__(kFbThreads) filter_bwd_dtaps_kernel(Dims d, const T* __restrict__ g,
                                                                      const T* __restrict__ x, T* __restrict__ dtaps) {
    const long long p = (long long)blockIdx.x * kFbThreads + threadIdx.x;
    if (p >= d.HW) return;
    const int c = blockIdx.y, b = blockIdx.z;
    const int h = (int)(p / d.W), w = (int)(p - (long long)h * d.W);
    constexpr int r = K / 2, K2 = K * K;
    const T* xp = x + ((long long)b * d.C + c) * d.HW;
#pragma unroll
    for (int di = 0; di < 3; ++di) {
        const int dil = d.dil[di];
        const float gv = to_f(g[((long long)b * 4 * d.C + (long long)(1 + di) * d.C + c) * d.HW + p]);
        T* out = dtaps + ((long long)b * d.O + (long long)(di * d.C + c) * K2) * d.HW + p;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            const int hs = h + (ky - r) * dil;
            const bool row_in = hs >= 0 && hs < d.H;
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int ws = w + (kx - r) * dil;
                const float xv = (row_in && ws >= 0 && ws < d.W) ? to_f(xp[(long long)hs * d.W + ws]) : 0.0f;
                out[(long long)(ky * K + kx) * d.HW] = from_f<T>(gv * xv);
            }
        }
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kFbThreads) filter_bwd_dx_kernel(Dims d, const T* __restrict__ g,
                                                                   const T* __restrict__ taps, T* __restrict__ dx) {
    const long long p = (long long)blockIdx.x * kFbThreads + threadIdx.x;
    if (p >= d.HW) return;
    const int c = blockIdx.y, b = blockIdx.z;
    const int h = (int)(p / d.W), w = (int)(p - (long long)h * d.W);
    constexpr int r = K / 2, K2 = K * K;
    float acc = to_f(g[((long long)b * 4 * d.C + c) * d.HW + p]);
#pragma unroll
    for (int di = 0; di < 3; ++di) {
        const int dil = d.dil[di];
        const T* gp = g + ((long long)b * 4 * d.C + (long long)(1 + di) * d.C + c) * d.HW;
        const T* tp = taps + ((long long)b * d.O + (long long)(di * d.C + c) * K2) * d.HW;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            const int hs = h - (ky - r) * dil;
            const bool row_in = hs >= 0 && hs < d.H;
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int ws = w - (kx - r) * dil;
                if (row_in && ws >= 0 && ws < d.W) {
                    const long long q = (long long)hs * d.W + ws;
                    acc = fmaf(to_f(tp[(long long)(ky * K + kx) * d.HW + q]), to_f(gp[q]), acc);
                }
            }
        }
    }
    dx[((long long)b * d.C + c) * d.HW + p] = from_f<T>(acc);
}

template <typename T, int K>
cudaError_t launch_k(const Dims& d, const void* g, const void* x, const void* taps, void* dx, void* dtaps,
                     cudaStream_t s) {
    const dim3 grid((unsigned)((d.HW + kFbThreads - 1) / kFbThreads), (unsigned)d.C, (unsigned)d.B);
    if (dx != nullptr) {
        trace_begin(s, kKFilterBwdDx);
        filter_bwd_dx_kernel<T, K><<<grid, kFbThreads, 0, s>>>(d, static_cast<const T*>(g),
                                                               static_cast<const T*>(taps), static_cast<T*>(dx));
        trace_end(s);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (dtaps != nullptr) {
        trace_begin(s, kKFilterBwdDtaps);
        filter_bwd_dtaps_kernel<T, K><<<grid, kFbThreads, 0, s>>>(d, static_cast<const T*>(g),
                                                                  static_cast<const T*>(x), static_cast<T*>(dtaps));
        trace_end(s);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_t(const Dims& d, const void* g, const void* x, const void* taps, void* dx, void* dtaps,
                     cudaStream_t s) {
    switch (d.K) {
        case 1: return launch_k<T, 1>(d, g, x, taps, dx, dtaps, s);
        case 3: return launch_k<T, 3>(d, g, x, taps, dx, dtaps, s);
        case 5: return launch_k<T, 5>(d, g, x, taps, dx, dtaps, s);
        case 7: return launch_k<T, 7>(d, g, x, taps, dx, dtaps, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_filter_backward_simt(const Dims& d, const void* g, const void* x, const void* taps, void* dx,
                                        void* dtaps, cudaStream_t s) {
    if (d.dtype == 1) return launch_t<__nv_bfloat16>(d, g, x, taps, dx, dtaps, s);
    return launch_t<float>(d, g, x, taps, dx, dtaps, s);
}

}  // namespace ddpm
