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
// per pixel, each exactly once.  Products and sums are FP32; each output is
// rounded once to its dtype.
//
// Tiled kernels (W a multiple of the 16-byte vector, 16-byte aligned tensors,
// halo radius <= 16): a block owns one (b, c) plane tile and a thread VEC
// consecutive pixels of a row (filter_tile.cuh).
//   dtaps: x is staged over the tile with a zero halo; each product vector of
//     tap (ky, kx) is the thread's grad vector times the x segment shifted by
//     ((ky-r)d, (kx-r)d), cut from two aligned shared vectors, and leaves with
//     one 16-byte store.
//   dx:    the three grad blocks are staged with a zero halo; for each tap the
//     thread reads the two aligned tap-plane vectors that cover its source
//     segment (shifted by -off; a vector outside the image reads as zero, and
//     with W a multiple of VEC a vector is never partly outside), cuts both
//     operands at the block-uniform shift and accumulates their products.
//     Every tap value is read from HBM once; the neighbour's overlapping
//     vector comes from L1.
// Other shapes use one thread per pixel (a warp covers 32 consecutive pixels of
// a row, so every tap-plane access is one coalesced 64- or 128-byte access).
#include "filter_tile.cuh"
#include "launch.h"

namespace ddpm {
namespace {

using namespace ftile;

// out[i] = a[i] * b[i] for the VEC elements packed in two 16-byte words, rounded once
__device__ __forceinline__ uint4 mul_vec_f32(const uint4& a, const uint4& b) {
    return make_uint4(__float_as_uint(__uint_as_float(a.x) * __uint_as_float(b.x)),
                      __float_as_uint(__uint_as_float(a.y) * __uint_as_float(b.y)),
                      __float_as_uint(__uint_as_float(a.z) * __uint_as_float(b.z)),
                      __float_as_uint(__uint_as_float(a.w) * __uint_as_float(b.w)));
}
// bf16 pairs: the exact FP32 product of each pair, rounded to bf16 (nearest even)
__device__ __forceinline__ uint32_t mul_pair_bf16(uint32_t a, uint32_t b) {
    const float lo = __uint_as_float(a << 16) * __uint_as_float(b << 16);
    const float hi = __uint_as_float(a & 0xFFFF0000u) * __uint_as_float(b & 0xFFFF0000u);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
template <typename T>
__device__ __forceinline__ uint4 mul_vec(const uint4& a, const uint4& b) {
    if constexpr (sizeof(T) == 4) return mul_vec_f32(a, b);
    else return make_uint4(mul_pair_bf16(a.x, b.x), mul_pair_bf16(a.y, b.y), mul_pair_bf16(a.z, b.z),
                           mul_pair_bf16(a.w, b.w));
}

template <typename T, int K>
__global__ void __launch_bounds__(kFThreads) filter_bwd_dtaps_tiled(Dims d, const T* __restrict__ g,
                                                                    const T* __restrict__ x, T* __restrict__ dtaps,
                                                                    int tiles_w, int tiles_h) {
    constexpr int VEC = FilterTile<T>::VEC, TH = FilterTile<T>::TH;
    constexpr int K2 = K * K, r = K / 2, TPR = kFTW / VEC, VPR = kFRowElems / VEC;
    extern __shared__ __align__(16) unsigned char fsm[];
    T* xs = reinterpret_cast<T*>(fsm);                    // [(TH + 2R) rows][kFRowElems]
    const int R = d.R();
    const int tile = blockIdx.x % (tiles_w * tiles_h);
    const long long bc = blockIdx.x / (tiles_w * tiles_h);
    const int c = (int)(bc % d.C), b = (int)(bc / d.C);
    const int h0 = (tile / tiles_w) * TH, w0 = (tile % tiles_w) * kFTW;
    const T* xp = x + bc * d.HW;
    const int srows = TH + 2 * R;
    for (int i = threadIdx.x; i < srows * VPR; i += kFThreads) {
        const int sr = i / VPR, sv = i % VPR;
        const int hh = h0 - R + sr, ww = w0 - kFHalo + sv * VEC;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (hh >= 0 && hh < d.H && ww >= 0 && ww + VEC <= d.W)
            v = __ldg(reinterpret_cast<const uint4*>(xp + (long long)hh * d.W + ww));
        *reinterpret_cast<uint4*>(xs + sr * kFRowElems + sv * VEC) = v;
    }
    __syncthreads();
    const int tr = threadIdx.x / TPR, tc = (threadIdx.x % TPR) * VEC;
    const int h = h0 + tr, w = w0 + tc;
    if (h >= d.H || w >= d.W) return;
    const long long p0 = (long long)h * d.W + w;
    const T* xrow0 = xs + (tr + R) * kFRowElems + kFHalo + tc;
#pragma unroll 1
    for (int di = 0; di < 3; ++di) {
        const int dil = dil_of(d, di);
        const uint4 gv =
            __ldg(reinterpret_cast<const uint4*>(g + ((long long)b * 4 * d.C + (long long)(1 + di) * d.C + c) * d.HW + p0));
        T* out = dtaps + ((long long)b * d.O + (long long)(di * d.C + c) * K2) * d.HW + p0;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            const T* xrow = xrow0 + (ky - r) * dil * kFRowElems;
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int o = (kx - r) * dil;
                const int sh = (o + kFHalo) & (VEC - 1);
                const T* row = xrow + (o - sh);
                const uint4 v0 = *reinterpret_cast<const uint4*>(row);
                const uint4 v1 = *reinterpret_cast<const uint4*>(row + VEC);
                *reinterpret_cast<uint4*>(out + (long long)(ky * K + kx) * d.HW) = mul_vec<T>(gv, cut_vec<T>(v0, v1, sh));
            }
        }
    }
}

template <typename T, int K>
__global__ void __launch_bounds__(kFThreads) filter_bwd_dx_tiled(Dims d, const T* __restrict__ g,
                                                                 const T* __restrict__ taps, T* __restrict__ dx,
                                                                 int tiles_w, int tiles_h) {
    constexpr int VEC = FilterTile<T>::VEC, TH = FilterTile<T>::TH;
    constexpr int K2 = K * K, r = K / 2, TPR = kFTW / VEC, VPR = kFRowElems / VEC;
    extern __shared__ __align__(16) unsigned char fsm[];
    T* gs = reinterpret_cast<T*>(fsm);                    // 3 x [(TH + 2R) rows][kFRowElems]
    const int R = d.R();
    const int tile = blockIdx.x % (tiles_w * tiles_h);
    const long long bc = blockIdx.x / (tiles_w * tiles_h);
    const int c = (int)(bc % d.C), b = (int)(bc / d.C);
    const int h0 = (tile / tiles_w) * TH, w0 = (tile % tiles_w) * kFTW;
    const int srows = TH + 2 * R, plane = srows * kFRowElems;
    // stage grad blocks 1..3 of channel c over the tile with a zero halo
    for (int i = threadIdx.x; i < 3 * srows * VPR; i += kFThreads) {
        const int di = i / (srows * VPR), rem = i - di * srows * VPR;
        const int sr = rem / VPR, sv = rem % VPR;
        const int hh = h0 - R + sr, ww = w0 - kFHalo + sv * VEC;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (hh >= 0 && hh < d.H && ww >= 0 && ww + VEC <= d.W)
            v = __ldg(reinterpret_cast<const uint4*>(
                g + ((long long)b * 4 * d.C + (long long)(1 + di) * d.C + c) * d.HW + (long long)hh * d.W + ww));
        *reinterpret_cast<uint4*>(gs + di * plane + sr * kFRowElems + sv * VEC) = v;
    }
    __syncthreads();
    const int tr = threadIdx.x / TPR, tc = (threadIdx.x % TPR) * VEC;
    const int h = h0 + tr, w = w0 + tc;
    if (h >= d.H || w >= d.W) return;
    const long long p0 = (long long)h * d.W + w;
    float acc[VEC];
    {
        const uint4 g0 = __ldg(reinterpret_cast<const uint4*>(g + ((long long)b * 4 * d.C + c) * d.HW + p0));
        const T* gt = reinterpret_cast<const T*>(&g0);
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = to_f(gt[i]);
    }
#pragma unroll 1
    for (int di = 0; di < 3; ++di) {
        const int dil = dil_of(d, di);
        const T* tp = taps + ((long long)b * d.O + (long long)(di * d.C + c) * K2) * d.HW;
        const T* grow0 = gs + di * plane + (tr + R) * kFRowElems + kFHalo + tc;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            const int hs = h - (ky - r) * dil;            // source row
            if (hs < 0 || hs >= d.H) continue;            // its grad row is zero: no contribution
            const T* grow = grow0 - (ky - r) * dil * kFRowElems;
            const T* trow = tp + (long long)(ky * K) * d.HW + (long long)hs * d.W;
            uint4 tv0[K], tv1[K];                         // one tap row: all its loads in flight
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int o = -(kx - r) * dil;            // source column shift
                const int sh = (o + kFHalo) & (VEC - 1);
                const int cb = w + o - sh;                // aligned start of the covering vectors
                const T* tpl = trow + (long long)kx * d.HW;
                tv0[kx] = (cb >= 0 && cb + VEC <= d.W) ? __ldg(reinterpret_cast<const uint4*>(tpl + cb))
                                                       : make_uint4(0u, 0u, 0u, 0u);
                tv1[kx] = (sh != 0 && cb + VEC >= 0 && cb + 2 * VEC <= d.W)
                              ? __ldg(reinterpret_cast<const uint4*>(tpl + cb + VEC))
                              : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int o = -(kx - r) * dil;
                const int sh = (o + kFHalo) & (VEC - 1);
                const T* row = grow + (o - sh);
                const uint4 v0 = *reinterpret_cast<const uint4*>(row);
                const uint4 v1 = *reinterpret_cast<const uint4*>(row + VEC);
                fma_vec(acc, cut_vec<T>(tv0[kx], tv1[kx], sh), cut_vec<T>(v0, v1, sh));
            }
        }
    }
    T res[VEC];
#pragma unroll
    for (int i = 0; i < VEC; ++i) res[i] = from_f<T>(acc[i]);
    *reinterpret_cast<uint4*>(dx + ((long long)b * d.C + c) * d.HW + p0) = *reinterpret_cast<const uint4*>(res);
}

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
    constexpr int V = 16 / sizeof(T);
    const bool aligned = (uintptr_t)g % 16 == 0 && (uintptr_t)x % 16 == 0 && (uintptr_t)taps % 16 == 0 &&
                         (uintptr_t)dx % 16 == 0 && (uintptr_t)dtaps % 16 == 0;
    if (aligned && d.W % V == 0 && d.R() <= kFHalo) {
        constexpr int TH = FilterTile<T>::TH;
        const int tiles_w = (d.W + kFTW - 1) / kFTW, tiles_h = (d.H + TH - 1) / TH;
        const long long blocks = (long long)d.B * d.C * tiles_w * tiles_h;
        const size_t plane = (size_t)(TH + 2 * d.R()) * kFRowElems * sizeof(T);
        // + one vector: the second vector of the last row's rightmost cut is read (and unused)
        const size_t smem_dx = 3 * plane + 16, smem_dt = plane + 16;
        if (blocks <= 0x7fffffffLL && smem_dx <= 48 * 1024) {
            if (dx != nullptr) {
                trace_begin(s, kKFilterBwdDx);
                filter_bwd_dx_tiled<T, K><<<(unsigned)blocks, kFThreads, smem_dx, s>>>(
                    d, static_cast<const T*>(g), static_cast<const T*>(taps), static_cast<T*>(dx), tiles_w, tiles_h);
                trace_end(s);
                const cudaError_t e = cudaGetLastError();
                if (e != cudaSuccess) return e;
            }
            if (dtaps != nullptr) {
                trace_begin(s, kKFilterBwdDtaps);
                filter_bwd_dtaps_tiled<T, K><<<(unsigned)blocks, kFThreads, smem_dt, s>>>(
                    d, static_cast<const T*>(g), static_cast<const T*>(x), static_cast<T*>(dtaps), tiles_w, tiles_h);
                trace_end(s);
                const cudaError_t e = cudaGetLastError();
                if (e != cudaSuccess) return e;
            }
            return cudaSuccess;
        }
    }
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
