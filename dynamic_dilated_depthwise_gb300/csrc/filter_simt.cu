// filter_simt.cu -- dynamic dilated depthwise filter with pregenerated taps.
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA 动态过滤": with the
// dynamic kernels already generated, one kernel handles all three dilations,
// reads the neighbourhood per spatial tile, accumulates in FP32 and writes
// [x, d1, d3, d5] directly, without Unfold.
//
// The op is bound by HBM: every tap is read exactly once (3*C*K*K values per
// pixel), x once from DRAM (its neighbours come from L1/L2) and 4C outputs are
// written.  Each thread owns VEC consecutive pixels of one (b, c) plane so that
// the 3*K*K tap planes are read with 16-byte loads, fully coalesced across the
// warp; the neighbour reads of x hit L1 (a plane is at most a few hundred KB).
#include "launch.h"

namespace ddpm {
namespace {

template <typename T, int VEC>
struct alignas(16) VecT {
    T v[VEC];
};

template <typename T, int VEC>
__device__ __forceinline__ void load_vec(const T* __restrict__ p, float (&f)[VEC]) {
    if constexpr (VEC == 1) {
        f[0] = to_f(__ldg(p));
    } else {
        static_assert(sizeof(T) * VEC == 16, "vector loads are 16 bytes");
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(p));
        const VecT<T, VEC> t = *reinterpret_cast<const VecT<T, VEC>*>(&raw);
#pragma unroll
        for (int i = 0; i < VEC; ++i) f[i] = to_f(t.v[i]);
    }
}

template <typename T, int VEC>
__device__ __forceinline__ void store_vec(T* __restrict__ p, const float (&f)[VEC]) {
    if constexpr (VEC == 1) {
        p[0] = from_f<T>(f[0]);
    } else {
        VecT<T, VEC> t;
#pragma unroll
        for (int i = 0; i < VEC; ++i) t.v[i] = from_f<T>(f[i]);
        *reinterpret_cast<uint4*>(p) = *reinterpret_cast<const uint4*>(&t);
    }
}

template <typename T, int K, int VEC>
__global__ void __launch_bounds__(256) filter_pregenerated_kernel(Dims d, const T* __restrict__ x,
                                                                  const T* __restrict__ taps,
                                                                  T* __restrict__ out) {
    constexpr int K2 = K * K;
    const int r = K / 2;
    const long long nvec = d.HW / VEC;  // VEC divides W whenever VEC > 1
    const long long total = (long long)d.B * d.C * nvec;
    for (long long item = (long long)blockIdx.x * blockDim.x + threadIdx.x; item < total;
         item += (long long)gridDim.x * blockDim.x) {
        const long long pv = item % nvec;
        const long long bc = item / nvec;
        const int c = (int)(bc % d.C);
        const int b = (int)(bc / d.C);
        const long long p0 = pv * VEC;
        const int h = (int)(p0 / d.W);
        const int w0 = (int)(p0 % d.W);
        const T* xp = x + ((long long)b * d.C + c) * d.HW;

        // channel c of the output is x itself (bit-exact copy)
        float xc[VEC];
        load_vec<T, VEC>(xp + p0, xc);
        store_vec<T, VEC>(out + ((long long)b * 4 * d.C + c) * d.HW + p0, xc);

#pragma unroll 1
        for (int di = 0; di < 3; ++di) {
            const int dil = dil_of(d, di);
            const T* tp = taps + ((long long)b * d.O + (long long)(di * d.C + c) * K2) * d.HW + p0;
            float acc[VEC];
#pragma unroll
            for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int ky = 0; ky < K; ++ky) {
                const int hh = h + (ky - r) * dil;
                const bool row_ok = hh >= 0 && hh < d.H;
                const T* xrow = xp + (long long)hh * d.W;
#pragma unroll
                for (int kx = 0; kx < K; ++kx) {
                    float tv[VEC];
                    load_vec<T, VEC>(tp + (long long)(ky * K + kx) * d.HW, tv);
                    const int ww = w0 + (kx - r) * dil;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        const int wi = ww + i;
                        const float xv = (row_ok && wi >= 0 && wi < d.W) ? to_f(__ldg(xrow + wi)) : 0.0f;
                        acc[i] = fmaf(tv[i], xv, acc[i]);
                    }
                }
            }
            store_vec<T, VEC>(out + ((long long)b * 4 * d.C + (1 + di) * d.C + c) * d.HW + p0, acc);
        }
    }
}

template <typename T, int K>
cudaError_t launch_k(const Dims& d, const void* x, const void* taps, void* out, cudaStream_t s, bool vec_ok) {
    constexpr int V = 16 / sizeof(T);
    const int threads = 256;
    const int vec = vec_ok ? V : 1;
    const long long items = (long long)d.B * d.C * (d.HW / vec);
    long long blocks = (items + threads - 1) / threads;
    if (blocks > 152LL * 64) blocks = 152LL * 64;  // grid-stride beyond this
    trace_begin(s, kKFilterSimt);
    if (vec_ok) {
        filter_pregenerated_kernel<T, K, V><<<(unsigned)blocks, threads, 0, s>>>(
            d, (const T*)x, (const T*)taps, (T*)out);
    } else {
        filter_pregenerated_kernel<T, K, 1><<<(unsigned)blocks, threads, 0, s>>>(
            d, (const T*)x, (const T*)taps, (T*)out);
    }
    trace_end(s);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const Dims& d, const void* x, const void* taps, void* out, cudaStream_t s) {
    constexpr int V = 16 / sizeof(T);
    const bool vec_ok = (d.W % V == 0) && ((uintptr_t)x % 16 == 0) && ((uintptr_t)taps % 16 == 0) &&
                        ((uintptr_t)out % 16 == 0);
    switch (d.K) {
        case 1: return launch_k<T, 1>(d, x, taps, out, s, vec_ok);
        case 3: return launch_k<T, 3>(d, x, taps, out, s, vec_ok);
        case 5: return launch_k<T, 5>(d, x, taps, out, s, vec_ok);
        case 7: return launch_k<T, 7>(d, x, taps, out, s, vec_ok);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_filter_simt(const Dims& d, const void* x, const void* taps, void* out, cudaStream_t s) {
    if (d.dtype == 1) return launch_t<__nv_bfloat16>(d, x, taps, out, s);
    return launch_t<float>(d, x, taps, out, s);
}

}  // namespace ddpm
