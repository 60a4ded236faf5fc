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
#include "filter_tile.cuh"
#include "launch.h"

namespace ddpm {
namespace {

using namespace ftile;

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

// ------------------------------------------------------------------ tiled
// The vectorised kernel.  A block owns one (b, c) plane tile of kFTH(T) rows x 64
// columns and first stages x over it with a halo of R rows and 16 columns on each
// side in shared memory, zeros outside the image, so the inner loop has no bounds
// checks.  A thread owns VEC consecutive pixels of a row: each tap plane is read
// with one 16-byte load, and the VEC neighbours of tap (ky, kx) -- a row segment
// shifted by o = (kx - r) * d columns -- come from the two aligned 16-byte vectors
// of shared memory that cover it, cut at o mod VEC, which is the same for every
// thread of the block (a uniform switch, no divergence).
template <typename T, int K>
__global__ void __launch_bounds__(kFThreads) filter_tiled_kernel(Dims d, const T* __restrict__ x,
                                                                 const T* __restrict__ taps, T* __restrict__ out,
                                                                 int tiles_w, int tiles_h) {
    constexpr int VEC = FilterTile<T>::VEC, TH = FilterTile<T>::TH;
    constexpr int K2 = K * K, r = K / 2;
    constexpr int TPR = kFTW / VEC;                       // threads per tile row
    extern __shared__ __align__(16) unsigned char fsm[];
    T* xs = reinterpret_cast<T*>(fsm);                    // [(TH + 2R) rows][kFRowElems]
    const int R = d.R();
    const int tile = blockIdx.x % (tiles_w * tiles_h);
    const long long bc = blockIdx.x / (tiles_w * tiles_h);
    const int c = (int)(bc % d.C), b = (int)(bc / d.C);
    const int h0 = (tile / tiles_w) * TH, w0 = (tile % tiles_w) * kFTW;
    const T* xp = x + bc * d.HW;

    // stage x rows h0-R .. h0+TH+R-1, columns w0-16 .. w0+64+15, zeros outside the image
    const int srows = TH + 2 * R;
    constexpr int VPR = kFRowElems / VEC;                 // vectors per staged row
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
    if (h >= d.H || w >= d.W) return;                     // W is a multiple of VEC: vectors are whole
    const long long p0 = (long long)h * d.W + w;
    const T* xrow0 = xs + (tr + R) * kFRowElems + kFHalo + tc;   // this thread's pixels in the stage
    T* ob = out + ((long long)b * 4 * d.C) * d.HW + p0;
    // channel c of the output is x itself (bit-exact copy)
    *reinterpret_cast<uint4*>(ob + (long long)c * d.HW) = *reinterpret_cast<const uint4*>(xrow0);
#pragma unroll 1
    for (int di = 0; di < 3; ++di) {
        const int dil = dil_of(d, di);
        const T* tp = taps + ((long long)b * d.O + (long long)(di * d.C + c) * K2) * d.HW + p0;
        float acc[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            uint4 tv[K];                                  // one tap row: K 16-byte loads in flight
#pragma unroll
            for (int kx = 0; kx < K; ++kx)
                tv[kx] = __ldg(reinterpret_cast<const uint4*>(tp + (long long)(ky * K + kx) * d.HW));
            const T* xrow = xrow0 + (ky - r) * dil * kFRowElems;
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int o = (kx - r) * dil;             // column shift, |o| <= R <= 16
                const int sh = (o + kFHalo) & (VEC - 1);  // the same for every thread
                const T* row = xrow + (o - sh);           // o - sh: a multiple of VEC
                const uint4 v0 = *reinterpret_cast<const uint4*>(row);
                const uint4 v1 = *reinterpret_cast<const uint4*>(row + VEC);
                fma_vec(acc, tv[kx], cut_vec<T>(v0, v1, sh));
            }
        }
        T res[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) res[i] = from_f<T>(acc[i]);
        *reinterpret_cast<uint4*>(ob + (long long)((1 + di) * d.C + c) * d.HW) = *reinterpret_cast<const uint4*>(res);
    }
}

template <typename T, int K>
cudaError_t launch_k(const Dims& d, const void* x, const void* taps, void* out, cudaStream_t s, bool vec_ok) {
    constexpr int V = 16 / sizeof(T);
    if (vec_ok && d.R() <= kFHalo) {
        constexpr int TH = FilterTile<T>::TH;
        const int tiles_w = (d.W + kFTW - 1) / kFTW, tiles_h = (d.H + TH - 1) / TH;
        const long long blocks = (long long)d.B * d.C * tiles_w * tiles_h;
        // + one vector: the second vector of the last row's rightmost cut is read (and unused)
        const size_t smem = ((size_t)(TH + 2 * d.R()) * kFRowElems + V) * sizeof(T);
        if (blocks <= 0x7fffffffLL && smem <= 48 * 1024) {
            trace_begin(s, kKFilterSimt);
            filter_tiled_kernel<T, K><<<(unsigned)blocks, kFThreads, smem, s>>>(d, (const T*)x, (const T*)taps,
                                                                               (T*)out, tiles_w, tiles_h);
            trace_end(s);
            return cudaGetLastError();
        }
    }
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
