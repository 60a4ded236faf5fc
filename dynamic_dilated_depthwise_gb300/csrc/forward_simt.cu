// forward_simt.cu -- fused generator + dynamic filter on CUDA cores.
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA 融合生成器推理":
// y tile -> dot(weight, y) -> dynamic taps -> consume with shifted x -> output,
// with the taps kept on chip.  Section "CUDA Flash 式融合训练" fixes the
// precision: the FP32 forward uses IEEE FP32 dot products (no TF32), so this
// kernel is the FP32 path; it accepts bf16 too (taps rounded to bf16 before use).
//
// One thread owns one pixel; a block owns 128 pixels of one image and a group
// of CG output channels.  For each (channel c, dilation di) the block stages
// the K*K generator rows of that (di, c) in shared memory, each thread forms its
// K*K taps from y at its pixel, rounds them for bf16, and applies them to the
// zero-padded shifted x.  With K <= 3 and C a multiple of 4 (up to 64) y stays
// in registers and the rows are staged as they lie in memory, Ws[k][j]: a
// 16-byte broadcast load gives four input channels of one tap, with no padded
// taps.  Otherwise Ws[j][k], k padded to a multiple of 4 (four taps' weights of
// one input channel per 16-byte load) and y streamed from L1.
#include "launch.h"

namespace ddpm {
namespace {

constexpr int kThreads = 128;
constexpr int kCG = 8;  // output channels per block

template <typename T, int K>
__global__ void __launch_bounds__(kThreads, K <= 3 ? 4 : 0) forward_simt_kernel(Dims d, const T* __restrict__ x,
                                                                const T* __restrict__ y,
                                                                const T* __restrict__ wgt,
                                                                const T* __restrict__ bias,
                                                                T* __restrict__ out) {
    constexpr int K2 = K * K;
    constexpr int KP = (K2 + 3) / 4 * 4;
    extern __shared__ __align__(16) float Ws[];  // [C][KP]
    const int r = K / 2;
    const int C = d.C;
    const int b = blockIdx.z;
    const int c0 = blockIdx.y * kCG;
    const long long p = (long long)blockIdx.x * kThreads + threadIdx.x;
    const bool active = p < d.HW;
    const int h = active ? (int)(p / d.W) : 0;
    const int w = active ? (int)(p % d.W) : 0;
    const T* yb = y + (long long)b * C * d.HW;

    // y of this pixel stays in registers across the block's channels and dilations when
    // C <= 64 and K <= 3 (one load per input channel instead of one per (channel,
    // dilation, input)); larger kernels need the registers for their taps
    constexpr int kYR = K <= 3 ? 64 : 1;
    const bool y_in_regs = K <= 3 && C <= kYR && C % 4 == 0;
    float yr[kYR];
#pragma unroll
    for (int j = 0; j < kYR; ++j) yr[j] = (y_in_regs && active && j < C) ? ldg_f(yb + (long long)j * d.HW + p) : 0.0f;
    // the generator rows of the next (channel, dilation) are loaded into registers while
    // the current ones are applied, so the staging latency overlaps
    constexpr int ITW = K <= 3 ? (kYR * KP + kThreads - 1) / kThreads : 1;
    float wn[ITW];
    // Ws[k][j] = W[o0 + k][j]: K2 contiguous rows of C, one coalesced copy
    auto load_rows = [&](long long o0) {
#pragma unroll
        for (int it = 0; it < ITW; ++it) {
            const int i = threadIdx.x + it * kThreads;
            wn[it] = i < K2 * C ? to_f(wgt[o0 * C + i]) : 0.0f;
        }
    };
    if (y_in_regs) load_rows((long long)c0 * K2);

    for (int cc = 0; cc < kCG; ++cc) {
        const int c = c0 + cc;
        if (c >= C) break;  // uniform across the block
        const T* xp = x + ((long long)b * C + c) * d.HW;
        if (active) out[((long long)b * 4 * C + c) * d.HW + p] = xp[p];
#pragma unroll 1
        for (int di = 0; di < 3; ++di) {
            __syncthreads();
            const long long o0 = (long long)(di * C + c) * K2;
            if (y_in_regs) {
#pragma unroll
                for (int it = 0; it < ITW; ++it) {
                    const int i = threadIdx.x + it * kThreads;
                    if (i < K2 * C) Ws[i] = wn[it];
                }
            } else {
                for (int i = threadIdx.x; i < C * KP; i += kThreads) {
                    const int j = i / KP, k = i % KP;
                    Ws[i] = k < K2 ? to_f(wgt[(o0 + k) * C + j]) : 0.0f;
                }
            }
            __syncthreads();
            if (y_in_regs) {
                // next (channel, dilation) of the block, if any
                const int ndi = di < 2 ? di + 1 : 0, nc = di < 2 ? c : c + 1;
                if (nc < C && nc < c0 + kCG) load_rows((long long)(ndi * C + nc) * K2);
            }
            if (!active) continue;
            float t[KP];
#pragma unroll
            for (int k = 0; k < KP; ++k) t[k] = (bias != nullptr && k < K2) ? to_f(bias[o0 + k]) : 0.0f;
            if (y_in_regs) {
                // input channels in fours, every tap per four: t[k] still sums j = 0, 1, 2, ... in order
#pragma unroll
                for (int q = 0; q < kYR / 4; ++q) {
                    if (4 * q >= C) break;
#pragma unroll
                    for (int k = 0; k < K2; ++k) {
                        const float4 w4 = *reinterpret_cast<const float4*>(Ws + k * C + 4 * q);
                        t[k] = __fmaf_rn(w4.x, yr[4 * q + 0], t[k]);
                        t[k] = __fmaf_rn(w4.y, yr[4 * q + 1], t[k]);
                        t[k] = __fmaf_rn(w4.z, yr[4 * q + 2], t[k]);
                        t[k] = __fmaf_rn(w4.w, yr[4 * q + 3], t[k]);
                    }
                }
            } else {
                for (int j = 0; j < C; ++j) {
                    const float yv = ldg_f(yb + (long long)j * d.HW + p);
                    const float4* wr = reinterpret_cast<const float4*>(Ws + j * KP);
#pragma unroll
                    for (int q = 0; q < KP / 4; ++q) {
                        const float4 w4 = wr[q];
                        t[4 * q + 0] = __fmaf_rn(w4.x, yv, t[4 * q + 0]);
                        t[4 * q + 1] = __fmaf_rn(w4.y, yv, t[4 * q + 1]);
                        t[4 * q + 2] = __fmaf_rn(w4.z, yv, t[4 * q + 2]);
                        t[4 * q + 3] = __fmaf_rn(w4.w, yv, t[4 * q + 3]);
                    }
                }
            }
            const int dil = dil_of(d, di);
            float acc = 0.0f;
#pragma unroll
            for (int ky = 0; ky < K; ++ky)
#pragma unroll
                for (int kx = 0; kx < K; ++kx) {
                    const float tq = quantise_tap<T>(t[ky * K + kx]);
                    acc = __fmaf_rn(tq, x_at(xp, d.H, d.W, h + (ky - r) * dil, w + (kx - r) * dil), acc);
                }
            out[((long long)b * 4 * C + (1 + di) * C + c) * d.HW + p] = from_f<T>(acc);
        }
    }
}

template <typename T, int K>
cudaError_t launch_k(const Dims& d, const void* x, const void* y, const void* w, const void* bias,
                     void* out, cudaStream_t s) {
    constexpr int K2 = K * K;
    constexpr int KP = (K2 + 3) / 4 * 4;
    const size_t smem = sizeof(float) * (size_t)d.C * KP;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(forward_simt_kernel<T, K>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((d.HW + kThreads - 1) / kThreads), (unsigned)((d.C + kCG - 1) / kCG), (unsigned)d.B);
    trace_begin(s, kKForwardSimt);
    forward_simt_kernel<T, K><<<grid, kThreads, smem, s>>>(d, (const T*)x, (const T*)y, (const T*)w,
                                                           (const T*)bias, (T*)out);
    trace_end(s);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const Dims& d, const void* x, const void* y, const void* w, const void* bias,
                     void* out, cudaStream_t s) {
    switch (d.K) {
        case 1: return launch_k<T, 1>(d, x, y, w, bias, out, s);
        case 3: return launch_k<T, 3>(d, x, y, w, bias, out, s);
        case 5: return launch_k<T, 5>(d, x, y, w, bias, out, s);
        case 7: return launch_k<T, 7>(d, x, y, w, bias, out, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_forward_simt(const Dims& d, const void* x, const void* y, const void* w,
                                const void* bias, void* out, cudaStream_t s) {
    if (d.dtype == 1) return launch_t<__nv_bfloat16>(d, x, y, w, bias, out, s);
    return launch_t<float>(d, x, y, w, bias, out, s);
}

}  // namespace ddpm
