// backward_simt.cu -- DDPM core backward on CUDA cores (any dtype and shape).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
//   dX     : recompute the dynamic taps and gather each dilation's contribution;
//   dY     : form dK = shifted(x) * grad on chip and multiply it by the generator
//            weight straight away;
//   dW/db  : form dK on chip and reduce over space -- the tokens are split into
//            at most 16 FP32 partials and a second short kernel sums them.
// Taps are recomputed, never written out.  In bf16 problems the tap rounding
// is straight-through: dx multiplies grad by the rounded taps.
//
// Four kernels: dx_kernel, dy_kernel, dw_partial_kernel, dw_reduce_kernel.
// The partial sums are summed in a fixed order, so results are reproducible
// bit for bit from run to run.
#include "launch.h"

namespace ddpm {
namespace {

constexpr int kThreads = 128;
constexpr int kCG = 8;          // dx: channels per block
constexpr int kJC = 64;         // dy: j per register chunk
constexpr int kMaxSplits = 16;  // "最多 16 个 FP32 partial"

// ---------------------------------------------------------------- dX --
// dx[b,c,q] = g[b,c,q] + sum_{di,ky,kx} Tq[b,o,q-off] * g[b,(1+di)C+c,q-off]
// One thread per pixel q, CG channels per block.  For each tap (di,k) the
// block stages the CG generator rows {o(di, c0+cc, k)} as Ws[j][cc]; each
// thread evaluates the taps of its CG channels at the neighbour p = q - off
// (one y load feeds CG FMAs) and accumulates tap * grad there.
template <typename T, int K>
__global__ void __launch_bounds__(kThreads) dx_kernel(Dims d, const T* __restrict__ g,
                                                      const T* __restrict__ y, const T* __restrict__ wgt,
                                                      const T* __restrict__ bias, T* __restrict__ dx) {
    constexpr int K2 = K * K;
    extern __shared__ __align__(16) float Ws[];  // [C][kCG]
    __shared__ float bs[kCG];
    const int r = K / 2;
    const int C = d.C;
    const int b = blockIdx.z;
    const int c0 = blockIdx.y * kCG;
    const long long q = (long long)blockIdx.x * kThreads + threadIdx.x;
    const bool active = q < d.HW;
    const int h = active ? (int)(q / d.W) : 0;
    const int w = active ? (int)(q % d.W) : 0;
    const T* yb = y + (long long)b * C * d.HW;
    const T* gb = g + (long long)b * 4 * C * d.HW;

    float acc[kCG];
#pragma unroll
    for (int cc = 0; cc < kCG; ++cc)
        acc[cc] = (active && c0 + cc < C) ? to_f(gb[(long long)(c0 + cc) * d.HW + q]) : 0.0f;

    // the generator rows of the next tap are loaded into registers while this tap is
    // applied (C <= 128: at most 8 values a thread), so the staging latency overlaps
    constexpr int ITX = 8;
    const bool ahead = C * kCG <= ITX * kThreads;
    float wn[ITX];
    auto load_tap = [&](int di, int k) {
#pragma unroll
        for (int it = 0; it < ITX; ++it) {
            const int i = threadIdx.x + it * kThreads;
            const int j = i / kCG, cc = i % kCG;
            const int c = c0 + cc;
            wn[it] = (i < C * kCG && c < C) ? to_f(wgt[((long long)(di * C + c) * K2 + k) * C + j]) : 0.0f;
        }
    };
    if (ahead) load_tap(0, 0);
#pragma unroll 1
    for (int di = 0; di < 3; ++di) {
        const int dil = dil_of(d, di);
#pragma unroll 1
        for (int k = 0; k < K2; ++k) {
            __syncthreads();
            if (ahead) {
#pragma unroll
                for (int it = 0; it < ITX; ++it) {
                    const int i = threadIdx.x + it * kThreads;
                    if (i < C * kCG) Ws[i] = wn[it];
                }
                const int nk = k + 1 < K2 ? k + 1 : 0, ndi = k + 1 < K2 ? di : di + 1;
                if (ndi < 3) load_tap(ndi, nk);
            } else {
                for (int i = threadIdx.x; i < C * kCG; i += kThreads) {
                    const int j = i / kCG, cc = i % kCG;
                    const int c = c0 + cc;
                    Ws[i] = c < C ? to_f(wgt[((long long)(di * C + c) * K2 + k) * C + j]) : 0.0f;
                }
            }
            if (threadIdx.x < kCG) {
                const int c = c0 + threadIdx.x;
                bs[threadIdx.x] = (c < C && bias != nullptr) ? to_f(bias[(long long)(di * C + c) * K2 + k]) : 0.0f;
            }
            __syncthreads();
            const int ky = k / K, kx = k % K;
            const int hs = h - (ky - r) * dil, ws = w - (kx - r) * dil;
            if (!active || hs < 0 || hs >= d.H || ws < 0 || ws >= d.W) continue;
            const long long ps = (long long)hs * d.W + ws;
            float t[kCG];
#pragma unroll
            for (int cc = 0; cc < kCG; ++cc) t[cc] = bs[cc];
            for (int j = 0; j < C; ++j) {
                const float yv = ldg_f(yb + (long long)j * d.HW + ps);
                const float4 w0 = reinterpret_cast<const float4*>(Ws + j * kCG)[0];
                const float4 w1 = reinterpret_cast<const float4*>(Ws + j * kCG)[1];
                t[0] = fmaf(w0.x, yv, t[0]); t[1] = fmaf(w0.y, yv, t[1]);
                t[2] = fmaf(w0.z, yv, t[2]); t[3] = fmaf(w0.w, yv, t[3]);
                t[4] = fmaf(w1.x, yv, t[4]); t[5] = fmaf(w1.y, yv, t[5]);
                t[6] = fmaf(w1.z, yv, t[6]); t[7] = fmaf(w1.w, yv, t[7]);
            }
#pragma unroll
            for (int cc = 0; cc < kCG; ++cc) {
                if (c0 + cc < C) {
                    const float gv = to_f(gb[(long long)((1 + di) * C + c0 + cc) * d.HW + ps]);
                    acc[cc] = fmaf(quantise_tap<T>(t[cc]), gv, acc[cc]);
                }
            }
        }
    }
    if (active) {
#pragma unroll
        for (int cc = 0; cc < kCG; ++cc)
            if (c0 + cc < C) dx[((long long)b * C + c0 + cc) * d.HW + q] = from_f<T>(acc[cc]);
    }
}

// ---------------------------------------------------------------- dY --
// dy[b,j,p] = sum_o W[o,j] * dK[b,o,p],  dK = g[b,(1+di)C+c,p] * x[b,c,p+off].
// One thread per pixel keeps kJC accumulators; per channel c the block stages
// the 3*K*K generator rows of c (Ws[(di*K2+k)][jj]) and each thread forms the
// dK of its pixel and applies it to the kJC weights (16-byte broadcasts).
template <typename T, int K>
__global__ void __launch_bounds__(kThreads) dy_kernel(Dims d, const T* __restrict__ g,
                                                      const T* __restrict__ x, const T* __restrict__ wgt,
                                                      T* __restrict__ dy) {
    constexpr int K2 = K * K;
    __shared__ __align__(16) float Ws[3 * K2 * kJC];
    const int r = K / 2;
    const int C = d.C;
    const int b = blockIdx.z;
    const int j0 = blockIdx.y * kJC;
    const long long p = (long long)blockIdx.x * kThreads + threadIdx.x;
    const bool active = p < d.HW;
    const int h = active ? (int)(p / d.W) : 0;
    const int w = active ? (int)(p % d.W) : 0;
    const T* gb = g + (long long)b * 4 * C * d.HW;

    float acc[kJC];
#pragma unroll
    for (int jj = 0; jj < kJC; ++jj) acc[jj] = 0.0f;

    // the generator rows of channel c are staged through registers one channel ahead:
    // channel c+1's loads are in flight while channel c is applied (for K <= 5; K = 7
    // would need 74 registers a thread and stages directly)
    constexpr int ITW0 = (3 * K2 * kJC + kThreads - 1) / kThreads;
    constexpr bool kAhead = ITW0 <= 40;
    constexpr int ITW = kAhead ? ITW0 : 1;
    float wn[ITW];
    auto load_rows = [&](int c) {
#pragma unroll
        for (int it = 0; it < ITW; ++it) {
            const int i = threadIdx.x + it * kThreads;
            const int row = i / kJC, jj = i % kJC;  // row = di*K2 + k
            const int di = row / K2, k = row % K2;
            wn[it] = (i < 3 * K2 * kJC && j0 + jj < C) ? to_f(wgt[((long long)(di * C + c) * K2 + k) * C + j0 + jj])
                                                        : 0.0f;
        }
    };
    if constexpr (kAhead) load_rows(0);
#pragma unroll 1
    for (int c = 0; c < C; ++c) {
        __syncthreads();
        if constexpr (kAhead) {
#pragma unroll
            for (int it = 0; it < ITW; ++it) {
                const int i = threadIdx.x + it * kThreads;
                if (i < 3 * K2 * kJC) Ws[i] = wn[it];
            }
        } else {
            for (int i = threadIdx.x; i < 3 * K2 * kJC; i += kThreads) {
                const int row = i / kJC, jj = i % kJC;  // row = di*K2 + k
                const int di = row / K2, k = row % K2;
                Ws[i] = (j0 + jj < C) ? to_f(wgt[((long long)(di * C + c) * K2 + k) * C + j0 + jj]) : 0.0f;
            }
        }
        __syncthreads();
        if constexpr (kAhead)
            if (c + 1 < C) load_rows(c + 1);
        if (!active) continue;
        const T* xp = x + ((long long)b * C + c) * d.HW;
#pragma unroll 1
        for (int di = 0; di < 3; ++di) {
            const int dil = dil_of(d, di);
            const float gv = to_f(gb[(long long)((1 + di) * C + c) * d.HW + p]);
#pragma unroll
            for (int k = 0; k < K2; ++k) {
                const int ky = k / K, kx = k % K;
                const float dk = gv * x_at(xp, d.H, d.W, h + (ky - r) * dil, w + (kx - r) * dil);
                const float4* wr = reinterpret_cast<const float4*>(Ws + (di * K2 + k) * kJC);
#pragma unroll
                for (int q4 = 0; q4 < kJC / 4; ++q4) {
                    const float4 w4 = wr[q4];
                    acc[4 * q4 + 0] = fmaf(w4.x, dk, acc[4 * q4 + 0]);
                    acc[4 * q4 + 1] = fmaf(w4.y, dk, acc[4 * q4 + 1]);
                    acc[4 * q4 + 2] = fmaf(w4.z, dk, acc[4 * q4 + 2]);
                    acc[4 * q4 + 3] = fmaf(w4.w, dk, acc[4 * q4 + 3]);
                }
            }
        }
    }
    if (active) {
#pragma unroll
        for (int jj = 0; jj < kJC; ++jj)
            if (j0 + jj < C) dy[((long long)b * C + j0 + jj) * d.HW + p] = from_f<T>(acc[jj]);
    }
}

// ------------------------------------------------------------- dW, db --
// Partial sums over split s of the flattened pixels (b, p):
//   ws[s][o][j] = sum_{(b,p) in s} dK[b,o,p] * y[b,j,p]   (j < C)
//   ws[s][o][C] = sum_{(b,p) in s} dK[b,o,p]               (the dbias column)
// A block is a small GEMM: M = the taps of CGW channels of one dilation (CGW*K*K,
// about 72 rows), N = 64 columns of j plus a column of ones that yields dbias, and
// the split's pixels as the reduction, walked in tiles of kPT pixels.  Per tile the
// block stages dK_s[m][pp] (formed from grad and shifted x) and y_s[n][pp] once --
// so y is read once per CGW channels, not once per channel -- and each thread owns
// one 4x4 output micro-tile that it accumulates over the tile's pixels in order
// (16-byte shared loads, no cross-thread reduction).
constexpr int kPT = 64;
constexpr int kNJ = 68;  // 64 j columns + ones column + 3 zero columns
constexpr int kRS = kPT + 4;   // shared row stride (floats): consecutive rows start one 16-byte bank group apart

template <int K>
struct DwTile {
    static constexpr int K2 = K * K;
    static constexpr int CGW = (72 / K2) > 1 ? 72 / K2 : 1;        // channels per block
    static constexpr int MT = (CGW * K2 + 3) / 4 * 4;              // tap rows, padded to the micro-tile
    static constexpr int NM = (MT / 4) * (kNJ / 4);                // 4x4 micro-tiles
    static constexpr int THREADS = (NM + 31) / 32 * 32;
};

template <typename T, int K>
__global__ void __launch_bounds__(DwTile<K>::THREADS, 2) dw_partial_kernel(Dims d, const T* __restrict__ g,
                                                                       const T* __restrict__ x,
                                                                       const T* __restrict__ y,
                                                                       float* __restrict__ ws, long long chunk) {
    using Tl = DwTile<K>;
    constexpr int K2 = K * K, CGW = Tl::CGW, MT = Tl::MT, NM = Tl::NM, NT = Tl::THREADS;
    __shared__ __align__(16) float dK_s[MT * kRS];
    __shared__ __align__(16) float y_s[kNJ * kRS];
    __shared__ int pix_b[kPT], pix_h[kPT], pix_w[kPT];

    const int r = K / 2;
    const int C = d.C;
    const int c0 = blockIdx.x * CGW;
    const int JT = (C + 63) / 64;
    const int di = blockIdx.y / JT;
    const int jt = blockIdx.y % JT;
    const int j0 = jt * 64;
    const int s = blockIdx.z;
    const int dil = dil_of(d, di);
    const long long NP = (long long)d.B * d.HW;
    const long long P0 = (long long)s * chunk;
    const long long P1 = P0 + chunk < NP ? P0 + chunk : NP;
    const int tid = threadIdx.x;
    const bool computes = tid < NM;
    const int mr = tid / (kNJ / 4), mc = tid % (kNJ / 4);

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    for (long long base = P0; base < P1; base += kPT) {
        __syncthreads();
        // pixel coordinates of the tile (b = -1 past the split)
        for (int pp = tid; pp < kPT; pp += NT) {
            const long long P = base + pp;
            if (P < P1) {
                const int b = (int)(P / d.HW);
                const long long p = P - (long long)b * d.HW;
                pix_b[pp] = b;
                pix_h[pp] = (int)(p / d.W);
                pix_w[pp] = (int)(p - (long long)pix_h[pp] * d.W);
            } else {
                pix_b[pp] = -1;
                pix_h[pp] = 0;
                pix_w[pp] = 0;
            }
        }
        __syncthreads();
        // every thread's loads of the tile are issued before any is used (the loops are
        // unrolled into registers), so their latencies overlap instead of adding up
        constexpr int ITK = (MT * kPT + NT - 1) / NT, ITY = (kNJ * kPT + NT - 1) / NT;
        float vk[ITK], vy[ITY];
#pragma unroll
        for (int it = 0; it < ITK; ++it) {
            const int i = tid + it * NT;
            const int m = i / kPT, pp = i - m * kPT;
            const int cl = m / K2, k = m - cl * K2;
            const int c = c0 + cl;
            const int b = i < MT * kPT ? pix_b[pp] : -1;
            float v = 0.0f;
            if (m < CGW * K2 && c < C && b >= 0) {
                const int h = pix_h[pp], w = pix_w[pp];
                const int ky = k / K, kx = k - ky * K;
                const long long p = (long long)h * d.W + w;
                const float gv = to_f(g[((long long)b * 4 * C + (1 + di) * C + c) * d.HW + p]);
                v = gv * x_at(x + ((long long)b * C + c) * d.HW, d.H, d.W, h + (ky - r) * dil, w + (kx - r) * dil);
            }
            vk[it] = v;
        }
#pragma unroll
        for (int it = 0; it < ITY; ++it) {
            const int i = tid + it * NT;
            const int jj = i / kPT, pp = i - jj * kPT;
            const int b = i < kNJ * kPT ? pix_b[pp] : -1;
            float v = 0.0f;
            if (b >= 0) {
                if (jj < 64) {
                    if (j0 + jj < C) v = to_f(y[((long long)b * C + j0 + jj) * d.HW + (long long)pix_h[pp] * d.W + pix_w[pp]]);
                } else if (jj == 64 && jt == 0) {
                    v = 1.0f;
                }
            }
            vy[it] = v;
        }
#pragma unroll
        for (int it = 0; it < ITK; ++it) {
            const int i = tid + it * NT;
            if (i < MT * kPT) dK_s[(i / kPT) * kRS + i % kPT] = vk[it];
        }
#pragma unroll
        for (int it = 0; it < ITY; ++it) {
            const int i = tid + it * NT;
            if (i < kNJ * kPT) y_s[(i / kPT) * kRS + i % kPT] = vy[it];
        }
        __syncthreads();
        if (computes) {
#pragma unroll 4
            for (int qd = 0; qd < kPT / 4; ++qd) {
                float4 a[4], bq[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = reinterpret_cast<const float4*>(dK_s + (4 * mr + i) * kRS)[qd];
#pragma unroll
                for (int j = 0; j < 4; ++j) bq[j] = reinterpret_cast<const float4*>(y_s + (4 * mc + j) * kRS)[qd];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[i][j] = fmaf(a[i].x, bq[j].x, acc[i][j]);
                        acc[i][j] = fmaf(a[i].y, bq[j].y, acc[i][j]);
                        acc[i][j] = fmaf(a[i].z, bq[j].z, acc[i][j]);
                        acc[i][j] = fmaf(a[i].w, bq[j].w, acc[i][j]);
                    }
            }
        }
    }
    if (!computes) return;
    float* wsb = ws + (long long)s * d.O * (C + 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = 4 * mr + i;
        const int cl = m / K2, k = m - cl * K2;
        if (m >= CGW * K2 || c0 + cl >= C) continue;
        const long long o = (long long)(di * C + c0 + cl) * K2 + k;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int jj = 4 * mc + j;
            if (jj < 64) {
                if (j0 + jj < C) wsb[o * (C + 1) + j0 + jj] = acc[i][j];
            } else if (jj == 64 && jt == 0) {
                wsb[o * (C + 1) + C] = acc[i][j];
            }
        }
    }
}

// Sum the partials in split order; cast to the gradient dtype.
template <typename T>
__global__ void __launch_bounds__(256) dw_reduce_kernel(Dims d, const float* __restrict__ ws, int S,
                                                        T* __restrict__ dw, T* __restrict__ db) {
    const long long n = d.O * (d.C + 1);
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        // all partial loads are issued before the sum, which then runs in the fixed order s = 0, 1, ...
        float part[kMaxSplits];
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s) part[s] = s < S ? __ldcs(ws + (long long)s * n + e) : 0.0f;
        float v = 0.0f;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
            if (s < S) v += part[s];
        const long long o = e / (d.C + 1);
        const int j = (int)(e % (d.C + 1));
        if (j < d.C) dw[o * d.C + j] = from_f<T>(v);
        else if (db != nullptr) db[o] = from_f<T>(v);
    }
}

long long split_chunk(const Dims& d, int S) {
    const long long NP = (long long)d.B * d.HW;
    long long chunk = (NP + S - 1) / S;
    return (chunk + kPT - 1) / kPT * kPT;
}

template <typename T, int K>
cudaError_t launch_dx_k(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                        cudaStream_t s) {
    const unsigned pix_blocks = (unsigned)((d.HW + kThreads - 1) / kThreads);
    const size_t smem = sizeof(float) * (size_t)d.C * kCG;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(dx_kernel<T, K>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid(pix_blocks, (unsigned)((d.C + kCG - 1) / kCG), (unsigned)d.B);
    trace_begin(s, kKBwdDxSimt);
    dx_kernel<T, K><<<grid, kThreads, smem, s>>>(d, (const T*)g, (const T*)y, (const T*)w, (const T*)bias, (T*)dx);
    trace_end(s);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t launch_dy_k(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s) {
    const unsigned pix_blocks = (unsigned)((d.HW + kThreads - 1) / kThreads);
    dim3 grid(pix_blocks, (unsigned)((d.C + kJC - 1) / kJC), (unsigned)d.B);
    trace_begin(s, kKBwdDySimt);
    dy_kernel<T, K><<<grid, kThreads, 0, s>>>(d, (const T*)g, (const T*)x, (const T*)w, (T*)dy);
    trace_end(s);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t launch_dw_k(const Dims& d, const void* g, const void* x, const void* y, void* ws, cudaStream_t s) {
    const int S = backward_num_splits(d);
    const int JT = (d.C + 63) / 64;
    dim3 grid((unsigned)((d.C + DwTile<K>::CGW - 1) / DwTile<K>::CGW), (unsigned)(3 * JT), (unsigned)S);
    trace_begin(s, kKBwdDwPartialSimt);
    dw_partial_kernel<T, K><<<grid, DwTile<K>::THREADS, 0, s>>>(d, (const T*)g, (const T*)x, (const T*)y,
                                                                (float*)ws, split_chunk(d, S));
    trace_end(s);
    return cudaGetLastError();
}

template <typename T>
cudaError_t reduce_t(const Dims& d, const float* ws, int S, void* dw, void* db, cudaStream_t s) {
    const long long n = d.O * (d.C + 1);
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    trace_begin(s, kKBwdDwReduce);
    dw_reduce_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(d, ws, S, (T*)dw, (T*)db);
    trace_end(s);
    return cudaGetLastError();
}

template <typename T>
cudaError_t dx_t(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                 cudaStream_t s) {
    switch (d.K) {
        case 1: return launch_dx_k<T, 1>(d, g, y, w, bias, dx, s);
        case 3: return launch_dx_k<T, 3>(d, g, y, w, bias, dx, s);
        case 5: return launch_dx_k<T, 5>(d, g, y, w, bias, dx, s);
        case 7: return launch_dx_k<T, 7>(d, g, y, w, bias, dx, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t dy_t(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s) {
    switch (d.K) {
        case 1: return launch_dy_k<T, 1>(d, g, x, w, dy, s);
        case 3: return launch_dy_k<T, 3>(d, g, x, w, dy, s);
        case 5: return launch_dy_k<T, 5>(d, g, x, w, dy, s);
        case 7: return launch_dy_k<T, 7>(d, g, x, w, dy, s);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t dw_t(const Dims& d, const void* g, const void* x, const void* y, void* ws, cudaStream_t s) {
    switch (d.K) {
        case 1: return launch_dw_k<T, 1>(d, g, x, y, ws, s);
        case 3: return launch_dw_k<T, 3>(d, g, x, y, ws, s);
        case 5: return launch_dw_k<T, 5>(d, g, x, y, ws, s);
        case 7: return launch_dw_k<T, 7>(d, g, x, y, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int backward_num_splits(const Dims& d) {
    const long long NP = (long long)d.B * d.HW;
    long long S = (NP + 2047) / 2048;
    if (S < 1) S = 1;
    if (S > kMaxSplits) S = kMaxSplits;
    return (int)S;
}

size_t backward_simt_workspace(const Dims& d) {
    return sizeof(float) * (size_t)backward_num_splits(d) * (size_t)d.O * (size_t)(d.C + 1);
}

cudaError_t launch_bwd_dx_simt(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                               cudaStream_t s) {
    if (d.dtype == 1) return dx_t<__nv_bfloat16>(d, g, y, w, bias, dx, s);
    return dx_t<float>(d, g, y, w, bias, dx, s);
}

cudaError_t launch_bwd_dy_simt(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s) {
    if (d.dtype == 1) return dy_t<__nv_bfloat16>(d, g, x, w, dy, s);
    return dy_t<float>(d, g, x, w, dy, s);
}

cudaError_t launch_bwd_dw_partial_simt(const Dims& d, const void* g, const void* x, const void* y, void* ws,
                                       cudaStream_t s) {
    if (d.dtype == 1) return dw_t<__nv_bfloat16>(d, g, x, y, ws, s);
    return dw_t<float>(d, g, x, y, ws, s);
}

cudaError_t launch_bwd_reduce(const Dims& d, const float* ws, int S, void* dw, void* db, cudaStream_t s) {
    if (d.dtype == 1) return reduce_t<__nv_bfloat16>(d, ws, S, dw, db, s);
    return reduce_t<float>(d, ws, S, dw, db, s);
}

cudaError_t launch_backward_simt(const Dims& d, const void* g, const void* x, const void* y, const void* w,
                                 const void* bias, void* dx, void* dy, void* dw, void* db, void* ws,
                                 cudaStream_t s) {
    cudaError_t e = launch_bwd_dx_simt(d, g, y, w, bias, dx, s);
    if (e != cudaSuccess) return e;
    e = launch_bwd_dy_simt(d, g, x, w, dy, s);
    if (e != cudaSuccess) return e;
    e = launch_bwd_dw_partial_simt(d, g, x, y, ws, s);
    if (e != cudaSuccess) return e;
    return launch_bwd_reduce(d, (const float*)ws, backward_num_splits(d), dw, db, s);
}

}  // namespace ddpm
