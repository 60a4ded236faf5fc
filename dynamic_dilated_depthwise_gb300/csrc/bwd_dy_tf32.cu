// bwd_dy_tf32.cu -- dY of FP32 problems on tcgen05 tensor cores (TF32), under
// DDPM_FLAG_TF32_BACKWARD.
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练": dY forms
// dK = shifted(x) * grad on chip and contracts it with the weight at once,
//   dy[b,j,p] = sum_o W[o,j] * dK[b,o,p],  dK[o,p] = grad[(1+d)C+c, p] * x[c, p+off(d,k)],
// o = (d*C + c)*9 + k; the page's precision policy allows TF32 for the FP32 backward's
// contractions.
//
// GB300 design.  tcgen05 reads TF32 operands K-major, so the contraction is laid out with
// the pixels as M and (tap, channel) as K:
//   D[px, j] += sum_{k, c in block} dK[px, (k, c)] * Wt[(k, c), j]
// A persistent CTA owns a 4 x 32 pixel tile (M = 128, slot m = r*32 + col) and walks
// units of (dilation d, block of 16 channels cb) -- 3 * C/16 units per tile -- and in each
// unit the 9 taps:
//   - a producer warp's TMA brings the unit's grad plane [16 ch][4 x 32 px] and x window
//     [16 ch][4 + 2R rows][48 cols] (zero outside the image) into a 2-stage ring;
//   - eight former warps form each tap's A operand dK[128 px x 16 ch] in FP32 (thread =
//     pixel and 8 channels; grad read once per unit, x at the tap's offset) into a 4-stage
//     ring, in the no-swizzle K-major core-matrix layout (element (m, q) at
//     (m/8)*512 + (q/4)*128 + (m%8)*16 + (q%4)*4);
//   - another producer warp streams the matching B operand, the weight rows of those taps
//     and channels transposed to [N = C][16] in the same core-matrix layout, with one bulk
//     copy per tap from a copy of W that a small kernel rearranges once per call (Wt);
//   - one thread issues two kind::tf32 MMAs (K = 8 each) per tap into one TMEM
//     accumulator [128 x C], FP32;
//   - after the tile's last unit the formers read the accumulator (TMEM lane = pixel) and
//     write dy directly (a warp stores 32 consecutive pixels of one channel).
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

constexpr int kTH = 4, kTW = 32, kTile = kTH * kTW;   // pixel tile (MMA M = 128)
constexpr int kCB = 16;                               // channels per unit (K per tap)
constexpr int kMaxHalo = 6;                           // halo radius the window buffers hold
constexpr int kWinRows = kTH + 2 * kMaxHalo;          // 16
constexpr int kWinCols = kTW + 16;                    // 48: columns w0 - 8 .. w0 + 39
constexpr int kFormWarps = 8;
constexpr int kThreads = 32 * (3 + kFormWarps);       // window producer, MMA, Wt producer, formers
constexpr int kWinStages = 2, kDkStages = 4, kWtStages = 8;
constexpr int kGBytes = kCB * kTile * 4;              // 8 KiB
constexpr int kXBytesMax = kCB * kWinRows * kWinCols * 4;   // 48 KiB
constexpr int kWinStage = kGBytes + kXBytesMax;
constexpr int kDkBytes = kTile * kCB * 4;             // 8 KiB
constexpr int kWtMax = 64 * kCB * 4;                  // 4 KiB (N = C <= 64)

// shared memory (bytes from a 1024-aligned base)
constexpr int kSWin = 0;
constexpr int kSDk = kSWin + kWinStages * kWinStage;
constexpr int kSWt = kSDk + kDkStages * kDkBytes;
constexpr int kSmemBytes = kSWt + kWtStages * kWtMax + 1024;
static_assert(kWinStage % 128 == 0 && kSDk % 128 == 0 && kSWt % 128 == 0, "TMA / bulk destinations");
static_assert(kSmemBytes <= 227 * 1024 - 512, "shared memory");

struct DyTf32Params {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int n_cb, units;            // C / 16 channel blocks; 3 * n_cb units per tile
    int R, win_rows;            // halo radius; x window rows of the TMA box (4 + 2R)
    uint32_t x_bytes;           // bytes of one x window box
    uint32_t wt_bytes;          // bytes of one Wt tap tile (C * 16 * 4)
    const float* wt;            // rearranged weight, [d][k][cb] tiles of wt_bytes
    float* dy;
    unsigned int* err;
};

// Wt tile (d, k, cb): element (n = j, q = local channel) at (n/8)*512 + (q/4)*128 + (n%8)*16
// + (q%4)*4 bytes holds W[(d*C + cb*16 + q)*9 + k][j] -- the B operand of tap (d, k) for
// channel block cb, ready for one bulk copy.
__global__ void __launch_bounds__(256) wt_pack_kernel(const float* __restrict__ w, float* __restrict__ wt, int C) {
    const long long total = 27LL * C * C;     // 3 dilations x 9 taps x C channels x C outputs j
    const int n_cb = C / kCB;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        // destination order: tile (d, k, cb), then n/8, q/4, n%8, q%4
        const long long tile = i / (C * kCB), rem = i % (C * kCB);
        const int n8 = (int)(rem / 128), r2 = (int)(rem % 128);
        const int q4 = r2 / 32, r3 = r2 % 32, nm = r3 / 4, qm = r3 % 4;
        const int n = n8 * 8 + nm, q = q4 * 4 + qm;
        const int cb = (int)(tile % n_cb), dk = (int)(tile / n_cb), d = dk / 9, k = dk % 9;
        wt[i] = w[((long long)(d * C + cb * kCB + q) * 9 + k) * C + n];
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dy_tf32_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                       const DyTf32Params P) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base by pointer arithmetic on the shared array (accesses stay shared-space)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t win_full[kWinStages], win_empty[kWinStages], dk_full[kDkStages], dk_empty[kDkStages],
        wt_full[kWtStages], wt_empty[kWtStages], acc_full, acc_empty, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.d.C, H = P.d.H, W = P.d.W;
    const int n_my = blockIdx.x < P.n_tiles ? (P.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int units = P.units;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kWinStages; ++i) {
            mbar_init(&win_full[i], 1);
            mbar_init(&win_empty[i], kFormWarps);
        }
        for (int i = 0; i < kDkStages; ++i) {
            mbar_init(&dk_full[i], kFormWarps);
            mbar_init(&dk_empty[i], 1);
        }
        for (int i = 0; i < kWtStages; ++i) {
            mbar_init(&wt_full[i], 1);
            mbar_init(&wt_empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, kFormWarps);
        mbar_init(&mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- window producer
        if (lane == 0) {
            prefetch_tmap(&tmG);
            prefetch_tmap(&tmX);
            int issued = 0;
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                const int t = blockIdx.x + tl * gridDim.x;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kTH, w0 = (ti % P.tiles_w) * kTW;
                for (int u = 0; u < units; ++u) {
                    const int i = tl * units + u, s = i % kWinStages, ph = (i / kWinStages) & 1;
                    if (!mbar_wait(&win_empty[s], ph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    const int dd = u / P.n_cb, cb = u % P.n_cb;
                    uint8_t* st = sm + kSWin + s * kWinStage;
                    mbar_arrive_expect_tx(&win_full[s], kGBytes + P.x_bytes);
                    tma_load_4d(st, &tmG, &win_full[s], w0, h0, (1 + dd) * C + cb * kCB, b);
                    tma_load_4d(st + kGBytes, &tmX, &win_full[s], w0 - 8, h0 - P.R, cb * kCB, b);
                    issued = i + 1;
                }
            }
            int never = 0;
            for (int i = issued > kWinStages ? issued - kWinStages : 0; i < issued; ++i)
                mbar_wait(&win_full[i % kWinStages], (i / kWinStages) & 1, P.err, &never);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------- Wt producer: one bulk copy per tap
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl)
                for (int u = 0; u < units && ok; ++u) {
                    const int dd = u / P.n_cb, cb = u % P.n_cb;
                    for (int k = 0; k < 9; ++k) {
                        const int i = (tl * units + u) * 9 + k, s = i % kWtStages, ph = (i / kWtStages) & 1;
                        if (!mbar_wait(&wt_empty[s], ph ^ 1, P.err, abort_v)) {
                            ok = false;
                            break;
                        }
                        const float* src = P.wt + ((long long)(dd * 9 + k) * P.n_cb + cb) * (P.wt_bytes / 4);
                        mbar_arrive_expect_tx(&wt_full[s], P.wt_bytes);
                        bulk_load(sm + kSWt + s * kWtMax, src, P.wt_bytes, &wt_full[s]);
                        issued = i + 1;
                    }
                }
            int never = 0;
            for (int i = issued > kWtStages ? issued - kWtStages : 0; i < issued; ++i)
                mbar_wait(&wt_full[i % kWtStages], (i / kWtStages) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(2, 0, 0, kTile, (uint32_t)C);   // TF32, both K-major
            const uint64_t a_base = smem_desc(smem_u32(sm + kSDk), 128, 512, kSwizzleNone);
            const uint64_t b_base = smem_desc(smem_u32(sm + kSWt), 128, 512, kSwizzleNone);
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                if (!mbar_wait(&acc_empty, (tl & 1) ^ 1, P.err, abort_v)) break;
                tc_fence_after();
                for (int u = 0; u < units && ok; ++u)
                    for (int k = 0; k < 9; ++k) {
                        const int i = (tl * units + u) * 9 + k;
                        const int sd = i % kDkStages, pd = (i / kDkStages) & 1;
                        const int sw = i % kWtStages, pw = (i / kWtStages) & 1;
                        if (!mbar_wait(&dk_full[sd], pd, P.err, abort_v) || !mbar_wait(&wt_full[sw], pw, P.err, abort_v)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t a = desc_advance(a_base, (uint32_t)(sd * kDkBytes));
                        const uint64_t b = desc_advance(b_base, (uint32_t)(sw * kWtMax));
                        const uint32_t first = (u == 0 && k == 0) ? 0u : 1u;
                        mma_tf32(tmem, a, b, idesc, first);
                        mma_tf32(tmem, desc_advance(a, 256), desc_advance(b, 256), idesc, 1u);
                        mma_commit(&dk_empty[sd]);
                        mma_commit(&wt_empty[sw]);
                    }
                if (ok) mma_commit(&acc_full);
            }
            mma_commit(&mma_done);
            int never = 0;
            mbar_wait(&mma_done, 0, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- formers + epilogue
        const int q = warp & 3;                          // TMEM lane quadrant this warp may access
        const int m = q * 32 + lane;                     // pixel slot == TMEM lane: one tile row per warp
        const int half = (warp - 3) >> 2;                // channels 8*half .. 8*half+7 of the unit
        const int r = m / kTW, col = m % kTW;
        bool ok = true;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            const int t = blockIdx.x + tl * gridDim.x;
            const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
            const int h0 = (ti / P.tiles_w) * kTH, w0 = (ti % P.tiles_w) * kTW;
            for (int u = 0; u < units && ok; ++u) {
                const int iw = tl * units + u, s = iw % kWinStages, ph = (iw / kWinStages) & 1;
                if (!mbar_wait(&win_full[s], ph, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                const int dd = u / P.n_cb;
                const int dil = dil_of(P.d, dd);
                const float* gs = reinterpret_cast<const float*>(sm + kSWin + s * kWinStage);   // [16][128]
                const float* xs = reinterpret_cast<const float*>(sm + kSWin + s * kWinStage + kGBytes);
                float g[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = gs[(half * 8 + e) * kTile + m];
                // this pixel's window position at tap offset 0
                const int xc = (r + P.R) * kWinCols + col + 8;
                const int plane = P.win_rows * kWinCols;
                for (int k = 0; k < 9; ++k) {
                    const int i = iw * 9 + k, sd = i % kDkStages, pd = (i / kDkStages) & 1;
                    if (!mbar_wait(&dk_empty[sd], pd ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    const int off = ((k / 3 - 1) * kWinCols + (k % 3 - 1)) * dil;
                    uint8_t* dk = sm + kSDk + sd * kDkBytes + (m / 8) * 512 + (m % 8) * 16;
#pragma unroll
                    for (int cq = 0; cq < 2; ++cq) {
                        const int c = half * 8 + cq * 4;
                        float4 v;
                        v.x = g[cq * 4 + 0] * xs[(c + 0) * plane + xc + off];
                        v.y = g[cq * 4 + 1] * xs[(c + 1) * plane + xc + off];
                        v.z = g[cq * 4 + 2] * xs[(c + 2) * plane + xc + off];
                        v.w = g[cq * 4 + 3] * xs[(c + 3) * plane + xc + off];
                        *reinterpret_cast<float4*>(dk + (c / 4) * 128) = v;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dk_full[sd]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&win_empty[s]);
            }
            if (!ok) break;
            // epilogue: D[m, j] for this thread's 32 output channels j = 32*half .. (TMEM lane m)
            if (!mbar_wait(&acc_full, tl & 1, P.err, abort_v)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[32];
            const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 32);
            if (half * 32 < C) {
                DDPM_TMEM_LD_X16(ta, v);
                DDPM_TMEM_LD_X16(ta + 16, (v + 16));
                tmem_ld_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty);
            const int h = h0 + r, w = w0 + col;
            if (h < H && w < W && half * 32 < C) {
                float* dyp = P.dy + (long long)b * C * P.d.HW + (long long)h * W + w;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int j = half * 32 + jj;
                    if (j < C) dyp[(long long)j * P.d.HW] = __uint_as_float(v[jj]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// 4-D FP32 tensor map over an NCHW tensor with `ch` channels: dims (W, H, ch, B).
bool encode_f32(CUtensorMap* m, const void* base, const Dims& d, int ch, uint32_t bw, uint32_t bh, uint32_t bc) {
    const cuuint64_t dims[4] = {(cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)ch, (cuuint64_t)d.B};
    const cuuint64_t str[3] = {(cuuint64_t)d.W * 4, (cuuint64_t)d.HW * 4, (cuuint64_t)d.HW * ch * 4};
    const cuuint32_t box[4] = {bw, bh, bc, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return bwdtc::encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, str, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// FP32 problems that asked for TF32 backward contractions: K = 3, C a multiple of 16 up to
// 64 (N = C, 16-channel units), W a multiple of 4, halo radius <= 6, 16-byte aligned.
bool bwd_dy_tf32_shape_ok(const Dims& d) {
    if (d.dtype != 0 || !(d.flags & kFlagTf32Backward) || (d.flags & kFlagCudaCores) || d.K != 3) return false;
    if (d.C % kCB != 0 || d.C > 64 || d.W % 4 != 0 || d.R() > kMaxHalo) return false;
    return d.O <= (1LL << 30) && d.HW <= (1LL << 31) - 1024;
}

bool bwd_dy_tf32_eligible(const Dims& d, const void* g, const void* x, const void* w, const void* dy) {
    if (!bwd_dy_tf32_shape_ok(d)) return false;
    if ((uintptr_t)g % 16 || (uintptr_t)x % 16 || (uintptr_t)w % 16 || (uintptr_t)dy % 4) return false;
    return bwdtc::encode_fn() != nullptr;
}

size_t bwd_dy_tf32_wt_bytes(const Dims& d) { return (size_t)27 * d.C * d.C * sizeof(float); }

cudaError_t launch_bwd_dy_tf32(const Dims& d, const void* g, const void* x, const void* w, void* dy, void* wt,
                               cudaStream_t s) {
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dy_tf32_kernel, kSmemBytes, attr_done);
        if (e != cudaSuccess) return e;
    }
    if ((uintptr_t)wt % 16 != 0) return cudaErrorInvalidValue;
    DyTf32Params P;
    P.d = d;
    P.tiles_w = (d.W + kTW - 1) / kTW;
    P.tiles_per_img = ((d.H + kTH - 1) / kTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.n_cb = d.C / kCB;
    P.units = 3 * P.n_cb;
    P.R = d.R();
    P.win_rows = kTH + 2 * P.R;
    P.x_bytes = (uint32_t)(kCB * P.win_rows * kWinCols * 4);
    P.wt_bytes = (uint32_t)(d.C * kCB * 4);
    P.wt = static_cast<const float*>(wt);
    P.dy = static_cast<float*>(dy);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    CUtensorMap tmG, tmX;
    if (!encode_f32(&tmG, g, d, 4 * d.C, kTW, kTH, kCB) ||
        !encode_f32(&tmX, x, d, d.C, kWinCols, (uint32_t)P.win_rows, kCB))
        return cudaErrorInvalidValue;
    trace_begin(s, kKBwdDyTf32);
    wt_pack_kernel<<<num_sms() * 2, 256, 0, s>>>(static_cast<const float*>(w), static_cast<float*>(wt), d.C);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) {
        int grid = num_sms();
        if (grid > P.n_tiles) grid = P.n_tiles;
        bwd_dy_tf32_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmG, tmX, P);
        e = cudaGetLastError();
    }
    trace_end(s);
    return e;
}

}  // namespace ddpm
