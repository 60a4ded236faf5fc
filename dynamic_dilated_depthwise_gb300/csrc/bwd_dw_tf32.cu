// bwd_dw_tf32.cu -- dW / dbias split partials of FP32 problems on tcgen05 tensor cores (TF32).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dWeight/dbias form dK = shifted(x) * grad on chip and reduce it over space,
// split into at most 16 FP32 partials that a second short kernel sums; the
// page's precision policy allows TF32 for the FP32 backward's reductions.
//
//   ws[s][o][j] = sum_{pixels p of split s} dK[o, p] * y[j, p]     (j < C)
//   ws[s][o][C] = sum_p dK[o, p]                                    (dbias)
//
// The FP32 counterpart of bwd_dw_tc.cu.  dK[o, p] = grad * x is formed in FP32 on
// CUDA cores; the tensor cores read it (and y) as TF32 and accumulate in FP32.
// A CTA owns a block of taps (14 channels of one dilation, 126 taps, for K = 3; 5
// channels, 125 taps, for K = 5; padded to M = 128) and one pixel split; per 1x64
// pixel tile:
//   - one producer warp's TMA brings y [64 j x 64 px] FP32 as two 128-byte
//     swizzled halves of 32 pixels (K-major operand) into a 2-stage ring the
//     MMA releases;
//   - another brings the block's grad rows [CB x 64 px] and x windows
//     [CB x (1+2R) x (64 + 2 halo)] (zero outside the image) into a 2-stage ring the
//     formers release as soon as dK is formed;
//   - two groups of eight warps (even and odd tiles) form dK^T[o, px] into a 128B-swizzled K-major tile (32 KiB);
//   - one thread issues D[o, n] += dK^T[o, px] * Y[n, px], kind::tf32, M = 128,
//     N = 80 (64 y channels, a ones row for dbias, 15 zero rows), K = 8 per
//     instruction: eight instructions per tile.
// The accumulator stays in TMEM for the whole split and is written once.
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using namespace bwdtc;

constexpr int kTW32 = 64;                          // pixels of a tile (one image row)
constexpr int kNY = 80;                            // MMA N: 64 y channels + ones row + 15 zero rows
constexpr int kGroupWarps = 8;                     // warps of one former group
constexpr int kFormWarps = 2 * kGroupWarps;        // two groups: even and odd tiles
constexpr int kThreads = 32 * (3 + kFormWarps);    // x/grad producer, MMA, formers, y producer
constexpr int kYWarp = 2 + kFormWarps;
constexpr int kYStages = 2, kXgStages = 2;
// tile i uses x/grad stage i % 2 and is formed by group i % 2: each stage serves one group,
// so each group waits on a barrier whose previous phase it has seen itself
static_assert(kXgStages == 2, "one x/grad stage per former group");
constexpr int kSmemCap = 232448 - 1024;            // dynamic shared memory: the opt-in 227 KiB less the static part

// Per kernel size: channels per block of taps, the x window's column halo (left and
// right of the tile, a 32-byte TMA coordinate, >= the taps' horizontal reach), its
// width, and the halo radius two x/grad stages hold.
template <int K> struct Tf32Geom;
template <> struct Tf32Geom<3> { static constexpr int CB = 14, HALO = 8, WIN = kTW32 + 16, MAXR = 6; };
template <> struct Tf32Geom<5> { static constexpr int CB = 5, HALO = 16, WIN = kTW32 + 32, MAXR = 10; };

// shared memory (bytes from a 1024-aligned base)
constexpr int kDK = 0;                             // 2 x dK^T tiles [128 taps x 64 px] FP32, 32 KiB each
constexpr int kDK32 = kBlockRows * kTW32 * 4;
constexpr int kYS = kDK + 2 * kDK32;               // y ring: stages x 2 halves x [80 rows x 128 B]
constexpr int kYHalf = kNY * 128;
constexpr int kYStage = 2 * kYHalf;
constexpr int kXG = kYS + kYStages * kYStage;      // x/grad ring
static_assert(kDK32 == 32768 && kYS % 1024 == 0 && kYHalf % 1024 == 0, "SW128 atoms need 1 KiB");

template <int K>
struct Tf32Layout {
    using G = Tf32Geom<K>;
    static constexpr int kGStage = G::CB * kTW32 * 4;   // grad rows of the block [CB x 64 px] FP32
    static constexpr int kXgMax = kGStage + G::CB * (1 + 2 * G::MAXR) * G::WIN * 4;
    static constexpr int kSmemBytes = kXG + kXgStages * kXgMax + 1024 + 128;   // + alignment slack + over-read margin
    static_assert(kXG % 128 == 0 && kGStage % 128 == 0, "TMA dst 128 B");
    static_assert(kSmemBytes <= kSmemCap, "shared memory");
};

struct DwTf32Params {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int n_cblk, n_oblk, tiles_per_split;
    int R, WHx;            // halo radius, window rows (1 + 2R)
    int xslot;             // bytes of one channel's x window: WHx * window columns * 4
    int xg_stage;          // bytes of one x/grad stage, a multiple of 128
    float* ws;             // [S][O][C+1]
    unsigned int* err;
};

// Form one dK^T tile in FP32: dK[r, px] = grad_d[c, px] * x[c, px + off(d, k)], r = c*K*K + k.
// Layout: pixel half h (px / 32) at +16 KiB * h, tap row r at (r/8)*1024 + (r%8)*128,
// 16-byte chunk (px%32)/4 XOR (r%8).  Work unit = (channel, 4-pixel chunk j): the
// grad chunk is one 16-byte load; each of the K window rows gives the aligned vectors
// of window columns 4j .. 4j+3+2H (H = the window's column halo; the chunk sits at
// columns 4j+H .. 4j+H+3), from which the K horizontal taps are taken at compile-time
// offsets H + (kx-r)*DIL; only the vectors the taps reach are loaded.  A warp's loads
// and stores touch each bank once per eight threads.  Rows of channels >= nc are
// written as zeros.
template <int K, int DIL>
__device__ __forceinline__ void form_dk_f32_dil(uint8_t* dk, const float* xs, const float* gs, int nc, int xslot_f,
                                                int R, int tid, int nthr) {
    using G = Tf32Geom<K>;
    constexpr int kH = G::HALO, kNV = (4 + 2 * kH) / 4, r0 = K / 2;
    static_assert(DIL >= 1 && r0 * DIL <= kH, "the window holds the taps' horizontal reach");
    for (int u = tid; u < G::CB * 16; u += nthr) {
        const int cl = u >> 4, j = u & 15;
        uint8_t* colbase = dk + (j >> 3) * 16384;
        const int sw = j & 7;
        if (cl >= nc) {
#pragma unroll
            for (int k = 0; k < K * K; ++k) {
                const int r = cl * K * K + k;
                *reinterpret_cast<float4*>(colbase + (r >> 3) * 1024 + (r & 7) * 128 + ((sw ^ (r & 7)) << 4)) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
            }
            continue;
        }
        const float4 gv = *reinterpret_cast<const float4*>(gs + cl * kTW32 + j * 4);
        const float g[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            const float* row = xs + cl * xslot_f + (R + (ky - r0) * DIL) * G::WIN + j * 4;
            float w[4 * kNV];
#pragma unroll
            for (int v = 0; v < kNV; ++v) {
                // only the vectors the K taps reach are loaded (compile-time indices)
                if (v * 4 + 3 >= kH - r0 * DIL && v * 4 <= kH + 3 + r0 * DIL) {
                    const float4 q = *reinterpret_cast<const float4*>(row + v * 4);
                    w[v * 4 + 0] = q.x;
                    w[v * 4 + 1] = q.y;
                    w[v * 4 + 2] = q.z;
                    w[v * 4 + 3] = q.w;
                }
            }
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int off = kH + (kx - r0) * DIL;
                const int r = cl * K * K + ky * K + kx;
                float4 o;
                o.x = g[0] * w[off + 0];
                o.y = g[1] * w[off + 1];
                o.z = g[2] * w[off + 2];
                o.w = g[3] * w[off + 3];
                *reinterpret_cast<float4*>(colbase + (r >> 3) * 1024 + (r & 7) * 128 + ((sw ^ (r & 7)) << 4)) = o;
            }
        }
    }
}

template <int K>
__device__ __forceinline__ void form_dk_f32(uint8_t* dk, const float* xs, const float* gs, int nc, int xslot_f, int R,
                                            int dil, int tid, int nthr) {
    switch (dil) {
        case 1: form_dk_f32_dil<K, 1>(dk, xs, gs, nc, xslot_f, R, tid, nthr); break;
        case 2: form_dk_f32_dil<K, 2>(dk, xs, gs, nc, xslot_f, R, tid, nthr); break;
        case 3: form_dk_f32_dil<K, 3>(dk, xs, gs, nc, xslot_f, R, tid, nthr); break;
        case 4: form_dk_f32_dil<K, 4>(dk, xs, gs, nc, xslot_f, R, tid, nthr); break;
        case 5: form_dk_f32_dil<K, 5>(dk, xs, gs, nc, xslot_f, R, tid, nthr); break;
        default: form_dk_f32_dil<K, (K == 3 ? 6 : 5)>(dk, xs, gs, nc, xslot_f, R, tid, nthr); break;
    }
}

// Zero the padding rows (CB*K*K .. 127) of an FP32 dK^T tile.
template <int K>
__device__ __forceinline__ void zero_pad_rows_f32(uint8_t* dk, int tid, int nthr) {
    constexpr int r0 = Tf32Geom<K>::CB * K * K, npad = kBlockRows - r0;
    for (int u = tid; u < npad * 2 * 8; u += nthr) {   // pad rows x 2 halves x 8 chunks
        const int r = r0 + (u >> 4), half = (u >> 3) & 1, c = u & 7;
        *reinterpret_cast<float4*>(dk + half * 16384 + (r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4)) =
            make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <int K>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dw_tf32_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmG,
                       const __grid_constant__ CUtensorMap tmX, const DwTf32Params P) {
    using namespace tc;
    using G = Tf32Geom<K>;
    constexpr int kCB = G::CB, kTaps = K * K, kGStage = Tf32Layout<K>::kGStage;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base, derived by pointer arithmetic on the shared array so that every
    // access through it stays a shared-memory access
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t y_full[kYStages], y_empty[kYStages], xg_full[kXgStages], xg_empty[kXgStages];
    __shared__ uint64_t dk_full[2], dk_empty[2], acc_done, mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.d.C;
    const long long O = P.d.O;
    const int ob = blockIdx.x % P.n_oblk;
    const int split = blockIdx.x / P.n_oblk;
    const int t_begin = split * P.tiles_per_split;
    const int t_end = min(t_begin + P.tiles_per_split, P.n_tiles);
    const int n_my = max(0, t_end - t_begin);

    // this block of taps: dilation dd, channels [c_first, c_first + nc)
    const int dd = ob / P.n_cblk;
    const int c_first = (ob % P.n_cblk) * kCB;
    const int nc = min(kCB, C - c_first);
    const int nrows = nc * kTaps;
    const int dil = dil_of(P.d, dd);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kYStages; ++s) {
            mbar_init(&y_full[s], 1);
            mbar_init(&y_empty[s], 1);
        }
        for (int s = 0; s < kXgStages; ++s) {
            mbar_init(&xg_full[s], 1);
            mbar_init(&xg_empty[s], kGroupWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&dk_full[s], kGroupWarps);
            mbar_init(&dk_empty[s], 1);
        }
        mbar_init(&acc_done, 1);
        mbar_init(&mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 128);
    if (warp >= 2 && warp < 2 + kFormWarps) {
        // rows 64..79 of every y stage / half: a row of ones (dbias) and 15 zero rows
        const int et = threadIdx.x - 64;
        for (int i = et; i < kYStages * 2 * 16 * 32; i += 32 * kFormWarps) {
            const int word = i % 32, row = (i / 32) % 16, half = (i / 512) % 2, st = i / 1024;
            const uint32_t v = row == 0 ? 0x3F800000u : 0u;   // FP32 1.0
            reinterpret_cast<uint32_t*>(sm + kYS + st * kYStage + half * kYHalf + (64 + row) * 128)[word] = v;
        }
        zero_pad_rows_f32<K>(sm + kDK, et, 32 * kFormWarps);
        zero_pad_rows_f32<K>(sm + kDK + kDK32, et, 32 * kFormWarps);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- x / grad producer
        if (lane == 0) {
            prefetch_tmap(&tmG);
            prefetch_tmap(&tmX);
            const uint32_t bytes = kGStage + kCB * P.xslot;
            int issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % kXgStages, ph = (i / kXgStages) & 1;
                if (!mbar_wait(&xg_empty[s], ph ^ 1, P.err, abort_v)) break;
                const int t = t_begin + i;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = ti / P.tiles_w, w0 = (ti % P.tiles_w) * kTW32;
                uint8_t* st = sm + kXG + s * P.xg_stage;
                mbar_arrive_expect_tx(&xg_full[s], bytes);
                tma_load_4d(st, &tmG, &xg_full[s], w0, h0, (1 + dd) * C + c_first, b);
                tma_load_4d(st + kGStage, &tmX, &xg_full[s], w0 - G::HALO, h0 - P.R, c_first, b);
                issued = i + 1;
            }
            // drain: every copy this thread started lands before its shared memory is released
            int never = 0;
            for (int i = issued > kXgStages ? issued - kXgStages : 0; i < issued; ++i)
                mbar_wait(&xg_full[i % kXgStages], (i / kXgStages) & 1, P.err, &never);
        }
    } else if (warp == kYWarp) {
        // ------------------------------------------------------- y producer
        if (lane == 0) {
            prefetch_tmap(&tmY);
            int issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % kYStages, ph = (i / kYStages) & 1;
                if (!mbar_wait(&y_empty[s], ph ^ 1, P.err, abort_v)) break;
                const int t = t_begin + i;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = ti / P.tiles_w, w0 = (ti % P.tiles_w) * kTW32;
                uint8_t* ys = sm + kYS + s * kYStage;
                mbar_arrive_expect_tx(&y_full[s], 2 * 8192);
                tma_load_4d(ys, &tmY, &y_full[s], w0, h0, 0, b);
                tma_load_4d(ys + kYHalf, &tmY, &y_full[s], w0 + 32, h0, 0, b);
                issued = i + 1;
            }
            int never = 0;
            for (int i = issued > kYStages ? issued - kYStages : 0; i < issued; ++i)
                mbar_wait(&y_full[i % kYStages], (i / kYStages) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(2, 0, 0, kBlockRows, kNY);   // TF32, both operands K-major
            const uint64_t dk_base = smem_desc(smem_u32(sm + kDK), 16, 1024, kSwizzle128B);
            const uint64_t y_base = smem_desc(smem_u32(sm + kYS), 16, 1024, kSwizzle128B);
            bool ok = true;
            for (int i = 0; i < n_my && ok; ++i) {
                const int s = i & 1, ph = (i >> 1) & 1;
                const int sy = i % kYStages, yph = (i / kYStages) & 1;
                if (!mbar_wait(&dk_full[s], ph, P.err, abort_v) || !mbar_wait(&y_full[sy], yph, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t da = desc_advance(dk_base, (uint32_t)s * kDK32);
                const uint64_t ya = desc_advance(y_base, (uint32_t)sy * kYStage);
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_tf32(tmem, desc_advance(da, half * 16384 + kk * 32), desc_advance(ya, half * kYHalf + kk * 32),
                                 idesc, (i > 0 || half > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&dk_empty[s]);
                mma_commit(&y_empty[sy]);
            }
            if (ok) mma_commit(&acc_done);
            mma_commit(&mma_done);
            int never = 0;
            mbar_wait(&mma_done, 0, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- dK formers + epilogue
        // group grp forms tiles grp, grp + 2, ... into dK^T buffer grp
        const int grp = (warp - 2) / kGroupWarps;
        const int et = threadIdx.x - 64 - grp * 32 * kGroupWarps;
        bool ok = true;
        for (int i = grp; i < n_my && ok; i += 2) {
            const int s = i & 1, ph = (i >> 1) & 1;
            const int sx = i % kXgStages, xph = (i / kXgStages) & 1;
            if (!mbar_wait(&xg_full[sx], xph, P.err, abort_v) || !mbar_wait(&dk_empty[s], ph ^ 1, P.err, abort_v)) {
                ok = false;
                break;
            }
            const uint8_t* st = sm + kXG + sx * P.xg_stage;
            form_dk_f32<K>(sm + kDK + s * kDK32, reinterpret_cast<const float*>(st + kGStage),
                        reinterpret_cast<const float*>(st), nc, P.xslot / 4, P.R, dil, et, 32 * kGroupWarps);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&dk_full[s]);
                mbar_arrive(&xg_empty[sx]);
            }
        }
        // epilogue (group 0): this split's partial sums for the block of taps
        if (grp != 0) ok = false;
        const int q = warp & 3, hc = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const int rc = row / kTaps;
        const long long o = (long long)(dd * C + c_first + rc) * kTaps + (row - rc * kTaps);
        float* wsrow = P.ws + ((long long)split * O + o) * (C + 1);
        uint32_t v[40];
        if (n_my > 0) {
            if (ok && mbar_wait(&acc_done, 0, P.err, abort_v)) {
                tc_fence_after();
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + hc * 40;
                DDPM_TMEM_LD_X16(ta, (v + 0));
                DDPM_TMEM_LD_X16(ta + 16, (v + 16));
                DDPM_TMEM_LD_X8(ta + 32, (v + 32));
                tmem_ld_wait();
            } else {
                ok = false;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 40; ++j) v[j] = 0u;
        }
        if (ok && row < nrows) {
#pragma unroll
            for (int jj = 0; jj < 40; ++jj) {
                const int j = hc * 40 + jj;
                if (j < C) wsrow[j] = __uint_as_float(v[jj]);
                else if (j == 64) wsrow[C] = __uint_as_float(v[jj]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// 4-D FP32 tensor map over an NCHW tensor with `ch` channels: dims (W, H, ch, B).
bool encode_nchw_f32(CUtensorMap* m, const void* base, const Dims& d, int ch, uint32_t bw, uint32_t bh, uint32_t bc,
                     CUtensorMapSwizzle swz) {
    const cuuint64_t dims[4] = {(cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)ch, (cuuint64_t)d.B};
    const cuuint64_t str[3] = {(cuuint64_t)d.W * 4, (cuuint64_t)d.HW * 4, (cuuint64_t)d.HW * ch * 4};
    const cuuint32_t box[4] = {bw, bh, bc, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, str, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int K>
cudaError_t launch_k(const Dims& d, const void* g, const void* x, const void* y, float* ws, int S, cudaStream_t s) {
    using G = Tf32Geom<K>;
    using L = Tf32Layout<K>;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dw_tf32_kernel<K>, L::kSmemBytes, attr_done);
        if (e != cudaSuccess) return e;
    }
    DwTf32Params P;
    P.d = d;
    P.tiles_w = (d.W + kTW32 - 1) / kTW32;
    P.tiles_per_img = d.H * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.n_cblk = (d.C + G::CB - 1) / G::CB;
    P.n_oblk = 3 * P.n_cblk;
    P.tiles_per_split = (P.n_tiles + S - 1) / S;
    P.R = d.R();
    P.WHx = 1 + 2 * P.R;
    P.xslot = P.WHx * G::WIN * 4;
    P.xg_stage = (L::kGStage + G::CB * P.xslot + 127) / 128 * 128;
    P.ws = ws;
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    CUtensorMap tmY, tmG, tmX;
    if (!encode_nchw_f32(&tmY, y, d, d.C, 32, 1, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_nchw_f32(&tmG, g, d, 4 * d.C, kTW32, 1, G::CB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_nchw_f32(&tmX, x, d, d.C, G::WIN, (uint32_t)P.WHx, G::CB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    trace_begin(s, kKBwdDwTf32);
    bwd_dw_tf32_kernel<K><<<P.n_oblk * S, kThreads, L::kSmemBytes, s>>>(tmY, tmG, tmX, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace

// FP32 problems that asked for TF32 backward contractions, K = 3 (halo radius <= 6) or
// 5 (halo radius <= 10), C <= 64, W a multiple of 4 (16-byte TMA strides), 16-byte
// aligned tensors.
bool bwd_dw_tf32_eligible(const Dims& d, const void* g, const void* x, const void* y) {
    if (d.dtype != 0 || !(d.flags & kFlagTf32Backward) || (d.flags & kFlagCudaCores)) return false;
    if (!(d.K == 3 || d.K == 5)) return false;
    if (d.C > 64 || d.W % 4 != 0 || d.R() > (d.K == 3 ? Tf32Geom<3>::MAXR : Tf32Geom<5>::MAXR)) return false;
    if (d.O > (1LL << 30) || d.HW > (1LL << 31) - 1024) return false;
    if ((uintptr_t)g % 16 || (uintptr_t)x % 16 || (uintptr_t)y % 16) return false;
    return encode_fn() != nullptr;
}

int bwd_dw_tf32_splits(const Dims& d, size_t workspace_bytes) {
    const int cb = d.K == 3 ? Tf32Geom<3>::CB : Tf32Geom<5>::CB;
    const int n_oblk = 3 * ((d.C + cb - 1) / cb);
    const long long n_tiles = (long long)d.B * d.H * ((d.W + kTW32 - 1) / kTW32);
    int S = num_sms() / n_oblk;
    if (S < 1) S = 1;
    if (S > 16) S = 16;
    if (S > n_tiles) S = (int)n_tiles;
    const long long cap = (long long)(workspace_bytes / (sizeof(float) * (size_t)d.O * (size_t)(d.C + 1)));
    if (S > cap) S = (int)cap;
    return S < 1 ? 1 : S;
}

cudaError_t launch_bwd_dw_tf32(const Dims& d, const void* g, const void* x, const void* y, float* ws, int S,
                               cudaStream_t s) {
    return d.K == 3 ? launch_k<3>(d, g, x, y, ws, S, s) : launch_k<5>(d, g, x, y, ws, S, s);
}

}  // namespace ddpm
