// forward_tf32.cu -- FP32 fused generator + filter with the generator GEMM on tcgen05 tensor
// cores in three TF32 products (opt-in: DDPM_FLAG_TF32X3_FORWARD).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA 融合生成器推理": y tile ->
// dot(weight, y) -> dynamic taps -> consume with shifted x -> output, the taps living only
// on chip.  Section "已验证但未采用的方案" lists tf32x3 for the FP32 forward as tried on
// the page's card and not adopted there; GB300's TF32 rate (about 12x its FP32 FMA rate)
// is the reason to offer it here.  The filter itself stays IEEE FP32 FMA.
//
// Each FP32 operand a is split as hi = tf32(a) (round to nearest) and lo = a - hi (exact),
// and the GEMM is accumulated in FP32 as hi_y*hi_W + hi_y*lo_W + lo_y*hi_W: the neglected
// lo*lo term and the TF32 reading of lo leave a relative error of about 2^-21 per product.
// The epilogue adds the bias to each tap in FP32.
//
// GB300 design (the FP32 counterpart of forward_tc.cu).  A persistent CTA (one per SM)
// owns CG output channels (K = 3: CG = 4, 36 taps per dilation in 48 rows; K = 5: CG = 2,
// 50 taps in 56 rows) and walks 128-pixel tiles (2 rows x 64 columns, or whole rows when
// W < 64).  TMEM lane = pixel, so each epilogue thread owns every tap of its pixel.
//   warp 0      TMA: the group's W rows (once, 128B-swizzled K-major) and each tile's raw
//               y [64 j][128 px], one K-atom of 32 input channels at a time
//   warp 1      TMEM owner + MMA issuer: per tile 8 K-steps x 3 products, kind::tf32,
//               M = 128, N = the three dilations' rows side by side (144 for K = 3, 176
//               for K = 5), into one of two TMEM accumulators; the y operand is released
//               one K-atom (32 input channels) at a time
//   warp 2      TMA: the x window of each tile, one box per channel (2 buffers)
//   warps 3-6   splitters: W hi/lo once; per tile y hi/lo, transposed into
//               128B-swizzled K-major tiles (the MMA reads both operands K-major)
//   warps 7-14  epilogue: each thread owns one pixel and CG/2 channels; it reads their
//               taps of the three dilations from TMEM, adds the bias and, per dilation,
//               accumulates tap * x in IEEE FP32 FMA,
//               x read from the window at the tap's offset; each tile's four output
//               blocks are staged (two staging buffers) and leave by TMA store after one
//               epilogue-wide barrier
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

constexpr int kTile = 128;               // pixels per tile (MMA M)
constexpr int kKPad = 64;                // generator K (channels of y), zero padded
constexpr int kSplit0 = 3, kSplitWarps = 4;
constexpr int kEpi0 = kSplit0 + kSplitWarps, kEpiWarps = 8;
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kTmemCols = 512;           // two accumulators of NALL columns
constexpr int kRawBufs = 2;

// Per-kernel-size configuration: CG output channels per CTA group; ND rows of W per
// dilation (CG*K*K taps padded to a multiple of 8, so each dilation's rows start on a
// swizzle atom); NALL = the MMA N (3 * ND, padded to a multiple of 16); HALO x-window
// columns left and right of the tile (a 16-byte TMA coordinate, >= the halo radius);
// WINMAX x-window positions (TH + 2R) x (TW + 2 HALO).
template <int K> struct Tf32Cfg;
template <> struct Tf32Cfg<3> { static constexpr int CG = 4, ND = 48, NALL = 144, HALO = 8, WINMAX = 960; };
template <> struct Tf32Cfg<5> { static constexpr int CG = 2, ND = 56, NALL = 176, HALO = 12, WINMAX = 1936; };

template <int K>
struct Tf32Layout {
    using F = Tf32Cfg<K>;
    static constexpr int kCG = F::CG, kTaps = K * K, kN = F::ND, kNAll = F::NALL, kHalo = F::HALO;
    static constexpr int kWinMax = F::WINMAX;
    static constexpr int kCPT = kCG / (kEpiWarps / 4);   // channels per epilogue thread
    // shared memory (bytes from a 1024-aligned base)
    static constexpr int kWAtom = kNAll * 128;                  // one K-atom (32 fp32 of K) of NALL rows, SW128
    static constexpr int kSW = 0;                               // W hi [2 K-atoms][dilation][ND rows x 128 B]
    static constexpr int kSWlo = kSW + 2 * kWAtom;              // W lo, same layout
    static constexpr int kSYr = kSWlo + 2 * kWAtom;             // raw y [2 K-atoms][2 pixel halves][32 j][64 px] fp32
    static constexpr int kSYhi = kSYr + 2 * 64 * 64 * 4;        // y hi [2 K-atoms][128 rows x 128 B], SW128 K-major
    static constexpr int kSYlo = kSYhi + 2 * kTile * 128;       // y lo, same layout
    static constexpr int kSBias = kSYlo + 2 * kTile * 128;      // bias of the group's taps [3][CG*K*K] fp32
    static constexpr int kSX = kSBias + (3 * kCG * kTaps * 4 + 127) / 128 * 128;   // x windows 2 x [CG][kWinMax] fp32
    static constexpr int kSlot = (kWinMax * 4 + 127) / 128 * 128;
    static constexpr int kRawBuf = kCG * kSlot;
    static constexpr int kSStage = kSX + kRawBufs * kRawBuf;    // output staging 2 x 4 blocks x [CG][TH][TW] fp32
    static constexpr int kStageBlk = kCG * kTile * 4;
    static constexpr int kStageBuf = 4 * kStageBlk;
    static constexpr int kSmemBytes = kSStage + 2 * kStageBuf + 1024;
    static_assert(kWAtom % 1024 == 0 && kSWlo % 1024 == 0 && kSYhi % 1024 == 0 && kSYlo % 1024 == 0 &&
                      (kN * 128) % 1024 == 0, "SW128 atoms need 1 KiB alignment");
    static_assert(kSX % 128 == 0 && kSlot % 128 == 0 && kSStage % 128 == 0, "TMA alignment");
    static_assert(2 * kNAll <= kTmemCols && kCG * kTaps <= kN && 3 * kN <= kNAll && kNAll % 16 == 0 && kNAll <= 256,
                  "MMA N, TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024 - 512, "shared memory");
};

struct Tf32Params {
    Dims d;
    int TH, TW, tiles_per_row, tiles_per_img, n_tiles, n_groups, ctas_per_group;
    int R, WH, WC;
    const float* bias;     // may be null
    unsigned int* err;
};

struct TileCoord {
    int b, h0, w0;
};

__device__ __forceinline__ TileCoord tile_coord(const Tf32Params& P, int t) {
    TileCoord c;
    c.b = t / P.tiles_per_img;
    const int ti = t % P.tiles_per_img;
    c.h0 = (ti / P.tiles_per_row) * P.TH;
    c.w0 = (ti % P.tiles_per_row) * P.TW;
    return c;
}

// tf32 (nearest, ties away from zero) of an fp32 value, as fp32 with the low 13 bits clear
__device__ __forceinline__ float tf32_hi(float a) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(a));
    return __uint_as_float(r);
}

template <int NTHREADS>
__device__ __forceinline__ void named_bar(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(NTHREADS) : "memory");
}

template <int K>
__global__ void __launch_bounds__(kThreads, 1)
    forward_tf32_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO,
                        const Tf32Params P) {
    using namespace tc;
    using L = Tf32Layout<K>;
    constexpr int kCG = L::kCG, kTaps = L::kTaps, kN = L::kN, kNAll = L::kNAll, kHalo = L::kHalo, kCPT = L::kCPT;
    constexpr int kWAtom = L::kWAtom, kSW = L::kSW, kSWlo = L::kSWlo, kSYr = L::kSYr, kSYhi = L::kSYhi,
                  kSYlo = L::kSYlo, kSBias = L::kSBias, kSX = L::kSX, kSlot = L::kSlot, kRawBuf = L::kRawBuf,
                  kSStage = L::kSStage, kStageBlk = L::kStageBlk, kStageBuf = L::kStageBuf;
    constexpr int r0 = K / 2;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base by pointer arithmetic on the shared array (accesses stay shared-space)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_w, bar_wsplit, bar_yraw_full[2], bar_yraw_empty[2], bar_ysplit_full[2], bar_ysplit_empty[2],
        bar_acc_full[2], bar_acc_empty[2], bar_raw_full[kRawBufs], bar_raw_empty[kRawBufs], bar_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = blockIdx.x % P.n_groups;
    const int cta_in_group = blockIdx.x / P.n_groups;
    const int c0 = group * kCG;
    const int C = P.d.C;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar_w, 1);
        mbar_init(&bar_wsplit, kSplitWarps);
        for (int kh = 0; kh < 2; ++kh) {
            mbar_init(&bar_yraw_full[kh], 1);
            mbar_init(&bar_yraw_empty[kh], kSplitWarps);
            mbar_init(&bar_ysplit_full[kh], kSplitWarps);
            mbar_init(&bar_ysplit_empty[kh], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bar_acc_full[b], 1);
            mbar_init(&bar_acc_empty[b], kEpiWarps);
        }
        for (int s = 0; s < kRawBufs; ++s) {
            mbar_init(&bar_raw_full[s], 1);
            mbar_init(&bar_raw_empty[s], kEpiWarps);
        }
        mbar_init(&bar_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
    if (warp >= kEpi0) {
        // the bias of the group's taps, [dilation][local channel * K*K + k], added by the epilogue
        const int et = threadIdx.x - 32 * kEpi0;
        float* bt = reinterpret_cast<float*>(sm + kSBias);
        for (int i = et; i < 3 * kCG * kTaps; i += 32 * kEpiWarps) {
            const int dd = i / (kCG * kTaps), n = i % (kCG * kTaps);
            const long long o = (long long)(dd * C + c0) * kTaps + n;
            bt[i] = (P.bias != nullptr && o < P.d.O) ? P.bias[o] : 0.0f;
        }
        // rows 3*ND .. NALL-1 of the W operand (no TMA box writes them) are zero
        constexpr int kPadF = (kNAll - 3 * kN) * 32;   // floats per K-atom
        if constexpr (kPadF > 0) {
            for (int i = et; i < 2 * kPadF; i += 32 * kEpiWarps) {
                const int kh = i / kPadF, e = i % kPadF;
                reinterpret_cast<float*>(sm + kSW + kh * kWAtom + 3 * kN * 128)[e] = 0.0f;
            }
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int n_my = cta_in_group < P.n_tiles ? (P.n_tiles - 1 - cta_in_group) / P.ctas_per_group + 1 : 0;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer: W, raw y
        if (lane == 0) {
            prefetch_tmap(&tmY);
            prefetch_tmap(&tmW);
            mbar_arrive_expect_tx(&bar_w, 2 * 3 * kN * 128);
            for (int dd = 0; dd < 3; ++dd)
                for (int kh = 0; kh < 2; ++kh)
                    tma_load_2d(sm + kSW + kh * kWAtom + dd * kN * 128, &tmW, &bar_w, kh * 32, (dd * C + c0) * kTaps);
            // raw y arrives one K-atom (32 input channels) at a time, so the next tile's first
            // atom is on its way while the splitters still work on this tile's second
            const int half_step = P.TW == 64 ? P.d.W : 64;
            int issued = 0;
            bool ok = true;
            for (int i = 0; i < n_my && ok; ++i) {
                const TileCoord tcd = tile_coord(P, cta_in_group + i * P.ctas_per_group);
                const int pb = tcd.h0 * P.d.W + tcd.w0;
                for (int kh = 0; kh < 2; ++kh) {
                    if (!mbar_wait(&bar_yraw_empty[kh], (i & 1) ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = sm + kSYr + kh * 2 * 32 * 64 * 4;
                    mbar_arrive_expect_tx(&bar_yraw_full[kh], 2 * 32 * 64 * 4);
                    tma_load_3d(dst, &tmY, &bar_yraw_full[kh], pb, 32 * kh, tcd.b);
                    tma_load_3d(dst + 32 * 64 * 4, &tmY, &bar_yraw_full[kh], pb + half_step, 32 * kh, tcd.b);
                    issued = 2 * i + kh + 1;
                }
            }
            // drain: every copy this thread started lands before shared memory is released
            int never = 0;
            mbar_wait(&bar_w, 0, P.err, &never);
            for (int n = issued > 2 ? issued - 2 : 0; n < issued; ++n)
                mbar_wait(&bar_yraw_full[n & 1], (n >> 1) & 1, P.err, &never);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------- TMA producer: x windows
        if (lane == 0) {
            prefetch_tmap(&tmX);
            const int nch = min(kCG, C - c0);
            const uint32_t raw_bytes = (uint32_t)(nch * P.WH * P.WC * 4);
            int issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % kRawBufs, ph = (i / kRawBufs) & 1;
                const TileCoord tcd = tile_coord(P, cta_in_group + i * P.ctas_per_group);
                if (!mbar_wait(&bar_raw_empty[s], ph ^ 1, P.err, abort_v)) break;
                mbar_arrive_expect_tx(&bar_raw_full[s], raw_bytes);
                uint8_t* rb = sm + kSX + s * kRawBuf;
                for (int c = 0; c < nch; ++c)
                    tma_load_4d(rb + c * kSlot, &tmX, &bar_raw_full[s], tcd.w0 - kHalo, tcd.h0 - P.R, c0 + c, tcd.b);
                issued = i + 1;
            }
            int never = 0;
            for (int i = issued > kRawBufs ? issued - kRawBufs : 0; i < issued; ++i)
                mbar_wait(&bar_raw_full[i % kRawBufs], (i / kRawBufs) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(&bar_wsplit, 0, P.err, abort_v);
            const uint32_t idesc = instr_desc(2, 0, 0, kTile, kNAll);   // TF32, both operands K-major
            const uint64_t yhi = smem_desc(smem_u32(sm + kSYhi), 16, 1024, kSwizzle128B);
            const uint64_t ylo = smem_desc(smem_u32(sm + kSYlo), 16, 1024, kSwizzle128B);
            const uint64_t whi = smem_desc(smem_u32(sm + kSW), 16, 1024, kSwizzle128B);
            const uint64_t wlo = smem_desc(smem_u32(sm + kSWlo), 16, 1024, kSwizzle128B);
            for (int i = 0; ok && i < n_my; ++i) {
                const int tb = i & 1;                  // TMEM accumulator of this tile
                if (!mbar_wait(&bar_acc_empty[tb], ((i >> 1) & 1) ^ 1, P.err, abort_v)) break;
                tc_fence_after();
                const uint32_t dt = tmem + tb * kNAll;
                // K-atom by K-atom, so that the splitters refill the first atom for the next
                // tile while the MMAs read the second
                for (int kh = 0; kh < 2 && ok; ++kh) {
                    if (!mbar_wait(&bar_ysplit_full[kh], i & 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t ya = (uint32_t)(kh * kTile * 128 + kk * 32);
                        const uint32_t wa = (uint32_t)(kh * kWAtom + kk * 32);
                        mma_tf32(dt, desc_advance(yhi, ya), desc_advance(whi, wa), idesc, (kh | kk) ? 1u : 0u);
                        mma_tf32(dt, desc_advance(yhi, ya), desc_advance(wlo, wa), idesc, 1u);
                        mma_tf32(dt, desc_advance(ylo, ya), desc_advance(whi, wa), idesc, 1u);
                    }
                    mma_commit(&bar_ysplit_empty[kh]);
                }
                if (!ok) break;
                mma_commit(&bar_acc_full[tb]);
            }
            // all issued MMAs retire before TMEM is released
            mma_commit(&bar_done);
            int never = 0;
            mbar_wait(&bar_done, 0, P.err, &never);
        }
    } else if (warp < kEpi0) {
        // ------------------------------------------------------- splitters
        const int st = threadIdx.x - 32 * kSplit0, nst = 32 * kSplitWarps;
        bool ok = mbar_wait(&bar_w, 0, P.err, abort_v);
        if (ok) {
            // W hi in place, W lo beside it (same swizzled offsets: the split is elementwise)
            for (int i = st; i < 2 * kWAtom / 16; i += nst) {
                float4* ph = reinterpret_cast<float4*>(sm + kSW) + i;
                float4* pl = reinterpret_cast<float4*>(sm + kSWlo) + i;
                const float4 v = *ph;
                float4 h, l;
                h.x = tf32_hi(v.x); l.x = v.x - h.x;
                h.y = tf32_hi(v.y); l.y = v.y - h.y;
                h.z = tf32_hi(v.z); l.z = v.z - h.z;
                h.w = tf32_hi(v.w); l.w = v.w - h.w;
                *ph = h;
                *pl = l;
            }
            fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_wsplit);
        for (int i = 0; ok && i < n_my; ++i) {
            // unit = (pixel px, group of 4 input channels jc): a warp covers 32 consecutive
            // pixels of one jc, so its raw reads are 128 contiguous bytes per channel and its
            // 16-byte stores touch each bank once per 8 rows.  K-atom kh holds jc 8kh .. 8kh+7.
            for (int kh = 0; kh < 2 && ok; ++kh) {
                if (!mbar_wait(&bar_yraw_full[kh], i & 1, P.err, abort_v) ||
                    !mbar_wait(&bar_ysplit_empty[kh], (i & 1) ^ 1, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                for (int u = st; u < kTile * 8; u += nst) {
                    const int px = u % kTile, jc = kh * 8 + u / kTile;
                    // raw atom kh: [pixel half][32 j][64 px]; local channel jl = 4 * (jc % 8)
                    const float* raw = reinterpret_cast<const float*>(sm + kSYr + kh * 2 * 32 * 64 * 4 +
                                                                      (px / 64) * 32 * 64 * 4) + (px % 64);
                    const int jl = 4 * (jc % 8);
                    float4 h, l;
                    const float y0 = raw[(jl + 0) * 64], y1 = raw[(jl + 1) * 64];
                    const float y2 = raw[(jl + 2) * 64], y3 = raw[(jl + 3) * 64];
                    h.x = tf32_hi(y0); l.x = y0 - h.x;
                    h.y = tf32_hi(y1); l.y = y1 - h.y;
                    h.z = tf32_hi(y2); l.z = y2 - h.z;
                    h.w = tf32_hi(y3); l.w = y3 - h.w;
                    const int off = kh * kTile * 128 + (px / 8) * 1024 + (px % 8) * 128 + (((jc % 8) ^ (px % 8)) << 4);
                    *reinterpret_cast<float4*>(sm + kSYhi + off) = h;
                    *reinterpret_cast<float4*>(sm + kSYlo + off) = l;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar_ysplit_full[kh]);
                    mbar_arrive(&bar_yraw_empty[kh]);
                }
            }
        }
    } else {
        // ------------------------------------------------------- epilogue
        const int ew = warp - kEpi0;
        const int q = warp & 3;                  // TMEM lane quadrant this warp may access
        const int cl0 = (ew >> 2) * kCPT;        // first local channel of this thread
        const int s = q * 32 + lane;             // pixel slot == TMEM lane
        const bool leader = ew == 0 && lane == 0;
        const int tpix = P.TH * P.TW;
        const bool in_tile = s < tpix;
        const int rr = in_tile ? s / P.TW : 0, cc = in_tile ? s % P.TW : 0;
        const int WC = P.WC;
        const int center = (rr + P.R) * WC + cc + kHalo;
        // this thread's element of staging buffer 0, block 0 (buffer sb at + sb * kStageBuf)
        const int st_off = cl0 * tpix + (in_tile ? s : 0);
        int buf = 0, bph = 0;
        bool ok = true;
        for (int i = 0; i < n_my; ++i) {
            const TileCoord tcd = tile_coord(P, cta_in_group + i * P.ctas_per_group);
            const int sb = i & 1;                // staging buffer: the stores of tile i - 1 may still read the other
            float* stage0 = reinterpret_cast<float*>(sm + kSStage + sb * kStageBuf) + st_off;
            const float* xw = reinterpret_cast<const float*>(sm + kSX + buf * kRawBuf + cl0 * kSlot) + center;
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar_raw_full[buf], bph, P.err, abort_v));
            // all three dilations' taps of this thread, then the accumulator goes back to the MMA
            const int tb = i & 1;
            uint32_t t[3][kCPT * kTaps];
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc_full[tb], (i >> 1) & 1, P.err, abort_v));
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int dd = 0; dd < 3; ++dd)
                    tmem_load_cols<kCPT * kTaps>(tmem + ((uint32_t)(q * 32) << 16) + tb * kNAll + dd * kN + cl0 * kTaps,
                                                 t[dd]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_acc_empty[tb]);
            }
            if (ok && in_tile) {
                // block 0: channels c0 .. c0+CG-1 of the output are x itself
#pragma unroll
                for (int c = 0; c < kCPT; ++c) stage0[c * tpix] = xw[c * (kSlot / 4)];
                const float* bt = reinterpret_cast<const float*>(sm + kSBias) + cl0 * kTaps;
#pragma unroll
                for (int dd = 0; dd < 3; ++dd) {
                    const int dil = dil_of(P.d, dd);
                    float acc[kCPT];
#pragma unroll
                    for (int c = 0; c < kCPT; ++c) acc[c] = 0.0f;
#pragma unroll
                    for (int k = 0; k < kTaps; ++k) {
                        const int off = ((k / K - r0) * WC + (k % K - r0)) * dil;
#pragma unroll
                        for (int c = 0; c < kCPT; ++c) {
                            const float tap = __uint_as_float(t[dd][c * kTaps + k]) + bt[dd * kCG * kTaps + c * kTaps + k];
                            acc[c] = fmaf(tap, xw[c * (kSlot / 4) + off], acc[c]);
                        }
                    }
                    float* sa = stage0 + (1 + dd) * (kStageBlk / 4);
#pragma unroll
                    for (int c = 0; c < kCPT; ++c) sa[c * tpix] = acc[c];
                }
            }
            // the window has been read for the last time
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_raw_empty[buf]);
            // one hand-off per tile: the leader first makes sure the stores of tile i - 1 have
            // read their staging buffer (the one tile i + 1 writes next), then every epilogue
            // thread's values are in place and the four blocks leave by TMA
            fence_proxy_async_smem();
            if (leader) bulk_wait_read<0>();
            named_bar<32 * kEpiWarps>(1);
            if (leader && ok) {
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    const int cbase = (blk == 0 ? 0 : blk * C) + c0;
                    tma_store_4d(&tmO, sm + kSStage + sb * kStageBuf + blk * kStageBlk, tcd.w0, tcd.h0, cbase, tcd.b);
                }
                bulk_commit();
            }
            if (++buf == kRawBufs) {
                buf = 0;
                bph ^= 1;
            }
        }
        if (leader) bulk_wait<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// fp32 NCHW tensor map, dims (W, H, ch, B)
bool encode_nchw_f32(CUtensorMap* m, const void* base, const Dims& d, int ch, uint32_t bw, uint32_t bh, uint32_t bc) {
    const cuuint64_t dims[4] = {(cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)ch, (cuuint64_t)d.B};
    const cuuint64_t str[3] = {(cuuint64_t)d.W * 4, (cuuint64_t)d.HW * 4, (cuuint64_t)d.HW * ch * 4};
    const cuuint32_t box[4] = {bw, bh, bc, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return bwdtc::encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, str, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Tiling {
    int TH, TW, tiles_per_row, tiles_per_img;
};

Tiling tiling_of(const Dims& d) {
    Tiling t;
    if (d.W >= 64) {
        t.TW = 64;
        t.TH = 2;
        t.tiles_per_row = (d.W + 63) / 64;
    } else {
        t.TW = d.W;
        t.TH = kTile / d.W < d.H ? kTile / d.W : d.H;
        t.tiles_per_row = 1;
    }
    t.tiles_per_img = ((d.H + t.TH - 1) / t.TH) * t.tiles_per_row;
    return t;
}

template <int K>
bool eligible_k(const Dims& d) {
    using L = Tf32Layout<K>;
    // 16-byte TMA strides (W rows: C % 4; images: W % 4) and whole channel groups
    if (d.C % 4 != 0 || d.C % L::kCG != 0 || d.C > kKPad || d.W % 4 != 0) return false;
    if (d.R() > L::kHalo) return false;
    const Tiling t = tiling_of(d);
    return (long long)(t.TH + 2 * d.R()) * (t.TW + 2 * L::kHalo) <= L::kWinMax;
}

template <int K>
cudaError_t launch_k(const Dims& d, const void* x, const void* y, const void* w, const void* bias, void* out,
                     cudaStream_t s) {
    using L = Tf32Layout<K>;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)forward_tf32_kernel<K>, L::kSmemBytes, attr_done, true);
        if (e != cudaSuccess) return e;
    }
    auto enc = bwdtc::encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const Tiling t = tiling_of(d);
    const int R = d.R();
    CUtensorMap tmY, tmW, tmX, tmO;
    const cuuint64_t dimY[3] = {(cuuint64_t)d.HW, (cuuint64_t)d.C, (cuuint64_t)d.B};
    const cuuint64_t strY[2] = {(cuuint64_t)d.HW * 4, (cuuint64_t)d.HW * d.C * 4};
    const cuuint32_t boxY[3] = {64, 32, 1};   // 64 pixels x one K-atom of input channels
    const cuuint32_t one3[3] = {1, 1, 1};
    if (enc(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(y), dimY, strY, boxY, one3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // W [O, C] fp32: boxes of 32 input channels (one 128-byte swizzle row) x ND rows
    const cuuint64_t dimW[2] = {(cuuint64_t)d.C, (cuuint64_t)d.O};
    const cuuint64_t strW[1] = {(cuuint64_t)d.C * 4};
    const cuuint32_t boxW[2] = {32, (cuuint32_t)L::kN};   // one dilation's rows of one K-atom
    const cuuint32_t one2[2] = {1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(w), dimW, strW, boxW, one2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int WH = t.TH + 2 * R, WC = t.TW + 2 * L::kHalo;
    if (!encode_nchw_f32(&tmX, x, d, d.C, (uint32_t)WC, (uint32_t)WH, 1) ||
        !encode_nchw_f32(&tmO, out, d, 4 * d.C, (uint32_t)t.TW, (uint32_t)t.TH, (uint32_t)L::kCG))
        return cudaErrorInvalidValue;

    Tf32Params P;
    P.d = d;
    P.TH = t.TH;
    P.TW = t.TW;
    P.tiles_per_row = t.tiles_per_row;
    P.tiles_per_img = t.tiles_per_img;
    P.n_tiles = d.B * t.tiles_per_img;
    P.n_groups = d.C / L::kCG;
    int cpg = num_sms() / P.n_groups;
    if (cpg < 1) cpg = 1;
    if (cpg > P.n_tiles) cpg = P.n_tiles;
    P.ctas_per_group = cpg;
    P.R = R;
    P.WH = WH;
    P.WC = WC;
    P.bias = static_cast<const float*>(bias);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    trace_begin(s, kKForwardTf32);
    forward_tf32_kernel<K><<<P.n_groups * cpg, kThreads, L::kSmemBytes, s>>>(tmY, tmW, tmX, tmO, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace

bool forward_tf32_eligible(const Dims& d, const void* x, const void* y, const void* w, const void* out) {
    if (d.dtype != 0 || !(d.flags & kFlagTf32x3Forward) || (d.flags & kFlagCudaCores)) return false;
    if (!(d.K == 3 ? eligible_k<3>(d) : d.K == 5 ? eligible_k<5>(d) : false)) return false;
    if ((uintptr_t)x % 16 || (uintptr_t)y % 16 || (uintptr_t)w % 16 || (uintptr_t)out % 16) return false;
    const long long tiles = (long long)d.B * tiling_of(d).tiles_per_img;
    return tiles <= (1LL << 30) && d.O <= (1LL << 30) && d.HW <= (1LL << 31) - 1024 && bwdtc::encode_fn() != nullptr;
}

cudaError_t launch_forward_tf32(const Dims& d, const void* x, const void* y, const void* w, const void* bias,
                                void* out, cudaStream_t s) {
    return d.K == 3 ? launch_k<3>(d, x, y, w, bias, out, s) : launch_k<5>(d, x, y, w, bias, out, s);
}

}  // namespace ddpm
