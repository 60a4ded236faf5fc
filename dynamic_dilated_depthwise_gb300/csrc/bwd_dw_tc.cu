// bwd_dw_tc.cu -- dW / dbias split partials on tcgen05 tensor cores (bf16).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dWeight/dbias form dK = shifted(x) * grad on chip and reduce it over space;
// the tokens are split into at most 16 FP32 partials that a second short
// kernel sums (dw_reduce_kernel in backward_simt.cu, fixed order).
//
//   ws[s][o][j] = sum_{pixels p of split s} dK[o, p] * y[j, p]     (j < C)
//   ws[s][o][C] = sum_p dK[o, p]                                    (dbias)
//
// GB300 design.  A CTA owns a block of taps -- 14 channels of one dilation,
// 126 taps, for K = 3, or 5 channels, 125 taps, for K = 5, padded to the MMA M
// of 128 -- and one pixel split.  Per 2x64
// pixel tile:
//   - one producer warp's TMA brings y [64 j x 128 px] (one 128-byte row per
//     channel and tile row, 128B-swizzled: a K-major operand) into a 3-stage
//     ring that the MMA releases;
//   - another brings the block's grad planes [CB x 128 px] and the matching
//     x windows [CB x (2+2R) x (64 + 2 halo) px], zero-filled outside the image, into a
//     ring of 2-4 stages (as many as shared memory holds for the halo) that
//     the formers release as soon as dK is formed;
//   - two groups of eight warps form dK^T[o, px] (bwdtc::form_dk_tile) into a
//     128B-swizzled K-major operand, even tiles in one group and buffer, odd
//     tiles in the other: one group's formation of a tile is a short chain of
//     shared-memory loads and stores per thread, so two tiles in flight keep the
//     formers' loads overlapped;
//   - one thread issues D[o, n] += dK^T[o, px] * Y[n, px] with N = 80 rows: the
//     64 y channels plus a constant ones row (row 64) that yields dbias; the
//     descriptors are built once and each MMA adds 32-bit offsets to their low
//     halves.
// The accumulator stays in TMEM for the whole split and is written once.
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using namespace bwdtc;

constexpr int kNY = 80;           // MMA N: 64 y channels + ones row + 15 zero rows
constexpr int kGroupWarps = 8;                     // warps of one former group
constexpr int kFormWarps = 2 * kGroupWarps;        // two groups: even and odd tiles
constexpr int kThreads = 32 * (3 + kFormWarps);   // x/grad producer, MMA, formers, y producer
constexpr int kYWarp = 2 + kFormWarps;             // warp of the y producer
constexpr int kYStages = 3;
constexpr int kMaxXgStages = 4;
constexpr int kSmemCap = 232448 - 1024;            // dynamic shared memory: the opt-in 227 KiB less the static part

// shared memory (bytes from a 1024-aligned base): two dK^T tiles, the y ring, then the
// x/grad ring (its stage size depends on the halo radius)
constexpr int kDK = 0;                               // 2 x dK^T tiles
constexpr int kYS = kDK + 2 * kDKBytes;              // y ring: stages x 2 halves x [80 rows x 128 B]
constexpr int kYHalf = kNY * 128;                    // 10240
constexpr int kYStage = 2 * kYHalf;                  // 20480
constexpr int kXG = kYS + kYStages * kYStage;        // x/grad ring
template <int K>
__host__ __device__ constexpr int gstage_bytes() { return BwdGeom<K>::kCB * kPx * 2; }   // grad planes of the block [CB x 128 px] bf16
constexpr int kSlack = 1024 + 128;                   // alignment slack + over-read margin
static_assert(kYS % 1024 == 0 && kYStage % 1024 == 0 && kYHalf % 1024 == 0, "SW128 atoms need 1 KiB");
static_assert(kXG % 128 == 0 && gstage_bytes<3>() % 128 == 0 && gstage_bytes<5>() % 128 == 0, "TMA dst 128 B");

struct XgLayout {
    int stage_bytes;   // grad planes + x windows, rounded up to 128 B
    int stages;        // 0 when even two stages do not fit
};

// The x/grad stage holds the block's grad planes and its x windows [CB x (2+2R) x cols].
template <int K>
inline XgLayout xg_layout(int R) {
    using G = BwdGeom<K>;
    XgLayout L;
    const int xbytes = G::kCB * (kTH + 2 * R) * G::kWinCols * 2;
    L.stage_bytes = (gstage_bytes<K>() + xbytes + 127) / 128 * 128;
    int n = (kSmemCap - kSlack - kXG) / L.stage_bytes;
    L.stages = n > kMaxXgStages ? kMaxXgStages : (n < 2 ? 0 : n);
    return L;
}

struct DwTcParams {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int n_cblk;        // ceil(C / CB) blocks of channels per dilation
    int n_oblk;        // 3 * n_cblk
    int tiles_per_split;
    int R, WHx;        // halo radius, window rows (2 + 2R)
    int xslot_bytes;   // WHx * window columns * 2
    int xg_stage, xg_stages;
    float* ws;         // [S][O][C+1]
    unsigned int* err;
};

// Pipeline per pixel tile i:
//   x/grad producer --xg_full--> formers --dk_full--> MMA <--y_full-- y producer
// The formers release the x/grad stage (xg_empty) as soon as dK^T is formed, and the
// MMA releases the y stage and the dK^T buffer through commits, so the next windows
// load while the tensor cores still read the previous tile.
template <int K>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dw_tc_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmX, const DwTcParams P) {
    using namespace tc;
    using G = BwdGeom<K>;
    constexpr int kCB = G::kCB, kTaps = K * K, kGStage = gstage_bytes<K>();
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base, derived by pointer arithmetic on the shared array so that every
    // access through it stays a shared-memory access (an integer round trip would make
    // them generic loads and stores with 64-bit addresses)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    // xg_full has one barrier per stage and former group: a parity wait is only sound
    // for a waiter that has seen the barrier's previous phase, and the two groups take
    // turns on the shared stages
    __shared__ uint64_t y_full[kYStages], y_empty[kYStages], xg_full[2][kMaxXgStages], xg_empty[kMaxXgStages];
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
    const int NX = P.xg_stages;
    const int NL = (NX & 1) ? 2 * NX : NX;   // tiles between two uses of one (stage, group) barrier

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
        for (int s = 0; s < NX; ++s) {
            mbar_init(&xg_full[0][s], 1);
            mbar_init(&xg_full[1][s], 1);
            mbar_init(&xg_empty[s], kGroupWarps);   // the group that formed the tile
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
            const uint32_t v = row == 0 ? 0x3F803F80u : 0u;  // bf16 pair (1.0, 1.0)
            reinterpret_cast<uint32_t*>(sm + kYS + st * kYStage + half * kYHalf + (64 + row) * 128)[word] = v;
        }
        zero_dk_pad_rows<K>(sm + kDK, et, 32 * kFormWarps);
        zero_dk_pad_rows<K>(sm + kDK + kDKBytes, et, 32 * kFormWarps);
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
            const uint32_t bytes = kGStage + kCB * P.xslot_bytes;
            int issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % NX, ph = (i / NX) & 1;
                if (!mbar_wait(&xg_empty[s], ph ^ 1, P.err, abort_v)) break;
                const int t = t_begin + i;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kTH, w0 = (ti % P.tiles_w) * kTW;
                uint8_t* st = sm + kXG + s * P.xg_stage;
                uint64_t* full = &xg_full[i & 1][s];
                mbar_arrive_expect_tx(full, bytes);
                tma_load_4d(st, &tmG, full, w0, h0, (1 + dd) * C + c_first, b);
                tma_load_4d(st + kGStage, &tmX, full, w0 - G::kHaloCols, h0 - P.R, c_first, b);
                issued = i + 1;
            }
            // drain: every copy this thread started lands before its shared memory is released
            int never = 0;
            for (int i = issued > NX ? issued - NX : 0; i < issued; ++i)
                mbar_wait(&xg_full[i & 1][i % NX], (i / NL) & 1, P.err, &never);
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
                const int h0 = (ti / P.tiles_w) * kTH, w0 = (ti % P.tiles_w) * kTW;
                uint8_t* ys = sm + kYS + s * kYStage;
                mbar_arrive_expect_tx(&y_full[s], 2 * 8192);
                tma_load_4d(ys, &tmY, &y_full[s], w0, h0, 0, b);
                tma_load_4d(ys + kYHalf, &tmY, &y_full[s], w0, h0 + 1, 0, b);
                issued = i + 1;
            }
            int never = 0;
            for (int i = issued > kYStages ? issued - kYStages : 0; i < issued; ++i)
                mbar_wait(&y_full[i % kYStages], (i / kYStages) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(1, 0, 0, kBlockRows, kNY);   // both operands K-major
            // descriptors are built once; each MMA only moves a start address (desc_advance)
            const uint64_t dk_base = smem_desc(smem_u32(sm + kDK), 16, 1024, kSwizzle128B);
            const uint64_t y_base = smem_desc(smem_u32(sm + kYS), 16, 1024, kSwizzle128B);
            const uint32_t dk_hi = (uint32_t)(dk_base >> 32), y_hi = (uint32_t)(y_base >> 32);
            bool ok = true;
            int sy = 0, yph = 0;   // y ring stage and phase, stepped by a counter
            for (int i = 0; i < n_my && ok; ++i) {
                const int s = i & 1, ph = (i >> 1) & 1;
                if (!mbar_wait(&dk_full[s], ph, P.err, abort_v) || !mbar_wait(&y_full[sy], yph, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t da = (uint32_t)dk_base + (uint32_t)((s * kDKBytes) >> 4);
                const uint32_t ya = (uint32_t)y_base + (uint32_t)((sy * kYStage) >> 4);
#pragma unroll
                for (int half = 0; half < 2; ++half)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16_lh(tmem, da + (uint32_t)((half * 16384 + kk * 32) >> 4), dk_hi,
                                   ya + (uint32_t)((half * kYHalf + kk * 32) >> 4), y_hi, idesc,
                                   (i > 0 || half > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&dk_empty[s]);
                mma_commit(&y_empty[sy]);
                if (++sy == kYStages) {
                    sy = 0;
                    yph ^= 1;
                }
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
        const int slot_elems = P.xslot_bytes / 2;
        bool ok = true;
        for (int i = grp; i < n_my && ok; i += 2) {
            const int s = i & 1, ph = (i >> 1) & 1;
            const int sx = i % NX, xph = (i / NL) & 1;
            if (!mbar_wait(&xg_full[grp][sx], xph, P.err, abort_v) || !mbar_wait(&dk_empty[s], ph ^ 1, P.err, abort_v)) {
                ok = false;
                break;
            }
            const uint8_t* st = sm + kXG + sx * P.xg_stage;
            form_dk_tile<K>(sm + kDK + s * kDKBytes, reinterpret_cast<const uint32_t*>(st + kGStage),
                         reinterpret_cast<const bf16*>(st), kPx, nrows, slot_elems, P.R, dil, 0, et, 32 * kGroupWarps);
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

template <int K>
cudaError_t launch_k(const Dims& d, const void* g, const void* x, const void* y, float* ws, int S, cudaStream_t s) {
    using G = BwdGeom<K>;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dw_tc_kernel<K>, kSmemCap, attr_done);
        if (e != cudaSuccess) return e;
    }
    DwTcParams P;
    P.d = d;
    P.tiles_w = (d.W + kTW - 1) / kTW;
    P.tiles_per_img = ((d.H + kTH - 1) / kTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.n_cblk = (d.C + G::kCB - 1) / G::kCB;
    P.n_oblk = 3 * P.n_cblk;
    P.tiles_per_split = (P.n_tiles + S - 1) / S;
    P.R = d.R();
    P.WHx = kTH + 2 * P.R;
    P.xslot_bytes = P.WHx * G::kWinCols * 2;
    const XgLayout L = xg_layout<K>(P.R);
    if (L.stages < 2) return cudaErrorInvalidValue;
    P.xg_stage = L.stage_bytes;
    P.xg_stages = L.stages;
    const int smem_bytes = kXG + L.stages * L.stage_bytes + kSlack;
    P.ws = ws;
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    CUtensorMap tmY, tmG, tmX;
    if (!encode_nchw(&tmY, y, d, d.C, kTW, 1, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_nchw(&tmG, g, d, 4 * d.C, kTW, kTH, G::kCB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_nchw(&tmX, x, d, d.C, G::kWinCols, (uint32_t)P.WHx, G::kCB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    trace_begin(s, kKBwdDwTc);
    bwd_dw_tc_kernel<K><<<P.n_oblk * S, kThreads, smem_bytes, s>>>(tmY, tmG, tmX, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace

bool bwd_dw_tc_eligible(const Dims& d, const void* g, const void* x, const void* y) {
    if (!bwdtc::eligible(d, g, x, y, true)) return false;
    return (d.K == 3 ? xg_layout<3>(d.R()).stages : xg_layout<5>(d.R()).stages) >= 2;
}

int bwd_dw_tc_splits(const Dims& d, size_t workspace_bytes) {
    const int cb = d.K == 3 ? BwdGeom<3>::kCB : BwdGeom<5>::kCB;
    const int n_oblk = 3 * ((d.C + cb - 1) / cb);
    const long long n_tiles = (long long)d.B * ((d.H + kTH - 1) / kTH) * ((d.W + kTW - 1) / kTW);
    int S = num_sms() / n_oblk;
    if (S < 1) S = 1;
    if (S > 16) S = 16;
    if (S > n_tiles) S = (int)n_tiles;
    const long long cap = (long long)(workspace_bytes / (sizeof(float) * (size_t)d.O * (size_t)(d.C + 1)));
    if (S > cap) S = (int)cap;
    return S < 1 ? 1 : S;
}

cudaError_t launch_bwd_dw_tc(const Dims& d, const void* g, const void* x, const void* y, float* ws, int S,
                             cudaStream_t s) {
    return d.K == 3 ? launch_k<3>(d, g, x, y, ws, S, s) : launch_k<5>(d, g, x, y, ws, S, s);
}

}  // namespace ddpm
