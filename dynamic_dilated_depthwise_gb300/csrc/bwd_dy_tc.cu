// bwd_dy_tc.cu -- dY on tcgen05 tensor cores (bf16).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dY forms dK = shifted(x) * grad on chip and multiplies it by the generator
// weight straight away:
//   dy[b, j, p] = sum_o W[o, j] * dK[b, o, p].
//
// GB300 design.  Persistent CTAs walk super tiles of 8 rows x 64 columns (four
// 2x64 sub-tiles, 512 pixels).  For each super tile the CTA visits every block
// of taps (14 channels of one dilation, 126 taps, for K = 3; 5 channels, 125
// taps, for K = 5); per block one producer
// warp's TMA brings the block's W rows [128 o x 64 j] into a 3-stage ring that
// the MMA releases, and another brings its grad planes [CB x 512 px] and x
// windows [CB x (8+2R) x (64 + 2 halo)] into a 2-stage ring that the formers release once
// the four sub-tiles are formed; per block:
//   - two groups of eight warps form the sub-tiles' dK^T tiles
//     (bwdtc::form_dk_tile), alternate sub-tiles in alternate buffers, so that
//     two formations are in flight (each is a short chain of shared-memory
//     loads and stores per thread); with one sub-tile per block the groups
//     take alternate blocks, and each x/grad stage serves one group;
//   - one thread issues D_st[px, j] += dK[px, o] * W[o, j] (M = 128 pixels read
//     MN-major from the dK^T tile, N = 64, K = 128 taps in eight K=16 steps).
// Four accumulators [128 px x 64 j] fp32 per super tile, double-buffered, fill
// the 512 TMEM columns; four epilogue warps store super tile i while i+1 runs.
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using namespace bwdtc;

constexpr int kN = 64;            // MMA N: output channels j (zero padded beyond C)
// Sub-tiles of 2x64 per super tile: 4 (8 rows, 512 pixels), or 1 for images whose
// 8-row super tiles would leave most SMs idle (the W block is then read per 128
// pixels instead of per 512).
constexpr int kDyMaxR = 5;        // K = 3: halo radius the window buffers hold (10 for K = 5)
constexpr int kGroupWarps = 8;    // warps of one former group
constexpr int kFormWarps = 2 * kGroupWarps;
constexpr int kEpiWarps = 4;
constexpr int kWWarp = 2 + kFormWarps + kEpiWarps;   // warp of the W producer
constexpr int kThreads = 32 * (3 + kFormWarps + kEpiWarps);
constexpr int kWStages = 3, kXgStages = 2;

// shared memory (bytes from a 1024-aligned base)
constexpr int kDK = 0;                               // 2 x dK^T tiles
constexpr int kWS = kDK + 2 * kDKBytes;              // W ring: stages x W block [128 o x 128 B] SW128
constexpr int kWStage = kBlockRows * 128;            // 16384
constexpr int kXG = kWS + kWStages * kWStage;        // x/grad ring
static_assert(kWS % 1024 == 0 && kWStage % 1024 == 0, "SW128 atoms need 1 KiB");

// The x/grad stage of kernel size K: grad planes [CB x 512 px] and x windows
// [CB x (8 + 2 maxR) x cols], bf16.
template <int K, int SUB>
struct DyLayout {
    using G = BwdGeom<K>;
    static constexpr int kSTH = SUB * kTH, kSPx = SUB * kPx;
    static constexpr int kMaxR = K == 3 ? kDyMaxR : 10;
    static constexpr int kGStage = G::kCB * kSPx * 2;
    static constexpr int kXgStage = kGStage + G::kCB * (kSTH + 2 * kMaxR) * G::kWinCols * 2;
    static constexpr int kSmemBytes = kXG + kXgStages * kXgStage + 1024 + 128;   // + alignment slack + over-read margin
    static_assert(kXG % 128 == 0 && kGStage % 128 == 0 && kXgStage % 128 == 0, "TMA dst 128 B");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct DyTcParams {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;   // super tiles
    int n_cblk, n_oblk;
    int R, WHx, xslot_bytes;
    bf16* dy;
    unsigned int* err;
};

template <int K, int SUB>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dy_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmG,
                     const __grid_constant__ CUtensorMap tmX, const DyTcParams P) {
    using namespace tc;
    using G = BwdGeom<K>;
    using L = DyLayout<K, SUB>;
    constexpr int kCB = G::kCB, kTaps = K * K, kGStage = L::kGStage, kXgStage = L::kXgStage;
    constexpr int kSub = SUB, kSTH = L::kSTH, kSPx = L::kSPx;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base, derived by pointer arithmetic on the shared array so that every
    // access through it stays a shared-memory access (an integer round trip would make
    // them generic loads and stores with 64-bit addresses)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t w_full[kWStages], w_empty[kWStages], xg_full[kXgStages], xg_empty[kXgStages];
    __shared__ uint64_t dk_full[2], dk_empty[2], acc_full[2], acc_empty[2], mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.d.C;
    const int n_my = blockIdx.x < P.n_tiles ? (P.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int NB = P.n_oblk;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], 1);
        }
        for (int s = 0; s < kXgStages; ++s) {
            mbar_init(&xg_full[s], 1);
            mbar_init(&xg_empty[s], kSub > 1 ? kFormWarps : kGroupWarps);   // the groups that read the block
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&dk_full[s], kGroupWarps);
            mbar_init(&dk_empty[s], 1);
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kEpiWarps);
        }
        mbar_init(&mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    if (warp >= 2 && warp < 2 + kFormWarps) {
        zero_dk_pad_rows<K>(sm + kDK, threadIdx.x - 64, 32 * kFormWarps);
        zero_dk_pad_rows<K>(sm + kDK + kDKBytes, threadIdx.x - 64, 32 * kFormWarps);
        tc::fence_proxy_async_smem();
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
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                const int t = blockIdx.x + tl * gridDim.x;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kSTH, w0 = (ti % P.tiles_w) * kTW;
                for (int ob = 0; ob < NB; ++ob) {
                    const int i = tl * NB + ob, s = i % kXgStages, ph = (i / kXgStages) & 1;
                    if (!mbar_wait(&xg_empty[s], ph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    const int dd = ob / P.n_cblk, c_first = (ob % P.n_cblk) * kCB;
                    uint8_t* st = sm + kXG + s * kXgStage;
                    mbar_arrive_expect_tx(&xg_full[s], bytes);
                    tma_load_4d(st, &tmG, &xg_full[s], w0, h0, (1 + dd) * C + c_first, b);
                    tma_load_4d(st + kGStage, &tmX, &xg_full[s], w0 - G::kHaloCols, h0 - P.R, c_first, b);
                    issued = i + 1;
                }
            }
            // drain: every copy this thread started lands before its shared memory is released
            int never = 0;
            for (int i = issued > kXgStages ? issued - kXgStages : 0; i < issued; ++i)
                mbar_wait(&xg_full[i % kXgStages], (i / kXgStages) & 1, P.err, &never);
        }
    } else if (warp == kWWarp) {
        // ------------------------------------------------------- W producer
        if (lane == 0) {
            prefetch_tmap(&tmW);
            int issued = 0;
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                for (int ob = 0; ob < NB; ++ob) {
                    const int i = tl * NB + ob, s = i % kWStages, ph = (i / kWStages) & 1;
                    if (!mbar_wait(&w_empty[s], ph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    const int dd = ob / P.n_cblk, c_first = (ob % P.n_cblk) * kCB;
                    mbar_arrive_expect_tx(&w_full[s], kWStage);
                    tma_load_2d(sm + kWS + s * kWStage, &tmW, &w_full[s], 0, (dd * C + c_first) * kTaps);
                    issued = i + 1;
                }
            }
            int never = 0;
            for (int i = issued > kWStages ? issued - kWStages : 0; i < issued; ++i)
                mbar_wait(&w_full[i % kWStages], (i / kWStages) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(1, 1, 1, kPx, kN);   // A (dK) and B (W) MN-major
            // descriptors are built once; each MMA only moves a start address (desc_advance)
            const uint64_t dk_base = smem_desc(smem_u32(sm + kDK), 16384, 1024, kSwizzle128B);
            const uint64_t w_base = smem_desc(smem_u32(sm + kWS), 8192, 1024, kSwizzle128B);
            const uint32_t dk_hi = (uint32_t)(dk_base >> 32), w_hi = (uint32_t)(w_base >> 32);
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                const int tb = tl & 1, tph = (tl >> 1) & 1;
                if (!mbar_wait(&acc_empty[tb], tph ^ 1, P.err, abort_v)) break;
                tc_fence_after();
                for (int ob = 0; ob < NB && ok; ++ob) {
                    const int i = tl * NB + ob, s = i % kWStages, ph = (i / kWStages) & 1;
                    if (!mbar_wait(&w_full[s], ph, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    const uint32_t wa = (uint32_t)w_base + (uint32_t)((s * kWStage) >> 4);
                    for (int st = 0; st < kSub; ++st) {
                        const int kd = i * kSub + st, db = kd & 1;
                        if (!mbar_wait(&dk_full[db], (kd >> 1) & 1, P.err, abort_v)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t da = (uint32_t)dk_base + (uint32_t)((db * kDKBytes) >> 4);
                        const uint32_t dt = tmem + (tb * kSub + st) * kN;
#pragma unroll
                        for (int kk = 0; kk < kBlockRows / 16; ++kk)
                            mma_f16_lh(dt, da + (uint32_t)(kk * 128), dk_hi, wa + (uint32_t)(kk * 128), w_hi, idesc,
                                       (ob > 0 || kk > 0) ? 1u : 0u);
                        mma_commit(&dk_empty[db]);
                    }
                    mma_commit(&w_empty[s]);
                }
                if (ok) mma_commit(&acc_full[tb]);
            }
            mma_commit(&mma_done);
            int never = 0;
            mbar_wait(&mma_done, 0, P.err, &never);
        }
    } else if (warp < 2 + kFormWarps) {
        // ------------------------------------------------------- dK formers
        // group grp forms the sub-tiles kd with kd % 2 == grp into dK^T buffer grp
        const int grp = (warp - 2) / kGroupWarps;
        const int et = threadIdx.x - 64 - grp * 32 * kGroupWarps;
        const int slot_elems = P.xslot_bytes / 2;
        bool ok = true;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            for (int ob = 0; ob < NB && ok; ++ob) {
                const int i = tl * NB + ob, s = i % kXgStages, ph = (i / kXgStages) & 1;
                if (kSub == 1 && (i & 1) != grp) continue;   // the other group's block
                if (!mbar_wait(&xg_full[s], ph, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                const int dd = ob / P.n_cblk, c_first = (ob % P.n_cblk) * kCB;
                const int nrows = min(kCB, C - c_first) * kTaps;
                const int dil = dil_of(P.d, dd);
                const bf16* gs = reinterpret_cast<const bf16*>(sm + kXG + s * kXgStage);
                const uint32_t* xs32 = reinterpret_cast<const uint32_t*>(sm + kXG + s * kXgStage + kGStage);
                for (int st = kSub > 1 ? grp : 0; st < kSub; st += 2) {
                    const int kd = i * kSub + st, db = kd & 1;
                    if (!mbar_wait(&dk_empty[db], ((kd >> 1) & 1) ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    form_dk_tile<K>(sm + kDK + db * kDKBytes, xs32, gs + st * kPx, kSPx, nrows, slot_elems, P.R, dil,
                                 st * kTH, et, 32 * kGroupWarps);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dk_full[db]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&xg_empty[s]);
            }
        }
    } else if (warp < kWWarp) {
        // ------------------------------------------------------- epilogue: dy stores
        const int q = warp & 3;
        const int m = q * 32 + lane;              // pixel slot == TMEM lane
        const int tr = m / kTW, tcol = m % kTW;
        for (int tl = 0; tl < n_my; ++tl) {
            const int tb = tl & 1, tph = (tl >> 1) & 1;
            if (!mbar_wait(&acc_full[tb], tph, P.err, abort_v)) break;
            tc_fence_after();
            const int t = blockIdx.x + tl * gridDim.x;
            const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
            const int h0 = (ti / P.tiles_w) * kSTH, w0 = (ti % P.tiles_w) * kTW;
            for (int st = 0; st < kSub; ++st) {
                const int h = h0 + st * kTH + tr, w = w0 + tcol;
                bf16* out = P.dy + (long long)b * C * P.d.HW + (long long)h * P.d.W + w;
#pragma unroll
                for (int jh = 0; jh < kN; jh += 32) {   // 32 columns at a time (register budget)
                    uint32_t v[32];
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (tb * kSub + st) * kN + jh;
                    DDPM_TMEM_LD_X16(ta, (v + 0));
                    DDPM_TMEM_LD_X16(ta + 16, (v + 16));
                    tmem_ld_wait();
                    if (h < P.d.H && w < P.d.W) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (jh + j < C)
                                out[(long long)(jh + j) * P.d.HW] = __float2bfloat16_rn(__uint_as_float(v[j]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[tb]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int K, int SUB>
cudaError_t launch_k(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s) {
    using G = BwdGeom<K>;
    using L = DyLayout<K, SUB>;
    constexpr int kSTH = L::kSTH;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dy_tc_kernel<K, SUB>, L::kSmemBytes, attr_done);
        if (e != cudaSuccess) return e;
    }
    DyTcParams P;
    P.d = d;
    P.tiles_w = (d.W + kTW - 1) / kTW;
    P.tiles_per_img = ((d.H + kSTH - 1) / kSTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.n_cblk = (d.C + G::kCB - 1) / G::kCB;
    P.n_oblk = 3 * P.n_cblk;
    P.R = d.R();
    P.WHx = kSTH + 2 * P.R;
    P.xslot_bytes = P.WHx * G::kWinCols * 2;
    P.dy = static_cast<bf16*>(dy);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    CUtensorMap tmW, tmG, tmX;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)d.C, (cuuint64_t)d.O};
        const cuuint64_t str[1] = {(cuuint64_t)d.C * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)kBlockRows};
        const cuuint32_t es[2] = {1, 1};
        if (encode_fn()(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, str, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (!encode_nchw(&tmG, g, d, 4 * d.C, kTW, kSTH, G::kCB, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_nchw(&tmX, x, d, d.C, G::kWinCols, (uint32_t)P.WHx, G::kCB, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int grid = num_sms();
    if (grid > P.n_tiles) grid = P.n_tiles;
    trace_begin(s, kKBwdDyTc);
    bwd_dy_tc_kernel<K, SUB><<<grid, kThreads, L::kSmemBytes, s>>>(tmW, tmG, tmX, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace

bool bwd_dy_tc_eligible(const Dims& d, const void* g, const void* x, const void* w) {
    return bwdtc::eligible(d, g, x, w, true) &&
           d.R() <= (d.K == 3 ? DyLayout<3, 4>::kMaxR : DyLayout<5, 4>::kMaxR);
}

cudaError_t launch_bwd_dy_tc(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s) {
    const long long super_tiles = (long long)d.B * ((d.H + 4 * kTH - 1) / (4 * kTH)) * ((d.W + kTW - 1) / kTW);
    const bool small = super_tiles < num_sms() / 2;
    if (d.K == 3) return small ? launch_k<3, 1>(d, g, x, w, dy, s) : launch_k<3, 4>(d, g, x, w, dy, s);
    return small ? launch_k<5, 1>(d, g, x, w, dy, s) : launch_k<5, 4>(d, g, x, w, dy, s);
}

}  // namespace ddpm
