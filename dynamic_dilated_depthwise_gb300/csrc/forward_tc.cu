// forward_tc.cu -- fused generator + dynamic filter on tcgen05 tensor cores (bf16).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA 融合生成器推理":
//   y tile -> dot(weight, y) -> dynamic taps -> consume with shifted x -> output,
// with the taps living only on chip; BF16 taps are rounded to bf16 before use.
//
// GB300 design.  A persistent CTA owns one group of CG output channels (CG = 8
// for K = 3, two CTAs per SM; CG = 4 for K = 5, one CTA per SM) and walks pixel
// tiles of 128 pixels (2 rows x 64 columns, or several whole rows when W < 64).
// Per tile and dilation d the generator GEMM is
//   D[p, n] = sum_j y[j, p] * W[o_n, j] + bias[o_n],  n = c_local*K*K + k
// (CG*K*K taps, padded to N = 80 for K = 3 and N = 112 for K = 5), issued as
// tcgen05.mma (M = 128 pixels, N, K = 64 in four K=16 steps, plus one K=16 step
// that adds the bias through a ones column) into TMEM:
// TMEM lane = pixel, so each epilogue thread owns every tap of its pixel and
// filters without any cross-thread reduction.
//
//   warp 0      TMA producer: W slice of the group (once), y tiles (2 stages)
//   warp 1      TMEM owner + MMA issuer (one elected lane)
//   warp 2      TMA producer: the x window of each tile, one box per channel
//               into a slot of fixed stride (2 buffers)
//   warps 3..   epilogue: each thread owns one pixel and kCPT channels.  Per
//               dilation it reads its K*K*kCPT taps from TMEM, rounds each pair
//               of channels' taps to bf16 with one conversion, and accumulates
//               tap * x with the mixed-precision FMA (bf16 operands, FP32
//               accumulator, exact product), x read as bf16 straight from the
//               window at immediate offsets.
// Three TMEM regions (one per dilation, N columns each) form the MMA /
// epilogue pipeline: a region is released as soon as its taps are in registers.
#include <utility>

#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kTile = 128;               // pixels per tile (MMA M)
constexpr int kKPad = 64;                // generator K (channels of y), zero padded
constexpr int kEpi0 = 3;                 // first epilogue warp

// Per-kernel-size configuration.  A CTA owns CG output channels: its MMA N per
// dilation is the group's CG*K*K taps padded to a multiple of 16, and its x window
// keeps HALO columns left and right of the tile (the tile start minus HALO stays a
// 16-byte TMA coordinate; HALO >= the halo radius R).
template <int K>
struct FwdCfg;
template <>
struct FwdCfg<3> {
    static constexpr int CG = 8, N = 80, HALO = 8, WINMAX = 960, CTAS = 2, TMEM_COLS = 256;
};
template <>
struct FwdCfg<5> {
    static constexpr int CG = 4, N = 112, HALO = 16, WINMAX = 2112, CTAS = 1, TMEM_COLS = 512;
};

template <int K>
struct FwdLayout {
    using F = FwdCfg<K>;
    static constexpr int kCG = F::CG;                  // output channels per CTA group
    static constexpr int kTaps = K * K;
    static constexpr int kN = F::N;                    // MMA N per dilation
    static constexpr int kEpiWarps = 8;                // 4 TMEM lane quadrants x (kCG / kCPT) channel sets
    static constexpr int kCPT = kCG / (kEpiWarps / 4); // channels per epilogue thread
    static constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
    static constexpr int kCtasPerSm = F::CTAS;
    static constexpr int kTmemCols = F::TMEM_COLS;
    static constexpr int kHalo = F::HALO;
    static constexpr int kWinMax = F::WINMAX;          // x window positions: (TH + 2R) x (TW + 2 HALO)
    static constexpr int kSlot = kWinMax * 2;          // bytes per channel slot of an x window buffer
    static constexpr int kRawBufs = 2;                 // x window buffers
    // shared-memory carve-up (bytes, from a 1024-aligned base).  The 128-byte
    // swizzled operands come first so that every swizzle atom starts on 1024 B.
    static constexpr int kSW = 0;                      // W slice, 3 x [N x 128 B], SW128 K-major
    static constexpr int kSWBytes = 3 * kN * 128;
    static constexpr int kSY = kSW + kSWBytes;         // y tiles, 2 x [64 j x 128 px] SW128 MN-major
    static constexpr int kSYBytes = 2 * kTile * kKPad * 2;
    static constexpr int kSBias = kSY + kSYBytes;      // bias B operand, 3 x [N x 16] no swizzle
    static constexpr int kSBiasBytes = 3 * kN * 32;
    static constexpr int kSOnes = kSBias + kSBiasBytes;   // ones A operand [128 x 16] no swizzle
    static constexpr int kSOnesBytes = kTile * 32;
    static constexpr int kSRaw = kSOnes + kSOnesBytes; // 2 x x window [CG slots of kSlot B][rows][cols] bf16
    static constexpr int kRawBuf = kCG * kSlot;
    static constexpr int kSStage = kSRaw + kRawBufs * kRawBuf;   // output staging, 4 blocks x [CG][TH][TW] bf16
    static constexpr int kStageBlk = kCG * kTile * 2;
    static constexpr int kSmemBytes = kSStage + 4 * kStageBlk + 1024;   // + alignment slack
    static_assert(kCG * kTaps <= kN && kN % 16 == 0 && 3 * kN <= kTmemCols, "MMA N and TMEM columns");
    static_assert(kCPT % 2 == 0 && kCG % kCPT == 0, "channel pairs per thread");
    static_assert(kSW % 1024 == 0 && kSY % 1024 == 0 && (kSY + kSYBytes / 2) % 1024 == 0, "SW128 atoms need 1 KiB");
    static_assert(kSBias % 16 == 0 && kSOnes % 16 == 0 && kSRaw % 128 == 0 && kSlot % 128 == 0 && kSStage % 128 == 0,
                  "operand alignment");
    // co-resident blocks: each takes dynamic + ~0.2 KiB static + 1 KiB reserved of the SM's 228 KiB
    static_assert(kCtasPerSm * (kSmemBytes + 256 + 1024) <= 228 * 1024, "shared memory of co-resident blocks");
};

struct FwdTcParams {
    Dims d;
    int TH, TW;            // tile rows / columns (TH * TW = 128, or whole rows when W < 64)
    int tiles_per_row;     // W >= 64: ceil(W / 64); else 1
    int tiles_per_img;
    int n_tiles;           // B * tiles_per_img
    int n_groups;          // C / CG
    int ctas_per_group;
    int R;                 // halo radius = max dilation * (K / 2)
    int WH, WC;            // x window rows (TH + 2R) / columns (TW + 2 HALO, origin w0 - HALO)
    const bf16* bias;      // may be null
    unsigned int* err;
};

struct TileCoord {
    int b, h0, w0;
};

__device__ __forceinline__ TileCoord tile_coord(const FwdTcParams& P, int t) {
    TileCoord c;
    c.b = t / P.tiles_per_img;
    const int ti = t % P.tiles_per_img;
    c.h0 = (ti / P.tiles_per_row) * P.TH;
    c.w0 = (ti % P.tiles_per_row) * P.TW;
    return c;
}

// bf16x2 of two fp32 values (round to nearest even): lo in bits 0..15, hi in 16..31
__device__ __forceinline__ uint32_t round_pair(uint32_t lo, uint32_t hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(__uint_as_float(hi)), "f"(__uint_as_float(lo)));
    return r;
}

// a0 += lo(t) * x0, a1 += hi(t) * x1: bf16 operands, exact product, FP32 accumulate
__device__ __forceinline__ void fma_pair(float& a0, float& a1, uint32_t t, unsigned short x0, unsigned short x1) {
    asm("{\n\t.reg .b16 tl, th;\n\t"
        "mov.b32 {tl, th}, %2;\n\t"
        "fma.rn.f32.bf16 %0, tl, %3, %0;\n\t"
        "fma.rn.f32.bf16 %1, th, %4, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(t), "h"(x0), "h"(x1));
}

template <int NTHREADS>
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(NTHREADS) : "memory"); }

// v[I] = the 16-bit value at addr + I * SLOT, I = 0 .. N-1 (compile-time offsets)
template <int SLOT, int... I>
__device__ __forceinline__ void lds_slots(uint32_t addr, unsigned short* v, std::integer_sequence<int, I...>) {
    ((v[I] = tc::lds_u16<I * SLOT>(addr)), ...);
}

// The constant MMA operands of a CTA: a ones column (A, [128 x 16]) and the bias column of
// each dilation (B, [N x 16]), K = 16, no swizzle.  In the core-matrix layout row r's k = 0..7
// sit at (r/8)*256 + (r%8)*16 and k = 8..15 128 bytes further; one thread per row writes both
// 16-byte halves, and each bias value is one load (a loop of dependent cold loads here cost
// microseconds).  Kept out of line: it runs once per CTA and leaves the epilogue's registers alone.
template <int K>
__device__ __noinline__ void fill_const_operands(uint8_t* sm, const bf16* bias, int C, int c0, int et) {
    using L = FwdLayout<K>;
    constexpr int kN = L::kN, kTaps = L::kTaps, kCG = L::kCG, nthr = 32 * L::kEpiWarps;
    for (int m = et; m < kTile; m += nthr) {
        uint8_t* r = sm + L::kSOnes + (m / 8) * 256 + (m % 8) * 16;
        *reinterpret_cast<uint4*>(r) = make_uint4(0x3F80u, 0u, 0u, 0u);   // bf16 1.0 in column 0
        *reinterpret_cast<uint4*>(r + 128) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int i = et; i < 3 * kN; i += nthr) {
        const int dd = i / kN, n = i - dd * kN;
        // columns n < CG*K*K are this group's taps (o < O: C is a multiple of CG), the rest padding
        uint32_t v = 0u;
        if (bias != nullptr && n < kCG * kTaps) v = __bfloat16_as_ushort(bias[(dd * C + c0) * kTaps + n]);
        uint8_t* r = sm + L::kSBias + dd * kN * 32 + (n / 8) * 256 + (n % 8) * 16;
        *reinterpret_cast<uint4*>(r) = make_uint4(v, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(r + 128) = make_uint4(0u, 0u, 0u, 0u);
    }
}

template <int K>
__global__ void __launch_bounds__(FwdLayout<K>::kThreads, FwdLayout<K>::kCtasPerSm)
    forward_tc_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmO,
                      const FwdTcParams P) {
    using namespace tc;
    using L = FwdLayout<K>;
    constexpr int kCG = L::kCG, kTaps = L::kTaps, kN = L::kN, kEpiWarps = L::kEpiWarps, kCPT = L::kCPT;
    constexpr int kTmemCols = L::kTmemCols, kHalo = L::kHalo, kSlot = L::kSlot, kRawBufs = L::kRawBufs;
    constexpr int kSW = L::kSW, kSY = L::kSY, kSBias = L::kSBias, kSOnes = L::kSOnes, kSRaw = L::kSRaw;
    constexpr int kRawBuf = L::kRawBuf, kSStage = L::kSStage, kStageBlk = L::kStageBlk;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base, derived by pointer arithmetic on the shared array so that every
    // access through it stays a shared-memory access (an integer round trip would make
    // them generic loads and stores with 64-bit addresses)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bar_w, bar_y_full[2], bar_y_empty[2], bar_acc_full[3], bar_acc_empty[3],
        bar_raw_full[kRawBufs], bar_raw_empty[kRawBufs], bar_done;
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
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_y_full[s], 1);
            mbar_init(&bar_y_empty[s], 1);
        }
        for (int s = 0; s < kRawBufs; ++s) {
            mbar_init(&bar_raw_full[s], 1);
            mbar_init(&bar_raw_empty[s], kEpiWarps);
        }
        for (int dd = 0; dd < 3; ++dd) {
            mbar_init(&bar_acc_full[dd], 1);
            mbar_init(&bar_acc_empty[dd], kEpiWarps);
        }
        mbar_init(&bar_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
    if (warp >= kEpi0) {
        // constant MMA operands: a ones column (A) and the bias column (B), K = 16, no swizzle
        fill_const_operands<K>(sm, P.bias, C, c0, threadIdx.x - 32 * kEpi0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int n_my = cta_in_group < P.n_tiles ? (P.n_tiles - 1 - cta_in_group) / P.ctas_per_group + 1 : 0;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmY);
            prefetch_tmap(&tmW);
            mbar_arrive_expect_tx(&bar_w, 3 * kN * 128);
            for (int dd = 0; dd < 3; ++dd)
                tma_load_2d(sm + kSW + dd * kN * 128, &tmW, &bar_w, 0, (dd * C + c0) * kTaps);
            // second 64-pixel half: the next row of a 2 x 64 tile, or the next 64 pixels of whole rows
            const int half_step = P.TW == 64 ? P.d.W : 64;
            int issued_y = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i & 1, ph = (i >> 1) & 1;
                const TileCoord tcd = tile_coord(P, cta_in_group + i * P.ctas_per_group);
                if (!mbar_wait(&bar_y_empty[s], ph ^ 1, P.err, abort_v)) break;
                const int pb = tcd.h0 * P.d.W + tcd.w0;
                mbar_arrive_expect_tx(&bar_y_full[s], kTile * kKPad * 2);
                tma_load_3d(sm + kSY + s * 16384, &tmY, &bar_y_full[s], pb, 0, tcd.b);
                tma_load_3d(sm + kSY + s * 16384 + 8192, &tmY, &bar_y_full[s], pb + half_step, 0, tcd.b);
                issued_y = i + 1;
            }
            // drain: every copy this thread started must land before shared memory is released
            int never = 0;
            mbar_wait(&bar_w, 0, P.err, &never);
            for (int i = issued_y > 2 ? issued_y - 2 : 0; i < issued_y; ++i)
                mbar_wait(&bar_y_full[i & 1], (i >> 1) & 1, P.err, &never);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------- TMA producer: x windows
        if (lane == 0) {
            prefetch_tmap(&tmX);
            const int nch = min(kCG, C - c0);                  // channel boxes inside the tensor
            const uint32_t raw_bytes = (uint32_t)(nch * P.WH * P.WC * 2);
            int issued_x = 0, s = 0, ph = 0;
            for (int i = 0; i < n_my; ++i) {
                const TileCoord tcd = tile_coord(P, cta_in_group + i * P.ctas_per_group);
                if (!mbar_wait(&bar_raw_empty[s], ph ^ 1, P.err, abort_v)) break;
                mbar_arrive_expect_tx(&bar_raw_full[s], raw_bytes);
                uint8_t* rb = sm + kSRaw + s * kRawBuf;
                for (int c = 0; c < nch; ++c)
                    tma_load_4d(rb + c * kSlot, &tmX, &bar_raw_full[s], tcd.w0 - kHalo, tcd.h0 - P.R, c0 + c, tcd.b);
                issued_x = i + 1;
                if (++s == kRawBufs) {
                    s = 0;
                    ph ^= 1;
                }
            }
            int never = 0;
            for (int i = issued_x > kRawBufs ? issued_x - kRawBufs : 0; i < issued_x; ++i)
                mbar_wait(&bar_raw_full[i % kRawBufs], (i / kRawBufs) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(&bar_w, 0, P.err, abort_v);
            const uint32_t idesc = instr_desc(1, 1, 0, kTile, kN);     // A (y) MN-major, B (W) K-major
            const uint32_t idesc_b = instr_desc(1, 0, 0, kTile, kN);   // ones x bias, both K-major
            // descriptors are built once; each MMA only moves a start address (desc_advance)
            const uint64_t d_ones = smem_desc(smem_u32(sm + kSOnes), 128, 256, kSwizzleNone);
            const uint64_t y_base = smem_desc(smem_u32(sm + kSY), 8192, 1024, kSwizzle128B);
            const uint64_t w_base = smem_desc(smem_u32(sm + kSW), 16, 1024, kSwizzle128B);
            const uint64_t b_base = smem_desc(smem_u32(sm + kSBias), 128, 256, kSwizzleNone);
            for (int i = 0; ok && i < n_my; ++i) {
                const int s = i & 1, ph = (i >> 1) & 1;
                if (!mbar_wait(&bar_y_full[s], ph, P.err, abort_v)) break;
                tc_fence_after();
                const uint64_t ya = desc_advance(y_base, (uint32_t)s * 16384);
                for (int dd = 0; dd < 3 && ok; ++dd) {
                    if (!mbar_wait(&bar_acc_empty[dd], (i & 1) ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + dd * kN;
                    const uint64_t wa = desc_advance(w_base, (uint32_t)dd * kN * 128);
#pragma unroll
                    for (int kk = 0; kk < kKPad / 16; ++kk)
                        mma_f16(dt, desc_advance(ya, kk * 2048), desc_advance(wa, kk * 32), idesc, kk > 0);
                    mma_f16(dt, d_ones, desc_advance(b_base, (uint32_t)dd * kN * 32), idesc_b, 1);
                    mma_commit(&bar_acc_full[dd]);
                }
                if (!ok) break;
                mma_commit(&bar_y_empty[s]);
            }
            // all issued MMAs must retire before TMEM is released
            mma_commit(&bar_done);
            int never = 0;
            mbar_wait(&bar_done, 0, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- epilogue
        // Results go to a staging block [8 ch][TH][TW] per output block (x, d1, d3, d5),
        // which one thread writes out with TMA stores, two blocks at a time once every
        // epilogue warp has filled them; the stores clip pixels outside the image.
        const int ew = warp - kEpi0;
        const int q = warp & 3;          // TMEM lane quadrant this warp may access
        const int cl0 = (ew >> 2) * kCPT;   // first local channel of this thread
        const int s = q * 32 + lane;     // pixel slot == TMEM lane
        const bool leader = ew == 0 && lane == 0;   // issues the TMA stores
        // slots beyond the tile (whole-row tiles of fewer than 128 pixels) read the window at
        // pixel (0, 0) and store nothing, so every shared-memory access stays inside its buffer
        const int tpix = P.TH * P.TW;
        const bool in_tile = s < tpix;
        const int rr = in_tile ? s / P.TW : 0, cc = in_tile ? s % P.TW : 0;
        const int WC = P.WC;
        const int center = (rr + P.R) * WC + cc + kHalo;   // window position of this pixel
        const uint32_t ch_stride = (uint32_t)tpix * 2;   // staging bytes per channel
        // this thread's first staging element of block 0
        const uint32_t st0 = smem_u32(sm + kSStage) + (uint32_t)cl0 * ch_stride + (uint32_t)(in_tile ? s : 0) * 2;
        int buf = 0, bph = 0;
        // hand staging blocks blk and blk+1 of tile tcd to the TMA (twice per tile: blocks 0, 1
        // after the first dilation, 2, 3 after the last): called by every epilogue thread after
        // writing its values, the same number of times by all of them even after a failed wait
        // (the named barrier has no time limit).  Before the barrier the leader waits until the
        // previous pair's stores have read their blocks, so that past the barrier every thread
        // may write the blocks that pair used (the next pair's writes come after it).
        bool ok = true;
        auto flush_pair = [&](int blk, const TileCoord& tcd) {
            fence_proxy_async_smem();
            if (leader) bulk_wait_read<0>();
            epi_bar<32 * kEpiWarps>();
            if (leader && ok) {
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int cbase = (blk + bb == 0 ? 0 : (blk + bb) * C) + c0;
                    const uint8_t* src = sm + kSStage + (blk + bb) * kStageBlk;
                    tma_store_4d(&tmO, src, tcd.w0, tcd.h0, cbase, tcd.b);
                }
                bulk_commit();
            }
        };
        for (int i = 0; i < n_my; ++i) {
            const TileCoord tcd = tile_coord(P, cta_in_group + i * P.ctas_per_group);
            // this thread's channel slots of the window: slot c at xa + c * kSlot
            const uint32_t xa = smem_u32(sm + kSRaw + buf * kRawBuf + cl0 * kSlot) + (uint32_t)center * 2;
            // waits are made warp-uniform (tcgen05.ld is a whole-warp instruction) and sticky:
            // after a failure the thread only keeps the barrier sequence
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar_raw_full[buf], bph, P.err, abort_v));
            // channels c0 .. c0+7 of the output are x itself
            if (ok && in_tile) {
                unsigned short v[kCPT];
                lds_slots<kSlot>(xa, v, std::make_integer_sequence<int, kCPT>{});
#pragma unroll
                for (int c = 0; c < kCPT; ++c)
                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(st0 + c * ch_stride), "h"(v[c]) : "memory");
            }
            for (int dd = 0; dd < 3; ++dd) {
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc_full[dd], i & 1, P.err, abort_v));
                if (!ok) {
                    if (dd != 1) flush_pair(dd, tcd);
                    continue;
                }
                tc_fence_after();
                uint32_t t[kCPT * kTaps];
                tmem_load_cols<kCPT * kTaps>(tmem + ((uint32_t)(q * 32) << 16) + dd * kN + cl0 * kTaps, t);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_acc_empty[dd]);
                const int dil = dil_of(P.d, dd);
                unsigned short xv[kTaps][kCPT];
#pragma unroll
                for (int k = 0; k < kTaps; ++k) {
                    constexpr int r0 = K / 2;
                    const uint32_t a = xa + (uint32_t)(((k / K - r0) * WC + (k % K - r0)) * dil * 2);
                    lds_slots<kSlot>(a, xv[k], std::make_integer_sequence<int, kCPT>{});
                }
                float acc[kCPT];
#pragma unroll
                for (int c = 0; c < kCPT; ++c) acc[c] = 0.0f;
#pragma unroll
                for (int k = 0; k < kTaps; ++k) {
#pragma unroll
                    for (int c = 0; c < kCPT; c += 2) {
                        const uint32_t tp = round_pair(t[c * kTaps + k], t[(c + 1) * kTaps + k]);
                        fma_pair(acc[c], acc[c + 1], tp, xv[k][c], xv[k][c + 1]);
                    }
                }
                if (in_tile) {
                    const uint32_t sa = st0 + (uint32_t)(1 + dd) * kStageBlk;
#pragma unroll
                    for (int c = 0; c < kCPT; c += 2) {
                        const uint32_t o = round_pair(__float_as_uint(acc[c]), __float_as_uint(acc[c + 1]));
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(sa + c * ch_stride), "h"((unsigned short)(o & 0xFFFFu))
                                     : "memory");
                        asm volatile("st.shared.u16 [%0], %1;" ::"r"(sa + (c + 1) * ch_stride), "h"((unsigned short)(o >> 16))
                                     : "memory");
                    }
                }
                if (dd == 2) {
                    // the window has been read for the last time
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar_raw_empty[buf]);
                }
                if (dd != 1) flush_pair(dd, tcd);   // blocks 0, 1 after dilation 0; 2, 3 after dilation 2
            }
            if (++buf == kRawBufs) {
                buf = 0;
                bph ^= 1;
            }
        }
        // every store has finished writing global memory (and reading shared memory)
        if (leader) bulk_wait<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

struct Tiling {
    int TH, TW, tiles_per_row, tiles_per_img, R, WH, WC;
};

Tiling tiling_of(const Dims& d, int halo) {
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
    t.R = d.R();
    t.WH = t.TH + 2 * t.R;
    t.WC = t.TW + 2 * halo;
    return t;
}

template <int K>
bool eligible_k(const Dims& d) {
    using L = FwdLayout<K>;
    if (d.C % 8 != 0 || d.C % L::kCG != 0 || d.C > kKPad) return false;   // TMA row stride of W; one 64-wide K block
    if (d.R() > L::kHalo) return false;                 // the x window spans w0 - HALO .. w0 + TW + HALO
    const Tiling t = tiling_of(d, L::kHalo);
    if ((long long)t.WH * t.WC > L::kWinMax || t.WH > 256) return false;
    const long long tiles = (long long)d.B * t.tiles_per_img;
    return tiles <= (1LL << 30) && d.O <= (1LL << 30) && d.HW <= (1LL << 31) - 1024;
}

template <int K>
cudaError_t launch_k(const Dims& d, const void* x, const void* y, const void* w, const void* bias, void* out,
                     cudaStream_t s) {
    using L = FwdLayout<K>;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)forward_tc_kernel<K>, L::kSmemBytes, attr_done, true);
        if (e != cudaSuccess) return e;
    }
    auto enc = bwdtc::encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    if ((uintptr_t)x % 16 != 0) return cudaErrorInvalidValue;
    const Tiling t = tiling_of(d, L::kHalo);
    CUtensorMap tmY, tmW, tmX, tmO;
    const cuuint64_t dimY[3] = {(cuuint64_t)d.HW, (cuuint64_t)d.C, (cuuint64_t)d.B};
    const cuuint64_t strY[2] = {(cuuint64_t)d.HW * 2, (cuuint64_t)d.HW * d.C * 2};
    const cuuint32_t boxY[3] = {64, (cuuint32_t)kKPad, 1};
    const cuuint32_t one3[3] = {1, 1, 1};
    if (enc(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(y), dimY, strY, boxY, one3,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const cuuint64_t dimW[2] = {(cuuint64_t)d.C, (cuuint64_t)d.O};
    const cuuint64_t strW[1] = {(cuuint64_t)d.C * 2};
    const cuuint32_t boxW[2] = {(cuuint32_t)kKPad, (cuuint32_t)L::kN};
    const cuuint32_t one2[2] = {1, 1};
    if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dimW, strW, boxW, one2,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (!bwdtc::encode_nchw(&tmX, x, d, d.C, (uint32_t)t.WC, (uint32_t)t.WH, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    // output [B, 4C, H, W]: boxes of CG channels x one tile, written from the staging blocks
    if ((uintptr_t)out % 16 != 0 || !bwdtc::encode_nchw(&tmO, out, d, 4 * d.C, (uint32_t)t.TW, (uint32_t)t.TH,
                                                        (uint32_t)L::kCG, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;

    FwdTcParams P;
    P.d = d;
    P.TH = t.TH;
    P.TW = t.TW;
    P.tiles_per_row = t.tiles_per_row;
    P.tiles_per_img = t.tiles_per_img;
    P.n_tiles = d.B * t.tiles_per_img;
    P.n_groups = d.C / L::kCG;
    const int ctas = num_sms() * L::kCtasPerSm;
    int cpg = ctas / P.n_groups;
    if (cpg < 1) cpg = 1;
    if (cpg > P.n_tiles) cpg = P.n_tiles;
    P.ctas_per_group = cpg;
    P.R = t.R;
    P.WH = t.WH;
    P.WC = t.WC;
    P.bias = static_cast<const bf16*>(bias);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    trace_begin(s, kKForwardTc);
    forward_tc_kernel<K><<<P.n_groups * cpg, L::kThreads, L::kSmemBytes, s>>>(tmY, tmW, tmX, tmO, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace

bool forward_tc_eligible(const Dims& d, const void* y, const void* w) {
    if (d.dtype != 1 || (d.flags & kFlagCudaCores)) return false;
    if (d.W % 8 != 0) return false;                     // every tile start is a 16-byte TMA coordinate
    if ((uintptr_t)y % 16 != 0 || (uintptr_t)w % 16 != 0) return false;
    const bool shape = d.K == 3 ? eligible_k<3>(d) : d.K == 5 ? eligible_k<5>(d) : false;
    return shape && bwdtc::encode_fn() != nullptr;
}

cudaError_t launch_forward_tc(const Dims& d, const void* x, const void* y, const void* w, const void* bias,
                              void* out, cudaStream_t s) {
    if (d.K == 3) return launch_k<3>(d, x, y, w, bias, out, s);
    if (d.K == 5) return launch_k<5>(d, x, y, w, bias, out, s);
    return cudaErrorInvalidValue;
}

}  // namespace ddpm
