// bwd_dx_tc.cu -- dX on tcgen05 tensor cores (bf16).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dX recomputes the dynamic taps and gathers each dilation's contribution:
//   dx[b,c,q] = grad[b,c,q] + sum_{d,ky,kx} Tq[b,o,q-off] * grad[b,(1+d)C+c,q-off],
//   Tq = bf16(bias[o] + sum_j W[o,j] y[b,j,q-off]),  o = (d*C + c)*9 + ky*3 + kx.
//
// GB300 design: one shifted GEMM per tap, so the taps are recomputed exactly
// once per (pixel, tap) with no halo recompute.  A CTA owns a 16x8 pixel tile
// (MMA M = 128, slot s = r*8 + c) and all 64 channels (N = 64):
//   - the y window of the tile, (16+2R) x (8+2R) positions, is staged once as
//     unswizzled K-major core matrices [8-channel chunk][position][8]: eight
//     consecutive slots are eight consecutive positions of one window row, so
//     the A operand of tap (dy, dx) is the same window at a start offset of
//     ((R-dy)*WW + (R-dx)) * 16 bytes (row-group stride WW * 16);
//   - a fifth K=16 step adds the bias: A is a constant 8-row ones column read
//     by every row group (row-group stride 0), B the bias tile the producer
//     writes per tap;
//   - the producer brings W's rows of tap (d, k) for all channels by TMA
//     (a 3-D view of W: [dc][k][j]) into a 3-stage ring;
//   - D of each tap lands in one of eight TMEM buffers [128 x 64];
//   - a second producer warp streams the raw windows -- 8-channel chunks
//     [8 ch][16+2R rows][24 cols] of y and of each dilation's grad planes, then
//     the tile's own grad block 0 (the identity term) as two [32 ch][16][8] chunks --
//     by TMA through a 4-stage ring; eight worker warps transpose each chunk
//     into the K-major y window or the position-major grad window, then per
//     tap round the taps to bf16 and accumulate tap * grad at the gathered
//     position.
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using namespace bwdtc;

constexpr int kDxTH = 16, kDxTW = 8;      // pixel tile
constexpr int kDxMaxR = 6;                // halo radius supported by the window buffers
constexpr int kMaxPos = (kDxTH + 2 * kDxMaxR) * (kDxTW + 2 * kDxMaxR);   // 560
constexpr int kN = 64;
constexpr int kTaps = 27;
constexpr int kWorkWarps = 8;
constexpr int kThreads = 32 * (3 + kWorkWarps);   // W producer, MMA, 8 workers, raw producer
constexpr int kRawWarp = 2 + kWorkWarps;
constexpr int kStages = 3;               // W ring
constexpr int kRawStages = 4;            // raw chunk ring
constexpr int kDBufs = 8;
constexpr int kRawCols = 24;              // raw window columns: origin w0 - 8 keeps TMA 16-byte aligned
constexpr int kRawStage = 8 * (kDxTH + 2 * kDxMaxR) * kRawCols * 2;   // 10752
// raw chunks per tile: y, the grad of each dilation, then the identity term (grad block 0 of
// the tile itself, [32 ch][16 rows][8 cols] per chunk)
constexpr int kChunks = 8 + 3 * 8 + 2;
constexpr int kIdChunk = 8 + 3 * 8;
constexpr int kIdBytes = 32 * kDxTH * kDxTW * 2;      // 8192
static_assert(kIdBytes <= 8 * (kDxTH + 2 * kDxMaxR) * kRawCols * 2, "an identity chunk fits a raw stage");

// shared memory (bytes from a 1024-aligned base)
constexpr int kWTStage = 8192 + 2048;                 // W tap tile (SW128, 64 rows) + bias tile
constexpr int kWT = 0;
constexpr int kRaw = kWT + kStages * kWTStage;        // raw chunk ring [8 ch][rows][24] bf16
constexpr int kYW = kRaw + kRawStages * kRawStage;    // 8 chunks x positions x 16 B
constexpr int kYWBytes = 8 * kMaxPos * 16;            // 71680
constexpr int kGW = kYW + kYWBytes;                   // [position][64] bf16, 16-byte chunks swizzled
constexpr int kGWBytes = kMaxPos * 128;               // 71680
constexpr int kBC = kGW + kGWBytes;                   // copy of the bias [3 d][64 c][9 k] bf16
constexpr int kBCBytes = 3 * 64 * 9 * 2;              // 3456
constexpr int kOnes = kBC + kBCBytes;                 // bias K-step A: [8 rows][16 k], column 0 ones
constexpr int kSmemBytes = kOnes + 256 + 1024;
static_assert(kSmemBytes <= 232448 - 1024, "shared memory");
static_assert(kRaw % 128 == 0 && kRawStage % 128 == 0 && kYW % 16 == 0 && kGW % 16 == 0 && kOnes % 16 == 0,
              "staging alignment");
static_assert(kWTStage % 1024 == 0, "W tap tiles need 1 KiB alignment");

struct DxTcParams {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int R, WH, WW, npos;
    const bf16* y;
    const bf16* g;
    const bf16* bias;
    bf16* dx;
    unsigned int* err;
};

__device__ __forceinline__ void work_bar() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kWorkWarps) : "memory"); }

// Window positions per worker thread: every position of the window at one pass.
constexpr int kPosPerThread = (kMaxPos + 32 * kWorkWarps - 1) / (32 * kWorkWarps);   // 3

// The eight channels of a raw chunk [8 ch][rows][kRawCols] at this thread's window positions
// et, et + 256, ... as bf16 pairs; every load is issued before any result is used (one
// shared-memory latency instead of one per position).  Positions beyond the window read
// position 0 (inside the chunk) and are not stored.
__device__ __forceinline__ void gather_positions(uint32_t (&pk)[kPosPerThread][4], const unsigned short* raw, int et,
                                                 int npos, int WW, int R, int rplane) {
#pragma unroll
    for (int u = 0; u < kPosPerThread; ++u) {
        int pos = et + u * 32 * kWorkWarps;
        if (pos >= npos) pos = 0;
        const int row = pos / WW, re = row * kRawCols + (pos - row * WW) + (8 - R);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            pk[u][e] = (uint32_t)raw[(2 * e) * rplane + re] | ((uint32_t)raw[(2 * e + 1) * rplane + re] << 16);
    }
}

// bf16x2 of two fp32 values (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// a0 += lo(t) * lo(g), a1 += hi(t) * hi(g): bf16 operands, FP32 accumulate, one rounding
__device__ __forceinline__ void fma2_bf16_f32(float& a0, float& a1, uint32_t t, uint32_t g) {
    asm("{\n\t.reg .b16 tl, th, gl, gh;\n\t"
        "mov.b32 {tl, th}, %2;\n\t"
        "mov.b32 {gl, gh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, tl, gl, %0;\n\t"
        "fma.rn.f32.bf16 %1, th, gh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(t), "r"(g));
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dx_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
                     const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmI,
                     const DxTcParams P) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base, derived by pointer arithmetic on the shared array so that every
    // access through it stays a shared-memory access (an integer round trip would make
    // them generic loads and stores with 64-bit addresses)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t wt_full[kStages], wt_empty[kStages], d_full[kDBufs], d_empty[kDBufs], yw_full, yw_empty,
        raw_full[kRawStages], raw_empty[kRawStages], mma_done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.d.C, H = P.d.H, W = P.d.W;
    const long long HW = P.d.HW;
    const int n_my = blockIdx.x < P.n_tiles ? (P.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int R = P.R, WW = P.WW, npos = P.npos;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&wt_full[i], 1);
            mbar_init(&wt_empty[i], 1);
        }
        for (int i = 0; i < kDBufs; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kWorkWarps);
        }
        mbar_init(&yw_full, kWorkWarps);
        mbar_init(&yw_empty, 1);
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(&raw_full[i], 1);
            mbar_init(&raw_empty[i], kWorkWarps);
        }
        mbar_init(&mma_done, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    {
        // the bias into shared memory once ([d][c][k], zero for c >= C): the W producer writes
        // each tap's bias tile from there, with no global load on its per-tap path.  All of a
        // thread's loads are issued before its stores.
        constexpr int kN = 3 * 64 * 9, kPer = (kN + kThreads - 1) / kThreads;
        unsigned short v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = threadIdx.x + j * kThreads;
            const int dd = i / 576, c = (i / 9) % 64, k = i % 9;
            v[j] = (i < kN && P.bias != nullptr && c < C)
                       ? reinterpret_cast<const unsigned short*>(P.bias)[((long long)dd * C + c) * 9 + k]
                       : (unsigned short)0;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int i = threadIdx.x + j * kThreads;
            if (i < kN) reinterpret_cast<unsigned short*>(sm + kBC)[i] = v[j];
        }
    }
    if (warp >= 2 && warp < kRawWarp) {
        // the bias K-step's A operand: one 8-row core-matrix pair (k = 0..7, then 8..15 at +128)
        // with a one in column 0, read by every row group (stride 0)
        const int et = threadIdx.x - 64;
        if (et < 16)
            *reinterpret_cast<uint4*>(sm + kOnes + et * 16) =
                et < 8 ? make_uint4(0x3F80u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- producer: W tap tiles + bias tiles
        if (lane == 0) prefetch_tmap(&tmW);
        bool ok = true;
        int issued = 0;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            for (int u = 0; u < kTaps; ++u) {
                const int i = tl * kTaps + u, st = i % kStages, ph = (i / kStages) & 1;
                int good = 1;
                if (lane == 0) good = mbar_wait(&wt_empty[st], ph ^ 1, P.err, abort_v) ? 1 : 0;
                good = __shfl_sync(0xffffffffu, good, 0);
                if (!good) {
                    ok = false;
                    break;
                }
                const int dd = u / 9, k = u % 9;
                uint8_t* bt = sm + kWT + st * kWTStage + 8192;
                for (int rr = 0; rr < 2; ++rr) {
                    const int c = 2 * lane + rr;
                    const uint32_t bv = reinterpret_cast<const unsigned short*>(sm + kBC)[(dd * 64 + c) * 9 + k];
                    *reinterpret_cast<uint4*>(bt + (c / 8) * 256 + (c % 8) * 16) = make_uint4(bv, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(bt + (c / 8) * 256 + 128 + (c % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(&wt_full[st], 8192);
                    tma_load_3d(sm + kWT + st * kWTStage, &tmW, &wt_full[st], 0, k, dd * C);
                }
                issued = i + 1;
            }
        }
        if (lane == 0) {
            // drain: every copy this CTA started lands before its shared memory is released
            int never = 0;
            for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                mbar_wait(&wt_full[i % kStages], (i / kStages) & 1, P.err, &never);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(1, 0, 0, 128, kN);
            const uint32_t lbo_y = (uint32_t)npos * 16, sbo_y = (uint32_t)WW * 16;
            // descriptors are built once; each MMA only moves a start address (desc_advance)
            const uint64_t y_base = smem_desc(smem_u32(sm + kYW), lbo_y, sbo_y, kSwizzleNone);
            const uint64_t w_base = smem_desc(smem_u32(sm + kWT), 16, 1024, kSwizzle128B);
            const uint64_t bias_base = smem_desc(smem_u32(sm + kWT + 8192), 128, 256, kSwizzleNone);
            const uint64_t ones = smem_desc(smem_u32(sm + kOnes), 128, 0, kSwizzleNone);
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                if (!mbar_wait(&yw_full, tl & 1, P.err, abort_v)) break;
                tc_fence_after();
                for (int u = 0; u < kTaps; ++u) {
                    const int i = tl * kTaps + u, st = i % kStages, buf = i % kDBufs;
                    if (!mbar_wait(&wt_full[st], (i / kStages) & 1, P.err, abort_v) ||
                        !mbar_wait(&d_empty[buf], ((i / kDBufs) & 1) ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int dd = u / 9, k = u % 9, dil = dil_of(P.d, dd);
                    const int ky = k / 3, kx = k - ky * 3;
                    const uint32_t shift = (uint32_t)((R - (ky - 1) * dil) * WW + (R - (kx - 1) * dil)) * 16;
                    const uint64_t ya = desc_advance(y_base, shift);
                    const uint64_t wt = desc_advance(w_base, (uint32_t)st * kWTStage);
                    const uint32_t dt = tmem + buf * kN;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_f16(dt, desc_advance(ya, 2 * kk * lbo_y), desc_advance(wt, kk * 32), idesc, kk > 0);
                    mma_f16(dt, ones, desc_advance(bias_base, (uint32_t)st * kWTStage), idesc, 1);
                    mma_commit(&d_full[buf]);
                    mma_commit(&wt_empty[st]);
                }
                if (ok) mma_commit(&yw_empty);
            }
            mma_commit(&mma_done);
            int never = 0;
            mbar_wait(&mma_done, 0, P.err, &never);
        }
    } else if (warp == kRawWarp) {
        // ------------------------------------------------------- raw window producer
        if (lane == 0) {
            prefetch_tmap(&tmY);
            prefetch_tmap(&tmG);
            prefetch_tmap(&tmI);
            const uint32_t raw_bytes = 8u * (uint32_t)P.WH * kRawCols * 2;
            int issued = 0;
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                const int t = blockIdx.x + tl * gridDim.x;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kDxTH, w0 = (ti % P.tiles_w) * kDxTW;
                for (int idx = 0; idx < kChunks; ++idx) {
                    const int i = tl * kChunks + idx, rs = i % kRawStages;
                    if (!mbar_wait(&raw_empty[rs], ((i / kRawStages) & 1) ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = sm + kRaw + rs * kRawStage;
                    mbar_arrive_expect_tx(&raw_full[rs], idx < kIdChunk ? raw_bytes : (uint32_t)kIdBytes);
                    if (idx < 8) {
                        tma_load_4d(dst, &tmY, &raw_full[rs], w0 - 8, h0 - R, idx * 8, b);
                    } else {
                        const int dd = (idx - 8) / 8, jc = (idx - 8) % 8;
                        if (idx < kIdChunk)
                            tma_load_4d(dst, &tmG, &raw_full[rs], w0 - 8, h0 - R, (1 + dd) * C + jc * 8, b);
                        else
                            tma_load_4d(dst, &tmI, &raw_full[rs], w0, h0, (idx - kIdChunk) * 32, b);
                    }
                    issued = i + 1;
                }
            }
            int never = 0;
            for (int i = issued > kRawStages ? issued - kRawStages : 0; i < issued; ++i)
                mbar_wait(&raw_full[i % kRawStages], (i / kRawStages) & 1, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- workers
        const int et = threadIdx.x - 64;
        const int q = warp & 3, hc = (warp - 2) >> 2;   // lane quadrant, channel half [32 hc, 32 hc + 32)
        const int s = q * 32 + lane;                    // slot == TMEM lane
        const int r = s >> 3, c = s & 7;
        uint8_t* ywp = sm + kYW;
        uint8_t* gwp = sm + kGW;
        const int rplane = P.WH * kRawCols;             // elements per channel of a raw chunk
        bool ok = true;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            const int t = blockIdx.x + tl * gridDim.x;
            const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
            const int h0 = (ti / P.tiles_w) * kDxTH, w0 = (ti % P.tiles_w) * kDxTW;
            // y window: [chunk][position][8 channels] from the raw chunks (zero outside the image / beyond C)
            if (!mbar_wait(&yw_empty, (tl & 1) ^ 1, P.err, abort_v)) break;
            for (int jc = 0; jc < 8 && ok; ++jc) {
                const int i = tl * kChunks + jc, rs = i % kRawStages;
                if (!mbar_wait(&raw_full[rs], (i / kRawStages) & 1, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                const unsigned short* raw = reinterpret_cast<const unsigned short*>(sm + kRaw + rs * kRawStage);
                uint32_t pk[kPosPerThread][4];
                gather_positions(pk, raw, et, npos, WW, R, rplane);
#pragma unroll
                for (int u = 0; u < kPosPerThread; ++u) {
                    const int pos = et + u * 32 * kWorkWarps;
                    if (pos < npos)
                        *reinterpret_cast<uint4*>(ywp + (jc * npos + pos) * 16) =
                            make_uint4(pk[u][0], pk[u][1], pk[u][2], pk[u][3]);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[rs]);
            }
            if (!ok) break;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&yw_full);

            // dx = grad (channel block 0) + the gathered sum; the identity term arrives as the
            // tile's last two raw chunks
            const int h = h0 + r, w = w0 + c;
            const bool inside = h < H && w < W;
            const long long pix = inside ? (long long)h * W + w : 0;
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            for (int dd = 0; dd < 3 && ok; ++dd) {
                const int dil = dil_of(P.d, dd);
                // grad window of dilation dd: [position][64 channels] bf16, 16-byte chunks rotated by position
                work_bar();
                for (int jc = 0; jc < 8 && ok; ++jc) {
                    const int i = tl * kChunks + 8 + dd * 8 + jc, rs = i % kRawStages;
                    if (!mbar_wait(&raw_full[rs], (i / kRawStages) & 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    const unsigned short* raw = reinterpret_cast<const unsigned short*>(sm + kRaw + rs * kRawStage);
                    uint32_t pk[kPosPerThread][4];
                    gather_positions(pk, raw, et, npos, WW, R, rplane);
#pragma unroll
                    for (int u = 0; u < kPosPerThread; ++u) {
                        const int pos = et + u * 32 * kWorkWarps;
                        if (pos < npos)
                            *reinterpret_cast<uint4*>(gwp + pos * 128 + ((jc ^ (pos & 7)) << 4)) =
                                make_uint4(pk[u][0], pk[u][1], pk[u][2], pk[u][3]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&raw_empty[rs]);
                }
                if (!ok) break;
                work_bar();
                for (int k = 0; k < 9; ++k) {
                    const int i = tl * kTaps + dd * 9 + k, buf = i % kDBufs;
                    if (!mbar_wait(&d_full[buf], (i / kDBufs) & 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t v[32];
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * kN + hc * 32;
                    DDPM_TMEM_LD_X16(ta, (v + 0));
                    DDPM_TMEM_LD_X16(ta + 16, (v + 16));
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&d_empty[buf]);
                    const int ky = k / 3, kx = k - ky * 3;
                    const int pos = (r + R - (ky - 1) * dil) * WW + (c + R - (kx - 1) * dil);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint4 gv = *reinterpret_cast<const uint4*>(gwp + pos * 128 + (((4 * hc + e) ^ (pos & 7)) << 4));
                        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            // the tap rounded to bf16, times grad: exact product, FP32 accumulate
                            const int ci = e * 8 + 2 * f;
                            fma2_bf16_f32(acc[ci], acc[ci + 1],
                                          pack_bf16x2(__uint_as_float(v[ci]), __uint_as_float(v[ci + 1])), gw[f]);
                        }
                    }
                }
            }
            if (!ok) break;
            // the identity term: chunk kIdChunk + hc holds this thread's 32 channels, [ch][row][col]
            for (int j = 0; j < 2 && ok; ++j) {
                const int i = tl * kChunks + kIdChunk + j, rs = i % kRawStages;
                if (!mbar_wait(&raw_full[rs], (i / kRawStages) & 1, P.err, abort_v)) ok = false;
            }
            if (!ok) break;
            {
                const unsigned short* id = reinterpret_cast<const unsigned short*>(
                    sm + kRaw + ((tl * kChunks + kIdChunk + hc) % kRawStages) * kRawStage);
                bf16* dxp = P.dx + (long long)b * C * HW + pix;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int ch = hc * 32 + i;
                    const float g0 = __uint_as_float((uint32_t)id[(i * kDxTH + r) * kDxTW + c] << 16);
                    if (inside && ch < C) dxp[(long long)ch * HW] = __float2bfloat16_rn(g0 + acc[i]);
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int j = 0; j < 2; ++j) mbar_arrive(&raw_empty[(tl * kChunks + kIdChunk + j) % kRawStages]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

bool bwd_dx_tc_eligible(const Dims& d, const void* g, const void* y, const void* w) {
    return bwdtc::eligible(d, g, y, w) && d.R() <= kDxMaxR;
}

cudaError_t launch_bwd_dx_tc(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                             cudaStream_t s) {
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dx_tc_kernel, kSmemBytes, attr_done);
        if (e != cudaSuccess) return e;
    }
    DxTcParams P;
    P.d = d;
    P.tiles_w = (d.W + kDxTW - 1) / kDxTW;
    P.tiles_per_img = ((d.H + kDxTH - 1) / kDxTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.R = d.R();
    P.WH = kDxTH + 2 * P.R;
    P.WW = kDxTW + 2 * P.R;
    P.npos = P.WH * P.WW;
    P.y = static_cast<const bf16*>(y);
    P.g = static_cast<const bf16*>(g);
    P.bias = static_cast<const bf16*>(bias);
    P.dx = static_cast<bf16*>(dx);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    CUtensorMap tmW;
    {
        // W viewed as [3C (dc)][9 (k)][C (j)]: box {64 j, 1 k, 64 dc} = rows (d*C + c, k) for 64 channels
        const cuuint64_t dims[3] = {(cuuint64_t)d.C, 9, (cuuint64_t)(3 * d.C)};
        const cuuint64_t str[2] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.C * 9 * 2};
        const cuuint32_t box[3] = {64, 1, 64};
        const cuuint32_t es[3] = {1, 1, 1};
        if (encode_fn()(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, str, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    CUtensorMap tmY, tmG, tmI;
    if (!encode_nchw(&tmY, y, d, d.C, kRawCols, (uint32_t)P.WH, 8, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_nchw(&tmG, g, d, 4 * d.C, kRawCols, (uint32_t)P.WH, 8, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_nchw(&tmI, g, d, 4 * d.C, kDxTW, kDxTH, 32, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    int grid = num_sms();
    if (grid > P.n_tiles) grid = P.n_tiles;
    trace_begin(s, kKBwdDxTc);
    bwd_dx_tc_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmW, tmY, tmG, tmI, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace ddpm
