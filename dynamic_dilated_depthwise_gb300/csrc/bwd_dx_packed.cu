// bwd_dx_packed.cu -- dX on tcgen05 tensor cores from channel-chunked copies of y and grad (bf16).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dX recomputes the dynamic taps and gathers each dilation's contribution:
//   dx[b,c,q] = grad[b,c,q] + sum_{d,ky,kx} Tq[b,o,q-off] * grad[b,(1+d)C+c,q-off],
//   Tq = bf16(bias[o] + sum_j W[o,j] y[b,j,q-off]),  o = (d*C + c)*9 + ky*3 + kx.
//
// Two launches.
// pack_chunks: y and the three dilation blocks of grad are copied once into a
//   channel-chunked layout [B][group][C/8][H][W][8] -- the eight channels of a
//   chunk at one pixel in 16 contiguous bytes.  An HBM-bound transposition.
// bwd_dx_tc_packed: one shifted GEMM per tap.  A CTA owns a 16x8 pixel tile (MMA
//   M = 128, slot s = r*8 + c) and all channels (N = 64):
//   - TMA brings the tile's y window [chunk][(16+2R) x (8+2R) positions][8] from the
//     packed copy as it is (one contiguous run per window row and chunk); eight consecutive slots are eight consecutive positions
//     of one window row, so the A operand of tap (ky, kx) is the window at a start
//     offset (K-major, no swizzle, row-group stride WW*16 bytes);
//   - TMA brings each dilation's grad window [chunk][(16+2d) x (8+2d)][8] into a
//     buffer of its own, reloaded for the next tile as soon as the tile's nine taps
//     of that dilation are gathered, so the load overlaps the other dilations;
//   - W rows of one tap for all channels stream through a ring (3-D view of W) fed by
//     a producer warp of its own, so the window loads never queue behind W stages;
//   - the bias is a last K=16 step: A is a one-hot row selecting tap k (the same
//     eight rows for every slot group: row-group stride 0), B a resident table of
//     bias[d, c, k];
//   - two threads in different warps issue the MMAs, even and odd taps: tcgen05.mma
//     issue waits for the tensor pipe to accept the instruction, so one thread's waits
//     and bookkeeping between taps would leave the pipe idle; the other thread's taps
//     fill those gaps (each thread commits its own MMAs);
//   - D of each tap lands in one of eight TMEM buffers [128 x 64]; eight worker
//     warps round it to bf16 and accumulate tap * grad in FP32 with one
//     mixed-precision FMA per channel (bf16 operands, exact product).
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using namespace bwdtc;

constexpr int kPTH = 16, kPTW = 8;         // pixel tile
constexpr int kPN = 64;                    // MMA N: channels (zero padded beyond C)
constexpr int kPTaps = 27;
constexpr int kPWork = 8;                  // worker warps
constexpr int kPIssuers = 2;               // MMA-issuing threads (warp 1 and the last warp), alternate taps
constexpr int kPIssuer2 = 2 + kPWork;      // warp of the second issuer
constexpr int kPWProd = 3 + kPWork;        // warp of the W-ring producer
constexpr int kPThreads = 32 * (4 + kPWork);
constexpr int kPDBufs = 8;                 // TMEM accumulators of 64 columns
constexpr int kPMaxStages = 8;             // W ring depth cap
constexpr int kPMinStages = 2;
constexpr int kPMaxR = 6;
constexpr int kPWTile = 8192;              // W rows of one tap: [64 c][64 j] bf16, SW128
constexpr int kPOneHot = 9 * 256;          // one-hot A rows, 9 taps x 2 chunks x 8 rows x 16 B
constexpr int kPBiasTab = 3 * 2048;        // bias B tiles, 3 dilations x [64 c][16 k] bf16
constexpr int kPSmemCap = 227 * 1024 - 1024;   // shared memory one block may use, less the static barriers
constexpr int kPackThreads = 256;

struct DxPackedParams {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int R, WW, WH, npos, nch, nks, stages;
    int wwd[3], npd[3];
    int oyw, ogw[3], ooh, obt;             // shared-memory offsets from the aligned base
    const bf16* g;                         // grad, NCHW (block 0 gives the identity term)
    const bf16* bias;                      // may be null
    bf16* dx;
    unsigned int* err;
};

// Shared-memory plan for a problem; stages == 0 when it does not fit.
struct DxPackedLayout {
    int stages, oyw, ogw[3], ooh, obt, bytes;
};

DxPackedLayout dx_packed_layout(const Dims& d) {
    DxPackedLayout L{};
    const int R = d.R();
    const int npos = (kPTH + 2 * R) * (kPTW + 2 * R);
    int gsz[3], rest = 8 * npos * 16;
    for (int dd = 0; dd < 3; ++dd) {
        const int dil = dil_of(d, dd);
        gsz[dd] = 8 * (kPTH + 2 * dil) * (kPTW + 2 * dil) * 16;
        rest += gsz[dd];
    }
    rest += kPOneHot + kPBiasTab;
    int stages = (kPSmemCap - 1024 - rest) / kPWTile;
    if (stages > kPMaxStages) stages = kPMaxStages;
    // an even number of stages: tap i uses stage i % stages, so every use of a stage falls
    // to the same issuer (taps alternate between the two) and its phase waits stay in order
    stages &= ~1;
    if (stages < kPMinStages || R > kPMaxR) return L;
    L.stages = stages;
    L.oyw = stages * kPWTile;
    L.ogw[0] = L.oyw + 8 * npos * 16;
    L.ogw[1] = L.ogw[0] + gsz[0];
    L.ogw[2] = L.ogw[1] + gsz[1];
    L.ooh = L.ogw[2] + gsz[2];
    L.obt = L.ooh + kPOneHot;
    L.bytes = L.obt + kPBiasTab + 1024;
    return L;
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

// ----------------------------------------------------------------------------- pack
// Thread = (tensor, b, group, chunk, 8-pixel run): eight 16-byte channel rows in,
// eight 16-byte pixel rows out.  HW is a multiple of 8 (W is).  Run idx (y runs
// first, then the grad runs) lands at bytes [128 idx, 128 idx + 128) of the packed
// buffer (gc follows yc), so the 256 runs of a block fill one contiguous 32 KiB range:
// the block transposes through shared memory and writes that range with 512-byte
// warp stores instead of 16-byte pieces 128 bytes apart.
__global__ void __launch_bounds__(kPackThreads, 2)
    pack_chunks_kernel(const bf16* __restrict__ y, const bf16* __restrict__ g, bf16* __restrict__ yc,
                       int B, int C, long long HW, long long n_y, long long n_all) {
    // [run][8 pixel rows of 16 B], pixel row p of run r at column p ^ (r & 7)
    __shared__ uint4 stage[kPackThreads * 8];
    const int nch = C / 8;
    const long long runs = HW / 8;
    const int tid = threadIdx.x;
    uint4* out = reinterpret_cast<uint4*>(yc);
    for (long long r0 = (long long)blockIdx.x * kPackThreads; r0 < n_all; r0 += (long long)gridDim.x * kPackThreads) {
        const long long idx = r0 + tid;
        if (idx < n_all) {
            const bf16* src;
            if (idx < n_y) {
                const long long o = idx % runs, bc = idx / runs;   // bc = b * nch + cb
                const long long b = bc / nch, cb = bc % nch;
                src = y + (b * C + cb * 8) * HW + o * 8;
            } else {
                const long long j = idx - n_y;
                const long long o = j % runs, bgc = j / runs;      // bgc = (b * 3 + grp) * nch + cb
                const long long cb = bgc % nch, bg = bgc / nch;
                const long long b = bg / 3, grp = bg % 3;
                src = g + (b * 4 * C + C + grp * C + cb * 8) * HW + o * 8;
            }
            uint4 in[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) in[e] = __ldg(reinterpret_cast<const uint4*>(src + e * HW));
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                const uint32_t sel = (p & 1) ? 0x7632u : 0x5410u;
                uint32_t w[4];
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const uint4 a = in[2 * f], b = in[2 * f + 1];
                    const uint32_t aw = (p >> 1) == 0 ? a.x : (p >> 1) == 1 ? a.y : (p >> 1) == 2 ? a.z : a.w;
                    const uint32_t bw = (p >> 1) == 0 ? b.x : (p >> 1) == 1 ? b.y : (p >> 1) == 2 ? b.z : b.w;
                    w[f] = __byte_perm(aw, bw, sel);
                }
                stage[tid * 8 + (p ^ (tid & 7))] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        __syncthreads();
        // copy out: 16-byte piece k of the block's range is pixel row (k & 7) of run k >> 3
        const long long n_pieces = (n_all - r0 < kPackThreads ? n_all - r0 : kPackThreads) * 8;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = i * kPackThreads + tid;
            if (k < n_pieces) {
                const int r = k >> 3, pr = k & 7;
                out[r0 * 8 + k] = stage[r * 8 + (pr ^ (r & 7))];
            }
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------- pack (TMA)
// Persistent variant for H*W a multiple of 2048, on half of the SMs: the pack is
// bound by HBM, not by SMs, and the SMs it leaves free run the dY and dW kernels
// that start beside it.  Unit = 2048 pixels of one chunk (eight channel rows of
// 4 KiB): eight untiled bulk copies bring it into a 4-stage ring; 256 threads each
// transpose one 8-pixel run into a 128B-swizzled staging block (conflict-free
// writes), and one 2-D tensor store with the same swizzle writes the unit's
// contiguous 32 KiB of output (runs are rows of 64 bf16 in the packed buffer).
constexpr int kPkWorkers = 256;
constexpr int kPkThreads = kPkWorkers + 32;   // + a producer warp
constexpr int kPkPx = 8 * kPkWorkers;         // 2048 pixels per unit
constexpr int kPkStages = 4;
constexpr int kPkRow = kPkPx * 2;             // 4 KiB: one channel row of a unit
constexpr int kPkIn = 8 * kPkRow;             // 32 KiB
constexpr int kPkOut = kPkWorkers * 128;      // 32 KiB
constexpr int kPkSmem = kPkStages * kPkIn + 2 * kPkOut + 1024;

struct PackParams {
    const bf16* y;
    const bf16* g;
    int C, nch;
    long long HW;
    int units_per_chunk;   // HW / 2048
    int n_ychunks;         // B * nch: y chunks come first, then the 3 * B * nch grad chunks
    int n_units;
    unsigned int* err;
};

__global__ void __launch_bounds__(kPkThreads, 1)
    pack_chunks_tma_kernel(const __grid_constant__ CUtensorMap tmOut, const PackParams P) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t full[kPkStages], empty[kPkStages];
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_my = blockIdx.x < P.n_units ? (P.n_units - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < kPkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPkWorkers / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == kPkWorkers / 32) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < n_my; ++i) {
                const int s = i % kPkStages, ph = (i / kPkStages) & 1;
                if (!mbar_wait(&empty[s], ph ^ 1, P.err, abort_v)) break;
                const int u = blockIdx.x + i * gridDim.x;
                const int chunk = u / P.units_per_chunk;
                const long long px0 = (long long)(u % P.units_per_chunk) * kPkPx;
                const bf16* src;
                if (chunk < P.n_ychunks) {
                    const int b = chunk / P.nch, cb = chunk % P.nch;
                    src = P.y + ((long long)b * P.C + cb * 8) * P.HW + px0;
                } else {
                    const int j = chunk - P.n_ychunks;   // (b * 3 + grp) * nch + cb
                    const int cb = j % P.nch, bg = j / P.nch, b = bg / 3, grp = bg % 3;
                    src = P.g + ((long long)b * 4 * P.C + P.C + (long long)grp * P.C + cb * 8) * P.HW + px0;
                }
                uint8_t* dst = sm + s * kPkIn;
                mbar_arrive_expect_tx(&full[s], kPkIn);
                for (int e = 0; e < 8; ++e) bulk_load(dst + e * kPkRow, src + e * P.HW, kPkRow, &full[s]);
                issued = i + 1;
            }
            // drain: every copy this thread started lands before its shared memory is released
            int never = 0;
            for (int i = issued > kPkStages ? issued - kPkStages : 0; i < issued; ++i)
                mbar_wait(&full[i % kPkStages], (i / kPkStages) & 1, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- workers: run tid of each unit
        uint8_t* const out0 = sm + kPkStages * kPkIn;
        bool ok = true;
        for (int i = 0; i < n_my; ++i) {
            const int s = i % kPkStages, ph = (i / kPkStages) & 1, ob = i & 1;
            if (ok) ok = mbar_wait(&full[s], ph, P.err, abort_v);
            // staging block ob was last read by the store of unit i - 2
            if (tid == 0) bulk_wait_read<1>();
            asm volatile("bar.sync 1, %0;" ::"n"(kPkWorkers) : "memory");
            if (ok) {
                const uint8_t* in = sm + s * kPkIn + tid * 16;
                uint4 q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) q[e] = *reinterpret_cast<const uint4*>(in + e * kPkRow);
                uint8_t* out = out0 + ob * kPkOut + tid * 128;
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const uint32_t sel = (p & 1) ? 0x7632u : 0x5410u;
                    uint32_t w[4];
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const uint4 a = q[2 * f], b = q[2 * f + 1];
                        const uint32_t aw = (p >> 1) == 0 ? a.x : (p >> 1) == 1 ? a.y : (p >> 1) == 2 ? a.z : a.w;
                        const uint32_t bw = (p >> 1) == 0 ? b.x : (p >> 1) == 1 ? b.y : (p >> 1) == 2 ? b.z : b.w;
                        w[f] = __byte_perm(aw, bw, sel);
                    }
                    *reinterpret_cast<uint4*>(out + ((p ^ (tid & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            fence_proxy_async_smem();
            asm volatile("bar.sync 1, %0;" ::"n"(kPkWorkers) : "memory");
            if (tid == 0 && ok) {
                const int u = blockIdx.x + i * gridDim.x;
                const int chunk = u / P.units_per_chunk, blk = u % P.units_per_chunk;
                const int row0 = (int)((long long)chunk * (P.HW / 8) + (long long)blk * kPkWorkers);
                tma_store_2d(&tmOut, out0 + ob * kPkOut, 0, row0);
                bulk_commit();
            }
        }
        // every store has written global memory before the kernel ends
        if (tid == 0) bulk_wait<0>();
    }
}

// ----------------------------------------------------------------------------- dX
__global__ void __launch_bounds__(kPThreads, 1)
    bwd_dx_tc_packed_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
                            const __grid_constant__ CUtensorMap tmG0, const __grid_constant__ CUtensorMap tmG1,
                            const __grid_constant__ CUtensorMap tmG2, const DxPackedParams P) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base, derived by pointer arithmetic on the shared array so that every
    // access through it stays a shared-memory access (an integer round trip would make
    // them generic loads and stores with 64-bit addresses)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t wt_full[kPMaxStages], wt_empty[kPMaxStages], d_full[kPDBufs], d_empty[kPDBufs];
    __shared__ uint64_t yw_full, yw_empty, gw_full[3], gw_empty[3], mma_done[kPIssuers];
    __shared__ uint32_t tmem_slot;
    __shared__ uint32_t a_shift[kPTaps];   // per-tap start offset of the A operand in the y window, bytes
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.d.C, H = P.d.H, W = P.d.W;
    const long long HW = P.d.HW;
    const int n_my = blockIdx.x < P.n_tiles ? (P.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int S = P.stages, R = P.R;

    if (threadIdx.x < kPTaps) {
        // tap (ky, kx) of dilation d reads y at q - ((ky-1) d, (kx-1) d): window position (r + R - (ky-1) d, c + R - (kx-1) d)
        const int u = threadIdx.x, dil = dil_of(P.d, u / 9), ky = (u % 9) / 3, kx = u % 3;
        a_shift[u] = (uint32_t)((R - (ky - 1) * dil) * P.WW + (R - (kx - 1) * dil)) * 16;
    }

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < S; ++i) {
            mbar_init(&wt_full[i], 1);
            mbar_init(&wt_empty[i], 1);
        }
        for (int i = 0; i < kPDBufs; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kPWork);
        }
        mbar_init(&yw_full, 1);
        mbar_init(&yw_empty, kPIssuers);   // each issuer commits once per tile
        for (int i = 0; i < 3; ++i) {
            mbar_init(&gw_full[i], 1);
            mbar_init(&gw_empty[i], kPWork);
        }
        for (int i = 0; i < kPIssuers; ++i) mbar_init(&mma_done[i], 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    if (warp >= 2 && warp < 2 + kPWork) {
        // constant operands: one-hot tap selectors, bias tables, zero chunks of the y window
        const int et = threadIdx.x - 64, nt = 32 * kPWork;
        unsigned short* oh = reinterpret_cast<unsigned short*>(sm + P.ooh);
        for (int i = et; i < kPOneHot / 2; i += nt) {       // [tap k][chunk kc][row][e]
            const int k = i >> 7, kc = (i >> 6) & 1, e = i & 7;
            oh[i] = (kc * 8 + e == k) ? (unsigned short)0x3F80u : (unsigned short)0u;
        }
        // bias table [d][c/8][chunk kc][c%8][e], k = kc*8 + e: one thread per (d, c) loads the
        // channel's nine taps (independent loads, one latency) and writes its two 16-byte chunks
        for (int i = et; i < 3 * 64; i += nt) {
            const int dd = i >> 6, c = i & 63;
            uint32_t v[5] = {0u, 0u, 0u, 0u, 0u};
            if (P.bias != nullptr && c < C) {
                const unsigned short* bp = reinterpret_cast<const unsigned short*>(P.bias) + ((long long)dd * C + c) * 9;
                unsigned short b[9];
#pragma unroll
                for (int k = 0; k < 9; ++k) b[k] = bp[k];
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] = (uint32_t)b[2 * k] | ((uint32_t)b[2 * k + 1] << 16);
                v[4] = b[8];
            }
            uint8_t* ch = sm + P.obt + (dd * 1024 + (c >> 3) * 128 + (c & 7) * 8) * 2;
            *reinterpret_cast<uint4*>(ch) = make_uint4(v[0], v[1], v[2], v[3]);
            *reinterpret_cast<uint4*>(ch + 128) = make_uint4(v[4], 0u, 0u, 0u);
        }
        const int nzero = (2 * P.nks - P.nch) * P.npos;     // chunk nch when C/8 is odd
        for (int i = et; i < nzero; i += nt)
            *reinterpret_cast<uint4*>(sm + P.oyw + ((long long)P.nch * P.npos + i) * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer: y window, grad windows
        // Per tile the dilation-0 grad window goes first: its buffer is free a third of
        // the way into the previous tile, while the y window waits for that tile's last MMA.
        if (lane == 0) {
            prefetch_tmap(&tmY);
            prefetch_tmap(&tmG0);
            prefetch_tmap(&tmG1);
            prefetch_tmap(&tmG2);
            const CUtensorMap* tmg[3] = {&tmG0, &tmG1, &tmG2};
            const uint32_t ybytes = (uint32_t)P.nch * P.npos * 16;
            int ny = 0, ng[3] = {0, 0, 0};
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                const int t = blockIdx.x + tl * gridDim.x;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kPTH, w0 = (ti % P.tiles_w) * kPTW;
                for (int step = 0; step < 4 && ok; ++step) {
                    if (step == 1) {
                        if (!mbar_wait(&yw_empty, (tl & 1) ^ 1, P.err, abort_v)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&yw_full, ybytes);
                        tma_load_4d(sm + P.oyw, &tmY, &yw_full, (w0 - R) * 8, h0 - R, 0, b);
                        ny = tl + 1;
                        continue;
                    }
                    const int dd = step == 0 ? 0 : step - 1;
                    const int dil = dil_of(P.d, dd);
                    if (!mbar_wait(&gw_empty[dd], (tl & 1) ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&gw_full[dd], (uint32_t)P.nch * P.npd[dd] * 16);
                    tma_load_4d(sm + P.ogw[dd], tmg[dd], &gw_full[dd], (w0 - dil) * 8, h0 - dil, dd * P.nch, b);
                    ng[dd] = tl + 1;
                }
            }
            // drain: every copy this thread started lands before its shared memory is released
            int never = 0;
            if (ny > 0) mbar_wait(&yw_full, (ny - 1) & 1, P.err, &never);
            for (int dd = 0; dd < 3; ++dd)
                if (ng[dd] > 0) mbar_wait(&gw_full[dd], (ng[dd] - 1) & 1, P.err, &never);
        }
    } else if (warp == kPWProd) {
        // ------------------------------------------------------- TMA producer: W ring, one tap per stage
        if (lane == 0) {
            prefetch_tmap(&tmW);
            int iw = 0;
            int st = 0, sph = 0;                       // W ring stage and its phase parity
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl)
                for (int u = 0; u < kPTaps; ++u) {
                    const int dd = u / 9, k = u - dd * 9;
                    if (!mbar_wait(&wt_empty[st], sph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&wt_full[st], kPWTile);
                    tma_load_3d(sm + st * kPWTile, &tmW, &wt_full[st], 0, k, dd * C);
                    ++iw;
                    if (++st == S) {
                        st = 0;
                        sph ^= 1;
                    }
                }
            int never = 0;
            for (int i = iw > S ? iw - S : 0; i < iw; ++i) mbar_wait(&wt_full[i % S], (i / S) & 1, P.err, &never);
        }
    } else if (warp == 1 || warp == kPIssuer2) {
        // ------------------------------------------------------- MMA issuers: taps of parity `par`
        // An issuing thread spends tens of cycles on every instruction between two MMAs, so
        // the loop keeps them few: stage, buffer and tap advance by counters (no division),
        // the descriptors are built once and each MMA adds a 32-bit offset to the low half
        // of one, and the K steps of a tap are one unrolled burst.
        const int par = warp == 1 ? 0 : 1;
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(1, 0, 0, 128, kPN);
            const uint32_t lbo_y = (uint32_t)P.npos * 16, sbo_y = (uint32_t)P.WW * 16;
            const uint64_t a_base = smem_desc(smem_u32(sm + P.oyw), lbo_y, sbo_y, kSwizzleNone);
            const uint64_t w_base = smem_desc(smem_u32(sm), 16, 1024, kSwizzle128B);
            const uint64_t oh_base = smem_desc(smem_u32(sm + P.ooh), 128, 0, kSwizzleNone);
            const uint64_t bt_base = smem_desc(smem_u32(sm + P.obt), 128, 256, kSwizzleNone);
            const uint32_t a_hi = (uint32_t)(a_base >> 32), w_hi = (uint32_t)(w_base >> 32);
            const uint32_t oh_hi = (uint32_t)(oh_base >> 32), bt_hi = (uint32_t)(bt_base >> 32);
            const uint32_t astep = (2 * lbo_y) >> 4;              // one K step of A, descriptor units
            const int nks = P.nks;
            const bool full_k = nks == 4;
            int st = par, sph = 0;            // W ring stage of this issuer's next tap and its phase
            int buf = par, bph = 0;           // TMEM buffer of this issuer's next tap and its phase
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                if (!mbar_wait(&yw_full, tl & 1, P.err, abort_v)) break;
                tc_fence_after();
                // the first tap of tile tl for this issuer: (27 tl + u) % 2 == par
                int u = par ^ (tl & 1), dd = 0, k = u;
                for (; u < kPTaps; u += 2) {
                    const uint32_t a_lo = (uint32_t)a_base + (a_shift[u] >> 4);
                    const uint32_t w_lo = (uint32_t)w_base + (uint32_t)((st * kPWTile) >> 4);
                    const uint32_t oh_lo = (uint32_t)oh_base + (uint32_t)(k * 16);
                    const uint32_t bt_lo = (uint32_t)bt_base + (uint32_t)(dd * 128);
                    const uint32_t dt = tmem + (uint32_t)(buf * kPN);
                    if (!mbar_wait(&wt_full[st], sph, P.err, abort_v) ||
                        !mbar_wait(&d_empty[buf], bph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (full_k) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f16_lh(dt, a_lo + kk * astep, a_hi, w_lo + (uint32_t)(kk * 2), w_hi, idesc,
                                       kk > 0 ? 1u : 0u);
                    } else {
                        for (int kk = 0; kk < nks; ++kk)
                            mma_f16_lh(dt, a_lo + kk * astep, a_hi, w_lo + (uint32_t)(kk * 2), w_hi, idesc,
                                       kk > 0 ? 1u : 0u);
                    }
                    mma_f16_lh(dt, oh_lo, oh_hi, bt_lo, bt_hi, idesc, 1u);
                    mma_commit(&d_full[buf]);
                    mma_commit(&wt_empty[st]);
                    st += 2;
                    if (st >= S) {
                        st -= S;
                        sph ^= 1;
                    }
                    buf += 2;
                    if (buf >= kPDBufs) {
                        buf -= kPDBufs;
                        bph ^= 1;
                    }
                    k += 2;
                    if (k >= 9) {
                        k -= 9;
                        ++dd;
                    }
                }
                if (ok) mma_commit(&yw_empty);
            }
            // every MMA this thread issued retires before TMEM is released
            mma_commit(&mma_done[par]);
            int never = 0;
            mbar_wait(&mma_done[par], 0, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- workers: round, gather, accumulate
        const int q = warp & 3, hc = (warp - 2) >> 2;   // lane quadrant, channel half [32 hc, 32 hc + 32)
        const int s = q * 32 + lane;                    // slot == TMEM lane
        const int r = s >> 3, c = s & 7;
        bool ok = true;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            const int t = blockIdx.x + tl * gridDim.x;
            const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
            const int h0 = (ti / P.tiles_w) * kPTH, w0 = (ti % P.tiles_w) * kPTW;
            // dx = grad (channel block 0) + the gathered sum.  The identity term is only
            // prefetched into L2 here and loaded after the gather: a load still in flight
            // would hold up the next mbarrier wait (its acquire orders it after the load),
            // stalling the workers at the start of every tile.  Addresses are clamped into
            // the tensor (validity is applied at the store).
            const int h = h0 + r, w = w0 + c;
            const bool inside = h < H && w < W;
            const long long pix = inside ? (long long)h * W + w : 0;
            const unsigned short* g0p = reinterpret_cast<const unsigned short*>(P.g) + (long long)b * 4 * C * HW + pix;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(g0p + (long long)min(hc * 32 + i, C - 1) * HW));
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            for (int dd = 0; dd < 3 && ok; ++dd) {
                const int dil = dil_of(P.d, dd), wwd = P.wwd[dd];
                const uint8_t* gw = sm + P.ogw[dd] + (4 * hc) * P.npd[dd] * 16;
                const int cstride = P.npd[dd] * 16;
                if (!mbar_wait(&gw_full[dd], tl & 1, P.err, abort_v)) {
                    ok = false;
                    break;
                }
                for (int k = 0; k < 9; ++k) {
                    const int i = tl * kPTaps + dd * 9 + k, buf = i % kPDBufs;
                    if (!mbar_wait(&d_full[buf], (i / kPDBufs) & 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t v[32];
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * kPN + hc * 32;
                    DDPM_TMEM_LD_X16(ta, (v + 0));
                    DDPM_TMEM_LD_X16(ta + 16, (v + 16));
                    const int ky = k / 3, kx = k - ky * 3;
                    const int pos = (r + dil - (ky - 1) * dil) * wwd + (c + dil - (kx - 1) * dil);
                    uint4 gv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) gv[e] = *reinterpret_cast<const uint4*>(gw + e * cstride + pos * 16);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&d_empty[buf]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t gw4[4] = {gv[e].x, gv[e].y, gv[e].z, gv[e].w};
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            const int ci = e * 8 + 2 * f;
                            const uint32_t t2 = pack_bf16x2(__uint_as_float(v[ci]), __uint_as_float(v[ci + 1]));
                            fma2_bf16_f32(acc[ci], acc[ci + 1], t2, gw4[f]);
                        }
                    }
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&gw_empty[dd]);
            }
            if (!ok) break;
            unsigned short g0raw[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) g0raw[i] = __ldg(g0p + (long long)min(hc * 32 + i, C - 1) * HW);
            if (inside) {
                bf16* dxp = P.dx + (long long)b * C * HW + pix;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int ch = hc * 32 + i;
                    if (ch < C) dxp[(long long)ch * HW] = __float2bfloat16_rn(__uint_as_float((uint32_t)g0raw[i] << 16) + acc[i]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// 4-D view of a packed tensor [B][nchunks][H][W][8] bf16 whose innermost dimension is a
// whole row, W*8 elements: a window of bw positions is one contiguous run of bw*16
// bytes per (row, chunk) -- one TMA request instead of bw 16-byte ones -- and
// positions left or right of the image (x < 0 or x >= W*8) still read as zeros.
bool encode_packed(CUtensorMap* m, const void* base, const Dims& d, int nchunks, uint32_t bw, uint32_t bh,
                   uint32_t bc) {
    const cuuint64_t dims[4] = {(cuuint64_t)d.W * 8, (cuuint64_t)d.H, (cuuint64_t)nchunks, (cuuint64_t)d.B};
    const cuuint64_t str[3] = {(cuuint64_t)d.W * 16, (cuuint64_t)d.HW * 16, (cuuint64_t)d.HW * 16 * nchunks};
    const cuuint32_t box[4] = {bw * 8, bh, bc, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return bw * 8 <= 256 &&
           encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, str, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool bwd_dx_packed_shape_ok(const Dims& d) { return bwdtc::shape_ok(d) && dx_packed_layout(d).stages > 0; }

bool bwd_dx_packed_eligible(const Dims& d, const void* g, const void* y, const void* w) {
    return bwdtc::eligible(d, g, y, w) && dx_packed_layout(d).stages > 0;
}

size_t bwd_dx_packed_bytes(const Dims& d) { return (size_t)4 * (size_t)d.B * (size_t)d.C * (size_t)d.HW * 2; }

cudaError_t launch_pack_chunks(const Dims& d, const void* g, const void* y, void* packed, cudaStream_t s) {
    bf16* yc = static_cast<bf16*>(packed);
    const int nch = d.C / 8;
    const long long n_rows = 4LL * d.B * nch * (d.HW / 8);   // 16-byte pixel rows of the copies
    if (d.HW % kPkPx == 0 && n_rows <= INT_MAX && (uintptr_t)y % 16 == 0 && (uintptr_t)g % 16 == 0) {
        static int attr_pk[64] = {};
        {
            const cudaError_t e = set_max_dynamic_smem((const void*)pack_chunks_tma_kernel, kPkSmem, attr_pk);
            if (e != cudaSuccess) return e;
        }
        CUtensorMap tmOut;
        const cuuint64_t dims[2] = {64, (cuuint64_t)n_rows};
        const cuuint64_t str[1] = {128};
        const cuuint32_t box[2] = {64, (cuuint32_t)kPkWorkers};
        const cuuint32_t es[2] = {1, 1};
        if (encode_fn()(&tmOut, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, packed, dims, str, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        PackParams Q;
        Q.y = static_cast<const bf16*>(y);
        Q.g = static_cast<const bf16*>(g);
        Q.C = d.C;
        Q.nch = nch;
        Q.HW = d.HW;
        Q.units_per_chunk = (int)(d.HW / kPkPx);
        Q.n_ychunks = d.B * nch;
        Q.n_units = 4 * d.B * nch * Q.units_per_chunk;
        Q.err = device_error_word();
        if (Q.err == nullptr) return cudaErrorUnknown;
        int grid = num_sms() / 2;
        if (grid < 1) grid = 1;
        if (grid > Q.n_units) grid = Q.n_units;
        trace_begin(s, kKPackChunks);
        pack_chunks_tma_kernel<<<grid, kPkThreads, kPkSmem, s>>>(tmOut, Q);
        trace_end(s);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else {
        const long long runs = d.HW / 8;
        const long long n_y = (long long)d.B * nch * runs;
        const long long n_all = n_y * 4;
        long long blocks = (n_all + kPackThreads - 1) / kPackThreads;
        const long long cap = (long long)num_sms() * 8;
        if (blocks > cap) blocks = cap;
        trace_begin(s, kKPackChunks);
        pack_chunks_kernel<<<(unsigned)blocks, kPackThreads, 0, s>>>(static_cast<const bf16*>(y),
                                                                     static_cast<const bf16*>(g), yc, d.B, d.C, d.HW,
                                                                     n_y, n_all);
        trace_end(s);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    return cudaSuccess;
}

cudaError_t launch_bwd_dx_packed(const Dims& d, const void* g, const void* y, const void* w, const void* bias,
                                 void* dx, void* packed, cudaStream_t s) {
    const DxPackedLayout L = dx_packed_layout(d);
    if (L.stages == 0) return cudaErrorInvalidValue;
    static int attr_bytes[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dx_tc_packed_kernel, L.bytes, attr_bytes);
        if (e != cudaSuccess) return e;
    }
    bf16* yc = static_cast<bf16*>(packed);
    bf16* gc = yc + (size_t)d.B * d.C * d.HW;
    const int nch = d.C / 8;

    // 1. channel-chunked copies of y and of the three dilation blocks of grad
    {
        const cudaError_t e = launch_pack_chunks(d, g, y, packed, s);
        if (e != cudaSuccess) return e;
    }

    // 2. the shifted-GEMM dX
    DxPackedParams P;
    P.d = d;
    P.tiles_w = (d.W + kPTW - 1) / kPTW;
    P.tiles_per_img = ((d.H + kPTH - 1) / kPTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.R = d.R();
    P.WW = kPTW + 2 * P.R;
    P.WH = kPTH + 2 * P.R;
    P.npos = P.WW * P.WH;
    P.nch = nch;
    P.nks = (nch + 1) / 2;
    P.stages = L.stages;
    for (int dd = 0; dd < 3; ++dd) {
        const int dil = dil_of(d, dd);
        P.wwd[dd] = kPTW + 2 * dil;
        P.npd[dd] = P.wwd[dd] * (kPTH + 2 * dil);
        P.ogw[dd] = L.ogw[dd];
    }
    P.oyw = L.oyw;
    P.ooh = L.ooh;
    P.obt = L.obt;
    P.g = static_cast<const bf16*>(g);
    P.bias = static_cast<const bf16*>(bias);
    P.dx = static_cast<bf16*>(dx);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;
    CUtensorMap tmW, tmY, tmG[3];
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
    if (!encode_packed(&tmY, yc, d, nch, (uint32_t)P.WW, (uint32_t)P.WH, (uint32_t)nch)) return cudaErrorInvalidValue;
    for (int dd = 0; dd < 3; ++dd) {
        const int dil = dil_of(d, dd);
        if (!encode_packed(&tmG[dd], gc, d, 3 * nch, (uint32_t)(kPTW + 2 * dil), (uint32_t)(kPTH + 2 * dil),
                           (uint32_t)nch))
            return cudaErrorInvalidValue;
    }
    int grid = num_sms();
    if (grid > P.n_tiles) grid = P.n_tiles;
    trace_begin(s, kKBwdDxTcPacked);
    bwd_dx_tc_packed_kernel<<<grid, kPThreads, L.bytes, s>>>(tmW, tmY, tmG[0], tmG[1], tmG[2], P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace ddpm
