// bwd_dx_tf32.cu -- dX of FP32 problems on TF32 tensor cores (DDPM_FLAG_TF32_BACKWARD).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dX recomputes the dynamic taps and gathers each dilation's contribution,
//   dx[b,c,q] = grad[b,c,q] + sum_{d,ky,kx} T[b,o,q-off] * grad[b,(1+d)C+c,q-off],
//   T = bias[o] + sum_j W[o,j] y[b,j,q-off],  o = (d*C + c)*9 + ky*3 + kx,
// and the section's precision policy lets an FP32 backward run its recompute on TF32
// tensor cores (FP32 accumulation).
//
// Two launches.
// pack_f32: y and the three dilation blocks of grad are copied once into a channel-chunked
//   layout ([B][C/4][H][W][4] and [B][3][C/4][H][W][4]) -- the four channels of a chunk at
//   one pixel in 16 contiguous bytes (HBM-bound).
// bwd_dx_tf32: one shifted TF32 GEMM per tap.  A persistent CTA walks 16x8 pixel tiles
//   (MMA M = 128, slot s = r*8 + c) with all channels (N = 64):
//   - TMA brings the tile's y window [chunk][(16+2R) x (8+2R) positions][4] from the
//     packed copy (one contiguous run per window row and chunk); eight consecutive
//     slots are eight consecutive positions of one window row, so the A operand of tap
//     (ky, kx) is the window at a start offset (K-major, no swizzle, core matrices of
//     8 positions x 4 channels, row-group stride WW*16 bytes);
//   - the W rows of one tap for all channels ([64 c][64 j] fp32, two 128B-swizzled
//     K-atoms) stream through a ring fed by a producer warp of its own;
//   - the bias is two last K=8 steps: A a one-hot row selecting tap k (every row group
//     the same: stride 0), B a resident table of bias[d, c, k];
//   - two threads in different warps issue the MMAs of even and odd taps (an issuing
//     thread waits for the tensor pipe to accept each MMA; the other one fills the gaps);
//   - D of each tap lands in one of eight TMEM buffers [128 x 64]; eight worker warps
//     accumulate tap * grad in IEEE FP32.  Four-byte grad windows of all 64 channels do
//     not fit in shared memory beside the y window, so each worker gathers its grad
//     values from the chunked copy in global memory (L2), two taps ahead of their use:
//     eight 16-byte loads per tap for its pixel's 32 channels.
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

constexpr int kTH = 16, kTW = 8;          // pixel tile
constexpr int kN = 64;                    // MMA N: channels (rows of W beyond C are never read back)
constexpr int kTaps = 27;
constexpr int kWork = 8;                  // worker warps
constexpr int kIssuers = 2;               // MMA-issuing threads (warp 1 and warp kIssuer2), alternate taps
constexpr int kIssuer2 = 2 + kWork;
constexpr int kWProd = 3 + kWork;         // W-ring producer warp
constexpr int kThreads = 32 * (4 + kWork);
constexpr int kDBufs = 8;                 // TMEM accumulators of 64 columns
constexpr int kMaxStages = 8;
constexpr int kMinStages = 2;
constexpr int kMaxR = 6;
constexpr int kWAtom = 64 * 128;          // [64 c][32 j] fp32, SW128
constexpr int kWTile = 2 * kWAtom;        // one tap: j 0..31 and 32..63
constexpr int kOneHot = 9 * 512;          // [tap k][4 K-groups][8 rows][4] fp32
constexpr int kBiasTab = 3 * 4096;        // [d][c/8][k/4][c%8][k%4] fp32
constexpr int kSmemCap = 227 * 1024 - 1024;
constexpr int kPackThreads = 256;

struct DxTf32Params {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int R, WW, WH, npos, nch4, nks, stages;
    int oyw, ooh, obt;                     // shared-memory offsets from the aligned base
    const float* g;                        // grad, NCHW [B][4C][H][W] (block 0 gives the identity term)
    const float4* gc;                      // grad blocks 1..3, chunked [B][3][C/4][H*W] float4
    const float* bias;                     // may be null
    float* dx;
    unsigned int* err;
};

// Shared-memory plan for a problem; stages == 0 when it does not fit.
struct DxTf32Layout {
    int stages, oyw, ooh, obt, bytes;
};

DxTf32Layout dx_tf32_layout(const Dims& d) {
    DxTf32Layout L{};
    const int R = d.R();
    if (R > kMaxR) return L;
    const int npos = (kTH + 2 * R) * (kTW + 2 * R);
    const int nks = (d.C + 7) / 8;
    const int ybytes = 2 * nks * npos * 16;
    const int rest = ybytes + kOneHot + kBiasTab;
    int stages = (kSmemCap - 1024 - rest) / kWTile;
    if (stages > kMaxStages) stages = kMaxStages;
    // an even number of stages: tap i uses stage i % stages and the taps alternate between
    // the two issuers, so every use of a stage falls to the same issuer
    stages &= ~1;
    if (stages < kMinStages) return L;
    L.stages = stages;
    L.oyw = stages * kWTile;
    L.ooh = L.oyw + ybytes;
    L.obt = L.ooh + kOneHot;
    L.bytes = L.obt + kBiasTab + 1024;
    return L;
}

// ----------------------------------------------------------------------------- pack
// Thread = (tensor, b, chunk, 4-pixel group): four 16-byte channel rows in, four 16-byte
// pixel rows out.  Units [0, n_y) copy y ([B][C/4] chunks), the rest the grad channels
// C .. 4C-1 ([B][3C/4] chunks).  HW is a multiple of 4 (W is).
__global__ void __launch_bounds__(kPackThreads)
    pack_f32_kernel(const float* __restrict__ y, const float* __restrict__ g, float* __restrict__ yc,
                    float* __restrict__ gc, int C, long long HW, long long n_y, long long n_all) {
    const long long groups = HW / 4;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < n_all;
         u += (long long)gridDim.x * blockDim.x) {
        const bool is_y = u < n_y;
        const long long v = is_y ? u : u - n_y;
        const int nch4 = is_y ? C / 4 : 3 * C / 4;
        const long long p4 = v % groups, bc = v / groups;   // bc = b * nch4 + cb
        const long long b = bc / nch4, cb = bc % nch4;
        const float* src = is_y ? y + (b * C + cb * 4) * HW + p4 * 4 : g + (b * 4 * C + C + cb * 4) * HW + p4 * 4;
        float4 in[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) in[e] = __ldg(reinterpret_cast<const float4*>(src + e * HW));
        float4* dst = reinterpret_cast<float4*>((is_y ? yc : gc) + (bc * HW + p4 * 4) * 4);
        dst[0] = make_float4(in[0].x, in[1].x, in[2].x, in[3].x);
        dst[1] = make_float4(in[0].y, in[1].y, in[2].y, in[3].y);
        dst[2] = make_float4(in[0].z, in[1].z, in[2].z, in[3].z);
        dst[3] = make_float4(in[0].w, in[1].w, in[2].w, in[3].w);
    }
}

// ----------------------------------------------------------------------------- dX
// The grad values of one tap for this thread's pixel and its 32 channels, from the
// chunked copy gci = [3][C/4][HW] float4 of this image (zero where the source pixel lies
// outside the image or the chunk beyond C).
__device__ __forceinline__ void gather_tap(float4 (&g)[8], const float4* gci, int u, const DxTf32Params& P, int h,
                                           int w, bool inside, int cq0) {
    const int dd = u / 9, k = u - dd * 9;
    const int dil = dil_of(P.d, dd);
    const int sh = h - (k / 3 - 1) * dil, sw = w - (k % 3 - 1) * dil;
    const bool valid = inside && sh >= 0 && sh < P.d.H && sw >= 0 && sw < P.d.W;
    const long long HW = P.d.HW;
    const float4* p = gci + ((long long)dd * P.nch4 + cq0) * HW + (long long)sh * P.d.W + sw;
    const int nq = P.nch4 - cq0;
#pragma unroll
    for (int j = 0; j < 8; ++j) g[j] = (valid && j < nq) ? __ldg(p + j * HW) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_dx_tf32_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
                       const DxTf32Params P) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    // 1 KiB-aligned base by pointer arithmetic on the shared array (accesses stay shared-space)
    uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t wt_full[kMaxStages], wt_empty[kMaxStages], d_full[kDBufs], d_empty[kDBufs];
    __shared__ uint64_t yw_full, yw_empty, mma_done[kIssuers];
    __shared__ uint32_t tmem_slot;
    __shared__ uint32_t a_shift[kTaps];   // per-tap start offset of the A operand in the y window, bytes
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.d.C, H = P.d.H, W = P.d.W;
    const long long HW = P.d.HW;
    const int n_my = blockIdx.x < P.n_tiles ? (P.n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    const int S = P.stages, R = P.R;

    if (threadIdx.x < kTaps) {
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
        for (int i = 0; i < kDBufs; ++i) {
            mbar_init(&d_full[i], 1);
            mbar_init(&d_empty[i], kWork);
        }
        mbar_init(&yw_full, 1);
        mbar_init(&yw_empty, kIssuers);   // each issuer commits once per tile
        for (int i = 0; i < kIssuers; ++i) mbar_init(&mma_done[i], 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    if (warp >= 2 && warp < 2 + kWork) {
        // constant operands: one-hot tap selectors, bias tables, the zero chunk of the y window
        const int et = threadIdx.x - 64, nt = 32 * kWork;
        float* oh = reinterpret_cast<float*>(sm + P.ooh);
        for (int i = et; i < kOneHot / 4; i += nt) {        // [tap k][K-group g][row][e], column g*4 + e
            const int k = i >> 7, g = (i >> 5) & 3, e = i & 3;
            oh[i] = (g * 4 + e == k) ? 1.0f : 0.0f;
        }
        // bias table [d][c/8][k/4][c%8][k%4]: one thread per (d, c) loads the channel's nine taps
        // (independent loads, one latency) and writes its four 16-byte chunks
        for (int i = et; i < 3 * 64; i += nt) {
            const int dd = i >> 6, c = i & 63;
            float b[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) b[k] = 0.0f;
            if (P.bias != nullptr && c < C) {
                const float* bp = P.bias + ((long long)dd * C + c) * 9;
#pragma unroll
                for (int k = 0; k < 9; ++k) b[k] = bp[k];
            }
            float* ch = reinterpret_cast<float*>(sm + P.obt) + dd * 1024 + (c >> 3) * 128 + (c & 7) * 4;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                *reinterpret_cast<float4*>(ch + g * 32) = make_float4(b[4 * g], b[4 * g + 1], b[4 * g + 2], b[4 * g + 3]);
        }
        const int nzero = (2 * P.nks - P.nch4) * P.npos;    // chunk nch4 when C/4 is odd
        for (int i = et; i < nzero; i += nt)
            *reinterpret_cast<uint4*>(sm + P.oyw + ((long long)P.nch4 * P.npos + i) * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer: y window
        if (lane == 0) {
            prefetch_tmap(&tmY);
            const uint32_t ybytes = (uint32_t)P.nch4 * P.npos * 16;
            int ny = 0;
            for (int tl = 0; tl < n_my; ++tl) {
                const int t = blockIdx.x + tl * gridDim.x;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kTH, w0 = (ti % P.tiles_w) * kTW;
                if (!mbar_wait(&yw_empty, (tl & 1) ^ 1, P.err, abort_v)) break;
                mbar_arrive_expect_tx(&yw_full, ybytes);
                tma_load_4d(sm + P.oyw, &tmY, &yw_full, (w0 - R) * 4, h0 - R, 0, b);
                ny = tl + 1;
            }
            // drain: every copy this thread started lands before its shared memory is released
            int never = 0;
            if (ny > 0) mbar_wait(&yw_full, (ny - 1) & 1, P.err, &never);
        }
    } else if (warp == kWProd) {
        // ------------------------------------------------------- TMA producer: W ring, one tap per stage
        if (lane == 0) {
            prefetch_tmap(&tmW);
            int iw = 0, st = 0, sph = 0;               // taps issued, ring stage and its phase parity
            const bool two_atoms = C > 32;             // j 32..63 exist
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl)
                for (int u = 0; u < kTaps; ++u) {
                    const int dd = u / 9, k = u - dd * 9;
                    if (!mbar_wait(&wt_empty[st], sph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&wt_full[st], two_atoms ? kWTile : kWAtom);
                    tma_load_3d(sm + st * kWTile, &tmW, &wt_full[st], 0, k, dd * C);
                    if (two_atoms) tma_load_3d(sm + st * kWTile + kWAtom, &tmW, &wt_full[st], 32, k, dd * C);
                    ++iw;
                    if (++st == S) {
                        st = 0;
                        sph ^= 1;
                    }
                }
            int never = 0;
            for (int i = iw > S ? iw - S : 0; i < iw; ++i) mbar_wait(&wt_full[i % S], (i / S) & 1, P.err, &never);
        }
    } else if (warp == 1 || warp == kIssuer2) {
        // ------------------------------------------------------- MMA issuers: taps of parity `par`
        // An issuing thread spends tens of cycles on every instruction between two MMAs,
        // so the loop keeps them few: ring stage, buffer and tap advance by counters (no
        // division), the descriptors are built once and each MMA adds a 32-bit offset to
        // the low half of one, and the eight K steps of a tap are one unrolled burst.
        const int par = warp == 1 ? 0 : 1;
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(2, 0, 0, 128, kN);   // TF32, both operands K-major
            const uint32_t lbo_y = (uint32_t)P.npos * 16, sbo_y = (uint32_t)P.WW * 16;
            const uint64_t a_base = smem_desc(smem_u32(sm + P.oyw), lbo_y, sbo_y, kSwizzleNone);
            const uint64_t w_base = smem_desc(smem_u32(sm), 16, 1024, kSwizzle128B);
            const uint64_t oh_base = smem_desc(smem_u32(sm + P.ooh), 128, 0, kSwizzleNone);
            const uint64_t bt_base = smem_desc(smem_u32(sm + P.obt), 128, 512, kSwizzleNone);
            const uint32_t a_hi = (uint32_t)(a_base >> 32), w_hi = (uint32_t)(w_base >> 32);
            const uint32_t oh_hi = (uint32_t)(oh_base >> 32), bt_hi = (uint32_t)(bt_base >> 32);
            const uint32_t astep = (2 * lbo_y) >> 4;              // one K step of A, descriptor units
            const bool full_k = P.nks == 8;
            const int nks = P.nks;
            int st = par, sph = 0;            // W ring stage of this issuer's next tap and its phase
            int buf = par, bph = 0;           // TMEM buffer of this issuer's next tap and its phase
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                if (!mbar_wait(&yw_full, tl & 1, P.err, abort_v)) break;
                tc_fence_after();
                // the first tap of tile tl for this issuer: (27 tl + u) % 2 == par
                int u = par ^ (tl & 1), dd = 0, k = u;
                for (; u < kTaps; u += 2) {
                    const uint32_t a_lo = (uint32_t)a_base + (a_shift[u] >> 4);
                    const uint32_t w_lo = (uint32_t)w_base + (uint32_t)((st * kWTile) >> 4);
                    const uint32_t oh_lo = (uint32_t)oh_base + (uint32_t)(k * 32);
                    const uint32_t bt_lo = (uint32_t)bt_base + (uint32_t)(dd * 256);
                    const uint32_t dt = tmem + (uint32_t)(buf * kN);
                    if (!mbar_wait(&wt_full[st], sph, P.err, abort_v) ||
                        !mbar_wait(&d_empty[buf], bph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (full_k) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_tf32_lh(dt, a_lo + kk * astep, a_hi,
                                        w_lo + (uint32_t)(((kk >> 2) * kWAtom + (kk & 3) * 32) >> 4), w_hi, idesc,
                                        kk > 0 ? 1u : 0u);
                    } else {
                        for (int kk = 0; kk < nks; ++kk)
                            mma_tf32_lh(dt, a_lo + kk * astep, a_hi,
                                        w_lo + (uint32_t)(((kk >> 2) * kWAtom + (kk & 3) * 32) >> 4), w_hi, idesc,
                                        kk > 0 ? 1u : 0u);
                    }
                    mma_tf32_lh(dt, oh_lo, oh_hi, bt_lo, bt_hi, idesc, 1u);
                    mma_tf32_lh(dt, oh_lo + 16, oh_hi, bt_lo + 16, bt_hi, idesc, 1u);
                    mma_commit(&d_full[buf]);
                    mma_commit(&wt_empty[st]);
                    st += 2;
                    if (st >= S) {
                        st -= S;
                        sph ^= 1;
                    }
                    buf += 2;
                    if (buf >= kDBufs) {
                        buf -= kDBufs;
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
        // ------------------------------------------------------- workers: gather, accumulate
        const int q = warp & 3, hc = (warp - 2) >> 2;   // lane quadrant, channel half [32 hc, 32 hc + 32)
        const int s = q * 32 + lane;                    // slot == TMEM lane
        const int r = s >> 3, c = s & 7;
        const int c0 = hc * 32;
        const long long gimg = 3LL * P.nch4 * HW;   // float4 per image of the chunked grad
        bool ok = true;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            const int t = blockIdx.x + tl * gridDim.x;
            const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
            const int h = (ti / P.tiles_w) * kTH + r, w = (ti % P.tiles_w) * kTW + c;
            const bool inside = h < H && w < W;
            const long long pix = inside ? (long long)h * W + w : 0;
            const float* gb = P.g + (long long)b * 4 * C * HW;
            const float4* gci = P.gc + (long long)b * gimg;
            // the identity term (channel block 0) is loaded after the gather (an L2 prefetch of
            // it here cost the workers more at every tile change than it saved)
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            // the grad of tap u sits in buffer u % 2; it is consumed after tap u's accumulator
            // has been read and the buffer is refilled at once with tap u + 2, so every gather
            // has two taps' time to arrive
            float4 ga[8], gb2[8];
            gather_tap(ga, gci, 0, P, h, w, inside, c0 / 4);
            gather_tap(gb2, gci, 1, P, h, w, inside, c0 / 4);
            auto step = [&](int u, float4(&g)[8]) {
                const int i = tl * kTaps + u, buf = i % kDBufs;
                if (!__all_sync(0xffffffffu, mbar_wait(&d_full[buf], (i / kDBufs) & 1, P.err, abort_v))) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                uint32_t v[32];
                const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + buf * kN + c0;
                DDPM_TMEM_LD_X16(ta, (v + 0));
                DDPM_TMEM_LD_X16(ta + 16, (v + 16));
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_empty[buf]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    acc[4 * j + 0] = fmaf(__uint_as_float(v[4 * j + 0]), g[j].x, acc[4 * j + 0]);
                    acc[4 * j + 1] = fmaf(__uint_as_float(v[4 * j + 1]), g[j].y, acc[4 * j + 1]);
                    acc[4 * j + 2] = fmaf(__uint_as_float(v[4 * j + 2]), g[j].z, acc[4 * j + 2]);
                    acc[4 * j + 3] = fmaf(__uint_as_float(v[4 * j + 3]), g[j].w, acc[4 * j + 3]);
                }
                if (u + 2 < kTaps) gather_tap(g, gci, u + 2, P, h, w, inside, c0 / 4);
            };
            for (int u = 0; u + 1 < kTaps && ok; u += 2) {
                step(u, ga);
                if (ok) step(u + 1, gb2);
            }
            if (ok) step(kTaps - 1, ga);
            if (!ok) break;
            if (inside) {
                const float* g0p = gb + (long long)c0 * HW + pix;
                float* dxp = P.dx + ((long long)b * C + c0) * HW + pix;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (c0 + i < C) dxp[(long long)i * HW] = __ldg(g0p + (long long)i * HW) + acc[i];
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

}  // namespace

bool bwd_dx_tf32_shape_ok(const Dims& d) {
    if (d.dtype != 0 || !(d.flags & kFlagTf32Backward) || (d.flags & kFlagCudaCores) || d.K != 3) return false;
    if (d.C % 4 != 0 || d.C > 64 || d.W % 4 != 0) return false;   // 16-byte chunks, strides and TMA coordinates
    if (4LL * d.C * d.HW >= (1LL << 31)) return false;
    return dx_tf32_layout(d).stages > 0 && d.O <= (1LL << 30);
}

bool bwd_dx_tf32_eligible(const Dims& d, const void* g, const void* y, const void* w, const void* dx) {
    if (!bwd_dx_tf32_shape_ok(d)) return false;
    if ((uintptr_t)g % 16 || (uintptr_t)y % 16 || (uintptr_t)w % 16 || (uintptr_t)dx % 4) return false;
    return bwdtc::encode_fn() != nullptr;
}

size_t bwd_dx_tf32_bytes(const Dims& d) { return (size_t)4 * d.B * (size_t)d.C * (size_t)d.HW * sizeof(float); }

cudaError_t launch_bwd_dx_tf32(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                               void* packed, cudaStream_t s) {
    const DxTf32Layout L = dx_tf32_layout(d);
    if (L.stages == 0 || (uintptr_t)packed % 16 != 0) return cudaErrorInvalidValue;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dx_tf32_kernel, L.bytes, attr_done);
        if (e != cudaSuccess) return e;
    }
    auto enc = bwdtc::encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    float* yc = static_cast<float*>(packed);
    float* gc = yc + (size_t)d.B * d.C * d.HW;
    const int nch4 = d.C / 4;

    DxTf32Params P;
    P.d = d;
    P.tiles_w = (d.W + kTW - 1) / kTW;
    P.tiles_per_img = ((d.H + kTH - 1) / kTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.R = d.R();
    P.WW = kTW + 2 * P.R;
    P.WH = kTH + 2 * P.R;
    P.npos = P.WW * P.WH;
    P.nch4 = nch4;
    P.nks = (d.C + 7) / 8;
    P.stages = L.stages;
    P.oyw = L.oyw;
    P.ooh = L.ooh;
    P.obt = L.obt;
    P.g = static_cast<const float*>(g);
    P.gc = reinterpret_cast<const float4*>(gc);
    P.bias = static_cast<const float*>(bias);
    P.dx = static_cast<float*>(dx);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;

    CUtensorMap tmW, tmY;
    {
        // W viewed as [3C (dc)][9 (k)][C (j)]: box {32 j, 1 k, 64 dc} = one K-atom of the rows (d*C + c, k)
        const cuuint64_t dims[3] = {(cuuint64_t)d.C, 9, (cuuint64_t)(3 * d.C)};
        const cuuint64_t str[2] = {(cuuint64_t)d.C * 4, (cuuint64_t)d.C * 9 * 4};
        const cuuint32_t box[3] = {32, 1, 64};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(w), dims, str, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // the packed copy [B][C/4][H][W*4] fp32: a window row of one chunk is one run of WW*16 bytes;
        // positions outside the image (x < 0 or x >= W*4, rows outside) read as zeros
        const cuuint64_t dims[4] = {(cuuint64_t)d.W * 4, (cuuint64_t)d.H, (cuuint64_t)nch4, (cuuint64_t)d.B};
        const cuuint64_t str[3] = {(cuuint64_t)d.W * 16, (cuuint64_t)d.HW * 16, (cuuint64_t)d.HW * 16 * nch4};
        const cuuint32_t box[4] = {(cuuint32_t)P.WW * 4, (cuuint32_t)P.WH, (cuuint32_t)nch4, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (P.WW * 4 > 256 || P.WH > 256 ||
            enc(&tmY, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, yc, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    // 1. the channel-chunked copies of y and of the three dilation blocks of grad
    const long long n_y = (long long)d.B * nch4 * (d.HW / 4), n_all = 4 * n_y;
    long long blocks = (n_all + kPackThreads - 1) / kPackThreads;
    const long long cap = (long long)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    trace_begin(s, kKPackF32);
    pack_f32_kernel<<<(unsigned)blocks, kPackThreads, 0, s>>>(static_cast<const float*>(y),
                                                              static_cast<const float*>(g), yc, gc, d.C, d.HW, n_y,
                                                              n_all);
    trace_end(s);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    // 2. the shifted-GEMM dX
    int grid = num_sms();
    if (grid > P.n_tiles) grid = P.n_tiles;
    trace_begin(s, kKBwdDxTf32);
    bwd_dx_tf32_kernel<<<grid, kThreads, L.bytes, s>>>(tmW, tmY, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace ddpm
