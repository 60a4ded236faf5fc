// bwd_dx_gather.cu -- bf16 dX on tcgen05 tensor cores with grad gathered from L2 (K = 3, 5).
//
// README "lartpang/DynamicConvolutionOperator", section "CUDA Flash 式融合训练":
// dX recomputes the dynamic taps and gathers each dilation's contribution:
//   dx[b,c,q] = grad[b,c,q] + sum_{d,ky,kx} Tq[b,o,q-off] * grad[b,(1+d)C+c,q-off],
//   Tq = bf16(bias[o] + sum_j W[o,j] y[b,j,q-off]),  o = (d*C + c)*K*K + ky*K + kx.
//
// The variant of the packed dX (bwd_dx_packed.cu) for halos whose grad windows do not
// fit in shared memory beside the y window -- K = 5, halo radius up to 10.  It reads
// the same channel-chunked copies ([B][C/8][H][W][8] for y, [B][3][C/8][H][W][8] for
// grad, written by the same pack) and computes the same taps, but keeps only the y
// window in shared memory:
//   - per 16x8 pixel tile (MMA M = 128, slot s = r*8 + c) each of the 3*K*K taps is one
//     shifted GEMM over all channels (N = 64): A is the y window (TMA, one contiguous
//     run per window row and chunk) at a start offset, B the tap's W rows [64 c][64 j]
//     (128B-swizzled, a ring fed by its own producer warp);
//   - the bias is one or two last K=16 steps: A a one-hot row selecting tap k (every row
//     group the same: stride 0), B a resident table of bias[d, c, k];
//   - two threads in different warps issue the MMAs of even and odd taps, from a compact
//     loop (counters, precomputed descriptor halves, one burst per tap);
//   - D of each tap lands in one of eight TMEM buffers [128 x 64]; eight worker warps
//     round it to bf16 and accumulate tap * grad in FP32 with one mixed-precision FMA
//     per channel (bf16 operands, exact product), the grad of each tap gathered from
//     the chunked copy in global memory (L2) two taps ahead: four 16-byte loads for
//     the thread's pixel and 32 channels.
#include "bwd_tc_common.cuh"
#include "tc.cuh"

namespace ddpm {
namespace {

using namespace bwdtc;

constexpr int kTH = 16, kTW = 8;           // pixel tile
constexpr int kN = 64;                     // MMA N: channels
constexpr int kWork = 8;                   // worker warps
constexpr int kIssuers = 2;
constexpr int kIssuer2 = 2 + kWork;
constexpr int kWProd = 3 + kWork;
constexpr int kThreads = 32 * (4 + kWork);
constexpr int kDBufs = 8;
constexpr int kMaxStages = 8;
constexpr int kMinStages = 2;
constexpr int kWTile = 8192;               // W rows of one tap: [64 c][64 j] bf16, SW128
constexpr int kSmemCap = 227 * 1024 - 1024;

// one-hot A rows per tap: [K-group of 8 taps][8 rows][8] bf16, NB16 K=16 steps
template <int K> struct GatherCfg {
    static constexpr int kTaps = 3 * K * K;
    static constexpr int kNBias = (K * K + 15) / 16;          // K=16 bias steps per tap
    static constexpr int kOneHot = K * K * kNBias * 256;      // [tap][2 NBias groups][8 rows][16 B]
    static constexpr int kBiasTab = 3 * 8 * kNBias * 256;     // [d][c/8][2 NBias k-groups][8][8] bf16
    static constexpr int kMaxR = K == 3 ? 8 : 10;
};

struct DxGatherParams {
    Dims d;
    int tiles_w, tiles_per_img, n_tiles;
    int R, WW, WH, npos, nch, nks, stages;
    int oyw, ooh, obt;
    const bf16* g;                         // grad, NCHW (block 0 gives the identity term)
    const uint4* gc;                       // grad blocks 1..3, chunked [B][3][C/8][H*W] x 16 B
    const bf16* bias;
    bf16* dx;
    unsigned int* err;
};

struct DxGatherLayout {
    int stages, oyw, ooh, obt, bytes;
};

template <int K>
DxGatherLayout dx_gather_layout(const Dims& d) {
    using F = GatherCfg<K>;
    DxGatherLayout L{};
    const int R = d.R();
    if (R > F::kMaxR) return L;
    const int npos = (kTH + 2 * R) * (kTW + 2 * R);
    const int nks = (d.C / 8 + 1) / 2;
    const int ybytes = 2 * nks * npos * 16;
    const int rest = ybytes + F::kOneHot + F::kBiasTab;
    int stages = (kSmemCap - 1024 - rest) / kWTile;
    if (stages > kMaxStages) stages = kMaxStages;
    stages &= ~1;   // tap i uses stage i % stages; even: every use of a stage falls to one issuer
    if (stages < kMinStages) return L;
    L.stages = stages;
    L.oyw = stages * kWTile;
    L.ooh = L.oyw + ybytes;
    L.obt = L.ooh + F::kOneHot;
    L.bytes = L.obt + F::kBiasTab + 1024;
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

// The grad of one tap for this thread's pixel and its 32 channels (4 chunks of 8), from
// the chunked copy gci = [3][C/8][HW] x 16 B of this image (zero outside the image or
// beyond C).
template <int K>
__device__ __forceinline__ void gather_tap(uint4 (&g)[4], const uint4* gci, int u, const DxGatherParams& P, int h,
                                           int w, bool inside, int cq0) {
    const int dd = u / (K * K), k = u - dd * (K * K);
    const int dil = dil_of(P.d, dd);
    const int sh = h - (k / K - K / 2) * dil, sw = w - (k % K - K / 2) * dil;
    const bool valid = inside && sh >= 0 && sh < P.d.H && sw >= 0 && sw < P.d.W;
    const long long HW = P.d.HW;
    const uint4* p = gci + ((long long)dd * P.nch + cq0) * HW + (long long)sh * P.d.W + sw;
    const int nq = P.nch - cq0;
#pragma unroll
    for (int j = 0; j < 4; ++j) g[j] = (valid && j < nq) ? __ldg(p + j * HW) : make_uint4(0u, 0u, 0u, 0u);
}

template <int K>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dx_gather_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmY,
                         const DxGatherParams P) {
    using namespace tc;
    using F = GatherCfg<K>;
    constexpr int kTaps = F::kTaps, kKK = K * K, kNBias = F::kNBias;
    extern __shared__ uint8_t smem_raw[];
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

    for (int u = threadIdx.x; u < kTaps; u += blockDim.x) {
        // tap (ky, kx) of dilation d reads y at q - ((ky-r) d, (kx-r) d): window position
        // (r_q + R - (ky-r) d, c_q + R - (kx-r) d)
        const int dil = dil_of(P.d, u / kKK), k = u % kKK, ky = k / K, kx = k % K;
        a_shift[u] = (uint32_t)((R - (ky - K / 2) * dil) * P.WW + (R - (kx - K / 2) * dil)) * 16;
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
        mbar_init(&yw_empty, kIssuers);
        for (int i = 0; i < kIssuers; ++i) mbar_init(&mma_done[i], 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 512);
    if (warp >= 2 && warp < 2 + kWork) {
        // constant operands: one-hot tap selectors, bias tables, the zero chunk of the y window
        const int et = threadIdx.x - 64, nt = 32 * kWork;
        unsigned short* oh = reinterpret_cast<unsigned short*>(sm + P.ooh);
        for (int i = et; i < F::kOneHot / 2; i += nt) {     // [tap k][K-group g][row][e], column g*8 + e
            const int k = i / (kNBias * 128), g = (i / 64) % (2 * kNBias), e = i & 7;
            oh[i] = (g * 8 + e == k) ? (unsigned short)0x3F80u : (unsigned short)0u;
        }
        // bias table [d][c/8][k-group g][c%8][e], k = g*8 + e: one thread per (d, c) loads the
        // channel's K*K taps (independent loads, one latency) and writes its 16-byte chunks
        for (int i = et; i < 3 * 64; i += nt) {
            const int dd = i >> 6, c = i & 63;
            unsigned short b[16 * kNBias];
#pragma unroll
            for (int k = 0; k < 16 * kNBias; ++k) b[k] = 0;
            if (P.bias != nullptr && c < C) {
                const unsigned short* bp =
                    reinterpret_cast<const unsigned short*>(P.bias) + ((long long)dd * C + c) * kKK;
#pragma unroll
                for (int k = 0; k < kKK; ++k) b[k] = bp[k];
            }
            uint8_t* ch = sm + P.obt + (dd * 8 * kNBias * 128 + (c >> 3) * (kNBias * 128) + (c & 7) * 8) * 2;
#pragma unroll
            for (int g = 0; g < 2 * kNBias; ++g) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) w[e] = (uint32_t)b[g * 8 + 2 * e] | ((uint32_t)b[g * 8 + 2 * e + 1] << 16);
                *reinterpret_cast<uint4*>(ch + g * 128) = make_uint4(w[0], w[1], w[2], w[3]);
            }
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
        // ------------------------------------------------------- TMA producer: y window
        if (lane == 0) {
            prefetch_tmap(&tmY);
            const uint32_t ybytes = (uint32_t)P.nch * P.npos * 16;
            int ny = 0;
            for (int tl = 0; tl < n_my; ++tl) {
                const int t = blockIdx.x + tl * gridDim.x;
                const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
                const int h0 = (ti / P.tiles_w) * kTH, w0 = (ti % P.tiles_w) * kTW;
                if (!mbar_wait(&yw_empty, (tl & 1) ^ 1, P.err, abort_v)) break;
                mbar_arrive_expect_tx(&yw_full, ybytes);
                tma_load_4d(sm + P.oyw, &tmY, &yw_full, (w0 - R) * 8, h0 - R, 0, b);
                ny = tl + 1;
            }
            int never = 0;
            if (ny > 0) mbar_wait(&yw_full, (ny - 1) & 1, P.err, &never);
        }
    } else if (warp == kWProd) {
        // ------------------------------------------------------- TMA producer: W ring, one tap per stage
        if (lane == 0) {
            prefetch_tmap(&tmW);
            int iw = 0, st = 0, sph = 0;
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl)
                for (int u = 0; u < kTaps; ++u) {
                    const int dd = u / kKK, k = u - dd * kKK;
                    if (!mbar_wait(&wt_empty[st], sph ^ 1, P.err, abort_v)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&wt_full[st], kWTile);
                    tma_load_3d(sm + st * kWTile, &tmW, &wt_full[st], 0, k, dd * C);
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
        const int par = warp == 1 ? 0 : 1;
        if (lane == 0 && n_my > 0) {
            const uint32_t idesc = instr_desc(1, 0, 0, 128, kN);
            const uint32_t lbo_y = (uint32_t)P.npos * 16, sbo_y = (uint32_t)P.WW * 16;
            const uint64_t a_base = smem_desc(smem_u32(sm + P.oyw), lbo_y, sbo_y, kSwizzleNone);
            const uint64_t w_base = smem_desc(smem_u32(sm), 16, 1024, kSwizzle128B);
            const uint64_t oh_base = smem_desc(smem_u32(sm + P.ooh), 128, 0, kSwizzleNone);
            const uint64_t bt_base = smem_desc(smem_u32(sm + P.obt), 128, 2 * kNBias * 128, kSwizzleNone);
            const uint32_t a_hi = (uint32_t)(a_base >> 32), w_hi = (uint32_t)(w_base >> 32);
            const uint32_t oh_hi = (uint32_t)(oh_base >> 32), bt_hi = (uint32_t)(bt_base >> 32);
            const uint32_t astep = (2 * lbo_y) >> 4;
            const int nks = P.nks;
            const bool full_k = nks == 4;
            int st = par, sph = 0, buf = par, bph = 0;
            bool ok = true;
            for (int tl = 0; tl < n_my && ok; ++tl) {
                if (!mbar_wait(&yw_full, tl & 1, P.err, abort_v)) break;
                tc_fence_after();
                // the first tap of tile tl for this issuer: (kTaps tl + u) % 2 == par
                int u = par ^ ((tl * kTaps) & 1), dd = 0, k = u;
                for (; u < kTaps; u += 2) {
                    const uint32_t a_lo = (uint32_t)a_base + (a_shift[u] >> 4);
                    const uint32_t w_lo = (uint32_t)w_base + (uint32_t)((st * kWTile) >> 4);
                    const uint32_t oh_lo = (uint32_t)oh_base + (uint32_t)(k * kNBias * 16);
                    const uint32_t bt_lo = (uint32_t)bt_base + (uint32_t)(dd * 8 * kNBias * 16);
                    const uint32_t dt = tmem + (uint32_t)(buf * kN);
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
#pragma unroll
                    for (int nb = 0; nb < kNBias; ++nb)
                        mma_f16_lh(dt, oh_lo + nb * 16, oh_hi, bt_lo + nb * 16, bt_hi, idesc, 1u);
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
                    if (k >= kKK) {
                        k -= kKK;
                        ++dd;
                    }
                }
                if (ok) mma_commit(&yw_empty);
            }
            mma_commit(&mma_done[par]);
            int never = 0;
            mbar_wait(&mma_done[par], 0, P.err, &never);
        }
    } else {
        // ------------------------------------------------------- workers: round, gather, accumulate
        const int q = warp & 3, hc = (warp - 2) >> 2;   // lane quadrant, channel half [32 hc, 32 hc + 32)
        const int s = q * 32 + lane;                    // slot == TMEM lane
        const int r = s >> 3, c = s & 7;
        const int c0 = hc * 32;
        const long long gimg = 3LL * P.nch * HW;        // 16-byte chunks per image of the chunked grad
        bool ok = true;
        for (int tl = 0; tl < n_my && ok; ++tl) {
            const int t = blockIdx.x + tl * gridDim.x;
            const int b = t / P.tiles_per_img, ti = t % P.tiles_per_img;
            const int h = (ti / P.tiles_w) * kTH + r, w = (ti % P.tiles_w) * kTW + c;
            const bool inside = h < H && w < W;
            const long long pix = inside ? (long long)h * W + w : 0;
            const unsigned short* g0p = reinterpret_cast<const unsigned short*>(P.g) + (long long)b * 4 * C * HW + pix;
            const uint4* gci = P.gc + (long long)b * gimg;
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
            // the grad of tap u sits in buffer u % 2; it is consumed after tap u's accumulator
            // has been read and refilled at once with tap u + 2
            uint4 ga[4], gb[4];
            gather_tap<K>(ga, gci, 0, P, h, w, inside, c0 / 8);
            gather_tap<K>(gb, gci, 1, P, h, w, inside, c0 / 8);
            auto step = [&](int u, uint4(&g)[4]) {
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
                for (int e = 0; e < 4; ++e) {
                    const uint32_t gw4[4] = {g[e].x, g[e].y, g[e].z, g[e].w};
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const int ci = e * 8 + 2 * f;
                        const uint32_t t2 = pack_bf16x2(__uint_as_float(v[ci]), __uint_as_float(v[ci + 1]));
                        fma2_bf16_f32(acc[ci], acc[ci + 1], t2, gw4[f]);
                    }
                }
                if (u + 2 < kTaps) gather_tap<K>(g, gci, u + 2, P, h, w, inside, c0 / 8);
            };
            for (int u = 0; u + 1 < kTaps && ok; u += 2) {
                step(u, ga);
                if (ok) step(u + 1, gb);
            }
            if (ok && (kTaps & 1)) step(kTaps - 1, ga);
            if (!ok) break;
            if (inside) {
                bf16* dxp = P.dx + (long long)b * C * HW + pix;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int ch = c0 + i;
                    if (ch < C) {
                        const unsigned short g0 = __ldg(g0p + (long long)ch * HW);
                        dxp[(long long)ch * HW] = __float2bfloat16_rn(__uint_as_float((uint32_t)g0 << 16) + acc[i]);
                    }
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

template <int K>
cudaError_t launch_k(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                     void* packed, cudaStream_t s) {
    const DxGatherLayout L = dx_gather_layout<K>(d);
    if (L.stages == 0 || (uintptr_t)packed % 16 != 0) return cudaErrorInvalidValue;
    static int attr_done[64] = {};
    {
        const cudaError_t e = set_max_dynamic_smem((const void*)bwd_dx_gather_kernel<K>, L.bytes, attr_done);
        if (e != cudaSuccess) return e;
    }
    auto enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int nch = d.C / 8;
    bf16* yc = static_cast<bf16*>(packed);
    bf16* gc = yc + (size_t)d.B * d.C * d.HW;

    DxGatherParams P;
    P.d = d;
    P.tiles_w = (d.W + kTW - 1) / kTW;
    P.tiles_per_img = ((d.H + kTH - 1) / kTH) * P.tiles_w;
    P.n_tiles = d.B * P.tiles_per_img;
    P.R = d.R();
    P.WW = kTW + 2 * P.R;
    P.WH = kTH + 2 * P.R;
    P.npos = P.WW * P.WH;
    P.nch = nch;
    P.nks = (nch + 1) / 2;
    P.stages = L.stages;
    P.oyw = L.oyw;
    P.ooh = L.ooh;
    P.obt = L.obt;
    P.g = static_cast<const bf16*>(g);
    P.gc = reinterpret_cast<const uint4*>(gc);
    P.bias = static_cast<const bf16*>(bias);
    P.dx = static_cast<bf16*>(dx);
    P.err = device_error_word();
    if (P.err == nullptr) return cudaErrorUnknown;

    CUtensorMap tmW, tmY;
    {
        // W viewed as [3C (dc)][K*K (k)][C (j)]: box {64 j, 1 k, 64 dc} = rows (d*C + c, k) for 64 channels
        const cuuint64_t dims[3] = {(cuuint64_t)d.C, (cuuint64_t)(K * K), (cuuint64_t)(3 * d.C)};
        const cuuint64_t str[2] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.C * K * K * 2};
        const cuuint32_t box[3] = {64, 1, 64};
        const cuuint32_t es[3] = {1, 1, 1};
        if (enc(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, str, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // the packed y [B][C/8][H][W*8]: a window row of one chunk is one run of WW*16 bytes;
        // positions outside the image read as zeros
        const cuuint64_t dims[4] = {(cuuint64_t)d.W * 8, (cuuint64_t)d.H, (cuuint64_t)nch, (cuuint64_t)d.B};
        const cuuint64_t str[3] = {(cuuint64_t)d.W * 16, (cuuint64_t)d.HW * 16, (cuuint64_t)d.HW * 16 * nch};
        const cuuint32_t box[4] = {(cuuint32_t)P.WW * 8, (cuuint32_t)P.WH, (cuuint32_t)nch, 1};
        const cuuint32_t es[4] = {1, 1, 1, 1};
        if (P.WW * 8 > 256 || P.WH > 256 ||
            enc(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, yc, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cudaError_t e = launch_pack_chunks(d, g, y, packed, s);
        if (e != cudaSuccess) return e;
    }
    int grid = num_sms();
    if (grid > P.n_tiles) grid = P.n_tiles;
    trace_begin(s, kKBwdDxGather);
    bwd_dx_gather_kernel<K><<<grid, kThreads, L.bytes, s>>>(tmW, tmY, P);
    trace_end(s);
    return cudaGetLastError();
}

}  // namespace

bool bwd_dx_gather_shape_ok(const Dims& d) {
    if (!bwdtc::shape_ok(d, true)) return false;
    return (d.K == 3 ? dx_gather_layout<3>(d).stages : dx_gather_layout<5>(d).stages) > 0;
}

bool bwd_dx_gather_eligible(const Dims& d, const void* g, const void* y, const void* w) {
    return bwdtc::eligible(d, g, y, w, true) && bwd_dx_gather_shape_ok(d);
}

cudaError_t launch_bwd_dx_gather(const Dims& d, const void* g, const void* y, const void* w, const void* bias,
                                 void* dx, void* packed, cudaStream_t s) {
    return d.K == 3 ? launch_k<3>(d, g, y, w, bias, dx, packed, s) : launch_k<5>(d, g, y, w, bias, dx, packed, s);
}

}  // namespace ddpm
