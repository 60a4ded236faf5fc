// bwd_tc_common.cuh -- pieces shared by the tensor-core backward kernels.
//
// Pixel tiles are 2 rows x 64 columns (128 pixels, m = r * 64 + c), so that
// each 64-pixel half of a tile is one contiguous 128-byte row per channel:
// the shape a 128B-swizzled TMA box delivers as an MMA operand atom.
// Taps are processed in blocks of channels of one dilation, padded to the MMA
// M / K of 128: 14 channels (126 taps) for K = 3, 5 channels (125 taps) for
// K = 5.  Row r of a block is tap o = (d*C + c_first + r/K^2)*K^2 + r%K^2.
//
// dK^T tiles ([128 taps x 128 pixels], bf16) live in shared memory in the
// 128B-swizzled layout: pixel half h at +16 KiB * h, tap row r at
// (r/8)*1024 + (r%8)*128, 16-byte chunk (px%64)/8 XOR (r%8).  Read with
// M = taps it is a K-major operand (dW); read with M = pixels it is an
// MN-major operand (dY): the same bytes serve both.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "launch.h"

namespace ddpm {
namespace bwdtc {

using bf16 = __nv_bfloat16;

constexpr int kCB = 14;            // K = 3: channels per block of taps (126 rows)
constexpr int kBlockRows = 128;    // MMA extent of a block of taps
constexpr int kTH = 2, kTW = 64;   // pixel tile
constexpr int kPx = kTH * kTW;     // 128
constexpr int kSlots = 16;         // channel slots of a 16-channel TMA box
constexpr int kMaxR = 8;           // K = 3: halo radius supported
constexpr int kWinCols = kTW + 16; // K = 3: x window columns; origin w0 - 8 keeps TMA coordinates 16-byte aligned
constexpr int kDKBytes = kBlockRows * kPx * 2;  // 32 KiB

// Per kernel size: channels per block of taps (CB * K^2 <= 128), the x window's
// column halo left and right of the tile (a 16-byte TMA coordinate, >= the widest
// horizontal tap reach), its width, and the largest halo radius the kernels take.
template <int K> struct BwdGeom;
template <> struct BwdGeom<3> {
    static constexpr int kCB = 14, kHaloCols = 8, kWinCols = kTW + 16, kMaxR = 8;
};
template <> struct BwdGeom<5> {
    static constexpr int kCB = 5, kHaloCols = 16, kWinCols = kTW + 32, kMaxR = 10;
};

// (a * b) for two bf16 pairs: the exact product rounded once to bf16 (nearest even).
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
    __nv_bfloat162 z = __hmul2(x, y);
    return *reinterpret_cast<uint32_t*>(&z);
}

// Form one dK^T tile: dK[r, px] = grad_d[c, px] * x[c, px + off(d, k)], r = c_local*K*K + k.
//   dk        destination tile (32 KiB, swizzled as described above)
//   xs32      x window of the block's channels: slot c_local, rows (tile rows + 2R),
//             G::kWinCols columns, bf16, origin (h0 - R + row_off, w0 - G::kHaloCols)
//   gs        grad planes of the block: slot c_local, the 128 pixels of this tile
//             at gs + c_local * gstride
//   row_off   first window row of this tile (tiles stacked in one window)
//   tid/nthr  this thread among the forming threads
// One work unit is (channel c_local, 8-pixel chunk) for all K*K taps: the grad
// chunk is loaded once, and each of the K window rows as aligned 16-byte vectors
// (elements c8 .. c8+8+2H-1 of the row, H = G::kHaloCols, i.e. columns -H .. 7+H
// around the chunk) from which the K horizontal taps, shifted by compile-time
// multiples of the dilation DIL, are cut with byte permutes.  A warp's 16-byte loads
// and stores touch each bank once per eight threads, so they run without shared-memory
// bank conflicts.  Rows of channels c_local >= nc are written as zeros; rows
// CB*K*K .. 127 of the block are never written (the caller zeroes them once).
template <int K, int DIL>
__device__ __forceinline__ void form_dk_tile_dil(uint8_t* dk, const uint32_t* xs32, const bf16* gs, int gstride,
                                                 int nc, int slot_elems, int R, int row_off, int tid, int nthr) {
    using G = BwdGeom<K>;
    constexpr int kH = G::kHaloCols, kNV = (8 + 2 * kH) / 8, kNW = 4 * kNV, r0 = K / 2;
    static_assert(DIL >= 1 && r0 * DIL <= kH, "the window holds the taps' horizontal reach");
    const uint4* xs4 = reinterpret_cast<const uint4*>(xs32);
    for (int u = tid; u < G::kCB * 16; u += nthr) {
        const int cl = u >> 4, chunk = u & 15;
        const int tr = chunk >> 3, c8 = (chunk & 7) * 8;
        uint8_t* rowbase = dk + tr * 16384;
        const int sw = chunk & 7;
        if (cl >= nc) {
#pragma unroll
            for (int k = 0; k < K * K; ++k) {
                const int ol = cl * K * K + k;
                *reinterpret_cast<uint4*>(rowbase + (ol >> 3) * 1024 + (ol & 7) * 128 + ((sw ^ (ol & 7)) << 4)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            continue;
        }
        const uint4 gv = *reinterpret_cast<const uint4*>(gs + cl * gstride + chunk * 8);
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            const int e = cl * slot_elems + (row_off + tr + R + (ky - r0) * DIL) * G::kWinCols + c8;   // multiple of 8
            uint32_t w[kNW];
#pragma unroll
            for (int v = 0; v < kNV; ++v) {
                const uint4 q = xs4[(e >> 3) + v];
                w[4 * v + 0] = q.x;
                w[4 * v + 1] = q.y;
                w[4 * v + 2] = q.z;
                w[4 * v + 3] = q.w;
            }
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int off = kH + (kx - r0) * DIL;            // element of tap kx's first pixel
                uint32_t a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int wi = (off >> 1) + i;
                    a[i] = (off & 1) ? __byte_perm(w[wi], w[(wi + 1) < kNW ? wi + 1 : kNW - 1], 0x5432) : w[wi];
                }
                const int ol = cl * K * K + ky * K + kx;
                uint4 v;
                v.x = bf2_mul(gv.x, a[0]);
                v.y = bf2_mul(gv.y, a[1]);
                v.z = bf2_mul(gv.z, a[2]);
                v.w = bf2_mul(gv.w, a[3]);
                *reinterpret_cast<uint4*>(rowbase + (ol >> 3) * 1024 + (ol & 7) * 128 + ((sw ^ (ol & 7)) << 4)) = v;
            }
        }
    }
}

template <int K>
__device__ __forceinline__ void form_dk_tile(uint8_t* dk, const uint32_t* xs32, const bf16* gs, int gstride, int nrows,
                                             int slot_elems, int R, int dil, int row_off, int tid, int nthr) {
    const int nc = nrows / (K * K);
    switch (dil) {
        case 1: form_dk_tile_dil<K, 1>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        case 2: form_dk_tile_dil<K, 2>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        case 3: form_dk_tile_dil<K, 3>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        case 4: form_dk_tile_dil<K, 4>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        case 5: form_dk_tile_dil<K, 5>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        case 6: form_dk_tile_dil<K, (K == 3 ? 6 : 5)>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        case 7: form_dk_tile_dil<K, (K == 3 ? 7 : 5)>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
        default: form_dk_tile_dil<K, (K == 3 ? 8 : 5)>(dk, xs32, gs, gstride, nc, slot_elems, R, row_off, tid, nthr); break;
    }
}

// Zero the padding rows (CB*K*K .. 127) of a dK^T tile.
template <int K>
__device__ __forceinline__ void zero_dk_pad_rows(uint8_t* dk, int tid, int nthr) {
    constexpr int r0 = BwdGeom<K>::kCB * K * K, npad = kBlockRows - r0;
    for (int u = tid; u < npad * 2 * 8; u += nthr) {   // pad rows x 2 halves x 8 chunks
        const int ol = r0 + (u >> 4), half = (u >> 3) & 1, c = u & 7;
        *reinterpret_cast<uint4*>(dk + half * 16384 + (ol >> 3) * 1024 + (ol & 7) * 128 + ((c ^ (ol & 7)) << 4)) =
            make_uint4(0u, 0u, 0u, 0u);
    }
}

// Driver entry point for tensor-map encoding (looked up once).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 4-D bf16 tensor map over an NCHW tensor with `ch` channels: dims (W, H, ch, B).
inline bool encode_nchw(CUtensorMap* m, const void* base, const Dims& d, int ch, uint32_t bw, uint32_t bh,
                        uint32_t bc, CUtensorMapSwizzle swz) {
    const cuuint64_t dims[4] = {(cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)ch, (cuuint64_t)d.B};
    const cuuint64_t str[3] = {(cuuint64_t)d.W * 2, (cuuint64_t)d.HW * 2, (cuuint64_t)d.HW * ch * 2};
    const cuuint32_t box[4] = {bw, bh, bc, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, str, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shapes the tensor-core backward handles: bf16, K = 3 (K = 5 as well where k5 is
// set: the dW and dY kernels), C a multiple of 8 up to 64, W a multiple of 8 (16-byte
// TMA strides), the halo radius within the window (8 for K = 3, 10 for K = 5),
// 16-byte aligned tensors.  shape_ok() is the part that depends on the problem alone.
inline bool shape_ok(const Dims& d, bool k5 = false) {
    if (d.dtype != 1 || (d.flags & kFlagCudaCores)) return false;
    if (!(d.K == 3 || (k5 && d.K == 5))) return false;
    if (d.C > 64 || d.C % 8 != 0 || d.W % 8 != 0) return false;
    if (d.R() > (d.K == 3 ? BwdGeom<3>::kMaxR : BwdGeom<5>::kMaxR)) return false;
    return d.O <= (1LL << 30) && d.HW <= (1LL << 31) - 1024;
}

inline bool eligible(const Dims& d, const void* a, const void* b, const void* c, bool k5 = false) {
    if (!shape_ok(d, k5)) return false;
    if ((uintptr_t)a % 16 || (uintptr_t)b % 16 || (uintptr_t)c % 16) return false;
    return encode_fn() != nullptr;
}

}  // namespace bwdtc
}  // namespace ddpm
