// bwd_tc_common.cuh -- pieces shared by the tensor-core backward kernels.
//
// Pixel tiles are 2 rows x 64 columns (128 pixels, m = r * 64 + c), so that
// each 64-pixel half of a tile is one contiguous 128-byte row per channel:
// the shape a 128B-swizzled TMA box delivers as an MMA operand atom.
// Taps are processed in blocks of 14 channels of one dilation (126 taps,
// padded to the MMA M / K of 128): row r of a block is tap
// o = (d*C + c_first + r/9)*9 + r%9.
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

constexpr int kCB = 14;            // channels per block of taps (126 rows)
constexpr int kBlockRows = 128;    // MMA extent of a block of taps
constexpr int kTH = 2, kTW = 64;   // pixel tile
constexpr int kPx = kTH * kTW;     // 128
constexpr int kSlots = 16;         // channel slots of a 16-channel TMA box
constexpr int kMaxR = 8;           // halo radius supported
constexpr int kWinCols = kTW + 16; // x window columns: origin w0 - 8 keeps TMA coordinates 16-byte aligned
constexpr int kDKBytes = kBlockRows * kPx * 2;  // 32 KiB

// (a * b) for two bf16 pairs: the exact product rounded once to bf16 (nearest even).
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162*>(&a);
    __nv_bfloat162 y = *reinterpret_cast<__nv_bfloat162*>(&b);
    __nv_bfloat162 z = __hmul2(x, y);
    return *reinterpret_cast<uint32_t*>(&z);
}

// Form one dK^T tile: dK[r, px] = grad_d[c, px] * x[c, px + off(d, k)], r = c_local*9 + k.
//   dk        destination tile (32 KiB, swizzled as described above)
//   xs32      x window of the block's channels: slot c_local, rows (tile rows + 2R),
//             kWinCols columns, bf16, origin (h0 - R + row_off, w0 - 8)
//   gs        grad planes of the block: slot c_local, 128 pixels of this tile
//   row_off   first window row of this tile (tiles stacked in one window)
//   tid/nthr  this thread among the forming threads
// Rows r >= nrows (the padding of a 126-tap block) are written as zeros.
__device__ __forceinline__ void form_dk_tile(uint8_t* dk, const uint32_t* xs32, const bf16* gs, int nrows,
                                             int slot_elems, int R, int dil, int row_off, int tid, int nthr) {
    for (int u = tid; u < kBlockRows * 16; u += nthr) {
        const int ol = u >> 4, chunk = u & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ol < nrows) {
            const int cl = ol / 9, k = ol - cl * 9;
            const int ky = k / 3, kx = k - ky * 3;
            const int tr = chunk >> 3, c8 = (chunk & 7) * 8;
            const int e0 = cl * slot_elems + (row_off + tr + R + (ky - 1) * dil) * kWinCols + (c8 + 8 + (kx - 1) * dil);
            const uint32_t* wp = xs32 + (e0 >> 1);
            uint32_t a0 = wp[0], a1 = wp[1], a2 = wp[2], a3 = wp[3];
            if (e0 & 1) {
                const uint32_t a4 = wp[4];
                a0 = __byte_perm(a0, a1, 0x5432);
                a1 = __byte_perm(a1, a2, 0x5432);
                a2 = __byte_perm(a2, a3, 0x5432);
                a3 = __byte_perm(a3, a4, 0x5432);
            }
            const uint4 gv = *reinterpret_cast<const uint4*>(gs + cl * kPx + chunk * 8);
            v.x = bf2_mul(gv.x, a0);
            v.y = bf2_mul(gv.y, a1);
            v.z = bf2_mul(gv.z, a2);
            v.w = bf2_mul(gv.w, a3);
        }
        *reinterpret_cast<uint4*>(dk + (chunk >> 3) * 16384 + (ol >> 3) * 1024 + (ol & 7) * 128 +
                                  (((chunk & 7) ^ (ol & 7)) << 4)) = v;
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

// Shapes the tensor-core backward handles: bf16, K = 3, C a multiple of 8 up to 64,
// W a multiple of 8 (16-byte TMA strides), halo radius <= 8, 16-byte aligned tensors.
inline bool eligible(const Dims& d, const void* a, const void* b, const void* c) {
    if (d.dtype != 1 || d.K != 3 || (d.flags & kFlagCudaCores)) return false;
    if (d.C > 64 || d.C % 8 != 0 || d.W % 8 != 0) return false;
    if (d.R() > kMaxR) return false;
    if ((uintptr_t)a % 16 || (uintptr_t)b % 16 || (uintptr_t)c % 16) return false;
    if (d.O > (1LL << 30) || d.HW > (1LL << 31) - 1024) return false;
    return encode_fn() != nullptr;
}

}  // namespace bwdtc
}  // namespace ddpm
