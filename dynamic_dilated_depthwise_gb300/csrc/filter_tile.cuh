// filter_tile.cuh -- the vectorised plane tile shared by the filter kernels.
//
// A block owns one (b, c) plane tile of kFTH(T) rows x 64 columns; a thread owns
// VEC consecutive pixels of a row (one 16-byte vector).  A row segment shifted by
// o columns is cut out of the two aligned 16-byte vectors that cover it at
// o mod VEC, which is the same for every thread of the block (a uniform switch,
// no divergence).  Staged planes keep kFHalo columns of zeros left and right.
#pragma once

#include "common.cuh"

namespace ddpm {
namespace ftile {

constexpr int kFTW = 64;          // tile columns
constexpr int kFHalo = 16;        // staged columns left and right of the tile (R <= 16)
constexpr int kFRowElems = kFTW + 2 * kFHalo;
constexpr int kFThreads = 128;   // (64 / VEC) threads per row x TH rows

template <typename T> struct FilterTile;
template <> struct FilterTile<__nv_bfloat16> { static constexpr int VEC = 8, TH = 16; };
template <> struct FilterTile<float> { static constexpr int VEC = 4, TH = 8; };
static_assert((kFTW / 8) * 16 == kFThreads && (kFTW / 4) * 8 == kFThreads, "one thread per vector of the tile");

// VEC elements starting `sh` elements into the 2*VEC elements (v0, v1), as raw 32-bit words
template <typename T>
__device__ __forceinline__ uint4 cut_vec(const uint4& v0, const uint4& v1, int sh) {
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint4 r;
    if constexpr (sizeof(T) == 4) {
        switch (sh) {
            case 0: r = v0; break;
            case 1: r = make_uint4(w[1], w[2], w[3], w[4]); break;
            case 2: r = make_uint4(w[2], w[3], w[4], w[5]); break;
            default: r = make_uint4(w[3], w[4], w[5], w[6]); break;
        }
    } else {
#define DDPM_CUT(S)                                                                                        \
    case S: {                                                                                              \
        constexpr int q = (S) >> 1;                                                                        \
        if constexpr (((S) & 1) == 0) r = make_uint4(w[q], w[q + 1], w[q + 2], w[q + 3]);                 \
        else r = make_uint4(__byte_perm(w[q], w[q + 1], 0x5432), __byte_perm(w[q + 1], w[q + 2], 0x5432),  \
                            __byte_perm(w[q + 2], w[q + 3], 0x5432), __byte_perm(w[q + 3], w[q + 4], 0x5432)); \
        break;                                                                                             \
    }
        switch (sh) {
            DDPM_CUT(0) DDPM_CUT(1) DDPM_CUT(2) DDPM_CUT(3) DDPM_CUT(4) DDPM_CUT(5) DDPM_CUT(6)
            default: r = make_uint4(__byte_perm(w[3], w[4], 0x5432), __byte_perm(w[4], w[5], 0x5432),
                                    __byte_perm(w[5], w[6], 0x5432), __byte_perm(w[6], w[7], 0x5432));
        }
#undef DDPM_CUT
    }
    return r;
}

// acc[i] += tap[i] * x[i] for the VEC elements packed in two 16-byte words
__device__ __forceinline__ void fma_vec(float (&acc)[4], const uint4& t, const uint4& x) {
    acc[0] = fmaf(__uint_as_float(t.x), __uint_as_float(x.x), acc[0]);
    acc[1] = fmaf(__uint_as_float(t.y), __uint_as_float(x.y), acc[1]);
    acc[2] = fmaf(__uint_as_float(t.z), __uint_as_float(x.z), acc[2]);
    acc[3] = fmaf(__uint_as_float(t.w), __uint_as_float(x.w), acc[3]);
}
// bf16 operands, exact product, FP32 accumulate (fma.rn.f32.bf16)
__device__ __forceinline__ void fma_pair_bf16(float& a0, float& a1, uint32_t t, uint32_t x) {
    asm("{\n\t.reg .b16 tl, th, xl, xh;\n\t"
        "mov.b32 {tl, th}, %2;\n\t"
        "mov.b32 {xl, xh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, tl, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, th, xh, %1;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "r"(t), "r"(x));
}
__device__ __forceinline__ void fma_vec(float (&acc)[8], const uint4& t, const uint4& x) {
    fma_pair_bf16(acc[0], acc[1], t.x, x.x);
    fma_pair_bf16(acc[2], acc[3], t.y, x.y);
    fma_pair_bf16(acc[4], acc[5], t.z, x.z);
    fma_pair_bf16(acc[6], acc[7], t.w, x.w);
}


}  // namespace ftile
}  // namespace ddpm
