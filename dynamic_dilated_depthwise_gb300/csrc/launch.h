// launch.h -- internal launcher interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

#include "common.cuh"

namespace ddpm {

// Kernel ids reported by the tracing facility (ddpm_trace_read).
enum KernelId : int {
    kKFilterSimt = 0,
    kKForwardSimt = 1,
    kKForwardTc = 2,
    kKBwdDxSimt = 3,
    kKBwdDySimt = 4,
    kKBwdDwPartialSimt = 5,
    kKBwdDwReduce = 6,
    kKBwdDxTc = 7,
    kKBwdDyTc = 8,
    kKBwdDwTc = 9,
    kKPackChunks = 10,
    kKBwdDxTcPacked = 11,
    kKBwdDwTf32 = 12,
    kKFilterBwdDx = 13,
    kKFilterBwdDtaps = 14,
    kKForwardTf32 = 15,
    kKBwdDyTf32 = 16,
    kKPackF32 = 17,
    kKBwdDxTf32 = 18,
    kKBwdDxGather = 19,
    kKNumKernels = 20
};

// Tracing hooks around each launch (cheap no-ops while tracing is off).
void trace_begin(cudaStream_t s, int kernel_id);
bool trace_enabled();
void trace_end(cudaStream_t s);

// ddpm_problem.flags bits: force the CUDA-core kernels (DDPM_FLAG_CUDA_CORES); allow
// TF32 tensor-core contractions in an FP32 backward (DDPM_FLAG_TF32_BACKWARD).
constexpr unsigned kFlagCudaCores = 0x2u;
constexpr unsigned kFlagTf32Backward = 0x1u;
// FP32 forward with the generator GEMM as three TF32 tensor-core products (DDPM_FLAG_TF32X3_FORWARD).
constexpr unsigned kFlagTf32x3Forward = 0x4u;

// Multiprocessor count of the current device (cached per device).
int num_sms();

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current device,
// once per device (done[] remembers the largest value set on each device).  With
// prefer_max the kernel also asks for the largest shared-memory carve-out.
inline cudaError_t set_max_dynamic_smem(const void* func, int bytes, int (&done)[64], bool prefer_max = false) {
    int dev = 0;
    const bool cached = cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64;
    if (cached && done[dev] >= bytes) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && prefer_max) e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess && cached) done[dev] = bytes;
    return e;
}

// Device address of the library's error word (set by kernels whose bounded
// waits expire).
unsigned int* device_error_word();

// Dynamic filter with pregenerated taps (README section "CUDA 动态过滤").
cudaError_t launch_filter_simt(const Dims& d, const void* x, const void* taps, void* out,
                               cudaStream_t s);
// Backward of the filter with given taps (dx and, when dtaps is non-null, the taps' gradient).
cudaError_t launch_filter_backward_simt(const Dims& d, const void* g, const void* x, const void* taps, void* dx,
                                        void* dtaps, cudaStream_t s);

// Fused generator + filter on CUDA cores (IEEE FP32 FMA; also any dtype/shape).
cudaError_t launch_forward_simt(const Dims& d, const void* x, const void* y, const void* w,
                                const void* bias, void* out, cudaStream_t s);

// Fused generator + filter on tcgen05 tensor cores (bf16, K = 3, C <= 64).
bool forward_tc_eligible(const Dims& d, const void* y, const void* w);
cudaError_t launch_forward_tc(const Dims& d, const void* x, const void* y, const void* w,
                              const void* bias, void* out, cudaStream_t s);

// FP32 fused generator + filter, generator GEMM as hi*hi + hi*lo + lo*hi TF32 products
// on tcgen05 tensor cores, filter in IEEE FP32 FMA (K = 3, C a multiple of 4 up to 64).
bool forward_tf32_eligible(const Dims& d, const void* x, const void* y, const void* w, const void* out);
cudaError_t launch_forward_tf32(const Dims& d, const void* x, const void* y, const void* w,
                                const void* bias, void* out, cudaStream_t s);

// Backward on CUDA cores: dX gather, dY, dW/dbias split partials + reduce.
size_t backward_simt_workspace(const Dims& d);
cudaError_t launch_backward_simt(const Dims& d, const void* g, const void* x, const void* y,
                                 const void* w, const void* bias, void* dx, void* dy, void* dw,
                                 void* db, void* ws, cudaStream_t s);

// Number of fp32 partial slices used for dW / dbias (at most 16).
int backward_num_splits(const Dims& d);

// The backward's pieces, launched separately so that each can run on the
// kernel that suits the problem.
cudaError_t launch_bwd_dx_simt(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                               cudaStream_t s);
cudaError_t launch_bwd_dy_simt(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s);
cudaError_t launch_bwd_dw_partial_simt(const Dims& d, const void* g, const void* x, const void* y, void* ws,
                                       cudaStream_t s);
cudaError_t launch_bwd_reduce(const Dims& d, const float* ws, int S, void* dw, void* db, cudaStream_t s);

// dW / dbias split partials on tcgen05 tensor cores (bf16, K = 3, 16 <= C <= 64).
bool bwd_dw_tc_eligible(const Dims& d, const void* g, const void* x, const void* y);
int bwd_dw_tc_splits(const Dims& d, size_t workspace_bytes);
cudaError_t launch_bwd_dw_tc(const Dims& d, const void* g, const void* x, const void* y, float* ws, int S,
                             cudaStream_t s);
bool bwd_dw_tf32_eligible(const Dims& d, const void* g, const void* x, const void* y);
int bwd_dw_tf32_splits(const Dims& d, size_t workspace_bytes);
cudaError_t launch_bwd_dw_tf32(const Dims& d, const void* g, const void* x, const void* y, float* ws, int S,
                               cudaStream_t s);

// dX on tcgen05 tensor cores: one shifted GEMM per tap (halo radius <= 6).
bool bwd_dx_tc_eligible(const Dims& d, const void* g, const void* y, const void* w);
cudaError_t launch_bwd_dx_tc(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                             cudaStream_t s);

// dX on tcgen05 tensor cores from channel-chunked copies of y and grad that the
// launcher first writes into `packed` (bwd_dx_packed_bytes(d) bytes, 16-byte
// aligned); the copies make the staging a plain TMA load (halo radius <= 6).
// The copies alone: y into packed[0, B*C*H*W) and grad blocks 1..3 after it, bf16
// [B][C/8][H][W][8] and [B][3][C/8][H][W][8] (C a multiple of 8, H*W of 8).
cudaError_t launch_pack_chunks(const Dims& d, const void* g, const void* y, void* packed, cudaStream_t s);
bool bwd_dx_packed_shape_ok(const Dims& d);   // the problem alone (sizes the workspace)
bool bwd_dx_packed_eligible(const Dims& d, const void* g, const void* y, const void* w);
size_t bwd_dx_packed_bytes(const Dims& d);
cudaError_t launch_bwd_dx_packed(const Dims& d, const void* g, const void* y, const void* w, const void* bias,
                                 void* dx, void* packed, cudaStream_t s);

// dY of FP32 problems on TF32 tensor cores (DDPM_FLAG_TF32_BACKWARD): K = 3, C a multiple
// of 16 up to 64.  Needs bwd_dy_tf32_wt_bytes(d) bytes of workspace (16-byte aligned) for
// the rearranged weight, which the launch writes first.
bool bwd_dy_tf32_shape_ok(const Dims& d);   // the problem alone (sizes the workspace)
bool bwd_dy_tf32_eligible(const Dims& d, const void* g, const void* x, const void* w, const void* dy);
size_t bwd_dy_tf32_wt_bytes(const Dims& d);
cudaError_t launch_bwd_dy_tf32(const Dims& d, const void* g, const void* x, const void* w, void* dy, void* wt,
                               cudaStream_t s);

// dX of FP32 problems on TF32 tensor cores (DDPM_FLAG_TF32_BACKWARD): K = 3, C a multiple
// of 4 up to 64, W a multiple of 4, halo radius <= 6.  The launch first writes
// channel-chunked copies of y and of grad's three dilation blocks into `packed`
// (bwd_dx_tf32_bytes(d) bytes, 16-byte aligned).
bool bwd_dx_tf32_shape_ok(const Dims& d);   // the problem alone (sizes the workspace)
bool bwd_dx_tf32_eligible(const Dims& d, const void* g, const void* y, const void* w, const void* dx);
size_t bwd_dx_tf32_bytes(const Dims& d);
cudaError_t launch_bwd_dx_tf32(const Dims& d, const void* g, const void* y, const void* w, const void* bias, void* dx,
                               void* packed, cudaStream_t s);

// bf16 dX on tcgen05 tensor cores from the same channel-chunked copies as the packed
// dX (bwd_dx_packed_bytes(d) bytes in `packed`, written by the launch), with grad
// gathered from L2: K = 3 or 5 (halo radius <= 10).  Taken for K = 5.
bool bwd_dx_gather_shape_ok(const Dims& d);
bool bwd_dx_gather_eligible(const Dims& d, const void* g, const void* y, const void* w);
cudaError_t launch_bwd_dx_gather(const Dims& d, const void* g, const void* y, const void* w, const void* bias,
                                 void* dx, void* packed, cudaStream_t s);

// dY on tcgen05 tensor cores (same shapes as the dW kernel).
bool bwd_dy_tc_eligible(const Dims& d, const void* g, const void* x, const void* w);
cudaError_t launch_bwd_dy_tc(const Dims& d, const void* g, const void* x, const void* w, void* dy, cudaStream_t s);

}  // namespace ddpm
