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
    kKBwdDyDwTc = 8,
    kKNumKernels = 9
};

// Tracing hooks around each launch (cheap no-ops while tracing is off).
void trace_begin(cudaStream_t s, int kernel_id);
void trace_end(cudaStream_t s);

// ddpm_problem.flags bit that forces the CUDA-core kernels (DDPM_FLAG_CUDA_CORES).
constexpr unsigned kFlagCudaCores = 0x2u;

// Multiprocessor count of the current device (cached per device).
int num_sms();

// Device address of the library's error word (set by kernels whose bounded
// waits expire).
unsigned int* device_error_word();

// Dynamic filter with pregenerated taps (README section "CUDA 动态过滤").
cudaError_t launch_filter_simt(const Dims& d, const void* x, const void* taps, void* out,
                               cudaStream_t s);

// Fused generator + filter on CUDA cores (IEEE FP32 FMA; also any dtype/shape).
cudaError_t launch_forward_simt(const Dims& d, const void* x, const void* y, const void* w,
                                const void* bias, void* out, cudaStream_t s);

// Fused generator + filter on tcgen05 tensor cores (bf16, K = 3, C <= 64).
bool forward_tc_eligible(const Dims& d, const void* y, const void* w);
cudaError_t launch_forward_tc(const Dims& d, const void* x, const void* y, const void* w,
                              const void* bias, void* out, cudaStream_t s);

// Backward on CUDA cores: dX gather, dY, dW/dbias split partials + reduce.
size_t backward_simt_workspace(const Dims& d);
cudaError_t launch_backward_simt(const Dims& d, const void* g, const void* x, const void* y,
                                 const void* w, const void* bias, void* dx, void* dy, void* dw,
                                 void* db, void* ws, cudaStream_t s);

// Number of fp32 partial slices used for dW / dbias (at most 16).
int backward_num_splits(const Dims& d);

}  // namespace ddpm
