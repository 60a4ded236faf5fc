// api.cu -- the C ABI of libddpm_gb300.so (declared in include/ddpm.h).
//
// Host-side validation, kernel selection and launch on the caller's stream.
// The library never allocates device memory, never synchronises (except in
// ddpm_get_device_error) and never throws across the boundary.  The backward's
// three independent pieces (dX, dY, dW) run side by side: dY and dW on two
// library streams forked from and joined back into the caller's stream.
#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/ddpm.h"
#include "launch.h"

namespace ddpm {

// Device-side error word: kernels with bounded waits set a nonzero code here
// when a wait expires, instead of trapping.  Passed to kernels by address.
__device__ unsigned int g_device_error = 0;

unsigned int* device_error_word() {
    static std::mutex mu;
    static unsigned int* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned int*>(p);
    }
    return addr[dev];
}

int num_sms() {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// Two non-blocking streams per device, and the events that fork them from and join
// them back into a caller's stream.  The events are re-recorded by every call, so a
// call holds g_side_mu from the fork to the join.
struct SideStreams {
    cudaStream_t s[2];
    cudaEvent_t fork, join[2];
};

std::mutex g_side_mu;

cudaError_t side_streams(SideStreams** out) {
    static SideStreams side[64];
    static bool ready[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev]) {
        SideStreams& t = side[dev];
        for (int i = 0; i < 2; ++i)
            if ((e = cudaStreamCreateWithFlags(&t.s[i], cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&t.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int i = 0; i < 2; ++i)
            if ((e = cudaEventCreateWithFlags(&t.join[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        ready[dev] = true;
    }
    *out = &side[dev];
    return cudaSuccess;
}

}  // namespace ddpm

namespace {

using ddpm::Dims;

constexpr size_t kMaxSmem = 227 * 1024;

size_t elem_size(int dtype) { return dtype == DDPM_BFLOAT16 ? 2 : 4; }

// Workspace layout of ddpm_backward: the FP32 dW/dbias partial sums (the minimum
// a caller must supply), then -- when the workspace is large enough -- for BF16
// problems the channel-chunked copies of y and grad that the packed dX kernel
// reads, for FP32 problems with TF32 contractions the rearranged weight that the
// TF32 dY kernel reads.
size_t packed_offset(const Dims& d) { return (ddpm::backward_simt_workspace(d) + 255) & ~size_t(255); }

// FP32 workspace after the partials: the TF32 dY's rearranged weight, then (256-byte
// aligned) the TF32 dX's channel-chunked copy of y.  The offsets depend on the problem
// alone, so a workspace sized for both serves either.
size_t dx_tf32_offset(const Dims& d) {
    const size_t wt = ddpm::bwd_dy_tf32_shape_ok(d) ? ddpm::bwd_dy_tf32_wt_bytes(d) : 0;
    return (packed_offset(d) + wt + 255) & ~size_t(255);
}

ddpm_status validate(const ddpm_problem* p, Dims* d) {
    if (p == nullptr) return DDPM_ERR_INVALID_ARGUMENT;
    if (p->B < 1 || p->C < 1 || p->H < 1 || p->W < 1) return DDPM_ERR_INVALID_ARGUMENT;
    if (p->K < 1 || p->K % 2 == 0) return DDPM_ERR_INVALID_ARGUMENT;
    if (p->dtype != DDPM_FLOAT32 && p->dtype != DDPM_BFLOAT16) return DDPM_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < 3; ++i)
        if (p->dilations[i] < 1) return DDPM_ERR_INVALID_ARGUMENT;
    if ((p->flags & ~(DDPM_FLAG_TF32_BACKWARD | DDPM_FLAG_CUDA_CORES | DDPM_FLAG_TF32X3_FORWARD)) != 0)
        return DDPM_ERR_INVALID_ARGUMENT;
    if (p->K > 7) return DDPM_ERR_UNSUPPORTED;
    // grid-dimension and index-width limits of this build
    if (p->B > 65535 || p->C > 65535) return DDPM_ERR_UNSUPPORTED;
    for (int i = 0; i < 3; ++i)
        if (p->dilations[i] > (1 << 20)) return DDPM_ERR_UNSUPPORTED;
    const long long HW = (long long)p->H * p->W;
    if (HW > INT_MAX) return DDPM_ERR_UNSUPPORTED;
    const long long O = 3LL * p->C * p->K * p->K;
    // largest tensor: taps [B, O, H, W]; keep every flat index inside int64 with margin
    if ((double)p->B * (double)O * (double)HW > 4.0e18) return DDPM_ERR_UNSUPPORTED;
    // shared-memory staging of the CUDA-core kernels
    const long long K2 = (long long)p->K * p->K;
    const long long KP = (K2 + 3) / 4 * 4;
    if ((size_t)p->C * KP * sizeof(float) > kMaxSmem) return DDPM_ERR_UNSUPPORTED;
    if ((size_t)p->C * 8 * sizeof(float) > kMaxSmem) return DDPM_ERR_UNSUPPORTED;
    d->B = p->B; d->C = p->C; d->H = p->H; d->W = p->W; d->K = p->K; d->r = p->K / 2;
    for (int i = 0; i < 3; ++i) d->dil[i] = p->dilations[i];
    d->dtype = p->dtype;
    d->flags = p->flags;
    d->HW = HW;
    d->O = O;
    return DDPM_OK;
}

ddpm_status check_ptr(const void* ptr, size_t align, bool nullable) {
    if (ptr == nullptr) return nullable ? DDPM_OK : DDPM_ERR_INVALID_ARGUMENT;
    if ((uintptr_t)ptr % align != 0) return DDPM_ERR_MISALIGNED;
    return DDPM_OK;
}

#define DDPM_TRY(expr)                         \
    do {                                       \
        const ddpm_status s_ = (expr);         \
        if (s_ != DDPM_OK) return s_;          \
    } while (0)

ddpm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DDPM_OK : DDPM_ERR_CUDA; }

}  // namespace

namespace ddpm {
ddpm_status backward_workspace_min(const ddpm_problem* problem, size_t* bytes);
}

extern "C" {

ddpm_status ddpm_forward(const ddpm_problem* problem, const void* x, const void* y, const void* weight,
                         const void* bias, void* out, ddpm_stream_t stream) {
    Dims d;
    DDPM_TRY(validate(problem, &d));
    const size_t es = elem_size(d.dtype);
    DDPM_TRY(check_ptr(x, es, false));
    DDPM_TRY(check_ptr(y, es, false));
    DDPM_TRY(check_ptr(weight, es, false));
    DDPM_TRY(check_ptr(bias, es, true));
    DDPM_TRY(check_ptr(out, es, false));
    try {
        if (ddpm::forward_tc_eligible(d, y, weight) && (uintptr_t)x % 16 == 0)
            return from_cuda(ddpm::launch_forward_tc(d, x, y, weight, bias, out, (cudaStream_t)stream));
        if (ddpm::forward_tf32_eligible(d, x, y, weight, out))
            return from_cuda(ddpm::launch_forward_tf32(d, x, y, weight, bias, out, (cudaStream_t)stream));
        return from_cuda(ddpm::launch_forward_simt(d, x, y, weight, bias, out, (cudaStream_t)stream));
    } catch (...) {
        return DDPM_ERR_CUDA;
    }
}

ddpm_status ddpm_filter_pregenerated(const ddpm_problem* problem, const void* x, const void* taps, void* out,
                                     ddpm_stream_t stream) {
    Dims d;
    DDPM_TRY(validate(problem, &d));
    const size_t es = elem_size(d.dtype);
    DDPM_TRY(check_ptr(x, es, false));
    DDPM_TRY(check_ptr(taps, es, false));
    DDPM_TRY(check_ptr(out, es, false));
    try {
        return from_cuda(ddpm::launch_filter_simt(d, x, taps, out, (cudaStream_t)stream));
    } catch (...) {
        return DDPM_ERR_CUDA;
    }
}

ddpm_status ddpm_filter_pregenerated_backward(const ddpm_problem* problem, const void* grad_out, const void* x,
                                              const void* taps, void* dx, void* dtaps, ddpm_stream_t stream) {
    Dims d;
    DDPM_TRY(validate(problem, &d));
    const size_t es = elem_size(d.dtype);
    DDPM_TRY(check_ptr(grad_out, es, false));
    DDPM_TRY(check_ptr(x, es, false));
    DDPM_TRY(check_ptr(taps, es, false));
    DDPM_TRY(check_ptr(dx, es, false));
    DDPM_TRY(check_ptr(dtaps, es, true));
    try {
        return from_cuda(ddpm::launch_filter_backward_simt(d, grad_out, x, taps, dx, dtaps, (cudaStream_t)stream));
    } catch (...) {
        return DDPM_ERR_CUDA;
    }
}

ddpm_status ddpm_backward_workspace_size(const ddpm_problem* problem, size_t* bytes) {
    Dims d;
    DDPM_TRY(validate(problem, &d));
    if (bytes == nullptr) return DDPM_ERR_INVALID_ARGUMENT;
    if (ddpm::bwd_dx_packed_shape_ok(d) || (d.K != 3 && ddpm::bwd_dx_gather_shape_ok(d)))
        *bytes = packed_offset(d) + ddpm::bwd_dx_packed_bytes(d);
    else if (ddpm::bwd_dx_tf32_shape_ok(d))
        *bytes = dx_tf32_offset(d) + ddpm::bwd_dx_tf32_bytes(d);
    else if (ddpm::bwd_dy_tf32_shape_ok(d))
        *bytes = packed_offset(d) + ddpm::bwd_dy_tf32_wt_bytes(d);
    else
        *bytes = ddpm::backward_simt_workspace(d);
    return DDPM_OK;
}

ddpm_status ddpm_backward_workspace_min_size(const ddpm_problem* problem, size_t* bytes) {
    return ddpm::backward_workspace_min(problem, bytes);
}

ddpm_status ddpm_backward(const ddpm_problem* problem, const void* grad_out, const void* x, const void* y,
                          const void* weight, const void* bias, void* dx, void* dy, void* dweight,
                          void* dbias, void* workspace, size_t workspace_bytes, ddpm_stream_t stream) {
    Dims d;
    DDPM_TRY(validate(problem, &d));
    const size_t es = elem_size(d.dtype);
    DDPM_TRY(check_ptr(grad_out, es, false));
    DDPM_TRY(check_ptr(x, es, false));
    DDPM_TRY(check_ptr(y, es, false));
    DDPM_TRY(check_ptr(weight, es, false));
    DDPM_TRY(check_ptr(bias, es, true));
    DDPM_TRY(check_ptr(dx, es, false));
    DDPM_TRY(check_ptr(dy, es, false));
    DDPM_TRY(check_ptr(dweight, es, false));
    DDPM_TRY(check_ptr(dbias, es, true));
    DDPM_TRY(check_ptr(workspace, 16, false));
    if (workspace_bytes < ddpm::backward_simt_workspace(d)) return DDPM_ERR_WORKSPACE_TOO_SMALL;
    try {
        const cudaStream_t s = (cudaStream_t)stream;
        // each piece runs on the tensor-core kernel where one exists for the problem;
        // dX takes the packed-operand kernel when the workspace also holds the copies
        const size_t poff = packed_offset(d);
        const bool packed = ddpm::bwd_dx_packed_eligible(d, grad_out, y, weight) &&
                            workspace_bytes >= poff + ddpm::bwd_dx_packed_bytes(d);
        // halos whose grad windows do not fit the packed kernel's shared memory (K = 5)
        const bool gather = !packed && d.K != 3 && ddpm::bwd_dx_gather_eligible(d, grad_out, y, weight) &&
                            workspace_bytes >= poff + ddpm::bwd_dx_packed_bytes(d);
        const bool dy_tf32 = ddpm::bwd_dy_tf32_eligible(d, grad_out, x, weight, dy) &&
                             workspace_bytes >= poff + ddpm::bwd_dy_tf32_wt_bytes(d);
        const size_t xoff = dx_tf32_offset(d);
        const bool dx_tf32 = ddpm::bwd_dx_tf32_eligible(d, grad_out, y, weight, dx) &&
                             workspace_bytes >= xoff + ddpm::bwd_dx_tf32_bytes(d);
        const size_t part_bytes = (packed || gather || dy_tf32 || dx_tf32) ? poff : workspace_bytes;
        // dX on the caller's stream, dY and dW (+ reduce) on the two side streams: the
        // pieces share only inputs, and each one's last partial wave of CTAs leaves SMs
        // that the others fill.  While kernels are traced the pieces run one after
        // another on the caller's stream, so each traced interval holds one kernel.
        const bool fork = !ddpm::trace_enabled();
        std::lock_guard<std::mutex> lock(ddpm::g_side_mu);
        ddpm::SideStreams* ss = nullptr;
        cudaError_t e = ddpm::side_streams(&ss);
        if (e != cudaSuccess) return from_cuda(e);
        const cudaStream_t s_dy = fork ? ss->s[0] : s, s_dw = fork ? ss->s[1] : s;
        if (fork) {
            if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return from_cuda(e);
            for (int i = 0; i < 2; ++i)
                if ((e = cudaStreamWaitEvent(ss->s[i], ss->fork, 0)) != cudaSuccess) return from_cuda(e);
        }
        if (packed)
            e = ddpm::launch_bwd_dx_packed(d, grad_out, y, weight, bias, dx, static_cast<char*>(workspace) + poff, s);
        else if (ddpm::bwd_dx_tc_eligible(d, grad_out, y, weight))
            e = ddpm::launch_bwd_dx_tc(d, grad_out, y, weight, bias, dx, s);
        else if (gather)
            e = ddpm::launch_bwd_dx_gather(d, grad_out, y, weight, bias, dx, static_cast<char*>(workspace) + poff, s);
        else if (dx_tf32)
            e = ddpm::launch_bwd_dx_tf32(d, grad_out, y, weight, bias, dx, static_cast<char*>(workspace) + xoff, s);
        else
            e = ddpm::launch_bwd_dx_simt(d, grad_out, y, weight, bias, dx, s);
        if (e == cudaSuccess) {
            if (ddpm::bwd_dy_tc_eligible(d, grad_out, x, weight))
                e = ddpm::launch_bwd_dy_tc(d, grad_out, x, weight, dy, s_dy);
            else if (dy_tf32)
                e = ddpm::launch_bwd_dy_tf32(d, grad_out, x, weight, dy, static_cast<char*>(workspace) + poff, s_dy);
            else
                e = ddpm::launch_bwd_dy_simt(d, grad_out, x, weight, dy, s_dy);
        }
        if (e == cudaSuccess) {
            const cudaStream_t sw = s_dw;
            if (ddpm::bwd_dw_tc_eligible(d, grad_out, x, y)) {
                const int S = ddpm::bwd_dw_tc_splits(d, part_bytes);
                e = ddpm::launch_bwd_dw_tc(d, grad_out, x, y, (float*)workspace, S, sw);
                if (e == cudaSuccess) e = ddpm::launch_bwd_reduce(d, (const float*)workspace, S, dweight, dbias, sw);
            } else if (ddpm::bwd_dw_tf32_eligible(d, grad_out, x, y)) {
                const int S = ddpm::bwd_dw_tf32_splits(d, part_bytes);
                e = ddpm::launch_bwd_dw_tf32(d, grad_out, x, y, (float*)workspace, S, sw);
                if (e == cudaSuccess) e = ddpm::launch_bwd_reduce(d, (const float*)workspace, S, dweight, dbias, sw);
            } else {
                e = ddpm::launch_bwd_dw_partial_simt(d, grad_out, x, y, workspace, sw);
                if (e == cudaSuccess)
                    e = ddpm::launch_bwd_reduce(d, (const float*)workspace, ddpm::backward_num_splits(d), dweight,
                                                dbias, sw);
            }
        }
        // join, whatever happened above, so the side streams never run ahead of `stream`
        for (int i = 0; i < 2 && fork; ++i) {
            const cudaError_t er = cudaEventRecord(ss->join[i], ss->s[i]);
            const cudaError_t ew = er == cudaSuccess ? cudaStreamWaitEvent(s, ss->join[i], 0) : er;
            if (e == cudaSuccess) e = ew;
        }
        return from_cuda(e);
    } catch (...) {
        return DDPM_ERR_CUDA;
    }
}

ddpm_status ddpm_get_device_error(ddpm_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DDPM_ERR_CUDA;
    unsigned int* word = ddpm::device_error_word();
    if (word == nullptr) return DDPM_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DDPM_ERR_CUDA;
    if (v != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return DDPM_ERR_CUDA;
        return DDPM_ERR_DEVICE_TIMEOUT;
    }
    return DDPM_OK;
}

const char* ddpm_status_string(ddpm_status status) {
    switch (status) {
        case DDPM_OK: return "DDPM_OK";
        case DDPM_ERR_INVALID_ARGUMENT: return "DDPM_ERR_INVALID_ARGUMENT: invalid argument";
        case DDPM_ERR_UNSUPPORTED: return "DDPM_ERR_UNSUPPORTED: problem outside what this build implements";
        case DDPM_ERR_MISALIGNED: return "DDPM_ERR_MISALIGNED: pointer not aligned to its element size";
        case DDPM_ERR_WORKSPACE_TOO_SMALL: return "DDPM_ERR_WORKSPACE_TOO_SMALL: workspace below the queried size";
        case DDPM_ERR_CUDA: return "DDPM_ERR_CUDA: a CUDA call or kernel launch failed";
        case DDPM_ERR_DEVICE_TIMEOUT: return "DDPM_ERR_DEVICE_TIMEOUT: a kernel's bounded wait expired";
    }
    return "DDPM: unknown status";
}

int ddpm_version(void) { return 100; }

}  // extern "C"

namespace ddpm {

// Smallest workspace ddpm_backward accepts (the FP32 dW/dbias partial sums).
ddpm_status backward_workspace_min(const ddpm_problem* problem, size_t* bytes) {
    Dims d;
    DDPM_TRY(validate(problem, &d));
    if (bytes == nullptr) return DDPM_ERR_INVALID_ARGUMENT;
    *bytes = backward_simt_workspace(d);
    return DDPM_OK;
}

}  // namespace ddpm
