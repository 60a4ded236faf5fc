// backward_noalloc.cu -- ddpm_backward_noalloc: the backward with built-in scratch.
//
// Some callers cannot hand the library a workspace: code that runs where
// cudaMalloc is off limits (a plugin inside a host application that owns all
// device memory, a real-time loop that forbids allocation after start-up, or
// a plain C caller with no allocator for temporaries).  For them this entry
// point keeps the backward's scratch -- the <= 16 FP32 dW/dbias partial sums
// -- in a fixed device array that is part of the library itself.  The whole
// array is handed to ddpm_backward as its workspace: where it also has room for
// the channel-chunked copies of y and grad (BF16 problems with small images)
// dX takes the packed kernel, as ddpm_backward would with a workspace of that
// size; otherwise dX runs on the kernel that stages its operands itself.
//
// The array is a file-scope __device__ object of DDPM_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads this library holds it until the process exits.  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should therefore come before any
// stream capture.  The address is kept for the life of the process: after a
// cudaDeviceReset it would no longer be the array's, so this entry point must
// not be called again after one.  All calls share the one array, and it keeps whatever the
// last call left in it.  Nothing in it needs to start at zero: the partial
// kernel overwrites every slot the reduce kernel then reads.  Two calls whose
// work overlaps on the GPU (different streams, or different host threads on
// the same device) race on the array and give wrong results.
#include <mutex>

#include "../../include/ddpm.h"
#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DDPM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
ddpm_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DDPM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DDPM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return DDPM_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DDPM_OK;
}

}  // namespace

namespace ddpm {
ddpm_status backward_workspace_min(const ddpm_problem* problem, size_t* bytes);  // api.cu
}

extern "C" ddpm_status ddpm_backward_noalloc(const ddpm_problem* problem, const void* grad_out, const void* x,
                                             const void* y, const void* weight, const void* bias, void* dx,
                                             void* dy, void* dweight, void* dbias, ddpm_stream_t stream) {
    size_t need = 0;
    const ddpm_status s = ddpm::backward_workspace_min(problem, &need);  // validates the problem
    if (s != DDPM_OK) return s;
    if (need > DDPM_NOALLOC_SCRATCH_BYTES) return DDPM_ERR_UNSUPPORTED;  // partials exceed the fixed scratch
    void* scratch = nullptr;
    const ddpm_status a = scratch_address(&scratch);
    if (a != DDPM_OK) return a;
    return ddpm_backward(problem, grad_out, x, y, weight, bias, dx, dy, dweight, dbias, scratch,
                         DDPM_NOALLOC_SCRATCH_BYTES, stream);
}
