// diag.cu -- ddpm_debug_wait_probe: exercises the bounded-wait failure path.
//
// Every tensor-core kernel of the library waits on shared-memory mbarriers with
// a time limit; when a limit runs out, the waiting thread records a timeout in
// the library's device error word, raises the block's abort flag so that the
// block's other waiters leave too, and the block frees its tensor memory and
// returns -- it never traps, so the CUDA context stays usable.  This probe runs
// that path on purpose with a short limit: a block with the kernels' warp roles
// (one warp owning a TMEM allocation, one waiting on a barrier that nothing
// arrives on, two waiting on a barrier that the first waiter would arrive on
// only after its own wait) so that a test can check the error status the host
// then reads and that the next calls on the same context still work.
#include "../../include/ddpm.h"
#include "launch.h"
#include "tc.cuh"

namespace ddpm {
namespace {

constexpr int kProbeThreads = 128;

__global__ void __launch_bounds__(kProbeThreads, 1)
    wait_probe_kernel(unsigned long long limit_ns, unsigned int* err) {
    using namespace tc;
    __shared__ uint64_t never, after;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    volatile int* abort_v = &abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&never, 1);   // nothing ever arrives
        mbar_init(&after, 1);   // warp 0 arrives once its own wait has succeeded
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(&tmem_slot, 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        if (lane == 0 && mbar_wait_for(&never, 0, err, abort_v, limit_ns)) mbar_arrive(&after);
    } else if (warp >= 2) {
        // leave through the abort flag (or, failing that, the library's own limit)
        if (lane == 0) mbar_wait(&after, 0, err, abort_v);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_slot, 32);
    }
}

}  // namespace
}  // namespace ddpm

extern "C" ddpm_status ddpm_debug_wait_probe(unsigned int limit_us, ddpm_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000u) return DDPM_ERR_INVALID_ARGUMENT;
    unsigned int* err = ddpm::device_error_word();
    if (err == nullptr) return DDPM_ERR_CUDA;
    ddpm::wait_probe_kernel<<<2, ddpm::kProbeThreads, 0, (cudaStream_t)stream>>>(1000ull * limit_us, err);
    return cudaGetLastError() == cudaSuccess ? DDPM_OK : DDPM_ERR_CUDA;
}
