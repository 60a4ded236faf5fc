// trace.cu -- optional per-kernel device timing (ddpm_trace_enable / ddpm_trace_read).
//
// While tracing is on, each launch site calls trace_begin / trace_end, which
// record a pair of CUDA events on the launching stream.  Events come from a
// pool that is reused across reads, so steady-state tracing creates nothing.
#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/ddpm.h"
#include "launch.h"

namespace ddpm {
namespace {

struct Record {
    int id;
    cudaEvent_t start, stop;
};

constexpr size_t kMaxRecords = 65536;

std::atomic<bool> g_enabled{false};
std::mutex g_mu;
std::vector<Record> g_records;
std::vector<cudaEvent_t> g_pool;
bool g_open = false;  // a begin without its end yet

cudaEvent_t take_event() {
    if (!g_pool.empty()) {
        cudaEvent_t e = g_pool.back();
        g_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

const char* const kNames[kKNumKernels] = {
    "filter_pregenerated_simt", "forward_simt", "forward_tc", "bwd_dx_simt", "bwd_dy_simt",
    "bwd_dw_partial_simt", "bwd_dw_reduce", "bwd_dx_tc", "bwd_dy_tc", "bwd_dw_tc",
    "pack_chunks", "bwd_dx_tc_packed", "bwd_dw_tf32", "filter_bwd_dx", "filter_bwd_dtaps", "forward_tf32",
    "bwd_dy_tf32", "pack_f32", "bwd_dx_tf32", "bwd_dx_gather",
};

}  // namespace

void trace_begin(cudaStream_t s, int kernel_id) {
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    g_open = false;
    if (g_records.size() >= kMaxRecords) return;
    Record r{kernel_id, take_event(), take_event()};
    if (r.start == nullptr || r.stop == nullptr || cudaEventRecord(r.start, s) != cudaSuccess) {
        if (r.start) g_pool.push_back(r.start);
        if (r.stop) g_pool.push_back(r.stop);
        return;
    }
    g_records.push_back(r);
    g_open = true;
}

bool trace_enabled() { return g_enabled.load(std::memory_order_relaxed); }

void trace_end(cudaStream_t s) {
    if (!g_enabled.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_open || g_records.empty()) return;
    cudaEventRecord(g_records.back().stop, s);
    g_open = false;
}

// Eight independent FMA chains per thread: with every SM full, the FP32 pipes
// issue one FMA per lane per cycle once each chain's latency is covered.  a and b
// come from the host, so nothing folds; the sum is written only if it takes a
// value it cannot reach, which keeps the chains live.
__device__ float g_ffma_sink;

__global__ void __launch_bounds__(256) ffma_chain_kernel(int iters, float a, float b) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 1e-3f * (float)threadIdx.x + (float)i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = fmaf(v[i], a, b);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i];
    if (s == -1.0f) g_ffma_sink = s;
}

}  // namespace ddpm

extern "C" {

ddpm_status ddpm_measure_ffma_tflops(double* tflops) {
    using namespace ddpm;
    if (tflops == nullptr) return DDPM_ERR_INVALID_ARGUMENT;
    const int blocks = num_sms() * 8, threads = 256, iters = 4096;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return DDPM_ERR_CUDA;
    ddpm_status st = DDPM_OK;
    float best = 1e30f;
    for (int rep = 0; rep < 4 && st == DDPM_OK; ++rep) {
        cudaEventRecord(e0, nullptr);
        ffma_chain_kernel<<<blocks, threads>>>(iters, 0.999999f, 1e-7f);
        cudaEventRecord(e1, nullptr);
        float ms = 0.0f;
        if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
            cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
            st = DDPM_ERR_CUDA;
        else if (rep > 0 && ms < best)
            best = ms;   // the first launch is a warm-up
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != DDPM_OK) return st;
    const double flops = 2.0 * 32.0 * (double)iters * (double)blocks * (double)threads;
    *tflops = flops / ((double)best * 1e-3) / 1e12;
    return DDPM_OK;
}

ddpm_status ddpm_trace_enable(int enable) {
    ddpm::g_enabled.store(enable != 0);
    return DDPM_OK;
}

int ddpm_trace_read(int* kernel_ids, float* milliseconds, int max_records) {
    using namespace ddpm;
    std::lock_guard<std::mutex> lock(g_mu);
    int n = 0;
    int rc = 0;
    for (const Record& r : g_records) {
        float ms = -1.0f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            rc = -1;
        if (n < max_records && kernel_ids != nullptr && milliseconds != nullptr) {
            kernel_ids[n] = r.id;
            milliseconds[n] = ms;
            ++n;
        }
        g_pool.push_back(r.start);
        g_pool.push_back(r.stop);
    }
    g_records.clear();
    g_open = false;
    return rc < 0 ? -1 : n;
}

const char* ddpm_kernel_name(int kernel_id) {
    if (kernel_id < 0 || kernel_id >= ddpm::kKNumKernels) return "unknown";
    return ddpm::kNames[kernel_id];
}

}  // extern "C"
