/*
 * ddpm.h -- C ABI of the GB300 (sm_103a) DDPM core library, libddpm_gb300.so.
 *
 * The Dynamic Dilated Pyramid Module core of HDFNet (ECCV 2020), as described
 * in the "lartpang/DynamicConvolutionOperator" README:
 *
 *   taps  T[b,o,h,w] = bias[o] + sum_j weight[o,j] * y[b,j,h,w]      (1x1 generator)
 *         with o = (di*C + c)*K*K + ky*K + kx, di indexing the three dilations;
 *   out   [B,4C,H,W] = [x, d1, d3, d5], where
 *         out[b,(1+di)*C+c,h,w] = sum_{ky,kx} T[b,o,h,w] * x[b,c,h+(ky-r)d,w+(kx-r)d],
 *         r = K/2, d = dilations[di], x = 0 outside the image (Unfold semantics).
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, contiguous, NCHW (weight [O, C], bias [O]) with
 *     O = 3*C*K*K, and all share the problem's dtype.
 *   - Every pointer is a DEVICE pointer owned by the caller.  The library never
 *     allocates device memory, frees or synchronises; it enqueues kernels on
 *     `stream` (NULL = the legacy default stream) and returns.  The backward
 *     also runs pieces on two streams of its own per device, forked from and
 *     joined back into `stream` with events: its work still starts after the
 *     work before it on `stream` and ends before the work after it.  The first
 *     backward call on a device creates those streams; make it before any
 *     stream capture.  Inputs are read-only; outputs are
 *     fully overwritten (no accumulation into them).  Outputs must not alias
 *     inputs.
 *   - Pointers must be aligned to the element size; 16-byte alignment enables
 *     the vectorised paths but is not required.
 *   - Arguments are validated on the host before anything is enqueued; on any
 *     error nothing is enqueued.  A launch failure maps to DDPM_ERR_CUDA.
 *     No C++ exception crosses this boundary.
 *   - Reductions accumulate in FP32.  FP32 problems compute the forward with
 *     IEEE FP32 FMA; BF16 problems round each generated tap to bf16 (round to
 *     nearest even) before the filter uses it, as the page's precision policy
 *     states (section "CUDA Flash 式融合训练", last paragraph).
 */
#ifndef DDPM_GB300_H
#define DDPM_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__) || defined(__clang__)
#define DDPM_API __attribute__((visibility("default")))
#else
#define DDPM_API
#endif

struct CUstream_st;
/* Same type as cudaStream_t / CUstream; NULL selects the legacy default stream. */
typedef struct CUstream_st* ddpm_stream_t;

typedef enum {
    DDPM_OK = 0,
    DDPM_ERR_INVALID_ARGUMENT = 1,    /* bad shape, NULL pointer, even K, dilation < 1 ... */
    DDPM_ERR_UNSUPPORTED = 2,         /* valid but outside what this build implements */
    DDPM_ERR_MISALIGNED = 3,          /* a pointer is not aligned to its element size */
    DDPM_ERR_WORKSPACE_TOO_SMALL = 4, /* ddpm_backward workspace below the queried size */
    DDPM_ERR_CUDA = 5,                /* a CUDA runtime call or a launch failed */
    DDPM_ERR_DEVICE_TIMEOUT = 6       /* a kernel's bounded wait expired (ddpm_get_device_error) */
} ddpm_status;

typedef enum { DDPM_FLOAT32 = 0, DDPM_BFLOAT16 = 1 } ddpm_dtype;

/* Flags for ddpm_problem.flags.
 * DDPM_FLAG_TF32_BACKWARD: FP32 problems may run the backward contractions on
 *   TF32 tensor cores (the page allows TF32 for FP32 backward reductions and
 *   recompute, never for the forward).  With it the dW/dbias partial sums run
 *   on tensor cores (TF32 operands, FP32 accumulation) for C <= 64, W a
 *   multiple of 4, 16-byte aligned tensors and K = 3 with dilations <= 6 or
 *   K = 5 with dilations <= 5.  For K = 3 so does dY
 *   where C is also a multiple of 16 and the workspace holds the rearranged
 *   weight, and so does dX's recompute of the taps (T = bias + W y as a TF32
 *   GEMM per tap, FP32 accumulation; the products T * grad and their sum stay
 *   IEEE FP32) where C is a multiple of 4 and the workspace holds
 *   channel-chunked FP32 copies of y and of grad's three dilation blocks.
 *   ddpm_backward_workspace_size counts both.
 *   Ignored for BF16 and under DDPM_FLAG_CUDA_CORES. */
#define DDPM_FLAG_TF32_BACKWARD 0x1u
/* DDPM_FLAG_CUDA_CORES: run the CUDA-core (FFMA) kernels even where a
 *   tensor-core kernel exists for the problem (BF16 forward / backward). */
#define DDPM_FLAG_CUDA_CORES 0x2u
/* DDPM_FLAG_TF32X3_FORWARD: FP32 problems compute the forward's generator GEMM on
 *   TF32 tensor cores as three products of split operands, a = hi + lo with
 *   hi = tf32(a): hi_y*hi_W + hi_y*lo_W + lo_y*hi_W, accumulated in FP32 (about
 *   2^-21 relative error per product, within the FP32 forward tolerance); the
 *   dynamic filter stays IEEE FP32 FMA.  The page lists tf32x3 among the
 *   variants it tried for the FP32 forward and did not adopt on its card
 *   (section "已验证但未采用的方案"); without the flag the FP32 forward is the
 *   page's IEEE FP32 dot.  Applies for K = 3 with halo radius <= 5 or K = 5 with
 *   halo radius <= 10 (up to 8 and 12 on images narrower than 64 pixels), C a
 *   multiple of 4 up to 64, W a multiple of 4 and 16-byte aligned tensors; other
 *   FP32 problems run the IEEE kernel.  Ignored for BF16 and under
 *   DDPM_FLAG_CUDA_CORES. */
#define DDPM_FLAG_TF32X3_FORWARD 0x4u

typedef struct {
    int B, C, H, W;    /* batch, channels, height, width: all >= 1 */
    int K;             /* kernel size: odd, 1 <= K <= 7 */
    int dilations[3];  /* the three pyramid dilations, each >= 1; (1,3,5) in the method */
    int dtype;         /* a ddpm_dtype */
    unsigned flags;    /* DDPM_FLAG_* bits */
} ddpm_problem;

/*
 * ddpm_forward -- fused generator + dynamic dilated depthwise filter.
 * Source: README section "CUDA 融合生成器推理" (fused generator inference:
 * y tile -> dot(weight, y) -> dynamic taps -> consume with shifted x -> output;
 * taps live only on chip) and "CUDA 动态过滤" (output [x, d1, d3, d5]).
 *   x, y    [B, C, H, W]   inputs
 *   weight  [O, C]         generator weight, O = 3*C*K*K
 *   bias    [O] or NULL    generator bias (NULL = zero bias)
 *   out     [B, 4C, H, W]  output; out[:, :C] is a bit-exact copy of x
 * The taps are never written to global memory.
 */
DDPM_API ddpm_status ddpm_forward(const ddpm_problem* problem, const void* x, const void* y,
                         const void* weight, const void* bias, void* out, ddpm_stream_t stream);

/*
 * ddpm_filter_pregenerated -- the dynamic filter alone, taps given.
 * Source: README section "CUDA 动态过滤" (with the dynamic kernels already
 * generated, one kernel handles dilations (1,3,5), reads the neighbourhood per
 * spatial tile, accumulates in FP32 and writes [x, d1, d3, d5] without Unfold).
 *   x     [B, C, H, W]
 *   taps  [B, O, H, W]    channel o = (di*C + c)*K*K + ky*K + kx; used as given
 *   out   [B, 4C, H, W]
 */
DDPM_API ddpm_status ddpm_filter_pregenerated(const ddpm_problem* problem, const void* x, const void* taps,
                                     void* out, ddpm_stream_t stream);

/*
 * ddpm_filter_pregenerated_backward -- gradients of L = <grad_out, out> for
 * ddpm_filter_pregenerated.  Source: README section "CUDA 动态过滤" (with the
 * taps given, the backward forms dX and dK directly, without a patch matrix):
 *   dx[b,c,q]    = grad[b,c,q] + sum_{di,ky,kx} taps[b,o,q-off] * grad[b,(1+di)C+c,q-off]
 *                  (terms whose q-off lies outside the image are dropped);
 *   dtaps[b,o,p] = grad[b,(1+di)C+c,p] * x[b,c,p+off]  (0 where p+off lies outside),
 *   o = (di*C + c)*K*K + ky*K + kx, off = ((ky-K/2)*d, (kx-K/2)*d), d = dilations[di].
 * Products and sums in FP32, each output rounded once to the problem's dtype.
 *   grad_out  [B, 4C, H, W];  x [B, C, H, W];  taps [B, O, H, W]
 *   dx        [B, C, H, W]    output
 *   dtaps     [B, O, H, W]    output, or NULL to compute dx alone
 */
DDPM_API ddpm_status ddpm_filter_pregenerated_backward(const ddpm_problem* problem, const void* grad_out,
                                                      const void* x, const void* taps, void* dx, void* dtaps,
                                                      ddpm_stream_t stream);

/*
 * ddpm_backward_workspace_size -- bytes of device workspace ddpm_backward needs.
 * Host only; enqueues nothing.  The workspace holds at most 16 FP32 partial
 * sums of [O, C+1] (dW and dbias), per README section "CUDA Flash 式融合训练"
 * (dWeight/dbias: split tokens into at most 16 FP32 partials, reduce them in a
 * second short kernel): 16 * O * (C+1) * 4 bytes at most, independent of the
 * image size (7.2 MB for C = 64, K = 3).  For BF16 problems whose dX runs on the
 * packed tensor-core kernel, the returned size also covers channel-chunked
 * copies of y and of the three dilation blocks of grad (4 * B * C * H * W bf16
 * elements, which does grow with the image); for FP32 problems whose dY and dX
 * run on TF32 tensor cores, a rearranged copy of the weight (27 * C * C FP32
 * values) and channel-chunked copies of y and of the three dilation blocks of
 * grad (4 * B * C * H * W FP32 values, which grow with the image).  ddpm_backward accepts any workspace of at least the
 * partials' size; with less than the returned size a BF16 dX stages its
 * operands inside the kernel, and an FP32 dY or dX that finds no room for its
 * copy runs on CUDA cores.
 */
DDPM_API ddpm_status ddpm_backward_workspace_size(const ddpm_problem* problem, size_t* bytes);

/*
 * ddpm_backward_workspace_min_size -- the smallest workspace ddpm_backward
 * accepts: the <= 16 FP32 partial sums of [O, C+1] alone (same section), i.e. at
 * most 16 * O * (C+1) * 4 bytes whatever the image size.  With a workspace of
 * this size dX stages its operands inside the kernel.  Host only.
 */
DDPM_API ddpm_status ddpm_backward_workspace_min_size(const ddpm_problem* problem, size_t* bytes);

/*
 * ddpm_backward -- gradients of L = <grad_out, out> for ddpm_forward.
 * Source: README section "CUDA Flash 式融合训练":
 *   dX : recompute the taps and gather each dilation's contribution
 *        dx[b,c,q] = grad[b,c,q] + sum_{di,ky,kx} T[b,o,q-off] * grad[b,(1+di)C+c,q-off];
 *   dY : form dK = shifted(x) * grad on chip and contract with the weight,
 *        dy[b,j,p] = sum_o weight[o,j] * dK[b,o,p];
 *   dW, dbias : spatial reductions of dK, dW[o,j] = sum_{b,p} dK[b,o,p] y[b,j,p],
 *        dbias[o] = sum_{b,p} dK[b,o,p], via <= 16 FP32 partials + a reduce kernel.
 * Taps are recomputed, never materialised.  In BF16 the tap rounding is
 * straight-through (dx uses the rounded taps).
 *   grad_out  [B, 4C, H, W]
 *   x, y      [B, C, H, W];  weight [O, C];  bias [O] or NULL
 *   dx, dy    [B, C, H, W]   outputs
 *   dweight   [O, C]         output
 *   dbias     [O] or NULL    output (NULL: not computed)
 *   workspace device buffer of at least ddpm_backward_workspace_size() bytes,
 *             16-byte aligned; its contents on entry do not matter
 */
DDPM_API ddpm_status ddpm_backward(const ddpm_problem* problem, const void* grad_out, const void* x,
                          const void* y, const void* weight, const void* bias, void* dx, void* dy,
                          void* dweight, void* dbias, void* workspace, size_t workspace_bytes,
                          ddpm_stream_t stream);

/* Bytes of device scratch that ddpm_backward_noalloc keeps inside the library. */
#define DDPM_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * ddpm_backward_noalloc -- ddpm_backward without a caller-supplied workspace.
 * The paper has no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory when they call the backward -- for example a
 * plugin running inside an application that owns every device allocation, a
 * real-time loop that forbids allocation after start-up, or a C caller with no
 * allocator for temporary buffers.
 *   Arguments and results are those of ddpm_backward, minus the workspace.
 *   The FP32 dW/dbias partial sums live in a fixed device array of
 *   DDPM_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library; every GPU that loads
 *   the library holds it until the process exits.  The criterion is the
 *   partials alone: problems whose partials need more than the array
 *   (16 * 3*C*K*K * (C+1) * 4 bytes at most; e.g. C=64 with K=5 needs 20 MB)
 *   are rejected with DDPM_ERR_UNSUPPORTED before anything is enqueued; C=64,
 *   K=3 needs 7.2 MB at any image size.  ddpm_backward_workspace_size() may
 *   report more for the same problem, because it also counts the optional
 *   packed copies that only speed up dX.
 *   No device memory is allocated or freed.  The first call on each device looks
 *   up the array's device address (cudaGetSymbolAddress with that device
 *   current) and keeps it for the life of the process; make that first call
 *   before any stream capture, and do not call this entry point again after a
 *   cudaDeviceReset (the kept address would no longer be the array's).
 *   All calls share the one array and it keeps the last call's contents (no
 *   slot needs to start at zero: each call overwrites every slot it reads).
 *   Calls that overlap on the GPU -- on different streams or from different
 *   host threads on one device -- race on the array and give wrong results.
 */
DDPM_API ddpm_status ddpm_backward_noalloc(const ddpm_problem* problem, const void* grad_out, const void* x,
                                          const void* y, const void* weight, const void* bias, void* dx,
                                          void* dy, void* dweight, void* dbias, ddpm_stream_t stream);

/*
 * ddpm_get_device_error -- synchronise `stream`, then report (and clear) the
 * device-side error word that kernels set when a bounded wait expires.
 * Returns DDPM_OK, DDPM_ERR_DEVICE_TIMEOUT or DDPM_ERR_CUDA.
 */
DDPM_API ddpm_status ddpm_get_device_error(ddpm_stream_t stream);

/*
 * ddpm_debug_wait_probe -- run the library's bounded-wait failure path once, on
 * purpose (a diagnostic; the pages have no counterpart).  Every tensor-core
 * kernel here waits on shared-memory barriers with a time limit (2 s); when a
 * limit runs out, the block records DDPM_ERR_DEVICE_TIMEOUT in the device error
 * word, makes its other waiters leave, frees its tensor memory and returns
 * instead of trapping, so the CUDA context stays usable.  This enqueues on
 * `stream` a kernel with the same warp roles whose wait can never be satisfied,
 * limited to `limit_us` microseconds (1 .. 1,000,000).  Afterwards
 * ddpm_get_device_error(stream) reports (and clears) DDPM_ERR_DEVICE_TIMEOUT.
 * Returns DDPM_ERR_INVALID_ARGUMENT for a limit outside the range (nothing is
 * enqueued), DDPM_ERR_CUDA if the launch fails, else DDPM_OK.
 */
DDPM_API ddpm_status ddpm_debug_wait_probe(unsigned int limit_us, ddpm_stream_t stream);

/*
 * Kernel tracing (profiling aid; off by default).
 * While enabled, every kernel an entry point launches is bracketed by a pair of
 * CUDA events recorded on the caller's stream, so per-kernel device time can be
 * read back without a profiler; the backward's pieces, which otherwise overlap
 * on the library's own streams, then run one after another on that stream so
 * that each interval holds one kernel alone.  Enabling creates CUDA events lazily (no device
 * memory is allocated); at most 65536 records are kept, later ones are dropped.
 *   ddpm_trace_enable(1|0)      switch tracing on or off (returns DDPM_OK)
 *   ddpm_trace_read(ids, ms, n) wait for the recorded kernels, copy up to n
 *                               (kernel id, milliseconds) pairs in launch order,
 *                               clear the list; returns the number copied, or
 *                               -1 on a CUDA error
 *   ddpm_kernel_name(id)        name of a kernel id (never NULL)
 */
DDPM_API ddpm_status ddpm_trace_enable(int enable);
/*
 * ddpm_measure_ffma_tflops -- measured FP32 FMA throughput of the current device
 * (profiling aid for the CUDA-core kernels' roofline).  Launches a kernel of
 * eight independent FMA chains per thread on every SM on the legacy default
 * stream, synchronises, and writes the best of three timed launches, in
 * TFLOP/s (2 flops per FMA), to *tflops.  Returns DDPM_OK, or
 * DDPM_ERR_INVALID_ARGUMENT for a NULL pointer, or DDPM_ERR_CUDA.
 */
DDPM_API ddpm_status ddpm_measure_ffma_tflops(double* tflops);
DDPM_API int ddpm_trace_read(int* kernel_ids, float* milliseconds, int max_records);
DDPM_API const char* ddpm_kernel_name(int kernel_id);

/* Human-readable name of a status code (static storage, never NULL). */
DDPM_API const char* ddpm_status_string(ddpm_status status);

/* Library version, major*10000 + minor*100 + patch. */
DDPM_API int ddpm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DDPM_GB300_H */
