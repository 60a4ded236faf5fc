/*
 * ddpm_oracle.h -- C interface of the CPU FP64 oracle (test infrastructure).
 *
 * Only tests, the smoke check and the benchmark's CPU-baseline leg use this.
 * It is unrelated to the CUDA library's public header and shares nothing
 * with it.  All arrays are FP64, NCHW, contiguous; every function returns 0
 * on success, 1 for an invalid shape and 2 when host memory runs out.
 */
#ifndef DDPM_ORACLE_H
#define DDPM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int B, C, H, W, K;  /* batch, channels, height, width, kernel size (odd) */
    int dil[3];         /* the three dilations, (1,3,5) in the method */
    int bf16;           /* nonzero: round each tap to bfloat16 before use */
} ddpmo_shape;

double ddpmo_round_bf16(double v);
double ddpmo_tap(const ddpmo_shape* s, const double* y, const double* Wg, const double* bias,
                 int b, int o, int h, int w);
int ddpmo_generate_taps(const ddpmo_shape* s, const double* y, const double* Wg,
                        const double* bias, double* T);
int ddpmo_forward(const ddpmo_shape* s, const double* x, const double* y, const double* Wg,
                  const double* bias, double* out);
int ddpmo_filter(const ddpmo_shape* s, const double* x, const double* T, double* out);
int ddpmo_forward_points(const ddpmo_shape* s, const double* x, const double* y, const double* Wg,
                         const double* bias, int64_t n, const int64_t* idx, double* vals);
int ddpmo_filter_points(const ddpmo_shape* s, const double* x, const double* T, int64_t n,
                        const int64_t* idx, double* vals);
int ddpmo_backward(const ddpmo_shape* s, const double* g, const double* x, const double* y,
                   const double* Wg, const double* bias, double* dx, double* dy, double* dW,
                   double* dbias);
int ddpmo_backward_points(const ddpmo_shape* s, const double* g, const double* x, const double* y,
                          const double* Wg, const double* bias, int which, int64_t n,
                          const int64_t* idx, double* vals);
int ddpmo_filter_backward(const ddpmo_shape* s, const double* g, const double* x, const double* T, double* dx,
                          double* dT);
int ddpmo_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
