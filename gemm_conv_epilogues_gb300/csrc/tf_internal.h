// Internal declarations shared by the library's translation units: the host
// launchers each kernel file exports, and the small device helpers they use.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tf_epilogue.h"
#include "gelu_poly.h"

namespace tf {

// Device error word of the current device (a __device__ symbol in tf_api.cu)
// and the wait limit every bounded spin-wait uses.
uint32_t *device_error_word();
uint64_t wait_limit_ns();
int sm_count();

// Conv launchers.  `epilogue` is 1 for the fused BN+SiLU epilogue, 0 for a
// plain bf16 store of the accumulator (the unfused chain's first kernel).
struct ConvArgs {
    const void *x;
    const void *w;
    const float *scale;
    const float *bias;
    void *y;
    tf_conv_shape s;
    int Ho, Wo;
    int epilogue;
};
cudaError_t launch_conv_direct(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_tiled(const ConvArgs &a, cudaStream_t st);
// Returns cudaErrorNotSupported when the shape does not fit the kernel.
cudaError_t launch_conv_umma(const ConvArgs &a, cudaStream_t st);
bool conv_umma_supports(const tf_conv_shape &s, int Ho, int Wo);

cudaError_t launch_pack_filter(const void *w_oihw, void *w_ohwi, int C_out, int C_in, int KH, int KW,
                               cudaStream_t st);
cudaError_t launch_bias_gelu(const void *x, const void *bias, void *y, int64_t rows, int64_t cols,
                             cudaStream_t st);
cudaError_t launch_residual_layernorm(const void *act, const void *res, const float *gamma,
                                      const float *beta, void *y, int64_t rows, int64_t hidden,
                                      float eps, cudaStream_t st);
cudaError_t launch_unfused_bn(const void *t1, const float *scale, const float *bias, void *t2,
                              int64_t M, int64_t C, cudaStream_t st);
cudaError_t launch_unfused_silu(const void *t2, void *y, int64_t n, cudaStream_t st);
cudaError_t launch_unfused_bias_add(const void *x, const void *bias, void *t, int64_t rows,
                                    int64_t cols, cudaStream_t st);
cudaError_t launch_unfused_gelu(const void *t, void *y, int64_t n, cudaStream_t st);
cudaError_t launch_unfused_residual_add(const void *a, const void *r, void *s, int64_t n,
                                        cudaStream_t st);
cudaError_t launch_unfused_layernorm(const void *s, void *nrm, int64_t rows, int64_t hidden,
                                     float eps, cudaStream_t st);
cudaError_t launch_unfused_affine(const void *nrm, const float *gamma, const float *beta, void *y,
                                  int64_t rows, int64_t hidden, cudaStream_t st);
cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st);

}  // namespace tf

#ifdef __CUDACC__
namespace tf {
// SiLU(v) = v * sigmoid(v) = v / (1 + e^-v), fp32 ("Fusing an Epilogue",
// "The shape of it").  For v below about -88 e^-v overflows to +inf and the
// quotient is -0, the correctly rounded fp32 limit.
__device__ __forceinline__ float silu_f32(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU(s) = s * Phi(s), Phi the standard normal distribution function (the
// erf definition).  The upper tail Q(t) = 1 - Phi(t) is evaluated as
// 2^P(t/3 - 1) with P a degree-7 fit of log2 Q on [0, 6] (gelu_poly.h,
// generated and checked by gen_gelu_poly.py); Phi(s) = 1 - Q(s) for s >= 0
// and Q(-s) for s < 0, so the negative tail keeps its relative accuracy
// without the cancellation of 1 + erf.  Beyond |s| = 6 the tail is clamped:
// |s| * Q(6) is below half the smallest fp16 subnormal.  Cost: 9 FMA-pipe
// operations and one ex2 per value.
__device__ __forceinline__ float gelu_f32(float s)
{
    const float t = fminf(fabsf(s), TF_GELU_TMAX);
    const float v = fmaf(t, 1.0f / (TF_GELU_TMAX * 0.5f), -1.0f);
    float acc = TF_GELU_C7;
    acc = fmaf(acc, v, TF_GELU_C6);
    acc = fmaf(acc, v, TF_GELU_C5);
    acc = fmaf(acc, v, TF_GELU_C4);
    acc = fmaf(acc, v, TF_GELU_C3);
    acc = fmaf(acc, v, TF_GELU_C2);
    acc = fmaf(acc, v, TF_GELU_C1);
    acc = fmaf(acc, v, TF_GELU_C0);
    const float q = ex2_approx(acc);
    return s * (s >= 0.0f ? 1.0f - q : q);
}
}  // namespace tf
#endif
