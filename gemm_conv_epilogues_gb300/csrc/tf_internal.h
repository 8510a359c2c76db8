// Internal declarations shared by the library's translation units: the host
// launchers each kernel file exports, and the small device helpers they use.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
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
    int splits = 1;          // tensor-core kernel only: K splits, fp32 partials to ws
    float *ws = nullptr;
    int cluster = 1;         // tensor-core kernel only: 2 = CTA pairs running paired (cta_group::2) MMAs
    bool wide = false;       // tensor-core kernel only: 256-row tiles per CTA (two MMAs per K step)
};
cudaError_t launch_conv_direct(const ConvArgs &a, cudaStream_t st);
cudaError_t launch_conv_tiled(const ConvArgs &a, cudaStream_t st);
// Returns cudaErrorNotSupported when the shape does not fit the kernel.
cudaError_t launch_conv_umma(const ConvArgs &a, cudaStream_t st);
bool conv_umma_supports(const tf_conv_shape &s, int Ho, int Wo);
// K splits worth using for this shape (1: none), and the reduction that sums
// the splits' fp32 partials and applies the epilogue.
int conv_umma_splits(const tf_conv_shape &s, int Ho, int Wo);
cudaError_t launch_splitk_reduce(const float *ws, int splits, int64_t M, int C_out, const float *scale,
                                 const float *bias, void *y, int epilogue, cudaStream_t st);

cudaError_t launch_pack_filter(const void *w_oihw, void *w_ohwi, int C_out, int C_in, int KH, int KW,
                               cudaStream_t st);
cudaError_t launch_bias_gelu(const void *x, const void *bias, void *y, int64_t rows, int64_t cols,
                             cudaStream_t st);
// Row-reduction strategy boundaries of the LayerNorm kernels (hidden widths).
constexpr int64_t kWarpMaxHidden = 1024;      // warp per row: up to 4 vectors per lane
constexpr int64_t kCtaMaxHidden = 16384;      // CTA per row: up to 1024 threads x 16 values
constexpr int64_t kClusterMaxHidden = 131072; // cluster of <= 8 CTAs per row
// Measured on GB300 (gemm_conv_epilogues_gb300/ln_sweep.py): one warp per row
// is faster up to this width, one CTA per row above it.
constexpr int64_t kWarpBoundary = 1024;
int layernorm_select(int64_t hidden);
cudaError_t launch_residual_layernorm(const void *act, const void *res, const float *gamma,
                                      const float *beta, void *y, int64_t rows, int64_t hidden,
                                      float eps, int variant, cudaStream_t st);
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
cudaError_t launch_bias_gelu_rowsum(const void *x, const void *bias, void *y, float *rowsum, int64_t rows,
                                    int64_t cols, cudaStream_t st);
cudaError_t launch_unfused_rowsum(const void *y, float *rowsum, int64_t rows, int64_t cols, cudaStream_t st);
cudaError_t launch_wait_probe(uint64_t limit_ns, cudaStream_t st);

}  // namespace tf

#ifdef __CUDACC__
namespace tf {

// Programmatic dependent launch.  Every kernel of the library starts with
// pdl_begin(): it waits until the stream's previous kernel has completed and
// its memory is visible (at once when launched without the attribute), then
// lets the stream's next kernel be scheduled, so that kernel's launch and
// set-up overlap this one's tail.  Nothing before pdl_begin() may touch
// global memory.
__device__ __forceinline__ void pdl_begin()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// CTA-wide barriers for code in which the lanes of a warp may have taken
// different paths (a role run by lane 0 alone, a divergent loop exit).  The
// barrier instruction is warp-aligned: it counts a whole warp as arrived as
// soon as any of its lanes arrives, so lanes that get there early would let
// it complete before the rest of the CTA (and count the warp again later).
// Each warp is reconverged first.  Every lane of the CTA must still be live.
__device__ __forceinline__ void cta_sync()
{
    __syncwarp();
    __syncthreads();
}

__device__ __forceinline__ int cta_sync_and(int pred)
{
    __syncwarp();
    return __syncthreads_and(pred);
}

// Kernels launched by this library in this process (tf_launch_count);
// every launch site passes its cudaLaunchKernelEx result through counted().
extern std::atomic<unsigned long long> g_launch_count;
inline cudaError_t counted(cudaError_t e)
{
    if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
    return e;
}

// kern<<<grid, block, smem, st>>>(args...) with programmatic dependent launch allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return counted(cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...));
}

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
// without the cancellation of 1 + erf.  With w = s*Q(|s|) that is s - w for
// s >= 0 and w for s < 0, which is max(s - w, w) since Q <= 1/2.  |s| is
// clamped at 12: past the fit range the polynomial keeps falling (below
// 2^-29 from |s| = 6, 2^-111 at 12), so |s*Q| rounds to zero in fp16 for every
// |s| > 6, as the exact value does.  Cost: 9 FMA-pipe operations and one ex2
// per value.
__device__ __forceinline__ float gelu_f32(float s)
{
    const float t = fminf(fabsf(s), TF_GELU_TCLAMP);
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
    const float w = s * q;
    return fmaxf(s - w, w);
}
// ---- packed fp32 pairs (sm_100 family f32x2 instructions): two lanes of
// work per FMA-pipe issue slot.
__device__ __forceinline__ unsigned long long pk2(float2 a)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a.x), "f"(a.y));
    return r;
}

__device__ __forceinline__ float2 upk2(unsigned long long r)
{
    float2 a;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a.x), "=f"(a.y) : "l"(r));
    return a;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)), "l"(pk2(c)));
    return upk2(d);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b)
{
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(d);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(d);
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b)
{
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pk2(a)), "l"(pk2(b)));
    return upk2(d);
}

// gelu_f32 on a pair, same arithmetic: with w = s*Q(|s|), GELU(s) is s - w
// for s >= 0 and w for s < 0, and in both cases the larger of the two
// (Q <= 1/2), so the sign test becomes a max.
__device__ __forceinline__ float2 gelu_f32x2(float2 s)
{
    const float2 t = make_float2(fminf(fabsf(s.x), TF_GELU_TCLAMP), fminf(fabsf(s.y), TF_GELU_TCLAMP));
    const float k = 1.0f / (TF_GELU_TMAX * 0.5f);
    const float2 v = ffma2(t, make_float2(k, k), make_float2(-1.0f, -1.0f));
    float2 acc = ffma2(make_float2(TF_GELU_C7, TF_GELU_C7), v, make_float2(TF_GELU_C6, TF_GELU_C6));
    acc = ffma2(acc, v, make_float2(TF_GELU_C5, TF_GELU_C5));
    acc = ffma2(acc, v, make_float2(TF_GELU_C4, TF_GELU_C4));
    acc = ffma2(acc, v, make_float2(TF_GELU_C3, TF_GELU_C3));
    acc = ffma2(acc, v, make_float2(TF_GELU_C2, TF_GELU_C2));
    acc = ffma2(acc, v, make_float2(TF_GELU_C1, TF_GELU_C1));
    acc = ffma2(acc, v, make_float2(TF_GELU_C0, TF_GELU_C0));
    const float2 q = make_float2(ex2_approx(acc.x), ex2_approx(acc.y));
    const float2 w = fmul2(s, q);
    const float2 d = fsub2(s, w);
    return make_float2(fmaxf(d.x, w.x), fmaxf(d.y, w.y));
}
// SiLU(v) = v * sigmoid(v) = v / (1 + 2^(-v*log2 e)) ("Fusing an Epilogue",
// "The shape of it"): one ex2.approx and one rcp.approx per value on the
// special-function unit (GB300's has room for both beside the epilogue's FMA
// work).  Relative error of a few fp32 ulp; for v < -88 the exponential is
// +inf and 1/inf gives the exact limit 0 (a signed zero), with no clamp.
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float silu_f32(float v)
{
    return v * rcp_approx(1.0f + ex2_approx(-kLog2e * v));
}

__device__ __forceinline__ float2 silu_f32x2(float2 v)
{
    const float2 x = fmul2(v, make_float2(-kLog2e, -kLog2e));
    const float2 d = make_float2(1.0f + ex2_approx(x.x), 1.0f + ex2_approx(x.y));
    return fmul2(v, make_float2(rcp_approx(d.x), rcp_approx(d.y)));
}
}  // namespace tf
#endif
