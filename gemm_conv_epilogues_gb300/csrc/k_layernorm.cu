// Residual + LayerNorm + affine, fused into one pass over HBM, plus the
// separate normalisation and scale-and-bias kernels of the unfused chain.
//
// "Costs and benefits of kernel fusion", "Worked example: Fusing a residual
// and normalization chain": load activation and residual once, compute the
// row statistics, normalise, apply scale and bias, write the final output.
// One CTA owns one row ("whether one block can own a row efficiently across
// hidden sizes"): each thread keeps its slice of s = act + res in fp32
// registers, the CTA reduces the sum (mean), then the sum of squared
// deviations from those registers (variance, two-pass), then writes
// (s - mean) * rsqrt(var + eps) * gamma + beta.  s is never written to HBM.
#include <cuda_fp16.h>

#include "tf_internal.h"

namespace tf {
namespace {

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// Sum of `v` over the CTA, returned to every thread.  `red` holds 32 floats.
__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = (blockDim.x + 31) >> 5;
    __syncthreads();  // `red` may still be read by the previous reduction
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < nwarps ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// NV: 16-byte vectors (8 values) per thread.  RESIDUAL: s = a + b, else s = a.
// AFFINE: multiply by gamma and add beta.
template <int NV, bool RESIDUAL, bool AFFINE>
__global__ void __launch_bounds__(1024) layernorm_kernel(const __half *__restrict__ a,
                                                         const __half *__restrict__ b,
                                                         const float *__restrict__ gamma,
                                                         const float *__restrict__ beta,
                                                         __half *__restrict__ y, int hidden, float eps)
{
    __shared__ float red[32];
    const int64_t row = blockIdx.x;
    const int nvec = hidden >> 3;
    const __half *ar = a + row * hidden;
    const __half *br = RESIDUAL ? b + row * hidden : nullptr;

    float s[NV][8];
    uint4 av[NV] = {}, bv[NV] = {};
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        if (v < nvec) {
            av[k] = ld_stream(ar + 8 * v);
            if (RESIDUAL) bv[k] = ld_stream(br + 8 * v);
        }
    }
    float sum = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        const __half2 *ah = reinterpret_cast<const __half2 *>(&av[k]);
        const __half2 *bh = reinterpret_cast<const __half2 *>(&bv[k]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 t = v < nvec ? __half22float2(ah[j]) : make_float2(0.0f, 0.0f);
            if (RESIDUAL && v < nvec) {
                const float2 u = __half22float2(bh[j]);
                t.x += u.x;
                t.y += u.y;
            }
            s[k][2 * j] = t.x;
            s[k][2 * j + 1] = t.y;
            sum += t.x + t.y;
        }
    }
    const float inv_h = 1.0f / (float)hidden;
    const float mean = block_sum(sum, red) * inv_h;
    float sq = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        if (v < nvec) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float d = s[k][j] - mean;
                sq += d * d;
            }
        }
    }
    const float var = block_sum(sq, red) * inv_h;
    const float rstd = rsqrtf(var + eps);
    __half *yr = y + row * hidden;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
        if (v < nvec) {
            float o[8];
            if (AFFINE) {
                const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * v));
                const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * v + 4));
                const float4 b0 = __ldg(reinterpret_cast<const float4 *>(beta + 8 * v));
                const float4 b1 = __ldg(reinterpret_cast<const float4 *>(beta + 8 * v + 4));
                const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
                const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = (s[k][j] - mean) * rstd * g[j] + bb[j];
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) o[j] = (s[k][j] - mean) * rstd;
            }
            uint4 out;
            __half2 *oh = reinterpret_cast<__half2 *>(&out);
#pragma unroll
            for (int j = 0; j < 4; ++j) oh[j] = __floats2half2_rn(o[2 * j], o[2 * j + 1]);
            st_stream(yr + 8 * v, out);
        }
    }
}

// y[i][j] = nrm[i][j] * gamma[j] + beta[j] (the unfused chain's last kernel).
__global__ void __launch_bounds__(256) affine_kernel(const uint4 *__restrict__ nrm,
                                                     const float *__restrict__ gamma,
                                                     const float *__restrict__ beta,
                                                     uint4 *__restrict__ y, int64_t nvec, int64_t cvec)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
        const uint4 v = ld_stream(nrm + i);
        const int64_t c0 = (i % cvec) * 8;
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
        uint4 out;
        __half2 *oh = reinterpret_cast<__half2 *>(&out);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 t = __half22float2(h[j]);
            oh[j] = __floats2half2_rn(t.x * __ldg(gamma + c0 + 2 * j) + __ldg(beta + c0 + 2 * j),
                                      t.y * __ldg(gamma + c0 + 2 * j + 1) + __ldg(beta + c0 + 2 * j + 1));
        }
        st_stream(y + i, out);
    }
}

// Threads per row for NV vectors per thread: a whole number of warps.
int threads_for(int64_t hidden, int nv)
{
    const int64_t nvec = hidden / 8;
    int64_t t = (nvec + nv - 1) / nv;
    t = (t + 31) / 32 * 32;
    return (int)(t < 32 ? 32 : t);
}

template <bool RESIDUAL, bool AFFINE>
cudaError_t launch_ln(const void *a, const void *b, const float *gamma, const float *beta, void *y,
                      int64_t rows, int64_t hidden, float eps, cudaStream_t st)
{
    const __half *ah = reinterpret_cast<const __half *>(a);
    const __half *bh = reinterpret_cast<const __half *>(b);
    __half *yh = reinterpret_cast<__half *>(y);
    if (hidden <= 2048 * 8) {
        layernorm_kernel<2, RESIDUAL, AFFINE>
            <<<(unsigned)rows, threads_for(hidden, 2), 0, st>>>(ah, bh, gamma, beta, yh, (int)hidden, eps);
    } else {
        return cudaErrorNotSupported;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_residual_layernorm(const void *act, const void *res, const float *gamma,
                                      const float *beta, void *y, int64_t rows, int64_t hidden,
                                      float eps, cudaStream_t st)
{
    return launch_ln<true, true>(act, res, gamma, beta, y, rows, hidden, eps, st);
}

cudaError_t launch_unfused_layernorm(const void *s, void *nrm, int64_t rows, int64_t hidden, float eps,
                                     cudaStream_t st)
{
    return launch_ln<false, false>(s, nullptr, nullptr, nullptr, nrm, rows, hidden, eps, st);
}

cudaError_t launch_unfused_affine(const void *nrm, const float *gamma, const float *beta, void *y,
                                  int64_t rows, int64_t hidden, cudaStream_t st)
{
    const int64_t nvec = rows * hidden / 8;
    int64_t g = (nvec + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (g > cap) g = cap;
    affine_kernel<<<(unsigned)g, 256, 0, st>>>(reinterpret_cast<const uint4 *>(nrm), gamma, beta,
                                               reinterpret_cast<uint4 *>(y), nvec, hidden / 8);
    return cudaGetLastError();
}

}  // namespace tf
