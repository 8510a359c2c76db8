// Residual + LayerNorm + affine, fused into one pass over HBM, plus the
// separate normalisation and scale-and-bias kernels of the unfused chain.
//
// "Costs and benefits of kernel fusion", "Worked example: Fusing a residual
// and normalization chain": load activation and residual once, compute the
// row statistics, normalise, apply scale and bias, write the final output.
// One CTA owns one row at a time ("whether one block can own a row efficiently
// across hidden sizes"): each thread keeps its slice of s = act + res in fp32
// registers, the CTA reduces the sum (mean), then the sum of squared
// deviations from those registers (variance, two-pass), then writes
// (s - mean) * rsqrt(var + eps) * gamma + beta.  s is never written to HBM.
#include <cuda_fp16.h>

#include "ptx_sm100.cuh"
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

// Persistent CTAs walk the rows blockIdx.x, blockIdx.x + gridDim.x, ...
// Thread 0 streams the input rows into a `stages`-deep shared-memory ring with
// 1-D bulk copies (cp.async.bulk, completion on an mbarrier), so several rows
// per CTA are in flight while the CTA reduces and writes the current one.
// Each thread converts its NV 16-byte vectors (8 values each) of the row to
// fp32 registers; the statistics come from those registers in two passes.
// NV: vectors per thread.  RESIDUAL: s = a + b, else s = a.  AFFINE: apply
// gamma and beta.
template <int NV, bool RESIDUAL, bool AFFINE>
__global__ void __launch_bounds__(1024) layernorm_kernel(const __half *__restrict__ a,
                                                         const __half *__restrict__ b,
                                                         const float *__restrict__ gamma,
                                                         const float *__restrict__ beta,
                                                         __half *__restrict__ y, int64_t rows, int hidden,
                                                         float eps, int stages, uint32_t *err, uint64_t wait_ns)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[32];
    const int nvec = hidden >> 3;
    const uint32_t row_bytes = (uint32_t)hidden * 2u;
    const uint32_t stage_bytes = RESIDUAL ? 2u * row_bytes : row_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);
    const int64_t G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int st = 0; st < stages; ++st) ptx::mbar_init(&full[st], 1);
        ptx::mbar_init_fence();
        for (int st = 0; st < stages; ++st) {
            const int64_t row = blockIdx.x + st * G;
            if (row >= rows) break;
            unsigned char *dst = smem + (size_t)st * stage_bytes;
            ptx::mbar_arrive_expect_tx(&full[st], stage_bytes);
            ptx::bulk_load(dst, a + row * hidden, row_bytes, &full[st]);
            if (RESIDUAL) ptx::bulk_load(dst + row_bytes, b + row * hidden, row_bytes, &full[st]);
        }
    }
    __syncthreads();

    // gamma and beta stay in registers for every row this CTA handles
    float g[NV][8], bb[NV][8];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            g[k][j] = 1.0f;
            bb[k][j] = 0.0f;
        }
        if (AFFINE && v < nvec) {
            const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * v));
            const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * v + 4));
            const float4 b0 = __ldg(reinterpret_cast<const float4 *>(beta + 8 * v));
            const float4 b1 = __ldg(reinterpret_cast<const float4 *>(beta + 8 * v + 4));
            g[k][0] = g0.x; g[k][1] = g0.y; g[k][2] = g0.z; g[k][3] = g0.w;
            g[k][4] = g1.x; g[k][5] = g1.y; g[k][6] = g1.z; g[k][7] = g1.w;
            bb[k][0] = b0.x; bb[k][1] = b0.y; bb[k][2] = b0.z; bb[k][3] = b0.w;
            bb[k][4] = b1.x; bb[k][5] = b1.y; bb[k][6] = b1.z; bb[k][7] = b1.w;
        }
    }

    const float inv_h = 1.0f / (float)hidden;
    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += G, ++it) {
        const int st = it % stages;
        const uint32_t parity = (uint32_t)(it / stages) & 1u;
        const bool ok = ptx::mbar_wait(&full[st], parity, wait_ns);
        if (!__syncthreads_and(ok)) {
            if (threadIdx.x == 0) atomicOr(err, TF_DEVERR_PRODUCER_WAIT);
            break;
        }
        const unsigned char *src = smem + (size_t)st * stage_bytes;
        float s[NV][8];
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            uint4 av = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
            if (v < nvec) {
                av = reinterpret_cast<const uint4 *>(src)[v];
                if (RESIDUAL) bv = reinterpret_cast<const uint4 *>(src + row_bytes)[v];
            }
            const __half2 *ah = reinterpret_cast<const __half2 *>(&av);
            const __half2 *bh = reinterpret_cast<const __half2 *>(&bv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 t = __half22float2(ah[j]);
                if (RESIDUAL) {
                    const float2 u = __half22float2(bh[j]);
                    t.x += u.x;
                    t.y += u.y;
                }
                s[k][2 * j] = t.x;
                s[k][2 * j + 1] = t.y;
                sum += t.x + t.y;
            }
        }
        const float mean = block_sum(sum, red) * inv_h;
        // every thread has read stage `st`: refill it with the row `stages` ahead
        if (threadIdx.x == 0) {
            const int64_t next = row + (int64_t)stages * G;
            if (next < rows) {
                unsigned char *dst = smem + (size_t)st * stage_bytes;
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive_expect_tx(&full[st], stage_bytes);
                ptx::bulk_load(dst, a + next * hidden, row_bytes, &full[st]);
                if (RESIDUAL) ptx::bulk_load(dst + row_bytes, b + next * hidden, row_bytes, &full[st]);
            }
        }
        float sq = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            if (v < nvec) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float d = s[k][j] - mean;
                    sq = fmaf(d, d, sq);
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
                uint4 out;
                __half2 *oh = reinterpret_cast<__half2 *>(&out);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float o0 = (s[k][2 * j] - mean) * rstd, o1 = (s[k][2 * j + 1] - mean) * rstd;
                    oh[j] = AFFINE ? __floats2half2_rn(fmaf(o0, g[k][2 * j], bb[k][2 * j]),
                                                       fmaf(o1, g[k][2 * j + 1], bb[k][2 * j + 1]))
                                   : __floats2half2_rn(o0, o1);
                }
                st_stream(yr + 8 * v, out);
            }
        }
    }
    // Copies issued for rows this CTA never consumed (only after a time-out)
    // must land before the CTA exits.
    if (threadIdx.x == 0) {
        for (int k = 0; k < stages; ++k) {
            const int64_t row = blockIdx.x + (int64_t)(it + k) * G;
            if (row >= rows) break;
            const int st = (it + k) % stages;
            if (!ptx::mbar_wait(&full[st], (uint32_t)((it + k) / stages) & 1u, wait_ns))
                atomicOr(err, TF_DEVERR_DRAIN_WAIT);
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
    if (hidden > 2048 * 8) return cudaErrorNotSupported;
    uint32_t *err = device_error_word();
    if (!err) return cudaErrorInitializationError;
    const int threads = threads_for(hidden, 2);
    const size_t stage_bytes = (size_t)hidden * 2 * (RESIDUAL ? 2 : 1);
    // Ring depth: up to 4 rows, within ~96 KB of shared memory per CTA.
    int stages = (int)((96 * 1024) / stage_bytes);
    stages = stages < 2 ? 2 : (stages > 4 ? 4 : stages);
    const size_t smem = (size_t)stages * stage_bytes + 8 * (size_t)stages;
    // CTAs per SM: limited by shared memory (~220 KB usable) and 2048 threads.
    int per_sm = (int)((220 * 1024) / (smem + 1024));
    if (per_sm > 2048 / threads) per_sm = 2048 / threads;
    if (per_sm > 8) per_sm = 8;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)sm_count() * per_sm;
    if (grid > rows) grid = rows;
    auto kern = layernorm_kernel<2, RESIDUAL, AFFINE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, threads, smem, st>>>(reinterpret_cast<const __half *>(a), reinterpret_cast<const __half *>(b),
                                                gamma, beta, reinterpret_cast<__half *>(y), rows, (int)hidden, eps,
                                                stages, err, wait_limit_ns());
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
