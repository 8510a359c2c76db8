// Bias + GELU + per-row sum, fused and split.
//
// "Costs and benefits of kernel fusion", "Compare fused and split
// bias-activation-reduction paths": on fp16 [8192, 8192], a fused path applies
// bias, GELU and a per-row reduction in one pass; the split path writes the
// GELU result first and then runs the reduction over it.
//
// Both kernels are persistent: each CTA walks the rows blockIdx.x,
// +gridDim.x, ... and thread 0 streams input rows into a shared-memory ring
// with 1-D bulk copies, as the LayerNorm kernel does.  Each thread owns NV
// 16-byte column vectors of every row (so its bias stays in registers), and
// the row sum is reduced in fp32 with warp shuffles and one shared-memory
// step.  The fused kernel sums the fp32 GELU values before rounding y to
// fp16; the split path's reduction sums the stored fp16 values.
#include <cuda_fp16.h>

#include "ptx_sm100.cuh"
#include "tf_internal.h"

namespace tf {
namespace {

__device__ __forceinline__ void st_stream(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float block_sum(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = (blockDim.x + 31) >> 5;
    __syncthreads();  // `red` may still be read from the previous row
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = lane < nwarps ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// FUSED: x, bias -> y = GELU(x + bias) (fp16) and rowsum (fp32).
// !FUSED: x is the stored GELU result; only rowsum is written.
template <int NV, bool FUSED>
__global__ void __launch_bounds__(1024) rowsum_kernel(const __half *__restrict__ x, const __half *__restrict__ bias,
                                                      __half *__restrict__ y, float *__restrict__ rowsum,
                                                      int64_t rows, int cols, int stages, uint32_t *err,
                                                      uint64_t wait_ns)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[32];
    const int nvec = cols >> 3;
    const uint32_t row_bytes = (uint32_t)cols * 2u;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * row_bytes);
    const int64_t G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int st = 0; st < stages; ++st) ptx::mbar_init(&full[st], 1);
        ptx::mbar_init_fence();
        for (int st = 0; st < stages; ++st) {
            const int64_t row = blockIdx.x + st * G;
            if (row >= rows) break;
            ptx::mbar_arrive_expect_tx(&full[st], row_bytes);
            ptx::bulk_load(smem + (size_t)st * row_bytes, x + row * cols, row_bytes, &full[st]);
        }
    }
    __syncthreads();

    float bv[NV][8];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int v = threadIdx.x + k * blockDim.x;
#pragma unroll
        for (int j = 0; j < 8; ++j) bv[k][j] = 0.0f;
        if (FUSED && v < nvec) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(bias) + v);
            const __half2 *h = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 t = __half22float2(h[j]);
                bv[k][2 * j] = t.x;
                bv[k][2 * j + 1] = t.y;
            }
        }
    }

    int it = 0;
    for (int64_t row = blockIdx.x; row < rows; row += G, ++it) {
        const int st = it % stages;
        const bool ok = ptx::mbar_wait(&full[st], (uint32_t)(it / stages) & 1u, wait_ns);
        if (!__syncthreads_and(ok)) {
            if (threadIdx.x == 0) atomicOr(err, TF_DEVERR_PRODUCER_WAIT);
            break;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(smem + (size_t)st * row_bytes);
        uint4 raw[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            raw[k] = v < nvec ? src[v] : make_uint4(0, 0, 0, 0);
        }
        // every thread holds its part of the row: the stage can be refilled
        // after the barrier inside block_sum; results are written first
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            if (v >= nvec) continue;
            const __half2 *h = reinterpret_cast<const __half2 *>(&raw[k]);
            if (FUSED) {
                uint4 o;
                __half2 *oh = reinterpret_cast<__half2 *>(&o);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 g =
                        gelu_f32x2(fadd2(__half22float2(h[j]), make_float2(bv[k][2 * j], bv[k][2 * j + 1])));
                    sum += g.x + g.y;
                    oh[j] = __floats2half2_rn(g.x, g.y);
                }
                st_stream(y + row * cols + 8 * v, o);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 t = __half22float2(h[j]);
                    sum += t.x + t.y;
                }
            }
        }
        const float total = block_sum(sum, red);
        if (threadIdx.x == 0) {
            rowsum[row] = total;
            const int64_t next = row + (int64_t)stages * G;
            if (next < rows) {
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive_expect_tx(&full[st], row_bytes);
                ptx::bulk_load(smem + (size_t)st * row_bytes, x + next * cols, row_bytes, &full[st]);
            }
        }
    }
    if (threadIdx.x == 0) {   // copies for rows never consumed (only after a time-out) land before exit
        for (int k = 0; k < stages; ++k) {
            const int64_t row = blockIdx.x + (int64_t)(it + k) * G;
            if (row >= rows) break;
            const int st = (it + k) % stages;
            if (!ptx::mbar_wait(&full[st], (uint32_t)((it + k) / stages) & 1u, wait_ns))
                atomicOr(err, TF_DEVERR_DRAIN_WAIT);
        }
    }
}

template <bool FUSED>
cudaError_t launch_rowsum(const void *x, const void *bias, void *y, float *rowsum, int64_t rows, int64_t cols,
                          cudaStream_t st)
{
    if (cols > 2048 * 8) return cudaErrorNotSupported;
    uint32_t *err = device_error_word();
    if (!err) return cudaErrorInitializationError;
    int threads = (int)((cols / 8 + 1) / 2);
    threads = (threads + 31) / 32 * 32;
    const size_t row_bytes = (size_t)cols * 2;
    int stages = (int)((64 * 1024) / row_bytes);
    stages = stages < 2 ? 2 : (stages > 4 ? 4 : stages);
    const size_t smem = (size_t)stages * row_bytes + 8 * (size_t)stages;
    auto kern = rowsum_kernel<2, FUSED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t grid = (int64_t)sm_count() * per_sm;
    if (grid > rows) grid = rows;
    kern<<<(unsigned)grid, threads, smem, st>>>(reinterpret_cast<const __half *>(x),
                                                reinterpret_cast<const __half *>(bias), reinterpret_cast<__half *>(y),
                                                rowsum, rows, (int)cols, stages, err, wait_limit_ns());
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bias_gelu_rowsum(const void *x, const void *bias, void *y, float *rowsum, int64_t rows,
                                    int64_t cols, cudaStream_t st)
{
    return launch_rowsum<true>(x, bias, y, rowsum, rows, cols, st);
}

cudaError_t launch_unfused_rowsum(const void *y, float *rowsum, int64_t rows, int64_t cols, cudaStream_t st)
{
    return launch_rowsum<false>(y, nullptr, nullptr, rowsum, rows, cols, st);
}

}  // namespace tf
