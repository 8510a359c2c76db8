// Bias + GELU + per-row sum, fused and split.
//
// "Costs and benefits of kernel fusion", "Compare fused and split
// bias-activation-reduction paths": on fp16 [8192, 8192], a fused path applies
// bias, GELU and a per-row reduction in one pass; the split path writes the
// GELU result first and then runs the reduction over it.
//
// Both kernels work on tiles of a few rows.  A persistent CTA of 256 threads
// walks the tiles blockIdx.x, +gridDim.x, ...; thread t owns the 16-byte
// column vectors t, t+256, ... of every row and keeps one fp32 partial sum
// per row of the tile; all of its loads of a tile are in flight together.
// At the end of a tile the CTA reduces the tile's partial sums at once (warp
// shuffles, one shared-memory step): one pair of barriers per tile.  The fused kernel sums the fp32
// GELU values before rounding y to fp16; the split path's reduction sums the
// stored fp16 values.
#include <cuda_fp16.h>

#include "tf_internal.h"

namespace tf {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxChunks = 8; // column vectors per thread: cols <= 8 * 256 * 8 = 16384

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

// FUSED: x, bias -> y = GELU(x + bias) (fp16) and rowsum (fp32).
// !FUSED: x is the stored GELU result; only rowsum is written.
// A tile is R rows; a thread owns the column vectors t + 256k, k < C, of each
// of them (C = ceil(cvec / 256)), so R * C = 8 independent 16-byte loads are in
// flight per thread, and small R keeps the tiles fine-grained enough to spread
// evenly over the persistent CTAs.
// (The fused kernels on tiles of 4 or 8 rows keep that many row sums and
// their GELU temporaries beside the 32 loaded values; they get the registers
// of three CTAs per SM.)
template <bool FUSED, int R, int C>
__global__ void __launch_bounds__(kThreads, FUSED && R >= 4 ? 3 : 4) rowsum_kernel(const uint4 *__restrict__ x,
                                                             const uint4 *__restrict__ bias,
                                                             uint4 *__restrict__ y, float *__restrict__ rowsum,
                                                             int64_t rows, int cvec)
{
    pdl_begin();
    __shared__ float red[kThreads / 32][R];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ntiles = (rows + R - 1) / R;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t r0 = tile * R;
        uint4 xv[R][C];
#pragma unroll
        for (int k = 0; k < C; ++k) {
            const int v = threadIdx.x + k * kThreads;
#pragma unroll
            for (int r = 0; r < R; ++r)
                xv[r][k] = (v < cvec && r0 + r < rows) ? ld_stream(x + (r0 + r) * cvec + v) : make_uint4(0, 0, 0, 0);
        }
        float sum[R];
#pragma unroll
        for (int r = 0; r < R; ++r) sum[r] = 0.0f;
#pragma unroll
        for (int k = 0; k < C; ++k) {
            const int v = threadIdx.x + k * kThreads;
            if (v >= cvec) continue;
            uint4 braw = make_uint4(0, 0, 0, 0);
            if (FUSED) braw = __ldg(bias + v);   // 16 KB of bias: L1 hits after the first tile
            const __half2 *bh = reinterpret_cast<const __half2 *>(&braw);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const __half2 *h = reinterpret_cast<const __half2 *>(&xv[r][k]);
                if (FUSED) {
                    uint4 o;
                    __half2 *oh = reinterpret_cast<__half2 *>(&o);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 g = gelu_f32x2(fadd2(__half22float2(h[j]), __half22float2(bh[j])));
                        sum[r] += g.x + g.y;
                        oh[j] = __floats2half2_rn(g.x, g.y);
                    }
                    if (r0 + r < rows) st_stream(y + (r0 + r) * cvec + v, o);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 t = __half22float2(h[j]);
                        sum[r] += t.x + t.y;
                    }
                }
            }
        }
        // the tile's R sums: shuffle within each warp, then across warps
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum[r] += __shfl_xor_sync(0xffffffffu, sum[r], o);
        }
        cta_sync();   // `red` of the previous tile has been read
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) red[warp][r] = sum[r];
        }
        cta_sync();
        if (threadIdx.x < R && r0 + threadIdx.x < rows) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) t += red[w][threadIdx.x];
            rowsum[r0 + threadIdx.x] = t;
        }
    }
}

template <bool FUSED>
cudaError_t launch_rowsum(const void *x, const void *bias, void *y, float *rowsum, int64_t rows, int64_t cols,
                          cudaStream_t st)
{
    const int64_t cvec = cols / 8;
    if (cvec > (int64_t)kThreads * kMaxChunks) return cudaErrorNotSupported;
    auto go = [&](auto kern, int R) -> cudaError_t {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        const int64_t ntiles = (rows + R - 1) / R;
        int64_t grid = (int64_t)sm_count() * per_sm;
        if (grid > ntiles) grid = ntiles;
        return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), 0, st, reinterpret_cast<const uint4 *>(x),
                          reinterpret_cast<const uint4 *>(bias), reinterpret_cast<uint4 *>(y), rowsum, rows,
                          (int)cvec);
    };
    const int64_t chunks = (cvec + kThreads - 1) / kThreads;
    if (chunks <= 1) return go(rowsum_kernel<FUSED, 8, 1>, 8);
    if (chunks <= 2) return go(rowsum_kernel<FUSED, 4, 2>, 4);
    if (chunks <= 4) return go(rowsum_kernel<FUSED, 2, 4>, 2);
    return go(rowsum_kernel<FUSED, 1, 8>, 1);
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
