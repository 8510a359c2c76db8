// Residual + LayerNorm + affine, fused into one pass over HBM, plus the
// separate normalisation kernel of the unfused chain (its residual-add and
// scale-and-bias kernels are the elementwise chain kernels).
//
// "Costs and benefits of kernel fusion", "Worked example: Fusing a residual
// and normalization chain": load activation and residual once, compute the
// row statistics, normalise, apply scale and bias, write the final output.
// One CTA owns one row at a time (the page asks how far that stays efficient
// as the hidden size grows): each thread keeps its slice of s = act + res in fp32
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
    cta_sync();  // `red` may still be read by the previous reduction
    if (lane == 0) red[warp] = v;
    cta_sync();
    float t = lane < nwarps ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// The same sum with ONE barrier: shuffles within each warp, one shared-memory
// step.  `red` must be a buffer no thread can still be reading:
// callers alternate two, with a CTA barrier between uses of the same one.
__device__ __forceinline__ float cta_sum_alt(float v, float *red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = (blockDim.x + 31) >> 5;
    if (lane == 0) red[warp] = v;
    cta_sync();
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
    pdl_begin();
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
    cta_sync();

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
        if (!cta_sync_and(ok)) {
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

// ---------------------------------------------------------------- one warp per row

// Narrow rows (hidden <= 1024): a warp owns a row, so both reductions are
// warp shuffles with no block barrier.  Lane l holds the 16-byte vectors
// l, l+32, ... (NV of them) of act and res; a CTA of 8 warps works on 8
// rows at once and the grid strides over the rest.
template <int NV, bool RESIDUAL, bool AFFINE>
__global__ void __launch_bounds__(256) layernorm_warp_kernel(const __half *__restrict__ a,
                                                             const __half *__restrict__ b,
                                                             const float *__restrict__ gamma,
                                                             const float *__restrict__ beta,
                                                             __half *__restrict__ y, int64_t rows, int hidden,
                                                             float eps)
{
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nvec = hidden >> 3;
    const float inv_h = 1.0f / (float)hidden;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows; row += nwarps) {
        uint4 av[NV], bv[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = lane + 32 * k;
            av[k] = make_uint4(0, 0, 0, 0);
            bv[k] = make_uint4(0, 0, 0, 0);
            if (v < nvec) {
                av[k] = ld_stream(a + row * hidden + 8 * v);
                if (RESIDUAL) bv[k] = ld_stream(b + row * hidden + 8 * v);
            }
        }
        float s[NV][8];
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const __half2 *ah = reinterpret_cast<const __half2 *>(&av[k]);
            const __half2 *bh = reinterpret_cast<const __half2 *>(&bv[k]);
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
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float mean = sum * inv_h;
        float sq = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (lane + 32 * k < nvec) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float d = s[k][j] - mean;
                    sq = fmaf(d, d, sq);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        const float rstd = rsqrtf(sq * inv_h + eps);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = lane + 32 * k;
            if (v >= nvec) continue;
            float g[8], bb[8];
            if (AFFINE) {
                const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * v));
                const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gamma + 8 * v + 4));
                const float4 b0 = __ldg(reinterpret_cast<const float4 *>(beta + 8 * v));
                const float4 b1 = __ldg(reinterpret_cast<const float4 *>(beta + 8 * v + 4));
                g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w; g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
                bb[0] = b0.x; bb[1] = b0.y; bb[2] = b0.z; bb[3] = b0.w; bb[4] = b1.x; bb[5] = b1.y; bb[6] = b1.z; bb[7] = b1.w;
            }
            uint4 out;
            __half2 *oh = reinterpret_cast<__half2 *>(&out);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float o0 = (s[k][2 * j] - mean) * rstd, o1 = (s[k][2 * j + 1] - mean) * rstd;
                oh[j] = AFFINE ? __floats2half2_rn(fmaf(o0, g[2 * j], bb[2 * j]), fmaf(o1, g[2 * j + 1], bb[2 * j + 1]))
                               : __floats2half2_rn(o0, o1);
            }
            st_stream(y + row * hidden + 8 * v, out);
        }
    }
}

// ---------------------------------------------------------------- a cluster per row

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}


// Wide rows (hidden > 16384): a thread-block cluster owns a row; CTA r of the
// cluster owns the slice [r*slice, (r+1)*slice).  Clusters are persistent and
// walk the rows c, c + nclusters, ...; like the CTA-per-row kernel, thread 0
// of every CTA streams its slice of the coming rows (act and res) into a
// shared-memory ring with bulk copies, and each thread holds NV vectors of
// the current row in fp32 registers, so a row is still read from HBM exactly
// once (the page's test of a width too large for one CTA per row).  Each CTA
// reduces its slice to
// (sum, M2), M2 the sum of squared deviations from the slice's own mean (two
// CTA sums), and exchanges that pair once: thread r pushes it into slot
// [rank] of CTA r with st.async, which completes on CTA r's own mbarrier.
// Every CTA then merges the nranks pairs in rank order with Chan et al.'s
// pairwise update (the same statistics in every CTA, and no cancellation of
// a one-pass sum of squares).  No cluster-wide barrier is taken per row.
// Slots and mbarriers are double-buffered by row parity: a peer can only be
// one row ahead, since it cannot finish row i+1 without this CTA's pair for
// row i+1, which is sent after this CTA has read every slot of row i.
//
// NV = 4, REGP: 32 columns per thread with their gamma and beta in registers
// for the whole kernel (slices of up to 8192 columns, 256 threads, two CTAs
// per SM): the per-row cost of the reductions and the exchange is spread
// over twice the columns of NV = 2.  NV = 2 with 1024 threads (only when
// 16-CTA clusters cannot be had) re-reads gamma and beta for every row.
template <bool RESIDUAL, bool AFFINE, int NV, int MAXT, bool REGP>
__global__ void __launch_bounds__(MAXT, 512 / MAXT > 0 ? 512 / MAXT : 1) layernorm_cluster_kernel(const __half *__restrict__ a,
                                                                 const __half *__restrict__ b,
                                                                 const float *__restrict__ gamma,
                                                                 const float *__restrict__ beta,
                                                                 __half *__restrict__ y, int64_t rows, int hidden,
                                                                 int slice, float eps, int stages, uint32_t *err,
                                                                 uint64_t wait_ns)
{
    pdl_begin();
    constexpr int kMaxRanks = 16;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float red[2][32];   // the row's two reductions alternate buffers
    __shared__ int copy_fail;      // set by any thread whose wait for a stage ran out
    __shared__ __align__(8) float2 slot[2][kMaxRanks];   // [row parity][sending rank]: (sum, M2) of its slice
    __shared__ __align__(8) uint64_t xbar[2];
    const uint32_t rank = ptx::cluster_ctarank(), nranks = cluster_nctarank();
    const int64_t cid = blockIdx.x / nranks, ncl = gridDim.x / nranks;
    const int c0 = (int)rank * slice;                    // first column of this CTA's slice
    const int width = min(hidden - c0, slice);           // columns in the slice (a multiple of 8, >= 8)
    const int nvec = width >> 3;
    const uint32_t part_bytes = (uint32_t)width * 2u;
    const uint32_t stage_bytes = (uint32_t)slice * 2u * (RESIDUAL ? 2u : 1u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * stage_bytes);

    auto issue = [&](int st, int64_t row) {
        unsigned char *dst = smem + (size_t)st * stage_bytes;
        ptx::mbar_arrive_expect_tx(&full[st], RESIDUAL ? 2u * part_bytes : part_bytes);
        ptx::bulk_load(dst, a + row * hidden + c0, part_bytes, &full[st]);
        if (RESIDUAL) ptx::bulk_load(dst + (size_t)slice * 2, b + row * hidden + c0, part_bytes, &full[st]);
    };
    if (threadIdx.x == 0) {
        copy_fail = 0;
        for (int st = 0; st < stages; ++st) ptx::mbar_init(&full[st], 1);
        for (int p = 0; p < 2; ++p) ptx::mbar_init(&xbar[p], 1);
        ptx::mbar_init_fence();
        for (int st = 0; st < stages; ++st) {
            const int64_t row = cid + st * ncl;
            if (row >= rows) break;
            issue(st, row);
        }
    }
    ptx::cluster_sync();   // every CTA's exchange barriers exist before the first push

    float g[NV][8], bb[NV][8];
    auto load_params = [&](int k) {
        const int v = threadIdx.x + k * blockDim.x;
        const float4 g0 = __ldg(reinterpret_cast<const float4 *>(gamma + c0 + 8 * v));
        const float4 g1 = __ldg(reinterpret_cast<const float4 *>(gamma + c0 + 8 * v + 4));
        const float4 b0 = __ldg(reinterpret_cast<const float4 *>(beta + c0 + 8 * v));
        const float4 b1 = __ldg(reinterpret_cast<const float4 *>(beta + c0 + 8 * v + 4));
        g[k][0] = g0.x; g[k][1] = g0.y; g[k][2] = g0.z; g[k][3] = g0.w;
        g[k][4] = g1.x; g[k][5] = g1.y; g[k][6] = g1.z; g[k][7] = g1.w;
        bb[k][0] = b0.x; bb[k][1] = b0.y; bb[k][2] = b0.z; bb[k][3] = b0.w;
        bb[k][4] = b1.x; bb[k][5] = b1.y; bb[k][6] = b1.z; bb[k][7] = b1.w;
    };
    if (AFFINE && REGP) {
#pragma unroll
        for (int k = 0; k < NV; ++k)
            if (threadIdx.x + k * blockDim.x < nvec) load_params(k);
    }

    // Sends this CTA's (sum, M2) (held by every thread) to slot[p][rank] of
    // every CTA of the cluster and waits until all nranks pairs have arrived.
    bool xfail = false;
    auto exchange = [&](float sum, float m2, int p, uint32_t parity) {
        if (threadIdx.x == 0 && !xfail) ptx::mbar_arrive_expect_tx(&xbar[p], nranks * 8u);
        if (threadIdx.x < nranks)
            ptx::st_async_f32x2(ptx::mapa_shared(&slot[p][rank], threadIdx.x), sum, m2,
                                ptx::mapa_shared(&xbar[p], threadIdx.x));
        const bool ok = !xfail && ptx::mbar_wait<true>(&xbar[p], parity, wait_ns);
        if (!ok && !xfail) {   // a peer stalled: stop using the barriers (results are void)
            xfail = true;
            atomicOr(err, TF_DEVERR_EXCHANGE_WAIT);
        }
    };

    const float inv_h = 1.0f / (float)hidden;
    const float inv_w = 1.0f / (float)width;
    // Merge terms of rank r (lane r of every warp): its column count and its
    // reciprocal, fixed for the kernel
    const uint32_t lane = threadIdx.x & 31u;
    const float n_l = lane < nranks ? (float)min(hidden - (int)lane * slice, slice) : 0.0f;
    const float inv_n_l = lane < nranks ? 1.0f / n_l : 0.0f;
    // After a copy time-out this CTA stops waiting for and issuing copies but
    // still runs every row and every exchange, so its peers never wait on it.
    bool failed = false;
    int fail_it = 0;                     // the first row whose copy timed out
    int issued_until = stages;           // this CTA's rows 0 .. issued_until-1 had copies issued
    int it = 0;
    for (int64_t row = cid; row < rows; row += ncl, ++it) {
        const int st = it % stages;
        const int pb = it & 1;
        const uint32_t xpar = (uint32_t)(it >> 1) & 1u;
        // a wait that runs out is reported through copy_fail, which every
        // thread reads after the row's first reduction barrier (the values read
        // from a stage that never filled are garbage, and the results void)
        if (!failed && !ptx::mbar_wait(&full[st], (uint32_t)(it / stages) & 1u, wait_ns)) copy_fail = 1;
        const unsigned char *src = smem + (size_t)st * stage_bytes;
        float sv[NV][8];
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            uint4 av = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
            if (v < nvec) {
                av = reinterpret_cast<const uint4 *>(src)[v];
                if (RESIDUAL) bv = reinterpret_cast<const uint4 *>(src + (size_t)slice * 2)[v];
            }
            const __half2 *ah = reinterpret_cast<const __half2 *>(&av);
            const __half2 *bh = reinterpret_cast<const __half2 *>(&bv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = __half22float2(ah[j]);
                if (RESIDUAL) {
                    const float2 u = __half22float2(bh[j]);
                    f.x += u.x;
                    f.y += u.y;
                }
                sv[k][2 * j] = f.x;
                sv[k][2 * j + 1] = f.y;
                sum += f.x + f.y;
            }
        }
        // Two reductions per row, one barrier each: the sum uses red[0], the
        // squared deviations red[1], and between a reduction and the next use
        // of its buffer lies the other one's barrier.
        const float total = cta_sum_alt(sum, red[0]);
        if (copy_fail && !failed) {
            failed = true;
            fail_it = it;
            if (threadIdx.x == 0) atomicOr(err, TF_DEVERR_PRODUCER_WAIT);
        }
        // this slice's own mean and sum of squared deviations from it ...
        const float mean_c = total * inv_w;
        float sq = 0.0f;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            if (threadIdx.x + k * blockDim.x < nvec) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float d = sv[k][j] - mean_c;
                    sq = fmaf(d, d, sq);
                }
            }
        }
        exchange(total, cta_sum_alt(sq, red[1]), pb, xpar);
        // ... merged over the slices (Chan et al.'s pairwise update):
        // M2 = sum_r M2_r + sum_r n_r (mean_r - mean)^2.  Lane r of every warp
        // takes rank r's terms and the warp sums them with the same shuffle
        // butterfly (each level adds the same two values in either lane), so
        // every thread of the cluster gets the same mean and M2.
        const float2 pr = lane < nranks ? slot[pb][lane] : make_float2(0.0f, 0.0f);
        float tsum = pr.x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tsum += __shfl_xor_sync(0xffffffffu, tsum, o);
        const float mean = tsum * inv_h;
        const float dl = pr.x * inv_n_l - mean;
        float m2 = lane < nranks ? fmaf(n_l * dl, dl, pr.y) : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
        const float rstd = rsqrtf(m2 * inv_h + eps);
        __half *yr = y + row * hidden + c0;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int v = threadIdx.x + k * blockDim.x;
            if (v >= nvec) continue;
            if (AFFINE && !REGP) load_params(k);
            uint4 out;
            __half2 *oh = reinterpret_cast<__half2 *>(&out);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float o0 = (sv[k][2 * j] - mean) * rstd, o1 = (sv[k][2 * j + 1] - mean) * rstd;
                oh[j] = AFFINE ? __floats2half2_rn(fmaf(o0, g[k][2 * j], bb[k][2 * j]),
                                                   fmaf(o1, g[k][2 * j + 1], bb[k][2 * j + 1]))
                               : __floats2half2_rn(o0, o1);
            }
            st_stream(yr + 8 * v, out);
        }
        // stage `st` (read by every thread before the first reduction) takes the
        // row `stages` ahead; issued at the end of the row, off the path between
        // the row's two reductions
        if (threadIdx.x == blockDim.x - 1) {
            const int64_t next = row + (int64_t)stages * ncl;
            if (next < rows && !failed) {
                ptx::fence_proxy_async_smem();
                issue(st, next);
                issued_until = it + stages + 1;
            }
        }
    }
    if (threadIdx.x == blockDim.x - 1 && failed) {   // copies issued but never consumed land before exit
        for (int k = fail_it; k < issued_until; ++k) {
            const int64_t row = cid + (int64_t)k * ncl;
            if (row >= rows) break;
            if (!ptx::mbar_wait(&full[k % stages], (uint32_t)(k / stages) & 1u, wait_ns))
                atomicOr(err, TF_DEVERR_DRAIN_WAIT);
        }
    }
    ptx::cluster_sync();   // no CTA leaves while a peer's push to it may be in flight
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
cudaError_t launch_ln_cta(const void *a, const void *b, const float *gamma, const float *beta, void *y,
                          int64_t rows, int64_t hidden, float eps, cudaStream_t st)
{
    if (hidden > kCtaMaxHidden) return cudaErrorNotSupported;
    uint32_t *err = device_error_word();
    if (!err) return cudaErrorInitializationError;
    const int threads = threads_for(hidden, 2);
    const size_t stage_bytes = (size_t)hidden * 2 * (RESIDUAL ? 2 : 1);
    // Ring depth: up to 4 rows, within ~96 KB of shared memory per CTA.
    int stages = (int)((96 * 1024) / stage_bytes);
    stages = stages < 2 ? 2 : (stages > 4 ? 4 : stages);
    const size_t smem = (size_t)stages * stage_bytes + 8 * (size_t)stages;
    auto kern = layernorm_kernel<2, RESIDUAL, AFFINE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t grid = (int64_t)sm_count() * per_sm;
    if (grid > rows) grid = rows;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(threads), smem, st, reinterpret_cast<const __half *>(a),
                      reinterpret_cast<const __half *>(b), gamma, beta, reinterpret_cast<__half *>(y), rows,
                      (int)hidden, eps, stages, err, wait_limit_ns());
}

template <bool RESIDUAL, bool AFFINE>
cudaError_t launch_ln_warp(const void *a, const void *b, const float *gamma, const float *beta, void *y,
                           int64_t rows, int64_t hidden, float eps, cudaStream_t st)
{
    if (hidden > kWarpMaxHidden) return cudaErrorNotSupported;
    const int nvec = (int)(hidden / 8);
    auto pick = [&](auto kern) -> cudaError_t {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        int64_t grid = (int64_t)sm_count() * per_sm;
        const int64_t need = (rows + 7) / 8;
        if (grid > need) grid = need;
        return launch_pdl(kern, dim3((unsigned)grid), dim3(256), 0, st, reinterpret_cast<const __half *>(a),
                          reinterpret_cast<const __half *>(b), gamma, beta, reinterpret_cast<__half *>(y), rows,
                          (int)hidden, eps);
    };
    if (nvec <= 32) return pick(layernorm_warp_kernel<1, RESIDUAL, AFFINE>);
    if (nvec <= 64) return pick(layernorm_warp_kernel<2, RESIDUAL, AFFINE>);
    return pick(layernorm_warp_kernel<4, RESIDUAL, AFFINE>);
}

// Cluster size (2..max_csize CTAs) and slice width for a row of `hidden`
// columns cut into slices of at most about `target` columns; no CTA is left
// with an empty slice.
void cluster_geometry(int64_t hidden, int target, int max_csize, int &csize, int64_t &slice)
{
    csize = (int)((hidden + target - 1) / target);
    if (csize < 2) csize = 2;
    if (csize > max_csize) csize = max_csize;
    while (csize > 1 && (csize - 1) * (((hidden + csize - 1) / csize + 7) / 8 * 8) >= hidden) --csize;
    slice = ((hidden + csize - 1) / csize + 7) / 8 * 8;
}

template <bool RESIDUAL, bool AFFINE, int NV, int MAXT, bool REGP>
cudaError_t launch_ln_cluster_with(const void *a, const void *b, const float *gamma, const float *beta, void *y,
                                   int64_t rows, int64_t hidden, float eps, int csize, int64_t slice, uint32_t *err,
                                   cudaStream_t st)
{
    const int threads = threads_for(slice, NV);
    if (threads > MAXT) return cudaErrorNotSupported;
    const size_t stage_bytes = (size_t)slice * 2 * (RESIDUAL ? 2 : 1);
    int stages = (int)((96 * 1024) / stage_bytes);
    stages = stages < 2 ? 2 : (stages > 4 ? 4 : stages);
    const size_t smem = (size_t)stages * stage_bytes + 8 * (size_t)stages;
    auto kern = layernorm_cluster_kernel<RESIDUAL, AFFINE, NV, MAXT, REGP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess && csize > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        cudaGetLastError();   // a refused attribute is not an error of the caller's stream
        return cudaErrorNotSupported;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_begin()
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(sm_count() / csize * csize);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    if (clusters > rows) clusters = (int)rows;
    cfg.gridDim = dim3((unsigned)(clusters * csize));
    return counted(cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const __half *>(a), reinterpret_cast<const __half *>(b),
                              gamma, beta, reinterpret_cast<__half *>(y), rows, (int)hidden, (int)slice, eps, stages,
                              err, wait_limit_ns()));
}

template <bool RESIDUAL, bool AFFINE>
cudaError_t launch_ln_cluster(const void *a, const void *b, const float *gamma, const float *beta, void *y,
                              int64_t rows, int64_t hidden, float eps, cudaStream_t st)
{
    if (hidden > kClusterMaxHidden) return cudaErrorNotSupported;
    uint32_t *err = device_error_word();
    if (!err) return cudaErrorInitializationError;
    // Slices of at most 8192 columns (256 threads, two CTAs per SM) so that
    // gamma and beta fit in registers: clusters of up to 8 CTAs to 65536
    // columns, 16 beyond.  Where the GPU cannot form 16-CTA clusters,
    // portable clusters of 8 CTAs with slices of up to 16384 columns.
    int csize;
    int64_t slice;
    cluster_geometry(hidden, 8192, 16, csize, slice);
    cudaError_t e = launch_ln_cluster_with<RESIDUAL, AFFINE, 4, 256, true>(a, b, gamma, beta, y, rows, hidden, eps,
                                                                            csize, slice, err, st);
    if (e != cudaErrorNotSupported) return e;
    cluster_geometry(hidden, 8192, 8, csize, slice);
    return launch_ln_cluster_with<RESIDUAL, AFFINE, 2, 1024, false>(a, b, gamma, beta, y, rows, hidden, eps, csize,
                                                                    slice, err, st);
}

template <bool RESIDUAL, bool AFFINE>
cudaError_t launch_ln(const void *a, const void *b, const float *gamma, const float *beta, void *y,
                      int64_t rows, int64_t hidden, float eps, int variant, cudaStream_t st)
{
    if (variant == TF_LN_AUTO) variant = layernorm_select(hidden);
    switch (variant) {
    case TF_LN_WARP: return launch_ln_warp<RESIDUAL, AFFINE>(a, b, gamma, beta, y, rows, hidden, eps, st);
    case TF_LN_CTA: return launch_ln_cta<RESIDUAL, AFFINE>(a, b, gamma, beta, y, rows, hidden, eps, st);
    case TF_LN_CLUSTER: return launch_ln_cluster<RESIDUAL, AFFINE>(a, b, gamma, beta, y, rows, hidden, eps, st);
    default: return cudaErrorNotSupported;
    }
}

}  // namespace

int layernorm_select(int64_t hidden)
{
    if (hidden <= kWarpBoundary) return TF_LN_WARP;
    if (hidden <= kCtaMaxHidden) return TF_LN_CTA;
    if (hidden <= kClusterMaxHidden) return TF_LN_CLUSTER;
    return -TF_ERR_UNSUPPORTED;
}

cudaError_t launch_residual_layernorm(const void *act, const void *res, const float *gamma,
                                      const float *beta, void *y, int64_t rows, int64_t hidden,
                                      float eps, int variant, cudaStream_t st)
{
    return launch_ln<true, true>(act, res, gamma, beta, y, rows, hidden, eps, variant, st);
}

cudaError_t launch_unfused_layernorm(const void *s, void *nrm, int64_t rows, int64_t hidden, float eps,
                                     cudaStream_t st)
{
    return launch_ln<false, false>(s, nullptr, nullptr, nullptr, nrm, rows, hidden, eps, TF_LN_AUTO, st);
}

}  // namespace tf
