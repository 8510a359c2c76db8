// Memory-bound kernels: the channels-last filter pack, fused bias + GELU and
// the separate elementwise kernels of the unfused comparison chains.
//
// Every streaming kernel moves 16 bytes per thread per access (eight fp16 or
// bf16 values), reads with the non-coherent streaming path and writes with
// evict-first stores, and runs a grid of a few CTAs per SM that strides over
// the tensor, so each thread keeps several independent 16-byte loads in flight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx_sm100.cuh"
#include "tf_internal.h"

namespace tf {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // independent 16-byte vectors per thread per iteration

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

__device__ __forceinline__ void h8_to_f(const uint4 &v, float (&f)[8])
{
    const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 f_to_h8(const float (&f)[8])
{
    uint4 v;
    __half2 *h = reinterpret_cast<__half2 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

__device__ __forceinline__ void b8_to_f(const uint4 &v, float (&f)[8])
{
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 f_to_b8(const float (&f)[8])
{
    uint4 v;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

// Grid size for a grid-stride kernel over `nvec` 16-byte vectors: one wave
// of resident CTAs, never more than the work needs.
unsigned grid_for(const void *kernel, int64_t nvec)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t per_cta = (int64_t)kThreads * kUnroll;
    int64_t need = (nvec + per_cta - 1) / per_cta;
    int64_t cap = (int64_t)sm_count() * per_sm;
    int64_t g = need < cap ? need : cap;
    return (unsigned)(g > 0 ? g : 1);
}

// ---------------------------------------------------------------- bias + GELU

// y = GELU(x + bias[col]).  cols % 8 == 0.  A grid-stride loop over 16-byte
// vectors (8 values) whose stride S is a multiple of the row length in
// vectors whenever S >= cvec, so each thread's column -- and its bias, kept in
// registers -- never changes, while the whole grid reads one compact window
// of the tensor at a time.  Four independent loads are in flight per thread.
__global__ void __launch_bounds__(kThreads) bias_gelu_kernel(const uint4 *__restrict__ x,
                                                             const uint4 *__restrict__ bias,
                                                             uint4 *__restrict__ y, int64_t nvec,
                                                             int64_t cvec)
{
    pdl_begin();
    const int64_t S = (int64_t)gridDim.x * kThreads;
    int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool fixed_col = S % cvec == 0;
    float b[8];
    h8_to_f(__ldg(bias + i % cvec), b);
    for (; i + 3 * S < nvec; i += 4 * S) {
        uint4 xv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) xv[u] = ld_stream(x + i + u * S);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!fixed_col) h8_to_f(__ldg(bias + (i + u * S) % cvec), b);
            const __half2 *h = reinterpret_cast<const __half2 *>(&xv[u]);
            uint4 o;
            __half2 *oh = reinterpret_cast<__half2 *>(&o);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 sv = fadd2(__half22float2(h[k]), make_float2(b[2 * k], b[2 * k + 1]));
                const float2 g = gelu_f32x2(sv);
                oh[k] = __floats2half2_rn(g.x, g.y);
            }
            st_stream(y + i + u * S, o);
        }
    }
    for (; i < nvec; i += S) {
        if (!fixed_col) h8_to_f(__ldg(bias + i % cvec), b);
        const uint4 xv = ld_stream(x + i);
        const __half2 *h = reinterpret_cast<const __half2 *>(&xv);
        uint4 o;
        __half2 *oh = reinterpret_cast<__half2 *>(&o);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 sv = fadd2(__half22float2(h[k]), make_float2(b[2 * k], b[2 * k + 1]));
            const float2 g = gelu_f32x2(sv);
            oh[k] = __floats2half2_rn(g.x, g.y);
        }
        st_stream(y + i, o);
    }
}

// Rows of up to 16384 columns: persistent CTAs walk chunks of whole rows (at
// most 32 KB), chunk c, c + gridDim.x, ...  A 17th warp, the copy warp,
// streams the coming chunks of x into a 3-stage shared-memory ring with 1-D
// bulk copies and writes each computed chunk back with a bulk store, so both
// directions move through the copy engine; the 16 compute warps compute
// GELU(x + bias) in place.  Compute warps and copy warp meet only at two
// mbarriers per stage (loaded; computed by all 16 warps), never at a CTA-wide
// barrier, and a stage is refilled as soon as its store has read it (5% faster
// than one thread of a compute warp doing the copies between two CTA
// barriers per chunk).  A chunk holds whole rows, so thread t's vectors
// t + 512k always have the same columns: their bias stays in registers.
// Waits are bounded; after a time-out the warps stop, the copy warp drains
// its copies and the error is recorded.
constexpr int kRingThreads = 512;
constexpr int kRingVecs = 4;                       // vectors per thread per chunk: 512 * 4 * 16 B = 32 KB
constexpr int kRingChunkBytes = kRingThreads * kRingVecs * 16;

constexpr int kRingBlock = kRingThreads + 32;   // 16 compute warps + 1 copy warp

__global__ void __launch_bounds__(kRingBlock, 2) bias_gelu_ring_kernel(const uint4 *__restrict__ x,
                                                                      const uint4 *__restrict__ bias,
                                                                      uint4 *__restrict__ y, int64_t rows,
                                                                      int cvec, int rps, int stages,
                                                                      uint32_t *err, uint64_t wait_ns)
{
    pdl_begin();
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)stages * kRingChunkBytes);
    uint64_t *done = full + stages;   // a stage's chunk computed in place by all 16 warps
    const int64_t nchunks = (rows + rps - 1) / rps;
    const int64_t G = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto chunk_bytes = [&](int64_t c) -> uint32_t {
        const int64_t r = rows - c * rps < rps ? rows - c * rps : rps;
        return (uint32_t)(r * cvec * 16);
    };
    if (threadIdx.x == kRingThreads) {
        for (int st = 0; st < stages; ++st) {
            ptx::mbar_init(&full[st], 1);
            ptx::mbar_init(&done[st], kRingThreads / 32);
        }
        ptx::mbar_init_fence();
    }
    cta_sync();
    if (warp == kRingThreads / 32) {
        // the copy warp: loads into free stages, stores computed ones
        if (lane != 0) return;
        auto issue = [&](int st, int64_t c) {
            const uint32_t bytes = chunk_bytes(c);
            ptx::mbar_arrive_expect_tx(&full[st], bytes);
            ptx::bulk_load(smem + (size_t)st * kRingChunkBytes, x + c * rps * cvec, bytes, &full[st]);
        };
        int issued = 0;   // chunks of this CTA whose loads were issued
        for (int st = 0; st < stages; ++st) {
            if (blockIdx.x + st * G >= nchunks) break;
            issue(st, blockIdx.x + st * G);
            issued = st + 1;
        }
        int it = 0;
        for (int64_t c = blockIdx.x; c < nchunks; c += G, ++it) {
            const int st = it % stages;
            if (!ptx::mbar_wait(&done[st], (uint32_t)(it / stages) & 1u, wait_ns)) {
                atomicOr(err, TF_DEVERR_PRODUCER_WAIT);
                break;
            }
            ptx::bulk_store(y + c * rps * cvec, smem + (size_t)st * kRingChunkBytes, chunk_bytes(c));
            ptx::bulk_commit_group();
            const int64_t next = c + (int64_t)stages * G;
            if (next < nchunks) {
                ptx::bulk_wait_group_read<0>();   // the store has read the stage: refill it
                issue(st, next);
                issued = it + stages + 1;
            }
        }
        ptx::bulk_wait_group_all();   // every store has written y
        // loads issued for chunks never computed (only after a time-out) land before exit
        for (int k = it; k < issued; ++k)
            if (!ptx::mbar_wait(&full[k % stages], (uint32_t)(k / stages) & 1u, wait_ns))
                atomicOr(err, TF_DEVERR_DRAIN_WAIT);
        return;
    }
    float b[kRingVecs][8];
#pragma unroll
    for (int k = 0; k < kRingVecs; ++k) h8_to_f(__ldg(bias + (threadIdx.x + k * kRingThreads) % cvec), b[k]);

    int it = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += G, ++it) {
        const int st = it % stages;
        // one decision per warp, so that no lane leaves its warp-mates in a warp collective
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&full[st], (uint32_t)(it / stages) & 1u, wait_ns))) {
            if (lane == 0) atomicOr(err, TF_DEVERR_PRODUCER_WAIT);
            break;   // the copy warp's wait for this chunk then runs out too
        }
        uint4 *buf = reinterpret_cast<uint4 *>(smem + (size_t)st * kRingChunkBytes);
        const int nv = (int)(chunk_bytes(c) / 16);
#pragma unroll
        for (int k = 0; k < kRingVecs; ++k) {
            const int v = threadIdx.x + k * kRingThreads;
            if (v >= nv) break;
            const uint4 xv = buf[v];
            const __half2 *h = reinterpret_cast<const __half2 *>(&xv);
            uint4 o;
            __half2 *oh = reinterpret_cast<__half2 *>(&o);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 sv = fadd2(__half22float2(h[j]), make_float2(b[k][2 * j], b[k][2 * j + 1]));
                const float2 g = gelu_f32x2(sv);
                oh[j] = __floats2half2_rn(g.x, g.y);
            }
            buf[v] = o;
        }
        ptx::fence_proxy_async_smem();   // the generic-proxy writes, before the bulk store reads them
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&done[st]);
    }
}

// ---------------------------------------------------------------- unfused pieces

enum class Op { BiasAddF16, GeluF16, ResidualAddF16, BnBf16, SiluBf16, AffineF16 };

__host__ __device__ constexpr bool has_column_params(Op op) { return op == Op::BiasAddF16 || op == Op::BnBf16 || op == Op::AffineF16; }

// Per-column parameters of one 16-byte vector (columns c0 .. c0+7): the fp16
// bias (BiasAddF16), or the fp32 scale/gamma and bias/beta pairs.
template <Op OP>
__device__ __forceinline__ void column_params(const void *b, const float *p0, const float *p1, int64_t cv,
                                              float (&m)[8], float (&a)[8])
{
    if constexpr (OP == Op::BiasAddF16) {
        h8_to_f(__ldg(reinterpret_cast<const uint4 *>(b) + cv), a);
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] = 1.0f;
    } else if constexpr (OP == Op::BnBf16 || OP == Op::AffineF16) {
        const float4 *q0 = reinterpret_cast<const float4 *>(p0 + 8 * cv);
        const float4 *q1 = reinterpret_cast<const float4 *>(p1 + 8 * cv);
        const float4 x0 = __ldg(q0), x1 = __ldg(q0 + 1), y0 = __ldg(q1), y1 = __ldg(q1 + 1);
        m[0] = x0.x; m[1] = x0.y; m[2] = x0.z; m[3] = x0.w; m[4] = x1.x; m[5] = x1.y; m[6] = x1.z; m[7] = x1.w;
        a[0] = y0.x; a[1] = y0.y; a[2] = y0.z; a[3] = y0.w; a[4] = y1.x; a[5] = y1.y; a[6] = y1.z; a[7] = y1.w;
    }
}

template <Op OP>
__device__ __forceinline__ uint4 chain_op(const uint4 &va, const uint4 *bsrc, int64_t i, const float (&m)[8],
                                          const float (&a)[8])
{
    float f[8];
    if constexpr (OP == Op::BnBf16 || OP == Op::SiluBf16) b8_to_f(va, f);
    else h8_to_f(va, f);
    if constexpr (OP == Op::ResidualAddF16) {
        float g[8];
        h8_to_f(ld_stream(bsrc + i), g);
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] += g[k];
    } else if constexpr (OP == Op::GeluF16) {
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float2 t = gelu_f32x2(make_float2(f[k], f[k + 1]));
            f[k] = t.x;
            f[k + 1] = t.y;
        }
    } else if constexpr (OP == Op::SiluBf16) {
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const float2 t = silu_f32x2(make_float2(f[k], f[k + 1]));
            f[k] = t.x;
            f[k + 1] = t.y;
        }
    } else if constexpr (OP == Op::BiasAddF16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] += a[k];
    } else {   // BnBf16, AffineF16: f * m + a
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = fmaf(f[k], m[k], a[k]);
    }
    if constexpr (OP == Op::BnBf16 || OP == Op::SiluBf16) return f_to_b8(f);
    else return f_to_h8(f);
}

// One elementwise step of an unfused chain: reads one (or two) tensors,
// writes one, in the storage type of the chain (bf16 for the conv chain,
// fp16 otherwise).  Built like bias_gelu_kernel -- grid-stride over 16-byte
// vectors with a stride that is a multiple of the row length when it can be,
// so per-column parameters stay in registers, and four loads in flight -- so
// that the fused kernels are compared against equally careful kernels.
template <Op OP>
__global__ void __launch_bounds__(kThreads) chain_kernel(const uint4 *__restrict__ a, const void *__restrict__ b,
                                                         const float *__restrict__ p0, const float *__restrict__ p1,
                                                         uint4 *__restrict__ out, int64_t nvec, int64_t cvec)
{
    pdl_begin();
    const int64_t S = (int64_t)gridDim.x * kThreads;
    int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const bool fixed_col = S % cvec == 0;
    const uint4 *bsrc = reinterpret_cast<const uint4 *>(b);
    float m[8] = {}, ad[8] = {};
    if constexpr (has_column_params(OP)) column_params<OP>(b, p0, p1, i % cvec, m, ad);
    for (; i + 3 * S < nvec; i += 4 * S) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = ld_stream(a + i + u * S);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (has_column_params(OP) && !fixed_col) column_params<OP>(b, p0, p1, (i + u * S) % cvec, m, ad);
            st_stream(out + i + u * S, chain_op<OP>(v[u], bsrc, i + u * S, m, ad));
        }
    }
    for (; i < nvec; i += S) {
        if (has_column_params(OP) && !fixed_col) column_params<OP>(b, p0, p1, i % cvec, m, ad);
        st_stream(out + i, chain_op<OP>(ld_stream(a + i), bsrc, i, m, ad));
    }
}

// One wave of resident CTAs, the stride a multiple of cvec when possible.
template <Op OP>
cudaError_t launch_chain(const void *a, const void *b, const float *p0, const float *p1, void *out, int64_t n,
                         int64_t cols, cudaStream_t st)
{
    const int64_t nvec = n / 8, cvec = cols / 8;
    int64_t grid = grid_for(reinterpret_cast<const void *>(chain_kernel<OP>), nvec);
    int64_t x = cvec, y = kThreads;
    while (y) { const int64_t t = x % y; x = y; y = t; }   // gcd(cvec, threads)
    const int64_t unit = cvec / x;
    if (grid >= unit) grid = grid / unit * unit;
    return launch_pdl(chain_kernel<OP>, dim3((unsigned)grid), dim3(kThreads), 0, st, reinterpret_cast<const uint4 *>(a),
                      b, p0, p1, reinterpret_cast<uint4 *>(out), nvec, cvec);
}

// ---------------------------------------------------------------- filter pack

// w_ohwi[co][kh][kw][ci] = w_oihw[co][ci][kh][kw].  One thread per output
// word, so the writes are contiguous; runs once at load time.
__global__ void pack_filter_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                   int C_out, int C_in, int KH, int KW)
{
    pdl_begin();
    const int64_t total = (int64_t)C_out * C_in * KH * KW;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += stride) {
        int64_t r = o;
        const int ci = (int)(r % C_in);
        r /= C_in;
        const int kw = (int)(r % KW);
        r /= KW;
        const int kh = (int)(r % KH);
        const int64_t co = r / KH;
        dst[o] = src[((co * C_in + ci) * KH + kh) * KW + kw];
    }
}

}  // namespace

cudaError_t launch_bias_gelu(const void *x, const void *bias, void *y, int64_t rows, int64_t cols,
                             cudaStream_t st)
{
    const int64_t cvec = cols / 8;
    if (cols * 2 <= kRingChunkBytes) {
        // the bulk-copy ring: chunks of whole rows
        uint32_t *err = device_error_word();
        if (!err) return cudaErrorInitializationError;
        const int rps = (int)(kRingChunkBytes / (cols * 2));
        const int stages = 3;
        const size_t smem = (size_t)stages * kRingChunkBytes + 16 * stages;
        cudaError_t e = cudaFuncSetAttribute(bias_gelu_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bias_gelu_ring_kernel, kRingBlock, smem) !=
                cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int64_t nchunks = (rows + rps - 1) / rps;
        int64_t grid = (int64_t)sm_count() * per_sm;
        if (grid > nchunks) grid = nchunks;
        return launch_pdl(bias_gelu_ring_kernel, dim3((unsigned)grid), dim3(kRingBlock), smem, st,
                          reinterpret_cast<const uint4 *>(x), reinterpret_cast<const uint4 *>(bias),
                          reinterpret_cast<uint4 *>(y), rows, (int)cvec, rps, stages, err, wait_limit_ns());
    }
    const int64_t nvec = rows * cvec;
    int64_t grid = grid_for(reinterpret_cast<const void *>(bias_gelu_kernel), nvec);
    // make the stride (grid * threads) a multiple of cvec when it can be, so
    // every thread keeps one column
    int64_t a = cvec, bq = kThreads;
    while (bq) { const int64_t t = a % bq; a = bq; bq = t; }   // gcd(cvec, threads)
    const int64_t unit = cvec / a;                             // CTAs per whole number of rows
    if (grid >= unit) grid = grid / unit * unit;
    return launch_pdl(bias_gelu_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, reinterpret_cast<const uint4 *>(x),
                      reinterpret_cast<const uint4 *>(bias), reinterpret_cast<uint4 *>(y), nvec, cvec);
}

cudaError_t launch_unfused_bias_add(const void *x, const void *bias, void *t, int64_t rows,
                                    int64_t cols, cudaStream_t st)
{
    return launch_chain<Op::BiasAddF16>(x, bias, nullptr, nullptr, t, rows * cols, cols, st);
}

cudaError_t launch_unfused_gelu(const void *t, void *y, int64_t n, cudaStream_t st)
{
    return launch_chain<Op::GeluF16>(t, nullptr, nullptr, nullptr, y, n, 8, st);
}

cudaError_t launch_unfused_residual_add(const void *a, const void *r, void *s, int64_t n,
                                        cudaStream_t st)
{
    return launch_chain<Op::ResidualAddF16>(a, r, nullptr, nullptr, s, n, 8, st);
}

cudaError_t launch_unfused_bn(const void *t1, const float *scale, const float *bias, void *t2,
                              int64_t M, int64_t C, cudaStream_t st)
{
    return launch_chain<Op::BnBf16>(t1, nullptr, scale, bias, t2, M * C, C, st);
}

cudaError_t launch_unfused_silu(const void *t2, void *y, int64_t n, cudaStream_t st)
{
    return launch_chain<Op::SiluBf16>(t2, nullptr, nullptr, nullptr, y, n, 8, st);
}

cudaError_t launch_unfused_affine(const void *nrm, const float *gamma, const float *beta, void *y, int64_t rows,
                                  int64_t hidden, cudaStream_t st)
{
    return launch_chain<Op::AffineF16>(nrm, nullptr, gamma, beta, y, rows * hidden, hidden, st);
}

cudaError_t launch_pack_filter(const void *w_oihw, void *w_ohwi, int C_out, int C_in, int KH, int KW,
                               cudaStream_t st)
{
    const int64_t total = (int64_t)C_out * C_in * KH * KW;
    int64_t g = (total + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 16;
    if (g > cap) g = cap;
    return launch_pdl(pack_filter_kernel, dim3((unsigned)g), dim3(256), 0, st, reinterpret_cast<const uint16_t *>(w_oihw),
                      reinterpret_cast<uint16_t *>(w_ohwi), C_out, C_in, KH, KW);
}

}  // namespace tf
