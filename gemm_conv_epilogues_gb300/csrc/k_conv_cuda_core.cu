// CUDA-core conv2d + BN + SiLU kernels for shapes where tensor-core tiles
// would be mostly empty.  "Fusing an Epilogue", "Three kernels for one
// operation": a scalar kernel with one output element per lane (no set-up
// cost, best on small shapes) and a kernel tiled over the output spatial
// extent.  Both accumulate in fp32 and apply the same epilogue as the
// tensor-core path: v = acc*scale[co] + bias[co], y = v*sigmoid(v), bf16.
#include <cuda_bf16.h>

#include "tf_internal.h"

namespace tf {
namespace {

__device__ __forceinline__ void bf8(const uint4 &v, float (&f)[8])
{
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ float epilogue(float acc, int co, const float *scale, const float *bias, int epi)
{
    if (!epi) return acc;
    return silu_f32(acc * __ldg(scale + co) + __ldg(bias + co));
}

// ---------------------------------------------------------------- direct

// One thread per output element y[n][oh][ow][co]; co is the fastest index so a
// warp's x reads are broadcasts and its y writes are contiguous.
//
// BATCHED: the K loop runs over units of one filter tap and 8 input channels
// (one 16-byte x vector and one filter vector), kBatch units at a time, and a
// batch's vectors are all loaded (zeros where the tap lies in the padding)
// before its first FMA: a thread waits for memory once per batch (a 3x3 filter
// over 8 input channels is one batch).  That pays where each thread's
// reduction is a few taps of few channels and there are few threads (small
// 3x3 layers: the tiny workload's 1x16x16, 8 -> 16 takes 2.5 us against 4.2);
// with more threads, or long channel runs per tap, the registers it holds cost
// more occupancy than its loads gain, and the tap-by-tap loop (whose channel
// loop the compiler unrolls) is faster.  Batched layers have fewer than 2^31
// outputs by construction (see launch_conv_direct).
constexpr int kBatch = 9;

template <bool BATCHED>
__global__ void __launch_bounds__(256) conv_direct_kernel(ConvArgs a)
{
    pdl_begin();
    const tf_conv_shape s = a.s;
    const int64_t total = (int64_t)s.N * a.Ho * a.Wo * s.C_out;
    const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= total) return;
    float acc = 0.0f;
    int co;
    if constexpr (BATCHED) {
        // (launched only for small layers: 32-bit output index)
        int r = (int)o;
        co = r % s.C_out;
        r /= s.C_out;
        const int ow = r % a.Wo;
        r /= a.Wo;
        const int oh = r % a.Ho;
        const int n = r / a.Ho;
        const uint4 *x = reinterpret_cast<const uint4 *>(a.x);
        const int cch = s.C_in / 8;   // 16-byte chunks per pixel and per filter tap
        const int units = s.KH * s.KW * cch;
        const uint4 *w = reinterpret_cast<const uint4 *>(a.w) + (int64_t)co * units;   // unit u at w[u]
        const int ih0 = oh * s.stride_h - s.pad_h, iw0 = ow * s.stride_w - s.pad_w;
        const int64_t img = (int64_t)n * s.H;
        const uint4 zero = make_uint4(0, 0, 0, 0);
        int kh = 0, kw = 0, c = 0;   // the next unit's tap and chunk
        for (int u0 = 0; u0 < units; u0 += kBatch) {
            uint4 xv[kBatch], wv[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int ih = ih0 + kh, iw = iw0 + kw;
                const bool in = u0 + j < units && (unsigned)ih < (unsigned)s.H && (unsigned)iw < (unsigned)s.W;
                xv[j] = in ? __ldg(x + ((img + ih) * s.W + iw) * cch + c) : zero;
                wv[j] = in ? __ldg(w + u0 + j) : zero;
                if (++c == cch) {
                    c = 0;
                    if (++kw == s.KW) {
                        kw = 0;
                        ++kh;
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (u0 + j >= units) break;
                float xf[8], wf[8];
                bf8(xv[j], xf);
                bf8(wv[j], wf);
#pragma unroll
                for (int k = 0; k < 8; ++k) acc = fmaf(xf[k], wf[k], acc);
            }
        }
    } else {
        int64_t r = o;
        co = (int)(r % s.C_out);
        r /= s.C_out;
        const int ow = (int)(r % a.Wo);
        r /= a.Wo;
        const int oh = (int)(r % a.Ho);
        const int n = (int)(r / a.Ho);
        const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(a.x);
        const __nv_bfloat16 *w = reinterpret_cast<const __nv_bfloat16 *>(a.w) + (int64_t)co * s.KH * s.KW * s.C_in;
        for (int kh = 0; kh < s.KH; ++kh) {
            const int ih = oh * s.stride_h - s.pad_h + kh;
            if (ih < 0 || ih >= s.H) continue;
            for (int kw = 0; kw < s.KW; ++kw) {
                const int iw = ow * s.stride_w - s.pad_w + kw;
                if (iw < 0 || iw >= s.W) continue;
                const uint4 *xp = reinterpret_cast<const uint4 *>(x + (((int64_t)n * s.H + ih) * s.W + iw) * s.C_in);
                const uint4 *wp = reinterpret_cast<const uint4 *>(w + ((int64_t)kh * s.KW + kw) * s.C_in);
                for (int c = 0; c < s.C_in / 8; ++c) {
                    float xf[8], wf[8];
                    bf8(__ldg(xp + c), xf);
                    bf8(__ldg(wp + c), wf);
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc = fmaf(xf[j], wf[j], acc);
                }
            }
        }
    }
    reinterpret_cast<__nv_bfloat16 *>(a.y)[o] = __float2bfloat16_rn(epilogue(acc, co, a.scale, a.bias, a.epilogue));
}

// ---------------------------------------------------------------- tiled

// One CTA computes a TH x TW tile of output pixels of one image for CO_T
// output channels.  For each chunk of 8 input channels it stages the input
// halo of the tile and the CO_T filters in shared memory; each thread owns
// one output pixel and CO_T fp32 accumulators.
constexpr int TH = 8, TW = 16, CO_T = 16, CI_T = 8;

__global__ void __launch_bounds__(TH * TW) conv_tiled_kernel(ConvArgs a, int halo_h, int halo_w)
{
    pdl_begin();
    extern __shared__ __align__(16) unsigned char smem[];
    const tf_conv_shape s = a.s;
    uint4 *xs = reinterpret_cast<uint4 *>(smem);                       // [halo_h][halo_w] x 8 channels
    uint4 *ws = xs + halo_h * halo_w;                                   // [CO_T][KH][KW] x 8 channels
    const int tiles_w = (a.Wo + TW - 1) / TW;
    const int oh0 = (blockIdx.x / tiles_w) * TH, ow0 = (blockIdx.x % tiles_w) * TW;
    const int n = blockIdx.y;
    const int co0 = blockIdx.z * CO_T;
    const int ty = threadIdx.x / TW, tx = threadIdx.x % TW;
    const int oh = oh0 + ty, ow = ow0 + tx;
    const int ih0 = oh0 * s.stride_h - s.pad_h, iw0 = ow0 * s.stride_w - s.pad_w;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(a.x);
    const __nv_bfloat16 *w = reinterpret_cast<const __nv_bfloat16 *>(a.w);
    const int taps = s.KH * s.KW;

    float acc[CO_T];
#pragma unroll
    for (int j = 0; j < CO_T; ++j) acc[j] = 0.0f;

    for (int c0 = 0; c0 < s.C_in; c0 += CI_T) {
        cta_sync();
        for (int i = threadIdx.x; i < halo_h * halo_w; i += blockDim.x) {
            const int ih = ih0 + i / halo_w, iw = iw0 + i % halo_w;
            uint4 v = zero;
            if (ih >= 0 && ih < s.H && iw >= 0 && iw < s.W)
                v = __ldg(reinterpret_cast<const uint4 *>(x + (((int64_t)n * s.H + ih) * s.W + iw) * s.C_in + c0));
            xs[i] = v;
        }
        for (int i = threadIdx.x; i < CO_T * taps; i += blockDim.x) {
            const int co = co0 + i / taps, t = i % taps;
            uint4 v = zero;
            if (co < s.C_out) v = __ldg(reinterpret_cast<const uint4 *>(w + ((int64_t)co * taps + t) * s.C_in + c0));
            ws[i] = v;
        }
        cta_sync();
        for (int kh = 0; kh < s.KH; ++kh) {
            for (int kw = 0; kw < s.KW; ++kw) {
                float xf[8];
                bf8(xs[(ty * s.stride_h + kh) * halo_w + tx * s.stride_w + kw], xf);
#pragma unroll
                for (int j = 0; j < CO_T; ++j) {
                    float wf[8];
                    bf8(ws[j * taps + kh * s.KW + kw], wf);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[j] = fmaf(xf[q], wf[q], acc[j]);
                }
            }
        }
    }
    if (oh >= a.Ho || ow >= a.Wo) return;
    __nv_bfloat16 *y = reinterpret_cast<__nv_bfloat16 *>(a.y) + (((int64_t)n * a.Ho + oh) * a.Wo + ow) * s.C_out;
#pragma unroll
    for (int j = 0; j < CO_T; ++j) {
        const int co = co0 + j;
        if (co < s.C_out) y[co] = __float2bfloat16_rn(epilogue(acc[j], co, a.scale, a.bias, a.epilogue));
    }
}

}  // namespace

cudaError_t launch_conv_direct(const ConvArgs &a, cudaStream_t st)
{
    const int64_t total = (int64_t)a.s.N * a.Ho * a.Wo * a.s.C_out;
    const int64_t grid = (total + 255) / 256;
    if (grid > 0x7fffffff) return cudaErrorNotSupported;
    // batched tap loads for small layers with several taps of few channels
    // (measured crossovers on GB300: from ~128K outputs or 64 input channels
    // on, the tap-by-tap loop is as fast or faster)
    const bool batched = a.s.KH * a.s.KW > 1 && a.s.C_in < 64 && total < 131072;
    if (batched) return launch_pdl(conv_direct_kernel<true>, dim3((unsigned)grid), dim3(256), 0, st, a);
    return launch_pdl(conv_direct_kernel<false>, dim3((unsigned)grid), dim3(256), 0, st, a);
}

cudaError_t launch_conv_tiled(const ConvArgs &a, cudaStream_t st)
{
    const tf_conv_shape &s = a.s;
    const int halo_h = (TH - 1) * s.stride_h + s.KH, halo_w = (TW - 1) * s.stride_w + s.KW;
    const size_t smem = sizeof(uint4) * ((size_t)halo_h * halo_w + (size_t)CO_T * s.KH * s.KW);
    if (smem > 200 * 1024 || s.N > 65535 || (s.C_out + CO_T - 1) / CO_T > 65535) return cudaErrorNotSupported;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(conv_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const dim3 grid((unsigned)(((a.Ho + TH - 1) / TH) * ((a.Wo + TW - 1) / TW)), (unsigned)s.N,
                    (unsigned)((s.C_out + CO_T - 1) / CO_T));
    return launch_pdl(conv_tiled_kernel, grid, dim3(TH * TW), smem, st, a, halo_h, halo_w);
}

}  // namespace tf
