/*
 * tf_epilogue.h -- C ABI of the GB300 (sm_103a) epilogue-fusion library
 * (libtf_epilogue.so).
 *
 * Epilogue fusion: a producer's output tile gets its cheap per-element work
 * (per-channel BatchNorm scale/bias and SiLU, bias + GELU, residual +
 * LayerNorm + affine) while it is still on chip, and is written to HBM once.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library
 *    allocates no device memory in any call.  Outputs must not alias inputs.
 *  - Every call is asynchronous on the given stream (a cudaStream_t; NULL is
 *    the legacy default stream) and never synchronises the device.
 *  - Arguments are validated on the host before anything is launched:
 *      TF_ERR_INVALID_ARG  a required pointer is NULL or a size is <= 0
 *                          (or the shape has an empty output);
 *      TF_ERR_UNSUPPORTED  a layout or alignment the library has no kernel
 *                          for (e.g. a pointer not 16-byte aligned, a row
 *                          length not a multiple of 8);
 *      TF_ERR_CUDA         the CUDA runtime refused the launch;
 *      TF_ERR_TIMEOUT      a bounded device-side wait ran out (reported by
 *                          tf_read_device_error after the stream completes).
 *    Nothing is launched when a call returns an error before TF_ERR_CUDA.
 *    There is no CPU fallback: an unsupported case is an error.
 *  - No C++ exception crosses this boundary.
 *  - Storage types: bf16 = bfloat16, fp16 = IEEE binary16, both passed as
 *    void pointers; fp32 parameters as float pointers.  Arithmetic is fp32.
 *    Every cast to bf16/fp16 rounds to nearest even.
 */
#ifndef TF_EPILOGUE_H
#define TF_EPILOGUE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared here so that the header needs no CUDA include. */
typedef struct CUstream_st *tf_stream_t;

typedef enum {
    TF_OK = 0,
    TF_ERR_INVALID_ARG = 1,
    TF_ERR_UNSUPPORTED = 2,
    TF_ERR_CUDA = 3,
    TF_ERR_TIMEOUT = 4
} tf_status;

/* Convolution geometry.  Input x is NHWC [N][H][W][C_in]; output y is NHWC
 * [N][Ho][Wo][C_out] with Ho = (H + 2*pad_h - KH)/stride_h + 1 and
 * Wo = (W + 2*pad_w - KW)/stride_w + 1 (floor division); taps outside the
 * input read zero. */
typedef struct {
    int N, H, W, C_in, C_out, KH, KW;
    int stride_h, stride_w, pad_h, pad_w;
} tf_conv_shape;

/* Convolution kernels (see tf_conv2d_bn_silu_variant). */
typedef enum {
    TF_CONV_AUTO = -1,   /* dispatch by shape */
    TF_CONV_DIRECT = 0,  /* one output element per thread, CUDA-core fp32 */
    TF_CONV_TILED = 1,   /* output-space tiles with a shared-memory halo, CUDA cores */
    TF_CONV_UMMA = 2,    /* implicit GEMM: TMA im2col -> tcgen05.mma -> TMEM -> fused epilogue */
    TF_CONV_UMMA_PAIR = 3, /* the same on CTA pairs (2-CTA clusters) with the paired MMA
                              (tcgen05 .cta_group::2, M = 256): each CTA loads its own 128 output
                              pixels and HALF of every filter tile, and the two SMs' tensor cores
                              read both halves; the dispatch's choice for im2col shapes over at
                              least two waves of pair tiles with C_out % 256 == 0 and at most 16
                              K steps, or with C_in not a multiple of 64 and C_out >= 64 */
    TF_CONV_UMMA_PAIR_WIDE = 4, /* paired MMA with 256-pixel tiles per CTA: two M = 256 MMAs per K
                                  step read each half filter tile (C_out % 256 == 0 only); the
                                  dispatch's choice for im2col shapes (not plain 1x1 GEMMs) with
                                  C_out % 256 == 0, at least 32 K steps and at least a wave of
                                  512-pixel pair tiles (one per CTA pair) */
    TF_CONV_UMMA_WIDE = 5  /* 256-pixel tiles on single CTAs (C_out % 256 == 0 only) */
} tf_conv_variant;

/* Row-reduction strategies of the LayerNorm kernels (see
 * tf_residual_layernorm_variant). */
typedef enum {
    TF_LN_AUTO = -1,    /* by hidden width */
    TF_LN_WARP = 0,     /* one warp per row, shuffle reductions (hidden <= 1024) */
    TF_LN_CTA = 1,      /* one CTA per row, rows streamed through a bulk-copy ring (hidden <= 16384) */
    TF_LN_CLUSTER = 2   /* a thread-block cluster per row (slices of <= 8192 columns: up to 8
                           CTAs to 65536 columns, 16 beyond), each CTA's (sum, M2) pushed into
                           its peers' shared memory once per row (16384 < hidden <= 131072) */
} tf_ln_variant;

/* Human-readable name of a status code (static storage). */
const char *tf_status_string(int status);

/* ---------------------------------------------------------------- filters */

/* Pack convolution filters channels-last, once, at load time.
 * "When the fusion you want is impossible, fuse into the producer"
 * (skandtandon.pages.dev), closing paragraphs: the filters were stored in the
 * wrong layout, so conversions wrapped every convolution; storing them
 * channels-last once at load time removed them with bit-identical output.
 *   w_oihw : bf16 [C_out][C_in][KH][KW]   (read)
 *   w_ohwi : bf16 [C_out][KH][KW][C_in]   (written; a pure permutation)
 * Both device pointers, no alignment requirement.  Sizes must be > 0. */
int tf_pack_filter_nhwc(const void *w_oihw, void *w_ohwi,
                        int C_out, int C_in, int KH, int KW, tf_stream_t stream);

/* ---------------------------------------------------------------- conv */

/* Fused conv2d + per-channel BatchNorm (scale, bias) + SiLU.
 * "Fusing an Epilogue" (docs.teenygrad.org), "The shape of it" and the
 * BatchNorm-epilog listing: after the K loop the accumulator tile gets
 * acc*bn_scale + bn_bias and then acc*sigmoid(acc) before the single store;
 * the per-channel parameters are loaded inside the same kernel, masked at
 * the C_out edge.
 *   x      : bf16 NHWC [N][H][W][C_in]
 *   w_ohwi : bf16 [C_out][KH][KW][C_in] (from tf_pack_filter_nhwc)
 *   scale, bias : fp32 [C_out] (BatchNorm already folded into a scale and a
 *            bias per output channel; no running statistics, no eps here)
 *   y      : bf16 NHWC [N][Ho][Wo][C_out]
 * y[n][oh][ow][co] = SiLU(acc*scale[co] + bias[co]) with
 * acc = sum_{kh,kw,ci} x[n][oh*sh-ph+kh][ow*sw-pw+kw][ci] * w[co][kh][kw][ci]
 * accumulated in fp32.  Requires C_in % 8 == 0 and 16-byte aligned x, w, y;
 * shapes that go to a tensor-core kernel also need 16-byte aligned scale and
 * bias (TF_ERR_UNSUPPORTED otherwise).  The kernel is chosen by shape (see
 * tf_conv2d_bn_silu_select); the wide-tile kernels may be followed by a
 * second launch on the same stream that computes the rows of their last,
 * partial wave on 128-row tiles (tf_launch_count counts both). */
int tf_conv2d_bn_silu(const void *x, const void *w_ohwi, const float *scale, const float *bias,
                      void *y, const tf_conv_shape *shape, tf_stream_t stream);

/* Same as tf_conv2d_bn_silu with the kernel forced (TF_CONV_*).  Returns
 * TF_ERR_UNSUPPORTED when the forced kernel cannot take the shape (the
 * tensor-core kernels: strides <= 8 and padding <= 128 for im2col shapes;
 * TF_CONV_UMMA takes any C_in % 8 == 0 and any C_out, TF_CONV_UMMA_PAIR needs
 * C_out % 32 == 0, TF_CONV_UMMA_PAIR_WIDE and TF_CONV_UMMA_WIDE
 * C_out % 256 == 0). */
int tf_conv2d_bn_silu_variant(const void *x, const void *w_ohwi, const float *scale,
                              const float *bias, void *y, const tf_conv_shape *shape,
                              int variant, tf_stream_t stream);

/* Bytes of device workspace tf_conv2d_bn_silu_ws can use for this shape: the
 * fp32 partial sums of a K split, splits * N*Ho*Wo * C_out * 4 bytes, or 0
 * when the shape fills the GPU without splitting (or is invalid).  Host only. */
int64_t tf_conv2d_bn_silu_workspace_size(const tf_conv_shape *shape);

/* Same result as tf_conv2d_bn_silu, with a caller-owned device workspace.
 * When the tensor-core kernel would leave SMs idle (fewer 128 x BN output
 * tiles than half the SMs) it splits the K loop (filter taps x input
 * channels) across CTAs -- the tile size and split chosen from the layer
 * shape and the SM count ("Fusing an Epilogue", "Three kernels for one
 * operation") -- writes fp32 partial sums to `workspace`, and a second kernel
 * adds them and applies the BatchNorm + SiLU epilogue.  With a workspace
 * smaller than tf_conv2d_bn_silu_workspace_size (including 0) it runs
 * tf_conv2d_bn_silu unchanged.  The workspace must be 16-byte aligned, must
 * not alias x, w, y, and is in use until the stream reaches the end of the
 * call; concurrent calls need separate workspaces. */
int tf_conv2d_bn_silu_ws(const void *x, const void *w_ohwi, const float *scale, const float *bias,
                         void *y, const tf_conv_shape *shape, void *workspace,
                         int64_t workspace_bytes, tf_stream_t stream);

/* tf_conv2d_bn_silu_ws for callers that cannot allocate device memory (no
 * counterpart in the pages: it exists for callers such as a serving runtime
 * or plugin host that plans and owns every device buffer, or code that must
 * not call cudaMalloc on the request path because it can synchronise the
 * device or fail when memory is fragmented).  Same arguments and result as
 * tf_conv2d_bn_silu, no workspace argument: the split-K partial sums go to
 * one library-owned device array of 8 MiB (8388608 bytes), a static
 * __device__ allocation that every GPU loading the library keeps until the
 * process exits.  The call allocates nothing.
 *   - Returns TF_ERR_UNSUPPORTED, launching nothing, when the shape's
 *     partial sums (tf_conv2d_bn_silu_workspace_size) exceed 8 MiB; shapes
 *     that do not split run unsplit, as tf_conv2d_bn_silu.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents
 *     (every split rewrites all its partials before they are read, so
 *     nothing needs clearing).  Calls whose GPU work overlaps -- on
 *     different streams or from different host threads without ordering --
 *     race on it; issue them on one stream. */
int tf_conv2d_bn_silu_static_ws(const void *x, const void *w_ohwi, const float *scale,
                                const float *bias, void *y, const tf_conv_shape *shape,
                                tf_stream_t stream);

/* The kernel tf_conv2d_bn_silu would run for this shape (host only, launches
 * nothing), or a negative tf_status value when the shape is rejected.
 * "Fusing an Epilogue", "Three kernels for one operation": the lowering picks
 * one of three kernels by shape with hand-chosen thresholds; this library's
 * thresholds are measured on GB300. */
int tf_conv2d_bn_silu_select(const tf_conv_shape *shape);

/* ---------------------------------------------------------------- bias + GELU */

/* y[i][j] = GELU(x[i][j] + bias[j]), GELU with the erf definition
 * s * Phi(s).  "Costs and benefits of kernel fusion"
 * (intro-to-ai-systems-performance), opening example: the fused kernel
 * computes the addition and GELU per value and writes y once instead of
 * materialising the fp16 x + bias tensor.
 *   x, y : fp16 [rows][cols] row-major;  bias : fp16 [cols], broadcast over rows.
 * Requires cols % 8 == 0 and 16-byte aligned x, bias, y. */
int tf_bias_gelu(const void *x, const void *bias, void *y, int64_t rows, int64_t cols,
                 tf_stream_t stream);

/* Bias + GELU + per-row sum in one pass.  "Costs and benefits of kernel
 * fusion", "Compare fused and split bias-activation-reduction paths": apply
 * bias, GELU and a per-row reduction without writing the GELU result before
 * the reduction reads it.
 *   x, y : fp16 [rows][cols];  bias : fp16 [cols];  rowsum : fp32 [rows]
 * y[i][j] = GELU(x[i][j] + bias[j]) as in tf_bias_gelu; rowsum[i] = sum over
 * j of the fp32 GELU values (before y is rounded to fp16), accumulated in
 * fp32.  Requires cols % 8 == 0, cols <= 16384, 16-byte aligned x, bias, y. */
int tf_bias_gelu_rowsum(const void *x, const void *bias, void *y, float *rowsum, int64_t rows,
                        int64_t cols, tf_stream_t stream);

/* ---------------------------------------------------------------- residual + LN */

/* y = LayerNorm(act + res) * gamma + beta, one HBM pass.  "Costs and benefits
 * of kernel fusion", "Worked example: Fusing a residual and normalization
 * chain": load activation and residual once, compute the row statistics,
 * normalise, apply scale and bias, write the final output.
 *   act, res, y : fp16 [rows][hidden];  gamma, beta : fp32 [hidden]
 * mean and biased variance of s = act + res per row, computed in fp32 from
 * registers in two passes (sum, then squared deviations; s is never
 * written); y = (s - mean) / sqrt(var + eps) * gamma + beta.  Requires
 * hidden % 8 == 0, hidden <= 131072, 16-byte aligned pointers, eps >= 0.
 * The row-reduction strategy is chosen by hidden width
 * (tf_residual_layernorm_select). */
int tf_residual_layernorm(const void *act, const void *res, const float *gamma, const float *beta,
                          void *y, int64_t rows, int64_t hidden, float eps, tf_stream_t stream);

/* Same with the strategy forced (TF_LN_*); TF_ERR_UNSUPPORTED when the width
 * is outside the strategy's range.  "Costs and benefits of kernel fusion",
 * worked example: test a hidden width large enough to require a different
 * row-reduction strategy, with an explicit dispatch boundary. */
int tf_residual_layernorm_variant(const void *act, const void *res, const float *gamma,
                                  const float *beta, void *y, int64_t rows, int64_t hidden,
                                  float eps, int variant, tf_stream_t stream);

/* The strategy tf_residual_layernorm uses for this width (host only), or a
 * negative tf_status value when no strategy takes it. */
int tf_residual_layernorm_select(int64_t hidden);

/* ---------------------------------------------------------------- unfused chains */

/* The separate kernels that the fused calls replace, for the traffic and time
 * comparison ("Fusing an Epilogue", "The problem": conv writes t1, batchnorm
 * reads t1 and writes t2, silu reads t2 and writes y; "Costs and benefits of
 * kernel fusion": the eager x + bias then GELU pair, and the eager residual
 * add, LayerNorm and scale-and-bias kernels).  Each materialises its result
 * in HBM in the storage type given.  Same validation rules as above. */

/* t1 = conv(x, w) in bf16 (no epilogue), same kernels and shape rules as
 * tf_conv2d_bn_silu_variant. */
int tf_unfused_conv2d(const void *x, const void *w_ohwi, void *t1, const tf_conv_shape *shape,
                      int variant, tf_stream_t stream);
/* t2[m][c] = t1[m][c]*scale[c] + bias[c]; bf16 [M][C], C % 8 == 0, all four
 * pointers 16-byte aligned. */
int tf_unfused_bn(const void *t1, const float *scale, const float *bias, void *t2,
                  int64_t M, int64_t C, tf_stream_t stream);
/* y = t2 * sigmoid(t2); bf16, n % 8 == 0. */
int tf_unfused_silu(const void *t2, void *y, int64_t n, tf_stream_t stream);
/* t[i][j] = x[i][j] + bias[j]; fp16, cols % 8 == 0. */
int tf_unfused_bias_add(const void *x, const void *bias, void *t, int64_t rows, int64_t cols,
                        tf_stream_t stream);
/* rowsum[i] = sum over j of y[i][j] (fp16 in, fp32 sum): the reduction of
 * the split bias-activation-reduction path, run after tf_bias_gelu has
 * written y.  cols % 8 == 0, cols <= 16384. */
int tf_unfused_rowsum(const void *y, float *rowsum, int64_t rows, int64_t cols, tf_stream_t stream);
/* y = GELU(t); fp16, n % 8 == 0. */
int tf_unfused_gelu(const void *t, void *y, int64_t n, tf_stream_t stream);
/* s = act + res; fp16, n % 8 == 0. */
int tf_unfused_residual_add(const void *act, const void *res, void *s, int64_t n,
                            tf_stream_t stream);
/* nrm = (s - mean)/sqrt(var + eps) per row, no affine; fp16 in and out
 * (hidden <= 131072, same strategies as tf_residual_layernorm). */
int tf_unfused_layernorm(const void *s, void *nrm, int64_t rows, int64_t hidden, float eps,
                         tf_stream_t stream);
/* y[i][j] = nrm[i][j]*gamma[j] + beta[j]; fp16 in and out, fp32 gamma/beta;
 * all four pointers 16-byte aligned. */
int tf_unfused_affine(const void *nrm, const float *gamma, const float *beta, void *y,
                      int64_t rows, int64_t hidden, tf_stream_t stream);

/* ---------------------------------------------------------------- device waits */

/* Every spin-wait inside the library's kernels (the mbarrier waits of the
 * tcgen05 pipeline and of the bulk-copy rings, and the cluster LayerNorm's
 * wait for its peers' partial sums) gives up after this many nanoseconds of
 * %globaltimer, records TF_DEVERR_* in a device error word and lets the
 * kernel finish cleanly.  Default 2e9 (2 s).  Host-side setting, applies to
 * later launches. */
void tf_set_wait_limit_ns(uint64_t limit_ns);
uint64_t tf_get_wait_limit_ns(void);

/* Bits of the device error word. */
#define TF_DEVERR_PRODUCER_WAIT 0x1u  /* conv TMA producer: a stage never freed; bulk-copy
                                        rings (bias + GELU, LayerNorm): a stage never filled */
#define TF_DEVERR_MMA_WAIT 0x2u       /* MMA issuer: operands or accumulator never ready */
#define TF_DEVERR_EPILOGUE_WAIT 0x4u  /* epilogue: accumulator never committed */
#define TF_DEVERR_DRAIN_WAIT 0x8u     /* in-flight copies/MMAs not drained on exit */
#define TF_DEVERR_PROBE_WAIT 0x10u    /* tf_wait_probe: the expected time-out */
#define TF_DEVERR_EXCHANGE_WAIT 0x20u /* cluster LayerNorm: a peer CTA's partial sum never arrived */
#define TF_DEVERR_PAIR_TMEM 0x40u     /* paired conv MMA: the two CTAs' TMEM allocations differ
                                         (the pair did no work) */
#define TF_DEVERR_SMEM_ALIGN 0x80u    /* tensor-core conv: dynamic shared memory not 1024-byte
                                         aligned (the CTA did no work) */

/* Synchronises the current device, copies the device error word of the
 * current device into *word (may be NULL), clears it, and returns TF_OK if it
 * was zero, TF_ERR_TIMEOUT if a wait gave up, TF_ERR_CUDA if the runtime
 * failed.  Not for use inside stream capture. */
int tf_read_device_error(uint32_t *word);

/* Number of kernels this library has launched in this process so far (every
 * entry point, every device and stream; launches the runtime accepted).  One
 * call may launch more than one kernel: tf_conv2d_bn_silu runs a wide-tile
 * kernel and then its partial last wave on 128-row tiles, the split-K path
 * adds a reduction.  For benchmarks that report how many kernels ran. */
uint64_t tf_launch_count(void);

/* Launches one small kernel that waits, with the given limit, on an mbarrier
 * that nothing ever arrives on; it gives up, sets TF_DEVERR_PROBE_WAIT and
 * returns.  Exercises the time-out path without disturbing the GPU. */
int tf_wait_probe(uint64_t limit_ns, tf_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TF_EPILOGUE_H */
