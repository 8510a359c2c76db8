// The C ABI of libtf_epilogue.so: argument validation, kernel selection and
// launch.  Every check runs on the host before anything is launched; an
// unsupported case is an error, never a silent fallback.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "tf_internal.h"

// Device error word, one per device that loads the library.  Kernels receive
// its device address (from cudaGetSymbolAddress) as a parameter.
static __device__ uint32_t g_tf_device_error;

namespace tf {

std::atomic<unsigned long long> g_launch_count{0};

static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];

int current_device()
{
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
    return d;
}
}  // namespace

uint32_t *device_error_word()
{
    const int d = current_device();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_ptr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tf_device_error) != cudaSuccess) return nullptr;
        g_err_ptr[d] = static_cast<uint32_t *>(p);
    }
    return g_err_ptr[d];
}

int sm_count()
{
    const int d = current_device();
    if (d < 0) return 148;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sms[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 148;
        g_sms[d] = n;
    }
    return g_sms[d];
}

}  // namespace tf

using namespace tf;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return TF_OK;
    if (e == cudaErrorNotSupported) {
        cudaGetLastError();
        return TF_ERR_UNSUPPORTED;
    }
    return TF_ERR_CUDA;
}

// Shape checks shared by every conv entry point.  Returns TF_OK and the
// output extent, or the error to report.
int check_conv_shape(const tf_conv_shape *s, int *Ho, int *Wo)
{
    if (!s) return TF_ERR_INVALID_ARG;
    if (s->N <= 0 || s->H <= 0 || s->W <= 0 || s->C_in <= 0 || s->C_out <= 0 || s->KH <= 0 || s->KW <= 0 ||
        s->stride_h <= 0 || s->stride_w <= 0 || s->pad_h < 0 || s->pad_w < 0)
        return TF_ERR_INVALID_ARG;
    const int64_t hn = (int64_t)s->H + 2 * (int64_t)s->pad_h - s->KH;
    const int64_t wn = (int64_t)s->W + 2 * (int64_t)s->pad_w - s->KW;
    if (hn < 0 || wn < 0) return TF_ERR_INVALID_ARG;  // empty output
    *Ho = (int)(hn / s->stride_h + 1);
    *Wo = (int)(wn / s->stride_w + 1);
    if (s->C_in % 8 != 0) return TF_ERR_UNSUPPORTED;
    if ((int64_t)s->N * *Ho * *Wo * s->C_out >= ((int64_t)1 << 40)) return TF_ERR_UNSUPPORTED;
    return TF_OK;
}

// Kernel choice by shape ("Fusing an Epilogue", "Three kernels for one
// operation").  Thresholds measured on GB300 by
// gemm_conv_epilogues_gb300/dispatch_sweep.py (GPU time of CUDA-graph
// replays over 200 shapes):
//  - the tensor-core kernel wins wherever it can run, except on tiny 1x1
//    reductions (K = C_in*KH*KW <= 64 under 6 MFLOP, or under 12 MFLOP when
//    C_in is not a multiple of 64), where its fixed cost (~3.2 us for one
//    persistent wave) ties or loses to the direct kernel, and for C_in < 16:
//    there each 64-channel K step carries 8 real channels, fetched in 16-byte
//    pieces, so it only pays from 15 MFLOP and 48 output channels (16 for a
//    plain 1x1, whose single K step per tile costs little);
//  - im2col shapes with 256-channel tiles, long reductions (>= 32 K steps of
//    64) and at least a wave of 512-pixel pair tiles run wide tiles on CTA
//    pairs with the paired MMA (tcgen05 cta_group::2: each CTA holds half of
//    every filter tile and the two SMs' tensor cores read both halves);
//  - im2col shapes over at least two waves of 128-pixel tiles run the paired
//    MMA on 128-pixel tiles per CTA when a single CTA would split the
//    channels further (C_out % 256 == 0 with a short K loop, where it drops
//    to 128-channel tiles) or when C_in is not a multiple of 64 (each CTA
//    then fetches half the zero-padded filter tiles), from 64 channels;
//  - among the CUDA-core kernels the tiled one wins from 16384 output pixels
//    up, or with few input channels (<= 16) once there are at least ~2M
//    output-channel-taps (M * C_out * KH * KW) to share each staged halo.
int select_variant(const tf_conv_shape &s, int Ho, int Wo)
{
    const int64_t M = (int64_t)s.N * Ho * Wo;
    const int64_t K = (int64_t)s.KH * s.KW * s.C_in;
    const double flops = 2.0 * (double)M * s.C_out * (double)K;
    const bool cin_tail = s.C_in % 64 != 0;
    const bool plain = s.KH == 1 && s.KW == 1 && s.stride_h == 1 && s.stride_w == 1 && s.pad_h == 0 &&
                       s.pad_w == 0;
    // small layers of several taps over few input channels: the direct
    // kernel's batched loads (one memory round trip per thread) beat the
    // tensor-core kernel's fill up to ~32K outputs
    if (s.KH * s.KW > 1 && s.C_in < 64 && M * s.C_out <= 32768) return TF_CONV_DIRECT;
    bool tc = conv_umma_supports(s, Ho, Wo);
    if (s.C_in < 16)
        tc = tc && flops >= 15.0e6 && s.C_out >= (plain ? 16 : 48);
    else if (K <= 64)
        tc = tc && flops >= (cin_tail ? 12.0e6 : 6.0e6);
    if (tc) {
        const int64_t sms = sm_count();
        const int64_t num_kb = (int64_t)s.KH * s.KW * ((s.C_in + 63) / 64);
        const int64_t wide_tiles = (M + 511) / 512 * (s.C_out / 256);
        if (!plain && s.C_out % 256 == 0 && num_kb >= 32 && wide_tiles >= sms / 2) return TF_CONV_UMMA_PAIR_WIDE;
        const bool pair_pays = cin_tail ? s.C_out >= 64 : (s.C_out % 256 == 0 && num_kb <= 16);
        if (!plain && s.C_out % 32 == 0 && M >= 2 * 128 * sms && pair_pays) return TF_CONV_UMMA_PAIR;
        return TF_CONV_UMMA;
    }
    const double taps = (double)M * s.C_out * s.KH * s.KW;
    if (M >= 16384 || (s.C_in <= 16 && taps >= 2.0e6)) return TF_CONV_TILED;
    return TF_CONV_DIRECT;
}

int run_conv(const void *x, const void *w, const float *scale, const float *bias, void *y,
             const tf_conv_shape *shape, int variant, int epilogue, cudaStream_t st)
{
    int Ho = 0, Wo = 0;
    if (!x || !w || !y || !shape || (epilogue && (!scale || !bias))) return TF_ERR_INVALID_ARG;
    int rc = check_conv_shape(shape, &Ho, &Wo);
    if (rc != TF_OK) return rc;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return TF_ERR_UNSUPPORTED;
    if (variant == TF_CONV_AUTO) variant = select_variant(*shape, Ho, Wo);
    ConvArgs a{x, w, scale, bias, y, *shape, Ho, Wo, epilogue};
    switch (variant) {
    case TF_CONV_DIRECT: return from_cuda(launch_conv_direct(a, st));
    case TF_CONV_TILED: return from_cuda(launch_conv_tiled(a, st));
    case TF_CONV_UMMA:
    case TF_CONV_UMMA_PAIR:
    case TF_CONV_UMMA_PAIR_WIDE:
    case TF_CONV_UMMA_WIDE:
        if (!conv_umma_supports(*shape, Ho, Wo)) return TF_ERR_UNSUPPORTED;
        a.wide = variant == TF_CONV_UMMA_PAIR_WIDE || variant == TF_CONV_UMMA_WIDE;
        if (a.wide && shape->C_out % 256 != 0) return TF_ERR_UNSUPPORTED;
        if (epilogue && (!aligned16(scale) || !aligned16(bias))) return TF_ERR_UNSUPPORTED;
        a.cluster = variant == TF_CONV_UMMA_PAIR || variant == TF_CONV_UMMA_PAIR_WIDE ? 2 : 1;
        return from_cuda(launch_conv_umma(a, st));
    default: return TF_ERR_INVALID_ARG;
    }
}

bool bad_rows_cols(int64_t rows, int64_t cols) { return rows <= 0 || cols <= 0; }

// Split-K bytes for a shape the dispatch sends to the tensor-core kernel
// (0 when it would not split).
int64_t splitk_bytes(const tf_conv_shape &s, int Ho, int Wo, int *splits)
{
    *splits = 1;
    // only the single-CTA tensor-core kernel splits K; the dispatch picks CTA
    // pairs only for shapes with at least two waves of tiles, which never split
    if (select_variant(s, Ho, Wo) != TF_CONV_UMMA) return 0;
    const int S = conv_umma_splits(s, Ho, Wo);
    if (S <= 1) return 0;
    *splits = S;
    return (int64_t)S * s.N * Ho * Wo * s.C_out * 4;
}

int run_conv_ws(const void *x, const void *w, const float *scale, const float *bias, void *y,
                const tf_conv_shape *shape, void *ws, int64_t ws_bytes, cudaStream_t st)
{
    int Ho = 0, Wo = 0;
    if (!x || !w || !y || !shape || !scale || !bias || ws_bytes < 0 || (ws_bytes > 0 && !ws))
        return TF_ERR_INVALID_ARG;
    int rc = check_conv_shape(shape, &Ho, &Wo);
    if (rc != TF_OK) return rc;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (ws && !aligned16(ws))) return TF_ERR_UNSUPPORTED;
    int splits = 1;
    const int64_t need = splitk_bytes(*shape, Ho, Wo, &splits);
    if (need == 0 || need > ws_bytes) return run_conv(x, w, scale, bias, y, shape, TF_CONV_AUTO, 1, st);
    if (!aligned16(scale) || !aligned16(bias)) return TF_ERR_UNSUPPORTED;
    ConvArgs a{x, w, scale, bias, y, *shape, Ho, Wo, 1};
    a.splits = splits;
    a.ws = static_cast<float *>(ws);
    rc = from_cuda(launch_conv_umma(a, st));
    if (rc != TF_OK) return rc;
    const int64_t M = (int64_t)shape->N * Ho * Wo;
    return from_cuda(launch_splitk_reduce(a.ws, splits, M, shape->C_out, scale, bias, y, 1, st));
}

}  // namespace

extern "C" {

const char *tf_status_string(int status)
{
    switch (status) {
    case TF_OK: return "TF_OK";
    case TF_ERR_INVALID_ARG: return "TF_ERR_INVALID_ARG: null pointer, non-positive size or empty output";
    case TF_ERR_UNSUPPORTED: return "TF_ERR_UNSUPPORTED: layout, alignment or shape without a kernel";
    case TF_ERR_CUDA: return "TF_ERR_CUDA: the CUDA runtime rejected a call";
    case TF_ERR_TIMEOUT: return "TF_ERR_TIMEOUT: a bounded device-side wait ran out";
    default: return "unknown tf_status";
    }
}

int tf_pack_filter_nhwc(const void *w_oihw, void *w_ohwi, int C_out, int C_in, int KH, int KW, tf_stream_t stream)
{
    if (!w_oihw || !w_ohwi || C_out <= 0 || C_in <= 0 || KH <= 0 || KW <= 0) return TF_ERR_INVALID_ARG;
    return from_cuda(launch_pack_filter(w_oihw, w_ohwi, C_out, C_in, KH, KW, (cudaStream_t)stream));
}

int tf_conv2d_bn_silu(const void *x, const void *w_ohwi, const float *scale, const float *bias, void *y,
                      const tf_conv_shape *shape, tf_stream_t stream)
{
    return run_conv(x, w_ohwi, scale, bias, y, shape, TF_CONV_AUTO, 1, (cudaStream_t)stream);
}

int tf_conv2d_bn_silu_variant(const void *x, const void *w_ohwi, const float *scale, const float *bias, void *y,
                              const tf_conv_shape *shape, int variant, tf_stream_t stream)
{
    if (variant < TF_CONV_AUTO || variant > TF_CONV_UMMA_WIDE) return TF_ERR_INVALID_ARG;
    return run_conv(x, w_ohwi, scale, bias, y, shape, variant, 1, (cudaStream_t)stream);
}

int64_t tf_conv2d_bn_silu_workspace_size(const tf_conv_shape *shape)
{
    int Ho = 0, Wo = 0;
    if (check_conv_shape(shape, &Ho, &Wo) != TF_OK) return 0;
    int splits = 1;
    return splitk_bytes(*shape, Ho, Wo, &splits);
}

int tf_conv2d_bn_silu_ws(const void *x, const void *w_ohwi, const float *scale, const float *bias, void *y,
                         const tf_conv_shape *shape, void *workspace, int64_t workspace_bytes, tf_stream_t stream)
{
    return run_conv_ws(x, w_ohwi, scale, bias, y, shape, workspace, workspace_bytes, (cudaStream_t)stream);
}

int tf_conv2d_bn_silu_select(const tf_conv_shape *shape)
{
    int Ho = 0, Wo = 0;
    const int rc = check_conv_shape(shape, &Ho, &Wo);
    if (rc != TF_OK) return -rc;
    return select_variant(*shape, Ho, Wo);
}

int tf_bias_gelu(const void *x, const void *bias, void *y, int64_t rows, int64_t cols, tf_stream_t stream)
{
    if (!x || !bias || !y || bad_rows_cols(rows, cols)) return TF_ERR_INVALID_ARG;
    if (cols % 8 != 0 || !aligned16(x) || !aligned16(bias) || !aligned16(y)) return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_bias_gelu(x, bias, y, rows, cols, (cudaStream_t)stream));
}

int tf_bias_gelu_rowsum(const void *x, const void *bias, void *y, float *rowsum, int64_t rows, int64_t cols,
                        tf_stream_t stream)
{
    if (!x || !bias || !y || !rowsum || bad_rows_cols(rows, cols)) return TF_ERR_INVALID_ARG;
    if (cols % 8 != 0 || cols > 16384 || !aligned16(x) || !aligned16(bias) || !aligned16(y))
        return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_bias_gelu_rowsum(x, bias, y, rowsum, rows, cols, (cudaStream_t)stream));
}

int tf_unfused_rowsum(const void *y, float *rowsum, int64_t rows, int64_t cols, tf_stream_t stream)
{
    if (!y || !rowsum || bad_rows_cols(rows, cols)) return TF_ERR_INVALID_ARG;
    if (cols % 8 != 0 || cols > 16384 || !aligned16(y)) return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_rowsum(y, rowsum, rows, cols, (cudaStream_t)stream));
}

int tf_residual_layernorm_variant(const void *act, const void *res, const float *gamma, const float *beta,
                                  void *y, int64_t rows, int64_t hidden, float eps, int variant, tf_stream_t stream)
{
    if (!act || !res || !gamma || !beta || !y || bad_rows_cols(rows, hidden) || !(eps >= 0.0f))
        return TF_ERR_INVALID_ARG;
    if (variant < TF_LN_AUTO || variant > TF_LN_CLUSTER) return TF_ERR_INVALID_ARG;
    if (hidden % 8 != 0 || hidden > kClusterMaxHidden || rows > 0x7fffffff) return TF_ERR_UNSUPPORTED;
    if (!aligned16(act) || !aligned16(res) || !aligned16(gamma) || !aligned16(beta) || !aligned16(y))
        return TF_ERR_UNSUPPORTED;
    return from_cuda(
        launch_residual_layernorm(act, res, gamma, beta, y, rows, hidden, eps, variant, (cudaStream_t)stream));
}

int tf_residual_layernorm(const void *act, const void *res, const float *gamma, const float *beta, void *y,
                          int64_t rows, int64_t hidden, float eps, tf_stream_t stream)
{
    return tf_residual_layernorm_variant(act, res, gamma, beta, y, rows, hidden, eps, TF_LN_AUTO, stream);
}

int tf_residual_layernorm_select(int64_t hidden)
{
    if (hidden <= 0) return -TF_ERR_INVALID_ARG;
    if (hidden % 8 != 0) return -TF_ERR_UNSUPPORTED;
    return layernorm_select(hidden);
}

int tf_unfused_conv2d(const void *x, const void *w_ohwi, void *t1, const tf_conv_shape *shape, int variant,
                      tf_stream_t stream)
{
    if (variant < TF_CONV_AUTO || variant > TF_CONV_UMMA_WIDE) return TF_ERR_INVALID_ARG;
    return run_conv(x, w_ohwi, nullptr, nullptr, t1, shape, variant, 0, (cudaStream_t)stream);
}

int tf_unfused_bn(const void *t1, const float *scale, const float *bias, void *t2, int64_t M, int64_t C,
                  tf_stream_t stream)
{
    if (!t1 || !scale || !bias || !t2 || bad_rows_cols(M, C)) return TF_ERR_INVALID_ARG;
    // scale and bias are read as 16-byte vectors
    if (C % 8 != 0 || !aligned16(t1) || !aligned16(t2) || !aligned16(scale) || !aligned16(bias))
        return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_bn(t1, scale, bias, t2, M, C, (cudaStream_t)stream));
}

int tf_unfused_silu(const void *t2, void *y, int64_t n, tf_stream_t stream)
{
    if (!t2 || !y || n <= 0) return TF_ERR_INVALID_ARG;
    if (n % 8 != 0 || !aligned16(t2) || !aligned16(y)) return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_silu(t2, y, n, (cudaStream_t)stream));
}

int tf_unfused_bias_add(const void *x, const void *bias, void *t, int64_t rows, int64_t cols, tf_stream_t stream)
{
    if (!x || !bias || !t || bad_rows_cols(rows, cols)) return TF_ERR_INVALID_ARG;
    if (cols % 8 != 0 || !aligned16(x) || !aligned16(bias) || !aligned16(t)) return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_bias_add(x, bias, t, rows, cols, (cudaStream_t)stream));
}

int tf_unfused_gelu(const void *t, void *y, int64_t n, tf_stream_t stream)
{
    if (!t || !y || n <= 0) return TF_ERR_INVALID_ARG;
    if (n % 8 != 0 || !aligned16(t) || !aligned16(y)) return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_gelu(t, y, n, (cudaStream_t)stream));
}

int tf_unfused_residual_add(const void *act, const void *res, void *s, int64_t n, tf_stream_t stream)
{
    if (!act || !res || !s || n <= 0) return TF_ERR_INVALID_ARG;
    if (n % 8 != 0 || !aligned16(act) || !aligned16(res) || !aligned16(s)) return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_residual_add(act, res, s, n, (cudaStream_t)stream));
}

int tf_unfused_layernorm(const void *s, void *nrm, int64_t rows, int64_t hidden, float eps, tf_stream_t stream)
{
    if (!s || !nrm || bad_rows_cols(rows, hidden) || !(eps >= 0.0f)) return TF_ERR_INVALID_ARG;
    if (hidden % 8 != 0 || hidden > kClusterMaxHidden || rows > 0x7fffffff || !aligned16(s) || !aligned16(nrm))
        return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_layernorm(s, nrm, rows, hidden, eps, (cudaStream_t)stream));
}

int tf_unfused_affine(const void *nrm, const float *gamma, const float *beta, void *y, int64_t rows, int64_t hidden,
                      tf_stream_t stream)
{
    if (!nrm || !gamma || !beta || !y || bad_rows_cols(rows, hidden)) return TF_ERR_INVALID_ARG;
    // gamma and beta are read as 16-byte vectors
    if (hidden % 8 != 0 || !aligned16(nrm) || !aligned16(y) || !aligned16(gamma) || !aligned16(beta))
        return TF_ERR_UNSUPPORTED;
    return from_cuda(launch_unfused_affine(nrm, gamma, beta, y, rows, hidden, (cudaStream_t)stream));
}

void tf_set_wait_limit_ns(uint64_t limit_ns) { g_wait_limit_ns.store(limit_ns, std::memory_order_relaxed); }

uint64_t tf_get_wait_limit_ns(void) { return wait_limit_ns(); }

uint64_t tf_launch_count(void) { return tf::g_launch_count.load(std::memory_order_relaxed); }

int tf_read_device_error(uint32_t *word)
{
    if (cudaDeviceSynchronize() != cudaSuccess) return TF_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tf_device_error, sizeof v) != cudaSuccess) return TF_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_tf_device_error, &zero, sizeof zero) != cudaSuccess) return TF_ERR_CUDA;
    if (word) *word = v;
    return v ? TF_ERR_TIMEOUT : TF_OK;
}

int tf_wait_probe(uint64_t limit_ns, tf_stream_t stream)
{
    return from_cuda(launch_wait_probe(limit_ns, (cudaStream_t)stream));
}

}  // extern "C"
