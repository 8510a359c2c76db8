// tf_conv2d_bn_silu_static_ws: the split-K conv + BN + SiLU of
// tf_conv2d_bn_silu_ws for callers that cannot hand the library a workspace.
//
// Some callers cannot call cudaMalloc on the path that runs the layer: a
// serving runtime or plugin host that plans every device buffer ahead of
// time and owns the whole memory pool, or code for which an allocation
// would be a device-wide synchronisation point or could fail under memory
// fragmentation in the middle of a request.  This entry point needs no
// buffer from them: the split-K partial sums live in one file-scope device
// array, kStaticWorkspaceBytes (8 MiB) long, that every GPU which loads the
// library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "tf_internal.h"

namespace {

constexpr int64_t kStaticWorkspaceBytes = 8ll << 20;

// The shared split-K workspace.  In host code this name is only a host-side
// stand-in for the symbol, never a device address: the device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_ws_mu;
void *g_ws_ptr[kMaxDevices];

// Device address of the static workspace on the current device, looked up
// once per device (with that device current) and cached; nullptr on failure.
void *static_workspace()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_ws_mu);
    if (!g_ws_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) {
            cudaGetLastError();   // reported as TF_ERR_CUDA; not left pending for a later call
            return nullptr;
        }
        g_ws_ptr[dev] = p;
    }
    return g_ws_ptr[dev];
}

}  // namespace

extern "C" int tf_conv2d_bn_silu_static_ws(const void *x, const void *w_ohwi, const float *scale,
                                           const float *bias, void *y, const tf_conv_shape *shape,
                                           tf_stream_t stream)
{
    if (!shape) return TF_ERR_INVALID_ARG;
    const int64_t need = tf_conv2d_bn_silu_workspace_size(shape);
    if (need > kStaticWorkspaceBytes) return TF_ERR_UNSUPPORTED;   // partials would not fit in 8 MiB
    if (need == 0) return tf_conv2d_bn_silu_ws(x, w_ohwi, scale, bias, y, shape, nullptr, 0, stream);
    void *ws = static_workspace();
    if (!ws) return TF_ERR_CUDA;
    // Every split writes all of its partial sums before the reduction reads
    // them, so the array's contents from an earlier call never leak in and
    // nothing has to be cleared.
    return tf_conv2d_bn_silu_ws(x, w_ohwi, scale, bias, y, shape, ws, kStaticWorkspaceBytes, stream);
}
