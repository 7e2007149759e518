// api_static_workspace.cu -- mha_forward_static_workspace(): the multi-head
// attention forward with its scratch memory inside the library, for callers
// that cannot allocate device memory themselves.
//
// The scratch is one file-scope device array of MHA_STATIC_WORKSPACE_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code may not pass the array's name to a kernel (on the host it is only a
// stand-in symbol), so on the first call on each device this file asks the
// runtime for the array's device address with cudaGetSymbolAddress, with
// that device current, and caches it; the kernels are then given that
// address exactly as mha_forward is given a caller's workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mha.h"

#define MHA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[MHA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_device_address[kMaxDevices] = {};

// Device address of g_static_workspace on the current device, or null.
void *static_workspace_address() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_device_address[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
        g_device_address[dev] = p;
    }
    return g_device_address[dev];
}

}  // namespace

MHA_EXPORT mha_status mha_forward_static_workspace(
    mha_dtype dt, const void *x_q, const void *x_kv, const void *w_q, const void *w_k,
    const void *w_v, const void *w_o, void *out, int B, int h, int T_q, int T_k, int d_model,
    int d_k, int d_v, float scale, mha_mask mask, const int32_t *key_lens, int *status_dev,
    cudaStream_t stream) {
    const size_t need = mha_workspace_bytes(B, h, T_q, T_k, d_k, d_v);
    if (need > static_cast<size_t>(MHA_STATIC_WORKSPACE_BYTES)) return MHA_ERR_WORKSPACE;
    void *ws = static_workspace_address();
    if (!ws) return MHA_ERR_CUDA;
    // Every workspace byte the kernels read is written earlier in the same
    // call (projections, then attention output), so nothing is cleared.
    return mha_forward(dt, x_q, x_kv, w_q, w_k, w_v, w_o, out, ws,
                       static_cast<size_t>(MHA_STATIC_WORKSPACE_BYTES), B, h, T_q, T_k, d_model,
                       d_k, d_v, scale, mask, key_lens, status_dev, stream);
}
