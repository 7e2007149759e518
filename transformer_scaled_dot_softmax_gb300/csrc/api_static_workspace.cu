// api_static_workspace.cu -- mha_forward_static_workspace(): the multi-head
// attention forward with its scratch memory inside the library, for callers
// that cannot allocate device memory themselves.
//
// The scratch is one file-scope device array of MHA_STATIC_WORKSPACE_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host
// code may not pass the array's name to a kernel (on the host it is only a
// stand-in symbol), so every call asks the runtime for the array's device
// address with cudaGetSymbolAddress, with the caller's device current, and
// gives the kernels that address exactly as mha_forward is given a caller's
// workspace.  The address is not cached: a context created anew on the same
// device (after cudaDeviceReset, or a different current context) loads the
// library's device code again, and the array may then live elsewhere.  The
// first call in a context is the one that loads the device code (the
// runtime's set-up for the context); later calls only look the address up.
#include <cuda_runtime.h>

#include "../../include/mha.h"
#include "kernels.h"

#define MHA_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[MHA_STATIC_WORKSPACE_BYTES];

}  // namespace

MHA_EXPORT mha_status mha_forward_static_workspace(
    mha_dtype dt, const void *x_q, const void *x_kv, const void *w_q, const void *w_k,
    const void *w_v, const void *w_o, void *out, int B, int h, int T_q, int T_k, int d_model,
    int d_k, int d_v, float scale, mha_mask mask, const int32_t *key_lens, int *status_dev,
    cudaStream_t stream) {
    // mha_forward's own argument checks, run without a workspace: they launch
    // nothing, and return MHA_ERR_WORKSPACE exactly when every check before
    // the workspace one passed and the problem is not empty.  Anything else
    // (an argument error, or MHA_OK for an empty problem) is the answer.
    const mha_status pre =
        mha_forward(dt, x_q, x_kv, w_q, w_k, w_v, w_o, out, nullptr, 0, B, h, T_q, T_k, d_model,
                    d_k, d_v, scale, mask, key_lens, status_dev, stream);
    if (pre != MHA_ERR_WORKSPACE) return pre;
    const size_t need = mha_workspace_bytes(B, h, T_q, T_k, d_k, d_v);
    if (need > static_cast<size_t>(MHA_STATIC_WORKSPACE_BYTES)) return MHA_ERR_WORKSPACE;
    void *ws = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ws, g_static_workspace);
    if (e != cudaSuccess || !ws)
        return mha::record_cuda_failure("static workspace address (cudaGetSymbolAddress)",
                                        e != cudaSuccess ? cudaGetErrorName(e) : "null address");
    // Every workspace byte the kernels read is written earlier in the same
    // call (projections, then attention output), so nothing is cleared.
    return mha_forward(dt, x_q, x_kv, w_q, w_k, w_v, w_o, out, ws,
                       static_cast<size_t>(MHA_STATIC_WORKSPACE_BYTES), B, h, T_q, T_k, d_model,
                       d_k, d_v, scale, mask, key_lens, status_dev, stream);
}
