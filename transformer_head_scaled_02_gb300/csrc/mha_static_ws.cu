// mha_static_ws.cu -- mha_forward_static_workspace: the forward pass for callers that are not
// allowed to allocate device memory.  Its scratch (status word, projected Q/K/V, Ocat) lives
// in one file-scope __device__ array of MHA_STATIC_WORKSPACE_BYTES instead of a caller-owned
// workspace.  The array is part of this library's device image, so every GPU that loads the
// library holds it until the process exits.
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/mha.h"
#include "internal.h"

namespace {

// The scratch itself.  In host code the name is only a host-side stand-in; the device
// address comes from cudaGetSymbolAddress below and is what the kernels receive.
static __device__ __align__(256) unsigned char g_static_ws[MHA_STATIC_WORKSPACE_BYTES];

// The array's device address, looked up once per device and CUDA context.  A context that is
// destroyed and created again (cudaDeviceReset, or the primary context released and retained
// again) loads the library's device image anew, possibly at another address, so the cached
// address is valid only for the context it was looked up in: each entry carries that
// context's process-unique id (cuCtxGetId), and a call from any other context looks the
// address up again.  g_mu serialises the lookups of concurrent first calls.
struct StaticAddr {
    unsigned long long ctx_id;
    void* addr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
StaticAddr g_addr[kMaxDevices];  // guarded by g_mu

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
int g_ctx_fns = 0;  // 0 not looked up, 1 available, -1 unavailable (guarded by g_mu)

bool context_fns() {
    if (g_ctx_fns == 0) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        const bool ok =
            cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1) ==
                cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess && f1 != nullptr &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
                cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess && f2 != nullptr;
        if (ok) {
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
        }
        g_ctx_fns = ok ? 1 : -1;
    }
    return g_ctx_fns == 1;
}

// Id of the calling thread's current context; false if none is current yet.
bool current_context_id(unsigned long long* id) {
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_ws in the current device's current context.
mha_status static_ws_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!context_fns()) return MHA_ERR_CUDA;
    unsigned long long id = 0;
    if (current_context_id(&id) && g_addr[dev].addr != nullptr && g_addr[dev].ctx_id == id) {
        *out = g_addr[dev].addr;
        return MHA_OK;
    }
    // set-up for this device and context, with the device current: the lookup also makes
    // the runtime's context current if no CUDA call has done so yet
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return MHA_ERR_CUDA;
    if (!current_context_id(&id)) return MHA_ERR_CUDA;
    g_addr[dev].ctx_id = id;
    g_addr[dev].addr = p;
    *out = p;
    return MHA_OK;
}

}  // namespace

extern "C" mha_status mha_forward_static_workspace(mha_t handle, const void* X_q,
                                                   const void* X_kv, int B, int T_q, int T_kv,
                                                   const void* W_qkv, const void* b_qkv,
                                                   const void* W_o, const void* b_o, int causal,
                                                   const int32_t* kv_lengths, void* out,
                                                   int32_t* status_out, void* stream) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    const size_t need = mha_workspace_size(handle, B, T_q, T_kv);
    if (need == 0) return MHA_ERR_INVALID_ARG;
    if (need > (size_t)MHA_STATIC_WORKSPACE_BYTES) return MHA_ERR_WORKSPACE;
    // every other argument check first: a call that is refused touches neither the array
    // (whose status word another call in flight may be using) nor *status_out
    mha_status st = mha::check_forward(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o,
                                       causal, nullptr, out);
    if (st != MHA_OK) return st;
    if (status_out != nullptr && (reinterpret_cast<uintptr_t>(status_out) & 3u) != 0)
        return MHA_ERR_INVALID_ARG;
    if (B == 0 || T_q == 0) return MHA_OK;

    void* ws = nullptr;
    st = static_ws_address(&ws);
    if (st != MHA_OK) return st;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents; the status word must start at zero.
    if (cudaMemsetAsync(ws, 0, 256, cs) != cudaSuccess) return MHA_ERR_CUDA;
    mha_s local = *handle;  // the caller's handle (and its own workspace) stay untouched
    local.ws = ws;
    local.ws_bytes = (size_t)MHA_STATIC_WORKSPACE_BYTES;
    st = mha_forward(&local, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal, kv_lengths,
                     out, stream);
    if (st != MHA_OK) return st;
    // the device status of this call, for a caller that asked for it
    if (status_out != nullptr &&
        cudaMemcpyAsync(status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, cs) != cudaSuccess)
        return MHA_ERR_CUDA;
    return MHA_OK;
}
