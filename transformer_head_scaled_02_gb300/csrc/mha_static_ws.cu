// mha_static_ws.cu -- mha_forward_static_workspace: the forward pass for callers that are not
// allowed to allocate device memory.  Its scratch (status word, projected Q/K/V, Ocat) lives
// in one file-scope __device__ array of MHA_STATIC_WORKSPACE_BYTES instead of a caller-owned
// workspace.  The array is part of this library's device image, so every GPU that loads the
// library holds it until the process exits.
#include <stddef.h>
#include <stdint.h>

#include "../../include/mha.h"
#include "internal.h"

namespace {

// The scratch itself.  In host code the name is only a host-side stand-in; the device
// address comes from cudaGetSymbolAddress below and is what the kernels receive.
static __device__ __align__(256) unsigned char g_static_ws[MHA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
static void* g_static_ws_addr[kMaxDevices];  // per device, filled on first use

}  // namespace

extern "C" mha_status mha_forward_static_workspace(mha_t handle, const void* X_q,
                                                   const void* X_kv, int B, int T_q, int T_kv,
                                                   const void* W_qkv, const void* b_qkv,
                                                   const void* W_o, const void* b_o, int causal,
                                                   const int32_t* kv_lengths, void* out,
                                                   void* stream) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    const size_t need = mha_workspace_size(handle, B, T_q, T_kv);
    if (need == 0) return MHA_ERR_INVALID_ARG;
    if (need > (size_t)MHA_STATIC_WORKSPACE_BYTES) return MHA_ERR_WORKSPACE;
    if (B == 0 || T_q == 0) return MHA_OK;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MHA_ERR_CUDA;
    if (g_static_ws_addr[dev] == nullptr) {
        // once per device, with that device current
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr)
            return MHA_ERR_CUDA;
        g_static_ws_addr[dev] = p;
    }
    void* ws = g_static_ws_addr[dev];
    // The array keeps the previous call's contents; the status word must start at zero.
    if (cudaMemsetAsync(ws, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MHA_ERR_CUDA;
    mha_s local = *handle;  // the caller's handle (and its own workspace) stay untouched
    local.ws = ws;
    local.ws_bytes = (size_t)MHA_STATIC_WORKSPACE_BYTES;
    return mha_forward(&local, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal,
                       kv_lengths, out, stream);
}
