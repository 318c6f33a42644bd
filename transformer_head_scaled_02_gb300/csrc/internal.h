// internal.h -- host-side declarations shared by the kernel translation units and the
// C-ABI layer.  Not part of the public interface (that is include/mha.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mha.h"

// The opaque handle of include/mha.h: the layer configuration and the caller's workspace.
// h_kv: K/V heads (h for plain multi-head attention, 1 for MQA); gated: the fused projection
// carries a fourth block of h*d_v gate pre-activations.
// aux_*: the two copy streams and the events of mha_forward_host, created with the first
// workspace on the device that was current then (aux_dev; -1: none yet).
constexpr int kHostMaxChunks = 16;
struct mha_s {
    int D, h, h_kv, dk, dv, gated;
    mha_dtype dtype;
    void* ws;
    size_t ws_bytes;
    int aux_dev;
    cudaStream_t aux_h2d, aux_d2h;
    cudaEvent_t aux_start, aux_done, aux_in[kHostMaxChunks], aux_out[kHostMaxChunks];
};

namespace mha {

// Every host-side check of mha_forward_ex except the one on the attached workspace
// (mha_api.cu).  MHA_OK: the call would launch its kernels, or nothing for B == 0 or T_q == 0.
mha_status check_forward(const mha_s* m, const void* X_q, const void* X_kv, int B, int T_q,
                         int T_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                         const void* b_o, int causal, const void* residual, const void* out);

// Launch a kernel that may start while the previous kernel on the stream is finishing
// (programmatic dependent launch): its CTAs run their set-up (barriers, TMEM allocation)
// early and wait in grid_dependency_wait() until the previous grid has completed and its
// memory is visible.  Every kernel launched this way calls grid_dependency_wait() before
// its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Encode a bf16 tiled tensor map with 128-byte swizzle (swizzle_bytes == 0: none) and zero
// fill out of bounds.  dims[0] is the innermost (contiguous) extent; strides_bytes has rank-1
// entries.  Returns false if the driver entry point is unavailable or rejects the map.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes = 128);

// C = A W + bias (+ R), fp32 everywhere.  A (M,K) lda; W (K,N) ldw; R (M,N) ldr or null;
// C (M,N) ldc.
cudaError_t launch_gemm_f32(const float* A, int64_t lda, const float* W, int64_t ldw,
                            const float* bias, const float* R, int64_t ldr, float* C, int64_t ldc,
                            int M, int N, int K, cudaStream_t stream);

// Attention for all heads, fp32.  See mha_attention_ex in include/mha.h for the layout;
// decode != 0 places the T_q rows at the end of each batch's L_b keys (mha_decode).
cudaError_t launch_attn_f32(const float* Q, int64_t ldq, const float* K, int64_t ldk,
                            const float* V, int64_t ldv, const float* G, int64_t ldg, float* O,
                            int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int d_k, int d_v,
                            int causal, int decode, const int32_t* kv_lengths, int* status,
                            cudaStream_t stream);

// C = A W + bias (+ R) on tcgen05: bf16 operands, fp32 accumulation in TMEM, bf16 output.
// Requires K, N, lda, ldw, ldc (and ldr) multiples of 8 and 16-byte aligned pointers.
// seg_len (device int32 per segment of seg_rows rows) or null: rows of a segment at or past
// its length rounded up to a multiple of 128 may be left unwritten (the key / value rows that
// the attention kernels never load).
cudaError_t launch_gemm_bf16(const void* A, int64_t lda, const void* W, int64_t ldw,
                             const void* bias, const void* R, int64_t ldr, void* C, int64_t ldc,
                             int M, int N, int K, int num_sms, int* status, cudaStream_t stream,
                             const int32_t* seg_len = nullptr, int seg_rows = 0);

// Two independent bf16 projections with the same K in one launch of the CTA-pair kernel
// (both M > 128; no residual): C = A W + bias, rows past the segment lengths optionally
// skipped as above, and C2 = A2 W2 + bias2.  cudaErrorInvalidValue if either M <= 128.
cudaError_t launch_gemm_bf16_two(const void* A, int64_t lda, const void* W, int64_t ldw,
                                 const void* bias, void* C, int64_t ldc, int M, int N,
                                 const int32_t* seg_len, int seg_rows, const void* A2, int64_t lda2,
                                 const void* W2, int64_t ldw2, const void* bias2, void* C2,
                                 int64_t ldc2, int M2, int N2, int K, int num_sms, int* status,
                                 cudaStream_t stream);

// Fused flash attention on tcgen05 for head dim 64 or 128 (d_k == d_v), grouped K/V heads
// (h_kv divides h) and an optional gate G.  num_sms sizes the persistent grid of the d = 64
// kernel.
cudaError_t launch_attn_bf16(const void* Q, int64_t ldq, const void* K, int64_t ldk,
                             const void* V, int64_t ldv, const void* G, int64_t ldg, void* O,
                             int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int d, int causal,
                             const int32_t* kv_lengths, int num_sms, int* status,
                             cudaStream_t stream);

// One decode step over a bf16 KV cache (head dim 64 or 128): the T_q new query rows of
// each batch are the last T_q of its L_b cached tokens.  ws: at least
// decode_workspace_bytes(B, h, T_q, d) bytes of device scratch.
size_t decode_workspace_bytes(int B, int h, int T_q, int d, int T_max);
cudaError_t launch_decode_bf16(const void* Q, int64_t ldq, const void* Kc, int64_t ldk,
                               const void* Vc, int64_t ldv, void* O, int64_t ldo, int B, int h,
                               int h_kv, int T_q, int T_max, int d, const int32_t* cache_lengths,
                               void* ws, int num_sms, int* status, cudaStream_t stream);

}  // namespace mha
