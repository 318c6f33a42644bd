// mha_api.cu -- the C ABI of include/mha.h: handle, host-side validation, workspace
// layout and the launch sequence of the forward pass.
//
// mha_forward (itwiki.kr "멀티 헤드 어텐션", tensor-shape table, all rows):
//   self-attention : one GEMM  X (B*T, D) x W_qkv (D, h*d_k + h_kv*(d_k+d_v) [+ h*d_v]) -> the
//                    fused buffer [Q | K | V (| G)]; attention reads Q, K, V (and the gate G) as
//                    strided column views of it (the head split is addressing, not a copy) and
//                    writes Ocat (B*T, h*d_v); GEMM  Ocat x W_o (+ residual) -> Y
//   cross-attention: GEMM X_q x W_qkv[:, Q block] -> Q (and X_q x W_qkv[:, G block] -> G);
//                    GEMM X_kv x W_qkv[:, K|V blocks] -> KV (iamjaehka13.blog "[Deep Learning 5]
//                    Attention의 내부 계산", section 19), then attention and the output GEMM.
// Variants (itwiki.kr, section 추론 비용과 변형; iamjaehka13.blog, section 14): grouped K/V
// heads (h_kv < h: MQA/GQA), the sigmoid output gate, the residual X' = X + O W_O, and the
// KV-cache decode step (mha_decode).
// All launches go to the caller's stream; nothing is allocated or synchronised here.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <atomic>

#include "../../include/mha.h"
#include "internal.h"

namespace mha {

// ------------------------------------------------------------------ tensor maps

// The driver's tensor-map encoder, looked up once (host threads may race to do it: the
// lookups agree, and the pointer is published before the state that says it is there).
static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};
static std::atomic<int> g_encode_state{0};  // 0 unknown, 1 ok, -1 unavailable

static bool get_encoder() {
    if (g_encode_state.load(std::memory_order_acquire) == 0) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t err =
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess && fn != nullptr) {
            g_encode.store(reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn), std::memory_order_relaxed);
            g_encode_state.store(1, std::memory_order_release);
        } else {
            g_encode_state.store(-1, std::memory_order_release);
        }
    }
    return g_encode_state.load(std::memory_order_acquire) == 1;
}

bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box, int swizzle_bytes) {
    if (!get_encoder()) return false;
    if (swizzle_bytes != 128 && swizzle_bytes != 0) return false;
    cuuint64_t gdim[5];
    cuuint64_t gstr[4];
    cuuint32_t bdim[5];
    cuuint32_t estr[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) gstr[i] = strides_bytes[i];
    }
    const CUresult r = g_encode.load(std::memory_order_relaxed)(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                                const_cast<void*>(base), gdim, gstr, bdim, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mha

namespace {

constexpr size_t kStatusBytes = 256;

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t elem_bytes(mha_dtype t) { return t == MHA_F32 ? 4 : 2; }

// Bytes of [p, p + n) overlap [q, q + m)?
inline bool overlaps(const void* p, size_t n, const void* q, size_t m) {
    if (!p || !q || n == 0 || m == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

// Column widths of the fused projection [Q | K | V | G].
struct Widths {
    int64_t q, k, v, g;  // h*dk, h_kv*dk, h_kv*dv, gated ? h*dv : 0
    int64_t all() const { return q + k + v + g; }
};

Widths widths(const mha_s* m) {
    Widths w;
    w.q = (int64_t)m->h * m->dk;
    w.k = (int64_t)m->h_kv * m->dk;
    w.v = (int64_t)m->h_kv * m->dv;
    w.g = m->gated ? (int64_t)m->h * m->dv : 0;
    return w;
}

struct WsLayout {
    size_t q_off, kv_off, o_off, total;
};

// status | Q and G (B,T_q,h*dk [+ h*dv]) | KV (B,T_kv,h_kv*(dk+dv)) | Ocat (B,T_q,h*dv).  For
// self-attention the Q and KV regions are used as one fused (B,T,[Q|K|V|G]) buffer starting
// at q_off, which needs no more bytes than the two regions together.
WsLayout ws_layout(const mha_s* m, int B, int T_q, int T_kv) {
    const size_t s = elem_bytes(m->dtype);
    const Widths wd = widths(m);
    const size_t hv = (size_t)m->h * m->dv;
    WsLayout w;
    w.q_off = kStatusBytes;
    w.kv_off = w.q_off + align256((size_t)B * T_q * (size_t)(wd.q + wd.g) * s);
    w.o_off = w.kv_off + align256((size_t)B * T_kv * (size_t)(wd.k + wd.v) * s);
    w.total = w.o_off + align256((size_t)B * T_q * hv * s);
    return w;
}

std::atomic<int> g_num_sms[64];  // SM count per device, 0 until asked

mha_status query_sms(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
    int n = dev >= 0 && dev < 64 ? g_num_sms[dev].load(std::memory_order_relaxed) : 0;
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return MHA_ERR_CUDA;
        if (dev >= 0 && dev < 64) g_num_sms[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return MHA_OK;
}

// Does this build have tensor-core kernels for the handle's shape?
bool bf16_shape_supported(const mha_s* m) {
    return m->dk == m->dv && (m->dk == 64 || m->dk == 128) && (m->D % 8) == 0;
}

int* status_ptr(const mha_s* m) { return m->ws ? reinterpret_cast<int*>(m->ws) : nullptr; }

// ---------------------------------------------------------------- step launchers (validated)

// seg_len / seg_rows: see launch_gemm_bf16 (rows the attention never reads may be skipped)
mha_status run_linear(const mha_s* m, const void* A, int64_t lda, int M, int K, const void* W,
                      int64_t ldw, int N, const void* bias, const void* R, int64_t ldr, void* C,
                      int64_t ldc, cudaStream_t stream, const int32_t* seg_len = nullptr,
                      int seg_rows = 0) {
    cudaError_t err;
    if (m->dtype == MHA_F32) {
        err = mha::launch_gemm_f32(static_cast<const float*>(A), lda, static_cast<const float*>(W),
                                   ldw, static_cast<const float*>(bias), static_cast<const float*>(R),
                                   ldr, static_cast<float*>(C), ldc, M, N, K, stream);
    } else {
        int sms = 0;
        const mha_status st = query_sms(&sms);
        if (st != MHA_OK) return st;
        err = mha::launch_gemm_bf16(A, lda, W, ldw, bias, R, ldr, C, ldc, M, N, K, sms,
                                    status_ptr(m), stream, seg_len, seg_rows);
    }
    return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// Two independent projections with the same K (validated): one launch for bf16 with both
// M > 128, else one after the other.  seg_len / seg_rows apply to the first.
mha_status run_linear_pair(const mha_s* m, const void* A, int64_t lda, int M, const void* W, int64_t ldw,
                           int N, const void* bias, const int32_t* seg_len, int seg_rows, void* C,
                           int64_t ldc, const void* A2, int64_t lda2, int M2, const void* W2,
                           int64_t ldw2, int N2, const void* bias2, void* C2, int64_t ldc2, int K,
                           cudaStream_t stream) {
    if (m->dtype == MHA_BF16 && M > 128 && M2 > 128) {
        int sms = 0;
        const mha_status st = query_sms(&sms);
        if (st != MHA_OK) return st;
        const cudaError_t err =
            mha::launch_gemm_bf16_two(A, lda, W, ldw, bias, C, ldc, M, N, seg_len, seg_rows, A2, lda2, W2,
                                      ldw2, bias2, C2, ldc2, M2, N2, K, sms, status_ptr(m), stream);
        return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
    }
    if (M > 0) {
        const mha_status st = run_linear(m, A, lda, M, K, W, ldw, N, bias, nullptr, 0, C, ldc, stream,
                                         seg_len, seg_len ? seg_rows : 0);
        if (st != MHA_OK) return st;
    }
    if (M2 > 0) return run_linear(m, A2, lda2, M2, K, W2, ldw2, N2, bias2, nullptr, 0, C2, ldc2, stream);
    return MHA_OK;
}

mha_status run_attention(const mha_s* m, int B, int T_q, int T_kv, const void* Q, int64_t ldq,
                         const void* K, int64_t ldk, const void* V, int64_t ldv, const void* G,
                         int64_t ldg, int causal, const int32_t* kv_lengths, void* O, int64_t ldo,
                         cudaStream_t stream) {
    cudaError_t err;
    if (m->dtype == MHA_F32) {
        err = mha::launch_attn_f32(static_cast<const float*>(Q), ldq, static_cast<const float*>(K),
                                   ldk, static_cast<const float*>(V), ldv,
                                   static_cast<const float*>(G), ldg, static_cast<float*>(O), ldo, B,
                                   m->h, m->h_kv, T_q, T_kv, m->dk, m->dv, causal, 0, kv_lengths,
                                   status_ptr(m), stream);
    } else {
        int sms = 0;
        const mha_status st = query_sms(&sms);
        if (st != MHA_OK) return st;
        err = mha::launch_attn_bf16(Q, ldq, K, ldk, V, ldv, G, ldg, O, ldo, B, m->h, m->h_kv, T_q, T_kv,
                                    m->dk, causal, kv_lengths, sms, status_ptr(m), stream);
    }
    return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// Checks shared by the public attention and forward entry points.
mha_status check_attention_shape(const mha_s* m, int B, int T_q, int T_kv, int causal) {
    if (B < 0 || T_q < 0 || T_kv < 0) return MHA_ERR_INVALID_ARG;
    if (causal && T_q != T_kv) return MHA_ERR_INVALID_ARG;
    if ((int64_t)B * m->h > INT32_MAX) return MHA_ERR_INVALID_ARG;
    if ((int64_t)B * T_q > INT32_MAX || (int64_t)B * T_kv > INT32_MAX) return MHA_ERR_INVALID_ARG;
    if (m->dtype == MHA_F32) {
        if (m->dk > 256 || m->dv > 256) return MHA_ERR_UNSUPPORTED;
        if ((T_q + 15) / 16 > 65535) return MHA_ERR_UNSUPPORTED;
    } else {
        if (!bf16_shape_supported(m)) return MHA_ERR_UNSUPPORTED;
        if ((T_q + 127) / 128 > 65535) return MHA_ERR_UNSUPPORTED;
        if ((int64_t)B * m->h * ((T_q + 127) / 128) > INT32_MAX) return MHA_ERR_UNSUPPORTED;
    }
    return MHA_OK;
}

// The copy streams and events of mha_forward_host, on the current device.  All or none.
mha_status create_aux(mha_s* m) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
    mha_s t = *m;
    bool ok = cudaStreamCreateWithFlags(&t.aux_h2d, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamCreateWithFlags(&t.aux_d2h, cudaStreamNonBlocking) == cudaSuccess;
    const unsigned fl = cudaEventDisableTiming;
    ok = ok && cudaEventCreateWithFlags(&t.aux_start, fl) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&t.aux_done, fl) == cudaSuccess;
    for (int i = 0; ok && i < kHostMaxChunks; ++i)
        ok = cudaEventCreateWithFlags(&t.aux_in[i], fl) == cudaSuccess &&
             cudaEventCreateWithFlags(&t.aux_out[i], fl) == cudaSuccess;
    if (!ok) return MHA_ERR_CUDA;  // (a partial set is left to the process teardown)
    t.aux_dev = dev;
    *m = t;
    return MHA_OK;
}

// mha_forward_host: the forward's scratch for one chunk of Bc batch elements, then device
// copies of X_q, X_kv, the residual and Y for the whole batch.
struct HostLayout {
    int chunks, Bc;
    size_t x_off, xkv_off, r_off, y_off, total;
};

// The batch cut of mha_forward_host: chunk c covers batch elements [bnd[c], bnd[c + 1]);
// returns the number of chunks.  Up to two chunks are equal (ceil(B / n) elements); from three
// on, the first and the last are half the size of the others, so that the copy-in before the
// first kernel and the copy-out after the last one, which nothing overlaps, are short.
int chunk_bounds(int B, int n, int* bnd) {
    int k = 0;
    bnd[0] = 0;
    if (n <= 2) {
        const int Bc = (B + n - 1) / n;
        for (int b = Bc; b < B; b += Bc) bnd[++k] = b;
        bnd[++k] = B;
        return k;
    }
    double cum = 0.0;
    for (int c = 0; c < n; ++c) {
        cum += (c == 0 || c == n - 1) ? 0.5 : 1.0;
        int e = (int)((double)B * cum / (n - 1) + 0.5);
        if (e > B) e = B;
        if (e > bnd[k]) bnd[++k] = e;
    }
    if (bnd[k] < B) bnd[++k] = B;
    return k;
}

bool host_layout(const mha_s* m, int B, int T_q, int T_kv, int chunks, HostLayout* L) {
    if (B <= 0 || T_q <= 0 || T_kv <= 0 || chunks < 1 || chunks > kHostMaxChunks) return false;
    const int c = chunks < B ? chunks : B;
    int bnd[kHostMaxChunks + 2];
    L->chunks = chunk_bounds(B, c, bnd);
    L->Bc = 0;  // the largest chunk
    for (int i = 0; i < L->chunks; ++i)
        if (bnd[i + 1] - bnd[i] > L->Bc) L->Bc = bnd[i + 1] - bnd[i];
    const size_t s = elem_bytes(m->dtype);
    const size_t xq = (size_t)B * T_q * (size_t)m->D * s, xkv = (size_t)B * T_kv * (size_t)m->D * s;
    L->x_off = align256(ws_layout(m, L->Bc, T_q, T_kv).total);
    L->xkv_off = L->x_off + align256(xq);
    L->r_off = L->xkv_off + align256(xkv);
    L->y_off = L->r_off + align256(xq);
    L->total = L->y_off + align256(xq);
    return true;
}

}  // namespace

extern "C" {

mha_status mha_create_ex(mha_t* out, int D, int h, int h_kv, int d_k, int d_v, int gated,
                         mha_dtype dtype) {
    if (out == nullptr) return MHA_ERR_INVALID_ARG;
    *out = nullptr;
    if (D <= 0 || h <= 0 || d_k <= 0 || d_v <= 0) return MHA_ERR_INVALID_ARG;
    if (h_kv <= 0 || h_kv > h || h % h_kv != 0) return MHA_ERR_INVALID_ARG;
    if (gated != 0 && gated != 1) return MHA_ERR_INVALID_ARG;
    if (dtype != MHA_F32 && dtype != MHA_BF16) return MHA_ERR_INVALID_ARG;
    if ((int64_t)h * d_k + (int64_t)h_kv * (d_k + d_v) + (int64_t)gated * h * d_v > INT32_MAX)
        return MHA_ERR_INVALID_ARG;
    mha_s* m = static_cast<mha_s*>(calloc(1, sizeof(mha_s)));
    if (m == nullptr) return MHA_ERR_INVALID_ARG;
    m->D = D;
    m->h = h;
    m->h_kv = h_kv;
    m->dk = d_k;
    m->dv = d_v;
    m->gated = gated;
    m->dtype = dtype;
    m->aux_dev = -1;
    *out = m;
    return MHA_OK;
}

mha_status mha_create(mha_t* out, int D, int h, int d_k, int d_v, mha_dtype dtype) {
    return mha_create_ex(out, D, h, h, d_k, d_v, 0, dtype);
}

void mha_destroy(mha_t handle) {
    if (handle == nullptr) return;
    if (handle->aux_dev >= 0) {
        int cur = 0;
        const bool swap = cudaGetDevice(&cur) == cudaSuccess && cur != handle->aux_dev &&
                          cudaSetDevice(handle->aux_dev) == cudaSuccess;
        cudaStreamDestroy(handle->aux_h2d);
        cudaStreamDestroy(handle->aux_d2h);
        cudaEventDestroy(handle->aux_start);
        cudaEventDestroy(handle->aux_done);
        for (int i = 0; i < kHostMaxChunks; ++i) {
            cudaEventDestroy(handle->aux_in[i]);
            cudaEventDestroy(handle->aux_out[i]);
        }
        if (swap) cudaSetDevice(cur);
    }
    free(handle);
}

size_t mha_workspace_size(mha_t handle, int B, int T_q, int T_kv) {
    if (handle == nullptr || B < 0 || T_q < 0 || T_kv < 0) return 0;
    return ws_layout(handle, B, T_q, T_kv).total;
}

mha_status mha_set_workspace(mha_t handle, void* dev_ptr, size_t bytes) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    if (dev_ptr == nullptr) {
        handle->ws = nullptr;
        handle->ws_bytes = 0;
        return MHA_OK;
    }
    if ((reinterpret_cast<uintptr_t>(dev_ptr) & 255u) != 0 || bytes < kStatusBytes)
        return MHA_ERR_INVALID_ARG;
    if (cudaMemset(dev_ptr, 0, kStatusBytes) != cudaSuccess) return MHA_ERR_CUDA;
    if (handle->aux_dev < 0) {
        const mha_status st = create_aux(handle);
        if (st != MHA_OK) return st;
    }
    handle->ws = dev_ptr;
    handle->ws_bytes = bytes;
    return MHA_OK;
}

}  // extern "C"

namespace {

// Host-side checks shared by the projection entry points (M == 0 passes: nothing to do).
mha_status check_linear(const mha_s* handle, const void* A, int64_t lda, int M, int K, const void* W,
                        int64_t ldw, int N, const void* bias, const void* R, int64_t ldr, const void* C,
                        int64_t ldc) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    if (M < 0 || K <= 0 || N <= 0) return MHA_ERR_INVALID_ARG;
    if (M == 0) return MHA_OK;
    if (A == nullptr || W == nullptr || C == nullptr) return MHA_ERR_INVALID_ARG;
    if (lda < K || ldw < N || ldc < N || (R && ldr < N)) return MHA_ERR_INVALID_ARG;
    if (handle->dtype == MHA_BF16) {
        if ((K % 8) || (N % 8) || (lda % 8) || (ldw % 8) || (ldc % 8) || (R && (ldr % 8)))
            return MHA_ERR_INVALID_ARG;
        if (!aligned16(A) || !aligned16(W) || !aligned16(C) || (bias && !aligned16(bias)) ||
            (R && !aligned16(R)))
            return MHA_ERR_INVALID_ARG;
    }
    const size_t s = elem_bytes(handle->dtype);
    const size_t c_bytes = ((size_t)(M - 1) * ldc + N) * s;
    if (overlaps(C, c_bytes, A, ((size_t)(M - 1) * lda + K) * s) ||
        overlaps(C, c_bytes, W, ((size_t)(K - 1) * ldw + N) * s))
        return MHA_ERR_INVALID_ARG;
    // the residual may be C itself (same rows), but not otherwise overlap it
    if (R && !(R == C && ldr == ldc) && overlaps(C, c_bytes, R, ((size_t)(M - 1) * ldr + N) * s))
        return MHA_ERR_INVALID_ARG;
    return MHA_OK;
}

}  // namespace

extern "C" {

mha_status mha_linear_ex(mha_t handle, const void* A, int64_t lda, int M, int K, const void* W,
                         int64_t ldw, int N, const void* bias, const void* R, int64_t ldr, void* C,
                         int64_t ldc, void* stream) {
    const mha_status st = check_linear(handle, A, lda, M, K, W, ldw, N, bias, R, ldr, C, ldc);
    if (st != MHA_OK || M == 0) return st;
    return run_linear(handle, A, lda, M, K, W, ldw, N, bias, R, R ? ldr : 0, C, ldc,
                      static_cast<cudaStream_t>(stream));
}

mha_status mha_linear_segments(mha_t handle, const void* A, int64_t lda, int M, int K, const void* W,
                               int64_t ldw, int N, const void* bias, const int32_t* seg_len,
                               int seg_rows, void* C, int64_t ldc, void* stream) {
    if (seg_len == nullptr || seg_rows <= 0 || M % seg_rows != 0) return MHA_ERR_INVALID_ARG;
    const mha_status st = check_linear(handle, A, lda, M, K, W, ldw, N, bias, nullptr, 0, C, ldc);
    if (st != MHA_OK || M == 0) return st;
    return run_linear(handle, A, lda, M, K, W, ldw, N, bias, nullptr, 0, C, ldc,
                      static_cast<cudaStream_t>(stream), seg_len, seg_rows);
}

mha_status mha_linear_pair(mha_t handle, const void* A, int64_t lda, int M, const void* W,
                           int64_t ldw, int N, const void* bias, const int32_t* seg_len,
                           int seg_rows, void* C, int64_t ldc, const void* A2, int64_t lda2,
                           int M2, const void* W2, int64_t ldw2, int N2, const void* bias2,
                           void* C2, int64_t ldc2, int K, void* stream) {
    if (seg_len != nullptr && (seg_rows <= 0 || M % seg_rows != 0)) return MHA_ERR_INVALID_ARG;
    mha_status st = check_linear(handle, A, lda, M, K, W, ldw, N, bias, nullptr, 0, C, ldc);
    if (st != MHA_OK) return st;
    st = check_linear(handle, A2, lda2, M2, K, W2, ldw2, N2, bias2, nullptr, 0, C2, ldc2);
    if (st != MHA_OK) return st;
    if (M > 0 && M2 > 0) {
        // neither output may overlap the other or the other projection's inputs
        const size_t s = elem_bytes(handle->dtype);
        const size_t c1 = ((size_t)(M - 1) * ldc + N) * s, c2 = ((size_t)(M2 - 1) * ldc2 + N2) * s;
        if (overlaps(C, c1, C2, c2) || overlaps(C, c1, A2, ((size_t)(M2 - 1) * lda2 + K) * s) ||
            overlaps(C, c1, W2, ((size_t)(K - 1) * ldw2 + N2) * s) ||
            overlaps(C2, c2, A, ((size_t)(M - 1) * lda + K) * s) ||
            overlaps(C2, c2, W, ((size_t)(K - 1) * ldw + N) * s))
            return MHA_ERR_INVALID_ARG;
    }
    if (M == 0 && M2 == 0) return MHA_OK;
    return run_linear_pair(handle, A, lda, M, W, ldw, N, bias, seg_len, seg_rows, C, ldc, A2, lda2, M2, W2,
                           ldw2, N2, bias2, C2, ldc2, K, static_cast<cudaStream_t>(stream));
}

mha_status mha_linear(mha_t handle, const void* A, int64_t lda, int M, int K, const void* W,
                      int64_t ldw, int N, const void* bias, void* C, int64_t ldc, void* stream) {
    return mha_linear_ex(handle, A, lda, M, K, W, ldw, N, bias, nullptr, 0, C, ldc, stream);
}

mha_status mha_attention_ex(mha_t handle, int B, int T_q, int T_kv, const void* Q, int64_t ldq,
                            const void* K, int64_t ldk, const void* V, int64_t ldv, const void* G,
                            int64_t ldg, int causal, const int32_t* kv_lengths, void* O, int64_t ldo,
                            void* stream) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    mha_status st = check_attention_shape(handle, B, T_q, T_kv, causal);
    if (st != MHA_OK) return st;
    if (B == 0 || T_q == 0) return MHA_OK;
    if (T_kv == 0) return MHA_ERR_INVALID_ARG;
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return MHA_ERR_INVALID_ARG;
    const Widths wd = widths(handle);
    const int64_t hv = (int64_t)handle->h * handle->dv;
    if (ldq < wd.q || ldk < wd.k || ldv < wd.v || ldo < hv || (G && ldg < hv)) return MHA_ERR_INVALID_ARG;
    if (handle->dtype == MHA_BF16) {
        if ((ldq % 8) || (ldk % 8) || (ldv % 8) || (ldo % 8) || (G && (ldg % 8))) return MHA_ERR_INVALID_ARG;
        if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || (G && !aligned16(G)))
            return MHA_ERR_INVALID_ARG;
    }
    return run_attention(handle, B, T_q, T_kv, Q, ldq, K, ldk, V, ldv, G, G ? ldg : 0, causal, kv_lengths,
                         O, ldo, static_cast<cudaStream_t>(stream));
}

mha_status mha_attention(mha_t handle, int B, int T_q, int T_kv, const void* Q, int64_t ldq,
                         const void* K, int64_t ldk, const void* V, int64_t ldv, int causal,
                         const int32_t* kv_lengths, void* O, int64_t ldo, void* stream) {
    return mha_attention_ex(handle, B, T_q, T_kv, Q, ldq, K, ldk, V, ldv, nullptr, 0, causal,
                            kv_lengths, O, ldo, stream);
}

}  // extern "C"

namespace mha {

// Every host-side check of mha_forward_ex except the workspace's: MHA_OK means the call
// launches its kernels (or, for B == 0 or T_q == 0, nothing) once a large enough workspace
// is attached.
mha_status check_forward(const mha_s* m, const void* X_q, const void* X_kv, int B, int T_q,
                         int T_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                         const void* b_o, int causal, const void* residual, const void* out) {
    if (m == nullptr) return MHA_ERR_INVALID_ARG;
    const bool self = (X_kv == nullptr || X_kv == X_q);
    if (self && T_kv != T_q) return MHA_ERR_INVALID_ARG;
    const mha_status st = check_attention_shape(m, B, T_q, T_kv, causal);
    if (st != MHA_OK) return st;
    if (B == 0 || T_q == 0) return MHA_OK;
    if (T_kv == 0) return MHA_ERR_INVALID_ARG;
    if (X_q == nullptr || W_qkv == nullptr || W_o == nullptr || out == nullptr)
        return MHA_ERR_INVALID_ARG;
    if (m->dtype == MHA_BF16) {
        if (!aligned16(X_q) || (X_kv && !aligned16(X_kv)) || !aligned16(W_qkv) ||
            !aligned16(W_o) || !aligned16(out) || (b_qkv && !aligned16(b_qkv)) ||
            (b_o && !aligned16(b_o)) || (residual && !aligned16(residual)))
            return MHA_ERR_INVALID_ARG;
    }
    const size_t s = elem_bytes(m->dtype);
    const int64_t D = m->D;
    const Widths wd = widths(m);
    const int64_t hv = (int64_t)m->h * m->dv;
    const int64_t ncols = wd.all();
    const size_t out_bytes = (size_t)B * T_q * D * s;
    if (overlaps(out, out_bytes, X_q, (size_t)B * T_q * D * s) ||
        (!self && overlaps(out, out_bytes, X_kv, (size_t)B * T_kv * D * s)) ||
        overlaps(out, out_bytes, W_qkv, (size_t)D * ncols * s) ||
        overlaps(out, out_bytes, W_o, (size_t)hv * D * s))
        return MHA_ERR_INVALID_ARG;
    // the residual is read in the output projection's epilogue, element by element before
    // the same element of Y is written: it may be Y itself, but not partly overlap it
    if (residual != nullptr && residual != out && overlaps(out, out_bytes, residual, out_bytes))
        return MHA_ERR_INVALID_ARG;
    return MHA_OK;
}

}  // namespace mha

extern "C" {

mha_status mha_forward_ex(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q, int T_kv,
                          const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                          int causal, const int32_t* kv_lengths, const void* residual, void* out,
                          void* stream) {
    const mha_s* m = handle;
    mha_status st = mha::check_forward(m, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal,
                                       residual, out);
    if (st != MHA_OK) return st;
    if (B == 0 || T_q == 0) return MHA_OK;
    const bool self = (X_kv == nullptr || X_kv == X_q);
    const size_t s = elem_bytes(m->dtype);
    const int64_t D = m->D;
    const Widths wd = widths(m);
    const int64_t hv = (int64_t)m->h * m->dv;
    const int64_t ncols = wd.all();
    const WsLayout w = ws_layout(m, B, T_q, T_kv);
    if (m->ws == nullptr || m->ws_bytes < w.total) return MHA_ERR_WORKSPACE;

    uint8_t* ws = static_cast<uint8_t*>(m->ws);
    void* ocat = ws + w.o_off;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const uint8_t* wqkv = static_cast<const uint8_t*>(W_qkv);
    const uint8_t* bqkv = static_cast<const uint8_t*>(b_qkv);
    const int64_t k_off = wd.q, v_off = wd.q + wd.k, g_off = wd.q + wd.k + wd.v;

    if (self) {
        // one projection into [Q | K | V | G]
        void* qkv = ws + w.q_off;
        st = run_linear(m, X_q, D, B * T_q, (int)D, W_qkv, ncols, (int)ncols, b_qkv, nullptr, 0, qkv,
                        ncols, cs);
        if (st != MHA_OK) return st;
        const uint8_t* base = static_cast<const uint8_t*>(qkv);
        st = run_attention(m, B, T_q, T_kv, base, ncols, base + k_off * s, ncols, base + v_off * s, ncols,
                           m->gated ? base + g_off * s : nullptr, ncols, causal, kv_lengths, ocat, hv, cs);
        if (st != MHA_OK) return st;
    } else {
        // query side [Q | G] from X_q, key/value side [K | V] from X_kv
        const int64_t qg = wd.q + wd.g;
        uint8_t* q = ws + w.q_off;
        uint8_t* kv = ws + w.kv_off;
        // key/value rows past each batch's key length (in whole 128-key tiles) are never read
        // by the attention step, so their projection may be skipped
        // (the query side [Q] next to them in the same launch; the gate block separately)
        st = run_linear_pair(m, X_kv, D, B * T_kv, wqkv + k_off * s, ncols, (int)(wd.k + wd.v),
                             bqkv ? bqkv + k_off * s : nullptr, kv_lengths, T_kv, kv, wd.k + wd.v, X_q, D,
                             B * T_q, W_qkv, ncols, (int)wd.q, b_qkv, q, qg, (int)D, cs);
        if (st != MHA_OK) return st;
        if (m->gated) {
            st = run_linear(m, X_q, D, B * T_q, (int)D, wqkv + g_off * s, ncols, (int)wd.g,
                            bqkv ? bqkv + g_off * s : nullptr, nullptr, 0, q + wd.q * s, qg, cs);
            if (st != MHA_OK) return st;
        }
        st = run_attention(m, B, T_q, T_kv, q, qg, kv, wd.k + wd.v, kv + wd.k * s, wd.k + wd.v,
                           m->gated ? q + wd.q * s : nullptr, qg, causal, kv_lengths, ocat, hv, cs);
        if (st != MHA_OK) return st;
    }
    return run_linear(m, ocat, hv, B * T_q, (int)hv, W_o, D, (int)D, b_o, residual, D, out, D, cs);
}

mha_status mha_forward_checked(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q,
                               int T_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                               const void* b_o, int causal, const int32_t* kv_lengths,
                               const int32_t* kv_lengths_host, void* out, void* stream) {
    if ((kv_lengths == nullptr) != (kv_lengths_host == nullptr)) return MHA_ERR_INVALID_ARG;
    if (kv_lengths_host != nullptr)
        for (int b = 0; b < B; ++b)
            if (kv_lengths_host[b] < 1 || kv_lengths_host[b] > T_kv) return MHA_ERR_BAD_LENGTH;
    return mha_forward(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal, kv_lengths, out,
                       stream);
}

mha_status mha_forward(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q, int T_kv,
                       const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                       int causal, const int32_t* kv_lengths, void* out, void* stream) {
    return mha_forward_ex(handle, X_q, X_kv, B, T_q, T_kv, W_qkv, b_qkv, W_o, b_o, causal, kv_lengths,
                          nullptr, out, stream);
}

size_t mha_decode_workspace_size(mha_t handle, int B, int T_q, int T_max) {
    if (handle == nullptr || B < 0 || T_q < 0 || T_max < 0) return 0;
    size_t part = 0;
    if (handle->dtype == MHA_BF16 && B > 0 && T_q > 0 && T_max > 0)
        part = mha::decode_workspace_bytes(B, handle->h, T_q, handle->dk, T_max);
    return kStatusBytes + align256(part);
}

mha_status mha_decode(mha_t handle, int B, int T_q, int T_max, const void* Q, int64_t ldq,
                      const void* K_cache, int64_t ldk, const void* V_cache, int64_t ldv,
                      const int32_t* cache_lengths, void* O, int64_t ldo, void* stream) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    const mha_s* m = handle;
    if (B < 0 || T_q < 0 || T_max < 0) return MHA_ERR_INVALID_ARG;
    if (B == 0 || T_q == 0) return MHA_OK;
    if (T_max == 0 || T_q > T_max || cache_lengths == nullptr) return MHA_ERR_INVALID_ARG;
    if ((int64_t)B * T_max > INT32_MAX || (int64_t)B * m->h * T_q > INT32_MAX) return MHA_ERR_INVALID_ARG;
    if (Q == nullptr || K_cache == nullptr || V_cache == nullptr || O == nullptr) return MHA_ERR_INVALID_ARG;
    const Widths wd = widths(m);
    const int64_t hv = (int64_t)m->h * m->dv;
    if (ldq < wd.q || ldk < wd.k || ldv < wd.v || ldo < hv) return MHA_ERR_INVALID_ARG;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (m->dtype == MHA_F32) {
        if (m->dk > 256 || m->dv > 256) return MHA_ERR_UNSUPPORTED;
        if ((T_q + 15) / 16 > 65535) return MHA_ERR_UNSUPPORTED;
        const cudaError_t err = mha::launch_attn_f32(
            static_cast<const float*>(Q), ldq, static_cast<const float*>(K_cache), ldk,
            static_cast<const float*>(V_cache), ldv, nullptr, 0, static_cast<float*>(O), ldo, B, m->h,
            m->h_kv, T_q, T_max, m->dk, m->dv, 0, 1, cache_lengths, status_ptr(m), cs);
        return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
    }
    if (!bf16_shape_supported(m)) return MHA_ERR_UNSUPPORTED;
    if ((ldq % 8) || (ldk % 8) || (ldv % 8) || (ldo % 8)) return MHA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K_cache) || !aligned16(V_cache) || !aligned16(O))
        return MHA_ERR_INVALID_ARG;
    const size_t need = mha_decode_workspace_size(handle, B, T_q, T_max);
    if (m->ws == nullptr || m->ws_bytes < need) return MHA_ERR_WORKSPACE;
    int sms = 0;
    const mha_status st = query_sms(&sms);
    if (st != MHA_OK) return st;
    const cudaError_t err = mha::launch_decode_bf16(
        Q, ldq, K_cache, ldk, V_cache, ldv, O, ldo, B, m->h, m->h_kv, T_q, T_max, m->dk, cache_lengths,
        static_cast<uint8_t*>(m->ws) + kStatusBytes, sms, status_ptr(m), cs);
    return err == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

size_t mha_forward_host_workspace_size(mha_t handle, int B, int T_q, int T_kv, int chunks) {
    HostLayout L;
    if (handle == nullptr || !host_layout(handle, B, T_q, T_kv, chunks, &L)) return 0;
    return L.total;
}

mha_status mha_forward_host(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q, int T_kv,
                            const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                            int causal, const int32_t* kv_lengths, const void* residual, void* out,
                            int chunks, void* stream) {
    if (handle == nullptr) return MHA_ERR_INVALID_ARG;
    mha_s* m = handle;
    const bool self = (X_kv == nullptr || X_kv == X_q);
    if (self && T_kv != T_q) return MHA_ERR_INVALID_ARG;
    if (chunks < 1 || chunks > kHostMaxChunks) return MHA_ERR_INVALID_ARG;
    mha_status st = check_attention_shape(m, B, T_q, T_kv, causal);
    if (st != MHA_OK) return st;
    if (B == 0 || T_q == 0) return MHA_OK;
    if (T_kv == 0) return MHA_ERR_INVALID_ARG;
    if (X_q == nullptr || W_qkv == nullptr || W_o == nullptr || out == nullptr) return MHA_ERR_INVALID_ARG;
    const size_t s = elem_bytes(m->dtype);
    const size_t row_q = (size_t)m->D * s;
    if (overlaps(out, (size_t)B * T_q * row_q, X_q, (size_t)B * T_q * row_q) ||
        (!self && overlaps(out, (size_t)B * T_q * row_q, X_kv, (size_t)B * T_kv * row_q)) ||
        (residual != nullptr && residual != X_q &&
         overlaps(out, (size_t)B * T_q * row_q, residual, (size_t)B * T_q * row_q)))
        return MHA_ERR_INVALID_ARG;
    HostLayout L;
    if (!host_layout(m, B, T_q, T_kv, chunks, &L)) return MHA_ERR_INVALID_ARG;
    if (m->ws == nullptr || m->ws_bytes < L.total || m->aux_dev < 0) return MHA_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MHA_ERR_CUDA;
    if (dev != m->aux_dev) return MHA_ERR_INVALID_ARG;

    int cb[kHostMaxChunks + 2];
    chunk_bounds(B, chunks < B ? chunks : B, cb);
    uint8_t* ws = static_cast<uint8_t*>(m->ws);
    uint8_t* xd = ws + L.x_off;
    uint8_t* xkvd = ws + L.xkv_off;
    uint8_t* rd = residual == nullptr ? nullptr : residual == X_q ? xd : ws + L.r_off;
    uint8_t* yd = ws + L.y_off;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto cuda = [](cudaError_t e) { return e == cudaSuccess; };
    // the copies start after the work already queued on the caller's stream
    if (!cuda(cudaEventRecord(m->aux_start, cs)) || !cuda(cudaStreamWaitEvent(m->aux_h2d, m->aux_start, 0)) ||
        !cuda(cudaStreamWaitEvent(m->aux_d2h, m->aux_start, 0)))
        return MHA_ERR_CUDA;
    // inputs, chunk by chunk, on the host-to-device stream
    for (int c = 0; c < L.chunks; ++c) {
        const int b0 = cb[c], nb = cb[c + 1] - cb[c];
        const size_t oq = (size_t)b0 * T_q * row_q, nq = (size_t)nb * T_q * row_q;
        if (!cuda(cudaMemcpyAsync(xd + oq, static_cast<const uint8_t*>(X_q) + oq, nq, cudaMemcpyHostToDevice,
                                  m->aux_h2d)))
            return MHA_ERR_CUDA;
        if (!self) {
            const size_t okv = (size_t)b0 * T_kv * row_q, nkv = (size_t)nb * T_kv * row_q;
            if (!cuda(cudaMemcpyAsync(xkvd + okv, static_cast<const uint8_t*>(X_kv) + okv, nkv,
                                      cudaMemcpyHostToDevice, m->aux_h2d)))
                return MHA_ERR_CUDA;
        }
        if (rd != nullptr && rd != xd &&
            !cuda(cudaMemcpyAsync(rd + oq, static_cast<const uint8_t*>(residual) + oq, nq,
                                  cudaMemcpyHostToDevice, m->aux_h2d)))
            return MHA_ERR_CUDA;
        if (!cuda(cudaEventRecord(m->aux_in[c], m->aux_h2d))) return MHA_ERR_CUDA;
    }
    // each chunk's forward on the caller's stream once its inputs are in; its output back on
    // the device-to-host stream while the next chunk computes
    for (int c = 0; c < L.chunks; ++c) {
        const int b0 = cb[c], nb = cb[c + 1] - cb[c];
        const size_t oq = (size_t)b0 * T_q * row_q, nq = (size_t)nb * T_q * row_q;
        if (!cuda(cudaStreamWaitEvent(cs, m->aux_in[c], 0))) return MHA_ERR_CUDA;
        st = mha_forward_ex(m, xd + oq, self ? nullptr : xkvd + (size_t)b0 * T_kv * row_q, nb, T_q, T_kv,
                            W_qkv, b_qkv, W_o, b_o, causal, kv_lengths == nullptr ? nullptr : kv_lengths + b0,
                            rd == nullptr ? nullptr : rd + oq, yd + oq, stream);
        if (st != MHA_OK) return st;
        if (!cuda(cudaEventRecord(m->aux_out[c], cs)) || !cuda(cudaStreamWaitEvent(m->aux_d2h, m->aux_out[c], 0)) ||
            !cuda(cudaMemcpyAsync(static_cast<uint8_t*>(out) + oq, yd + oq, nq, cudaMemcpyDeviceToHost,
                                  m->aux_d2h)))
            return MHA_ERR_CUDA;
    }
    // the caller's stream completes only after the last output has landed in host memory
    if (!cuda(cudaEventRecord(m->aux_done, m->aux_d2h)) || !cuda(cudaStreamWaitEvent(cs, m->aux_done, 0)))
        return MHA_ERR_CUDA;
    return MHA_OK;
}

mha_status mha_get_status(mha_t handle, int32_t* status_out, void* stream) {
    if (handle == nullptr || status_out == nullptr) return MHA_ERR_INVALID_ARG;
    if (handle->ws == nullptr) return MHA_ERR_WORKSPACE;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, handle->ws, sizeof(v), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return MHA_ERR_CUDA;
    if (cudaMemsetAsync(handle->ws, 0, sizeof(v), cs) != cudaSuccess) return MHA_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return MHA_ERR_CUDA;
    *status_out = v;
    return MHA_OK;
}

const char* mha_strerror(mha_status status) {
    switch (status) {
        case MHA_OK: return "ok";
        case MHA_ERR_INVALID_ARG: return "invalid argument";
        case MHA_ERR_UNSUPPORTED: return "shape or dtype not supported by this build";
        case MHA_ERR_WORKSPACE: return "workspace missing or too small";
        case MHA_ERR_CUDA: return "CUDA call or kernel launch failed";
        case MHA_ERR_TIMEOUT: return "a device pipeline wait timed out";
        case MHA_ERR_BAD_LENGTH: return "a key length is outside [1, T_kv]; its rows are NaN";
    }
    return "unknown status";
}

}  // extern "C"
