// simt_f32.cu -- the fp32 path on CUDA cores (FFMA), for layers stored in fp32.
// fp32 results must agree with the exact result to about 1e-5 relative; TF32 tensor cores
// (10-bit mantissa) cannot, so both steps run in full fp32:
//   gemm_f32_kernel  C = A W + bias (+ R)   (itwiki.kr "멀티 헤드 어텐션", table rows 투영,
//                    출력 투영; the residual R of iamjaehka13.blog "[Deep Learning 5]
//                    Attention의 내부 계산", section 14)
//   attn_f32_kernel  online-softmax attention for every head, any d_k, d_v <= 256, written
//                    into the Concat layout (same page, 수식 and the shape table;
//                    iamjaehka13.blog sections 9-10), with grouped K/V heads and the sigmoid
//                    output gate (itwiki.kr, 추론 비용과 변형), and a decode mode in which
//                    the T_q rows are the last T_q of the L_b keys (a KV-cache step)
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int F_BM = 64, F_BN = 64, F_BK = 16;

// 64x64 output tile per 256-thread block, 4x4 outputs per thread; the K loop runs in
// order (k = 0, 1, ...) with one FFMA per product.
__global__ void __launch_bounds__(256)
    gemm_f32_kernel(const float* __restrict__ A, int64_t lda, const float* __restrict__ W,
                    int64_t ldw, const float* __restrict__ bias, const float* R, int64_t ldr,
                    float* C, int64_t ldc, int M, int N, int K) {
    __shared__ float As[F_BK][F_BM + 4];  // As[k][m]
    __shared__ float Ws[F_BK][F_BN + 4];  // Ws[k][n]
    const int tx = threadIdx.x & 15;
    const int ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * F_BM;
    const int n0 = blockIdx.x * F_BN;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += F_BK) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int idx = threadIdx.x + p * 256;
            const int r = idx >> 4, c = idx & 15;  // A: 64 rows x 16 k
            const int gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < M && gk < K) ? A[(int64_t)gm * lda + gk] : 0.f;
            const int wr = idx >> 6, wc = idx & 63;  // W: 16 k x 64 cols
            const int wk = k0 + wr, wn = n0 + wc;
            Ws[wr][wc] = (wk < K && wn < N) ? W[(int64_t)wk * ldw + wn] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < F_BK; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Ws[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + ty * 4 + i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tx * 4 + j;
            if (gn < N)
                C[(int64_t)gm * ldc + gn] =
                    acc[i][j] + (bias ? bias[gn] : 0.f) + (R ? R[(int64_t)gm * ldr + gn] : 0.f);
        }
    }
}

constexpr int FA_BQ = 16;      // query rows per block (4 per warp)
constexpr int FA_BKEY = 32;    // keys per tile (one per lane)
constexpr int FA_THREADS = 128;
constexpr int FA_MAXV = 8;     // d_v <= 256: up to 8 output columns per lane

// One block = 16 query rows of one (batch, head).  Per key tile each lane scores one key;
// the row maximum and sum come from warp shuffles; every lane owns d_v/32 output columns.
// Query head `head` reads K/V head head / (h / h_kv).  G (gate pre-activations, (B, T_q)
// rows of stride ldg, head at columns head*d_v) or nullptr.  decode: row t sees keys
// j <= L_b - T_q + t, and L_b < T_q is invalid.
__global__ void __launch_bounds__(FA_THREADS)
    attn_f32_kernel(const float* __restrict__ Q, int64_t ldq, const float* __restrict__ K,
                    int64_t ldk, const float* __restrict__ V, int64_t ldv,
                    const float* __restrict__ G, int64_t ldg, float* __restrict__ O,
                    int64_t ldo, int h, int h_kv, int T_q, int T_kv, int dk, int dv, int causal,
                    int decode, const int32_t* __restrict__ kv_lengths, float scale, int* status) {
    extern __shared__ float fsm[];
    float* Qs = fsm;                       // [FA_BQ][dk]
    float* Ks = Qs + FA_BQ * dk;           // [FA_BKEY][dk + 1]
    float* Vs = Ks + FA_BKEY * (dk + 1);   // [FA_BKEY][dv]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int b = bh / h, head = bh - b * h;
    const int kvh = head / (h / h_kv);
    const int q0 = blockIdx.y * FA_BQ;
    const int L = kv_lengths ? kv_lengths[b] : T_kv;
    const bool bad = L < (decode ? T_q : 1) || L > T_kv;
    const int shift = decode ? L - T_q : 0;  // row t is token t + shift

    if (bad) {
        if (threadIdx.x == 0) record_status(status, kStatusBadLength);
        for (int i = threadIdx.x; i < FA_BQ * dv; i += FA_THREADS) {
            const int r = i / dv, e = i - (i / dv) * dv;
            if (q0 + r < T_q) O[((int64_t)b * T_q + q0 + r) * ldo + (int64_t)head * dv + e] = NAN;
        }
        return;
    }
    for (int i = threadIdx.x; i < FA_BQ * dk; i += FA_THREADS) {
        const int r = i / dk, e = i - (i / dk) * dk;
        const int t = q0 + r;
        Qs[i] = t < T_q ? Q[((int64_t)b * T_q + t) * ldq + (int64_t)head * dk + e] : 0.f;
    }
    int kv_end = L;
    if ((causal || decode) && kv_end > q0 + FA_BQ + shift) kv_end = q0 + FA_BQ + shift;

    float m[4], l[4], o[4][FA_MAXV];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int u = 0; u < FA_MAXV; ++u) o[rr][u] = 0.f;
    }

    for (int kt0 = 0; kt0 < kv_end; kt0 += FA_BKEY) {
        __syncthreads();
        for (int i = threadIdx.x; i < FA_BKEY * dk; i += FA_THREADS) {
            const int j = i / dk, e = i - (i / dk) * dk;
            const int key = kt0 + j;
            Ks[j * (dk + 1) + e] = key < T_kv ? K[((int64_t)b * T_kv + key) * ldk + (int64_t)kvh * dk + e] : 0.f;
        }
        for (int i = threadIdx.x; i < FA_BKEY * dv; i += FA_THREADS) {
            const int j = i / dv, e = i - (i / dv) * dv;
            const int key = kt0 + j;
            Vs[i] = key < T_kv ? V[((int64_t)b * T_kv + key) * ldv + (int64_t)kvh * dv + e] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = warp * 4 + rr;
            const int t = q0 + r;
            if (t >= T_q) continue;  // warp-uniform
            const int key = kt0 + lane;
            const bool visible = key < L && !((causal || decode) && key > t + shift);
            float s = -INFINITY;
            if (visible) {
                float dot = 0.f;
                const float* qr = Qs + r * dk;
                const float* kr = Ks + lane * (dk + 1);
                for (int e = 0; e < dk; ++e) dot = fmaf(qr[e], kr[e], dot);
                s = dot * scale;
            }
            float tmax = s;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_new = fmaxf(m[rr], tmax);
            if (m_new == -INFINITY) continue;  // nothing visible yet (warp-uniform)
            const float p = visible ? expf(s - m_new) : 0.f;
            const float alpha = expf(m[rr] - m_new);
            float psum = p;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l[rr] = l[rr] * alpha + psum;
#pragma unroll
            for (int u = 0; u < FA_MAXV; ++u) {
                if (32 * u >= dv) break;  // uniform: only the column groups that exist
                const int e = lane + 32 * u;
                float acc = o[rr][u] * alpha;
                for (int jj = 0; jj < FA_BKEY; ++jj) {
                    const float pj = __shfl_sync(0xffffffffu, p, jj);
                    if (e < dv) acc = fmaf(pj, Vs[jj * dv + e], acc);
                }
                o[rr][u] = acc;
            }
            m[rr] = m_new;
        }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
        const int t = q0 + warp * 4 + rr;
        if (t >= T_q) continue;
        const float inv = 1.f / l[rr];
#pragma unroll
        for (int u = 0; u < FA_MAXV; ++u) {
            const int e = lane + 32 * u;
            if (e >= dv) continue;
            float y = o[rr][u] * inv;
            if (G != nullptr) y *= 1.f / (1.f + expf(-G[((int64_t)b * T_q + t) * ldg + (int64_t)head * dv + e]));
            O[((int64_t)b * T_q + t) * ldo + (int64_t)head * dv + e] = y;
        }
    }
}

}  // namespace

cudaError_t launch_gemm_f32(const float* A, int64_t lda, const float* W, int64_t ldw,
                            const float* bias, const float* R, int64_t ldr, float* C, int64_t ldc,
                            int M, int N, int K, cudaStream_t stream) {
    const dim3 grid((unsigned)((N + F_BN - 1) / F_BN), (unsigned)((M + F_BM - 1) / F_BM));
    gemm_f32_kernel<<<grid, 256, 0, stream>>>(A, lda, W, ldw, bias, R, ldr, C, ldc, M, N, K);
    return cudaGetLastError();
}

cudaError_t launch_attn_f32(const float* Q, int64_t ldq, const float* K, int64_t ldk,
                            const float* V, int64_t ldv, const float* G, int64_t ldg, float* O,
                            int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int d_k, int d_v,
                            int causal, int decode, const int32_t* kv_lengths, int* status,
                            cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)(FA_BQ * d_k + FA_BKEY * (d_k + 1) + FA_BKEY * d_v);
    cudaError_t err = cudaFuncSetAttribute(attn_f32_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const float scale = (float)(1.0 / sqrt((double)d_k));
    const dim3 grid((unsigned)(B * h), (unsigned)((T_q + FA_BQ - 1) / FA_BQ));
    attn_f32_kernel<<<grid, FA_THREADS, smem, stream>>>(Q, ldq, K, ldk, V, ldv, G, ldg, O, ldo, h,
                                                        h_kv, T_q, T_kv, d_k, d_v, causal, decode,
                                                        kv_lengths, scale, status);
    return cudaGetLastError();
}

}  // namespace mha
