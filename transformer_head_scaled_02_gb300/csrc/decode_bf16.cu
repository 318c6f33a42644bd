// decode_bf16.cu -- one decode step over a key/value cache (itwiki.kr "멀티 헤드 어텐션",
// section 추론 비용과 변형: the keys and values of earlier tokens are kept in a KV cache and
// every generation step reads the whole cache, so the step is bound by memory bandwidth; with
// grouped K/V heads (MQA/GQA) h / h_kv query heads share each cached head).
//
// The T_q new tokens of batch b are the last T_q of its L_b cached tokens: new token t (row
// t) sees cache entries j <= L_b - T_q + t.  For cached K/V head g the query rows are the
// (query head, new token) pairs of its group, R = (h / h_kv) * T_q of them.
//
// Split over the cache (flash-decoding): CTA (chunk, g, b, row block) reads DEC_KEYS cached
// keys and values of head g once and, for up to DEC_ROWS query rows, computes the partial
// softmax statistics of its chunk -- the maximum m, the sum l of 2^(s - m) and the weighted
// value sum o -- and writes them to the workspace; a second kernel merges the chunks of each
// row: M = max m_c, O = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c.  Scores are kept in
// base 2 with log2(e)/sqrt(d) folded into the query.  The cache is bf16, all arithmetic fp32.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int DEC_KEYS = 128;     // cached keys per CTA (one per thread in the score phase)
constexpr int DEC_ROWS = 16;      // query rows per CTA
constexpr int DEC_THREADS = 128;

inline int dec_chunks(int T_max) { return (T_max + DEC_KEYS - 1) / DEC_KEYS; }

// Workspace: partials [B][h][T_q][chunk] of (m, l, o[d]) floats.
__host__ __device__ constexpr int dec_partial_floats(int d) { return d + 2; }

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

template <int HD>
__global__ void __launch_bounds__(DEC_THREADS)
    decode_partial_kernel(const __nv_bfloat16* __restrict__ Q, int64_t ldq,
                          const __nv_bfloat16* __restrict__ Kc, int64_t ldk,
                          const __nv_bfloat16* __restrict__ Vc, int64_t ldv, int h, int h_kv,
                          int T_q, int T_max, const int32_t* __restrict__ cache_lengths,
                          float scale_log2, float* __restrict__ part, int* status) {
    __shared__ __align__(16) float q_s[DEC_ROWS][HD];  // scaled query rows
    __shared__ float p_s[DEC_ROWS][DEC_KEYS];       // 2^(s - m) of this chunk
    __shared__ __align__(16) __nv_bfloat16 v_s[DEC_KEYS][HD];
    __shared__ float red_s[DEC_THREADS / 32][DEC_ROWS];
    __shared__ float m_s[DEC_ROWS], l_s[DEC_ROWS];

    grid_dependency_wait();  // Q and the cache may come from the previous kernel
    grid_launch_dependents();

    const int chunk = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = h / h_kv;                      // query heads per K/V head
    const int R = per * T_q;                       // query rows of this group
    const int nrb = (R + DEC_ROWS - 1) / DEC_ROWS; // row blocks
    const int bz = (int)blockIdx.z;
    const int bb = bz / nrb, rb = bz - bb * nrb;
    const int L = cache_lengths[bb];
    const int n_chunks = gridDim.x;
    const int c0 = chunk * DEC_KEYS;
    if (L < T_q || L > T_max) {
        if (tid == 0 && chunk == 0 && g == 0 && rb == 0) record_status(status, kStatusBadLength);
        return;  // the merge writes NaN rows
    }
    if (c0 >= L) return;  // the merge skips chunks past the cache length

    // query rows of this block: local row r -> (query head, new token)
    for (int i = tid; i < DEC_ROWS * HD; i += DEC_THREADS) {
        const int r = i / HD, e = i - r * HD;
        const int rr = rb * DEC_ROWS + r;
        float v = 0.f;
        if (rr < R) {
            const int head = g * per + rr / T_q, t = rr - (rr / T_q) * T_q;
            v = __bfloat162float(Q[((int64_t)bb * T_q + t) * ldq + (int64_t)head * HD + e]) * scale_log2;
        }
        q_s[r][e] = v;
    }
    // this chunk's values, 16-byte pieces
    for (int i = tid; i < DEC_KEYS * (HD / 8); i += DEC_THREADS) {
        const int j = i / (HD / 8), e8 = i - j * (HD / 8);
        const int key = c0 + j;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (key < L) w = __ldg(reinterpret_cast<const uint4*>(Vc + ((int64_t)bb * T_max + key) * ldv + (int64_t)g * HD) + e8);
        *reinterpret_cast<uint4*>(&v_s[j][e8 * 8]) = w;
    }
    __syncthreads();

    // scores: thread = cached key
    const int key = c0 + tid;
    float s[DEC_ROWS];
#pragma unroll
    for (int r = 0; r < DEC_ROWS; ++r) s[r] = 0.f;
    if (key < L) {
        const uint4* kp = reinterpret_cast<const uint4*>(Kc + ((int64_t)bb * T_max + key) * ldk + (int64_t)g * HD);
#pragma unroll
        for (int e8 = 0; e8 < HD / 8; ++e8) {
            float kf[8];
            bf16x8_to_f32(__ldg(kp + e8), kf);
#pragma unroll
            for (int r = 0; r < DEC_ROWS; ++r) {
                const float4 qa = *reinterpret_cast<const float4*>(&q_s[r][e8 * 8]);
                const float4 qb = *reinterpret_cast<const float4*>(&q_s[r][e8 * 8 + 4]);
                s[r] = fmaf(qa.x, kf[0], s[r]);
                s[r] = fmaf(qa.y, kf[1], s[r]);
                s[r] = fmaf(qa.z, kf[2], s[r]);
                s[r] = fmaf(qa.w, kf[3], s[r]);
                s[r] = fmaf(qb.x, kf[4], s[r]);
                s[r] = fmaf(qb.y, kf[5], s[r]);
                s[r] = fmaf(qb.z, kf[6], s[r]);
                s[r] = fmaf(qb.w, kf[7], s[r]);
            }
        }
    }
    // visibility: row (head, t) sees keys j <= L - T_q + t
#pragma unroll
    for (int r = 0; r < DEC_ROWS; ++r) {
        const int rr = rb * DEC_ROWS + r;
        const int t = rr - (rr / T_q) * T_q;
        if (rr >= R || key >= L - T_q + t + 1) s[r] = -INFINITY;
    }
    // per-row maximum over the chunk
#pragma unroll
    for (int r = 0; r < DEC_ROWS; ++r) {
        float mx = s[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        if (lane == 0) red_s[warp][r] = mx;
    }
    __syncthreads();
    if (tid < DEC_ROWS) {
        float mx = red_s[0][tid];
#pragma unroll
        for (int w = 1; w < DEC_THREADS / 32; ++w) mx = fmaxf(mx, red_s[w][tid]);
        m_s[tid] = mx;
    }
    __syncthreads();
    // 2^(s - m) and its per-row sum
#pragma unroll
    for (int r = 0; r < DEC_ROWS; ++r) {
        const float m = m_s[r];
        const float p = m == -INFINITY ? 0.f : ex2_approx(s[r] - m);
        p_s[r][tid] = p;
        float sum = p;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (lane == 0) red_s[warp][r] = sum;
    }
    __syncthreads();
    if (tid < DEC_ROWS) {
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < DEC_THREADS / 32; ++w) sum += red_s[w][tid];
        l_s[tid] = sum;
    }
    // weighted values: thread = (output column, group of rows)
    constexpr int RPT = DEC_ROWS * HD / DEC_THREADS;  // rows per thread
    const int e = tid % HD, r0 = (tid / HD) * RPT;
    float o[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) o[i] = 0.f;
    for (int j = 0; j < DEC_KEYS; ++j) {
        const float v = __bfloat162float(v_s[j][e]);
#pragma unroll
        for (int i = 0; i < RPT; ++i) o[i] = fmaf(p_s[r0 + i][j], v, o[i]);
    }
    __syncthreads();
    // partials of the rows that exist: part[((b*h + head)*T_q + t)*n_chunks + chunk]
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = r0 + i, rr = rb * DEC_ROWS + r;
        if (rr >= R) continue;
        const int head = g * per + rr / T_q, t = rr - (rr / T_q) * T_q;
        float* pp = part + ((((int64_t)bb * h + head) * T_q + t) * n_chunks + chunk) * dec_partial_floats(HD);
        pp[2 + e] = o[i];
        if (e == 0) {
            pp[0] = m_s[r];
            pp[1] = l_s[r];
        }
    }
}

// Merge of the chunk partials of one row: thread = output column.
template <int HD>
__global__ void __launch_bounds__(HD)
    decode_merge_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ O, int64_t ldo,
                        int h, int T_q, int T_max, int n_chunks,
                        const int32_t* __restrict__ cache_lengths) {
    grid_dependency_wait();  // the partials come from the previous kernel
    grid_launch_dependents();
    const int row = blockIdx.x;  // (b * h + head) * T_q + t
    const int t = row % T_q, bh = row / T_q;
    const int b = bh / h, head = bh - b * h;
    const int e = threadIdx.x;
    const int L = cache_lengths[b];
    __nv_bfloat16* out = O + ((int64_t)b * T_q + t) * ldo + (int64_t)head * HD + e;
    if (L < T_q || L > T_max) {
        *out = __float2bfloat16_rn(NAN);
        return;
    }
    const int nc = (L + DEC_KEYS - 1) / DEC_KEYS;  // chunks holding keys of this batch
    const float* pp = part + (int64_t)row * n_chunks * dec_partial_floats(HD);
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, pp[c * dec_partial_floats(HD)]);
    float l = 0.f, o = 0.f;
    for (int c = 0; c < nc; ++c) {
        const float* q = pp + c * dec_partial_floats(HD);
        const float w = q[0] == -INFINITY ? 0.f : ex2_approx(q[0] - M);
        l = fmaf(w, q[1], l);
        o = fmaf(w, q[2 + e], o);
    }
    *out = __float2bfloat16_rn(o / l);
}

template <int HD>
cudaError_t launch_decode_hd(const void* Q, int64_t ldq, const void* Kc, int64_t ldk, const void* Vc,
                             int64_t ldv, void* O, int64_t ldo, int B, int h, int h_kv, int T_q,
                             int T_max, const int32_t* cache_lengths, void* ws, int* status,
                             cudaStream_t stream) {
    const int n_chunks = dec_chunks(T_max);
    const int R = (h / h_kv) * T_q;
    const int nrb = (R + DEC_ROWS - 1) / DEC_ROWS;
    if ((int64_t)B * nrb > 65535 || h_kv > 65535) return cudaErrorInvalidValue;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    float* part = static_cast<float*>(ws);
    cudaError_t err = launch_pdl(decode_partial_kernel<HD>, dim3(n_chunks, h_kv, B * nrb),
                                 dim3(DEC_THREADS), 0, stream,
                                 reinterpret_cast<const __nv_bfloat16*>(Q), ldq,
                                 reinterpret_cast<const __nv_bfloat16*>(Kc), ldk,
                                 reinterpret_cast<const __nv_bfloat16*>(Vc), ldv, h, h_kv, T_q, T_max,
                                 cache_lengths, scale_log2, part, status);
    if (err != cudaSuccess) return err;
    return launch_pdl(decode_merge_kernel<HD>, dim3(B * h * T_q), dim3(HD), 0, stream,
                      static_cast<const float*>(part), reinterpret_cast<__nv_bfloat16*>(O), ldo, h, T_q,
                      T_max, n_chunks, cache_lengths);
}

}  // namespace

size_t decode_workspace_bytes(int B, int h, int T_q, int d, int T_max) {
    return sizeof(float) * (size_t)B * h * T_q * dec_chunks(T_max) * dec_partial_floats(d);
}

cudaError_t launch_decode_bf16(const void* Q, int64_t ldq, const void* Kc, int64_t ldk,
                               const void* Vc, int64_t ldv, void* O, int64_t ldo, int B, int h,
                               int h_kv, int T_q, int T_max, int d, const int32_t* cache_lengths,
                               void* ws, int num_sms, int* status, cudaStream_t stream) {
    (void)num_sms;
    if (d == 64)
        return launch_decode_hd<64>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                    cache_lengths, ws, status, stream);
    if (d == 128)
        return launch_decode_hd<128>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                     cache_lengths, ws, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mha
