// decode_bf16.cu -- one decode step over a key/value cache (itwiki.kr "멀티 헤드 어텐션",
// section 추론 비용과 변형: the keys and values of earlier tokens are kept in a KV cache and
// every generation step reads the whole cache, so the step is bound by memory bandwidth; with
// grouped K/V heads (MQA/GQA) h / h_kv query heads share each cached head).
//
// The T_q new tokens of batch b are the last T_q of its L_b cached tokens: new token t (row
// t) sees cache entries j <= L_b - T_q + t.  For cached K/V head g the query rows are the
// (query head, new token) pairs of its group, R = (h / h_kv) * T_q of them.
//
// Split over the cache (flash-decoding): CTA (split, g, b, row block) streams a span of the
// cached keys and values of head g through shared memory once and, for its query rows,
// computes the softmax statistics of its span -- the maximum m, the sum l of 2^(s - m) and
// the weighted value sum o -- and writes them to the workspace; a second kernel merges the
// spans of each row: M = max m_c, O = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c.  Scores
// are kept in base 2 with log2(e)/sqrt(d) folded into the query.  The cache is bf16, all
// arithmetic fp32, on CUDA cores: the step is bound by the cache reads, not by arithmetic.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int DEC_TK = 64;        // cached keys per tile
constexpr int DEC_THREADS = 128;

// Workspace: partials [B][h][T_q][split] of (m, l, o[d]) floats.
__host__ __device__ constexpr int dec_partial_floats(int d) { return d + 2; }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    // 16 bytes global -> shared; a key past the cache length is filled with zeros instead
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float (&f)[8]) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}

// CTA (split, g, b * row blocks): keys [split * span, (split + 1) * span) of cached head g,
// ROWS query rows (R = (h / h_kv) * T_q rows per group, split into row blocks).  K and V
// tiles of DEC_TK keys stream through a double-buffered shared-memory ring (cp.async, rows
// padded to HD + 8 elements so that the per-key reads do not collide in one bank); the
// softmax over the split is online (running maximum and sum per row, base 2).
template <int HD, int ROWS>
__global__ void __launch_bounds__(DEC_THREADS)
    decode_partial_kernel(const __nv_bfloat16* __restrict__ Q, int64_t ldq,
                          const __nv_bfloat16* __restrict__ Kc, int64_t ldk,
                          const __nv_bfloat16* __restrict__ Vc, int64_t ldv, int h, int h_kv,
                          int T_q, int T_max, int span, const int32_t* __restrict__ cache_lengths,
                          float scale_log2, float* __restrict__ part, int* status) {
    constexpr int LD = HD + 8;                       // padded row (elements)
    constexpr int TILE = DEC_TK * LD;                // elements per K or V tile
    constexpr int CH = HD / 8;                       // 16-byte chunks per row
    extern __shared__ __align__(16) uint8_t dsm[];
    __nv_bfloat16* kv_s = reinterpret_cast<__nv_bfloat16*>(dsm);   // [2 buffers][K, V][TILE]
    float* q_s = reinterpret_cast<float*>(dsm + 2 * 2 * TILE * 2);   // [ROWS][HD]
    float* s_s = q_s + ROWS * HD;                                    // [ROWS][DEC_TK]
    float* m_s = s_s + ROWS * DEC_TK;                                // running max [ROWS]
    float* l_s = m_s + ROWS;                                         // running sum [ROWS]
    float* a_s = l_s + ROWS;                                         // rescale of this tile

    grid_dependency_wait();  // Q and the cache may come from the previous kernel
    grid_launch_dependents();

    const int split = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x;
    const int per = h / h_kv;
    const int R = per * T_q;
    const int nrb = (R + ROWS - 1) / ROWS;
    const int bb = (int)blockIdx.z / nrb, rb = (int)blockIdx.z - bb * nrb;
    const int L = cache_lengths[bb];
    if (L < T_q || L > T_max) {
        if (tid == 0 && split == 0 && g == 0 && rb == 0) record_status(status, kStatusBadLength);
        return;  // the merge writes NaN rows
    }
    const int k0 = split * span;
    const int k1 = min(L, k0 + span);
    if (k0 >= k1) return;  // the merge skips splits past the cache length
    const int n_tiles = (k1 - k0 + DEC_TK - 1) / DEC_TK;

    const uint32_t kv_base = smem_u32(kv_s);
    auto load_tile = [&](int t, int buf) {
        const int kt = k0 + t * DEC_TK;
#pragma unroll
        for (int i = tid; i < DEC_TK * CH; i += DEC_THREADS) {
            const int j = i / CH, c = i - j * CH;
            const int key = kt + j;
            const bool ok = key < k1;
            const int64_t krow = ((int64_t)bb * T_max + (ok ? key : k0)) ;
            const uint32_t off = (uint32_t)((j * LD + c * 8) * 2);
            cp_async16(kv_base + (uint32_t)(buf * 2 * TILE * 2) + off, Kc + krow * ldk + (int64_t)g * HD + c * 8, ok);
            cp_async16(kv_base + (uint32_t)((buf * 2 + 1) * TILE * 2) + off, Vc + krow * ldv + (int64_t)g * HD + c * 8, ok);
        }
        cp_async_commit();
    };
    load_tile(0, 0);

    // query rows (pre-scaled to base 2): local row r -> (query head, new token)
    for (int i = tid; i < ROWS * HD; i += DEC_THREADS) {
        const int r = i / HD, e = i - r * HD;
        const int rr = rb * ROWS + r;
        float v = 0.f;
        if (rr < R) {
            const int head = g * per + rr / T_q, t = rr - (rr / T_q) * T_q;
            v = __bfloat162float(Q[((int64_t)bb * T_q + t) * ldq + (int64_t)head * HD + e]) * scale_log2;
        }
        q_s[i] = v;
    }
    if (tid < ROWS) {
        m_s[tid] = -INFINITY;
        l_s[tid] = 0.f;
    }
    // row -> last visible key + 1, for the rows this block holds
    auto row_end = [&](int r) -> int {
        const int rr = rb * ROWS + r;
        if (rr >= R) return -1;
        const int t = rr - (rr / T_q) * T_q;
        return L - T_q + t + 1;
    };

    // PV mapping: thread = (output column, group of rows)
    constexpr int TPR = DEC_THREADS / HD > 0 ? DEC_THREADS / HD : 1;  // threads per column
    constexpr int RPT = (ROWS + TPR - 1) / TPR;                         // rows per thread
    const int e_col = tid % HD, r_base = (tid / HD) * RPT;
    float o[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) o[i] = 0.f;

    for (int t = 0; t < n_tiles; ++t) {
        const int buf = t & 1;
        if (t + 1 < n_tiles) {
            load_tile(t + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const __nv_bfloat16* k_s = kv_s + buf * 2 * TILE;
        const __nv_bfloat16* v_s = k_s + TILE;
        const int kt = k0 + t * DEC_TK;
        // scores: two adjacent lanes per key, each half of the head dimension
        {
            const int j = tid >> 1, half = tid & 1;
            float sc[ROWS];
#pragma unroll
            for (int r = 0; r < ROWS; ++r) sc[r] = 0.f;
            const uint4* kp = reinterpret_cast<const uint4*>(k_s + j * LD + half * (HD / 2));
#pragma unroll
            for (int c = 0; c < HD / 16; ++c) {
                float kf[8];
                bf16x8_to_f32(kp[c], kf);
#pragma unroll
                for (int r = 0; r < ROWS; ++r) {
                    const float* qr = q_s + r * HD + half * (HD / 2) + c * 8;
                    const float4 qa = *reinterpret_cast<const float4*>(qr);
                    const float4 qb = *reinterpret_cast<const float4*>(qr + 4);
                    sc[r] = fmaf(qa.x, kf[0], sc[r]);
                    sc[r] = fmaf(qa.y, kf[1], sc[r]);
                    sc[r] = fmaf(qa.z, kf[2], sc[r]);
                    sc[r] = fmaf(qa.w, kf[3], sc[r]);
                    sc[r] = fmaf(qb.x, kf[4], sc[r]);
                    sc[r] = fmaf(qb.y, kf[5], sc[r]);
                    sc[r] = fmaf(qb.z, kf[6], sc[r]);
                    sc[r] = fmaf(qb.w, kf[7], sc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < ROWS; ++r) {
                const float full = sc[r] + __shfl_xor_sync(0xffffffffu, sc[r], 1);
                if (half == 0) s_s[r * DEC_TK + j] = kt + j < row_end(r) ? full : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax per row: 128 / ROWS threads per row (a power of two, <= 32)
        {
            constexpr int TPROW = DEC_THREADS / ROWS < 32 ? DEC_THREADS / ROWS : 32;
            constexpr int KPT = DEC_TK / TPROW;  // keys per thread
            const int r = tid / TPROW, sub = tid - r * TPROW;
            if (r < ROWS) {
                float* sr = s_s + r * DEC_TK + sub * KPT;
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < KPT; ++i) mx = fmaxf(mx, sr[i]);
#pragma unroll
                for (int off = TPROW / 2; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off, TPROW));
                const float m_old = m_s[r];
                const float m_new = fmaxf(m_old, mx);
                float sum = 0.f;
#pragma unroll
                for (int i = 0; i < KPT; ++i) {
                    const float p = m_new == -INFINITY ? 0.f : ex2_approx(sr[i] - m_new);
                    sr[i] = p;
                    sum += p;
                }
#pragma unroll
                for (int off = TPROW / 2; off > 0; off >>= 1)
                    sum += __shfl_xor_sync(0xffffffffu, sum, off, TPROW);
                __syncwarp();
                if (sub == 0) {
                    const float a = m_new == -INFINITY ? 1.f : ex2_approx(m_old - m_new);
                    a_s[r] = a;
                    l_s[r] = l_s[r] * a + sum;
                    m_s[r] = m_new;
                }
            }
        }
        __syncthreads();
        // weighted values
#pragma unroll
        for (int i = 0; i < RPT; ++i)
            if (r_base + i < ROWS) o[i] *= a_s[r_base + i];
        for (int j = 0; j < DEC_TK; ++j) {
            const float v = __bfloat162float(v_s[j * LD + e_col]);
#pragma unroll
            for (int i = 0; i < RPT; ++i)
                if (r_base + i < ROWS) o[i] = fmaf(s_s[(r_base + i) * DEC_TK + j], v, o[i]);
        }
        __syncthreads();  // the buffer of tile t is reloaded by the next iteration's prefetch
    }
    // partials of the rows that exist
    const int n_splits = gridDim.x;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = r_base + i, rr = rb * ROWS + r;
        if (r >= ROWS || rr >= R) continue;
        const int head = g * per + rr / T_q, t = rr - (rr / T_q) * T_q;
        float* pp = part + ((((int64_t)bb * h + head) * T_q + t) * n_splits + split) * dec_partial_floats(HD);
        pp[2 + e_col] = o[i];
        if (e_col == 0) {
            pp[0] = m_s[r];
            pp[1] = l_s[r];
        }
    }
}

// Merge of the split partials of one row: thread = output column.
template <int HD>
__global__ void __launch_bounds__(HD)
    decode_merge_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ O, int64_t ldo,
                        int h, int T_q, int T_max, int n_splits, int span,
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
    const int ns = (L + span - 1) / span;  // splits holding keys of this batch
    const float* pp = part + (int64_t)row * n_splits * dec_partial_floats(HD);
    float M = -INFINITY;
    for (int c = 0; c < ns; ++c) M = fmaxf(M, pp[c * dec_partial_floats(HD)]);
    float l = 0.f, o = 0.f;
    for (int c = 0; c < ns; ++c) {
        const float* q = pp + c * dec_partial_floats(HD);
        const float w = q[0] == -INFINITY ? 0.f : ex2_approx(q[0] - M);
        l = fmaf(w, q[1], l);
        o = fmaf(w, q[2 + e], o);
    }
    *out = __float2bfloat16_rn(o / l);
}

// Keys per CTA: enough CTAs to fill the GPU a few times over, at least 4 tiles per CTA.
int decode_span(int B, int h_kv, int nrb, int T_max, int num_sms) {
    const int64_t groups = (int64_t)B * h_kv * nrb;
    const int64_t target = 4LL * (num_sms > 0 ? num_sms : 148);
    int64_t splits = (target + groups - 1) / groups;
    const int64_t max_splits = (T_max + 4 * DEC_TK - 1) / (4 * DEC_TK);
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t span = (T_max + splits - 1) / splits;
    span = (span + DEC_TK - 1) / DEC_TK * DEC_TK;
    return (int)span;
}

template <int HD, int ROWS>
size_t decode_smem() {
    return (size_t)2 * 2 * DEC_TK * (HD + 8) * 2 + sizeof(float) * ((size_t)ROWS * HD + (size_t)ROWS * DEC_TK + 3 * ROWS);
}

template <int HD, int ROWS>
cudaError_t launch_decode_rows(const void* Q, int64_t ldq, const void* Kc, int64_t ldk, const void* Vc,
                               int64_t ldv, void* O, int64_t ldo, int B, int h, int h_kv, int T_q,
                               int T_max, const int32_t* cache_lengths, void* ws, int num_sms,
                               int* status, cudaStream_t stream) {
    const int R = (h / h_kv) * T_q;
    const int nrb = (R + ROWS - 1) / ROWS;
    if ((int64_t)B * nrb > 65535 || h_kv > 65535) return cudaErrorInvalidValue;
    const int span = decode_span(B, h_kv, nrb, T_max, num_sms);
    const int n_splits = (T_max + span - 1) / span;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    const size_t smem = decode_smem<HD, ROWS>();
    cudaError_t err = cudaFuncSetAttribute(decode_partial_kernel<HD, ROWS>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    float* part = static_cast<float*>(ws);
    err = launch_pdl(decode_partial_kernel<HD, ROWS>, dim3(n_splits, h_kv, B * nrb), dim3(DEC_THREADS), smem,
                     stream, reinterpret_cast<const __nv_bfloat16*>(Q), ldq,
                     reinterpret_cast<const __nv_bfloat16*>(Kc), ldk,
                     reinterpret_cast<const __nv_bfloat16*>(Vc), ldv, h, h_kv, T_q, T_max, span,
                     cache_lengths, scale_log2, part, status);
    if (err != cudaSuccess) return err;
    return launch_pdl(decode_merge_kernel<HD>, dim3(B * h * T_q), dim3(HD), 0, stream,
                      static_cast<const float*>(part), reinterpret_cast<__nv_bfloat16*>(O), ldo, h, T_q,
                      T_max, n_splits, span, cache_lengths);
}

template <int HD>
cudaError_t launch_decode_hd(const void* Q, int64_t ldq, const void* Kc, int64_t ldk, const void* Vc,
                             int64_t ldv, void* O, int64_t ldo, int B, int h, int h_kv, int T_q,
                             int T_max, const int32_t* cache_lengths, void* ws, int num_sms, int* status,
                             cudaStream_t stream) {
    // query rows per K/V head: one for plain multi-head attention at one new token, more
    // for grouped heads or several new tokens
    const int R = (h / h_kv) * T_q;
    if (R <= 1)
        return launch_decode_rows<HD, 1>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                         cache_lengths, ws, num_sms, status, stream);
    if (R <= 4)
        return launch_decode_rows<HD, 4>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                         cache_lengths, ws, num_sms, status, stream);
    return launch_decode_rows<HD, 16>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                      cache_lengths, ws, num_sms, status, stream);
}

}  // namespace

// The partials hold one record per split; splits are at least 4 key tiles long, so
// T_max / (4 * 64) + 1 records per row bound the count for every launch configuration.
size_t decode_workspace_bytes(int B, int h, int T_q, int d, int T_max) {
    const size_t max_splits = (size_t)(T_max + 4 * DEC_TK - 1) / (4 * DEC_TK);
    return sizeof(float) * (size_t)B * h * T_q * max_splits * dec_partial_floats(d);
}

cudaError_t launch_decode_bf16(const void* Q, int64_t ldq, const void* Kc, int64_t ldk,
                               const void* Vc, int64_t ldv, void* O, int64_t ldo, int B, int h,
                               int h_kv, int T_q, int T_max, int d, const int32_t* cache_lengths,
                               void* ws, int num_sms, int* status, cudaStream_t stream) {
    if (d == 64)
        return launch_decode_hd<64>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                    cache_lengths, ws, num_sms, status, stream);
    if (d == 128)
        return launch_decode_hd<128>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                     cache_lengths, ws, num_sms, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mha
