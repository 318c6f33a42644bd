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
// are kept in base 2 with log2(e)/sqrt(d) folded in.  The cache is bf16, accumulation fp32.
// One query row per cached head (plain multi-head attention, one new token) runs on CUDA
// cores, bound by the cache reads; grouped heads or several new tokens put R >= 2 rows on
// each cached head, and those run on the tensor core (decode_tc_kernel below).
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

// ---------------------------------------------------------------------------------------
// Grouped heads (R = (h / h_kv) * T_q >= 2 query rows per cached head) on tcgen05: the R rows
// of head group g form one 128-row query tile (rows past R are zero), so every cached key and
// value is read once for the whole group and the score and weighted-value products run on the
// tensor core (S = Q K^T and O += P V with the accumulators in TMEM), leaving the CUDA cores
// only the softmax.  CTA (split, g, b * row blocks) streams its span of the cache in 128-key
// tiles through a TMA ring and writes the same per-split partials (m, l, o) as the CUDA-core
// kernel above, merged by decode_merge_kernel.
//
// Warp roles (256 threads): warp 0 TMA (K and V tiles), warp 1 TMEM owner and MMA issuer
// (S(i+1) as soon as the softmax has read S(i), then O += P(i) V(i)), warps 4-7 softmax (one
// query row per thread; warps whose 32 rows are all padding stay idle).
template <int HD>
struct DtcCfg {
    static constexpr int CH = HD / 64;                   // 64-column chunks of a row
    static constexpr int CHUNK = 128 * 128;              // 128 rows x 64 bf16 = 16 KB
    static constexpr int TILE = CH * CHUNK;              // one Q, K or V tile
    static constexpr int STAGES = 2;
    static constexpr int SMEM = TILE + 2 * STAGES * TILE + 256 + 1024;
    static constexpr uint32_t TMEM_COLS = HD == 64 ? 256 : 512;
    static constexpr uint32_t S_COL = 0, O_COL = 128, P_COL = 128 + HD;
};
static_assert(DtcCfg<128>::SMEM <= 232448, "decode smem budget");
constexpr int DTC_THREADS = 256;
constexpr int DTC_TK = 128;  // keys per tile

template <int HD>
__global__ void __launch_bounds__(DTC_THREADS, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __nv_bfloat16* __restrict__ Q, int64_t ldq, int h, int h_kv, int T_q,
                     int T_max, int span, const int32_t* __restrict__ cache_lengths, float scale_log2,
                     float* __restrict__ part, int* status) {
    using C = DtcCfg<HD>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base;
    const uint32_t sK = sQ + C::TILE;
    const uint32_t sV = sK + S * C::TILE;
    const uint32_t sBar = sV + S * C::TILE;
    // barriers: k_full[S], k_empty[S], v_full[S], v_empty[S], s_full, s_free, p_full, pv_done, drain
    const uint32_t bar_kfull = sBar;
    const uint32_t bar_kempty = bar_kfull + 8u * S;
    const uint32_t bar_vfull = bar_kempty + 8u * S;
    const uint32_t bar_vempty = bar_vfull + 8u * S;
    const uint32_t bar_sfull = bar_vempty + 8u * S;
    const uint32_t bar_sfree = bar_sfull + 8u;
    const uint32_t bar_pfull = bar_sfree + 8u;
    const uint32_t bar_pvdone = bar_pfull + 8u;
    const uint32_t bar_drain = bar_pvdone + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    grid_dependency_wait();  // Q and the cache may come from the previous kernel
    grid_launch_dependents();

    const int split = blockIdx.x, g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int per = h / h_kv;
    const int R = per * T_q;
    const int nrb = (R + 127) / 128;
    const int bb = (int)blockIdx.z / nrb, rb = (int)blockIdx.z - bb * nrb;
    const int L = cache_lengths[bb];
    if (L < T_q || L > T_max) {
        if (threadIdx.x == 0 && split == 0 && g == 0 && rb == 0) record_status(status, kStatusBadLength);
        return;  // the merge writes NaN rows
    }
    const int k0 = split * span;
    const int k1 = min(L, k0 + span);
    if (k0 >= k1) return;  // the merge skips splits past the cache length
    const int n_tiles = (k1 - k0 + DTC_TK - 1) / DTC_TK;
    const int rows = min(128, R - rb * 128);      // real query rows of this block
    const int arrivals = 32 * ((rows + 31) / 32);  // threads of the softmax warps holding them

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_kfull + 8u * s, 1);
            mbar_init(bar_kempty + 8u * s, 1);
            mbar_init(bar_vfull + 8u * s, 1);
            mbar_init(bar_vempty + 8u * s, 1);
        }
        mbar_init(bar_sfull, 1);
        mbar_init(bar_sfree, arrivals);
        mbar_init(bar_pfull, arrivals);
        mbar_init(bar_pvdone, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    // the query tile: local row r = (query head g * per + r / T_q, new token r % T_q), 128-byte
    // swizzled like a TMA box; rows past R are zero
    for (int i = threadIdx.x; i < 128 * C::CH * 8; i += DTC_THREADS) {
        const int r = i / (C::CH * 8), cu = i - r * (C::CH * 8), c = cu >> 3, u = cu & 7;
        const int rr = rb * 128 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (rr < R) {
            const int head = g * per + rr / T_q, t = rr - (rr / T_q) * T_q;
            v = *reinterpret_cast<const uint4*>(Q + ((int64_t)bb * T_q + t) * ldq + (int64_t)head * HD + c * 64 + u * 8);
        }
        st_shared_v4(sQ + (uint32_t)(c * C::CHUNK + r * 128) + ((uint32_t)(u ^ (r & 7)) << 4), v.x, v.y, v.z, v.w);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA: K and V tiles of the span
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int nk = 0, nv = 0;  // K, V tiles issued
            for (int i = 0; i < n_tiles; ++i) {
                const uint32_t st = (uint32_t)(i % S), ph = ((uint32_t)(i / S) & 1u) ^ 1u;
                const int key0 = k0 + i * DTC_TK;
                if (!mbar_wait(bar_kempty + 8u * st, ph, abort_flag, status)) break;
                mbar_arrive_expect_tx(bar_kfull + 8u * st, C::TILE);
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sK + st * C::TILE + c * C::CHUNK, &tmK, g * HD + c * 64, key0, bb, bar_kfull + 8u * st);
                ++nk;
                if (!mbar_wait(bar_vempty + 8u * st, ph, abort_flag, status)) break;
                mbar_arrive_expect_tx(bar_vfull + 8u * st, C::TILE);
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sV + st * C::TILE + c * C::CHUNK, &tmV, g * HD + c * 64, key0, bb, bar_vfull + 8u * st);
                ++nv;
            }
            // every load issued lands before the CTA exits
            for (int i = nk > S ? nk - S : 0; i < nk; ++i)
                drain_wait_a(bar_kfull + 8u * (uint32_t)(i % S), (uint32_t)(i / S) & 1u);
            for (int i = nv > S ? nv - S : 0; i < nv; ++i)
                drain_wait_a(bar_vfull + 8u * (uint32_t)(i % S), (uint32_t)(i / S) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc_s = idesc_bf16_f32(128, DTC_TK, false, false);
            const uint32_t idesc_o = idesc_bf16_f32(128, HD, false, true);
            const uint64_t qdesc = sdesc_sw128(sQ, 16, 1024);
            const uint64_t kdesc0 = sdesc_sw128(sK, 16, 1024);
            const uint64_t vdesc0 = sdesc_sw128(sV, C::CHUNK, 1024);
            auto issue_s = [&](int i) -> bool {
                const uint32_t st = (uint32_t)(i % S);
                if (!mbar_wait(bar_kfull + 8u * st, (uint32_t)(i / S) & 1u, abort_flag, status)) return false;
                if (i > 0 && !mbar_wait(bar_sfree, (uint32_t)(i - 1) & 1u, abort_flag, status)) return false;
                tc_fence_after();
                const uint64_t kdesc = kdesc0 + (uint64_t)((st * C::TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off16 = (uint32_t)(((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(tmem_base + C::S_COL, qdesc + off16, kdesc + off16, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar_sfull);
                tc_commit(bar_kempty + 8u * st);
                return true;
            };
            bool ok = issue_s(0);
            for (int i = 0; i < n_tiles && ok; ++i) {
                if (i + 1 < n_tiles) ok = issue_s(i + 1);
                if (!ok) break;
                const uint32_t st = (uint32_t)(i % S);
                ok = mbar_wait(bar_vfull + 8u * st, (uint32_t)(i / S) & 1u, abort_flag, status) &&
                     mbar_wait(bar_pfull, (uint32_t)i & 1u, abort_flag, status);
                if (!ok) break;
                tc_fence_after();
                const uint64_t vdesc = vdesc0 + (uint64_t)((st * C::TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < DTC_TK / 16; ++kk)
                    mma_bf16_ts(tmem_base + C::O_COL, tmem_base + C::P_COL + kk * 8,
                                vdesc + (uint64_t)((kk * 2048) >> 4), idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar_pvdone);
                tc_commit(bar_vempty + 8u * st);
            }
            tc_commit(bar_drain);
            drain_wait_a(bar_drain, 0);
        }
    } else if (warp >= 4 && (warp - 4) * 32 < rows) {
        // ---------------- softmax: thread = query row
        const int r = (warp & 3) * 32 + lane;
        const uint32_t trow = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
        const int rr = rb * 128 + r;
        const bool real = r < rows;
        const int t = real ? rr - (rr / T_q) * T_q : 0;
        const int lim = real ? min(k1, L - T_q + t + 1) : k0;  // keys [k0, lim) are visible
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull, (uint32_t)i & 1u, abort_flag, status))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int key0 = k0 + i * DTC_TK;
            float x[128];
            {
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(trow + C::S_COL + c * 32, sr[c]);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    x[c] = key0 + c < lim ? __uint_as_float(sr[c >> 5][c & 31]) : -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(bar_sfree);
            // base-2 online softmax; the reference moves only when P would otherwise exceed 2^32
            const float m_tile = row_max(x) * scale_log2;
            const float m_new = m_tile > m + 32.0f ? m_tile : m;
            // 0 when m leaves -inf; 1 while a row has seen no visible key of the split
            const float alpha = m_new == -INFINITY ? 1.f : ex2_approx(m - m_new);
            uint32_t pk[64];
            const float rowsum = exp_tile(x, pack2(scale_log2, scale_log2), m_new == -INFINITY ? 0.f : -m_new, pk);
            if (i > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(bar_pvdone, (uint32_t)(i - 1) & 1u, abort_flag, status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool rescale = m_new != m;
                if (__any_sync(0xffffffffu, rescale)) {
                    const float a = rescale ? alpha : 1.f;
#pragma unroll
                    for (int cc = 0; cc < HD / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(trow + C::O_COL + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * a);
                        tmem_st32(trow + C::O_COL + cc * 32, o);
                    }
                }
            }
            {
                uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
                uint32_t (&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
                tmem_st32(trow + C::P_COL, p0);
                tmem_st32(trow + C::P_COL + 32, p1);
            }
            // cached rows at or past L may hold anything: zero the V rows the PV product would
            // multiply by P = 0 (a NaN there would survive the product)
            if (key0 + DTC_TK > L) {
                const uint32_t st = (uint32_t)(i % S);
                if (!__all_sync(0xffffffffu, mbar_wait(bar_vfull + 8u * st, (uint32_t)(i / S) & 1u, abort_flag, status))) {
                    ok = false;
                    break;
                }
                const int first = L - key0;  // first row to clear
                for (int z = (warp - 4) * 32 + lane; z < (DTC_TK - first) * C::CH * 8; z += arrivals) {
                    const int row = first + z / (C::CH * 8), cu = z - (z / (C::CH * 8)) * (C::CH * 8);
                    st_shared_v4(sV + st * C::TILE + (uint32_t)((cu >> 3) * C::CHUNK + row * 128 + ((cu & 7) << 4)),
                                 0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar_pfull);
            l = l * alpha + rowsum;
            m = m_new;
        }
        if (ok && __all_sync(0xffffffffu, mbar_wait(bar_pvdone, (uint32_t)(n_tiles - 1) & 1u, abort_flag, status))) {
            tc_fence_after();
            // this split's partial for the row: reference maximum, sum and weighted values
            float* pp = nullptr;
            if (real) {
                const int head = g * per + rr / T_q;
                pp = part + ((((int64_t)bb * h + head) * T_q + t) * gridDim.x + split) * dec_partial_floats(HD);
                pp[0] = m;
                pp[1] = l;
            }
#pragma unroll
            for (int cc = 0; cc < HD / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32(trow + C::O_COL + cc * 32, o);
                tmem_wait_ld();
                if (real) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) pp[2 + cc * 32 + e] = __uint_as_float(o[e]);
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// Keys per CTA for the tensor-core kernel: the split count that minimises (waves of CTAs over
// the resident slots) x (128-key tiles per CTA + a fixed cost of about three tiles for the
// CTA's set-up: query gather, TMEM allocation, pipeline fill, partial record), splits at
// least two tiles long.
int decode_span_tc(int B, int h_kv, int nrb, int T_max, int num_sms, int ctas_per_sm) {
    const int64_t groups = (int64_t)B * h_kv * nrb;
    const int64_t slots = (int64_t)(num_sms > 0 ? num_sms : 148) * ctas_per_sm;
    const int64_t max_splits = (T_max + 2 * DTC_TK - 1) / (2 * DTC_TK);
    int64_t best_span = 0, best_cost = -1;
    for (int64_t s = 1; s <= max_splits; ++s) {
        const int64_t span = ((T_max + s - 1) / s + DTC_TK - 1) / DTC_TK * DTC_TK;
        const int64_t splits = (T_max + span - 1) / span;
        const int64_t waves = (groups * splits + slots - 1) / slots;
        const int64_t cost = waves * (span / DTC_TK + 3);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_span = span;
        }
    }
    return (int)best_span;
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
cudaError_t launch_decode_tc(const void* Q, int64_t ldq, const void* Kc, int64_t ldk, const void* Vc,
                             int64_t ldv, void* O, int64_t ldo, int B, int h, int h_kv, int T_q,
                             int T_max, const int32_t* cache_lengths, void* ws, int num_sms, int* status,
                             cudaStream_t stream) {
    using C = DtcCfg<HD>;
    const int R = (h / h_kv) * T_q;
    const int nrb = (R + 127) / 128;
    if ((int64_t)B * nrb > 65535 || h_kv > 65535) return cudaErrorInvalidValue;
    CUtensorMap tK, tV;
    const uint32_t box[3] = {64, 128, 1};
    {
        const uint64_t dims[3] = {(uint64_t)h_kv * HD, (uint64_t)T_max, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldk * 2, (uint64_t)ldk * 2 * (uint64_t)T_max};
        if (!encode_tmap_bf16(&tK, Kc, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h_kv * HD, (uint64_t)T_max, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldv * 2, (uint64_t)ldv * 2 * (uint64_t)T_max};
        if (!encode_tmap_bf16(&tV, Vc, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const int span = decode_span_tc(B, h_kv, nrb, T_max, num_sms, HD == 64 ? 2 : 1);
    const int n_splits = (T_max + span - 1) / span;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    cudaError_t err = cudaFuncSetAttribute(decode_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           C::SMEM);
    if (err != cudaSuccess) return err;
    float* part = static_cast<float*>(ws);
    err = launch_pdl(decode_tc_kernel<HD>, dim3(n_splits, h_kv, B * nrb), dim3(DTC_THREADS), C::SMEM, stream,
                     tK, tV, reinterpret_cast<const __nv_bfloat16*>(Q), ldq, h, h_kv, T_q, T_max, span,
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
    // for grouped heads or several new tokens, the tensor-core kernel; one row per cached head
    // (plain multi-head attention at one new token) streams at most of HBM bandwidth on CUDA
    // cores already
    const int R = (h / h_kv) * T_q;
    if (R <= 1)
        return launch_decode_rows<HD, 1>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                         cache_lengths, ws, num_sms, status, stream);
    return launch_decode_tc<HD>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max, cache_lengths,
                                ws, num_sms, status, stream);
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
