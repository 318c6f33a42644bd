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
// cached keys and values of head g once and, for its query rows, computes the softmax
// statistics of its span -- the maximum m, the sum l of 2^(s - m) and the weighted value sum
// o -- and writes them to the workspace; a second kernel merges the spans of each row:
// M = max m_c, O = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c.  Scores are kept in base 2
// with log2(e)/sqrt(d) folded in.  The cache is bf16, accumulation fp32, and the score and
// weighted-value products run on the tensor core (decode_tc_kernel below) for every row count:
// with one row per cached head the MMAs are mostly padding, but the tensor core has the time
// to spare and the CUDA cores keep only the softmax, so the step streams the cache at close
// to the HBM copy bandwidth.
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

// Workspace: partials [B][h][T_q][split] of (m, l, o[d]) floats.
__host__ __device__ constexpr int dec_partial_floats(int d) { return d + 2; }

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
// The decode step on tcgen05: the R = (h / h_kv) * T_q query rows of head group g form one
// 128-row query tile (rows past R are zero), so every cached key and value is read once for
// the whole group and the score and weighted-value products run on the tensor core (S = Q K^T
// and O += P V with the accumulators in TMEM), leaving the CUDA cores only the softmax.  CTA (split, g, b * row blocks) streams its span of the cache in 128-key
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
    static constexpr int STAGES = HD == 128 ? 3 : 2;  // d = 64 keeps two CTAs per SM
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

}  // namespace

// The partials hold one record per split; splits are at least two 128-key tiles long, so
// ceil(T_max / 256) records per row bound the count for every launch configuration.
size_t decode_workspace_bytes(int B, int h, int T_q, int d, int T_max) {
    const size_t max_splits = (size_t)(T_max + 2 * DTC_TK - 1) / (2 * DTC_TK);
    return sizeof(float) * (size_t)B * h * T_q * max_splits * dec_partial_floats(d);
}

cudaError_t launch_decode_bf16(const void* Q, int64_t ldq, const void* Kc, int64_t ldk,
                               const void* Vc, int64_t ldv, void* O, int64_t ldo, int B, int h,
                               int h_kv, int T_q, int T_max, int d, const int32_t* cache_lengths,
                               void* ws, int num_sms, int* status, cudaStream_t stream) {
    if (d == 64)
        return launch_decode_tc<64>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                    cache_lengths, ws, num_sms, status, stream);
    if (d == 128)
        return launch_decode_tc<128>(Q, ldq, Kc, ldk, Vc, ldv, O, ldo, B, h, h_kv, T_q, T_max,
                                     cache_lengths, ws, num_sms, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mha
