// attn_bf16.cu -- the fused attention step on tcgen05 tensor cores, for every head:
//   S = Q_i K_i^T / sqrt(d)  [+ causal / key-padding mask]      (never written to memory)
//   O_i = softmax_rows(S) V_i                                   (written into Concat layout)
// itwiki.kr "멀티 헤드 어텐션": 수식 (scaled dot-product attention), the tensor-shape table
// (view+transpose head split, (B,h,T,T) scores, last-axis softmax, weighted sum, Concat),
// and 매개변수와 계산량 (flash attention removes the memory traffic of the T^2 term);
// iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", sections 9-10 (mask as -inf,
// row softmax) and 19 (cross-attention).
//
// One CTA computes one (batch, head, 128-row query tile).  The softmax is the online form:
// a running row maximum m and sum l, with O rescaled when m grows, so the result equals the
// row softmax after the final division by l.  Everything stays in base 2: p = 2^(s*c - m)
// with c = log2(e)/sqrt(d) folded into one FFMA per score.
//
// Warp roles (192 threads):
//   warp 0      TMA loads: the Q tile once, then K and V tiles (128 keys) into a ring;
//   warp 1      TMEM owner and single-thread MMA issuer:
//                 S_j = Q K_j^T   (M=128, N=128, K=d; double-buffered S in TMEM)
//                 O  += P_j V_j   (M=128, N=d, K=128; O accumulates in TMEM)
//               S_{j+1} is issued before waiting for P_j, so the tensor core computes the
//               next scores while the softmax warps work on the current ones;
//   warps 2..5  softmax, one query row per thread (TMEM lane = row): read S_j, mask, row
//               max, exponentials, row sum, write P_j (bf16, swizzled K-major) to shared
//               memory, rescale O in TMEM when needed; at the end O/l is rounded to bf16
//               and written by TMA straight into column block i*d of the (B,T,h*d) output.
// The rescale is lazy: the reference maximum only moves when a tile's maximum exceeds it by
// more than 8 (a factor 256 in base 2), so most tiles skip the O read-modify-write; the
// final O/l is the same because numerator and denominator share the reference.
// Causal: query tile qt needs key tiles 0..qt only; the grid runs the heaviest tiles first.
// Key padding: key tiles stop at ceil(L_b/128); the last one is masked in registers.
#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

template <int HD>
struct AttnCfg {
    static constexpr int BM = 128;                 // query rows per CTA
    static constexpr int BN = 128;                 // keys per tile
    static constexpr int CH = HD / 64;             // 64-column chunks per head
    static constexpr int CHUNK = 128 * 128;        // 128 rows x 64 bf16 (128 B) = 16 KB
    static constexpr int Q_BYTES = CH * CHUNK;
    static constexpr int KV_BYTES = CH * CHUNK;    // one K (or V) tile
    static constexpr int P_BYTES = 2 * CHUNK;      // 128 rows x 128 keys
    static constexpr int STAGES = HD == 64 ? 4 : 2;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = Q_BYTES + 2 * STAGES * KV_BYTES + P_BYTES + BAR_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;         // S buffers at columns 0 and 128
};

static_assert(AttnCfg<64>::SMEM <= 232448, "smem budget d=64");
static_assert(AttnCfg<128>::SMEM <= 232448, "smem budget d=128");

constexpr int A_THREADS = 192;

__device__ __forceinline__ void drain_wait_a(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

template <int HD>
__global__ void __launch_bounds__(A_THREADS, 1)
    attn_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, int h, int T_kv, int causal,
                        const int32_t* __restrict__ kv_lengths, float scale_log2, int* status) {
    using C = AttnCfg<HD>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sQ = base;
    const uint32_t sK = sQ + C::Q_BYTES;
    const uint32_t sV = sK + S * C::KV_BYTES;
    const uint32_t sP = sV + S * C::KV_BYTES;
    const uint32_t sBar = sP + C::P_BYTES;
    // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], s_free[2], p_full,
    //           pv_done, mma_drain
    const uint32_t bar_q = sBar;
    const uint32_t bar_kfull = sBar + 8u;
    const uint32_t bar_vfull = bar_kfull + 8u * S;
    const uint32_t bar_kvempty = bar_vfull + 8u * S;
    const uint32_t bar_sfull = bar_kvempty + 8u * S;
    const uint32_t bar_sfree = bar_sfull + 16u;
    const uint32_t bar_pfull = bar_sfree + 16u;
    const uint32_t bar_pvdone = bar_pfull + 8u;
    const uint32_t bar_drain = bar_pvdone + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int b = bh / h;
    const int head = bh - b * h;
    const int qt = causal ? (int)(gridDim.y - 1 - blockIdx.y) : (int)blockIdx.y;
    const int q0 = qt * C::BM;

    const int L = kv_lengths != nullptr ? kv_lengths[b] : T_kv;
    const bool bad = L < 1 || L > T_kv;
    int kv_hi = L;
    if (causal && kv_hi > q0 + C::BM) kv_hi = q0 + C::BM;
    const int n_tiles = bad ? 0 : (kv_hi + C::BN - 1) / C::BN;

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_kfull + 8u * s, 1);
            mbar_init(bar_vfull + 8u * s, 1);
            mbar_init(bar_kvempty + 8u * s, 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar_sfull + 8u * s, 1);
            mbar_init(bar_sfree + 8u * s, 128);
        }
        mbar_init(bar_pfull, 128);
        mbar_init(bar_pvdone, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        if (bad) record_status(status, kStatusBadLength);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0 && n_tiles > 0) {
            // ---------------- TMA loads
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(bar_q, C::Q_BYTES);
#pragma unroll
            for (int c = 0; c < C::CH; ++c)
                tma_load_3d(sQ + c * C::CHUNK, &tmQ, head * HD + c * 64, q0, b, bar_q);
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % S;
                const uint32_t ph = (uint32_t)(j / S) & 1u;
                if (!mbar_wait(bar_kvempty + 8u * st, ph ^ 1u, abort_flag, status)) break;
                const uint32_t kb = bar_kfull + 8u * st, vb = bar_vfull + 8u * st;
                mbar_arrive_expect_tx(kb, C::KV_BYTES);
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sK + st * C::KV_BYTES + c * C::CHUNK, &tmK, head * HD + c * 64,
                                j * C::BN, b, kb);
                mbar_arrive_expect_tx(vb, C::KV_BYTES);
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sV + st * C::KV_BYTES + c * C::CHUNK, &tmV, head * HD + c * 64,
                                j * C::BN, b, vb);
                ++issued;
            }
            // every copy issued lands before the CTA exits
            drain_wait_a(bar_q, 0);
            for (int j = issued - 1; j >= 0 && j >= issued - S; --j) {
                const int st = j % S;
                const uint32_t ph = (uint32_t)(j / S) & 1u;
                drain_wait_a(bar_kfull + 8u * st, ph);
                drain_wait_a(bar_vfull + 8u * st, ph);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && n_tiles > 0) {
            // ---------------- MMA issuer
            const uint32_t idesc_s = idesc_bf16_f32(128, C::BN, false, false);
            const uint32_t idesc_o = idesc_bf16_f32(128, HD, false, true);
            bool ok = mbar_wait(bar_q, 0, abort_flag, status);
            for (int j = 0; j <= n_tiles && ok; ++j) {
                if (j < n_tiles) {
                    const int st = j % S;
                    const uint32_t ph = (uint32_t)(j / S) & 1u;
                    const int sb = j & 1;
                    const uint32_t sph = (uint32_t)(j >> 1) & 1u;
                    if (!mbar_wait(bar_kfull + 8u * st, ph, abort_flag, status)) break;
                    if (!mbar_wait(bar_sfree + 8u * sb, sph ^ 1u, abort_flag, status)) break;
                    tc_fence_after();
                    const uint32_t kbase = sK + st * C::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < HD / 16; ++kk) {
                        const uint32_t off = (uint32_t)((kk >> 2) * C::CHUNK + (kk & 3) * 32);
                        mma_bf16_ss(tmem_base + (uint32_t)(sb * 128), sdesc_sw128(sQ + off, 16, 1024),
                                    sdesc_sw128(kbase + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar_sfull + 8u * sb);
                }
                if (j > 0) {
                    const int i = j - 1;
                    const int st = i % S;
                    const uint32_t ph = (uint32_t)(i / S) & 1u;
                    if (!mbar_wait(bar_pfull, (uint32_t)i & 1u, abort_flag, status)) break;
                    if (!mbar_wait(bar_vfull + 8u * st, ph, abort_flag, status)) break;
                    tc_fence_after();
                    const uint32_t vbase = sV + st * C::KV_BYTES;
#pragma unroll
                    for (int kk = 0; kk < C::BN / 16; ++kk) {
                        const uint32_t poff = (uint32_t)((kk >> 2) * C::CHUNK + (kk & 3) * 32);
                        mma_bf16_ss(tmem_base + C::O_COL, sdesc_sw128(sP + poff, 16, 1024),
                                    sdesc_sw128(vbase + kk * 2048, C::CHUNK, 1024), idesc_o,
                                    (i > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(bar_kvempty + 8u * st);
                    tc_commit(bar_pvdone);
                }
            }
            tc_commit(bar_drain);
            drain_wait_a(bar_drain, 0);
        }
    } else {
        // ---------------- softmax: warps 2..5, thread = query row
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int t = q0 + r;
        const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t srow_sw = (uint32_t)(r & 7);
        if (n_tiles == 0) {
            // no valid key: the softmax is undefined, the rows are NaN
#pragma unroll
            for (int c = 0; c < C::CH; ++c)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(sQ + c * C::CHUNK + r * 128 + ((u ^ srow_sw) << 4), 0x7FC07FC0u,
                                 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
        } else {
            float m = -INFINITY;  // reference maximum, already scaled to base 2
            float l = 0.f;
            bool ok = true;
            for (int j = 0; j < n_tiles; ++j) {
                const int sb = j & 1;
                // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
                if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull + 8u * sb, (uint32_t)(j >> 1) & 1u,
                                                       abort_flag, status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(trow + (uint32_t)(sb * 128 + c * 32), sr[c]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(bar_sfree + 8u * sb);

                float x[128];
#pragma unroll
                for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
                const int kv0 = j * C::BN;
                if (kv0 + C::BN > L || (causal && kv0 + C::BN - 1 > q0)) {
                    const int lim = causal ? min(L, t + 1) : L;  // keys [0, lim) are visible
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (kv0 + c >= lim) x[c] = -INFINITY;
                }
                float mx = x[0];
#pragma unroll
                for (int c = 1; c < 128; ++c) mx = fmaxf(mx, x[c]);
                const float m_tile = mx * scale_log2;
                float m_new = m;
                if (m_tile > m + 8.0f) m_new = m_tile;
                const bool rescale = (m_new != m) && j > 0;
                const float alpha = ex2_approx(m - m_new);
                const float neg = m_new == -INFINITY ? 0.f : -m_new;
                float rowsum = 0.f;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    x[c] = ex2_approx(fmaf(x[c], scale_log2, neg));
                    rowsum += x[c];
                }
                if (j > 0) {
                    // P_{j-1} V_{j-1} finished: O is stable and the P buffer is free
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_pvdone, (uint32_t)(j - 1) & 1u,
                                                           abort_flag, status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, rescale)) {
                        const float a = rescale ? alpha : 1.f;
#pragma unroll
                        for (int cc = 0; cc < HD / 32; ++cc) {
                            uint32_t o[32];
                            tmem_ld32(trow + C::O_COL + cc * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                            tmem_st32(trow + C::O_COL + cc * 32, o);
                        }
                        tmem_wait_st();
                    }
                }
                // P_j as bf16, K-major with 128-byte swizzle: keys [64c, 64c+64) in chunk c
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int k = c * 64 + u * 8;
                        st_shared_v4(sP + c * C::CHUNK + r * 128 + ((u ^ srow_sw) << 4),
                                     pack_bf16x2(x[k], x[k + 1]), pack_bf16x2(x[k + 2], x[k + 3]),
                                     pack_bf16x2(x[k + 4], x[k + 5]),
                                     pack_bf16x2(x[k + 6], x[k + 7]));
                    }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar_pfull);
                l = l * alpha + rowsum;
                m = m_new;
            }
            if (ok && __all_sync(0xffffffffu, mbar_wait(bar_pvdone, (uint32_t)(n_tiles - 1) & 1u,
                                                        abort_flag, status))) {
                tc_fence_after();
                const float inv = 1.f / l;
                // O / l as bf16 into the (now idle) Q buffer, same swizzled layout as the TMA box
#pragma unroll
                for (int cc = 0; cc < HD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(trow + C::O_COL + cc * 32, o);
                    tmem_wait_ld();
                    const int c = cc >> 1;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const int u = (cc & 1) * 4 + u4;
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(o[u4 * 8 + i]) * inv;
                        st_shared_v4(sQ + c * C::CHUNK + r * 128 + ((u ^ srow_sw) << 4),
                                     pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                     pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
            }
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, 128);
        if (threadIdx.x == 64 && !*abort_flag) {
#pragma unroll
            for (int c = 0; c < C::CH; ++c) tma_store_3d(&tmO, sQ + c * C::CHUNK, head * HD + c * 64, q0, b);
            bulk_commit_group();
            bulk_wait_group<0>();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int HD>
cudaError_t launch_attn_hd(const void* Q, int64_t ldq, const void* K, int64_t ldk, const void* V,
                           int64_t ldv, void* O, int64_t ldo, int B, int h, int T_q, int T_kv,
                           int causal, const int32_t* kv_lengths, int* status,
                           cudaStream_t stream) {
    using C = AttnCfg<HD>;
    CUtensorMap tQ, tK, tV, tO;
    const uint32_t box[3] = {64, 128, 1};
    {
        const uint64_t dims[3] = {(uint64_t)h * HD, (uint64_t)T_q, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldq * 2, (uint64_t)ldq * 2 * (uint64_t)T_q};
        if (!encode_tmap_bf16(&tQ, Q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h * HD, (uint64_t)T_kv, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldk * 2, (uint64_t)ldk * 2 * (uint64_t)T_kv};
        if (!encode_tmap_bf16(&tK, K, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h * HD, (uint64_t)T_kv, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldv * 2, (uint64_t)ldv * 2 * (uint64_t)T_kv};
        if (!encode_tmap_bf16(&tV, V, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h * HD, (uint64_t)T_q, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldo * 2, (uint64_t)ldo * 2 * (uint64_t)T_q};
        if (!encode_tmap_bf16(&tO, O, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaFuncSetAttribute(attn_bf16_tc_kernel<HD>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    const dim3 grid((unsigned)(B * h), (unsigned)((T_q + C::BM - 1) / C::BM));
    attn_bf16_tc_kernel<HD><<<grid, A_THREADS, C::SMEM, stream>>>(tQ, tK, tV, tO, h, T_kv, causal,
                                                                   kv_lengths, scale_log2, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bf16(const void* Q, int64_t ldq, const void* K, int64_t ldk,
                             const void* V, int64_t ldv, void* O, int64_t ldo, int B, int h,
                             int T_q, int T_kv, int d, int causal, const int32_t* kv_lengths,
                             int* status, cudaStream_t stream) {
    if (d == 64)
        return launch_attn_hd<64>(Q, ldq, K, ldk, V, ldv, O, ldo, B, h, T_q, T_kv, causal,
                                  kv_lengths, status, stream);
    if (d == 128)
        return launch_attn_hd<128>(Q, ldq, K, ldk, V, ldv, O, ldo, B, h, T_q, T_kv, causal,
                                   kv_lengths, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mha
