// attn_bf16.cu -- the fused attention step on tcgen05 tensor cores, for every head:
//   S = Q_i K_i^T / sqrt(d)  [+ causal / key-padding mask]      (never written to memory)
//   O_i = softmax_rows(S) V_i                                   (written into Concat layout)
// itwiki.kr "멀티 헤드 어텐션": 수식 (scaled dot-product attention), the tensor-shape table
// (view+transpose head split, (B,h,T,T) scores, last-axis softmax, weighted sum, Concat),
// and 매개변수와 계산량 (flash attention removes the memory traffic of the T^2 term);
// iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", sections 9-10 (mask as -inf,
// row softmax) and 19 (cross-attention).
//
// Two kernels share the softmax scheme below:
//   attn_bf16_tc_kernel   d = 128: one CTA = two 128-row query tiles of one (batch, head)
//                         that share every K/V tile the TMA brings in;
//   attn_bf16_d64_kernel  d = 64: persistent, two CTAs per SM, one query tile at a time
//                         (described with the kernel further down).
// The softmax is the online form: a running row maximum m and sum l, with O rescaled when m
// grows, so the result equals the row softmax after the final division by l.  Everything
// stays in base 2: p = 2^(s*c - m) with c = log2(e)/sqrt(d) folded into one FMA per score.
//
// d = 128 tensor memory (512 columns, one CTA per SM):
//   S_t  [128 t, 128 t + 128)          scores of query tile t, fp32
//   O_t  [256 + 128 t, 256 + 128 t + 128)  output accumulator of tile t, fp32
//   P_t  the first 64 columns of S_t (TMEM is full: S0, S1, O0, O1 use all 512)
// The PV product reads P from TMEM (A operand in tensor memory); Q and K come from shared
// memory.  With P inside S, S_{j+1} must wait until P_j has been consumed, and the two
// query tiles take turns on the tensor core.
//
// d = 128 warp roles (384 threads):
//   warp 0      TMA: Q0 and Q1 once, then K and V tiles (128 keys) into a ring of stages;
//   warp 1      TMEM owner and MMA issuer, alternating the tiles per key tile j:
//                 O_0 += P_0 V_j, S_0(j+1), O_1 += P_1 V_j, S_1(j+1)
//               (tcgen05 MMAs of one thread execute in issue order, so S_t may overwrite the
//               P_t columns right after the MMA that reads them);
//   warps 2-3   otherwise idle;
//   warps 4-7   softmax of query tile 0, warps 8-11 of tile 1 -- one row per thread (TMEM
//               lane = row): read S, mask, exponentials, row sum, P -> TMEM, lazy O rescale;
//               while one group works, the tensor core runs the other tile's MMAs.
//               At the end O/l is rounded to bf16 and stored by TMA straight into column
//               block (head * d) of the (B, T, h*d) Concat output.
// Reference maximum: P = 2^(s*c - m_ref) gives the same O / l for any reference m_ref (the
// numerator and the denominator carry the same factor); the reference only has to keep P
// finite.  So the first key tile sets m_ref to the exact row maximum, and later tiles skip
// the maximum altogether: their P is computed against the current m_ref and only if a row's
// sum exceeds 2^64 (or is not finite) does the warp redo the tile with the exact maximum and
// rescale O and l.  Every exponential runs on the MUFU unit (ex2.approx), which retires 32
// results per clock per SM on GB300 -- a key tile's 32768 exponentials in 1024 clocks, within
// the tensor core's time for the same tile.
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

template <int HD>
struct AttnCfg {
    static constexpr int BM = 128;                  // rows per query tile
    static constexpr int NQ = 2;                    // query tiles per CTA
    static constexpr int BN = 128;                  // keys per tile
    static constexpr int CH = HD / 64;              // 64-column chunks per head
    static constexpr int CHUNK = 128 * 128;         // 128 rows x 64 bf16 (128 B) = 16 KB
    static constexpr int Q_BYTES = CH * CHUNK;      // one query tile
    static constexpr int KV_BYTES = CH * CHUNK;     // one K (or V) tile
    static constexpr int STAGES = 2;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = NQ * Q_BYTES + 2 * STAGES * KV_BYTES + BAR_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t S_COL(int t) { return (uint32_t)(128 * t); }
    __host__ __device__ static constexpr uint32_t O_COL(int t) { return (uint32_t)(256 + HD * t); }
    __host__ __device__ static constexpr uint32_t P_COL(int t) { return (uint32_t)(128 * t); }
};

static_assert(AttnCfg<128>::SMEM <= 232448, "smem budget d=128");

constexpr int A_THREADS = 384;

// K/V bytes of one group of (batch, head) pairs in the d = 128 kernel's CTA order
#ifndef MHA_D128_GROUP_BYTES
#define MHA_D128_GROUP_BYTES (64ll << 20)
#endif

// One row of a 128-key score tile from TMEM into registers (warp-collective), with the
// causal / key-length mask applied (keys [0, lim) are visible).
__device__ __forceinline__ void load_s_tile(uint32_t taddr, bool masked, int kv0, int lim,
                                            float (&x)[128]) {
    uint32_t sr[4][32];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(taddr + c * 32, sr[c]);
    tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c >> 5][c & 31]);
    if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
            if (kv0 + c >= lim) x[c] = -INFINITY;
    }
}

// p = 2^(s*c + neg) for the 64 scores [64 h, 64 h + 64) of a row; returns their sum and
// writes P as packed bf16 pairs.
__device__ __forceinline__ float exp_half(const float (&x)[128], int h, uint64_t c2, float neg,
                                          uint32_t (&pk)[32]) {
    const uint64_t neg2 = pack2(neg, neg);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        float a0, a1;
        unpack2(fma2(pack2(x[64 * h + 2 * k], x[64 * h + 2 * k + 1]), c2, neg2), a0, a1);
        const float y0 = ex2_approx(a0), y1 = ex2_approx(a1);
        acc[k & 3] = add2(acc[k & 3], pack2(y0, y1));
        pk[k] = pack_bf16x2(y0, y1);
    }
    const uint64_t s01 = add2(acc[0], acc[1]), s23 = add2(acc[2], acc[3]);
    float a0, a1;
    unpack2(add2(s01, s23), a0, a1);
    return a0 + a1;
}

// The output gate of gated attention: f[i] *= sigmoid(g_i) for 8 consecutive outputs, w the
// 8 bf16 gate pre-activations of this row.  sigmoid(x) = 1 / (1 + 2^(-x log2 e)).
__device__ __forceinline__ void apply_gate8(const uint4 w, float (&f)[8]) {
    const uint32_t gw[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float g0 = __uint_as_float(gw[i] << 16), g1 = __uint_as_float(gw[i] & 0xFFFF0000u);
        f[2 * i] *= __fdividef(1.f, 1.f + ex2_approx(-1.4426950408889634f * g0));
        f[2 * i + 1] *= __fdividef(1.f, 1.f + ex2_approx(-1.4426950408889634f * g1));
    }
}

template <int HD, bool GATE>
__global__ void __launch_bounds__(A_THREADS, 1)
    attn_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, int h, int h_kv, int T_q, int T_kv,
                        int causal, const int32_t* __restrict__ kv_lengths,
                        const __nv_bfloat16* __restrict__ gate, int64_t ldg, float scale_log2,
                        int* status, int BH, int n_qb, int head_group) {
    static_assert(HD == 128, "head dim 64 runs on attn_bf16_d64_kernel");
    using C = AttnCfg<HD>;
    constexpr int S = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sQ = base;  // Q0 then Q1; each later reused as that tile's output staging
    const uint32_t sK = sQ + C::NQ * C::Q_BYTES;
    const uint32_t sV = sK + S * C::KV_BYTES;
    const uint32_t sBar = sV + S * C::KV_BYTES;
    // barriers: q_full, k_full[S], v_full[S], kv_empty[S], s_full[2], s_free[2], p_full[2],
    //           pv_done[2], mma_drain
    const uint32_t bar_q = sBar;
    const uint32_t bar_kfull = sBar + 8u;
    const uint32_t bar_vfull = bar_kfull + 8u * S;
    const uint32_t bar_kvempty = bar_vfull + 8u * S;
    const uint32_t bar_sfull = bar_kvempty + 8u * S;
    const uint32_t bar_sfree = bar_sfull + 16u;
    const uint32_t bar_pfull = bar_sfree + 16u;
    const uint32_t bar_pvdone = bar_pfull + 16u;
    const uint32_t bar_drain = bar_pvdone + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA i of the 1-D grid (CTAs start roughly in index order): the (batch, head) pairs form
    // groups of head_group; a group's CTAs come before the next group's, and within a group the
    // query-tile pairs are numbered longest first (causal: the last pair of every (batch, head)
    // first), the group's (batch, head) pairs fastest.  The CTAs in flight then read the K/V
    // of about two groups, which stays in L2 while each of its query-tile pairs streams it.
    const int gi = (int)blockIdx.x / (head_group * n_qb);
    const int gr = (int)blockIdx.x - gi * head_group * n_qb;
    const int gsz = min(head_group, BH - gi * head_group);
    const int rank = gr / gsz;
    const int bh = gi * head_group + (gr - rank * gsz);
    const int b = bh / h;
    const int head = bh - b * h;
    const int kvh = head / (h / h_kv);  // grouped K/V heads: the K/V head of this query head
    const int qb = causal ? n_qb - 1 - rank : rank;
    const int q0 = qb * (C::NQ * C::BM);

    if (threadIdx.x == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_kfull + 8u * s, 1);
            mbar_init(bar_vfull + 8u * s, 1);
            mbar_init(bar_kvempty + 8u * s, 1);  // committed by the thread issuing the PV MMAs
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar_sfull + 8u * t, 1);
            mbar_init(bar_sfree + 8u * t, 128);
            mbar_init(bar_pfull + 8u * t, 128);
            mbar_init(bar_pvdone + 8u * t, 1);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Q, K, V and the key lengths may come from the previous kernel on the stream
    grid_dependency_wait();
    grid_launch_dependents();

    const int L = kv_lengths != nullptr ? kv_lengths[b] : T_kv;
    const bool bad = L < 1 || L > T_kv;
    const int nL = (L + C::BN - 1) / C::BN;
    int n_t[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        int n = nL;
        if (causal) {
            const int nc = (q0 + C::BM * t + C::BM + C::BN - 1) / C::BN;  // key tiles up to the diagonal
            n = n < nc ? n : nc;
        }
        n_t[t] = bad ? 0 : n;
    }
    const int n_max = n_t[0] > n_t[1] ? n_t[0] : n_t[1];
    if (threadIdx.x == 0 && bad) record_status(status, kStatusBadLength);

    if (warp == 0) {
        if (lane == 0 && n_max > 0) {
            // ---------------- TMA loads
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(bar_q, C::NQ * C::Q_BYTES);
#pragma unroll
            for (int t = 0; t < C::NQ; ++t)
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sQ + t * C::Q_BYTES + c * C::CHUNK, &tmQ, head * HD + c * 64,
                                q0 + t * C::BM, b, bar_q);
            int issued = 0;
            for (int j = 0; j < n_max; ++j) {
                const int st = j % S;
                const uint32_t ph = (uint32_t)(j / S) & 1u;
                if (!mbar_wait(bar_kvempty + 8u * st, ph ^ 1u, abort_flag, status)) break;
                const uint32_t kb = bar_kfull + 8u * st, vb = bar_vfull + 8u * st;
                mbar_arrive_expect_tx(kb, C::KV_BYTES);
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sK + st * C::KV_BYTES + c * C::CHUNK, &tmK, kvh * HD + c * 64,
                                j * C::BN, b, kb);
                mbar_arrive_expect_tx(vb, C::KV_BYTES);
#pragma unroll
                for (int c = 0; c < C::CH; ++c)
                    tma_load_3d(sV + st * C::KV_BYTES + c * C::CHUNK, &tmV, kvh * HD + c * 64,
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
        if (lane == 0) {
            // ---------------- single MMA issuer for both query tiles, strictly alternating:
            //   O_0 += P_0 V_j ; S_0(j+1) ; O_1 += P_1 V_j ; S_1(j+1)
            const uint32_t idesc_s = idesc_bf16_f32(128, C::BN, false, false);
            const uint32_t idesc_o = idesc_bf16_f32(128, HD, false, true);
            const uint64_t kdesc0 = sdesc_sw128(sK, 16, 1024);
            const uint64_t vdesc0 = sdesc_sw128(sV, C::CHUNK, 1024);
            const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024);
            auto issue_s = [&](int t, int j) {
                const uint64_t kdesc = kdesc0 + (uint64_t)(((j % S) * C::KV_BYTES) >> 4);
                const uint64_t qdesc = qdesc0 + (uint64_t)((t * C::Q_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off16 = (uint32_t)(((kk >> 2) * C::CHUNK + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(tmem_base + C::S_COL(t), qdesc + off16, kdesc + off16, idesc_s,
                                kk > 0 ? 1u : 0u);
                }
                tc_commit(bar_sfull + 8u * t);
            };
            auto issue_pv = [&](int t, int j) {
                const uint64_t vdesc = vdesc0 + (uint64_t)(((j % S) * C::KV_BYTES) >> 4);
#pragma unroll
                for (int kk = 0; kk < C::BN / 16; ++kk)
                    mma_bf16_ts(tmem_base + C::O_COL(t), tmem_base + C::P_COL(t) + kk * 8,
                                vdesc + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar_pvdone + 8u * t);
            };
            bool ok = true;
            if (n_max > 0) {
                ok = mbar_wait(bar_q, 0, abort_flag, status) &&
                     mbar_wait(bar_kfull, 0, abort_flag, status);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t)
                        if (n_t[t] > 0) issue_s(t, 0);
                }
            }
            int k_ready = 0;  // highest key tile whose K has been waited for
            for (int j = 0; j < n_max && ok; ++j) {
                const int jn = j + 1;
                ok = mbar_wait(bar_vfull + 8u * (j % S), (uint32_t)(j / S) & 1u, abort_flag, status);
#pragma unroll
                for (int t = 0; t < 2 && ok; ++t) {
                    if (j >= n_t[t]) continue;
                    ok = mbar_wait(bar_pfull + 8u * t, (uint32_t)j & 1u, abort_flag, status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(t, j);
                    if (jn < n_t[t]) {
                        if (jn > k_ready) {
                            ok = mbar_wait(bar_kfull + 8u * (jn % S), (uint32_t)(jn / S) & 1u,
                                           abort_flag, status);
                            k_ready = jn;
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_s(t, jn);
                    }
                }
                if (!ok) break;
                tc_commit(bar_kvempty + 8u * (j % S));
            }
            tc_commit(bar_drain);
            drain_wait_a(bar_drain, 0);
        }
    } else if (warp >= 4) {
        // ---------------- softmax: warps 4-7 tile 0, warps 8-11 tile 1; thread = query row
        const int t = (warp - 4) >> 2;
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int qrow0 = q0 + t * C::BM;      // first row of this query tile
        const int row = qrow0 + r;             // this thread's query row
        const int n = n_t[t];
        if constexpr (GATE)  // this row's gate pre-activations, into L2 for the epilogue
            if (row < T_q)
#pragma unroll
                for (int c = 0; c < HD / 64; ++c)
                    prefetch_l2(gate + ((int64_t)b * T_q + row) * ldg + (int64_t)head * HD + 64 * c);
        const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t sw = (uint32_t)(r & 7);
        const uint32_t sQt = sQ + t * C::Q_BYTES;
        const uint32_t bar_s = bar_sfull + 8u * t, bar_p = bar_pfull + 8u * t;
        bool ok = true;

        if (n == 0) {
            // no valid key: the softmax is undefined, the rows are NaN
#pragma unroll
            for (int c = 0; c < C::CH; ++c)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(sQt + c * C::CHUNK + r * 128 + ((u ^ sw) << 4), 0x7FC07FC0u,
                                 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
        } else {
            float m = -INFINITY;  // reference maximum, already scaled to base 2
            float l = 0.f;
            for (int j = 0; j < n && ok; ++j) {
                // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
                if (!__all_sync(0xffffffffu, mbar_wait(bar_s, (uint32_t)j & 1u, abort_flag, status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int kv0 = j * C::BN;
                const bool masked = kv0 + C::BN > L || (causal && kv0 + C::BN - 1 > qrow0);
                const int lim = causal ? min(L, row + 1) : L;  // keys [0, lim) are visible
                uint32_t pk[64];
                float x[128];
                float rowsum, alpha = 1.f, m_new = m;
                {
                    // P overwrites S in place, so S_t(j) stays readable until P is written.
                    // Fast path (every key tile after the first): no row maximum.  P is computed
                    // against the current reference m; any reference gives the same O / l, it
                    // only has to keep P finite.  If some row's sum exceeds 2^64 (or is not
                    // finite) the warp redoes the tile with the exact maximum (slow path, also
                    // used for j = 0).
                    bool slow = j == 0;
                    if (!slow) {
                        load_s_tile(trow + C::S_COL(t), masked, kv0, lim, x);
                        rowsum = exp_tile(x, pack2(scale_log2, scale_log2), -m, pk);
                        slow = !__all_sync(0xffffffffu, rowsum <= 18446744073709551616.f);
                    }
                    if (slow) {
                        load_s_tile(trow + C::S_COL(t), masked, kv0, lim, x);
                        const float m_tile = row_max(x) * scale_log2;
                        m_new = m_tile > m ? m_tile : m;
                        alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)
                        rowsum = exp_tile(x, pack2(scale_log2, scale_log2),
                                          m_new == -INFINITY ? 0.f : -m_new, pk);
                    }
                }
                const bool rescale = (m_new != m) && j > 0;
                // S_t(j) was issued after PV_t(j-1), so O_t is already complete
                if (__any_sync(0xffffffffu, rescale)) {
                    const float a = rescale ? alpha : 1.f;
#pragma unroll
                    for (int cc = 0; cc < HD / 32; ++cc) {
                        uint32_t o[32];
                        tmem_ld32(trow + C::O_COL(t) + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                        tmem_st32(trow + C::O_COL(t) + cc * 32, o);
                    }
                }
                {
                    uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[0]);
                    uint32_t (&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&pk[32]);
                    tmem_st32(trow + C::P_COL(t), p0);
                    tmem_st32(trow + C::P_COL(t) + 32, p1);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar_p);
                l = l * alpha + rowsum;
                m = m_new;
            }
            // the gate pre-activations of this row, loaded while the last PV product runs
            uint4 gv[GATE ? HD / 8 : 1];
            if constexpr (GATE) {
                const uint4* g4 = reinterpret_cast<const uint4*>(gate + ((int64_t)b * T_q + row) * ldg +
                                                                 (int64_t)head * HD);
#pragma unroll
                for (int i = 0; i < HD / 8; ++i) gv[i] = row < T_q ? __ldg(g4 + i) : make_uint4(0u, 0u, 0u, 0u);
            }
            if (ok && __all_sync(0xffffffffu, mbar_wait(bar_pvdone + 8u * t, (uint32_t)(n - 1) & 1u,
                                                        abort_flag, status))) {
                tc_fence_after();
                const float inv = 1.f / l;
                // O / l (times the gate) as bf16 into this tile's Q buffer (idle now), in the
                // TMA box layout
#pragma unroll
                for (int cc = 0; cc < HD / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(trow + C::O_COL(t) + cc * 32, o);
                    tmem_wait_ld();
                    const int c = cc >> 1;
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const int u = (cc & 1) * 4 + u4;
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(o[u4 * 8 + i]) * inv;
                        if constexpr (GATE) apply_gate8(gv[cc * 4 + u4], f);
                        st_shared_v4(sQt + c * C::CHUNK + r * 128 + ((u ^ sw) << 4),
                                     pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                     pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
            }
        }
        fence_proxy_async_smem();
        named_barrier_sync(1 + t, 128);
        if ((threadIdx.x & 127) == 0 && !*abort_flag && qrow0 < T_q) {
#pragma unroll
            for (int c = 0; c < C::CH; ++c)
                tma_store_3d(&tmO, sQt + c * C::CHUNK, head * HD + c * 64, qrow0, b);
            bulk_commit_group();
            bulk_wait_group<0>();
        }
    }

    // lanes that skipped a one-thread role wait here for it: the CTA barrier below must
    // see whole warps, or it can complete while a role is still running
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------
// d = 64: persistent CTAs, two per SM, one 128-row query tile at a time.
//
// With d = 64 a 128x128 key tile costs the tensor core 2 x 256 cycles per query tile and the
// softmax 16384 exponentials, which the MUFU retires at 32 per clock per SM at best, so the
// softmax must never wait.  Two CTAs per SM (256 TMEM columns each: S 128, O 64, P 64; 96 KB
// of shared memory) advance independently, so one CTA's softmax keeps the MUFU busy while the
// other reads S or stores P.  Each CTA is persistent: it walks a list of work items (one
// query tile of one (batch, head)), and the start of item i+1 -- its Q tile, its first K/V
// tiles and its first score MMA -- overlaps the end of item i (last softmax, last PV product,
// output store), which would otherwise leave the SM idle for thousands of cycles per item.
//
// Work items are numbered longest first (causal: the last query tiles of every head first)
// and dealt to the CTAs in a snake order (0..G-1, then G-1..0, ...), which balances the
// causal triangle across CTAs.
//
// Warp roles (256 threads; warps 0-3 run on 56 registers, the softmax warps on 200):
//   warp 0      TMA: per item the Q tile into one of two Q buffers (once the output of the
//               item two back has left it), then the K tiles through a ring of DK_STAGES
//               (freed when the score MMA that read them completes);
//   warp 1      TMEM owner and MMA issuer: S = Q K^T for the next key tile (of this item or
//               the next) as soon as the softmax has read the current S, then O += P V as
//               soon as P is in TMEM;
//   warp 2      TMA: the V tiles through a ring of DV_STAGES (freed when the PV MMA completes);
//   warp 3      TMA: stores each item's output, which the softmax leaves in the item's Q buffer;
//   warps 4-7   softmax, one query row per thread (TMEM lane quarter = warp & 3).
constexpr int DK_STAGES = 2;
constexpr int DV_STAGES = 2;
constexpr int D64_THREADS = 256;
constexpr int D64_REGS_CTRL = 56;
constexpr int D64_REGS_SOFTMAX = 200;
constexpr int D64_TILE = 128 * 128;  // one 128-row x 64-column bf16 box, 16 KB
constexpr int D64_BAR_BYTES = 512;
// batches ordered by key length (longest first) when the lengths vary: up to this many
constexpr int D64_SORT_MAX_B = 64;
constexpr int D64_SMEM = D64_TILE * (2 + DK_STAGES + DV_STAGES) + D64_BAR_BYTES + 1024;
// two CTAs (each with its 1 KB of reserved shared memory) must fit one SM's 228 KB
static_assert(2 * (D64_SMEM + 1024) <= 233472, "two d=64 CTAs per SM");
// the register split must fit the 128 registers per thread two CTAs are launched with
static_assert(128 * D64_REGS_CTRL + 128 * D64_REGS_SOFTMAX <= D64_THREADS * 128, "register split");
constexpr uint32_t D64_TMEM_COLS = 256;
constexpr uint32_t D64_S_COL = 0, D64_O_COL = 128, D64_P_COL = 192;

struct D64Item {
    int b, head, kvh, qrow0, n;  // kvh: the K/V head; n = key tiles to visit (0: no valid key)
    bool bad;
};

// Item k of the longest-first numbering.  Causal: by query tile, the last tiles of every
// (batch, head) first.  With key lengths and no causal mask (bperm: the batches sorted by
// length, longest first): by batch in that order, then head, then query tile, so that the
// items dealt out at one time share their K/V tiles.
__device__ __forceinline__ D64Item d64_item(int k, int BH, int h, int group, int n_qt, int causal,
                                            const int32_t* kv_lengths, int T_kv, const int* bperm) {
    D64Item it;
    int qt;
    if (bperm != nullptr) {
        const int per_b = h * n_qt;
        const int bs = k / per_b;
        const int rem = k - bs * per_b;
        it.b = bperm[bs];
        it.head = rem / n_qt;
        qt = rem - it.head * n_qt;
    } else {
        const int rank = k / BH;
        const int bh = k - rank * BH;
        qt = causal ? n_qt - 1 - rank : rank;
        it.b = bh / h;
        it.head = bh - it.b * h;
    }
    it.kvh = it.head / group;
    it.qrow0 = qt * 128;
    const int L = kv_lengths != nullptr ? kv_lengths[it.b] : T_kv;
    it.bad = L < 1 || L > T_kv;
    int n = (L + 127) / 128;
    if (causal) n = n < qt + 1 ? n : qt + 1;  // key tiles up to the diagonal
    it.n = it.bad ? 0 : n;
    return it;
}

// The r-th item of CTA c among G CTAs (snake order).
__device__ __forceinline__ int d64_item_index(int r, int G, int c) {
    return r * G + ((r & 1) ? G - 1 - c : c);
}

// SORTED: key lengths given, no causal mask, B <= D64_SORT_MAX_B -- items by batch, longest
// first (a separate instantiation: the plain order's code is left exactly as it is)
template <bool GATE, bool SORTED>
__global__ void __launch_bounds__(D64_THREADS, 2)
    attn_bf16_d64_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmO, int B, int h, int h_kv, int T_q,
                         int T_kv, int causal, const int32_t* __restrict__ kv_lengths,
                         const __nv_bfloat16* __restrict__ gate, int64_t ldg, float scale_log2,
                         int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sQ = base;  // two Q buffers; item r uses buffer r & 1, also for its output
    const uint32_t sK = sQ + 2 * D64_TILE;
    const uint32_t sV = sK + DK_STAGES * D64_TILE;
    const uint32_t sBar = sV + DV_STAGES * D64_TILE;
    // barriers: q_full[2], staged[2], q_free[2], k_full[DK], k_empty[DK], v_full[DV],
    //           v_empty[DV], s_full, s_free, p_full, pv_done, mma_drain
    const uint32_t bar_qfull = sBar;
    const uint32_t bar_staged = bar_qfull + 16u;
    const uint32_t bar_qfree = bar_staged + 16u;
    const uint32_t bar_kfull = bar_qfree + 16u;
    const uint32_t bar_kempty = bar_kfull + 8u * DK_STAGES;
    const uint32_t bar_vfull = bar_kempty + 8u * DK_STAGES;
    const uint32_t bar_vempty = bar_vfull + 8u * DV_STAGES;
    const uint32_t bar_sfull = bar_vempty + 8u * DV_STAGES;
    const uint32_t bar_sfree = bar_sfull + 8u;
    const uint32_t bar_pfull = bar_sfree + 8u;
    const uint32_t bar_pvdone = bar_pfull + 8u;
    const uint32_t bar_drain = bar_pvdone + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* bperm_s = reinterpret_cast<int*>(gbase + (bar_drain + 16u - base));  // [D64_SORT_MAX_B]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int BH = B * h;
    const int n_qt = (T_q + 127) / 128;
    const int N = BH * n_qt;
    const int G = (int)gridDim.x;
    const int c = (int)blockIdx.x;
    const int* bperm = SORTED ? bperm_s : nullptr;
    int R = 0;  // items of this CTA
    while (d64_item_index(R, G, c) < N) ++R;
    auto item = [&](int r) {
        return d64_item(d64_item_index(r, G, c), BH, h, h / h_kv, n_qt, causal, kv_lengths, T_kv, bperm);
    };

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_qfull + 8u * i, 1);
            mbar_init(bar_staged + 8u * i, 128);
            mbar_init(bar_qfree + 8u * i, 1);
        }
        for (int s = 0; s < DK_STAGES; ++s) {
            mbar_init(bar_kfull + 8u * s, 1);
            mbar_init(bar_kempty + 8u * s, 1);
        }
        for (int s = 0; s < DV_STAGES; ++s) {
            mbar_init(bar_vfull + 8u * s, 1);
            mbar_init(bar_vempty + 8u * s, 1);
        }
        mbar_init(bar_sfull, 1);
        mbar_init(bar_sfree, 128);
        mbar_init(bar_pfull, 128);
        mbar_init(bar_pvdone, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), D64_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Q, K, V and the key lengths may come from the previous kernel on the stream
    grid_dependency_wait();
    grid_launch_dependents();
    if constexpr (SORTED) {
        // rank of each batch by key length (longest first, ties by index)
        if (threadIdx.x < B) {
            const int t = (int)threadIdx.x;
            const int Lt = kv_lengths[t];
            int rank = 0;
            for (int u = 0; u < B; ++u) {
                const int Lu = kv_lengths[u];
                rank += (Lu > Lt) || (Lu == Lt && u < t);
            }
            bperm_s[rank] = t;
        }
        __syncthreads();
    }

    if (warp < 4) {
      setmaxnreg_dec<D64_REGS_CTRL>();
      if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA: Q and K
            tma_prefetch_desc(&tmK);
            uint32_t gk = 0;  // K tiles issued
            int rq = -1;      // last item whose Q load was issued
            bool ok = true;
            for (int r = 0; r < R && ok; ++r) {
                const D64Item it = item(r);
                // the Q buffer of item r held the output of item r-2 until it was stored
                if (r >= 2 && !mbar_wait(bar_qfree + 8u * (r & 1), (uint32_t)((r - 2) >> 1) & 1u,
                                         abort_flag, status))
                    break;
                if (it.bad) record_status(status, kStatusBadLength);
                const uint32_t qb = bar_qfull + 8u * (r & 1);
                mbar_arrive_expect_tx(qb, D64_TILE);
                tma_load_3d(sQ + (uint32_t)(r & 1) * D64_TILE, &tmQ, it.head * 64, it.qrow0, it.b, qb);
                rq = r;
                for (int j = 0; j < it.n; ++j) {
                    const uint32_t st = gk % DK_STAGES;
                    ok = mbar_wait(bar_kempty + 8u * st, ((gk / DK_STAGES) & 1u) ^ 1u, abort_flag, status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar_kfull + 8u * st, D64_TILE);
                    tma_load_3d(sK + st * D64_TILE, &tmK, it.kvh * 64, j * 128, it.b, bar_kfull + 8u * st);
                    ++gk;
                }
            }
            // every load issued lands before the CTA exits
            for (uint32_t g = gk > DK_STAGES ? gk - DK_STAGES : 0; g < gk; ++g)
                drain_wait_a(bar_kfull + 8u * (g % DK_STAGES), (g / DK_STAGES) & 1u);
            for (int r = rq > 1 ? rq - 1 : 0; r <= rq; ++r)
                drain_wait_a(bar_qfull + 8u * (r & 1), (uint32_t)(r >> 1) & 1u);
        }
      } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- TMA: V
            tma_prefetch_desc(&tmV);
            uint32_t gv = 0;  // V tiles issued
            bool ok = true;
            for (int r = 0; r < R && ok; ++r) {
                const D64Item it = item(r);
                for (int j = 0; j < it.n; ++j) {
                    const uint32_t st = gv % DV_STAGES;
                    ok = mbar_wait(bar_vempty + 8u * st, ((gv / DV_STAGES) & 1u) ^ 1u, abort_flag, status);
                    if (!ok) break;
                    mbar_arrive_expect_tx(bar_vfull + 8u * st, D64_TILE);
                    tma_load_3d(sV + st * D64_TILE, &tmV, it.kvh * 64, j * 128, it.b, bar_vfull + 8u * st);
                    ++gv;
                }
            }
            for (uint32_t g = gv > DV_STAGES ? gv - DV_STAGES : 0; g < gv; ++g)
                drain_wait_a(bar_vfull + 8u * (g % DV_STAGES), (g / DV_STAGES) & 1u);
        }
      } else if (warp == 3) {
        if (lane == 0) {
            // ---------------- TMA: outputs, each as soon as the softmax has staged it
            for (int r = 0; r < R; ++r) {
                if (!mbar_wait(bar_staged + 8u * (r & 1), (uint32_t)(r >> 1) & 1u, abort_flag, status))
                    break;
                const D64Item it = item(r);
                if (!*abort_flag && it.qrow0 < T_q) {
                    tma_store_3d(&tmO, sQ + (uint32_t)(r & 1) * D64_TILE, it.head * 64, it.qrow0, it.b);
                    bulk_commit_group();
                    bulk_wait_group_read<0>();
                }
                mbar_arrive(bar_qfree + 8u * (r & 1));
            }
            bulk_wait_group<0>();
        }
      } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
            const uint32_t idesc_o = idesc_bf16_f32(128, 64, false, true);
            const uint64_t kdesc0 = sdesc_sw128(sK, 16, 1024);
            const uint64_t vdesc0 = sdesc_sw128(sV, D64_TILE, 1024);
            const uint64_t qdesc0 = sdesc_sw128(sQ, 16, 1024);
            uint32_t gk = 0, gv = 0, gs = 0, gp = 0;  // K, V consumed; S, PV issued
            bool ok = true;
            // S = Q_r K^T for the next K tile, once the softmax has read the previous S
            auto issue_s = [&](int r) -> bool {
                const uint32_t st = gk % DK_STAGES;
                if (!mbar_wait(bar_kfull + 8u * st, (gk / DK_STAGES) & 1u, abort_flag, status)) return false;
                if (gs > 0 && !mbar_wait(bar_sfree, (gs - 1) & 1u, abort_flag, status)) return false;
                tc_fence_after();
                const uint64_t kdesc = kdesc0 + (uint64_t)((st * D64_TILE) >> 4);
                const uint64_t qdesc = qdesc0 + (uint64_t)(((uint32_t)(r & 1) * D64_TILE) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ss(tmem_base + D64_S_COL, qdesc + (uint64_t)(kk * 2),
                                kdesc + (uint64_t)(kk * 2), idesc_s, kk > 0 ? 1u : 0u);
                tc_commit(bar_sfull);
                tc_commit(bar_kempty + 8u * st);
                ++gk;
                ++gs;
                return true;
            };
            // the first score MMA of item r (an item without keys has none; its Q load is
            // waited for by the softmax instead)
            auto start_item = [&](int r, const D64Item& it) -> bool {
                if (it.n == 0) return true;
                if (!mbar_wait(bar_qfull + 8u * (r & 1), (uint32_t)(r >> 1) & 1u, abort_flag, status))
                    return false;
                return issue_s(r);
            };
            D64Item cur = item(0);
            ok = start_item(0, cur);
            for (int r = 0; r < R && ok; ++r) {
                D64Item nxt;
                nxt.n = 0;
                if (r + 1 < R) nxt = item(r + 1);
                if (cur.n == 0 && r + 1 < R) ok = start_item(r + 1, nxt);
                for (int j = 0; j < cur.n && ok; ++j) {
                    if (j + 1 < cur.n)
                        ok = issue_s(r);
                    else if (r + 1 < R)
                        ok = start_item(r + 1, nxt);
                    if (!ok) break;
                    const uint32_t st = gv % DV_STAGES;
                    ok = mbar_wait(bar_vfull + 8u * st, (gv / DV_STAGES) & 1u, abort_flag, status) &&
                         mbar_wait(bar_pfull, gp & 1u, abort_flag, status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t vdesc = vdesc0 + (uint64_t)((st * D64_TILE) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_bf16_ts(tmem_base + D64_O_COL, tmem_base + D64_P_COL + kk * 8,
                                    vdesc + (uint64_t)((kk * 2048) >> 4), idesc_o,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_pvdone);
                    tc_commit(bar_vempty + 8u * st);
                    ++gv;
                    ++gp;
                }
                cur = nxt;
            }
            tc_commit(bar_drain);
            drain_wait_a(bar_drain, 0);
        }
      }
    } else {
        setmaxnreg_inc<D64_REGS_SOFTMAX>();
        // ---------------- softmax: thread = query row
        const int q = warp & 3;
        const int r_ = q * 32 + lane;
        const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
        const uint32_t sw = (uint32_t)(r_ & 7);
        uint32_t gs = 0, gp = 0;  // S read, P written
        bool ok = true;
        for (int r = 0; r < R && ok; ++r) {
            const D64Item it = item(r);
            const uint32_t sOut = sQ + (uint32_t)(r & 1) * D64_TILE;
            const int row = it.qrow0 + r_;
            if constexpr (GATE)  // this row's gate pre-activations, into L2 for the epilogue
                if (row < T_q) prefetch_l2(gate + ((int64_t)it.b * T_q + row) * ldg + (int64_t)it.head * 64);
            if (it.n == 0) {
                // no valid key: the softmax is undefined, the rows are NaN (written once the
                // item's Q load, which targets the same buffer, has landed)
                ok = __all_sync(0xffffffffu, mbar_wait(bar_qfull + 8u * (r & 1), (uint32_t)(r >> 1) & 1u,
                                                       abort_flag, status));
                if (!ok) break;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(sOut + r_ * 128 + ((u ^ sw) << 4), 0x7FC07FC0u, 0x7FC07FC0u,
                                 0x7FC07FC0u, 0x7FC07FC0u);
            } else {
                float m = -INFINITY;  // reference maximum, already scaled to base 2
                float l = 0.f;
                const int L = kv_lengths != nullptr ? kv_lengths[it.b] : T_kv;
                for (int j = 0; j < it.n && ok; ++j) {
                    // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
                    if (!__all_sync(0xffffffffu, mbar_wait(bar_sfull, gs & 1u, abort_flag, status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int kv0 = j * 128;
                    const bool masked = kv0 + 128 > L || (causal && kv0 + 127 > it.qrow0);
                    const int lim = causal ? min(L, row + 1) : L;  // keys [0, lim) are visible
                    float x[128];
                    load_s_tile(trow + D64_S_COL, masked, kv0, lim, x);
                    tc_fence_before();
                    mbar_arrive(bar_sfree);
                    ++gs;
                    // P against the current reference m, each half stored to TMEM as soon as it
                    // is computed; any reference gives the same O / l, it only has to keep P
                    // finite.  The first tile, or any tile where some row's sum would exceed
                    // 2^64, takes the exact row maximum as the new reference instead (and
                    // rescales O); the P stores of the fast attempt are simply overwritten.
                    const uint64_t c2 = pack2(scale_log2, scale_log2);
                    float rowsum = 0.f, alpha = 1.f;
                    bool slow = j == 0;
                    if (!slow) {
                        uint32_t pk[32];
                        rowsum = exp_half(x, 0, c2, -m, pk);
                        // the previous PV product is done: O is stable and the P columns are free
                        if (!__all_sync(0xffffffffu, mbar_wait(bar_pvdone, (gp - 1) & 1u, abort_flag, status))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        tmem_st32(trow + D64_P_COL, pk);
                        rowsum += exp_half(x, 1, c2, -m, pk);
                        tmem_st32(trow + D64_P_COL + 32, pk);
                        slow = !__all_sync(0xffffffffu, rowsum <= 18446744073709551616.f);
                    }
                    if (slow) {
                        const float m_tile = row_max(x) * scale_log2;
                        const float m_new = m_tile > m ? m_tile : m;
                        alpha = ex2_approx(m - m_new);  // 0 on the first tile (m = -inf)
                        const bool rescale = (m_new != m) && j > 0;
                        if (__any_sync(0xffffffffu, rescale)) {
                            const float a = rescale ? alpha : 1.f;
#pragma unroll
                            for (int cc = 0; cc < 2; ++cc) {
                                uint32_t o[32];
                                tmem_ld32(trow + D64_O_COL + cc * 32, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                                tmem_st32(trow + D64_O_COL + cc * 32, o);
                            }
                        }
                        const float neg = m_new == -INFINITY ? 0.f : -m_new;
                        uint32_t pk[32];
                        rowsum = exp_half(x, 0, c2, neg, pk);
                        tmem_st32(trow + D64_P_COL, pk);
                        rowsum += exp_half(x, 1, c2, neg, pk);
                        tmem_st32(trow + D64_P_COL + 32, pk);
                        m = m_new;
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar_pfull);
                    ++gp;
                    l = l * alpha + rowsum;
                }
                // the gate pre-activations of this row, loaded while the last PV product runs
                uint4 gv[GATE ? 8 : 1];
                if constexpr (GATE) {
                    const uint4* g4 = reinterpret_cast<const uint4*>(gate + ((int64_t)it.b * T_q + row) * ldg +
                                                                     (int64_t)it.head * 64);
#pragma unroll
                    for (int i = 0; i < 8; ++i) gv[i] = row < T_q ? __ldg(g4 + i) : make_uint4(0u, 0u, 0u, 0u);
                }
                if (!ok || !__all_sync(0xffffffffu, mbar_wait(bar_pvdone, (gp - 1) & 1u, abort_flag, status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float inv = 1.f / l;
                // O / l (times the gate) as bf16 into the item's Q buffer (its last score MMA
                // has completed)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(trow + D64_O_COL + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int u4 = 0; u4 < 4; ++u4) {
                        const int u = cc * 4 + u4;
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(o[u4 * 8 + i]) * inv;
                        if constexpr (GATE) apply_gate8(gv[cc * 4 + u4], f);
                        st_shared_v4(sOut + r_ * 128 + (((uint32_t)u ^ sw) << 4),
                                     pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                     pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
                // the next item's PV product overwrites O: the reads above must be complete
                tc_fence_before();
            }
            fence_proxy_async_smem();
            mbar_arrive(bar_staged + 8u * (r & 1));
        }
    }

    // lanes that skipped a one-thread role wait here for it: the CTA barrier below must
    // see whole warps, or it can complete while a role is still running
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, D64_TMEM_COLS);
    }
}

cudaError_t launch_attn_d64(const void* Q, int64_t ldq, const void* K, int64_t ldk,
                            const void* V, int64_t ldv, const void* G, int64_t ldg, void* O,
                            int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int causal,
                            const int32_t* kv_lengths, int num_sms, int* status,
                            cudaStream_t stream) {
    CUtensorMap tQ, tK, tV, tO;
    const uint32_t box[3] = {64, 128, 1};
    {
        const uint64_t dims[3] = {(uint64_t)h * 64, (uint64_t)T_q, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldq * 2, (uint64_t)ldq * 2 * (uint64_t)T_q};
        if (!encode_tmap_bf16(&tQ, Q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h_kv * 64, (uint64_t)T_kv, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldk * 2, (uint64_t)ldk * 2 * (uint64_t)T_kv};
        if (!encode_tmap_bf16(&tK, K, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h_kv * 64, (uint64_t)T_kv, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldv * 2, (uint64_t)ldv * 2 * (uint64_t)T_kv};
        if (!encode_tmap_bf16(&tV, V, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h * 64, (uint64_t)T_q, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldo * 2, (uint64_t)ldo * 2 * (uint64_t)T_q};
        if (!encode_tmap_bf16(&tO, O, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    // setmaxnreg.inc waits until the CTA's register pool (threads x registers at launch) can
    // grant the rise: refuse to launch a build whose register count cannot cover the split
    const bool sorted = kv_lengths != nullptr && !causal && B <= D64_SORT_MAX_B;
    auto kernel = G != nullptr ? (sorted ? attn_bf16_d64_kernel<true, true> : attn_bf16_d64_kernel<true, false>)
                               : (sorted ? attn_bf16_d64_kernel<false, true> : attn_bf16_d64_kernel<false, false>);
    static std::atomic<int> pool_ok[4] = {{-1}, {-1}, {-1}, {-1}};
    std::atomic<int>& slot = pool_ok[(G != nullptr ? 2 : 0) + (sorted ? 1 : 0)];
    int ok = slot.load(std::memory_order_relaxed);
    if (ok < 0) {
        cudaFuncAttributes fa;
        const cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        ok = fa.numRegs * D64_THREADS >= 128 * (D64_REGS_CTRL + D64_REGS_SOFTMAX) ? 1 : 0;
        slot.store(ok, std::memory_order_relaxed);
    }
    if (!ok) return cudaErrorInvalidConfiguration;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, D64_SMEM);
    if (err != cudaSuccess) return err;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt(64.0));
    const int64_t items = (int64_t)B * h * ((T_q + 127) / 128);
    if (items > INT32_MAX) return cudaErrorInvalidValue;
    const int64_t slots = 2 * (int64_t)(num_sms > 0 ? num_sms : 1);
    const int grid = (int)(items < slots ? items : slots);
    return launch_pdl(kernel, dim3(grid), dim3(D64_THREADS), D64_SMEM, stream, tQ, tK, tV,
                      tO, B, h, h_kv, T_q, T_kv, causal, kv_lengths,
                      reinterpret_cast<const __nv_bfloat16*>(G), ldg, scale_log2, status);
}

template <int HD>
cudaError_t launch_attn_hd(const void* Q, int64_t ldq, const void* K, int64_t ldk, const void* V,
                           int64_t ldv, const void* G, int64_t ldg, void* O, int64_t ldo, int B,
                           int h, int h_kv, int T_q, int T_kv, int causal,
                           const int32_t* kv_lengths, int* status, cudaStream_t stream) {
    using C = AttnCfg<HD>;
    CUtensorMap tQ, tK, tV, tO;
    const uint32_t box[3] = {64, 128, 1};
    {
        const uint64_t dims[3] = {(uint64_t)h * HD, (uint64_t)T_q, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldq * 2, (uint64_t)ldq * 2 * (uint64_t)T_q};
        if (!encode_tmap_bf16(&tQ, Q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h_kv * HD, (uint64_t)T_kv, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldk * 2, (uint64_t)ldk * 2 * (uint64_t)T_kv};
        if (!encode_tmap_bf16(&tK, K, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h_kv * HD, (uint64_t)T_kv, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldv * 2, (uint64_t)ldv * 2 * (uint64_t)T_kv};
        if (!encode_tmap_bf16(&tV, V, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {(uint64_t)h * HD, (uint64_t)T_q, (uint64_t)B};
        const uint64_t strides[2] = {(uint64_t)ldo * 2, (uint64_t)ldo * 2 * (uint64_t)T_q};
        if (!encode_tmap_bf16(&tO, O, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    auto kernel = G != nullptr ? attn_bf16_tc_kernel<HD, true> : attn_bf16_tc_kernel<HD, false>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    const float scale_log2 = (float)(1.4426950408889634 / sqrt((double)HD));
    const int rows_per_cta = C::NQ * C::BM;
    const int BH = B * h;
    const int n_qb = (T_q + rows_per_cta - 1) / rows_per_cta;
    // (batch, head) pairs per group: the K/V of one group (4 T_kv d bytes per pair) within
    // MHA_D128_GROUP_BYTES
    const int64_t kv_head_bytes = 4 * (int64_t)T_kv * HD;
    int64_t hg = (int64_t)MHA_D128_GROUP_BYTES / (kv_head_bytes > 0 ? kv_head_bytes : 1);
    hg = hg < 1 ? 1 : (hg > BH ? BH : hg);
    const int64_t ctas = (int64_t)BH * n_qb;
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    return launch_pdl(kernel, dim3((unsigned)ctas), dim3(A_THREADS), C::SMEM, stream, tQ, tK, tV, tO,
                      h, h_kv, T_q, T_kv, causal, kv_lengths, reinterpret_cast<const __nv_bfloat16*>(G),
                      ldg, scale_log2, status, BH, n_qb, (int)hg);
}

}  // namespace

cudaError_t launch_attn_bf16(const void* Q, int64_t ldq, const void* K, int64_t ldk,
                             const void* V, int64_t ldv, const void* G, int64_t ldg, void* O,
                             int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int d, int causal,
                             const int32_t* kv_lengths, int num_sms, int* status,
                             cudaStream_t stream) {
    // d = 64: the persistent kernel, two CTAs per SM, whose fixed longest-first item order
    // balances the causal triangle and, with key lengths, the batches' lengths
    if (d == 64)
        return launch_attn_d64(Q, ldq, K, ldk, V, ldv, G, ldg, O, ldo, B, h, h_kv, T_q, T_kv, causal,
                               kv_lengths, num_sms, status, stream);
    if (d == 128)
        return launch_attn_hd<128>(Q, ldq, K, ldk, V, ldv, G, ldg, O, ldo, B, h, h_kv, T_q, T_kv, causal,
                                   kv_lengths, status, stream);
    return cudaErrorInvalidValue;
}

}  // namespace mha
