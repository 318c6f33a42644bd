// simt_f32.cu -- the fp32 path on CUDA cores (FFMA), for layers stored in fp32.
// fp32 results must agree with the exact result to about 1e-5 relative; TF32 tensor cores
// (10-bit mantissa) cannot, so both steps run in full fp32:
//   gemm_f32_kernel  C = A W + bias (+ R)   (itwiki.kr "멀티 헤드 어텐션", table rows 투영,
//                    출력 투영; the residual R of iamjaehka13.blog "[Deep Learning 5]
//                    Attention의 내부 계산", section 14)
//   attn_f32_tiled_kernel (the forward) and attn_f32_kernel (the decode step)
//                    online-softmax attention for every head, any d_k, d_v <= 256, written
//                    into the Concat layout (same page, 수식 and the shape table;
//                    iamjaehka13.blog sections 9-10), with grouped K/V heads and the sigmoid
//                    output gate (itwiki.kr, 추론 비용과 변형), and a decode mode in which
//                    the T_q rows are the last T_q of the L_b keys (a KV-cache step)
#include <math.h>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int F_BN = 64;

// 64 x 64 output tile per block of 128 threads, 8 x 4 outputs per thread (rows 8 ty..,
// columns 4 tx..), K consumed in slices of BK.  Per k step a thread reads 8 A and 4 W values
// (three 16-byte shared loads) for 32 multiply-adds, issued as 16 packed `fma.rn.f32x2`
// (two IEEE fp32 fmas each: row pairs of A times a broadcast W value), so the FMA pipe, not
// instruction issue, sets the pace.  Shared-memory tiles are double-buffered: the next slice
// is loaded from global memory into registers while the current one is multiplied, then
// stored to the other buffer, one barrier per slice.  A is staged transposed (As[k][m]) so
// that both operands of a product step are 16-byte shared loads.  The K loop runs in order
// (k = 0, 1, ...) with one fma per product.  VEC: A and W 16-byte aligned with row strides a
// multiple of 4 floats, so that four consecutive elements of a row are one 16-byte global
// load.
//
// SPLIT: a cluster of gridDim.z CTAs (2, 4 or 8) shares each tile, rank z multiplying the K slices
// [z * kper, (z + 1) * kper); the fp32 partial tiles meet in distributed shared memory, where
// rank z adds rows [z * 64 / S, (z + 1) * 64 / S) of all S partials in rank order (so the sum
// does not depend on timing), then bias and residual, and writes C.  For grids of too few tiles
// to keep several warps per scheduler busy.
template <int BK, bool VEC, bool SPLIT>
__global__ void __launch_bounds__(128)
    gemm_f32_kernel(const float* __restrict__ A, int64_t lda, const float* __restrict__ W,
                    int64_t ldw, const float* __restrict__ bias, const float* R, int64_t ldr,
                    float* C, int64_t ldc, int M, int N, int K, int kper) {
    constexpr int BM = 64, THREADS = 128;
    constexpr int NA = BM * BK / 4 / THREADS;  // 4-element pieces of A per thread and slice
    constexpr int NW = BK * F_BN / 4 / THREADS;
    static_assert(NA >= 1 && NW >= 1, "slice smaller than the block");
    __shared__ __align__(16) float As[2][BK][BM + 4];     // As[buf][k][m]
    __shared__ __align__(16) float Ws[2][BK][F_BN + 4];   // Ws[buf][k][n]
    const int tid = (int)threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int m0 = blockIdx.y * BM;
    const int n0 = blockIdx.x * F_BN;
    const int kbeg = SPLIT ? (int)blockIdx.z * kper : 0;
    const int kend = SPLIT ? min(K, kbeg + kper) : K;  // loads past kend read as zeros
    float ra[NA][4], rw[NW][4];
    auto load = [&](int k0) {
#pragma unroll
        for (int c = 0; c < NA; ++c) {
            const int idx = tid + c * THREADS;
            const int gm = m0 + idx / (BK / 4), gk = k0 + (idx % (BK / 4)) * 4;
            if (VEC && gm < M && gk + 3 < kend) {
                const float4 v = *reinterpret_cast<const float4*>(A + (int64_t)gm * lda + gk);
                ra[c][0] = v.x; ra[c][1] = v.y; ra[c][2] = v.z; ra[c][3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    ra[c][i] = (gm < M && gk + i < kend) ? A[(int64_t)gm * lda + gk + i] : 0.f;
            }
        }
#pragma unroll
        for (int c = 0; c < NW; ++c) {
            const int idx = tid + c * THREADS;
            const int gw = k0 + idx / 16, gn = n0 + (idx % 16) * 4;
            if (VEC && gw < kend && gn + 3 < N) {
                const float4 v = *reinterpret_cast<const float4*>(W + (int64_t)gw * ldw + gn);
                rw[c][0] = v.x; rw[c][1] = v.y; rw[c][2] = v.z; rw[c][3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    rw[c][i] = (gw < kend && gn + i < N) ? W[(int64_t)gw * ldw + gn + i] : 0.f;
            }
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int c = 0; c < NA; ++c) {
            const int idx = tid + c * THREADS;
            const int r = idx / (BK / 4), k4 = (idx % (BK / 4)) * 4;
#pragma unroll
            for (int i = 0; i < 4; ++i) As[buf][k4 + i][r] = ra[c][i];
        }
#pragma unroll
        for (int c = 0; c < NW; ++c) {
            const int idx = tid + c * THREADS;
            *reinterpret_cast<float4*>(&Ws[buf][idx / 16][(idx % 16) * 4]) =
                make_float4(rw[c][0], rw[c][1], rw[c][2], rw[c][3]);
        }
    };

    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    load(kbeg);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = kbeg; k0 < kend; k0 += BK) {
        const bool more = k0 + BK < kend;
        if (more) load(k0 + BK);  // in flight while this slice is multiplied
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 8 + 4]);
            const float4 b4 = *reinterpret_cast<const float4*>(&Ws[buf][kk][tx * 4]);
            // rows (2p, 2p + 1) of the thread's eight, each W value in both halves
            const uint64_t ap[4] = {pack2(a0.x, a0.y), pack2(a0.z, a0.w), pack2(a1.x, a1.y),
                                    pack2(a1.z, a1.w)};
            const uint64_t bp[4] = {pack2(b4.x, b4.x), pack2(b4.y, b4.y), pack2(b4.z, b4.z),
                                    pack2(b4.w, b4.w)};
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    unpack2(fma2(ap[p], bp[j], pack2(acc[2 * p][j], acc[2 * p + 1][j])), acc[2 * p][j],
                            acc[2 * p + 1][j]);
        }
        if (more) store(buf ^ 1);  // the other buffer was last read before the previous barrier
        __syncthreads();
        buf ^= 1;
    }
    if constexpr (SPLIT) {
        // the partial tile, row-major 64 x 64, over the A buffers (free after the last barrier)
        float* part = &As[0][0][0];
        static_assert(sizeof(As) >= BM * F_BN * sizeof(float), "partial tile does not fit");
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(part + (ty * 8 + i) * F_BN + tx * 4) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        cluster_sync_all();
        const int S = (int)gridDim.z;
        const int rank = (int)cluster_ctarank();
        const int rows = BM / S;  // S divides 64
        const uint32_t pbase = smem_u32(part);
        for (int e = tid; e < rows * (F_BN / 4); e += THREADS) {
            const int r = rank * rows + e / (F_BN / 4);
            const int c4 = (e % (F_BN / 4)) * 4;
            const uint32_t off = pbase + (uint32_t)((r * F_BN + c4) * 4);
            float4 sum = ld_shared_cluster_v4(mapa_shared(off, 0));
            for (int z = 1; z < S; ++z) {
                const float4 p = ld_shared_cluster_v4(mapa_shared(off, (uint32_t)z));
                sum.x += p.x;
                sum.y += p.y;
                sum.z += p.z;
                sum.w += p.w;
            }
            const int gm = m0 + r;
            if (gm < M) {
                const float v[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int gn = n0 + c4 + j;
                    if (gn < N)
                        C[(int64_t)gm * ldc + gn] =
                            v[j] + (bias ? bias[gn] : 0.f) + (R ? R[(int64_t)gm * ldr + gn] : 0.f);
                }
            }
        }
        __syncwarp();
        cluster_sync_all();  // every partial stays until its readers are done
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gm = m0 + ty * 8 + i;
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

// ---------------------------------------------------------------------------------------
// Tiled fp32 attention (the forward; the decode step keeps the kernel above): one block =
// BQ = 16 RQ query rows of one (batch, head), 256 threads, key tiles of 64.  Per key tile the
// block forms the BQ x 64 score tile as a small matrix product (thread = RQ rows x 4 keys),
// masks it, updates the online softmax (row maximum and sum over the 16 threads sharing the
// rows, by shuffles), stages P in shared memory and adds P V to its RQ x (4 CV) outputs
// (columns c*64 + 4 tx + i).  Q and K are staged transposed (Qs[e][q], Ks[e][j]) so that a
// product step reads 16 bytes of each; V and P row-major.  Causal: key tiles past the block's
// last row are skipped.  d_k any size, d_v <= 64 CV.
constexpr int FT_BK = 64;
constexpr int FT_THREADS = 256;
constexpr int FT_PAD = 4;  // row padding of the transposed and P tiles (floats)

__host__ __device__ constexpr int ft_bq(int RQ) { return 16 * RQ; }

template <int RQ, int CV>
__global__ void __launch_bounds__(FT_THREADS)
    attn_f32_tiled_kernel(const float* __restrict__ Q, int64_t ldq, const float* __restrict__ K,
                          int64_t ldk, const float* __restrict__ V, int64_t ldv,
                          const float* __restrict__ G, int64_t ldg, float* __restrict__ O,
                          int64_t ldo, int h, int h_kv, int T_q, int T_kv, int dk, int dv,
                          int causal, const int32_t* __restrict__ kv_lengths, float scale,
                          int* status) {
    constexpr int BQ = ft_bq(RQ);
    constexpr int QS = BQ + FT_PAD;      // row stride of Qs
    constexpr int KS = FT_BK + FT_PAD;   // row stride of Ks and Ps
    constexpr int VS = 64 * CV;          // row stride of Vs
    extern __shared__ __align__(16) float fsm[];
    const int dk4 = (dk + 3) & ~3;
    float* Qs = fsm;                 // [dk4][QS]
    float* Ks = Qs + dk4 * QS;       // [dk4][KS]
    float* Vs = Ks + dk4 * KS;       // [FT_BK][VS]
    float* Ps = Vs + FT_BK * VS;     // [BQ][KS]
    const int tid = (int)threadIdx.x;
    const int tx = tid & 15;  // keys 4 tx .. 4 tx + 3 of a score tile; output columns c*64 + 4 tx ..
    const int ty = tid >> 4;  // rows RQ ty .. RQ ty + RQ - 1
    const int bh = blockIdx.x;
    const int b = bh / h, head = bh - b * h;
    const int kvh = head / (h / h_kv);
    const int qb = causal ? (int)(gridDim.y - 1 - blockIdx.y) : (int)blockIdx.y;  // long blocks first
    const int q0 = qb * BQ;
    const int L = kv_lengths ? kv_lengths[b] : T_kv;
    if (L < 1 || L > T_kv) {
        if (tid == 0) record_status(status, kStatusBadLength);
        for (int i = tid; i < BQ * dv; i += FT_THREADS) {
            const int r = i / dv, e = i - r * dv;
            if (q0 + r < T_q) O[((int64_t)b * T_q + q0 + r) * ldo + (int64_t)head * dv + e] = NAN;
        }
        return;
    }
    // Q tile, transposed; rows past T_q and columns past d_k are zero
    for (int i = tid; i < BQ * (dk4 / 4); i += FT_THREADS) {
        const int q = i % BQ, e4 = (i / BQ) * 4;
        const int t = q0 + q;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            Qs[(e4 + c) * QS + q] = (t < T_q && e4 + c < dk)
                                        ? Q[((int64_t)b * T_q + t) * ldq + (int64_t)head * dk + e4 + c] : 0.f;
    }
    int kv_end = L;
    if (causal && kv_end > q0 + BQ) kv_end = q0 + BQ;

    float m[RQ], l[RQ], o[RQ][4 * CV];
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int u = 0; u < 4 * CV; ++u) o[r][u] = 0.f;
    }
    for (int kt0 = 0; kt0 < kv_end; kt0 += FT_BK) {
        __syncthreads();  // the previous tile's K, V and P are no longer read
        for (int i = tid; i < FT_BK * (dk4 / 4); i += FT_THREADS) {
            const int j = i % FT_BK, e4 = (i / FT_BK) * 4;
            const int key = kt0 + j;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                Ks[(e4 + c) * KS + j] = (key < T_kv && e4 + c < dk)
                                            ? K[((int64_t)b * T_kv + key) * ldk + (int64_t)kvh * dk + e4 + c] : 0.f;
        }
        for (int i = tid; i < FT_BK * (VS / 4); i += FT_THREADS) {
            const int j = i / (VS / 4), e4 = (i - j * (VS / 4)) * 4;
            const int key = kt0 + j;
            float v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                v[c] = (key < T_kv && e4 + c < dv) ? V[((int64_t)b * T_kv + key) * ldv + (int64_t)kvh * dv + e4 + c] : 0.f;
            *reinterpret_cast<float4*>(&Vs[j * VS + e4]) = make_float4(v[0], v[1], v[2], v[3]);
        }
        __syncthreads();
        // scores of this thread's RQ rows x 4 keys
        float sc[RQ][4];
#pragma unroll
        for (int r = 0; r < RQ; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) sc[r][c] = 0.f;
#pragma unroll 4
        for (int e = 0; e < dk4; ++e) {
            float a[RQ];
            if constexpr (RQ == 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(&Qs[e * QS + ty * 4]);
                a[0] = a4.x; a[1] = a4.y; a[2] = a4.z; a[3] = a4.w;
            } else {
                const float2 a2 = *reinterpret_cast<const float2*>(&Qs[e * QS + ty * RQ]);
                a[0] = a2.x; a[1] = a2.y;
            }
            const float4 k4 = *reinterpret_cast<const float4*>(&Ks[e * KS + tx * 4]);
            const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int r = 0; r < RQ; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[r][c] = fmaf(a[r], kk[c], sc[r][c]);
        }
        // mask, online softmax (the 16 threads of a half-warp share their rows)
#pragma unroll
        for (int r = 0; r < RQ; ++r) {
            const int t = q0 + ty * RQ + r;
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = kt0 + tx * 4 + c;
                const bool visible = key < L && !(causal && key > t);
                sc[r][c] = visible ? sc[r][c] * scale : -INFINITY;
                tmax = fmaxf(tmax, sc[r][c]);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
            const float m_new = fmaxf(m[r], tmax);
            float psum = 0.f;
            if (m_new == -INFINITY) {  // nothing visible to this row yet
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[r][c] = 0.f;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    sc[r][c] = expf(sc[r][c] - m_new);  // masked: exp(-inf) = 0
                    psum += sc[r][c];
                }
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            const float alpha = m_new == -INFINITY ? 1.f : expf(m[r] - m_new);  // 0 when m = -inf
            l[r] = l[r] * alpha + psum;
#pragma unroll
            for (int u = 0; u < 4 * CV; ++u) o[r][u] *= alpha;
            m[r] = m_new;
            *reinterpret_cast<float4*>(&Ps[(ty * RQ + r) * KS + tx * 4]) =
                make_float4(sc[r][0], sc[r][1], sc[r][2], sc[r][3]);
        }
        __syncthreads();
        // O += P V over the tile's keys, four at a time
        const int nk = min(FT_BK, kv_end - kt0);
        for (int j4 = 0; j4 < nk; j4 += 4) {
            float p[RQ][4];
#pragma unroll
            for (int r = 0; r < RQ; ++r) {
                const float4 p4 = *reinterpret_cast<const float4*>(&Ps[(ty * RQ + r) * KS + j4]);
                p[r][0] = p4.x; p[r][1] = p4.y; p[r][2] = p4.z; p[r][3] = p4.w;
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                for (int c = 0; c < CV; ++c) {
                    const float4 v4 = *reinterpret_cast<const float4*>(&Vs[(j4 + jj) * VS + c * 64 + tx * 4]);
                    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int r = 0; r < RQ; ++r)
#pragma unroll
                        for (int u = 0; u < 4; ++u) o[r][c * 4 + u] = fmaf(p[r][jj], v[u], o[r][c * 4 + u]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
        const int t = q0 + ty * RQ + r;
        if (t >= T_q) continue;
        const float inv = 1.f / l[r];
#pragma unroll
        for (int c = 0; c < CV; ++c)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = c * 64 + tx * 4 + u;
                if (e >= dv) continue;
                float y = o[r][c * 4 + u] * inv;
                if (G != nullptr) y *= 1.f / (1.f + expf(-G[((int64_t)b * T_q + t) * ldg + (int64_t)head * dv + e]));
                O[((int64_t)b * T_q + t) * ldo + (int64_t)head * dv + e] = y;
            }
    }
}

template <int RQ, int CV>
cudaError_t launch_attn_f32_tiled(const float* Q, int64_t ldq, const float* K, int64_t ldk,
                                  const float* V, int64_t ldv, const float* G, int64_t ldg, float* O,
                                  int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int d_k,
                                  int d_v, int causal, const int32_t* kv_lengths, int* status,
                                  cudaStream_t stream) {
    constexpr int BQ = ft_bq(RQ);
    const int dk4 = (d_k + 3) & ~3;
    const size_t smem = sizeof(float) * ((size_t)dk4 * (BQ + FT_PAD) + (size_t)dk4 * (FT_BK + FT_PAD) +
                                         (size_t)FT_BK * 64 * CV + (size_t)BQ * (FT_BK + FT_PAD));
    if (smem > 232448) return cudaErrorInvalidValue;
    auto kernel = attn_f32_tiled_kernel<RQ, CV>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const float scale = (float)(1.0 / sqrt((double)d_k));
    const dim3 grid((unsigned)(B * h), (unsigned)((T_q + BQ - 1) / BQ));
    kernel<<<grid, FT_THREADS, smem, stream>>>(Q, ldq, K, ldk, V, ldv, G, ldg, O, ldo, h, h_kv, T_q,
                                               T_kv, d_k, d_v, causal, kv_lengths, scale, status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_f32(const float* A, int64_t lda, const float* W, int64_t ldw,
                            const float* bias, const float* R, int64_t ldr, float* C, int64_t ldc,
                            int M, int N, int K, cudaStream_t stream) {
    // 32-wide K slices: 16-wide ones measured slower on the 1024 x 512 x {1536, 512}
    // projections of the fp32 causal workload (43.7 / 28.4 against 42.4 / 20.3 us)
    constexpr int BK = 32;
    const dim3 grid((unsigned)((N + F_BN - 1) / F_BN), (unsigned)((M + 63) / 64));
    const bool vec = (reinterpret_cast<uintptr_t>(A) % 16 == 0) && (reinterpret_cast<uintptr_t>(W) % 16 == 0) &&
                     lda % 4 == 0 && ldw % 4 == 0;
    // no more tiles than SMs: split K over clusters of 4, of 8 up to half as many tiles as
    // SMs (measured on 64-1024 rows: 8 beats 4 beats 2 wherever all CTAs stay resident, 2 lost
    // 4% at 240 tiles), each rank at least two K slices
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    const int64_t tiles = (int64_t)grid.x * grid.y;
    const int slices = (K + BK - 1) / BK;
    int S = 1;
    if (tiles <= (int64_t)sms) S = tiles * 2 <= (int64_t)sms ? 8 : 4;
    while (S > 1 && slices < 2 * S) S /= 2;
    if (S > 1) {
        const int kper = (slices + S - 1) / S * BK;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid.x, grid.y, (unsigned)S);
        cfg.blockDim = dim3(128);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = (unsigned)S;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t err =
            vec ? cudaLaunchKernelEx(&cfg, gemm_f32_kernel<BK, true, true>, A, lda, W, ldw, bias, R, ldr, C, ldc,
                                     M, N, K, kper)
                : cudaLaunchKernelEx(&cfg, gemm_f32_kernel<BK, false, true>, A, lda, W, ldw, bias, R, ldr, C, ldc,
                                     M, N, K, kper);
        if (err == cudaSuccess) return err;
        cudaGetLastError();  // no room for the clusters here: one CTA per tile below
    }
    if (vec)
        gemm_f32_kernel<BK, true, false><<<grid, 128, 0, stream>>>(A, lda, W, ldw, bias, R, ldr, C, ldc, M, N, K, K);
    else
        gemm_f32_kernel<BK, false, false><<<grid, 128, 0, stream>>>(A, lda, W, ldw, bias, R, ldr, C, ldc, M, N, K, K);
    return cudaGetLastError();
}

cudaError_t launch_attn_f32(const float* Q, int64_t ldq, const float* K, int64_t ldk,
                            const float* V, int64_t ldv, const float* G, int64_t ldg, float* O,
                            int64_t ldo, int B, int h, int h_kv, int T_q, int T_kv, int d_k, int d_v,
                            int causal, int decode, const int32_t* kv_lengths, int* status,
                            cudaStream_t stream) {
    if (!decode && d_v <= 256) {
        // the forward: tiled kernel; 32-row blocks when 64-row ones would not fill the GPU twice
        const bool small = (int64_t)B * h * ((T_q + 63) / 64) < 256;
        const int cv = (d_v + 63) / 64;
#define MHA_FT(RQ, CV)                                                                                  \
    if ((small ? 2 : 4) == RQ && cv == CV)                                                              \
        return launch_attn_f32_tiled<RQ, CV>(Q, ldq, K, ldk, V, ldv, G, ldg, O, ldo, B, h, h_kv, T_q, \
                                             T_kv, d_k, d_v, causal, kv_lengths, status, stream);
        MHA_FT(2, 1) MHA_FT(2, 2) MHA_FT(2, 3) MHA_FT(2, 4)
        MHA_FT(4, 1) MHA_FT(4, 2) MHA_FT(4, 3) MHA_FT(4, 4)
#undef MHA_FT
    }
    // the decode step (a few new rows over a long cache): 16-row blocks
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
