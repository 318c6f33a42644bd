// gemm_bf16.cu -- the projection steps on tcgen05 tensor cores:
//   C = A W + bias (+ R)   (A (M,K) bf16, W (K,N) bf16 (in,out) row-major, fp32 accumulate,
//                           optional bf16 residual R (M,N), C bf16)
// which is [Q|K|V] = X W_qkv + b_qkv and Y = Ocat W_o + b_o of
// itwiki.kr "멀티 헤드 어텐션", tensor-shape table rows 투영 and 출력 투영, and the residual
// form X' = X + O W_O of iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", section 14.
//
// Four warp-specialised kernels (the host picks one per shape):
//   gemm_bf16_splitk_kernel M <= 128 (a decode step's tokens): clusters of CTAs split K over
//                           128 x 128 tiles (128 x 256 where clusters of two over the narrow
//                           ones would not all fit at once) and add their fp32 partials
//                           through distributed shared memory;
//   gemm_bf16_tc_kernel     M <= 128 where no split applies: one CTA per SM, persistent over
//                           128 x 256 tiles;
//   gemm_bf16_pair_kernel   CTA pairs (cta_group::2), 256 x 256 tiles, persistent; optionally
//                           a second, independent projection in the same grid
//                           (cross-attention's query side next to its key / value side);
//   gemm_bf16_pairT_kernel  CTA pairs with the accumulator transposed, 192 x 256 tiles, where
//                           their rounds over the pairs cost less.
// Roles, as in the one-CTA kernel:
//   warp 0      TMA producer: A tile 128x64 (K-major, 128B swizzle) and W tile 64x256
//               (N-major: four 64x64 boxes) into a 4-stage shared-memory ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma (M=128, N=256, K=16)
//               from one thread; accumulators double-buffered in TMEM (2 x 256 columns) so
//               the epilogue of tile i overlaps the main loop of tile i+1;
//   warps 2..5  epilogue: tcgen05.ld the fp32 accumulator (one TMEM lane = one output row),
//               add bias, round to bf16, stage 32x64 sub-tiles in swizzled shared memory
//               and write them with TMA stores (double-buffered per warp).
// W stays in its natural (in,out) layout: the MMA reads it as an MN-major operand, so no
// transpose pass over the weights is needed.  Ragged M, N, K are handled by TMA bounds
// (zero fill on loads, clipping on stores).
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace mha {
namespace {

constexpr int G_BM = 128;
constexpr int G_BN = 256;
constexpr int G_BK = 64;
constexpr int G_STAGES = 4;
constexpr int G_A_BYTES = G_BM * G_BK * 2;  // 16 KB
constexpr int G_B_CHUNK = G_BK * 64 * 2;    // 8 KB: 64 K-rows x 64 N-columns
constexpr int G_B_BYTES = G_BK * G_BN * 2;  // 32 KB
constexpr int G_EPI_BUF = 32 * 64 * 2;      // 4 KB: 32 rows x 64 columns
constexpr int G_EPI_BYTES = 4 * 2 * G_EPI_BUF;
constexpr int G_BAR_BYTES = 256;
constexpr int G_SMEM = G_STAGES * (G_A_BYTES + G_B_BYTES) + G_EPI_BYTES + G_BAR_BYTES + 1024;
constexpr int G_THREADS = 192;
constexpr uint32_t G_TMEM_COLS = 512;

static_assert(G_SMEM <= 232448, "shared memory budget");

// Bounded wait that ignores the abort flag: used only to drain copies / MMAs still in
// flight before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) return;
    }
}

// One bf16 (x rounded to nearest even) to shared memory.
__device__ __forceinline__ void st_shared_b16(uint32_t addr, float x) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<const unsigned short*>(&h))
                 : "memory");
}

// Residual of one thread's row for the 64 columns of chunk c (zeros outside C).
__device__ __forceinline__ void load_residual(const __nv_bfloat16* R, int64_t ldr, int row, int nc, int M,
                                              int N, uint4 (&dst)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u)
        dst[u] = row < M && nc + u * 8 < N
                     ? __ldg(reinterpret_cast<const uint4*>(R + (int64_t)row * ldr + nc + u * 8))
                     : make_uint4(0u, 0u, 0u, 0u);
}

// The bias of a tile's G_BN columns spread over one warp: lane l holds columns n0 + 8l .. 8l + 7
// (N is a multiple of 8).  Loaded before the accumulator is ready, so that the epilogue reads
// it by shuffles instead of waiting on global loads.
__device__ __forceinline__ uint4 load_bias_lanes(const __nv_bfloat16* bias, int n0, int N, int lane) {
    const int c = n0 + lane * 8;
    return bias != nullptr && c < N ? __ldg(reinterpret_cast<const uint4*>(bias + c))
                                    : make_uint4(0u, 0u, 0u, 0u);
}

// Epilogue of one warp's share of an accumulator tile: 32 rows (the warp's TMEM lane quarter,
// one row per thread, starting at row m0w of C) x G_BN columns from TMEM address t0, written as
// C = acc + bias (+ R) in bf16 through the warp's two 4 KB staging buffers (buf0, buf0 + 4 KB)
// and 32x64 TMA stores.  The TMEM read of chunk c + 1 is in flight while chunk c is converted,
// so only the first read's latency is exposed; release() runs as soon as the whole accumulator
// has been read, before the last chunk is converted.
template <bool RESID, typename Release>
__device__ __forceinline__ void epilogue_rows(uint32_t t0, uint4 bvec, bool has_bias, int m0w, int n0, int lane,
                                              uint32_t buf0, uint32_t& bufsel, const CUtensorMap* tmC,
                                              const __nv_bfloat16* R, int64_t ldr, int M, int N,
                                              uint4 (&res)[RESID ? 8 : 1], Release release) {
    constexpr int NCH = G_BN / 64;
    uint32_t va[2][32], vb[2][32];
    uint4 rnext[RESID ? 8 : 1];
    const int row = m0w + lane;
    tmem_ld32(t0, va[0]);
    tmem_ld32(t0 + 32, va[1]);
    tmem_wait_ld();
    reg_fence(va[0]);
    reg_fence(va[1]);
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        uint32_t(&cur)[2][32] = (c & 1) ? vb : va;
        uint32_t(&nxt)[2][32] = (c & 1) ? va : vb;
        if (c + 1 < NCH) {
            tmem_ld32(t0 + (c + 1) * 64, nxt[0]);
            tmem_ld32(t0 + (c + 1) * 64 + 32, nxt[1]);
        } else {
            release();  // every column of the accumulator is in registers
        }
        if constexpr (RESID) {
            if (c + 1 < NCH) load_residual(R, ldr, row, n0 + (c + 1) * 64, M, N, rnext);
        }
        const int nc = n0 + c * 64;
        if (nc < N && m0w < M) {  // else the sub-tile lies wholly outside C
            const uint32_t buf = buf0 + bufsel * (uint32_t)G_EPI_BUF;
            if (lane == 0) bulk_wait_group_read<1>();  // the store that last used buf has read it
            __syncwarp();
            const uint32_t srow = buf + (uint32_t)lane * 128u;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                float x[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(cur[u >> 2][(u & 3) * 8 + i]);
                if constexpr (RESID) {
                    const uint32_t rw[4] = {res[u].x, res[u].y, res[u].z, res[u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[2 * i] += __uint_as_float(rw[i] << 16);
                        x[2 * i + 1] += __uint_as_float(rw[i] & 0xFFFF0000u);
                    }
                }
                if (has_bias) {
                    const int src = c * 8 + u;
                    const uint32_t bw[4] = {__shfl_sync(0xffffffffu, bvec.x, src),
                                            __shfl_sync(0xffffffffu, bvec.y, src),
                                            __shfl_sync(0xffffffffu, bvec.z, src),
                                            __shfl_sync(0xffffffffu, bvec.w, src)};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[2 * i] += __uint_as_float(bw[i] << 16);
                        x[2 * i + 1] += __uint_as_float(bw[i] & 0xFFFF0000u);
                    }
                }
                st_shared_v4(srow + ((uint32_t)(u ^ (lane & 7)) << 4), pack_bf16x2(x[0], x[1]),
                             pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(tmC, buf, nc, m0w);
                bulk_commit_group();
            }
            bufsel ^= 1u;
        }
        if constexpr (RESID) {
            if (c + 1 < NCH)
#pragma unroll
                for (int u = 0; u < 8; ++u) res[u] = rnext[u];
        }
        if (c + 1 < NCH) {
            tmem_wait_ld();
            reg_fence(nxt[0]);
            reg_fence(nxt[1]);
        }
    }
}

// RESID: the epilogue adds the residual R (a separate instantiation, so that the plain
// projection carries none of its code or registers).
template <bool RESID>
__global__ void __launch_bounds__(G_THREADS, 1)
    gemm_bf16_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmC,
                        const __nv_bfloat16* __restrict__ bias, const __nv_bfloat16* R,
                        int64_t ldr, int M, int N, int K, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sA = base;
    const uint32_t sB = sA + G_STAGES * G_A_BYTES;
    const uint32_t sE = sB + G_STAGES * G_B_BYTES;
    const uint32_t sBar = sE + G_EPI_BYTES;
    // barrier layout: full[S], empty[S], tfull[2], tempty[2], mma_drain
    const uint32_t bar_full = sBar;
    const uint32_t bar_empty = sBar + 8u * G_STAGES;
    const uint32_t bar_tfull = sBar + 16u * G_STAGES;
    const uint32_t bar_tempty = bar_tfull + 16u;
    const uint32_t bar_drain = bar_tempty + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_m = (M + G_BM - 1) / G_BM;
    const int num_n = (N + G_BN - 1) / G_BN;
    const int num_tiles = num_m * num_n;
    const int num_k = (K + G_BK - 1) / G_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G_STAGES; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8u * a, 1);
            mbar_init(bar_tempty + 8u * a, 128);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), G_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // inputs may come from the previous kernel on the stream
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const int m0 = (tile % num_m) * G_BM;
                const int n0 = (tile / num_m) * G_BN;
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(bar_empty + 8u * stage, phase ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_full + 8u * stage;
                    mbar_arrive_expect_tx(fb, G_A_BYTES + G_B_BYTES);
                    tma_load_2d(sA + stage * G_A_BYTES, &tmA, kb * G_BK, m0, fb);
#pragma unroll
                    for (int c = 0; c < G_BN / 64; ++c)
                        tma_load_2d(sB + stage * G_B_BYTES + c * G_B_CHUNK, &tmW, n0 + c * 64,
                                    kb * G_BK, fb);
                    ++issued;
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every load issued must have landed before the CTA exits (on the normal path
            // these phases completed long ago and the waits return at once).
            for (int back = 0; back < G_STAGES && back < issued; ++back) {
                stage = stage == 0 ? G_STAGES - 1 : stage - 1;
                if (stage == G_STAGES - 1) phase ^= 1u;
                drain_wait(bar_full + 8u * stage, phase);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = idesc_bf16_f32(G_BM, G_BN, false, true);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(bar_tempty + 8u * acc, acc_phase ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * G_BN);
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(bar_full + 8u * stage, phase, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + stage * G_A_BYTES;
                    const uint32_t b0 = sB + stage * G_B_BYTES;
#pragma unroll
                    for (int k = 0; k < G_BK / 16; ++k) {
                        const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(b0 + k * 2048, G_B_CHUNK, 1024);
                        mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    tc_commit(bar_empty + 8u * stage);
                    if (++stage == G_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(bar_tfull + 8u * acc);
            }
            // all MMAs issued by this thread complete before TMEM is released
            tc_commit(bar_drain);
            drain_wait(bar_drain, 0);
        }
    } else {
        // ---------------- epilogue: warps 2..5, one TMEM lane (= output row) per thread
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int e = warp - 2;  // staging-buffer owner index
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint32_t bufsel = 0;
        int it = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
            const int m0 = (tile % num_m) * G_BM;
            const int n0 = (tile / num_m) * G_BN;
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            // bias and the first 64 residual columns are fetched while the tile's MMAs run
            const uint4 bvec = load_bias_lanes(bias, n0, N, lane);
            uint4 res[RESID ? 8 : 1];
            if constexpr (RESID) load_residual(R, ldr, m0 + q * 32 + lane, n0, M, N, res);
            // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8u * acc, acc_phase, abort_flag, status)))
                break;
            tc_fence_after();
            epilogue_rows<RESID>(tmem_base + lane_off + (uint32_t)(acc * G_BN), bvec, bias != nullptr,
                                 m0 + q * 32, n0, lane, sE + (uint32_t)(e * 2 * G_EPI_BUF), bufsel, &tmC, R,
                                 ldr, M, N, res, [&] {
                                     // accumulator read: hand it back to the MMA warp
                                     tc_fence_before();
                                     mbar_arrive(bar_tempty + 8u * acc);
                                 });
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // lanes that skipped a one-thread role wait here for it: the CTA barrier below must
    // see whole warps, or it can complete while a role is still running
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, G_TMEM_COLS);
    }
}


// ---------------------------------------------------------------------------------------
// At most 128 rows (the new tokens of a decode step) over few column tiles: the one-CTA kernel
// above reads all of W through a handful of SMs.  Here a cluster of S CTAs shares one 128 x BN
// tile (BN a multiple of 64; launched with 128): CTA r (its rank) runs the K blocks
// [r * kb_per, (r + 1) * kb_per), puts its fp32 partial tile into its own (by then idle) stage
// buffers, and after a cluster barrier reduces columns [r * BN / S, (r + 1) * BN / S) of the
// tile over all S partials, read in rank order through distributed shared memory (so the sum
// does not depend on timing), adds bias and residual and writes C.  A second cluster barrier
// keeps every partial alive until its readers are done.  Roles as above (warp 0 TMA, warp 1
// MMA, warps 2..5 epilogue); all six warps reduce.  Distributed shared memory moves only
// ~20-30 GB/s into each SM (measured, by loads, stores or bulk copies alike), so the exchange,
// M x BN x 4 x (S - 1) / S bytes per rank, is what bounds this kernel from a few dozen rows up.
// Partial layout: row r at r * BN * 4 bytes, its BN / 4 groups of four columns as float4s,
// the low three bits of the group index XORed with r & 7 so that the eight rows a
// quarter-warp writes hit different banks.
// One rank's share of the split kernel's reduction: column groups [g0, g0 + w) of rows [0, M),
// each the sum of the S partials in rank order (+ bias, + residual), written to C.  A thread
// takes U elements at a time and has all their U x S loads from distributed shared memory in
// flight before it adds any: each load is a round trip of several hundred cycles.
template <int S, int BN>
__device__ __forceinline__ void splitk_reduce(uint32_t sPart, int g0, int w, int M, int N, int n0,
                                              const __nv_bfloat16* __restrict__ bias,
                                              const __nv_bfloat16* __restrict__ R, int64_t ldr,
                                              __nv_bfloat16* __restrict__ C, int64_t ldc) {
    constexpr int U = S <= 2 ? 8 : (S <= 4 ? 4 : 2);  // at most 64 registers of loads
    const int count = M * w;
#pragma unroll 1
    for (int e0 = threadIdx.x; e0 < count; e0 += U * G_THREADS) {
        float4 p[U][S];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * G_THREADS;
            if (e < count) {
                const int row = e / w;
                const int g = g0 + e % w;
                const uint32_t off = (uint32_t)(row * BN * 4) + ((uint32_t)((g & ~7) | ((g ^ row) & 7)) << 4);
#pragma unroll
                for (int r = 0; r < S; ++r) p[u][r] = ld_shared_cluster_v4(mapa_shared(sPart + off, (uint32_t)r));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int e = e0 + u * G_THREADS;
            if (e >= count) break;
            const int row = e / w;
            const int n = n0 + (g0 + e % w) * 4;
            if (n >= N) continue;  // N is a multiple of 8: a group of four is all in or out
            float4 acc = p[u][0];
#pragma unroll
            for (int r = 1; r < S; ++r) {
                acc.x += p[u][r].x;
                acc.y += p[u][r].y;
                acc.z += p[u][r].z;
                acc.w += p[u][r].w;
            }
            if (bias != nullptr) {
                const uint2 bb = *reinterpret_cast<const uint2*>(bias + n);
                acc.x += __uint_as_float(bb.x << 16);
                acc.y += __uint_as_float(bb.x & 0xffff0000u);
                acc.z += __uint_as_float(bb.y << 16);
                acc.w += __uint_as_float(bb.y & 0xffff0000u);
            }
            if (R != nullptr) {
                const uint2 rr = *reinterpret_cast<const uint2*>(R + (int64_t)row * ldr + n);
                acc.x += __uint_as_float(rr.x << 16);
                acc.y += __uint_as_float(rr.x & 0xffff0000u);
                acc.z += __uint_as_float(rr.y << 16);
                acc.w += __uint_as_float(rr.y & 0xffff0000u);
            }
            *reinterpret_cast<uint2*>(C + (int64_t)row * ldc + n) =
                make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(G_THREADS, 1)
    gemm_bf16_splitk_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmW,
                            const __nv_bfloat16* __restrict__ bias,
                            const __nv_bfloat16* __restrict__ R, int64_t ldr,
                            __nv_bfloat16* __restrict__ C, int64_t ldc, int M, int N, int K,
                            int kb_per, int a_rows, int nst, int* status) {
    constexpr int B_BYTES = G_BK * BN * 2;  // W stage: BN / 64 chunks of 64 columns
    constexpr int GROUPS = BN / 4;          // float4 column groups of a partial row
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    // nst stages of [A: a_rows x 64 K][W: 64 K x BN].  The MMA reads 128 rows of A; those past
    // a_rows (which hold no row below M) come from the stage's own W bytes, so they are
    // complete when the stage is, and only fill accumulator rows that are never stored.
    const uint32_t a_bytes = (uint32_t)a_rows * 128u;
    const uint32_t stage_bytes = a_bytes + (uint32_t)B_BYTES;
    const uint32_t sBar = base + (uint32_t)nst * stage_bytes;
    const uint32_t sPart = base;  // the partial tile reuses the stage buffers (<= 64 KB)
    // barriers: full[nst], empty[nst], tfull, drain
    const uint32_t bar_full = sBar;
    const uint32_t bar_empty = sBar + 8u * (uint32_t)nst;
    const uint32_t bar_tfull = sBar + 16u * (uint32_t)nst;
    const uint32_t bar_drain = bar_tfull + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = (int)blockIdx.x * BN;
    const int S = (int)gridDim.y;  // the cluster spans the whole y extent
    const int rank = (int)cluster_ctarank();
    const int num_k = (K + G_BK - 1) / G_BK;
    const int kb0 = rank * kb_per;
    const int kb1 = min(num_k, kb0 + kb_per);  // the host makes every range non-empty

    if (threadIdx.x == 0) {
        for (int st = 0; st < nst; ++st) {
            mbar_init(bar_full + 8u * st, 1);
            mbar_init(bar_empty + 8u * st, 1);
        }
        mbar_init(bar_tfull, 1);
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (rows past M arrive as zeros)
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(bar_empty + 8u * stage, phase ^ 1u, abort_flag, status)) break;
                const uint32_t fb = bar_full + 8u * stage;
                const uint32_t st0 = base + (uint32_t)stage * stage_bytes;
                mbar_arrive_expect_tx(fb, stage_bytes);
                tma_load_2d(st0, &tmA, kb * G_BK, 0, fb);
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                    tma_load_2d(st0 + a_bytes + c * G_B_CHUNK, &tmW, n0 + c * 64, kb * G_BK, fb);
                ++issued;
                if (++stage == nst) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            for (int back = 0; back < nst && back < issued; ++back) {
                stage = stage == 0 ? nst - 1 : stage - 1;
                if (stage == nst - 1) phase ^= 1u;
                drain_wait(bar_full + 8u * stage, phase);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            const uint32_t idesc = idesc_bf16_f32(G_BM, BN, false, true);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(bar_full + 8u * stage, phase, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = base + (uint32_t)stage * stage_bytes;
                const uint32_t b0 = a0 + a_bytes;
#pragma unroll
                for (int k = 0; k < G_BK / 16; ++k) {
                    const uint64_t ad = sdesc_sw128(a0 + k * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(b0 + k * 2048, G_B_CHUNK, 1024);
                    mma_bf16_ss(tmem_base, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                }
                tc_commit(bar_empty + 8u * stage);
                if (++stage == nst) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) tc_commit(bar_tfull);
            tc_commit(bar_drain);
            drain_wait(bar_drain, 0);
        }
    } else {
        // ---------------- epilogue: warps 2..5, thread = row q * 32 + lane of the tile.  Once
        // the accumulator is complete every MMA has read its operands and every load has
        // landed, so the stage buffers are free for the partial.
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t t0 = tmem_base + ((uint32_t)(q * 32) << 16);
        if (__all_sync(0xffffffffu, mbar_wait(bar_tfull, 0, abort_flag, status))) {
            tc_fence_after();
            const uint32_t prow = sPart + (uint32_t)(row * BN * 4);
            const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(t0 + c * 32, v);
                tmem_wait_ld();
                if (row < M)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        st_shared_v4(prow + (((uint32_t)(c * 8) + ((uint32_t)u ^ sw)) << 4), v[4 * u],
                                     v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            }
        }
    }

    // every thread of every CTA of the cluster passes both barriers, whatever its role did
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    {
        // ---------------- reduction of this rank's column groups [g0, g0 + w) over the S partials
        const int gs = (GROUPS + S - 1) / S;
        const int g0 = rank * gs;
        const int w = min(GROUPS, g0 + gs) - g0;
        if (w > 0) {
            switch (S) {
                case 2: splitk_reduce<2, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
                case 3: splitk_reduce<3, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
                case 4: splitk_reduce<4, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
                case 5: splitk_reduce<5, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
                case 6: splitk_reduce<6, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
                case 7: splitk_reduce<7, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
                default: splitk_reduce<8, BN>(sPart, g0, w, M, N, n0, bias, R, ldr, C, ldc); break;
            }
        }
    }
    __syncwarp();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, BN);
    }
}

// ---------------------------------------------------------------------------------------
// CTA-pair version (cta_group::2): a cluster of two CTAs on two SMs computes a 256x256
// output tile with M = 256 MMAs.  Each CTA stages its own 128 rows of A and 128 of the 256
// columns of B, so per SM the operand traffic through shared memory is A 4 KB + B 4 KB per
// 128-clock MMA instead of A 4 KB + B 8 KB (plus the TMA fills, likewise halved for B): the
// one-SM kernel above is bound by shared-memory bandwidth at about two thirds of the tensor
// rate; the pair is not.
//   warp 0 (both CTAs)   TMA: own A rows and own half of B, completing on the even CTA's
//                        stage barrier (which expects both CTAs' bytes);
//   warp 1               TMEM owner (pair allocation) and, in the even CTA only, the single
//                        MMA issuer; its commits are multicast to both CTAs' barriers;
//   warps 2..5 (both)    epilogue of the CTA's own 128 rows, as above; they release the
//                        accumulator by arriving on the even CTA's barrier.
// Tiles are numbered with N fastest, so the pairs running at the same time work on the same
// 256 rows of A (read from HBM once, then from L2) while the weights, a few MB, stay in L2;
// numbered M-first, every column block re-read the whole of A (a 65536 x 768 A six times).
// A stage holds 128 K-columns as two 64-wide halves (the 128-byte swizzle atom is 64 bf16
// wide): per CTA and half, one 128-row A box and two 64x64 B boxes.  A half that lies wholly
// past K is neither loaded nor multiplied.
constexpr int P_BK = 128;
constexpr int P_STAGES = 3;
constexpr int P_HALF_A = 128 * 64 * 2;             // 16 KB: 128 rows x 64 K of A
constexpr int P_B_CHUNK = 64 * 64 * 2;             // 8 KB: 64 K-rows x 64 N-columns
constexpr int P_HALF_B = 2 * P_B_CHUNK;            // 16 KB: 64 K-rows x this CTA's 128 columns
constexpr int P_A_BYTES = 2 * P_HALF_A;            // 32 KB: this CTA's 128 rows of A
constexpr int P_B_BYTES = 2 * P_HALF_B;            // 32 KB: this CTA's half of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
// Row-block list for a projection whose later rows of each segment are never read (the key /
// value rows past a batch's key length): one flag byte and one list entry per 256-row block.
constexpr int P_MLIST_MAX = 512;
constexpr int P_LIST_BYTES = P_MLIST_MAX + 2 * P_MLIST_MAX + 16;
constexpr int P_SMEM = P_STAGES * P_STAGE_BYTES + G_EPI_BYTES + G_BAR_BYTES + P_LIST_BYTES + 1024;

static_assert(P_SMEM <= 232448, "shared memory budget (pair)");

// TWO: a second, independent projection with the same K (tmA2 / tmW2 / tmC2, bias2, M2 x N2)
// runs in the same launch, its tiles numbered after the first's: the cross-attention query
// projection next to the key / value one, whose rounds it would otherwise add to the step.
template <bool RESID, bool TWO>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G_THREADS, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmW,
                          const __grid_constant__ CUtensorMap tmC,
                          const __nv_bfloat16* __restrict__ bias, const __nv_bfloat16* R,
                          int64_t ldr, int M, int N, int K, int* status,
                          const int32_t* __restrict__ seg_len, int seg_rows,
                          const __grid_constant__ CUtensorMap tmA2,
                          const __grid_constant__ CUtensorMap tmW2,
                          const __grid_constant__ CUtensorMap tmC2,
                          const __nv_bfloat16* __restrict__ bias2, int M2, int N2) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sA = base;
    const uint32_t sB = sA + P_STAGES * P_A_BYTES;
    const uint32_t sE = sB + P_STAGES * P_B_BYTES;
    const uint32_t sBar = sE + G_EPI_BYTES;
    // barrier layout (same offsets in both CTAs): full[S], empty[S], tfull[2], tempty[2], drain
    const uint32_t bar_full = sBar;
    const uint32_t bar_empty = sBar + 8u * P_STAGES;
    const uint32_t bar_tfull = sBar + 16u * P_STAGES;
    const uint32_t bar_tempty = bar_tfull + 16u;
    const uint32_t bar_drain = bar_tempty + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint8_t* mflag = gbase + (sBar + G_BAR_BYTES - base);         // [P_MLIST_MAX]
    uint16_t* mlist = reinterpret_cast<uint16_t*>(mflag + P_MLIST_MAX);  // [P_MLIST_MAX]
    int* mcount = reinterpret_cast<int*>(mlist + P_MLIST_MAX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x >> 1);
    const int npairs = (int)(gridDim.x >> 1);
    const int num_m_all = (M + 255) / 256;
    const int num_n = (N + G_BN - 1) / G_BN;
    const int num_k = (K + P_BK - 1) / P_BK;
    const bool listed = seg_len != nullptr;  // the host guarantees num_m_all <= P_MLIST_MAX

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(bar_full + 8u * s, 1);   // used in the even CTA: its producer's arrival
            mbar_init(bar_empty + 8u * s, 1);  // one multicast commit per use of the stage
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8u * a, 1);
            mbar_init(bar_tempty + 8u * a, 8);  // 4 epilogue warps in each CTA
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmC);
        if constexpr (TWO) {
            tma_prefetch_desc(&tmA2);
            tma_prefetch_desc(&tmW2);
            tma_prefetch_desc(&tmC2);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), G_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // inputs may come from the previous kernel on the stream
    grid_dependency_wait();
    grid_launch_dependents();

    // With segment lengths, only the 256-row blocks that hold a needed row are computed: row r
    // of segment b = r / seg_rows is needed if r - b * seg_rows < seg_len[b] rounded up to a
    // multiple of 128 (the reader loads whole 128-row tiles).  Every CTA builds the same list.
    int num_m = num_m_all;
    if (listed) {
        for (int mb = (int)threadIdx.x; mb < num_m_all; mb += (int)blockDim.x) {
            const int r0 = mb * 256;
            const int r1 = min(r0 + 256, M);
            bool need = false;
            for (int b = r0 / seg_rows; b * seg_rows < r1 && !need; ++b) {
                const int len = min(max(seg_len[b], 0), seg_rows);
                const int upto = min((len + 127) / 128 * 128, seg_rows);
                need = max(r0 - b * seg_rows, 0) < upto;
            }
            mflag[mb] = need ? 1 : 0;
        }
        __syncthreads();
        if (warp == 0) {
            int cnt = 0;
            for (int c0 = 0; c0 < num_m_all; c0 += 32) {
                const int mb = c0 + lane;
                const bool f = mb < num_m_all && mflag[mb] != 0;
                const uint32_t bal = __ballot_sync(0xffffffffu, f);
                if (f) mlist[cnt + __popc(bal & ((1u << lane) - 1u))] = (uint16_t)mb;
                cnt += __popc(bal);
            }
            if (lane == 0) *mcount = cnt;
        }
        __syncthreads();
        num_m = *mcount;
    }
    const int tiles1 = num_m * num_n;
    const int num_n2 = TWO ? (N2 + G_BN - 1) / G_BN : 1;
    const int num_tiles = TWO ? tiles1 + ((M2 + 255) / 256) * num_n2 : tiles1;
    // tile -> problem, first row of its 256-row block and first column (N fastest: see above)
    auto decode = [&](int tile, int& prob, int& row0, int& n0) {
        if (!TWO || tile < tiles1) {
            prob = 0;
            row0 = (listed ? (int)mlist[tile / num_n] : tile / num_n) * 256;
            n0 = (tile % num_n) * G_BN;
        } else {
            const int t = tile - tiles1;
            prob = 1;
            row0 = (t / num_n2) * 256;
            n0 = (t % num_n2) * G_BN;
        }
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
                int prob, row0, n0;
                decode(tile, prob, row0, n0);
                const CUtensorMap* mA = TWO && prob ? &tmA2 : &tmA;
                const CUtensorMap* mW = TWO && prob ? &tmW2 : &tmW;
                const int m0 = row0 + (int)rank * 128;
                const int nb = n0 + (int)rank * 128;
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(bar_empty + 8u * stage, phase ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(bar_full + 8u * stage, 0);
                    const int halves = kb * P_BK + 64 < K ? 2 : 1;
                    if (leader)
                        mbar_arrive_expect_tx(bar_full + 8u * stage, 2 * halves * (P_HALF_A + P_HALF_B));
                    for (int hh = 0; hh < halves; ++hh) {
                        const int k0 = kb * P_BK + hh * 64;
                        tma_load_2d_pair(sA + stage * P_A_BYTES + hh * P_HALF_A, mA, k0, m0, fb);
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tma_load_2d_pair(sB + stage * P_B_BYTES + hh * P_HALF_B + c * P_B_CHUNK, mW,
                                             nb + c * 64, k0, fb);
                    }
                    ++issued;
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // the even CTA waits for every stage it expected (its own and the odd CTA's
            // copies); the odd CTA's copies land before that barrier completes
            if (leader)
                for (int back = 0; back < P_STAGES && back < issued; ++back) {
                    stage = stage == 0 ? P_STAGES - 1 : stage - 1;
                    if (stage == P_STAGES - 1) phase ^= 1u;
                    drain_wait(bar_full + 8u * stage, phase);
                }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA only)
            const uint32_t idesc = idesc_bf16_f32(256, G_BN, false, true);
            const uint64_t adesc0 = sdesc_sw128(sA, 16, 1024);
            const uint64_t bdesc0 = sdesc_sw128(sB, P_B_CHUNK, 1024);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int tile = pair; tile < num_tiles && ok; tile += npairs, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(bar_tempty + 8u * acc, acc_phase ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * G_BN);
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(bar_full + 8u * stage, phase, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = adesc0 + (uint64_t)((stage * P_A_BYTES) >> 4);
                    const uint64_t bd = bdesc0 + (uint64_t)((stage * P_B_BYTES) >> 4);
                    const int ksteps = kb * P_BK + 64 < K ? P_BK / 16 : 64 / 16;
                    for (int k = 0; k < ksteps; ++k)
                        mma_bf16_ss_pair(d_tmem, ad + (uint64_t)(((k >> 2) * P_HALF_A + (k & 3) * 32) >> 4),
                                         bd + (uint64_t)(((k >> 2) * P_HALF_B + (k & 3) * 2048) >> 4), idesc,
                                         (kb | k) != 0 ? 1u : 0u);
                    tc_commit_pair_mc(bar_empty + 8u * stage, 0x3);
                    if (++stage == P_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(bar_tfull + 8u * acc, 0x3);
            }
            // all MMAs complete before either CTA releases its TMEM or shared memory
            tc_commit_pair_mc(bar_drain, 0x1);
            drain_wait(bar_drain, 0);
        }
    } else {
        // ---------------- epilogue: this CTA's 128 rows, one TMEM lane per thread
        const int q = warp & 3;
        const int e = warp - 2;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        uint32_t bufsel = 0;
        int it = 0;
        for (int tile = pair; tile < num_tiles; tile += npairs, ++it) {
            int prob, row0, n0;
            decode(tile, prob, row0, n0);
            const int m0 = row0 + (int)rank * 128;
            const bool p2 = TWO && prob;
            const __nv_bfloat16* tb = p2 ? bias2 : bias;
            const int tM = p2 ? M2 : M, tN = p2 ? N2 : N;
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            // bias and the first 64 residual columns are fetched while the tile's MMAs run
            const uint4 bvec = load_bias_lanes(tb, n0, tN, lane);
            uint4 res[RESID ? 8 : 1];
            if constexpr (RESID) load_residual(R, ldr, m0 + q * 32 + lane, n0, M, N, res);
            // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8u * acc, acc_phase, abort_flag, status)))
                break;
            tc_fence_after();
            epilogue_rows<RESID>(tmem_base + lane_off + (uint32_t)(acc * G_BN), bvec, tb != nullptr,
                                 m0 + q * 32, n0, lane, sE + (uint32_t)(e * 2 * G_EPI_BUF), bufsel,
                                 p2 ? &tmC2 : &tmC, R, ldr, tM, tN, res, [&] {
                                     // accumulator read: release it to the MMA issuer in the even CTA
                                     tc_fence_before();
                                     __syncwarp();
                                     if (lane == 0) {
                                         if (leader)
                                             mbar_arrive(bar_tempty + 8u * acc);
                                         else
                                             mbar_arrive_cluster(mapa_shared(bar_tempty + 8u * acc, 0));
                                     }
                                 });
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // lanes that skipped a one-thread role wait here for it: the CTA barrier below must
    // see whole warps, or it can complete while a role is still running
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the pair's MMAs may touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, G_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------
// CTA-pair version with the accumulator transposed: tiles of 192 rows of A (the MMA's N
// dimension) x 256 columns of W (the MMA's M dimension, 128 per CTA), for shapes where
// 192-row tiles fill the pairs in less time than 256 x 256 ones (M = 8192, N = K = 768: 129
// tiles in two rounds of smaller tiles against 96 in two full rounds).  The 192-row side comes
// from A, whose K-major layout allows 96 rows per CTA; W, MN-major, could not be split into
// 96-column halves in its 128-byte swizzled 64-column chunks.
//   MMA A operand  W^T: each CTA's 128 columns of W, MN-major (W's rows are K), 128-byte
//                  swizzled 64-column chunks, exactly as the other kernel stages its half of B;
//   MMA B operand  A^T: 96 rows of A per CTA, K-major, 128-byte swizzle (a 96-row half of a
//                  192-row tile is twelve 8-row groups, which a K-major operand allows);
//   accumulator    TMEM lane = output column n (the CTA's 128), TMEM column = output row m
//                  (all 192 of the tile, from both CTAs' halves of A).
// Epilogue: each thread holds one output column across the tile's rows; it adds that column's
// bias, rounds, and writes 64-row x 32-column boxes (row-major, no swizzle: the 32 lanes of a
// warp write one 64-byte row segment per store) that a TMA store sends to C.
constexpr int T_BM = 192;                          // rows of A per tile (96 per CTA)
constexpr int T_HALF_X = 96 * 64 * 2;              // 12 KB: 96 rows x 64 K of A
constexpr int T_X_BYTES = 2 * T_HALF_X;            // 24 KB per stage
constexpr int T_W_CHUNK = 64 * 64 * 2;             // 8 KB: 64 K-rows x 64 columns of W
constexpr int T_HALF_W = 2 * T_W_CHUNK;            // 16 KB: 64 K-rows x this CTA's 128 columns
constexpr int T_W_BYTES = 2 * T_HALF_W;            // 32 KB per stage
constexpr int T_STAGES = 3;
constexpr int T_EPI_BUF = 64 * 32 * 2;             // 4 KB: 64 rows x 32 columns
constexpr int T_EPI_BYTES = 4 * 2 * T_EPI_BUF;
constexpr int T_SMEM = T_STAGES * (T_X_BYTES + T_W_BYTES) + T_EPI_BYTES + G_BAR_BYTES + 1024;
static_assert(T_SMEM <= 232448, "shared memory budget (transposed pair)");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(G_THREADS, 1)
    gemm_bf16_pairT_kernel(const __grid_constant__ CUtensorMap tmX,
                           const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmC,
                           const __nv_bfloat16* __restrict__ bias, int M, int N, int K, int* status) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);

    const uint32_t sX = base;
    const uint32_t sW = sX + T_STAGES * T_X_BYTES;
    const uint32_t sE = sW + T_STAGES * T_W_BYTES;
    const uint32_t sBar = sE + T_EPI_BYTES;
    // barrier layout (same offsets in both CTAs): full[S], empty[S], tfull[2], tempty[2], drain
    const uint32_t bar_full = sBar;
    const uint32_t bar_empty = sBar + 8u * T_STAGES;
    const uint32_t bar_tfull = sBar + 16u * T_STAGES;
    const uint32_t bar_tempty = bar_tfull + 16u;
    const uint32_t bar_drain = bar_tempty + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar_drain + 8u - base));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x >> 1);
    const int npairs = (int)(gridDim.x >> 1);
    const int num_m = (M + T_BM - 1) / T_BM;
    const int num_n = (N + G_BN - 1) / G_BN;
    const int num_tiles = num_m * num_n;
    const int num_k = (K + P_BK - 1) / P_BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < T_STAGES; ++s) {
            mbar_init(bar_full + 8u * s, 1);
            mbar_init(bar_empty + 8u * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + 8u * a, 1);
            mbar_init(bar_tempty + 8u * a, 8);  // 4 epilogue warps in each CTA
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), G_TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // inputs may come from the previous kernel on the stream
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs): own 96 rows of A, own 128 columns of W
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int tile = pair; tile < num_tiles && ok; tile += npairs) {
                const int m0 = (tile / num_n) * T_BM + (int)rank * 96;
                const int nb = (tile % num_n) * G_BN + (int)rank * 128;
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(bar_empty + 8u * stage, phase ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(bar_full + 8u * stage, 0);
                    const int halves = kb * P_BK + 64 < K ? 2 : 1;
                    if (leader)
                        mbar_arrive_expect_tx(bar_full + 8u * stage, 2 * halves * (T_HALF_X + T_HALF_W));
                    for (int hh = 0; hh < halves; ++hh) {
                        const int k0 = kb * P_BK + hh * 64;
                        tma_load_2d_pair(sX + stage * T_X_BYTES + hh * T_HALF_X, &tmX, k0, m0, fb);
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tma_load_2d_pair(sW + stage * T_W_BYTES + hh * T_HALF_W + c * T_W_CHUNK, &tmW,
                                             nb + c * 64, k0, fb);
                    }
                    ++issued;
                    if (++stage == T_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader)
                for (int back = 0; back < T_STAGES && back < issued; ++back) {
                    stage = stage == 0 ? T_STAGES - 1 : stage - 1;
                    if (stage == T_STAGES - 1) phase ^= 1u;
                    drain_wait(bar_full + 8u * stage, phase);
                }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (even CTA only): D (256 columns of W x 192 rows of A)
            const uint32_t idesc = idesc_bf16_f32(256, T_BM, true, false);
            const uint64_t wdesc0 = sdesc_sw128(sW, T_W_CHUNK, 1024);
            const uint64_t xdesc0 = sdesc_sw128(sX, 16, 1024);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int it = 0;
            for (int tile = pair; tile < num_tiles && ok; tile += npairs, ++it) {
                const int acc = it & 1;
                const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(bar_tempty + 8u * acc, acc_phase ^ 1u, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * T_BM);
                for (int kb = 0; kb < num_k; ++kb) {
                    if (!mbar_wait(bar_full + 8u * stage, phase, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t wd = wdesc0 + (uint64_t)((stage * T_W_BYTES) >> 4);
                    const uint64_t xd = xdesc0 + (uint64_t)((stage * T_X_BYTES) >> 4);
                    const int ksteps = kb * P_BK + 64 < K ? P_BK / 16 : 64 / 16;
                    for (int k = 0; k < ksteps; ++k)
                        mma_bf16_ss_pair(d_tmem, wd + (uint64_t)(((k >> 2) * T_HALF_W + (k & 3) * 2048) >> 4),
                                         xd + (uint64_t)(((k >> 2) * T_HALF_X + (k & 3) * 32) >> 4), idesc,
                                         (kb | k) != 0 ? 1u : 0u);
                    tc_commit_pair_mc(bar_empty + 8u * stage, 0x3);
                    if (++stage == T_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc(bar_tfull + 8u * acc, 0x3);
            }
            tc_commit_pair_mc(bar_drain, 0x1);
            drain_wait(bar_drain, 0);
        }
    } else {
        // ---------------- epilogue: this CTA's 128 output columns, one per thread
        const int q = warp & 3;
        const int e = warp - 2;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const uint32_t buf0 = sE + (uint32_t)(e * 2 * T_EPI_BUF);
        uint32_t bufsel = 0;
        int it = 0;
        for (int tile = pair; tile < num_tiles; tile += npairs, ++it) {
            const int m0 = (tile / num_n) * T_BM;
            const int nw = (tile % num_n) * G_BN + (int)rank * 128 + q * 32;  // this warp's columns
            const int n = nw + lane;
            const int acc = it & 1;
            const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
            const float bv = bias != nullptr && n < N ? __bfloat162float(bias[n]) : 0.f;
            // warp-uniform outcome: the tcgen05.ld below is .sync.aligned
            if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8u * acc, acc_phase, abort_flag, status)))
                break;
            tc_fence_after();
            const uint32_t t0 = tmem_base + lane_off + (uint32_t)(acc * T_BM);
#pragma unroll 1
            for (int ch = 0; ch < T_BM / 64; ++ch) {
                uint32_t va[32], vb[32];
                tmem_ld32(t0 + ch * 64, va);
                tmem_ld32(t0 + ch * 64 + 32, vb);
                tmem_wait_ld();
                reg_fence(va);
                reg_fence(vb);
                if (ch == T_BM / 64 - 1) {
                    // accumulator read: release it to the MMA issuer in the even CTA
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            mbar_arrive(bar_tempty + 8u * acc);
                        else
                            mbar_arrive_cluster(mapa_shared(bar_tempty + 8u * acc, 0));
                    }
                }
                const int mr = m0 + ch * 64;
                if (mr < M && nw < N) {  // else the box lies wholly outside C
                    const uint32_t buf = buf0 + bufsel * (uint32_t)T_EPI_BUF;
                    if (lane == 0) bulk_wait_group_read<1>();  // the store that last used buf has read it
                    __syncwarp();
                    // row i of the box: this lane's column at byte 2 * lane of a 64-byte row
                    const uint32_t col = buf + 2u * (uint32_t)lane;
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        st_shared_b16(col + (uint32_t)i * 64u, __uint_as_float(va[i]) + bv);
                        st_shared_b16(col + (uint32_t)(i + 32) * 64u, __uint_as_float(vb[i]) + bv);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmC, buf, nw, mr);
                        bulk_commit_group();
                    }
                    bufsel ^= 1u;
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    // lanes that skipped a one-thread role wait here for it: the CTA barrier below must
    // see whole warps, or it can complete while a role is still running
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the pair's MMAs may touch its memory
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, G_TMEM_COLS);
    }
}

// Co-resident clusters of a pair kernel (cached per kernel variant and device): the persistent
// grid's size.
template <typename Kernel>
int pair_occupancy(Kernel kernel, int variant, int num_sms) {
    static std::atomic<int> cache[3][64];  // 0 until asked
    int dev = 0;
    cudaGetDevice(&dev);
    int n = dev >= 0 && dev < 64 ? cache[variant][dev].load(std::memory_order_relaxed) : 0;
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2));
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = P_SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) n = num_sms / 2;
    if (dev >= 0 && dev < 64) cache[variant][dev].store(n, std::memory_order_relaxed);
    return n;
}

// The three tensor maps of one pair-kernel projection: A (K-major, 64 x 128 boxes), W (64 x 64
// boxes of its (in, out) rows) and C (64 x 32 store boxes).
bool encode_pair_maps(const void* A, int64_t lda, const void* W, int64_t ldw, void* C, int64_t ldc,
                      int M, int N, int K, CUtensorMap* tA, CUtensorMap* tW, CUtensorMap* tC) {
    const uint64_t da[2] = {(uint64_t)K, (uint64_t)M}, sa[1] = {(uint64_t)lda * 2};
    const uint32_t ba[2] = {64, G_BM};
    const uint64_t dw[2] = {(uint64_t)N, (uint64_t)K}, sw[1] = {(uint64_t)ldw * 2};
    const uint32_t bw[2] = {64, G_BK};
    const uint64_t dc[2] = {(uint64_t)N, (uint64_t)M}, sc[1] = {(uint64_t)ldc * 2};
    const uint32_t bc[2] = {64, 32};
    return encode_tmap_bf16(tA, A, 2, da, sa, ba) && encode_tmap_bf16(tW, W, 2, dw, sw, bw) &&
           encode_tmap_bf16(tC, C, 2, dc, sc, bc);
}

// Shared memory of the split kernel: up to 8 stages of (A rows rounded up to 8) x 64 K plus
// 64 K x BN of W, within the per-CTA limit.  Every launch takes more than half an SM's shared
// memory (at least 8 x 17 KB), so one CTA runs per SM whatever the row count.
constexpr int SK_SMEM_MAX = 232448;
constexpr int SK_SMEM_EXTRA = G_BAR_BYTES + 1024;
template <int BN>
int splitk_stages(int a_rows) {
    const int stage = a_rows * 128 + G_BK * BN * 2;
    const int n = (SK_SMEM_MAX - SK_SMEM_EXTRA) / stage;
    return n < 8 ? n : 8;
}

// Clusters of S CTAs of the split kernel that the device runs at once (0: none), per device,
// tile width and S.
template <int BN>
int splitk_max_clusters(int S) {
    static std::atomic<int> cache[64][9];  // count + 1; 0 = not asked yet
    int dev = -1;
    if (S < 1 || S > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int c = cache[dev][S].load(std::memory_order_relaxed);
    if (c == 0) {
        int n = 0;
        if (cudaFuncSetAttribute(gemm_bf16_splitk_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SK_SMEM_MAX) == cudaSuccess) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, S);
            cfg.blockDim = dim3(G_THREADS);
            cfg.dynamicSmemBytes = SK_SMEM_MAX;  // one CTA per SM, as every launch
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = (unsigned)S;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_splitk_kernel<BN>, &cfg) != cudaSuccess) n = 0;
        }
        cudaGetLastError();
        c = n + 1;
        cache[dev][S].store(c, std::memory_order_relaxed);
    }
    return c - 1;
}

// Clusters of S CTAs share each 128 x BN tile of a projection of at most 128 rows: returns S
// (0: one CTA per 256-column tile of the kernel above instead) and the K blocks of each rank.
// About one CTA per SM in all, at most 8 to a cluster (the portable limit), no more clusters
// than the device runs at once (a second wave of clusters would double the time), every rank
// at least one K block.
template <int BN>
int splitk_plan(int M, int N, int K, int num_sms, int* kb_per) {
    if (M <= 0 || M > G_BM || N <= 0 || K <= 0) return 0;
    const int tiles = (N + BN - 1) / BN, num_k = (K + G_BK - 1) / G_BK;
    int S = num_sms / tiles;
    if (S > 8) S = 8;
    if (S > num_k) S = num_k;
    while (S >= 2 && tiles > splitk_max_clusters<BN>(S)) --S;
    if (S < 2) return 0;
    const int per = (num_k + S - 1) / S;
    S = (num_k + per - 1) / per;
    if (S < 2) return 0;
    *kb_per = per;
    return S;
}

template <int BN>
cudaError_t launch_splitk(const void* A, int64_t lda, const CUtensorMap& tW, const void* bias,
                          const void* R, int64_t ldr, void* C, int64_t ldc, int M, int N, int K,
                          int S, int kb_per, int* status, cudaStream_t stream) {
    // A in boxes of only the rows that exist (rounded up to 8: whole 128-byte swizzle atoms)
    const int a_rows = (M + 7) & ~7;
    CUtensorMap tA;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)lda * 2};
        const uint32_t box[2] = {G_BK, (uint32_t)a_rows};
        if (!encode_tmap_bf16(&tA, A, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const int nst = splitk_stages<BN>(a_rows);
    const int smem = nst * (a_rows * 128 + G_BK * BN * 2) + SK_SMEM_EXTRA;
    cudaError_t err = cudaFuncSetAttribute(gemm_bf16_splitk_kernel<BN>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM_MAX);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + BN - 1) / BN, S);
    cfg.blockDim = dim3(G_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gemm_bf16_splitk_kernel<BN>, tA, tW,
                              reinterpret_cast<const __nv_bfloat16*>(bias),
                              reinterpret_cast<const __nv_bfloat16*>(R), ldr,
                              static_cast<__nv_bfloat16*>(C), ldc, M, N, K, kb_per, a_rows, nst, status);
}

}  // namespace

cudaError_t launch_gemm_bf16_two(const void* A, int64_t lda, const void* W, int64_t ldw,
                                 const void* bias, void* C, int64_t ldc, int M, int N,
                                 const int32_t* seg_len, int seg_rows, const void* A2, int64_t lda2,
                                 const void* W2, int64_t ldw2, const void* bias2, void* C2,
                                 int64_t ldc2, int M2, int N2, int K, int num_sms, int* status,
                                 cudaStream_t stream) {
    if (M <= 128 || M2 <= 128) return cudaErrorInvalidValue;
    CUtensorMap tA, tW, tC, tA2, tW2, tC2;
    if (!encode_pair_maps(A, lda, W, ldw, C, ldc, M, N, K, &tA, &tW, &tC) ||
        !encode_pair_maps(A2, lda2, W2, ldw2, C2, ldc2, M2, N2, K, &tA2, &tW2, &tC2))
        return cudaErrorInvalidValue;
    auto kernel = gemm_bf16_pair_kernel<false, true>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
    if (err != cudaSuccess) return err;
    const int max_pairs = pair_occupancy(kernel, 2, num_sms);
    const int64_t tiles = (int64_t)((M + 255) / 256) * ((N + G_BN - 1) / G_BN) +
                          (int64_t)((M2 + 255) / 256) * ((N2 + G_BN - 1) / G_BN);
    const int pairs = tiles < max_pairs ? (int)tiles : max_pairs;
    const bool listed = seg_len != nullptr && seg_rows >= 128 && (M + 255) / 256 <= P_MLIST_MAX;
    return launch_pdl(kernel, dim3(2 * pairs), dim3(G_THREADS), P_SMEM, stream, tA, tW, tC,
                      reinterpret_cast<const __nv_bfloat16*>(bias),
                      static_cast<const __nv_bfloat16*>(nullptr), (int64_t)0, M, N, K, status,
                      listed ? seg_len : nullptr, listed ? seg_rows : 0, tA2, tW2, tC2,
                      reinterpret_cast<const __nv_bfloat16*>(bias2), M2, N2);
}

cudaError_t launch_gemm_bf16(const void* A, int64_t lda, const void* W, int64_t ldw,
                             const void* bias, const void* R, int64_t ldr, void* C, int64_t ldc,
                             int M, int N, int K, int num_sms, int* status, cudaStream_t stream,
                             const int32_t* seg_len, int seg_rows) {
    CUtensorMap tA, tW, tC;
    if (!encode_pair_maps(A, lda, W, ldw, C, ldc, M, N, K, &tA, &tW, &tC)) return cudaErrorInvalidValue;
    const int num_tiles = ((M + G_BM - 1) / G_BM) * ((N + G_BN - 1) / G_BN);
    auto pair_kernel = R != nullptr ? gemm_bf16_pair_kernel<true, false> : gemm_bf16_pair_kernel<false, false>;
    auto tc_kernel = R != nullptr ? gemm_bf16_tc_kernel<true> : gemm_bf16_tc_kernel<false>;
    if (M > 128 && R == nullptr && seg_len == nullptr) {
        // 192-row tiles with the accumulator transposed, where they fill the pairs in less time
        // than 256 x 256 ones: rounds of tiles over the resident pairs, a 192-row tile taking
        // 0.91 of a 256-row one (measured: c3's QKV projection, 7 rounds of 192-row tiles
        // against 6 of 256-row ones, 41.1 against 38.8 us; M = 8192, N = K = 768, 2 rounds
        // each, 15.1 against 16.9 us)
        static std::atomic<int> t_pairs_cache[64];  // 0 until asked
        int dev = 0;
        cudaGetDevice(&dev);
        int t_pairs = dev >= 0 && dev < 64 ? t_pairs_cache[dev].load(std::memory_order_relaxed) : 0;
        if (t_pairs == 0) {
            if (cudaFuncSetAttribute(gemm_bf16_pairT_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     T_SMEM) != cudaSuccess)
                return cudaErrorInvalidValue;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2 * (unsigned)(num_sms / 2));
            cfg.blockDim = dim3(G_THREADS);
            cfg.dynamicSmemBytes = T_SMEM;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 2;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, gemm_bf16_pairT_kernel, &cfg) != cudaSuccess || n <= 0)
                n = num_sms / 2;
            t_pairs = n;
            if (dev >= 0 && dev < 64) t_pairs_cache[dev].store(n, std::memory_order_relaxed);
        }
        const int64_t nb = (N + G_BN - 1) / G_BN;
        const int64_t tiles_t = ((M + T_BM - 1) / T_BM) * nb, tiles_s = ((M + 255) / 256) * nb;
        const int64_t cost_t = 91 * ((tiles_t + t_pairs - 1) / t_pairs);
        const int64_t cost_s = 100 * ((tiles_s + t_pairs - 1) / t_pairs);
        if (cost_t < cost_s) {
            CUtensorMap tX, tCT;
            {
                const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
                const uint64_t strides[1] = {(uint64_t)lda * 2};
                const uint32_t box[2] = {64, 96};
                if (!encode_tmap_bf16(&tX, A, 2, dims, strides, box)) return cudaErrorInvalidValue;
            }
            {
                const uint64_t dims[2] = {(uint64_t)N, (uint64_t)M};
                const uint64_t strides[1] = {(uint64_t)ldc * 2};
                const uint32_t box[2] = {32, 64};
                if (!encode_tmap_bf16(&tCT, C, 2, dims, strides, box, 0)) return cudaErrorInvalidValue;
            }
            cudaError_t err = cudaFuncSetAttribute(gemm_bf16_pairT_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, T_SMEM);
            if (err != cudaSuccess) return err;
            const int pairs = tiles_t < t_pairs ? (int)tiles_t : t_pairs;
            return launch_pdl(gemm_bf16_pairT_kernel, dim3(2 * pairs), dim3(G_THREADS), T_SMEM, stream, tX, tW,
                              tCT, reinterpret_cast<const __nv_bfloat16*>(bias), M, N, K, status);
        }
    }
    if (M > 128) {
        // CTA pairs: the W box is 64 columns x 64 K-rows, the A box 64 K x 128 rows (as
        // above); each CTA of a pair loads its own A rows and its half of the W tile.
        cudaError_t err = cudaFuncSetAttribute(pair_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, P_SMEM);
        if (err != cudaSuccess) return err;
        const int max_pairs = pair_occupancy(pair_kernel, R != nullptr ? 1 : 0, num_sms);
        const int pair_tiles = ((M + 255) / 256) * ((N + G_BN - 1) / G_BN);
        const int pairs = pair_tiles < max_pairs ? pair_tiles : max_pairs;
        // the row-block list fits up to P_MLIST_MAX blocks; beyond that every row is computed
        const bool listed = seg_len != nullptr && seg_rows >= 128 && (M + 255) / 256 <= P_MLIST_MAX;
        return launch_pdl(pair_kernel, dim3(2 * pairs), dim3(G_THREADS), P_SMEM, stream,
                          tA, tW, tC, reinterpret_cast<const __nv_bfloat16*>(bias),
                          reinterpret_cast<const __nv_bfloat16*>(R), ldr, M, N, K, status,
                          listed ? seg_len : nullptr, listed ? seg_rows : 0, tA, tW, tC,
                          static_cast<const __nv_bfloat16*>(nullptr), 0, 0);
    }
    // few rows: clusters of S CTAs split K over 128-column tiles (every row is written, seg_len
    // or not).  128 columns rather than 256: each rank exchanges half the partial bytes, and
    // measured 1-20% faster from 32 rows up, the same at one row, and still faster where
    // 256-column tiles would allow more CTAs (32 x 2048 x 6144: 11.6 against 12.1 us).  Where
    // clusters of two over 128-column tiles would not all fit at once (N > 9728 on 152 SMs),
    // 256-column tiles still leave room for them.
    int kb_per = 0;
    int S = splitk_plan<128>(M, N, K, num_sms, &kb_per);
    if (S > 0) return launch_splitk<128>(A, lda, tW, bias, R, ldr, C, ldc, M, N, K, S, kb_per, status, stream);
    S = splitk_plan<256>(M, N, K, num_sms, &kb_per);
    if (S > 0) return launch_splitk<256>(A, lda, tW, bias, R, ldr, C, ldc, M, N, K, S, kb_per, status, stream);
    cudaError_t err = cudaFuncSetAttribute(tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, G_SMEM);
    if (err != cudaSuccess) return err;
    const int grid = num_tiles < num_sms ? num_tiles : num_sms;
    return launch_pdl(tc_kernel, dim3(grid), dim3(G_THREADS), G_SMEM, stream, tA, tW, tC,
                      reinterpret_cast<const __nv_bfloat16*>(bias),
                      reinterpret_cast<const __nv_bfloat16*>(R), ldr, M, N, K, status);
}

}  // namespace mha
