/*
 * mha.h -- C ABI of the GB300 (sm_103a) multi-head attention forward.
 *
 * The operation (itwiki.kr "멀티 헤드 어텐션", section 수식, and the tensor-shape
 * table of section 텐서 모양으로 본 계산):
 *
 *   [Q | K | V] = X W_qkv + b_qkv                    one fused projection
 *   head_i      = softmax(Q_i K_i^T / sqrt(d_k) [+ M]) V_i
 *   Ocat        = Concat(head_1, ..., head_h)        head i at columns i*d_v
 *   Y           = Ocat W_o + b_o
 *
 * Q_i, K_i, V_i are column slices of the projection output ("a head is not a
 * separate matrix, only a slice of one matrix's output dimension", same
 * table).  M is the causal mask (-inf for key j > query i; iamjaehka13.blog
 * "[Deep Learning 5] Attention의 내부 계산", section 9) and/or key padding
 * (keys j >= L_b excluded; molayo1419.me "MHA란 무엇인가?", pitfall 2).
 * Cross-attention takes Q from X_q and K, V from X_kv (iamjaehka13.blog,
 * section 19).
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers, row-major, in the handle's
 *    dtype (fp32 or bf16) unless stated; kv_lengths is device int32.
 *  - Strides ("ld*") are in elements.
 *  - Nothing is allocated, freed or synchronised inside the compute calls;
 *    every kernel is launched asynchronously on `stream` (a cudaStream_t; NULL
 *    is the legacy default stream).  All memory is owned by the caller.
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing.  Errors found on the device (an out-of-range L_b, a
 *    pipeline wait that ran out of time) are recorded in a status word kept in
 *    the workspace; read it with mha_get_status.
 *  - Outputs must not alias inputs.
 *  - Every function is thread-compatible: one handle must not be used from
 *    two host threads at once.
 *  - The work a handle launches must not overlap on the GPU: its workspace
 *    (the status word and the scratch tensors) is shared by all its calls, so
 *    issue them on one stream or order the streams with events.
 */
#ifndef MHA_H_
#define MHA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mha_s* mha_t; /* opaque; holds the layer configuration only */

typedef enum {
    MHA_F32 = 0,  /* fp32 storage, fp32 arithmetic (CUDA-core FFMA) */
    MHA_BF16 = 1  /* bf16 storage, fp32 accumulation (tcgen05 tensor cores) */
} mha_dtype;

typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = 1, /* a size, pointer, stride or flag is invalid */
    MHA_ERR_UNSUPPORTED = 2, /* valid, but this build has no kernel for it */
    MHA_ERR_WORKSPACE = 3,   /* no workspace set, or it is too small */
    MHA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
    MHA_ERR_TIMEOUT = 5,     /* device status: a pipeline wait gave up */
    MHA_ERR_BAD_LENGTH = 6   /* device status: some L_b outside [1, T_kv]; its rows are NaN */
} mha_status;

/*
 * mha_create -- make a handle for one layer shape.
 *   D    model width (d_model);  h  number of heads;
 *   d_k  query/key width per head;  d_v  value width per head
 *   (itwiki.kr "멀티 헤드 어텐션", 수식: W_i^Q, W_i^K in R^{d_model x d_k},
 *   W_i^V in R^{d_model x d_v}, W^O in R^{h d_v x d_model}).
 * Any positive D, h, d_k, d_v is accepted here; a dtype/shape pair without a
 * kernel is reported by the compute calls as MHA_ERR_UNSUPPORTED.
 * Returns MHA_ERR_INVALID_ARG for out == NULL, a non-positive size or an
 * unknown dtype.  Host memory only; makes no CUDA call, so it also works on a
 * machine without a GPU.
 */
mha_status mha_create(mha_t* out, int D, int h, int d_k, int d_v, mha_dtype dtype);

/*
 * mha_create_ex -- mha_create with the variants of itwiki.kr "멀티 헤드 어텐션", section
 * 추론 비용과 변형:
 *   h_kv   number of K/V heads, a divisor of h: h_kv == h is plain multi-head attention,
 *          h_kv == 1 multi-query attention (MQA), anything between grouped-query attention
 *          (GQA).  Query head i uses K/V head i / (h / h_kv) (consecutive query heads form
 *          a group).
 *   gated  0 or 1: gated attention -- the output of every head is multiplied element by
 *          element by sigmoid(X_q W_G + b_G) (a head-specific sigmoid gate on the scaled
 *          dot-product attention output) before the output projection.
 * The fused projection W_qkv then has the column blocks [W^Q | W^K | W^V (| W^G)] of widths
 * h*d_k, h_kv*d_k, h_kv*d_v (and h*d_v).  MHA_ERR_INVALID_ARG as for mha_create, and for
 * h_kv not dividing h or gated not 0/1.  mha_create(D, h, d_k, d_v) is
 * mha_create_ex(D, h, h, d_k, d_v, 0).
 */
mha_status mha_create_ex(mha_t* out, int D, int h, int h_kv, int d_k, int d_v, int gated,
                         mha_dtype dtype);

/* mha_destroy -- free the handle and the copy streams and events mha_set_workspace
 * created for it (NULL is ignored).  Does not touch the caller's workspace; no work
 * of the handle may still be in flight. */
void mha_destroy(mha_t handle);

/*
 * mha_workspace_size -- bytes of device workspace mha_forward needs for
 * batch B, T_q query rows and T_kv key rows (self-attention: T_kv = T_q).
 * Layout: a 256-byte status block, the projected query side Q (and the gate
 * pre-activations) (B,T_q,h*d_k [+h*d_v]) and K,V (B,T_kv,h_kv*(d_k+d_v)) -- for
 * self-attention one fused buffer of the projection's width -- and Ocat
 * (B,T_q,h*d_v), each 256-byte aligned.  Returns 0 for an invalid handle or size.
 */
size_t mha_workspace_size(mha_t handle, int B, int T_q, int T_kv);

/*
 * mha_set_workspace -- attach caller-owned device memory (256-byte aligned,
 * `bytes` long) to the handle, and zero its status block (a synchronous
 * cudaMemset of 256 bytes).  The memory must stay valid while calls using
 * the handle are in flight.  NULL detaches.  The first attach also creates the
 * two copy streams and the events mha_forward_host uses, on the current device
 * (MHA_ERR_CUDA if that fails); they live until mha_destroy.
 */
mha_status mha_set_workspace(mha_t handle, void* dev_ptr, size_t bytes);

/*
 * mha_forward -- Y = MultiHead(X_q, X_kv) for the whole batch.
 *   X_q    (B, T_q, D)
 *   X_kv   (B, T_kv, D); NULL or == X_q means self-attention (T_kv must equal
 *          T_q), done with ONE fused GEMM against all of W_qkv
 *   W_qkv  (D, 2*h*d_k + h*d_v), column blocks [W^Q | W^K | W^V]; head i of
 *          each block is its columns [i*d, (i+1)*d)
 *   b_qkv  (2*h*d_k + h*d_v) or NULL
 *   W_o    (h*d_v, D);  b_o  (D) or NULL
 *   causal nonzero applies the causal mask (key j > query i excluded);
 *          requires T_q == T_kv
 *   kv_lengths  device int32[B] or NULL; keys j >= kv_lengths[b] excluded.
 *          Values outside [1, T_kv] make that batch's output NaN and record
 *          MHA_ERR_BAD_LENGTH in the status word (an all-masked softmax row is
 *          undefined, molayo1419.me pitfall 3)
 *   out    (B, T_q, D)
 * Needs a workspace of mha_workspace_size(B, T_q, T_kv) bytes.  Launches
 * three kernels on `stream` (projection, attention, output projection; bf16 cross-
 * attention with more than 128 query and 128 key rows projects both sides in one launch,
 * see mha_linear_pair), four for other cross-attention, one more for the gate block of a
 * gated cross-attention.
 * bf16 requires d_k == d_v in {64, 128} and D a multiple of 8 (else
 * MHA_ERR_UNSUPPORTED) and 16-byte aligned pointers (else MHA_ERR_INVALID_ARG);
 * fp32 accepts any shape with d_k, d_v <= 256.  B == 0 or T_q == 0 is a no-op;
 * T_kv == 0 with T_q > 0 is MHA_ERR_INVALID_ARG.
 */
mha_status mha_forward(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q, int T_kv,
                       const void* W_qkv, const void* b_qkv, const void* W_o, const void* b_o,
                       int causal, const int32_t* kv_lengths, void* out, void* stream);

/*
 * mha_forward_checked -- mha_forward that first validates the key lengths on the host, for
 * debugging and for callers that want an invalid length reported before any work instead of
 * NaN rows plus a device status.
 *   kv_lengths_host  host int32[B], a copy of the device array kv_lengths (the caller keeps
 *                    the two equal; both NULL, or both non-NULL, else MHA_ERR_INVALID_ARG).
 * Every L_b must lie in [1, T_kv] (molayo1419.me "MHA란 무엇인가?", pitfall 3: a row with no
 * visible key has no softmax); otherwise MHA_ERR_BAD_LENGTH is returned and nothing is launched.
 * All other arguments, checks and behaviour are those of mha_forward.  Reads only host memory
 * before launching; asynchronous like mha_forward.
 */
mha_status mha_forward_checked(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q,
                               int T_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                               const void* b_o, int causal, const int32_t* kv_lengths,
                               const int32_t* kv_lengths_host, void* out, void* stream);

/*
 * mha_forward_ex -- mha_forward for a handle of any mha_create_ex shape (W_qkv with the
 * column blocks described there), plus an optional residual:
 *   residual  (B, T_q, D) or NULL; added to the output in the output projection's epilogue,
 *             Y = residual + Concat(heads) W_o + b_o (iamjaehka13.blog "[Deep Learning 5]
 *             Attention의 내부 계산", sections 14 and 16: X' = X + O W_O, so normally
 *             residual == X_q).  It may be `out` itself (in place) but must not otherwise
 *             overlap it (MHA_ERR_INVALID_ARG); bf16 needs it 16-byte aligned.
 * With a gate and X_kv != X_q the gate pre-activations come from X_q (one more GEMM).
 * mha_forward(...) is mha_forward_ex(..., residual = NULL, out, stream).
 */
mha_status mha_forward_ex(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q,
                          int T_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                          const void* b_o, int causal, const int32_t* kv_lengths,
                          const void* residual, void* out, void* stream);

/*
 * mha_forward_host_workspace_size -- workspace bytes mha_forward_host needs: the forward's
 * scratch (mha_workspace_size) for its largest chunk of batch elements (see mha_forward_host),
 * then device copies of X_q (B,T_q,D), X_kv (B,T_kv,D), the residual (B,T_q,D) and Y
 * (B,T_q,D), each 256-byte aligned.  0 for an invalid handle, a size <= 0 or chunks outside
 * [1, 16].
 */
size_t mha_forward_host_workspace_size(mha_t handle, int B, int T_q, int T_kv, int chunks);

/*
 * mha_forward_host -- mha_forward_ex with the activations in HOST memory: X_q, X_kv (NULL
 * or == X_q for self-attention), residual (NULL, == X_q, or another (B,T_q,D) buffer) and
 * out are host pointers; W_qkv, b_qkv, W_o, b_o and kv_lengths stay device pointers
 * (resident weights).  Host buffers should be pinned (cudaHostAlloc/cudaHostRegister) for
 * the copies to run asynchronously.
 * The batch is cut into at most min(chunks, B) chunks of whole batch elements (every batch
 * element is an independent problem, so the result is the same as one mha_forward_ex over
 * the whole batch, bit for bit): one or two chunks of ceil(B / n) elements; from three on,
 * the first and last chunks half the size of the others (B = 4, chunks = 3: 1, 2, 1), so
 * that the first copy-in and the last copy-out, which no kernel overlaps, are short.  Chunk c's inputs go to the device on the handle's
 * host-to-device stream, its forward runs on `stream` once they are in, and its output
 * goes back on the handle's device-to-host stream while chunk c+1 computes, so copies in
 * both directions overlap the kernels.  The copies start after the work already queued on
 * `stream`, and `stream` completes only once all of `out` has landed: synchronise on
 * `stream` before reading `out` or reusing the host inputs.  Asynchronous; allocates
 * nothing.
 * Needs a workspace of mha_forward_host_workspace_size(B, T_q, T_kv, chunks) bytes attached
 * on the current device (else MHA_ERR_WORKSPACE; another current device:
 * MHA_ERR_INVALID_ARG).  chunks outside [1, 16] is MHA_ERR_INVALID_ARG; other arguments as
 * for mha_forward_ex.  Launches the kernels of mha_forward_ex once per chunk.
 */
mha_status mha_forward_host(mha_t handle, const void* X_q, const void* X_kv, int B, int T_q,
                            int T_kv, const void* W_qkv, const void* b_qkv, const void* W_o,
                            const void* b_o, int causal, const int32_t* kv_lengths,
                            const void* residual, void* out, int chunks, void* stream);

/*
 * mha_linear -- one projection step, C = A W + bias
 * (itwiki.kr "멀티 헤드 어텐션", tensor-shape table rows 투영 and 출력 투영).
 *   A (M, K) row stride lda;  W (K, N) row stride ldw;  bias (N) or NULL;
 *   C (M, N) row stride ldc.   fp32 accumulate in both dtypes.
 * bf16 requires K, N, lda, ldw, ldc multiples of 8 and 16-byte aligned
 * pointers.  M, N, K >= 1.  bf16 with M <= 128 (a decode step's new tokens) splits K over a
 * cluster of CTAs per output tile and adds their fp32 partials in a fixed order: the result is
 * the same on every call, and differs from the unsplit sum only by fp32 rounding.
 */
mha_status mha_linear(mha_t handle, const void* A, int64_t lda, int M, int K,
                      const void* W, int64_t ldw, int N, const void* bias,
                      void* C, int64_t ldc, void* stream);

/*
 * mha_linear_ex -- mha_linear plus a residual, C = A W + bias + R: the output projection of
 * the residual form X' = X + O W_O (iamjaehka13.blog "[Deep Learning 5] Attention의 내부
 * 계산", section 14) with the addition in the GEMM's epilogue.  R (M, N) row stride ldr, or
 * NULL; it may be C itself with ldr == ldc (in place), but must not otherwise overlap C
 * (MHA_ERR_INVALID_ARG).  bf16 needs ldr a multiple of 8 and R 16-byte aligned.
 */
mha_status mha_linear_ex(mha_t handle, const void* A, int64_t lda, int M, int K,
                         const void* W, int64_t ldw, int N, const void* bias, const void* R,
                         int64_t ldr, void* C, int64_t ldc, void* stream);

/*
 * mha_linear_segments -- mha_linear for the key/value projection of cross-attention with key
 * padding (molayo1419.me "MHA란 무엇인가?", pitfalls 2 and 3: padded keys are excluded, so
 * their projections are never used).  The M rows form M / seg_rows segments of seg_rows
 * consecutive rows (segment b = batch b of a (B, T_kv, *) tensor, seg_rows = T_kv);
 * seg_len is a device int32[M / seg_rows] of valid lengths.  Rows of segment b at or past
 * seg_len[b] rounded up to a multiple of 128 may be left unwritten (their contents are then
 * unspecified); every other row is exactly what mha_linear writes.  The attention step
 * (mha_attention with the same lengths) reads only whole 128-key tiles up to each length, so
 * it never reads an unwritten row.  The skipped rows are whole 256-row blocks; for fp32
 * handles, or more than 131072 rows, every row is written.
 * seg_len NULL, seg_rows <= 0 or M not a multiple of seg_rows: MHA_ERR_INVALID_ARG; other
 * arguments as for mha_linear.
 */
/*
 * mha_linear_pair -- two independent projections that share the inner dimension K, in one
 * launch where possible: C = A W + bias (M x N; with seg_len, the rows of each segment past
 * its length may be left unwritten exactly as in mha_linear_segments) and C2 = A2 W2 + bias2
 * (M2 x N2).  Cross-attention projects its key/value side and its query side this way
 * (itwiki.kr "멀티 헤드 어텐션", tensor-shape table row 투영, with the query and key/value inputs
 * of the cross-attention form): for bf16 handles with M > 128 and M2 > 128 both run on one
 * persistent grid of CTA pairs, so the smaller one fills the larger one's last round instead of
 * adding rounds of its own; otherwise they run one after the other on `stream`.
 * Arguments as for mha_linear (both) and mha_linear_segments (seg_len, seg_rows; seg_len may be
 * NULL, then seg_rows is ignored).  M2 == 0 or M == 0 skips that projection.  C and C2 may not
 * overlap each other or any input of either projection (MHA_ERR_INVALID_ARG).
 */
mha_status mha_linear_pair(mha_t handle, const void* A, int64_t lda, int M, const void* W,
                           int64_t ldw, int N, const void* bias, const int32_t* seg_len,
                           int seg_rows, void* C, int64_t ldc, const void* A2, int64_t lda2,
                           int M2, const void* W2, int64_t ldw2, int N2, const void* bias2,
                           void* C2, int64_t ldc2, int K, void* stream);

mha_status mha_linear_segments(mha_t handle, const void* A, int64_t lda, int M, int K,
                               const void* W, int64_t ldw, int N, const void* bias,
                               const int32_t* seg_len, int seg_rows, void* C, int64_t ldc,
                               void* stream);

/*
 * mha_attention -- the fused attention step for all heads: scores, scale,
 * mask, row softmax and weighted sum, written straight into the
 * concatenated layout (itwiki.kr "멀티 헤드 어텐션", table rows 헤드 분리
 * through 헤드 결합).  The (B,h,T_q,T_kv) scores never reach memory.
 *   Q  rows (B, T_q) of stride ldq; head i reads columns [i*d_k, (i+1)*d_k)
 *   K  rows (B, T_kv) of stride ldk; head i reads columns [i*d_k, (i+1)*d_k)
 *   V  rows (B, T_kv) of stride ldv; head i reads columns [i*d_v, (i+1)*d_v)
 *   O  rows (B, T_q) of stride ldo; head i writes columns [i*d_v, (i+1)*d_v)
 * causal / kv_lengths as for mha_forward.  The head split is this strided
 * addressing: the projection output is read in place, never copied.
 */
mha_status mha_attention(mha_t handle, int B, int T_q, int T_kv,
                         const void* Q, int64_t ldq, const void* K, int64_t ldk,
                         const void* V, int64_t ldv, int causal, const int32_t* kv_lengths,
                         void* O, int64_t ldo, void* stream);

/*
 * mha_attention_ex -- mha_attention with the handle's K/V head count and an optional gate.
 *   K, V  head g of the h_kv K/V heads at columns [g*d_k, (g+1)*d_k) / [g*d_v, (g+1)*d_v);
 *         query head i reads K/V head i / (h / h_kv)
 *   G     NULL, or the gate pre-activations, rows (B, T_q) of stride ldg, head i at
 *         columns [i*d_v, (i+1)*d_v): O = softmax(...) V * sigmoid(G), element by element
 * mha_attention(...) is mha_attention_ex(..., G = NULL, ldg = 0, ...).
 */
mha_status mha_attention_ex(mha_t handle, int B, int T_q, int T_kv,
                            const void* Q, int64_t ldq, const void* K, int64_t ldk,
                            const void* V, int64_t ldv, const void* G, int64_t ldg, int causal,
                            const int32_t* kv_lengths, void* O, int64_t ldo, void* stream);

/*
 * mha_decode_workspace_size -- bytes of workspace mha_decode needs: the 256-byte status
 * block and, for bf16, the per-chunk partial results of the split over the cache (B*h*T_q
 * rows, one (max, sum, d_v values) record per 128 cached tokens).  0 for an invalid handle.
 */
size_t mha_decode_workspace_size(mha_t handle, int B, int T_q, int T_max);

/*
 * mha_decode -- one decode step over a key/value cache (itwiki.kr "멀티 헤드 어텐션",
 * section 추론 비용과 변형: generation keeps the keys and values of earlier tokens and
 * every step reads the whole cache, so the step is bound by memory bandwidth).
 *   Q        the T_q new tokens' queries, rows (B, T_q) of stride ldq, head i at columns
 *            [i*d_k, (i+1)*d_k)
 *   K_cache  rows (B, T_max) of stride ldk, K/V head g at columns [g*d_k, (g+1)*d_k)
 *   V_cache  rows (B, T_max) of stride ldv, K/V head g at columns [g*d_v, (g+1)*d_v)
 *   cache_lengths  device int32[B]: L_b cached tokens, the T_q new ones included (their keys
 *            and values already written at rows L_b - T_q .. L_b - 1)
 *   O        rows (B, T_q) of stride ldo, head i at columns [i*d_v, (i+1)*d_v)
 * New token t sees cache rows j <= L_b - T_q + t; query head i uses K/V head i / (h / h_kv).
 * L_b outside [T_q, T_max] makes that batch's rows NaN and records MHA_ERR_BAD_LENGTH.
 * bf16 (d_k == d_v in {64, 128}) splits the cache over many CTAs and needs a workspace of
 * mha_decode_workspace_size bytes (MHA_ERR_WORKSPACE otherwise); fp32 (d_k, d_v <= 256) needs
 * none.  B == 0 or T_q == 0 is a no-op; T_q > T_max or cache_lengths == NULL is
 * MHA_ERR_INVALID_ARG.  Launches two kernels (bf16) or one (fp32) on `stream`.
 */
mha_status mha_decode(mha_t handle, int B, int T_q, int T_max, const void* Q, int64_t ldq,
                      const void* K_cache, int64_t ldk, const void* V_cache, int64_t ldv,
                      const int32_t* cache_lengths, void* O, int64_t ldo, void* stream);

/*
 * mha_get_status -- copy the device status word of the attached workspace to
 * *status_out (an mha_status: MHA_OK, MHA_ERR_TIMEOUT or MHA_ERR_BAD_LENGTH;
 * the first error recorded wins) and reset it to MHA_OK.  Synchronises
 * `stream`.  Returns MHA_ERR_WORKSPACE if no workspace is attached.
 */
mha_status mha_get_status(mha_t handle, int32_t* status_out, void* stream);

/*
 * mha_check_wait_timeout -- exercise the failure path of the kernels' pipeline waits.  (The
 * pages have no counterpart: this is the library's own failure detection.)  Every wait on a
 * pipeline barrier inside the kernels gives up after one second, records MHA_ERR_TIMEOUT in
 * the workspace status word and lets the kernel drain and exit instead of hanging.  This call
 * launches one small kernel whose waits are on a barrier that nothing ever completes, with
 * the given limit (1 ns .. 10 s), so a test can check that the timeout is reported through
 * mha_get_status and that the CUDA context stays usable.  Needs an attached workspace
 * (MHA_ERR_WORKSPACE otherwise); MHA_ERR_INVALID_ARG for a NULL handle or a limit out of
 * range.  Asynchronous on `stream`.
 */
mha_status mha_check_wait_timeout(mha_t handle, int64_t limit_ns, void* stream);

/* mha_strerror -- static description of a status code. */
const char* mha_strerror(mha_status status);

/* Size of the library-owned scratch array behind mha_forward_static_workspace: 32 MiB. */
#define MHA_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * mha_forward_static_workspace -- mha_forward for callers that may not allocate device
 * memory.  The pages have no counterpart to this call: they define the operation, not how
 * its scratch memory is provided.
 *
 * Who needs it: code that cannot call cudaMalloc (or ask anyone to) -- for example a library
 * embedded in a host framework that owns every device allocation through its own pool and
 * hands plugins no scratch buffer, or a latency-critical serving loop where cudaMalloc's
 * implicit device-wide synchronisation is not acceptable.  Such a caller still owns and
 * passes every input and the output; only the scratch (status word, projected Q/K/V, Ocat)
 * comes from a file-scope __device__ array of MHA_STATIC_WORKSPACE_BYTES inside this library.
 * Every GPU that loads the library holds that array until the process exits.
 *
 *  - Arguments, layouts and result are those of mha_forward.  The handle's own workspace
 *    (mha_set_workspace) is neither used nor modified.
 *  - status_out: NULL, or a 4-byte aligned device int32 that receives this call's device
 *    status (MHA_OK, MHA_ERR_TIMEOUT or MHA_ERR_BAD_LENGTH, as mha_get_status reports it for
 *    mha_forward), copied on `stream` after the last kernel.  mha_get_status cannot see it:
 *    it reads the handle's own workspace.
 *  - Returns MHA_ERR_WORKSPACE, before any CUDA call, when mha_workspace_size(B, T_q, T_kv)
 *    exceeds MHA_STATIC_WORKSPACE_BYTES; every other argument error of mha_forward is also
 *    reported before the array or *status_out is touched.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - The first call on a device (and again after that device's context was destroyed and
 *    created anew, as by cudaDeviceReset) looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and remembers it for that context;
 *    make that first call before any stream capture.  Concurrent first calls from several
 *    host threads are safe.
 *  - All calls share the one array, which keeps the previous call's contents: calls that
 *    overlap on the GPU (other streams or host threads on the same device) race on it and
 *    must be serialised by the caller.
 *  - Each call zeroes the array's status word first (cudaMemsetAsync on `stream`).
 */
mha_status mha_forward_static_workspace(mha_t handle, const void* X_q, const void* X_kv, int B,
                                        int T_q, int T_kv, const void* W_qkv, const void* b_qkv,
                                        const void* W_o, const void* b_o, int causal,
                                        const int32_t* kv_lengths, void* out,
                                        int32_t* status_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MHA_H_ */
