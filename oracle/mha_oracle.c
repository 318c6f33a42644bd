/*
 * mha_oracle.c -- plain fp64 CPU reference of the multi-head attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the library under
 * transformer_head_scaled_02_gb300/ never links, imports or calls it, and it
 * shares no code, header, table or helper with that library.
 *
 * What it computes is the textbook definition, written out with no blocking,
 * fusion or reordering beyond what the definition states:
 *
 *   itwiki.kr "멀티 헤드 어텐션", section 수식 (equations):
 *     Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V
 *     MultiHead = Concat(head_1..head_h) W^O,  head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V)
 *   same page, section 텐서 모양으로 본 계산 (tensor-shape table):
 *     projections fused into one D x 3D matrix, head split by view+transpose
 *     (head i = column slice [i*d_k, (i+1)*d_k) of its Q/K/V block),
 *     scores (B,h,T,T) with optional causal mask, softmax over the last axis,
 *     weighted sum, Concat (head i at columns [i*d_v, (i+1)*d_v)), W^O.
 *   iamjaehka13.blog "[Deep Learning 5] Attention의 내부 계산", sections 9-10:
 *     causal mask M_ij = -inf for j > i, 0 otherwise; A = softmax(S/sqrt(d_k) + M)
 *     row-wise; masked weights are exactly exp(-inf) = 0.
 *   same page, section 19: cross-attention takes Q from the target sequence
 *     and K, V from the source sequence.
 *   molayo1419.me "MHA란 무엇인가?", pitfall 2/3: key padding excludes keys; a
 *     row whose keys are all excluded has an undefined softmax (NaN).
 *
 * Variants (same pages):
 *   - residual (iamjaehka13.blog, sections 14 and 16): X' = X + O W_O; here the
 *     residual is any (B, T_q, D) tensor added to Y, normally X_q itself;
 *   - grouped K/V heads, MQA / GQA (itwiki.kr "멀티 헤드 어텐션", section 추론 비용과
 *     변형, its table): h query heads share h_kv K/V head sets, h_kv = 1 is MQA and
 *     h_kv = h is plain MHA;
 *   - gated attention (same section): a per-head sigmoid gate multiplies the scaled
 *     dot-product attention output before W^O;
 *   - KV-cache decode (same section): new query rows attend to the key/value cache
 *     of the tokens so far.
 *
 * Readings of points the pages leave open (each also listed in the design notes):
 *   - weights are (in, out) row-major so that Y = X W + b;
 *   - key padding is given as a per-batch valid length L_b: keys j >= L_b are
 *     masked; L_b outside [1, T_kv] is invalid and its rows come out NaN;
 *   - causal masking is defined only for T_q == T_kv (top-left aligned);
 *   - causal and padding masks combine by logical OR;
 *   - grouped heads: query head i uses K/V head i / (h / h_kv) (consecutive query heads
 *     form a group); the fused projection's column blocks are [Q | K | V], of widths
 *     h*d_k, h_kv*d_k, h_kv*d_v;
 *   - the gate is elementwise and head-specific: G = sigmoid(X_q W_G + b_G), W_G of
 *     shape (D, h*d_v) stored as a fourth column block of the fused projection, and
 *     O_cat is multiplied by G element by element;
 *   - decode: the T_q new tokens are the last T_q of each batch's L_b cached tokens,
 *     so new token t sees cache entries j <= L_b - T_q + t (causal, bottom-aligned);
 *     L_b < T_q or L_b > T_max is invalid and gives NaN rows.
 *
 * Precision: every operation is IEEE fp64; exp is libm exp().
 *
 * Rounded mode (oracle_mha_forward_rounded, a secondary diagnostic): the same steps, with the
 * values the bf16 GPU path stores rounded to bf16 (round to nearest, ties to even) where it
 * stores them -- the projections Q, K, V (and the gate pre-activations), the unnormalised
 * softmax weights exp(s_j - m) that enter the weighted sum (their sum, the denominator, is
 * not rounded), the attention output after the gate, and Y.  The pass/fail reference stays
 * the unrounded forward.
 * Threads: OpenMP over independent output rows / (batch, head) pairs; the
 * arithmetic done for any one output element does not depend on the thread
 * count.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEM 2

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/*
 * x rounded to the nearest bfloat16 value (8 significant bits), ties to even: with
 * x = m * 2^e and 0.5 <= |m| < 1, keep m * 2^8 rounded to an integer (nearbyint rounds to
 * nearest, ties to even, in the default rounding mode).  Values below the bf16 normal range
 * (2^-126) are rounded as if it extended further; none arise here.
 */
double oracle_round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    const double m = frexp(x, &e);
    return ldexp(nearbyint(ldexp(m, 8)), e - 8);
}

static void round_all(double* a, long n) {
    for (long i = 0; i < n; ++i) a[i] = oracle_round_bf16(a[i]);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Linear projection, one row at a time:
 *   Y[m, n] = sum_{k=0}^{K-1} X[m, k] * W[k, n]  (+ b[n] if b != NULL)
 * X is (M, K) with row stride ldx, W is (K, N) with row stride ldw, Y is (M, N)
 * with row stride ldy.  The sum over k runs in increasing k.
 * itwiki.kr "멀티 헤드 어텐션", tensor-shape table rows 투영 and 출력 투영.
 */
int oracle_linear(long M, long K, long N,
                  const double* X, long ldx,
                  const double* W, long ldw,
                  const double* b,
                  double* Y, long ldy, int nthreads) {
    if (M < 0 || K < 0 || N < 0 || !X || !W || !Y) return ORACLE_BAD_ARG;
    set_threads(nthreads);
    long m;
#pragma omp parallel for schedule(static)
    for (m = 0; m < M; ++m) {
        double* y = Y + m * ldy;
        for (long n = 0; n < N; ++n) y[n] = 0.0;
        for (long k = 0; k < K; ++k) {
            const double xk = X[m * ldx + k];
            const double* w = W + k * ldw;
            for (long n = 0; n < N; ++n) y[n] += xk * w[n];
        }
        if (b)
            for (long n = 0; n < N; ++n) y[n] += b[n];
    }
    return ORACLE_OK;
}

/*
 * Scaled dot-product attention for every (batch, head, query row).
 *
 * Q is (B, Tq) rows of stride ldq; head i reads columns [i*dk, (i+1)*dk).
 * K is (B, Tkv) rows of stride ldk; head i reads columns [i*dk, (i+1)*dk).
 * V is (B, Tkv) rows of stride ldv; head i reads columns [i*dv, (i+1)*dv).
 * O is (B, n_out) rows of stride ldo; head i writes columns [i*dv, (i+1)*dv)
 *   (this is the Concat of the heads).
 * rows: if non-NULL, the n_rows query indices (the same for every batch) to
 *   compute; output row r of batch b is query rows[r].  If NULL, all Tq rows.
 * kv_lengths: if non-NULL, L_b per batch; keys j >= L_b are masked.
 * P: if non-NULL, receives the softmax weights, shape (B, h, n_out, Tkv).
 *
 * Per output row (the definition, in order):
 *   s_j = (sum_e q_e k_je) / sqrt(dk)                  for j in [0, Tkv)
 *   s_j = -inf  if (causal and j > t) or j >= L_b
 *   m   = max_j s_j
 *   w_j = exp(s_j - m) / sum_j' exp(s_j' - m)
 *   o_e = sum_j w_j v_je
 * The whole score row is materialised before the softmax.
 */
static int attention_impl(int B, int Tq, int Tkv, int h, int h_kv, int dk, int dv,
                          const double* Q, long ldq,
                          const double* K, long ldk,
                          const double* V, long ldv,
                          int causal, const int* kv_lengths,
                          const int* rows, int n_rows,
                          double* O, long ldo, double* P, int nthreads, int round_p) {
    if (B < 0 || Tq < 0 || Tkv < 0 || h <= 0 || dk <= 0 || dv <= 0) return ORACLE_BAD_ARG;
    if (h_kv <= 0 || h % h_kv != 0) return ORACLE_BAD_ARG;
    if (!Q || !K || !V || !O) return ORACLE_BAD_ARG;
    if (causal && Tq != Tkv) return ORACLE_BAD_ARG;
    const int n_out = rows ? n_rows : Tq;
    if (rows)
        for (int r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= Tq) return ORACLE_BAD_ARG;
    set_threads(nthreads);
    const double scale = 1.0 / sqrt((double)dk);
    int status = ORACLE_OK;
    long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long)B * h; ++bh) {
        const int b = (int)(bh / h);
        const int i = (int)(bh % h);
        const int g = i / (h / h_kv); /* the K/V head of query head i */
        const int L = kv_lengths ? kv_lengths[b] : Tkv;
        const int valid_len = (L >= 1 && L <= Tkv);
        double* s = (double*)malloc(sizeof(double) * (size_t)(Tkv > 0 ? Tkv : 1));
        if (!s) {
#pragma omp atomic write
            status = ORACLE_NO_MEM;
            continue;
        }
        for (int r = 0; r < n_out; ++r) {
            const int t = rows ? rows[r] : r;
            const double* q = Q + ((long)b * Tq + t) * ldq + (long)i * dk;
            double* o = O + ((long)b * n_out + r) * ldo + (long)i * dv;
            double* prow = P ? P + (((long)b * h + i) * n_out + r) * (long)Tkv : NULL;
            if (!valid_len) {
                /* every key is excluded (or the length is out of range): the
                   softmax is undefined and the row is NaN */
                for (int e = 0; e < dv; ++e) o[e] = NAN;
                if (prow)
                    for (int j = 0; j < Tkv; ++j) prow[j] = NAN;
                continue;
            }
            /* scores, scaled, masked */
            for (int j = 0; j < Tkv; ++j) {
                const double* kj = K + ((long)b * Tkv + j) * ldk + (long)g * dk;
                double dot = 0.0;
                for (int e = 0; e < dk; ++e) dot += q[e] * kj[e];
                s[j] = dot * scale;
                if ((causal && j > t) || j >= L) s[j] = -INFINITY;
            }
            /* row softmax */
            double m = -INFINITY;
            for (int j = 0; j < Tkv; ++j)
                if (s[j] > m) m = s[j];
            double sum = 0.0;
            for (int j = 0; j < Tkv; ++j) {
                s[j] = exp(s[j] - m);
                sum += s[j];
            }
            /* rounded mode: the weights enter the weighted sum as bf16, the sum does not */
            for (int j = 0; j < Tkv; ++j) s[j] = (round_p ? oracle_round_bf16(s[j]) : s[j]) / sum;
            if (prow) memcpy(prow, s, sizeof(double) * (size_t)Tkv);
            /* weighted sum of values */
            for (int e = 0; e < dv; ++e) o[e] = 0.0;
            for (int j = 0; j < Tkv; ++j) {
                const double w = s[j];
                const double* vj = V + ((long)b * Tkv + j) * ldv + (long)g * dv;
                for (int e = 0; e < dv; ++e) o[e] += w * vj[e];
            }
        }
        free(s);
    }
    return status;
}

int oracle_attention_grouped(int B, int Tq, int Tkv, int h, int h_kv, int dk, int dv,
                             const double* Q, long ldq,
                             const double* K, long ldk,
                             const double* V, long ldv,
                             int causal, const int* kv_lengths,
                             const int* rows, int n_rows,
                             double* O, long ldo, double* P, int nthreads) {
    return attention_impl(B, Tq, Tkv, h, h_kv, dk, dv, Q, ldq, K, ldk, V, ldv, causal, kv_lengths,
                          rows, n_rows, O, ldo, P, nthreads, 0);
}

/* Plain multi-head attention: every query head has its own K/V head. */
int oracle_attention(int B, int Tq, int Tkv, int h, int dk, int dv,
                     const double* Q, long ldq,
                     const double* K, long ldk,
                     const double* V, long ldv,
                     int causal, const int* kv_lengths,
                     const int* rows, int n_rows,
                     double* O, long ldo, double* P, int nthreads) {
    return oracle_attention_grouped(B, Tq, Tkv, h, h, dk, dv, Q, ldq, K, ldk, V, ldv, causal,
                                    kv_lengths, rows, n_rows, O, ldo, P, nthreads);
}

/*
 * The whole forward: projections, attention of every head, Concat, W^O, and the
 * variants (grouped K/V heads, output gate, residual).
 *
 *   Xq  (B, Tq, D);  Xkv (B, Tkv, D), or NULL for self-attention (Xkv = Xq)
 *   Wqkv (D, h*dk + h_kv*dk + h_kv*dv [+ h*dv if gated]), column blocks
 *        [Q | K | V (| G)]; bqkv the same width or NULL
 *   Wo  (h*dv, D); bo (D) or NULL
 *   R   (B, Tq, D) residual or NULL
 *   Y   (B, n_out, D) where n_out = n_rows if rows != NULL else Tq
 *
 * Only the query rows asked for are projected; every key/value row is
 * projected.  Steps:
 *   Qf = Xq  W[:, Q block] + b[Q block]
 *   Kf = Xkv W[:, K block] + b[K block]
 *   Vf = Xkv W[:, V block] + b[V block]
 *   Ocat = attention(Qf, Kf, Vf)      (head i at columns i*dv, K/V head i/(h/h_kv))
 *   if gated:  Gf = Xq W[:, G block] + b[G block];  Ocat *= 1 / (1 + exp(-Gf))
 *   Y  = Ocat Wo + bo  (+ R)
 */
static int forward_impl(int B, int Tq, int Tkv, int D, int h, int h_kv, int dk, int dv,
                        int gated, const double* Xq, const double* Xkv,
                        const double* Wqkv, const double* bqkv,
                        const double* Wo, const double* bo, const double* R,
                        int causal, const int* kv_lengths,
                        const int* rows, int n_rows,
                        double* Y, int nthreads, int rounded) {
    if (B < 0 || Tq < 0 || Tkv < 0 || D <= 0 || h <= 0 || dk <= 0 || dv <= 0) return ORACLE_BAD_ARG;
    if (h_kv <= 0 || h % h_kv != 0) return ORACLE_BAD_ARG;
    if (!Xq || !Wqkv || !Wo || !Y) return ORACLE_BAD_ARG;
    if (!Xkv) {
        Xkv = Xq;
        if (Tkv != Tq) return ORACLE_BAD_ARG;
    }
    if (causal && Tq != Tkv) return ORACLE_BAD_ARG;
    const int n_out = rows ? n_rows : Tq;
    const long hq = (long)h * dk, hk = (long)h_kv * dk, hkv = (long)h_kv * dv, hv = (long)h * dv;
    const long wcols = hq + hk + hkv + (gated ? hv : 0);
    const long k_off = hq, v_off = hq + hk, g_off = hq + hk + hkv;
    double* Xsel = (double*)malloc(sizeof(double) * (size_t)((long)B * n_out * D + 1));
    double* Qf = (double*)malloc(sizeof(double) * (size_t)((long)B * n_out * hq + 1));
    double* Kf = (double*)malloc(sizeof(double) * (size_t)((long)B * Tkv * hk + 1));
    double* Vf = (double*)malloc(sizeof(double) * (size_t)((long)B * Tkv * hkv + 1));
    double* Oc = (double*)malloc(sizeof(double) * (size_t)((long)B * n_out * hv + 1));
    double* Gf = gated ? (double*)malloc(sizeof(double) * (size_t)((long)B * n_out * hv + 1)) : NULL;
    int rc = ORACLE_OK;
    if (!Xsel || !Qf || !Kf || !Vf || !Oc || (gated && !Gf)) {
        rc = ORACLE_NO_MEM;
        goto done;
    }
    /* the query rows asked for, batch by batch */
    for (int b = 0; b < B; ++b)
        for (int r = 0; r < n_out; ++r) {
            const int t = rows ? rows[r] : r;
            if (t < 0 || t >= Tq) {
                rc = ORACLE_BAD_ARG;
                goto done;
            }
            memcpy(Xsel + ((long)b * n_out + r) * D, Xq + ((long)b * Tq + t) * D, sizeof(double) * (size_t)D);
        }
    rc = oracle_linear((long)B * n_out, D, hq, Xsel, D, Wqkv, wcols, bqkv, Qf, hq, nthreads);
    if (rc) goto done;
    rc = oracle_linear((long)B * Tkv, D, hk, Xkv, D, Wqkv + k_off, wcols, bqkv ? bqkv + k_off : NULL, Kf,
                       hk, nthreads);
    if (rc) goto done;
    rc = oracle_linear((long)B * Tkv, D, hkv, Xkv, D, Wqkv + v_off, wcols, bqkv ? bqkv + v_off : NULL, Vf,
                       hkv, nthreads);
    if (rc) goto done;
    if (rounded) {
        round_all(Qf, (long)B * n_out * hq);
        round_all(Kf, (long)B * Tkv * hk);
        round_all(Vf, (long)B * Tkv * hkv);
    }
    {
        /* the attention step sees the selected rows as a (B, n_out) query
           block; the causal test needs each row's original index t, so the
           rows are computed one original index at a time */
        if (rows) {
            double* Qfull = (double*)calloc((size_t)((long)B * Tq * hq + 1), sizeof(double));
            if (!Qfull) {
                rc = ORACLE_NO_MEM;
                goto done;
            }
            for (int b = 0; b < B; ++b)
                for (int r = 0; r < n_out; ++r)
                    memcpy(Qfull + ((long)b * Tq + rows[r]) * hq, Qf + ((long)b * n_out + r) * hq,
                           sizeof(double) * (size_t)hq);
            rc = attention_impl(B, Tq, Tkv, h, h_kv, dk, dv, Qfull, hq, Kf, hk, Vf, hkv, causal,
                                kv_lengths, rows, n_rows, Oc, hv, NULL, nthreads, rounded);
            free(Qfull);
        } else {
            rc = attention_impl(B, Tq, Tkv, h, h_kv, dk, dv, Qf, hq, Kf, hk, Vf, hkv, causal,
                                kv_lengths, NULL, 0, Oc, hv, NULL, nthreads, rounded);
        }
        if (rc) goto done;
    }
    if (gated) {
        /* the gate of every output element, from the query-side input */
        rc = oracle_linear((long)B * n_out, D, hv, Xsel, D, Wqkv + g_off, wcols, bqkv ? bqkv + g_off : NULL,
                           Gf, hv, nthreads);
        if (rc) goto done;
        if (rounded) round_all(Gf, (long)B * n_out * hv);
        for (long e = 0; e < (long)B * n_out * hv; ++e) Oc[e] = Oc[e] * (1.0 / (1.0 + exp(-Gf[e])));
    }
    if (rounded) round_all(Oc, (long)B * n_out * hv);
    rc = oracle_linear((long)B * n_out, hv, D, Oc, hv, Wo, D, bo, Y, D, nthreads);
    if (rc) goto done;
    if (R) {
        for (int b = 0; b < B; ++b)
            for (int r = 0; r < n_out; ++r) {
                const int t = rows ? rows[r] : r;
                const double* rr = R + ((long)b * Tq + t) * D;
                double* y = Y + ((long)b * n_out + r) * D;
                for (int c = 0; c < D; ++c) y[c] += rr[c];
            }
    }
    if (rounded) round_all(Y, (long)B * n_out * D);
done:
    free(Xsel);
    free(Qf);
    free(Kf);
    free(Vf);
    free(Oc);
    free(Gf);
    return rc;
}

int oracle_mha_forward_ex(int B, int Tq, int Tkv, int D, int h, int h_kv, int dk, int dv,
                          int gated, const double* Xq, const double* Xkv,
                          const double* Wqkv, const double* bqkv,
                          const double* Wo, const double* bo, const double* R,
                          int causal, const int* kv_lengths,
                          const int* rows, int n_rows,
                          double* Y, int nthreads) {
    return forward_impl(B, Tq, Tkv, D, h, h_kv, dk, dv, gated, Xq, Xkv, Wqkv, bqkv, Wo, bo, R, causal,
                        kv_lengths, rows, n_rows, Y, nthreads, 0);
}

/* The forward with bf16 rounding at the GPU path's storage points (see the header). */
int oracle_mha_forward_rounded(int B, int Tq, int Tkv, int D, int h, int h_kv, int dk, int dv,
                               int gated, const double* Xq, const double* Xkv,
                               const double* Wqkv, const double* bqkv,
                               const double* Wo, const double* bo, const double* R,
                               int causal, const int* kv_lengths,
                               const int* rows, int n_rows,
                               double* Y, int nthreads) {
    return forward_impl(B, Tq, Tkv, D, h, h_kv, dk, dv, gated, Xq, Xkv, Wqkv, bqkv, Wo, bo, R, causal,
                        kv_lengths, rows, n_rows, Y, nthreads, 1);
}

/* The plain forward: h K/V heads, no gate, no residual. */
int oracle_mha_forward(int B, int Tq, int Tkv, int D, int h, int dk, int dv,
                       const double* Xq, const double* Xkv,
                       const double* Wqkv, const double* bqkv,
                       const double* Wo, const double* bo,
                       int causal, const int* kv_lengths,
                       const int* rows, int n_rows,
                       double* Y, int nthreads) {
    return oracle_mha_forward_ex(B, Tq, Tkv, D, h, h, dk, dv, 0, Xq, Xkv, Wqkv, bqkv, Wo, bo, NULL,
                                 causal, kv_lengths, rows, n_rows, Y, nthreads);
}

/*
 * Attention of new query rows over a key/value cache (one decode step).
 *
 * Q  (B, Tq) rows of stride ldq, head i at columns [i*dk, (i+1)*dk);
 * Kc (B, Tmax) rows of stride ldk, K/V head g at columns [g*dk, (g+1)*dk);
 * Vc (B, Tmax) rows of stride ldv, K/V head g at columns [g*dv, (g+1)*dv);
 * cache_lengths: L_b per batch, the tokens cached so far including the Tq new ones;
 * O  (B, Tq) rows of stride ldo, head i at columns [i*dv, (i+1)*dv).
 *
 * New row t of batch b is token L_b - Tq + t and sees cache entries
 * j <= L_b - Tq + t; query head i uses K/V head i / (h / h_kv).  Per row:
 *   s_j = (sum_e q_e k_je) / sqrt(dk)   for visible j
 *   w_j = exp(s_j - max s) / sum exp(s - max s),   o_e = sum_j w_j v_je
 */
int oracle_decode(int B, int Tq, int Tmax, int h, int h_kv, int dk, int dv,
                  const double* Q, long ldq, const double* Kc, long ldk, const double* Vc, long ldv,
                  const int* cache_lengths, double* O, long ldo, int nthreads) {
    if (B < 0 || Tq <= 0 || Tmax <= 0 || h <= 0 || dk <= 0 || dv <= 0) return ORACLE_BAD_ARG;
    if (h_kv <= 0 || h % h_kv != 0 || !Q || !Kc || !Vc || !O || !cache_lengths) return ORACLE_BAD_ARG;
    set_threads(nthreads);
    const double scale = 1.0 / sqrt((double)dk);
    int status = ORACLE_OK;
    long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long)B * h; ++bh) {
        const int b = (int)(bh / h);
        const int i = (int)(bh % h);
        const int g = i / (h / h_kv);
        const int L = cache_lengths[b];
        double* s = (double*)malloc(sizeof(double) * (size_t)Tmax);
        if (!s) {
#pragma omp atomic write
            status = ORACLE_NO_MEM;
            continue;
        }
        for (int t = 0; t < Tq; ++t) {
            double* o = O + ((long)b * Tq + t) * ldo + (long)i * dv;
            if (L < Tq || L > Tmax) {
                for (int e = 0; e < dv; ++e) o[e] = NAN;
                continue;
            }
            const int n = L - Tq + t + 1; /* visible cache entries [0, n) */
            const double* q = Q + ((long)b * Tq + t) * ldq + (long)i * dk;
            double m = -INFINITY;
            for (int j = 0; j < n; ++j) {
                const double* kj = Kc + ((long)b * Tmax + j) * ldk + (long)g * dk;
                double dot = 0.0;
                for (int e = 0; e < dk; ++e) dot += q[e] * kj[e];
                s[j] = dot * scale;
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (int j = 0; j < n; ++j) {
                s[j] = exp(s[j] - m);
                sum += s[j];
            }
            for (int e = 0; e < dv; ++e) o[e] = 0.0;
            for (int j = 0; j < n; ++j) {
                const double w = s[j] / sum;
                const double* vj = Vc + ((long)b * Tmax + j) * ldv + (long)g * dv;
                for (int e = 0; e < dv; ++e) o[e] += w * vj[e];
            }
        }
        free(s);
    }
    return status;
}
