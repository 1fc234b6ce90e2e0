/*
 * oracle.c -- plain fp64 CPU oracle for the fused attention forward pass
 * (MHA/GQA prefill) and for MLA decode.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library.  The product
 * path (the CUDA library and its Python binding) never calls it, and the two
 * share no code.
 *
 * What it computes is the plain definition of attention, written out with no
 * tiling, no online rescaling and no fusion:
 *
 *   S = scale * Q K^T (+ mask),  P = softmax(S) row-wise,  O = P V
 *
 * following "TileLang 学习笔记" (sealessland.top), section "FlashAttention 的实现"
 * -> "为什么需要 FlashAttention" (S = Q K^T, P = softmax(S), O = P V).  The
 * softmax is the explicit two-pass form: pass 1 takes the row maximum M, pass 2
 * sums Z = sum_j exp(s_j - M); P_j = exp(s_j - M) / Z.  The max subtraction is
 * the one the same page ("Online softmax 的数值稳定性") says cannot be dropped.
 * LSE_i = M + ln Z (natural log) of the scaled scores.
 *
 * MLA decode follows the devpress.csdn.net FlashMLA article, section 2.2
 * ("计算流水线设计"): the score is the sum of two products, the latent part
 * Q_nope . KV_latent and the RoPE part Q_pe . K_pe, into one accumulator; the
 * value matrix is KV_latent itself (one shared KV head), one query token.
 *
 * Readings where the pages are silent:
 *  - the mask is additive 0 / -inf: a masked key is excluded entirely;
 *  - causal alignment is bottom-right: key j is allowed for query i iff
 *    j <= i + (N_kv - N_q);
 *  - with causal, a window w > 0 keeps keys j >= i + (N_kv - N_q) - w + 1;
 *  - without causal, a window w > 0 is the symmetric local window of the
 *    TileLang study notes ("TileLang 学习笔记", section on local attention
 *    variants: keys from seqpos - w to seqpos + w): with i' = i + (N_kv - N_q),
 *    key j is visible iff i' - w <= j <= i' + w;
 *  - GQA maps query head h to key/value head h / (H / H_kv) (contiguous
 *    groups; the FlashMLA article's section 5.1 shows only kv_head_num = 1);
 *  - a row with no allowed key has O = 0 and LSE = -inf;
 *  - a block-sparse mask (the TileLang study notes' block-sparse variant:
 *    attention computed only where a block-level mask is set) is a byte per
 *    (batch, head, block of `blk` query rows, block of `blk` keys); a zero
 *    byte removes those keys from those rows, on top of the causal / window
 *    rules.
 *
 * Inputs are bf16 bit patterns (uint16), converted exactly to double.  All
 * arithmetic is fp64.  Rows are independent, so threads split the rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Is key j visible to query i?  See the readings in the header comment. */
static int key_allowed(long i, long j, long n_q, long n_kv, int causal, long window)
{
    long off = n_kv - n_q;
    if (causal) {
        if (j > i + off) return 0;
        if (window > 0 && j < i + off - window + 1) return 0;
    } else if (window > 0) {
        if (j < i + off - window || j > i + off + window) return 0;
    }
    return 1;
}

/*
 * Softmax of one score row s[0..n) (masked entries are -INFINITY) and the
 * weighted sum of value rows.  Two passes over s: max, then sum of exp.
 * p_out (may be NULL) receives the normalised probabilities.
 */
static void softmax_weighted_sum(const double *s, long n, const uint16_t *V, long v_row_stride,
                                 int dv, double *o, double *lse, double *p_out)
{
    double M = -INFINITY;
    for (long j = 0; j < n; j++)
        if (s[j] > M) M = s[j];

    for (int c = 0; c < dv; c++) o[c] = 0.0;
    if (M == -INFINITY) {              /* no allowed key */
        *lse = -INFINITY;
        if (p_out)
            for (long j = 0; j < n; j++) p_out[j] = 0.0;
        return;
    }

    double Z = 0.0;
    for (long j = 0; j < n; j++)
        if (s[j] != -INFINITY) Z += exp(s[j] - M);

    for (long j = 0; j < n; j++) {
        double p = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - M) / Z;
        if (p_out) p_out[j] = p;
        if (p == 0.0) continue;
        const uint16_t *v = V + j * v_row_stride;
        for (int c = 0; c < dv; c++) o[c] += p * bf16_to_f64(v[c]);
    }
    *lse = M + log(Z);
}

/* ------------------------------------------------------------------------ */
/* Prefill: O[B,H,N_q,d], LSE[B,H,N_q] from Q[B,H,N_q,d], K,V[B,H_kv,N_kv,d] */

typedef struct {
    const uint16_t *Q, *K, *V;
    double *O, *LSE, *P;
    int B, H, H_kv, N_q, N_kv, d, causal, window;
    double scale;
    const int64_t *rows;   /* flat (b*H + h)*N_q + i, or NULL for all rows */
    int64_t n_rows;
    int n_threads, tid;
    const uint8_t *block_mask;   /* [B][H][ceil(N_q/blk)][ceil(N_kv/blk)], or NULL */
    int blk;
} attn_job;

static void attn_one_row(const attn_job *J, int64_t flat, int64_t out_idx, double *s)
{
    const long n_q = J->N_q, n_kv = J->N_kv;
    const int d = J->d;
    long i = (long)(flat % n_q);
    long bh = (long)(flat / n_q);
    long b = bh / J->H, h = bh % J->H;
    long g = h / (J->H / J->H_kv);                 /* GQA: contiguous head groups */

    const uint16_t *q = J->Q + ((b * J->H + h) * n_q + i) * d;
    const uint16_t *K = J->K + (b * J->H_kv + g) * n_kv * d;
    const uint16_t *V = J->V + (b * J->H_kv + g) * n_kv * d;
    const uint8_t *mrow = NULL;
    if (J->block_mask) {
        const long nqb = (n_q + J->blk - 1) / J->blk, nkb = (n_kv + J->blk - 1) / J->blk;
        mrow = J->block_mask + ((b * J->H + h) * nqb + i / J->blk) * nkb;
    }

    for (long j = 0; j < n_kv; j++) {
        if (!key_allowed(i, j, n_q, n_kv, J->causal, J->window) || (mrow && !mrow[j / J->blk])) {
            s[j] = -INFINITY;
            continue;
        }
        double dot = 0.0;
        const uint16_t *k = K + j * d;
        for (int c = 0; c < d; c++) dot += bf16_to_f64(q[c]) * bf16_to_f64(k[c]);
        s[j] = J->scale * dot;
    }
    softmax_weighted_sum(s, n_kv, V, d, d, J->O + out_idx * d, J->LSE + out_idx,
                         J->P ? J->P + out_idx * n_kv : NULL);
}

static void *attn_worker(void *arg)
{
    const attn_job *J = (const attn_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (J->N_kv > 0 ? J->N_kv : 1));
    if (!s) return (void *)1;
    for (int64_t k = J->tid; k < J->n_rows; k += J->n_threads) {
        int64_t flat = J->rows ? J->rows[k] : k;
        attn_one_row(J, flat, k, s);
    }
    free(s);
    return NULL;
}

static int run_threads(void *(*fn)(void *), void *jobs, size_t job_size, int n_threads)
{
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
    if (!th) return -1;
    int rc = 0;
    for (int t = 0; t < n_threads; t++)
        if (pthread_create(&th[t], NULL, fn, (char *)jobs + t * job_size)) rc = -1;
    for (int t = 0; t < n_threads; t++) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret) rc = -1;
    }
    free(th);
    return rc;
}

/*
 * oracle_attn_fwd: O and LSE for the listed rows (or all rows when rows is
 * NULL, in which case O is [B,H,N_q,d] and LSE [B,H,N_q]).  P, if not NULL,
 * receives the full probability row of each computed row ([n_rows, N_kv]).
 * Returns 0, or -1 on invalid arguments / allocation failure.
 */
int oracle_attn_fwd_masked(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *O, double *LSE,
                           double *P, int B, int H, int H_kv, int N_q, int N_kv, int d, int causal,
                           int window, double scale, const uint8_t *block_mask, int blk,
                           const int64_t *rows, int64_t n_rows, int n_threads);

int oracle_attn_fwd(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *O, double *LSE,
                    double *P, int B, int H, int H_kv, int N_q, int N_kv, int d, int causal,
                    int window, double scale, const int64_t *rows, int64_t n_rows, int n_threads)
{
    return oracle_attn_fwd_masked(Q, K, V, O, LSE, P, B, H, H_kv, N_q, N_kv, d, causal, window, scale,
                                  NULL, 1, rows, n_rows, n_threads);
}

/*
 * oracle_attn_fwd_masked: oracle_attn_fwd with an optional block-sparse mask
 * (NULL: none) of blk x blk (query rows x keys) blocks.
 */
int oracle_attn_fwd_masked(const uint16_t *Q, const uint16_t *K, const uint16_t *V, double *O, double *LSE,
                           double *P, int B, int H, int H_kv, int N_q, int N_kv, int d, int causal,
                           int window, double scale, const uint8_t *block_mask, int blk,
                           const int64_t *rows, int64_t n_rows, int n_threads)
{
    if (blk < 1) return -1;
    if (B < 0 || H <= 0 || H_kv <= 0 || H % H_kv || N_q < 0 || N_kv < 0 || d <= 0) return -1;
    int64_t total = (int64_t)B * H * N_q;
    if (!rows) n_rows = total;
    if (n_rows == 0) return 0;
    for (int64_t k = 0; rows && k < n_rows; k++)
        if (rows[k] < 0 || rows[k] >= total) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_rows) n_threads = (int)n_rows;

    attn_job *jobs = (attn_job *)malloc(sizeof(attn_job) * n_threads);
    if (!jobs) return -1;
    for (int t = 0; t < n_threads; t++) {
        attn_job j = {Q, K, V, O, LSE, P, B, H, H_kv, N_q, N_kv, d, causal, window,
                      scale, rows, n_rows, n_threads, t, block_mask, blk};
        jobs[t] = j;
    }
    int rc = run_threads(attn_worker, jobs, sizeof(attn_job), n_threads);
    free(jobs);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* MLA decode: one query token per sequence, one shared latent KV head.       */
/*   s_j = scale * (Q_nope[b,h,:] . KV_latent[b,j,:] + Q_pe[b,h,:] . K_pe[b,j,:]) */
/*   O[b,h,:] = sum_j softmax(s)_j * KV_latent[b,j,:]                         */

typedef struct {
    const uint16_t *Qn, *Qp, *KV, *Kp;
    double *O, *LSE;
    int B, H, N_kv, d_c, d_r;
    double scale;
    const int64_t *rows;   /* flat b*H + h, or NULL */
    int64_t n_rows;
    int n_threads, tid;
} mla_job;

static void *mla_worker(void *arg)
{
    const mla_job *J = (const mla_job *)arg;
    const long n_kv = J->N_kv;
    const int dc = J->d_c, dr = J->d_r;
    double *s = (double *)malloc(sizeof(double) * (n_kv > 0 ? n_kv : 1));
    if (!s) return (void *)1;
    for (int64_t k = J->tid; k < J->n_rows; k += J->n_threads) {
        int64_t flat = J->rows ? J->rows[k] : k;
        long b = (long)(flat / J->H), h = (long)(flat % J->H);
        const uint16_t *qn = J->Qn + (b * J->H + h) * dc;
        const uint16_t *qp = J->Qp + (b * J->H + h) * dr;
        const uint16_t *KV = J->KV + b * n_kv * dc;
        const uint16_t *Kp = J->Kp + b * n_kv * dr;
        for (long j = 0; j < n_kv; j++) {
            double nope = 0.0, rope = 0.0;
            for (int c = 0; c < dc; c++) nope += bf16_to_f64(qn[c]) * bf16_to_f64(KV[j * dc + c]);
            for (int c = 0; c < dr; c++) rope += bf16_to_f64(qp[c]) * bf16_to_f64(Kp[j * dr + c]);
            s[j] = J->scale * (nope + rope);
        }
        softmax_weighted_sum(s, n_kv, KV, dc, dc, J->O + k * dc, J->LSE + k, NULL);
    }
    free(s);
    return NULL;
}

int oracle_mla_decode(const uint16_t *Q_nope, const uint16_t *Q_pe, const uint16_t *KV_latent,
                      const uint16_t *K_pe, double *O, double *LSE, int B, int H, int N_kv, int d_c,
                      int d_r, double scale, const int64_t *rows, int64_t n_rows, int n_threads)
{
    if (B < 0 || H <= 0 || N_kv < 0 || d_c <= 0 || d_r < 0) return -1;
    int64_t total = (int64_t)B * H;
    if (!rows) n_rows = total;
    if (n_rows == 0) return 0;
    for (int64_t k = 0; rows && k < n_rows; k++)
        if (rows[k] < 0 || rows[k] >= total) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_rows) n_threads = (int)n_rows;

    mla_job *jobs = (mla_job *)malloc(sizeof(mla_job) * n_threads);
    if (!jobs) return -1;
    for (int t = 0; t < n_threads; t++) {
        mla_job j = {Q_nope, Q_pe, KV_latent, K_pe, O, LSE, B, H, N_kv, d_c, d_r,
                     scale, rows, n_rows, n_threads, t};
        jobs[t] = j;
    }
    int rc = run_threads(mla_worker, jobs, sizeof(mla_job), n_threads);
    free(jobs);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* MLA decode over a paged KV cache with per-sequence lengths (the loop bound */
/* of the FlashMLA article's section 2.2, ceildiv(seqlen_kv, block_N), taken  */
/* per sequence).  Key j < seqlens[b] of sequence b is row j % page of page   */
/* block_table[b * max_pages + j / page] of the caches                        */
/*   KV_cache [num_pages][page][d_c],  K_pe_cache [num_pages][page][d_r];     */
/* otherwise the same definition as oracle_mla_decode.  With s_q query tokens */
/* per sequence (Q [B][s_q][H][d], O [B][s_q][H][d_c]), the tokens are the    */
/* last s_q positions of the sequence and attend causally: token t sees keys  */
/* j < seqlens[b] - (s_q - 1 - t).  A row with no key has O = 0, LSE = -inf.  */

typedef struct {
    const uint16_t *Qn, *Qp, *KV, *Kp;
    const int32_t *table, *seqlens;
    double *O, *LSE;
    int B, s_q, H, max_pages, page, d_c, d_r;
    double scale;
    const int64_t *rows;   /* flat b*H + h, or NULL */
    int64_t n_rows;
    int n_threads, tid;
} mla_paged_job;

static void *mla_paged_worker(void *arg)
{
    const mla_paged_job *J = (const mla_paged_job *)arg;
    const int dc = J->d_c, dr = J->d_r;
    const long cap = (long)J->max_pages * J->page;
    double *s = (double *)malloc(sizeof(double) * (cap > 0 ? cap : 1));
    uint16_t *kv = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(cap > 0 ? cap : 1) * dc);
    uint16_t *kp = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(cap > 0 ? cap : 1) * dr);
    if (!s || !kv || !kp) {
        free(s);
        free(kv);
        free(kp);
        return (void *)1;
    }
    for (int64_t k = J->tid; k < J->n_rows; k += J->n_threads) {
        int64_t flat = J->rows ? J->rows[k] : k;   /* (b * s_q + t) * H + h */
        long bt = (long)(flat / J->H), h = (long)(flat % J->H);
        long b = bt / J->s_q, tok = bt % J->s_q;
        long n = (long)J->seqlens[b] - (J->s_q - 1 - tok);
        if (n < 0) n = 0;
        /* gather this sequence's key rows in order */
        for (long j = 0; j < n; j++) {
            const long pg = J->table[b * J->max_pages + j / J->page];
            const long r = pg * J->page + j % J->page;
            memcpy(kv + j * dc, J->KV + r * dc, sizeof(uint16_t) * dc);
            memcpy(kp + j * dr, J->Kp + r * dr, sizeof(uint16_t) * dr);
        }
        const uint16_t *qn = J->Qn + (bt * J->H + h) * dc;
        const uint16_t *qp = J->Qp + (bt * J->H + h) * dr;
        for (long j = 0; j < n; j++) {
            double nope = 0.0, rope = 0.0;
            for (int c = 0; c < dc; c++) nope += bf16_to_f64(qn[c]) * bf16_to_f64(kv[j * dc + c]);
            for (int c = 0; c < dr; c++) rope += bf16_to_f64(qp[c]) * bf16_to_f64(kp[j * dr + c]);
            s[j] = J->scale * (nope + rope);
        }
        softmax_weighted_sum(s, n, kv, dc, dc, J->O + k * dc, J->LSE + k, NULL);
    }
    free(s);
    free(kv);
    free(kp);
    return NULL;
}

int oracle_mla_decode_paged(const uint16_t *Q_nope, const uint16_t *Q_pe, const uint16_t *KV_cache,
                            const uint16_t *K_pe_cache, const int32_t *block_table, const int32_t *seqlens,
                            double *O, double *LSE, int B, int s_q, int H, int num_pages, int max_pages, int page,
                            int d_c, int d_r, double scale, const int64_t *rows, int64_t n_rows, int n_threads)
{
    if (B < 0 || s_q < 1 || H <= 0 || num_pages < 0 || max_pages < 0 || page <= 0 || d_c <= 0 || d_r < 0)
        return -1;
    for (int b = 0; b < B; b++) {
        if (seqlens[b] < 0 || (long)seqlens[b] > (long)max_pages * page) return -1;
        for (long j = 0; j < seqlens[b]; j += page) {
            const int32_t pg = block_table[(long)b * max_pages + j / page];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    int64_t total = (int64_t)B * s_q * H;
    if (!rows) n_rows = total;
    if (n_rows == 0) return 0;
    for (int64_t k = 0; rows && k < n_rows; k++)
        if (rows[k] < 0 || rows[k] >= total) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_rows) n_threads = (int)n_rows;

    mla_paged_job *jobs = (mla_paged_job *)malloc(sizeof(mla_paged_job) * n_threads);
    if (!jobs) return -1;
    for (int t = 0; t < n_threads; t++) {
        mla_paged_job j = {Q_nope, Q_pe, KV_cache, K_pe_cache, block_table, seqlens, O, LSE, B, s_q, H,
                           max_pages, page, d_c, d_r, scale, rows, n_rows, n_threads, t};
        jobs[t] = j;
    }
    int rc = run_threads(mla_paged_worker, jobs, sizeof(mla_paged_job), n_threads);
    free(jobs);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Mamba-2 SSD scan (the chunk-state / chunk-scan linear-attention functions */
/* named in "TileLang: 面向AI系统的可组合分块编程模型" (results, linear        */
/* attention on H100), with the selective-scan recurrence sketched in        */
/* "从FlashAttention到通用内核" section 4), written as the plain recurrence:  */
/* per batch b and head h (group g = h / (H / G)), with state S [P][N]:      */
/*   S_t = exp(dt_t * A_h) * S_{t-1} + dt_t * x_t (outer) B_t                */
/*   y_t = S_t . C_t  (+ D_h * x_t)                                          */
/* x [B][L][H][P] bf16, dt [B][L][H] fp32, A [H] fp32, B_, C_ [B][L][G][N]   */
/* bf16, D [H] fp32 or NULL; y [B][L][H][P] and the final state             */
/* [B][H][P][N] (may be NULL) in fp64.                                       */

static double f32_to_f64(float f) { return (double)f; }

typedef struct {
    const uint16_t *x, *Bm, *Cm;
    const float *dt, *A, *D;
    double *y, *S_out;
    int Bsz, L, H, P, G, N;
    int n_threads, tid;
} ssd_job;

static void *ssd_worker(void *arg)
{
    const ssd_job *J = (const ssd_job *)arg;
    const int P = J->P, N = J->N, H = J->H, G = J->G, L = J->L;
    double *S = (double *)malloc(sizeof(double) * (size_t)P * N);
    if (!S) return (void *)1;
    for (long bh = J->tid; bh < (long)J->Bsz * H; bh += J->n_threads) {
        const long b = bh / H, h = bh % H, g = h / (H / G);
        for (long i = 0; i < (long)P * N; i++) S[i] = 0.0;
        for (long t = 0; t < L; t++) {
            const double dt = f32_to_f64(J->dt[(b * L + t) * H + h]);
            const double decay = exp(dt * f32_to_f64(J->A[h]));
            const uint16_t *xt = J->x + ((b * L + t) * H + h) * P;
            const uint16_t *Bt = J->Bm + ((b * L + t) * G + g) * N;
            const uint16_t *Ct = J->Cm + ((b * L + t) * G + g) * N;
            double *yt = J->y + ((b * L + t) * H + h) * P;
            for (int p = 0; p < P; p++) {
                const double xp = bf16_to_f64(xt[p]);
                double acc = 0.0;
                for (int n = 0; n < N; n++) {
                    double *s = S + (long)p * N + n;
                    *s = decay * *s + dt * xp * bf16_to_f64(Bt[n]);
                    acc += *s * bf16_to_f64(Ct[n]);
                }
                yt[p] = acc + (J->D ? f32_to_f64(J->D[h]) * xp : 0.0);
            }
        }
        if (J->S_out) memcpy(J->S_out + bh * (long)P * N, S, sizeof(double) * (size_t)P * N);
    }
    free(S);
    return NULL;
}

int oracle_ssd_scan(const uint16_t *x, const float *dt, const float *A, const uint16_t *Bm, const uint16_t *Cm,
                    const float *D, double *y, double *S_out, int Bsz, int L, int H, int P, int G, int N,
                    int n_threads)
{
    if (Bsz < 0 || L < 0 || H <= 0 || P <= 0 || G <= 0 || N <= 0 || H % G) return -1;
    const long total = (long)Bsz * H;
    if (total == 0) return 0;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > total) n_threads = (int)total;
    ssd_job *jobs = (ssd_job *)malloc(sizeof(ssd_job) * n_threads);
    if (!jobs) return -1;
    for (int t = 0; t < n_threads; t++) {
        ssd_job j = {x, Bm, Cm, dt, A, D, y, S_out, Bsz, L, H, P, G, N, n_threads, t};
        jobs[t] = j;
    }
    int rc = run_threads(ssd_worker, jobs, sizeof(ssd_job), n_threads);
    free(jobs);
    return rc;
}
