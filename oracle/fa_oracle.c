/*
 * fa_oracle.c — plain, slow, obviously correct CPU oracle for the non-causal
 * scaled-dot-product attention forward with row log-sum-exp.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline /
 * reference arm do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes (the plain definition, in fp64 throughout):
 *
 *   s_ij   = scale * sum_d q[b,h,i,d] * k[b,h,j,d]   (+ mask[b,j] if a mask is given)
 *   m_i    = max_j s_ij
 *   l_i    = sum_j exp(s_ij - m_i)
 *   O[i,:] = sum_j exp(s_ij - m_i) * v[b,h,j,:] / l_i
 *   LSE_i  = m_i + ln(l_i)
 *
 * Sources, by page and section:
 *  - "算子加速：注意力、编译与融合" (anrans.github.io ai-infra-handbooks, perf/kernels),
 *    section "注意力：从O(N²)显存到分块", worked example function `naive`:
 *    scores = q k^T / sqrt(D), softmax over the key axis, times v.
 *  - "FlashAttention原理与工业实战" (sheratonhq.com), §2.1: a mask entry of
 *    "ignore" becomes -inf before the softmax.
 *  - "Step 3.7 Flash" SD1.5 case study (pwwt.cn), §2.3: the scores are scaled
 *    first and the additive mask is added after the scale (large negative for
 *    ignored positions).
 *  - "FlashAttention原理与工业实战" §2.3 kernel signature: the forward also
 *    writes a per-row Lse; its base is not stated, the natural log is used.
 *
 * General masking (fa_oracle_fwd_ex): an additive mask per (query, key) pair,
 * [B, 1 or H, Nq, Nk], added after the scale like the key-padding mask; a
 * boolean mask (keep where nonzero) is the additive mask 0 / -inf, as in
 * "FlashAttention原理与工业实战" §2.1; causal excludes key j > query i (the
 * lower-triangular mask of that page's §4.3 causal example, top-left aligned).
 *
 * Readings where the pages are silent:
 *  - the mask is an additive fp32 key-padding mask of shape [B, Nk], broadcast
 *    over heads and query rows; it is not multiplied by `scale`;
 *  - a row whose every score is -inf (all keys masked) gives O = 0 and
 *    LSE = -inf;
 *  - the softmax is two-pass over a materialised fp64 score row (max, then
 *    exp/sum), which is exactly the textbook definition.
 *
 * Inputs are fp32 or raw bf16 bit patterns (uint16), widened exactly to fp64.
 * Layout: q [B,H,Nq,D], k and v [B,H,Nk,D], contiguous row-major.
 * Outputs are fp64: O [B,H,Nq,D] (or [B,H,nrows,D] in sampled mode), LSE
 * [B,H,Nq] (or [B,H,nrows]).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_F32 0
#define ORACLE_DTYPE_BF16 1

/* Widen one input element to fp64.  bf16 is the upper half of an fp32. */
static double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORACLE_DTYPE_BF16) {
        uint16_t bits = ((const uint16_t*)base)[idx];
        uint32_t wide = ((uint32_t)bits) << 16;
        float f;
        memcpy(&f, &wide, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const float* mask; /* [B, Nk] or NULL */
    const float* full_mask; /* [B, mask_heads, Nq, Nk] additive, or NULL */
    int mask_heads;         /* 1 (broadcast over heads) or H */
    int causal;             /* key j > query i is excluded */
    int win;                /* window attention: tokens are an img_h x img_w grid */
    int img_h, img_w, win_h, win_w, shift_h, shift_w;
    int dtype;
    int B, H, Nq, Nk, D;
    double scale;
    const int64_t* rows; /* NULL: every row; else [B*H, nrows] query indices */
    int nrows;
    double* out;
    double* lse;
    int64_t total_items;          /* number of (head, row) items */
    int64_t next_item;            /* shared work counter */
} oracle_job;

/* Window of token t (row-major on the img_h x img_w grid) after the grid is
 * rolled by (-shift_h, -shift_w), as a cyclic shift moves the token at (r, c)
 * to (r - shift_h, c - shift_w); windows are win_h x win_w tiles of that grid. */
static int64_t window_of(const oracle_job* job, int64_t t) {
    const int64_t r = t / job->img_w, c = t % job->img_w;
    const int64_t rs = ((r - job->shift_h) % job->img_h + job->img_h) % job->img_h;
    const int64_t cs = ((c - job->shift_w) % job->img_w + job->img_w) % job->img_w;
    return (rs / job->win_h) * (job->img_w / job->win_w) + cs / job->win_w;
}

/* One query row of one head: materialise the score row, then softmax, then the
 * weighted sum of V rows.  s and p are scratch buffers of length Nk.  When
 * probs_out is not NULL the row's softmax probabilities p_j / l are also
 * written there (all zeros for a fully masked row). */
static void attend_one_row(const oracle_job* job, int64_t bh, int64_t i, double* o_row,
                           double* lse_out, double* s, double* p, double* probs_out) {
    const int Nk = job->Nk, D = job->D, Nq = job->Nq;
    const int64_t b = bh / job->H;
    const int64_t q_base = (bh * Nq + i) * D;
    const int64_t kv_base = bh * (int64_t)Nk * D;

    /* s_ij = scale * (q_i . k_j) + mask_bj */
    for (int j = 0; j < Nk; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) {
            dot += load_elem(job->q, job->dtype, q_base + d) *
                   load_elem(job->k, job->dtype, kv_base + (int64_t)j * D + d);
        }
        double sij = job->scale * dot;
        if (job->mask) sij += (double)job->mask[b * Nk + j];
        if (job->full_mask) {
            const int64_t hm = job->mask_heads == 1 ? 0 : bh % job->H;
            sij += (double)job->full_mask[((b * job->mask_heads + hm) * Nq + i) * Nk + j];
        }
        if (job->causal && j > i) sij = -INFINITY;
        if (job->win && window_of(job, j) != window_of(job, i)) sij = -INFINITY;
        s[j] = sij;
    }

    /* m_i = max_j s_ij */
    double m = -INFINITY;
    for (int j = 0; j < Nk; ++j)
        if (s[j] > m) m = s[j];

    if (m == -INFINITY) { /* every key masked */
        for (int d = 0; d < D; ++d) o_row[d] = 0.0;
        *lse_out = -INFINITY;
        if (probs_out)
            for (int j = 0; j < Nk; ++j) probs_out[j] = 0.0;
        return;
    }

    /* p_ij = exp(s_ij - m_i), l_i = sum_j p_ij */
    double l = 0.0;
    for (int j = 0; j < Nk; ++j) {
        p[j] = exp(s[j] - m);
        l += p[j];
    }

    /* O_i = sum_j p_ij v_j / l_i */
    for (int d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int j = 0; j < Nk; ++j) {
        for (int d = 0; d < D; ++d)
            o_row[d] += p[j] * load_elem(job->v, job->dtype, kv_base + (int64_t)j * D + d);
    }
    for (int d = 0; d < D; ++d) o_row[d] /= l;

    *lse_out = m + log(l);
    if (probs_out)
        for (int j = 0; j < Nk; ++j) probs_out[j] = p[j] / l;
}

static void* worker(void* arg) {
    oracle_job* job = (oracle_job*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)job->Nk);
    double* p = (double*)malloc(sizeof(double) * (size_t)job->Nk);
    if (!s || !p) {
        free(s);
        free(p);
        return (void*)1;
    }
    const int64_t per_head = job->rows ? job->nrows : job->Nq;
    for (;;) {
        int64_t item = __atomic_fetch_add(&job->next_item, 1, __ATOMIC_RELAXED);
        if (item >= job->total_items) break;
        int64_t bh = item / per_head;
        int64_t r = item % per_head;
        int64_t i = job->rows ? job->rows[bh * job->nrows + r] : r;
        attend_one_row(job, bh, i, job->out + item * job->D, job->lse + item, s, p, NULL);
    }
    free(s);
    free(p);
    return NULL;
}

static int run_job(oracle_job* job, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if (job->total_items < nthreads) nthreads = (int)(job->total_items > 0 ? job->total_items : 1);
    pthread_t* tids = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!tids) return 2;
    int started = 0, failed = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, worker, job) != 0) break;
        ++started;
    }
    if (started == 0) { /* run inline */
        if (worker(job) != NULL) failed = 1;
    }
    for (int t = 0; t < started; ++t) {
        void* rv = NULL;
        pthread_join(tids[t], &rv);
        if (rv != NULL) failed = 1;
    }
    free(tids);
    return failed ? 2 : 0;
}

static int check_shape(int B, int H, int Nq, int Nk, int D) {
    return (B >= 1 && H >= 1 && Nq >= 1 && Nk >= 1 && D >= 1) ? 0 : 1;
}

/* Full forward: O [B,H,Nq,D] and LSE [B,H,Nq], both fp64.
 * Returns 0 on success, 1 on a bad shape or pointer, 2 on an allocation or
 * thread failure. */
int fa_oracle_fwd(const void* q, const void* k, const void* v, const float* mask, int dtype,
                  double* out, double* lse, int B, int H, int Nq, int Nk, int D, double scale,
                  int nthreads) {
    if (!q || !k || !v || !out || !lse || check_shape(B, H, Nq, Nk, D)) return 1;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return 1;
    oracle_job job = {q, k, v, mask, NULL, 1, 0, 0, 0, 0, 0, 0, 0, 0, dtype, B, H, Nq, Nk, D, scale,
                      NULL, 0, out, lse, (int64_t)B * H * Nq, 0};
    return run_job(&job, nthreads);
}

/* Forward with general masking: the key-padding mask [B, Nk] (or NULL), an
 * additive mask over every (query, key) pair [B, mask_heads, Nq, Nk] (or
 * NULL; mask_heads 1 broadcasts over heads), and `causal` (key j excluded
 * for query i when j > i, the top-left-aligned triangle).  `rows` NULL
 * computes every row, else the rows[B*H*nrows] query indices per head. */
int fa_oracle_fwd_ex(const void* q, const void* k, const void* v, const float* mask,
                     const float* full_mask, int mask_heads, int causal, int dtype,
                     const int64_t* rows, int nrows, double* out, double* lse, int B, int H,
                     int Nq, int Nk, int D, double scale, int nthreads) {
    if (!q || !k || !v || !out || !lse || check_shape(B, H, Nq, Nk, D)) return 1;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return 1;
    if (full_mask && mask_heads != 1 && mask_heads != H) return 1;
    if (rows) {
        if (nrows < 1) return 1;
        for (int64_t t = 0; t < (int64_t)B * H * nrows; ++t)
            if (rows[t] < 0 || rows[t] >= Nq) return 1;
    }
    oracle_job job = {q, k, v, mask, full_mask, mask_heads < 1 ? 1 : mask_heads, causal ? 1 : 0,
                      0, 0, 0, 0, 0, 0, 0, dtype, B, H, Nq, Nk, D, scale, rows, rows ? nrows : 0,
                      out, lse, (int64_t)B * H * (rows ? nrows : Nq), 0};
    return run_job(&job, nthreads);
}

/* Sampled forward: for each head bh, the query rows rows[bh*nrows + r].
 * O [B,H,nrows,D] and LSE [B,H,nrows], fp64. */
int fa_oracle_rows(const void* q, const void* k, const void* v, const float* mask, int dtype,
                   const int64_t* rows, int nrows, double* out, double* lse, int B, int H, int Nq,
                   int Nk, int D, double scale, int nthreads) {
    if (!q || !k || !v || !out || !lse || !rows || nrows < 1 || check_shape(B, H, Nq, Nk, D))
        return 1;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return 1;
    for (int64_t t = 0; t < (int64_t)B * H * nrows; ++t)
        if (rows[t] < 0 || rows[t] >= Nq) return 1;
    oracle_job job = {q, k, v, mask, NULL, 1, 0, 0, 0, 0, 0, 0, 0, 0, dtype, B, H, Nq, Nk, D, scale,
                      rows, nrows, out, lse, (int64_t)B * H * nrows, 0};
    return run_job(&job, nthreads);
}

/* Window attention on an img_h x img_w token grid (N = img_h * img_w tokens,
 * q, k, v [B, H, N, D] in row-major token order): the grid is cyclically
 * shifted by (-shift_h, -shift_w), cut into win_h x win_w windows, and each
 * token attends only to the tokens of its own window (the "Step 3.7 Flash"
 * §2.1 / §3.2 window and shifted-window attention, read as a cyclic shift
 * with no further mask).  O [B, H, N, D], LSE [B, H, N] in the original
 * token order.  img_h % win_h == 0 and img_w % win_w == 0 are required. */
int fa_oracle_window(const void* q, const void* k, const void* v, int dtype, int img_h, int img_w,
                     int win_h, int win_w, int shift_h, int shift_w, double* out, double* lse,
                     int B, int H, int D, double scale, int nthreads) {
    if (img_h < 1 || img_w < 1 || win_h < 1 || win_w < 1) return 1;
    if (img_h % win_h || img_w % win_w) return 1;
    const int N = img_h * img_w;
    if (!q || !k || !v || !out || !lse || check_shape(B, H, N, N, D)) return 1;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return 1;
    oracle_job job = {q, k, v, NULL, NULL, 1, 0, 1, img_h, img_w, win_h, win_w, shift_h, shift_w,
                      dtype, B, H, N, N, D, scale, NULL, 0, out, lse, (int64_t)B * H * N, 0};
    return run_job(&job, nthreads);
}

/* One row (b, h, i) of the forward through the same function every other
 * entry point uses (attend_one_row), also returning that row's softmax
 * probabilities p_j = exp(s_ij - m_i) / l_i in probs[Nk] (all zeros for a
 * fully masked row), its O row in o_row[D] and its LSE.  Used to check that
 * each row of the attention matrix is a probability distribution and that
 * O_i = sum_j p_j v_j. */
int fa_oracle_probs(const void* q, const void* k, const void* v, const float* mask, int dtype,
                    int b, int h, int i, double* probs, double* o_row, double* lse, int B, int H,
                    int Nq, int Nk, int D, double scale) {
    if (!q || !k || !v || !probs || !o_row || !lse || check_shape(B, H, Nq, Nk, D)) return 1;
    if (dtype != ORACLE_DTYPE_F32 && dtype != ORACLE_DTYPE_BF16) return 1;
    if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Nq) return 1;
    oracle_job job = {q, k, v, mask, NULL, 1, 0, 0, 0, 0, 0, 0, 0, 0, dtype, B, H, Nq, Nk, D, scale,
                      NULL, 0, NULL, NULL, 1, 0};
    double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
    double* p = (double*)malloc(sizeof(double) * (size_t)Nk);
    if (!s || !p) {
        free(s);
        free(p);
        return 2;
    }
    attend_one_row(&job, (int64_t)b * H + h, i, o_row, lse, s, p, probs);
    free(s);
    free(p);
    return 0;
}
