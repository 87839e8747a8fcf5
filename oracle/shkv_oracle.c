/*
 * shkv_oracle.c -- plain, slow fp64 CPU oracle for shared-KV multi-decoder
 * paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and
 * the benchmark's CPU-baseline leg may load this file's library.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * What it computes (each function cites the passage it follows):
 *
 *  - ICaRus, key design 2: every task model's logical encoder is the frozen
 *    base encoder, so all N decoders see one bitwise-identical KV cache; one
 *    block table serves every model.
 *  - ICaRus, key design 3: the decoders' queries are concatenated along the
 *    head axis and attend the same KV.  The result for each query row is
 *    ordinary softmax attention; concatenation only changes how often the
 *    cache is read, never the value.
 *  - PrefillShare, Sec. 3.3 and Sec. 7: the cache lives in vLLM-style
 *    PagedAttention blocks (pages); a returning session runs a partial
 *    prefill on its new tokens only and extends the cached prefix.
 *
 * Readings where the pages are silent (the same readings the library uses):
 *  - q head h of a decoder uses KV head g = h / (Hq / Hkv) (contiguous GQA);
 *  - stacked rows are model-major: row r = m * Hq + h;
 *  - decode attends every cached token t < L_b (no causal mask);
 *  - scores are scale * <q, k>; the caller passes scale (1/sqrt(d) in all
 *    configured workloads);
 *  - lse is the natural-log log-sum-exp of the scaled scores.
 *
 * Every value is widened exactly from bf16 and all arithmetic is fp64.  The
 * softmax is the two-pass definition (max, then normalised exponentials),
 * not an online recurrence.
 */
#include <limits.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EARG 1
#define ORACLE_EPAGE 2
#define ORACLE_ENOMEM 3

static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* KV head of q head h (contiguous GQA); stacked row of decoder m, q head h
 * (model-major); token slot t of (page, KV head g) in a [pages, Hkv, P, D]
 * pool. */
static int kv_head(int Hq, int Hkv, int h) { return h / (Hq / Hkv); }
static long stacked_row(int N, int Hq, int m, int h)
{
    (void)N;
    return (long)m * Hq + h;
}
static const uint16_t *page_slot(const uint16_t *pool, int Hkv, int P, int D, int32_t page, int g, int t)
{
    return pool + (((long)page * Hkv + g) * P + t % P) * (long)D;
}

/*
 * Softmax attention of one query row over n tokens given by their K and V
 * rows (the definition, two-pass, fp64):
 *   s_i = scale * <q, K_i>,  p_i = exp(s_i - max s) / sum_j exp(s_j - max s),
 *   o = sum_i p_i V_i,       lse = max s + ln sum_i exp(s_i - max s).
 * n = 0 gives o = 0 and lse = -inf.  s is scratch of n doubles.
 */
static void softmax_attend(const uint16_t *q, int D, double scale, int n, const uint16_t *const *kt,
                           const uint16_t *const *vt, double *s, double *o, double *lse)
{
    for (int k = 0; k < D; ++k)
        o[k] = 0.0;
    if (n <= 0) {
        if (lse)
            *lse = -INFINITY;
        return;
    }
    double smax = -INFINITY;
    for (int i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int k = 0; k < D; ++k)
            acc += widen_bf16(q[k]) * widen_bf16(kt[i][k]);
        s[i] = scale * acc;
        if (s[i] > smax)
            smax = s[i];
    }
    double denom = 0.0;
    for (int i = 0; i < n; ++i)
        denom += exp(s[i] - smax);
    for (int i = 0; i < n; ++i) {
        double p = exp(s[i] - smax) / denom;
        for (int k = 0; k < D; ++k)
            o[k] += p * widen_bf16(vt[i][k]);
    }
    if (lse)
        *lse = smax + log(denom);
}

/* per-thread scratch: scores and the token list of one row */
typedef struct {
    double *s;
    const uint16_t **kt, **vt;
} row_scratch;

static int scratch_alloc(row_scratch *sc, int max_len)
{
    size_t n = (size_t)(max_len > 0 ? max_len : 1);
    sc->s = (double *)malloc(sizeof(double) * n);
    sc->kt = (const uint16_t **)malloc(sizeof(uint16_t *) * n);
    sc->vt = (const uint16_t **)malloc(sizeof(uint16_t *) * n);
    return sc->s && sc->kt && sc->vt;
}

static void scratch_free(row_scratch *sc)
{
    free(sc->s);
    free(sc->kt);
    free(sc->vt);
}

typedef struct {
    int B, N, Hq, Hkv, D, P, num_pages, max_pages;
    const uint16_t *q, *k_pages, *v_pages;
    const int32_t *block_table, *seq_lens;
    int32_t t_begin, t_end;
    double scale;
    double *out, *lse;
    /* work distribution */
    long next_row;
    long total_rows;
    int status;
    pthread_mutex_t lock;
} decode_job;

/* Address of token t of request b, KV head g, in a [num_pages, Hkv, P, D]
 * pool, read through the block table.  Returns NULL for a bad page index. */
static const uint16_t *token_ptr(const decode_job *j, const uint16_t *pool, int b, int g, int t)
{
    int32_t page = j->block_table[(long)b * j->max_pages + t / j->P];
    if (page < 0 || page >= j->num_pages)
        return NULL;
    return page_slot(pool, j->Hkv, j->P, j->D, page, g, t);
}

/*
 * One query row: request b, decoder m, q head h.  Attention over the cached
 * tokens t in [t_begin, t_end) intersected with [0, L_b):
 *   s_t   = scale * sum_k q[k] K_t[k]
 *   p_t   = exp(s_t - max s) / sum_u exp(s_u - max s)
 *   o     = sum_t p_t V_t
 *   lse   = max s + ln sum_t exp(s_t - max s)
 * An empty token range gives o = 0 and lse = -inf.
 */
static int attend_row(const decode_job *j, int b, int m, int h, row_scratch *sc)
{
    const int g = kv_head(j->Hq, j->Hkv, h);
    const long r = stacked_row(j->N, j->Hq, m, h);
    const long rows = (long)j->N * j->Hq;
    const uint16_t *q = j->q + ((long)b * rows + r) * j->D;
    double *o = j->out + ((long)b * rows + r) * j->D;
    double *lse = j->lse ? j->lse + (long)b * rows + r : NULL;

    int L = j->seq_lens[b];
    int t0 = j->t_begin < 0 ? 0 : j->t_begin;
    int t1 = j->t_end < L ? j->t_end : L;
    int n = t1 > t0 ? t1 - t0 : 0;
    for (int i = 0; i < n; ++i) {
        sc->kt[i] = token_ptr(j, j->k_pages, b, g, t0 + i);
        sc->vt[i] = token_ptr(j, j->v_pages, b, g, t0 + i);
        if (!sc->kt[i] || !sc->vt[i])
            return ORACLE_EPAGE;
    }
    softmax_attend(q, j->D, j->scale, n, sc->kt, sc->vt, sc->s, o, lse);
    return ORACLE_OK;
}

static void *decode_worker(void *arg)
{
    decode_job *j = (decode_job *)arg;
    int max_len = 0;
    for (int b = 0; b < j->B; ++b)
        if (j->seq_lens[b] > max_len)
            max_len = j->seq_lens[b];
    row_scratch sc;
    if (!scratch_alloc(&sc, max_len)) {
        scratch_free(&sc);
        pthread_mutex_lock(&j->lock);
        j->status = ORACLE_ENOMEM;
        pthread_mutex_unlock(&j->lock);
        return NULL;
    }
    const long rows = (long)j->N * j->Hq;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        long idx = j->next_row++;
        int stop = j->status != ORACLE_OK;
        pthread_mutex_unlock(&j->lock);
        if (stop || idx >= j->total_rows)
            break;
        int b = (int)(idx / rows);
        int r = (int)(idx % rows);
        int st = attend_row(j, b, r / j->Hq, r % j->Hq, &sc);
        if (st != ORACLE_OK) {
            pthread_mutex_lock(&j->lock);
            j->status = st;
            pthread_mutex_unlock(&j->lock);
        }
    }
    scratch_free(&sc);
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0)
        return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Decode attention of N stacked decoders over one shared paged cache
 * (ICaRus key designs 2-3; PrefillShare Sec. 3.3 paged blocks).
 *
 *   q           bf16 bits [B, N*Hq, D], model-major rows
 *   k/v_pages   bf16 bits [num_pages, Hkv, P, D]
 *   block_table int32 [B, max_pages]; seq_lens int32 [B]
 *   t_begin/end token window applied to every request (use 0 and INT_MAX
 *               for full attention; a window gives a split partial)
 *   out         fp64 [B, N*Hq, D];  lse fp64 [B, N*Hq] (nullable)
 *   nthreads    worker threads (<= 0: all online cores)
 * Returns 0, or ORACLE_EARG / ORACLE_EPAGE (page index outside the pool) /
 * ORACLE_ENOMEM.
 */
int oracle_decode_attention(int B, int N, int Hq, int Hkv, int D, int P, int num_pages,
                            int max_pages, const uint16_t *q, const uint16_t *k_pages,
                            const uint16_t *v_pages, const int32_t *block_table,
                            const int32_t *seq_lens, int32_t t_begin, int32_t t_end,
                            double scale, double *out, double *lse, int nthreads)
{
    if (B < 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || P <= 0 || !out)
        return ORACLE_EARG;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > (long)max_pages * P)
            return ORACLE_EARG;
    decode_job j;
    memset(&j, 0, sizeof j);
    j.B = B; j.N = N; j.Hq = Hq; j.Hkv = Hkv; j.D = D; j.P = P;
    j.num_pages = num_pages; j.max_pages = max_pages;
    j.q = q; j.k_pages = k_pages; j.v_pages = v_pages;
    j.block_table = block_table; j.seq_lens = seq_lens;
    j.t_begin = t_begin; j.t_end = t_end; j.scale = scale;
    j.out = out; j.lse = lse;
    j.total_rows = (long)B * N * Hq;
    j.status = ORACLE_OK;
    pthread_mutex_init(&j.lock, NULL);

    int nt = resolve_threads(nthreads);
    if (nt > j.total_rows)
        nt = j.total_rows > 0 ? (int)j.total_rows : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th)
        return ORACLE_ENOMEM;
    for (int i = 0; i < nt; ++i)
        pthread_create(&th[i], NULL, decode_worker, &j);
    for (int i = 0; i < nt; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.lock);
    return j.status;
}

/*
 * Per-decoder unique tails (PrefillShare Sec. 3.3 and Sec. 4, Eqs. 8-9): a
 * decoder starts from the shared base cache C_base and extends it with its
 * own generated-token cache Delta C_t, so decoder m of request b attends the
 * concatenation [shared prefix tokens 0 .. L_b) ++ [its tail tokens
 * 0 .. T_{b,m}).  The shared prefix is stored once (L_shared); each decoder's
 * tail is its own (N * L_unique).  Both live in the same page pool:
 *
 *   block_table      int32 [B, max_pages], seq_lens int32 [B]       (shared)
 *   tail_table       int32 [B, N, max_tail_pages], tail_lens int32 [B, N]
 *   out fp64 [B, N*Hq, D], lse fp64 [B, N*Hq] (nullable)
 *
 * Same definition as oracle_decode_attention over the concatenated token
 * list: two-pass softmax in fp64.  An empty concatenation gives o = 0 and
 * lse = -inf.
 */
typedef struct {
    int B, N, Hq, Hkv, D, P, num_pages, max_pages, max_tail_pages;
    const uint16_t *q, *k_pages, *v_pages;
    const int32_t *block_table, *seq_lens, *tail_table, *tail_lens;
    double scale;
    double *out, *lse;
    long next_row, total_rows;
    int status;
    pthread_mutex_t lock;
} tails_job;

/* token i of the concatenation for (b, m), KV head g; NULL for a bad page */
static const uint16_t *concat_token(const tails_job *j, const uint16_t *pool, int b, int m, int g, int i)
{
    int L = j->seq_lens[b];
    int32_t page;
    int t;
    if (i < L) {
        t = i;
        page = j->block_table[(long)b * j->max_pages + t / j->P];
    } else {
        t = i - L;
        page = j->tail_table[((long)b * j->N + m) * j->max_tail_pages + t / j->P];
    }
    if (page < 0 || page >= j->num_pages)
        return NULL;
    return page_slot(pool, j->Hkv, j->P, j->D, page, g, t);
}

static int attend_row_tails(const tails_job *j, int b, int m, int h, row_scratch *sc)
{
    const int g = kv_head(j->Hq, j->Hkv, h);
    const long r = stacked_row(j->N, j->Hq, m, h);
    const long rows = (long)j->N * j->Hq;
    const uint16_t *q = j->q + ((long)b * rows + r) * j->D;
    double *o = j->out + ((long)b * rows + r) * j->D;
    double *lse = j->lse ? j->lse + (long)b * rows + r : NULL;
    const int n = j->seq_lens[b] + j->tail_lens[(long)b * j->N + m];
    for (int i = 0; i < n; ++i) {
        sc->kt[i] = concat_token(j, j->k_pages, b, m, g, i);
        sc->vt[i] = concat_token(j, j->v_pages, b, m, g, i);
        if (!sc->kt[i] || !sc->vt[i])
            return ORACLE_EPAGE;
    }
    softmax_attend(q, j->D, j->scale, n, sc->kt, sc->vt, sc->s, o, lse);
    return ORACLE_OK;
}

static void *tails_worker(void *arg)
{
    tails_job *j = (tails_job *)arg;
    int max_len = 1;
    for (int b = 0; b < j->B; ++b)
        for (int m = 0; m < j->N; ++m) {
            int n = j->seq_lens[b] + j->tail_lens[(long)b * j->N + m];
            if (n > max_len)
                max_len = n;
        }
    row_scratch sc;
    if (!scratch_alloc(&sc, max_len)) {
        scratch_free(&sc);
        pthread_mutex_lock(&j->lock);
        j->status = ORACLE_ENOMEM;
        pthread_mutex_unlock(&j->lock);
        return NULL;
    }
    const long rows = (long)j->N * j->Hq;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        long idx = j->next_row++;
        int stop = j->status != ORACLE_OK;
        pthread_mutex_unlock(&j->lock);
        if (stop || idx >= j->total_rows)
            break;
        int b = (int)(idx / rows);
        int r = (int)(idx % rows);
        int st = attend_row_tails(j, b, r / j->Hq, r % j->Hq, &sc);
        if (st != ORACLE_OK) {
            pthread_mutex_lock(&j->lock);
            j->status = st;
            pthread_mutex_unlock(&j->lock);
        }
    }
    scratch_free(&sc);
    return NULL;
}

int oracle_decode_attention_tails(int B, int N, int Hq, int Hkv, int D, int P, int num_pages,
                                  int max_pages, int max_tail_pages, const uint16_t *q,
                                  const uint16_t *k_pages, const uint16_t *v_pages,
                                  const int32_t *block_table, const int32_t *seq_lens,
                                  const int32_t *tail_table, const int32_t *tail_lens, double scale,
                                  double *out, double *lse, int nthreads)
{
    if (B < 0 || N <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || P <= 0 || !out)
        return ORACLE_EARG;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0 || seq_lens[b] > (long)max_pages * P)
            return ORACLE_EARG;
        for (int m = 0; m < N; ++m) {
            int T = tail_lens[(long)b * N + m];
            if (T < 0 || T > (long)max_tail_pages * P)
                return ORACLE_EARG;
        }
    }
    tails_job j;
    memset(&j, 0, sizeof j);
    j.B = B; j.N = N; j.Hq = Hq; j.Hkv = Hkv; j.D = D; j.P = P;
    j.num_pages = num_pages; j.max_pages = max_pages; j.max_tail_pages = max_tail_pages;
    j.q = q; j.k_pages = k_pages; j.v_pages = v_pages;
    j.block_table = block_table; j.seq_lens = seq_lens;
    j.tail_table = tail_table; j.tail_lens = tail_lens;
    j.scale = scale; j.out = out; j.lse = lse;
    j.total_rows = (long)B * N * Hq;
    j.status = ORACLE_OK;
    pthread_mutex_init(&j.lock, NULL);
    int nt = resolve_threads(nthreads);
    if (nt > j.total_rows)
        nt = j.total_rows > 0 ? (int)j.total_rows : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th)
        return ORACLE_ENOMEM;
    for (int i = 0; i < nt; ++i)
        pthread_create(&th[i], NULL, tails_worker, &j);
    for (int i = 0; i < nt; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.lock);
    return j.status;
}

/*
 * Partial-prefill attention (PrefillShare Sec. 3.3: on a prefix-cache hit the
 * shared prefill module runs only on the new tokens, extending the cached
 * prefix).  The caller has appended the n_new tokens' K/V, so request b holds
 * L_b = seq_lens[b] tokens of which the last n_new are new; new token i sits
 * at position L_b - n_new + i and attends every key at a position <= its own
 * (the whole cached prefix, and the new tokens causally).
 *
 *   q      bf16 bits [B, n_new, Hq, D]     (the prefill module's query heads)
 *   out    fp64 [B, n_new, Hq, D];  lse fp64 [B, n_new, Hq] (nullable)
 *
 * Same two-pass fp64 softmax as the decode oracle, over keys 0 .. position.
 */
typedef struct {
    int B, n_new, Hq, Hkv, D, P, num_pages, max_pages;
    const uint16_t *q, *k_pages, *v_pages;
    const int32_t *block_table, *seq_lens;
    double scale;
    double *out, *lse;
    long next_row, total_rows;
    int status;
    pthread_mutex_t lock;
} prefill_job;

static int attend_prefill_row(const prefill_job *j, int b, int i, int h, row_scratch *sc)
{
    const int g = kv_head(j->Hq, j->Hkv, h);
    const long row = ((long)b * j->n_new + i) * j->Hq + h;
    const uint16_t *q = j->q + row * j->D;
    double *o = j->out + row * j->D;
    double *lse = j->lse ? j->lse + row : NULL;
    const int L = j->seq_lens[b];
    const int n = L - j->n_new + i + 1;                /* keys 0 .. own position */
    for (int t = 0; t < n; ++t) {
        int32_t page = j->block_table[(long)b * j->max_pages + t / j->P];
        if (page < 0 || page >= j->num_pages)
            return ORACLE_EPAGE;
        sc->kt[t] = page_slot(j->k_pages, j->Hkv, j->P, j->D, page, g, t);
        sc->vt[t] = page_slot(j->v_pages, j->Hkv, j->P, j->D, page, g, t);
    }
    softmax_attend(q, j->D, j->scale, n, sc->kt, sc->vt, sc->s, o, lse);
    return ORACLE_OK;
}

static void *prefill_worker(void *arg)
{
    prefill_job *j = (prefill_job *)arg;
    int max_len = 1;
    for (int b = 0; b < j->B; ++b)
        if (j->seq_lens[b] > max_len)
            max_len = j->seq_lens[b];
    row_scratch sc;
    if (!scratch_alloc(&sc, max_len)) {
        scratch_free(&sc);
        pthread_mutex_lock(&j->lock);
        j->status = ORACLE_ENOMEM;
        pthread_mutex_unlock(&j->lock);
        return NULL;
    }
    const long per_b = (long)j->n_new * j->Hq;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        long idx = j->next_row++;
        int stop = j->status != ORACLE_OK;
        pthread_mutex_unlock(&j->lock);
        if (stop || idx >= j->total_rows)
            break;
        int b = (int)(idx / per_b);
        long rem = idx % per_b;
        int st = attend_prefill_row(j, b, (int)(rem / j->Hq), (int)(rem % j->Hq), &sc);
        if (st != ORACLE_OK) {
            pthread_mutex_lock(&j->lock);
            j->status = st;
            pthread_mutex_unlock(&j->lock);
        }
    }
    scratch_free(&sc);
    return NULL;
}

int oracle_prefill_attention(int B, int n_new, int Hq, int Hkv, int D, int P, int num_pages, int max_pages,
                             const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                             const int32_t *block_table, const int32_t *seq_lens, double scale, double *out,
                             double *lse, int nthreads)
{
    if (B < 0 || n_new < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || P <= 0 || !out)
        return ORACLE_EARG;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < n_new || seq_lens[b] > (long)max_pages * P)
            return ORACLE_EARG;
    prefill_job j;
    memset(&j, 0, sizeof j);
    j.B = B; j.n_new = n_new; j.Hq = Hq; j.Hkv = Hkv; j.D = D; j.P = P;
    j.num_pages = num_pages; j.max_pages = max_pages;
    j.q = q; j.k_pages = k_pages; j.v_pages = v_pages;
    j.block_table = block_table; j.seq_lens = seq_lens;
    j.scale = scale; j.out = out; j.lse = lse;
    j.total_rows = (long)B * n_new * Hq;
    j.status = ORACLE_OK;
    pthread_mutex_init(&j.lock, NULL);
    int nt = resolve_threads(nthreads);
    if (nt > j.total_rows)
        nt = j.total_rows > 0 ? (int)j.total_rows : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!th)
        return ORACLE_ENOMEM;
    for (int i = 0; i < nt; ++i)
        pthread_create(&th[i], NULL, prefill_worker, &j);
    for (int i = 0; i < nt; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&j.lock);
    return j.status;
}

/*
 * Log-sum-exp merge of S partial attentions over disjoint token ranges of
 * the same rows (the split-KV reduction named for long contexts):
 *   M   = max_s lse_s
 *   w_s = exp(lse_s - M)
 *   out = sum_s w_s o_s / sum_s w_s,   lse = M + ln sum_s w_s
 * Partials with lse = -inf carry no weight; if all are -inf the row is
 * out = 0, lse = -inf.
 *   o_part fp64 [S, B, rows, D], lse_part fp64 [S, B, rows]
 *   out fp64 [B, rows, D], lse_out fp64 [B, rows] (nullable)
 */
int oracle_splitkv_merge(int S, int B, int rows, int D, const double *o_part,
                         const double *lse_part, double *out, double *lse_out)
{
    if (S <= 0 || B < 0 || rows < 0 || D <= 0)
        return ORACLE_EARG;
    const long R = (long)B * rows;
    for (long i = 0; i < R; ++i) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (lse_part[s * R + i] > M)
                M = lse_part[s * R + i];
        double *o = out + i * D;
        for (int k = 0; k < D; ++k)
            o[k] = 0.0;
        if (M == -INFINITY) {
            if (lse_out)
                lse_out[i] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int s = 0; s < S; ++s) {
            double l = lse_part[s * R + i];
            if (l == -INFINITY)
                continue;
            double w = exp(l - M);
            wsum += w;
            const double *os = o_part + (s * R + i) * D;
            for (int k = 0; k < D; ++k)
                o[k] += w * os[k];
        }
        for (int k = 0; k < D; ++k)
            o[k] /= wsum;
        if (lse_out)
            lse_out[i] = M + log(wsum);
    }
    return ORACLE_OK;
}

/*
 * Partial-prefill append (PrefillShare Sec. 3.3: a cache hit runs prefill on
 * the new tokens only and hands the extended cache on).  Token t of request
 * b lands at logical position L_b + t:
 *   pool[bt[b][(L_b+t)/P], g, (L_b+t)%P, :] = new[b, t, g, :]
 * then L_b += T.  A pure byte copy.
 *   k_new/v_new bf16 bits [B, T, Hkv, D]
 */
int oracle_append_kv(int B, int T, int Hkv, int D, int P, int num_pages, int max_pages,
                     uint16_t *k_pages, uint16_t *v_pages, const int32_t *block_table,
                     int32_t *seq_lens, const uint16_t *k_new, const uint16_t *v_new)
{
    if (B < 0 || T < 0 || Hkv <= 0 || D <= 0 || P <= 0)
        return ORACLE_EARG;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || (long)seq_lens[b] + T > (long)max_pages * P)
            return ORACLE_EARG;
    for (int b = 0; b < B; ++b) {
        for (int t = 0; t < T; ++t) {
            long pos = (long)seq_lens[b] + t;
            int32_t page = block_table[(long)b * max_pages + pos / P];
            if (page < 0 || page >= num_pages)
                return ORACLE_EPAGE;
            for (int g = 0; g < Hkv; ++g) {
                long dst = (((long)page * Hkv + g) * P + pos % P) * (long)D;
                long src = (((long)b * T + t) * Hkv + g) * (long)D;
                memcpy(k_pages + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
                memcpy(v_pages + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
            }
        }
    }
    for (int b = 0; b < B; ++b)
        seq_lens[b] += T;
    return ORACLE_OK;
}

/*
 * Logical view of one request's cache: out[t, g, :] = pool[bt[b][t/P], g,
 * t%P, :] for t < L_b (bf16 bits, [L_b, Hkv, D]).  The block-table gather
 * every decoder performs (PrefillShare Sec. 3.3).
 */
int oracle_gather_kv(int b, int Hkv, int D, int P, int num_pages, int max_pages,
                     const uint16_t *pool, const int32_t *block_table,
                     const int32_t *seq_lens, uint16_t *out)
{
    int L = seq_lens[b];
    for (int t = 0; t < L; ++t) {
        int32_t page = block_table[(long)b * max_pages + t / P];
        if (page < 0 || page >= num_pages)
            return ORACLE_EPAGE;
        for (int g = 0; g < Hkv; ++g)
            memcpy(out + ((long)t * Hkv + g) * D,
                   pool + (((long)page * Hkv + g) * P + t % P) * (long)D,
                   sizeof(uint16_t) * (size_t)D);
    }
    return ORACLE_OK;
}

int oracle_num_threads(void) { return resolve_threads(0); }
