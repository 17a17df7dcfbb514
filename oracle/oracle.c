/*
 * oracle.c -- plain, slow, obviously correct fp64 CPU reference for exact
 * scaled dot-product attention: dense and packed (varlen) prefill with a
 * bottom-right causal mask and grouped-query heads, and paged decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * calls it, and the two share no code, header or table.
 *
 * What one output row is (the definition, written out; no tiling and no online
 * recurrence -- two plain passes over the allowed keys):
 *
 *   A_i   = { j : 0 <= j < Nk_b  and  (not causal  or  j <= i + Nk_b - Nq_b)
 *                and (left < 0 or j >= i + Nk_b - Nq_b - left)
 *                and (right < 0 or j <= i + Nk_b - Nq_b + right) }
 *   s_j   = scale * sum_c q[i,c] * k[j,c]                 for j in A_i
 *   m     = max_{j in A_i} s_j
 *   l     = sum_{j in A_i} exp(s_j - m)
 *   O_i,c = sum_{j in A_i} exp(s_j - m) * v[j,c] / l
 *   lse_i = m + ln(l)
 *   A_i empty  ->  O_i = 0 and lse_i = -inf.
 *
 * Passages followed:
 *  - the operator: softmax(Q K^T * scale) V, "Deep Dive - FlashAttention",
 *    opening section; "FlashAttention: Part 1", sections 1.2 and 3.2;
 *  - max subtraction before the exponentials: "Flash Attention: A Complete
 *    Architectural Autopsy", part 2, "The Online Softmax Recurrence" (the
 *    plain softmax formula for row i);
 *  - lse = m + log l, defined for a nonempty row: "Deep Dive - FlashAttention",
 *    section "Exact attention without an n x n workspace";
 *  - an entirely masked row returns zero: same page, section "Online softmax
 *    is what makes the tiles exact"; its lse is read as log 0 = -inf (the page
 *    defines lse only for nonempty rows; -inf is the value that leaves a
 *    log-sum-exp merge unchanged);
 *  - keep rule j <= i + Nk - Nq (bottom-right corner): same page, section
 *    "Causal 2.1 is the decode gotcha";
 *  - local window (left, right): keep i + Nk - Nq - left <= j <= i + Nk - Nq
 *    + right, a side of -1 being unbounded, intersected with the causal rule
 *    when both are given: same section, paragraph on local attention;
 *  - query head h reads K/V head h / (Hq / Hkv) (consecutive groups): same
 *    page, section "The public interface is several kernels";
 *  - packed sequences: sequence b owns tokens [cu[b], cu[b+1]), section
 *    "Paged KV is a lookup, not a cache manager";
 *  - paged keys: logical token t of sequence b sits in physical page
 *    block_table[b][t / page] at slot t % page: "FlashAttention-3 and
 *    PagedAttention", sections "Block tables and what the kernel does" and
 *    "Runnable Example: Measuring the IO Gap" (the block-table gather);
 *  - several new queries per sequence over the paged cache: query i of Nq is
 *    the position len - Nq + i and takes the bottom-right rule with Nq
 *    queries and len keys ("Deep Dive - FlashAttention", sections "Causal 2.1
 *    is the decode gotcha" and "Paged KV is a lookup, not a cache manager").
 *
 * Backward (oracle_backward), for one nonempty row i with G = dL/dO
 * ("Deep Dive - FlashAttention", section "Backward recomputes tiles on
 * purpose"; "FlashAttention: Part 1", section 3.6):
 *   P_ij  = exp(s_ij - m) / l            over the allowed keys (else 0)
 *   dV_j += P_ij G_i                     dP_ij = G_i . v_j
 *   D_i   = sum_j P_ij dP_ij             (= G_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j      dK_j += scale * dS_ij q_i
 * with the K/V gradients of a grouped head summed over its query heads.
 *
 * 8-bit inputs (oracle_quantize_fp8 / oracle_dequantize_fp8, at the end of
 * this file): per-tile E4M3 codes and fp32 scales, and the values they stand
 * for; attention on those values is the same definition on fp64 inputs
 * (oracle_prefill_rows_f64).
 *
 * Inputs are bf16 bit patterns (uint16), each widened exactly to double, or
 * doubles.
 * Threads: POSIX threads over output rows; each row is computed by one thread
 * in the order written above, so results do not depend on the thread count.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---- bf16 -> double (exact: bf16 is the top half of an IEEE binary32) ---- */
static double bf16_value(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* ---- the mask: is key j allowed for query row i of a (nq, nk) sequence? ---- */
static int key_allowed(long i, long j, long nq, long nk, int causal, long left, long right)
{
    if (j < 0 || j >= nk)
        return 0;
    if (causal && j > i + nk - nq) /* bottom-right aligned corner */
        return 0;
    if (left >= 0 && j < i + nk - nq - left) /* local window, left side */
        return 0;
    if (right >= 0 && j > i + nk - nq + right) /* local window, right side */
        return 0;
    return 1;
}

/* ---- one element of an input tensor: bf16 bits, or (f64 = 1) a double ---- */
static double elem(const void *base, int f64, long idx)
{
    return f64 ? ((const double *)base)[idx] : bf16_value(((const uint16_t *)base)[idx]);
}

/* ---- where the key/value rows of one sequence live ---- */
typedef struct {
    const void *k, *v;        /* K and V base pointers */
    int f64;                  /* element type of q, k, v: 0 bf16 bits, 1 double */
    long first_token;         /* contiguous: token row of key 0 */
    const int32_t *pages;     /* paged: this sequence's block-table row, else NULL */
    int page_size;
    int hkv, d;
} key_store;

static long token_of_key(const key_store *ks, long j)
{
    if (ks->pages) {
        long page = ks->pages[j / ks->page_size];
        return page * ks->page_size + j % ks->page_size;
    }
    return ks->first_token + j;
}

/* element index of channel 0 of key j, K/V head g */
static long key_row(const key_store *ks, long j, int g)
{
    return (token_of_key(ks, j) * ks->hkv + g) * (long)ks->d;
}

/* ---- one output row, by the definition ---- */
static void attend_row(const void *q, long q_row, const key_store *ks, int g,
                       long i, long nq, long nk, int causal, long left, long right, double scale,
                       double *s, double *out, double *lse)
{
    const int d = ks->d;
    double m = -INFINITY;
    long n_allowed = 0;

    /* pass 1: scores of the allowed keys and their maximum */
    for (long j = 0; j < nk; ++j) {
        if (!key_allowed(i, j, nq, nk, causal, left, right))
            continue;
        const long k_row = key_row(ks, j, g);
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += elem(q, ks->f64, q_row + c) * elem(ks->k, ks->f64, k_row + c);
        s[j] = scale * dot;
        if (n_allowed == 0 || s[j] > m)
            m = s[j];
        ++n_allowed;
    }

    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    if (n_allowed == 0) {
        *lse = -INFINITY;
        return;
    }

    /* pass 2: normaliser and value-weighted sum, relative to the maximum */
    double l = 0.0;
    for (long j = 0; j < nk; ++j) {
        if (!key_allowed(i, j, nq, nk, causal, left, right))
            continue;
        double w = exp(s[j] - m);
        l += w;
        const long v_row = key_row(ks, j, g);
        for (int c = 0; c < d; ++c)
            out[c] += w * elem(ks->v, ks->f64, v_row + c);
    }
    for (int c = 0; c < d; ++c)
        out[c] /= l;
    *lse = m + log(l);
}

/* ---- row jobs ---- */
typedef struct {
    /* shared inputs */
    const void *q, *k, *v;
    int f64;   /* element type of q, k, v: 0 bf16 bits, 1 double */
    int B, Hq, Hkv, Nq, Nk, d, causal, paged, page_size, max_pages;
    long win_left, win_right;
    double scale;
    const int32_t *cu_q, *cu_k, *block_table, *seq_lens;
    const int32_t *rows;   /* prefill: (b, h, i) triples; decode: (b, h) pairs */
    long n_rows;
    double *out, *lse;
    long max_keys;
    /* work distribution */
    long next;
    int status;
} job;

static void run_row(job *jb, long r, double *s)
{
    double *out = jb->out + r * (long)jb->d;
    double *lse = jb->lse + r;
    const int group = jb->Hq / jb->Hkv;
    key_store ks;
    memset(&ks, 0, sizeof ks);
    ks.k = jb->k;
    ks.v = jb->v;
    ks.f64 = jb->f64;
    ks.hkv = jb->Hkv;
    ks.d = jb->d;

    if (!jb->paged) {
        int b = jb->rows[3 * r], h = jb->rows[3 * r + 1], i = jb->rows[3 * r + 2];
        long q_first, nq, nk;
        if (jb->cu_q) {
            q_first = jb->cu_q[b];
            nq = jb->cu_q[b + 1] - jb->cu_q[b];
            ks.first_token = jb->cu_k[b];
            nk = jb->cu_k[b + 1] - jb->cu_k[b];
        } else {
            q_first = (long)b * jb->Nq;
            nq = jb->Nq;
            ks.first_token = (long)b * jb->Nk;
            nk = jb->Nk;
        }
        const long q_row = ((q_first + i) * jb->Hq + h) * (long)jb->d;
        attend_row(jb->q, q_row, &ks, h / group, i, nq, nk, jb->causal, jb->win_left, jb->win_right, jb->scale, s,
                   out, lse);
    } else if (jb->paged == 1) {
        int b = jb->rows[2 * r], h = jb->rows[2 * r + 1];
        long len = jb->seq_lens[b];
        ks.pages = jb->block_table + (long)b * jb->max_pages;
        ks.page_size = jb->page_size;
        const long q_row = ((long)b * jb->Hq + h) * (long)jb->d;
        /* one query per sequence: it is the last position, so under the
         * bottom-right rule it sees every cached key (i = 0, nq = 1). */
        attend_row(jb->q, q_row, &ks, h / group, 0, 1, len, 0, -1, -1, jb->scale, s, out, lse);
    } else {
        /* Nq queries per sequence over the paged cache: query i is position
         * len - Nq + i, so under the bottom-right rule (with causal) it sees
         * keys j <= i + len - Nq; without causal it sees all len keys. */
        int b = jb->rows[3 * r], h = jb->rows[3 * r + 1], i = jb->rows[3 * r + 2];
        long len = jb->seq_lens[b];
        ks.pages = jb->block_table + (long)b * jb->max_pages;
        ks.page_size = jb->page_size;
        const long q_row = (((long)b * jb->Nq + i) * jb->Hq + h) * (long)jb->d;
        attend_row(jb->q, q_row, &ks, h / group, i, jb->Nq, len, jb->causal, -1, -1, jb->scale, s, out, lse);
    }
}

static void *worker(void *arg)
{
    job *jb = (job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->max_keys > 0 ? jb->max_keys : 1));
    if (!s) {
        __atomic_store_n(&jb->status, -2, __ATOMIC_SEQ_CST);
        return NULL;
    }
    for (;;) {
        long r = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (r >= jb->n_rows)
            break;
        run_row(jb, r, s);
    }
    free(s);
    return NULL;
}

static int run_job(job *jb, int n_threads)
{
    if (n_threads <= 0)
        n_threads = 1;
    if (n_threads > 1024)
        n_threads = 1024;
    if ((long)n_threads > jb->n_rows)
        n_threads = jb->n_rows > 0 ? (int)jb->n_rows : 1;
    jb->next = 0;
    jb->status = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th)
        return -2;
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&th[t], NULL, worker, jb) != 0)
            break;
        ++started;
    }
    if (started == 0)
        worker(jb);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    return jb->status;
}

/* ---- exported API ---- */

/* Number of CPUs this process may run on. */
int oracle_num_threads(void)
{
    cpu_set_t set;
    CPU_ZERO(&set);
    if (sched_getaffinity(0, sizeof set, &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0)
            return n;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Prefill rows.  q [T_q, Hq, d], k/v [T_k, Hkv, d] bf16 bits, token-major.
 * Dense when cu_q == cu_k == NULL (sequence b = tokens [b*Nq, (b+1)*Nq) and
 * [b*Nk, (b+1)*Nk)); packed otherwise.  rows: n_rows triples (b, h, i) with i
 * local to sequence b.  out [n_rows, d] and lse [n_rows] in fp64.
 * Returns 0, or -1 for invalid arguments, -2 when out of memory.
 */
int oracle_prefill_rows_window(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               int B, int Hq, int Hkv, int Nq, int Nk, int d,
                               double scale, int causal, int win_left, int win_right,
                               const int32_t *cu_q, const int32_t *cu_k,
                               const int32_t *rows, long n_rows,
                               double *out, double *lse, int n_threads);

int oracle_prefill_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        double scale, int causal,
                        const int32_t *cu_q, const int32_t *cu_k,
                        const int32_t *rows, long n_rows,
                        double *out, double *lse, int n_threads)
{
    return oracle_prefill_rows_window(q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal, -1, -1, cu_q, cu_k,
                                      rows, n_rows, out, lse, n_threads);
}

static int prefill_rows(const void *q, const void *k, const void *v, int f64,
                        int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        double scale, int causal, int win_left, int win_right,
                        const int32_t *cu_q, const int32_t *cu_k,
                        const int32_t *rows, long n_rows,
                        double *out, double *lse, int n_threads);

/* As oracle_prefill_rows, with a local window (win_left, win_right); -1 on a
 * side leaves it unbounded. */
int oracle_prefill_rows_window(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               int B, int Hq, int Hkv, int Nq, int Nk, int d,
                               double scale, int causal, int win_left, int win_right,
                               const int32_t *cu_q, const int32_t *cu_k,
                               const int32_t *rows, long n_rows,
                               double *out, double *lse, int n_threads)
{
    return prefill_rows(q, k, v, 0, B, Hq, Hkv, Nq, Nk, d, scale, causal, win_left, win_right, cu_q, cu_k,
                        rows, n_rows, out, lse, n_threads);
}

/* As oracle_prefill_rows_window on inputs given as doubles (used for the
 * values an 8-bit encoding and its per-tile scales stand for, which bf16
 * cannot hold). */
int oracle_prefill_rows_f64(const double *q, const double *k, const double *v,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d,
                            double scale, int causal, int win_left, int win_right,
                            const int32_t *cu_q, const int32_t *cu_k,
                            const int32_t *rows, long n_rows,
                            double *out, double *lse, int n_threads)
{
    return prefill_rows(q, k, v, 1, B, Hq, Hkv, Nq, Nk, d, scale, causal, win_left, win_right, cu_q, cu_k,
                        rows, n_rows, out, lse, n_threads);
}

static int prefill_rows(const void *q, const void *k, const void *v, int f64,
                        int B, int Hq, int Hkv, int Nq, int Nk, int d,
                        double scale, int causal, int win_left, int win_right,
                        const int32_t *cu_q, const int32_t *cu_k,
                        const int32_t *rows, long n_rows,
                        double *out, double *lse, int n_threads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || n_rows < 0)
        return -1;
    if ((cu_q == NULL) != (cu_k == NULL))
        return -1;
    long max_keys = Nk;
    for (long r = 0; r < n_rows; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0)
            return -1;
        long nq = cu_q ? cu_q[b + 1] - cu_q[b] : Nq;
        long nk = cu_k ? cu_k[b + 1] - cu_k[b] : Nk;
        if (i >= nq || nk < 0)
            return -1;
        if (nk > max_keys)
            max_keys = nk;
    }
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.f64 = f64;
    jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.Nq = Nq; jb.Nk = Nk; jb.d = d;
    jb.causal = causal; jb.scale = scale;
    jb.win_left = win_left < 0 ? -1 : win_left;
    jb.win_right = win_right < 0 ? -1 : win_right;
    jb.cu_q = cu_q; jb.cu_k = cu_k;
    jb.rows = rows; jb.n_rows = n_rows;
    jb.out = out; jb.lse = lse;
    jb.max_keys = max_keys;
    return run_job(&jb, n_threads);
}

/*
 * Paged decode rows: one query per sequence, q [B, Hq, d]; caches
 * [num_pages, page_size, Hkv, d]; block_table [B, max_pages]; seq_lens [B].
 * rows: n_rows pairs (b, h).  out [n_rows, d], lse [n_rows] in fp64.
 */
int oracle_decode_rows(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                       int B, int Hq, int Hkv, int d, int page_size, double scale,
                       const int32_t *rows, long n_rows,
                       double *out, double *lse, int n_threads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || page_size <= 0 || n_rows < 0)
        return -1;
    long max_keys = 1;
    for (long r = 0; r < n_rows; ++r) {
        int b = rows[2 * r], h = rows[2 * r + 1];
        if (b < 0 || b >= B || h < 0 || h >= Hq)
            return -1;
        long len = seq_lens[b];
        if (len < 0 || len > (long)max_pages * page_size)
            return -1;
        if (len > max_keys)
            max_keys = len;
    }
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k_cache; jb.v = v_cache;
    jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.d = d;
    jb.paged = 1; jb.page_size = page_size; jb.max_pages = max_pages;
    jb.scale = scale;
    jb.block_table = block_table; jb.seq_lens = seq_lens;
    jb.rows = rows; jb.n_rows = n_rows;
    jb.out = out; jb.lse = lse;
    jb.max_keys = max_keys;
    return run_job(&jb, n_threads);
}

/*
 * Several queries per sequence over the paged cache.  q [B, Nq, Hq, d] (query
 * i of sequence b is its position seq_lens[b] - Nq + i); caches and block
 * table as oracle_decode_rows; rows: n_rows triples (b, h, i).
 * Returns 0, or -1 for invalid arguments, -2 when out of memory.
 */
int oracle_decode_multi_rows(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                             const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                             int B, int Nq, int Hq, int Hkv, int d, int page_size, double scale, int causal,
                             const int32_t *rows, long n_rows,
                             double *out, double *lse, int n_threads)
{
    if (B < 0 || Nq <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || page_size <= 0 || n_rows < 0)
        return -1;
    long max_keys = 1;
    for (long r = 0; r < n_rows; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Nq)
            return -1;
        long len = seq_lens[b];
        if (len < 0 || len > (long)max_pages * page_size)
            return -1;
        if (len > max_keys)
            max_keys = len;
    }
    job jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k_cache; jb.v = v_cache;
    jb.B = B; jb.Nq = Nq; jb.Hq = Hq; jb.Hkv = Hkv; jb.d = d;
    jb.causal = causal ? 1 : 0;
    jb.paged = 2; jb.page_size = page_size; jb.max_pages = max_pages;
    jb.scale = scale;
    jb.block_table = block_table; jb.seq_lens = seq_lens;
    jb.rows = rows; jb.n_rows = n_rows;
    jb.out = out; jb.lse = lse;
    jb.max_keys = max_keys;
    return run_job(&jb, n_threads);
}

/* ---- backward by the definition ---- */
typedef struct {
    const uint16_t *q, *k, *v, *g;   /* g = dL/dO, laid out like q */
    int B, Hq, Hkv, Nq, Nk, d, causal;
    long win_left, win_right;
    double scale;
    const int32_t *cu_q, *cu_k;
    const int32_t *pairs;            /* (b, kv head) pairs to compute */
    long n_pairs;
    long row_stride;                 /* 1: every row; k: rows i = 0, k, 2k, ... (a timing sample) */
    double *dq, *dk, *dv;
    long max_keys;
    long next;
    int status;
} bwd_job;

static void bwd_pair(bwd_job *jb, long r, double *sc, double *p, double *dp)
{
    const int b = jb->pairs[2 * r], g = jb->pairs[2 * r + 1];
    const int d = jb->d, group = jb->Hq / jb->Hkv;
    long q_first, k_first, nq, nk;
    if (jb->cu_q) {
        q_first = jb->cu_q[b];
        nq = jb->cu_q[b + 1] - jb->cu_q[b];
        k_first = jb->cu_k[b];
        nk = jb->cu_k[b + 1] - jb->cu_k[b];
    } else {
        q_first = (long)b * jb->Nq;
        nq = jb->Nq;
        k_first = (long)b * jb->Nk;
        nk = jb->Nk;
    }
    for (int h = g * group; h < (g + 1) * group; ++h) {
        for (long i = 0; i < nq; i += jb->row_stride) {
            const uint16_t *q_row = jb->q + ((q_first + i) * jb->Hq + h) * (long)d;
            const uint16_t *g_row = jb->g + ((q_first + i) * jb->Hq + h) * (long)d;
            double *dq_row = jb->dq + ((q_first + i) * jb->Hq + h) * (long)d;
            double m = -INFINITY;
            long n_allowed = 0;
            for (long j = 0; j < nk; ++j) {
                if (!key_allowed(i, j, nq, nk, jb->causal, jb->win_left, jb->win_right))
                    continue;
                const uint16_t *k_row = jb->k + ((k_first + j) * jb->Hkv + g) * (long)d;
                double dot = 0.0;
                for (int c = 0; c < d; ++c)
                    dot += bf16_value(q_row[c]) * bf16_value(k_row[c]);
                sc[j] = jb->scale * dot;
                if (n_allowed == 0 || sc[j] > m)
                    m = sc[j];
                ++n_allowed;
            }
            for (int c = 0; c < d; ++c)
                dq_row[c] = 0.0;
            if (n_allowed == 0)
                continue;   /* an empty row has O = 0 and passes no gradient */
            double l = 0.0;
            for (long j = 0; j < nk; ++j)
                if (key_allowed(i, j, nq, nk, jb->causal, jb->win_left, jb->win_right))
                    l += exp(sc[j] - m);
            double D = 0.0;
            for (long j = 0; j < nk; ++j) {
                if (!key_allowed(i, j, nq, nk, jb->causal, jb->win_left, jb->win_right))
                    continue;
                const uint16_t *v_row = jb->v + ((k_first + j) * jb->Hkv + g) * (long)d;
                p[j] = exp(sc[j] - m) / l;
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += bf16_value(g_row[c]) * bf16_value(v_row[c]);
                dp[j] = acc;
                D += p[j] * dp[j];
            }
            for (long j = 0; j < nk; ++j) {
                if (!key_allowed(i, j, nq, nk, jb->causal, jb->win_left, jb->win_right))
                    continue;
                const double ds = p[j] * (dp[j] - D);
                const uint16_t *k_row = jb->k + ((k_first + j) * jb->Hkv + g) * (long)d;
                double *dk_row = jb->dk + ((k_first + j) * jb->Hkv + g) * (long)d;
                double *dv_row = jb->dv + ((k_first + j) * jb->Hkv + g) * (long)d;
                for (int c = 0; c < d; ++c) {
                    dq_row[c] += jb->scale * ds * bf16_value(k_row[c]);
                    dk_row[c] += jb->scale * ds * bf16_value(q_row[c]);
                    dv_row[c] += p[j] * bf16_value(g_row[c]);
                }
            }
        }
    }
}

static void *bwd_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    size_t n = (size_t)(jb->max_keys > 0 ? jb->max_keys : 1);
    double *buf = (double *)malloc(sizeof(double) * 3 * n);
    if (!buf) {
        __atomic_store_n(&jb->status, -2, __ATOMIC_SEQ_CST);
        return NULL;
    }
    for (;;) {
        long r = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (r >= jb->n_pairs)
            break;
        bwd_pair(jb, r, buf, buf + n, buf + 2 * n);
    }
    free(buf);
    return NULL;
}

/*
 * Gradients dQ, dK, dV of L = <G, O> for the (b, kv head) pairs listed
 * (n_pairs pairs; each pair covers its group's query heads), dense or packed
 * like oracle_prefill_rows_window.  g [T_q, Hq, d] bf16 bits.  dq [T_q, Hq, d],
 * dk/dv [T_k, Hkv, d] fp64: the rows of the listed pairs are overwritten (dq)
 * or accumulated into (dk, dv: the caller zero-fills them).  row_stride > 1
 * takes only rows 0, row_stride, 2 row_stride, ... of each sequence (their
 * contributions; a timing sample, not a gradient).
 * Returns 0, or -1 for invalid arguments, -2 when out of memory.
 */
int oracle_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *g,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d,
                    double scale, int causal, int win_left, int win_right,
                    const int32_t *cu_q, const int32_t *cu_k,
                    const int32_t *pairs, long n_pairs, long row_stride,
                    double *dq, double *dk, double *dv, int n_threads)
{
    if (row_stride < 1)
        return -1;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || n_pairs < 0)
        return -1;
    if ((cu_q == NULL) != (cu_k == NULL))
        return -1;
    long max_keys = 1;
    for (long r = 0; r < n_pairs; ++r) {
        int b = pairs[2 * r], gg = pairs[2 * r + 1];
        if (b < 0 || b >= B || gg < 0 || gg >= Hkv)
            return -1;
        long nk = cu_k ? (long)cu_k[b + 1] - cu_k[b] : Nk;
        if (nk > max_keys)
            max_keys = nk;
    }
    bwd_job jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.g = g;
    jb.B = B; jb.Hq = Hq; jb.Hkv = Hkv; jb.Nq = Nq; jb.Nk = Nk; jb.d = d;
    jb.causal = causal ? 1 : 0;
    jb.win_left = win_left < 0 ? -1 : win_left;
    jb.win_right = win_right < 0 ? -1 : win_right;
    jb.scale = scale;
    jb.cu_q = cu_q; jb.cu_k = cu_k;
    jb.pairs = pairs; jb.n_pairs = n_pairs;
    jb.row_stride = row_stride;
    jb.dq = dq; jb.dk = dk; jb.dv = dv;
    jb.max_keys = max_keys;
    if (n_threads <= 0)
        n_threads = 1;
    if ((long)n_threads > n_pairs)
        n_threads = n_pairs > 0 ? (int)n_pairs : 1;
    if (n_threads > 1024)
        n_threads = 1024;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th)
        return -2;
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &jb) != 0)
            break;
        ++started;
    }
    if (started == 0)
        bwd_worker(&jb);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    return jb.status;
}


/* ---- 8-bit floating point, E4M3 ----
 *
 * "FP8 Path and Quantization" ("Flash Attention: A Complete Architectural
 * Autopsy", part 4) and "FlashAttention-3: asynchrony and low precision on
 * Hopper" ("FlashAttention-3 and PagedAttention") name the E4M3 format and
 * per-tile (block) quantization: a tile is scaled by a factor taken from its
 * absolute maximum before it is cast to 8 bits, and the scores are turned
 * back into fp32 before the softmax.
 *
 * E4M3 as this file reads it: 1 sign bit, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 holds the subnormals m * 2^-9; no
 * infinities; the one pattern S.1111.111 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_value(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7)
        return NAN;
    /* (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10) for e >= 1 */
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return sign ? -mag : mag;
}

/* x rounded to the nearest E4M3 value, ties to the even mantissa; magnitudes
 * from 448 up give 448 (saturation), NaN gives NaN. */
uint8_t oracle_e4m3_from_float(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x))
        return (uint8_t)(sign | 0x7f);
    const double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    if (a == 0.0)
        return sign;
    /* spacing of the representable values around a: 2^(floor(log2 a) - 3) in
     * the normal range, 2^-9 among the subnormals (below 2^-6) */
    int e2;
    frexp(a, &e2);
    int ue = e2 - 1;   /* floor(log2 a) */
    if (ue < -6)
        ue = -6;
    const double ulp = ldexp(1.0, ue - 3);
    const double v = rint(a / ulp) * ulp;   /* a / ulp is exact; rint ties to even */
    if (v < ldexp(1.0, -6))                 /* subnormal: the code is v / 2^-9 */
        return (uint8_t)(sign | (int)(v / ldexp(1.0, -9)));
    frexp(v, &e2);
    const int ve = e2 - 1;                  /* rounding may have reached the next binade */
    const int m = (int)((v / ldexp(1.0, ve) - 1.0) * 8.0);
    return (uint8_t)(sign | ((ve + 7) << 3) | m);
}

/*
 * Per-tile quantization of x [T, H, d] (bf16 bits) to E4M3 codes.
 *
 * A tile is 128 consecutive tokens of one sequence, counted from the
 * sequence's first token (the last tile of a sequence may be shorter), for
 * one head and all d channels.  Sequence b owns tokens [b*N, (b+1)*N) when cu
 * is NULL (dense), else [cu[b], cu[b+1]).  For each tile, in fp32:
 *   amax  = max |x| over the tile (exact: bf16 values are fp32 values)
 *   scale = amax / 448,  inv = 448 / amax          (each rounded to fp32)
 *   code  = E4M3(x * inv)  (the product rounded to fp32, then to E4M3)
 * so the tile's largest magnitude lands on 448 and x is represented as
 * E4M3(code) * scale.  A tile whose amax is below 2^-100 (all zero, or so
 * small that 448 / amax would overflow) gets scale 1 and all-zero codes.
 * scales [H, n_scale]: tile t of sequence b is entry floor(s_b / 128) + b + t,
 * s_b the sequence's first token; n_scale = T / 128 + B covers every
 * sequence (entries between sequences are left untouched).
 * Returns 0, or -1 for invalid arguments.
 */
int oracle_quantize_fp8(const uint16_t *x, int B, int H, int N, int d, const int32_t *cu,
                        uint8_t *codes, float *scales, long n_scale)
{
    if (B < 0 || H <= 0 || d <= 0 || (!cu && N < 0))
        return -1;
    for (int b = 0; b < B; ++b) {
        const long first = cu ? cu[b] : (long)b * N;
        const long len = cu ? (long)cu[b + 1] - cu[b] : N;
        if (first < 0 || len < 0)
            return -1;
        for (long t = 0; t * 128 < len; ++t) {
            const long idx = first / 128 + b + t;
            if (idx >= n_scale)
                return -1;
            const long r0 = first + 128 * t;
            const long rows = len - 128 * t < 128 ? len - 128 * t : 128;
            for (int h = 0; h < H; ++h) {
                float amax = 0.0f;
                for (long r = r0; r < r0 + rows; ++r)
                    for (int c = 0; c < d; ++c) {
                        const float a = (float)fabs(bf16_value(x[(r * H + h) * (long)d + c]));
                        if (a > amax)
                            amax = a;
                    }
                const int zero = !(amax >= 0x1p-100f);
                const float scale = zero ? 1.0f : amax / 448.0f;
                const float inv = zero ? 0.0f : 448.0f / amax;
                for (long r = r0; r < r0 + rows; ++r)
                    for (int c = 0; c < d; ++c) {
                        const long at = (r * H + h) * (long)d + c;
                        const float y = (float)bf16_value(x[at]) * inv;
                        codes[at] = zero ? 0 : oracle_e4m3_from_float(y);
                    }
                scales[(long)h * n_scale + idx] = scale;
            }
        }
    }
    return 0;
}

/* The values quantized tiles stand for: out = E4M3(code) * scale of the
 * code's tile, in fp64 (exact), with the tiles and the scale layout of
 * oracle_quantize_fp8. */
int oracle_dequantize_fp8(const uint8_t *codes, const float *scales, long n_scale, int B, int H, int N, int d,
                          const int32_t *cu, double *out)
{
    if (B < 0 || H <= 0 || d <= 0 || (!cu && N < 0))
        return -1;
    for (int b = 0; b < B; ++b) {
        const long first = cu ? cu[b] : (long)b * N;
        const long len = cu ? (long)cu[b + 1] - cu[b] : N;
        for (long r = first; r < first + len; ++r) {
            const long idx = first / 128 + b + (r - first) / 128;
            if (idx >= n_scale)
                return -1;
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < d; ++c) {
                    const long at = (r * H + h) * (long)d + c;
                    out[at] = oracle_e4m3_value(codes[at]) * (double)scales[(long)h * n_scale + idx];
                }
        }
    }
    return 0;
}
