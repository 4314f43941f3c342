/*
 * oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: it is written from the definition of attention, not from the
 * kernels.
 *
 * Sources (page title, section):
 *   [FP]  "Flash Attention, From First Principles" (adithyag73.github.io)
 *   [LAR] "LLM Architecture Refresh [3]: Flash Attention Is Exact, and Here's
 *          the Proof" (bearbearyu1223.github.io)
 *   [FAS] "FlashAttention from scratch: how it works and how to code it"
 *          (interview.clozo.ai)
 *
 * Tensor layout everywhere: contiguous [B][H][N][d] row-major doubles, the
 * (batch, heads, seq, dim) order of [LAR] section 4.  A "head" is one (b, h)
 * slice of N*d numbers.
 *
 * Definition ([FP] "What is attention?", Stop 1-3; [LAR] section 4 applies the
 * scale; [FAS] follow-up "How do you implement the backward pass"):
 *   s_rk  = scale * <q_r, k_k>            (k > r is -inf when causal; with a
 *                                          sliding window of w keys, also
 *                                          k < r - w + 1: [LAR] section 5's
 *                                          contrast, "each query attends only
 *                                          to the last w keys")
 *   m_r   = max_k s_rk
 *   l_r   = sum_k exp(s_rk - m_r)
 *   p_rk  = exp(s_rk - m_r) / l_r
 *   o_r   = sum_k p_rk v_k
 *   LSE_r = m_r + ln l_r                  (natural log)
 * Backward, with upstream gradient dO:
 *   dP_rk = <dO_r, v_k>
 *   D_r   = sum_k p_rk dP_rk              (equals <dO_r, o_r>)
 *   dS_rk = p_rk (dP_rk - D_r)
 *   dQ_r  = scale * sum_k dS_rk k_k
 *   dK_k  = scale * sum_r dS_rk q_r
 *   dV_k  = sum_r p_rk dO_r
 *
 * Dropout (the reading of the pages' "algorithm 2's extra lines", [FP]
 * "What's left out"): after the softmax, p_rk is replaced by p_rk * M_rk with
 * M_rk = keep_rk * 256 / (256 - t), keep_rk in {0, 1}, so O = (P o M) V while
 * LSE stays that of the undropped row.  Then D_r = sum_k p_rk M_rk dP_rk
 * (still <dO_r, o_r>), dS_rk = p_rk (M_rk dP_rk - D_r), dV_k = sum_r p_rk M_rk
 * dO_r.  keep_rk comes from the counter-based generator Philox4x32-10
 * (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2,
 * 3", SC'11): key = (seed low word, seed high word), counter = (k/4, r/4,
 * head, 0); of the 16 output bytes, byte (k mod 4) of word (r mod 4) is the
 * one of (r, k), and keep_rk = (byte >= t).  t = round(256 * dropout
 * probability) in 0..255.
 *
 * Every function returns 0 on success and a negative number on bad arguments.
 * Parity pins for every exported function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_PLANT_NO_RESCALE 1 /* negative control: drop the rescale */

typedef long long i64;

/* ------------------------------------------------------------------ */
/* A tiny parallel-for over [0, n): each worker takes a contiguous slice. */

typedef void (*range_fn)(void *ctx, i64 begin, i64 end);

typedef struct {
    range_fn fn;
    void *ctx;
    i64 begin, end;
} worker_arg;

static void *worker_main(void *p) {
    worker_arg *a = (worker_arg *)p;
    a->fn(a->ctx, a->begin, a->end);
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

static void parallel_for(i64 n, int nthreads, range_fn fn, void *ctx) {
    int t = resolve_threads(nthreads);
    if ((i64)t > n) t = (int)(n > 0 ? n : 1);
    if (t <= 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)t);
    worker_arg *args = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)t);
    for (int i = 0; i < t; ++i) {
        args[i].fn = fn;
        args[i].ctx = ctx;
        args[i].begin = n * i / t;
        args[i].end = n * (i + 1) / t;
        if (pthread_create(&th[i], NULL, worker_main, &args[i]) != 0) {
            /* could not start a thread: do its slice here */
            worker_main(&args[i]);
            th[i] = 0;
        }
    }
    for (int i = 0; i < t; ++i)
        if (th[i]) pthread_join(th[i], NULL);
    free(args);
    free(th);
}

static int bad_shape(int B, int H, int N, int d) {
    return B < 1 || H < 1 || N < 1 || d < 1;
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10, written from its published definition: ten rounds of two
 * 32x32->64-bit products (multipliers 0xD2511F53 and 0xCD9E8D57) whose
 * halves are crossed and xored with the key, the key advancing by the Weyl
 * constants 0x9E3779B9 and 0xBB67AE85 between rounds. */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

/* Dropout decision for (head bh, query r, key k); see the header comment. */
static int drop_keep(uint64_t seed, i64 bh, int r, int k, int t) {
    uint32_t ctr[4] = {(uint32_t)(k >> 2), (uint32_t)(r >> 2), (uint32_t)bh, 0};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    int byte = (int)((out[r & 3] >> (8 * (k & 3))) & 0xFFu);
    return byte >= t;
}

/* keep[bh][r][k] as bytes (0/1) for t in 0..255; pins and tests only. */
int oracle_dropout_keep(int B, int H, int N, int t, uint64_t seed,
                        uint8_t *keep) {
    if (B < 1 || H < 1 || N < 1 || t < 0 || t > 255 || !keep) return -1;
    for (i64 bh = 0; bh < (i64)B * H; ++bh)
        for (int r = 0; r < N; ++r)
            for (int k = 0; k < N; ++k)
                keep[(bh * N + r) * N + k] = (uint8_t)drop_keep(seed, bh, r, k, t);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Scores and probabilities of one query row, straight from the definition
 * ([FP] Stop 1 and Stop 2.5: subtract the row max, exponentiate, divide by
 * the sum).  s and p are caller buffers of N doubles. */

static double dot(const double *a, const double *b, int d) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += a[i] * b[i];
    return acc;
}

/* Is key k visible to query r?  Causal: k <= r ([LAR] section 5: scores
 * above the diagonal forced to -inf).  A sliding window of w > 0 keys (which
 * implies causal) also hides k < r - w + 1 ([LAR] section 5, the
 * sliding-window contrast: the query and the w - 1 keys before it). */
static int visible(int causal, int window, int r, int k) {
    if (window > 0) return k <= r && k >= r - window + 1;
    return !causal || k <= r;
}

/* Fills s[0..N) with the scaled scores of row r; invisible keys are -inf. */
static void row_scores(const double *Qh, const double *Kh, int N, int d,
                       double scale, int causal, int window, int r,
                       double *s) {
    const double *q = Qh + (i64)r * d;
    for (int k = 0; k < N; ++k) {
        if (!visible(causal, window, r, k))
            s[k] = -INFINITY;
        else
            s[k] = scale * dot(q, Kh + (i64)k * d, d);
    }
}

/* Turns scores into probabilities in place (p may alias s); returns the row
 * max and writes the normaliser l. */
static double row_softmax(const double *s, double *p, int N, double *l_out) {
    double m = -INFINITY;
    for (int k = 0; k < N; ++k)
        if (s[k] > m) m = s[k];
    double l = 0.0;
    for (int k = 0; k < N; ++k) {
        double e = (s[k] == -INFINITY) ? 0.0 : exp(s[k] - m);
        p[k] = e;
        l += e;
    }
    for (int k = 0; k < N; ++k) p[k] = p[k] / l;
    *l_out = l;
    return m;
}

/* Dropout of one call: t = 0 disables it. */
typedef struct {
    int t;
    uint64_t seed;
} drop_spec;

/* M_rk of the header comment (1 without dropout). */
static double drop_factor(const drop_spec *dr, i64 bh, int r, int k) {
    if (!dr || dr->t == 0) return 1.0;
    return drop_keep(dr->seed, bh, r, k, dr->t) ? 256.0 / (256 - dr->t) : 0.0;
}

/* o_r = sum_k p_k M_k v_k and LSE_r = m + ln l for row r of head bh. */
static void attend_row(const double *Qh, const double *Kh, const double *Vh,
                       int N, int d, double scale, int causal, int window,
                       const drop_spec *dr, i64 bh, int r, double *work,
                       double *o, double *lse) {
    double l;
    row_scores(Qh, Kh, N, d, scale, causal, window, r, work);
    double m = row_softmax(work, work, N, &l);
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int k = 0; k < N; ++k) {
        double pk = work[k] * drop_factor(dr, bh, r, k);
        if (pk == 0.0) continue;
        const double *v = Vh + (i64)k * d;
        for (int c = 0; c < d; ++c) o[c] += pk * v[c];
    }
    if (lse) *lse = m + log(l);
}

/* ------------------------------------------------------------------ */
/* Full score and probability matrices for small inputs (pins only). */

int oracle_scores(const double *Q, const double *K, double *S, int B, int H,
                  int N, int d, double scale, int causal) {
    if (bad_shape(B, H, N, d) || !Q || !K || !S) return -1;
    i64 heads = (i64)B * H;
    for (i64 bh = 0; bh < heads; ++bh)
        for (int r = 0; r < N; ++r)
            row_scores(Q + bh * N * d, K + bh * N * d, N, d, scale, causal, 0,
                       r, S + (bh * N + r) * N);
    return 0;
}

int oracle_probs(const double *Q, const double *K, double *P, int B, int H,
                 int N, int d, double scale, int causal) {
    if (oracle_scores(Q, K, P, B, H, N, d, scale, causal) != 0) return -1;
    i64 rows = (i64)B * H * N;
    for (i64 r = 0; r < rows; ++r) {
        double l;
        row_softmax(P + r * N, P + r * N, N, &l);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Forward: every row, or a chosen list of rows. */

typedef struct {
    const double *Q, *K, *V;
    double *O, *LSE;
    int N, d, causal, window;
    double scale;
    const i64 *rows; /* NULL: all rows in order */
    drop_spec drop;
} fwd_ctx;

static void fwd_range(void *p, i64 begin, i64 end) {
    fwd_ctx *c = (fwd_ctx *)p;
    double *work = (double *)malloc(sizeof(double) * (size_t)c->N);
    for (i64 i = begin; i < end; ++i) {
        i64 flat = c->rows ? c->rows[i] : i;
        i64 bh = flat / c->N;
        int r = (int)(flat % c->N);
        i64 off = bh * c->N * c->d;
        attend_row(c->Q + off, c->K + off, c->V + off, c->N, c->d, c->scale,
                   c->causal, c->window, &c->drop, bh, r, work, c->O + i * c->d,
                   c->LSE ? c->LSE + i : NULL);
    }
    free(work);
}

int oracle_fwd(const double *Q, const double *K, const double *V, double *O,
               double *LSE, int B, int H, int N, int d, double scale,
               int causal, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !O) return -1;
    fwd_ctx c = {Q, K, V, O, LSE, N, d, causal, 0, scale, NULL, {0, 0}};
    parallel_for((i64)B * H * N, nthreads, fwd_range, &c);
    return 0;
}

/* Every option at once: causal, sliding window (0: none), dropout threshold
 * t (0: none) and seed.  With t = 0 this is oracle_fwd / oracle_fwd_w. */
int oracle_fwd_x(const double *Q, const double *K, const double *V, double *O,
                 double *LSE, int B, int H, int N, int d, double scale,
                 int causal, int window, int t, uint64_t seed, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !O || window < 0 || t < 0 ||
        t > 255)
        return -1;
    fwd_ctx c = {Q, K, V, O, LSE, N, d, causal || window > 0, window, scale,
                 NULL, {t, seed}};
    parallel_for((i64)B * H * N, nthreads, fwd_range, &c);
    return 0;
}

/* Causal sliding window of `window` >= 1 keys (query r sees keys
 * r - window + 1 .. r). */
int oracle_fwd_w(const double *Q, const double *K, const double *V, double *O,
                 double *LSE, int B, int H, int N, int d, double scale,
                 int window, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !O || window < 1) return -1;
    fwd_ctx c = {Q, K, V, O, LSE, N, d, 1, window, scale, NULL, {0, 0}};
    parallel_for((i64)B * H * N, nthreads, fwd_range, &c);
    return 0;
}

int oracle_fwd_rows_w(const double *Q, const double *K, const double *V,
                      double *O, double *LSE, int B, int H, int N, int d,
                      double scale, int causal, int window, const i64 *rows,
                      i64 nrows, int nthreads);

/* rows[i] is a flat row index (b*H + h)*N + r; O is [nrows][d], LSE [nrows]. */
int oracle_fwd_rows(const double *Q, const double *K, const double *V,
                    double *O, double *LSE, int B, int H, int N, int d,
                    double scale, int causal, const i64 *rows, i64 nrows,
                    int nthreads) {
    return oracle_fwd_rows_w(Q, K, V, O, LSE, B, H, N, d, scale, causal, 0,
                             rows, nrows, nthreads);
}

int oracle_fwd_rows_x(const double *Q, const double *K, const double *V,
                      double *O, double *LSE, int B, int H, int N, int d,
                      double scale, int causal, int window, int t,
                      uint64_t seed, const i64 *rows, i64 nrows, int nthreads);

/* As oracle_fwd_rows; window > 0 selects the causal sliding window. */
int oracle_fwd_rows_w(const double *Q, const double *K, const double *V,
                      double *O, double *LSE, int B, int H, int N, int d,
                      double scale, int causal, int window, const i64 *rows,
                      i64 nrows, int nthreads) {
    return oracle_fwd_rows_x(Q, K, V, O, LSE, B, H, N, d, scale, causal, window,
                             0, 0, rows, nrows, nthreads);
}

/* As oracle_fwd_rows with every option (see oracle_fwd_x). */
int oracle_fwd_rows_x(const double *Q, const double *K, const double *V,
                      double *O, double *LSE, int B, int H, int N, int d,
                      double scale, int causal, int window, int t,
                      uint64_t seed, const i64 *rows, i64 nrows, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !O || !rows || nrows < 0 ||
        window < 0 || t < 0 || t > 255)
        return -1;
    i64 total = (i64)B * H * N;
    for (i64 i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= total) return -2;
    fwd_ctx c = {Q, K, V, O, LSE, N, d, causal || window > 0, window, scale,
                 rows, {t, seed}};
    parallel_for(nrows, nthreads, fwd_range, &c);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Backward ([FAS] follow-up on the backward pass; [FP] "The ghost at the
 * door": C = AB gives dA = dC B^T, dB = A^T dC).  Heads are independent, so
 * each worker owns whole heads and accumulates dK, dV without races.
 * Dvec (optional) receives D_r = sum_k p_rk dP_rk. */

typedef struct {
    const double *Q, *K, *V, *dO;
    double *dQ, *dK, *dV, *Dvec;
    int N, d, causal, window;
    double scale;
    drop_spec drop;
} bwd_ctx;

static void bwd_range(void *p, i64 begin, i64 end) {
    bwd_ctx *c = (bwd_ctx *)p;
    int N = c->N, d = c->d;
    double *prob = (double *)malloc(sizeof(double) * (size_t)N);
    double *dP = (double *)malloc(sizeof(double) * (size_t)N);
    for (i64 bh = begin; bh < end; ++bh) {
        i64 off = bh * N * d;
        const double *Qh = c->Q + off, *Kh = c->K + off, *Vh = c->V + off;
        const double *dOh = c->dO + off;
        double *dQh = c->dQ + off, *dKh = c->dK + off, *dVh = c->dV + off;
        memset(dKh, 0, sizeof(double) * (size_t)N * d);
        memset(dVh, 0, sizeof(double) * (size_t)N * d);
        for (int r = 0; r < N; ++r) {
            double l;
            row_scores(Qh, Kh, N, d, c->scale, c->causal, c->window, r, prob);
            row_softmax(prob, prob, N, &l);
            const double *dOr = dOh + (i64)r * d;
            const double *qr = Qh + (i64)r * d;
            double D = 0.0;
            for (int k = 0; k < N; ++k) {
                dP[k] = dot(dOr, Vh + (i64)k * d, d);
                D += prob[k] * drop_factor(&c->drop, bh, r, k) * dP[k];
            }
            if (c->Dvec) c->Dvec[bh * N + r] = D;
            double *dQr = dQh + (i64)r * d;
            for (int i = 0; i < d; ++i) dQr[i] = 0.0;
            for (int k = 0; k < N; ++k) {
                double pk = prob[k];
                if (pk == 0.0) continue;
                double mk = drop_factor(&c->drop, bh, r, k);
                double dS = pk * (mk * dP[k] - D);
                const double *kk = Kh + (i64)k * d;
                double *dKk = dKh + (i64)k * d;
                double *dVk = dVh + (i64)k * d;
                for (int i = 0; i < d; ++i) {
                    dQr[i] += c->scale * dS * kk[i];
                    dKk[i] += c->scale * dS * qr[i];
                    dVk[i] += pk * mk * dOr[i];
                }
            }
        }
    }
    free(dP);
    free(prob);
}

int oracle_bwd(const double *Q, const double *K, const double *V,
               const double *dO, double *dQ, double *dK, double *dV,
               double *Dvec, int B, int H, int N, int d, double scale,
               int causal, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !dO || !dQ || !dK || !dV)
        return -1;
    bwd_ctx c = {Q, K, V, dO, dQ, dK, dV, Dvec, N, d, causal, 0, scale, {0, 0}};
    parallel_for((i64)B * H, nthreads, bwd_range, &c);
    return 0;
}

/* Every option at once (see oracle_fwd_x). */
int oracle_bwd_x(const double *Q, const double *K, const double *V,
                 const double *dO, double *dQ, double *dK, double *dV,
                 double *Dvec, int B, int H, int N, int d, double scale,
                 int causal, int window, int t, uint64_t seed, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !dO || !dQ || !dK || !dV ||
        window < 0 || t < 0 || t > 255)
        return -1;
    bwd_ctx c = {Q, K, V, dO, dQ, dK, dV, Dvec, N, d, causal || window > 0,
                 window, scale, {t, seed}};
    parallel_for((i64)B * H, nthreads, bwd_range, &c);
    return 0;
}

/* Backward of the causal sliding window of `window` >= 1 keys. */
int oracle_bwd_w(const double *Q, const double *K, const double *V,
                 const double *dO, double *dQ, double *dK, double *dV,
                 double *Dvec, int B, int H, int N, int d, double scale,
                 int window, int nthreads) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !dO || !dQ || !dK || !dV ||
        window < 1)
        return -1;
    bwd_ctx c = {Q, K, V, dO, dQ, dK, dV, Dvec, N, d, 1, window, scale, {0, 0}};
    parallel_for((i64)B * H, nthreads, bwd_range, &c);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Tiled companion: the online-softmax loop with queries outer and key/value
 * blocks inner ([LAR] section 4, deferred division at the end; causal tiles
 * whose first key lies after the block's last query are skipped, [LAR]
 * section 7).  It exists to check tiled == untiled in fp64, to count tiles
 * and matmul FLOPs the way [LAR] sections 7-8 count them, and to replay the
 * worked examples block by block.
 *
 * counters (optional, 3 entries): matmul FLOPs (2 matmuls of
 * 2*rows*cols*d each per computed tile), tiles computed, tiles skipped.
 * trace (optional): for head trace_bh and row trace_row, after each key block
 * that row's running (m, l, o[0..d)) is appended: (2+d) doubles per block,
 * at most ceil(N/block_k) blocks.
 * flags: ORACLE_PLANT_NO_RESCALE drops the rebase of l and o (the mistake the
 * [FAS] worked example warns about); only the negative-control test sets it.
 * window > 0 selects the causal sliding window: tiles whose last key is
 * older than the block's first query's window are skipped too. */
static int fwd_tiled(const double *Q, const double *K, const double *V,
                     double *O, double *LSE, int B, int H, int N, int d,
                     double scale, int causal, int window, int block_q,
                     int block_k, int flags, i64 *counters, i64 trace_bh,
                     int trace_row, double *trace) {
    if (bad_shape(B, H, N, d) || !Q || !K || !V || !O || block_q < 1 ||
        block_k < 1 || window < 0)
        return -1;
    if (window > 0) causal = 1;
    i64 heads = (i64)B * H;
    i64 flops = 0, computed = 0, skipped = 0;
    double *m = (double *)malloc(sizeof(double) * (size_t)block_q);
    double *l = (double *)malloc(sizeof(double) * (size_t)block_q);
    double *acc = (double *)malloc(sizeof(double) * (size_t)block_q * d);
    double *sc = (double *)malloc(sizeof(double) * (size_t)block_q * block_k);
    for (i64 bh = 0; bh < heads; ++bh) {
        const double *Qh = Q + bh * N * d, *Kh = K + bh * N * d;
        const double *Vh = V + bh * N * d;
        int trace_n = 0;
        for (int i = 0; i < N; i += block_q) {
            int rows = (N - i < block_q) ? N - i : block_q;
            for (int a = 0; a < rows; ++a) {
                m[a] = -INFINITY;
                l[a] = 0.0;
                for (int c = 0; c < d; ++c) acc[(i64)a * d + c] = 0.0;
            }
            for (int j = 0; j < N; j += block_k) {
                int cols = (N - j < block_k) ? N - j : block_k;
                if ((causal && j > i + rows - 1) ||
                    (window > 0 && j + cols - 1 < i - window + 1)) {
                    skipped += 1;
                    continue;
                }
                computed += 1;
                flops += 2 * (2 * (i64)rows * cols * d);
                /* score tile, with the mask inside the tiles it cuts */
                for (int a = 0; a < rows; ++a)
                    for (int b = 0; b < cols; ++b) {
                        int qi = i + a, kj = j + b;
                        sc[(i64)a * block_k + b] =
                            !visible(causal, window, qi, kj)
                                ? -INFINITY
                                : scale * dot(Qh + (i64)qi * d,
                                              Kh + (i64)kj * d, d);
                    }
                for (int a = 0; a < rows; ++a) {
                    double tile_max = -INFINITY;
                    for (int b = 0; b < cols; ++b)
                        if (sc[(i64)a * block_k + b] > tile_max)
                            tile_max = sc[(i64)a * block_k + b];
                    double m_new = m[a] > tile_max ? m[a] : tile_max;
                    /* a fully masked row so far: nothing to rebase, nothing
                     * to add ([FAS] edge cases: guard exp(-inf - -inf)) */
                    double corr = (m_new == -INFINITY) ? 1.0 : exp(m[a] - m_new);
                    if (flags & ORACLE_PLANT_NO_RESCALE) corr = 1.0;
                    double rowsum = 0.0;
                    double *o = acc + (i64)a * d;
                    for (int c = 0; c < d; ++c) o[c] *= corr;
                    for (int b = 0; b < cols; ++b) {
                        double s = sc[(i64)a * block_k + b];
                        double p = (s == -INFINITY) ? 0.0 : exp(s - m_new);
                        rowsum += p;
                        const double *v = Vh + (i64)(j + b) * d;
                        for (int c = 0; c < d; ++c) o[c] += p * v[c];
                    }
                    l[a] = l[a] * corr + rowsum;
                    m[a] = m_new;
                    if (trace && bh == trace_bh && i + a == trace_row) {
                        double *t = trace + (i64)trace_n * (2 + d);
                        t[0] = m[a];
                        t[1] = l[a];
                        for (int c = 0; c < d; ++c) t[2 + c] = o[c];
                        trace_n += 1;
                    }
                }
            }
            for (int a = 0; a < rows; ++a) {
                double *out = O + (bh * N + i + a) * d;
                for (int c = 0; c < d; ++c) out[c] = acc[(i64)a * d + c] / l[a];
                if (LSE) LSE[bh * N + i + a] = m[a] + log(l[a]);
            }
        }
    }
    free(sc);
    free(acc);
    free(l);
    free(m);
    if (counters) {
        counters[0] = flops;
        counters[1] = computed;
        counters[2] = skipped;
    }
    return 0;
}

int oracle_fwd_tiled(const double *Q, const double *K, const double *V,
                     double *O, double *LSE, int B, int H, int N, int d,
                     double scale, int causal, int block_q, int block_k,
                     int flags, i64 *counters, i64 trace_bh, int trace_row,
                     double *trace) {
    return fwd_tiled(Q, K, V, O, LSE, B, H, N, d, scale, causal, 0, block_q,
                     block_k, flags, counters, trace_bh, trace_row, trace);
}

int oracle_fwd_tiled_w(const double *Q, const double *K, const double *V,
                       double *O, double *LSE, int B, int H, int N, int d,
                       double scale, int window, int block_q, int block_k,
                       i64 *counters) {
    if (window < 1) return -1;
    return fwd_tiled(Q, K, V, O, LSE, B, H, N, d, scale, 1, window, block_q,
                     block_k, 0, counters, -1, 0, NULL);
}

/* ------------------------------------------------------------------ */
/* The online normaliser on one row of logits, one block at a time ([FP]
 * "The citizenship laws"; [LAR] section 2).  After block t, m_trace[t] is the
 * running max and l_trace[t] the running sum of exp(x - m). */
int oracle_online_normalizer(const double *x, int n, int block,
                             double *m_trace, double *l_trace) {
    if (!x || n < 1 || block < 1 || !m_trace || !l_trace) return -1;
    double m = -INFINITY, l = 0.0;
    int t = 0;
    for (int start = 0; start < n; start += block) {
        int end = start + block < n ? start + block : n;
        double bmax = -INFINITY;
        for (int i = start; i < end; ++i)
            if (x[i] > bmax) bmax = x[i];
        double m_new = m > bmax ? m : bmax;
        double corr = exp(m - m_new);
        double add = 0.0;
        for (int i = start; i < end; ++i) add += exp(x[i] - m_new);
        l = l * corr + add;
        m = m_new;
        m_trace[t] = m;
        l_trace[t] = l;
        ++t;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Tile census without arithmetic ([LAR] sections 7 and 8): walks the same
 * (query block, key block) grid as oracle_fwd_tiled and counts computed and
 * skipped tiles and the matmul FLOPs of the computed ones, for `heads`
 * independent heads.  out = {flops, computed, skipped}. */
int oracle_tile_census(i64 heads, int N, int d, int block_q, int block_k,
                       int causal, i64 *out) {
    if (heads < 1 || N < 1 || d < 1 || block_q < 1 || block_k < 1 || !out)
        return -1;
    i64 flops = 0, computed = 0, skipped = 0;
    for (int i = 0; i < N; i += block_q) {
        int rows = (N - i < block_q) ? N - i : block_q;
        for (int j = 0; j < N; j += block_k) {
            int cols = (N - j < block_k) ? N - j : block_k;
            if (causal && j > i + rows - 1) {
                skipped += 1;
                continue;
            }
            computed += 1;
            flops += 2 * (2 * (i64)rows * cols * d);
        }
    }
    out[0] = flops * heads;
    out[1] = computed * heads;
    out[2] = skipped * heads;
    return 0;
}
