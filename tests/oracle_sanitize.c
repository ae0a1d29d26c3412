/*
 * Runs every oracle function on small seeded inputs, including the degenerate
 * cases the oracle accepts (no history, one tap, one position, one candidate,
 * rows holding NaN and -inf, rejected arguments), so that a build of the
 * oracle with -fsanitize=address,undefined can report any out-of-bounds
 * access, leak or undefined behaviour.  Exit status 0 means every call
 * returned what the arguments call for; the sanitizers abort on a finding.
 * Test infrastructure only: compiled together with oracle/dflash2_oracle.c by
 * tests/test_oracle_sanitize.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

int oracle_max_threads(void);
int oracle_dynconv(const double* x, const double* hist, const double* base, const double* delta,
                   double* out, long S, long n, long C, long T, long G);
void oracle_project(const double* h, const double* W, double* u, long P, long d, long R);
int oracle_edges(const int32_t* cand_ids, const double* u, const double* A, const double* B,
                 const double* unary, long S, long n, long K, long R, long V, double* edges,
                 int32_t* best_slot, double* best_score);
int oracle_select(const double* h, const double* W, const int32_t* cand_ids, const double* A,
                  const double* B, const double* unary, long S, long n, long d, long K, long R,
                  long V, double* u, double* edges, int32_t* best_slot, double* best_score);
int oracle_topk(const double* z, long rows, long V, long K, int32_t* ids, double* vals);
int oracle_chain(const int32_t* cand_ids, const double* unary, const double* edges,
                 const int32_t* best_slot, const int32_t* start_slot, long S, long n, long K,
                 double p_min, int32_t* tokens, double* probs, int32_t* length);

static uint64_t g_state = 0x9E3779B97F4A7C15ull;

static double rnd(void) { /* xorshift64*, uniform in [-1, 1) */
    g_state ^= g_state >> 12;
    g_state ^= g_state << 25;
    g_state ^= g_state >> 27;
    const uint64_t v = g_state * 0x2545F4914F6CDD1Dull;
    return (double)(v >> 11) / 4503599627370496.0 - 1.0;
}

static double* vec(long n) {
    double* p = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    for (long i = 0; i < n; ++i) p[i] = rnd();
    return p;
}

static int fails = 0;
#define CHECK(c)                                                      \
    do {                                                              \
        if (!(c)) {                                                   \
            fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
            ++fails;                                                  \
        }                                                             \
    } while (0)

static void conv_case(long S, long n, long C, long T, long G, int with_hist) {
    double *x = vec(S * n * C), *h = vec(S * (T - 1) * C), *b = vec(T * C);
    double *d = vec(S * n * T * G), *o = vec(S * n * C);
    CHECK(oracle_dynconv(x, with_hist ? h : NULL, b, d, o, S, n, C, T, G) == 0);
    for (long i = 0; i < S * n * C; ++i) CHECK(isfinite(o[i]));
    free(x); free(h); free(b); free(d); free(o);
}

static void select_case(long S, long n, long d, long K, long R, long V) {
    double *h = vec(S * n * d), *W = vec(R * d), *A = vec(V * R), *B = vec(V * R);
    double *un = vec(S * n * K), *u = vec(S * n * R);
    const long E = S * (n > 1 ? n - 1 : 0);
    double *e = vec(E * K * K), *sc = vec(E * K);
    int32_t* slot = (int32_t*)malloc((size_t)(E * K > 0 ? E * K : 1) * 4);
    int32_t* ids = (int32_t*)malloc((size_t)(S * n * K) * 4);
    for (long i = 0; i < S * n * K; ++i) ids[i] = (int32_t)((i * 7919) % V);
    CHECK(oracle_select(h, W, ids, A, B, un, S, n, d, K, R, V, u, e, slot, sc) == 0);
    CHECK(oracle_edges(ids, u, A, B, un, S, n, K, R, V, NULL, slot, sc) == 0);
    for (long i = 0; i < E * K; ++i) CHECK(slot[i] >= 0 && slot[i] < K);
    if (S * n * K > 0) {  /* an id outside [0, V) is rejected, not read */
        ids[0] = (int32_t)V;
        CHECK(oracle_edges(ids, u, A, B, un, S, n, K, R, V, e, slot, sc) == 1);
        ids[0] = -1;
        CHECK(oracle_edges(ids, u, A, B, un, S, n, K, R, V, e, slot, sc) == 1);
    }
    if (E > 0) {  /* chain on the argmax table just written */
        int32_t *tok = (int32_t*)malloc((size_t)(S * n) * 4), *len = (int32_t*)malloc((size_t)S * 4);
        int32_t* st = (int32_t*)malloc((size_t)S * 4);
        double* pr = vec(S * n);
        for (long i = 0; i < S * n * K; ++i) ids[i] = (int32_t)((i * 7919) % V);
        CHECK(oracle_edges(ids, u, A, B, un, S, n, K, R, V, e, slot, sc) == 0);
        CHECK(oracle_chain(ids, un, e, slot, NULL, S, n, K, 0.1, tok, pr, len) == 0);
        for (long s = 0; s < S; ++s) st[s] = (int32_t)(s % K);
        CHECK(oracle_chain(ids, un, e, slot, st, S, n, K, 0.0, tok, pr, len) == 0);
        for (long s = 0; s < S; ++s) CHECK(len[s] == n);
        st[0] = (int32_t)K;  /* bad start slot */
        CHECK(oracle_chain(ids, un, e, slot, st, S, n, K, 0.0, tok, pr, len) == 1);
        for (long i = 0; i < E * K; ++i) slot[i] = (int32_t)K;  /* every table entry bad */
        CHECK(oracle_chain(ids, un, e, slot, NULL, S, n, K, 0.0, tok, pr, len) == 1);
        free(tok); free(len); free(st); free(pr);
    }
    free(h); free(W); free(A); free(B); free(un); free(u); free(e); free(sc); free(slot);
    free(ids);
}

static void topk_case(long rows, long V, long K) {
    double* z = vec(rows * V);
    if (rows * V > 3) {
        z[0] = NAN;
        z[1] = -INFINITY;
        z[2] = -0.0;
        z[3] = 0.0;
    }
    int32_t* ids = (int32_t*)malloc((size_t)(rows * K) * 4);
    double* v = vec(rows * K);
    CHECK(oracle_topk(z, rows, V, K, ids, v) == 0);
    for (long i = 0; i < rows * K; ++i) CHECK(ids[i] >= -1 && ids[i] < V);
    CHECK(oracle_topk(z, rows, V, V + 1, ids, v) == 1);
    CHECK(oracle_topk(z, rows, V, 0, ids, v) == 1);
    for (long j = 0; j < V; ++j) z[j] = NAN;  /* an all-NaN row pads with -1 */
    CHECK(oracle_topk(z, 1, V, K, ids, v) == 0);
    CHECK(ids[0] == -1 && isnan(v[0]));
    free(z); free(ids); free(v);
}

int main(void) {
    CHECK(oracle_max_threads() >= 1);
    conv_case(2, 9, 32, 4, 4, 1);
    conv_case(2, 9, 32, 4, 4, 0);   /* NULL history */
    conv_case(1, 1, 16, 1, 16, 0);  /* one tap, one position, one channel per group */
    conv_case(3, 2, 24, 8, 3, 1);   /* n < T: the history reaches every position */
    {
        double* x = vec(16);
        CHECK(oracle_dynconv(x, NULL, x, x, x, 1, 1, 16, 1, 3) == 1);  /* C % G != 0 */
        free(x);
    }
    select_case(2, 5, 24, 4, 8, 50);
    select_case(1, 1, 16, 3, 4, 10);  /* one position: no transitions */
    select_case(3, 4, 8, 1, 1, 7);    /* K = 1, R = 1 */
    topk_case(3, 40, 5);
    topk_case(1, 6, 6);               /* K = V */
    if (fails == 0) printf("oracle sanitize ok\n");
    return fails == 0 ? 0 : 1;
}
