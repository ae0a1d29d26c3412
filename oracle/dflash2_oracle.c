/*
 * DFlash2 draft-head oracle: plain, slow, fp64 CPU definitions of the hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code with the CUDA library.
 *
 * Source of every formula: ggml-org/llama.cpp pull request #27342,
 * "spec : add DFlash2 support (local convolution + candidate selector)",
 * section "Overview" (the two printed formulas), together with the tensor names
 * in the same thread's review ("selector_predecessor", "selector_successor",
 * "selector_hidden") and the codebook-size exchange further down that thread.
 *
 * Readings taken where the page is silent (each is also listed in the design
 * notes of the repository):
 *   - taps t = 0..T-1, tap t multiplies x[i-t] (causal, not flipped);
 *   - positions before the block come from a (T-1)-row history window, oldest
 *     row first, so hist row T-1+j holds position j for j = -(T-1)..-1; a NULL
 *     history means zeros;
 *   - groups are contiguous: g(c) = c / (C/G);
 *   - project(h) is a plain linear map u = h W^T with W stored [R, d];
 *   - predecessors of position i are the K candidates of position i-1, so the
 *     transitions of a block are i = 1..n-1;
 *   - unary is per (position, candidate slot);
 *   - the argmax keeps the lowest slot on ties (strict ">" scan).
 *
 * All arithmetic is IEEE double.  Inputs arrive as double arrays; callers that
 * model bf16 data round to bf16 before converting, so both sides read the same
 * values.  OpenMP only splits the outermost independent loop; it changes no
 * arithmetic and no summation order.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Grouped dynamic depthwise causal convolution (Overview, first formula):
 *   out[s,i,c] = sum_{t=0}^{T-1} (base[t,c] + delta[s,i,t,g(c)]) * x~[s,i-t,c]
 * with x~[s,j,c] = x[s,j,c] for j >= 0 and hist[s,T-1+j,c] for j < 0.
 * Layouts (row-major): x, out [S,n,C]; hist [S,T-1,C] or NULL; base [T,C];
 * delta [S,n,T,G].  Returns 0, or 1 when C is not a multiple of G.
 */
int oracle_dynconv(const double* x, const double* hist, const double* base,
                   const double* delta, double* out,
                   long S, long n, long C, long T, long G) {
    if (C % G != 0) return 1;
    const long cg = C / G;
    long si;
#pragma omp parallel for schedule(static)
    for (si = 0; si < S * n; ++si) {
        const long s = si / n, i = si % n;
        for (long c = 0; c < C; ++c) {
            const long g = c / cg;
            double acc = 0.0;
            for (long t = 0; t < T; ++t) {
                const long j = i - t;
                double xv;
                if (j >= 0)
                    xv = x[(s * n + j) * C + c];
                else if (hist != NULL)
                    xv = hist[(s * (T - 1) + (T - 1 + j)) * C + c];
                else
                    xv = 0.0;
                const double w = base[t * C + c] + delta[((s * n + i) * T + t) * G + g];
                acc += w * xv;
            }
            out[(s * n + i) * C + c] = acc;
        }
    }
    return 0;
}

/*
 * project(h): the dense d -> R map of each position's hidden state ("This
 * position's hidden is projected ... to the same rank"; weight tensor
 * "selector_hidden").  u[r,k] = sum_j h[r,j] * W[k,j].
 * Layouts: h [P,d], W [R,d], u [P,R].
 */
void oracle_project(const double* h, const double* W, double* u,
                    long P, long d, long R) {
    long r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < P; ++r) {
        for (long k = 0; k < R; ++k) {
            double acc = 0.0;
            for (long j = 0; j < d; ++j) acc += h[r * d + j] * W[k * d + j];
            u[r * R + k] = acc;
        }
    }
}

/*
 * Edge scores and the per-predecessor argmax (Overview, second formula):
 *   edge(p -> c) = < A[p] (.) project(h), B[c] > + unary[c]
 * For sequence s and position i in 1..n-1, predecessor slot p and candidate
 * slot c:
 *   e[s,i-1,p,c] = sum_r A[id_p,r] * u[s*n+i,r] * B[id_c,r] + unary[s,i,c],
 *   id_p = cand_ids[s,i-1,p], id_c = cand_ids[s,i,c].
 * The readout for (s,i-1,p) is the lowest slot c reaching max_c e, and that max.
 * Layouts: cand_ids, unary [S,n,K]; u [S*n,R]; A, B [V,R];
 * edges [S,n-1,K,K] or NULL; best_slot, best_score [S,n-1,K].
 * Returns 0, or 1 if any candidate id lies outside [0,V) (nothing written for
 * that transition's rows beyond what was computed before the check).
 */
int oracle_edges(const int32_t* cand_ids, const double* u, const double* A,
                 const double* B, const double* unary,
                 long S, long n, long K, long R, long V,
                 double* edges, int32_t* best_slot, double* best_score) {
    for (long q = 0; q < S * n * K; ++q)
        if (cand_ids[q] < 0 || (long)cand_ids[q] >= V) return 1;
    if (n < 2) return 0;
    const long E = n - 1;
    long se;
#pragma omp parallel for schedule(static)
    for (se = 0; se < S * E; ++se) {
        const long s = se / E, i = se % E + 1;
        const double* urow = u + (s * n + i) * R;
        for (long p = 0; p < K; ++p) {
            const long idp = cand_ids[(s * n + i - 1) * K + p];
            double best = 0.0;
            int32_t arg = 0;
            for (long c = 0; c < K; ++c) {
                const long idc = cand_ids[(s * n + i) * K + c];
                double acc = 0.0;
                for (long r = 0; r < R; ++r)
                    acc += A[idp * R + r] * urow[r] * B[idc * R + r];
                const double e = acc + unary[(s * n + i) * K + c];
                if (edges != NULL) edges[((s * E + (i - 1)) * K + p) * K + c] = e;
                if (c == 0 || e > best) {
                    best = e;
                    arg = (int32_t)c;
                }
            }
            best_slot[(s * E + (i - 1)) * K + p] = arg;
            best_score[(s * E + (i - 1)) * K + p] = best;
        }
    }
    return 0;
}

/* The composite selector: project every position's hidden state, then score
 * the edges and read out the argmax.  u [S*n,R] receives the projection. */
int oracle_select(const double* h, const double* W, const int32_t* cand_ids,
                  const double* A, const double* B, const double* unary,
                  long S, long n, long d, long K, long R, long V,
                  double* u, double* edges, int32_t* best_slot, double* best_score) {
    oracle_project(h, W, u, S * n, d, R);
    return oracle_edges(cand_ids, u, A, B, unary, S, n, K, R, V, edges, best_slot,
                        best_score);
}

/*
 * Top-K candidate extraction, the step before the selector (the pull request's
 * review thread: the selector works on the top K of V-wide rows with small K).
 * Reading taken: for row r of draft logits z[r, 0..V-1], ids[r, 0..K-1] are the
 * K indices with the largest values, in descending order of value, equal
 * values ordered by ascending index; vals[r, k] = z[r, ids[r, k]] (the
 * draft's own score of that candidate).  K rounds of a full scan for the best
 * element not yet taken.  Degenerate inputs (the text says nothing of them):
 * a NaN entry is never a candidate, and when a row holds fewer than K entries
 * that are not NaN the remaining slots get id -1 and value NaN; -0 and +0 are
 * equal (the lower index comes first), as the comparison below already gives.
 * Returns 0, or 1 if K > V or K < 1 (or no memory).
 */
int oracle_topk(const double* z, long rows, long V, long K, int32_t* ids, double* vals) {
    if (K < 1 || K > V) return 1;
    int fail = 0;
    long r;
#pragma omp parallel for schedule(static) reduction(| : fail)
    for (r = 0; r < rows; ++r) {
        const double* zr = z + r * V;
        unsigned char* taken = (unsigned char*)calloc((size_t)V, 1);
        if (taken == NULL) {
            fail = 1;
            continue;
        }
        for (long k = 0; k < K; ++k) {
            long best = -1;
            for (long j = 0; j < V; ++j) {
                if (taken[j] || isnan(zr[j])) continue;
                if (best < 0 || zr[j] > zr[best]) best = j;  /* strict: lower index wins ties */
            }
            if (best < 0) {
                ids[r * K + k] = -1;
                vals[r * K + k] = NAN;
                continue;
            }
            taken[best] = 1;
            ids[r * K + k] = (int32_t)best;
            vals[r * K + k] = zr[best];
        }
        free(taken);
    }
    return fail;
}

/*
 * Greedy chain readout with a p_min cut, the step after the selector (the
 * pull request names "selector + p_min" as the DFlash2 draft path but gives no
 * formula; readings taken here):
 *   slot_0 = start_slot[s] if given (>= 0), else the argmax over k of
 *            unary[s,0,k] (lowest k on ties);
 *   slot_i = best_slot[s,i-1,slot_{i-1}]  (each predecessor's argmax candidate);
 *   p_0 = softmax_k(unary[s,0,:])[slot_0];
 *   p_i = softmax_c(edges[s,i-1,slot_{i-1},:])[slot_i], the chosen candidate's
 *         share among the K scores leaving the chosen predecessor;
 *   tokens[s,i] = cand_ids[s,i,slot_i];
 *   length[s] = the number of leading positions with p_i >= p_min.
 * The softmax is taken about the row maximum (exp(x - max) / sum exp(y - max)).
 * Returns 0, or 1 if a slot falls outside [0, K).
 */
int oracle_chain(const int32_t* cand_ids, const double* unary, const double* edges,
                 const int32_t* best_slot, const int32_t* start_slot, long S, long n, long K,
                 double p_min, int32_t* tokens, double* probs, int32_t* length) {
    int bad = 0;
    long s;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (s = 0; s < S; ++s) {
        const double* u0 = unary + (s * n) * K;
        long slot = start_slot != NULL ? start_slot[s] : -1;
        if (slot < 0) {
            slot = 0;
            for (long k = 1; k < K; ++k)
                if (u0[k] > u0[slot]) slot = k;
        }
        if (slot >= K) { bad = 1; continue; }
        double mx = u0[0];
        for (long k = 1; k < K; ++k) if (u0[k] > mx) mx = u0[k];
        double z = 0.0;
        for (long k = 0; k < K; ++k) z += exp(u0[k] - mx);
        double p = exp(u0[slot] - mx) / z;
        int32_t len = 0;
        int open = 1;
        for (long i = 0; i < n; ++i) {
            if (i > 0) {
                const double* row = edges + (((s * (n - 1) + (i - 1)) * K) + slot) * K;
                const long next = best_slot[(s * (n - 1) + (i - 1)) * K + slot];
                if (next < 0 || next >= K) { bad = 1; break; }
                double m2 = row[0];
                for (long c = 1; c < K; ++c) if (row[c] > m2) m2 = row[c];
                double z2 = 0.0;
                for (long c = 0; c < K; ++c) z2 += exp(row[c] - m2);
                p = exp(row[next] - m2) / z2;
                slot = next;
            }
            tokens[s * n + i] = cand_ids[(s * n + i) * K + slot];
            probs[s * n + i] = p;
            if (open && p >= p_min) ++len; else open = 0;
        }
        length[s] = len;
    }
    return bad;
}
