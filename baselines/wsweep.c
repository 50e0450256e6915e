/*
 * CPU grammar sweep: Theorem 2.3's W-array evaluation of y = M x over the raw
 * RePair grammar (rules R in creation order, the final sequence C), in
 * float64. A CPU baseline, reported beside the GPU figures; TEST
 * INFRASTRUCTURE like the rest of this directory, never on the product path.
 *
 *   W[i] = cv(A_i) + cv(B_i)          cv(N_j) = W[j], cv(<l, j>) = V[l] * x[j]
 *   y[r] = sum of cv over row r's symbols of C, in order   (Lemma 2.2)
 *
 * Symbols: s >= 0 is rule N_s, s < 0 is terminal -s-1 (the library's exported
 * encoding). With threads > 1 the rules of one Eq. 3.1 level run in parallel
 * (a level's rules read only lower levels, Lemma 3.1), levels in order, and
 * the rows in parallel; every value is computed by the same additions in the
 * same order either way, so y does not depend on the thread count.
 */
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double cv(int32_t s, const double* W, const double* T) { return s >= 0 ? W[s] : T[-(int64_t)s - 1]; }

/* level_off[k] .. level_off[k+1]: positions in by_level of the rules of level k + 1 */
int ws_sweep(int64_t n_rules, const int32_t* rule_a, const int32_t* rule_b, const int64_t* level_off,
             const int32_t* by_level, int64_t depth, int64_t n, const int64_t* c_off, const int32_t* c_sym,
             int64_t n_terms, const int32_t* term_col, const int32_t* term_vidx, const double* V, const double* x,
             double* y, double* W, double* T, int threads) {
    if (threads < 1) return -1;
#ifdef _OPENMP
    omp_set_num_threads(threads);
#endif
    for (int64_t p = 0; p < n_terms; ++p) T[p] = V[term_vidx[p]] * x[term_col[p]];
    if (threads == 1) {
        for (int64_t i = 0; i < n_rules; ++i) W[i] = cv(rule_a[i], W, T) + cv(rule_b[i], W, T);
    } else {
        for (int64_t k = 0; k < depth; ++k) {
            const int64_t lo = level_off[k], hi = level_off[k + 1];
#pragma omp parallel for schedule(static) if (threads > 1)
            for (int64_t q = lo; q < hi; ++q) {
                const int32_t i = by_level[q];
                W[i] = cv(rule_a[i], W, T) + cv(rule_b[i], W, T);
            }
        }
    }
#pragma omp parallel for schedule(dynamic, 64) if (threads > 1)
    for (int64_t r = 0; r < n; ++r) {
        double acc = 0.0;
        for (int64_t q = c_off[r]; q < c_off[r + 1]; ++q) acc += cv(c_sym[q], W, T);
        y[r] = acc;
    }
    return 0;
}

/*
 * The same product from the uncompressed CSR matrix, float64: y[i] = sum of
 * val[e] * x[col[e]] over row i, rows in parallel. The CSR CPU baseline
 * (the direct product of Sec. 2, on every host core).
 */
int ws_csr(int64_t n, const int64_t* row_ptr, const int32_t* col, const float* val, const double* x, double* y,
           int threads) {
    if (threads < 1) return -1;
#ifdef _OPENMP
    omp_set_num_threads(threads);
#endif
#pragma omp parallel for schedule(dynamic, 16) if (threads > 1)
    for (int64_t i = 0; i < n; ++i) {
        double acc = 0.0;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) acc += (double)val[e] * x[col[e]];
        y[i] = acc;
    }
    return 0;
}
