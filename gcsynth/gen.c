/*
 * Seeded synthetic inputs for the grammar-compressed right product.
 *
 * This file makes matrices and graphs; it holds none of the product's
 * arithmetic (no encoding, no grammar, no evaluation). Both the CUDA path
 * and the CPU oracle read what it writes.
 *
 * Random numbers come from a counter-based hash: every draw is a pure
 * function of (seed, stream, i, j), so any row block can be regenerated on
 * its own, in any order and on any number of threads, with the same result.
 * The hash is the SplitMix64 output function (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014), applied to
 * an incremented state.
 *
 * Genotype model (founder mosaic). Stated here because the pages simulate
 * their panels with msprime and give no generator of their own:
 *   p_j           = 0.05 + 0.45 * U(FREQ; j)                 allele frequency
 *   A[f][j]       = U(ALLELE; f, j) < p_j                    founder allele
 *   founder(h,0)  = floor(F * U(START; h))
 *   founder(h,j)  = floor(F * U(PICK; h, j)) if switch(h,j) else founder(h,j-1)
 *   switch(h,j)   = lo32(H(SWMUT; h, j)) < s * 2^32           (j >= 1)
 *   hap(h,j)      = A[founder(h,j)][j] XOR (hi32(H(SWMUT; h, j)) < mu * 2^32)
 *   G[i][j]       = hap(2i, j) + hap(2i+1, j)                in {0,1,2}
 *
 * Copy-model graph: nodes 0..n0-1 draw d0 uniform targets in [0,N); node
 * i >= n0 copies the (final) list of a uniform prototype in [0,i), replaces
 * each entry with probability p_edit by a uniform target, then sorts and
 * removes duplicates. Row i of the adjacency is node i's out-list.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { S_FREQ = 1, S_ALLELE = 2, S_START = 3, S_PICK = 4, S_SWMUT = 5,
       S_PROTO = 6, S_EDIT = 7, S_TARGET = 8, S_SOURCE = 9 };

static inline uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* key for (seed, stream, a): one hash per extra coordinate */
static inline uint64_t key2(uint64_t seed, uint64_t stream, uint64_t a) {
    return sm64(sm64(seed ^ (stream * 0xD1B54A32D192ED03ull)) ^ a);
}
static inline uint64_t hash3(uint64_t seed, uint64_t stream, uint64_t a, uint64_t b) {
    return sm64(key2(seed, stream, a) ^ b);
}
static inline double unit53(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

/* uniform integer in [0, n) from a 64-bit hash (multiply-shift, n < 2^32) */
static inline uint32_t below(uint64_t h, uint32_t n) {
    return (uint32_t)(((h >> 32) * (uint64_t)n) >> 32);
}

uint64_t gcs_hash3(uint64_t seed, uint64_t stream, uint64_t a, uint64_t b) {
    return hash3(seed, stream, a, b);
}

/* founder alleles A[F][m] as bytes (0/1) */
static void founders(int64_t m, int32_t F, uint64_t seed, uint8_t* A) {
    double* p = (double*)malloc(sizeof(double) * (size_t)m);
    for (int64_t j = 0; j < m; ++j) p[j] = 0.05 + 0.45 * unit53(hash3(seed, S_FREQ, (uint64_t)j, 0));
#pragma omp parallel for schedule(static)
    for (int32_t f = 0; f < F; ++f) {
        uint64_t k = key2(seed, S_ALLELE, (uint64_t)f);
        for (int64_t j = 0; j < m; ++j) A[(int64_t)f * m + j] = unit53(sm64(k ^ (uint64_t)j)) < p[j];
    }
    free(p);
}

static void haplotype(int64_t h, int64_t m, int32_t F, uint64_t thr_s, uint64_t thr_mu,
                      uint64_t seed, const uint8_t* A, uint8_t* out) {
    uint32_t f = below(hash3(seed, S_START, (uint64_t)h, 0), (uint32_t)F);
    uint64_t ksw = key2(seed, S_SWMUT, (uint64_t)h);
    uint64_t kpk = key2(seed, S_PICK, (uint64_t)h);
    for (int64_t j = 0; j < m; ++j) {
        uint64_t r = sm64(ksw ^ (uint64_t)j);
        if (j > 0 && (r & 0xffffffffull) < thr_s) f = below(sm64(kpk ^ (uint64_t)j), (uint32_t)F);
        out[j] = (uint8_t)(A[(int64_t)f * m + j] ^ ((r >> 32) < thr_mu));
    }
}

/*
 * Dense genotype rows [r0, r1) into out[(r1-r0) * m]. Returns 0, or -1 on bad
 * arguments / allocation failure.
 */
int gcs_genotype_dense(int64_t m, int32_t F, double s, double mu, uint64_t seed,
                       int64_t r0, int64_t r1, uint8_t* out) {
    if (m <= 0 || F <= 0 || r1 < r0 || s < 0 || s > 1 || mu < 0 || mu > 1) return -1;
    uint8_t* A = (uint8_t*)malloc((size_t)F * (size_t)m);
    if (!A) return -1;
    founders(m, F, seed, A);
    uint64_t thr_s = (uint64_t)(s * 4294967296.0), thr_mu = (uint64_t)(mu * 4294967296.0);
    int err = 0;
#pragma omp parallel
    {
        uint8_t* hb = (uint8_t*)malloc((size_t)m);
        if (!hb) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t i = r0; i < r1; ++i) {
                uint8_t* row = out + (i - r0) * m;
                haplotype(2 * i, m, F, thr_s, thr_mu, seed, A, row);
                haplotype(2 * i + 1, m, F, thr_s, thr_mu, seed, A, hb);
                for (int64_t j = 0; j < m; ++j) row[j] = (uint8_t)(row[j] + hb[j]);
            }
            free(hb);
        }
    }
    free(A);
    return err ? -1 : 0;
}

/*
 * Genotype rows [r0, r1) straight to CSR in two passes over the same draws.
 * Pass 1 (row_ptr == NULL): writes per-row non-zero counts into nnz[r1-r0].
 * Pass 2: row_ptr[0..r1-r0] (absolute offsets into col/val, any base) given;
 * writes col (int32) and val (float, 1 or 2).
 */
int gcs_genotype_csr(int64_t m, int32_t F, double s, double mu, uint64_t seed,
                     int64_t r0, int64_t r1, int64_t* nnz, const int64_t* row_ptr,
                     int32_t* col, float* val) {
    if (m <= 0 || F <= 0 || r1 < r0 || s < 0 || s > 1 || mu < 0 || mu > 1) return -1;
    uint8_t* A = (uint8_t*)malloc((size_t)F * (size_t)m);
    if (!A) return -1;
    founders(m, F, seed, A);
    uint64_t thr_s = (uint64_t)(s * 4294967296.0), thr_mu = (uint64_t)(mu * 4294967296.0);
    int err = 0;
    int64_t base = row_ptr ? row_ptr[0] : 0;
#pragma omp parallel
    {
        uint8_t* ha = (uint8_t*)malloc((size_t)m);
        uint8_t* hb = (uint8_t*)malloc((size_t)m);
        if (!ha || !hb) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t i = r0; i < r1; ++i) {
                haplotype(2 * i, m, F, thr_s, thr_mu, seed, A, ha);
                haplotype(2 * i + 1, m, F, thr_s, thr_mu, seed, A, hb);
                if (!row_ptr) {
                    int64_t c = 0;
                    for (int64_t j = 0; j < m; ++j) c += (ha[j] | hb[j]) != 0;
                    nnz[i - r0] = c;
                } else {
                    int64_t o = row_ptr[i - r0] - base;
                    for (int64_t j = 0; j < m; ++j) {
                        uint8_t g = (uint8_t)(ha[j] + hb[j]);
                        if (g) { col[o] = (int32_t)j; val[o] = (float)g; ++o; }
                    }
                }
            }
        }
        free(ha);
        free(hb);
    }
    free(A);
    return err ? -1 : 0;
}

/* per-row non-zero counts of a dense u8 block */
void gcs_dense_row_nnz(const uint8_t* d, int64_t rows, int64_t m, int64_t* nnz) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        const uint8_t* r = d + i * m;
        int64_t c = 0;
        for (int64_t j = 0; j < m; ++j) c += r[j] != 0;
        nnz[i] = c;
    }
}

/* CSR fill from a dense u8 block; row_ptr[0..rows] (absolute, any base) */
void gcs_dense_to_csr(const uint8_t* d, int64_t rows, int64_t m, const int64_t* row_ptr,
                      int32_t* col, float* val) {
    int64_t base = row_ptr[0];
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < rows; ++i) {
        const uint8_t* r = d + i * m;
        int64_t o = row_ptr[i] - base;
        for (int64_t j = 0; j < m; ++j)
            if (r[j]) { col[o] = (int32_t)j; val[o] = (float)r[j]; ++o; }
    }
}

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/*
 * Copy-model graph (sequential by construction: a node copies an earlier
 * node's final list). col must hold N*d0 entries; row_ptr N+1. Returns the
 * edge count, or -1 on bad arguments.
 */
int64_t gcs_copy_model(int32_t N, int32_t n0, int32_t d0, double p_edit, uint64_t seed,
                       int64_t* row_ptr, int32_t* col) {
    if (N <= 0 || n0 <= 0 || n0 > N || d0 <= 0 || p_edit < 0 || p_edit > 1) return -1;
    uint64_t thr = (uint64_t)(p_edit * 4294967296.0);
    int32_t* tmp = (int32_t*)malloc(sizeof(int32_t) * (size_t)d0);
    if (!tmp) return -1;
    int64_t e = 0;
    row_ptr[0] = 0;
    for (int32_t i = 0; i < N; ++i) {
        int32_t len;
        if (i < n0) {
            for (int32_t t = 0; t < d0; ++t) tmp[t] = (int32_t)below(hash3(seed, S_TARGET, (uint64_t)i, (uint64_t)t), (uint32_t)N);
            len = d0;
        } else {
            int32_t pr = (int32_t)below(hash3(seed, S_PROTO, (uint64_t)i, 0), (uint32_t)i);
            len = (int32_t)(row_ptr[pr + 1] - row_ptr[pr]);
            uint64_t ke = key2(seed, S_EDIT, (uint64_t)i);
            for (int32_t t = 0; t < len; ++t) {
                uint64_t r = sm64(ke ^ (uint64_t)t);
                tmp[t] = ((r & 0xffffffffull) < thr) ? (int32_t)below(hash3(seed, S_TARGET, (uint64_t)i, (uint64_t)t), (uint32_t)N)
                                                      : col[row_ptr[pr] + t];
            }
        }
        qsort(tmp, (size_t)len, sizeof(int32_t), cmp_i32);
        int32_t w = 0;
        for (int32_t t = 0; t < len; ++t)
            if (w == 0 || tmp[t] != tmp[w - 1]) tmp[w++] = tmp[t];
        memcpy(col + e, tmp, sizeof(int32_t) * (size_t)w);
        e += w;
        row_ptr[i + 1] = e;
    }
    free(tmp);
    return e;
}

/* 64 (or fewer) distinct uniform source nodes in [0, N) */
int gcs_sources(int32_t N, int32_t count, uint64_t seed, int32_t* out) {
    if (count < 0 || count > N) return -1;
    int32_t got = 0;
    for (uint64_t t = 0; got < count; ++t) {
        int32_t v = (int32_t)below(hash3(seed, S_SOURCE, t, 0), (uint32_t)N);
        int dup = 0;
        for (int32_t q = 0; q < got; ++q) dup |= out[q] == v;
        if (!dup) out[got++] = v;
    }
    return 0;
}
