// CSRV encoding (Sec. 2 "CSRV" of the pages, Eqs. 2.1-2.2): the distinct
// non-zero values of M form V (ascending), every stored non-zero M[i][j] =
// V[l] becomes the terminal <l, j>, and each row is the string of its
// terminals in column order. Terminals are numbered by (column, value index),
// so a terminal's id order is also its column order.
#include <cmath>
#include <cstring>
#include <numeric>

#include "common.hpp"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace gcs {
namespace {

inline uint32_t float_bits(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}

inline bool is_zero_bits(uint32_t u) { return (u & 0x7fffffffu) == 0; }

// Small open-addressing map from a float's bit pattern to an index.
struct BitsMap {
    std::vector<uint32_t> key;
    std::vector<int32_t> idx;
    size_t mask = 0, count = 0;
    explicit BitsMap(size_t cap = 64) { reset(cap); }
    void reset(size_t cap) {
        size_t c = 16;
        while (c < cap * 2) c <<= 1;
        key.assign(c, 0);
        idx.assign(c, -1);
        mask = c - 1;
        count = 0;
    }
    static size_t h(uint32_t k) { return (size_t)((k * 0x9E3779B1u) ^ (k >> 16)); }
    int32_t find(uint32_t k) const {
        for (size_t p = h(k) & mask;; p = (p + 1) & mask) {
            if (idx[p] < 0) return -1;
            if (key[p] == k) return idx[p];
        }
    }
    void insert(uint32_t k, int32_t v) {
        if ((count + 1) * 2 > key.size()) {
            std::vector<uint32_t> ok = key;
            std::vector<int32_t> oi = idx;
            reset(key.size());
            for (size_t p = 0; p < ok.size(); ++p)
                if (oi[p] >= 0) insert(ok[p], oi[p]);
        }
        size_t p = h(k) & mask;
        while (idx[p] >= 0 && key[p] != k) p = (p + 1) & mask;
        if (idx[p] < 0) ++count;
        key[p] = k;
        idx[p] = v;
    }
};

}  // namespace

Csrv csrv_encode(int64_t n, int64_t m, const int64_t* row_ptr, const int32_t* col,
                 const float* val, int threads) {
    if (n < 0 || m < 0) fail(GC_ERR_ARG, "negative matrix shape");
    if (m > INT32_MAX) fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 columns");
    if (!row_ptr) fail(GC_ERR_ARG, "row_ptr is NULL");
    if (row_ptr[0] != 0) fail(GC_ERR_ARG, "row_ptr[0] must be 0");
    for (int64_t i = 0; i < n; ++i)
        if (row_ptr[i + 1] < row_ptr[i]) fail(GC_ERR_ARG, "row_ptr must be non-decreasing");
    const int64_t nnz_in = row_ptr[n];
    if (nnz_in > 0 && !col) fail(GC_ERR_ARG, "col is NULL");
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#else
    threads = 1;
#endif

    Csrv s;
    s.n = n;
    s.m = m;

    // 1. value dictionary: distinct non-zero bit patterns, finite only
    BitsMap vmap(64);
    std::vector<uint32_t> vbits;
    if (val) {
        uint32_t last = 0;
        bool have_last = false;
        for (int64_t e = 0; e < nnz_in; ++e) {
            uint32_t u = float_bits(val[e]);
            if (have_last && u == last) continue;
            if (is_zero_bits(u)) continue;
            if (!std::isfinite(val[e])) fail(GC_ERR_ARG, "matrix value is NaN or infinite");
            if (vmap.find(u) < 0) {
                if (vbits.size() >= (size_t)INT32_MAX) fail(GC_ERR_UNSUPPORTED, "too many distinct values");
                vmap.insert(u, (int32_t)vbits.size());
                vbits.push_back(u);
            }
            last = u;
            have_last = true;
        }
    } else if (nnz_in > 0) {
        vbits.push_back(float_bits(1.0f));
    }
    std::vector<float> vals(vbits.size());
    for (size_t i = 0; i < vbits.size(); ++i) std::memcpy(&vals[i], &vbits[i], 4);
    std::vector<int32_t> order(vals.size());
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return vals[a] < vals[b]; });
    s.V.resize(vals.size());
    BitsMap rank((size_t)std::max<size_t>(vals.size(), 16));
    for (size_t r = 0; r < order.size(); ++r) {
        s.V[r] = vals[order[r]];
        rank.insert(vbits[order[r]], (int32_t)r);
    }
    const int64_t nv = (int64_t)s.V.size();

    // 2. per-entry value index (-1 for a stored zero), column bounds
    std::vector<int32_t> vidx((size_t)nnz_in);
    int bad_col = 0;
#pragma omp parallel for num_threads(threads) schedule(static) reduction(| : bad_col)
    for (int64_t e = 0; e < nnz_in; ++e) {
        if (col[e] < 0 || col[e] >= m) bad_col = 1;
        if (!val) {
            vidx[e] = 0;
        } else {
            uint32_t u = float_bits(val[e]);
            vidx[e] = is_zero_bits(u) ? -1 : rank.find(u);
        }
    }
    if (bad_col) fail(GC_ERR_ARG, "column index out of range");

    // 3. rows: drop zeros, order by column, reject repeated columns
    s.row_off.assign((size_t)n + 1, 0);
    for (int64_t i = 0; i < n; ++i) {
        int64_t c = 0;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) c += vidx[e] >= 0;
        s.row_off[i + 1] = s.row_off[i] + c;
    }
    const int64_t nnz = s.row_off[n];
    std::vector<int32_t> rcol((size_t)nnz), rvid((size_t)nnz);
    int dup = 0;
#pragma omp parallel for num_threads(threads) schedule(dynamic, 64) reduction(| : dup)
    for (int64_t i = 0; i < n; ++i) {
        int64_t o = s.row_off[i];
        bool sorted = true;
        int32_t prev = -1;
        for (int64_t e = row_ptr[i]; e < row_ptr[i + 1]; ++e) {
            if (vidx[e] < 0) continue;
            if (col[e] <= prev) sorted = false;
            prev = col[e];
            rcol[o] = col[e];
            rvid[o] = vidx[e];
            ++o;
        }
        if (!sorted) {
            int64_t a = s.row_off[i], b = s.row_off[i + 1];
            std::vector<std::pair<int32_t, int32_t>> tmp;
            tmp.reserve((size_t)(b - a));
            for (int64_t q = a; q < b; ++q) tmp.emplace_back(rcol[q], rvid[q]);
            std::sort(tmp.begin(), tmp.end());
            for (int64_t q = a; q < b; ++q) {
                rcol[q] = tmp[q - a].first;
                rvid[q] = tmp[q - a].second;
                if (q > a && rcol[q] == rcol[q - 1]) dup = 1;
            }
        }
    }
    if (dup) fail(GC_ERR_ARG, "a row repeats a column");

    // 4. terminal table sorted by (col, vidx) and the terminal id of each entry
    s.sym.resize((size_t)nnz);
    if (nv <= 64) {
        std::vector<uint64_t> mask((size_t)m, 0);
        for (int64_t e = 0; e < nnz; ++e) mask[rcol[e]] |= 1ull << rvid[e];
        std::vector<int64_t> base((size_t)m + 1, 0);
        for (int64_t j = 0; j < m; ++j) base[j + 1] = base[j] + __builtin_popcountll(mask[j]);
        if (base[m] > INT32_MAX - 2) fail(GC_ERR_UNSUPPORTED, "more than 2^31-3 distinct terminals");
        s.term_col.resize((size_t)base[m]);
        s.term_vidx.resize((size_t)base[m]);
        for (int64_t j = 0; j < m; ++j) {
            int64_t t = base[j];
            for (uint64_t w = mask[j]; w; w &= w - 1) {
                s.term_col[t] = (int32_t)j;
                s.term_vidx[t] = __builtin_ctzll(w);
                ++t;
            }
        }
#pragma omp parallel for num_threads(threads) schedule(static)
        for (int64_t e = 0; e < nnz; ++e) {
            uint64_t below = mask[rcol[e]] & ((1ull << rvid[e]) - 1ull);
            s.sym[e] = (int32_t)(base[rcol[e]] + __builtin_popcountll(below));
        }
    } else {
        std::vector<uint64_t> keys((size_t)nnz);
        for (int64_t e = 0; e < nnz; ++e) keys[e] = ((uint64_t)(uint32_t)rcol[e] << 32) | (uint32_t)rvid[e];
        std::vector<uint64_t> uk = keys;
        std::sort(uk.begin(), uk.end());
        uk.erase(std::unique(uk.begin(), uk.end()), uk.end());
        if ((int64_t)uk.size() > INT32_MAX - 2) fail(GC_ERR_UNSUPPORTED, "more than 2^31-3 distinct terminals");
        s.term_col.resize(uk.size());
        s.term_vidx.resize(uk.size());
        for (size_t t = 0; t < uk.size(); ++t) {
            s.term_col[t] = (int32_t)(uk[t] >> 32);
            s.term_vidx[t] = (int32_t)(uk[t] & 0xffffffffu);
        }
#pragma omp parallel for num_threads(threads) schedule(static)
        for (int64_t e = 0; e < nnz; ++e)
            s.sym[e] = (int32_t)(std::lower_bound(uk.begin(), uk.end(), keys[e]) - uk.begin());
    }
    return s;
}

}  // namespace gcs
