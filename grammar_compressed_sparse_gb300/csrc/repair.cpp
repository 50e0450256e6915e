// RePair with row boundaries (Sec. 2 "Grammar" and Sec. 4.1 of the pages):
// repeatedly replace the most frequent pair of adjacent symbols by a new
// nonterminal N_i -> A_i B_i, never pairing across a row end, and stop when
// no pair occurs twice. Rules are numbered in creation order, so every child
// precedes its parent (the topological numbering of Eq. 2.3).
//
// Data structures (after Larsson and Moffat's linear-time RePair):
//   seq/nxt/prv      the working sequence with links over live positions;
//                    a row end is a DELIM position, a replaced right symbol
//                    becomes EMPTY and is unlinked
//   pid[i]           id of the pair that starts at live position i (or -1)
//   onext/oprev      each pair's occurrences, threaded through positions
//   pair records     (a, b, freq, first occurrence, bucket links)
//   buckets          frequency buckets 2..B plus one unsorted list above B
// Because a row never holds the same symbol twice (its symbols cover disjoint
// column ranges), occurrences never overlap. Every pair created while
// replacing (a, b) by N contains N, so new pairs are found through two small
// per-round maps keyed by the neighbour symbol; no global pair hash is needed
// after the initial count, and decrements go through pid[].
#include <cstring>
#include <numeric>

#include "common.hpp"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace gcs {
namespace {

constexpr int32_t DELIM = -1;
constexpr int32_t EMPTY = -2;

// int32 -> int32 map cleared in O(1) by a generation stamp.
struct StampMap {
    std::vector<int32_t> key, val, stamp;
    int32_t gen = 1;
    size_t mask = 0;
    void prepare(size_t expected) {
        size_t c = 64;
        while (c < expected * 2) c <<= 1;
        if (c > key.size()) {
            key.assign(c, 0);
            val.assign(c, 0);
            stamp.assign(c, 0);
            mask = c - 1;
            gen = 1;
        } else if (++gen == INT32_MAX) {
            std::fill(stamp.begin(), stamp.end(), 0);
            gen = 1;
        }
    }
    // returns slot; found tells whether the key was present
    size_t slot(int32_t k, bool& found) {
        size_t p = ((uint32_t)k * 0x9E3779B1u) & mask;
        while (stamp[p] == gen) {
            if (key[p] == k) {
                found = true;
                return p;
            }
            p = (p + 1) & mask;
        }
        found = false;
        return p;
    }
    void put(size_t p, int32_t k, int32_t v) {
        stamp[p] = gen;
        key[p] = k;
        val[p] = v;
    }
};

class RePair {
public:
    RePair(const Csrv& s, int64_t r0, int64_t r1) : alpha_((int32_t)s.term_col.size()) {
        const int64_t nsym = s.row_off[r1] - s.row_off[r0];
        const int64_t ns = nsym + (r1 - r0);
        if (ns >= INT32_MAX - 1)
            fail(GC_ERR_UNSUPPORTED,
                 "a RePair block holds more than 2^31-2 symbols; compress in row blocks (block_rows)");
        ns_ = (int32_t)ns;
        rows_ = r1 - r0;
        seq_.resize(ns_);
        row_start_.resize((size_t)rows_);
        int64_t p = 0;
        for (int64_t r = r0; r < r1; ++r) {
            row_start_[r - r0] = (int32_t)p;
            for (int64_t e = s.row_off[r]; e < s.row_off[r + 1]; ++e) seq_[p++] = s.sym[e];
            seq_[p++] = DELIM;
        }
        nxt_.resize(ns_);
        prv_.resize(ns_);
        for (int32_t i = 0; i < ns_; ++i) {
            nxt_[i] = i + 1;
            prv_[i] = i - 1;
        }
        pid_.assign(ns_, -1);
        onext_.assign(ns_, -1);
        oprev_.assign(ns_, -1);
        int64_t b = 2;
        while (b * b < ns) ++b;
        B_ = (int32_t)std::max<int64_t>(b, 2);
        bucket_.assign((size_t)B_ + 2, -1);
        btail_.assign((size_t)B_ + 2, -1);
        maxb_ = 0;
    }

    Slp run() {
        count_initial_pairs();
        for (;;) {
            int32_t p = pop_max();
            if (p < 0) break;
            replace(p);
        }
        Slp out;
        out.rule_a.resize(ra_.size());
        out.rule_b.resize(rb_.size());
        for (size_t i = 0; i < ra_.size(); ++i) {
            out.rule_a[i] = to_export(ra_[i]);
            out.rule_b[i] = to_export(rb_[i]);
        }
        out.c_off.assign((size_t)rows_ + 1, 0);
        for (int64_t r = 0; r < rows_; ++r) {
            int64_t c = 0;
            for (int32_t q = row_start_[r]; seq_[q] != DELIM; q = nxt_[q]) ++c;
            out.c_off[r + 1] = out.c_off[r] + c;
        }
        out.c_sym.resize((size_t)out.c_off[rows_]);
        for (int64_t r = 0; r < rows_; ++r) {
            int64_t o = out.c_off[r];
            for (int32_t q = row_start_[r]; seq_[q] != DELIM; q = nxt_[q]) out.c_sym[o++] = to_export(seq_[q]);
        }
        return out;
    }

private:
    int32_t alpha_;
    int32_t ns_ = 0;
    int64_t rows_ = 0;
    std::vector<int32_t> seq_, nxt_, prv_, pid_, onext_, oprev_, row_start_;
    // pair records
    std::vector<int32_t> pa_, pb_, pf_, ph_, qp_, qn_, free_;
    // buckets
    int32_t B_ = 2, maxb_ = 0;
    std::vector<int32_t> bucket_, btail_, qb_;
    std::vector<int32_t> fresh_;   // pairs created in the current round
    // rules in internal symbols
    std::vector<int32_t> ra_, rb_;
    StampMap lmap_, rmap_;

    int32_t to_export(int32_t s) const { return s < alpha_ ? -(s + 1) : s - alpha_; }

    int32_t new_pair(int32_t a, int32_t b) {
        int32_t id;
        if (!free_.empty()) {
            id = free_.back();
            free_.pop_back();
            pa_[id] = a;
            pb_[id] = b;
            pf_[id] = 0;
            ph_[id] = -1;
            qp_[id] = qn_[id] = -1;
            qb_[id] = -1;
        } else {
            if (pa_.size() >= (size_t)INT32_MAX) fail(GC_ERR_UNSUPPORTED, "too many pairs");
            id = (int32_t)pa_.size();
            pa_.push_back(a);
            pb_.push_back(b);
            pf_.push_back(0);
            ph_.push_back(-1);
            qp_.push_back(-1);
            qn_.push_back(-1);
            qb_.push_back(-1);
        }
        fresh_.push_back(id);
        return id;
    }

    // ---- occurrence lists
    void occ_push(int32_t id, int32_t pos) {
        int32_t h = ph_[id];
        onext_[pos] = h;
        oprev_[pos] = -1;
        if (h >= 0) oprev_[h] = pos;
        ph_[id] = pos;
    }
    void occ_remove(int32_t id, int32_t pos) {
        int32_t a = oprev_[pos], b = onext_[pos];
        if (a >= 0) onext_[a] = b; else ph_[id] = b;
        if (b >= 0) oprev_[b] = a;
        onext_[pos] = oprev_[pos] = -1;
    }

    // ---- frequency buckets: FIFO queues per frequency 2..B, one list above B.
    // Ties between equally frequent pairs go to the oldest pair (the pages
    // leave the tie-break open). Older pairs hold shallower symbols, so over a
    // repeated segment this pairs neighbours level by level and keeps the
    // grammar's depth near log2 of the segment length; a newest-first order
    // instead grows left-deep chains.
    // Decrements are lazy: a pair stays in the bucket it was filed in (which
    // is then >= its frequency) and is re-filed when it reaches the front.
    // Increments only ever happen to the pairs created in the current round
    // (they all contain the new symbol); those are filed once, after it.
    int32_t list_of(int32_t f) const { return f > B_ ? B_ + 1 : f; }
    void pq_insert(int32_t id) {
        const int32_t l = list_of(pf_[id]);
        const int32_t t = btail_[l];
        qp_[id] = t;
        qn_[id] = -1;
        if (t >= 0) qn_[t] = id; else bucket_[l] = id;
        btail_[l] = id;
        qb_[id] = l;
        if (l <= B_ && l > maxb_) maxb_ = l;
    }
    void pq_unlink(int32_t id) {
        const int32_t l = qb_[id];
        const int32_t a = qp_[id], b = qn_[id];
        if (a >= 0) qn_[a] = b; else bucket_[l] = b;
        if (b >= 0) qp_[b] = a; else btail_[l] = a;
        qp_[id] = qn_[id] = -1;
        qb_[id] = -1;
    }
    // Takes id out of the queue; returns true if it is still a candidate.
    bool settle(int32_t id) {
        pq_unlink(id);
        if (pf_[id] >= 2) return true;
        if (pf_[id] == 0) free_.push_back(id);
        return false;
    }
    int32_t pop_max() {
        // above B: exact maximum by scan, re-filing entries that fell to <= B
        for (;;) {
            int32_t best = -1;
            for (int32_t q = bucket_[B_ + 1]; q >= 0;) {
                const int32_t nx = qn_[q];
                if (pf_[q] <= B_) {
                    if (settle(q)) pq_insert(q);
                } else if (best < 0 || pf_[q] > pf_[best]) {
                    best = q;
                }
                q = nx;
            }
            if (best >= 0) {
                pq_unlink(best);
                return best;
            }
            break;
        }
        for (;;) {
            while (maxb_ >= 2 && bucket_[maxb_] < 0) --maxb_;
            if (maxb_ < 2) return -1;
            const int32_t id = bucket_[maxb_];
            if (pf_[id] == maxb_) {
                pq_unlink(id);
                return id;
            }
            if (settle(id)) pq_insert(id);   // stale: frequency dropped since filing
        }
    }
    void inc(int32_t id, int32_t pos) {   // only pairs created in this round
        occ_push(id, pos);
        ++pf_[id];
    }
    void dec(int32_t id, int32_t pos) {
        occ_remove(id, pos);
        if (--pf_[id] == 0 && qb_[id] < 0) free_.push_back(id);
    }

    // Initial digram count, grouped by left symbol (parallel over groups).
    void count_initial_pairs() {
        const int32_t A = alpha_;
        std::vector<int64_t> cnt((size_t)A + 1, 0);
        for (int32_t i = 0; i + 1 < ns_; ++i)
            if (seq_[i] >= 0 && seq_[i + 1] >= 0) ++cnt[seq_[i] + 1];
        for (int32_t a = 0; a < A; ++a) cnt[a + 1] += cnt[a];
        std::vector<int32_t> grp((size_t)cnt[A]);
        {
            std::vector<int64_t> w(cnt.begin(), cnt.end() - 1);
            for (int32_t i = 0; i + 1 < ns_; ++i)
                if (seq_[i] >= 0 && seq_[i + 1] >= 0) grp[w[seq_[i]]++] = i;
        }
        // distinct right symbols per group -> local pair ids
        std::vector<int32_t> ndist((size_t)A + 1, 0);
#pragma omp parallel
        {
            StampMap m;
#pragma omp for schedule(dynamic, 256)
            for (int32_t a = 0; a < A; ++a) {
                const int64_t g0 = cnt[a], g1 = cnt[a + 1];
                if (g0 == g1) continue;
                m.prepare((size_t)(g1 - g0));
                int32_t d = 0;
                for (int64_t q = g0; q < g1; ++q) {
                    const int32_t pos = grp[q];
                    const int32_t bsym = seq_[pos + 1];
                    bool f;
                    size_t s = m.slot(bsym, f);
                    if (!f) m.put(s, bsym, d++);
                    pid_[pos] = m.val[s];
                }
                ndist[a + 1] = d;
            }
        }
        for (int32_t a = 0; a < A; ++a) ndist[a + 1] += ndist[a];
        const int32_t np = ndist[A];
        pa_.resize(np);
        pb_.resize(np);
        pf_.assign(np, 0);
        ph_.assign(np, -1);
        qp_.assign(np, -1);
        qn_.assign(np, -1);
        qb_.assign(np, -1);
        // global ids, records, occurrence lists (each group owns its positions)
#pragma omp parallel for schedule(dynamic, 256)
        for (int32_t a = 0; a < A; ++a) {
            for (int64_t q = cnt[a]; q < cnt[a + 1]; ++q) {
                int32_t pos = grp[q];
                int32_t id = ndist[a] + pid_[pos];
                pid_[pos] = id;
                pa_[id] = a;
                pb_[id] = seq_[pos + 1];
                ++pf_[id];
                int32_t h = ph_[id];
                onext_[pos] = h;
                if (h >= 0) oprev_[h] = pos;
                ph_[id] = pos;
            }
        }
        for (int32_t id = 0; id < np; ++id)
            if (pf_[id] >= 2) pq_insert(id);
    }

    void replace(int32_t p) {
        const int32_t a = pa_[p], b = pb_[p];
        if ((int64_t)alpha_ + (int64_t)ra_.size() >= INT32_MAX)
            fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 symbols");
        const int32_t N = alpha_ + (int32_t)ra_.size();
        ra_.push_back(a);
        rb_.push_back(b);
        lmap_.prepare((size_t)pf_[p]);
        rmap_.prepare((size_t)pf_[p]);
        fresh_.clear();
        while (ph_[p] >= 0) {
            const int32_t i = ph_[p];
            occ_remove(p, i);
            const int32_t j = nxt_[i];
            if (j >= ns_ || seq_[i] != a || seq_[j] != b) continue;   // cannot happen; defensive
            const int32_t xp = prv_[i];
            const int32_t yp = nxt_[j];
            const bool hx = xp >= 0 && seq_[xp] >= 0;
            const bool hy = yp < ns_ && seq_[yp] >= 0;
            if (hx) dec(pid_[xp], xp);
            if (hy) dec(pid_[j], j);
            seq_[i] = N;
            seq_[j] = EMPTY;
            pid_[j] = -1;
            nxt_[i] = yp;
            if (yp < ns_) prv_[yp] = i;
            if (hx) {
                const int32_t x = seq_[xp];
                bool f;
                size_t s = lmap_.slot(x, f);
                int32_t id;
                if (f) id = lmap_.val[s];
                else { id = new_pair(x, N); lmap_.put(s, x, id); }
                pid_[xp] = id;
                inc(id, xp);
            }
            if (hy) {
                const int32_t y = seq_[yp];
                bool f;
                size_t s = rmap_.slot(y, f);
                int32_t id;
                if (f) id = rmap_.val[s];
                else { id = new_pair(N, y); rmap_.put(s, y, id); }
                pid_[i] = id;
                inc(id, i);
            } else {
                pid_[i] = -1;
            }
        }
        pf_[p] = 0;
        free_.push_back(p);
        for (int32_t id : fresh_)
            if (pf_[id] >= 2) pq_insert(id);
        fresh_.clear();
    }
};

}  // namespace

Slp repair(const Csrv& s, int64_t r0, int64_t r1) {
    RePair rp(s, r0, r1);
    return rp.run();
}

}  // namespace gcs
