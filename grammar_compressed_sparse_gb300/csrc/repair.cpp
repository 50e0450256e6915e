// RePair with row boundaries (Sec. 2 "Grammar" and Sec. 4.1 of the pages):
// repeatedly replace the most frequent pair of adjacent symbols by a new
// nonterminal N_i -> A_i B_i, never pairing across a row end, and stop when
// no pair occurs twice. Rules are numbered in creation order, so every child
// precedes its parent (the topological numbering of Eq. 2.3).
//
// Data structures (after Larsson and Moffat's linear-time RePair):
//   Pos[i]     one record per position of the working sequence: its symbol
//              (a row end is DELIM, a replaced right symbol EMPTY), links to
//              the neighbouring live positions, the id of the pair starting
//              here, and this occurrence's links in that pair's list
//   Pair[id]   (a, b, frequency, first occurrence, queue links)
//   queues     FIFO per frequency 2..B plus one list above B
// Because a row never holds the same symbol twice (its symbols cover disjoint
// column ranges), occurrences never overlap. Every pair created while
// replacing (a, b) by N contains N, so new pairs are found through two small
// per-round maps keyed by the neighbour symbol; no global pair hash is needed
// after the initial count, and decrements go through Pos[i].pid.
//
// The main loop is bound by memory latency, so each record fits one cache
// line and a round first collects the pair's occurrences, then walks them
// with a three-stage software prefetch (the position; its neighbours; their
// list neighbours and pair records).
#include <sys/mman.h>

#include <cstring>
#include <memory>
#include <numeric>

#include "common.hpp"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace gcs {
namespace {

constexpr int32_t DELIM = -1;
constexpr int32_t EMPTY = -2;

struct Pos {
    int32_t seq, nxt, prv, pid, onext, oprev;
};
struct alignas(32) PairRec {
    int32_t a, b, freq, head, qp, qn, qb, pad;
};

template <class T>
inline void prefetch(const T* p) {
    __builtin_prefetch(p, 1, 3);
}

// Fixed-capacity array in anonymous memory, backed by transparent huge pages
// where the kernel allows it: the random accesses of the main loop would
// otherwise miss the TLB on almost every step. Pages are zero until touched.
template <class T>
class HugeArray {
public:
    HugeArray() = default;
    explicit HugeArray(size_t n) { reset(n); }
    HugeArray(const HugeArray&) = delete;
    HugeArray& operator=(const HugeArray&) = delete;
    ~HugeArray() { release(); }
    void reset(size_t n) {
        release();
        bytes_ = std::max<size_t>(n * sizeof(T), 1);
        void* p = mmap(nullptr, bytes_, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS | MAP_NORESERVE, -1, 0);
        if (p == MAP_FAILED) throw std::bad_alloc();
        madvise(p, bytes_, MADV_HUGEPAGE);
        p_ = static_cast<T*>(p);
        cap_ = n;
    }
    T* get() const { return p_; }
    T& operator[](size_t i) const { return p_[i]; }
    size_t capacity() const { return cap_; }

private:
    void release() {
        if (p_) munmap(p_, bytes_);
        p_ = nullptr;
        cap_ = 0;
    }
    T* p_ = nullptr;
    size_t bytes_ = 0, cap_ = 0;
};

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
    // slot of key k; found tells whether it is present
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
        S_.reset((size_t)ns_ + 1);
        // ids are recycled, so records in use never exceed all ever created:
        // the initial pairs (<= ns) plus two per replacement (<= 2 ns)
        P_.reset(3 * (size_t)ns_ + 2);
        row_start_.resize((size_t)rows_);
        int64_t p = 0;
        for (int64_t r = r0; r < r1; ++r) {
            row_start_[r - r0] = (int32_t)p;
            for (int64_t e = s.row_off[r]; e < s.row_off[r + 1]; ++e) S_[p++].seq = s.sym[e];
            S_[p++].seq = DELIM;
        }
        Pos* S = S_.get();
#pragma omp parallel for schedule(static)
        for (int32_t i = 0; i < ns_; ++i) {
            S[i].nxt = i + 1;
            S[i].prv = i - 1;
            S[i].pid = -1;
            S[i].onext = -1;
            S[i].oprev = -1;
        }
        S[ns_] = Pos{DELIM, ns_, ns_ - 1, -1, -1, -1};   // sentinel read by prefetches
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
            const int32_t p = pop_max();
            if (p < 0) break;
            replace(p);
        }
        const Pos* S = S_.get();
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
            for (int32_t q = row_start_[r]; S[q].seq != DELIM; q = S[q].nxt) ++c;
            out.c_off[r + 1] = out.c_off[r] + c;
        }
        out.c_sym.resize((size_t)out.c_off[rows_]);
        for (int64_t r = 0; r < rows_; ++r) {
            int64_t o = out.c_off[r];
            for (int32_t q = row_start_[r]; S[q].seq != DELIM; q = S[q].nxt) out.c_sym[o++] = to_export(S[q].seq);
        }
        return out;
    }

private:
    int32_t alpha_;
    int32_t ns_ = 0;
    int64_t rows_ = 0;
    HugeArray<Pos> S_;
    std::vector<int32_t> row_start_;
    HugeArray<PairRec> P_;
    int32_t np_ = 0;   // pair records in use
    std::vector<int32_t> free_;
    int32_t B_ = 2, maxb_ = 0;
    std::vector<int32_t> bucket_, btail_;
    std::vector<int32_t> fresh_, occ_;
    std::vector<int32_t> ra_, rb_;   // rules in internal symbols
    StampMap lmap_, rmap_;

    int32_t to_export(int32_t s) const { return s < alpha_ ? -(s + 1) : s - alpha_; }

    int32_t new_pair(int32_t a, int32_t b) {
        int32_t id;
        if (!free_.empty()) {
            id = free_.back();
            free_.pop_back();
        } else {
            if ((size_t)np_ >= P_.capacity()) fail(GC_ERR_UNSUPPORTED, "pair table full");
            id = np_++;
        }
        P_[id] = PairRec{a, b, 0, -1, -1, -1, -1, 0};
        fresh_.push_back(id);
        return id;
    }

    // ---- occurrence lists
    void occ_push(int32_t id, int32_t pos) {
        Pos* S = S_.get();
        const int32_t h = P_[id].head;
        S[pos].onext = h;
        S[pos].oprev = -1;
        if (h >= 0) S[h].oprev = pos;
        P_[id].head = pos;
    }
    void occ_remove(int32_t id, int32_t pos) {
        Pos* S = S_.get();
        const int32_t a = S[pos].oprev, b = S[pos].onext;
        if (a >= 0) S[a].onext = b; else P_[id].head = b;
        if (b >= 0) S[b].oprev = a;
    }

    // ---- frequency queues: FIFO per frequency 2..B, one list above B.
    // Ties between equally frequent pairs go to the oldest pair (the pages
    // leave the tie-break open). Older pairs hold shallower symbols, so over a
    // repeated segment this pairs neighbours level by level and keeps the
    // grammar's depth near log2 of the segment length; a newest-first order
    // instead grows left-deep chains.
    // Decrements are lazy: a pair stays in the queue it was filed in (which
    // is then >= its frequency) and is re-filed when it reaches the front.
    // Increments only ever happen to the pairs created in the current round
    // (they all contain the new symbol); those are filed once, after it.
    int32_t list_of(int32_t f) const { return f > B_ ? B_ + 1 : f; }
    void pq_insert(int32_t id) {
        PairRec& r = P_[id];
        const int32_t l = list_of(r.freq);
        const int32_t t = btail_[l];
        r.qp = t;
        r.qn = -1;
        if (t >= 0) P_[t].qn = id; else bucket_[l] = id;
        btail_[l] = id;
        r.qb = l;
        if (l <= B_ && l > maxb_) maxb_ = l;
    }
    void pq_unlink(int32_t id) {
        PairRec& r = P_[id];
        const int32_t l = r.qb;
        if (r.qp >= 0) P_[r.qp].qn = r.qn; else bucket_[l] = r.qn;
        if (r.qn >= 0) P_[r.qn].qp = r.qp; else btail_[l] = r.qp;
        r.qp = r.qn = -1;
        r.qb = -1;
    }
    // Takes id out of its queue; true if it is still a candidate (freq >= 2).
    bool settle(int32_t id) {
        pq_unlink(id);
        if (P_[id].freq >= 2) return true;
        if (P_[id].freq == 0) free_.push_back(id);
        return false;
    }
    int32_t pop_max() {
        // above B: exact maximum by scan, re-filing entries that fell to <= B
        int32_t best = -1;
        for (int32_t q = bucket_[B_ + 1]; q >= 0;) {
            const int32_t nx = P_[q].qn;
            if (P_[q].freq <= B_) {
                if (settle(q)) pq_insert(q);
            } else if (best < 0 || P_[q].freq > P_[best].freq) {
                best = q;
            }
            q = nx;
        }
        if (best >= 0) {
            pq_unlink(best);
            return best;
        }
        for (;;) {
            while (maxb_ >= 2 && bucket_[maxb_] < 0) --maxb_;
            if (maxb_ < 2) return -1;
            const int32_t id = bucket_[maxb_];
            if (P_[id].freq == maxb_) {
                pq_unlink(id);
                return id;
            }
            if (settle(id)) pq_insert(id);   // stale: frequency dropped since filing
        }
    }
    void inc(int32_t id, int32_t pos) {   // only pairs created in this round
        occ_push(id, pos);
        ++P_[id].freq;
    }
    void dec(int32_t id, int32_t pos) {
        occ_remove(id, pos);
        if (--P_[id].freq == 0 && P_[id].qb < 0) free_.push_back(id);
    }

    // Initial digram count, grouped by left symbol (parallel over groups).
    void count_initial_pairs() {
        Pos* S = S_.get();
        const int32_t A = alpha_;
        std::vector<int64_t> cnt((size_t)A + 1, 0);
        for (int32_t i = 0; i + 1 < ns_; ++i)
            if (S[i].seq >= 0 && S[i + 1].seq >= 0) ++cnt[S[i].seq + 1];
        for (int32_t a = 0; a < A; ++a) cnt[a + 1] += cnt[a];
        std::unique_ptr<int32_t[]> grp(new int32_t[(size_t)cnt[A] + 1]);
        {
            std::vector<int64_t> w(cnt.begin(), cnt.end() - 1);
            for (int32_t i = 0; i + 1 < ns_; ++i)
                if (S[i].seq >= 0 && S[i + 1].seq >= 0) grp[w[S[i].seq]++] = i;
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
                    const int32_t bsym = S[pos + 1].seq;
                    bool f;
                    const size_t sl = m.slot(bsym, f);
                    if (!f) m.put(sl, bsym, d++);
                    S[pos].pid = m.val[sl];
                }
                ndist[a + 1] = d;
            }
        }
        for (int32_t a = 0; a < A; ++a) ndist[a + 1] += ndist[a];
        const int32_t np = ndist[A];
        np_ = np;
#pragma omp parallel for schedule(static)
        for (int32_t id = 0; id < np; ++id) P_[id] = PairRec{0, 0, 0, -1, -1, -1, -1, 0};
        // global ids, records, occurrence lists (each group owns its positions)
#pragma omp parallel for schedule(dynamic, 256)
        for (int32_t a = 0; a < A; ++a) {
            for (int64_t q = cnt[a]; q < cnt[a + 1]; ++q) {
                const int32_t pos = grp[q];
                const int32_t id = ndist[a] + S[pos].pid;
                S[pos].pid = id;
                PairRec& r = P_[id];
                r.a = a;
                r.b = S[pos + 1].seq;
                ++r.freq;
                const int32_t h = r.head;
                S[pos].onext = h;
                if (h >= 0) S[h].oprev = pos;
                r.head = pos;
            }
        }
        for (int32_t id = 0; id < np; ++id)
            if (P_[id].freq >= 2) pq_insert(id);
    }

    void replace(int32_t p) {
        Pos* S = S_.get();
        const int32_t a = P_[p].a, b = P_[p].b;
        if ((int64_t)alpha_ + (int64_t)ra_.size() >= INT32_MAX)
            fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 symbols");
        const int32_t N = alpha_ + (int32_t)ra_.size();
        ra_.push_back(a);
        rb_.push_back(b);
        // Every occurrence of p is consumed this round, so its list is only
        // read (the positions are re-threaded into new lists as they go).
        occ_.clear();
        for (int32_t q = P_[p].head; q >= 0; q = S[q].onext) occ_.push_back(q);
        P_[p].head = -1;
        lmap_.prepare(occ_.size());
        rmap_.prepare(occ_.size());
        fresh_.clear();
        const int64_t K = (int64_t)occ_.size();
        constexpr int64_t D = 6;
        for (int64_t t = 0; t < K; ++t) {
            if (t + 3 * D < K) prefetch(&S[occ_[t + 3 * D]]);
            if (t + 2 * D < K) {
                const Pos& s2 = S[occ_[t + 2 * D]];
                if (s2.prv >= 0) prefetch(&S[s2.prv]);
                prefetch(&S[s2.nxt]);
            }
            if (t + D < K) {
                const Pos& s1 = S[occ_[t + D]];
                if (s1.prv >= 0) {
                    const Pos& sx = S[s1.prv];
                    if (sx.onext >= 0) prefetch(&S[sx.onext]);
                    if (sx.oprev >= 0) prefetch(&S[sx.oprev]);
                    if (sx.pid >= 0) prefetch(&P_[sx.pid]);
                }
                const Pos& sj = S[s1.nxt];
                if (sj.onext >= 0) prefetch(&S[sj.onext]);
                if (sj.oprev >= 0) prefetch(&S[sj.oprev]);
                if (sj.pid >= 0) prefetch(&P_[sj.pid]);
                if (sj.nxt < ns_) prefetch(&S[sj.nxt]);
            }
            const int32_t i = occ_[t];
            const int32_t j = S[i].nxt;
            if (j >= ns_ || S[i].seq != a || S[j].seq != b) continue;   // cannot happen; defensive
            const int32_t xp = S[i].prv;
            const int32_t yp = S[j].nxt;
            const bool hx = xp >= 0 && S[xp].seq >= 0;
            const bool hy = yp < ns_ && S[yp].seq >= 0;
            if (hx) dec(S[xp].pid, xp);
            if (hy) dec(S[j].pid, j);
            S[i].seq = N;
            S[j].seq = EMPTY;
            S[j].pid = -1;
            S[i].nxt = yp;
            if (yp < ns_) S[yp].prv = i;
            if (hx) {
                const int32_t x = S[xp].seq;
                bool f;
                const size_t sl = lmap_.slot(x, f);
                int32_t id;
                if (f) {
                    id = lmap_.val[sl];
                } else {
                    id = new_pair(x, N);
                    lmap_.put(sl, x, id);
                }
                S[xp].pid = id;
                inc(id, xp);
            }
            if (hy) {
                const int32_t y = S[yp].seq;
                bool f;
                const size_t sl = rmap_.slot(y, f);
                int32_t id;
                if (f) {
                    id = rmap_.val[sl];
                } else {
                    id = new_pair(N, y);
                    rmap_.put(sl, y, id);
                }
                S[i].pid = id;
                inc(id, i);
            } else {
                S[i].pid = -1;
            }
        }
        P_[p].freq = 0;
        free_.push_back(p);
        for (int32_t id : fresh_)
            if (P_[id].freq >= 2) pq_insert(id);
        fresh_.clear();
    }
};

}  // namespace

Slp repair(const Csrv& s, int64_t r0, int64_t r1) {
    RePair rp(s, r0, r1);
    return rp.run();
}

}  // namespace gcs
