// Host-side plan of the left product x^T = y^T M (x = M^T y) over the packed,
// properly layered grammar: the dual of the right product, which the pages
// leave to future work ("left multiplication via pull-based reduction",
// Sec. 8). Written here as a top-down sweep in which every value is a pulled
// sum, so there are no atomics and the result is the same bit for bit on
// every run.
//
// Every layered node u gets a weight W[u]: the sum of y[r] over the
// occurrences of u in the expansions of the rows r (Lemma 2.2 read
// backwards). Top-down, level L first:
//   seed     RS[s]  = sum of y[r] over the rows r whose C names s, for the
//                     root slots s < rho and the terminals (slot rho + p)
//   level k  W[u]   = (RS[slot of u] if u is a root) + sum of W[p] over the
//                     parents p of u, all at level k + 1 (proper layering,
//                     Def. 3.2: a pass-through carries its child's weight
//                     down as it carries its value up)
//   terms    TIN[p] = RS[rho + p] + sum of W[q] over the nodes q with
//                     terminal p as a child (any level)
//   columns  x[j]   = sum over the terminals p = <l, j> of V[l] * TIN[p]
//
// Each step is a set of segments (a sum over a list of references). A warp
// task reduces either up to 32 consecutive segments, one per lane, each in
// order (LIGHT; a lane whose segment holds more than kLeftLightMax items
// leaves it to a HEAVY task), or one long segment over all 32 lanes: lane l
// sums items l, l + 32, ... in order, then the lanes combine by a fixed
// butterfly (HEAVY). So no sum is a sequential chain longer than
// kLeftLightMax + count / 32 + 5 additions.
#pragma once

#include <cstdint>
#include <vector>

#include "common.hpp"

namespace gcs {

constexpr int32_t kLeftLightMax = 64;   // items of a segment one lane sums alone

// Segment sets, in sweep order: 0 seed, 1..L levels (level L first in time,
// set k is level k), L+1 terminals, L+2 columns.
struct LeftPlan {
    int64_t n = 0, m = 0, L = 0, N = 0, rho = 0, alpha = 0;
    std::vector<int64_t> lvl_off, lvl_roots, root_off;   // L+2 each (as in Grammar)
    // seed: segments s < rho + alpha, references are rows
    std::vector<int32_t> soff, srow;
    // parents: segments are node positions (0..N), references node positions
    std::vector<int32_t> poff, pref;
    // terminal parents: segments are terminals, references node positions
    std::vector<int32_t> toff, tref;
    // columns: segments are columns, references terminals (contiguous: the
    // terminal table is sorted by column)
    std::vector<int32_t> coff;
    std::vector<int32_t> term_vidx;
    std::vector<float> V;
    // warp tasks of every set: (first segment, count > 0: LIGHT over
    // segments first .. first + count - 1; -1: HEAVY for segment first); set
    // s owns tasks[task_off[s] .. task_off[s+1])
    std::vector<int32_t> task;      // 2 per task
    std::vector<int64_t> task_off;  // L+4
    int64_t n_tasks() const { return (int64_t)task.size() / 2; }
};

// Tasks of one segment set: the segments in runs of 32 (LIGHT; their heavy
// segments, over kLeftLightMax items, skipped), then one task per heavy
// segment.
inline bool left_heavy(const std::vector<int32_t>& off, int64_t s) {
    return (int64_t)off[s + 1] - off[s] > kLeftLightMax;
}
inline void left_tasks(LeftPlan& p, int64_t first, int64_t count, const std::vector<int32_t>& off) {
    for (int64_t s = first; s < first + count; s += 32) {
        p.task.push_back((int32_t)s);
        p.task.push_back((int32_t)std::min<int64_t>(32, first + count - s));
    }
    for (int64_t s = first; s < first + count; ++s)
        if (left_heavy(off, s)) {
            p.task.push_back((int32_t)s);
            p.task.push_back(-1);
        }
}

// CSR by counting: for keys key[e] < nkeys, the values val[e] grouped by key,
// each group in the order of e.
inline void left_csr(int64_t nkeys, const std::vector<int32_t>& key, const std::vector<int32_t>& val,
                     std::vector<int32_t>& off, std::vector<int32_t>& out) {
    std::vector<int64_t> o((size_t)nkeys + 1, 0);
    for (int32_t k : key) ++o[(size_t)k + 1];
    for (int64_t i = 0; i < nkeys; ++i) o[i + 1] += o[i];
    if (o[nkeys] >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "left product: a reference list longer than 2^31");
    off.assign(o.begin(), o.end());
    out.assign(key.size(), 0);
    std::vector<int64_t> at(o.begin(), o.end() - 1);
    for (size_t e = 0; e < key.size(); ++e) out[at[key[e]]++] = val[e];
}

// The plan of the packed layered grammar g (not a device view: pass-throughs
// are nodes here, each with one child and the identity).
inline LeftPlan plan_left(const Grammar& g) {
    LeftPlan p;
    p.n = g.n;
    p.m = g.m;
    p.L = g.L;
    p.N = g.n_nodes();
    p.rho = g.n_roots;
    p.alpha = g.alpha();
    p.lvl_off = g.lvl_off;
    p.lvl_roots = g.lvl_roots;
    p.root_off = g.root_off;
    p.term_vidx = g.term_vidx;
    p.V = g.V;
    if (p.N >= INT32_MAX || p.rho + p.alpha >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "left product: grammar too large");
    const int64_t A = p.alpha, L = p.L;
    // seed: C's references, by target (root slot, or rho + terminal)
    {
        std::vector<int32_t> key, val;
        key.reserve(g.c_ref.size());
        val.reserve(g.c_ref.size());
        for (int64_t r = 0; r < g.n; ++r)
            for (int64_t q = g.slp.c_off[r]; q < g.slp.c_off[r + 1]; ++q) {
                const int32_t c = g.c_ref[q];
                key.push_back(c >= 0 ? c : (int32_t)(p.rho + (-(int64_t)c - 2)));
                val.push_back((int32_t)r);
            }
        left_csr(p.rho + A, key, val, p.soff, p.srow);
    }
    // parents and terminal parents, from every node's children
    {
        std::vector<int32_t> pk, pv, tk, tv;
        for (int64_t k = 1; k <= L; ++k)
            for (int64_t t = 0; t < g.lvl_off[k + 1] - g.lvl_off[k]; ++t) {
                const int64_t u = g.lvl_off[k] + t;
                for (int h = 0; h < 2; ++h) {
                    const int32_t c = g.nodes[2 * u + h];
                    if (c >= 0) {
                        if (k < 2 || c >= g.lvl_off[k] - g.lvl_off[k - 1])
                            fail(GC_ERR_INVALID_GRAMMAR, "left plan: child outside the level below");
                        pk.push_back((int32_t)(g.lvl_off[k - 1] + c));
                        pv.push_back((int32_t)u);
                    } else if (c <= -2) {
                        if (-(int64_t)c - 2 >= A) fail(GC_ERR_INVALID_GRAMMAR, "left plan: terminal out of range");
                        tk.push_back(-c - 2);
                        tv.push_back((int32_t)u);
                    }
                }
            }
        left_csr(p.N, pk, pv, p.poff, p.pref);
        left_csr(A, tk, tv, p.toff, p.tref);
    }
    // columns: the terminal table is sorted by column
    p.coff.assign((size_t)p.m + 1, 0);
    for (int64_t q = 0; q < A; ++q) {
        if (q > 0 && g.term_col[q] < g.term_col[q - 1]) fail(GC_ERR_INVALID_GRAMMAR, "terminals not sorted by column");
        ++p.coff[(size_t)g.term_col[q] + 1];
    }
    for (int64_t j = 0; j < p.m; ++j) p.coff[j + 1] += p.coff[j];
    // tasks: seed, levels 1..L, terminals, columns
    p.task_off.assign((size_t)L + 4, 0);
    left_tasks(p, 0, p.rho + A, p.soff);
    for (int64_t k = 1; k <= L; ++k) {
        p.task_off[k] = p.n_tasks();
        left_tasks(p, g.lvl_off[k], g.lvl_off[k + 1] - g.lvl_off[k], p.poff);
    }
    p.task_off[L + 1] = p.n_tasks();
    left_tasks(p, 0, A, p.toff);
    p.task_off[L + 2] = p.n_tasks();
    left_tasks(p, 0, p.m, p.coff);
    p.task_off[L + 3] = p.n_tasks();
    return p;
}

// Bounds of every array the kernels index, before any device access.
inline void validate_left_plan(const LeftPlan& p) {
    auto bad = [](const char* what) { fail(GC_ERR_INVALID_GRAMMAR, std::string("left plan: ") + what); };
    auto check_csr = [&](const std::vector<int32_t>& off, const std::vector<int32_t>& ref, int64_t nseg,
                         int64_t bound, const char* what) {
        if ((int64_t)off.size() != nseg + 1 || off[0] != 0 || off[nseg] != (int64_t)ref.size()) bad(what);
        for (int64_t s = 0; s < nseg; ++s)
            if (off[s + 1] < off[s]) bad(what);
        for (int32_t r : ref)
            if (r < 0 || r >= bound) bad(what);
    };
    check_csr(p.soff, p.srow, p.rho + p.alpha, p.n, "seed rows");
    check_csr(p.poff, p.pref, p.N, p.N, "parents");
    check_csr(p.toff, p.tref, p.alpha, p.N, "terminal parents");
    if ((int64_t)p.coff.size() != p.m + 1 || p.coff[p.m] != p.alpha) bad("columns");
    for (int64_t j = 0; j < p.m; ++j)
        if (p.coff[j + 1] < p.coff[j]) bad("columns");
    for (int32_t v : p.term_vidx)
        if (v < 0 || v >= (int64_t)p.V.size()) bad("value index");
    // every parent of a level-k node is at level k + 1, and each segment set's
    // tasks name only its own segments
    for (int64_t k = 1; k <= p.L; ++k)
        for (int64_t u = p.lvl_off[k]; u < p.lvl_off[k + 1]; ++u)
            for (int32_t q = p.poff[u]; q < p.poff[u + 1]; ++q)
                if (k == p.L || p.pref[q] < p.lvl_off[k + 1] || p.pref[q] >= p.lvl_off[k + 2]) bad("parent level");
    auto set_range = [&](int64_t s, int64_t& lo, int64_t& hi) {
        if (s == 0) lo = 0, hi = p.rho + p.alpha;
        else if (s <= p.L) lo = p.lvl_off[s], hi = p.lvl_off[s + 1];
        else if (s == p.L + 1) lo = 0, hi = p.alpha;
        else lo = 0, hi = p.m;
    };
    if ((int64_t)p.task_off.size() != p.L + 4 || p.task_off[p.L + 3] != p.n_tasks()) bad("task table");
    std::vector<int32_t> seen;
    for (int64_t s = 0; s <= p.L + 2; ++s) {
        int64_t lo = 0, hi = 0;
        set_range(s, lo, hi);
        const std::vector<int32_t>& off = s == 0 ? p.soff : s <= p.L ? p.poff : s == p.L + 1 ? p.toff : p.coff;
        seen.assign((size_t)(hi - lo), 0);
        for (int64_t t = p.task_off[s]; t < p.task_off[s + 1]; ++t) {
            const int32_t first = p.task[2 * t], cnt = p.task[2 * t + 1];
            const int32_t k = cnt < 0 ? 1 : cnt;
            if (cnt == 0 || cnt > 32 || cnt < -1 || first < lo || (int64_t)first + k > hi) bad("task");
            for (int32_t i = 0; i < k; ++i) {
                const int32_t sg = first + i;
                const bool heavy = left_heavy(off, sg);
                if (cnt < 0 && !heavy) bad("heavy task on a short segment");
                if ((cnt < 0) == heavy && seen[sg - lo]++) bad("segment summed twice");
            }
        }
        for (int32_t c : seen)
            if (c != 1) bad("segment not covered exactly once");
    }
}

}  // namespace gcs
