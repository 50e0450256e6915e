// Device arena layout of an uploaded grammar (host-side arithmetic only; used
// by gc_layout and gc_upload). Every part starts on a 256-byte boundary.
//
//   read-only grammar   nodes     int2[sum of padded widths]  child references,
//                                 each level starting on a 16-node (128 B)
//                                 boundary and padded to a multiple of 16
//                       levels    int64[6 (L+2)]   per level k: padded start,
//                                 width, roots, first RV slot, first emit chunk,
//                                 offset in the tail buffer
//                       V         policy[|V|]      value dictionary
//                       leaf      int32[alpha]     leaf code of terminal p
//     level / chunk     cref      int32[early]     C without the references to
//     emit:                                        the tail levels: by level, then
//                                                  row (level emit); by row (chunk)
//                       echunk    int4[chunks]     (start, length, id, 0) per chunk
//                       row_ech   int32[n+1]       row r's chunk ids
//                       late_off  int32[n+1]       row r's references into the
//                       late_ref  int32[late]      narrow top levels (tail indices)
//     row emit:         c_off     int32[n+1]
//                       c_ref     int32[|C|]       C in row order (RV slots / T)
//   scratch             buf0X     value[TB + w*]   leaf table T, then a level's
//                       buf1X     value[TB + w*]   values (the two streaming buffers)
//                       tbuf      value[tail]      the narrow top levels' values,
//                                                  level after level
//     level / chunk:    esum      value[chunks]    chunk sums
//     chunk / row:      RVX       value[TB + rho]  leaf table T, then root values
//                       status    256 B            status word, fixpoint flag,
//                                                  grid-barrier arrival counter
//   staging             xs        value[m]         x / y copies for the
//                       ys        value[n]         host-buffer entry point
// "value" is k_max elements of the policy's type (float, int64, uint64);
// TB = alpha + 1 rounded up to a multiple of 64 values.
//
// Leaf table: T[0] is the combine identity and T[p+1] = V[l_p] (x) x[j_p] for
// terminal p = <l_p, j_p> (Sec. 4.3's T). Its copies sit in front of each
// buffer, so that one index space covers both: a child or C reference is
//   0            the identity (second child of a pass-through)
//   p + 1        terminal p
//   TB + s       slot s of a level's buffer (or root slot s of RV)
// and every read is a single load, without a branch. Level 1, whose children
// are all terminals, instead stores leaf codes (column << vbits | value index)
// and evaluates its leaves in the sweep while the T copies are being written.
//
// Levels 1..Lg are wide and use the whole grid; the narrow levels above them
// (each at most tail_nodes wide, two or more of them) form the tail, computed
// by one CTA into the tail buffer, where they all stay until the product ends.
//
// Emit modes (Lemma 2.2, y[r] = sum of row r's symbols of C). C's references
// to the tail levels ("late" references, few) are kept per row and added by
// the last pass, from the tail buffer; the others are "early" references.
//   level emit  rows of C average 128 symbols or more, 16-wide values. Early
//               references are grouped by level, then row; chunks of at most
//               512 references of one (level, row) are reduced right after
//               their level is computed, straight from that level's buffer
//               (the pages' emit on the spot). A last pass adds each row's
//               chunk sums in order, then its late references.
//   chunk emit  rows average 128 symbols or more, one-wide values: roots are
//               also stored to RV when their level is computed (RV stays in
//               L2), and the early references, in row order and cut into
//               chunks of at most 512 of one row, are reduced from RV while
//               one CTA computes the tail levels; a last pass as above.
//   row emit    shorter rows: roots are stored to RV, and rows are reduced at
//               the end, a few lanes per row.
#pragma once

#include "common.hpp"

namespace gcs {

constexpr int64_t kNodeAlign = 16;        // nodes per 128-byte granule
constexpr int64_t kEmitChunkSyms = 512;   // references per emit chunk
constexpr int64_t kLongRowAvg = 128;      // average |C| per row for chunked emits
constexpr int64_t kLevelRows = 6;         // rows of the level table

enum EmitMode : int32_t { EMIT_LEVEL = 0, EMIT_CHUNK = 1, EMIT_ROWS = 2 };

struct DevLayout {
    int64_t nodes, levels, V, leaf;
    int64_t cref, echunk, row_ech;        // level and chunk emit
    int64_t late_off, late_ref;
    int64_t c_off, c_ref;                 // row emit
    int64_t buf0, buf1, esum, tbuf, RV, status, xs, ys;
    int64_t total, grammar_bytes, scratch_bytes, staging_bytes;
    int64_t value_bytes;   // bytes of one node value (k_max elements)
    int64_t n_nodes_padded;
    int64_t n_echunks, n_late;
    int64_t tail_nodes;    // widest level the single-CTA tail takes
    int64_t grid_levels;   // Lg: levels 1..Lg use the whole grid
    int64_t tail_total;    // nodes of the tail buffer (levels Lg+1..L, padded)
    int64_t TB;            // leaf-table block length in values
    int32_t vbits;         // bits of the value index inside a leaf code
    EmitMode emit;

    bool chunked() const { return emit != EMIT_ROWS; }
    bool has_rv() const { return emit != EMIT_LEVEL; }
};

inline int64_t policy_elem_bytes(gc_policy p) { return p == GC_F32_SUM ? 4 : 8; }

inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

inline int64_t pad_nodes(int64_t w) { return (w + kNodeAlign - 1) / kNodeAlign * kNodeAlign; }

inline int32_t value_bits(int64_t n_values) {
    int32_t b = 0;
    while (((int64_t)1 << b) < n_values) ++b;
    return b;
}

inline int64_t leaf_block(int64_t alpha) { return (alpha + 1 + 63) / 64 * 64; }

inline EmitMode emit_mode(const Grammar& g, int32_t k_max) {
    const bool long_rows = g.n > 0 && (int64_t)g.c_ref.size() >= kLongRowAvg * g.n;
    return !long_rows ? EMIT_ROWS : k_max == 1 ? EMIT_CHUNK : EMIT_LEVEL;
}

inline int64_t tail_width(int32_t k_max) { return k_max == 16 ? 1024 : 4096; }

// Lg: the narrow levels at the top (each at most tail_nodes wide) form the
// tail when there are two or more of them; otherwise every level is wide.
inline int64_t grid_level_count(const Grammar& g, int64_t tail_nodes) {
    const int64_t L = g.L;
    int64_t first_narrow = L + 1;
    while (first_narrow > 1 && g.lvl_off[first_narrow] - g.lvl_off[first_narrow - 1] <= tail_nodes) --first_narrow;
    return L - first_narrow + 1 >= 2 ? first_narrow - 1 : L;
}

// Offset of level k in the tail buffer (k > Lg; 0 otherwise); entry L+1 is the total.
inline std::vector<int64_t> tail_offsets(const Grammar& g, int64_t Lg) {
    std::vector<int64_t> t((size_t)g.L + 2, 0);
    int64_t o = 0;
    for (int64_t k = Lg + 1; k <= g.L; ++k) {
        t[k] = o;
        o += pad_nodes(g.lvl_off[k + 1] - g.lvl_off[k]);
    }
    t[g.L + 1] = o;
    return t;
}

// Chunks of C's early references (terminals and levels 1..Lg): with by_level,
// grouped by the level of their symbol and indexed into that level's
// [T | buffer] space, in chunks of one (level, row); otherwise in row order,
// indexed into [T | RV], in chunks of one row (all in group 0). References to
// the tail levels are kept per row as tail-buffer indices.
struct EmitPlan {
    std::vector<int32_t> cref;      // grouped by (level, row), as [T | buffer] indices
    std::vector<int32_t> echunk;    // 4 per chunk: start, length, id, 0 (level-major)
    std::vector<int64_t> ech;       // L+2: chunk range of level k
    std::vector<int32_t> row_ech;   // n+1
    std::vector<int32_t> late_off;  // n+1
    std::vector<int32_t> late_ref;  // tail-buffer node indices, row by row
};

inline int64_t ref_level(const Grammar& g, int32_t c) {
    if (c < 0) return 0;
    // root slot c lies in level k with root_off[k] <= c < root_off[k+1]
    return std::upper_bound(g.root_off.begin() + 1, g.root_off.begin() + g.L + 2, (int64_t)c) -
           g.root_off.begin() - 1;
}

inline EmitPlan plan_emit(const Grammar& g, int64_t TB, int64_t Lg, bool by_level) {
    const int64_t L = g.L, n = g.n;
    const std::vector<int64_t>& co = g.slp.c_off;
    const std::vector<int64_t> toff = tail_offsets(g, Lg);
    const size_t C = g.c_ref.size();
    std::vector<int32_t> lev(C), pos(C);
    std::vector<char> early(C);
    EmitPlan p;
    p.late_off.assign((size_t)n + 1, 0);
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            const int32_t c = g.c_ref[e];
            const int64_t k = ref_level(g, c);
            early[e] = k <= Lg;
            lev[e] = by_level ? (int32_t)k : 0;
            if (c < 0) {
                pos[e] = -c - 1;   // terminal p = -c-2 -> T[p+1]
            } else if (k <= Lg) {
                pos[e] = (int32_t)(by_level ? TB + c - g.root_off[k] : TB + c);
            } else {
                p.late_ref.push_back((int32_t)(toff[k] + c - g.root_off[k]));
            }
        }
        p.late_off[r + 1] = (int32_t)p.late_ref.size();
    }
    // counting sort of the wide references by level, stable in row-major order
    std::vector<int64_t> cnt((size_t)Lg + 2, 0);
    for (size_t e = 0; e < C; ++e)
        if (early[e]) ++cnt[lev[e] + 1];
    for (int64_t k = 0; k <= Lg; ++k) cnt[k + 1] += cnt[k];
    p.cref.resize((size_t)cnt[Lg + 1]);
    std::vector<int64_t> at(cnt.begin(), cnt.end() - 1);
    std::vector<int32_t> row_of(p.cref.size());
    for (int64_t r = 0; r < n; ++r)
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            if (!early[e]) continue;
            const int64_t d = at[lev[e]]++;
            p.cref[d] = pos[e];
            row_of[d] = (int32_t)r;
        }
    // chunks: runs of one (level, row), cut every kEmitChunkSyms references
    struct Ch { int32_t row, lev, start, len; };
    std::vector<Ch> ch;
    p.ech.assign((size_t)L + 2, 0);
    for (int64_t k = 0; k <= L; ++k) {
        p.ech[k] = (int64_t)ch.size();
        if (k > Lg) continue;
        for (int64_t d = cnt[k]; d < cnt[k + 1];) {
            int64_t e = d;
            while (e < cnt[k + 1] && row_of[e] == row_of[d] && e - d < kEmitChunkSyms) ++e;
            ch.push_back({row_of[d], (int32_t)k, (int32_t)d, (int32_t)(e - d)});
            d = e;
        }
    }
    p.ech[L + 1] = (int64_t)ch.size();
    // ids in (row, level, start) order: a row's chunks are contiguous
    std::vector<int32_t> order(ch.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = (int32_t)i;
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        if (ch[a].row != ch[b].row) return ch[a].row < ch[b].row;
        if (ch[a].lev != ch[b].lev) return ch[a].lev < ch[b].lev;
        return ch[a].start < ch[b].start;
    });
    p.echunk.assign(4 * ch.size(), 0);
    p.row_ech.assign((size_t)n + 1, 0);
    for (size_t id = 0; id < order.size(); ++id) {
        const Ch& c = ch[order[id]];
        p.echunk[4 * order[id]] = c.start;
        p.echunk[4 * order[id] + 1] = c.len;
        p.echunk[4 * order[id] + 2] = (int32_t)id;
        ++p.row_ech[c.row + 1];
    }
    for (int64_t r = 0; r < n; ++r) p.row_ech[r + 1] += p.row_ech[r];
    return p;
}

// Checks a plan against the grammar before it reaches the device: every
// chunk lies inside cref and holds references of its own level only (T for
// level 0, that level's roots otherwise), chunk ids are a permutation that
// row_ech splits by row, and every tail reference lies inside the tail buffer.
inline void validate_emit_plan(const EmitPlan& p, const Grammar& g, int64_t TB, int64_t Lg, bool by_level) {
    const int64_t n = g.n, L = g.L, nch = (int64_t)p.echunk.size() / 4;
    const std::vector<int64_t> toff = tail_offsets(g, Lg);
    auto bad = [](const char* what) { fail(GC_ERR_INVALID_GRAMMAR, std::string("emit plan: ") + what); };
    if ((int64_t)p.ech.size() != L + 2 || p.ech[0] != 0 || p.ech[L + 1] != nch) bad("level chunk ranges");
    if ((int64_t)p.row_ech.size() != n + 1 || p.row_ech[0] != 0 || p.row_ech[n] != nch) bad("row chunk ranges");
    if ((int64_t)p.late_off.size() != n + 1 || p.late_off[0] != 0 || p.late_off[n] != (int64_t)p.late_ref.size())
        bad("tail reference ranges");
    std::vector<char> seen((size_t)nch, 0);
    for (int64_t k = 0; k <= L; ++k) {
        if (p.ech[k + 1] < p.ech[k] || ((k > Lg || (!by_level && k > 0)) && p.ech[k + 1] != p.ech[k]))
            bad("level chunk ranges");
        // terminals (level 0), one level's roots (by level), or terminals and
        // the roots of levels 1..Lg in RV (row order)
        const int64_t t_hi = k == 0 ? g.alpha() + 1 : 0;
        const int64_t r_hi = TB + (!by_level ? g.root_off[Lg + 1] : k == 0 ? 0 : g.lvl_roots[k]);
        auto ok = [&](int64_t v) { return (v >= 0 && v < t_hi) || (v >= TB && v < r_hi); };
        for (int64_t j = p.ech[k]; j < p.ech[k + 1]; ++j) {
            const int64_t st = p.echunk[4 * j], len = p.echunk[4 * j + 1], id = p.echunk[4 * j + 2];
            if (st < 0 || len < 1 || len > kEmitChunkSyms || st + len > (int64_t)p.cref.size()) bad("chunk extent");
            if (id < 0 || id >= nch || seen[id]) bad("chunk ids");
            seen[id] = 1;
            for (int64_t e = st; e < st + len; ++e)
                if (!ok(p.cref[e])) bad("reference outside its level");
        }
    }
    for (int64_t r = 0; r < n; ++r)
        if (p.row_ech[r + 1] < p.row_ech[r] || p.late_off[r + 1] < p.late_off[r]) bad("row ranges decrease");
    for (int32_t t : p.late_ref)
        if (t < 0 || t >= toff[L + 1]) bad("tail reference outside the tail buffer");
}

// Sizes of plan_emit's arrays, counted without building the plan:
// chunks, wide references and tail references.
struct EmitCounts {
    int64_t chunks = 0, wide = 0, late = 0;
};
inline EmitCounts count_emit(const Grammar& g, int64_t Lg, bool by_level) {
    const int64_t n = g.n;
    const std::vector<int64_t>& co = g.slp.c_off;
    std::vector<int64_t> per((size_t)Lg + 1, 0);
    EmitCounts t;
    for (int64_t r = 0; r < n; ++r) {
        std::fill(per.begin(), per.end(), 0);
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            const int64_t k = ref_level(g, g.c_ref[e]);
            if (k > Lg) ++t.late;
            else ++per[by_level ? k : 0];
        }
        for (int64_t k = 0; k <= Lg; ++k) {
            t.chunks += (per[k] + kEmitChunkSyms - 1) / kEmitChunkSyms;
            t.wide += per[k];
        }
    }
    return t;
}

inline DevLayout device_layout(const Grammar& g, gc_policy p, int32_t k_max) {
    DevLayout d{};
    const int64_t L = g.L, C = (int64_t)g.c_ref.size(), A = g.alpha();
    d.value_bytes = policy_elem_bytes(p) * k_max;
    d.vbits = value_bits((int64_t)g.V.size());
    d.TB = leaf_block(A);
    d.emit = emit_mode(g, k_max);
    d.tail_nodes = tail_width(k_max);
    d.grid_levels = grid_level_count(g, d.tail_nodes);
    d.tail_total = tail_offsets(g, d.grid_levels)[L + 1];
    d.n_nodes_padded = 0;
    for (int64_t k = 1; k <= L; ++k) d.n_nodes_padded += pad_nodes(g.lvl_off[k + 1] - g.lvl_off[k]);
    EmitCounts ec;
    if (d.chunked()) ec = count_emit(g, d.grid_levels, d.emit == EMIT_LEVEL);
    d.n_echunks = ec.chunks;
    d.n_late = ec.late;
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        int64_t at = o;
        o = align256(o + bytes);
        return at;
    };
    d.nodes = take(8 * d.n_nodes_padded);
    d.levels = take(8 * kLevelRows * (L + 2));
    d.V = take(policy_elem_bytes(p) * std::max<int64_t>(1, (int64_t)g.V.size()));
    d.leaf = take(4 * A);
    if (d.chunked()) {
        d.cref = take(4 * ec.wide);
        d.echunk = take(16 * d.n_echunks);
        d.row_ech = take(4 * (g.n + 1));
        d.late_off = take(4 * (g.n + 1));
        d.late_ref = take(4 * d.n_late);
    } else {
        d.c_off = take(4 * (g.n + 1));
        d.c_ref = take(4 * C);
    }
    d.grammar_bytes = o;
    const int64_t w = g.max_width();
    d.buf0 = take(d.value_bytes * (d.TB + w));
    d.buf1 = take(d.value_bytes * (d.TB + w));
    d.tbuf = take(d.value_bytes * d.tail_total);
    if (d.chunked()) d.esum = take(d.value_bytes * d.n_echunks);
    if (d.has_rv()) d.RV = take(d.value_bytes * (d.TB + g.n_roots));
    d.status = take(256);
    d.scratch_bytes = o - d.grammar_bytes;
    d.xs = take(d.value_bytes * g.m);
    d.ys = take(d.value_bytes * g.n);
    d.staging_bytes = o - d.grammar_bytes - d.scratch_bytes;
    d.total = o;
    return d;
}

// Checks a (policy, k) request against the grammar's values.
inline void check_policy(const Grammar& g, gc_policy p, int32_t k_max) {
    if (p != GC_F32_SUM && p != GC_I64_SUM && p != GC_BOOL_OR) fail(GC_ERR_ARG, "unknown policy");
    if (p == GC_F32_SUM ? (k_max != 1 && k_max != 16) : k_max != 1)
        fail(GC_ERR_ARG, "k_max must be 1 (or 16 for GC_F32_SUM)");
    if (p == GC_I64_SUM)
        for (float v : g.V)
            if (v != (float)(int64_t)v || v > 9.0e15f || v < -9.0e15f)
                fail(GC_ERR_UNSUPPORTED, "GC_I64_SUM needs integer matrix values");
    if (p == GC_BOOL_OR)
        for (float v : g.V)
            if (v != 1.0f) fail(GC_ERR_UNSUPPORTED, "GC_BOOL_OR needs every stored entry to be 1");
    if ((int64_t)g.c_ref.size() >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "|C| >= 2^31");
    if ((((int64_t)g.m) << value_bits((int64_t)g.V.size())) >= INT32_MAX)
        fail(GC_ERR_UNSUPPORTED, "columns x distinct values too large for 31-bit leaf codes");
    if (leaf_block(g.alpha()) + std::max(g.max_width(), g.n_roots) >= INT32_MAX)
        fail(GC_ERR_UNSUPPORTED, "leaf table plus level width exceeds 31-bit indices");
}

}  // namespace gcs
