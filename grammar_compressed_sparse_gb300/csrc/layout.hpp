// Device arena layout of an uploaded grammar (host-side arithmetic only; used
// by gc_layout and gc_upload). Every part starts on a 256-byte boundary.
//
//   read-only grammar   nodes     int2[sum of padded widths]  child references,
//                                 each level starting on a 16-node (128 B)
//                                 boundary and padded to a multiple of 16
//                       levels    int64[10 (L+2)]  per level k: padded start,
//                                 width, roots, first RV slot, first emit chunk,
//                                 offset in the tail buffer, carried roots,
//                                 carried other nodes, first carry slot,
//                                 dataflow blocks of the level
//                       V         policy[|V|]      value dictionary
//                       leaf      int32[alpha]     leaf code of terminal p
//     level emit:       cref      int32[early]     C without the references to
//                                                  the tail levels, by level, then row
//                       echunk    int4[chunks]     (start, length, id, 0) per chunk
//     slice emit:       sref      uint16[256 tiles] offsets into slices of [T | RV],
//                                                  in tiles of 256 references
//                       sflag     uint8[32 tiles]  bit i of byte j: reference 8j+i
//                                                  of the tile starts a segment
//                       tile_sid  int32[tiles+1]   first segment start of each tile
//                       row_pos   int32[ids]       for each id (a row's segments and
//                                                  pieces in slice order), the index
//                                                  of its segment start
//                       sx0       int32[slices+1]  first value of each slice
//                       stile     int32[slices+1]  tile range of each slice
//                       sorder    int32[slices]    slices by decreasing tile count
//     level / slice:    row_ech   int32[n+1]       row r's chunk / segment ids
//                       late_off  int32[n+1]       row r's references into the
//                       late_ref  int32[late]      narrow top levels (tail indices)
//     row emit:         c_off     int32[n+1]
//                       c_ref     int32[|C|]       C in row order (RV slots / T)
//   scratch             buf0X     value[w*]        a level's values (the two
//                       buf1X     value[w*]        streaming buffers)
//                       tbuf      value[tail]      the narrow top levels' values,
//                                                  level after level
//                       carry     value[carried]   values of the nodes read two or
//                                                  more levels up (device view)
//     level / slice:    esum      value[chunks     chunk sums, or one sum per
//                                       / starts]  segment start
//     slice / row:      RVX       value[TB + rho]  leaf table T, then root values
//                       status    256 B            status word, fixpoint flag, grid-
//                                                  barrier and tail-group arrival counters
//   dataflow sweep (one value a node, flow.hpp): nodes holds the block-local
//   child references; fblk int32[16 blocks] block records, forder int32[blocks]
//   the processing order, fdeps / fgran int32 dependency and outlier-granule lists; scratch fb0..fb2 value[buf]
//   three level buffers, fflags int32[blocks] ready flags, fdone
//   uint64[L+2] finished blocks per level; no tail and no buf0 / buf1
//   staging             xs        value[m]         x / y copies for the
//                       ys        value[n]         host-buffer entry point
// "value" is k_max elements of the policy's type (float, int64, uint64);
// TB = alpha + 1 rounded up to a multiple of 64 values.
//
// Terminals are evaluated where the sweep reads them (Sec. 4.3's leaf values
// V[l_p] (x) x[j_p], without a leaf table in front of the level buffers, so
// the buffers hold w* values at every batch width): a child reference of a
// level k >= 2 node, and a C reference of the level emit, is
//   c >= 0       slot c of the level below (of its own level for C), or a
//                carry slot (kCarryBase + s, the device view's carried rules)
//   -1           the identity (second child of a pass-through)
//   -2 - q       a terminal by its leaf code q = column << vbits | value index
// and level 1, whose children are all terminals, stores the leaf codes
// themselves. The slice and row emits read C's bare terminals from a leaf
// table in front of RV: T[0] the identity, T[p+1] = V[l_p] (x) x[j_p] for
// terminal p, and root slot s at TB + s.
//
// Levels 1..Lg are wide and use the whole grid; the narrow levels above them
// (each at most tail_nodes wide, two or more of them) form the tail, computed
// into the tail buffer, where they all stay until the product ends: by one CTA
// in the level and row emits, by a group of CTAs beside the slices in the
// slice emit (whose tail takes wider levels).
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
//   slice emit  rows average 128 symbols or more, one-wide values: roots are
//               also stored to RV when their level is computed. After the wide
//               levels, a second kernel cuts [T | RV] into slices that fit a
//               CTA's shared memory; each CTA loads a slice and sums, for
//               every row, that row's references into the slice (a segment,
//               in C order), reading shared memory instead of scattered global
//               lines. One CTA computes the tail levels meanwhile; a last pass
//               adds each row's segment sums in slice order, then its late
//               references.
//   row emit    shorter rows: roots are stored to RV, and rows are reduced at
//               the end, a few lanes per row.
#pragma once

#include "common.hpp"

namespace gcs {

constexpr int64_t kNodeAlign = 16;        // nodes per 128-byte granule
constexpr int64_t kEmitChunkSyms = 512;   // references per emit chunk
constexpr int64_t kLongRowAvg = 128;      // average |C| per row for chunked emits
constexpr int64_t kLevelRows = 10;        // rows of the level table
constexpr int64_t kFlowBlkBytes = 64;     // bytes of a dataflow block record (flow.hpp)

enum EmitMode : int32_t { EMIT_LEVEL = 0, EMIT_SLICE = 1, EMIT_ROWS = 2 };

constexpr int64_t kSliceBytes = 192 << 10;   // shared memory of one slice
constexpr int64_t kSliceTarget = 136;         // slices per round: a 152-SM part's CTAs less the tail group's 16
constexpr int64_t kSliceValueCost = 4;        // staged values that cost as much as one reference
constexpr int64_t kSliceStep = 256;           // slices start on multiples of this many values
inline int64_t slice_len(int64_t value_bytes) { return std::min<int64_t>(kSliceBytes / value_bytes, 65536); }

struct DevLayout {
    int64_t nodes, levels, V, leaf;
    int64_t cref, echunk;                 // level emit
    int64_t sref, sflag, tile_sid, row_pos, sx0, stile, sorder;   // slice emit
    int64_t row_ech, late_off, late_ref;  // level and slice emit
    int64_t c_off, c_ref;                 // row emit
    int64_t buf0, buf1, esum, tbuf, carry, RV, status, xs, ys;
    int64_t total, grammar_bytes, scratch_bytes, staging_bytes;
    int64_t value_bytes;   // bytes of one node value (k_max elements)
    int64_t n_nodes_padded;
    int64_t n_echunks, n_late;   // chunk or segment ids; late references
    int64_t n_early;             // level emit: early references
    int64_t slice, n_slices;     // slice emit: most values a slice holds, slices,
    int64_t n_tiles, n_starts;   //   tiles, segment starts
    int64_t n_esum;              // level emit: chunks; slice emit: segment starts
    int64_t tail_nodes;    // widest level the single-CTA tail takes
    int64_t grid_levels;   // Lg: levels 1..Lg use the whole grid
    int64_t tail_total;    // nodes of the tail buffer (levels Lg+1..L, padded)
    int64_t TB;            // leaf-table block length in values
    int32_t vbits;         // bits of the value index inside a leaf code
    EmitMode emit;
    // dataflow sweep (flow.hpp): one value a node; replaces the tail and the
    // two level buffers with three level buffers, block records and flags
    bool flow = false;
    int64_t fblk, fdeps, fgran, forder;   // grammar part: block records, dependencies, granules, order
    int64_t fb0, fb1, fb2, fflags, fdone; // scratch: level buffers, ready flags, per-level counters
    int64_t n_fblocks, n_fdeps, n_fgran, fbuf_values, final_k0;

    bool chunked() const { return emit != EMIT_ROWS; }   // chunk or segment sums, esum
    bool has_rv() const { return emit != EMIT_LEVEL; }
};

inline bool policy_is_f32(gc_policy p) { return p == GC_F32_SUM || p == GC_F32_MIN_PLUS; }
// Right-hand sides a node's value may hold: the float32 sum takes the batch
// widths of Appendix A (1, 4, 8, ..., 256), the tropical policy 1 or 16, the
// exact and Boolean policies one.
inline bool policy_width_ok(gc_policy p, int64_t k) {
    if (p == GC_F32_SUM) return k == 1 || k == 4 || k == 8 || k == 16 || k == 32 || k == 64 || k == 128 || k == 256;
    if (p == GC_F32_MIN_PLUS) return k == 1 || k == 16;
    return k == 1;
}
inline int64_t policy_elem_bytes(gc_policy p) { return policy_is_f32(p) ? 4 : 8; }

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
    return !long_rows ? EMIT_ROWS : k_max == 1 ? EMIT_SLICE : EMIT_LEVEL;
}

// Device view of a layered grammar. The pages' pass-through nodes (Sec. 4.2)
// copy a value one level up; a chain of them carries a rule u to its highest
// parent. With carry slots (used for 16-wide values, whose level buffers do
// not stay in L2, so each copy costs a DRAM round trip) the device does not
// execute the copies: every rule a parent reads two or more levels above it
// (u has pass-throughs) stores its value once, when its level is computed,
// into a carry slot, and parents read the slot where the layered grammar
// reads u's chain element. Without carry slots (one-wide values, whose copies
// read the level just written, in L2) the view is the layered grammar itself. x (+) identity = x for every
// policy, so the values are the same; the node stream shrinks by the
// pass-throughs. Each level lists its roots first (carried ones first), then
// its other rules (carried ones first), each group in the packed order, so a
// level's carried nodes are two runs of positions and their carry slots
// follow from position. Child references: >= 0 a slot of the level below,
// -2 - p terminal p, below -1 - alpha a carry slot (carry_ref / carry_slot).
inline int32_t carry_ref(int64_t slot, int64_t alpha) { return (int32_t)(-(alpha + 2) - slot); }
inline int64_t carry_slot(int32_t c, int64_t alpha) { return -(int64_t)c - (alpha + 2); }

inline Grammar device_view(const Grammar& g, bool carry) {
    const int64_t L = g.L, R = g.n_rules(), A = g.alpha();
    Grammar d;
    if (!carry) {
        d.n = g.n;
        d.m = g.m;
        d.nnz = g.nnz;
        d.L = L;
        d.V = g.V;
        d.term_col = g.term_col;
        d.term_vidx = g.term_vidx;
        d.slp.c_off = g.slp.c_off;
        d.lvl_off = g.lvl_off;
        d.lvl_roots = g.lvl_roots;
        d.root_off = g.root_off;
        d.n_roots = g.n_roots;
        d.nodes = g.nodes;
        d.node_id = g.node_id;
        d.c_ref = g.c_ref;
        d.carry_roots.assign((size_t)L + 2, 0);
        d.carry_rest.assign((size_t)L + 2, 0);
        d.carry_off.assign((size_t)L + 2, 0);
        return d;
    }
    d.n = g.n;
    d.m = g.m;
    d.nnz = g.nnz;
    d.L = L;
    d.V = g.V;
    d.term_col = g.term_col;
    d.term_vidx = g.term_vidx;
    d.slp.c_off = g.slp.c_off;
    d.lvl_roots = g.lvl_roots;
    d.root_off = g.root_off;
    d.n_roots = g.n_roots;
    std::vector<char> carried((size_t)R, 0);
    for (int32_t id : g.node_id)
        if (id < 0) carried[-(int64_t)id - 1] = 1;
    std::vector<int32_t> pos((size_t)R, -1), cslot((size_t)R, -1);
    d.lvl_off.assign((size_t)L + 2, 0);
    d.carry_roots.assign((size_t)L + 2, 0);
    d.carry_rest.assign((size_t)L + 2, 0);
    d.carry_off.assign((size_t)L + 2, 0);
    d.node_id.reserve((size_t)R);
    int64_t off = 0, coff = 0;
    for (int64_t k = 1; k <= L; ++k) {
        d.lvl_off[k] = off;
        d.carry_off[k] = coff;
        const int64_t q0 = g.lvl_off[k], qr = q0 + g.lvl_roots[k], q1 = g.lvl_off[k + 1];
        auto take = [&](int64_t a, int64_t b, bool want_carried, int64_t& count) {
            for (int64_t q = a; q < b; ++q) {
                const int32_t u = g.node_id[q];
                if (u < 0 || (bool)carried[u] != want_carried) continue;   // pass-throughs are dropped
                pos[u] = (int32_t)(off - d.lvl_off[k]);
                if (want_carried) cslot[u] = (int32_t)coff++;
                d.node_id.push_back(u);
                ++off;
                ++count;
            }
        };
        int64_t cr = 0, cn = 0, rest = 0;
        take(q0, qr, true, cr);
        take(q0, qr, false, rest);
        take(qr, q1, true, cn);
        take(qr, q1, false, rest);
        d.carry_roots[k] = cr;
        d.carry_rest[k] = cn;
    }
    d.lvl_off[L + 1] = off;
    d.carry_off[L + 1] = coff;
    d.n_carry = coff;
    if (coff >= (int64_t)INT32_MAX - A - 2) fail(GC_ERR_UNSUPPORTED, "too many carried nodes for 31-bit references");
    // children: a rule at level k reads level k-1 slots; a host chain element
    // there stands for its rule's carry slot
    d.nodes.assign((size_t)2 * off, 0);
    for (int64_t k = 1; k <= L; ++k)
        for (int64_t i = d.lvl_off[k]; i < d.lvl_off[k + 1]; ++i) {
            const int32_t u = d.node_id[i];
            const int32_t kids[2] = {g.slp.rule_a[u], g.slp.rule_b[u]};
            for (int t = 0; t < 2; ++t) {
                const int32_t c = kids[t];
                int32_t ref;
                if (c < 0) {
                    ref = c - 1;                                   // terminal -c-1 -> -2 - p
                } else if (g.rule_level[c] == k - 1) {
                    ref = pos[c];
                } else {
                    if (cslot[c] < 0) fail(GC_ERR_INVALID_GRAMMAR, "a rule skips levels without a carry slot");
                    ref = carry_ref(cslot[c], A);
                }
                d.nodes[2 * i + t] = ref;
            }
        }
    // C's root slots in the new order
    d.c_ref.resize(g.c_ref.size());
    for (size_t e = 0; e < g.c_ref.size(); ++e) {
        const int32_t c = g.c_ref[e];
        if (c < 0) {
            d.c_ref[e] = c;
            continue;
        }
        const int64_t k = std::upper_bound(g.root_off.begin() + 1, g.root_off.begin() + L + 2, (int64_t)c) -
                          g.root_off.begin() - 1;
        const int32_t u = g.node_id[g.lvl_off[k] + (c - g.root_off[k])];
        d.c_ref[e] = (int32_t)(g.root_off[k] + pos[u]);
    }
    return d;
}

// Checks a device view: every child of a level-k node is a terminal, a slot
// of level k-1, the identity (a pass-through's second child) or the carry slot
// of a rule at least two levels down; carried runs lie inside their levels; C
// names terminals and roots.
inline void validate_device_view(const Grammar& d) {
    const int64_t L = d.L, A = d.alpha();
    auto bad = [](const char* what) { fail(GC_ERR_INVALID_GRAMMAR, std::string("device view: ") + what); };
    if ((int64_t)d.lvl_off.size() != L + 2 || (int64_t)d.carry_off.size() != L + 2 ||
        d.lvl_off[L + 1] * 2 != (int64_t)d.nodes.size() || d.carry_off[L + 1] != d.n_carry)
        bad("level tables");
    std::vector<int64_t> slot_level((size_t)d.n_carry, 0);
    for (int64_t k = 1; k <= L; ++k) {
        const int64_t w = d.lvl_off[k + 1] - d.lvl_off[k];
        if (w < 0 || d.lvl_roots[k] > w || d.carry_roots[k] > d.lvl_roots[k] ||
            d.lvl_roots[k] + d.carry_rest[k] > w || d.carry_off[k + 1] - d.carry_off[k] != d.carry_roots[k] + d.carry_rest[k])
            bad("level sizes");
        for (int64_t s = d.carry_off[k]; s < d.carry_off[k + 1]; ++s) slot_level[s] = k;
    }
    for (int64_t k = 1; k <= L; ++k) {
        const int64_t wprev = k > 1 ? d.lvl_off[k] - d.lvl_off[k - 1] : 0;
        for (int64_t i = 2 * d.lvl_off[k]; i < 2 * d.lvl_off[k + 1]; ++i) {
            const int32_t c = d.nodes[i];
            const bool ok = c >= 0                 ? c < wprev
                            : c == -1              ? (i & 1) == 1 && k >= 2
                            : c >= -(A + 1)        ? true
                            : (carry_slot(c, A) < d.n_carry && slot_level[carry_slot(c, A)] < k - 1);
            if (!ok || (k == 1 && c > -2) || (k == 1 && c < -(A + 1))) bad("child reference out of range");
        }
    }
    for (int32_t c : d.c_ref)
        if (c >= 0 ? c >= d.n_roots : (-(int64_t)c - 1) > A) bad("C reference out of range");
}

// widest level of the tail that one CTA finishes: 4,096 one-lane values,
// 16 KB of values a level for wider ones (1,024 16-wide values), at least 256
inline int64_t tail_width(int32_t k_max) { return k_max == 1 ? 4096 : std::max<int64_t>(256, 16384 / k_max); }
// the slice emit's tail runs on a group of CTAs beside the slices, so it
// takes the levels up to this width
constexpr int64_t kSliceTailNodes = 65536;

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

// Level emit: chunks of C's early references (terminals and levels 1..Lg),
// grouped by the level of their symbol, in chunks of one (level, row): a root
// slot of that level's buffer, or a terminal as -2 - its leaf code. References
// to the tail levels are kept per row as tail-buffer indices.
struct EmitPlan {
    std::vector<int32_t> cref;      // grouped by (level, row): root slots, or -2 - leaf code
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

// Row r's references into the tail levels (levels > Lg), as tail-buffer indices.
inline void plan_late(const Grammar& g, int64_t Lg, std::vector<int32_t>& off, std::vector<int32_t>& ref) {
    const std::vector<int64_t>& co = g.slp.c_off;
    const std::vector<int64_t> toff = tail_offsets(g, Lg);
    off.assign((size_t)g.n + 1, 0);
    ref.clear();
    for (int64_t r = 0; r < g.n; ++r) {
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            const int32_t c = g.c_ref[e];
            const int64_t k = ref_level(g, c);
            if (k > Lg) ref.push_back((int32_t)(toff[k] + c - g.root_off[k]));
        }
        off[r + 1] = (int32_t)ref.size();
    }
}

inline EmitPlan plan_level_emit(const Grammar& g, int64_t Lg) {
    const int64_t L = g.L, n = g.n;
    const std::vector<int64_t>& co = g.slp.c_off;
    const size_t C = g.c_ref.size();
    const int32_t vbits = value_bits((int64_t)g.V.size());
    EmitPlan p;
    plan_late(g, Lg, p.late_off, p.late_ref);
    std::vector<int32_t> lev(C), pos(C);
    for (size_t e = 0; e < C; ++e) {
        const int32_t c = g.c_ref[e];
        const int64_t k = ref_level(g, c);
        lev[e] = (int32_t)k;
        // a terminal p = -c-2 as -2 - its leaf code (evaluated where it is
        // read); a root as its slot in its level's buffer
        pos[e] = c < 0 ? (int32_t)(-2 - (((int64_t)g.term_col[-c - 2] << vbits) | g.term_vidx[-c - 2]))
                       : (int32_t)(c - g.root_off[k]);
    }
    // counting sort of the early references by level, stable in row-major order
    std::vector<int64_t> cnt((size_t)Lg + 2, 0);
    for (size_t e = 0; e < C; ++e)
        if (lev[e] <= Lg) ++cnt[lev[e] + 1];
    for (int64_t k = 0; k <= Lg; ++k) cnt[k + 1] += cnt[k];
    p.cref.resize((size_t)cnt[Lg + 1]);
    std::vector<int64_t> at(cnt.begin(), cnt.end() - 1);
    std::vector<int32_t> row_of(p.cref.size());
    for (int64_t r = 0; r < n; ++r)
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            if (lev[e] > Lg) continue;
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

// Slice emit: the early references as [T | RV] indices x. Slices are runs of
// values [x0[s], x0[s+1]) that start on multiples of kSliceStep, at most S
// values wide, with their costs balanced (slice_bounds); slice s holds offset
// x - x0[s]. Within a slice the references
// keep row-major C order, so a row's references into it form one segment.
// A slice's segments are packed back to back, in order, into tiles of
// kTileRefs references (32 lanes x 8): a segment that runs past the end of a
// tile goes on in the next one as a new piece, and only the slice's last tile
// is padded (the rest is a segment with id -1), so a slice of R references
// takes ceil(R / kTileRefs) tiles. Every piece gets its own id, in (row,
// slice, piece) order, so a row's sums are contiguous.
constexpr int64_t kTileRefs = 256;

struct SlicePlan {
    int64_t S = 0, nslices = 0, ntiles = 0, nids = 0;
    std::vector<int32_t> x0;        // nslices+1
    std::vector<int32_t> stile;     // nslices+1
    std::vector<int32_t> sorder;    // nslices: slices by decreasing tile count
    std::vector<uint16_t> sref;     // kTileRefs per tile
    std::vector<uint8_t> sflag;     // kTileRefs/8 per tile
    std::vector<int32_t> tsid;      // one per segment start: its id (-1: padding)
    std::vector<int32_t> tile_sid;  // ntiles+1
    std::vector<int32_t> row_seg;   // n+1: row r's ids
    std::vector<int32_t> row_pos;   // nids: segment start of each id
    std::vector<int32_t> late_off, late_ref;
};

// [T | RV] index of an early reference (terminal or root of levels 1..Lg).
inline int64_t slice_index(int64_t TB, int32_t c) { return c < 0 ? -c - 1 : TB + c; }

// Slice boundaries from the references' counts per kSliceStep values. A
// slice's cost is its references plus its values / kSliceValueCost (the
// staging); slices are cut greedily at the smallest cost cap that gives at
// most kSliceTarget * r slices (r rounds of slices over the CTAs).
inline std::vector<int32_t> slice_bounds(const Grammar& g, int64_t TB, int64_t Lg, int64_t S) {
    const int64_t X = TB + (Lg >= 1 ? g.root_off[Lg + 1] : 0);   // early references lie below X
    const int64_t nb = (X + kSliceStep - 1) / kSliceStep;
    std::vector<int64_t> cost((size_t)nb, kSliceStep / kSliceValueCost);
    for (int32_t c : g.c_ref)
        if (ref_level(g, c) <= Lg) ++cost[slice_index(TB, c) / kSliceStep];
    auto cut = [&](int64_t cap, std::vector<int32_t>* x0) {
        int64_t count = nb > 0 ? 1 : 0, sum = 0, width = 0;
        for (int64_t b = 0; b < nb; ++b) {
            if (width > 0 && (width + kSliceStep > S || sum + cost[b] > cap)) {
                if (x0) x0->push_back((int32_t)(b * kSliceStep));
                ++count;
                sum = width = 0;
            }
            sum += cost[b];
            width += kSliceStep;
        }
        return count;
    };
    int64_t total = 0;
    for (int64_t c : cost) total += c;
    // one round more than the S-value limit alone needs, so that the costs can
    // be balanced (in one round, slices full of values leave the few others
    // all the densely referenced values)
    const int64_t fewest = cut(total, nullptr);
    const int64_t target = kSliceTarget * ((fewest + kSliceTarget - 1) / kSliceTarget + 1);
    int64_t lo = 1, hi = std::max<int64_t>(total, 1);   // cut(hi) <= target
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (cut(mid, nullptr) <= target) hi = mid;
        else lo = mid + 1;
    }
    std::vector<int32_t> x0{0};
    cut(hi, &x0);
    if (nb > 0) x0.push_back((int32_t)X);
    return x0;
}

inline int64_t slice_of(const std::vector<int32_t>& x0, int64_t x) {
    return std::upper_bound(x0.begin() + 1, x0.end(), (int32_t)x) - x0.begin() - 1;
}

// Segments of the early references: for each slice, (row, first, length) in
// row order, with the references' offsets in `off` (slice by slice).
struct SliceSegments {
    std::vector<int32_t> x0;
    std::vector<int64_t> sseg;                 // nslices+1
    std::vector<int32_t> seg_row;
    std::vector<int64_t> seg_first, seg_len;   // into off
    std::vector<uint16_t> off;
};

inline SliceSegments slice_segments(const Grammar& g, int64_t TB, int64_t Lg, int64_t S, bool with_offsets) {
    const std::vector<int64_t>& co = g.slp.c_off;
    const size_t C = g.c_ref.size();
    SliceSegments z;
    z.x0 = slice_bounds(g, TB, Lg, S);
    const int64_t NS = (int64_t)z.x0.size() - 1;
    std::vector<int32_t> sl(C, -1);   // slice of each early reference, -1 for late ones
    for (size_t e = 0; e < C; ++e)
        if (ref_level(g, g.c_ref[e]) <= Lg) sl[e] = (int32_t)slice_of(z.x0, slice_index(TB, g.c_ref[e]));
    std::vector<int64_t> last((size_t)NS, -1), nref((size_t)NS + 1, 0), nseg((size_t)NS + 1, 0);
    for (int64_t r = 0; r < g.n; ++r)
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            if (sl[e] < 0) continue;
            ++nref[sl[e] + 1];
            if (last[sl[e]] != r) {
                last[sl[e]] = r;
                ++nseg[sl[e] + 1];
            }
        }
    for (int64_t s = 0; s < NS; ++s) {
        nref[s + 1] += nref[s];
        nseg[s + 1] += nseg[s];
    }
    z.sseg = nseg;
    z.seg_row.assign((size_t)nseg[NS], 0);
    z.seg_first.assign((size_t)nseg[NS], 0);
    z.seg_len.assign((size_t)nseg[NS], 0);
    if (with_offsets) z.off.resize((size_t)nref[NS]);
    std::vector<int64_t> at_ref(nref.begin(), nref.end() - 1), at_seg(nseg.begin(), nseg.end() - 1);
    std::fill(last.begin(), last.end(), -1);
    for (int64_t r = 0; r < g.n; ++r)
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            if (sl[e] < 0) continue;
            const int32_t s = sl[e];
            if (last[s] != r) {
                last[s] = r;
                z.seg_row[at_seg[s]] = (int32_t)r;
                z.seg_first[at_seg[s]] = at_ref[s];
                ++at_seg[s];
            }
            ++z.seg_len[at_seg[s] - 1];
            if (with_offsets) z.off[at_ref[s]] = (uint16_t)(slice_index(TB, g.c_ref[e]) - z.x0[s]);
            ++at_ref[s];
        }
    return z;
}

// Tiles and ids of the packing described above, from a slice's segment lengths.
struct TileCounts {
    int64_t tiles = 0, starts = 0, ids = 0;
};
// Pieces of each segment under that packing (pieces[j] for segment j).
inline TileCounts count_tiles(const SliceSegments& z, std::vector<int32_t>* pieces = nullptr) {
    TileCounts t;
    const int64_t NS = (int64_t)z.x0.size() - 1;
    if (pieces) pieces->assign(z.seg_len.size(), 0);
    for (int64_t s = 0; s < NS; ++s) {
        int64_t fill = kTileRefs;   // no open tile yet
        for (int64_t j = z.sseg[s]; j < z.sseg[s + 1]; ++j)
            for (int64_t left = z.seg_len[j]; left > 0;) {
                if (fill == kTileRefs) {
                    ++t.tiles;
                    fill = 0;
                }
                const int64_t take = std::min(left, kTileRefs - fill);
                ++t.starts;
                ++t.ids;
                if (pieces) ++(*pieces)[j];
                fill += take;
                left -= take;
            }
        if (fill > 0 && fill < kTileRefs) ++t.starts;   // padding of the slice's last tile
    }
    return t;
}

inline SlicePlan plan_slice_emit(const Grammar& g, int64_t TB, int64_t Lg, int64_t S) {
    const int64_t n = g.n;
    SliceSegments z = slice_segments(g, TB, Lg, S, true);
    SlicePlan p;
    p.S = S;
    p.x0 = z.x0;
    p.nslices = (int64_t)z.x0.size() - 1;
    plan_late(g, Lg, p.late_off, p.late_ref);
    const int64_t NS = p.nslices;
    // ids: per row, its pieces in (slice, piece) order
    std::vector<int32_t> pieces;
    count_tiles(z, &pieces);
    std::vector<int64_t> row_ids((size_t)n + 1, 0);
    for (int64_t j = 0; j < (int64_t)z.seg_row.size(); ++j) row_ids[z.seg_row[j] + 1] += pieces[j];
    for (int64_t r = 0; r < n; ++r) row_ids[r + 1] += row_ids[r];
    p.row_seg.assign(row_ids.begin(), row_ids.end());
    p.nids = row_ids[n];
    std::vector<int64_t> next_id(row_ids.begin(), row_ids.end() - 1);
    // slices in order: each row's pieces are met in (slice, piece) order
    p.stile.assign((size_t)NS + 1, 0);
    int64_t fill = kTileRefs;
    auto open_tile = [&]() {
        p.sref.resize(p.sref.size() + kTileRefs, 0);
        p.sflag.resize(p.sflag.size() + kTileRefs / 8, 0);
        p.tile_sid.push_back((int32_t)p.tsid.size());
        ++p.ntiles;
        fill = 0;
    };
    for (int64_t s = 0; s < NS; ++s) {
        p.stile[s] = p.ntiles;
        fill = kTileRefs;
        for (int64_t j = z.sseg[s]; j < z.sseg[s + 1]; ++j) {
            int64_t q = z.seg_first[j];
            for (int64_t left = z.seg_len[j]; left > 0;) {
                if (fill == kTileRefs) open_tile();
                const int64_t take = std::min(left, kTileRefs - fill);
                const int64_t base = (p.ntiles - 1) * kTileRefs + fill;
                p.sflag[(p.ntiles - 1) * (kTileRefs / 8) + fill / 8] |= (uint8_t)(1u << (fill % 8));
                p.tsid.push_back((int32_t)next_id[z.seg_row[j]]++);
                for (int64_t i = 0; i < take; ++i) p.sref[base + i] = z.off[q + i];
                q += take;
                fill += take;
                left -= take;
            }
        }
        if (fill > 0 && fill < kTileRefs) {   // pad the slice's last tile
            p.sflag[(p.ntiles - 1) * (kTileRefs / 8) + fill / 8] |= (uint8_t)(1u << (fill % 8));
            p.tsid.push_back(-1);
        }
    }
    p.stile[NS] = p.ntiles;
    p.tile_sid.push_back((int32_t)p.tsid.size());
    p.row_pos.assign((size_t)p.nids, -1);
    for (size_t k = 0; k < p.tsid.size(); ++k)
        if (p.tsid[k] >= 0) p.row_pos[p.tsid[k]] = (int32_t)k;
    // processing order: heaviest slices first, so that CTAs taking a second
    // slice take light ones
    p.sorder.resize((size_t)NS);
    for (int64_t i = 0; i < NS; ++i) p.sorder[i] = (int32_t)i;
    std::stable_sort(p.sorder.begin(), p.sorder.end(), [&](int32_t a, int32_t b) {
        return p.stile[a + 1] - p.stile[a] > p.stile[b + 1] - p.stile[b];
    });
    return p;
}

// Counts of plan_slice_emit's arrays, without building it.
struct SliceCounts {
    int64_t slices = 0, tiles = 0, starts = 0, ids = 0, late = 0;
};
inline SliceCounts count_slice_emit(const Grammar& g, int64_t TB, int64_t Lg, int64_t S) {
    const SliceSegments z = slice_segments(g, TB, Lg, S, false);
    const TileCounts t = count_tiles(z);
    SliceCounts c;
    c.slices = (int64_t)z.x0.size() - 1;
    c.tiles = t.tiles;
    c.starts = t.starts;
    c.ids = t.ids;
    for (int32_t r : g.c_ref)
        if (ref_level(g, r) > Lg) ++c.late;
    return c;
}

// Checks a plan against the grammar before it reaches the device: every
// chunk lies inside cref and holds references of its own level only (T for
// level 0, that level's roots otherwise), chunk ids are a permutation that
// row_ech splits by row, and every tail reference lies inside the tail buffer.
inline void check_late(const std::vector<int32_t>& off, const std::vector<int32_t>& ref, const Grammar& g,
                       int64_t Lg, const char* what) {
    const std::vector<int64_t> toff = tail_offsets(g, Lg);
    auto bad = [&](const char* why) { fail(GC_ERR_INVALID_GRAMMAR, std::string(what) + ": " + why); };
    if ((int64_t)off.size() != g.n + 1 || off[0] != 0 || off[g.n] != (int64_t)ref.size()) bad("tail reference ranges");
    for (int64_t r = 0; r < g.n; ++r)
        if (off[r + 1] < off[r]) bad("tail reference ranges decrease");
    for (int32_t t : ref)
        if (t < 0 || t >= toff[g.L + 1]) bad("tail reference outside the tail buffer");
}

inline void validate_emit_plan(const EmitPlan& p, const Grammar& g, int64_t Lg) {
    const int64_t n = g.n, L = g.L, nch = (int64_t)p.echunk.size() / 4;
    auto bad = [](const char* what) { fail(GC_ERR_INVALID_GRAMMAR, std::string("emit plan: ") + what); };
    if ((int64_t)p.ech.size() != L + 2 || p.ech[0] != 0 || p.ech[L + 1] != nch) bad("level chunk ranges");
    if ((int64_t)p.row_ech.size() != n + 1 || p.row_ech[0] != 0 || p.row_ech[n] != nch) bad("row chunk ranges");
    check_late(p.late_off, p.late_ref, g, Lg, "emit plan");
    std::vector<char> seen((size_t)nch, 0);
    for (int64_t k = 0; k <= L; ++k) {
        if (p.ech[k + 1] < p.ech[k] || (k > Lg && p.ech[k + 1] != p.ech[k])) bad("level chunk ranges");
        // terminals (level 0: -2 - a leaf code) or level k's roots (their slots)
        const int32_t vbits = value_bits((int64_t)g.V.size());
        const int64_t nv = (int64_t)g.V.size(), leaf_max = (int64_t)g.m << vbits;
        auto ok = [&](int64_t v) {
            if (k == 0) return v <= -2 && -v - 2 < leaf_max && ((-v - 2) & ((1 << vbits) - 1)) < nv;
            return v >= 0 && v < g.lvl_roots[k];
        };
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
        if (p.row_ech[r + 1] < p.row_ech[r]) bad("row ranges decrease");
}

// Same for a slice plan: slice bounds and tile ranges are consistent, every
// tile starts a segment at its first reference, its starts match its ids,
// every id is -1 or names one esum slot exactly once, every reference of a
// real segment names a T entry or a root of levels 1..Lg inside its slice,
// and row_seg covers the ids.
inline void validate_slice_plan(const SlicePlan& p, const Grammar& g, int64_t TB, int64_t Lg) {
    const int64_t n = g.n, NS = p.nslices, S = p.S, NT = p.ntiles;
    auto bad = [](const char* what) { fail(GC_ERR_INVALID_GRAMMAR, std::string("slice plan: ") + what); };
    if (S < 1 || S > 65536 || (int64_t)p.x0.size() != NS + 1 || (int64_t)p.stile.size() != NS + 1) bad("slice size");
    if ((int64_t)p.sref.size() != NT * kTileRefs || (int64_t)p.sflag.size() != NT * (kTileRefs / 8) ||
        (int64_t)p.tile_sid.size() != NT + 1 || p.tile_sid[0] != 0 || p.tile_sid[NT] != (int64_t)p.tsid.size())
        bad("tile arrays");
    if ((int64_t)p.row_seg.size() != n + 1 || p.row_seg[0] != 0 || p.row_seg[n] != p.nids) bad("row id ranges");
    for (int64_t r = 0; r < n; ++r)
        if (p.row_seg[r + 1] < p.row_seg[r]) bad("row id ranges decrease");
    check_late(p.late_off, p.late_ref, g, Lg, "slice plan");
    const int64_t x_hi = TB + (Lg >= 1 ? g.root_off[Lg + 1] : 0);
    std::vector<char> seen((size_t)p.nids, 0);
    if (p.stile[0] != 0 || p.stile[NS] != NT) bad("slice tile ranges");
    for (int64_t s = 0; s < NS; ++s) {
        if (p.x0[s] % kSliceStep != 0 || p.x0[s + 1] <= p.x0[s] || p.x0[s + 1] - p.x0[s] > S) bad("slice bounds");
        if (p.stile[s + 1] < p.stile[s]) bad("slice tile ranges decrease");
        for (int64_t t = p.stile[s]; t < p.stile[s + 1]; ++t) {
            if (!(p.sflag[t * (kTileRefs / 8)] & 1u)) bad("tile does not start a segment");
            int64_t k = p.tile_sid[t] - 1, id = -1;
            for (int64_t i = 0; i < kTileRefs; ++i) {
                if (p.sflag[t * (kTileRefs / 8) + i / 8] & (1u << (i % 8))) {
                    if (++k >= p.tile_sid[t + 1]) bad("tile starts exceed its ids");
                    id = p.tsid[k];
                    if (id < -1 || id >= p.nids || (id >= 0 && seen[id])) bad("segment ids");
                    if (id >= 0) seen[id] = 1;
                }
                if (id < 0) continue;   // padding
                const int64_t x = p.x0[s] + p.sref[t * kTileRefs + i];
                if (x >= p.x0[s + 1] || !((x >= 0 && x <= g.alpha()) || (x >= TB && x < x_hi)))
                    bad("reference outside its slice, T and RV");
            }
            if (k + 1 != p.tile_sid[t + 1]) bad("tile starts and ids differ");
        }
    }
    for (int64_t i = 0; i < p.nids; ++i)
        if (!seen[i]) bad("an id is never written");
    if ((int64_t)p.sorder.size() != NS) bad("slice order");
    {
        std::vector<char> sseen((size_t)NS, 0);
        for (int32_t v : p.sorder) {
            if (v < 0 || v >= NS || sseen[v]) bad("slice order");
            sseen[v] = 1;
        }
    }
    if ((int64_t)p.row_pos.size() != p.nids) bad("row positions");
    for (int64_t i = 0; i < p.nids; ++i)
        if (p.row_pos[i] < 0 || p.row_pos[i] >= (int64_t)p.tsid.size() || p.tsid[p.row_pos[i]] != i)
            bad("row positions");
}

// Counts of plan_level_emit's arrays, without building it: chunks, early
// references and tail references.
struct EmitCounts {
    int64_t chunks = 0, wide = 0, late = 0;
};
inline EmitCounts count_level_emit(const Grammar& g, int64_t Lg) {
    const std::vector<int64_t>& co = g.slp.c_off;
    std::vector<int64_t> per((size_t)Lg + 1, 0);
    EmitCounts t;
    for (int64_t r = 0; r < g.n; ++r) {
        std::fill(per.begin(), per.end(), 0);
        for (int64_t e = co[r]; e < co[r + 1]; ++e) {
            const int64_t k = ref_level(g, g.c_ref[e]);
            if (k > Lg) ++t.late;
            else ++per[k];
        }
        for (int64_t k = 0; k <= Lg; ++k) {
            t.chunks += (per[k] + kEmitChunkSyms - 1) / kEmitChunkSyms;
            t.wide += per[k];
        }
    }
    return t;
}

// Counts of a dataflow block plan (flow.hpp) that size the arena.
struct FlowCounts {
    int64_t nblocks = 0, ndeps = 0, ngran = 0, buf_values = 0, final_k0 = 0;
};

// Sizes of the arena for the device view g (device_view) of a grammar; with
// fc, for the dataflow sweep of that block plan (every level is swept by the
// blocks, so there is no tail: grid_levels = L).
inline DevLayout device_layout(const Grammar& g, gc_policy p, int32_t k_max, const FlowCounts* fc = nullptr) {
    DevLayout d{};
    const int64_t L = g.L, C = (int64_t)g.c_ref.size(), A = g.alpha();
    d.value_bytes = policy_elem_bytes(p) * k_max;
    d.vbits = value_bits((int64_t)g.V.size());
    d.TB = leaf_block(A);
    d.emit = emit_mode(g, k_max);
    d.flow = fc != nullptr;
    d.tail_nodes = d.emit == EMIT_SLICE ? kSliceTailNodes : tail_width(k_max);
    d.grid_levels = d.flow ? L : grid_level_count(g, d.tail_nodes);
    d.tail_total = tail_offsets(g, d.grid_levels)[L + 1];
    if (d.flow) {
        d.n_fblocks = fc->nblocks;
        d.n_fdeps = fc->ndeps;
        d.n_fgran = fc->ngran;
        d.fbuf_values = fc->buf_values;
        d.final_k0 = fc->final_k0;
    }
    d.n_nodes_padded = 0;
    for (int64_t k = 1; k <= L; ++k) d.n_nodes_padded += pad_nodes(g.lvl_off[k + 1] - g.lvl_off[k]);
    EmitCounts ec;
    SliceCounts sc;
    if (d.emit == EMIT_LEVEL) {
        ec = count_level_emit(g, d.grid_levels);
        d.n_echunks = ec.chunks;
        d.n_esum = ec.chunks;
        d.n_late = ec.late;
        d.n_early = ec.wide;
    } else if (d.emit == EMIT_SLICE) {
        d.slice = slice_len(d.value_bytes);
        sc = count_slice_emit(g, d.TB, d.grid_levels, d.slice);
        d.n_slices = sc.slices;
        d.n_tiles = sc.tiles;
        d.n_starts = sc.starts;
        d.n_echunks = sc.ids;
        d.n_esum = sc.starts;
        d.n_late = sc.late;
    }
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        int64_t at = o;
        o = align256(o + bytes);
        return at;
    };
    d.nodes = take(8 * d.n_nodes_padded);
    d.levels = take(8 * kLevelRows * (L + 2));
    if (d.flow) {
        d.fblk = take(kFlowBlkBytes * d.n_fblocks);
        d.forder = take(4 * d.n_fblocks);
        d.fdeps = take(4 * d.n_fdeps);
        d.fgran = take(4 * d.n_fgran);
    }
    d.V = take(policy_elem_bytes(p) * std::max<int64_t>(1, (int64_t)g.V.size()));
    d.leaf = take(4 * A);
    if (d.emit == EMIT_LEVEL) {
        d.cref = take(4 * d.n_early);
        d.echunk = take(16 * d.n_echunks);
    } else if (d.emit == EMIT_SLICE) {
        d.sref = take(2 * kTileRefs * d.n_tiles);
        d.sflag = take(kTileRefs / 8 * d.n_tiles);
        d.tile_sid = take(4 * (d.n_tiles + 1));
        d.row_pos = take(4 * d.n_echunks);
        d.sx0 = take(4 * (d.n_slices + 1));
        d.stile = take(4 * (d.n_slices + 1));
        d.sorder = take(4 * d.n_slices);
    }
    if (d.chunked()) {
        d.row_ech = take(4 * (g.n + 1));
        d.late_off = take(4 * (g.n + 1));
        d.late_ref = take(4 * d.n_late);
    } else {
        d.c_off = take(4 * (g.n + 1));
        d.c_ref = take(4 * C);
    }
    d.grammar_bytes = o;
    const int64_t w = g.max_width();
    if (d.flow) {
        d.fb0 = take(d.value_bytes * d.fbuf_values);
        d.fb1 = take(d.value_bytes * d.fbuf_values);
        d.fb2 = take(d.value_bytes * d.fbuf_values);
        d.fflags = take(4 * std::max<int64_t>(1, d.n_fblocks));
        d.fdone = take(8 * (L + 2));
        d.buf0 = d.buf1 = d.tbuf = d.carry = take(0);
    } else {
        d.buf0 = take(d.value_bytes * std::max<int64_t>(1, w));
        d.buf1 = take(d.value_bytes * std::max<int64_t>(1, w));
        d.tbuf = take(d.value_bytes * d.tail_total);
        d.carry = take(d.value_bytes * std::max<int64_t>(1, g.n_carry));
    }
    if (d.chunked()) d.esum = take(d.value_bytes * d.n_esum);
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
    if (p != GC_F32_SUM && p != GC_I64_SUM && p != GC_BOOL_OR && p != GC_F32_MIN_PLUS)
        fail(GC_ERR_ARG, "unknown policy");
    if (!policy_width_ok(p, k_max))
        fail(GC_ERR_ARG, "k_max must be 1, or 4, 8, ..., 256 for GC_F32_SUM, or 16 for GC_F32_MIN_PLUS");
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
