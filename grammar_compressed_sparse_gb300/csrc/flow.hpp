// Block plan of the dataflow sweep (host-side arithmetic only; used by
// gc_layout and gc_upload for handles with one value per node).
//
// The level-synchronous sweep of Sec. 4.3 evaluates level k from level k-1
// only (Lemma 3.3), and any order within a level is correct (Lemma 3.1). The
// packed order sorts each level by the first column of a node's expansion
// (roots first), so the children of a run of consecutive level-k nodes lie
// in two narrow slot ranges of level k-1: one among its roots, one among its
// other nodes. The dataflow sweep cuts every level into blocks of consecutive
// nodes and gives each block
//   * up to two windows: slot ranges of level k-1 that hold almost all of its
//     children, copied into shared memory with one bulk copy each;
//   * outlier granules: 16-byte pieces of level k-1 around the few children
//     outside the windows, copied the same way;
//   * its dependencies: the level k-1 blocks that write any of those slots.
// A block starts once its dependencies have published their values (per-block
// ready flags instead of a grid barrier per level). Every child reference of
// the block is re-encoded as an index into the block's staged values, so a
// node reads its two children from shared memory.
//
// The narrow top levels form one final block: the whole level below them is
// its window, and the block computes its levels one after the other inside
// shared memory, where the top levels' values stay.
//
// Node references in the uploaded pair array (one int2 per padded node, the
// layout of the packed grammar):
//   c >= 0   index into the block's staged values (window 1, window 2, outlier
//            granules, then in the final block its own levels' values)
//   c == -1  the combine identity (second child of a pass-through, Sec. 4.2)
//   c <= -2  a terminal, as its leaf code q = -c - 2 = column << vbits | value
//            index, evaluated in place as V[l] (x) x[j]
//
// Level buffers: three, level k written to buffer k % 3. A block of level k
// reads buffer (k-1) % 3; the buffer it writes last held level k-3, which
// level k-2 reads, so a block of level k also waits for level k-2 to finish.
#pragma once

#include <algorithm>
#include <cmath>

#include "layout.hpp"

namespace gcs {

constexpr int64_t kFlowStages = 4;              // staging buffers per CTA
constexpr int64_t kFlowStageBytes = 48 << 10;   // shared memory of one staging buffer
constexpr int64_t kFlowMaxNodes = 2048;         // nodes of a regular block
constexpr int64_t kFlowMaxGran = 256;           // outlier granules of a block
constexpr int64_t kFlowMinNodes = 16;           // smallest block when windows do not fit
constexpr double kFlowCover = 0.98;             // share of a region's children a window holds
constexpr int64_t kFlowBlkInts = 16;            // ints per block record

// Fields of a block record (int32 each).
enum FlowField : int32_t {
    FB_NODE0 = 0,   // first node of the block in the pair array
    FB_PAIRS,       // pairs staged (even; the final block: all its levels, padded)
    FB_K0,          // level (the final block: first level)
    FB_K1,          // last level (= FB_K0 for a regular block)
    FB_SLOT0,       // slot of the first node within its level
    FB_WS1,         // window 1: first slot of level k-1, values
    FB_WL1,
    FB_WS2,         // window 2
    FB_WL2,
    FB_GOFF,        // outlier granules: first entry in the granule list, count
    FB_NGRAN,
    FB_DOFF,        // dependencies: first entry in the dependency list, count
    FB_NDEP,
    FB_PB,          // bytes of staged pairs (multiple of 16)
    FB_BYTES,       // staged bytes in all (pairs, then values)
    FB_NNODES       // nodes computed (the final block: all its levels)
};

struct FlowPlan {
    std::vector<int32_t> pairs;     // 2 per padded node
    std::vector<int32_t> blk;       // kFlowBlkInts per block
    std::vector<int32_t> deps;      // producer blocks, per block
    std::vector<int32_t> gran;      // first slot of each outlier granule, per block
    std::vector<int64_t> lvl_blk;   // L+2: first block of level k; [L+1] = blocks
    std::vector<int64_t> lvl_start; // L+2: first padded node of level k
    int64_t nblocks = 0;
    int64_t final_k0 = 0;           // first level of the final block (L+1: none)
    int64_t buf_values = 0;         // values per level buffer
    int64_t value_bytes = 4;
};

inline int64_t flow_granule(int64_t value_bytes) { return 16 / value_bytes; }

// Values a level buffer holds: the widest level rounded up to a granule, plus
// room for windows rounded past a level's end.
inline int64_t flow_buf_values(const Grammar& g, int64_t value_bytes) {
    const int64_t G = flow_granule(value_bytes);
    return (g.max_width() + G - 1) / G * G + 2 * G;
}

// Shared memory the final block needs when it starts at level k0.
inline int64_t flow_final_bytes(const Grammar& g, int64_t k0, int64_t value_bytes) {
    const int64_t G = flow_granule(value_bytes);
    auto rup = [&](int64_t v) { return (v + G - 1) / G * G; };
    auto width = [&](int64_t k) { return g.lvl_off[k + 1] - g.lvl_off[k]; };
    int64_t pairs = 0, vals = k0 > 1 ? rup(width(k0 - 1)) : 0;
    for (int64_t k = k0; k <= g.L; ++k) {
        pairs += pad_nodes(width(k));
        vals += rup(width(k));
    }
    return pairs * 8 + vals * value_bytes;
}

// First level of the final block: the lowest level from which the top levels
// fit the shared memory of all staging buffers together (L+1 if not even the
// top level fits).
inline int64_t flow_final_level(const Grammar& g, int64_t value_bytes) {
    int64_t k0 = g.L + 1;
    while (k0 > 1 && flow_final_bytes(g, k0 - 1, value_bytes) <= kFlowStages * kFlowStageBytes) --k0;
    return k0;
}

// Shortest run of sorted v holding at least ceil(q * n) of its entries: [lo, hi].
inline void flow_cover(const std::vector<int32_t>& v, double q, int64_t& lo, int64_t& hi) {
    const int64_t n = (int64_t)v.size();
    if (n == 0) {
        lo = 0;
        hi = -1;
        return;
    }
    int64_t need = (int64_t)std::ceil(q * (double)n);
    need = std::min(std::max<int64_t>(need, 1), n);
    int64_t best = 0;
    for (int64_t i = 0; i + need - 1 < n; ++i)
        if (v[i + need - 1] - v[i] < v[best + need - 1] - v[best]) best = i;
    lo = v[best];
    hi = v[best + need - 1];
}

inline FlowPlan plan_flow(const Grammar& g, int64_t value_bytes) {
    const int64_t L = g.L, G = flow_granule(value_bytes);
    auto rdn = [&](int64_t s) { return s / G * G; };
    auto rup = [&](int64_t s) { return (s + G - 1) / G * G; };
    auto width = [&](int64_t k) { return g.lvl_off[k + 1] - g.lvl_off[k]; };
    auto rup2 = [](int64_t s) { return (s + 1) / 2 * 2; };
    FlowPlan p;
    p.value_bytes = value_bytes;
    p.buf_values = flow_buf_values(g, value_bytes);
    p.final_k0 = flow_final_level(g, value_bytes);
    p.lvl_start.assign((size_t)L + 2, 0);
    for (int64_t k = 1; k <= L; ++k) p.lvl_start[k + 1] = p.lvl_start[k] + pad_nodes(width(k));
    p.pairs.assign((size_t)(2 * p.lvl_start[L + 1]), -1);
    p.lvl_blk.assign((size_t)L + 2, 0);
    const int32_t vbits = value_bits((int64_t)g.V.size());
    auto leaf_ref = [&](int32_t c) {   // terminal -c-2 -> -2 - leaf code
        const int64_t t = -(int64_t)c - 2;
        const int64_t q = ((int64_t)g.term_col[t] << vbits) | g.term_vidx[t];
        return (int32_t)(-2 - q);
    };
    std::vector<int64_t> prev_slot0, cur_slot0;   // first slot of each block of level k-1, k
    int64_t prev_b0 = 0;                          // first block id of level k-1
    std::vector<int32_t> r, o, gr, dl;
    for (int64_t k = 1; k <= L; ++k) {
        p.lvl_blk[k] = p.nblocks;
        if (k >= p.final_k0) break;
        const int64_t w = width(k), R = k > 1 ? g.lvl_roots[k - 1] : 0, wprev = k > 1 ? width(k - 1) : 0;
        const int32_t* kids = g.nodes.data() + 2 * g.lvl_off[k];
        cur_slot0.clear();
        // producer blocks of level k-1 for the slots [a, b)
        auto deps_of = [&](int64_t a, int64_t b) {
            a = std::max<int64_t>(a, 0);
            b = std::min(b, wprev);
            if (a >= b) return;
            int64_t i = std::upper_bound(prev_slot0.begin(), prev_slot0.end(), a) - prev_slot0.begin() - 1;
            for (; i < (int64_t)prev_slot0.size() && prev_slot0[i] < b; ++i) dl.push_back((int32_t)(prev_b0 + i));
        };
        for (int64_t i = 0; i < w;) {
            int64_t S = std::min(kFlowMaxNodes, w - i);
            int64_t ws1 = 0, we1 = 0, ws2 = 0, we2 = 0, bytes = 0;
            for (;;) {
                r.clear();
                o.clear();
                for (int64_t t = 2 * i; t < 2 * (i + S); ++t) {
                    const int32_t c = kids[t];
                    if (c >= 0) (c < R ? r : o).push_back(c);
                }
                std::sort(r.begin(), r.end());
                std::sort(o.begin(), o.end());
                int64_t lo, hi;
                flow_cover(r, kFlowCover, lo, hi);
                ws1 = rdn(lo);
                we1 = hi >= lo ? rup(hi + 1) : ws1;
                flow_cover(o, kFlowCover, lo, hi);
                ws2 = rdn(lo);
                we2 = hi >= lo ? rup(hi + 1) : ws2;
                if (we1 > ws2 && we2 > ws1) {   // rounding made them meet: one window
                    ws1 = std::min(ws1, ws2);
                    we1 = std::max(we1, we2);
                    ws2 = we2 = 0;
                }
                auto outside = [&](int64_t c) { return !(c >= ws1 && c < we1) && !(c >= ws2 && c < we2); };
                gr.clear();
                for (int32_t c : r)
                    if (outside(c)) gr.push_back((int32_t)rdn(c));
                for (int32_t c : o)
                    if (outside(c)) gr.push_back((int32_t)rdn(c));
                std::sort(gr.begin(), gr.end());
                gr.erase(std::unique(gr.begin(), gr.end()), gr.end());
                const int64_t vals = (we1 - ws1) + (we2 - ws2) + (int64_t)gr.size() * G;
                bytes = rup2(S) * 8 + vals * value_bytes;
                if ((bytes <= kFlowStageBytes && (int64_t)gr.size() <= kFlowMaxGran) || S <= kFlowMinNodes) break;
                S = std::max<int64_t>(kFlowMinNodes, S / 2 / kNodeAlign * kNodeAlign);
            }
            if (bytes > kFlowStageBytes || (int64_t)gr.size() > kFlowMaxGran) {
                // the smallest block still does not fit: no windows, every child a granule
                ws1 = we1 = ws2 = we2 = 0;
                gr.clear();
                for (int64_t t = 2 * i; t < 2 * (i + S); ++t)
                    if (kids[t] >= 0) gr.push_back((int32_t)rdn(kids[t]));
                std::sort(gr.begin(), gr.end());
                gr.erase(std::unique(gr.begin(), gr.end()), gr.end());
                bytes = rup2(S) * 8 + (int64_t)gr.size() * G * value_bytes;
                if (bytes > kFlowStageBytes || (int64_t)gr.size() > kFlowMaxGran)
                    fail(GC_ERR_UNSUPPORTED, "dataflow plan: a block does not fit its staging buffer");
            }
            // dependencies
            dl.clear();
            deps_of(ws1, we1);
            deps_of(ws2, we2);
            for (int32_t s : gr) deps_of(s, s + G);
            std::sort(dl.begin(), dl.end());
            dl.erase(std::unique(dl.begin(), dl.end()), dl.end());
            // re-encode the block's child references
            const int64_t W1 = we1 - ws1, W2 = we2 - ws2;
            for (int64_t t = 2 * i; t < 2 * (i + S); ++t) {
                const int32_t c = kids[t];
                int32_t e;
                if (c == -1) {
                    e = -1;
                } else if (c <= -2) {
                    e = leaf_ref(c);
                } else if (c >= ws1 && c < we1) {
                    e = (int32_t)(c - ws1);
                } else if (c >= ws2 && c < we2) {
                    e = (int32_t)(W1 + c - ws2);
                } else {
                    const int64_t j = std::lower_bound(gr.begin(), gr.end(), (int32_t)rdn(c)) - gr.begin();
                    e = (int32_t)(W1 + W2 + j * G + (c - rdn(c)));
                }
                p.pairs[2 * p.lvl_start[k] + t] = e;
            }
            const int32_t rec[kFlowBlkInts] = {
                (int32_t)(p.lvl_start[k] + i), (int32_t)rup2(S), (int32_t)k, (int32_t)k, (int32_t)i,
                (int32_t)ws1, (int32_t)W1, (int32_t)ws2, (int32_t)W2,
                (int32_t)p.gran.size(), (int32_t)gr.size(), (int32_t)p.deps.size(), (int32_t)dl.size(),
                (int32_t)(rup2(S) * 8), (int32_t)bytes, (int32_t)S};
            p.blk.insert(p.blk.end(), rec, rec + kFlowBlkInts);
            p.gran.insert(p.gran.end(), gr.begin(), gr.end());
            p.deps.insert(p.deps.end(), dl.begin(), dl.end());
            cur_slot0.push_back(i);
            ++p.nblocks;
            i += S;
        }
        prev_slot0.swap(cur_slot0);
        prev_b0 = p.lvl_blk[k];
    }
    if (p.final_k0 <= L) {
        const int64_t k0 = p.final_k0;
        const int64_t W0 = k0 > 1 ? rup(width(k0 - 1)) : 0;
        std::vector<int64_t> own((size_t)L + 2, 0);   // offset of level k's values after the window
        int64_t vals = W0, pairs = 0, nn = 0;
        for (int64_t k = k0; k <= L; ++k) {
            own[k] = vals;
            vals += rup(width(k));
            pairs += pad_nodes(width(k));
            nn += width(k);
        }
        for (int64_t k = k0; k <= L; ++k) {
            const int32_t* kids = g.nodes.data() + 2 * g.lvl_off[k];
            for (int64_t t = 0; t < 2 * width(k); ++t) {
                const int32_t c = kids[t];
                p.pairs[2 * p.lvl_start[k] + t] = c == -1 ? -1 : c <= -2 ? leaf_ref(c)
                                                   : k == k0 ? c : (int32_t)(own[k - 1] + c);
            }
        }
        dl.clear();
        if (k0 > 1)
            for (int64_t b = p.lvl_blk[k0 - 1]; b < p.nblocks; ++b) dl.push_back((int32_t)b);
        const int64_t bytes = pairs * 8 + vals * value_bytes;
        const int32_t rec[kFlowBlkInts] = {
            (int32_t)p.lvl_start[k0], (int32_t)pairs, (int32_t)k0, (int32_t)L, 0, 0, (int32_t)W0, 0, 0,
            (int32_t)p.gran.size(), 0, (int32_t)p.deps.size(), (int32_t)dl.size(),
            (int32_t)(pairs * 8), (int32_t)bytes, (int32_t)nn};
        p.blk.insert(p.blk.end(), rec, rec + kFlowBlkInts);
        p.deps.insert(p.deps.end(), dl.begin(), dl.end());
        ++p.nblocks;
        for (int64_t k = k0 + 1; k <= L; ++k) p.lvl_blk[k] = p.lvl_blk[k0];
    }
    p.lvl_blk[L + 1] = p.nblocks;
    return p;
}

// Checks a plan before anything reaches the device: every staged range inside
// its buffer, every block within its staging bytes, every child reference
// inside its block's staged values (and, in the final block, only into lower
// levels), dependencies earlier blocks of the level below that cover every
// staged slot, and the block sequence covering each level once.
inline void validate_flow_plan(const FlowPlan& p, const Grammar& g) {
    auto bad = [](const std::string& what) { fail(GC_ERR_INVALID_GRAMMAR, "dataflow plan: " + what); };
    const int64_t L = g.L, G = flow_granule(p.value_bytes), NB = p.nblocks;
    auto width = [&](int64_t k) { return g.lvl_off[k + 1] - g.lvl_off[k]; };
    if ((int64_t)p.blk.size() != NB * kFlowBlkInts || (int64_t)p.lvl_blk.size() != L + 2 || p.lvl_blk[L + 1] != NB ||
        (int64_t)p.pairs.size() != 2 * p.lvl_start[L + 1])
        bad("table sizes");
    const int32_t vbits = value_bits((int64_t)g.V.size());
    const int64_t leaf_max = (int64_t)g.m << vbits, nv = (int64_t)g.V.size();
    auto leaf_ok = [&](int64_t q) { return q >= 0 && q < leaf_max && (q & ((1 << vbits) - 1)) < nv; };
    std::vector<int64_t> covered((size_t)L + 2, 0);
    for (int64_t b = 0; b < NB; ++b) {
        const int32_t* f = p.blk.data() + b * kFlowBlkInts;
        const int64_t k0 = f[FB_K0], k1 = f[FB_K1];
        const bool fin = k0 >= p.final_k0;
        if (k0 < 1 || k1 > L || k1 < k0) bad("levels");
        if (f[FB_WL1] < 0 || f[FB_WL2] < 0 || f[FB_NGRAN] < 0 || f[FB_NDEP] < 0 || f[FB_PAIRS] < 0 || f[FB_NNODES] < 0)
            bad("negative sizes");
        const int64_t W1 = f[FB_WL1], W2 = f[FB_WL2], vals_staged = W1 + W2 + (int64_t)f[FB_NGRAN] * G;
        if (f[FB_PB] != (int64_t)f[FB_PAIRS] * 8 || f[FB_PB] % 16 != 0) bad("pair bytes");
        if (f[FB_NODE0] % 2 != 0 || f[FB_NODE0] < 0 || (int64_t)f[FB_NODE0] + f[FB_PAIRS] > p.lvl_start[L + 1]) bad("pair range");
        if (f[FB_WS1] % G || f[FB_WL1] % G || f[FB_WS2] % G || f[FB_WL2] % G) bad("window alignment");
        if ((int64_t)f[FB_WS1] + W1 > p.buf_values || (int64_t)f[FB_WS2] + W2 > p.buf_values || f[FB_WS1] < 0 || f[FB_WS2] < 0)
            bad("window outside the level buffer");
        if ((int64_t)f[FB_GOFF] + f[FB_NGRAN] > (int64_t)p.gran.size() || (int64_t)f[FB_DOFF] + f[FB_NDEP] > (int64_t)p.deps.size())
            bad("list ranges");
        for (int64_t j = 0; j < f[FB_NGRAN]; ++j) {
            const int64_t s = p.gran[f[FB_GOFF] + j];
            if (s < 0 || s % G || s + G > p.buf_values) bad("granule outside the level buffer");
        }
        // dependencies: earlier blocks of level k0-1 (ascending), whose slot
        // ranges cover every staged slot below that level's width
        const int64_t kp = k0 - 1;
        if (kp < 1 && W1 + W2 + f[FB_NGRAN] != 0) bad("level-1 block with staged values");
        for (int64_t j = 0; j < f[FB_NDEP]; ++j) {
            const int64_t d = p.deps[f[FB_DOFF] + j];
            if (d < 0 || d >= b || kp < 1 || d < p.lvl_blk[kp] || d >= p.lvl_blk[kp + 1] ||
                (j > 0 && d <= p.deps[f[FB_DOFF] + j - 1]))
                bad("dependency outside the level below");
        }
        auto covers = [&](int64_t a, int64_t e) {
            a = std::max<int64_t>(a, 0);
            e = std::min<int64_t>(e, kp >= 1 ? width(kp) : 0);
            for (int64_t j = 0; j < f[FB_NDEP] && a < e; ++j) {
                const int32_t* fd = p.blk.data() + (int64_t)p.deps[f[FB_DOFF] + j] * kFlowBlkInts;
                const int64_t s0 = fd[FB_SLOT0], s1 = s0 + fd[FB_NNODES];
                if (s0 <= a && a < s1) a = s1;
            }
            return a >= e;
        };
        if (!covers(f[FB_WS1], f[FB_WS1] + W1) || !covers(f[FB_WS2], f[FB_WS2] + W2))
            bad("a window slot without its producer among the dependencies");
        for (int64_t j = 0; j < f[FB_NGRAN]; ++j)
            if (!covers(p.gran[f[FB_GOFF] + j], p.gran[f[FB_GOFF] + j] + G))
                bad("a granule slot without its producer among the dependencies");
        // bytes
        const int64_t vbytes = p.value_bytes;
        int64_t own = 0;
        if (fin)
            for (int64_t k = k0; k <= k1; ++k) own += (width(k) + G - 1) / G * G;
        if ((int64_t)f[FB_BYTES] != f[FB_PB] + (vals_staged + own) * vbytes) bad("staged bytes");
        if (f[FB_BYTES] > (fin ? kFlowStages * kFlowStageBytes : kFlowStageBytes)) bad("block larger than its staging");
        // child references
        if (!fin) {
            if (k0 >= p.final_k0) bad("a regular block above the final level");
            if (f[FB_SLOT0] != covered[k0]) bad("blocks do not tile their level");
            if (p.lvl_start[k0] + f[FB_SLOT0] != f[FB_NODE0] || f[FB_NNODES] > f[FB_PAIRS] || f[FB_PAIRS] > f[FB_NNODES] + 1)
                bad("block nodes");
            covered[k0] += f[FB_NNODES];
            for (int64_t t = 0; t < 2 * f[FB_NNODES]; ++t) {
                const int64_t c = p.pairs[2 * (int64_t)f[FB_NODE0] + t];
                if (c >= 0 ? c >= vals_staged : c == -1 ? (t & 1) == 0 : !leaf_ok(-c - 2))
                    bad("child reference outside the block");
            }
        } else {
            if (b != NB - 1 || k0 != p.final_k0 || k1 != L || f[FB_NODE0] != p.lvl_start[k0] ||
                f[FB_PAIRS] != p.lvl_start[L + 1] - p.lvl_start[k0] || W2 != 0 || f[FB_NGRAN] != 0)
                bad("final block");
            const int64_t W0 = k0 > 1 ? (width(k0 - 1) + G - 1) / G * G : 0;
            if (W1 != W0 || f[FB_WS1] != 0) bad("final block window");
            int64_t lo = 0, hi = W0, nn = 0;   // a level-k node reads values in [lo, hi)
            for (int64_t k = k0; k <= L; ++k) {
                for (int64_t t = 0; t < 2 * width(k); ++t) {
                    const int64_t c = p.pairs[2 * p.lvl_start[k] + t];
                    const bool okc = c >= 0 ? (k > 1 && c >= lo && c < hi && c - lo < width(k - 1))
                                     : c == -1 ? (t & 1) == 1 : leaf_ok(-c - 2);
                    if (!okc) bad("final block reference");
                }
                lo = hi;
                hi += (width(k) + G - 1) / G * G;
                nn += width(k);
                covered[k] = width(k);
            }
            if (nn != f[FB_NNODES]) bad("final block nodes");
        }
    }
    for (int64_t k = 1; k <= L; ++k)
        if (covered[k] != width(k)) bad("a level not covered by its blocks");
}

// The plan of gg's grammar for values of value_bytes, made on first use and
// kept with the grammar (gc_layout and gc_upload both need it).
inline std::shared_ptr<const FlowPlan> flow_plan_for(const gc_grammar* gg, int64_t value_bytes) {
    std::lock_guard<std::mutex> lock(gg->flow_mu);
    std::shared_ptr<const void>& slot = gg->flow_plan[value_bytes == 4 ? 0 : 1];
    if (!slot) slot = std::make_shared<const FlowPlan>(plan_flow(gg->g, value_bytes));
    return std::static_pointer_cast<const FlowPlan>(slot);
}

inline FlowCounts flow_counts(const FlowPlan& p) {
    FlowCounts c;
    c.nblocks = p.nblocks;
    c.ndeps = (int64_t)p.deps.size();
    c.ngran = (int64_t)p.gran.size();
    c.buf_values = p.buf_values;
    c.final_k0 = p.final_k0;
    return c;
}

// Handles with one value a node (k_max = 1) run the dataflow sweep.
inline bool uses_flow(int32_t k_max) { return k_max == 1; }

}  // namespace gcs
