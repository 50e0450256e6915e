// Block plan of the dataflow sweep (host-side arithmetic only; used by
// gc_layout and gc_upload for handles with one value per node).
//
// The level-synchronous sweep of Sec. 4.3 evaluates level k from level k-1
// only (Lemma 3.3), and any order within a level is correct (Lemma 3.1). The
// dataflow sweep cuts every level into blocks of consecutive nodes (4,096 at
// most) and gives each block the list of blocks of level k-1 that write its
// children's slots: its dependencies. A block starts once its dependencies
// have published their values (per-block ready flags instead of a grid
// barrier per level); its node pairs are staged in shared memory by one bulk
// copy, and its nodes gather their children from the level buffer of k-1.
//
// The narrow top levels form one final block: the whole level below them is
// copied into shared memory, and the block computes its levels one after the
// other there, where the top levels' values stay.
//
// Node references in the uploaded pair array (one int2 per padded node, the
// layout of the packed grammar):
//   c >= 0   regular block: slot c of level k-1 (in its level buffer);
//            final block: index into its staged values (the level below,
//            then its own levels' values)
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
constexpr int64_t kFlowMaxNodes = 4096;         // nodes of a regular block (a multiple of 16)
constexpr int64_t kFlowStageBytes = 8 * kFlowMaxNodes;   // a staging buffer: one block's node pairs
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
    std::vector<int32_t> order;     // the blocks in processing order (see plan_flow)
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

inline FlowPlan plan_flow(const Grammar& g, int64_t value_bytes) {
    const int64_t L = g.L, G = flow_granule(value_bytes);
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
    std::vector<int32_t> dl;
    for (int64_t k = 1; k <= L; ++k) {
        p.lvl_blk[k] = p.nblocks;
        if (k >= p.final_k0) break;
        const int64_t w = width(k), b_prev = k > 1 ? p.lvl_blk[k - 1] : 0;
        const int32_t* kids = g.nodes.data() + 2 * g.lvl_off[k];
        for (int64_t i = 0; i < w; i += kFlowMaxNodes) {
            const int64_t S = std::min(kFlowMaxNodes, w - i);
            dl.clear();
            for (int64_t t = 2 * i; t < 2 * (i + S); ++t) {
                const int32_t c = kids[t];
                // a child slot c of level k-1 is written by that level's block c / kFlowMaxNodes
                if (c >= 0) dl.push_back((int32_t)(b_prev + c / kFlowMaxNodes));
                p.pairs[2 * p.lvl_start[k] + t] = c <= -2 ? leaf_ref(c) : c;
            }
            std::sort(dl.begin(), dl.end());
            dl.erase(std::unique(dl.begin(), dl.end()), dl.end());
            const int32_t rec[kFlowBlkInts] = {
                (int32_t)(p.lvl_start[k] + i), (int32_t)rup2(S), (int32_t)k, (int32_t)k, (int32_t)i,
                0, 0, 0, 0, (int32_t)p.gran.size(), 0, (int32_t)p.deps.size(), (int32_t)dl.size(),
                (int32_t)(rup2(S) * 8), (int32_t)(rup2(S) * 8), (int32_t)S};
            p.blk.insert(p.blk.end(), rec, rec + kFlowBlkInts);
            p.deps.insert(p.deps.end(), dl.begin(), dl.end());
            ++p.nblocks;
        }
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
    // Processing order: level after level (every dependency lies in the level
    // below, so this is a topological order), and within a level by the
    // position of the block's latest dependency in the order, then by id. A
    // block's children span both halves of the level below (roots first,
    // then the other nodes, each sorted by column), so by id the first blocks
    // of a level would wait for the last of the one below; in this order
    // they wait for the earliest ones.
    std::vector<int32_t> pos((size_t)p.nblocks, 0);
    std::vector<std::pair<int64_t, int32_t>> key;
    for (int64_t k = 1; k < std::min(p.final_k0, L + 1); ++k) {
        key.clear();
        for (int64_t b = p.lvl_blk[k]; b < p.lvl_blk[k + 1]; ++b) {
            const int32_t* f = p.blk.data() + b * kFlowBlkInts;
            int64_t latest = -1;
            for (int32_t j = 0; j < f[FB_NDEP]; ++j) latest = std::max<int64_t>(latest, pos[p.deps[f[FB_DOFF] + j]]);
            key.push_back({latest, (int32_t)b});
        }
        std::sort(key.begin(), key.end());
        for (const auto& kb : key) {
            pos[kb.second] = (int32_t)p.order.size();
            p.order.push_back(kb.second);
        }
    }
    if (p.final_k0 <= L) p.order.push_back((int32_t)(p.nblocks - 1));   // the final block last
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
            if (vals_staged != 0) bad("a regular block with staged values");
            const int32_t* d0 = p.deps.data() + f[FB_DOFF];
            for (int64_t t = 0; t < 2 * f[FB_NNODES]; ++t) {
                const int64_t c = p.pairs[2 * (int64_t)f[FB_NODE0] + t];
                if (c >= 0) {
                    // a slot of level k0-1, whose producer is among the dependencies
                    if (k0 < 2 || c >= width(k0 - 1)) bad("child reference outside the level below");
                    const int32_t pbk = (int32_t)(p.lvl_blk[k0 - 1] + c / kFlowMaxNodes);
                    if (!std::binary_search(d0, d0 + f[FB_NDEP], pbk)) bad("a child's producer is not a dependency");
                    const int32_t* fp = p.blk.data() + (int64_t)pbk * kFlowBlkInts;
                    if (fp[FB_K0] != k0 - 1 || c < fp[FB_SLOT0] || c >= fp[FB_SLOT0] + fp[FB_NNODES])
                        bad("a child's producer does not hold its slot");
                } else if (c == -1 ? (t & 1) == 0 : !leaf_ok(-c - 2)) {
                    bad("child reference outside the block");
                }
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
    // the processing order: a permutation that keeps each level's blocks in
    // that level's id range and puts every dependency before its block
    if ((int64_t)p.order.size() != NB) bad("processing order size");
    std::vector<int64_t> pos((size_t)NB, -1);
    for (int64_t q = 0; q < NB; ++q) {
        const int64_t b = p.order[q];
        if (b < 0 || b >= NB || pos[b] >= 0) bad("processing order is not a permutation");
        pos[b] = q;
    }
    for (int64_t b = 0; b < NB; ++b) {
        const int32_t* f = p.blk.data() + b * kFlowBlkInts;
        const int64_t k0 = f[FB_K0];
        if (pos[b] < p.lvl_blk[k0] || pos[b] >= (k0 >= p.final_k0 ? NB : p.lvl_blk[k0 + 1])) bad("processing order mixes levels");
        for (int64_t j = 0; j < f[FB_NDEP]; ++j)
            if (pos[p.deps[f[FB_DOFF] + j]] >= pos[b]) bad("a dependency after its block in the processing order");
    }
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

// The dataflow layout is made on request (schedule GC_SCHED_DATAFLOW at
// upload) for handles with one value a node; anything else is refused.
inline bool wants_flow(int32_t schedule, int32_t k_max) {
    if (schedule != GC_SCHED_PERSISTENT && schedule != GC_SCHED_PER_LEVEL && schedule != GC_SCHED_DATAFLOW)
        fail(GC_ERR_ARG, "unknown schedule");
    if (schedule == GC_SCHED_DATAFLOW && k_max != 1)
        fail(GC_ERR_UNSUPPORTED, "the dataflow schedule serves handles with one value a node (k_max = 1)");
    return schedule == GC_SCHED_DATAFLOW;
}

}  // namespace gcs
