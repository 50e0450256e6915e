// Levels, pass-through completion and level-major packing.
//
//   Eq. 3.1     lvl(terminal) = 0, lvl(N -> A B) = 1 + max(lvl A, lvl B)
//   Def. 3.2    properly layered: every nonterminal child one level below
//   Sec. 4.2    pass-through completion: a nonterminal u whose highest parent
//               sits d > 1 levels above it is carried upward by identity
//               nodes at levels lvl(u)+1 .. maxpar(u)-1. One chain per node,
//               shared by all its skipping parents, so the width of a level
//               equals its live set; each parent reads the chain element one
//               level below itself.
//   Sec. 4.3    nodes are laid out level by level in one flat array; a child
//               reference c >= 0 is a slot of the previous level's buffer,
//               c < 0 reads the terminal array T[-c-1] with T[0] the combine
//               identity (a pass-through is (c, -1)).
//   Lemma 3.3 / emit-on-the-spot: a root (symbol of C) is captured when its
//               level is computed; each level lists its roots first, so level
//               k's roots fill RV[root_off[k] ..] contiguously and C is
//               rewritten into RV slots / T indices.
// Any order within a level is correct (Lemma 3.1); the default orders nodes
// by the first column of their expansion so that neighbouring threads read
// neighbouring children.
#include <numeric>

#include "common.hpp"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace gcs {

void layer_and_pack(Grammar& g, int order) {
    const double t0 = now_seconds();
    const Slp& s = g.slp;
    const int64_t R = g.n_rules();
    if (R >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 rules");

    // Eq. 3.1 levels, in rule order (children precede parents)
    g.rule_level.assign((size_t)R, 0);
    int32_t L = 0;
    for (int64_t i = 0; i < R; ++i) {
        int32_t a = s.rule_a[i], b = s.rule_b[i];
        int32_t la = a >= 0 ? g.rule_level[a] : 0, lb = b >= 0 ? g.rule_level[b] : 0;
        g.rule_level[i] = 1 + std::max(la, lb);
        L = std::max(L, g.rule_level[i]);
    }
    const std::vector<int32_t>& lvl = g.rule_level;
    g.L = L;

    // highest parent level and root flags
    std::vector<int32_t> mp((size_t)R, 0);
    for (int64_t i = 0; i < R; ++i) {
        int32_t a = s.rule_a[i], b = s.rule_b[i];
        if (a >= 0) mp[a] = std::max(mp[a], lvl[i]);
        if (b >= 0) mp[b] = std::max(mp[b], lvl[i]);
    }
    std::vector<uint8_t> is_root((size_t)R, 0);
    for (int32_t c : s.c_sym)
        if (c >= 0) is_root[c] = 1;

    // per-level counts: rules, roots, pass-throughs (difference array)
    std::vector<int64_t> cnt((size_t)L + 2, 0), roots((size_t)L + 2, 0), dpt((size_t)L + 2, 0);
    std::vector<int64_t> chain_base((size_t)R + 1, 0);
    for (int64_t u = 0; u < R; ++u) {
        cnt[lvl[u]]++;
        if (is_root[u]) roots[lvl[u]]++;
        int64_t len = std::max<int64_t>(0, (int64_t)mp[u] - lvl[u] - 1);
        chain_base[u + 1] = chain_base[u] + len;
        if (len > 0) {
            dpt[lvl[u] + 1]++;
            dpt[mp[u]]--;
        }
    }
    g.n_pass = chain_base[R];
    int64_t run = 0;
    for (int32_t k = 1; k <= L; ++k) {
        run += dpt[k];
        cnt[k] += run;
    }
    g.n_roots = 0;
    for (int32_t k = 1; k <= L; ++k) g.n_roots += roots[k];
    const int64_t N = R + g.n_pass;
    if (N >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 layered nodes");

    g.lvl_off.assign((size_t)L + 2, 0);
    g.lvl_roots.assign((size_t)L + 2, 0);
    g.root_off.assign((size_t)L + 2, 0);
    for (int32_t k = 1; k <= L; ++k) {
        g.lvl_off[k + 1] = g.lvl_off[k] + cnt[k];
        g.lvl_roots[k] = roots[k];
        g.root_off[k + 1] = g.root_off[k] + roots[k];
    }
    g.root_off[0] = 0;

    // first column of each rule's expansion (locality key)
    std::vector<int32_t> fc((size_t)R);
    for (int64_t i = 0; i < R; ++i) {
        int32_t a = s.rule_a[i];
        fc[i] = a >= 0 ? fc[a] : g.term_col[-a - 1];
    }

    // sort keys per level: group (roots first) | order key | kind | id
    //   kind 0 = rule i, kind 1 = pass-through of u (at this level)
    std::vector<uint64_t> ent((size_t)N);
    {
        std::vector<int64_t> w(g.lvl_off.begin(), g.lvl_off.end());
        auto key = [&](uint64_t grp, uint64_t col, uint64_t kind, uint64_t id) -> uint64_t {
            if (order == 1) return (grp << 63) | (id << 1) | kind;
            return (grp << 63) | (col << 32) | (kind << 31) | id;
        };
        for (int64_t i = 0; i < R; ++i)
            ent[w[lvl[i]]++] = key(is_root[i] ? 0 : 1, (uint64_t)fc[i], 0, (uint64_t)i);
        for (int64_t u = 0; u < R; ++u)
            for (int32_t k = lvl[u] + 1; k < mp[u]; ++k)
                ent[w[k]++] = key(1, (uint64_t)fc[u], 1, (uint64_t)u);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t k = 1; k <= L; ++k)
        std::sort(ent.begin() + g.lvl_off[k], ent.begin() + g.lvl_off[k + 1]);

    // positions of rules and chain elements within their level
    std::vector<int32_t> pos_rule((size_t)R, -1), pos_chain((size_t)g.n_pass, -1);
    g.node_id.assign((size_t)N, 0);
    auto decode = [&](uint64_t e, int32_t& kind, int32_t& id) {
        if (order == 1) {
            uint64_t v = e & ~(1ull << 63);
            kind = (int32_t)(v & 1);
            id = (int32_t)(v >> 1);
        } else {
            kind = (int32_t)((e >> 31) & 1);
            id = (int32_t)(e & 0x7fffffffu);
        }
    };
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t k = 1; k <= L; ++k) {
        for (int64_t q = g.lvl_off[k]; q < g.lvl_off[k + 1]; ++q) {
            int32_t kind, id;
            decode(ent[q], kind, id);
            int32_t pos = (int32_t)(q - g.lvl_off[k]);
            if (kind == 0) {
                pos_rule[id] = pos;
                g.node_id[q] = id;
            } else {
                pos_chain[chain_base[id] + (k - lvl[id] - 1)] = pos;
                g.node_id[q] = -(id + 1);
            }
        }
    }
    std::vector<uint64_t>().swap(ent);

    // packed child references
    auto node_ref = [&](int32_t u, int32_t K) -> int32_t {   // nonterminal u read at level K
        if (lvl[u] == K - 1) return pos_rule[u];
        return pos_chain[chain_base[u] + (K - 1 - lvl[u] - 1)];
    };
    g.nodes.assign((size_t)(2 * N), 0);
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t k = 1; k <= L; ++k) {
        for (int64_t q = g.lvl_off[k]; q < g.lvl_off[k + 1]; ++q) {
            int32_t id = g.node_id[q];
            int32_t a, b;
            if (id >= 0) {
                int32_t ca = s.rule_a[id], cb = s.rule_b[id];
                a = ca < 0 ? ca - 1 : node_ref(ca, k);
                b = cb < 0 ? cb - 1 : node_ref(cb, k);
            } else {
                a = node_ref(-id - 1, k);
                b = -1;
            }
            g.nodes[2 * q] = a;
            g.nodes[2 * q + 1] = b;
        }
    }

    // C rewritten into RV slots (roots) and T indices (terminals)
    g.c_ref.resize(s.c_sym.size());
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < (int64_t)s.c_sym.size(); ++e) {
        int32_t c = s.c_sym[e];
        g.c_ref[e] = c < 0 ? c - 1 : (int32_t)(g.root_off[lvl[c]] + pos_rule[c]);
    }
    g.layer_seconds += now_seconds() - t0;
}

void validate_packed(const Grammar& g) {
    const int64_t A = g.alpha();
    const int64_t N = g.n_nodes();
    if ((int64_t)g.lvl_off.size() != g.L + 2 || g.lvl_off[g.L + 1] != N)
        fail(GC_ERR_INVALID_GRAMMAR, "level offsets do not cover the nodes");
    if ((int64_t)g.nodes.size() != 2 * N) fail(GC_ERR_INVALID_GRAMMAR, "node array size");
    int64_t rv = 0;
    for (int64_t k = 1; k <= g.L; ++k) {
        const int64_t w = g.lvl_off[k + 1] - g.lvl_off[k];
        const int64_t wprev = k > 1 ? g.lvl_off[k] - g.lvl_off[k - 1] : 0;
        if (w < 0) fail(GC_ERR_INVALID_GRAMMAR, "level offsets decrease");
        if (g.lvl_roots[k] < 0 || g.lvl_roots[k] > w) fail(GC_ERR_INVALID_GRAMMAR, "root count exceeds level");
        if (g.root_off[k] != rv) fail(GC_ERR_INVALID_GRAMMAR, "root offsets inconsistent");
        rv += g.lvl_roots[k];
        for (int64_t q = g.lvl_off[k]; q < g.lvl_off[k + 1]; ++q) {
            for (int t = 0; t < 2; ++t) {
                const int64_t c = g.nodes[2 * q + t];
                if (c >= 0 ? c >= wprev : (-c - 1) > A)
                    fail(GC_ERR_INVALID_GRAMMAR, "child reference out of range at level " + std::to_string(k));
            }
        }
    }
    if (rv != g.n_roots) fail(GC_ERR_INVALID_GRAMMAR, "root total mismatch");
    const std::vector<int64_t>& co = g.slp.c_off;
    if ((int64_t)co.size() != g.n + 1 || co[0] != 0 || co[g.n] != (int64_t)g.c_ref.size())
        fail(GC_ERR_INVALID_GRAMMAR, "C offsets do not cover C");
    for (int64_t r = 0; r < g.n; ++r)
        if (co[r + 1] < co[r]) fail(GC_ERR_INVALID_GRAMMAR, "C offsets decrease");
    for (int32_t c : g.c_ref)
        if (c >= 0 ? c >= g.n_roots : (-(int64_t)c - 1) > A)
            fail(GC_ERR_INVALID_GRAMMAR, "C reference out of range");
}

}  // namespace gcs
