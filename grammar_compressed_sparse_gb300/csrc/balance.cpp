// Height balancing of the grammar (Sec. 4.2: RePair's grammars can be
// "pre-balanced to a logarithmic height", which bounds the number of levels L
// -- the sweep's sequential steps -- but not the live set, so completion is
// still needed; Sec. 8 leaves it as future work). The pages name no
// construction; this one rebuilds the straight-line program bottom-up as an
// AVL grammar: every rule's expansion is the concatenation of its children's
// balanced forms, joined the way two AVL trees are joined under a new root,
// so the heights of any rule's two children differ by at most one and a
// symbol of expansion length n has height at most about 1.44 log2(n). A join
// of heights h1, h2 creates O(|h1 - h2|) rules; equal pairs are shared (one
// rule per distinct (left, right) pair). The expansions do not change, so
// every product over the balanced grammar equals the original's.
#include "common.hpp"

namespace gcs {
namespace {

// (left, right) -> rule id, open addressing with linear probing; the table
// holds rule ids only (the pair is read back from the rule arrays).
struct PairTable {
    std::vector<int32_t> slot;   // -1 empty
    uint64_t mask = 0;

    static uint64_t hash(int32_t x, int32_t y) {
        uint64_t k = ((uint64_t)(uint32_t)x << 32) | (uint32_t)y;
        k ^= k >> 33;   // splitmix64 finaliser
        k *= 0xff51afd7ed558ccdULL;
        k ^= k >> 33;
        k *= 0xc4ceb9fe1a85ec53ULL;
        k ^= k >> 33;
        return k;
    }
    void init(int64_t expected) {
        uint64_t cap = 1024;
        while (cap < (uint64_t)expected * 2) cap <<= 1;
        slot.assign(cap, -1);
        mask = cap - 1;
    }
};

struct Balancer {
    std::vector<int32_t> a, b, h;   // new rules: children (GC_A_RULES encoding) and heights
    PairTable pairs;

    int32_t height(int32_t s) const { return s < 0 ? 0 : h[s]; }

    void grow() {
        PairTable t;
        t.init((int64_t)a.size() * 2);
        for (int32_t id = 0; id < (int32_t)a.size(); ++id) {
            uint64_t i = PairTable::hash(a[id], b[id]) & t.mask;
            while (t.slot[i] >= 0) i = (i + 1) & t.mask;
            t.slot[i] = id;
        }
        pairs = std::move(t);
    }

    // The rule (x, y), made once.
    int32_t mk(int32_t x, int32_t y) {
        uint64_t i = PairTable::hash(x, y) & pairs.mask;
        for (; pairs.slot[i] >= 0; i = (i + 1) & pairs.mask) {
            const int32_t id = pairs.slot[i];
            if (a[id] == x && b[id] == y) return id;
        }
        if ((int64_t)a.size() >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "balancing: more than 2^31-1 rules");
        const int32_t id = (int32_t)a.size();
        a.push_back(x);
        b.push_back(y);
        h.push_back(1 + std::max(height(x), height(y)));
        pairs.slot[i] = id;
        if ((uint64_t)a.size() * 2 > pairs.mask + 1) grow();   // load factor <= 1/2
        return id;
    }

    // A symbol expanding to exp(x) exp(y), balanced when x and y are.
    int32_t concat(int32_t x, int32_t y) {
        const int32_t hx = height(x), hy = height(y);
        if (hx <= hy + 1 && hy <= hx + 1) return mk(x, y);
        if (hx > hy) {
            const int32_t x1 = a[x], x2 = b[x];
            const int32_t t = concat(x2, y);
            if (height(t) <= height(x1) + 1) return mk(x1, t);
            // height(t) = height(x1) + 2: rotate
            const int32_t t1 = a[t], t2 = b[t];
            if (height(t2) >= height(t1)) return mk(mk(x1, t1), t2);
            return mk(mk(x1, a[t1]), mk(b[t1], t2));
        }
        const int32_t y1 = a[y], y2 = b[y];
        const int32_t t = concat(x, y1);
        if (height(t) <= height(y2) + 1) return mk(t, y2);
        const int32_t t1 = a[t], t2 = b[t];
        if (height(t1) >= height(t2)) return mk(t1, mk(t2, y2));
        return mk(mk(t1, a[t2]), mk(b[t2], y2));
    }
};

}  // namespace

Slp balance_slp(const Slp& s) {
    const int64_t R = (int64_t)s.rule_a.size();
    Balancer z;
    z.a.reserve((size_t)(R + R / 2));
    z.b.reserve((size_t)(R + R / 2));
    z.h.reserve((size_t)(R + R / 2));
    z.pairs.init(R + R / 2);
    std::vector<int32_t> bal((size_t)R, -1);   // original rule -> balanced symbol
    auto sym = [&](int32_t c) { return c < 0 ? c : bal[c]; };
    for (int64_t i = 0; i < R; ++i) {   // children precede parents in rule order
        if (s.rule_a[i] >= i || s.rule_b[i] >= i) fail(GC_ERR_INVALID_GRAMMAR, "balancing: a rule names a later rule");
        bal[i] = z.concat(sym(s.rule_a[i]), sym(s.rule_b[i]));
    }
    // keep the rules C reaches, renumbered in creation order (children first)
    const int64_t Rn = (int64_t)z.a.size();
    std::vector<char> live((size_t)Rn, 0);
    std::vector<int32_t> stack;
    Slp out;
    out.c_off = s.c_off;
    out.c_sym.resize(s.c_sym.size());
    for (size_t e = 0; e < s.c_sym.size(); ++e) {
        const int32_t c = sym(s.c_sym[e]);
        out.c_sym[e] = c;
        if (c >= 0 && !live[c]) {
            live[c] = 1;
            stack.push_back(c);
        }
    }
    while (!stack.empty()) {
        const int32_t u = stack.back();
        stack.pop_back();
        for (int32_t c : {z.a[u], z.b[u]})
            if (c >= 0 && !live[c]) {
                live[c] = 1;
                stack.push_back(c);
            }
    }
    std::vector<int32_t> id((size_t)Rn, -1);
    for (int64_t u = 0; u < Rn; ++u)
        if (live[u]) {
            id[u] = (int32_t)out.rule_a.size();
            out.rule_a.push_back(z.a[u] < 0 ? z.a[u] : id[z.a[u]]);
            out.rule_b.push_back(z.b[u] < 0 ? z.b[u] : id[z.b[u]]);
        }
    for (int32_t& c : out.c_sym)
        if (c >= 0) c = id[c];
    return out;
}

}  // namespace gcs
