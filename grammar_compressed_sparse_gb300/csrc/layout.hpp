// Device arena layout of an uploaded grammar (host-side arithmetic only; used
// by gc_layout and gc_upload). Every part starts on a 256-byte boundary.
//
//   read-only grammar   nodes     int2[sum of padded widths]  child references,
//                                 each level starting on a 16-node (128 B)
//                                 boundary and padded to a multiple of 16
//                       levels    int64[4 (L+2)]   per level k: padded start,
//                                 width, number of roots, RV slot of the first root
//                       V         policy[|V|]      value dictionary
//                       leaf      int32[alpha]     leaf code of terminal p
//                       c_off     int32[n+1]
//                       c_ref     int32[|C|]
//   scratch             RVX       value[TB + rho]  leaf table T, then root values
//                       buf0X     value[TB + w*]   leaf table T, then a level's
//                       buf1X     value[TB + w*]   values (the two streaming buffers)
//                       status    256 B            status word, fixpoint flag,
//                                                  grid-barrier arrival counter
//   staging             xs        value[m]         x / y copies for the
//                       ys        value[n]         host-buffer entry point
// "value" is k_max elements of the policy's type (float, int64, uint64);
// TB = alpha + 1 rounded up to a multiple of 64 values.
//
// Leaf table: T[0] is the combine identity and T[p+1] = V[l_p] (x) x[j_p] for
// terminal p = <l_p, j_p> (Sec. 4.3's T). Its three copies sit in front of
// each buffer, so that one index space covers both: a child or C reference is
//   0            the identity (second child of a pass-through)
//   p + 1        terminal p
//   TB + s       slot s of the previous level (nodes) or root slot s (C)
// and every read is a single load, without a branch. Level 1, whose children
// are all terminals, instead stores leaf codes (column << vbits | value index)
// and evaluates its leaves in the sweep while the T copies are being written.
#pragma once

#include "common.hpp"

namespace gcs {

constexpr int64_t kNodeAlign = 16;   // nodes per 128-byte granule

struct DevLayout {
    int64_t nodes, levels, V, leaf, c_off, c_ref;
    int64_t RV, buf0, buf1, status, xs, ys;
    int64_t total, grammar_bytes, scratch_bytes, staging_bytes;
    int64_t value_bytes;   // bytes of one node value (k_max elements)
    int64_t n_nodes_padded;
    int64_t TB;            // leaf-table block length in values
    int32_t vbits;         // bits of the value index inside a leaf code
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

inline DevLayout device_layout(const Grammar& g, gc_policy p, int32_t k_max) {
    DevLayout d{};
    const int64_t L = g.L, C = (int64_t)g.c_ref.size(), A = g.alpha();
    d.value_bytes = policy_elem_bytes(p) * k_max;
    d.vbits = value_bits((int64_t)g.V.size());
    d.TB = leaf_block(A);
    d.n_nodes_padded = 0;
    for (int64_t k = 1; k <= L; ++k) d.n_nodes_padded += pad_nodes(g.lvl_off[k + 1] - g.lvl_off[k]);
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        int64_t at = o;
        o = align256(o + bytes);
        return at;
    };
    d.nodes = take(8 * d.n_nodes_padded);
    d.levels = take(8 * 4 * (L + 2));
    d.V = take(policy_elem_bytes(p) * std::max<int64_t>(1, (int64_t)g.V.size()));
    d.leaf = take(4 * A);
    d.c_off = take(4 * (g.n + 1));
    d.c_ref = take(4 * C);
    d.grammar_bytes = o;
    d.RV = take(d.value_bytes * (d.TB + g.n_roots));
    const int64_t w = g.max_width();
    d.buf0 = take(d.value_bytes * (d.TB + w));
    d.buf1 = take(d.value_bytes * (d.TB + w));
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
