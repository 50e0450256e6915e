// Device arena layout of an uploaded grammar (host-side arithmetic only; used
// by gc_layout and gc_upload). Every part starts on a 256-byte boundary.
//
//   read-only grammar   nodes     int2[sum of padded widths]  (a, b) child refs,
//                                 each level starting on a 16-node (128 B)
//                                 boundary and padded to a multiple of 16
//                       levels    int64[4 (L+2)]   per level k: padded start,
//                                 width, number of roots, RV slot of the first root
//                       V         policy[|V|]      value dictionary
//                       c_off     int32[n+1]
//                       c_ref     int32[|C|]
//   scratch             RV        value[rho]       root values
//                       buf0/1    value[w*]        level ping-pong buffers
//                       status    256 B            status word, fixpoint flag,
//                                                  grid-barrier arrival counter
//   staging             xs        value[m]         x / y copies for the
//                       ys        value[n]         host-buffer entry point
// "value" is k_max elements of the policy's type (float, int64, uint64).
//
// Device child references (rewritten from the packed T-index form at upload):
//   c >= 0    slot c of the previous level's buffer
//   c == -1   the combine identity (second child of a pass-through)
//   c <= -2   leaf q = -c - 2 = (column << vbits) | value index: the leaf value
//             V[l] (x) x[j] is evaluated in the sweep, no terminal array.
#pragma once

#include "common.hpp"

namespace gcs {

constexpr int64_t kNodeAlign = 16;   // nodes per 128-byte bulk-copy granule

struct DevLayout {
    int64_t nodes, levels, V, c_off, c_ref;
    int64_t RV, buf0, buf1, status, xs, ys;
    int64_t total, grammar_bytes, scratch_bytes, staging_bytes;
    int64_t value_bytes;   // bytes of one node value (k_max elements)
    int64_t n_nodes_padded;
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

inline DevLayout device_layout(const Grammar& g, gc_policy p, int32_t k_max) {
    DevLayout d{};
    const int64_t L = g.L, C = (int64_t)g.c_ref.size();
    d.value_bytes = policy_elem_bytes(p) * k_max;
    d.vbits = value_bits((int64_t)g.V.size());
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
    d.c_off = take(4 * (g.n + 1));
    d.c_ref = take(4 * C);
    d.grammar_bytes = o;
    d.RV = take(d.value_bytes * g.n_roots);
    const int64_t w = g.max_width();
    d.buf0 = take(d.value_bytes * w);
    d.buf1 = take(d.value_bytes * w);
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
    if ((((int64_t)g.m) << value_bits((int64_t)g.V.size())) + 2 > INT32_MAX)
        fail(GC_ERR_UNSUPPORTED, "columns x distinct values too large for 31-bit leaf codes");
}

}  // namespace gcs
