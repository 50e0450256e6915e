// Device arena layout of an uploaded grammar (host-side arithmetic only; used
// by gc_layout and gc_upload). Every part starts on a 256-byte boundary.
//
//   read-only grammar            nodes        int2[N]        (a, b) child refs
//                                lvl_off      int64[L+2]
//                                lvl_roots    int64[L+2]
//                                root_off     int64[L+2]
//                                leaf_col     int32[alpha]
//                                leaf_val     policy[alpha]  V[l] of each leaf (none for OR)
//                                c_off        int32[n+1]
//                                c_ref        int32[|C|]
//   scratch (overwritten)        T            value[alpha+1]  T[0] identity
//                                RV           value[rho]      root values
//                                buf0, buf1   value[w*]       level ping-pong
//                                status       256 B           device status word, flags
//   staging (host-buffer calls)  xs           value[m]
//                                ys           value[n]
// "value" is k_max elements of the policy's type (float, int64, uint64).
#pragma once

#include "common.hpp"

namespace gcs {

struct DevLayout {
    int64_t nodes, lvl_off, lvl_roots, root_off, leaf_col, leaf_val, c_off, c_ref;
    int64_t T, RV, buf0, buf1, status, xs, ys;
    int64_t total, grammar_bytes, scratch_bytes, staging_bytes;
    int64_t value_bytes;   // bytes of one node value (k_max elements)
    int64_t leaf_bytes;    // bytes of one leaf value
};

inline int64_t policy_elem_bytes(gc_policy p) { return p == GC_F32_SUM ? 4 : 8; }

inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

inline DevLayout device_layout(const Grammar& g, gc_policy p, int32_t k_max) {
    DevLayout d{};
    const int64_t N = g.n_nodes(), L = g.L, A = g.alpha(), C = (int64_t)g.c_ref.size();
    d.value_bytes = policy_elem_bytes(p) * k_max;
    d.leaf_bytes = p == GC_BOOL_OR ? 0 : policy_elem_bytes(p);
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        int64_t at = o;
        o = align256(o + bytes);
        return at;
    };
    d.nodes = take(8 * N);
    d.lvl_off = take(8 * (L + 2));
    d.lvl_roots = take(8 * (L + 2));
    d.root_off = take(8 * (L + 2));
    d.leaf_col = take(4 * A);
    d.leaf_val = take(d.leaf_bytes * A);
    d.c_off = take(4 * (g.n + 1));
    d.c_ref = take(4 * C);
    d.grammar_bytes = o;
    d.T = take(d.value_bytes * (A + 1));
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
}

}  // namespace gcs
