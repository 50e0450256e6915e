// Internal host-side types of the gcsparse library (not part of the C ABI).
#pragma once

#include <algorithm>
#include <chrono>
#include <memory>
#include <mutex>
#include <cstdint>
#include <new>
#include <stdexcept>
#include <string>
#include <vector>

#include "../../include/gcsparse.h"

namespace gcs {

// A failure carrying the C ABI status it maps to.
struct Error : std::runtime_error {
    gc_status status;
    Error(gc_status s, const std::string& msg) : std::runtime_error(msg), status(s) {}
};

[[noreturn]] inline void fail(gc_status s, const std::string& msg) { throw Error(s, msg); }

void set_last_error(const std::string& msg);

inline double now_seconds() {
    using clk = std::chrono::steady_clock;
    return std::chrono::duration<double>(clk::now().time_since_epoch()).count();
}

// CSRV form of a matrix (Sec. 2 "CSRV"): value dictionary, terminal table and
// one terminal string per row.
struct Csrv {
    int64_t n = 0, m = 0;
    std::vector<float> V;             // distinct non-zero values, ascending
    std::vector<int32_t> term_col;    // terminal t = <term_vidx[t], term_col[t]>,
    std::vector<int32_t> term_vidx;   //   sorted by (col, vidx)
    std::vector<int64_t> row_off;     // n+1 offsets into sym
    std::vector<int32_t> sym;         // terminal ids, each row in column order
};

// RePair output in the exported symbol encoding: a child s >= 0 is rule N_s,
// s < 0 is terminal -s-1.
struct Slp {
    std::vector<int32_t> rule_a, rule_b;   // |R|
    std::vector<int64_t> c_off;            // n+1
    std::vector<int32_t> c_sym;            // |C|
};

// Everything a built grammar holds: CSRV tables, the raw SLP and the packed,
// properly layered form the device sweeps.
struct Grammar {
    int64_t n = 0, m = 0, nnz = 0;
    std::vector<float> V;
    std::vector<int32_t> term_col, term_vidx;
    Slp slp;
    std::vector<int32_t> rule_level;       // Eq. 3.1 level of each rule
    // packed, level-major (levels 1..L; index 0 and L+1 are sentinels)
    int64_t L = 0;
    std::vector<int64_t> lvl_off;          // L+2
    std::vector<int64_t> lvl_roots;        // L+2
    std::vector<int64_t> root_off;         // L+2
    std::vector<int32_t> nodes;            // 2 * n_nodes: (a, b) child references
    std::vector<int32_t> node_id;          // n_nodes: rule i, or -(u+1) pass-through of u
    std::vector<int32_t> c_ref;            // |C|: >= 0 RV slot, < 0 T[-c-1]
    int64_t n_pass = 0, n_roots = 0, n_blocks = 1;
    // device view only (see device_view in layout.hpp): carried nodes per
    // level (roots, others) and the first carry slot of each level
    std::vector<int64_t> carry_roots, carry_rest, carry_off;
    int64_t n_carry = 0;
    double repair_seconds = 0, layer_seconds = 0;

    int64_t n_rules() const { return (int64_t)slp.rule_a.size(); }
    int64_t n_nodes() const { return (int64_t)node_id.size(); }
    int64_t alpha() const { return (int64_t)term_col.size(); }
    int64_t max_width() const {
        int64_t w = 0;
        for (int64_t k = 1; k <= L; ++k) w = std::max(w, lvl_off[k + 1] - lvl_off[k]);
        return w;
    }
};

// Sec. 2 "CSRV": validate the CSR input and encode it.
Csrv csrv_encode(int64_t n, int64_t m, const int64_t* row_ptr, const int32_t* col,
                 const float* val, int threads);

// Sec. 2 "Grammar" / Sec. 4.1: RePair over rows [r0, r1) of the CSRV strings,
// never pairing across a row end. alpha = terminal count.
Slp repair(const Csrv& s, int64_t r0, int64_t r1);

// Sec. 3 (Eq. 3.1), Sec. 4.2 (pass-through completion), Sec. 4.3 (level-major
// packing with roots first in each level). Fills g's level and packed fields.
void layer_and_pack(Grammar& g, int order);

// Host-side validation of the packed arrays (bounds of every reference).
void validate_packed(const Grammar& g);

// Sec. 4.2 pre-balancing: the same expansions as an AVL grammar (children's
// heights differ by at most one), rules in creation order, C remapped.
Slp balance_slp(const Slp& s);

// Runs f at the C ABI boundary: maps exceptions to a status and records the
// message for gc_last_error().
template <class F>
gc_status guard(F&& f) {
    try {
        f();
        return GC_OK;
    } catch (const Error& e) {
        set_last_error(e.what());
        return e.status;
    } catch (const std::bad_alloc&) {
        set_last_error("host allocation failed");
        return GC_ERR_OOM;
    } catch (const std::exception& e) {
        set_last_error(e.what());
        return GC_ERR_ARG;
    } catch (...) {
        set_last_error("unknown failure");
        return GC_ERR_ARG;
    }
}

}  // namespace gcs

struct gc_grammar {
    gcs::Grammar g;
    // dataflow block plans of this grammar for 4- and 8-byte values, made on
    // first use by gc_layout / gc_upload (flow.hpp) and kept with the grammar
    mutable std::mutex flow_mu;
    mutable std::shared_ptr<const void> flow_plan[2];
};
