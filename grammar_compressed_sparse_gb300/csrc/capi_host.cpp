// Host entry points of the C ABI: build, statistics, export, layout,
// save / load. Nothing here touches a GPU.
#include <cstdio>
#include <cstring>
#include <exception>
#include <memory>
#include <mutex>

#include "common.hpp"
#include "flow.hpp"
#include "layout.hpp"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace gcs {

static thread_local std::string g_last_error;

static int32_t value_bits_host(int64_t n_values) {
    int32_t b = 0;
    while (((int64_t)1 << b) < n_values) ++b;
    return b;
}

void set_last_error(const std::string& msg) { g_last_error = msg; }

namespace {

// RePair on every row block (in parallel) and the merge of their rules into
// one rule list: block b's rule i becomes rule offset_b + i. The blocks share
// the terminal table, so their leaves are the same T entries.
Slp repair_blocks(const Csrv& s, int64_t block_rows, int threads, int64_t& n_blocks) {
    const int64_t n = s.n;
    if (block_rows <= 0 || block_rows >= n) {
        n_blocks = 1;
        return repair(s, 0, n);
    }
    n_blocks = (n + block_rows - 1) / block_rows;
    std::vector<Slp> parts((size_t)n_blocks);
    std::exception_ptr err;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#endif
    (void)threads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
    for (int64_t b = 0; b < n_blocks; ++b) {
        try {
            parts[b] = repair(s, b * block_rows, std::min(n, (b + 1) * block_rows));
        } catch (...) {
#pragma omp critical
            if (!err) err = std::current_exception();
        }
    }
    if (err) std::rethrow_exception(err);
    Slp out;
    int64_t R = 0, C = 0;
    for (auto& p : parts) {
        R += (int64_t)p.rule_a.size();
        C += (int64_t)p.c_sym.size();
    }
    if (R >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 rules over all blocks");
    out.rule_a.reserve((size_t)R);
    out.rule_b.reserve((size_t)R);
    out.c_sym.reserve((size_t)C);
    out.c_off.assign(1, 0);
    int32_t base = 0;
    for (auto& p : parts) {
        auto shift = [&](int32_t c) { return c >= 0 ? c + base : c; };
        for (size_t i = 0; i < p.rule_a.size(); ++i) {
            out.rule_a.push_back(shift(p.rule_a[i]));
            out.rule_b.push_back(shift(p.rule_b[i]));
        }
        const int64_t c0 = (int64_t)out.c_sym.size();
        for (int32_t c : p.c_sym) out.c_sym.push_back(shift(c));
        for (size_t r = 1; r < p.c_off.size(); ++r) out.c_off.push_back(c0 + p.c_off[r]);
        base += (int32_t)p.rule_a.size();
        p = Slp();   // release the block's arrays as soon as they are merged
    }
    return out;
}

struct ArrayView {
    const void* ptr;
    int64_t bytes;
};

template <class T>
ArrayView view(const std::vector<T>& v) {
    return {v.data(), (int64_t)(v.size() * sizeof(T))};
}

ArrayView array_of(const Grammar& g, gc_array which) {
    switch (which) {
        case GC_A_VALUES: return view(g.V);
        case GC_A_TERM_COL: return view(g.term_col);
        case GC_A_TERM_VIDX: return view(g.term_vidx);
        case GC_A_RULES: return {nullptr, (int64_t)(g.slp.rule_a.size() * 8)};
        case GC_A_C_OFF: return view(g.slp.c_off);
        case GC_A_C_SYM: return view(g.slp.c_sym);
        case GC_A_RULE_LEVEL: return view(g.rule_level);
        case GC_A_LVL_OFF: return view(g.lvl_off);
        case GC_A_NODES: return view(g.nodes);
        case GC_A_LVL_ROOTS: return view(g.lvl_roots);
        case GC_A_ROOT_OFF: return view(g.root_off);
        case GC_A_C_REF: return view(g.c_ref);
        case GC_A_NODE_ID: return view(g.node_id);
    }
    fail(GC_ERR_ARG, "unknown array");
}

// ---------------------------------------------------------------- save / load
constexpr char kMagic[8] = {'G', 'C', 'S', 'P', 'A', 'R', '0', '1'};

struct Writer {
    FILE* f;
    void raw(const void* p, size_t b) {
        if (b && fwrite(p, 1, b, f) != b) fail(GC_ERR_IO, "write failed");
    }
    void i64(int64_t v) { raw(&v, 8); }
    template <class T>
    void vec(const std::vector<T>& v) {
        i64((int64_t)v.size());
        raw(v.data(), v.size() * sizeof(T));
    }
};

struct Reader {
    FILE* f;
    void raw(void* p, size_t b) {
        if (b && fread(p, 1, b, f) != b) fail(GC_ERR_IO, "truncated grammar file");
    }
    int64_t i64() {
        int64_t v;
        raw(&v, 8);
        return v;
    }
    template <class T>
    void vec(std::vector<T>& v) {
        int64_t n = i64();
        if (n < 0 || n > (int64_t)1 << 40) fail(GC_ERR_IO, "corrupt array length");
        v.resize((size_t)n);
        raw(v.data(), (size_t)n * sizeof(T));
    }
};

template <class IO, class G>
void fields(IO& io, G& g) {
    io.vec(g.V);
    io.vec(g.term_col);
    io.vec(g.term_vidx);
    io.vec(g.slp.rule_a);
    io.vec(g.slp.rule_b);
    io.vec(g.slp.c_off);
    io.vec(g.slp.c_sym);
    io.vec(g.rule_level);
    io.vec(g.lvl_off);
    io.vec(g.lvl_roots);
    io.vec(g.root_off);
    io.vec(g.nodes);
    io.vec(g.node_id);
    io.vec(g.c_ref);
}

// One compressed row block of a streaming build: its own value dictionary,
// terminal table and SLP (terminals in the block's local numbering).
struct Block {
    int64_t r0 = 0, rows = 0;
    std::vector<float> V;
    std::vector<int32_t> term_col, term_vidx;
    Slp slp;
};

// Merges row blocks (sorted by first row, covering [0, n)) into one grammar:
// one value dictionary (sorted union), one terminal table (sorted union of
// <l, j>), rules numbered block after block, C rows in row order.
void merge_blocks(std::vector<Block>& blocks, Grammar& g) {
    std::vector<float> V;
    for (auto& b : blocks) V.insert(V.end(), b.V.begin(), b.V.end());
    std::sort(V.begin(), V.end());
    V.erase(std::unique(V.begin(), V.end(), [](float x, float y) {
                uint32_t a, c;
                std::memcpy(&a, &x, 4);
                std::memcpy(&c, &y, 4);
                return a == c;
            }),
            V.end());
    const int32_t vb = value_bits_host((int64_t)V.size());
    auto vglob = [&](const Block& b, int32_t l) {
        return (int32_t)(std::lower_bound(V.begin(), V.end(), b.V[l]) - V.begin());
    };
    std::vector<uint64_t> keys;
    for (auto& b : blocks)
        for (size_t t = 0; t < b.term_col.size(); ++t)
            keys.push_back(((uint64_t)(uint32_t)b.term_col[t] << vb) | (uint64_t)vglob(b, b.term_vidx[t]));
    std::sort(keys.begin(), keys.end());
    keys.erase(std::unique(keys.begin(), keys.end()), keys.end());
    if ((int64_t)keys.size() > INT32_MAX - 2) fail(GC_ERR_UNSUPPORTED, "more than 2^31-3 distinct terminals");
    g.V = V;
    g.term_col.resize(keys.size());
    g.term_vidx.resize(keys.size());
    for (size_t t = 0; t < keys.size(); ++t) {
        g.term_col[t] = (int32_t)(keys[t] >> vb);
        g.term_vidx[t] = (int32_t)(keys[t] & ((1ull << vb) - 1ull));
    }
    int64_t R = 0, C = 0;
    for (auto& b : blocks) {
        R += (int64_t)b.slp.rule_a.size();
        C += (int64_t)b.slp.c_sym.size();
    }
    if (R >= INT32_MAX) fail(GC_ERR_UNSUPPORTED, "more than 2^31-1 rules over all blocks");
    Slp& out = g.slp;
    out.rule_a.reserve((size_t)R);
    out.rule_b.reserve((size_t)R);
    out.c_sym.reserve((size_t)C);
    out.c_off.assign(1, 0);
    int32_t base = 0;
    for (auto& b : blocks) {
        std::vector<int32_t> tmap(b.term_col.size());
        for (size_t t = 0; t < tmap.size(); ++t) {
            const uint64_t key = ((uint64_t)(uint32_t)b.term_col[t] << vb) | (uint64_t)vglob(b, b.term_vidx[t]);
            tmap[t] = (int32_t)(std::lower_bound(keys.begin(), keys.end(), key) - keys.begin());
        }
        auto shift = [&](int32_t c) { return c >= 0 ? c + base : -(tmap[-c - 1] + 1); };
        for (size_t i = 0; i < b.slp.rule_a.size(); ++i) {
            out.rule_a.push_back(shift(b.slp.rule_a[i]));
            out.rule_b.push_back(shift(b.slp.rule_b[i]));
        }
        const int64_t c0 = (int64_t)out.c_sym.size();
        for (int32_t c : b.slp.c_sym) out.c_sym.push_back(shift(c));
        for (size_t r = 1; r < b.slp.c_off.size(); ++r) out.c_off.push_back(c0 + b.slp.c_off[r]);
        base += (int32_t)b.slp.rule_a.size();
        b = Block();   // release the block as soon as it is merged
    }
}

}  // namespace
}  // namespace gcs

using namespace gcs;

extern "C" {

const char* gc_last_error(void) { return g_last_error.c_str(); }

const char* gc_version(void) { return "gcsparse 0.1 sm_103a"; }

gc_status gc_build(int64_t n, int64_t m, const int64_t* row_ptr, const int32_t* col, const float* val,
                   const gc_build_opts* opts, gc_grammar** out) {
    return guard([&] {
        if (!out) fail(GC_ERR_ARG, "null output pointer");
        *out = nullptr;
        gc_build_opts o{0, 0, 0};
        if (opts) o = *opts;
        if (o.order != 0 && o.order != 1) fail(GC_ERR_ARG, "order must be 0 or 1");
        const double t0 = now_seconds();
        Csrv s = csrv_encode(n, m, row_ptr, col, val, o.threads);
        auto G = std::make_unique<gc_grammar>();
        Grammar& g = G->g;
        g.n = n;
        g.m = m;
        g.nnz = s.row_off[n];
        g.slp = repair_blocks(s, o.block_rows, o.threads, g.n_blocks);
        g.V = std::move(s.V);
        g.term_col = std::move(s.term_col);
        g.term_vidx = std::move(s.term_vidx);
        std::vector<int32_t>().swap(s.sym);
        g.repair_seconds = now_seconds() - t0;
        layer_and_pack(g, o.order);
        validate_packed(g);
        *out = G.release();
    });
}

gc_status gc_balance(const gc_grammar* gg, gc_grammar** out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null argument");
        *out = nullptr;
        const Grammar& g = gg->g;
        const double t0 = now_seconds();
        auto G = std::make_unique<gc_grammar>();
        Grammar& b = G->g;
        b.n = g.n;
        b.m = g.m;
        b.nnz = g.nnz;
        b.V = g.V;
        b.term_col = g.term_col;
        b.term_vidx = g.term_vidx;
        b.n_blocks = g.n_blocks;
        b.slp = balance_slp(g.slp);
        b.repair_seconds = g.repair_seconds + (now_seconds() - t0);
        layer_and_pack(b, 0);
        validate_packed(b);
        *out = G.release();
    });
}

gc_status gc_stats(const gc_grammar* gg, gc_grammar_stats* out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null argument");
        const Grammar& g = gg->g;
        gc_grammar_stats s{};
        s.n = g.n;
        s.m = g.m;
        s.nnz = g.nnz;
        s.n_values = (int64_t)g.V.size();
        s.n_terminals = g.alpha();
        s.n_rules = g.n_rules();
        s.n_pass = g.n_pass;
        s.n_nodes = g.n_nodes();
        s.depth = g.L;
        s.max_width = g.max_width();
        s.c_len = (int64_t)g.slp.c_sym.size();
        s.n_roots = g.n_roots;
        s.n_blocks = g.n_blocks;
        s.repair_seconds = g.repair_seconds;
        s.layer_seconds = g.layer_seconds;
        *out = s;
    });
}

gc_status gc_widths(const gc_grammar* gg, int64_t* w, int64_t cap) {
    return guard([&] {
        if (!gg || (!w && gg->g.L > 0)) fail(GC_ERR_ARG, "null argument");
        const Grammar& g = gg->g;
        if (cap < g.L) fail(GC_ERR_ARG, "width buffer shorter than depth");
        for (int64_t k = 1; k <= g.L; ++k) w[k - 1] = g.lvl_off[k + 1] - g.lvl_off[k];
    });
}

gc_status gc_export_size(const gc_grammar* gg, gc_array which, int64_t* bytes) {
    return guard([&] {
        if (!gg || !bytes) fail(GC_ERR_ARG, "null argument");
        *bytes = array_of(gg->g, which).bytes;
    });
}

gc_status gc_export(const gc_grammar* gg, gc_array which, void* dst, int64_t dst_bytes) {
    return guard([&] {
        if (!gg) fail(GC_ERR_ARG, "null grammar");
        const Grammar& g = gg->g;
        ArrayView a = array_of(g, which);
        if (dst_bytes < a.bytes) fail(GC_ERR_ARG, "destination too small");
        if (a.bytes == 0) return;
        if (!dst) fail(GC_ERR_ARG, "null destination");
        if (which == GC_A_RULES) {
            int32_t* d = static_cast<int32_t*>(dst);
            for (size_t i = 0; i < g.slp.rule_a.size(); ++i) {
                d[2 * i] = g.slp.rule_a[i];
                d[2 * i + 1] = g.slp.rule_b[i];
            }
        } else {
            std::memcpy(dst, a.ptr, (size_t)a.bytes);
        }
    });
}

gc_status gc_layout_ex(const gc_grammar* gg, gc_policy policy, int32_t k_max, int32_t schedule, gc_arena_layout* out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null argument");
        const Grammar& g = gg->g;
        check_policy(g, policy, k_max);
        const bool flow = wants_flow(schedule, k_max);
        DevLayout d;
        if (flow) {
            const FlowCounts fc = flow_counts(*flow_plan_for(gg, policy_elem_bytes(policy)));
            d = device_layout(g, policy, k_max, &fc);
        } else {
            d = device_layout(device_view(g, emit_mode(g, k_max) == EMIT_LEVEL), policy, k_max);
        }
        gc_arena_layout l{};
        l.arena_bytes = d.total;
        l.grammar_bytes = d.grammar_bytes;
        l.scratch_bytes = d.scratch_bytes;
        l.staging_bytes = d.staging_bytes;
        const int64_t rp = g.nnz >= INT32_MAX ? 8 * (g.n + 1) : 4 * (g.n + 1);
        l.csr_bytes = 8 * g.nnz + rp + d.value_bytes * (g.n + g.m);
        *out = l;
    });
}

gc_status gc_layout(const gc_grammar* gg, gc_policy policy, int32_t k_max, gc_arena_layout* out) {
    return gc_layout_ex(gg, policy, k_max, GC_SCHED_PERSISTENT, out);
}

gc_status gc_save(const gc_grammar* gg, const char* path) {
    return guard([&] {
        if (!gg || !path) fail(GC_ERR_ARG, "null argument");
        const Grammar& g = gg->g;
        FILE* f = std::fopen(path, "wb");
        if (!f) fail(GC_ERR_IO, std::string("cannot open ") + path);
        std::unique_ptr<FILE, int (*)(FILE*)> closer(f, &std::fclose);
        Writer w{f};
        w.raw(kMagic, 8);
        for (int64_t v : {g.n, g.m, g.nnz, g.L, g.n_pass, g.n_roots, g.n_blocks}) w.i64(v);
        w.raw(&g.repair_seconds, 8);
        w.raw(&g.layer_seconds, 8);
        fields(w, g);
    });
}

gc_status gc_load(const char* path, gc_grammar** out) {
    return guard([&] {
        if (!path || !out) fail(GC_ERR_ARG, "null argument");
        *out = nullptr;
        FILE* f = std::fopen(path, "rb");
        if (!f) fail(GC_ERR_IO, std::string("cannot open ") + path);
        std::unique_ptr<FILE, int (*)(FILE*)> closer(f, &std::fclose);
        Reader r{f};
        char magic[8];
        r.raw(magic, 8);
        if (std::memcmp(magic, kMagic, 8) != 0) fail(GC_ERR_IO, "not a gcsparse grammar file");
        auto G = std::make_unique<gc_grammar>();
        Grammar& g = G->g;
        g.n = r.i64();
        g.m = r.i64();
        g.nnz = r.i64();
        g.L = r.i64();
        g.n_pass = r.i64();
        g.n_roots = r.i64();
        g.n_blocks = r.i64();
        r.raw(&g.repair_seconds, 8);
        r.raw(&g.layer_seconds, 8);
        fields(r, g);
        validate_packed(g);
        *out = G.release();
    });
}

void gc_free_grammar(gc_grammar* g) { delete g; }

}  // extern "C"

struct gc_builder {
    int64_t n = 0, m = 0;
    gc_build_opts opts{0, 0, 0};
    std::mutex mu;
    std::vector<gcs::Block> blocks;
    int64_t rows_added = 0;
    double seconds = 0;
};

extern "C" {

gc_status gc_builder_create(int64_t n, int64_t m, const gc_build_opts* opts, gc_builder** out) {
    return guard([&] {
        if (!out) fail(GC_ERR_ARG, "null output pointer");
        if (n < 0 || m < 0) fail(GC_ERR_ARG, "negative matrix shape");
        auto b = std::make_unique<gc_builder>();
        b->n = n;
        b->m = m;
        if (opts) b->opts = *opts;
        if (b->opts.order != 0 && b->opts.order != 1) fail(GC_ERR_ARG, "order must be 0 or 1");
        *out = b.release();
    });
}

gc_status gc_builder_add_rows(gc_builder* b, int64_t r0, int64_t rows, const int64_t* row_ptr, const int32_t* col,
                              const float* val) {
    return guard([&] {
        if (!b) fail(GC_ERR_ARG, "null builder");
        if (r0 < 0 || rows < 0 || r0 + rows > b->n) fail(GC_ERR_ARG, "row block outside [0, n)");
        const double t0 = now_seconds();
        Block blk;
        blk.r0 = r0;
        blk.rows = rows;
        {
            Csrv s = csrv_encode(rows, b->m, row_ptr, col, val, b->opts.threads);
            blk.slp = repair(s, 0, rows);
            blk.V = std::move(s.V);
            blk.term_col = std::move(s.term_col);
            blk.term_vidx = std::move(s.term_vidx);
        }
        const double dt = now_seconds() - t0;
        std::lock_guard<std::mutex> lock(b->mu);
        for (auto& o : b->blocks)
            if (r0 < o.r0 + o.rows && o.r0 < r0 + rows) fail(GC_ERR_ARG, "row blocks overlap");
        b->blocks.push_back(std::move(blk));
        b->rows_added += rows;
        b->seconds += dt;
    });
}

gc_status gc_builder_finish(gc_builder* b, gc_grammar** out) {
    return guard([&] {
        if (!b || !out) fail(GC_ERR_ARG, "null argument");
        *out = nullptr;
        std::lock_guard<std::mutex> lock(b->mu);
        if (b->rows_added != b->n) fail(GC_ERR_ARG, "row blocks do not cover all n rows");
        std::sort(b->blocks.begin(), b->blocks.end(), [](const Block& x, const Block& y) { return x.r0 < y.r0; });
        auto G = std::make_unique<gc_grammar>();
        Grammar& g = G->g;
        g.n = b->n;
        g.m = b->m;
        g.n_blocks = (int64_t)b->blocks.size();
        const double t0 = now_seconds();
        merge_blocks(b->blocks, g);
        b->blocks.clear();
        g.nnz = 0;
        g.repair_seconds = b->seconds + (now_seconds() - t0);
        layer_and_pack(g, b->opts.order);
        validate_packed(g);
        // stored non-zeros: the expansion lengths of C
        {
            std::vector<int64_t> len(g.slp.rule_a.size());
            for (size_t i = 0; i < len.size(); ++i) {
                const int32_t a = g.slp.rule_a[i], c = g.slp.rule_b[i];
                len[i] = (a >= 0 ? len[a] : 1) + (c >= 0 ? len[c] : 1);
            }
            for (int32_t c : g.slp.c_sym) g.nnz += c >= 0 ? len[c] : 1;
        }
        *out = G.release();
    });
}

void gc_builder_free(gc_builder* b) { delete b; }

}  // extern "C"
