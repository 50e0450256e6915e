// Checks the dataflow sweep's block plan (flow.hpp) on the CPU.
//
// For each input matrix and value width (4 and 8 bytes) it builds the plan the
// library uploads, runs its host checks, and replays the blocks in order the
// way the device runs them: every node of a regular block reads its two
// children from the level buffer of the level below (or the identity, or a
// leaf code evaluated from x), writes its value to buffer k % 3 and, if it is
// a root, to RV; the final block copies the level below into its staging
// array and keeps its own levels there. y is then the sum of each row's C references (T for bare
// terminals, RV for roots), compared with the direct product of the input CSR
// matrix in float64.
//
// Input files: int64 n, m, nnz; int64 row_ptr[n+1]; int32 col[nnz];
// float32 val[nnz]. Exit status 0 when every check holds.
#include <cmath>
#include <cstdio>
#include <random>

#include "common.hpp"
#include "flow.hpp"
#include "gcsparse.h"

using namespace gcs;

static int check_flow(const Grammar& g, int64_t vb, const std::vector<int64_t>& rp, const std::vector<int32_t>& col,
                      const std::vector<float>& val) {
    const FlowPlan p = plan_flow(g, vb);
    validate_flow_plan(p, g);
    const int64_t L = g.L, G = flow_granule(vb), A = g.alpha();
    const int32_t vbits = value_bits((int64_t)g.V.size());
    std::mt19937_64 rng(11);
    std::uniform_real_distribution<double> U(-1, 1);
    std::vector<double> x((size_t)g.m);
    for (double& v : x) v = U(rng);
    auto leaf = [&](int64_t q) { return (double)g.V[q & ((1 << vbits) - 1)] * x[q >> vbits]; };
    // level buffers start with garbage: a read of a slot nobody wrote shows up
    std::vector<std::vector<double>> buf(3, std::vector<double>((size_t)p.buf_values, 1e300));
    std::vector<double> rv((size_t)g.n_roots, 1e300);
    int64_t regular = 0, finals = 0, staged = 0, nodes = 0, ngran = 0;
    for (int64_t q = 0; q < p.nblocks; ++q) {   // in the processing order
        const int64_t b = p.order[q];
        const int32_t* f = p.blk.data() + b * kFlowBlkInts;
        const int64_t k0 = f[FB_K0], k1 = f[FB_K1];
        const std::vector<double>& prev = buf[(k0 + 2) % 3];
        std::vector<double> st;
        for (int64_t s = f[FB_WS1]; s < f[FB_WS1] + f[FB_WL1]; ++s) st.push_back(prev[s]);
        for (int64_t s = f[FB_WS2]; s < f[FB_WS2] + f[FB_WL2]; ++s) st.push_back(prev[s]);
        for (int64_t j = 0; j < f[FB_NGRAN]; ++j)
            for (int64_t s = p.gran[f[FB_GOFF] + j]; s < p.gran[f[FB_GOFF] + j] + G; ++s) st.push_back(prev[s]);
        staged += (int64_t)st.size();
        ngran += f[FB_NGRAN];
        const bool fin = k0 >= p.final_k0;
        // a regular block reads its children from the level buffer of k0-1,
        // the final block from its staged values
        auto child = [&](int32_t c) -> double {
            if (c >= 0) return fin ? st.at((size_t)c) : prev.at((size_t)c);
            if (c == -1) return 0.0;
            return leaf(-(int64_t)c - 2);
        };
        if (fin) {
            ++finals;
            for (int64_t k = k0; k <= k1; ++k) {
                const int64_t w = g.lvl_off[k + 1] - g.lvl_off[k];
                std::vector<double> lv((size_t)((w + G - 1) / G * G), 1e300);
                for (int64_t t = 0; t < w; ++t) {
                    const int32_t* e = p.pairs.data() + 2 * (p.lvl_start[k] + t);
                    lv[t] = child(e[0]) + child(e[1]);
                    if (t < g.lvl_roots[k]) rv[g.root_off[k] + t] = lv[t];
                }
                nodes += w;
                st.insert(st.end(), lv.begin(), lv.end());
            }
        } else {
            ++regular;
            std::vector<double>& out = buf[k0 % 3];
            for (int64_t i = 0; i < f[FB_NNODES]; ++i) {
                const int32_t* e = p.pairs.data() + 2 * ((int64_t)f[FB_NODE0] + i);
                const int64_t t = f[FB_SLOT0] + i;
                out[t] = child(e[0]) + child(e[1]);
                if (t < g.lvl_roots[k0]) rv[g.root_off[k0] + t] = out[t];
            }
            nodes += f[FB_NNODES];
        }
    }
    double worst = 0;
    for (int64_t r = 0; r < g.n; ++r) {
        double got = 0, want = 0, mag = 0;
        for (int64_t e = g.slp.c_off[r]; e < g.slp.c_off[r + 1]; ++e) {
            const int32_t c = g.c_ref[e];
            got += c >= 0 ? rv[c] : (double)g.V[g.term_vidx[-c - 2]] * x[g.term_col[-c - 2]];
        }
        for (int64_t e = rp[r]; e < rp[r + 1]; ++e) {
            want += (double)val[e] * x[col[e]];
            mag += std::fabs((double)val[e] * x[col[e]]);
        }
        worst = std::max(worst, std::fabs(got - want) / (mag + 1e-300));
    }
    std::printf("flow vb=%ld: L %ld blocks %ld (final from level %ld) nodes %ld staged/node %.2f granules %ld "
                "max scaled |y difference| %.3g\n",
                (long)vb, (long)L, (long)p.nblocks, (long)p.final_k0, (long)nodes,
                nodes ? (double)staged / (double)nodes : 0.0, (long)ngran, worst);
    (void)A;
    return (worst < 1e-12 && nodes == g.n_nodes() && regular + finals == p.nblocks) ? 0 : 1;
}

int main(int argc, char** argv) {
    int bad = 0;
    for (int a = 1; a < argc; ++a) {
        FILE* fp = std::fopen(argv[a], "rb");
        if (!fp) return 2;
        int64_t hdr[3];
        if (std::fread(hdr, 8, 3, fp) != 3) return 2;
        const int64_t n = hdr[0], m = hdr[1], nnz = hdr[2];
        std::vector<int64_t> rp((size_t)n + 1);
        std::vector<int32_t> col((size_t)nnz);
        std::vector<float> v((size_t)nnz);
        if (std::fread(rp.data(), 8, rp.size(), fp) != rp.size() || std::fread(col.data(), 4, col.size(), fp) != col.size() ||
            std::fread(v.data(), 4, v.size(), fp) != v.size())
            return 2;
        std::fclose(fp);
        gc_grammar* gg = nullptr;
        if (gc_build(n, m, rp.data(), col.data(), v.data(), nullptr, &gg) != GC_OK) return 2;
        for (int64_t vb : {4, 8}) {
            try {
                bad |= check_flow(gg->g, vb, rp, col, v);
            } catch (const Error& e) {
                std::printf("%s: %s\n", argv[a], e.what());
                bad = 1;
            }
        }
        gc_free_grammar(gg);
    }
    std::printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
