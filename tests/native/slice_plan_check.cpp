// Checks two host-side constructions of the device path on the CPU.
//
// check_view: evaluates the device view of the grammar (pass-throughs replaced
// by carry slots, levels compacted, C's roots renumbered) level by level from a
// random x, exactly as the sweep reads it, and compares y with the direct
// product of the input CSR matrix.
//
// check_slices: builds the slice plan the library uploads, replays the
// per-lane runs and the segmented lane scan that tile_sums performs on the
// device (over random values standing in for [T | RV]), and compares every
// row's sum of segment sums with the direct sum of the row's early
// references. Also checks that every segment start is written exactly once
// and that the counts used to size the arena match the plan.
//
// Input files: int64 n, m, nnz; int64 row_ptr[n+1]; int32 col[nnz];
// float32 val[nnz]. Exit status 0 when every check holds.
#include <cmath>
#include <cstdio>
#include <random>

#include "common.hpp"
#include "gcsparse.h"
#include "layout.hpp"

using namespace gcs;

static int check_view(const Grammar& host, const Grammar& g, const std::vector<int64_t>& rp,
                      const std::vector<int32_t>& col, const std::vector<float>& val) {
    validate_device_view(g);
    const int64_t A = g.alpha(), L = g.L;
    std::mt19937_64 rng(7);
    std::uniform_real_distribution<double> U(-1, 1);
    std::vector<double> x((size_t)g.m);
    for (double& v : x) v = U(rng);
    std::vector<double> T((size_t)A);
    for (int64_t p = 0; p < A; ++p) T[p] = (double)g.V[g.term_vidx[p]] * x[g.term_col[p]];
    std::vector<std::vector<double>> lv((size_t)L + 1);
    std::vector<double> carry((size_t)std::max<int64_t>(1, g.n_carry));
    for (int64_t k = 1; k <= L; ++k) {
        const int64_t w = g.lvl_off[k + 1] - g.lvl_off[k];
        lv[k].assign((size_t)w, 0);
        auto child = [&](int32_t c) -> double {
            if (c >= 0) return lv[k - 1][c];
            if (c == -1) return 0.0;   // a pass-through's identity
            if (c >= -(A + 1)) return T[-c - 2];
            return carry[carry_slot(c, A)];
        };
        for (int64_t t = 0; t < w; ++t) {
            const double v = child(g.nodes[2 * (g.lvl_off[k] + t)]) + child(g.nodes[2 * (g.lvl_off[k] + t) + 1]);
            lv[k][t] = v;
            const int64_t cr = g.carry_roots[k], cn = g.carry_rest[k], nr = g.lvl_roots[k];
            const int64_t cs = t < cr ? t : (t >= nr && t - nr < cn) ? cr + (t - nr) : -1;
            if (cs >= 0) carry[g.carry_off[k] + cs] = v;
        }
    }
    double worst = 0;
    for (int64_t r = 0; r < g.n; ++r) {
        double got = 0, want = 0, mag = 0;
        for (int64_t e = g.slp.c_off[r]; e < g.slp.c_off[r + 1]; ++e) {
            const int32_t c = g.c_ref[e];
            if (c < 0) {
                got += T[-c - 2];
            } else {
                const int64_t k = ref_level(g, c);
                got += lv[k][c - g.root_off[k]];
            }
        }
        for (int64_t e = rp[r]; e < rp[r + 1]; ++e) {
            want += (double)val[e] * x[col[e]];
            mag += std::fabs((double)val[e] * x[col[e]]);
        }
        worst = std::max(worst, std::fabs(got - want) / (mag + 1e-300));
    }
    std::printf("view: n %ld nodes %ld (layered %ld) carried %ld  max scaled |y difference| %.3g\n", (long)g.n,
                (long)g.lvl_off[L + 1], (long)host.n_nodes(), (long)g.n_carry, worst);
    return worst < 1e-12 ? 0 : 1;
}

static int check_slices(const Grammar& g, int64_t value_bytes, int64_t tail_nodes) {
    const int64_t TB = leaf_block(g.alpha());
    const int64_t Lg = grid_level_count(g, tail_nodes);
    const int64_t S = slice_len(value_bytes);
    const SlicePlan p = plan_slice_emit(g, TB, Lg, S);
    validate_slice_plan(p, g, TB, Lg);
    const SliceCounts c = count_slice_emit(g, TB, Lg, S);
    if (c.ids != p.nids || c.tiles != p.ntiles || c.starts != (int64_t)p.tsid.size() || c.slices != p.nslices) {
        std::printf("arena counts differ from the plan\n");
        return 1;
    }
    std::mt19937_64 rng(1);
    std::uniform_real_distribution<double> U(-1, 1);
    std::vector<double> val((size_t)(TB + g.n_roots));
    for (double& v : val) v = U(rng);
    const int64_t NST = (int64_t)p.tsid.size();
    std::vector<double> esum((size_t)NST, NAN);
    std::vector<int> written((size_t)NST, 0);
    auto put = [&](int64_t i, double v) {
        esum[i] = v;
        ++written[i];
    };
    for (int64_t s = 0; s < p.nslices; ++s)
        for (int64_t t = p.stile[s]; t < p.stile[s + 1]; ++t) {
            const int64_t base = p.tile_sid[t];
            double v[32][8], cur[32], head[32], X[32];
            uint32_t f[32];
            int nf[32], before[32], incl[32];
            bool F[32];
            for (int l = 0; l < 32; ++l) {
                f[l] = p.sflag[t * 32 + l];
                nf[l] = __builtin_popcount(f[l]);
                for (int i = 0; i < 8; ++i) v[l][i] = val[p.x0[s] + p.sref[t * 256 + l * 8 + i]];
            }
            for (int l = 0, acc = 0; l < 32; ++l) {
                before[l] = acc;
                acc += nf[l];
                incl[l] = acc;
            }
            for (int l = 0; l < 32; ++l) {   // runs inside each lane
                cur[l] = head[l] = 0;
                bool open_head = true;
                int k = before[l] - 1;
                for (int i = 0; i < 8; ++i) {
                    if ((f[l] >> i) & 1u) {
                        if (open_head) {
                            head[l] = cur[l];
                            open_head = false;
                        } else {
                            put(base + k, cur[l]);
                        }
                        ++k;
                        cur[l] = 0;
                    }
                    cur[l] += v[l][i];
                }
                F[l] = f[l] != 0;
                X[l] = cur[l];
            }
            for (int d = 1; d < 32; d <<= 1) {   // Hillis-Steele segmented scan, as on the device
                bool Fn[32];
                double Xn[32];
                for (int l = 0; l < 32; ++l) {
                    Fn[l] = F[l];
                    Xn[l] = X[l];
                    if (l >= d) {
                        if (!F[l]) Xn[l] = X[l - d] + X[l];
                        Fn[l] = F[l] || F[l - d];
                    }
                }
                for (int l = 0; l < 32; ++l) {
                    F[l] = Fn[l];
                    X[l] = Xn[l];
                }
            }
            for (int l = 0; l < 32; ++l)
                if (f[l] && before[l] >= 1) put(base + before[l] - 1, (l >= 1 ? X[l - 1] : 0) + head[l]);
            if (incl[31] >= 1) put(base + incl[31] - 1, X[31]);
        }
    for (int64_t i = 0; i < NST; ++i)
        if (written[i] != 1) {
            std::printf("segment start %ld written %d times\n", (long)i, written[i]);
            return 1;
        }
    double worst = 0;
    for (int64_t r = 0; r < g.n; ++r) {
        double got = 0, want = 0;
        for (int32_t i = p.row_seg[r]; i < p.row_seg[r + 1]; ++i) got += esum[p.row_pos[i]];
        for (int64_t e = g.slp.c_off[r]; e < g.slp.c_off[r + 1]; ++e)
            if (ref_level(g, g.c_ref[e]) <= Lg) want += val[slice_index(TB, g.c_ref[e])];
        worst = std::max(worst, std::fabs(got - want));
    }
    std::printf("n %ld slices %ld tiles %ld sums %ld starts %ld max |row difference| %.3g\n", (long)g.n,
                (long)p.nslices, (long)p.ntiles, (long)p.nids, (long)NST, worst);
    return worst < 1e-9 ? 0 : 1;
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
        for (bool carry : {true, false}) bad |= check_view(gg->g, device_view(gg->g, carry), rp, col, v);
        const Grammar dv = device_view(gg->g, false);
        for (int64_t vb : {4, 8})
            for (int64_t tail : {kSliceTailNodes, (int64_t)4096, (int64_t)1024}) bad |= check_slices(dv, vb, tail);
        gc_free_grammar(gg);
    }
    std::printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
