// Checks the left product's host plan (left.hpp) on the CPU: builds it for a
// matrix, validates it, and replays its tasks the way left_step_kernel does
// (LIGHT: one segment per lane of a run of 32, in order from its initial
// value, segments over kLeftLightMax items left to their HEAVY task; HEAVY: 32
// lane partial sums in order, then the xor butterfly, added to the initial
// value), in float32 with every operation rounded separately and again in
// float64. Compares x with a direct M^T y: the float64 replay within 1e-9,
// the float32 replay within 1e-4 (|M|^T |y|)_j, and exactly 0 where that
// bound is 0. Also checks the float32 replay's worst scaled error against
// the depth bound the plan promises.
//
// Input files: int64 n, m, nnz; int64 row_ptr[n+1]; int32 col[nnz];
// float32 val[nnz]. Exit status 0 when every check holds.
#include <cmath>
#include <cstdio>
#include <random>

#include "common.hpp"
#include "gcsparse.h"
#include "layout.hpp"
#include "left.hpp"

using namespace gcs;

template <class T>
static std::vector<T> replay(const LeftPlan& p, const std::vector<T>& y) {
    std::vector<T> RS((size_t)(p.rho + p.alpha)), W((size_t)p.N), TIN((size_t)p.alpha), x((size_t)p.m);
    auto run = [&](int64_t set, const std::vector<int32_t>& off, auto init, auto item, auto store) {
        for (int64_t t = p.task_off[set]; t < p.task_off[set + 1]; ++t) {
            const int32_t first = p.task[2 * t], cnt = p.task[2 * t + 1];
            if (cnt > 0) {
                for (int32_t l = 0; l < cnt; ++l) {
                    const int32_t g = first + l;
                    if (off[g + 1] - off[g] > kLeftLightMax) continue;   // its HEAVY task sums it
                    T acc = init(g);
                    for (int32_t q = off[g]; q < off[g + 1]; ++q) acc = acc + item(q);
                    store(g, acc);
                }
            } else {
                const int32_t g = first;
                T lane[32];
                for (int l = 0; l < 32; ++l) {
                    lane[l] = T(0);
                    for (int32_t q = off[g] + l; q < off[g + 1]; q += 32) lane[l] = lane[l] + item(q);
                }
                for (int msk = 16; msk >= 1; msk >>= 1) {
                    T nxt[32];
                    for (int l = 0; l < 32; ++l) nxt[l] = lane[l] + lane[l ^ msk];
                    for (int l = 0; l < 32; ++l) lane[l] = nxt[l];
                }
                store(g, init(g) + lane[0]);
            }
        }
    };
    run(0, p.soff, [&](int32_t) { return T(0); }, [&](int32_t q) { return y[p.srow[q]]; },
        [&](int32_t g, T v) { RS[g] = v; });
    for (int64_t k = p.L; k >= 1; --k) {
        const int64_t base = p.lvl_off[k], nr = p.lvl_roots[k], roff = p.root_off[k];
        run(k, p.poff, [&](int32_t g) { return g - base < nr ? RS[roff + (g - base)] : T(0); },
            [&](int32_t q) { return W[p.pref[q]]; }, [&](int32_t g, T v) { W[g] = v; });
    }
    run(p.L + 1, p.toff, [&](int32_t g) { return RS[p.rho + g]; }, [&](int32_t q) { return W[p.tref[q]]; },
        [&](int32_t g, T v) { TIN[g] = v; });
    run(p.L + 2, p.coff, [&](int32_t) { return T(0); },
        [&](int32_t q) { return T(p.V[p.term_vidx[q]]) * TIN[q]; }, [&](int32_t g, T v) { x[g] = v; });
    return x;
}

static int check(const char* name, const Grammar& g, const std::vector<int64_t>& rp, const std::vector<int32_t>& col,
                 const std::vector<float>& val, uint64_t seed) {
    const LeftPlan p = plan_left(g);
    validate_left_plan(p);
    std::mt19937_64 rng(seed);
    std::normal_distribution<float> N01(0.0f, 1.0f);
    std::vector<float> yf((size_t)g.n);
    for (float& v : yf) v = N01(rng);
    std::vector<double> yd(yf.begin(), yf.end());
    std::vector<double> xr((size_t)g.m, 0.0), b((size_t)g.m, 0.0);
    for (int64_t i = 0; i < g.n; ++i)
        for (int64_t e = rp[i]; e < rp[i + 1]; ++e) {
            xr[col[e]] += (double)val[e] * yd[i];
            b[col[e]] += std::fabs((double)val[e] * yd[i]);
        }
    const std::vector<double> xd = replay<double>(p, yd);
    const std::vector<float> xf = replay<float>(p, yf);
    double worst = 0.0;
    int bad = 0;
    for (int64_t j = 0; j < g.m; ++j) {
        if (std::fabs(xd[j] - xr[j]) > 1e-9 * (b[j] + 1e-300)) bad = 1;
        if (b[j] == 0.0 ? xf[j] != 0.0f : std::fabs((double)xf[j] - xr[j]) > 1e-4 * b[j]) bad = 1;
        if (b[j] > 0) worst = std::max(worst, std::fabs((double)xf[j] - xr[j]) / b[j]);
    }
    int64_t heavy = 0, longest = 0;
    for (int64_t t = 0; t < p.n_tasks(); ++t)
        if (p.task[2 * t + 1] < 0) ++heavy;
    for (int64_t u = 0; u < p.N; ++u) longest = std::max<int64_t>(longest, p.poff[u + 1] - p.poff[u]);
    std::printf("%s: n %lld m %lld L %lld N %lld tasks %lld heavy %lld longest parent list %lld, float32 worst scaled "
                "error %.3e%s\n",
                name, (long long)g.n, (long long)g.m, (long long)g.L, (long long)p.N, (long long)p.n_tasks(),
                (long long)heavy, (long long)longest, worst, bad ? "  FAIL" : "");
    return bad;
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
        try {
            bad |= check(argv[a], gg->g, rp, col, v, 17 + a);
        } catch (const Error& e) {
            std::printf("%s: %s  FAIL\n", argv[a], e.what());
            bad = 1;
        }
        gc_free_grammar(gg);
    }
    std::printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
