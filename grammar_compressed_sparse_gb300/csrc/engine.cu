// Device side of gcsparse: upload of the packed grammar into a caller-owned
// arena, and the streaming bottom-up sweep of Sec. 4.3 of the pages ("Right
// Multiplication on Grammar-Compressed Matrices"), written for sm_103a.
//
//   leaf table      T[0] = identity, T[p+1] = V[l_p] (x) x[j_p]          (Sec. 4.3)
//   level combine   for k = 1..L: cur[t] = cv(a_t) (+) cv(b_t) with one load
//                   per child from the previous level's buffer, which has T
//                   in front (see layout.hpp); the level's roots (its first
//                   nodes) are also written to RV, the emit-on-the-spot
//                   capture                                  (Listing 1, Lemma 3.3)
//   row emit        y[r] = (+) over row r's symbols of RV / T entries   (Lemma 2.2)
//
// Schedule (differences from the pages' two launches per level, for this GPU):
//   * one persistent cooperative kernel per product, two CTAs of 512 threads
//     per SM; levels are separated by a grid barrier whose waits are bounded
//     (a wait that runs out sets the status word and the kernel returns);
//   * within a level every warp works on its own chunks of 128 nodes
//     (4 per lane, coalesced), with no block-wide synchronisation, and loads
//     the next chunk's child pairs -- possibly of the next level, since pairs
//     do not depend on values -- before gathering the current chunk's
//     children, so node-stream latency hides behind gathers and barriers;
//   * level 1 evaluates its (all-terminal) children in the sweep while the
//     grid writes the three T copies, so T costs no phase of its own;
//   * child values are gathered through L1/L2 (the grid barrier's gpu-scope
//     acquire orders them after the writers); root values are stored with an
//     L2 evict-last policy so the emit finds them in L2; the node and C
//     streams are loaded evict-first;
//   * the narrow top levels run on one CTA with block-level barriers;
//   * the pages emit with atomicAdd into y; here each row is reduced by a
//     fixed group of threads in a fixed order: deterministic, no atomics.
// A second schedule launches one kernel per level plus one emit kernel with
// the same device functions (bit-identical y): the launch sequence of
// Listing 1, kept as the reference point for the persistent one.
#include <cuda_runtime.h>

#include <cstring>
#include <memory>
#include <mutex>

#include "common.hpp"
#include "layout.hpp"
#include "policy.cuh"

struct gc_handle {
    gc_policy policy = GC_F32_SUM;
    int32_t k_max = 1;
    int64_t n = 0, m = 0, L = 0, n_roots = 0, c_len = 0, max_width = 0, alpha = 0;
    std::vector<int64_t> lv;      // host copy of the level table, 4 (L+2)
    char* arena = nullptr;
    gcs::DevLayout lay{};
    int sms = 1;
    int emit_group = 32;          // threads per row in the emit; 0 = one CTA per row
    int schedule = 0;             // 0 persistent (if cooperative launch works), 1 per level
    int coop = 0;                 // device supports cooperative launch
    int grid_levels = 0;          // levels 1..grid_levels use the whole grid
    unsigned long long bar_base = 0;
    long long timeout_cycles = 4000000000LL;
    int32_t inject = 0;           // test-only: 1 = CTA 0 skips its first barrier arrival
    int64_t launches = 0;
};

namespace gcs {
namespace {

constexpr int kThreads = 512;        // every kernel: 16 warps
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;                // nodes (or node lanes) per thread per chunk
constexpr int LV_START = 0, LV_W = 1, LV_ROOTS = 2, LV_ROFF = 3;

void cuda_check(cudaError_t e, const char* what) {
    if (e != cudaSuccess) fail(GC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

template <class P>
struct Chunk {
    static constexpr int NPW = 32 / P::LPN;          // nodes per warp row
    static constexpr int NODES = NPW * kU;           // nodes per warp chunk
    static constexpr int TAIL = NODES * kWarps * 2;  // widest level left to one CTA
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void red_add_release(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_volatile(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }

__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// stores that ask L2 to keep the line (root values, read again by the emit)
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(float4* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_keep(long long* p, long long v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(p), "l"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(unsigned long long* p, unsigned long long v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(p), "l"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ float shfl_x(float v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ long long shfl_x(long long v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ unsigned long long shfl_x(unsigned long long v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
}
__device__ __forceinline__ float4 shfl_x(float4 v, int m) {
    return make_float4(shfl_x(v.x, m), shfl_x(v.y, m), shfl_x(v.z, m), shfl_x(v.w, m));
}

// ---------------------------------------------------------------- arguments
template <class P>
struct SweepArgs {
    using V = typename P::V;
    const int2* nodes;
    const int64_t* lv;        // level table: 4 rows of L+2
    int32_t L, L2, grid_levels;
    int64_t TB;               // leaf-table block length (values)
    int64_t alpha;
    const typename P::Leaf* Vd;
    const int32_t* leaf;      // leaf code per terminal
    int32_t vbits;
    const V* x;
    V* y;
    V* buf0;                  // [T | level values]
    V* buf1;
    V* rv;                    // [T | root values]
    const int32_t* c_off;
    const int32_t* c_ref;
    int64_t n;
    int32_t emit_group;
    int32_t* status;
    unsigned long long* bar;
    unsigned long long bar_base;
    long long timeout;
    int32_t inject;

    __device__ __forceinline__ int64_t lvl(int row, int k) const { return __ldg(lv + (int64_t)row * L2 + k); }
};

// V[l] (x) x[j] for a leaf code (column << vbits | value index)
template <class P>
__device__ __forceinline__ typename P::V leaf_value(int32_t code, int part, const SweepArgs<P>& a) {
    const uint32_t q = (uint32_t)code;
    const uint32_t col = q >> a.vbits, vi = q & ((1u << a.vbits) - 1u);
    return P::leaf(__ldg(a.Vd + vi), __ldg(a.x + (int64_t)col * P::LPN + part));
}

// The three leaf-table copies (in front of buf0, buf1 and RV), grid-stride.
template <class P>
__device__ void write_leaf_tables(const SweepArgs<P>& a, int64_t tid, int64_t nthreads) {
    using V = typename P::V;
    const int64_t total = (a.alpha + 1) * P::LPN;
    for (int64_t i = tid; i < total; i += nthreads) {
        const int64_t p = i / P::LPN;
        const int part = (int)(i % P::LPN);
        const V v = p == 0 ? P::identity() : leaf_value<P>(__ldg(a.leaf + (p - 1)), part, a);
        a.buf0[i] = v;
        a.buf1[i] = v;
        a.rv[i] = v;
    }
}

// Loads the child pairs of chunk c of level k (this warp's lanes).
template <class P>
__device__ __forceinline__ void load_chunk(const SweepArgs<P>& a, int k, int64_t c, int2 (&ab)[kU]) {
    constexpr int NPW = Chunk<P>::NPW;
    const int lane = threadIdx.x & 31;
    const int64_t w = a.lvl(LV_W, k);
    const int2* src = a.nodes + a.lvl(LV_START, k);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
        ab[u] = node < w ? __ldcs(src + node) : make_int2(0, 0);
    }
}

// Combines chunk c of level k from its prefetched child pairs.
template <class P>
__device__ __forceinline__ void combine_chunk(const SweepArgs<P>& a, int k, int64_t c, const int2 (&ab)[kU],
                                              uint64_t keep) {
    using V = typename P::V;
    constexpr int NPW = Chunk<P>::NPW;
    const int lane = threadIdx.x & 31;
    const int part = lane % P::LPN;
    const int64_t w = a.lvl(LV_W, k), nroots = a.lvl(LV_ROOTS, k);
    const V* prev = (k & 1) ? a.buf0 : a.buf1;
    V* cur = ((k & 1) ? a.buf1 : a.buf0) + a.TB * P::LPN;
    V* rv = a.rv + (a.TB + a.lvl(LV_ROFF, k)) * P::LPN;
    V va[kU], vb[kU];
    if (k == 1) {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
            va[u] = node < w ? leaf_value<P>(ab[u].x, part, a) : P::identity();
            vb[u] = node < w ? leaf_value<P>(ab[u].y, part, a) : P::identity();
        }
    } else {
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            va[u] = prev[(int64_t)ab[u].x * P::LPN + part];
            vb[u] = prev[(int64_t)ab[u].y * P::LPN + part];
        }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
        if (node < w) {
            const V v = P::combine(va[u], vb[u]);
            cur[node * P::LPN + part] = v;
            if (node < nroots) st_keep(rv + node * P::LPN + part, v, keep);
        }
    }
}

// ---------------------------------------------------------------- row emit
constexpr int kEmitBatch = 4;

// G threads per row (G divides 32); warps walk rows in lockstep so the
// shuffles always see the full warp. Thread gl sums its symbols q = s+gl,
// s+gl+G, ... in order, then the group reduces by a fixed butterfly.
template <class P, int G>
__device__ void emit_groups(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    using V = typename P::V;
    constexpr int RPW = 32 / G;
    const int lane = threadIdx.x & 31;
    const int gl = lane % G;
    const int64_t warp = block * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = nblocks * kWarps;
    for (int64_t base = warp * RPW; base < a.n; base += nwarps * RPW) {
        const int64_t row = base + lane / G;
        V acc[P::LPN];
#pragma unroll
        for (int l = 0; l < P::LPN; ++l) acc[l] = P::identity();
        if (row < a.n) {
            const int32_t s = __ldg(a.c_off + row), e = __ldg(a.c_off + row + 1);
            for (int32_t q0 = s + gl; q0 < e; q0 += G * kEmitBatch) {
                int32_t c[kEmitBatch];
#pragma unroll
                for (int u = 0; u < kEmitBatch; ++u) c[u] = q0 + u * G < e ? __ldcs(a.c_ref + q0 + u * G) : 0;
                V v[kEmitBatch][P::LPN];
#pragma unroll
                for (int u = 0; u < kEmitBatch; ++u)
#pragma unroll
                    for (int l = 0; l < P::LPN; ++l) v[u][l] = a.rv[(int64_t)c[u] * P::LPN + l];
#pragma unroll
                for (int u = 0; u < kEmitBatch; ++u)
#pragma unroll
                    for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], v[u][l]);
            }
        }
#pragma unroll
        for (int msk = G / 2; msk >= 1; msk >>= 1)
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], shfl_x(acc[l], msk));
        if (row < a.n && gl == 0)
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) a.y[row * P::LPN + l] = acc[l];
    }
}

// One CTA per row, for long rows of C.
template <class P>
__device__ void emit_ctas(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    using V = typename P::V;
    __shared__ V red[kWarps][P::LPN];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t row = block; row < a.n; row += nblocks) {
        V acc[P::LPN];
#pragma unroll
        for (int l = 0; l < P::LPN; ++l) acc[l] = P::identity();
        const int32_t s = __ldg(a.c_off + row), e = __ldg(a.c_off + row + 1);
        for (int32_t q0 = s + threadIdx.x; q0 < e; q0 += kThreads * kEmitBatch) {
            int32_t c[kEmitBatch];
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u) c[u] = q0 + u * kThreads < e ? __ldcs(a.c_ref + q0 + u * kThreads) : 0;
            V v[kEmitBatch][P::LPN];
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u)
#pragma unroll
                for (int l = 0; l < P::LPN; ++l) v[u][l] = a.rv[(int64_t)c[u] * P::LPN + l];
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u)
#pragma unroll
                for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], v[u][l]);
        }
#pragma unroll
        for (int msk = 16; msk >= 1; msk >>= 1)
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], shfl_x(acc[l], msk));
        if (lane == 0)
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) red[wid][l] = acc[l];
        __syncthreads();
        if (threadIdx.x < P::LPN) {
            V t = red[0][threadIdx.x];
            for (int w = 1; w < kWarps; ++w) t = P::combine(t, red[w][threadIdx.x]);
            a.y[row * P::LPN + threadIdx.x] = t;
        }
        __syncthreads();
    }
}

template <class P>
__device__ void emit_rows(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    switch (a.emit_group) {
        case 0: emit_ctas<P>(a, block, nblocks); break;
        case 1: emit_groups<P, 1>(a, block, nblocks); break;
        case 2: emit_groups<P, 2>(a, block, nblocks); break;
        case 4: emit_groups<P, 4>(a, block, nblocks); break;
        case 8: emit_groups<P, 8>(a, block, nblocks); break;
        case 16: emit_groups<P, 16>(a, block, nblocks); break;
        default: emit_groups<P, 32>(a, block, nblocks); break;
    }
}

// ---------------------------------------------------------------- grid barrier
// Arrival counter that only grows; barrier j of this launch completes when it
// reaches (bar_base + j + 1) * gridDim.x. A wait gives up after a.timeout
// cycles (or when another CTA already reported a timeout), sets the status
// word and returns false. The acquire at gpu scope, followed by the block
// barrier, orders every thread's later loads after the other CTAs' writes.
template <class P>
__device__ bool grid_sync(const SweepArgs<P>& a, unsigned long long j) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const bool skip = a.inject == 1 && blockIdx.x == 0 && j == 0;   // test-only
        if (!skip) {
            __threadfence();
            red_add_release(a.bar, 1ull);
        }
        const unsigned long long target = (a.bar_base + j + 1) * (unsigned long long)gridDim.x;
        const long long t0 = clock64();
        unsigned it = 0;
        while (ld_acquire(a.bar) < target) {
            if ((++it & 63u) == 0) {
                if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) {
                    ok = 0;
                    break;
                }
                if (clock64() - t0 > a.timeout) {
                    atomicCAS(a.status, 0, (int32_t)GC_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
        if (skip) ok = 0;
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ---------------------------------------------------------------- persistent sweep
template <class P>
__global__ void __launch_bounds__(kThreads, 2) sweep_kernel(const SweepArgs<P> a) {
    // an unread earlier timeout left the barrier counter part-way: do nothing
    if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) return;
    const int Lg = a.grid_levels;
    const int64_t GW = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const uint64_t keep = l2_evict_last();
    auto nchunks = [&](int k) { return (a.lvl(LV_W, k) + Chunk<P>::NODES - 1) / Chunk<P>::NODES; };
    auto norm = [&](int& k, int64_t& c) {
        while (k <= Lg && c >= nchunks(k)) {
            ++k;
            c = gw;
        }
    };

    write_leaf_tables<P>(a, (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads);

    int kn = 1;
    int64_t cn = gw;
    norm(kn, cn);
    int2 nab[kU];
    if (kn <= Lg) load_chunk<P>(a, kn, cn, nab);
    unsigned long long nbar = 0;
    for (int k = 1; k <= Lg; ++k) {
        if (k > 1 && !grid_sync(a, nbar++)) return;
        while (kn == k) {
            int2 ab[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) ab[u] = nab[u];
            const int64_t c = cn;
            cn += GW;
            norm(kn, cn);
            if (kn <= Lg) load_chunk<P>(a, kn, cn, nab);   // next chunk, maybe of a later level
            combine_chunk<P>(a, k, c, ab, keep);
        }
    }
    // narrow top levels: CTA 0 alone, block barriers only
    if (Lg < a.L) {
        if (!grid_sync(a, nbar++)) return;
        if (blockIdx.x == 0) {
            const int w0 = threadIdx.x >> 5;
            for (int k = Lg + 1; k <= a.L; ++k) {
                for (int64_t c = w0; c < nchunks(k); c += kWarps) {
                    int2 ab[kU];
                    load_chunk<P>(a, k, c, ab);
                    combine_chunk<P>(a, k, c, ab, keep);
                }
                __syncthreads();
            }
        }
    }
    if (!grid_sync(a, nbar++)) return;
    emit_rows<P>(a, blockIdx.x, gridDim.x);
}

// ---------------------------------------------------------------- per-level schedule
template <class P>
__global__ void __launch_bounds__(kThreads, 2) level_kernel(const SweepArgs<P> a, int k) {
    const int64_t GW = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const uint64_t keep = l2_evict_last();
    if (k <= 1) write_leaf_tables<P>(a, (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads);
    if (k < 1) return;
    const int64_t nc = (a.lvl(LV_W, k) + Chunk<P>::NODES - 1) / Chunk<P>::NODES;
    int2 nab[kU];
    if (gw < nc) load_chunk<P>(a, k, gw, nab);
    for (int64_t c = gw; c < nc; c += GW) {
        int2 ab[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) ab[u] = nab[u];
        if (c + GW < nc) load_chunk<P>(a, k, c + GW, nab);
        combine_chunk<P>(a, k, c, ab, keep);
    }
}

template <class P>
__global__ void __launch_bounds__(kThreads, 2) emit_kernel(const SweepArgs<P> a) {
    emit_rows<P>(a, blockIdx.x, gridDim.x);
}

// x |= y elementwise; sets *changed if any word changed (Boolean fixpoint step).
__global__ void __launch_bounds__(kThreads)
or_update_kernel(unsigned long long* __restrict__ x, const unsigned long long* __restrict__ y, int64_t n,
                 int32_t* __restrict__ changed) {
    int ch = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const unsigned long long u = x[i], v = u | y[i];
        if (v != u) {
            x[i] = v;
            ch = 1;
        }
    }
    if (__syncthreads_or(ch) && threadIdx.x == 0) *changed = 1;
}

// ---------------------------------------------------------------- host side
int grid_for(int64_t items, int per_block, int sms, int per_sm = 2) {
    int64_t g = (items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)sms * per_sm;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

template <class P>
SweepArgs<P> make_args(gc_handle* h, const void* x, void* y) {
    using V = typename P::V;
    const DevLayout& d = h->lay;
    char* ar = h->arena;
    SweepArgs<P> a{};
    a.nodes = reinterpret_cast<const int2*>(ar + d.nodes);
    a.lv = reinterpret_cast<const int64_t*>(ar + d.levels);
    a.L = (int32_t)h->L;
    a.L2 = (int32_t)h->L + 2;
    a.grid_levels = h->grid_levels;
    a.TB = d.TB;
    a.alpha = h->alpha;
    a.Vd = reinterpret_cast<const typename P::Leaf*>(ar + d.V);
    a.leaf = reinterpret_cast<const int32_t*>(ar + d.leaf);
    a.vbits = d.vbits;
    a.x = static_cast<const V*>(x);
    a.y = static_cast<V*>(y);
    a.buf0 = reinterpret_cast<V*>(ar + d.buf0);
    a.buf1 = reinterpret_cast<V*>(ar + d.buf1);
    a.rv = reinterpret_cast<V*>(ar + d.RV);
    a.c_off = reinterpret_cast<const int32_t*>(ar + d.c_off);
    a.c_ref = reinterpret_cast<const int32_t*>(ar + d.c_ref);
    a.n = h->n;
    a.emit_group = h->emit_group;
    a.status = reinterpret_cast<int32_t*>(ar + d.status);
    a.bar = reinterpret_cast<unsigned long long*>(ar + d.status + 64);
    a.bar_base = h->bar_base;
    a.timeout = h->timeout_cycles;
    a.inject = h->inject;
    return a;
}

// CTAs the persistent kernel can keep resident (at most two per SM; 0 if none)
template <class P>
int sweep_grid(const gc_handle* h) {
    int per_sm = 0;
    cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sweep_kernel<P>, kThreads, 0),
               "sweep occupancy");
    return std::min(per_sm, 2) * h->sms;
}

int64_t barriers_per_product(const gc_handle* h) {
    const int Lg = h->grid_levels;
    return std::max(Lg - 1, 0) + (Lg < h->L ? 1 : 0) + 1;
}

// Enqueues one product with the arguments in a (persistent kernel when the
// device allows, else one kernel per level). Returns the launch count.
template <class P>
int64_t launch_product(const gc_handle* h, SweepArgs<P>& a, cudaStream_t st) {
    int grid = 0;
    if (h->schedule == 0 && h->coop) grid = sweep_grid<P>(h);
    int64_t launches = 0;
    if (grid > 0) {
        void* args[] = {&a};
        cuda_check(cudaLaunchCooperativeKernel((const void*)sweep_kernel<P>, dim3(grid), dim3(kThreads), args, 0, st),
                   "sweep launch");
        launches = 1;
    } else {
        a.grid_levels = (int32_t)h->L;
        // level 1 also writes the leaf tables; with no levels a table-only launch
        const int64_t w1 = h->L >= 1 ? h->lv[LV_W * (h->L + 2) + 1] : 0;
        const int64_t items = std::max<int64_t>(w1, (h->alpha + 1) * P::LPN);
        level_kernel<P><<<grid_for(items, Chunk<P>::NODES * kWarps, h->sms), kThreads, 0, st>>>(a, h->L >= 1 ? 1 : 0);
        ++launches;
        for (int k = 2; k <= h->L; ++k) {
            const int64_t w = h->lv[LV_W * (h->L + 2) + k];
            level_kernel<P><<<grid_for(w, Chunk<P>::NODES * kWarps, h->sms), kThreads, 0, st>>>(a, k);
            ++launches;
        }
        if (h->n > 0) {
            const int64_t rows_per_block = h->emit_group == 0 ? 1 : kWarps * (32 / h->emit_group);
            emit_kernel<P><<<grid_for(h->n, (int)rows_per_block, h->sms, 4), kThreads, 0, st>>>(a);
            ++launches;
        }
    }
    cuda_check(cudaGetLastError(), "kernel launch");
    return launches;
}

template <class P>
void run_product(gc_handle* h, const void* x, void* y, cudaStream_t st) {
    SweepArgs<P> a = make_args<P>(h, x, y);
    const bool persistent = h->schedule == 0 && h->coop;
    const int64_t launches = launch_product<P>(h, a, st);
    if (persistent && launches == 1) h->bar_base += (unsigned long long)barriers_per_product(h);
    h->launches = launches;
}

void dispatch_product(gc_handle* h, const void* x, void* y, int32_t k, cudaStream_t st) {
    switch (h->policy) {
        case GC_F32_SUM:
            if (k == 1) run_product<PolF32>(h, x, y, st);
            else run_product<PolF32x16>(h, x, y, st);
            break;
        case GC_I64_SUM: run_product<PolI64>(h, x, y, st); break;
        case GC_BOOL_OR: run_product<PolOr>(h, x, y, st); break;
    }
}

void check_k(const gc_handle* h, int32_t k) {
    if (h->policy == GC_F32_SUM) {
        if (k != 1 && k != 16) fail(GC_ERR_ARG, "k must be 1 or 16");
        if (k > h->k_max) fail(GC_ERR_ARG, "k exceeds the k_max the handle was uploaded with");
    } else if (k != 1) {
        fail(GC_ERR_ARG, "k must be 1 for this policy");
    }
}

template <class T>
void put(cudaStream_t st, char* arena, int64_t off, const T* p, size_t count) {
    if (count == 0) return;
    cuda_check(cudaMemcpyAsync(arena + off, p, count * sizeof(T), cudaMemcpyHostToDevice, st), "upload copy");
}

// ---------------------------------------------------------------- fixed scratch
// Scratch for gc_matvec_static: callers that cannot allocate device memory at
// the point of the call still get a product. Every GPU that loads the library
// holds this array until the process exits; every call shares it.
constexpr int64_t kStaticScratchBytes = GC_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch per device, looked up once with that
// device current (the host-side name is only a stand-in for it).
constexpr int kMaxDevices = 64;
static unsigned char* g_static_ptr[kMaxDevices] = {};
static std::mutex g_static_mu;

unsigned char* static_scratch_on_current_device() {
    int dev = 0;
    cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) fail(GC_ERR_UNSUPPORTED, "device index beyond the fixed-scratch table");
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        cuda_check(cudaGetSymbolAddress(&p, g_static_scratch), "cudaGetSymbolAddress(fixed scratch)");
        g_static_ptr[dev] = static_cast<unsigned char*>(p);
    }
    return g_static_ptr[dev];
}

// Bytes of fixed scratch a product with k right-hand sides needs: status
// block, [T | root values], two [T | level] buffers (the arena's scratch parts).
int64_t static_scratch_need(const gc_handle* h, int32_t k) {
    const int64_t vb = policy_elem_bytes(h->policy) * k;
    const int64_t TB = h->lay.TB;
    return 256 + align256(vb * (TB + h->n_roots)) + 2 * align256(vb * (TB + h->max_width));
}

// One product whose scratch is the fixed array: the same kernels and order of
// evaluation as gc_matvec, with RV, the level buffers, the status word and
// the barrier counter pointed into g_static_scratch.
template <class P>
void run_product_static(gc_handle* h, const void* x, void* y, cudaStream_t st, unsigned char* scratch) {
    using V = typename P::V;
    SweepArgs<P> a = make_args<P>(h, x, y);
    const int64_t vb = (int64_t)sizeof(V) * P::LPN;
    const int64_t rv_bytes = align256(vb * (a.TB + h->n_roots)), buf_bytes = align256(vb * (a.TB + h->max_width));
    a.status = reinterpret_cast<int32_t*>(scratch);
    a.bar = reinterpret_cast<unsigned long long*>(scratch + 64);
    a.bar_base = 0;
    a.rv = reinterpret_cast<V*>(scratch + 256);
    a.buf0 = reinterpret_cast<V*>(scratch + 256 + rv_bytes);
    a.buf1 = reinterpret_cast<V*>(scratch + 256 + rv_bytes + buf_bytes);
    a.inject = 0;
    // the array keeps the previous call's contents: start from a clear status
    // word and barrier counter
    cuda_check(cudaMemsetAsync(scratch, 0, 256, st), "fixed scratch clear");
    h->launches = launch_product<P>(h, a, st);
}

}  // namespace
}  // namespace gcs

using namespace gcs;

extern "C" {

gc_status gc_upload(const gc_grammar* gg, gc_policy policy, int32_t k_max, void* arena, int64_t arena_bytes,
                    void* stream, gc_handle** out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null grammar or output pointer");
        if (!arena) fail(GC_ERR_ARG, "null arena");
        if (reinterpret_cast<uintptr_t>(arena) % 256 != 0) fail(GC_ERR_ARG, "arena must be 256-byte aligned");
        const Grammar& g = gg->g;
        check_policy(g, policy, k_max);
        validate_packed(g);
        const DevLayout d = device_layout(g, policy, k_max);
        if (arena_bytes < d.total) fail(GC_ERR_ARG, "arena smaller than gc_layout().arena_bytes");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        auto h = std::make_unique<gc_handle>();
        h->policy = policy;
        h->k_max = k_max;
        h->n = g.n;
        h->m = g.m;
        h->L = g.L;
        h->alpha = g.alpha();
        h->n_roots = g.n_roots;
        h->c_len = (int64_t)g.c_ref.size();
        h->max_width = g.max_width();
        h->arena = static_cast<char*>(arena);
        h->lay = d;
        int dev = 0;
        cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
        cuda_check(cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
        cuda_check(cudaDeviceGetAttribute(&h->coop, cudaDevAttrCooperativeLaunch, dev), "cooperative attribute");
        // emit group: about one symbol per thread per pass, capped at a CTA
        const double avg = g.n > 0 ? (double)h->c_len / (double)g.n : 0.0;
        if (avg >= 128) {
            h->emit_group = 0;
        } else {
            int G = 1;
            while (G < 32 && G < avg) G <<= 1;
            h->emit_group = G;
        }
        // levels narrow enough for one CTA finish the sweep there (when two or more)
        const int64_t L = g.L;
        const int64_t tail_w = (policy == GC_F32_SUM && k_max == 16) ? Chunk<PolF32x16>::TAIL : Chunk<PolF32>::TAIL;
        int64_t first_narrow = L + 1;
        while (first_narrow > 1 && g.lvl_off[first_narrow] - g.lvl_off[first_narrow - 1] <= tail_w) --first_narrow;
        h->grid_levels = (int)(L - first_narrow + 1 >= 2 ? first_narrow - 1 : L);

        // level table; level 1 with leaf codes, later levels with indices into [T | buffer]
        auto leaf_code = [&](int32_t p) { return (int32_t)(((int64_t)g.term_col[p] << d.vbits) | g.term_vidx[p]); };
        auto ref = [&](int32_t c) -> int32_t {   // packed reference -> [T | buffer] index
            if (c >= 0) return (int32_t)(d.TB + c);
            if (c == -1) return 0;
            return -c - 1;                         // terminal p = -c-2 -> T[p+1]
        };
        h->lv.assign((size_t)(4 * (L + 2)), 0);
        std::vector<int32_t> nodes((size_t)(2 * d.n_nodes_padded), 0);
        int64_t start = 0;
        for (int64_t k = 1; k <= L; ++k) {
            const int64_t w = g.lvl_off[k + 1] - g.lvl_off[k];
            h->lv[LV_START * (L + 2) + k] = start;
            h->lv[LV_W * (L + 2) + k] = w;
            h->lv[LV_ROOTS * (L + 2) + k] = g.lvl_roots[k];
            h->lv[LV_ROFF * (L + 2) + k] = g.root_off[k];
            for (int64_t q = 0; q < w; ++q)
                for (int t = 0; t < 2; ++t) {
                    const int32_t c = g.nodes[2 * (g.lvl_off[k] + q) + t];
                    if (k == 1 && c > -2) fail(GC_ERR_INVALID_GRAMMAR, "a level-1 node has a non-terminal child");
                    nodes[2 * (start + q) + t] = k == 1 ? leaf_code(-c - 2) : ref(c);
                }
            start += pad_nodes(w);
        }
        std::vector<int32_t> leaf((size_t)g.alpha());
        for (int64_t p = 0; p < g.alpha(); ++p) leaf[p] = leaf_code((int32_t)p);
        std::vector<int32_t> cref(g.c_ref.size());
        for (size_t e = 0; e < cref.size(); ++e) cref[e] = ref(g.c_ref[e]);
        std::vector<int32_t> co(g.slp.c_off.size());
        for (size_t r = 0; r < co.size(); ++r) co[r] = (int32_t)g.slp.c_off[r];

        char* a = h->arena;
        put(st, a, d.nodes, nodes.data(), nodes.size());
        put(st, a, d.levels, h->lv.data(), h->lv.size());
        if (policy == GC_F32_SUM) {
            put(st, a, d.V, g.V.data(), g.V.size());
        } else {
            std::vector<long long> v(g.V.size());
            for (size_t i = 0; i < v.size(); ++i) v[i] = policy == GC_BOOL_OR ? ~0ll : (long long)g.V[i];
            put(st, a, d.V, v.data(), v.size());
        }
        put(st, a, d.leaf, leaf.data(), leaf.size());
        put(st, a, d.c_off, co.data(), co.size());
        put(st, a, d.c_ref, cref.data(), cref.size());
        cuda_check(cudaMemsetAsync(a + d.status, 0, 256, st), "status clear");
        cuda_check(cudaStreamSynchronize(st), "upload synchronize");
        *out = h.release();
    });
}

gc_status gc_matvec(gc_handle* h, const void* x, void* y, int32_t k, void* stream) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if ((!x && h->m > 0) || (!y && h->n > 0)) fail(GC_ERR_ARG, "null x or y");
        check_k(h, k);
        dispatch_product(h, x, y, k, static_cast<cudaStream_t>(stream));
    });
}

gc_status gc_matvec_host(gc_handle* h, const void* x_host, void* y_host, int32_t k, void* stream) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if ((!x_host && h->m > 0) || (!y_host && h->n > 0)) fail(GC_ERR_ARG, "null x or y");
        check_k(h, k);
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        const int64_t eb = policy_elem_bytes(h->policy) * k;
        char* xs = h->arena + h->lay.xs;
        char* ys = h->arena + h->lay.ys;
        if (h->m > 0) cuda_check(cudaMemcpyAsync(xs, x_host, h->m * eb, cudaMemcpyHostToDevice, st), "x upload");
        dispatch_product(h, xs, ys, k, st);
        if (h->n > 0) cuda_check(cudaMemcpyAsync(y_host, ys, h->n * eb, cudaMemcpyDeviceToHost, st), "y download");
        cuda_check(cudaStreamSynchronize(st), "stream synchronize");
    });
}

gc_status gc_reach(gc_handle* h, const uint64_t* x0, uint64_t* x, int32_t max_iter, int32_t* iters,
                   void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h || !x0 || !x || !iters) fail(GC_ERR_ARG, "null argument");
        if (h->policy != GC_BOOL_OR) fail(GC_ERR_ARG, "gc_reach needs the GC_BOOL_OR policy");
        if (h->n != h->m) fail(GC_ERR_ARG, "gc_reach needs a square matrix");
        if (max_iter < 1) fail(GC_ERR_ARG, "max_iter must be >= 1");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        const int64_t n = h->n;
        unsigned long long* xv = reinterpret_cast<unsigned long long*>(x);
        unsigned long long* yv = reinterpret_cast<unsigned long long*>(h->arena + h->lay.ys);
        int32_t* status = reinterpret_cast<int32_t*>(h->arena + h->lay.status);
        int32_t* changed = status + 1;
        if (x != x0 && n > 0)
            cuda_check(cudaMemcpyAsync(x, x0, n * 8, cudaMemcpyDeviceToDevice, st), "x0 copy");
        int32_t it = 0, done = 0;
        int64_t launches = 0;
        while (it < max_iter) {
            ++it;
            cuda_check(cudaMemsetAsync(changed, 0, 4, st), "flag clear");
            dispatch_product(h, xv, yv, 1, st);
            launches += h->launches;
            if (n > 0) {
                or_update_kernel<<<grid_for(n, kThreads, h->sms, 8), kThreads, 0, st>>>(xv, yv, n, changed);
                ++launches;
            }
            cuda_check(cudaGetLastError(), "kernel launch");
            int32_t c = 0;
            cuda_check(cudaMemcpyAsync(&c, changed, 4, cudaMemcpyDeviceToHost, st), "flag read");
            cuda_check(cudaStreamSynchronize(st), "stream synchronize");
            if (!c) {
                done = 1;
                break;
            }
        }
        h->launches = launches;
        int32_t result = done ? it : -1;
        cuda_check(cudaMemcpyAsync(iters, &result, 4, cudaMemcpyHostToDevice, st), "iters write");
        if (!done) {
            int32_t s = GC_ERR_NOT_CONVERGED;
            cuda_check(cudaMemcpyAsync(status, &s, 4, cudaMemcpyHostToDevice, st), "status write");
            rc = GC_ERR_NOT_CONVERGED;
        }
        cuda_check(cudaStreamSynchronize(st), "stream synchronize");
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_reach: max_iter reached before the fixpoint");
    return rc;
}

gc_status gc_check(gc_handle* h, void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int32_t* status = reinterpret_cast<int32_t*>(h->arena + h->lay.status);
        int32_t s = 0;
        cuda_check(cudaMemcpyAsync(&s, status, 4, cudaMemcpyDeviceToHost, st), "status read");
        cuda_check(cudaStreamSynchronize(st), "stream synchronize");
        if (s != 0) {
            // a failed launch leaves the barrier counter part-way: restart it
            cuda_check(cudaMemsetAsync(h->arena + h->lay.status, 0, 256, st), "status clear");
            cuda_check(cudaStreamSynchronize(st), "stream synchronize");
            h->bar_base = 0;
        }
        rc = (gc_status)s;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("device status word reported an error");
    return rc;
}

gc_status gc_launch_count(const gc_handle* h, int64_t* launches) {
    return guard([&] {
        if (!h || !launches) fail(GC_ERR_ARG, "null argument");
        *launches = h->launches;
    });
}

gc_status gc_set_schedule(gc_handle* h, int32_t schedule) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if (schedule != GC_SCHED_PERSISTENT && schedule != GC_SCHED_PER_LEVEL) fail(GC_ERR_ARG, "unknown schedule");
        h->schedule = schedule;
    });
}

gc_status gc_get_schedule(const gc_handle* h, int32_t* schedule) {
    return guard([&] {
        if (!h || !schedule) fail(GC_ERR_ARG, "null argument");
        *schedule = (h->schedule == GC_SCHED_PERSISTENT && h->coop) ? GC_SCHED_PERSISTENT : GC_SCHED_PER_LEVEL;
    });
}

gc_status gc_debug_inject(gc_handle* h, int32_t what, int64_t timeout_cycles) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if (what != 0 && what != 1) fail(GC_ERR_ARG, "unknown injection");
        if (timeout_cycles <= 0) fail(GC_ERR_ARG, "timeout must be positive");
        h->inject = what;
        h->timeout_cycles = timeout_cycles;
    });
}

gc_status gc_matvec_static(gc_handle* h, const void* x, void* y, int32_t k, void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if ((!x && h->m > 0) || (!y && h->n > 0)) fail(GC_ERR_ARG, "null x or y");
        check_k(h, k);
        const int64_t need = static_scratch_need(h, k);
        if (need > kStaticScratchBytes)
            fail(GC_ERR_UNSUPPORTED, "gc_matvec_static: this grammar needs " + std::to_string(need) +
                                         " bytes of scratch; the fixed array holds " +
                                         std::to_string(kStaticScratchBytes));
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        unsigned char* scratch = static_scratch_on_current_device();
        switch (h->policy) {
            case GC_F32_SUM:
                if (k == 1) run_product_static<PolF32>(h, x, y, st, scratch);
                else run_product_static<PolF32x16>(h, x, y, st, scratch);
                break;
            case GC_I64_SUM: run_product_static<PolI64>(h, x, y, st, scratch); break;
            case GC_BOOL_OR: run_product_static<PolOr>(h, x, y, st, scratch); break;
        }
        int32_t s = 0;
        cuda_check(cudaMemcpyAsync(&s, scratch, 4, cudaMemcpyDeviceToHost, st), "fixed scratch status read");
        cuda_check(cudaStreamSynchronize(st), "stream synchronize");
        rc = (gc_status)s;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_matvec_static: a device-side wait ran out");
    return rc;
}

void gc_free_handle(gc_handle* h) { delete h; }

}  // extern "C"
