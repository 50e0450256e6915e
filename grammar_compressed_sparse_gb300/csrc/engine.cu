// Device side of gcsparse: upload of the packed grammar into a caller-owned
// arena, and the streaming bottom-up sweep of Sec. 4.3 of the pages ("Right
// Multiplication on Grammar-Compressed Matrices"), written for sm_103a.
//
//   level combine   for k = 1..L: cur[t] = cv(a_t) (+) cv(b_t), where
//                   cv(c) = prev[c] for c >= 0, the identity for c = -1, and
//                   the leaf V[l] (x) x[j] for a terminal <l, j>; the level's
//                   roots (its first nodes) are also written to RV, the
//                   emit-on-the-spot capture (Listing 1, Lemma 3.3)
//   row emit        y[r] = (+) over row r's symbols of RV[c] or the leaf value
//                   (Lemma 2.2; a row of C may hold several symbols and bare
//                   terminals)
//
// Differences from the pages' design, for this GPU:
//   * one persistent cooperative kernel per product instead of two launches
//     per level; levels are separated by a grid barrier whose waits are
//     bounded (a wait that runs out sets the status word and the kernel
//     returns);
//   * each CTA streams its tiles of child pairs from HBM into shared memory
//     with cp.async.bulk (an mbarrier-tracked, three-stage pipeline with an
//     L2 evict-first hint) and keeps issuing across level barriers, since the
//     pairs do not depend on values; the child values are gathered from the
//     L2-resident level buffers, eight nodes per thread with all loads issued
//     first;
//   * leaves are evaluated where they are read (the pages' own future-work
//     item, Sec. 7 item 3), so there is no terminal array and no leaf phase;
//   * the narrow top levels run on one CTA with block-level barriers;
//   * the pages emit with atomicAdd into y; here each row is reduced by a
//     fixed group of threads in a fixed order: deterministic, no atomics.
// A second schedule launches one kernel per level plus one emit kernel; it
// computes every value with the same device functions (bit-identical y) and
// serves as the reference point for the persistent one.
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
    int64_t n = 0, m = 0, L = 0, n_roots = 0, c_len = 0, max_width = 0;
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

constexpr int kSweepThreads = 512;   // persistent kernel: one CTA of 512 per SM
constexpr int kLevelThreads = 256;   // per-level schedule
constexpr int kStages = 3;
constexpr int kNodesPerThread = 8;
constexpr int LV_START = 0, LV_W = 1, LV_ROOTS = 2, LV_ROFF = 3;

void cuda_check(cudaError_t e, const char* what) {
    if (e != cudaSuccess) fail(GC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

template <class P>
struct Tile {
    static constexpr int NODES = kSweepThreads * kNodesPerThread / P::LPN;   // nodes per bulk copy
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// global -> shared bulk copy (16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void atom_add_release(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_volatile(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }

// L2-only loads / stores for values written during the kernel (L1 is not
// coherent across SMs)
__device__ __forceinline__ float ldv(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ldv(const float4* p) { return __ldcg(p); }
__device__ __forceinline__ long long ldv(const long long* p) { return __ldcg(p); }
__device__ __forceinline__ unsigned long long ldv(const unsigned long long* p) { return __ldcg(p); }
__device__ __forceinline__ void stv(float* p, float v) { __stcg(p, v); }
__device__ __forceinline__ void stv(float4* p, float4 v) { __stcg(p, v); }
__device__ __forceinline__ void stv(long long* p, long long v) { __stcg(p, v); }
__device__ __forceinline__ void stv(unsigned long long* p, unsigned long long v) { __stcg(p, v); }

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
    const typename P::Leaf* Vd;
    int32_t vbits;
    const V* x;
    V* y;
    V* buf0;
    V* buf1;
    V* rv;
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

// value of child reference c (lane `lane` of the node value)
template <class P>
__device__ __forceinline__ typename P::V child(int32_t c, int lane, const typename P::V* prev,
                                               const SweepArgs<P>& a) {
    if (c >= 0) return ldv(prev + (int64_t)c * P::LPN + lane);
    if (c == -1) return P::identity();
    const uint32_t q = (uint32_t)(-(c + 2));
    const uint32_t col = q >> a.vbits, vi = q & ((1u << a.vbits) - 1u);
    return P::leaf(__ldg(a.Vd + vi), __ldg(a.x + (int64_t)col * P::LPN + lane));
}

// Combine cnt nodes (pairs at src, from shared memory or, with kGlobal,
// streamed from global) into cur[base ..], capturing roots into rv.
template <class P, int NT, bool kGlobal>
__device__ __forceinline__ void combine_block(const int2* src, int32_t cnt, int64_t base, int64_t nroots,
                                              const typename P::V* prev, typename P::V* cur, typename P::V* rv,
                                              const SweepArgs<P>& a) {
    using V = typename P::V;
    constexpr int NPP = NT / P::LPN;
    constexpr int U = kNodesPerThread;
    const int lane = threadIdx.x % P::LPN;
    const int sub = threadIdx.x / P::LPN;
    int2 ab[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int i = u * NPP + sub;
        ab[u] = i < cnt ? (kGlobal ? __ldcs(src + i) : src[i]) : make_int2(-1, -1);
    }
    V va[U], vb[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        va[u] = child<P>(ab[u].x, lane, prev, a);
        vb[u] = child<P>(ab[u].y, lane, prev, a);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int i = u * NPP + sub;
        if (i < cnt) {
            const V v = P::combine(va[u], vb[u]);
            const int64_t g = base + i;
            stv(cur + g * P::LPN + lane, v);
            if (g < nroots) stv(rv + g * P::LPN + lane, v);
        }
    }
}

// ---------------------------------------------------------------- row emit
template <class P>
__device__ __forceinline__ typename P::V emit_value(int32_t c, int lane, const SweepArgs<P>& a) {
    if (c >= 0) return ldv(a.rv + (int64_t)c * P::LPN + lane);
    return child<P>(c, lane, nullptr, a);   // leaf (or identity for -1)
}

constexpr int kEmitBatch = 4;

// G threads per row (G divides 32); warps walk rows in lockstep so the
// shuffles always see the full warp. Thread gl sums its symbols q = s+gl,
// s+gl+G, ... in order, then the group reduces by a fixed butterfly.
template <class P, int NT, int G>
__device__ void emit_groups(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    using V = typename P::V;
    constexpr int RPW = 32 / G;
    const int lane = threadIdx.x & 31;
    const int gl = lane % G;
    const int64_t warp = block * (NT / 32) + (threadIdx.x >> 5);
    const int64_t nwarps = nblocks * (NT / 32);
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
                for (int u = 0; u < kEmitBatch; ++u) c[u] = q0 + u * G < e ? __ldcs(a.c_ref + q0 + u * G) : -1;
                V v[kEmitBatch][P::LPN];
#pragma unroll
                for (int u = 0; u < kEmitBatch; ++u)
#pragma unroll
                    for (int l = 0; l < P::LPN; ++l) v[u][l] = emit_value<P>(c[u], l, a);
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
template <class P, int NT>
__device__ void emit_ctas(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    using V = typename P::V;
    __shared__ V red[NT / 32][P::LPN];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t row = block; row < a.n; row += nblocks) {
        V acc[P::LPN];
#pragma unroll
        for (int l = 0; l < P::LPN; ++l) acc[l] = P::identity();
        const int32_t s = __ldg(a.c_off + row), e = __ldg(a.c_off + row + 1);
        for (int32_t q0 = s + threadIdx.x; q0 < e; q0 += NT * kEmitBatch) {
            int32_t c[kEmitBatch];
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u) c[u] = q0 + u * NT < e ? __ldcs(a.c_ref + q0 + u * NT) : -1;
            V v[kEmitBatch][P::LPN];
#pragma unroll
            for (int u = 0; u < kEmitBatch; ++u)
#pragma unroll
                for (int l = 0; l < P::LPN; ++l) v[u][l] = emit_value<P>(c[u], l, a);
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
            for (int w = 1; w < NT / 32; ++w) t = P::combine(t, red[w][threadIdx.x]);
            a.y[row * P::LPN + threadIdx.x] = t;
        }
        __syncthreads();
    }
}

template <class P, int NT>
__device__ void emit_rows(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    switch (a.emit_group) {
        case 0: emit_ctas<P, NT>(a, block, nblocks); break;
        case 1: emit_groups<P, NT, 1>(a, block, nblocks); break;
        case 2: emit_groups<P, NT, 2>(a, block, nblocks); break;
        case 4: emit_groups<P, NT, 4>(a, block, nblocks); break;
        case 8: emit_groups<P, NT, 8>(a, block, nblocks); break;
        case 16: emit_groups<P, NT, 16>(a, block, nblocks); break;
        default: emit_groups<P, NT, 32>(a, block, nblocks); break;
    }
}

// ---------------------------------------------------------------- waits
// Grid barrier: arrival counter that only grows; barrier j of this launch
// completes when it reaches (bar_base + j + 1) * gridDim.x. A wait gives up
// after a.timeout cycles (or when another CTA already reported a failure),
// sets the status word and returns false.
template <class P>
__device__ bool grid_sync(const SweepArgs<P>& a, unsigned long long j) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const bool skip = a.inject == 1 && blockIdx.x == 0 && j == 0;   // test-only
        if (!skip) {
            __threadfence();
            atom_add_release(a.bar, 1ull);
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

// Bounded wait for a bulk copy to land; false (status set) if it does not.
template <class P>
__device__ bool stage_wait(const SweepArgs<P>& a, uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > a.timeout) {
            atomicCAS(a.status, 0, (int32_t)GC_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------- persistent sweep
template <class P>
__global__ void __launch_bounds__(kSweepThreads, 1) sweep_kernel(const SweepArgs<P> a) {
    using V = typename P::V;
    constexpr int TILE = Tile<P>::NODES;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    int2* stage = reinterpret_cast<int2*>(smem_raw);
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ int s_ok;

    // an unread earlier timeout left the barrier counter part-way: do nothing
    if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) return;
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int Lg = a.grid_levels;
    auto ntiles = [&](int k) { return (a.lvl(LV_W, k) + TILE - 1) / TILE; };
    // (level, tile) iterators over this CTA's tiles b, b+G, ... of levels 1..Lg
    auto norm = [&](int& k, int64_t& t) {
        while (k <= Lg && t >= ntiles(k)) {
            ++k;
            t = b;
        }
    };
    const uint64_t pol = l2_evict_first();
    auto issue = [&](int k, int64_t t, int s) {
        const int64_t node0 = t * TILE;
        const int64_t cnt = min((int64_t)TILE, a.lvl(LV_W, k) - node0);
        const uint32_t bytes = (uint32_t)(((cnt + kNodeAlign - 1) / kNodeAlign) * kNodeAlign * 8);
        mbar_expect_tx(&bars[s], bytes);
        bulk_g2s(stage + (int64_t)s * TILE, a.nodes + a.lvl(LV_START, k) + node0, bytes, &bars[s], pol);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    int pk = 1, ck = 1;
    int64_t pt = b, ct = b;
    norm(pk, pt);
    norm(ck, ct);
    int inflight = 0;   // meaningful in thread 0
    if (threadIdx.x == 0)
        for (int s = 0; s < kStages && pk <= Lg; ++s) {
            issue(pk, pt, s);
            ++inflight;
            pt += G;
            norm(pk, pt);
        }
    uint32_t parity = 0;
    int slot = 0;
    unsigned long long nbar = 0;
    bool ok = true;

    for (int k = 1; k <= Lg && ok; ++k) {
        if (k > 1 && !(ok = grid_sync(a, nbar++))) break;
        const V* prev = (k & 1) ? a.buf0 : a.buf1;
        V* cur = (k & 1) ? a.buf1 : a.buf0;
        const int64_t w = a.lvl(LV_W, k), nroots = a.lvl(LV_ROOTS, k);
        V* rv = a.rv + a.lvl(LV_ROFF, k) * P::LPN;
        while (ck == k) {
            const int got = stage_wait(a, &bars[slot], (parity >> slot) & 1u);
            if (!__syncthreads_and(got)) {
                ok = false;
                break;
            }
            parity ^= 1u << slot;
            const int64_t node0 = ct * TILE;
            combine_block<P, kSweepThreads, false>(stage + (int64_t)slot * TILE, (int32_t)min((int64_t)TILE, w - node0),
                                                   node0, nroots, prev, cur, rv, a);
            __syncthreads();   // every thread is done with this stage
            if (threadIdx.x == 0) {
                --inflight;
                if (pk <= Lg) {
                    issue(pk, pt, slot);
                    ++inflight;
                    pt += G;
                    norm(pk, pt);
                }
            }
            ct += G;
            norm(ck, ct);
            slot = slot + 1 == kStages ? 0 : slot + 1;
        }
    }

    if (!ok) {
        // leave no bulk copy writing into shared memory after the CTA exits
        if (threadIdx.x == 0) {
            for (int i = 0, s = slot; i < inflight; ++i, s = s + 1 == kStages ? 0 : s + 1) {
                const long long t0 = clock64();
                while (!mbar_try_wait(&bars[s], (parity >> s) & 1u) && clock64() - t0 < a.timeout) {
                }
                parity ^= 1u << s;
            }
        }
        __syncthreads();
        return;
    }

    // narrow top levels: CTA 0 alone, block barriers only
    if (Lg < a.L) {
        if (!grid_sync(a, nbar++)) return;
        if (b == 0) {
            constexpr int CH = kSweepThreads * kNodesPerThread / P::LPN;
            for (int k = Lg + 1; k <= a.L; ++k) {
                const V* prev = (k & 1) ? a.buf0 : a.buf1;
                V* cur = (k & 1) ? a.buf1 : a.buf0;
                const int64_t w = a.lvl(LV_W, k), nroots = a.lvl(LV_ROOTS, k);
                const int2* src = a.nodes + a.lvl(LV_START, k);
                V* rv = a.rv + a.lvl(LV_ROFF, k) * P::LPN;
                for (int64_t c0 = 0; c0 < w; c0 += CH)
                    combine_block<P, kSweepThreads, true>(src + c0, (int32_t)min((int64_t)CH, w - c0), c0, nroots,
                                                          prev, cur, rv, a);
                __syncthreads();
            }
        }
    }
    if (!grid_sync(a, nbar++)) return;
    emit_rows<P, kSweepThreads>(a, b, G);
    (void)s_ok;
}

// ---------------------------------------------------------------- per-level schedule
template <class P>
__global__ void __launch_bounds__(kLevelThreads) level_kernel(const SweepArgs<P> a, int k) {
    constexpr int CH = kLevelThreads * kNodesPerThread / P::LPN;
    const typename P::V* prev = (k & 1) ? a.buf0 : a.buf1;
    typename P::V* cur = (k & 1) ? a.buf1 : a.buf0;
    const int64_t w = a.lvl(LV_W, k), nroots = a.lvl(LV_ROOTS, k);
    const int2* src = a.nodes + a.lvl(LV_START, k);
    typename P::V* rv = a.rv + a.lvl(LV_ROFF, k) * P::LPN;
    for (int64_t c0 = (int64_t)blockIdx.x * CH; c0 < w; c0 += (int64_t)gridDim.x * CH)
        combine_block<P, kLevelThreads, true>(src + c0, (int32_t)min((int64_t)CH, w - c0), c0, nroots, prev, cur, rv,
                                              a);
}

// Same block size as the persistent kernel, so both schedules reduce every
// row in the same order.
template <class P>
__global__ void __launch_bounds__(kSweepThreads) emit_kernel(const SweepArgs<P> a) {
    emit_rows<P, kSweepThreads>(a, blockIdx.x, gridDim.x);
}

// x |= y elementwise; sets *changed if any word changed (Boolean fixpoint step).
__global__ void __launch_bounds__(kLevelThreads)
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
int grid_for(int64_t items, int threads, int sms, int per_sm = 8) {
    int64_t g = (items + threads - 1) / threads;
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
    a.Vd = reinterpret_cast<const typename P::Leaf*>(ar + d.V);
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

template <class P>
int sweep_grid(const gc_handle* h) {
    const size_t smem = (size_t)kStages * Tile<P>::NODES * sizeof(int2);
    cuda_check(cudaFuncSetAttribute(sweep_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
               "sweep smem attribute");
    int per_sm = 0;
    cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sweep_kernel<P>, kSweepThreads, smem),
               "sweep occupancy");
    return per_sm >= 1 ? h->sms : 0;   // one CTA per SM
}

template <class P>
void run_product(gc_handle* h, const void* x, void* y, cudaStream_t st) {
    SweepArgs<P> a = make_args<P>(h, x, y);
    int64_t launches = 0;
    int grid = 0;
    if (h->schedule == 0 && h->coop) grid = sweep_grid<P>(h);
    if (grid > 0) {
        const size_t smem = (size_t)kStages * Tile<P>::NODES * sizeof(int2);
        void* args[] = {&a};
        cuda_check(cudaLaunchCooperativeKernel((const void*)sweep_kernel<P>, dim3(grid), dim3(kSweepThreads), args,
                                               smem, st),
                   "sweep launch");
        const int Lg = h->grid_levels;
        h->bar_base += (unsigned long long)(std::max(Lg - 1, 0) + (Lg < h->L ? 1 : 0) + 1);
        launches = 1;
    } else {
        a.grid_levels = (int32_t)h->L;
        for (int k = 1; k <= h->L; ++k) {
            const int64_t w = h->lv[LV_W * (h->L + 2) + k];
            if (w == 0) continue;
            level_kernel<P><<<grid_for(w * P::LPN, kLevelThreads * kNodesPerThread, h->sms), kLevelThreads, 0, st>>>(
                a, k);
            ++launches;
        }
        if (h->n > 0) {
            const int64_t rows_per_block = h->emit_group == 0 ? 1 : (kSweepThreads / 32) * (32 / h->emit_group);
            emit_kernel<P><<<grid_for(h->n, (int)rows_per_block, h->sms, 8), kSweepThreads, 0, st>>>(a);
            ++launches;
        }
    }
    cuda_check(cudaGetLastError(), "kernel launch");
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
// block, root values, two level buffers (same parts as the arena's scratch).
int64_t static_scratch_need(const gc_handle* h, int32_t k) {
    const int64_t vb = policy_elem_bytes(h->policy) * k;
    return 256 + align256(vb * h->n_roots) + 2 * align256(vb * h->max_width);
}

// One product whose scratch is the fixed array: the same kernels and order of
// evaluation as run_product, with RV, the level buffers, the status word and
// the barrier counter pointed into g_static_scratch.
template <class P>
void run_product_static(gc_handle* h, const void* x, void* y, cudaStream_t st, unsigned char* scratch) {
    using V = typename P::V;
    SweepArgs<P> a = make_args<P>(h, x, y);
    const int64_t vb = (int64_t)sizeof(V) * P::LPN;
    a.status = reinterpret_cast<int32_t*>(scratch);
    a.bar = reinterpret_cast<unsigned long long*>(scratch + 64);
    a.bar_base = 0;
    a.rv = reinterpret_cast<V*>(scratch + 256);
    a.buf0 = reinterpret_cast<V*>(scratch + 256 + align256(vb * h->n_roots));
    a.buf1 = reinterpret_cast<V*>(scratch + 256 + align256(vb * h->n_roots) + align256(vb * h->max_width));
    a.inject = 0;
    // the array keeps the previous call's contents: start from a clear status
    // word and barrier counter
    cuda_check(cudaMemsetAsync(scratch, 0, 256, st), "fixed scratch clear");
    int64_t launches = 0;
    int grid = 0;
    if (h->schedule == 0 && h->coop) grid = sweep_grid<P>(h);
    if (grid > 0) {
        const size_t smem = (size_t)kStages * Tile<P>::NODES * sizeof(int2);
        void* args[] = {&a};
        cuda_check(cudaLaunchCooperativeKernel((const void*)sweep_kernel<P>, dim3(grid), dim3(kSweepThreads), args,
                                               smem, st),
                   "sweep launch");
        launches = 1;
    } else {
        a.grid_levels = (int32_t)h->L;
        for (int k = 1; k <= h->L; ++k) {
            const int64_t w = h->lv[LV_W * (h->L + 2) + k];
            if (w == 0) continue;
            level_kernel<P><<<grid_for(w * P::LPN, kLevelThreads * kNodesPerThread, h->sms), kLevelThreads, 0, st>>>(
                a, k);
            ++launches;
        }
        if (h->n > 0) {
            const int64_t rows_per_block = h->emit_group == 0 ? 1 : (kSweepThreads / 32) * (32 / h->emit_group);
            emit_kernel<P><<<grid_for(h->n, (int)rows_per_block, h->sms, 8), kSweepThreads, 0, st>>>(a);
            ++launches;
        }
    }
    cuda_check(cudaGetLastError(), "kernel launch");
    h->launches = launches;
}

// device leaf code of terminal p: -((col << vbits | vidx) + 2)
inline int32_t leaf_ref(const Grammar& g, int32_t p, int32_t vbits) {
    const int64_t q = ((int64_t)g.term_col[p] << vbits) | g.term_vidx[p];
    return (int32_t)(-(q + 2));
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
        const int64_t tail_w = (int64_t)kSweepThreads * kNodesPerThread / (policy == GC_F32_SUM && k_max == 16 ? 4 : 1);
        int64_t first_narrow = L + 1;
        while (first_narrow > 1 && g.lvl_off[first_narrow] - g.lvl_off[first_narrow - 1] <= tail_w) --first_narrow;
        h->grid_levels = (int)(L - first_narrow + 1 >= 2 ? first_narrow - 1 : L);

        // level table and nodes with leaf codes, each level padded to 16 nodes
        h->lv.assign((size_t)(4 * (L + 2)), 0);
        std::vector<int32_t> nodes((size_t)(2 * d.n_nodes_padded), -1);
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
                    nodes[2 * (start + q) + t] = c <= -2 ? leaf_ref(g, -c - 2, d.vbits) : c;
                }
            start += pad_nodes(w);
        }
        std::vector<int32_t> cref(g.c_ref.size());
        for (size_t e = 0; e < cref.size(); ++e) {
            const int32_t c = g.c_ref[e];
            cref[e] = c <= -2 ? leaf_ref(g, -c - 2, d.vbits) : c;
        }
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
                or_update_kernel<<<grid_for(n, kLevelThreads, h->sms), kLevelThreads, 0, st>>>(xv, yv, n, changed);
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
