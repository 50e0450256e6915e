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
//   row emit        y[r] = (+) over row r's symbols of C               (Lemma 2.2),
//                   in one of two modes (layout.hpp): long rows are reduced
//                   level by level in chunks, straight from the level buffer
//                   right after the level is computed (emit on the spot,
//                   Sec. 4.3) and summed per row at the end; short rows read
//                   root values captured into RV
//
// Schedule (differences from the pages' two launches per level, for this GPU):
//   * one persistent cooperative kernel per product, two CTAs of 512 threads
//     per SM; levels are separated by a grid barrier whose waits are bounded
//     (a wait that runs out sets the status word and the kernel returns);
//   * within a level every warp works on its own chunks of nodes (128
//     one-lane values, 4 per lane; or 16 four-lane values, 2 per lane),
//     coalesced, with no block-wide synchronisation, and loads
//     the next chunk's child pairs -- possibly of the next level, since pairs
//     do not depend on values -- before gathering the current chunk's
//     children, so node-stream latency hides behind gathers and barriers;
//   * level 1 evaluates its (all-terminal) children in the sweep while the
//     grid writes the T copies, so T costs no phase of its own;
//   * child values are gathered through L1/L2 (the grid barrier's gpu-scope
//     acquire orders them after the writers); the node and C streams are
//     loaded evict-first; root values for RV are stored evict-last;
//   * the narrow top levels run on one CTA with block-level barriers, in a
//     small buffer pair of their own, so that the other CTAs can reduce the
//     C chunks of the last wide level meanwhile;
//   * the pages emit with atomicAdd into y; here every partial sum has a
//     fixed order: deterministic, no atomics.
// A second schedule launches one kernel per level plus one emit kernel with
// the same device functions (bit-identical y): the launch sequence of
// Listing 1, kept as the reference point for the persistent one.
#include <cuda_runtime.h>

#include <cstring>
#include <type_traits>
#include <memory>
#include <mutex>

#include "common.hpp"
#include "flow.hpp"
#include "layout.hpp"
#include "loop.hpp"
#include "policy.cuh"

struct gc_handle {
    gc_policy policy = GC_F32_SUM;
    int32_t k_max = 1;
    int64_t n = 0, m = 0, L = 0, n_roots = 0, c_len = 0, max_width = 0, alpha = 0, n_carry = 0;
    std::vector<int64_t> lv;      // host copy of the level table, 4 (L+2)
    char* arena = nullptr;
    gcs::DevLayout lay{};
    int sms = 1;
    int device = 0;               // the device the arena lives on (current at gc_upload)
    int emit_group = 32;          // row emit: threads per row (0 in the chunked emits)
    int schedule = 0;             // 0 persistent (if cooperative launch works), 1 per level
    int coop = 0;                 // device supports cooperative launch
    int grid_levels = 0;          // levels 1..grid_levels use the whole grid
    unsigned long long bar_base = 0;   // barrier arrivals of all earlier persistent launches
    unsigned long long tbar_base = 0;  // arrivals on the slice kernel's tail-group counter
    long long timeout_cycles = 4000000000LL;
    int32_t inject = 0;           // test-only: 1 = CTA 0 skips its first barrier arrival
    int64_t launches = 0;
    // dataflow sweep (one value a node): block plan counts and the product
    // number its ready flags and level counters are stamped with
    bool flow = false;
    int64_t nblocks = 0, final_k0 = 0;
    std::vector<int64_t> lvl_blk;   // first block of each level (L+2)
    uint32_t epoch = 0;
    const int32_t* conv = nullptr;   // during a device-side fixpoint loop: its converged word
    gcs::LoopHost loop;              // the fixpoint loop's pinned words and events
};

namespace gcs {
namespace {

constexpr int kThreads = 512;        // every kernel: 16 warps
constexpr int kWarps = kThreads / 32;
constexpr int LV_START = 0, LV_W = 1, LV_ROOTS = 2, LV_ROFF = 3, LV_ECH = 4, LV_TOFF = 5;
constexpr int LV_CR = 6, LV_CN = 7, LV_COFF = 8;   // carried roots, carried others, first carry slot
constexpr int LV_ROWS = (int)kLevelRows;
static_assert(LV_COFF < LV_ROWS, "level table rows");
// device index of carry slot s: kCarryBase + s (above every slot of a level buffer)
constexpr int32_t kCarryBase = 1 << 30;


void cuda_check(cudaError_t e, const char* what) {
    if (e != cudaSuccess) fail(GC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// A warp's chunk: U rows of NPW nodes, LPN lanes per node. Values of 16 bytes
// a lane take two rows, of 32 bytes one, so that a lane's pairs and child
// values stay in registers.
template <class P>
struct Chunk {
    static constexpr int U = sizeof(typename P::V) <= 8 ? 4 : sizeof(typename P::V) <= 16 ? 2 : 1;   // nodes per lane
    static constexpr int NPW = 32 / P::LPN;          // nodes per warp row
    static constexpr int NODES = NPW * U;            // nodes per warp chunk
};

// ---------------------------------------------------------------- PTX helpers
// Every .global-qualified instruction below takes a global-window address:
// the generic pointer (always into the caller's arena, the fixed scratch
// array or x / y) is converted with cvta.to.global first, as the PTX state
// spaces require, instead of relying on the generic and global windows
// coinciding.
__device__ __forceinline__ size_t gaddr(const void* p) { return __cvta_generic_to_global(p); }
__device__ __forceinline__ void red_add_release(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(gaddr(p)), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(gaddr(p)) : "memory");
    return v;
}
__device__ __forceinline__ int ld_volatile(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }
__device__ __forceinline__ void st_volatile(int32_t* p, int32_t v) { *reinterpret_cast<volatile int32_t*>(p) = v; }

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(gaddr(p))); }

__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// stores that ask L2 to keep the line (root values, read again by the emit)
__device__ __forceinline__ void st_keep(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(gaddr(p)), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(float4* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(gaddr(p)), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_keep(long long* p, long long v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(gaddr(p)), "l"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(unsigned long long* p, unsigned long long v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(gaddr(p)), "l"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ float shfl_x(float v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ long long shfl_x(long long v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ unsigned long long shfl_x(unsigned long long v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
}
__device__ __forceinline__ float4 shfl_x(float4 v, int m) {
    return make_float4(shfl_x(v.x, m), shfl_x(v.y, m), shfl_x(v.z, m), shfl_x(v.w, m));
}
__device__ __forceinline__ F8 shfl_x(F8 v, int m) { return F8{shfl_x(v.lo, m), shfl_x(v.hi, m)}; }
// read-only loads of x: __ldg, and two 16-byte ones for the eight-float value
template <class T>
__device__ __forceinline__ T ldg_value(const T* p) { return __ldg(p); }
__device__ __forceinline__ F8 ldg_value(const F8* p) {
    const float4* q = reinterpret_cast<const float4*>(p);
    return F8{__ldg(q), __ldg(q + 1)};
}
__device__ __forceinline__ void st_keep(F8* p, F8 v, uint64_t pol) {
    st_keep(&p->lo, v.lo, pol);
    st_keep(&p->hi, v.hi, pol);
}
__device__ __forceinline__ float shfl_up(float v, int d) { return __shfl_up_sync(0xffffffffu, v, d); }
__device__ __forceinline__ long long shfl_up(long long v, int d) { return __shfl_up_sync(0xffffffffu, v, d); }
__device__ __forceinline__ unsigned long long shfl_up(unsigned long long v, int d) {
    return __shfl_up_sync(0xffffffffu, v, d);
}

// ---------------------------------------------------------------- arguments
template <class P>
struct SweepArgs {
    using V = typename P::V;
    const int2* nodes;
    const int64_t* lv;        // level table: LV_ROWS rows of L+2
    int32_t L, L2, grid_levels;
    int64_t TB;               // leaf-table block length (values)
    int64_t alpha;
    const typename P::Leaf* Vd;
    const int32_t* leaf;      // leaf code per terminal
    int32_t vbits;
    const V* x;
    V* y;
    V* buf0;                  // level values (the two buffers alternate by level)
    V* buf1;
    V* rv;                    // row emit: [T | root values]
    const int32_t* c_off;     // row emit: C in row order
    const int32_t* c_ref;
    const int4* echunk;       // level emit: (start, length, id, 0) per chunk
    const int32_t* cref;      //   C grouped by level, then row
    const uint4* sref;        // slice emit: offsets into slices of [T | RV], 256 a tile
    const uint8_t* sflag;     //   segment starts, one bit per reference
    const int32_t* tile_sid;  //   first segment start of each tile
    const int32_t* row_pos;   //   segment start of each of a row's sums (nullptr: level emit)
    const int32_t* sx0;       //   first value of each slice
    const int32_t* stile;     //   tile range of each slice
    const int32_t* sorder;    //   slices, heaviest first
    int64_t slice, nslices;   //   most values a slice holds, slices
    const int32_t* row_ech;   // level / slice emit: row r's chunk / segment ids
    const int32_t* late_off;  //   row r's references into the tail levels
    const int32_t* late_ref;
    V* esum;                  //   chunk sums
    V* tbuf;                  // the narrow top levels' values, level after level
    V* carry;                 // values of nodes read two or more levels up
    int64_t tail_total;       // nodes of the tail levels (padded)
    int64_t n;
    int32_t emode;            // EmitMode
    int32_t emit_group;       // row emit: G lanes per row
    int32_t* status;
    int32_t* fix;             // a fixpoint in one launch (see sweep_fixpoint), else nullptr
    int32_t fix_max;          //   at most this many products
    unsigned long long* bar;
    unsigned long long bar_base;
    unsigned long long* tbar;        // slice emit: the tail group's arrival counter
    unsigned long long tbar_base;
    int32_t tail_group;              //   CTAs of the slice kernel that run the tail
    int32_t tail_solo;               //   first tail level CTA 0 runs alone (L + 1: none)
    long long timeout;
    int32_t inject;
    const int32_t* conv;      // fixpoint loop: nonzero once it has converged (then skip), or nullptr

    __device__ __forceinline__ int64_t lvl(int row, int k) const { return __ldg(lv + (int64_t)row * L2 + k); }
};

// V[l] (x) x[j] for a leaf code (column << vbits | value index)
template <class P>
__device__ __forceinline__ typename P::V leaf_value(int32_t code, int part, const SweepArgs<P>& a) {
    const uint32_t q = (uint32_t)code;
    const uint32_t col = q >> a.vbits, vi = q & ((1u << a.vbits) - 1u);
    const typename P::V* xp = a.x + (int64_t)col * P::LPN + part;
    if constexpr (kFixpointPolicy<P>)
        if (a.fix != nullptr) return P::leaf(__ldg(a.Vd + vi), *xp);   // x changes inside the launch
    return P::leaf(__ldg(a.Vd + vi), ldg_value(xp));
}

// The leaf table in front of RV (slice and row emits: C's bare terminals),
// grid-stride. The sweep itself evaluates terminals where it reads them.
template <class P>
__device__ void write_leaf_tables(const SweepArgs<P>& a, int64_t tid, int64_t nthreads) {
    if (a.emode == EMIT_LEVEL) return;   // no RV: the level emit evaluates its terminals too
    const int64_t total = (a.alpha + 1) * P::LPN;
    for (int64_t i = tid; i < total; i += nthreads) {
        const int64_t p = i / P::LPN;
        const int part = (int)(i % P::LPN);
        a.rv[i] = p == 0 ? P::identity() : leaf_value<P>(__ldg(a.leaf + (p - 1)), part, a);
    }
}

// Loads the child pairs of chunk c of level k (this warp's lanes).
template <class P>
__device__ __forceinline__ void load_chunk(const SweepArgs<P>& a, int k, int64_t c, int2 (&ab)[Chunk<P>::U]) {
    constexpr int NPW = Chunk<P>::NPW;
    const int lane = threadIdx.x & 31;
    const int64_t w = a.lvl(LV_W, k);
    const int2* src = a.nodes + a.lvl(LV_START, k);
#pragma unroll
    for (int u = 0; u < Chunk<P>::U; ++u) {
        const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
        ab[u] = node < w ? __ldcs(src + node) : make_int2(0, 0);
    }
}

// Same, from node pairs staged elsewhere (shared memory): src holds level k.
template <class P>
__device__ __forceinline__ void load_chunk_staged(const SweepArgs<P>& a, int k, int64_t c, const int2* src,
                                                  int2 (&ab)[Chunk<P>::U]) {
    constexpr int NPW = Chunk<P>::NPW;
    const int lane = threadIdx.x & 31;
    const int64_t w = a.lvl(LV_W, k);
#pragma unroll
    for (int u = 0; u < Chunk<P>::U; ++u) {
        const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
        ab[u] = node < w ? src[node] : make_int2(0, 0);
    }
}

// Combines chunk c of level k from its prefetched child pairs. prev holds
// level k-1; with kTail, its slots come from prev_tail instead when that
// level is one of the narrow ones kept in the tail buffers. The values go to
// cur[t]; roots also to rv[t] when rv is given.
template <class P, bool kTail, bool kC>
__device__ __forceinline__ void combine_chunk(const SweepArgs<P>& a, int k, int64_t c, const int2 (&ab)[Chunk<P>::U],
                                              const typename P::V* prev, const typename P::V* prev_tail,
                                              typename P::V* cur, typename P::V* rv, uint64_t keep) {
    using V = typename P::V;
    constexpr int NPW = Chunk<P>::NPW;
    const int lane = threadIdx.x & 31;
    const int part = lane % P::LPN;
    const int64_t w = a.lvl(LV_W, k), nroots = a.lvl(LV_ROOTS, k);
    V va[Chunk<P>::U], vb[Chunk<P>::U];
    if (k == 1) {
#pragma unroll
        for (int u = 0; u < Chunk<P>::U; ++u) {
            const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
            va[u] = node < w ? leaf_value<P>(ab[u].x, part, a) : P::identity();
            vb[u] = node < w ? leaf_value<P>(ab[u].y, part, a) : P::identity();
        }
    } else {
        // a child is a carry slot (index >= kCarryBase), a slot of level k-1
        // (in the tail buffer with kTail when that level is there), the
        // identity (-1), or a terminal by its leaf code (-2 - code),
        // evaluated here
        auto child = [&](int32_t x) -> V {
            if (kC && x >= kCarryBase) return a.carry[(int64_t)(x - kCarryBase) * P::LPN + part];
            if (x >= 0) {
                if (kTail && prev_tail != nullptr) return prev_tail[(int64_t)x * P::LPN + part];
                return prev[(int64_t)x * P::LPN + part];
            }
            return x == -1 ? P::identity() : leaf_value<P>(-2 - x, part, a);
        };
#pragma unroll
        for (int u = 0; u < Chunk<P>::U; ++u) {
            va[u] = child(ab[u].x);
            vb[u] = child(ab[u].y);
        }
    }
    // carried nodes (kC): the first cr roots and the cn nodes after the roots,
    // in carry slots from coff on (level sizes fit 32 bits); read levels later,
    // so kept in L2
    [[maybe_unused]] int32_t cr = 0, cn = 0, nr = 0;
    [[maybe_unused]] V* carry = nullptr;
    if constexpr (kC) {
        cr = (int32_t)a.lvl(LV_CR, k);
        cn = (int32_t)a.lvl(LV_CN, k);
        nr = (int32_t)nroots;
        carry = a.carry + a.lvl(LV_COFF, k) * P::LPN;
    }
#pragma unroll
    for (int u = 0; u < Chunk<P>::U; ++u) {
        const int64_t node = c * Chunk<P>::NODES + u * NPW + lane / P::LPN;
        if (node < w) {
            const V v = P::combine(va[u], vb[u]);
            cur[node * P::LPN + part] = v;
            if (rv != nullptr && node < nroots) st_keep(rv + node * P::LPN + part, v, keep);
            if constexpr (kC) {
                const int32_t t = (int32_t)node;
                const int32_t cs = t < cr ? t : (t >= nr && t - nr < cn) ? cr + (t - nr) : -1;
                if (cs >= 0) st_keep(carry + (int64_t)cs * P::LPN + part, v, keep);
            }
        }
    }
}

// Buffer pointers of grid level k: level k-1 in, level k's values out.
template <class P>
struct LevelIO {
    const typename P::V* prev;
    typename P::V* cur;
    typename P::V* rv;
};
template <class P>
__device__ __forceinline__ LevelIO<P> level_io(const SweepArgs<P>& a, int k) {
    LevelIO<P> io;
    io.prev = (k & 1) ? a.buf0 : a.buf1;
    io.cur = (k & 1) ? a.buf1 : a.buf0;
    io.rv = a.emode != EMIT_LEVEL ? a.rv + (a.TB + a.lvl(LV_ROFF, k)) * P::LPN : nullptr;
    return io;
}

// Buffer pointers of tail level k > Lg: level k-1 from its full buffer
// (k-1 == Lg) or from the tail buffer, level k's values into the tail buffer.
template <class P>
struct TailIO {
    const typename P::V* prev;
    const typename P::V* prev_tail;   // nullptr: level k-1 is in prev
    typename P::V* cur;
    typename P::V* rv;
};
template <class P>
__device__ __forceinline__ TailIO<P> tail_io(const SweepArgs<P>& a, int k, typename P::V* tb) {
    TailIO<P> io;
    io.prev = (k & 1) ? a.buf0 : a.buf1;
    io.prev_tail = k - 1 > a.grid_levels ? tb + a.lvl(LV_TOFF, k - 1) * P::LPN : nullptr;
    io.cur = tb + a.lvl(LV_TOFF, k) * P::LPN;
    io.rv = a.emode == EMIT_ROWS ? a.rv + (a.TB + a.lvl(LV_ROFF, k)) * P::LPN : nullptr;   // late refs read tbuf
    return io;
}

// ---------------------------------------------------------------- row emit

// S symbol slots of LPN lanes each per row, S = min(G, 32 / LPN) (G divides
// 32); warps walk rows in lockstep so the shuffles always see the full warp.
// Lane (slot, part) sums part `part` of the row's symbols q = s+slot,
// s+slot+S, ... in order, then the group reduces the slots by a fixed butterfly.
template <class P, int G>
__device__ void emit_groups(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    using V = typename P::V;
    constexpr int S = G < 32 / P::LPN ? G : 32 / P::LPN;
    constexpr int GG = S * P::LPN;                     // lanes per row
    constexpr int RPW = 32 / GG;                       // rows per warp
    constexpr int BATCH = sizeof(V) <= 8 ? 4 : 2;      // symbols loaded together per lane
    const int lane = threadIdx.x & 31;
    const int gl = lane % GG;
    const int slot = gl / P::LPN, part = gl % P::LPN;
    const int64_t warp = block * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = nblocks * kWarps;
    // the next rows' C ranges are loaded before the current rows are reduced
    int64_t row = warp * RPW + lane / GG;
    int32_t s = 0, e = 0;
    if (row < a.n) {
        s = __ldg(a.c_off + row);
        e = __ldg(a.c_off + row + 1);
    }
    for (int64_t base = warp * RPW; base < a.n; base += nwarps * RPW) {
        const int64_t nrow = row + nwarps * RPW;
        int32_t ns = 0, ne = 0;
        if (nrow < a.n) {
            ns = __ldg(a.c_off + nrow);
            ne = __ldg(a.c_off + nrow + 1);
        }
        V acc = P::identity();
        if (row < a.n) {
            for (int32_t q0 = s + slot; q0 < e; q0 += S * BATCH) {
                int32_t c[BATCH];
#pragma unroll
                for (int u = 0; u < BATCH; ++u) c[u] = q0 + u * S < e ? __ldcs(a.c_ref + q0 + u * S) : 0;
                V v[BATCH];
#pragma unroll
                for (int u = 0; u < BATCH; ++u) v[u] = a.rv[(int64_t)c[u] * P::LPN + part];
#pragma unroll
                for (int u = 0; u < BATCH; ++u) acc = P::combine(acc, v[u]);
            }
        }
#pragma unroll
        for (int msk = GG / 2; msk >= P::LPN; msk >>= 1) acc = P::combine(acc, shfl_x(acc, msk));
        if (row < a.n && slot == 0) a.y[row * P::LPN + part] = acc;
        row = nrow;
        s = ns;
        e = ne;
    }
}

// Level and chunk emit: chunk j holds references cref[start .. start+len) of
// one row (and one level, in the level emit), len <= kEmitChunk. A warp takes
// 32/LPN references at a time, LPN lanes each; lane (slot, part) sums part
// `part` of references slot, slot + 32/LPN, ... in order, the warp reduces the
// slots by a fixed butterfly, and the sum goes to esum[id]. base is the
// level's buffer: a reference is one of its root slots, or a bare terminal
// of C by its leaf code (-2 - code), evaluated here.
constexpr int kEmitChunk = (int)kEmitChunkSyms;

template <class P>
__device__ __forceinline__ void emit_chunk(const SweepArgs<P>& a, int64_t j, const typename P::V* base) {
    using V = typename P::V;
    constexpr int NS = 32 / P::LPN;            // reference slots per warp row
    constexpr int PER = kEmitChunk / NS;       // references per lane
    constexpr int B = sizeof(V) <= 8 ? PER : 4;   // references loaded together
    const int lane = threadIdx.x & 31;
    const int part = lane % P::LPN, slot = lane / P::LPN;
    const int4 ch = __ldg(a.echunk + j);
    V acc = P::identity();
    auto batch = [&](int u0) {
        int32_t r[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int idx = (u0 + u) * NS + slot;
            r[u] = idx < ch.y ? __ldcs(a.cref + ch.x + idx) : -1;   // padding: the identity
        }
        V v[B];
#pragma unroll
        for (int u = 0; u < B; ++u) {
            v[u] = r[u] >= 0 ? base[(int64_t)r[u] * P::LPN + part]
                   : r[u] == -1 ? P::identity() : leaf_value<P>(-2 - r[u], part, a);
        }
#pragma unroll
        for (int u = 0; u < B; ++u) acc = P::combine(acc, v[u]);
    };
    if constexpr (PER / B <= 8) {
#pragma unroll
        for (int u0 = 0; u0 < PER; u0 += B) {
            if (u0 * NS >= ch.y) break;            // the same for the whole warp
            batch(u0);
        }
    } else {   // wide values: few slots per warp row, so many batches
#pragma unroll 1
        for (int u0 = 0; u0 < PER && u0 * NS < ch.y; u0 += B) batch(u0);
    }
#pragma unroll
    for (int msk = 16; msk >= P::LPN; msk >>= 1) acc = P::combine(acc, shfl_x(acc, msk));
    if (slot == 0) a.esum[(int64_t)ch.z * P::LPN + part] = acc;
}

// Chunks j0 <= j < j1, spread over warps gwarp, gwarp + nwarps, ...
template <class P>
__device__ void emit_chunks(const SweepArgs<P>& a, int64_t j0, int64_t j1, const typename P::V* base, int64_t gwarp,
                            int64_t nwarps) {
    for (int64_t j = j0 + gwarp; j < j1; j += nwarps) emit_chunk<P>(a, j, base);
}

// The chunks of level k (0 = bare terminals).
template <class P>
__device__ void emit_level(const SweepArgs<P>& a, int k, const typename P::V* base, int64_t gwarp, int64_t nwarps) {
    emit_chunks<P>(a, a.lvl(LV_ECH, k), a.lvl(LV_ECH, k + 1), base, gwarp, nwarps);
}

// y[r] = row r's chunk (or segment) sums, then its references into the tail
// levels: one warp per row, LPN lanes per item; lane (slot, part) adds part
// `part` of items slot, slot + 32/LPN, ... of the row's list [chunk sums |
// tail references] in order, and the warp reduces the slots by a fixed
// butterfly (identity for an empty row). The slice emit's sums sit at their
// segment starts, found through row_pos.
template <class P>
__device__ void emit_final(const SweepArgs<P>& a, int64_t gwarp, int64_t nwarps) {
    using V = typename P::V;
    constexpr int NS = 32 / P::LPN;
    const int lane = threadIdx.x & 31;
    const int part = lane % P::LPN, slot = lane / P::LPN;
    for (int64_t row = gwarp; row < a.n; row += nwarps) {
        const int32_t c0 = __ldg(a.row_ech + row), c1 = __ldg(a.row_ech + row + 1);
        const int32_t q0 = __ldg(a.late_off + row), q1 = __ldg(a.late_off + row + 1);
        const int32_t nc = c1 - c0, total = nc + (q1 - q0);
        V acc = P::identity();
        constexpr int B = sizeof(V) <= 8 ? 8 : 4;   // items a lane loads together
        for (int32_t i0 = 0; i0 < total; i0 += B * NS) {
            V v[B];
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int32_t i = i0 + u * NS + slot;
                const int64_t e = i < nc ? (a.row_pos ? (int64_t)__ldg(a.row_pos + c0 + i) : (int64_t)(c0 + i)) : 0;
                v[u] = i >= total ? P::identity()
                       : i < nc   ? a.esum[e * P::LPN + part]
                                  : a.tbuf[(int64_t)__ldg(a.late_ref + q0 + (i - nc)) * P::LPN + part];
            }
#pragma unroll
            for (int u = 0; u < B; ++u) acc = P::combine(acc, v[u]);
        }
#pragma unroll
        for (int msk = 16; msk >= P::LPN; msk >>= 1) acc = P::combine(acc, shfl_x(acc, msk));
        if (slot == 0) a.y[row * P::LPN + part] = acc;
    }
}

// The row pass of the slice kernel, split around its grid barrier. Which sums
// and tail values a row adds (its sum positions and late references) does not
// depend on the slices, so plan_rows reads them for the warp's first R rows
// before the barrier, as indices: e >= 0 a sum, e <= -2 tail value -2 - e,
// -1 nothing. finish_rows then only gathers; rows with more than B * NS items
// and rows past the first R go through emit_final's loop.
template <int R, int B>
struct RowPlan {
    int32_t e[R][B];
    int32_t total[R];
};

template <class P, int R, int B>
__device__ void plan_rows(const SweepArgs<P>& a, int64_t gwarp, int64_t nwarps, RowPlan<R, B>& pl) {
    constexpr int NS = 32 / P::LPN;
    const int slot = (threadIdx.x & 31) / P::LPN;
    int32_t c0[R], nc[R], q0[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int64_t row = gwarp + j * nwarps;
        if (row < a.n) {
            c0[j] = __ldg(a.row_ech + row);
            nc[j] = __ldg(a.row_ech + row + 1) - c0[j];
            q0[j] = __ldg(a.late_off + row);
            pl.total[j] = nc[j] + (__ldg(a.late_off + row + 1) - q0[j]);
        } else {
            c0[j] = nc[j] = q0[j] = pl.total[j] = 0;
        }
    }
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int32_t i = u * NS + slot;
            pl.e[j][u] = i >= pl.total[j] ? -1
                         : i < nc[j]      ? (a.row_pos ? __ldg(a.row_pos + c0[j] + i) : c0[j] + i)
                                          : -2 - __ldg(a.late_ref + q0[j] + (i - nc[j]));
        }
}

template <class P, int R, int B>
__device__ void finish_rows(const SweepArgs<P>& a, int64_t gwarp, int64_t nwarps, const RowPlan<R, B>& pl) {
    using V = typename P::V;
    constexpr int NS = 32 / P::LPN;
    const int lane = threadIdx.x & 31;
    const int part = lane % P::LPN, slot = lane / P::LPN;
    V v[R][B];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
        for (int u = 0; u < B; ++u) {
            const int32_t e = pl.e[j][u];
            v[j][u] = e == -1 ? P::identity()
                      : e >= 0 ? a.esum[(int64_t)e * P::LPN + part]
                               : a.tbuf[(int64_t)(-2 - e) * P::LPN + part];
        }
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int64_t row = gwarp + j * nwarps;
        if (row >= a.n) break;
        V acc = v[j][0];
#pragma unroll
        for (int u = 1; u < B; ++u) acc = P::combine(acc, v[j][u]);
        if (pl.total[j] > B * NS) {   // the rest of a long row
            const int32_t c0 = __ldg(a.row_ech + row), nc = __ldg(a.row_ech + row + 1) - c0;
            const int32_t q0 = __ldg(a.late_off + row);
            for (int32_t i = B * NS + slot; i < pl.total[j]; i += NS) {
                const V w = i < nc ? a.esum[(a.row_pos ? (int64_t)__ldg(a.row_pos + c0 + i) : (int64_t)(c0 + i)) * P::LPN + part]
                                   : a.tbuf[(int64_t)__ldg(a.late_ref + q0 + (i - nc)) * P::LPN + part];
                acc = P::combine(acc, w);
            }
        }
#pragma unroll
        for (int msk = 16; msk >= P::LPN; msk >>= 1) acc = P::combine(acc, shfl_x(acc, msk));
        if (slot == 0) a.y[row * P::LPN + part] = acc;
    }
    if (gwarp + R * nwarps < a.n) emit_final<P>(a, gwarp + R * nwarps, nwarps);
}

// Row emit: groups of G lanes per row (emit_group = G).
template <class P>
__device__ void emit_rows(const SweepArgs<P>& a, int64_t block, int64_t nblocks) {
    switch (a.emit_group) {
        case 1: emit_groups<P, 1>(a, block, nblocks); break;
        case 2: emit_groups<P, 2>(a, block, nblocks); break;
        case 4: emit_groups<P, 4>(a, block, nblocks); break;
        case 8: emit_groups<P, 8>(a, block, nblocks); break;
        case 16: emit_groups<P, 16>(a, block, nblocks); break;
        default: emit_groups<P, 32>(a, block, nblocks); break;
    }
}

// ---------------------------------------------------------------- grid barrier
// Arrival counter that only grows; bar_base is its value when the launch
// starts, and barrier j of this launch completes when it reaches
// bar_base + (j + 1) * gridDim.x. A wait gives up after a.timeout
// cycles (or when another CTA already reported a timeout), sets the status
// word and returns false. The acquire at gpu scope, followed by the block
// barrier, orders every thread's later loads after the other CTAs' writes.
// Barrier j of `members` CTAs on the arrival counter bar, whose value was
// base when the launch started.
template <class P>
__device__ bool sync_on(const SweepArgs<P>& a, unsigned long long* bar, unsigned long long base, unsigned long long j,
                        unsigned long long members) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const bool skip = a.inject == 1 && blockIdx.x == 0 && j == 0 && bar == a.bar;   // test-only
        if (!skip) {
            __threadfence();
            red_add_release(bar, 1ull);
        }
        const unsigned long long target = base + (j + 1) * members;
        const long long t0 = clock64();
        unsigned it = 0;
        while (ld_acquire(bar) < target) {
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

template <class P>
__device__ bool grid_sync(const SweepArgs<P>& a, unsigned long long j) {
    return sync_on<P>(a, a.bar, a.bar_base, j, gridDim.x);
}

// Arrival at a barrier of bar without waiting for it (a CTA that has no work
// after it, but whose writes the waiting CTAs read).
__device__ __forceinline__ void arrive_on(unsigned long long* bar) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_add_release(bar, 1ull);
    }
}

// ---------------------------------------------------------------- persistent sweep
// One product of the persistent sweep, this CTA's share: leaf tables, the
// wide levels, then (unless the slice kernel takes over) the tail and the
// emit. nbar counts the launch's grid barriers passed so far. False if a
// barrier timed out (the status word says so).
template <class P, bool kC>
__device__ __forceinline__ bool sweep_product(const SweepArgs<P>& a, unsigned long long& nbar) {
    const int Lg = a.grid_levels;
    const int64_t GW = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const uint64_t keep = l2_evict_last();
    const bool tail = Lg < a.L;
    const bool tail_cta = tail && blockIdx.x == 0;
    auto nchunks = [&](int k) { return (a.lvl(LV_W, k) + Chunk<P>::NODES - 1) / Chunk<P>::NODES; };
    auto norm = [&](int& k, int64_t& c) {
        while (k <= Lg && c >= nchunks(k)) {
            ++k;
            c = gw;
        }
    };

    // CTA 0 asks L2 for the tail's node pairs (levels Lg+1..L, contiguous at
    // the end of the node array) while the grid sweeps the wide levels
    if (tail_cta && a.emode != EMIT_SLICE) {
        const int2* src = a.nodes + a.lvl(LV_START, Lg + 1);
        for (int64_t i = (int64_t)threadIdx.x * 16; i < a.tail_total; i += (int64_t)kThreads * 16) prefetch_l2(src + i);
    }

    write_leaf_tables<P>(a, (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads);
    const bool lemit = a.emode == EMIT_LEVEL;

    int kn = 1;
    int64_t cn = gw;
    norm(kn, cn);
    int2 nab[Chunk<P>::U];
    if (kn <= Lg) load_chunk<P>(a, kn, cn, nab);
    for (int k = 1; k <= Lg; ++k) {
        if (k > 1 && !grid_sync(a, nbar++)) return false;
        const LevelIO<P> io = level_io<P>(a, k);
        while (kn == k) {
            int2 ab[Chunk<P>::U];
#pragma unroll
            for (int u = 0; u < Chunk<P>::U; ++u) ab[u] = nab[u];
            const int64_t c = cn;
            cn += GW;
            norm(kn, cn);
            if (kn <= Lg) load_chunk<P>(a, kn, cn, nab);   // next chunk, maybe of a later level
            combine_chunk<P, false, kC>(a, k, c, ab, io.prev, nullptr, io.cur, io.rv, keep);
        }
        if (lemit && k >= 2) {   // level k-1 is complete and still in its buffer
            emit_level<P>(a, k - 1, io.prev, gw, GW);
            if (k == 2) emit_level<P>(a, 0, a.buf0, gw, GW);
        }
    }
    // slice emit: the second kernel takes the tail, the emit and the row pass
    if (a.emode == EMIT_SLICE) return true;
    if (!grid_sync(a, nbar++)) return false;
    // while CTA 0 runs the tail, the others reduce what is left of the level
    // emit (level Lg, and the terminals if no phase took them)
    const int64_t skip = (tail && gridDim.x > 1) ? kWarps : 0;
    if (gw >= skip) {
        if (lemit) {
            if (Lg >= 1) emit_level<P>(a, Lg, (Lg & 1) ? a.buf1 : a.buf0, gw - skip, GW - skip);
            if (Lg < 2) emit_level<P>(a, 0, a.buf0, gw - skip, GW - skip);
        }
    }
    // narrow top levels: CTA 0 alone, block barriers only, into the tail buffer
    if (tail_cta) {
        const int w0 = threadIdx.x >> 5;
        for (int k = Lg + 1; k <= a.L; ++k) {
            const TailIO<P> io = tail_io<P>(a, k, a.tbuf);
            for (int64_t c = w0; c < nchunks(k); c += kWarps) {
                int2 ab[Chunk<P>::U];
                load_chunk<P>(a, k, c, ab);
                combine_chunk<P, true, kC>(a, k, c, ab, io.prev, io.prev_tail, io.cur, io.rv, keep);
            }
            __syncthreads();
        }
    }
    if (!grid_sync(a, nbar++)) return false;
    if (a.emode != EMIT_ROWS) emit_final<P>(a, gw, GW);
    else emit_rows<P>(a, blockIdx.x, gridDim.x);
    return true;
}

// A whole fixpoint x = x (+) (M (x) x) in one launch (handles whose product is
// this kernel alone: no slice kernel): product it into y, a grid barrier, then
// x = x (+) y over the grid with a changed flag, a grid barrier, and every CTA
// reads the flag. fix[0] / fix[1] are the changed flags of the even / odd
// products (a product's flag is cleared by CTA 0 during the product before
// it, after every CTA has read it), fix[2] = 1 and fix[3] = the product
// count on convergence; both stay 0 if a.fix_max products did not converge.
// Each product passes sweep_barriers + 2 grid barriers. (Folding the update
// into the row emit instead, one barrier fewer, measured slower.)
template <class P, bool kC>
__device__ void sweep_fixpoint(const SweepArgs<P>& a, unsigned long long& nbar) {
    using V = typename P::V;
    V* x = const_cast<V*>(a.x);   // x is the fixpoint's iterate, updated in place
    int32_t* fx = a.fix;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, nth = (int64_t)gridDim.x * blockDim.x;
    for (int32_t it = 1; it <= a.fix_max; ++it) {
        if (!sweep_product<P, kC>(a, nbar)) return;
        if (!grid_sync(a, nbar++)) return;   // every row of y is written and x no longer read
        int ch = 0;
        for (int64_t i = tid; i < a.n; i += nth) {
            const V u = x[i], v = P::combine(u, a.y[i]);
            if (v != u) {
                x[i] = v;
                ch = 1;
            }
        }
        if (__syncthreads_or(ch) && threadIdx.x == 0) st_volatile(fx + (it & 1), 1);
        if (blockIdx.x == 0 && threadIdx.x == 0) st_volatile(fx + ((it + 1) & 1), 0);
        if (!grid_sync(a, nbar++)) return;
        if (ld_volatile(fx + (it & 1)) == 0) {   // nothing changed: converged at product it
            if (blockIdx.x == 0 && threadIdx.x == 0) {
                fx[3] = it;
                fx[2] = 1;
            }
            return;
        }
    }
}

template <class P, bool kC>
__global__ void __launch_bounds__(kThreads, 2) sweep_kernel(const SweepArgs<P> a) {
    // an unread earlier timeout left the barrier counter part-way: do nothing
    if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) return;
    const int Lg = a.grid_levels;
    // a converged fixpoint loop skips the product: the CTA's arrivals at the
    // launch's grid barriers (one a level after the first; before the tail
    // and the emit unless the slice kernel takes them) in one addition
    if (a.conv != nullptr && ld_volatile(a.conv) != 0) {
        if (threadIdx.x == 0)
            red_add_release(a.bar, (unsigned long long)((Lg > 1 ? Lg - 1 : 0) + (a.emode == EMIT_SLICE ? 0 : 2)));
        return;
    }
    unsigned long long nbar = 0;
    if constexpr (kFixpointPolicy<P> && !kC)   // the one-launch fixpoint runs without carry slots
        if (a.fix != nullptr) {
            sweep_fixpoint<P, kC>(a, nbar);
            return;
        }
    sweep_product<P, kC>(a, nbar);
}

// ---------------------------------------------------------------- slice emit
constexpr int kSliceThreads = 1024;
constexpr int kTailGroup = 16;   // CTAs of the slice kernel that run the tail

// The narrow top levels on the slice kernel's first `group` CTAs, chunks
// dealt over their warps, a barrier of the group between levels (on its own
// counter), values in the tail buffer. From level a.tail_solo on (at most one
// chunk per warp of a CTA) CTA 0 goes on alone with block barriers: the other
// CTAs arrive at the barrier before that level and leave. As in the sweep, a
// warp loads its next chunk's child pairs, possibly of the next level, before
// gathering the current chunk's children.
template <class P, bool kC>
__device__ bool slice_tail(const SweepArgs<P>& a, int64_t group) {
    const int Lg = a.grid_levels, ks = a.tail_solo;
    const int32_t wpc = (int32_t)(blockDim.x >> 5), nw = (int32_t)group * wpc;
    const int32_t w0 = (int32_t)blockIdx.x * wpc + (int32_t)(threadIdx.x >> 5);
    const uint64_t keep = l2_evict_last();
    auto nchunks = [&](int k) { return (int32_t)((a.lvl(LV_W, k) + Chunk<P>::NODES - 1) / Chunk<P>::NODES); };
    auto stride = [&](int k) { return k < ks ? nw : wpc; };
    auto norm = [&](int& k, int32_t& c) {
        while (k <= a.L && c >= nchunks(k)) {
            ++k;
            c = w0;
        }
    };
    int kn = Lg + 1;
    int32_t cn = w0;
    norm(kn, cn);
    int2 nab[Chunk<P>::U];
    if (kn <= a.L) load_chunk<P>(a, kn, cn, nab);
    unsigned long long j = 0;
    for (int k = Lg + 1; k <= a.L; ++k) {
        if (k > Lg + 1) {
            if (group > 1 && k <= ks) {
                if (k == ks && blockIdx.x != 0) {
                    arrive_on(a.tbar);
                    return true;
                }
                if (!sync_on<P>(a, a.tbar, a.tbar_base, j++, (unsigned long long)group)) return false;
            } else {
                __syncthreads();
            }
        }
        const TailIO<P> io = tail_io<P>(a, k, a.tbuf);
        while (kn == k) {
            int2 ab[Chunk<P>::U];
#pragma unroll
            for (int u = 0; u < Chunk<P>::U; ++u) ab[u] = nab[u];
            const int32_t c = cn;
            cn += stride(kn);
            norm(kn, cn);
            if (kn <= a.L) load_chunk<P>(a, kn, cn, nab);
            combine_chunk<P, true, kC>(a, k, c, ab, io.prev, io.prev_tail, io.cur, io.rv, keep);
        }
    }
    return true;
}

// One tile of a slice, on one warp: lane l holds references 8l .. 8l+7 (their
// offsets o, their segment-start bits f). A lane adds its references in order,
// closing the runs that start and end inside it; a segmented scan over the
// lanes (Hillis-Steele, fixed order) carries each open run into the lane where
// the next segment starts, which closes it, and lane 31 closes the run open at
// the tile's end. The sum of the tile's k-th segment start goes to
// esum[base + k] (padding included: nothing reads it).
template <class P>
__device__ __forceinline__ void tile_sums(const SweepArgs<P>& a, int64_t base, uint4 o, uint32_t f,
                                          const typename P::V* sv) {
    using V = typename P::V;
    const int lane = threadIdx.x & 31;
    const uint32_t w[4] = {o.x, o.y, o.z, o.w};
    V v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = sv[(w[i / 2] >> (16 * (i % 2))) & 0xffffu];
    // segment starts before this lane, and in all lanes up to this one
    const int nf = __popc(f);
    int incl = nf;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += t;
    }
    const int before = incl - nf;
    // runs inside the lane
    V cur = P::identity(), head = P::identity();
    bool open_head = true;
    int k = before - 1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if ((f >> i) & 1u) {
            if (open_head) {
                head = cur;
                open_head = false;
            } else {
                a.esum[base + k] = cur;
            }
            ++k;
            cur = P::identity();
        }
        cur = P::combine(cur, v[i]);
    }
    // segmented inclusive scan of (lane holds a start, sum of its last run)
    bool F = f != 0u;
    V X = cur;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const bool Fp = __shfl_up_sync(0xffffffffu, F, d);
        const V Xp = shfl_up(X, d);
        if (lane >= d) {
            if (!F) X = P::combine(Xp, X);
            F = F || Fp;
        }
    }
    // the run open at this lane's start: the scan one lane down
    const V carry = shfl_up(X, 1);
    if (f != 0u && before >= 1) a.esum[base + before - 1] = P::combine(lane >= 1 ? carry : P::identity(), head);
    if (lane == 31 && incl >= 1) a.esum[base + incl - 1] = X;
}

// Slice s of [T | RV] into shared memory, then its tiles: a warp claims tiles
// from a counter in shared memory (so the CTA's warps finish together) and
// loads its next tile's offsets, starts and first start index before reducing
// the current one.
template <class P>
__device__ void slice_sums(const SweepArgs<P>& a, int64_t s, typename P::V* sv) {
    __shared__ int32_t next_tile;
    using V = typename P::V;
    static_assert(kScalarPolicy<P>, "the slice emit serves one-lane scalar values");
    // values [x0, x1) in 16-byte units (x0 is a multiple of 256 values; the
    // last unit may run up to 15 bytes past x1, inside RV's padded allocation)
    const int64_t x0 = __ldg(a.sx0 + s), x1 = __ldg(a.sx0 + s + 1);
    const int64_t n16 = ((x1 - x0) * (int64_t)sizeof(V) + 15) / 16;
    const int4* src = reinterpret_cast<const int4*>(a.rv + x0);
    int4* dst = reinterpret_cast<int4*>(sv);
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
    const int64_t t0 = __ldg(a.stile + s), nw = blockDim.x >> 5;
    if (threadIdx.x == 0) next_tile = (int32_t)nw;
    __syncthreads();
    {
        const int lane = threadIdx.x & 31;
        const int64_t t1 = __ldg(a.stile + s + 1);
        auto claim = [&]() {
            int32_t i = 0;
            if (lane == 0) i = atomicAdd(&next_tile, 1);
            return t0 + __shfl_sync(0xffffffffu, i, 0);
        };
        int64_t t = t0 + (threadIdx.x >> 5);
        uint4 o = make_uint4(0, 0, 0, 0);
        uint32_t f = 0;
        int32_t sb = 0;
        if (t < t1) {
            o = __ldcs(a.sref + t * 32 + lane);
            f = __ldcs(a.sflag + t * 32 + lane);
            sb = __ldg(a.tile_sid + t);
        }
        while (t < t1) {
            const int64_t tn = claim();
            uint4 on = make_uint4(0, 0, 0, 0);
            uint32_t fn = 0;
            int32_t sbn = 0;
            if (tn < t1) {
                on = __ldcs(a.sref + tn * 32 + lane);
                fn = __ldcs(a.sflag + tn * 32 + lane);
                sbn = __ldg(a.tile_sid + tn);
            }
            tile_sums<P>(a, sb, o, f, sv);
            t = tn;
            o = on;
            f = fn;
            sb = sbn;
        }
    }
    __syncthreads();
}

// After the wide levels: slices on every CTA (when the launch is cooperative,
// the first tail_group CTAs run the tail instead), and, cooperative, the row
// plan, a grid barrier and the row pass.
template <class P, bool kC>
__global__ void __launch_bounds__(kSliceThreads, 1) slice_kernel(const SweepArgs<P> a, int coop) {
    using V = typename P::V;
    extern __shared__ __align__(16) unsigned char slice_smem[];
    if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) return;
    // a converged fixpoint loop skips the product (one arrival at the grid
    // barrier, as if the launch had passed it)
    if (a.conv != nullptr && ld_volatile(a.conv) != 0) {
        if (coop && threadIdx.x == 0) {
            red_add_release(a.bar, 1ull);
            // the tail group's CTAs pass one group barrier a tail level up to tail_solo
            const bool tl = a.grid_levels < a.L;
            const int64_t grp = !tl ? 0 : gridDim.x > a.tail_group ? a.tail_group : gridDim.x;
            const int64_t per = (a.tail_solo < a.L ? a.tail_solo : a.L) - a.grid_levels - 1;
            if (grp > 1 && blockIdx.x < grp && per > 0) red_add_release(a.tbar, (unsigned long long)per);
        }
        return;
    }
    const bool tail = coop && a.grid_levels < a.L;
    // the first tail_group CTAs run the tail (all of them when the grid is
    // that small), the others the slices
    const int64_t group = !tail ? 0 : gridDim.x > a.tail_group ? a.tail_group : gridDim.x;
    if (tail && blockIdx.x < group && !slice_tail<P, kC>(a, group)) return;
    const int64_t first = group < gridDim.x ? group : 0;
    if (blockIdx.x >= first)
        // slices heaviest first, dealt out in snake order: round r goes to the
        // CTAs in reverse when r is odd
        for (int64_t r = 0, g = gridDim.x - first, c = blockIdx.x - first;; ++r) {
            const int64_t i = r * g + ((r & 1) ? g - 1 - c : c);
            if (i >= a.nslices) break;
            slice_sums<P>(a, __ldg(a.sorder + i), reinterpret_cast<V*>(slice_smem));
        }
    if (!coop) return;
    {
        // rows on the slice CTAs only: the tail's CTAs reach the barrier last
        const int64_t wpc = blockDim.x >> 5;
        const int64_t gw = (int64_t)(blockIdx.x - first) * wpc + (threadIdx.x >> 5), GW = (gridDim.x - first) * wpc;
        constexpr int R = sizeof(V) <= 4 ? 3 : 2;
        RowPlan<R, 10> pl;
        if (blockIdx.x >= first) plan_rows<P>(a, gw, GW, pl);
        if (!grid_sync(a, 0)) return;
        if (blockIdx.x >= first) finish_rows<P>(a, gw, GW, pl);
    }
}

// ---------------------------------------------------------------- dataflow sweep
// One value a node (flow.hpp has the block plan). A CTA per SM, three roles:
// kNS staging warps, warp s owning stage s of a ring of shared-memory
// buffers -- it waits until its stage is free, copies the next block's node
// pairs in with one bulk copy completing on the stage's mbarrier, and waits
// for the block's dependencies (the producers' ready flags, and level k-2
// finished before level k overwrites its buffer); 16 compute warps evaluate
// the staged blocks in order, gathering each child from the level buffer of
// the level below through L1/L2 (the flag acquire and the stage's mbarrier
// order the gathers after the producers' writes), the identity, or a leaf
// evaluated in place, and write the values to the level buffer (and RV for
// roots); a publishing warp, once all compute warps have reported a block,
// sets its ready flag (one gpu-scope fence, then relaxed stores) and adds it
// to its level's done counter, so the fence stays off the compute path.
// Blocks are dealt to CTAs round robin over a processing order sorted by
// readiness, and a CTA works through its blocks in that order; every
// dependency comes earlier in the order, so the earliest unfinished block can
// always proceed (all CTAs are resident: cooperative launch). The final block
// (the narrow top levels) takes every staging buffer of its CTA and computes
// its levels one after the other in shared memory. Every wait is bounded.
constexpr int kFlowCW = 16;                   // compute warps of a CTA
constexpr int kFlowCT = 32 * kFlowCW;         // compute threads
constexpr int kFlowThreads = kFlowCT + 32 * ((int)kFlowStages + 1);   // and kNS staging warps, one publishing warp
constexpr int kNS = (int)kFlowStages;
constexpr int kSB = (int)kFlowStageBytes;
constexpr int LV_NBLK = 9;                    // level table: regular blocks of level k
static_assert(LV_NBLK < LV_ROWS, "level table rows");

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bulk copy global -> this CTA's shared memory, completing on bar (16-byte
// aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(gaddr(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(gaddr(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// generic-proxy writes and async-proxy (bulk copy) reads of the level buffers
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ uint32_t ld_acquire_u32(const int32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(gaddr(p)) : "memory");
    return v;
}
// one fence, then relaxed writes: together a release of both writes
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ void st_relaxed_u32(int32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(gaddr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add(unsigned long long* p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(gaddr(p)), "l"(v) : "memory");
}

template <class P>
struct FlowArgs {
    using V = typename P::V;
    const int2* pairs;        // block-local child references
    const int32_t* blk;       // kFlowBlkInts per block
    const int32_t* order;     // blocks in processing order; a launch takes positions [b_begin, b_end)
    const int32_t* deps;
    const int32_t* gran;
    const int64_t* lv;        // level table
    int32_t L2;               // its row stride
    int32_t b_begin, b_end;   // positions in the processing order of this launch
    int32_t final_block;      // id of the final block, or -1
    int32_t waits;            // 1: one launch for all blocks, wait for dependencies
    int32_t write_t;          // write T in front of RV
    int64_t TB, alpha;
    const typename P::Leaf* Vd;
    const int32_t* leaf;
    int32_t vbits;
    const V* x;
    V* rv;
    V* fb0;                   // level k is written to buffer k % 3
    V* fb1;
    V* fb2;
    int32_t* flags;           // per block: the product number once it is ready
    unsigned long long* done; // per level: blocks finished over all products
    uint32_t epoch;           // this product's number
    int32_t* status;
    long long timeout;
    int32_t inject;
    const int32_t* conv;      // fixpoint loop: nonzero once it has converged (then skip), or nullptr
    int32_t nblocks;          // all blocks of the plan

    __device__ __forceinline__ int64_t lvl(int row, int k) const { return __ldg(lv + (int64_t)row * L2 + k); }
    __device__ __forceinline__ V* buf(int k) const { return k % 3 == 0 ? fb0 : k % 3 == 1 ? fb1 : fb2; }
};

template <class P>
__device__ __forceinline__ typename P::V flow_leaf(const FlowArgs<P>& a, uint32_t q) {
    return P::leaf(__ldg(a.Vd + (q & ((1u << a.vbits) - 1u))), __ldg(a.x + (q >> a.vbits)));
}

// Bounded waits: each gives up after a.timeout cycles, or as soon as another
// wait has reported a timeout, and then returns false.
template <class P>
__device__ __forceinline__ bool wait_give_up(const FlowArgs<P>& a, long long t0) {
    if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) return true;
    if (clock64() - t0 > a.timeout) {
        atomicCAS(a.status, 0, (int32_t)GC_ERR_TIMEOUT);
        return true;
    }
    return false;
}
template <class P>
__device__ bool wait_flag(const int32_t* p, uint32_t want, const FlowArgs<P>& a) {
    const long long t0 = clock64();
    for (unsigned n = 0;; ++n) {
        if (ld_acquire_u32(p) == want) return true;
        if ((n & 15u) == 15u && wait_give_up(a, t0)) return false;
    }
}
template <class P>
__device__ bool wait_count(const unsigned long long* p, unsigned long long want, const FlowArgs<P>& a) {
    const long long t0 = clock64();
    for (unsigned n = 0;; ++n) {
        if (ld_acquire(p) >= want) return true;
        if ((n & 15u) == 15u && wait_give_up(a, t0)) return false;
    }
}
template <class P>
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity, const FlowArgs<P>& a) {
    const long long t0 = clock64();
    for (unsigned n = 0;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 63u && wait_give_up(a, t0)) return false;
    }
}

// shared-memory counters: release / acquire at CTA scope
__device__ __forceinline__ void red_release_cta(int* p, int v) {
    asm volatile("red.release.cta.shared::cta.add.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int* p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_cta(int* p, int v) {
    asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// What the compute warps need of a staged block, written by its staging
// warp (so the compute path reads no block record or level table).
struct FlowHead {
    long long out;   // level-buffer address of the block's first node (regular blocks)
    long long rvo;   // RV address of the block's first node
    long long prev;  // level buffer of k0 - 1 (regular blocks read their children there)
    int k0, k1, pb, nn, nr, wl1;
};

// Per-CTA pipeline state in shared memory.
struct FlowSync {
    FlowHead head[kNS];
    uint64_t full[kNS];    // stage s filled (bulk-copy bytes)
    uint64_t empty[kNS];   // stage s read by every compute warp (one arrival a warp)
    uint64_t cbar;         // the compute warps between the final block's levels
    int done[kNS];         // compute warps finished with stage s, over all its uses
    int stop;              // first iteration that will never be staged (a wait gave up)
    int pub;               // blocks published so far
};

// Staging warp w (w < kNS) owns stage w and stages this CTA's iterations
// it = w, w + kNS, ...: once its stage is free (every compute warp has read
// its previous use) it starts the bulk copy of the block's node pairs, then
// waits for the block's dependencies (the producers' ready flags; level k0 - 2
// finished, once a level); the final block also waits for every earlier block
// of the CTA to be published and copies the level below into the stage area.
// Lane 0's arrival on the stage's barrier, after the waits, lets the phase
// complete once the copies have landed: the compute warps' child gathers are
// ordered after the producers' releases (flag acquire, then the barrier). On a
// failed wait it lowers sy.stop to this iteration, arrives (so the copies it
// issued can complete), waits for them (bounded) and leaves.
template <class P>
__device__ void flow_stage(const FlowArgs<P>& a, unsigned char* fsm, FlowSync& sy, int w) {
    using V = typename P::V;
    const int lane = threadIdx.x & 31;
    const uint64_t first = l2_evict_first();
    int lvl_ok = -1;      // highest level k found finished (levels only grow)
    int last = -1;        // last iteration this warp issued
    auto drain = [&]() {
        if (lane == 0 && last >= 0) mbar_wait(&sy.full[w], (uint32_t)(last / kNS) & 1u, a);
        __syncwarp();
    };
    int it = w;
    for (int q = a.b_begin + (int)blockIdx.x + w * (int)gridDim.x; q < a.b_end; q += kNS * (int)gridDim.x, it += kNS) {
        const int b = __ldg(a.order + q);
        const int32_t fv = lane < (int)kFlowBlkInts ? __ldg(a.blk + (int64_t)b * kFlowBlkInts + lane) : 0;
        // every lane reads every field here: F is a full-warp shuffle, so it
        // is never called inside a lane-dependent branch
        auto F = [&](int i) { return __shfl_sync(0xffffffffu, fv, i); };
        const int k0 = F(FB_K0), doff = F(FB_DOFF), nd = F(FB_NDEP), pb = F(FB_PB), wl1 = F(FB_WL1);
        const int node0 = F(FB_NODE0), k1 = F(FB_K1), nn = F(FB_NNODES), slot0 = F(FB_SLOT0);
        const bool fin = b == a.final_block;
        // (ok is the same in every lane before each branch that holds a shuffle)
        bool ok = __all_sync(0xffffffffu, ld_volatile(&sy.stop) > it);
        // the stage is free once every compute warp has read its previous use
        // (this warp issued that use itself, so the phase is not ambiguous);
        // the final block takes every stage: every earlier block of the CTA
        // must have been published (so computed)
        if (lane == 0 && ok && it >= kNS) ok = mbar_wait(&sy.empty[w], (uint32_t)(it / kNS - 1) & 1u, a);
        if (lane == 0 && ok && fin) {
            const long long t0 = clock64();
            for (unsigned n = 0; ld_acquire_cta(&sy.pub) < it; ++n)
                if ((n & 63u) == 63u && (ld_volatile(&sy.stop) <= it || wait_give_up(a, t0))) {
                    ok = false;
                    break;
                }
        }
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicMin(&sy.stop, it);
            drain();
            return;
        }
        unsigned char* base = fin ? fsm : fsm + w * kSB;
        if (lane == 0) {
            FlowHead& h = sy.head[w];
            h.k0 = k0;
            h.k1 = k1;
            h.pb = pb;
            h.nn = nn;
            h.wl1 = wl1;
            if (!fin) {
                const int64_t nroots = a.lvl(LV_ROOTS, k0);
                h.nr = (int)(nroots - slot0 < 0 ? 0 : nroots - slot0 < nn ? nroots - slot0 : nn);
                h.out = (long long)(a.buf(k0) + slot0);
                h.rvo = (long long)(a.rv + a.TB + a.lvl(LV_ROFF, k0) + slot0);
                h.prev = (long long)a.buf(k0 + 2);   // level k0 - 1
            }
            fence_proxy_async_shared();   // earlier generic reads of the stage before the copies' writes
            mbar_expect_tx_only(&sy.full[w], (uint32_t)pb + (uint32_t)(fin ? wl1 * (int)sizeof(V) : 0));
            bulk_g2s_hint(base, a.pairs + node0, (uint32_t)pb, &sy.full[w], first);
        }
        last = it;
        if (a.waits) {
            for (int j = lane; j < nd && ok; j += 32) ok = wait_flag(a.flags + __ldg(a.deps + doff + j), a.epoch, a);
            if (lane == 0 && ok && !fin && k0 >= 3 && k0 - 2 > lvl_ok) {
                ok = wait_count(a.done + (k0 - 2), (unsigned long long)a.epoch * (unsigned long long)a.lvl(LV_NBLK, k0 - 2), a);
                if (ok) lvl_ok = k0 - 2;
            }
            lvl_ok = __shfl_sync(0xffffffffu, lvl_ok, 0);
        }
        __syncwarp();   // every lane's flag acquires before lane 0's arrival below
        const bool all_ok = __all_sync(0xffffffffu, ok);
        if (lane == 0) {
            if (!all_ok) atomicMin(&sy.stop, it);
            else if (fin && wl1 > 0) {
                fence_proxy_async_global();   // the producers' values (acquired above) before the copy reads them
                bulk_g2s(base + pb, a.buf(k0 + 2), (uint32_t)(wl1 * sizeof(V)), &sy.full[w]);
            }
            // (on a failed wait the final block's window is not copied: its
            // bytes stay expected, the phase never completes, and the drain
            // below gives up after its bounded wait with nothing in flight)
            mbar_arrive(&sy.full[w]);
        }
        if (!all_ok) {
            drain();
            return;
        }
    }
    drain();
}

// Lane 0 of a warp waits (bounded) for phase `parity` of bar, giving up when
// sy.stop says the stage will never be filled (stop_at: this block's
// iteration; -1: do not look at stop); the whole warp gets the answer.
template <class P>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const FlowSync& sy, int stop_at,
                                          long long limit, const FlowArgs<P>& a) {
    const int lane = threadIdx.x & 31;
    int ok = 1;
    if (lane == 0) {
        const long long t0 = clock64();
        for (unsigned n = 0;; ++n) {
            if (mbar_try_wait(bar, parity)) break;
            if ((n & 63u) == 63u) {
                if (stop_at >= 0 && ld_volatile(&sy.stop) <= stop_at) {
                    ok = 0;
                    break;
                }
                if (clock64() - t0 > limit) {
                    atomicCAS(a.status, 0, (int32_t)GC_ERR_TIMEOUT);
                    ok = 0;
                    break;
                }
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();   // orders the other lanes' reads after lane 0's acquire
    return ok != 0;
}

// The compute warps (16): evaluate this CTA's staged blocks in order. Each
// warp takes its share of a block's nodes, then reports -- an arrival on the
// stage's `empty` barrier (the staging warp may refill it) and a count in
// sy.done (the publishing warp may release the block) -- and moves on to the
// next staged block at once; warps of one CTA may be on different blocks.
// Only the final block's levels need the compute warps together, on cbar.
template <class P>
__device__ void flow_compute(const FlowArgs<P>& a, unsigned char* fsm, FlowSync& sy, int ct) {
    using V = typename P::V;
    constexpr int G = 16 / (int)sizeof(V);
    constexpr int U = 8;   // nodes a thread evaluates together (their child loads in flight at once)
    const int lane = (int)threadIdx.x & 31;
    const uint64_t keep = l2_evict_last();
    uint32_t cphase = 0;
    int it = 0;
    for (int q = a.b_begin + (int)blockIdx.x; q < a.b_end; q += (int)gridDim.x, ++it) {
        const int b = __ldg(a.order + q);
        const int s = it % kNS;
        if (!warp_wait(&sy.full[s], (uint32_t)(it / kNS) & 1u, sy, it, 4 * a.timeout, a)) return;
        const FlowHead& h = sy.head[s];
        const int k0 = h.k0, pb = h.pb;
        const bool fin = b == a.final_block;
        unsigned char* base = fin ? fsm : fsm + s * kSB;
        const int2* pr = reinterpret_cast<const int2*>(base);
        V* vals = reinterpret_cast<V*>(base + pb);
        auto child = [&](int32_t c) -> V {
            return c >= 0 ? vals[c] : c == -1 ? P::identity() : flow_leaf<P>(a, (uint32_t)(-2 - c));
        };
        if (!fin) {
            const int nn = h.nn, nr = h.nr;
            V* out = reinterpret_cast<V*>(h.out);
            V* rvo = reinterpret_cast<V*>(h.rvo);
            const V* prev = reinterpret_cast<const V*>(h.prev);
            // children: slots of level k0 - 1 in its level buffer (through L1/L2)
            auto gchild = [&](int32_t c) -> V {
                return c >= 0 ? prev[c] : c == -1 ? P::identity() : flow_leaf<P>(a, (uint32_t)(-2 - c));
            };
            for (int i0 = ct; i0 < nn; i0 += U * kFlowCT) {
                int2 c[U];
#pragma unroll
                for (int u = 0; u < U; ++u) c[u] = i0 + u * kFlowCT < nn ? pr[i0 + u * kFlowCT] : make_int2(-1, -1);
                V va[U], vb[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    va[u] = gchild(c[u].x);
                    vb[u] = gchild(c[u].y);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int i = i0 + u * kFlowCT;
                    if (i < nn) {
                        const V v = P::combine(va[u], vb[u]);
                        out[i] = v;
                        if (i < nr) st_keep(rvo + i, v, keep);
                    }
                }
            }
        } else {
            // levels k0..k1 one after the other; level k's values follow the
            // window (and the levels before it) in shared memory; between
            // levels every compute warp reports on cbar and waits for the rest
            const int k1 = h.k1;
            int own = h.wl1;
            const int64_t start0 = a.lvl(LV_START, k0);
            for (int k = k0; k <= k1; ++k) {
                const int w = (int)a.lvl(LV_W, k), nr = (int)a.lvl(LV_ROOTS, k);
                const int p0 = (int)(a.lvl(LV_START, k) - start0);
                V* rvo = a.rv + a.TB + a.lvl(LV_ROFF, k);
                for (int i = ct; i < w; i += kFlowCT) {
                    const int2 c = pr[p0 + i];
                    const V v = P::combine(child(c.x), child(c.y));
                    vals[own + i] = v;
                    if (i < nr) st_keep(rvo + i, v, keep);
                }
                own += (w + G - 1) / G * G;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sy.cbar);
                if (!warp_wait(&sy.cbar, cphase++ & 1u, sy, -1, a.timeout, a)) return;
            }
        }
        __syncwarp();   // the warp's reads and writes before lane 0's report
        if (lane == 0) {
            mbar_arrive(&sy.empty[s]);
            red_release_cta(&sy.done[s], 1);
        }
    }
}

// The publishing warp, one lane: releases this CTA's blocks in order once
// every compute warp has counted it done -- the block's ready flag (and its
// level's count) -- off the compute warps' path.
template <class P>
__device__ void flow_publish(const FlowArgs<P>& a, FlowSync& sy) {
    if ((threadIdx.x & 31) != 0) return;
    int it = 0;
    for (int q = a.b_begin + (int)blockIdx.x; q < a.b_end; q += (int)gridDim.x, ++it) {
        const int b = __ldg(a.order + q);
        const int s = it % kNS, want = kFlowCW * (it / kNS + 1);   // sy.done only grows
        const long long t0 = clock64();
        for (unsigned n = 0; ld_acquire_cta(&sy.done[s]) < want; ++n)
            if ((n & 63u) == 63u) {
                if (ld_volatile(&sy.stop) <= it) return;
                if (clock64() - t0 > 4 * a.timeout) {
                    atomicCAS(a.status, 0, (int32_t)GC_ERR_TIMEOUT);
                    return;
                }
            }
        // (test-only injection: CTA 0 never publishes its first block)
        if (!(a.inject == 1 && a.waits && blockIdx.x == 0 && it == 0)) {
            // one gpu-scope fence releases the block's values (ordered before
            // it by the compute warps' counts, acquired above) with both writes
            fence_acq_rel_gpu();
            st_relaxed_u32(a.flags + b, a.epoch);
            if (b != a.final_block) red_relaxed_add(a.done + __ldg(a.blk + (int64_t)b * kFlowBlkInts + FB_K0), 1ull);
        }
        st_release_cta(&sy.pub, it + 1);   // the final block's staging warp waits on it
    }
}

template <class P>
__global__ void __launch_bounds__(kFlowThreads, 1) flow_kernel(const FlowArgs<P> a) {
    using V = typename P::V;
    extern __shared__ __align__(128) unsigned char fsm[];
    __shared__ __align__(8) FlowSync sy;
    // an unread earlier timeout: do nothing
    if (ld_volatile(a.status) == (int32_t)GC_ERR_TIMEOUT) return;
    // a converged fixpoint loop skips the product; the level counters still
    // advance by the blocks of this launch, as if they had run, so that the
    // next product's waits stay consistent
    if (a.conv != nullptr && ld_volatile(a.conv) != 0) {
        if (blockIdx.x == 0 && a.waits) {
            for (int k = (int)threadIdx.x; k < a.L2; k += (int)blockDim.x) {
                const int64_t nb = k >= 1 && k < a.L2 - 1 ? a.lvl(LV_NBLK, k) : 0;
                if (nb > 0) red_add_release(a.done + k, (unsigned long long)nb);
            }
        } else if (blockIdx.x == 0 && threadIdx.x == 0 && a.b_end > a.b_begin) {
            const int b0 = __ldg(a.order + a.b_begin);   // a launch of one level's blocks
            if (b0 != a.final_block)
                red_add_release(a.done + __ldg(a.blk + (int64_t)b0 * kFlowBlkInts + FB_K0),
                                (unsigned long long)(a.b_end - a.b_begin));
        }
        return;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kNS; ++s) {
            mbar_init(&sy.full[s], 1);
            mbar_init(&sy.empty[s], kFlowCW);
            sy.done[s] = 0;
        }
        mbar_init(&sy.cbar, kFlowCW);
        sy.stop = 0x7fffffff;
        sy.pub = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // T[0] = identity, T[p+1] = V[l_p] (x) x[j_p] in front of RV (the emit's
    // terminals), grid-stride
    if (a.write_t) {
        const int64_t nt = (int64_t)gridDim.x * blockDim.x;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= a.alpha; i += nt)
            a.rv[i] = i == 0 ? P::identity() : flow_leaf<P>(a, (uint32_t)__ldg(a.leaf + (i - 1)));
    }
    __syncthreads();
    const int warp = (int)threadIdx.x >> 5;
    if (warp < kNS) flow_stage<P>(a, fsm, sy, warp);
    else if (warp < kNS + kFlowCW) flow_compute<P>(a, fsm, sy, (int)threadIdx.x - 32 * kNS);
    else flow_publish<P>(a, sy);
}

// ---------------------------------------------------------------- per-level schedule
template <class P, bool kC>
__global__ void __launch_bounds__(kThreads, 2) level_kernel(const SweepArgs<P> a, int k) {
    if (a.conv != nullptr && ld_volatile(a.conv) != 0) return;   // a converged fixpoint loop
    const int64_t GW = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const uint64_t keep = l2_evict_last();
    if (k <= 1) write_leaf_tables<P>(a, (int64_t)blockIdx.x * kThreads + threadIdx.x, (int64_t)gridDim.x * kThreads);
    if (k < 1) return;
    const int64_t nc = (a.lvl(LV_W, k) + Chunk<P>::NODES - 1) / Chunk<P>::NODES;
    const bool tail = k > a.grid_levels;
    const LevelIO<P> io = level_io<P>(a, k);
    const TailIO<P> tio = tail_io<P>(a, k, a.tbuf);
    int2 nab[Chunk<P>::U];
    if (gw < nc) load_chunk<P>(a, k, gw, nab);
    for (int64_t c = gw; c < nc; c += GW) {
        int2 ab[Chunk<P>::U];
#pragma unroll
        for (int u = 0; u < Chunk<P>::U; ++u) ab[u] = nab[u];
        if (c + GW < nc) load_chunk<P>(a, k, c + GW, nab);
        if (tail) combine_chunk<P, true, kC>(a, k, c, ab, tio.prev, tio.prev_tail, tio.cur, tio.rv, keep);
        else combine_chunk<P, false, kC>(a, k, c, ab, io.prev, nullptr, io.cur, io.rv, keep);
    }
    // level k-1 (a wide one) is complete and still in its buffer
    if (a.emode == EMIT_LEVEL && k >= 2) {
        if (k - 1 <= a.grid_levels) emit_level<P>(a, k - 1, io.prev, gw, GW);
        if (k == 2) emit_level<P>(a, 0, a.buf0, gw, GW);
    }
}

// phase 0: what is left of the level emit (level L when it is a wide one,
// terminals if L < 2), every chunk of the chunk emit, or the whole row emit;
// phase 1: the chunked emits' row sums
template <class P>
__global__ void __launch_bounds__(kThreads, 1) emit_kernel(const SweepArgs<P> a, int phase) {
    if (a.conv != nullptr && ld_volatile(a.conv) != 0) return;   // a converged fixpoint loop
    const int64_t GW = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (a.emode == EMIT_ROWS) {
        emit_rows<P>(a, blockIdx.x, gridDim.x);
    } else if (phase == 0) {
        if (a.L >= 1 && a.grid_levels == a.L) emit_level<P>(a, a.L, (a.L & 1) ? a.buf1 : a.buf0, gw, GW);
        if (a.L < 2) emit_level<P>(a, 0, a.buf0, gw, GW);
    } else {
        emit_final<P>(a, gw, GW);
    }
}

// x = x (+) y elementwise (OR for reachability, min for shortest paths);
// sets *changed if any element changed (one fixpoint step).
struct OrUpdate {
    using T = unsigned long long;
    using Pol = PolOr;
    __device__ __forceinline__ static T apply(T u, T v) { return u | v; }
};
struct MinUpdate {
    using T = float;
    using Pol = PolMinPlus;
    __device__ __forceinline__ static T apply(T u, T v) { return fminf(u, v); }
};

// One fixpoint step on rows a caller holds (a rank's share of a row-sharded
// fixpoint): x = x (+) y; *changed = 1 if any element changed (untouched
// otherwise: every writer stores the same value).
template <class U>
__global__ void __launch_bounds__(kThreads)
update_rows_kernel(typename U::T* __restrict__ x, const typename U::T* __restrict__ y, int64_t n,
                   int32_t* __restrict__ changed) {
    int ch = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const typename U::T u = x[i], v = U::apply(u, y[i]);
        if (v != u) {
            x[i] = v;
            ch = 1;
        }
    }
    if (__syncthreads_or(ch) && threadIdx.x == 0) *changed = 1;
}

// Fixpoint control words (in the status block): ctl[0] changed in this
// step, ctl[1] converged, ctl[2] CTAs of this step finished, ctl[3] the
// product count at convergence. With ctl[1] set every later step (and, in the
// dataflow products, every later product) does nothing.
// One step of a fixpoint loop that runs on without the host, x = x (+) y:
// the last CTA to finish reads the changed word; if nothing changed, the loop has converged
// at product `it` (recorded in ctl[3]); it then clears the step's words.
template <class U>
__global__ void __launch_bounds__(kThreads)
update_loop_kernel(typename U::T* __restrict__ x, const typename U::T* __restrict__ y, int64_t n,
                   int32_t* __restrict__ ctl, int32_t it, int32_t max_it, int32_t* __restrict__ status) {
    __shared__ int s_last;
    if (ld_volatile(ctl + 1) != 0) return;   // converged at an earlier step
    // a product that timed out wrote no y: no step, no convergence (the loop
    // runs out at max_it and the status word keeps the timeout)
    if (ld_volatile(status) == (int32_t)GC_ERR_TIMEOUT) return;
    int ch = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const typename U::T u = x[i], v = U::apply(u, y[i]);
        if (v != u) {
            x[i] = v;
            ch = 1;
        }
    }
    const int any = __syncthreads_or(ch);
    if (threadIdx.x == 0) {
        if (any) atomicOr(ctl, 1);
        __threadfence();
        s_last = atomicAdd(ctl + 2, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (s_last && threadIdx.x == 0) {
        __threadfence();
        if (ld_volatile(ctl) == 0) {
            ctl[3] = it;
            ctl[1] = 1;
        } else if (it == max_it) {
            atomicCAS(status, 0, (int32_t)GC_ERR_NOT_CONVERGED);
        }
        ctl[0] = 0;
        ctl[2] = 0;
        __threadfence();
    }
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
    a.L2 = (int32_t)h->L + 2;   // row stride of the level table
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
    a.echunk = reinterpret_cast<const int4*>(ar + d.echunk);
    a.cref = reinterpret_cast<const int32_t*>(ar + d.cref);
    a.row_ech = reinterpret_cast<const int32_t*>(ar + d.row_ech);
    a.sref = reinterpret_cast<const uint4*>(ar + d.sref);
    a.sflag = reinterpret_cast<const uint8_t*>(ar + d.sflag);
    a.tile_sid = reinterpret_cast<const int32_t*>(ar + d.tile_sid);
    a.row_pos = d.emit == EMIT_SLICE ? reinterpret_cast<const int32_t*>(ar + d.row_pos) : nullptr;
    a.sx0 = reinterpret_cast<const int32_t*>(ar + d.sx0);
    a.stile = reinterpret_cast<const int32_t*>(ar + d.stile);
    a.sorder = reinterpret_cast<const int32_t*>(ar + d.sorder);
    a.slice = d.slice;
    a.nslices = d.n_slices;
    a.late_off = reinterpret_cast<const int32_t*>(ar + d.late_off);
    a.late_ref = reinterpret_cast<const int32_t*>(ar + d.late_ref);
    a.esum = reinterpret_cast<V*>(ar + d.esum);
    a.tbuf = reinterpret_cast<V*>(ar + d.tbuf);
    a.carry = reinterpret_cast<V*>(ar + d.carry);
    a.tail_total = d.tail_total;
    a.n = h->n;
    a.emode = d.emit;
    a.emit_group = h->emit_group;
    a.status = reinterpret_cast<int32_t*>(ar + d.status);
    a.bar = reinterpret_cast<unsigned long long*>(ar + d.status + 64);
    a.tbar = reinterpret_cast<unsigned long long*>(ar + d.status + 128);
    a.tbar_base = h->tbar_base;
    a.bar_base = h->bar_base;
    a.timeout = h->timeout_cycles;
    a.inject = h->inject;
    a.conv = h->conv;
    a.tail_group = 1;
    a.tail_solo = h->L + 1;
    return a;
}

// CTAs the persistent kernel can keep resident (at most two per SM; 0 if none)
template <class P, bool kC>
int sweep_grid(const gc_handle* h) {
    int per_sm = 0;
    cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sweep_kernel<P, kC>, kThreads, 0),
               "sweep occupancy");
    return std::min(per_sm, 2) * h->sms;
}

// Grid barriers one CTA of the persistent sweep passes: one per level after
// the first, then (unless the slice kernel takes over) one before the tail and
// one before the row pass.
int64_t sweep_barriers(const gc_handle* h) {
    return std::max(h->grid_levels - 1, 0) + (h->lay.emit == EMIT_SLICE ? 0 : 2);
}

// Shared memory of the slice kernel: one slice of values.
template <class P>
int64_t slice_smem(const gc_handle* h) {
    return h->lay.slice * (int64_t)sizeof(typename P::V);
}

// CTAs of the cooperative slice kernel (one per SM; 0 if it cannot be resident).
template <class P, bool kC>
int slice_grid(const gc_handle* h) {
    const int64_t smem = slice_smem<P>(h);
    cuda_check(cudaFuncSetAttribute((const void*)slice_kernel<P, kC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem),
               "slice shared memory");
    int per_sm = 0;
    cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, slice_kernel<P, kC>, kSliceThreads, (size_t)smem),
               "slice occupancy");
    return per_sm >= 1 ? h->sms : 0;
}

// Enqueues one product with the arguments in a (persistent kernels when the
// device allows, else one kernel per level). Returns the launch count and
// adds the grid-barrier arrivals of the cooperative launches to *arrivals;
// a.bar_base is the barrier counter's value when the first launch starts.
template <class P, bool kC>
int64_t launch_product_as(const gc_handle* h, SweepArgs<P>& a, cudaStream_t st, unsigned long long* arrivals,
                          unsigned long long* tail_arrivals) {
    const bool slice = h->lay.emit == EMIT_SLICE;
    // the slice emit (k_max = 1 handles) serves one-lane values only
    if (slice && !kScalarPolicy<P>) fail(GC_ERR_ARG, "a multi-vector product on a one-vector handle");
    int grid = 0, grid2 = 0;
    if (h->schedule == 0 && h->coop) {
        grid = sweep_grid<P, kC>(h);
        if constexpr (kScalarPolicy<P>)
            if (slice && grid > 0) grid2 = slice_grid<P, kC>(h);
        if (slice && grid2 == 0) grid = 0;
    }
    int64_t launches = 0;
    *arrivals = 0;
    *tail_arrivals = 0;
    if (grid > 0) {
        void* args[] = {&a};
        cuda_check(cudaLaunchCooperativeKernel((const void*)sweep_kernel<P, kC>, dim3(grid), dim3(kThreads), args, 0, st),
                   "sweep launch");
        launches = 1;
        *arrivals = (unsigned long long)sweep_barriers(h) * (unsigned long long)grid;
        if constexpr (kScalarPolicy<P>) if (slice) {
            SweepArgs<P> b = a;
            b.bar_base = a.bar_base + *arrivals;
            b.tail_group = std::min(kTailGroup, grid2);
            // the top levels of at most one chunk per warp of a CTA run on CTA 0 alone
            const int64_t solo_nodes = (int64_t)Chunk<P>::NODES * (kSliceThreads / 32);
            int ks = h->L + 1;
            while (ks - 1 > h->grid_levels && h->lv[LV_W * (h->L + 2) + ks - 1] <= solo_nodes) --ks;
            b.tail_solo = ks;
            if (ks == h->grid_levels + 1) b.tail_group = 1;
            int coop = 1;
            void* args2[] = {&b, &coop};
            cuda_check(cudaLaunchCooperativeKernel((const void*)slice_kernel<P, kC>, dim3(grid2), dim3(kSliceThreads),
                                                   args2, (size_t)slice_smem<P>(h), st),
                       "slice launch");
            ++launches;
            *arrivals += (unsigned long long)grid2;
            if (b.tail_group > 1 && h->L > h->grid_levels)   // group barriers before tail levels Lg+2 .. min(ks, L)
                *tail_arrivals = (unsigned long long)(std::min<int64_t>(b.tail_solo, h->L) - h->grid_levels - 1) *
                                 (unsigned long long)b.tail_group;
        }
    } else {
        // level 1 also writes the leaf tables; with no levels a table-only launch
        const int64_t w1 = h->L >= 1 ? h->lv[LV_W * (h->L + 2) + 1] : 0;
        const int64_t items = std::max<int64_t>(w1, (h->alpha + 1) * P::LPN);
        level_kernel<P, kC><<<grid_for(items, Chunk<P>::NODES * kWarps, h->sms), kThreads, 0, st>>>(a, h->L >= 1 ? 1 : 0);
        ++launches;
        for (int k = 2; k <= h->L; ++k) {
            const int64_t w = h->lv[LV_W * (h->L + 2) + k];
            level_kernel<P, kC><<<grid_for(w, Chunk<P>::NODES * kWarps, h->sms), kThreads, 0, st>>>(a, k);
            ++launches;
        }
        if (h->n > 0 && h->lay.emit == EMIT_ROWS) {
            emit_kernel<P><<<grid_for(h->n, kWarps * (32 / h->emit_group), h->sms, 4), kThreads, 0, st>>>(a, 0);
            ++launches;
        } else if (h->n > 0) {
            if constexpr (kScalarPolicy<P>) if (slice) {
                const int64_t smem = slice_smem<P>(h);
                cuda_check(cudaFuncSetAttribute((const void*)slice_kernel<P, kC>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                           "slice shared memory");
                const int g2 = (int)std::max<int64_t>(1, std::min<int64_t>(h->lay.n_slices, h->sms));
                slice_kernel<P, kC><<<g2, kSliceThreads, (size_t)smem, st>>>(a, 0);
            }
            if (!slice) emit_kernel<P><<<grid_for(h->lay.n_echunks, kWarps, h->sms, 4), kThreads, 0, st>>>(a, 0);
            emit_kernel<P><<<grid_for(h->n, kWarps, h->sms, 4), kThreads, 0, st>>>(a, 1);
            launches += 2;
        }
    }
    cuda_check(cudaGetLastError(), "kernel launch");
    return launches;
}

// Scratch of a dataflow product: the three level buffers, the ready flags
// and level counters, and the product number they are stamped with.
struct FlowScratch {
    char* fb0;
    char* fb1;
    char* fb2;
    int32_t* flags;
    unsigned long long* done;
    uint32_t epoch;
};

template <class P>
FlowArgs<P> make_flow_args(const gc_handle* h, const SweepArgs<P>& a, const FlowScratch& fs) {
    using V = typename P::V;
    const DevLayout& d = h->lay;
    char* ar = h->arena;
    FlowArgs<P> f{};
    f.pairs = reinterpret_cast<const int2*>(ar + d.nodes);
    f.blk = reinterpret_cast<const int32_t*>(ar + d.fblk);
    f.order = reinterpret_cast<const int32_t*>(ar + d.forder);
    f.deps = reinterpret_cast<const int32_t*>(ar + d.fdeps);
    f.gran = reinterpret_cast<const int32_t*>(ar + d.fgran);
    f.lv = a.lv;
    f.L2 = a.L2;
    f.final_block = h->final_k0 <= h->L ? (int32_t)(h->nblocks - 1) : -1;
    f.TB = a.TB;
    f.alpha = a.alpha;
    f.Vd = a.Vd;
    f.leaf = a.leaf;
    f.vbits = a.vbits;
    f.x = a.x;
    f.rv = a.rv;
    f.fb0 = reinterpret_cast<V*>(fs.fb0);
    f.fb1 = reinterpret_cast<V*>(fs.fb1);
    f.fb2 = reinterpret_cast<V*>(fs.fb2);
    f.flags = fs.flags;
    f.done = fs.done;
    f.epoch = fs.epoch;
    f.status = a.status;
    f.timeout = a.timeout;
    f.inject = a.inject;
    f.conv = a.conv;
    f.nblocks = (int32_t)h->nblocks;
    return f;
}

// One dataflow product: the sweep (one cooperative launch, or one launch per
// level without waits for the per-level schedule), then the emit from RV
// (slice emit with its row pass, or the row emit).
template <class P>
int64_t launch_flow(const gc_handle* h, SweepArgs<P>& a, const FlowScratch& fs, cudaStream_t st,
                    unsigned long long* arrivals) {
    FlowArgs<P> f = make_flow_args<P>(h, a, fs);
    const size_t smem = (size_t)kNS * kSB;
    cuda_check(cudaFuncSetAttribute((const void*)flow_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
               "dataflow shared memory");
    int64_t launches = 0;
    *arrivals = 0;
    int grid = 0;
    if (h->schedule != GC_SCHED_PER_LEVEL && h->coop) {
        int per_sm = 0;
        cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, flow_kernel<P>, kFlowThreads, smem),
                   "dataflow occupancy");
        grid = per_sm >= 1 ? h->sms : 0;
    }
    if (grid > 0) {
        f.b_begin = 0;
        f.b_end = (int32_t)h->nblocks;
        f.waits = 1;
        f.write_t = 1;
        void* args[] = {&f};
        cuda_check(cudaLaunchCooperativeKernel((const void*)flow_kernel<P>, dim3(grid), dim3(kFlowThreads), args, smem, st),
                   "dataflow launch");
        launches = 1;
    } else {
        // Listing 1's order: one launch per level (the final block last);
        // the launches order the levels, so nothing waits
        f.waits = 0;
        f.write_t = 1;
        auto one = [&](int64_t b0, int64_t b1) {
            f.b_begin = (int32_t)b0;
            f.b_end = (int32_t)b1;
            const int g = (int)std::max<int64_t>(1, std::min<int64_t>(b1 - b0, (int64_t)h->sms));
            flow_kernel<P><<<g, kFlowThreads, smem, st>>>(f);
            f.write_t = 0;
            ++launches;
        };
        const int64_t kreg = std::min<int64_t>(h->final_k0, h->L + 1);   // first level without regular blocks
        for (int64_t k = 1; k < kreg; ++k)
            if (h->lvl_blk[k + 1] > h->lvl_blk[k]) one(h->lvl_blk[k], h->lvl_blk[k + 1]);
        if (h->final_k0 <= h->L) one(h->nblocks - 1, h->nblocks);
        if (launches == 0) one(0, 0);   // no levels: the leaf table only
    }
    if (h->n > 0) {
        if (h->lay.emit == EMIT_SLICE) {
            if constexpr (kScalarPolicy<P>) {
                const int grid2 = grid > 0 ? slice_grid<P, false>(h) : 0;
                a.tail_group = 1;
                a.tail_solo = h->L + 1;
                if (grid2 > 0) {
                    int coop = 1;
                    void* args2[] = {&a, &coop};
                    cuda_check(cudaLaunchCooperativeKernel((const void*)slice_kernel<P, false>, dim3(grid2),
                                                           dim3(kSliceThreads), args2, (size_t)slice_smem<P>(h), st),
                               "slice launch");
                    *arrivals = (unsigned long long)grid2;
                    ++launches;
                } else {
                    const int64_t ss = slice_smem<P>(h);
                    cuda_check(cudaFuncSetAttribute((const void*)slice_kernel<P, false>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ss),
                               "slice shared memory");
                    const int g2 = (int)std::max<int64_t>(1, std::min<int64_t>(h->lay.n_slices, h->sms));
                    slice_kernel<P, false><<<g2, kSliceThreads, (size_t)ss, st>>>(a, 0);
                    emit_kernel<P><<<grid_for(h->n, kWarps, h->sms, 4), kThreads, 0, st>>>(a, 1);
                    launches += 2;
                }
            }
        } else {
            emit_kernel<P><<<grid_for(h->n, kWarps * (32 / h->emit_group), h->sms, 4), kThreads, 0, st>>>(a, 0);
            ++launches;
        }
    }
    cuda_check(cudaGetLastError(), "kernel launch");
    return launches;
}

// Carry slots exist only for the device view of 16-wide handles (the float32
// policies); the other policies are built without them. Handles with one
// value a node run the dataflow sweep (fs: its scratch).
template <class P>
int64_t launch_product(const gc_handle* h, SweepArgs<P>& a, cudaStream_t st, unsigned long long* arrivals,
                       unsigned long long* tail_arrivals, const FlowScratch* fs) {
    if (h->flow) {
        *tail_arrivals = 0;
        if constexpr (kScalarPolicy<P>) return launch_flow<P>(h, a, *fs, st, arrivals);
        fail(GC_ERR_ARG, "a multi-vector product on a one-vector handle");
    }
    if constexpr (std::is_same<typename P::Leaf, float>::value)
        if (h->n_carry > 0) return launch_product_as<P, true>(h, a, st, arrivals, tail_arrivals);
    if (h->n_carry > 0) fail(GC_ERR_UNSUPPORTED, "carry slots for a policy built without them");
    return launch_product_as<P, false>(h, a, st, arrivals, tail_arrivals);
}

template <class P>
void run_product(gc_handle* h, const void* x, void* y, cudaStream_t st) {
    SweepArgs<P> a = make_args<P>(h, x, y);
    unsigned long long arrivals = 0, tail_arrivals = 0;
    FlowScratch fs{};
    if (h->flow) {
        const DevLayout& d = h->lay;
        fs.fb0 = h->arena + d.fb0;
        fs.fb1 = h->arena + d.fb1;
        fs.fb2 = h->arena + d.fb2;
        fs.flags = reinterpret_cast<int32_t*>(h->arena + d.fflags);
        fs.done = reinterpret_cast<unsigned long long*>(h->arena + d.fdone);
        if (++h->epoch == 0) ++h->epoch;   // flags start at 0: never stamp 0
        fs.epoch = h->epoch;
    }
    h->launches = launch_product<P>(h, a, st, &arrivals, &tail_arrivals, h->flow ? &fs : nullptr);
    h->bar_base += arrivals;
    h->tbar_base += tail_arrivals;
}

// The float32 sum at k right-hand sides (k one of kF32Widths; checked before).
template <template <class> class Run, class... Args>
void for_f32_width(int32_t k, Args&&... args) {
    switch (k) {
        case 1: Run<PolF32>::go(args...); break;
        case 4: Run<PolF32xN<1>>::go(args...); break;
        case 8: Run<PolF32xN<2>>::go(args...); break;
        case 16: Run<PolF32xN<4>>::go(args...); break;
        case 32: Run<PolF32xN<8>>::go(args...); break;
        case 64: Run<PolF32xN<16>>::go(args...); break;
        case 128: Run<PolF32xN<32>>::go(args...); break;
        case 256: Run<PolF32x256>::go(args...); break;
        default: fail(GC_ERR_ARG, "unsupported k");
    }
}
template <class P>
struct RunProduct {
    static void go(gc_handle* h, const void* x, void* y, cudaStream_t st) { run_product<P>(h, x, y, st); }
};

void dispatch_product(gc_handle* h, const void* x, void* y, int32_t k, cudaStream_t st) {
    switch (h->policy) {
        case GC_F32_SUM: for_f32_width<RunProduct>(k, h, x, y, st); break;
        case GC_I64_SUM: run_product<PolI64>(h, x, y, st); break;
        case GC_BOOL_OR: run_product<PolOr>(h, x, y, st); break;
        case GC_F32_MIN_PLUS:
            if (k == 1) run_product<PolMinPlus>(h, x, y, st);
            else run_product<PolMinPlusx16>(h, x, y, st);
            break;
    }
}

// k: a width the policy supports (policy_width_ok), at most the handle's
// k_max (its buffers hold k_max values a node).
void check_k(const gc_handle* h, int32_t k) {
    if (!policy_width_ok(h->policy, k)) fail(GC_ERR_ARG, "k is not a width this policy supports");
    if (k > h->k_max) fail(GC_ERR_ARG, "k exceeds the k_max the handle was uploaded with");
}

// Products run on the current device; the handle's arena (and the fixed
// scratch picked for the current device) must be on that same device.
void check_device(const gc_handle* h) {
    int dev = 0;
    cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (dev != h->device)
        fail(GC_ERR_ARG, "the current device (" + std::to_string(dev) + ") is not the device the handle was uploaded on (" +
                             std::to_string(h->device) + ")");
}

template <class T>
void put(cudaStream_t st, char* arena, int64_t off, const T* p, size_t count) {
    if (count == 0) return;
    cuda_check(cudaMemcpyAsync(arena + off, p, count * sizeof(T), cudaMemcpyHostToDevice, st), "upload copy");
}

// x <- x (+) (M (x) x) from x0 until nothing changes, at most max_iter
// products; the product's y lives in the arena's staging area. Handles whose
// product is the persistent sweep alone run it in one launch
// (fused_fixpoint). Otherwise the loop runs on the device (drive_fixpoint):
// products and update steps are enqueued in batches of 1, 2, 4, 8, 8, ...,
// one batch ahead of the one the host waits for; the update step's last CTA
// records convergence (ctl, in the status block) and every kernel enqueued
// after it returns at once, keeping the barrier counters and level counters
// consistent. Writes the product count (or -1) to iters on the device.
// Returns false if max_iter was reached first (the status word then says
// GC_ERR_NOT_CONVERGED, unless a barrier timed out: GC_ERR_TIMEOUT).
// The whole fixpoint as one launch of the persistent sweep (sweep_fixpoint):
// for handles whose product is that kernel alone (persistent schedule, no
// slice kernel, no dataflow layout). Sets *result to the product count (or
// -1) and returns whether it converged; synchronises the stream.
template <class P, bool kC>
bool fused_fixpoint(gc_handle* h, typename P::V* x, int32_t max_iter, int32_t* result, cudaStream_t st) {
    int32_t* status = reinterpret_cast<int32_t*>(h->arena + h->lay.status);
    int32_t* fix = status + 8;   // bytes 32..47 of the status block
    const int grid = sweep_grid<P, kC>(h);
    if (!h->loop.words) {
        void* p = nullptr;
        cuda_check(cudaHostAlloc(&p, 8 * sizeof(int32_t), cudaHostAllocDefault), "loop words (pinned)");
        h->loop.words = static_cast<int32_t*>(p);
    }
    cuda_check(cudaMemsetAsync(fix, 0, 4 * sizeof(int32_t), st), "fixpoint words clear");
    SweepArgs<P> a = make_args<P>(h, x, h->arena + h->lay.ys);
    a.fix = fix;
    a.fix_max = max_iter;
    a.conv = nullptr;
    void* args[] = {&a};
    cuda_check(cudaLaunchCooperativeKernel((const void*)sweep_kernel<P, kC>, dim3(grid), dim3(kThreads), args, 0, st),
               "fixpoint launch");
    h->launches = 1;
    int32_t* w = h->loop.words;   // status word, then the fixpoint's four
    cuda_check(cudaMemcpyAsync(w, status, sizeof(int32_t), cudaMemcpyDeviceToHost, st), "status read");
    cuda_check(cudaMemcpyAsync(w + 4, fix, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, st), "fixpoint words read");
    cuda_check(cudaStreamSynchronize(st), "stream synchronize");
    const bool done = w[0] == 0 && w[6] != 0;
    *result = done ? w[7] : -1;
    // the launch's grid barriers: sweep_barriers + 2 a product (sweep_fixpoint; a timed-out
    // launch leaves the counter part-way; gc_check restarts it)
    const int64_t products = done ? w[7] : max_iter;
    if (w[0] == 0)
        h->bar_base += (unsigned long long)products *
                       (unsigned long long)(sweep_barriers(h) + 2) *
                       (unsigned long long)grid;
    return done;
}

template <class P>
bool fused_fixpoint_ok(const gc_handle* h) {
    if (h->schedule != 0 || !h->coop || h->flow || h->lay.emit == EMIT_SLICE) return false;
    if (h->n_carry > 0) return false;
    return sweep_grid<P, false>(h) > 0;
}

template <class U>
bool run_fixpoint(gc_handle* h, const typename U::T* x0, typename U::T* x, int32_t max_iter, int32_t* iters,
                  cudaStream_t st) {
    using T = typename U::T;
    const int64_t n = h->n;
    T* yv = reinterpret_cast<T*>(h->arena + h->lay.ys);
    int32_t* status = reinterpret_cast<int32_t*>(h->arena + h->lay.status);
    int32_t* ctl = status + 4;   // changed, converged, CTAs done, product count (bytes 16..31)
    after_last_loop(h->loop, st, cuda_check);
    if (x != x0 && n > 0)
        cuda_check(cudaMemcpyAsync(x, x0, n * sizeof(T), cudaMemcpyDeviceToDevice, st), "x0 copy");
    if (fused_fixpoint_ok<typename U::Pol>(h)) {
        int32_t result = -1;
        const bool done = fused_fixpoint<typename U::Pol, false>(h, x, max_iter, &result, st);
        cuda_check(cudaMemcpyAsync(iters, &result, 4, cudaMemcpyHostToDevice, st), "iters write");
        if (!done && h->loop.words[0] == 0) {
            int32_t sw = GC_ERR_NOT_CONVERGED;
            cuda_check(cudaMemcpyAsync(status, &sw, 4, cudaMemcpyHostToDevice, st), "status write");
        }
        return done;
    }
    cuda_check(cudaMemsetAsync(ctl, 0, 16, st), "loop words clear");
    int32_t result = -1;
    int64_t launches = 0;
    h->conv = ctl + 1;
    bool done = false;
    try {
        done = drive_fixpoint(h->loop, ctl, max_iter, st, cuda_check, [&](int32_t it) {
            dispatch_product(h, x, yv, 1, st);
            launches += h->launches;
            update_loop_kernel<U><<<grid_for(n, kThreads, h->sms, 8), kThreads, 0, st>>>(x, yv, n, ctl, it, max_iter,
                                                                                         status);
            ++launches;
        }, &result);
    } catch (...) {
        h->conv = nullptr;
        if (h->loop.end && cudaEventRecord(h->loop.end, st) == cudaSuccess) h->loop.ended = true;
        throw;
    }
    h->conv = nullptr;
    h->launches = launches;
    // a pageable source: the copy takes its value before it returns (the
    // last update step records GC_ERR_NOT_CONVERGED in the status word)
    cuda_check(cudaMemcpyAsync(iters, &result, 4, cudaMemcpyHostToDevice, st), "iters write");
    mark_loop_end(h->loop, st, cuda_check);
    return done;
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

// Offsets of the scratch parts inside the fixed array for a product with k
// right-hand sides, in the arena's order: buffers, tail buffers, level-emit
// sums or RV, then the status block.
struct StaticParts {
    int64_t buf0, buf1, esum, tbuf, carry, rv, status, total;
    int64_t fb0, fb1, fb2, fflags, fdone;   // dataflow handles
};
StaticParts static_parts(const gc_handle* h, int32_t k) {
    const DevLayout& d = h->lay;
    const int64_t vb = policy_elem_bytes(h->policy) * k;
    StaticParts s{};
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = o;
        o = align256(o + bytes);
        return at;
    };
    if (h->flow) {
        // the three level buffers, RV and the emit's sums, then the flags,
        // level counters and status block back to back (cleared by every call)
        s.fb0 = take(vb * d.fbuf_values);
        s.fb1 = take(vb * d.fbuf_values);
        s.fb2 = take(vb * d.fbuf_values);
        if (d.chunked()) s.esum = take(vb * d.n_esum);
        if (d.has_rv()) s.rv = take(vb * (d.TB + h->n_roots));
        s.fflags = take(4 * std::max<int64_t>(1, h->nblocks));
        s.fdone = take(8 * (h->L + 2));
        s.status = take(256);
        s.total = o;
        return s;
    }
    s.buf0 = take(vb * std::max<int64_t>(1, h->max_width));
    s.buf1 = take(vb * std::max<int64_t>(1, h->max_width));
    s.tbuf = take(vb * d.tail_total);
    s.carry = take(vb * std::max<int64_t>(1, h->n_carry));
    if (d.chunked()) s.esum = take(vb * d.n_esum);
    if (d.has_rv()) s.rv = take(vb * (d.TB + h->n_roots));
    s.status = take(256);
    s.total = o;
    return s;
}

int64_t static_scratch_need(const gc_handle* h, int32_t k) { return static_parts(h, k).total; }

// One product whose scratch is the fixed array: the same kernels and order of
// evaluation as gc_matvec, with the level buffers, emit sums or RV, status
// word and barrier counter pointed into g_static_scratch.
template <class P>
void run_product_static(gc_handle* h, const void* x, void* y, cudaStream_t st, unsigned char* scratch) {
    using V = typename P::V;
    SweepArgs<P> a = make_args<P>(h, x, y);
    const StaticParts sp = static_parts(h, P::LPN * (int32_t)(sizeof(V) / policy_elem_bytes(h->policy)));
    a.buf0 = reinterpret_cast<V*>(scratch + sp.buf0);
    a.buf1 = reinterpret_cast<V*>(scratch + sp.buf1);
    a.esum = reinterpret_cast<V*>(scratch + sp.esum);
    a.tbuf = reinterpret_cast<V*>(scratch + sp.tbuf);
    a.carry = reinterpret_cast<V*>(scratch + sp.carry);
    a.rv = reinterpret_cast<V*>(scratch + sp.rv);
    a.status = reinterpret_cast<int32_t*>(scratch + sp.status);
    a.bar = reinterpret_cast<unsigned long long*>(scratch + sp.status + 64);
    a.bar_base = 0;
    a.tbar = reinterpret_cast<unsigned long long*>(scratch + sp.status + 128);
    a.tbar_base = 0;
    a.inject = 0;
    // the array keeps the previous call's contents: start from a clear status
    // word and barrier counter (and, for the dataflow sweep, clear ready
    // flags and level counters, with product number 1)
    FlowScratch fs{};
    if (h->flow) {
        fs.fb0 = reinterpret_cast<char*>(scratch + sp.fb0);
        fs.fb1 = reinterpret_cast<char*>(scratch + sp.fb1);
        fs.fb2 = reinterpret_cast<char*>(scratch + sp.fb2);
        fs.flags = reinterpret_cast<int32_t*>(scratch + sp.fflags);
        fs.done = reinterpret_cast<unsigned long long*>(scratch + sp.fdone);
        fs.epoch = 1;
        cuda_check(cudaMemsetAsync(scratch + sp.fflags, 0, (size_t)(sp.total - sp.fflags), st), "fixed scratch clear");
    } else {
        cuda_check(cudaMemsetAsync(scratch + sp.status, 0, 256, st), "fixed scratch clear");
    }
    unsigned long long arrivals = 0, tail_arrivals = 0;
    h->launches = launch_product<P>(h, a, st, &arrivals, &tail_arrivals, h->flow ? &fs : nullptr);
}

template <class P>
struct RunStatic {
    static void go(gc_handle* h, const void* x, void* y, cudaStream_t st, unsigned char* scratch) {
        run_product_static<P>(h, x, y, st, scratch);
    }
};

}  // namespace
}  // namespace gcs

using namespace gcs;

extern "C" {

gc_status gc_upload_ex(const gc_grammar* gg, gc_policy policy, int32_t k_max, int32_t schedule, void* arena,
                       int64_t arena_bytes, void* stream, gc_handle** out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null grammar or output pointer");
        if (!arena) fail(GC_ERR_ARG, "null arena");
        if (reinterpret_cast<uintptr_t>(arena) % 256 != 0) fail(GC_ERR_ARG, "arena must be 256-byte aligned");
        check_policy(gg->g, policy, k_max);
        validate_packed(gg->g);
        // one value a node: the dataflow sweep over the layered grammar itself;
        // wider values: the device view (carry slots for the level emit)
        const bool flow = wants_flow(schedule, k_max);
        std::shared_ptr<const FlowPlan> fp;
        FlowCounts fc;
        Grammar view;
        if (flow) {
            fp = flow_plan_for(gg, policy_elem_bytes(policy));
            validate_flow_plan(*fp, gg->g);
            fc = flow_counts(*fp);
        } else {
            view = device_view(gg->g, emit_mode(gg->g, k_max) == EMIT_LEVEL);   // carry slots for 16-wide values
            validate_device_view(view);
        }
        const Grammar& g = flow ? gg->g : view;
        const DevLayout d = device_layout(g, policy, k_max, flow ? &fc : nullptr);
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
        h->n_carry = g.n_carry;
        h->arena = static_cast<char*>(arena);
        h->lay = d;
        h->flow = flow;
        if (flow) {
            h->nblocks = fp->nblocks;
            h->final_k0 = fp->final_k0;
            h->lvl_blk = fp->lvl_blk;
            h->schedule = GC_SCHED_DATAFLOW;
        } else if (schedule == GC_SCHED_PER_LEVEL) {
            h->schedule = GC_SCHED_PER_LEVEL;
        }
        // row emit (rows average < 128 symbols): G lanes per row, so that a
        // lane loads about one batch of a row's symbols (4 one-lane values, 2
        // four-lane ones) and a warp reduces 32 / G rows at a time
        const double avg = g.n > 0 ? (double)h->c_len / (double)g.n : 0.0;
        const int batch = k_max == 1 ? 4 : 2;
        int G = 1;
        while (G < 32 && G * batch < avg) G <<= 1;
        h->emit_group = d.emit == EMIT_ROWS ? G : 0;
        // levels narrow enough for one CTA finish the sweep there (when two or more)
        const int64_t L = g.L;
        h->grid_levels = (int)d.grid_levels;
        const std::vector<int64_t> toff = tail_offsets(g, d.grid_levels);

        // level table; node children as slots of the level below, the identity (-1), terminals as
        // -2 - leaf code, or carry slots
        auto leaf_code = [&](int32_t p) { return (int32_t)(((int64_t)g.term_col[p] << d.vbits) | g.term_vidx[p]); };
        const int64_t A = g.alpha();
        auto ref = [&](int32_t c) -> int32_t {   // device-view reference -> device index
            if (c >= 0) return c;                   // slot of the level below
            if (c == -1) return -1;                 // identity
            if (c >= -(A + 1)) return -2 - leaf_code(-c - 2);   // terminal p = -c-2, by its leaf code
            return kCarryBase + (int32_t)carry_slot(c, A);
        };
        h->lv.assign((size_t)(LV_ROWS * (L + 2)), 0);
        std::vector<int32_t> nodes;
        if (flow) nodes = fp->pairs;
        else nodes.assign((size_t)(2 * d.n_nodes_padded), 0);
        int64_t start = 0;
        for (int64_t k = 1; k <= L; ++k) {
            const int64_t w = g.lvl_off[k + 1] - g.lvl_off[k];
            h->lv[LV_START * (L + 2) + k] = start;
            h->lv[LV_W * (L + 2) + k] = w;
            h->lv[LV_ROOTS * (L + 2) + k] = g.lvl_roots[k];
            h->lv[LV_ROFF * (L + 2) + k] = g.root_off[k];
            h->lv[LV_TOFF * (L + 2) + k] = toff[k];
            if (flow) {
                h->lv[LV_NBLK * (L + 2) + k] = k < fp->final_k0 ? fp->lvl_blk[k + 1] - fp->lvl_blk[k] : 0;
                start += pad_nodes(w);
                continue;   // the plan's block-local references are the node array
            }
            h->lv[LV_CR * (L + 2) + k] = g.carry_roots[k];
            h->lv[LV_CN * (L + 2) + k] = g.carry_rest[k];
            h->lv[LV_COFF * (L + 2) + k] = g.carry_off[k];
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
        EmitPlan plan;
        SlicePlan sp;
        std::vector<int32_t> cref, co;
        if (d.emit == EMIT_LEVEL) {
            plan = plan_level_emit(g, d.grid_levels);
            if ((int64_t)plan.echunk.size() != 4 * d.n_echunks || (int64_t)plan.late_ref.size() != d.n_late ||
                (int64_t)plan.cref.size() != d.n_early)
                fail(GC_ERR_INVALID_GRAMMAR, "emit plan does not match the layout");
            validate_emit_plan(plan, g, d.grid_levels);
            for (int64_t k = 0; k <= L + 1; ++k) h->lv[LV_ECH * (L + 2) + k] = plan.ech[k];
        } else if (d.emit == EMIT_SLICE) {
            sp = plan_slice_emit(g, d.TB, d.grid_levels, d.slice);
            if (sp.nids != d.n_echunks || (int64_t)sp.late_ref.size() != d.n_late || sp.ntiles != d.n_tiles ||
                (int64_t)sp.tsid.size() != d.n_starts || sp.nslices != d.n_slices)
                fail(GC_ERR_INVALID_GRAMMAR, "slice plan does not match the layout");
            validate_slice_plan(sp, g, d.TB, d.grid_levels);
        } else {
            cref.resize(g.c_ref.size());
            // row emit: C's references index [T | RV] (root slot s at TB + s,
            // terminal p at T[p + 1])
            for (size_t e = 0; e < cref.size(); ++e) {
                const int32_t c = g.c_ref[e];
                cref[e] = c >= 0 ? (int32_t)(d.TB + c) : -c - 1;
            }
            co.resize(g.slp.c_off.size());
            for (size_t r = 0; r < co.size(); ++r) co[r] = (int32_t)g.slp.c_off[r];
        }

        // every host-side array is built and checked; now the device
        int dev = 0;
        cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
        h->device = dev;
        cuda_check(cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
        cuda_check(cudaDeviceGetAttribute(&h->coop, cudaDevAttrCooperativeLaunch, dev), "cooperative attribute");
        char* a = h->arena;
        put(st, a, d.nodes, nodes.data(), nodes.size());
        put(st, a, d.levels, h->lv.data(), h->lv.size());
        if (policy_is_f32(policy)) {
            put(st, a, d.V, g.V.data(), g.V.size());
        } else {
            std::vector<long long> v(g.V.size());
            for (size_t i = 0; i < v.size(); ++i) v[i] = policy == GC_BOOL_OR ? ~0ll : (long long)g.V[i];
            put(st, a, d.V, v.data(), v.size());
        }
        put(st, a, d.leaf, leaf.data(), leaf.size());
        if (d.emit == EMIT_LEVEL) {
            put(st, a, d.cref, plan.cref.data(), plan.cref.size());
            put(st, a, d.echunk, plan.echunk.data(), plan.echunk.size());
            put(st, a, d.row_ech, plan.row_ech.data(), plan.row_ech.size());
            put(st, a, d.late_off, plan.late_off.data(), plan.late_off.size());
            put(st, a, d.late_ref, plan.late_ref.data(), plan.late_ref.size());
        } else if (d.emit == EMIT_SLICE) {
            put(st, a, d.sref, sp.sref.data(), sp.sref.size());
            put(st, a, d.sflag, sp.sflag.data(), sp.sflag.size());
            put(st, a, d.tile_sid, sp.tile_sid.data(), sp.tile_sid.size());
            put(st, a, d.row_pos, sp.row_pos.data(), sp.row_pos.size());
            put(st, a, d.sx0, sp.x0.data(), sp.x0.size());
            put(st, a, d.stile, sp.stile.data(), sp.stile.size());
            put(st, a, d.sorder, sp.sorder.data(), sp.sorder.size());
            put(st, a, d.row_ech, sp.row_seg.data(), sp.row_seg.size());
            put(st, a, d.late_off, sp.late_off.data(), sp.late_off.size());
            put(st, a, d.late_ref, sp.late_ref.data(), sp.late_ref.size());
        } else {
            put(st, a, d.c_off, co.data(), co.size());
            put(st, a, d.c_ref, cref.data(), cref.size());
        }
        if (flow) {
            put(st, a, d.fblk, fp->blk.data(), fp->blk.size());
            put(st, a, d.forder, fp->order.data(), fp->order.size());
            put(st, a, d.fdeps, fp->deps.data(), fp->deps.size());
            put(st, a, d.fgran, fp->gran.data(), fp->gran.size());
            cuda_check(cudaMemsetAsync(a + d.fflags, 0, 4 * std::max<int64_t>(1, d.n_fblocks), st), "flags clear");
            cuda_check(cudaMemsetAsync(a + d.fdone, 0, 8 * (L + 2), st), "level counters clear");
        }
        cuda_check(cudaMemsetAsync(a + d.status, 0, 256, st), "status clear");
        cuda_check(cudaStreamSynchronize(st), "upload synchronize");
        *out = h.release();
    });
}

gc_status gc_upload(const gc_grammar* gg, gc_policy policy, int32_t k_max, void* arena, int64_t arena_bytes,
                    void* stream, gc_handle** out) {
    return gc_upload_ex(gg, policy, k_max, GC_SCHED_PERSISTENT, arena, arena_bytes, stream, out);
}

gc_status gc_matvec(gc_handle* h, const void* x, void* y, int32_t k, void* stream) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if ((!x && h->m > 0) || (!y && h->n > 0)) fail(GC_ERR_ARG, "null x or y");
        check_k(h, k);
        check_device(h);
        after_last_loop(h->loop, static_cast<cudaStream_t>(stream), cuda_check);
        dispatch_product(h, x, y, k, static_cast<cudaStream_t>(stream));
    });
}

gc_status gc_matvec_host(gc_handle* h, const void* x_host, void* y_host, int32_t k, void* stream) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if ((!x_host && h->m > 0) || (!y_host && h->n > 0)) fail(GC_ERR_ARG, "null x or y");
        check_k(h, k);
        check_device(h);
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        after_last_loop(h->loop, st, cuda_check);
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
        check_device(h);
        if (h->n != h->m) fail(GC_ERR_ARG, "gc_reach needs a square matrix");
        if (max_iter < 1) fail(GC_ERR_ARG, "max_iter must be >= 1");
        if (!run_fixpoint<OrUpdate>(h, reinterpret_cast<const unsigned long long*>(x0),
                                    reinterpret_cast<unsigned long long*>(x), max_iter, iters,
                                    static_cast<cudaStream_t>(stream)))
            rc = GC_ERR_NOT_CONVERGED;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_reach: max_iter reached before the fixpoint");
    return rc;
}

gc_status gc_sssp(gc_handle* h, const float* x0, float* x, int32_t max_iter, int32_t* iters, void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h || !x0 || !x || !iters) fail(GC_ERR_ARG, "null argument");
        if (h->policy != GC_F32_MIN_PLUS) fail(GC_ERR_ARG, "gc_sssp needs the GC_F32_MIN_PLUS policy");
        check_device(h);
        if (h->n != h->m) fail(GC_ERR_ARG, "gc_sssp needs a square matrix");
        if (max_iter < 1) fail(GC_ERR_ARG, "max_iter must be >= 1");
        if (!run_fixpoint<MinUpdate>(h, x0, x, max_iter, iters, static_cast<cudaStream_t>(stream)))
            rc = GC_ERR_NOT_CONVERGED;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_sssp: max_iter reached before the fixpoint");
    return rc;
}

gc_status gc_check(gc_handle* h, void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        int32_t* status = reinterpret_cast<int32_t*>(h->arena + h->lay.status);
        int32_t s = 0;
        after_last_loop(h->loop, st, cuda_check);
        cuda_check(cudaMemcpyAsync(&s, status, 4, cudaMemcpyDeviceToHost, st), "status read");
        cuda_check(cudaStreamSynchronize(st), "stream synchronize");
        if (s != 0) {
            // a failed launch leaves the barrier counter part-way: restart it
            cuda_check(cudaMemsetAsync(h->arena + h->lay.status, 0, 256, st), "status clear");
            if (h->flow) {   // a failed dataflow product leaves flags and counters part-way
                cuda_check(cudaMemsetAsync(h->arena + h->lay.fflags, 0, 4 * std::max<int64_t>(1, h->nblocks), st),
                           "flags clear");
                cuda_check(cudaMemsetAsync(h->arena + h->lay.fdone, 0, 8 * (h->L + 2), st), "level counters clear");
                h->epoch = 0;
            }
            cuda_check(cudaStreamSynchronize(st), "stream synchronize");
            h->bar_base = 0;
            h->tbar_base = 0;
        }
        rc = (gc_status)s;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("device status word reported an error");
    return rc;
}

gc_status gc_update(gc_policy policy, void* x, const void* y, int64_t n, int32_t* changed, void* stream) {
    return guard([&] {
        if (policy != GC_BOOL_OR && policy != GC_F32_MIN_PLUS)
            fail(GC_ERR_ARG, "gc_update needs the GC_BOOL_OR or GC_F32_MIN_PLUS policy");
        if (n < 0 || !changed || (n > 0 && (!x || !y))) fail(GC_ERR_ARG, "null argument or negative n");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        cuda_check(cudaMemsetAsync(changed, 0, sizeof(int32_t), st), "changed clear");
        if (n == 0) return;
        int dev = 0, sms = 1;
        cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
        cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
        const int grid = grid_for(n, kThreads, sms, 8);
        if (policy == GC_BOOL_OR)
            update_rows_kernel<OrUpdate><<<grid, kThreads, 0, st>>>(static_cast<unsigned long long*>(x),
                                                                   static_cast<const unsigned long long*>(y), n,
                                                                   changed);
        else
            update_rows_kernel<MinUpdate><<<grid, kThreads, 0, st>>>(static_cast<float*>(x),
                                                                    static_cast<const float*>(y), n, changed);
        cuda_check(cudaGetLastError(), "kernel launch");
    });
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
        if (schedule != GC_SCHED_PERSISTENT && schedule != GC_SCHED_PER_LEVEL && schedule != GC_SCHED_DATAFLOW)
            fail(GC_ERR_ARG, "unknown schedule");
        if (schedule == GC_SCHED_DATAFLOW && !h->flow)
            fail(GC_ERR_UNSUPPORTED, "the dataflow schedule serves handles with one value a node (k_max = 1)");
        // on a dataflow handle the persistent schedule is the dataflow sweep
        h->schedule = h->flow && schedule == GC_SCHED_PERSISTENT ? GC_SCHED_DATAFLOW : schedule;
    });
}

gc_status gc_get_schedule(const gc_handle* h, int32_t* schedule) {
    return guard([&] {
        if (!h || !schedule) fail(GC_ERR_ARG, "null argument");
        *schedule = (h->schedule != GC_SCHED_PER_LEVEL && h->coop) ? h->schedule : GC_SCHED_PER_LEVEL;
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
        check_device(h);
        const int64_t need = static_scratch_need(h, k);
        if (need > kStaticScratchBytes)
            fail(GC_ERR_UNSUPPORTED, "gc_matvec_static: this grammar needs " + std::to_string(need) +
                                         " bytes of scratch; the fixed array holds " +
                                         std::to_string(kStaticScratchBytes));
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        after_last_loop(h->loop, st, cuda_check);
        unsigned char* scratch = static_scratch_on_current_device();
        switch (h->policy) {
            case GC_F32_SUM: for_f32_width<RunStatic>(k, h, x, y, st, scratch); break;
            case GC_I64_SUM: run_product_static<PolI64>(h, x, y, st, scratch); break;
            case GC_BOOL_OR: run_product_static<PolOr>(h, x, y, st, scratch); break;
            case GC_F32_MIN_PLUS:
                if (k == 1) run_product_static<PolMinPlus>(h, x, y, st, scratch);
                else run_product_static<PolMinPlusx16>(h, x, y, st, scratch);
                break;
        }
        int32_t s = 0;
        cuda_check(cudaMemcpyAsync(&s, scratch + static_parts(h, k).status, 4, cudaMemcpyDeviceToHost, st),
                   "fixed scratch status read");
        cuda_check(cudaStreamSynchronize(st), "stream synchronize");
        rc = (gc_status)s;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_matvec_static: a device-side wait ran out");
    return rc;
}

void gc_free_handle(gc_handle* h) { delete h; }

}  // extern "C"
