// Device side of gcsparse: upload of the packed grammar into a caller-owned
// arena, and the streaming bottom-up sweep of Sec. 4.3 of the pages
// ("Right Multiplication on Grammar-Compressed Matrices"):
//
//   leaf gather     T[0] = identity, T[p+1] = V[l_p] (x) x[j_p]        (Sec. 4.3)
//   level combine   for k = 1..L: cur[t] = cv(a_t) (+) cv(b_t), where
//                   cv(c) = prev[c] for c >= 0 and T[-c-1] for c < 0;
//                   the level's roots (its first nodes) are also written to
//                   RV, the emit-on-the-spot capture                  (Listing 1,
//                   Lemma 3.3)
//   row emit        y[r] = (+) over row r's symbols of RV[c] / T[-c-1]  (Lemma 2.2)
//
// The pages emit with atomicAdd into y; here each row is reduced by a fixed
// group of threads in a fixed order, so the result is deterministic.
#include <cuda_runtime.h>

#include <cstring>
#include <memory>

#include "common.hpp"
#include "layout.hpp"
#include "policy.cuh"

struct gc_handle {
    gc_policy policy = GC_F32_SUM;
    int32_t k_max = 1;
    int64_t n = 0, m = 0, alpha = 0, L = 0, n_roots = 0, c_len = 0, max_width = 0;
    std::vector<int64_t> lvl_off, lvl_roots, root_off;
    char* arena = nullptr;
    gcs::DevLayout lay{};
    int sms = 1;
    int emit_group = 32;   // threads per row in the emit; 0 = one CTA per row
    int64_t launches = 0;
};

namespace gcs {

namespace {

constexpr int kThreads = 256;

void cuda_check(cudaError_t e, const char* what) {
    if (e != cudaSuccess) fail(GC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

__device__ __forceinline__ float shfl_x(float v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ long long shfl_x(long long v, int m) { return __shfl_xor_sync(0xffffffffu, v, m); }
__device__ __forceinline__ unsigned long long shfl_x(unsigned long long v, int m) {
    return __shfl_xor_sync(0xffffffffu, v, m);
}
__device__ __forceinline__ float4 shfl_x(float4 v, int m) {
    return make_float4(shfl_x(v.x, m), shfl_x(v.y, m), shfl_x(v.z, m), shfl_x(v.w, m));
}

// ---------------------------------------------------------------- leaf gather
template <class P>
__global__ void __launch_bounds__(kThreads)
leaf_kernel(const int32_t* __restrict__ leaf_col, const typename P::Leaf* __restrict__ leaf_val,
            const typename P::V* __restrict__ x, typename P::V* __restrict__ T, int64_t alpha) {
    const int64_t total = (alpha + 1) * P::LPN;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = i / P::LPN;
        const int lane = (int)(i % P::LPN);
        if (p == 0) {
            T[i] = P::identity();
        } else {
            const int64_t j = __ldg(leaf_col + (p - 1));
            T[i] = P::leaf(leaf_val, p - 1, __ldg(x + j * P::LPN + lane));
        }
    }
}

// ---------------------------------------------------------------- level combine
template <class P>
__global__ void __launch_bounds__(kThreads)
level_kernel(const int2* __restrict__ nodes, int64_t w, int64_t nroots,
             const typename P::V* __restrict__ prev, const typename P::V* __restrict__ T,
             typename P::V* __restrict__ cur, typename P::V* __restrict__ rv) {
    using V = typename P::V;
    const int64_t total = w * P::LPN;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / P::LPN;
        const int lane = (int)(i % P::LPN);
        const int2 ab = __ldcs(nodes + t);           // streamed once: evict first
        const V* pa = ab.x >= 0 ? prev + (int64_t)ab.x * P::LPN : T + (int64_t)(-ab.x - 1) * P::LPN;
        const V* pb = ab.y >= 0 ? prev + (int64_t)ab.y * P::LPN : T + (int64_t)(-ab.y - 1) * P::LPN;
        const V v = P::combine(pa[lane], pb[lane]);
        cur[i] = v;
        if (t < nroots) rv[i] = v;
    }
}

// ---------------------------------------------------------------- row emit
// G threads per row (G divides 32); warps iterate rows in lockstep so the
// shuffles always see the full warp.
template <class P, int G>
__global__ void __launch_bounds__(kThreads)
emit_group_kernel(const int32_t* __restrict__ c_off, const int32_t* __restrict__ c_ref,
                  const typename P::V* __restrict__ rv, const typename P::V* __restrict__ T,
                  typename P::V* __restrict__ y, int64_t n) {
    using V = typename P::V;
    constexpr int RPW = 32 / G;   // rows per warp per round
    const int lane = threadIdx.x & 31;
    const int gl = lane % G;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = warp * RPW; base < n; base += nwarps * RPW) {
        const int64_t row = base + lane / G;
        V acc[P::LPN];
#pragma unroll
        for (int l = 0; l < P::LPN; ++l) acc[l] = P::identity();
        if (row < n) {
            const int32_t s = __ldg(c_off + row), e = __ldg(c_off + row + 1);
            for (int32_t q = s + gl; q < e; q += G) {
                const int32_t c = __ldcs(c_ref + q);
                const V* src = c >= 0 ? rv + (int64_t)c * P::LPN : T + (int64_t)(-c - 1) * P::LPN;
#pragma unroll
                for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], src[l]);
            }
        }
#pragma unroll
        for (int msk = G / 2; msk >= 1; msk >>= 1)
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], shfl_x(acc[l], msk));
        if (row < n && gl == 0)
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) y[row * P::LPN + l] = acc[l];
    }
}

// One CTA per row, for long rows of C.
template <class P>
__global__ void __launch_bounds__(kThreads)
emit_cta_kernel(const int32_t* __restrict__ c_off, const int32_t* __restrict__ c_ref,
                const typename P::V* __restrict__ rv, const typename P::V* __restrict__ T,
                typename P::V* __restrict__ y, int64_t n) {
    using V = typename P::V;
    __shared__ V red[kThreads / 32][P::LPN];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t row = blockIdx.x; row < n; row += gridDim.x) {
        V acc[P::LPN];
#pragma unroll
        for (int l = 0; l < P::LPN; ++l) acc[l] = P::identity();
        const int32_t s = __ldg(c_off + row), e = __ldg(c_off + row + 1);
        for (int32_t q = s + threadIdx.x; q < e; q += kThreads) {
            const int32_t c = __ldcs(c_ref + q);
            const V* src = c >= 0 ? rv + (int64_t)c * P::LPN : T + (int64_t)(-c - 1) * P::LPN;
#pragma unroll
            for (int l = 0; l < P::LPN; ++l) acc[l] = P::combine(acc[l], src[l]);
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
            for (int w = 1; w < kThreads / 32; ++w) t = P::combine(t, red[w][threadIdx.x]);
            y[row * P::LPN + threadIdx.x] = t;
        }
        __syncthreads();
    }
}

// x |= y elementwise; sets *changed if any word changed (Boolean fixpoint step).
__global__ void __launch_bounds__(kThreads)
or_update_kernel(unsigned long long* __restrict__ x, const unsigned long long* __restrict__ y, int64_t n,
                 int32_t* __restrict__ changed) {
    int ch = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const unsigned long long a = x[i], b = a | y[i];
        if (b != a) {
            x[i] = b;
            ch = 1;
        }
    }
    if (__syncthreads_or(ch) && threadIdx.x == 0) *changed = 1;
}

int grid_for(int64_t items, int sms, int per_sm = 8) {
    int64_t g = (items + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)sms * per_sm;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

template <class P>
void run_product(gc_handle* h, const void* x, void* y, cudaStream_t st) {
    using V = typename P::V;
    const DevLayout& d = h->lay;
    char* a = h->arena;
    const V* xv = static_cast<const V*>(x);
    V* yv = static_cast<V*>(y);
    V* T = reinterpret_cast<V*>(a + d.T);
    V* RV = reinterpret_cast<V*>(a + d.RV);
    V* buf[2] = {reinterpret_cast<V*>(a + d.buf0), reinterpret_cast<V*>(a + d.buf1)};
    const int2* nodes = reinterpret_cast<const int2*>(a + d.nodes);
    int64_t launches = 0;

    leaf_kernel<P><<<grid_for((h->alpha + 1) * P::LPN, h->sms), kThreads, 0, st>>>(
        reinterpret_cast<const int32_t*>(a + d.leaf_col),
        reinterpret_cast<const typename P::Leaf*>(a + d.leaf_val), xv, T, h->alpha);
    ++launches;
    for (int64_t k = 1; k <= h->L; ++k) {
        const int64_t w = h->lvl_off[k + 1] - h->lvl_off[k];
        if (w == 0) continue;
        level_kernel<P><<<grid_for(w * P::LPN, h->sms), kThreads, 0, st>>>(
            nodes + h->lvl_off[k], w, h->lvl_roots[k], buf[(k - 1) & 1], T, buf[k & 1],
            RV + h->root_off[k] * P::LPN);
        ++launches;
    }
    if (h->n > 0) {
        const int32_t* c_off = reinterpret_cast<const int32_t*>(a + d.c_off);
        const int32_t* c_ref = reinterpret_cast<const int32_t*>(a + d.c_ref);
        switch (h->emit_group) {
            case 0:
                emit_cta_kernel<P><<<(int)std::min<int64_t>(h->n, (int64_t)h->sms * 8), kThreads, 0, st>>>(
                    c_off, c_ref, RV, T, yv, h->n);
                break;
#define GC_EMIT(G)                                                                                   \
    case G:                                                                                          \
        emit_group_kernel<P, G><<<grid_for((h->n + (32 / G) - 1) / (32 / G) * 32, h->sms), kThreads, 0, st>>>( \
            c_off, c_ref, RV, T, yv, h->n);                                                          \
        break;
            GC_EMIT(1) GC_EMIT(2) GC_EMIT(4) GC_EMIT(8) GC_EMIT(16) GC_EMIT(32)
#undef GC_EMIT
            default:
                fail(GC_ERR_ARG, "bad emit configuration");
        }
        ++launches;
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
void put(cudaStream_t st, char* arena, int64_t off, const std::vector<T>& v) {
    if (v.empty()) return;
    cuda_check(cudaMemcpyAsync(arena + off, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice, st),
               "upload copy");
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
        h->alpha = g.alpha();
        h->L = g.L;
        h->n_roots = g.n_roots;
        h->c_len = (int64_t)g.c_ref.size();
        h->max_width = g.max_width();
        h->lvl_off = g.lvl_off;
        h->lvl_roots = g.lvl_roots;
        h->root_off = g.root_off;
        h->arena = static_cast<char*>(arena);
        h->lay = d;
        int dev = 0;
        cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
        cuda_check(cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
        // emit group: about one symbol per thread per pass, capped at a CTA
        const double avg = g.n > 0 ? (double)h->c_len / (double)g.n : 0.0;
        if (avg >= 256) h->emit_group = 0;
        else {
            int G = 1;
            while (G < 32 && G < avg) G <<= 1;
            h->emit_group = G;
        }

        char* a = h->arena;
        put(st, a, d.nodes, g.nodes);
        put(st, a, d.lvl_off, g.lvl_off);
        put(st, a, d.lvl_roots, g.lvl_roots);
        put(st, a, d.root_off, g.root_off);
        put(st, a, d.leaf_col, g.term_col);
        if (policy == GC_F32_SUM) {
            std::vector<float> lv(g.term_vidx.size());
            for (size_t t = 0; t < lv.size(); ++t) lv[t] = g.V[g.term_vidx[t]];
            put(st, a, d.leaf_val, lv);
        } else if (policy == GC_I64_SUM) {
            std::vector<long long> lv(g.term_vidx.size());
            for (size_t t = 0; t < lv.size(); ++t) lv[t] = (long long)g.V[g.term_vidx[t]];
            put(st, a, d.leaf_val, lv);
        }
        std::vector<int32_t> co(g.slp.c_off.size());
        for (size_t r = 0; r < co.size(); ++r) co[r] = (int32_t)g.slp.c_off[r];
        put(st, a, d.c_off, co);
        put(st, a, d.c_ref, g.c_ref);
        cuda_check(cudaMemsetAsync(a + d.status, 0, 256, st), "status clear");
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
                or_update_kernel<<<grid_for(n, h->sms), kThreads, 0, st>>>(xv, yv, n, changed);
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
            cuda_check(cudaMemsetAsync(status, 0, 4, st), "status clear");
            cuda_check(cudaStreamSynchronize(st), "stream synchronize");
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

void gc_free_handle(gc_handle* h) { delete h; }

}  // extern "C"
