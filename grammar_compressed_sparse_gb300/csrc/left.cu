// Device side of the left product x = M^T y (x^T = y^T M) over the packed,
// properly layered grammar: the pull-based top-down sweep planned in
// left.hpp. The pages name left multiplication by pull-based reduction as
// future work (Sec. 8); this is its plainest reading: every value is a sum
// the reading thread gathers (no atomics, no scatter), the level sets run in
// stream order L, L-1, ..., 1, and each sum has a fixed order, so x is the
// same bit for bit on every run.
//
// One kernel serves every step: a grid of warps walks the step's tasks; a
// LIGHT task sums up to 32 consecutive segments, one per lane, each in order
// from its initial value (items loaded four at a time, added in order; a
// segment too long for one lane is left to its HEAVY task); a HEAVY task sums
// one segment over the warp (lane l takes items l, l + 32, ... in order, then
// a fixed xor butterfly) and adds it to the initial value.
//
// Policies (Sec. 5's semirings, as for the right product): the float32 sum
// (each addition and product rounded separately), the exact int64 sum,
// Boolean OR on 64-bit source sets, and tropical min-plus in float32. The
// weights are (+)-sums of y over occurrences in every policy; the column
// step applies the leaf map: V[l] * weight, or V[l] + weight for min-plus
// (+ distributes over min), or the weight itself for OR (every entry is 1).
//
// The L + 3 steps are one CUDA graph per handle, a chain of kernel nodes
// built on the first product; later products update the two nodes that read
// y and write x when those pointers change, and launch the graph, which
// spares the per-launch gaps of a stream of short dependent kernels.
#include <cuda_runtime.h>

#include <memory>
#include <string>

#include "common.hpp"
#include "layout.hpp"
#include "left.hpp"
#include "loop.hpp"

struct gc_left_handle {
    gc_policy policy = GC_F32_SUM;
    int64_t elem = 4;   // bytes of a value
    int64_t n = 0, m = 0, L = 0, N = 0, rho = 0, alpha = 0;
    std::vector<int64_t> lvl_off, lvl_roots, root_off, task_off;
    char* arena = nullptr;
    int sms = 1;
    int64_t launches = 0;
    // arena offsets
    int64_t soff, srow, poff, pref, toff, tref, coff, vidx, V, task, RS, W, TIN, tmp, flag, total, grammar_bytes;
    // the steps as a graph: its kernel nodes and the step set of each
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    gcs::LoopHost loop;   // the fixpoint loop's pinned words and events
    std::vector<cudaGraphNode_t> nodes;
    std::vector<int64_t> node_set;
    const void* y_last = nullptr;
    void* x_last = nullptr;
    ~gc_left_handle() {
        if (loop.ended) (void)cudaEventSynchronize(loop.end);   // a fixpoint's last batch may still run
        if (exec) cudaGraphExecDestroy(exec);
        if (graph) cudaGraphDestroy(graph);
    }
};

namespace gcs {
namespace {

constexpr int kLeftThreads = 256;

// What one step reads and writes: segment g covers references
// ref[off[g] .. off[g+1]) (ref == nullptr: the references are the indices
// themselves); item i is src[i], or leaf(V[vidx[i]], src[i]) in the column
// step. Value arrays are untyped here; the kernel's policy gives their type.
struct LeftStep {
    const int32_t* off;
    const int32_t* ref;
    const void* src;
    const int32_t* vidx;   // columns: terminal -> value index, else nullptr
    const void* V;
    // initial value of segment g: init[g - init_base + init_shift] when
    // init_base <= g < init_base + init_count, else the identity
    const void* init;
    int64_t init_base, init_count, init_shift;
    void* out;             // out[g - out_base]
    int64_t out_base;
    const int32_t* conv;   // nonzero while a converged fixpoint loop skips the rest of its products
};

// The combine, its identity and the column step's leaf map of each policy.
struct LeftSum {
    using V = float;
    using Leaf = float;
    __device__ __forceinline__ static V identity() { return 0.0f; }
    __device__ __forceinline__ static V combine(V a, V b) { return __fadd_rn(a, b); }
    __device__ __forceinline__ static V leaf(Leaf v, V w) { return __fmul_rn(v, w); }
};
struct LeftI64 {
    using V = long long;
    using Leaf = long long;
    __device__ __forceinline__ static V identity() { return 0; }
    __device__ __forceinline__ static V combine(V a, V b) { return a + b; }
    __device__ __forceinline__ static V leaf(Leaf v, V w) { return v * w; }
};
struct LeftOr {
    using V = unsigned long long;
    using Leaf = unsigned long long;   // every stored entry is 1: AND with all ones
    __device__ __forceinline__ static V identity() { return 0ull; }
    __device__ __forceinline__ static V combine(V a, V b) { return a | b; }
    __device__ __forceinline__ static V leaf(Leaf, V w) { return w; }
};
struct LeftMinPlus {
    using V = float;
    using Leaf = float;
    __device__ __forceinline__ static V identity() { return __int_as_float(0x7f800000); }
    __device__ __forceinline__ static V combine(V a, V b) { return fminf(a, b); }
    __device__ __forceinline__ static V leaf(Leaf v, V w) { return __fadd_rn(v, w); }
};

template <class Op>
__device__ __forceinline__ typename Op::V left_item(const LeftStep& s, int32_t q) {
    using V = typename Op::V;
    const int32_t i = s.ref ? __ldg(s.ref + q) : q;
    const V v = static_cast<const V*>(s.src)[i];
    return s.vidx ? Op::leaf(__ldg(static_cast<const typename Op::Leaf*>(s.V) + __ldg(s.vidx + i)), v) : v;
}

template <class Op>
__device__ __forceinline__ typename Op::V left_init(const LeftStep& s, int32_t g) {
    const int64_t r = (int64_t)g - s.init_base;
    return (s.init && r >= 0 && r < s.init_count) ? static_cast<const typename Op::V*>(s.init)[r + s.init_shift]
                                                  : Op::identity();
}

// A warp's tasks are t0 + w, t0 + w + warps, ...; the next task's header and
// segment offsets are loaded before the current task is summed, so their
// latency hides behind its gathers.
struct TaskHead {
    int32_t first, cnt, q0, q1;
};

__device__ __forceinline__ TaskHead load_head(const LeftStep& s, const int32_t* __restrict__ task, int64_t t,
                                              int64_t t1, int lane) {
    TaskHead h{0, 0, 0, 0};
    if (t < t1) {
        h.first = __ldg(task + 2 * t);
        h.cnt = __ldg(task + 2 * t + 1);
        // LIGHT: lane's own segment; HEAVY: the one segment
        const int32_t g = h.cnt > 0 ? h.first + lane : h.first;
        if (h.cnt < 0 || lane < h.cnt) {
            h.q0 = __ldg(s.off + g);
            h.q1 = __ldg(s.off + g + 1);
        }
    }
    return h;
}

template <class Op>
__global__ void __launch_bounds__(kLeftThreads) left_step_kernel(const LeftStep s, const int32_t* __restrict__ task,
                                                                 int64_t t0, int64_t t1) {
    using V = typename Op::V;
    if (*reinterpret_cast<const volatile int32_t*>(s.conv) != 0) return;
    const int lane = threadIdx.x & 31;
    V* const out = static_cast<V*>(s.out);
    const int64_t warps = (int64_t)gridDim.x * (kLeftThreads / 32);
    int64_t t = t0 + (int64_t)blockIdx.x * (kLeftThreads / 32) + (threadIdx.x >> 5);
    TaskHead h = load_head(s, task, t, t1, lane);
    while (t < t1) {
        const TaskHead c = h;
        t += warps;
        h = load_head(s, task, t, t1, lane);
        if (c.cnt > 0) {   // LIGHT: one segment per lane
            const int32_t g = c.first + lane;
            if (lane < c.cnt && c.q1 - c.q0 <= kLeftLightMax) {
                V acc = left_init<Op>(s, g);
                int32_t q = c.q0;
                for (; q + 4 <= c.q1; q += 4) {
                    const V v0 = left_item<Op>(s, q), v1 = left_item<Op>(s, q + 1), v2 = left_item<Op>(s, q + 2),
                            v3 = left_item<Op>(s, q + 3);
                    acc = Op::combine(Op::combine(Op::combine(Op::combine(acc, v0), v1), v2), v3);
                }
                for (; q < c.q1; ++q) acc = Op::combine(acc, left_item<Op>(s, q));
                out[g - s.out_base] = acc;
            }
        } else {           // HEAVY: one segment over the warp
            const int32_t g = c.first;
            V acc = Op::identity();
            for (int32_t q = c.q0 + lane; q < c.q1; q += 32) acc = Op::combine(acc, left_item<Op>(s, q));
#pragma unroll
            for (int msk = 16; msk >= 1; msk >>= 1) acc = Op::combine(acc, __shfl_xor_sync(0xffffffffu, acc, msk));
            if (lane == 0) out[g - s.out_base] = Op::combine(left_init<Op>(s, g), acc);
        }
    }
}

// One step of a forward fixpoint loop that runs on without the host, x = x
// (+) t elementwise (OR, or min). ctl: changed in this step, converged, CTAs
// of this step finished, product count at convergence. The last CTA to
// finish reads the changed word; if nothing changed the loop has converged
// at product `it`; it then clears the step's words. Once converged, every
// later step (and product) does nothing.
template <class Op>
__global__ void __launch_bounds__(kLeftThreads)
left_update_loop_kernel(typename Op::V* __restrict__ x, const typename Op::V* __restrict__ t, int64_t n,
                        int32_t* __restrict__ ctl, int32_t it) {
    __shared__ int s_last;
    if (*reinterpret_cast<const volatile int32_t*>(ctl + 1) != 0) return;
    int ch = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const typename Op::V u = x[i], v = Op::combine(u, t[i]);
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
        if (*reinterpret_cast<volatile int32_t*>(ctl) == 0) {
            ctl[3] = it;
            ctl[1] = 1;
        }
        ctl[0] = 0;
        ctl[2] = 0;
        __threadfence();
    }
}

void cuda_ok(cudaError_t e, const char* what) {
    if (e != cudaSuccess) fail(GC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Arena parts, 256-byte aligned: the plan's arrays (read-only), then the
// seed sums RS, the node weights W and the terminal sums TIN (h.elem bytes a
// value).
void left_layout(const LeftPlan& p, gc_left_handle& h) {
    int64_t o = 0;
    auto take = [&](int64_t bytes) {
        const int64_t at = o;
        o = align256(o + std::max<int64_t>(bytes, 4));
        return at;
    };
    h.soff = take(4 * (int64_t)p.soff.size());
    h.srow = take(4 * (int64_t)p.srow.size());
    h.poff = take(4 * (int64_t)p.poff.size());
    h.pref = take(4 * (int64_t)p.pref.size());
    h.toff = take(4 * (int64_t)p.toff.size());
    h.tref = take(4 * (int64_t)p.tref.size());
    h.coff = take(4 * (int64_t)p.coff.size());
    h.vidx = take(4 * (int64_t)p.term_vidx.size());
    h.V = take(h.elem * (int64_t)p.V.size());
    h.task = take(4 * (int64_t)p.task.size());
    h.grammar_bytes = o;
    h.RS = take(h.elem * (p.rho + p.alpha));
    h.W = take(h.elem * p.N);
    h.TIN = take(h.elem * p.alpha);
    h.tmp = take(h.elem * p.m);   // the fixpoints' M^T x
    h.flag = take(256);           // the fixpoints' changed flag
    h.total = o;
}

// One step of a product: its arguments and launch shape.
struct StepLaunch {
    LeftStep s;
    const int32_t* task;
    int64_t t0, t1, set;
    unsigned grid;
};

// The product's steps in order (steps with no task left out).
std::vector<StepLaunch> left_steps(const gc_left_handle* h, const void* y, void* x) {
    char* a = h->arena;
    auto I = [&](int64_t off) { return reinterpret_cast<const int32_t*>(a + off); };
    auto F = [&](int64_t off) { return static_cast<void*>(a + off); };
    std::vector<StepLaunch> out;
    const int32_t* conv = I(h->flag) + 1;   // the fixpoint loop's converged word (0 outside a loop)
    auto add = [&](LeftStep s, int64_t set) {
        const int64_t t0 = h->task_off[set], t1 = h->task_off[set + 1];
        if (t1 <= t0) return;
        s.conv = conv;
        const int64_t wpb = kLeftThreads / 32;
        const int64_t grid = std::min<int64_t>((t1 - t0 + wpb - 1) / wpb, (int64_t)h->sms * 8);
        out.push_back(StepLaunch{s, I(h->task), t0, t1, set, (unsigned)grid});
    };
    // seed: RS[s] = sum of y over C's references to s
    add(LeftStep{I(h->soff), I(h->srow), y, nullptr, nullptr, nullptr, 0, 0, 0, F(h->RS), 0, nullptr}, 0);
    // levels, top first: W[u] = RS[root slot] (roots) + sum of the parents' W
    for (int64_t k = h->L; k >= 1; --k)
        add(LeftStep{I(h->poff), I(h->pref), F(h->W), nullptr, nullptr, F(h->RS), h->lvl_off[k], h->lvl_roots[k],
                     h->root_off[k], F(h->W), 0, nullptr},
            k);
    // terminals: TIN[p] = RS[rho + p] + sum of the W of the nodes naming p
    add(LeftStep{I(h->toff), I(h->tref), F(h->W), nullptr, nullptr, F(h->RS), 0, h->alpha, h->rho, F(h->TIN), 0,
                 nullptr},
        h->L + 1);
    // columns: x[j] = sum over column j's terminals of V[l] * TIN[p]
    add(LeftStep{I(h->coff), nullptr, F(h->TIN), I(h->vidx), F(h->V), nullptr, 0, 0, 0, x, 0, nullptr}, h->L + 2);
    return out;
}

// Kernel-node parameters of a step; args holds the argument pointers and
// must live until the call that takes the parameters returns.
// The step kernel of a policy.
void* step_kernel(gc_policy p) {
    switch (p) {
        case GC_F32_SUM: return reinterpret_cast<void*>(left_step_kernel<LeftSum>);
        case GC_I64_SUM: return reinterpret_cast<void*>(left_step_kernel<LeftI64>);
        case GC_BOOL_OR: return reinterpret_cast<void*>(left_step_kernel<LeftOr>);
        case GC_F32_MIN_PLUS: return reinterpret_cast<void*>(left_step_kernel<LeftMinPlus>);
    }
    fail(GC_ERR_ARG, "unknown policy");
}

cudaKernelNodeParams node_params(gc_policy p, StepLaunch& l, void* (&args)[4]) {
    args[0] = &l.s;
    args[1] = &l.task;
    args[2] = &l.t0;
    args[3] = &l.t1;
    cudaKernelNodeParams kp{};
    kp.func = step_kernel(p);
    kp.gridDim = dim3(l.grid);
    kp.blockDim = dim3(kLeftThreads);
    kp.sharedMemBytes = 0;
    kp.kernelParams = args;
    kp.extra = nullptr;
    return kp;
}

template <class T>
void put(cudaStream_t st, char* arena, int64_t off, const std::vector<T>& v) {
    if (v.empty()) return;
    cuda_ok(cudaMemcpyAsync(arena + off, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice, st), "left upload copy");
}

// One left product on stream st: the handle's graph, built on the first
// call; a call with other y or x pointers updates the seed and column nodes.
void left_run(gc_left_handle* h, const void* y, void* x, cudaStream_t st) {
    std::vector<StepLaunch> steps = left_steps(h, y, x);
    if (steps.empty()) {
        h->launches = 0;
        return;
    }
    if (!h->exec) {
        // first product: the chain of kernel nodes, in step order
        cuda_ok(cudaGraphCreate(&h->graph, 0), "left graph create");
        for (StepLaunch& l : steps) {
            void* args[4];
            const cudaKernelNodeParams kp = node_params(h->policy, l, args);
            cudaGraphNode_t node = nullptr;
            const cudaGraphNode_t* dep = h->nodes.empty() ? nullptr : &h->nodes.back();
            cuda_ok(cudaGraphAddKernelNode(&node, h->graph, dep, dep ? 1 : 0, &kp), "left graph node");
            h->nodes.push_back(node);
            h->node_set.push_back(l.set);
        }
        cuda_ok(cudaGraphInstantiate(&h->exec, h->graph, 0), "left graph instantiate");
    } else if (y != h->y_last || x != h->x_last) {
        // new y or x: the seed and column nodes take the new pointers
        for (size_t i = 0; i < steps.size(); ++i)
            if (steps[i].set == 0 || steps[i].set == h->L + 2) {
                if (h->node_set[i] != steps[i].set) fail(GC_ERR_ARG, "left graph does not match its steps");
                void* args[4];
                const cudaKernelNodeParams kp = node_params(h->policy, steps[i], args);
                cuda_ok(cudaGraphExecKernelNodeSetParams(h->exec, h->nodes[i], &kp), "left graph update");
            }
    }
    h->y_last = y;
    h->x_last = x;
    cuda_ok(cudaGraphLaunch(h->exec, st), "left graph launch");
    h->launches = (int64_t)steps.size();
}

// x <- x (+) (M^T x) from x0 until nothing changes, at most max_iter products;
// M^T x goes to the arena's tmp. The loop runs on the device
// (drive_fixpoint): products (the handle's graph) and update steps are
// enqueued in batches of 1, 2, 4, 8, 8, ..., one batch ahead of the one the
// host waits for; the update step's last CTA records convergence and the
// kernels enqueued after it return at once. The loop's words are cleared at
// the end, so later products run. Writes the product count (or -1) to iters
// on the device; false if max_iter was reached first.
template <class Op>
bool left_fixpoint(gc_left_handle* h, const typename Op::V* x0, typename Op::V* x, int32_t max_iter, int32_t* iters,
                   cudaStream_t st) {
    using V = typename Op::V;
    const int64_t n = h->n;
    V* t = reinterpret_cast<V*>(h->arena + h->tmp);
    int32_t* ctl = reinterpret_cast<int32_t*>(h->arena + h->flag);
    after_last_loop(h->loop, st, cuda_ok);
    if (x != x0 && n > 0) cuda_ok(cudaMemcpyAsync(x, x0, n * sizeof(V), cudaMemcpyDeviceToDevice, st), "x0 copy");
    cuda_ok(cudaMemsetAsync(ctl, 0, 16, st), "loop words clear");
    int32_t result = -1;
    int64_t launches = 0;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((n + kLeftThreads - 1) / kLeftThreads, (int64_t)h->sms * 8));
    bool done = false;
    try {
        done = drive_fixpoint(h->loop, ctl, max_iter, st, cuda_ok, [&](int32_t it) {
            left_run(h, x, t, st);
            launches += h->launches;
            left_update_loop_kernel<Op><<<(unsigned)grid, kLeftThreads, 0, st>>>(x, t, n, ctl, it);
            ++launches;
        }, &result);
    } catch (...) {
        if (h->loop.end && cudaEventRecord(h->loop.end, st) == cudaSuccess) h->loop.ended = true;
        throw;
    }
    h->launches = launches;
    cuda_ok(cudaMemsetAsync(ctl, 0, 16, st), "loop words clear");   // later products run again
    // a pageable source: the copy takes its value before it returns
    cuda_ok(cudaMemcpyAsync(iters, &result, 4, cudaMemcpyHostToDevice, st), "iters write");
    mark_loop_end(h->loop, st, cuda_ok);
    return done;
}

}  // namespace
}  // namespace gcs

using namespace gcs;

extern "C" {

gc_status gc_left_layout(const gc_grammar* gg, gc_policy policy, gc_arena_layout* out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null argument");
        const Grammar& g = gg->g;
        check_policy(g, policy, 1);
        validate_packed(g);
        const LeftPlan p = plan_left(g);
        gc_left_handle h;
        h.elem = policy_elem_bytes(policy);
        left_layout(p, h);
        gc_arena_layout l{};
        l.arena_bytes = h.total;
        l.grammar_bytes = h.grammar_bytes;
        l.scratch_bytes = h.total - h.grammar_bytes;
        l.staging_bytes = 0;
        const int64_t rp = g.nnz >= INT32_MAX ? 8 * (g.n + 1) : 4 * (g.n + 1);
        l.csr_bytes = 8 * g.nnz + rp + h.elem * (g.n + g.m);
        *out = l;
    });
}

gc_status gc_left_upload(const gc_grammar* gg, gc_policy policy, void* arena, int64_t arena_bytes, void* stream,
                         gc_left_handle** out) {
    return guard([&] {
        if (!gg || !out) fail(GC_ERR_ARG, "null grammar or output pointer");
        if (!arena) fail(GC_ERR_ARG, "null arena");
        if (reinterpret_cast<uintptr_t>(arena) % 256 != 0) fail(GC_ERR_ARG, "arena must be 256-byte aligned");
        const Grammar& g = gg->g;
        check_policy(g, policy, 1);
        validate_packed(g);
        const LeftPlan p = plan_left(g);
        validate_left_plan(p);
        auto h = std::make_unique<gc_left_handle>();
        h->policy = policy;
        h->elem = policy_elem_bytes(policy);
        left_layout(p, *h);
        if (arena_bytes < h->total) fail(GC_ERR_ARG, "arena smaller than gc_left_layout().arena_bytes");
        h->n = p.n;
        h->m = p.m;
        h->L = p.L;
        h->N = p.N;
        h->rho = p.rho;
        h->alpha = p.alpha;
        h->lvl_off = p.lvl_off;
        h->lvl_roots = p.lvl_roots;
        h->root_off = p.root_off;
        h->task_off = p.task_off;
        h->arena = static_cast<char*>(arena);
        int dev = 0;
        cuda_ok(cudaGetDevice(&dev), "cudaGetDevice");
        cuda_ok(cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, dev), "SM count");
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        char* a = h->arena;
        put(st, a, h->soff, p.soff);
        put(st, a, h->srow, p.srow);
        put(st, a, h->poff, p.poff);
        put(st, a, h->pref, p.pref);
        put(st, a, h->toff, p.toff);
        put(st, a, h->tref, p.tref);
        put(st, a, h->coff, p.coff);
        put(st, a, h->vidx, p.term_vidx);
        if (policy_is_f32(policy)) {
            put(st, a, h->V, p.V);
        } else {   // exact integers, or all-ones masks for OR
            std::vector<long long> v(p.V.size());
            for (size_t i = 0; i < v.size(); ++i) v[i] = policy == GC_BOOL_OR ? ~0ll : (long long)p.V[i];
            put(st, a, h->V, v);
        }
        put(st, a, h->task, p.task);
        // the fixpoint loop's words: clear, so products run (a nonzero
        // converged word makes every step return at once)
        cuda_ok(cudaMemsetAsync(a + h->flag, 0, 256, st), "loop words clear");
        cuda_ok(cudaStreamSynchronize(st), "left upload synchronize");
        *out = h.release();
    });
}

gc_status gc_left_matvec(gc_left_handle* h, const void* y, void* x, void* stream) {
    return guard([&] {
        if (!h) fail(GC_ERR_ARG, "null handle");
        if ((!y && h->n > 0) || (!x && h->m > 0)) fail(GC_ERR_ARG, "null y or x");
        after_last_loop(h->loop, static_cast<cudaStream_t>(stream), cuda_ok);
        left_run(h, y, x, static_cast<cudaStream_t>(stream));
    });
}

gc_status gc_left_reach(gc_left_handle* h, const uint64_t* x0, uint64_t* x, int32_t max_iter, int32_t* iters,
                        void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h || !x0 || !x || !iters) fail(GC_ERR_ARG, "null argument");
        if (h->policy != GC_BOOL_OR) fail(GC_ERR_ARG, "gc_left_reach needs the GC_BOOL_OR policy");
        if (h->n != h->m) fail(GC_ERR_ARG, "gc_left_reach needs a square matrix");
        if (max_iter < 1) fail(GC_ERR_ARG, "max_iter must be >= 1");
        if (!left_fixpoint<LeftOr>(h, reinterpret_cast<const unsigned long long*>(x0),
                                   reinterpret_cast<unsigned long long*>(x), max_iter, iters,
                                   static_cast<cudaStream_t>(stream)))
            rc = GC_ERR_NOT_CONVERGED;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_left_reach: max_iter reached before the fixpoint");
    return rc;
}

gc_status gc_left_sssp(gc_left_handle* h, const float* x0, float* x, int32_t max_iter, int32_t* iters,
                       void* stream) {
    gc_status rc = GC_OK;
    gc_status g = guard([&] {
        if (!h || !x0 || !x || !iters) fail(GC_ERR_ARG, "null argument");
        if (h->policy != GC_F32_MIN_PLUS) fail(GC_ERR_ARG, "gc_left_sssp needs the GC_F32_MIN_PLUS policy");
        if (h->n != h->m) fail(GC_ERR_ARG, "gc_left_sssp needs a square matrix");
        if (max_iter < 1) fail(GC_ERR_ARG, "max_iter must be >= 1");
        if (!left_fixpoint<LeftMinPlus>(h, x0, x, max_iter, iters, static_cast<cudaStream_t>(stream)))
            rc = GC_ERR_NOT_CONVERGED;
    });
    if (g != GC_OK) return g;
    if (rc != GC_OK) set_last_error("gc_left_sssp: max_iter reached before the fixpoint");
    return rc;
}

gc_status gc_left_launch_count(const gc_left_handle* h, int64_t* launches) {
    return guard([&] {
        if (!h || !launches) fail(GC_ERR_ARG, "null argument");
        *launches = h->launches;
    });
}

void gc_free_left_handle(gc_left_handle* h) { delete h; }

}  // extern "C"
