// Host driver of the device-side fixpoint loops (right and left products).
//
// The iteration x <- x (+) (M (x) x) is enqueued in batches of 1, 2, 4, 8, 8,
// ... products, each product followed by the update step whose last CTA
// records convergence in four device words (changed, converged, CTAs done,
// product count). After each batch the words are copied into pinned host
// memory and an event is recorded. The driver keeps one batch enqueued ahead
// of the one it waits for, so the device never idles on a host round trip;
// once a batch reports convergence the kernels of the batch behind it return
// at once (they read the converged word), and the call returns without
// waiting for them.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

namespace gcs {

// Pinned words and events of one handle's fixpoint loop, made on first use.
struct LoopHost {
    int32_t* words = nullptr;   // 2 slots x 4 words, pinned
    cudaEvent_t ev[2] = {nullptr, nullptr};
    cudaEvent_t end = nullptr;   // recorded after all the work of the last call
    bool ended = false;

    ~LoopHost() {
        // teardown errors (a context already gone at exit) are ignored; the
        // last call's copies into the words end before they are freed
        if (ended) (void)cudaEventSynchronize(end);
        if (words) (void)cudaFreeHost(words);
        for (cudaEvent_t e : ev)
            if (e) (void)cudaEventDestroy(e);
        if (end) (void)cudaEventDestroy(end);
    }
};

// Work enqueued on st after this call starts after the whole of the handle's
// previous fixpoint call (which may still be running the early-return kernels
// of its last batch when it has returned). Every entry point of a handle that
// enqueues work calls it first.
template <class Check>
void after_last_loop(const LoopHost& lh, cudaStream_t st, Check&& check) {
    if (lh.ended) check(cudaStreamWaitEvent(st, lh.end, 0), "wait for the previous fixpoint loop");
}

// Marks the end of a fixpoint call: after drive_fixpoint and whatever the
// caller enqueued behind it.
template <class Check>
void mark_loop_end(LoopHost& lh, cudaStream_t st, Check&& check) {
    check(cudaEventRecord(lh.end, st), "loop end record");
    lh.ended = true;
}

// step(it) enqueues product number it (1-based) and its update step on st.
// Returns true on convergence with *result = the product count the device
// recorded; false (result -1) when max_iter products did not converge.
// check(err, what) throws on a CUDA error. The caller resets the words ctl
// points to (on st, after after_last_loop) before the call and calls
// mark_loop_end after it, also when it throws.
template <class Check, class Step>
bool drive_fixpoint(LoopHost& lh, const int32_t* ctl, int32_t max_iter, cudaStream_t st, Check&& check, Step&& step,
                    int32_t* result) {
    if (!lh.words) {
        void* p = nullptr;
        check(cudaHostAlloc(&p, 8 * sizeof(int32_t), cudaHostAllocDefault), "loop words (pinned)");
        lh.words = static_cast<int32_t*>(p);
        for (cudaEvent_t& e : lh.ev) check(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "loop event");
        check(cudaEventCreateWithFlags(&lh.end, cudaEventDisableTiming), "loop event");
    }
    int32_t it = 0, batch = 1;
    int slot = 0, oldest = 0, pending = 0;
    auto enqueue = [&] {
        const int32_t nb = std::min(batch, max_iter - it);
        for (int32_t j = 0; j < nb; ++j) step(++it);
        check(cudaGetLastError(), "kernel launch");
        check(cudaMemcpyAsync(lh.words + 4 * slot, ctl, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, st),
              "loop words read");
        check(cudaEventRecord(lh.ev[slot], st), "loop event record");
        slot ^= 1;
        ++pending;
        batch = std::min(batch * 2, 8);
    };
    *result = -1;
    if (it < max_iter) enqueue();
    while (pending > 0) {
        if (it < max_iter && pending < 2) enqueue();
        check(cudaEventSynchronize(lh.ev[oldest]), "loop event wait");
        const int32_t* w = lh.words + 4 * oldest;
        oldest ^= 1;
        --pending;
        if (w[1]) {
            *result = w[3];
            return true;
        }
    }
    return false;
}

}  // namespace gcs
