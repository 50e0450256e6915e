// Leaf / combine / emit policies of the sweep (Sec. 5 of the pages: the
// schedule needs only an associative combine, so swapping these evaluates
// any monoid homomorphism over the grammar).
//
// A node value is LPN lanes of type V:
//   F32   (+, x) float32, one right-hand side          V = float,  LPN = 1
//   F32x16 (+, x) float32, 16 right-hand sides          V = float4, LPN = 4
//          (Appendix A batched product; 64 B per node, four float4 lanes)
//   I64   (+, x) exact int64                            V = int64,  LPN = 1
//   OR    (OR, AND) on 64 sources per uint64 word       V = uint64, LPN = 1
// The leaf map is T[p] = V[l_p] (x) x[j_p]; the combine identity fills T[0]
// (0 for sums, all-zero bits for OR: the semiring zero, Sec. 5).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gcs {

struct PolF32 {
    using V = float;
    using Leaf = float;
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return 0.0f; }
    __device__ __forceinline__ static V combine(V a, V b) { return a + b; }
    __device__ __forceinline__ static V leaf(const Leaf* lv, int64_t p, V x) { return lv[p] * x; }
};

struct PolF32x16 {
    using V = float4;
    using Leaf = float;
    static constexpr int LPN = 4;
    __device__ __forceinline__ static V identity() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static V combine(V a, V b) {
        return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    }
    __device__ __forceinline__ static V leaf(const Leaf* lv, int64_t p, V x) {
        float s = lv[p];
        return make_float4(s * x.x, s * x.y, s * x.z, s * x.w);
    }
};

struct PolI64 {
    using V = long long;
    using Leaf = long long;
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return 0; }
    __device__ __forceinline__ static V combine(V a, V b) { return a + b; }
    __device__ __forceinline__ static V leaf(const Leaf* lv, int64_t p, V x) { return lv[p] * x; }
};

struct PolOr {
    using V = unsigned long long;
    using Leaf = unsigned long long;   // unused: every stored entry is 1
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return 0ull; }
    __device__ __forceinline__ static V combine(V a, V b) { return a | b; }
    __device__ __forceinline__ static V leaf(const Leaf*, int64_t, V x) { return x; }
};

}  // namespace gcs
