// Leaf / combine / emit policies of the sweep (Sec. 5 of the pages: the
// schedule needs only an associative combine, so swapping these evaluates
// any monoid homomorphism over the grammar).
//
// A node value is LPN lanes of type V:
//   F32   (+, x) float32, one right-hand side          V = float,  LPN = 1
//   F32xN  (+, x) float32, k = 4 LPN right-hand sides   V = float4, LPN = k / 4
//          (Appendix A batched product: k = 4 .. 128; F32x16 is LPN = 4,
//          64 B per node in four float4 lanes)
//   F32x256 (+, x) float32, 256 right-hand sides        V = F8 (8 floats), LPN = 32
//   I64   (+, x) exact int64                            V = int64,  LPN = 1
//   OR    (OR, AND) on 64 sources per uint64 word       V = uint64, LPN = 1
//   MinPlus   tropical (min, +) float32, one right-hand side      V = float
//   MinPlusx16 the same on 16 right-hand sides                      V = float4
// The leaf map is V[l] (x) x[j] for the terminal <l, j>, evaluated where the
// sweep reads the terminal; the combine identity (0 for sums, all-zero bits
// for OR, +inf for min: the semiring zero, Sec. 5) stands in for a missing
// child.
#pragma once

#include <type_traits>

#include <cstdint>
#include <cuda_runtime.h>

namespace gcs {

struct PolF32 {
    using V = float;
    using Leaf = float;
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return 0.0f; }
    // explicitly rounded: no FMA contraction, so every kernel that evaluates
    // the same node gets the same bits
    __device__ __forceinline__ static V combine(V a, V b) { return __fadd_rn(a, b); }
    __device__ __forceinline__ static V leaf(Leaf v, V x) { return __fmul_rn(v, x); }
};

template <int LPN_>
struct PolF32xN {
    using V = float4;
    using Leaf = float;
    static constexpr int LPN = LPN_;
    __device__ __forceinline__ static V identity() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static V combine(V a, V b) {
        return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
    }
    __device__ __forceinline__ static V leaf(Leaf s, V x) {
        return make_float4(__fmul_rn(s, x.x), __fmul_rn(s, x.y), __fmul_rn(s, x.z), __fmul_rn(s, x.w));
    }
};

using PolF32x16 = PolF32xN<4>;

// Eight floats of a 256-wide value: one lane's part (32 lanes a node).
struct __align__(16) F8 {
    float4 lo, hi;
};

struct PolF32x256 {
    using V = F8;
    using Leaf = float;
    static constexpr int LPN = 32;
    __device__ __forceinline__ static V identity() {
        return F8{make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    }
    __device__ __forceinline__ static V combine(V a, V b) {
        return F8{PolF32x16::combine(a.lo, b.lo), PolF32x16::combine(a.hi, b.hi)};
    }
    __device__ __forceinline__ static V leaf(Leaf s, V x) { return F8{PolF32x16::leaf(s, x.lo), PolF32x16::leaf(s, x.hi)}; }
};

// Values of one scalar per node (one lane): the slice emit serves only these.
template <class P>
constexpr bool kScalarPolicy = P::LPN == 1 && sizeof(typename P::V) <= 8;

struct PolI64 {
    using V = long long;
    using Leaf = long long;
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return 0; }
    __device__ __forceinline__ static V combine(V a, V b) { return a + b; }
    __device__ __forceinline__ static V leaf(Leaf v, V x) { return v * x; }
};

struct PolOr {
    using V = unsigned long long;
    using Leaf = unsigned long long;   // every stored entry is 1: AND with all-ones
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return 0ull; }
    __device__ __forceinline__ static V combine(V a, V b) { return a | b; }
    __device__ __forceinline__ static V leaf(Leaf, V x) { return x; }
};

// Tropical: min is exact and each leaf sum is rounded once, so every order of
// evaluation gives the same bits. A leaf sum is never -0 (stored values are
// non-zero), so min never has to choose between two zeros.
struct PolMinPlus {
    using V = float;
    using Leaf = float;
    static constexpr int LPN = 1;
    __device__ __forceinline__ static V identity() { return __int_as_float(0x7f800000); }
    __device__ __forceinline__ static V combine(V a, V b) { return fminf(a, b); }
    __device__ __forceinline__ static V leaf(Leaf v, V x) { return __fadd_rn(v, x); }
};

struct PolMinPlusx16 {
    using V = float4;
    using Leaf = float;
    static constexpr int LPN = 4;
    __device__ __forceinline__ static V identity() {
        const float inf = __int_as_float(0x7f800000);
        return make_float4(inf, inf, inf, inf);
    }
    __device__ __forceinline__ static V combine(V a, V b) {
        return make_float4(fminf(a.x, b.x), fminf(a.y, b.y), fminf(a.z, b.z), fminf(a.w, b.w));
    }
    __device__ __forceinline__ static V leaf(Leaf s, V x) {
        return make_float4(__fadd_rn(s, x.x), __fadd_rn(s, x.y), __fadd_rn(s, x.z), __fadd_rn(s, x.w));
    }
};

// The policies the fixpoints run in, x = x (+) (M (x) x) with one value a
// node: reachability (OR) and shortest paths (min); (+) is P::combine.
template <class P>
constexpr bool kFixpointPolicy = std::is_same<P, PolOr>::value || std::is_same<P, PolMinPlus>::value;

}  // namespace gcs
