// tm2_common.cuh -- device helpers shared by the libtm2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define TM2_DEV __device__ __forceinline__

// Bounds-checked build (-DTM2_DEBUG): TM2_CHECK(cond, status) is cond, and a false cond also
// records TM2_ERR_BOUNDS (-7) in the device status word `status` unless it already holds a
// status; the caller skips the access it guards (no trap, no assert).  Without TM2_DEBUG it is
// the constant true and costs nothing.
#ifdef TM2_DEBUG
#define TM2_CHECK(cond, status) (::tm2_debug_check((cond), (status)))
__device__ __forceinline__ bool tm2_debug_check(bool ok, int* status) {
    if (!ok && status) atomicCAS(status, 0, -7);
    return ok;
}
#else
#define TM2_CHECK(cond, status) true
#endif

namespace tm2 {

// ---- element conversion -------------------------------------------------------------
TM2_DEV float to_f(float x) { return x; }
TM2_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> TM2_DEV T from_f(float x);
template <> TM2_DEV float from_f<float>(float x) { return x; }
template <> TM2_DEV __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// element i of an output that is fp32, or of the input type T when lowp (the gradients'
// TM2_GRADS_INPUT_DTYPE form)
template <typename T> TM2_DEV void store_out(void* p, long i, float x, bool lowp) {
    if (lowp) reinterpret_cast<T*>(p)[i] = from_f<T>(x);
    else reinterpret_cast<float*>(p)[i] = x;
}

// ---- the A-mask ----------------------------------------------------------------------
// softplus(x) = log(1 + e^x) in the overflow-free form max(x,0) + log1p(e^-|x|).
TM2_DEV float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x))); }
TM2_DEV float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }

// ---- power-of-two operand scales ---------------------------------------------------------
// The factor 2^-e that brings a non-negative maximum m = f 2^e (f in [0.5, 1)) into [0.5, 1),
// from m's fp32 bit pattern; 1 when m is 0, subnormal-free zero, infinite or NaN.  e is
// clamped to [-40, 40], so products of a few such factors stay inside fp32.  Multiplying by
// it is exact, so a value scaled on the way into a 16-bit operand and unscaled afterwards is
// unchanged unless the unscaled value would have left the 16-bit range.
TM2_DEV float pow2_scale(uint32_t maxbits) {
    const float m = __uint_as_float(maxbits);
    if (!(m > 0.f) || !(m < INFINITY)) return 1.f;
    int e = (int)((maxbits >> 23) & 0xffu) - 126;
    e = max(-40, min(40, e));
    return __uint_as_float((uint32_t)(127 - e) << 23);
}

// ---- warp reductions -----------------------------------------------------------------
TM2_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
TM2_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// inclusive prefix sum over the 32 lanes of a warp
TM2_DEV float warp_inclusive_scan(float v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Double-float sums (an unevaluated pair hi + lo of fp32 values, about 48 significant bits)
// for long reductions (the reverse sums of the A-mask gradient, the convolution's weight
// gradients): the error-free sum of two floats is Knuth's TwoSum, and the pair is renormalised
// with Dekker's Fast2Sum.  fp64 arithmetic would do as well but runs at a small fraction of
// the fp32 rate on this part; these are plain fp32 adds and subtracts (no products, so
// nothing can be contracted into an FMA).  Used only in sources built without fast math.
struct df32 {
    float hi, lo;
};
TM2_DEV df32 df_two_sum(float a, float b) {
    const float s = a + b, bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}
TM2_DEV df32 df_fast_two_sum(float a, float b) {   // |a| >= |b|
    const float s = a + b;
    return {s, b - (s - a)};
}
// Sum of two pairs with both the high and the low parts added error-free, so that the
// cancelling sums stay accurate relative to the result.
TM2_DEV df32 df_add(df32 x, df32 y) {
    const df32 s = df_two_sum(x.hi, y.hi), t = df_two_sum(x.lo, y.lo);
    df32 r = df_fast_two_sum(s.hi, s.lo + t.hi);
    return df_fast_two_sum(r.hi, r.lo + t.lo);
}
// The exact product of two floats as a pair (the FMA form of Dekker's TwoProduct).
TM2_DEV df32 df_two_prod(float a, float b) {
    const float p = a * b;
    return {p, fmaf(a, b, -p)};
}

}  // namespace tm2
