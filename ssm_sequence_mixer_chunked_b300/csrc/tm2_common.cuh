// tm2_common.cuh -- device helpers shared by the libtm2 kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define TM2_DEV __device__ __forceinline__

namespace tm2 {

// ---- element conversion -------------------------------------------------------------
TM2_DEV float to_f(float x) { return x; }
TM2_DEV float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> TM2_DEV T from_f(float x);
template <> TM2_DEV float from_f<float>(float x) { return x; }
template <> TM2_DEV __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---- the A-mask ----------------------------------------------------------------------
// softplus(x) = log(1 + e^x) in the overflow-free form max(x,0) + log1p(e^-|x|).
TM2_DEV float softplus_f(float x) { return fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x))); }
TM2_DEV float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }

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

}  // namespace tm2
