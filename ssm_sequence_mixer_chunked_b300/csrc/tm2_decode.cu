// tm2_decode.cu -- one recurrent decode step of the second-order state
// ("2Mamba2Furious", App. A: recurrent inference with a fixed-size state;
//  Sec. 2: the state has size (d^2, dv)):
//   gamma = exp(-softplus(a)),  S <- gamma S + (k (x) k) v^T,  z <- gamma z + k (x) k,
//   y = (q (x) q)^T S,  zeta = (q (x) q)^T z,  o = y / zeta (normalised) or y.
//
// The step is bound by HBM bandwidth: each (sequence, head) state of d^2 x dv fp32
// (1 MiB at d = dv = 64) is read once and written once, in place.  One 256-thread
// block per (sequence, head); a thread owns one float4 of value columns and walks
// every (256 / (dv/4))-th state row, with 8 rows' loads issued before any store so
// that each thread keeps 128 bytes in flight.  Loads and stores use the streaming
// cache hints (each byte is touched once per step).
#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

template <int D, int DV, typename Tin>
__global__ void __launch_bounds__(256) decode_step_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ a, float* __restrict__ S, float* __restrict__ z, float* __restrict__ o,
    float* __restrict__ Zout, bool normalize) {
    constexpr int NQ = DV / 4;        // float4 column groups per state row
    constexpr int RG = 256 / NQ;      // row groups
    constexpr int R = D * D;          // state rows
    constexpr int U = (R / RG) < 8 ? (R / RG) : 8;   // rows in flight per thread
    static_assert(R % (RG * U) == 0, "row count must tile");
    __shared__ float sq[D], sk[D], sv[DV];
    __shared__ float4 sred[RG][NQ];
    __shared__ float zred[8];
    const long s = blockIdx.x;
    const int tid = threadIdx.x;
    for (int e = tid; e < D; e += 256) {
        sq[e] = to_f(q[s * D + e]);
        sk[e] = to_f(k[s * D + e]);
    }
    for (int e = tid; e < DV; e += 256) sv[e] = to_f(v[s * DV + e]);
    const float gamma = __expf(-softplus_f(a[s]));
    __syncthreads();

    const int cq = tid % NQ, rg = tid / NQ;
    const float4 vq = make_float4(sv[4 * cq], sv[4 * cq + 1], sv[4 * cq + 2], sv[4 * cq + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4* Sp = reinterpret_cast<float4*>(S + s * (long)R * DV);
    for (int r0 = rg; r0 < R; r0 += RG * U) {
        float4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) x[u] = __ldcs(Sp + (long)(r0 + u * RG) * NQ + cq);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * RG;
            const int m = r / D, n = r % D;
            const float kk = sk[m] * sk[n], qq = sq[m] * sq[n];
            float4 y;
            y.x = fmaf(gamma, x[u].x, kk * vq.x);
            y.y = fmaf(gamma, x[u].y, kk * vq.y);
            y.z = fmaf(gamma, x[u].z, kk * vq.z);
            y.w = fmaf(gamma, x[u].w, kk * vq.w);
            __stcs(Sp + (long)r * NQ + cq, y);
            acc.x = fmaf(qq, y.x, acc.x);
            acc.y = fmaf(qq, y.y, acc.y);
            acc.z = fmaf(qq, y.z, acc.z);
            acc.w = fmaf(qq, y.w, acc.w);
        }
    }
    float zacc = 0.f;
    if (z) {
        float* zp = z + s * (long)R;
        for (int r = tid; r < R; r += 256) {
            const int m = r / D, n = r % D;
            const float zn = fmaf(gamma, __ldcs(zp + r), sk[m] * sk[n]);
            __stcs(zp + r, zn);
            zacc = fmaf(sq[m] * sq[n], zn, zacc);
        }
    }
    sred[rg][cq] = acc;
    zacc = warp_sum(zacc);
    if ((tid & 31) == 0) zred[tid >> 5] = zacc;
    __syncthreads();
    if (tid < NQ) {
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g2 = 0; g2 < RG; ++g2) {
            const float4 t = sred[g2][tid];
            y.x += t.x; y.y += t.y; y.z += t.z; y.w += t.w;
        }
        float ze = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) ze += zred[w];
        const float inv = (normalize && ze != 0.f) ? 1.f / ze : (normalize ? 0.f : 1.f);
        reinterpret_cast<float4*>(o + s * DV)[tid] = make_float4(y.x * inv, y.y * inv, y.z * inv, y.w * inv);
        if (tid == 0 && Zout) Zout[s] = ze;
    }
}

cudaError_t launch_decode_step(int N, int H, int d, int dv, int dtype, bool normalize,
                               const void* q, const void* k, const void* v, const float* a,
                               float* S, float* z, void* o, float* Z, cudaStream_t s) {
    const unsigned blocks = (unsigned)((long)N * H);
#define TM2_DECODE(D, T)                                                                         \
    decode_step_kernel<D, D, T><<<blocks, 256, 0, s>>>((const T*)q, (const T*)k, (const T*)v, a, \
                                                        S, z, (float*)o, Z, normalize)
    if (dtype == 1) {
        if (d == 64) TM2_DECODE(64, __nv_bfloat16);
        else if (d == 32) TM2_DECODE(32, __nv_bfloat16);
        else TM2_DECODE(16, __nv_bfloat16);
    } else {
        if (d == 64) TM2_DECODE(64, float);
        else if (d == 32) TM2_DECODE(32, float);
        else TM2_DECODE(16, float);
    }
#undef TM2_DECODE
    (void)dv;
    return cudaGetLastError();
}

}  // namespace tm2
