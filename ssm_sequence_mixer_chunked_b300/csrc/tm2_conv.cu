// tm2_conv.cu -- the size-2 causal input convolution of Mamba-2S, kept by 2Mamba
// ("2Mamba2Furious", Sec. 3: a convolution of kernel size 2 is, after the A-mask, the
// component that helps linear attention most; Sec. 4: window 2, no activation; App. A: at
// inference the previous window - 1 = 1 raw token is cached).  Per channel c of head h of
// q, k or v (a depthwise convolution over time):
//   y_t[c] = w[h][c][0] x_t[c] + w[h][c][1] x_{t-1}[c] (+ b[h][c]),   x_{-1} = x_prev or 0,
// and its backward
//   dx_t = w0 dy_t + w1 dy_{t+1} (dy_T = 0),   dx_prev = w1 dy_0,
//   dw0 = sum_{b,t} dy_t x_t,   dw1 = sum_{b,t} dy_t x_{t-1},   db = sum_{b,t} dy_t.
// Both passes are elementwise over (B, H, T, C) and bound by HBM bandwidth: each thread owns
// 8 consecutive channels (one 16-byte load of bf16) of one token.  The weight gradients are
// reduced per head by a cluster of 8 blocks over token splits (compensated fp32 sums per
// thread, double-float pairs above).
#include <algorithm>

#include <cooperative_groups.h>

#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

namespace cg = cooperative_groups;

template <typename Tin>
TM2_DEV void ld8(const Tin* p, float* x);
template <>
TM2_DEV void ld8<float>(const float* p, float* x) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
TM2_DEV void ld8<__nv_bfloat16>(const __nv_bfloat16* p, float* x) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
template <typename Tout>
TM2_DEV void st8(Tout* p, const float* x);
template <>
TM2_DEV void st8<float>(float* p, const float* x) {
    reinterpret_cast<float4*>(p)[0] = make_float4(x[0], x[1], x[2], x[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(x[4], x[5], x[6], x[7]);
}
TM2_DEV uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
TM2_DEV void st8<__nv_bfloat16>(__nv_bfloat16* p, const float* x) {
    uint4 u;
    u.x = bf16x2_bits(x[0], x[1]);
    u.y = bf16x2_bits(x[2], x[3]);
    u.z = bf16x2_bits(x[4], x[5]);
    u.w = bf16x2_bits(x[6], x[7]);
    *reinterpret_cast<uint4*>(p) = u;
}

// y (B,H,T,C) in the input type from x (B,H,T,C): one thread per (token, 8 channels).
template <typename Tin>
__global__ void conv2_fwd_kernel(const Tin* __restrict__ x, const float* __restrict__ w, const float* __restrict__ b,
                                 const Tin* __restrict__ x_prev, Tin* __restrict__ y, long BH, int H, int T, int C) {
    const int P = C / 8;
    const long total = BH * (long)T * P;
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long)gridDim.x * blockDim.x) {
        const int pc = (int)(e % P);
        const long tok = e / P;
        const int t = (int)(tok % T);
        const long bh = tok / T;
        const int h = (int)(bh % H);
        float cur[8], prv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, out[8], wv[16], bv[8];
        ld8(x + tok * C + 8 * pc, cur);
        if (t > 0) ld8(x + (tok - 1) * C + 8 * pc, prv);
        else if (x_prev) ld8(x_prev + bh * C + 8 * pc, prv);
        ld8(w + ((long)h * C + 8 * pc) * 2, wv);   // (w0, w1) of the 8 channels
        ld8(w + ((long)h * C + 8 * pc) * 2 + 8, wv + 8);
        if (b) ld8(b + (long)h * C + 8 * pc, bv);
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = fmaf(wv[2 * i], cur[i], wv[2 * i + 1] * prv[i]) + (b ? bv[i] : 0.f);
        st8(y + tok * C + 8 * pc, out);
    }
}

// dx (B,H,T,C) fp32 and, optionally, dx_prev (B,H,C) fp32.
template <typename Tin>
__global__ void conv2_bwd_dx_kernel(const Tin* __restrict__ dy, const float* __restrict__ w, float* __restrict__ dx,
                                    float* __restrict__ dx_prev, long BH, int H, int T, int C) {
    const int P = C / 8;
    const long total = BH * (long)T * P;
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long)gridDim.x * blockDim.x) {
        const int pc = (int)(e % P);
        const long tok = e / P;
        const int t = (int)(tok % T);
        const long bh = tok / T;
        const int h = (int)(bh % H);
        float g0[8], g1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, out[8], wv[16];
        ld8(dy + tok * C + 8 * pc, g0);
        if (t + 1 < T) ld8(dy + (tok + 1) * C + 8 * pc, g1);
        ld8(w + ((long)h * C + 8 * pc) * 2, wv);
        ld8(w + ((long)h * C + 8 * pc) * 2 + 8, wv + 8);
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = fmaf(wv[2 * i], g0[i], wv[2 * i + 1] * g1[i]);
        st8(dx + tok * C + 8 * pc, out);
        if (t == 0 && dx_prev) {
#pragma unroll
            for (int i = 0; i < 8; ++i) out[i] = wv[2 * i + 1] * g0[i];
            st8(dx_prev + bh * C + 8 * pc, out);
        }
    }
}

// dw (H,C,2), db (H,C) (optional).  One cluster of DW_SPLIT blocks per head, grid
// (DW_SPLIT, H), DW_THREADS threads: block rank sp sums the (b, t) items
// [n sp / DW_SPLIT, n (sp + 1) / DW_SPLIT) of the head, n = B T; thread (token lane tl,
// channel group cg of 8 channels, one 16-byte load of bf16) takes every NL-th item and keeps
// its 24 sums in fp32 with Neumaier's compensation (the products dy x rounded once each).
// The token lanes of a warp are then added as double-float pairs by a butterfly, the warps
// in warp order, and block rank 0 adds the blocks' sums in rank order through distributed
// shared memory and writes the head's gradients: deterministic, no scratch in global memory.
constexpr int DW_SPLIT = 8, DW_THREADS = 512;

struct comp32 {   // Neumaier-compensated fp32 sum: s + c
    float s = 0.f, c = 0.f;
    TM2_DEV void add(float x) {
        const float t = s + x;
        c += fabsf(s) >= fabsf(x) ? (s - t) + x : (x - t) + s;
        s = t;
    }
};

TM2_DEV df32 df_shfl_xor(df32 v, int o) {
    return {__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

template <typename Tin>
__global__ void __cluster_dims__(DW_SPLIT, 1, 1) __launch_bounds__(DW_THREADS)
    conv2_bwd_dw_kernel(const Tin* __restrict__ x, const Tin* __restrict__ dy, const Tin* __restrict__ x_prev,
                        float* __restrict__ dw, float* __restrict__ db, int B, int H, int T, int C) {
    __shared__ df32 wred[DW_THREADS / 32][3][64];
    __shared__ df32 part[3][64];
    cg::cluster_group cluster = cg::this_cluster();
    const int h = blockIdx.y, sp = (int)cluster.block_rank(), tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = C / 8, cgp = tid % G, tl = tid / G, NL = DW_THREADS / G;
    const long n = (long)B * T, i0 = n * sp / DW_SPLIT, i1 = n * (sp + 1) / DW_SPLIT;
    comp32 s0[8], s1[8], sb[8];
    for (long i = i0 + tl; i < i1; i += NL) {
        const int bb = (int)(i / T), t = (int)(i % T);
        const long bh = (long)bb * H + h, tok = bh * T + t;
        float g[8], xc[8], xp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        ld8(dy + tok * C + 8 * cgp, g);
        ld8(x + tok * C + 8 * cgp, xc);
        if (t > 0) ld8(x + (tok - 1) * C + 8 * cgp, xp);
        else if (x_prev) ld8(x_prev + bh * C + 8 * cgp, xp);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s0[j].add(__fmul_rn(g[j], xc[j]));   // (never contracted into the compensated add)
            s1[j].add(__fmul_rn(g[j], xp[j]));
            sb[j].add(g[j]);
        }
    }
    // the warp's token lanes (lanes with the same channel group: lane mod G) as pairs
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        df32 v[3] = {df_two_sum(s0[j].s, s0[j].c), df_two_sum(s1[j].s, s1[j].c), df_two_sum(sb[j].s, sb[j].c)};
        for (int o = G; o < 32; o <<= 1)
#pragma unroll
            for (int k = 0; k < 3; ++k) v[k] = df_add(v[k], df_shfl_xor(v[k], o));
        if (lane < G)
#pragma unroll
            for (int k = 0; k < 3; ++k) wred[warp][k][8 * cgp + j] = v[k];
    }
    __syncthreads();
    const int k = tid / C, cc = tid % C;
    if (tid < 3 * C) {
        df32 acc = wred[0][k][cc];
        for (int q = 1; q < DW_THREADS / 32; ++q) acc = df_add(acc, wred[q][k][cc]);
        part[k][cc] = acc;
    }
    cluster.sync();   // every block's sums are in its shared memory
    if (sp == 0 && tid < 3 * C) {
        df32 acc = part[k][cc];
        for (int q = 1; q < DW_SPLIT; ++q) acc = df_add(acc, cluster.map_shared_rank(&part[0][0], q)[k * 64 + cc]);
        const float v = acc.hi + acc.lo;
        if (k < 2) dw[((long)h * C + cc) * 2 + k] = v;
        else if (db) db[(long)h * C + cc] = v;
    }
    cluster.sync();   // no block leaves while rank 0 reads its shared memory
}

static unsigned grid_for(long total) {
    return (unsigned)std::max<long>(1, std::min<long>((total + 255) / 256, 148L * 16));
}

cudaError_t launch_conv2_fwd(long BH, int H, int T, int C, int dtype, const void* x, const float* w, const float* b,
                             const void* x_prev, void* y, cudaStream_t s) {
    const long total = BH * (long)T * (C / 8);
    if (total == 0) return cudaSuccess;
    if (dtype == 1)
        conv2_fwd_kernel<__nv_bfloat16><<<grid_for(total), 256, 0, s>>>(
            (const __nv_bfloat16*)x, w, b, (const __nv_bfloat16*)x_prev, (__nv_bfloat16*)y, BH, H, T, C);
    else
        conv2_fwd_kernel<float><<<grid_for(total), 256, 0, s>>>((const float*)x, w, b, (const float*)x_prev,
                                                               (float*)y, BH, H, T, C);
    return cudaGetLastError();
}

cudaError_t launch_conv2_bwd(int B, int H, int T, int C, int dtype, const void* x, const float* w,
                             const void* x_prev, const void* dy, float* dx, float* dx_prev, float* dw, float* db,
                             cudaStream_t s) {
    const long BH = (long)B * H;
    const long total = BH * (long)T * (C / 8);
    if (total == 0) return cudaSuccess;
    const dim3 gw(DW_SPLIT, H);
    if (dtype == 1) {
        conv2_bwd_dx_kernel<__nv_bfloat16><<<grid_for(total), 256, 0, s>>>((const __nv_bfloat16*)dy, w, dx, dx_prev,
                                                                          BH, H, T, C);
        conv2_bwd_dw_kernel<__nv_bfloat16><<<gw, DW_THREADS, 0, s>>>((const __nv_bfloat16*)x, (const __nv_bfloat16*)dy,
                                                              (const __nv_bfloat16*)x_prev, dw, db, B, H, T, C);
    } else {
        conv2_bwd_dx_kernel<float><<<grid_for(total), 256, 0, s>>>((const float*)dy, w, dx, dx_prev, BH, H, T, C);
        conv2_bwd_dw_kernel<float><<<gw, DW_THREADS, 0, s>>>((const float*)x, (const float*)dy, (const float*)x_prev, dw, db,
                                                      B, H, T, C);
    }
    return cudaGetLastError();
}

}  // namespace tm2
