// tm2_scan.cu -- the fp32 A-mask kernels: chunked running sums of -softplus(a)
// ("2Mamba2Furious", Sec. 3/4: the softplus A-mask; the decay running sum always
// runs in fp32), the reverse running sum that turns dL/dcumA into dL/da (App. C.1),
// and small per-token preparation kernels of the backward passes.
#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

// Block-wide inclusive scan of one value per thread (blockDim.x <= 1024).
TM2_DEV float block_inclusive_scan(float v, float* wsum /* >= 32 floats */) {
    const int t = threadIdx.x, w = t >> 5, lane = t & 31, nw = (blockDim.x + 31) >> 5;
    float s = warp_inclusive_scan(v);
    if (lane == 31) wsum[w] = s;
    __syncthreads();
    if (w == 0) {
        float x = lane < nw ? wsum[lane] : 0.f;
        x = warp_inclusive_scan(x);
        wsum[lane] = x;
    }
    __syncthreads();
    if (w > 0) s += wsum[w - 1];
    __syncthreads();
    return s;
}

// (double-float pairs: tm2_common.cuh)
TM2_DEV df32 df_shfl_up(df32 v, int o) {
    return {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
TM2_DEV df32 block_inclusive_scan_df(df32 v, df32* wsum /* >= 32 */) {
    const int t = threadIdx.x, w = t >> 5, lane = t & 31, nw = (blockDim.x + 31) >> 5;
    df32 s = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const df32 u = df_shfl_up(s, o);
        if (lane >= o) s = df_add(s, u);
    }
    if (lane == 31) wsum[w] = s;
    __syncthreads();
    if (w == 0) {
        df32 x = lane < nw ? wsum[lane] : df32{0.f, 0.f};
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const df32 u = df_shfl_up(x, o);
            if (lane >= o) x = df_add(x, u);
        }
        wsum[lane] = x;
    }
    __syncthreads();
    if (w > 0) s = df_add(s, wsum[w - 1]);
    __syncthreads();
    return s;
}

// grid (NC, BH), block C threads: one chunk per block.
__global__ void decay_chunk_kernel(const float* __restrict__ a, float* __restrict__ Aloc,
                                   float* __restrict__ g, int T, int C, int NC) {
    __shared__ float wsum[32];
    const int c = blockIdx.x, t = threadIdx.x;
    const long bh = blockIdx.y;
    const long tok = (long)c * C + t;
    const float l = tok < T ? -softplus_f(a[bh * T + tok]) : 0.f;
    const float s = block_inclusive_scan(l, wsum);
    Aloc[bh * (long)NC * C + tok] = s;
    const int last = min(C, T - c * C) - 1;
    if (t == last) g[bh * NC + c] = s;
}

cudaError_t launch_decay(const Problem& p, const float* a, float* Aloc, float* g, cudaStream_t s) {
    dim3 grid(p.NC, (unsigned)p.BH());
    decay_chunk_kernel<<<grid, p.C, 0, s>>>(a, Aloc, g, p.T, p.C, p.NC);
    return cudaGetLastError();
}

// grid (ceil(T / GC_TOK), BH), block 256: each block writes the running sums of GC_TOK tokens.
// The offset at the start of chunk c is the fp64 sum of the chunk totals before it: a block
// reduction over the chunks before the tile, then one thread runs through the tile's own
// chunks, so only the final rounding to fp32 (and its residual cum_lo) enters cum.
constexpr int GC_TOK = 1024;

TM2_DEV double block_sum_d(double v, double* wsum /* >= 32 doubles */) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (blockDim.x + 31) >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) wsum[w] = v;
    __syncthreads();
    double t = 0.0;
    for (int i = 0; i < nw; ++i) t += wsum[i];
    __syncthreads();
    return t;
}

__global__ void __launch_bounds__(256) global_cumsum_kernel(const float* __restrict__ Aloc, const float* __restrict__ g,
                                                            float* __restrict__ cum, float* __restrict__ cum_lo, int T,
                                                            int C, int NC) {
    extern __shared__ double off[];   // offsets of the tile's chunks
    __shared__ double wsum[32];
    const long bh = blockIdx.y;
    const int t0 = blockIdx.x * GC_TOK, t1 = min(T, t0 + GC_TOK);
    const int c0 = t0 / C, c1 = (t1 - 1) / C;
    double before = 0.0;
    for (int c = threadIdx.x; c < c0; c += blockDim.x) before += (double)g[bh * NC + c];
    before = block_sum_d(before, wsum);
    if (threadIdx.x == 0) {
        double run = before;
        for (int c = c0; c <= c1; ++c) {
            off[c - c0] = run;
            run += (double)g[bh * NC + c];
        }
    }
    __syncthreads();
    for (int t = t0 + (int)threadIdx.x; t < t1; t += blockDim.x) {
        const double x = off[t / C - c0] + (double)Aloc[bh * (long)NC * C + t];
        const float hi = (float)x;
        cum[bh * T + t] = hi;
        if (cum_lo) cum_lo[bh * T + t] = (float)(x - (double)hi);
    }
}

cudaError_t launch_global_cumsum(const Problem& p, const float* Aloc, const float* g, float* cum, float* cum_lo,
                                 cudaStream_t s) {
    const size_t smem = sizeof(double) * (size_t)(GC_TOK / p.C + 2);
    dim3 grid((unsigned)((p.T + GC_TOK - 1) / GC_TOK), (unsigned)p.BH());
    global_cumsum_kernel<<<grid, 256, smem, s>>>(Aloc, g, cum, cum_lo, p.T, p.C, p.NC);
    return cudaGetLastError();
}

// grid (tiles, BH), block 1024: tile j holds the 1024 tokens ending at T - 1 - 1024 j (thread 0
// the latest).  Its carry is the sum over every later token, read directly (a block reduction:
// the later tokens of all tiles of a head total T^2 / 2048 reads, small next to the rest), so
// the tiles of a head run in parallel.  The sums are kept as double-float pairs: over
// thousands of tokens the terms largely cancel (their total is zero without an initial state),
// and an fp32 sum would leave a rounding error comparable to the result.  Each term
// row - col is formed exactly (TwoSum).
__global__ void __launch_bounds__(1024) reverse_cumsum_da_kernel(
    const float* __restrict__ a, const float* __restrict__ row, const float* __restrict__ col,
    float* __restrict__ da, int T) {
    __shared__ df32 wsum[32];
    __shared__ df32 carry_s;
    const int j = blockIdx.x;
    const long bh = blockIdx.y;
    const int top = T - 1 - 1024 * j;            // the latest token of this tile
    auto term = [&](int u) { return df_two_sum(row[bh * T + u], col ? -col[bh * T + u] : 0.f); };
    df32 part = {0.f, 0.f};
    for (int u = top + 1 + (int)threadIdx.x; u < T; u += blockDim.x) part = df_add(part, term(u));
    // block total of `part`: the last element of the inclusive scan
    const df32 run = block_inclusive_scan_df(part, wsum);
    if (threadIdx.x == blockDim.x - 1) carry_s = run;
    __syncthreads();
    const df32 carry = carry_s;
    __syncthreads();
    const int u = top - (int)threadIdx.x;
    const df32 x = u >= 0 ? term(u) : df32{0.f, 0.f};
    const df32 sres = df_add(block_inclusive_scan_df(x, wsum), carry);
    if (u >= 0) da[bh * T + u] = -sigmoid_f(a[bh * T + u]) * (sres.hi + sres.lo);
}

cudaError_t launch_reverse_cumsum_da(const Problem& p, const float* a, const float* row,
                                     const float* col, float* da, cudaStream_t s) {
    if (p.T <= 0 || p.BH() == 0) return cudaSuccess;
    dim3 grid((unsigned)((p.T + 1023) / 1024), (unsigned)p.BH());
    reverse_cumsum_da_kernel<<<grid, 1024, 0, s>>>(a, row, col, da, p.T);
    return cudaGetLastError();
}

// One warp per token: D = dO . o; dY = [dO/Z, -D/Z] (normalised) or [dO, 0];
// rowterm = dY . Y, which is exactly 0 when normalised (Y = [N, Z] and o = N/Z)
// and dO . o otherwise.
template <typename Tin>
__global__ void dy_prep_kernel(const float* __restrict__ o, const float* __restrict__ Z,
                               const Tin* __restrict__ dO, float* __restrict__ dY,
                               float* __restrict__ rowterm, long ntok, int dv, bool normalize) {
    const long tok = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= ntok) return;
    float D = 0.f;
    for (int c = lane; c < dv; c += 32) D += to_f(dO[tok * dv + c]) * o[tok * dv + c];
    D = warp_sum(D);
    const float z = normalize ? Z[tok] : 1.f;
    const float inv = (normalize && z != 0.f) ? 1.f / z : (normalize ? 0.f : 1.f);
    for (int c = lane; c < dv; c += 32) dY[tok * (dv + 1) + c] = to_f(dO[tok * dv + c]) * inv;
    if (lane == 0) {
        dY[tok * (dv + 1) + dv] = normalize ? -D * inv : 0.f;
        rowterm[tok] = normalize ? 0.f : D;
    }
}

cudaError_t launch_dy_prep(const Problem& p, const void* o, const float* Z, const void* dO,
                           float* dY, float* rowterm, cudaStream_t s) {
    const long ntok = p.BH() * p.T;
    const unsigned blocks = (unsigned)((ntok + 7) / 8);
    if (p.dtype == 1)
        dy_prep_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            (const float*)o, Z, (const __nv_bfloat16*)dO, dY, rowterm, ntok, p.dv, p.normalize);
    else
        dy_prep_kernel<float><<<blocks, 256, 0, s>>>((const float*)o, Z, (const float*)dO, dY,
                                                     rowterm, ntok, p.dv, p.normalize);
    return cudaGetLastError();
}

// Tensor-core backward preparation.  One block of 256 threads per (chunk, b, h), one warp
// per token at a time.  With D = dO . o:
//   zeta = 1/Z (normalised) or 1, ucol = -D (normalised) or 0, rowterm = 0 (normalised)
//   or D, so that dL/dY_i = zeta_i [dO_i, ucol_i];  zmax[c] = max over the chunk of
//   exp(A_i) zeta_i (the scale of the reverse state scan's generated operand).
__global__ void __launch_bounds__(256, 3) tc_dy_prep_kernel(const float* __restrict__ o, const float* __restrict__ Z,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         const float* __restrict__ Aloc, float* __restrict__ zeta,
                                                         float* __restrict__ ucol, float* __restrict__ rowterm,
                                                         float* __restrict__ zmax, unsigned* __restrict__ amax, int T,
                                                         int C, int NC, bool normalize) {
    __shared__ float wmax[8], wumax[8];
    const int c = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane >> 3, l8 = lane & 7;   // four tokens per warp pass, eight lanes per token
    const long bh = blockIdx.y;
    float mx = 0.f, umx = 0.f;
    constexpr int NP = 4;   // passes whose loads are in flight together
    for (int jp = 0; jp < C; jp += 32 * NP) {
        // elements 8*l8 .. 8*l8+7 of each pass's row: one 16-byte dO load, two 16-byte o loads
        uint4 d8[NP];
        float4 o0[NP], o1[NP];
        float zr[NP], ar[NP];
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const long t = (long)c * C + jp + 32 * k + warp * 4 + sub;
            const bool in = t < T && jp + 32 * k < C;
            const long tok = bh * T + (in ? t : 0);
            d8[k] = in ? *reinterpret_cast<const uint4*>(dO + tok * 64 + 8 * l8) : make_uint4(0, 0, 0, 0);
            o0[k] = in ? *reinterpret_cast<const float4*>(o + tok * 64 + 8 * l8) : make_float4(0.f, 0.f, 0.f, 0.f);
            o1[k] = in ? *reinterpret_cast<const float4*>(o + tok * 64 + 8 * l8 + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
            zr[k] = in && normalize ? Z[tok] : 1.f;
            ar[k] = in ? Aloc[bh * (long)NC * C + t] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const long t = (long)c * C + jp + 32 * k + warp * 4 + sub;
            const bool in = t < T && jp + 32 * k < C;
            const long tok = bh * T + (in ? t : 0);
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&d8[k]);
            const float2 f0 = __bfloat1622float2(b2[0]), f1 = __bfloat1622float2(b2[1]);
            const float2 f2 = __bfloat1622float2(b2[2]), f3 = __bfloat1622float2(b2[3]);
            float D = f0.x * o0[k].x + f0.y * o0[k].y + f1.x * o0[k].z + f1.y * o0[k].w + f2.x * o1[k].x +
                      f2.y * o1[k].y + f3.x * o1[k].z + f3.y * o1[k].w;
            D += __shfl_xor_sync(0xffffffffu, D, 1);
            D += __shfl_xor_sync(0xffffffffu, D, 2);
            D += __shfl_xor_sync(0xffffffffu, D, 4);
            if (in) {
                const float z = zr[k];
                const float ze = normalize ? (z != 0.f ? 1.f / z : 0.f) : 1.f;
                if (l8 == 0) {
                    zeta[tok] = ze;
                    ucol[tok] = normalize ? -D : 0.f;
                    rowterm[tok] = normalize ? 0.f : D;
                }
                mx = fmaxf(mx, __expf(ar[k]) * ze);
                if (normalize) umx = fmaxf(umx, fabsf(D));
            }
        }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    umx = fmaxf(umx, __shfl_xor_sync(0xffffffffu, umx, 8));
    umx = fmaxf(umx, __shfl_xor_sync(0xffffffffu, umx, 16));
    if (lane == 0) {
        wmax[warp] = mx;
        wumax[warp] = umx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f, um = 0.f;
        for (int w = 0; w < 8; ++w) {
            m = fmaxf(m, wmax[w]);
            um = fmaxf(um, wumax[w]);
        }
        zmax[bh * NC + c] = m > 0.f ? m : 1.f;
        atomicMax(amax + bh * 4 + 2, __float_as_uint(um));   // largest |ucol| of the head
    }
}

cudaError_t launch_tc_dy_prep(const Problem& p, const float* o, const float* Z, const void* dO, const float* Aloc,
                              float* zeta, float* ucol, float* rowterm, float* zmax, unsigned* amax, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned) * 4 * (size_t)p.BH(), s);
    if (e != cudaSuccess) return e;
    dim3 grid(p.NC, (unsigned)p.BH());
    tc_dy_prep_kernel<<<grid, 256, 0, s>>>(o, Z, (const __nv_bfloat16*)dO, Aloc, zeta, ucol, rowterm, zmax, amax, p.T,
                                          p.C, p.NC, p.normalize);
    return cudaGetLastError();
}

// Largest |x| of each (b, h) of two bf16 tensors (BH, T, 64), max-combined into amax[bh * 4]
// and amax[bh * 4 + 1] as fp32 bit patterns (non-negative floats order like their bits).
// grid (ceil(T / 128), BH), 256 threads: 128 tokens x 8 sixteen-byte pieces per block.
TM2_DEV uint32_t bf16x8_absmax_bits(uint4 a) {
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
    return m << 16;
}
__global__ void __launch_bounds__(256) head_absmax_kernel(const __nv_bfloat16* __restrict__ x,
                                                          const __nv_bfloat16* __restrict__ y,
                                                          unsigned* __restrict__ amax, int T) {
    __shared__ uint32_t red[2][8];
    const long bh = blockIdx.y;
    const long t0 = (long)blockIdx.x * 128;
    uint4 xr[4], yr[4];   // all eight 16-byte loads in flight before the reduction
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = threadIdx.x + 256 * i;
        const long t = t0 + (e >> 3);
        const long off = (bh * T + t) * 64 + 8 * (e & 7);
        xr[i] = t < T ? *reinterpret_cast<const uint4*>(x + off) : make_uint4(0, 0, 0, 0);
        yr[i] = t < T ? *reinterpret_cast<const uint4*>(y + off) : make_uint4(0, 0, 0, 0);
    }
    uint32_t mx = 0, my = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mx = max(mx, bf16x8_absmax_bits(xr[i]));
        my = max(my, bf16x8_absmax_bits(yr[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        my = max(my, __shfl_xor_sync(0xffffffffu, my, o));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[0][warp] = mx;
        red[1][warp] = my;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < 8; ++w) {
            mx = max(mx, red[0][w]);
            my = max(my, red[1][w]);
        }
        atomicMax(amax + bh * 4, mx);
        atomicMax(amax + bh * 4 + 1, my);
    }
}

cudaError_t launch_head_absmax(const Problem& p, const void* x, const void* y, unsigned* amax, bool zero_first,
                               cudaStream_t s) {
    if (zero_first) {
        cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(unsigned) * 4 * (size_t)p.BH(), s);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((p.T + 127) / 128), (unsigned)p.BH());
    head_absmax_kernel<<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, (const __nv_bfloat16*)y, amax, p.T);
    return cudaGetLastError();
}

// Operands of the tensor-core chunk-state scan, one thread per token (256 tokens per block of
// one (b, h)), written as one [144][64] fp16 block per 64-token stage (token j = stage*64 + column):
//   rows   0-63 : [n][j]   = fp16(ks key_j[n])         (the key block, transposed)
//   rows  64-127: [col][j] = fp16(vs w_j val_j[col])   (the weighted values, transposed)
//   row   128   : [j]      = fp16(zs w_j zc_j)         (the normaliser column)
//   rows 129-143: 0                                    (rows 64-143: the walk's N = 80 operand)
// with the scan's weight w_t = exp(g_c - A_t), zc = 1 (forward walk) or
// w_t = exp(A_t) zeta_t / zmax_c, zc = ucol_t (reverse walk); tokens past T give zeros.
// ks, vs, zs are the powers of two that bring the head's largest |key|, |val| and (reverse
// walk) |ucol| into [0.5, 1) (amax, from launch_head_absmax and launch_tc_dy_prep; zs = 1
// forward): the fp16 operands and the products k[m] k[n] then sit in fp16's normal range
// whatever the scale of the inputs, and the state comes out multiplied by ks^2 vs exactly.
__global__ void __launch_bounds__(256) tc_scan_operands_kernel(
    const __nv_bfloat16* __restrict__ key, const __nv_bfloat16* __restrict__ val, const float* __restrict__ Aloc,
    const float* __restrict__ g, const float* __restrict__ zeta, const float* __restrict__ ucol,
    const float* __restrict__ zmax, const unsigned* __restrict__ amax, __half* __restrict__ ops, int T, int C, int NC,
    int rev) {
    // one token per thread, one warp per 32 tokens (half a stage); the transposition goes
    // through registers: the lanes of a pair trade halves so that each writes two adjacent
    // tokens of one row (even lane: row 2p, odd lane: row 2p + 1), 128 bytes per warp store
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long bh = blockIdx.y;
    const int Tp = NC * C;
    const long tw = (long)blockIdx.x * 256 + warp * 32;   // the warp's first token
    if (tw >= Tp) return;
    const long t = tw + lane;
    const int st = (int)(tw / 64), c = (int)(t / C);
    const bool in = t < T;
    // the token's key and value rows first (16 loads in flight), then its weight's terms
    uint4 kr[8], vr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        kr[i] = in ? reinterpret_cast<const uint4*>(key + (bh * T + t) * 64)[i] : make_uint4(0, 0, 0, 0);
        vr[i] = in ? reinterpret_cast<const uint4*>(val + (bh * T + t) * 64)[i] : make_uint4(0, 0, 0, 0);
    }
    const float ks = pow2_scale(amax[bh * 4]), vs = pow2_scale(amax[bh * 4 + 1]);
    const float zs = rev ? pow2_scale(amax[bh * 4 + 2]) : 1.f;
    const float A = Aloc[bh * Tp + t];
    float w = 0.f, zc = 0.f;
    if (rev) {
        if (in) {
            w = __expf(A) * zeta[bh * T + t] / zmax[bh * NC + c];
            zc = ucol[bh * T + t];
        }
    } else {
        w = in ? __expf(g[bh * NC + c] - A) : 0.f;
        zc = 1.f;
    }
    const float wv = vs * w;
    // fp16(ks key[n]) and fp16(vs w val[col]) as half2 words (element pairs 2p, 2p + 1)
    uint32_t kh[32], vh[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __nv_bfloat162* kb = reinterpret_cast<const __nv_bfloat162*>(&kr[i]);
        const __nv_bfloat162* vb = reinterpret_cast<const __nv_bfloat162*>(&vr[i]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 kk = __bfloat1622float2(kb[u]), vv = __bfloat1622float2(vb[u]);
            const __half2 hk = __floats2half2_rn(kk.x * ks, kk.y * ks);
            const __half2 hv = __floats2half2_rn(vv.x * wv, vv.y * wv);
            kh[4 * i + u] = *reinterpret_cast<const uint32_t*>(&hk);
            vh[4 * i + u] = *reinterpret_cast<const uint32_t*>(&hv);
        }
    }
    __half* blk = ops + (bh * (Tp / 64) + st) * (long)(TC_OPS_ROWS * 64);
    const bool odd = lane & 1;
    const int j = (int)(tw % 64) + (lane & ~1);   // the pair's first token column in the stage
    uint32_t* rk = reinterpret_cast<uint32_t*>(blk + (odd ? 64 : 0) + j);         // row 2p (+1 odd) at 128 p
    uint32_t* rv = reinterpret_cast<uint32_t*>(blk + 64 * 64 + (odd ? 64 : 0) + j);
#pragma unroll
    for (int q = 0; q < 32; ++q) {
        const uint32_t sk = odd ? (kh[q] & 0xffffu) : (kh[q] >> 16);   // what the partner lane needs
        const uint32_t sv = odd ? (vh[q] & 0xffffu) : (vh[q] >> 16);
        const uint32_t gk = __shfl_xor_sync(0xffffffffu, sk, 1), gv = __shfl_xor_sync(0xffffffffu, sv, 1);
        rk[q * 64] = odd ? (gk | (kh[q] & 0xffff0000u)) : ((kh[q] & 0xffffu) | (gk << 16));
        rv[q * 64] = odd ? (gv | (vh[q] & 0xffff0000u)) : ((vh[q] & 0xffffu) | (gv << 16));
    }
    // the normaliser row (even lanes, two tokens a word) and this half-stage's part of the zero rows
    const __half hz = __float2half_rn(zs * w * zc);
    const uint32_t zb = *reinterpret_cast<const unsigned short*>(&hz);
    const uint32_t zo = __shfl_xor_sync(0xffffffffu, zb, 1);
    if (!odd) reinterpret_cast<uint32_t*>(blk + 128 * 64 + j)[0] = zb | (zo << 16);
    const int half = (int)(tw % 64) / 32;
    for (int e = lane; e < (TC_OPS_ROWS - 129) * 4; e += 32)   // 15 rows x 64 bytes, 16 bytes a store
        reinterpret_cast<uint4*>(blk + (129 + e / 4) * 64 + 32 * half)[e & 3] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_tc_scan_operands(const Problem& p, bool rev, const void* key, const void* val, const float* Aloc,
                                    const float* g, const float* zeta, const float* ucol, const float* zmax,
                                    const unsigned* amax, void* ops, cudaStream_t s) {
    dim3 grid((unsigned)((p.Tp() + 255) / 256), (unsigned)p.BH());
    tc_scan_operands_kernel<<<grid, 256, 0, s>>>((const __nv_bfloat16*)key, (const __nv_bfloat16*)val, Aloc, g, zeta,
                                                 ucol, zmax, amax, (__half*)ops, p.T, p.C, p.NC, rev ? 1 : 0);
    return cudaGetLastError();
}

// Backward preparation, one warp per token: D = dO . o (rowdot), and for the quadratic-form
// mixers zeta = 1/Z (0 where Z = 0) and D when normalised, D = 0 and zeta = 1 otherwise.
template <typename Tin, bool POLY>
__global__ void prep_kernel(const float* __restrict__ o, const float* __restrict__ Z, const Tin* __restrict__ dO,
                            float* __restrict__ Dv, float* __restrict__ zeta, long ntok, int dv, bool normalize) {
    const long tok = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= ntok) return;
    float D = 0.f;
    if (!POLY || normalize) {
        for (int c = lane; c < dv; c += 32) D += to_f(dO[tok * dv + c]) * o[tok * dv + c];
        D = warp_sum(D);
    }
    if (lane == 0) {
        Dv[tok] = D;
        if (POLY) {
            const float z = normalize ? Z[tok] : 1.f;
            zeta[tok] = z != 0.f ? 1.f / z : 0.f;
        }
    }
}

// The same for dv = 64 with 16-byte aligned rows: eight threads per token, eight elements each
// (one 16-byte load of bf16 dO, or two of fp32, and two of o), combined by shuffles.
TM2_DEV void load8(const __nv_bfloat16* p, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
TM2_DEV void load8(const float* p, float* f) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    f[0] = a.x, f[1] = a.y, f[2] = a.z, f[3] = a.w, f[4] = b.x, f[5] = b.y, f[6] = b.z, f[7] = b.w;
}

template <typename Tin, bool POLY>
__global__ void __launch_bounds__(256) prep64_kernel(const float* __restrict__ o, const float* __restrict__ Z,
                                                     const Tin* __restrict__ dO, float* __restrict__ Dv,
                                                     float* __restrict__ zeta, long ntok, bool normalize) {
    const long tok = (long)blockIdx.x * 32 + (threadIdx.x >> 3);
    const int part = threadIdx.x & 7;
    float D = 0.f;
    if (tok < ntok && (!POLY || normalize)) {
        float x[8], y[8];
        load8(dO + tok * 64 + part * 8, x);
        load8(o + tok * 64 + part * 8, y);
#pragma unroll
        for (int i = 0; i < 8; ++i) D = fmaf(x[i], y[i], D);
    }
    D += __shfl_xor_sync(0xffffffffu, D, 4);
    D += __shfl_xor_sync(0xffffffffu, D, 2);
    D += __shfl_xor_sync(0xffffffffu, D, 1);
    if (tok < ntok && part == 0) {
        Dv[tok] = D;
        if (POLY) {
            const float z = normalize ? Z[tok] : 1.f;
            zeta[tok] = z != 0.f ? 1.f / z : 0.f;
        }
    }
}

template <bool POLY>
static cudaError_t launch_prep(const Problem& p, const float* o, const float* Z, const void* dO, float* D, float* zeta,
                               cudaStream_t s) {
    const long ntok = p.BH() * p.T;
    const bool vec = p.dv == 64 && ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dO)) & 15) == 0;
    if (vec) {
        const unsigned blocks = (unsigned)((ntok + 31) / 32);
        if (p.dtype == 1)
            prep64_kernel<__nv_bfloat16, POLY><<<blocks, 256, 0, s>>>(o, Z, (const __nv_bfloat16*)dO, D, zeta, ntok,
                                                                     p.normalize);
        else
            prep64_kernel<float, POLY><<<blocks, 256, 0, s>>>(o, Z, (const float*)dO, D, zeta, ntok, p.normalize);
    } else {
        const unsigned blocks = (unsigned)((ntok + 7) / 8);
        if (p.dtype == 1)
            prep_kernel<__nv_bfloat16, POLY><<<blocks, 256, 0, s>>>(o, Z, (const __nv_bfloat16*)dO, D, zeta, ntok,
                                                                   p.dv, p.normalize);
        else
            prep_kernel<float, POLY><<<blocks, 256, 0, s>>>(o, Z, (const float*)dO, D, zeta, ntok, p.dv, p.normalize);
    }
    return cudaGetLastError();
}

cudaError_t launch_poly_prep(const Problem& p, const float* o, const float* Z, const void* dO, float* D,
                             float* zeta, cudaStream_t s) {
    return launch_prep<true>(p, o, Z, dO, D, zeta, s);
}

cudaError_t launch_rowdot(const Problem& p, const void* o, const void* dO, float* Dvec, cudaStream_t s) {
    return launch_prep<false>(p, (const float*)o, nullptr, dO, Dvec, nullptr, s);
}

}  // namespace tm2
