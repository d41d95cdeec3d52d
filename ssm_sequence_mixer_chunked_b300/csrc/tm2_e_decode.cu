// tm2_e_decode.cu -- 2Mamba-E decoding over a key/value cache.
//
// "2Mamba2Furious", Sec. 6: 2Mamba-E is softmax attention whose logits carry the softplus
// A-mask, and so, unlike 2Mamba, it "requires a KV cache" (Sec. 1): its recurrent state is the
// cache of every earlier key and value (Sec. 2, "Softmax as a Recurrent Neural Network": 2 N dh
// elements per head).  One decode step for token t = pos of each (sequence, head):
//   cumA_t = cumA_{t-1} - softplus(a_t)            (appended to the cache as fp32 hi + lo)
//   x_j    = scale q_t . k_j + cumA_t - cumA_j      (j <= t)
//   o_t    = sum_j softmax_j(x) v_j,   lse_t = log sum_j exp(x_j)
// with k_t, v_t appended to the cache.
//
// The step reads the whole cache once, so it is bound by HBM bandwidth.  The keys 0..t of a
// (sequence, head) are split into ranges (at least 512 keys each, as few as give about eight
// waves of blocks: per-block set-up and the combine cost less with long ranges, measured 0.49 ms
// at 512 keys against 0.445 at 2048 for 64 x 16 heads at context 8192); one block per (range,
// head): a producer warp
// streams the range's key and value rows into shared memory with bulk copies (stages of 64
// keys, four in flight, so the loads in flight do not depend on registers), and four consumer
// warps walk each stage with groups of D / 8 lanes per key (each lane 8 elements), an online
// maximum per group, and combine their groups in shared memory.  With one range the block writes o and lse itself; otherwise each block writes its
// (max, sum, weighted values) and a second kernel combines the ranges.  The block whose range
// holds t takes k_t, v_t from the inputs and writes them, and cumA_t, into the cache; every
// block computes cumA_t the same way (fp64 sum of the cached hi + lo and -softplus(a_t)).
#include <algorithm>

#include "tm2_common.cuh"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {

constexpr int E_DEC_KPS = 512;   // fewest keys per range (one block)
constexpr int E_DEC_STAGE = 64;  // keys per bulk-copy stage
constexpr int E_DEC_NST = 4;     // stages in flight

TM2_DEV void load8(const float* p, float* x) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
TM2_DEV void load8(const __nv_bfloat16* p, float* x) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <int D, int DV, typename Tin>
__global__ void __launch_bounds__(160) e_decode_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                       const Tin* __restrict__ v, const float* __restrict__ a,
                                                       Tin* __restrict__ Kc, Tin* __restrict__ Vc,
                                                       float* __restrict__ cumc, int pos, int L, int kps, float scale,
                                                       float* __restrict__ part, float* __restrict__ o,
                                                       float* __restrict__ lse, int* status) {
    static_assert(D == DV, "one group of lanes covers a key row and a value row");
    constexpr int G = D / 8;                  // lanes per key
    constexpr int NG = 128 / G;               // key groups of the four consumer warps
    constexpr int RB = D * (int)sizeof(Tin);  // bytes per cached row
    constexpr int SB = E_DEC_STAGE * RB;      // bytes of one stage's keys (and of its values)
    constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);   // [E_DEC_NST][K rows | V rows]
    __shared__ __align__(8) uint64_t bar_full[E_DEC_NST], bar_empty[E_DEC_NST];
    __shared__ float sm[NG], sl[NG];
    __shared__ float sacc[NG][DV + 1];
    const long s = blockIdx.y;
    const int sp = blockIdx.x, nsplit = gridDim.x;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int j0 = sp * kps, j1 = min(j0 + kps, pos + 1);
    const int nst = (j1 - j0 + E_DEC_STAGE - 1) / E_DEC_STAGE;
    const uint32_t sbase = smem_u32(smem);
    if (tid == 0) {
        for (int i = 0; i < E_DEC_NST; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), 4);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // the new token's running sum, the same in every block
    double cprev = 0.0;
    if (pos > 0) cprev = (double)cumc[(s * L + pos - 1) * 2] + (double)cumc[(s * L + pos - 1) * 2 + 1];
    const double cnew = cprev - (double)softplus_f(a[s]);
    const float cq_hi = (float)cnew, cq_lo = (float)(cnew - (double)cq_hi);

    if (warp == 4) {
        // ---------------------------------------------------------------- producer: the range's
        // rows in stages of E_DEC_STAGE keys through an E_DEC_NST-slot ring (the row at pos is read
        // from the inputs by the consumers, and written to the cache here once its stage is issued)
        if ((tid & 31) == 0) {
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int sl = i % E_DEC_NST;
                if (i >= E_DEC_NST && !mbar_wait(smem_u32(&bar_empty[sl]), (uint32_t)((i / E_DEC_NST) - 1) & 1, status))
                    break;
                const int js = j0 + i * E_DEC_STAGE, cnt = min(E_DEC_STAGE, j1 - js);
                const uint32_t fb = smem_u32(&bar_full[sl]), dst = sbase + sl * 2 * SB;
                mbar_arrive_expect_tx(fb, 2 * cnt * RB);
                bulk_load(dst, Kc + (s * L + js) * D, cnt * RB, fb);
                bulk_load(dst + SB, Vc + (s * L + js) * DV, cnt * RB, fb);
                issued = i + 1;
            }
            for (int i = issued - 1; i >= 0 && i >= issued - E_DEC_NST; --i)   // no copy in flight at exit
                mbar_wait(smem_u32(&bar_full[i % E_DEC_NST]), (uint32_t)(i / E_DEC_NST) & 1, status);
        }
        __syncwarp();   // the row at pos is written once every copy of the range has landed
        if (sp == nsplit - 1) {   // this block's range holds pos: append the token to the cache
            const int t = tid - 128;
            for (int e = t; e < D; e += 32) Kc[(s * L + pos) * D + e] = k[s * D + e];
            for (int e = t; e < DV; e += 32) Vc[(s * L + pos) * DV + e] = v[s * DV + e];
            if (t == 0) {
                cumc[(s * L + pos) * 2] = cq_hi;
                cumc[(s * L + pos) * 2 + 1] = cq_lo;
            }
        }
    } else {
        // ---------------------------------------------------------------- consumers
        const int grp = tid / G, gl = tid % G;
        float qv[8];
        load8(q + s * D + 8 * gl, qv);
        const float sl2 = scale * LOG2E;
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] *= sl2;
        float m = -INFINITY, lsum = 0.f, acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        constexpr int KPG = E_DEC_STAGE / NG;   // keys of a stage per group
        for (int i = 0; i < nst; ++i) {
            const int sl = i % E_DEC_NST;
            const int js = j0 + i * E_DEC_STAGE, cnt = min(E_DEC_STAGE, j1 - js);
            // this group's running sums of the stage, loaded before the wait so that their latency
            // overlaps the stage's bulk copy
            float2 cr[KPG];
#pragma unroll
            for (int u = 0; u < KPG; ++u) {
                const int r = u * NG + grp, j = js + r;
                cr[u] = (r < cnt && j != pos) ? *reinterpret_cast<const float2*>(cumc + (s * L + j) * 2)
                                              : make_float2(cq_hi, cq_lo);
            }
            if (!mbar_wait(smem_u32(&bar_full[sl]), (uint32_t)(i / E_DEC_NST) & 1, status)) break;
            const Tin* ks = reinterpret_cast<const Tin*>(smem + sl * 2 * SB);
            const Tin* vs = reinterpret_cast<const Tin*>(smem + sl * 2 * SB + SB);
            // the trip count is the same for every group, so all lanes reach the shuffles
#pragma unroll
            for (int u = 0; u < KPG; ++u) {
                const int r = u * NG + grp, j = js + r;
                const bool in = r < cnt;
                float kx[8], vx[8];
                const float c0 = cr[u].x, c1 = cr[u].y;
                if (in && j == pos) {
                    load8(k + s * D + 8 * gl, kx);
                    load8(v + s * DV + 8 * gl, vx);
                } else if (in) {
                    load8(ks + r * D + 8 * gl, kx);
                    load8(vs + r * DV + 8 * gl, vx);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kx[e] = vx[e] = 0.f;
                }
                float x = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) x = fmaf(qv[e], kx[e], x);
#pragma unroll
                for (int o2 = G / 2; o2 > 0; o2 >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o2, G);
                if (!in) continue;
                x += ((cq_hi - c0) + (cq_lo - c1)) * LOG2E;
                const float mn = fmaxf(m, x);
                const float al = exp2f(m - mn), p = exp2f(x - mn);
                lsum = lsum * al + p;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(acc[e], al, p * vx[e]);
                m = mn;
            }
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(smem_u32(&bar_empty[sl]));
        }
        if (gl == 0) {
            sm[grp] = m;
            sl[grp] = lsum;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) sacc[grp][8 * gl + i] = acc[i];
    }
    __syncthreads();
    if (tid < DV) {
        float M = -INFINITY;
        for (int g = 0; g < NG; ++g) M = fmaxf(M, sm[g]);
        float Ls = 0.f, A = 0.f;
        for (int g = 0; g < NG; ++g) {
            if (sm[g] == -INFINITY) continue;
            const float f = exp2f(sm[g] - M);
            Ls = fmaf(sl[g], f, Ls);
            A = fmaf(sacc[g][tid], f, A);
        }
        if (nsplit == 1) {
            o[s * DV + tid] = A / Ls;
            if (tid == 0 && lse) lse[s] = (M + log2f(Ls)) * LN2;
        } else {
            float* pp = part + (s * nsplit + sp) * (DV + 2);
            pp[2 + tid] = A;
            if (tid == 0) {
                pp[0] = M;
                pp[1] = Ls;
            }
        }
    }
}

// Combines the ranges of each (sequence, head): one block of DV threads per head.
template <int DV>
__global__ void e_decode_combine_kernel(const float* __restrict__ part, int nsplit, float* __restrict__ o,
                                        float* __restrict__ lse) {
    constexpr float LN2 = 0.6931471805599453f;
    const long s = blockIdx.x;
    const int c = threadIdx.x;
    const float* pp = part + s * nsplit * (DV + 2);
    float M = -INFINITY;
    for (int i = 0; i < nsplit; ++i) M = fmaxf(M, pp[i * (DV + 2)]);
    float Ls = 0.f, A = 0.f;
    for (int i = 0; i < nsplit; ++i) {
        const float f = exp2f(pp[i * (DV + 2)] - M);
        Ls = fmaf(pp[i * (DV + 2) + 1], f, Ls);
        A = fmaf(pp[i * (DV + 2) + 2 + c], f, A);
    }
    o[s * DV + c] = A / Ls;
    if (c == 0 && lse) lse[s] = (M + log2f(Ls)) * LN2;
}

// Ranges of the step at position pos: kps keys each (a multiple of the stage), ns of them; the
// last one holds pos.  About eight waves of blocks (three resident per SM), ranges of at least
// E_DEC_KPS keys.
static void e_decode_plan(long NH, int pos, int& ns, int& kps) {
    const int keys = pos + 1;
    int sms = 148, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long maxs = (keys + E_DEC_KPS - 1) / E_DEC_KPS;
    const long want = (8L * 3 * sms + NH - 1) / std::max(1L, NH);
    const int n0 = (int)std::max(1L, std::min(maxs, want));
    kps = ((keys + n0 - 1) / n0 + E_DEC_STAGE - 1) / E_DEC_STAGE * E_DEC_STAGE;
    ns = (keys + kps - 1) / kps;
}
int e_decode_splits(long NH, int pos) {
    int ns, kps;
    e_decode_plan(NH, pos, ns, kps);
    return ns;
}
int e_decode_max_splits(int L) { return (L + E_DEC_KPS - 1) / E_DEC_KPS; }

template <int D, typename Tin>
static cudaError_t e_decode_run(long NH, int pos, int L, float scale, const void* q, const void* k, const void* v,
                                const float* a, void* Kc, void* Vc, float* cumc, float* part, float* o, float* lse,
                                cudaStream_t s) {
    int ns, kps;
    e_decode_plan(NH, pos, ns, kps);
    dim3 grid((unsigned)ns, (unsigned)NH);
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    const int smem = E_DEC_NST * 2 * E_DEC_STAGE * D * (int)sizeof(Tin) + 1024;
    cudaError_t e = cudaFuncSetAttribute(e_decode_kernel<D, D, Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e_decode_kernel<D, D, Tin><<<grid, 160, smem, s>>>((const Tin*)q, (const Tin*)k, (const Tin*)v, a, (Tin*)Kc,
                                                       (Tin*)Vc, cumc, pos, L, kps, scale, part, o, lse, status);
    e = cudaGetLastError();
    if (e != cudaSuccess || ns == 1) return e;
    e_decode_combine_kernel<D><<<(unsigned)NH, D, 0, s>>>(part, ns, o, lse);
    return cudaGetLastError();
}

cudaError_t launch_e_decode(long NH, int d, int dtype, int pos, int L, float scale, const void* q, const void* k,
                            const void* v, const float* a, void* Kc, void* Vc, float* cumc, float* part, float* o,
                            float* lse, cudaStream_t s) {
#define TM2_ED(D, T) return e_decode_run<D, T>(NH, pos, L, scale, q, k, v, a, Kc, Vc, cumc, part, o, lse, s)
    if (dtype == 1) {
        if (d == 64) TM2_ED(64, __nv_bfloat16);
        if (d == 32) TM2_ED(32, __nv_bfloat16);
        if (d == 16) TM2_ED(16, __nv_bfloat16);
    } else {
        if (d == 64) TM2_ED(64, float);
        if (d == 32) TM2_ED(32, float);
        if (d == 16) TM2_ED(16, float);
    }
#undef TM2_ED
    return cudaErrorInvalidValue;
}

// Cache fill after a prefill of T tokens: K, V rows 0..T-1 copied into caches of capacity L,
// and the running sums (cum, cum_lo from launch_global_cumsum) stored as the cache's hi + lo.
template <typename Tin>
__global__ void e_cache_fill_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                                    const float* __restrict__ cum, const float* __restrict__ cum_lo,
                                    Tin* __restrict__ Kc, Tin* __restrict__ Vc, float* __restrict__ cumc, long NH,
                                    int T, int L, int d, int dv) {
    const long total = NH * (long)T;
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long)gridDim.x * blockDim.x) {
        const long h = e / T;
        const int t = (int)(e % T);
        for (int i = 0; i < d; ++i) Kc[(h * L + t) * d + i] = k[e * d + i];
        for (int i = 0; i < dv; ++i) Vc[(h * L + t) * dv + i] = v[e * dv + i];
        cumc[(h * L + t) * 2] = cum[e];
        cumc[(h * L + t) * 2 + 1] = cum_lo[e];
    }
}

cudaError_t launch_e_cache_fill(long NH, int T, int L, int d, int dv, int dtype, const void* k, const void* v,
                                const float* cum, const float* cum_lo, void* Kc, void* Vc, float* cumc,
                                cudaStream_t s) {
    const long total = NH * (long)T;
    if (total == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<long>((total + 255) / 256, 148L * 16);
    if (dtype == 1)
        e_cache_fill_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>((const __nv_bfloat16*)k, (const __nv_bfloat16*)v,
                                                                 cum, cum_lo, (__nv_bfloat16*)Kc,
                                                                 (__nv_bfloat16*)Vc, cumc, NH, T, L, d, dv);
    else
        e_cache_fill_kernel<float><<<blocks, 256, 0, s>>>((const float*)k, (const float*)v, cum, cum_lo, (float*)Kc,
                                                         (float*)Vc, cumc, NH, T, L, d, dv);
    return cudaGetLastError();
}

}  // namespace tm2
