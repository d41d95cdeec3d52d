// tm2_e_simt.cu -- 2Mamba-E ("2Mamba2Furious", Sec. 6) on CUDA cores (fp32 arithmetic):
// causal softmax attention whose logits carry the softplus A-mask,
//   x_ij = scale q_i . k_j + cumA_i - cumA_j   (j <= i),   o_i = sum_j softmax_j(x_i.) v_j,
// forward with a blockwise online maximum (running max and rescaled sum), backward with
// P_ij = exp(x_ij - lse_i), dx_ij = P_ij (dO_i . v_j - D_i), D_i = dO_i . o_i.
// Blocks of 64 queries x 64 keys; thread (ti, tc) of 16 x 16 owns rows ti + 16 r and
// columns tc + 16 s of each 64 x 64 tile.
//
// Instantiated with KIND = ATTN_P2 / ATTN_P1 the same kernels evaluate the quadratic (C = T)
// form of 2Mamba and of the first-order mixer ("2Mamba2Furious", Sec. 4-5):
//   w_ij = (q_i . k_j)^p exp(cumA_i - cumA_j),  o_i = sum_j w_ij v_j [/ Z_i],  Z_i = sum_j w_ij,
// with no running maximum (the weights are not exponentiated scores), and the backward
//   dw_ij = zeta_i (dO_i . v_j - D_i),  dv_j += w_ij zeta_i dO_i,  ds_ij = p s_ij^(p-1) e_ij dw_ij,
// the A-mask axis sums taking w_ij dw_ij (zeta = 1/Z, D = dO . o normalised; 1 and 0 otherwise).
#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

constexpr int EB = 64;

template <int KIND, int D, int DV, typename Tin>
__global__ void __launch_bounds__(256) e_fwd_kernel(const Tin* __restrict__ q, const Tin* __restrict__ k,
                                                    const Tin* __restrict__ v, const float* __restrict__ cum,
                                                    const float* __restrict__ cum_lo, float scale, float* __restrict__ o,
                                                    float* __restrict__ lse, int T, int normalize) {
    constexpr int LDQ = D + 1, LDP = EB + 1, NCOL = DV / 16;
    extern __shared__ float sm[];
    float* sq = sm;               // [EB][LDQ]
    float* sk = sq + EB * LDQ;    // [EB][LDQ]
    float* sv = sk + EB * LDQ;    // [EB][DV]
    float* sP = sv + EB * DV;     // [EB][LDP]
    float* scq = sP + EB * LDP;   // [EB]
    float* sck = scq + EB;        // [EB]
    float* scql = sck + EB;       // [EB] residuals of the running sums
    float* sckl = scql + EB;      // [EB]
    const int qb = blockIdx.x;
    const long bh = blockIdx.y;
    const int tid = threadIdx.x, ti = tid >> 4, tc = tid & 15;
    for (int e = tid; e < EB * D; e += 256) {
        const int i = e / D, f = e % D;
        const long t = (long)qb * EB + i;
        sq[i * LDQ + f] = t < T ? to_f(q[(bh * T + t) * D + f]) : 0.f;
    }
    for (int i = tid; i < EB; i += 256) {
        const long t = (long)qb * EB + i;
        scq[i] = t < T ? cum[bh * T + t] : 0.f;
        scql[i] = t < T ? cum_lo[bh * T + t] : 0.f;
    }
    float acc[4][NCOL], mrow[4], lrow[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        mrow[r] = -INFINITY;
        lrow[r] = 0.f;
#pragma unroll
        for (int s = 0; s < NCOL; ++s) acc[r][s] = 0.f;
    }
    for (int kb = 0; kb <= qb; ++kb) {
        __syncthreads();
        for (int e = tid; e < EB * D; e += 256) {
            const int j = e / D, f = e % D;
            const long t = (long)kb * EB + j;
            sk[j * LDQ + f] = t < T ? to_f(k[(bh * T + t) * D + f]) : 0.f;
        }
        for (int e = tid; e < EB * DV; e += 256) {
            const int j = e / DV, f = e % DV;
            const long t = (long)kb * EB + j;
            sv[e] = t < T ? to_f(v[(bh * T + t) * DV + f]) : 0.f;
        }
        for (int j = tid; j < EB; j += 256) {
            const long t = (long)kb * EB + j;
            sck[j] = t < T ? cum[bh * T + t] : 0.f;
            sckl[j] = t < T ? cum_lo[bh * T + t] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = ti + 16 * r;
            const long ig = (long)qb * EB + i;
            if constexpr (KIND != ATTN_E) {   // w = s^p e, no maximum; lrow holds Z
                float rs = 0.f;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const int j = tc + 16 * s;
                    const long jg = (long)kb * EB + j;
                    float w = 0.f;
                    if (jg <= ig && jg < T) {
                        float dot = 0.f;
#pragma unroll 16
                        for (int n = 0; n < D; ++n) dot = fmaf(sq[i * LDQ + n], sk[j * LDQ + n], dot);
                        const float e = expf((scq[i] - sck[j]) + (scql[i] - sckl[j]));
                        w = KIND == ATTN_P2 ? dot * dot * e : dot * e;
                    }
                    sP[i * LDP + j] = w;
                    rs += w;
                }
#pragma unroll
                for (int o2 = 8; o2 > 0; o2 >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o2);
                lrow[r] += rs;
                continue;
            }
            float x[4];
            float mx = -INFINITY;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int j = tc + 16 * s;
                const long jg = (long)kb * EB + j;
                float dot = 0.f;
#pragma unroll 16
                for (int n = 0; n < D; ++n) dot = fmaf(sq[i * LDQ + n], sk[j * LDQ + n], dot);
                x[s] = (jg <= ig && jg < T) ? scale * dot + (scq[i] - sck[j]) + (scql[i] - sckl[j]) : -INFINITY;
                mx = fmaxf(mx, x[s]);
            }
#pragma unroll
            for (int o2 = 8; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
            const float mnew = fmaxf(mrow[r], mx);
            const float msafe = mnew == -INFINITY ? 0.f : mnew;
            float rs = 0.f;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const float p = __expf(x[s] - msafe);
                sP[i * LDP + tc + 16 * s] = p;
                rs += p;
            }
#pragma unroll
            for (int o2 = 8; o2 > 0; o2 >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o2);
            const float alpha = __expf(mrow[r] - msafe);
            lrow[r] = lrow[r] * alpha + rs;
#pragma unroll
            for (int s = 0; s < NCOL; ++s) acc[r][s] *= alpha;
            mrow[r] = mnew;
        }
        __syncthreads();
        for (int j = 0; j < EB; ++j) {
            float vv[NCOL];
#pragma unroll
            for (int s = 0; s < NCOL; ++s) vv[s] = sv[j * DV + tc + 16 * s];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float p = sP[(ti + 16 * r) * LDP + j];
#pragma unroll
                for (int s = 0; s < NCOL; ++s) acc[r][s] = fmaf(p, vv[s], acc[r][s]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long t = (long)qb * EB + ti + 16 * r;
        if (t >= T) continue;
        float inv;
        if constexpr (KIND == ATTN_E) inv = 1.f / lrow[r];
        else inv = normalize ? (lrow[r] != 0.f ? 1.f / lrow[r] : 0.f) : 1.f;
#pragma unroll
        for (int s = 0; s < NCOL; ++s) o[(bh * T + t) * DV + tc + 16 * s] = acc[r][s] * inv;
        if (tc == 0) lse[bh * T + t] = KIND == ATTN_E ? mrow[r] + logf(lrow[r]) : lrow[r];
    }
}

// dk, dv and column sums of dx for one block of 64 keys, looping over query blocks.
template <int KIND, int D, int DV, typename Tin>
__global__ void __launch_bounds__(256) e_bwd_dkdv_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ cum, const float* __restrict__ cum_lo, const float* __restrict__ lse,
    const float* __restrict__ Dvec, const Tin* __restrict__ dO, float scale, void* __restrict__ dk, void* __restrict__ dvo,
    float* __restrict__ colsum, int T, int NQB, bool lowp) {
    constexpr int LDQ = D + 1, LDV = DV + 1, LDP = EB + 1, NCOL = DV / 16, NN = D / 16;
    extern __shared__ float sm[];
    float* sk = sm;                 // [EB][LDQ]
    float* sv = sk + EB * LDQ;      // [EB][LDV]
    float* sq = sv + EB * LDV;      // [EB][LDQ]
    float* sdo = sq + EB * LDQ;     // [EB][LDV]
    float* sP = sdo + EB * LDV;     // [EB][LDP]
    float* sX = sP + EB * LDP;      // [EB][LDP]
    float* sC = sX + EB * LDP;      // [EB][LDP] column-sum terms
    float* sck = sC + EB * LDP;     // [EB]
    float* scq = sck + EB;          // [EB]
    float* slse = scq + EB;         // [EB] lse (E) or zeta
    float* sD = slse + EB;          // [EB]
    float* sckl = sD + EB;          // [EB] residuals of the running sums
    float* scql = sckl + EB;        // [EB]
    const int kb = blockIdx.x;
    const long bh = blockIdx.y;
    const int tid = threadIdx.x, ti = tid >> 4, tc = tid & 15;
    for (int e = tid; e < EB * D; e += 256) {
        const int j = e / D, f = e % D;
        const long t = (long)kb * EB + j;
        sk[j * LDQ + f] = t < T ? to_f(k[(bh * T + t) * D + f]) : 0.f;
    }
    for (int e = tid; e < EB * DV; e += 256) {
        const int j = e / DV, f = e % DV;
        const long t = (long)kb * EB + j;
        sv[j * LDV + f] = t < T ? to_f(v[(bh * T + t) * DV + f]) : 0.f;
    }
    for (int j = tid; j < EB; j += 256) {
        const long t = (long)kb * EB + j;
        sck[j] = t < T ? cum[bh * T + t] : 0.f;
        sckl[j] = t < T ? cum_lo[bh * T + t] : 0.f;
    }
    float adk[4][NN], adv[4][NCOL], cs[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        cs[r] = 0.f;
#pragma unroll
        for (int s = 0; s < NN; ++s) adk[r][s] = 0.f;
#pragma unroll
        for (int s = 0; s < NCOL; ++s) adv[r][s] = 0.f;
    }
    for (int qb = kb; qb < NQB; ++qb) {
        __syncthreads();
        for (int e = tid; e < EB * D; e += 256) {
            const int i = e / D, f = e % D;
            const long t = (long)qb * EB + i;
            sq[i * LDQ + f] = t < T ? to_f(q[(bh * T + t) * D + f]) : 0.f;
        }
        for (int e = tid; e < EB * DV; e += 256) {
            const int i = e / DV, f = e % DV;
            const long t = (long)qb * EB + i;
            sdo[i * LDV + f] = t < T ? to_f(dO[(bh * T + t) * DV + f]) : 0.f;
        }
        for (int i = tid; i < EB; i += 256) {
            const long t = (long)qb * EB + i;
            scq[i] = t < T ? cum[bh * T + t] : 0.f;
            scql[i] = t < T ? cum_lo[bh * T + t] : 0.f;
            slse[i] = t < T ? lse[bh * T + t] : 0.f;
            sD[i] = (t < T && Dvec) ? Dvec[bh * T + t] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int i = ti + 16 * r, j = tc + 16 * s;
                const long ig = (long)qb * EB + i, jg = (long)kb * EB + j;
                float P = 0.f, dX = 0.f, cterm = 0.f;
                if (jg <= ig && ig < T) {
                    float dot = 0.f;
#pragma unroll 16
                    for (int n = 0; n < D; ++n) dot = fmaf(sq[i * LDQ + n], sk[j * LDQ + n], dot);
                    float dP = 0.f;
#pragma unroll 16
                    for (int cc = 0; cc < DV; ++cc) dP = fmaf(sdo[i * LDV + cc], sv[j * LDV + cc], dP);
                    if constexpr (KIND == ATTN_E) {
                        P = __expf(scale * dot + (scq[i] - sck[j]) + (scql[i] - sckl[j]) - slse[i]);
                        dX = P * (dP - sD[i]);
                        cterm = dX;
                    } else {   // slse holds zeta
                        const float e = expf((scq[i] - sck[j]) + (scql[i] - sckl[j]));
                        const float dw = slse[i] * (dP - sD[i]);
                        const float w = KIND == ATTN_P2 ? dot * dot * e : dot * e;
                        P = w * slse[i];
                        dX = (KIND == ATTN_P2 ? 2.f * dot * e : e) * dw;
                        cterm = w * dw;
                    }
                }
                sP[i * LDP + j] = P;
                sX[i * LDP + j] = dX;
                sC[i * LDP + j] = cterm;
            }
        __syncthreads();
        for (int i = 0; i < EB; ++i) {
            float qn[NN], dn[NCOL];
#pragma unroll
            for (int s = 0; s < NN; ++s) qn[s] = sq[i * LDQ + tc + 16 * s];
#pragma unroll
            for (int s = 0; s < NCOL; ++s) dn[s] = sdo[i * LDV + tc + 16 * s];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int j = ti + 16 * r;
                const float p = sP[i * LDP + j], dx = sX[i * LDP + j];
                cs[r] += sC[i * LDP + j];
#pragma unroll
                for (int s = 0; s < NN; ++s) adk[r][s] = fmaf(dx, qn[s], adk[r][s]);
#pragma unroll
                for (int s = 0; s < NCOL; ++s) adv[r][s] = fmaf(p, dn[s], adv[r][s]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const long t = (long)kb * EB + ti + 16 * r;
        if (t >= T) continue;
#pragma unroll
        for (int s = 0; s < NN; ++s) store_out<Tin>(dk, (bh * T + t) * D + tc + 16 * s, scale * adk[r][s], lowp);
#pragma unroll
        for (int s = 0; s < NCOL; ++s) store_out<Tin>(dvo, (bh * T + t) * DV + tc + 16 * s, adv[r][s], lowp);
        if (tc == 0) colsum[bh * T + t] = cs[r];
    }
}

// dq and row sums of dx for one block of 64 queries, looping over key blocks.
template <int KIND, int D, int DV, typename Tin>
__global__ void __launch_bounds__(256) e_bwd_dq_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ cum, const float* __restrict__ cum_lo, const float* __restrict__ lse,
    const float* __restrict__ Dvec, const Tin* __restrict__ dO, float scale, void* __restrict__ dq, float* __restrict__ rowsum, int T,
    bool lowp) {
    constexpr int LDQ = D + 1, LDV = DV + 1, LDP = EB + 1, NN = D / 16;
    extern __shared__ float sm[];
    float* sq = sm;                 // [EB][LDQ]
    float* sdo = sq + EB * LDQ;     // [EB][LDV]
    float* sk = sdo + EB * LDV;     // [EB][LDQ]
    float* sv = sk + EB * LDQ;      // [EB][LDV]
    float* sX = sv + EB * LDV;      // [EB][LDP]
    float* scq = sX + EB * LDP;     // [EB]
    float* sck = scq + EB;          // [EB]
    float* slse = sck + EB;         // [EB]
    float* sD = slse + EB;          // [EB]
    float* scql = sD + EB;          // [EB] residuals of the running sums
    float* sckl = scql + EB;        // [EB]
    const int qb = blockIdx.x;
    const long bh = blockIdx.y;
    const int tid = threadIdx.x, ti = tid >> 4, tc = tid & 15;
    for (int e = tid; e < EB * D; e += 256) {
        const int i = e / D, f = e % D;
        const long t = (long)qb * EB + i;
        sq[i * LDQ + f] = t < T ? to_f(q[(bh * T + t) * D + f]) : 0.f;
    }
    for (int e = tid; e < EB * DV; e += 256) {
        const int i = e / DV, f = e % DV;
        const long t = (long)qb * EB + i;
        sdo[i * LDV + f] = t < T ? to_f(dO[(bh * T + t) * DV + f]) : 0.f;
    }
    for (int i = tid; i < EB; i += 256) {
        const long t = (long)qb * EB + i;
        scq[i] = t < T ? cum[bh * T + t] : 0.f;
        scql[i] = t < T ? cum_lo[bh * T + t] : 0.f;
        slse[i] = t < T ? lse[bh * T + t] : 0.f;
        sD[i] = (t < T && Dvec) ? Dvec[bh * T + t] : 0.f;
    }
    float adq[4][NN], rs[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        rs[r] = 0.f;
#pragma unroll
        for (int s = 0; s < NN; ++s) adq[r][s] = 0.f;
    }
    for (int kb = 0; kb <= qb; ++kb) {
        __syncthreads();
        for (int e = tid; e < EB * D; e += 256) {
            const int j = e / D, f = e % D;
            const long t = (long)kb * EB + j;
            sk[j * LDQ + f] = t < T ? to_f(k[(bh * T + t) * D + f]) : 0.f;
        }
        for (int e = tid; e < EB * DV; e += 256) {
            const int j = e / DV, f = e % DV;
            const long t = (long)kb * EB + j;
            sv[j * LDV + f] = t < T ? to_f(v[(bh * T + t) * DV + f]) : 0.f;
        }
        for (int j = tid; j < EB; j += 256) {
            const long t = (long)kb * EB + j;
            sck[j] = t < T ? cum[bh * T + t] : 0.f;
            sckl[j] = t < T ? cum_lo[bh * T + t] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int i = ti + 16 * r, j = tc + 16 * s;
                const long ig = (long)qb * EB + i, jg = (long)kb * EB + j;
                float dX = 0.f, rterm = 0.f;
                if (jg <= ig && ig < T) {
                    float dot = 0.f;
#pragma unroll 16
                    for (int n = 0; n < D; ++n) dot = fmaf(sq[i * LDQ + n], sk[j * LDQ + n], dot);
                    float dP = 0.f;
#pragma unroll 16
                    for (int cc = 0; cc < DV; ++cc) dP = fmaf(sdo[i * LDV + cc], sv[j * LDV + cc], dP);
                    if constexpr (KIND == ATTN_E) {
                        const float P = __expf(scale * dot + (scq[i] - sck[j]) + (scql[i] - sckl[j]) - slse[i]);
                        dX = P * (dP - sD[i]);
                        rterm = dX;
                    } else {   // slse holds zeta
                        const float e = expf((scq[i] - sck[j]) + (scql[i] - sckl[j]));
                        const float dw = slse[i] * (dP - sD[i]);
                        dX = (KIND == ATTN_P2 ? 2.f * dot * e : e) * dw;
                        rterm = (KIND == ATTN_P2 ? dot * dot * e : dot * e) * dw;
                    }
                }
                sX[i * LDP + j] = dX;
                rs[r] += rterm;
            }
        __syncthreads();
        for (int j = 0; j < EB; ++j) {
            float kn[NN];
#pragma unroll
            for (int s = 0; s < NN; ++s) kn[s] = sk[j * LDQ + tc + 16 * s];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float dx = sX[(ti + 16 * r) * LDP + j];
#pragma unroll
                for (int s = 0; s < NN; ++s) adq[r][s] = fmaf(dx, kn[s], adq[r][s]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float x = rs[r];
#pragma unroll
        for (int o2 = 8; o2 > 0; o2 >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o2);
        const long t = (long)qb * EB + ti + 16 * r;
        if (t >= T) continue;
#pragma unroll
        for (int s = 0; s < NN; ++s) store_out<Tin>(dq, (bh * T + t) * D + tc + 16 * s, scale * adq[r][s], lowp);
        if (tc == 0) rowsum[bh * T + t] = x;
    }
}

template <int KIND, int D, int DV, typename Tin>
static cudaError_t run_e_fwd(const Problem& p, const void* q, const void* k, const void* v,
                             const float* cum, const float* cum_lo, float scale, void* o, float* lse,
                             cudaStream_t s) {
    const size_t smem = sizeof(float) * (size_t)(2 * EB * (D + 1) + EB * DV + EB * (EB + 1) + 4 * EB);
    auto kern = e_fwd_kernel<KIND, D, DV, Tin>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((p.T + EB - 1) / EB, (unsigned)p.BH());
    kern<<<grid, 256, smem, s>>>((const Tin*)q, (const Tin*)k, (const Tin*)v, cum, cum_lo, scale, (float*)o, lse,
                                 p.T, p.normalize ? 1 : 0);
    return cudaGetLastError();
}

template <int KIND, int D, int DV, typename Tin>
static cudaError_t run_e_bwd(const Problem& p, const void* q, const void* k, const void* v,
                             const float* cum, const float* cum_lo, const float* lse, const float* Dvec,
                             const void* dO, float scale, void* dq, void* dk, void* dv, float* rowsum,
                             float* colsum, cudaStream_t s) {
    const int NQB = (p.T + EB - 1) / EB;
    dim3 grid(NQB, (unsigned)p.BH());
    {
        const size_t smem = sizeof(float) * (size_t)(2 * EB * (D + 1) + 2 * EB * (DV + 1) +
                                                     3 * EB * (EB + 1) + 6 * EB);
        auto kern = e_bwd_dkdv_kernel<KIND, D, DV, Tin>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, 256, smem, s>>>((const Tin*)q, (const Tin*)k, (const Tin*)v, cum, cum_lo, lse, Dvec,
                                     (const Tin*)dO, scale, dk, dv, colsum, p.T, NQB, p.lowp_grads);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        const size_t smem = sizeof(float) * (size_t)(2 * EB * (D + 1) + 2 * EB * (DV + 1) +
                                                     EB * (EB + 1) + 6 * EB);
        auto kern = e_bwd_dq_kernel<KIND, D, DV, Tin>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, 256, smem, s>>>((const Tin*)q, (const Tin*)k, (const Tin*)v, cum, cum_lo, lse, Dvec,
                                     (const Tin*)dO, scale, dq, rowsum, p.T, p.lowp_grads);
    }
    return cudaGetLastError();
}

#define TM2_E_DISPATCH(P, CALL)                                                                  \
    do {                                                                                         \
        if ((P).dtype == 1) {                                                                    \
            typedef __nv_bfloat16 Tin;                                                           \
            if ((P).d == 64) { constexpr int D = 64; return CALL; }                              \
            if ((P).d == 32) { constexpr int D = 32; return CALL; }                              \
            if ((P).d == 16) { constexpr int D = 16; return CALL; }                              \
        } else {                                                                                 \
            typedef float Tin;                                                                   \
            if ((P).d == 64) { constexpr int D = 64; return CALL; }                              \
            if ((P).d == 32) { constexpr int D = 32; return CALL; }                              \
            if ((P).d == 16) { constexpr int D = 16; return CALL; }                              \
        }                                                                                        \
        return cudaErrorInvalidValue;                                                            \
    } while (0)

cudaError_t simt_e_fwd(const Problem& p, const void* q, const void* k, const void* v,
                       const float* cum, const float* cum_lo, float scale, void* o, float* lse, cudaStream_t s) {
    TM2_E_DISPATCH(p, (run_e_fwd<ATTN_E, D, D, Tin>(p, q, k, v, cum, cum_lo, scale, o, lse, s)));
}

cudaError_t simt_e_bwd(const Problem& p, const void* q, const void* k, const void* v,
                       const float* cum, const float* cum_lo, const float* lse, const float* Dvec,
                       const void* dO, float scale, void* dq, void* dk, void* dv, float* rowsum,
                       float* colsum, cudaStream_t s) {
    TM2_E_DISPATCH(p, (run_e_bwd<ATTN_E, D, D, Tin>(p, q, k, v, cum, cum_lo, lse, Dvec, dO, scale, dq, dk, dv,
                                                    rowsum, colsum, s)));
}

template <int KIND>
static cudaError_t simt_poly_fwd_k(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                                   const float* cum_lo, void* o, float* Z, cudaStream_t s) {
    TM2_E_DISPATCH(p, (run_e_fwd<KIND, D, D, Tin>(p, q, k, v, cum, cum_lo, 1.f, o, Z, s)));
}

template <int KIND>
static cudaError_t simt_poly_bwd_k(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                                   const float* cum_lo, const float* zeta, const float* Dvec, const void* dO, void* dq,
                                   void* dk, void* dv, float* rowsum, float* colsum, cudaStream_t s) {
    TM2_E_DISPATCH(p, (run_e_bwd<KIND, D, D, Tin>(p, q, k, v, cum, cum_lo, zeta, Dvec, dO, 1.f, dq, dk, dv, rowsum,
                                                  colsum, s)));
}

cudaError_t simt_poly_fwd(const Problem& p, int order, const void* q, const void* k, const void* v,
                          const float* cum, const float* cum_lo, void* o, float* Z, cudaStream_t s) {
    if (order == 2) return simt_poly_fwd_k<ATTN_P2>(p, q, k, v, cum, cum_lo, o, Z, s);
    if (order == 1) return simt_poly_fwd_k<ATTN_P1>(p, q, k, v, cum, cum_lo, o, Z, s);
    return cudaErrorInvalidValue;
}

cudaError_t simt_poly_bwd(const Problem& p, int order, const void* q, const void* k, const void* v,
                          const float* cum, const float* cum_lo, const float* zeta, const float* D, const void* dO,
                          void* dq, void* dk, void* dv, float* rowsum, float* colsum, cudaStream_t s) {
    if (order == 2) return simt_poly_bwd_k<ATTN_P2>(p, q, k, v, cum, cum_lo, zeta, D, dO, dq, dk, dv, rowsum, colsum, s);
    if (order == 1) return simt_poly_bwd_k<ATTN_P1>(p, q, k, v, cum, cum_lo, zeta, D, dO, dq, dk, dv, rowsum, colsum, s);
    return cudaErrorInvalidValue;
}

}  // namespace tm2
