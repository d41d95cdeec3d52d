// tm2_tc_bwd.cu -- per-chunk gradient kernels of the tensor-core path (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", App. C / C.1: the gradients of the attention kernel w.r.t. q, k, v and the
// A-mask.  Inside chunk c (chunk-local running sums A, chunk total g), with
//   s_ij = q_i . k_j,  E_ij = exp(A_i - A_j) [j <= i],  W_ij = s_ij^2 E_ij,  Vt_j = [v_j, 1],
//   dL/dY_i = zeta_i u_i,  u_i = [dO_i, ucol_i]  (zeta = 1/Z, ucol = -dO.o when normalised),
//   dSs_ij = 2 s_ij E_ij zeta_i (u_i . Vt_j)          (gradient w.r.t. s_ij),
// and the states S_{c-1} (entering the chunk) and dS_c (gradient at its end, both symmetric
// in (m, n) because the backward has no initial state):
//   dq_i   = sum_j dSs_ij k_j + 2 exp(A_i) zeta_i sum_n q_i[n] sum_col u_i[col] S_{c-1}[(m,n), col]
//   dk_j   = sum_i dSs_ij q_i + 2 w_j sum_n k_j[n] sum_col Vt_j[col] dS_c[(m,n), col]
//   dVt_j  = sum_i W_ij zeta_i u_i + w_j sum_n k_j[n] sum_m k_j[m] dS_c[(m,n), :]
//   dcumA_j = rowterm_j - Vt_j . dVt_j          (w_j = exp(g - A_j))
// (the row-axis sum minus the column-axis sum of the A-mask gradient; rowterm = dY.Y is 0
// when normalised).
//
// The inter-chunk sums run over 64 slices n of the state: for each n the tensor cores
// contract the chunk's token vectors (dO, or v and k: exact in fp16) with the state slice
// {S[(m, n), :]} (two fp16 planes, hi and residual), and the epilogue warps add the slice
// result times the per-token scalar q_i[n] / k_j[n] into fp32 registers.  No operand is a
// rounded product, which keeps the cancellation-prone contractions accurate.  A 65th slice
// carries the normaliser column (z as a 64 x 64 matrix).  The intra-chunk parts use bf16
// tiles and the hi + lo bf16 split of the fp32 epilogue values.
//
// One CTA per (128-token tile, chunk, b, h).  Warps 0-7 compute (warp w: tensor-memory lane
// quadrant w % 4, column half w / 4), warp 8 issues TMA, warp 9 the MMAs.  Every mbarrier
// wait is bounded (TM2_ERR_TIMEOUT on expiry).
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"
#include "tm2_tc_tiles.cuh"

namespace tm2 {
namespace tcbwd {
using namespace tctile;

constexpr int C = TC_CHUNK;
constexpr int THREADS = 10 * 32;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr int NP = 5;                         // stages of two state slices (hi + lo planes, 32 KB)
constexpr int NP_EARLY = 2;                   // stages free from the start; the rest alias the
                                              // intra-chunk tiles and open once those are done
constexpr int PBYTES = 32768;
constexpr int NSL = 65;                       // 64 state slices + the normaliser slice
constexpr uint32_t IDESC_BF_K = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_BF_MN = idesc_bf16_f32(128, 64, false, true);
constexpr uint32_t IDESC_H_K = idesc_f16_f32(128, 64, false, false);
constexpr uint32_t IDESC_H_MN = idesc_f16_f32(128, 64, false, true);

struct DkvArgs {
    const float* Aloc;    // [BH][Tp]
    const float* g;       // [BH][NC]
    const float* zeta;    // [BH][T]
    const float* ucol;    // [BH][T]
    const float* rowterm; // [BH][T]
    const float* dzx;     // [BH][NC][4096] gradient normaliser states (unscaled)
    const float* sscale;  // [BH][NC] scale of the gradient state planes
    float* dk;            // [BH][T][64]
    float* dv;            // [BH][T][64]
    float* dcum;          // [BH][T]
    int* status;
    int T, NC, Tp;
};

namespace kvm {
constexpr int STG = 0;                                             // NP x [plane][slice n, n+1][64][64]
constexpr int SK = 65536, SV = 81920;                              // [128][64] bf16 tiles (stage 2)
constexpr int SQ = 98304, SD = 131072;                             // [256][64] bf16 tiles (stages 3-4)
constexpr int SKH = 163840, SVH = 180224;                          // [128][64] fp16 copies
constexpr int SZH = 196608, SZL = 204800;
constexpr int SAV = 212992;                                        // A, zeta, ucol: 3 x 256 floats
constexpr int SRED = SAV + 3072;                                   // 2 x 128 partial sums
constexpr int BYTES = SRED + 1024 + 1024;
constexpr uint32_t TM_DK = 0, TM_DV = 64, TM_S = 128, TM_W = 192, TM_DH = 256, TM_DL = 288, TM_WH = 320, TM_WL = 352;
constexpr uint32_t TM_U0 = 128, TM_U1 = 384;                       // U at +0, U' at +64
}  // namespace kvm

}  // namespace tcbwd

using namespace tcbwd;

__global__ void __launch_bounds__(THREADS, 1) tc_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV,
                                                                 const __grid_constant__ CUtensorMap tmQ,
                                                                 const __grid_constant__ CUtensorMap tmD,
                                                                 const __grid_constant__ CUtensorMap tmS,
                                                                 const __grid_constant__ DkvArgs a) {
    using namespace kvm;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_ld, bar_full[NP], bar_empty[NP], bar_cvt, bar_sfull[4], bar_sfree[4],
        bar_pfull[4], bar_pfree[4], bar_ufull[2], bar_uempty[2], bar_kvfull, bar_red, bar_intra, bar_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int gflags[2];         // group waits of the compute warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tj = blockIdx.x & 1, c = blockIdx.x >> 1;
    const long bh = blockIdx.y;
    const int NC = a.NC;
    const int nblk = 4 - 2 * tj;                 // 64-query blocks at or after this key tile
    const uint32_t sb0 = smem_u32(smem);
    float* sAv = reinterpret_cast<float*>(smem + SAV);
    float* sZe = sAv + 256;
    float* sUc = sAv + 512;
    float* sRed = reinterpret_cast<float*>(smem + SRED);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_ld), 1);
        for (int i = 0; i < NP; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), 1);
        }
        mbar_init(smem_u32(&bar_cvt), 256);
        for (int b = 0; b < 4; ++b) {
            mbar_init(smem_u32(&bar_sfull[b]), 1);
            mbar_init(smem_u32(&bar_sfree[b]), 256);
            mbar_init(smem_u32(&bar_pfull[b]), 256);
            mbar_init(smem_u32(&bar_pfree[b]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_ufull[i]), 1);
            mbar_init(smem_u32(&bar_uempty[i]), 256);
        }
        mbar_init(smem_u32(&bar_kvfull), 1);
        mbar_init(smem_u32(&bar_intra), 1);
        mbar_init(smem_u32(&bar_red), 256);
        mbar_init(smem_u32(&bar_done), 1);
        abort_s = 0;
        fence_mbar_init();
    }
    for (int j = threadIdx.x; j < C; j += THREADS) {
        const long tok = (long)c * C + j;
        sAv[j] = a.Aloc[bh * a.Tp + tok];
        sZe[j] = tok < a.T ? a.zeta[bh * a.T + tok] : 0.f;
        sUc[j] = tok < a.T ? a.ucol[bh * a.T + tok] : 0.f;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == WARP_TMA) {
        if (lane == 0) {
            prefetch_tmap(&tmS);
            const uint32_t lb = smem_u32(&bar_ld);
            mbar_arrive_expect_tx(lb, 2 * 16384 + 2 * 32768);
            tma_load_3d(sb0 + SK, &tmK, lb, 0, c * C + tj * 128, (int)bh);
            tma_load_3d(sb0 + SV, &tmV, lb, 0, c * C + tj * 128, (int)bh);
            tma_load_3d(sb0 + SQ, &tmQ, lb, 0, c * C, (int)bh);
            tma_load_3d(sb0 + SD, &tmD, lb, 0, c * C, (int)bh);
            int issued = 0;
            const int chunk_id = (int)(bh * NC + c);
            for (int pp = 0; pp < 32 && !abort_s; ++pp) {   // slices 2pp, 2pp+1, both planes
                const int ps = pp % NP;
                if (pp >= NP && !mbar_wait(smem_u32(&bar_empty[ps]), ((pp / NP) - 1) & 1, a.status)) {
                    abort_s = 1;
                    break;
                }
                if (pp == NP_EARLY && (!mbar_wait(smem_u32(&bar_intra), 0, a.status) ||
                                       !mbar_wait(smem_u32(&bar_cvt), 0, a.status))) {   // tiles dead, copies made
                    abort_s = 1;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_full[ps]);
                mbar_arrive_expect_tx(fb, PBYTES);
                tma_load_5d(sb0 + STG + ps * PBYTES, &tmS, fb, 0, 0, 2 * pp, 0, chunk_id);
                issued = pp + 1;
            }
            mbar_wait(lb, 0, a.status);
            for (int pp = issued - 1; pp >= 0 && pp >= issued - NP; --pp)
                mbar_wait(smem_u32(&bar_full[pp % NP]), (pp / NP) & 1, a.status);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&bar_ld), 0, a.status);
            tc_fence_after();
            // ---- intra-chunk: dk += (dSs^T) Q, dv += (W zeta)^T dO over the 64-query blocks
            for (int b = 0; b < nblk && ok; ++b) {
                const int ib = 2 * tj + b;
                if (b > 0 && !(ok = mbar_wait(smem_u32(&bar_sfree[b - 1]), 0, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    umma_bf16(tmem + TM_S, sdesc_sw128(sb0 + SK + kk * 32), sdesc_sw128(sb0 + SQ + ib * 8192 + kk * 32),
                              IDESC_BF_K, kk > 0);
                    umma_bf16(tmem + TM_W, sdesc_sw128(sb0 + SV + kk * 32), sdesc_sw128(sb0 + SD + ib * 8192 + kk * 32),
                              IDESC_BF_K, kk > 0);
                }
                umma_commit(smem_u32(&bar_sfull[b]));
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[b]), 0, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t qd = sdesc_sw128_ex(sb0 + SQ + ib * 8192 + kk * 2048, 8192, 1024);
                    const uint64_t dd = sdesc_sw128_ex(sb0 + SD + ib * 8192 + kk * 2048, 8192, 1024);
                    const uint32_t acc0 = (b > 0 || kk > 0) ? 1u : 0u;
                    umma_bf16_ts(tmem + TM_DK, tmem + TM_DH + kk * 8, qd, IDESC_BF_MN, acc0);
                    umma_bf16_ts(tmem + TM_DK, tmem + TM_DL + kk * 8, qd, IDESC_BF_MN, 1u);
                    umma_bf16_ts(tmem + TM_DV, tmem + TM_WH + kk * 8, dd, IDESC_BF_MN, acc0);
                    umma_bf16_ts(tmem + TM_DV, tmem + TM_WL + kk * 8, dd, IDESC_BF_MN, 1u);
                }
                umma_commit(smem_u32(&bar_pfree[b]));
            }
            umma_commit(smem_u32(&bar_intra));   // arrives when every intra-chunk MMA has finished
            // ---- inter-chunk: U_n = K dS_n (N = column), U'_n = V dS_n^T (N = m); U'_64 = K dzm^T
            if (ok) ok = mbar_wait(smem_u32(&bar_cvt), 0, a.status);
            tc_fence_after();
            for (int n = 0; n < NSL && ok; ++n) {
                const int pp = n >> 1, ps = pp % NP, ub = n & 1;
                const uint32_t tu = tmem + (ub ? TM_U1 : TM_U0);
                if (abort_s) { ok = false; break; }
                if (n < 64 && (n & 1) == 0 && !(ok = mbar_wait(smem_u32(&bar_full[ps]), (pp / NP) & 1, a.status)))
                    break;
                if (n >= 2 && !(ok = mbar_wait(smem_u32(&bar_uempty[ub]), ((n >> 1) - 1) & 1, a.status))) break;
                tc_fence_after();
                if (n < 64) {
                    const uint32_t bhi = sb0 + STG + ps * PBYTES + (n & 1) * 8192, blo = bhi + 16384;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ak = sdesc_sw128(sb0 + SKH + kk * 32), av = sdesc_sw128(sb0 + SVH + kk * 32);
                        umma_bf16(tu, ak, sdesc_sw128_ex(bhi + kk * 2048, 8192, 1024), IDESC_H_MN, kk > 0);
                        umma_bf16(tu, ak, sdesc_sw128_ex(blo + kk * 2048, 8192, 1024), IDESC_H_MN, 1u);
                        umma_bf16(tu + 64, av, sdesc_sw128(bhi + kk * 32), IDESC_H_K, kk > 0);
                        umma_bf16(tu + 64, av, sdesc_sw128(blo + kk * 32), IDESC_H_K, 1u);
                    }
                    if (n & 1) umma_commit(smem_u32(&bar_empty[ps]));
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ak = sdesc_sw128(sb0 + SKH + kk * 32);
                        umma_bf16(tu + 64, ak, sdesc_sw128(sb0 + SZH + kk * 32), IDESC_H_K, kk > 0);
                        umma_bf16(tu + 64, ak, sdesc_sw128(sb0 + SZL + kk * 32), IDESC_H_K, 1u);
                    }
                }
                umma_commit(smem_u32(&bar_ufull[ub]));
            }
            if (ok) umma_commit(smem_u32(&bar_kvfull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;                  // tile row (key)
        const int j = tj * 128 + l;                      // chunk-local key index
        const long tok = (long)c * C + j;
        const bool in = tok < a.T;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float Aj = sAv[j];
        float dv64_in = 0.f;
        int kg = 0;                                      // group-wait counter
        bool ok = mbar_wait(smem_u32(&bar_ld), 0, a.status);
        if (ok) {   // fp16 copies of the key and value tiles; the normaliser gradient matrix / scale
            const int t256 = threadIdx.x;
            for (int pc = t256; pc < 1024; pc += 256) {
                tile_bf16_to_f16(sb0 + SK, sb0 + SKH, pc);
                tile_bf16_to_f16(sb0 + SV, sb0 + SVH, pc);
            }
            build_z_tiles(smem + SZH, smem + SZL, a.dzx + (bh * NC + c) * 4096, 1.f / a.sscale[bh * NC + c], t256);
            fence_proxy_async();
            mbar_arrive(smem_u32(&bar_cvt));
        }
        // ---- intra-chunk blocks (queries i >= j)
        for (int b = 0; b < nblk && ok; ++b) {
            const int ib = 2 * tj + b;
            if (!(ok = group_wait(smem_u32(&bar_sfull[b]), 0, a.status, warp == 0, 1, 256, gflags, kg, &abort_s))) break;
            if (b > 0 && !(ok = group_wait(smem_u32(&bar_pfree[b - 1]), 0, a.status, warp == 0, 1, 256, gflags, kg,
                                           &abort_s)))
                break;
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int cc = 2 * h + g2;
                float sv[16], wv[16];
                tmem_ld16(tmem + lane_base + TM_S + cc * 16, sv);
                tmem_ld16(tmem + lane_base + TM_W + cc * 16, wv);
                uint32_t dh[8], dl[8], wh[8], wl[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    float d2h[2], d2l[2], w2h[2], w2l[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int i = ib * 64 + cc * 16 + 2 * k2 + u;
                        const int kx = 2 * k2 + u;
                        float ds = 0.f, wz = 0.f;
                        if (i >= j) {
                            const float E = __expf(sAv[i] - Aj), ze = sZe[i], s = sv[kx];
                            ds = 2.f * s * E * (wv[kx] + sUc[i]) * ze;
                            wz = s * s * E * ze;
                            dv64_in = fmaf(wz, sUc[i], dv64_in);
                        }
                        d2h[u] = __bfloat162float(__float2bfloat16_rn(ds));
                        d2l[u] = ds - d2h[u];
                        w2h[u] = __bfloat162float(__float2bfloat16_rn(wz));
                        w2l[u] = wz - w2h[u];
                    }
                    dh[k2] = pack_bf16x2(d2h[0], d2h[1]);
                    dl[k2] = pack_bf16x2(d2l[0], d2l[1]);
                    wh[k2] = pack_bf16x2(w2h[0], w2h[1]);
                    wl[k2] = pack_bf16x2(w2l[0], w2l[1]);
                }
                tmem_st8(tmem + lane_base + TM_DH + cc * 8, dh);
                tmem_st8(tmem + lane_base + TM_DL + cc * 8, dl);
                tmem_st8(tmem + lane_base + TM_WH + cc * 8, wh);
                tmem_st8(tmem + lane_base + TM_WL + cc * 8, wl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[b]));
            mbar_arrive(smem_u32(&bar_pfull[b]));
        }
        // ---- inter-chunk slices
        float dkx[32], dvx[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) dkx[k] = dvx[k] = 0.f;
        float dv64x = 0.f;
        const uint8_t* krow = smem + SKH;            // fp16 copies (the bf16 tiles are reused for stages)
#pragma unroll 1
        for (int n = 0; n < NSL && ok; ++n) {
            const int ub = n & 1;
            const uint32_t tu = tmem + lane_base + (ub ? TM_U1 : TM_U0);
            if (!(ok = group_wait(smem_u32(&bar_ufull[ub]), (n >> 1) & 1, a.status, warp == 0, 1, 256, gflags, kg,
                                  &abort_s)))
                break;
            float up[32], uv[32];
            tmem_ld16(tu + 64 + h * 32, up);
            tmem_ld16(tu + 64 + h * 32 + 16, up + 16);
            if (n < 64) {
                tmem_ld16(tu + h * 32, uv);
                tmem_ld16(tu + h * 32 + 16, uv + 16);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_uempty[ub]));
            if (n < 64) {
                const float kn = __half2float(*reinterpret_cast<const __half*>(krow + swz_elem(l, n)));
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    dkx[k] = fmaf(kn, up[k], dkx[k]);
                    dvx[k] = fmaf(kn, uv[k], dvx[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    dkx[k] += up[k];
                    const float km = __half2float(*reinterpret_cast<const __half*>(krow + swz_elem(l, h * 32 + k)));
                    dv64x = fmaf(km, up[k], dv64x);
                }
            }
        }
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_kvfull), 0, a.status))) {
            tc_fence_after();
            float dk0[32], dv0[32];
            tmem_ld16(tmem + lane_base + TM_DK + h * 32, dk0);
            tmem_ld16(tmem + lane_base + TM_DK + h * 32 + 16, dk0 + 16);
            tmem_ld16(tmem + lane_base + TM_DV + h * 32, dv0);
            tmem_ld16(tmem + lane_base + TM_DV + h * 32 + 16, dv0 + 16);
            const float wj = __expf(a.g[bh * NC + c] - Aj);
            const float gsc = a.sscale[bh * NC + c];
            const float fk = 2.f * wj * gsc, fv = wj * gsc;
            float vdot = 0.f;
            const uint8_t* vrow = smem + SVH;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                dk0[k] += fk * dkx[k];
                dv0[k] += fv * dvx[k];
                const float vv = __half2float(*reinterpret_cast<const __half*>(vrow + swz_elem(l, h * 32 + k)));
                vdot = fmaf(vv, dv0[k], vdot);
            }
            const float part = vdot + dv64_in + fv * dv64x;   // this half's share of Vt_j . dVt_j
            if (h == 1) sRed[l] = part;
            mbar_arrive(smem_u32(&bar_red));
            ok = mbar_wait(smem_u32(&bar_red), 0, a.status);
            if (in) {
                float4* dkp = reinterpret_cast<float4*>(a.dk + (bh * a.T + tok) * 64 + h * 32);
                float4* dvp = reinterpret_cast<float4*>(a.dv + (bh * a.T + tok) * 64 + h * 32);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    dkp[u] = make_float4(dk0[4 * u], dk0[4 * u + 1], dk0[4 * u + 2], dk0[4 * u + 3]);
                    dvp[u] = make_float4(dv0[4 * u], dv0[4 * u + 1], dv0[4 * u + 2], dv0[4 * u + 3]);
                }
                if (h == 0 && ok) a.dcum[bh * a.T + tok] = a.rowterm[bh * a.T + tok] - (part + sRed[l]);
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t tc_bwd_dkdv(const Problem& p, const void* q, const void* k, const void* v, const void* dO,
                        const float* Aloc, const float* g, const float* zeta, const float* ucol, const float* rowterm,
                        const void* dSx, const float* dzx, const float* sscale, float* dk, float* dv, float* dcum,
                        cudaStream_t s) {
    CUtensorMap tk, tv, tq, td, ts;
    const uint64_t BH = (uint64_t)p.BH(), T = (uint64_t)p.T;
    if (!make_tmap_bf16_3d(&tk, k, BH, T, 64, 128) || !make_tmap_bf16_3d(&tv, v, BH, T, 64, 128) ||
        !make_tmap_bf16_3d(&tq, q, BH, T, 64, 256) || !make_tmap_bf16_3d(&td, dO, BH, T, 64, 256) ||
        !make_tmap_state_tpairs(&ts, dSx, BH * (uint64_t)p.NC))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    DkvArgs a{Aloc, g, zeta, ucol, rowterm, dzx, sscale, dk, dv, dcum, status, p.T, p.NC, (int)p.Tp()};
    cudaError_t e = cudaFuncSetAttribute(tc_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kvm::BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(2 * p.NC, (unsigned)p.BH());
    tc_bwd_dkdv_kernel<<<grid, THREADS, kvm::BYTES, s>>>(tk, tv, tq, td, ts, a);
    return cudaGetLastError();
}

}  // namespace tm2
