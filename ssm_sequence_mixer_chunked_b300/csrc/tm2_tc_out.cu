// tm2_tc_out.cu -- the per-chunk output kernel of the tensor-core path (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", Sec. 5: w_ij = exp(cumA_i - cumA_j) (q_i . k_j)^2, o_i = N_i / Z_i with
// N_i = sum_{j<=i} w_ij v_j and Z_i = sum_{j<=i} w_ij.  Split at the chunk boundary:
//   [N_i, Z_i] = sum_{j in c, j<=i} P_ij [v_j, 1]  +  exp(A_i) sum_{m,n} q_i[m] q_i[n] [S_{c-1}, z_{c-1}][(m,n), :]
// with P_ij = (q_i . k_j)^2 exp(A_i - A_j) and S_{c-1}, z_{c-1} the state entering the chunk
// (written by the chunk-state scan as two fp16 planes, hi and residual, and fp32 z).
//
// One CTA per (chunk, b, h); the chunk's 256 tokens form two 128-row tiles.
//  * Intra-chunk (causal 128 x 64 blocks: tile 0 x key blocks 0-1, tile 1 x key blocks 0-3):
//    s = Q K^T by tcgen05.mma from TMA tiles (bf16, K-major), the compute warps square it,
//    apply the decay mask in fp32, keep the row sums (Z) in fp32 and write P into tensor
//    memory as two bf16 terms P_hi + P_lo (one bf16 term alone costs ~2^-9 relative per
//    weight, enough to break the 2e-2 bar on unnormalised outputs); both are A operands
//    of P V (V MN-major, straight from its TMA tile).
//  * Inter-chunk readout: for each m, U_m = Q S_m with S_m[n][col] = S[(m,n), col] (the state
//    slice by TMA, MN-major, hi and residual plane: two MMAs; Q converted exactly to fp16),
//    and the compute warps accumulate N_x[col] += q_i[m] U_m[i][col] in fp32.  A 65th
//    product U = Q zm^T with zm[m][n] = z[(m,n)] gives Z_x = sum_m q_i[m] U[i][m].  No
//    operand is a rounded product; the readout of nearly orthogonal queries keeps its
//    precision.
//  * Epilogue: [N, Z] = intra + exp(A_i) [N_x, Z_x]; o = N / Z (or N), fp32; Z saved.
// Warps 0-15 compute (warp w: tile (w >> 2) & 1, tensor-memory lane quadrant w & 3, column
// half w >> 3), warp 16 issues TMA, warp 17 the MMAs.  Every mbarrier wait is bounded
// (TM2_ERR_TIMEOUT on expiry).
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {
namespace tcout {

constexpr int C = TC_CHUNK;
constexpr int NP = 5;                        // stages of two state slices (hi + residual planes, 32 KB)
constexpr int NP_EARLY = 2;                  // stages free from the start; the rest alias the
                                             // intra-chunk tiles and open once those are done
constexpr int PBYTES = 32768;
constexpr int NSL = 65;                      // 64 state slices + the normaliser product
constexpr int THREADS = 18 * 32;
constexpr int NCOMP = 512;                   // compute threads
constexpr int WARP_TMA = 16, WARP_MMA = 17;
constexpr int TILE_BYTES = C * 128;          // [256][64] 16-bit
constexpr int STG = 0;                                             // NP x [plane][slice m, m+1][64][64]
constexpr int SQ = 65536, SK = 98304, SV = 131072;                 // bf16 tiles (stages 2-4)
constexpr int SQH = 163840;                                        // fp16 copy of Q
constexpr int SZH = SQH + TILE_BYTES, SZL = SZH + 8192;            // zm hi / lo, [64][64] fp16
constexpr int SAV = SZL + 8192;                                    // A values, 256 floats
constexpr int SRED = SAV + 1024;                                   // [2 halves][256 tokens][2]
constexpr int SMEM_BYTES = SRED + 4096 + 1024;
constexpr int NBLK = 6;                      // intra-chunk blocks: (tile, 64-key block)
// tensor-memory columns
constexpr uint32_t TM_Y = 0;                 // intra N, tile t at t * 64
constexpr uint32_t TM_S = 128;               // Q K^T block, 64 columns
constexpr uint32_t TM_PH = 192, TM_PL = 224; // P hi / lo (bf16), 32 columns each
constexpr uint32_t TM_U = 256;               // U buffers: 256 + buf*128 + tile*64
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 64, false, true);
constexpr uint32_t IDESC_RD = idesc_f16_f32(128, 64, false, true);
constexpr uint32_t IDESC_RZ = idesc_f16_f32(128, 64, false, false);
TM2_DEV int blk_tile(int b) { return b < 2 ? 0 : 1; }
TM2_DEV int blk_key(int b) { return b < 2 ? b : b - 2; }
TM2_DEV uint32_t swz_elem(int row, int col) { return row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + (col & 7) * 2; }

struct Args {
    const float* Aloc;   // [BH][Tp]
    const float* zx;     // [BH][NC][4096]
    float* o;            // [BH][T][64]
    float* Z;            // [BH][T] or null
    int* status;
    int T, NC, Tp, normalize;
};

}  // namespace tcout

using namespace tcout;

__global__ void __launch_bounds__(THREADS, 1) tc_chunk_out_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                  const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const __grid_constant__ CUtensorMap tmS,
                                                                  const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_qkv, bar_full[NP], bar_empty[NP], bar_cvt, bar_sfull[NBLK], bar_sfree[NBLK],
        bar_pfull[NBLK], bar_pfree[NBLK], bar_ufull[2], bar_uempty[2], bar_yfull, bar_red, bar_intra, bar_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int gflags[3][2];      // group waits: all compute warps, tile 0, tile 1
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x;
    const long bh = blockIdx.y;
    const int NC = a.NC;
    const uint32_t sb0 = smem_u32(smem);
    float* sAv = reinterpret_cast<float*>(smem + SAV);
    float* sRed = reinterpret_cast<float*>(smem + SRED);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_qkv), 1);
        for (int i = 0; i < NP; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), 1);
        }
        mbar_init(smem_u32(&bar_cvt), NCOMP);
        for (int b = 0; b < NBLK; ++b) {   // one set per intra-chunk block, each used once
            mbar_init(smem_u32(&bar_sfull[b]), 1);
            mbar_init(smem_u32(&bar_sfree[b]), 256);
            mbar_init(smem_u32(&bar_pfull[b]), 256);
            mbar_init(smem_u32(&bar_pfree[b]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_ufull[i]), 1);
            mbar_init(smem_u32(&bar_uempty[i]), NCOMP);
        }
        mbar_init(smem_u32(&bar_yfull), 1);
        mbar_init(smem_u32(&bar_intra), 1);
        mbar_init(smem_u32(&bar_red), NCOMP);
        mbar_init(smem_u32(&bar_done), 1);
        abort_s = 0;
        fence_mbar_init();
    }
    for (int j = threadIdx.x; j < C; j += THREADS) sAv[j] = a.Aloc[bh * a.Tp + (long)c * C + j];
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == WARP_TMA) {
        if (lane == 0) {
            prefetch_tmap(&tmS);
            const uint32_t qb = smem_u32(&bar_qkv);
            mbar_arrive_expect_tx(qb, 3 * TILE_BYTES);
            tma_load_3d(sb0 + SQ, &tmQ, qb, 0, c * C, (int)bh);
            tma_load_3d(sb0 + SK, &tmK, qb, 0, c * C, (int)bh);
            tma_load_3d(sb0 + SV, &tmV, qb, 0, c * C, (int)bh);
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
                tma_load_4d(sb0 + STG + ps * PBYTES, &tmS, fb, 0, pp * 128, 0, chunk_id);
                issued = pp + 1;
            }
            mbar_wait(qb, 0, a.status);
            for (int pp = issued - 1; pp >= 0 && pp >= issued - NP; --pp)
                mbar_wait(smem_u32(&bar_full[pp % NP]), (pp / NP) & 1, a.status);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&bar_qkv), 0, a.status);
            tc_fence_after();
            // ---- intra-chunk blocks (tile t, 64-key block jb)
            for (int b = 0; b < NBLK && ok; ++b) {
                const int t = blk_tile(b), jb = blk_key(b);
                if (b > 0 && !(ok = mbar_wait(smem_u32(&bar_sfree[b - 1]), 0, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + TM_S, sdesc_sw128(sb0 + SQ + t * 16384 + kk * 32),
                              sdesc_sw128(sb0 + SK + jb * 8192 + kk * 32), IDESC_QK, kk > 0);
                umma_commit(smem_u32(&bar_sfull[b]));
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[b]), 0, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t vd = sdesc_sw128_ex(sb0 + SV + jb * 8192 + kk * 2048, 8192, 1024);
                    umma_bf16_ts(tmem + TM_Y + t * 64, tmem + TM_PH + kk * 8, vd, IDESC_PV, (jb > 0 || kk > 0) ? 1u : 0u);
                    umma_bf16_ts(tmem + TM_Y + t * 64, tmem + TM_PL + kk * 8, vd, IDESC_PV, 1u);
                }
                umma_commit(smem_u32(&bar_pfree[b]));
            }
            umma_commit(smem_u32(&bar_intra));   // arrives when every intra-chunk MMA has finished
            // ---- inter-chunk readout: U_m = Q S_m (m < 64), U_64 = Q zm^T
            if (ok) ok = mbar_wait(smem_u32(&bar_cvt), 0, a.status);
            tc_fence_after();
            for (int m = 0; m < NSL && ok; ++m) {
                const int pp = m >> 1, ps = pp % NP, ub = m & 1;
                if (abort_s) { ok = false; break; }
                if (m < 64 && (m & 1) == 0 && !(ok = mbar_wait(smem_u32(&bar_full[ps]), (pp / NP) & 1, a.status)))
                    break;
                if (m >= 2 && !(ok = mbar_wait(smem_u32(&bar_uempty[ub]), ((m >> 1) - 1) & 1, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint32_t d = tmem + TM_U + ub * 128 + t * 64;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = sdesc_sw128(sb0 + SQH + t * 16384 + kk * 32);
                        if (m < 64) {
                            const uint32_t bs = sb0 + STG + ps * PBYTES + (m & 1) * 8192 + kk * 2048;
                            umma_bf16(d, ad, sdesc_sw128_ex(bs, 8192, 1024), IDESC_RD, kk > 0);
                            umma_bf16(d, ad, sdesc_sw128_ex(bs + 16384, 8192, 1024), IDESC_RD, 1u);
                        } else {
                            umma_bf16(d, ad, sdesc_sw128(sb0 + SZH + kk * 32), IDESC_RZ, kk > 0);
                            umma_bf16(d, ad, sdesc_sw128(sb0 + SZL + kk * 32), IDESC_RZ, 1u);
                        }
                    }
                }
                if (m < 64 && (m & 1)) umma_commit(smem_u32(&bar_empty[ps]));
                umma_commit(smem_u32(&bar_ufull[ub]));
            }
            if (ok) umma_commit(smem_u32(&bar_yfull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, t = (warp >> 2) & 1, h = warp >> 3;
        const int l = quad * 32 + lane;              // row of tile t
        const int i = t * 128 + l;                   // token index inside the chunk
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float Ai = sAv[i];
        float zin = 0.f;
        int kall = 0, ktile = 0;                       // group-wait counters
        bool ok = mbar_wait(smem_u32(&bar_qkv), 0, a.status);
        if (ok) {   // fp16 copy of the Q tile; the normaliser matrix of the state as hi + lo fp16
            const int tt = threadIdx.x;
            for (int pc = tt; pc < 2048; pc += NCOMP) {
                uint32_t x[4];
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                             : "r"(sb0 + SQ + pc * 16));
                st_shared_v4(sb0 + SQH + pc * 16, bf16x2_to_f16x2(x[0]), bf16x2_to_f16x2(x[1]), bf16x2_to_f16x2(x[2]),
                             bf16x2_to_f16x2(x[3]));
            }
            const float* zc = a.zx + (bh * NC + c) * 4096;
            for (int pc = tt; pc < 512; pc += NCOMP) {
                const int m = pc >> 3, k8 = pc & 7;
                const float4 a0 = *reinterpret_cast<const float4*>(zc + m * 64 + k8 * 8);
                const float4 a1 = *reinterpret_cast<const float4*>(zc + m * 64 + k8 * 8 + 4);
                const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                uint32_t hh[4], ll[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    hh[u] = pack_f16x2(v[2 * u], v[2 * u + 1]);
                    const __half2 h2 = *reinterpret_cast<const __half2*>(&hh[u]);
                    ll[u] = pack_f16x2(v[2 * u] - __low2float(h2), v[2 * u + 1] - __high2float(h2));
                }
                const uint32_t off = m * 128 + ((k8 ^ (m & 7)) << 4);
                st_shared_v4(sb0 + SZH + off, hh[0], hh[1], hh[2], hh[3]);
                st_shared_v4(sb0 + SZL + off, ll[0], ll[1], ll[2], ll[3]);
            }
            fence_proxy_async();
            mbar_arrive(smem_u32(&bar_cvt));
        }
        // ---- intra-chunk: tile 0 owns blocks 0-1, tile 1 owns blocks 2-5; half h: 32 key columns
        for (int b = (t == 0 ? 0 : 2); b < (t == 0 ? 2 : NBLK) && ok; ++b) {
            const int jb = blk_key(b);
            if (!(ok = group_wait(smem_u32(&bar_sfull[b]), 0, a.status, warp == 4 * t, 2 + t, 256, gflags[1 + t],
                                  ktile, &abort_s)))
                break;
            if (b > 0 && !(ok = group_wait(smem_u32(&bar_pfree[b - 1]), 0, a.status, warp == 4 * t, 2 + t, 256,
                                           gflags[1 + t], ktile, &abort_s)))
                break;
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int cc = 2 * h + g2;
                float s[16];
                tmem_ld16(tmem + lane_base + TM_S + cc * 16, s);
                uint32_t ph[8], pl[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    float hi2[2], lo2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j = jb * 64 + cc * 16 + 2 * k2 + u;
                        const float sv = s[2 * k2 + u];
                        const float pv = j <= i ? sv * sv * __expf(Ai - sAv[j]) : 0.f;
                        zin += pv;
                        hi2[u] = __bfloat162float(__float2bfloat16_rn(pv));
                        lo2[u] = pv - hi2[u];
                    }
                    ph[k2] = pack_bf16x2(hi2[0], hi2[1]);
                    pl[k2] = pack_bf16x2(lo2[0], lo2[1]);
                }
                tmem_st8(tmem + lane_base + TM_PH + cc * 8, ph);
                tmem_st8(tmem + lane_base + TM_PL + cc * 8, pl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[b]));
            mbar_arrive(smem_u32(&bar_pfull[b]));
        }
        // ---- inter-chunk readout: nx[col] += q_i[m] U_m[i][col]; zx += q_i[m'] U_64[i][m']
        float nx[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) nx[k] = 0.f;
        float zxp = 0.f;
        const uint8_t* qrow = smem + SQH;            // fp16 copy (the bf16 tile is reused for stages)
#pragma unroll 1
        for (int m = 0; m < NSL && ok; ++m) {
            const int ub = m & 1;
            if (!(ok = group_wait(smem_u32(&bar_ufull[ub]), (m >> 1) & 1, a.status, warp == 0, 1, NCOMP, gflags[0], kall,
                                  &abort_s)))
                break;
            float u[32];
            const uint32_t ua = tmem + lane_base + TM_U + ub * 128 + t * 64 + h * 32;
            tmem_ld16(ua, u);
            tmem_ld16(ua + 16, u + 16);
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_uempty[ub]));
            if (m < 64) {
                const float qm = __half2float(*reinterpret_cast<const __half*>(qrow + swz_elem(i, m)));
#pragma unroll
                for (int k = 0; k < 32; ++k) nx[k] = fmaf(qm, u[k], nx[k]);
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    zxp = fmaf(__half2float(*reinterpret_cast<const __half*>(qrow + swz_elem(i, h * 32 + k))), u[k], zxp);
            }
        }
        // ---- combine the two column halves' shares of Z, then the epilogue
        if (ok) {
            sRed[(h * 256 + i) * 2] = zin;
            sRed[(h * 256 + i) * 2 + 1] = zxp;
        }
        mbar_arrive(smem_u32(&bar_red));
        if (ok) ok = mbar_wait(smem_u32(&bar_red), 0, a.status);
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_yfull), 0, a.status))) {
            tc_fence_after();
            const float eA = __expf(Ai);
            const float zi = sRed[i * 2] + sRed[(256 + i) * 2];
            const float zo = sRed[i * 2 + 1] + sRed[(256 + i) * 2 + 1];
            const float z = zi + eA * zo;
            float y[32];
            const uint32_t ya = tmem + lane_base + TM_Y + t * 64 + h * 32;
            tmem_ld16(ya, y);
            tmem_ld16(ya + 16, y + 16);
            const long tok = (long)c * C + i;
            if (tok < a.T) {
                const float inv = a.normalize ? (z != 0.f ? 1.f / z : 0.f) : 1.f;
                float4* dst = reinterpret_cast<float4*>(a.o + (bh * a.T + tok) * 64 + h * 32);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    dst[q4] = make_float4((y[4 * q4] + eA * nx[4 * q4]) * inv, (y[4 * q4 + 1] + eA * nx[4 * q4 + 1]) * inv,
                                          (y[4 * q4 + 2] + eA * nx[4 * q4 + 2]) * inv,
                                          (y[4 * q4 + 3] + eA * nx[4 * q4 + 3]) * inv);
                if (a.Z && h == 0) a.Z[bh * a.T + tok] = z;
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

cudaError_t tc_chunk_out(const Problem& p, const void* q, const void* k, const void* v, const float* Aloc,
                         const void* Sx, const float* zx, float* o, float* Z, cudaStream_t s) {
    CUtensorMap tq, tk, tv, ts;
    const uint64_t BH = (uint64_t)p.BH();
    if (!make_tmap_bf16_3d(&tq, q, BH, (uint64_t)p.T, 64, C) || !make_tmap_bf16_3d(&tk, k, BH, (uint64_t)p.T, 64, C) ||
        !make_tmap_bf16_3d(&tv, v, BH, (uint64_t)p.T, 64, C) ||
        !make_tmap_state_pairs(&ts, Sx, BH * (uint64_t)p.NC))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    Args a{Aloc, zx, o, Z, status, p.T, p.NC, (int)p.Tp(), p.normalize ? 1 : 0};
    cudaError_t e = cudaFuncSetAttribute(tc_chunk_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(p.NC, (unsigned)p.BH());
    tc_chunk_out_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(tq, tk, tv, ts, a);
    return cudaGetLastError();
}

}  // namespace tm2
