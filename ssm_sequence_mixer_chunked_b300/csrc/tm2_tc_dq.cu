// tm2_tc_dq.cu -- the query gradient of the tensor-core path (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", App. C / C.1: inside chunk c (chunk-local running sums A), with
//   s_ij = q_i . k_j,  E_ij = exp(A_i - A_j) [j <= i],  Vt_j = [v_j, 1],
//   dL/dY_i = zeta_i u_i,  u_i = [dO_i, ucol_i]  (zeta = 1/Z, ucol = -dO.o when normalised),
//   dSs_ij = 2 s_ij E_ij zeta_i (u_i . Vt_j)          (gradient w.r.t. s_ij),
// and S_{c-1}, z_{c-1} the state entering the chunk (symmetric in (m, n)):
//   dq_i[m] = sum_j dSs_ij k_j[m]
//           + 2 exp(A_i) zeta_i sum_n q_i[n] ( sum_col dO_i[col] S[(m,n), col] + ucol_i z[(m,n)] ).
//
// One CTA per (128-token tile, chunk, b, h).  The inter-chunk sum runs first, over the 10 blocks
// of the block-packed forward state (tm2_launch.h: the 16 x 16 blocks bm <= bn of the (m, n)
// index square, off-diagonal ones doubled): V_b[i][(m', n')] = sum_col dO_i[col] T_b[(m', n'),
// col] is one tcgen05.mma of N = 256 per K step and plane (the block plane K-major straight
// from its 32 KB TMA box; dO exact in fp16), and the compute warps fold it into fp32 registers
// on both sides, dqx[16 bm + m'] += q_i[16 bn + n'] V and dqx[16 bn + n'] += q_i[16 bm + m'] V,
// which over all blocks is 2 sum_n q_i[n] sum_col dO_i[col] S[(m, n), col] with 62.5% of the
// full state's products and bytes.  A tensor-core instruction costs about the same for any N up
// to 256, so a whole block per instruction is what keeps this part short.  An 11th product
// U_z = Q zm^T (zm[m][n] = z[(m, n)], the normaliser state, full layout) carries the
// normaliser column.
// The state planes hold ks^2 vs S and the normaliser state ks^2 z (the forward scan's operand
// scales, exact powers of two): the normaliser matrix is built times vs, so that both inter-chunk
// terms carry ks^2 vs, and their sum is divided by it at the end.
// The intra-chunk part follows in the same tensor memory: per 64-key block, s = Q K^T and
// u.Vt = dO V^T (bf16 MMAs), dSs as bf16 hi + lo in tensor memory, dq += dSs K.
// Warps 0-7 compute (warp w: tensor-memory lane quadrant w % 4, column half w / 4), warp 8
// issues TMA, warp 9 the MMAs.  Every mbarrier wait is bounded (TM2_ERR_TIMEOUT on expiry).
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"
#include "tm2_tc_tiles.cuh"

namespace tm2 {
namespace tcdq {
using namespace tctile;

constexpr int C = TC_CHUNK;
constexpr int THREADS = 10 * 32;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
// One TMA transaction per state block carries both planes (2 x 32 KB): a CTA streams at a fixed
// cost per transaction plus a small cost per byte, so few large transactions keep the inter
// part short.
constexpr int NR = 3;                         // ring slots of 64 KB
constexpr int RB = 65536;
constexpr int PLANE = 32768;                  // the lo plane of a block at +32 KB
static_assert(NR <= 5, "a slot is reused less than four groups later (gdone ring of four)");
constexpr int NG = TC_PACKED_BLOCKS;          // state blocks (block-packed layout), one product each
constexpr int NREQ = NG + 3;                  // both planes of each block, then Q|dO, K, V (intra part)
constexpr int EARLY = NR - 1;                 // slot NR-1 first holds the Q and dO tiles for conversion
// shared memory
constexpr int RING = 0;
constexpr int SQH = NR * RB;                  // fp16 copy of the Q tile [128][64]
constexpr int SDH = SQH + 16384;              // fp16 copy of the dO tile
// the normaliser matrix (hi, lo [64][64]) goes into the upper half of the slot of the Q|dO
// request (its tiles take the lower 32 KB; no later request uses the slot) once the slot's
// previous group, NG - NR, is done
constexpr int ZREQ = NG;
constexpr int ZFREE = NG - NR;
static_assert(ZFREE >= 0 && ZREQ + NR >= NREQ, "no later request may reuse the normaliser slot");
constexpr int SAV = SDH + 16384;              // chunk-local A, 256 floats
constexpr int BYTES = SAV + 1024 + 1024;
// tensor memory: U buffers at 0 and 256; the intra part reuses it after the inter part: dq
// accumulator, two (s, u.Vt) buffers and two (P hi, P lo) buffers, so that block b+1's scores
// are computed while block b's products run
constexpr uint32_t TM_DQ = 0, TM_SW = 64, TM_P = 320;   // SW buffer x: 64 + 128x (s, +64 u.Vt); P: 320 + 64x
constexpr uint32_t IDESC_U = idesc_f16_f32(128, 256, false, false);
constexpr uint32_t IDESC_Z = idesc_f16_f32(128, 64, false, false);
constexpr uint32_t IDESC_BF_K = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_BF_MN = idesc_bf16_f32(128, 64, false, true);

struct Args {
    const float* Aloc;   // [BH][Tp]
    const float* zeta;   // [BH][T]
    const float* ucol;   // [BH][T]
    const float* zx;     // [BH][NC][4096] forward normaliser states (slot c = entering chunk c)
    const unsigned* amax;   // [BH][4] the forward scan's operand maxima (key, value)
    void* dq;            // [BH][T][64] fp32, or bf16 with lowp
    int lowp;
    int* status;
    int T, NC, Tp;
};

TM2_DEV int slot_of(int r) { return r % NR; }
TM2_DEV uint32_t use_of(int r) { return (uint32_t)(r / NR); }

}  // namespace tcdq

using namespace tcdq;

__global__ void __launch_bounds__(THREADS, 1) tc_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                               const __grid_constant__ CUtensorMap tmD,
                                                               const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV,
                                                               const __grid_constant__ CUtensorMap tmS,
                                                               const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    // gdone[g % 4]: the products of group g are done (its ring slots are free and its U buffer
    // is full): one commit per group serves the TMA producer and the compute warps
    __shared__ __align__(8) uint64_t bar_ld, bar_full[NR], bar_gdone[4], bar_cvt, bar_sfull[4], bar_sfree[4],
        bar_pfull[4], bar_uempty[2], bar_dqfull, bar_zrdy, bar_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int gflags[2];         // group waits of the compute warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int it = blockIdx.x & 1, c = blockIdx.x >> 1;
    const long bh = blockIdx.y;
    const int NC = a.NC;
    const int nblk = 2 * (it + 1);               // 64-key blocks at or before this tile
    const uint32_t sb0 = smem_u32(smem);
    float* sAv = reinterpret_cast<float*>(smem + SAV);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_ld), 1);
        for (int i = 0; i < NR; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
        }
        mbar_init(smem_u32(&bar_cvt), 256);
        for (int b = 0; b < 4; ++b) {
            mbar_init(smem_u32(&bar_sfull[b]), 1);
            mbar_init(smem_u32(&bar_sfree[b]), 256);
            mbar_init(smem_u32(&bar_pfull[b]), 256);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_gdone[i]), 1);
            mbar_init(smem_u32(&bar_gdone[i + 2]), 1);
            mbar_init(smem_u32(&bar_uempty[i]), 256);
        }
        mbar_init(smem_u32(&bar_dqfull), 1);
        mbar_init(smem_u32(&bar_zrdy), 256);
        mbar_init(smem_u32(&bar_done), 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const uint32_t early = sb0 + RING + EARLY * RB;   // Q tile at +0, dO tile at +16384

    if (warp == WARP_TMA) {
        if (lane == 0) {
            prefetch_tmap(&tmS);
            const uint32_t lb = smem_u32(&bar_ld);
            mbar_arrive_expect_tx(lb, 2 * 16384);
            tma_load_3d(early, &tmQ, lb, 0, c * C + it * 128, (int)bh);
            tma_load_3d(early + 16384, &tmD, lb, 0, c * C + it * 128, (int)bh);
            const int chunk_id = (int)(bh * NC + c);
            int issued = 0;
            for (int r = 0; r < NREQ && !abort_s; ++r) {
                const int sl = slot_of(r);
                const uint32_t u = use_of(r);
                // the slot's previous request was group r - NR (fewer than four groups behind, so
                // gdone of that group cannot have moved on yet)
                if (u > 0 && !mbar_wait(smem_u32(&bar_gdone[(r - NR) & 3]), (uint32_t)((r - NR) >> 2) & 1, a.status)) {
                    abort_s = 1;
                    break;
                }
                if (r == EARLY && !mbar_wait(smem_u32(&bar_cvt), 0, a.status)) {   // copies made: slot free
                    abort_s = 1;
                    break;
                }
                if (!TM2_CHECK(sl >= 0 && sl < NR, a.status)) {
                    abort_s = 1;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_full[sl]), dst = sb0 + RING + sl * RB;
                if (r < NG) {
                    mbar_arrive_expect_tx(fb, 2 * PLANE);
                    tma_load_3d(dst, &tmS, fb, 0, 256 * r, 2 * chunk_id);
                    tma_load_3d(dst + PLANE, &tmS, fb, 0, 256 * r, 2 * chunk_id + 1);
                } else if (r == NG) {
                    mbar_arrive_expect_tx(fb, 2 * 16384);
                    tma_load_3d(dst, &tmQ, fb, 0, c * C + it * 128, (int)bh);
                    tma_load_3d(dst + 16384, &tmD, fb, 0, c * C + it * 128, (int)bh);
                } else {
                    mbar_arrive_expect_tx(fb, 32768);
                    tma_load_3d(dst, r == NG + 1 ? &tmK : &tmV, fb, 0, c * C, (int)bh);
                }
                issued = r + 1;
            }
            // no copy may be in flight at exit
            mbar_wait(lb, 0, a.status);
            for (int r = issued - 1; r >= 0 && r >= issued - NR; --r)
                mbar_wait(smem_u32(&bar_full[slot_of(r)]), use_of(r) & 1, a.status);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&bar_cvt), 0, a.status);
            tc_fence_after();
            // ---- inter-chunk: U_g = dO [S_{4g}..S_{4g+3}]^T (hi + lo plane), then U_z = Q zm^T
            for (int g = 0; g <= NG && ok; ++g) {
                const int ub = g & 1;
                const uint32_t k = (uint32_t)(g >> 1);
                if (abort_s) { ok = false; break; }
                if (g < NG && !(ok = mbar_wait(smem_u32(&bar_full[slot_of(g)]), use_of(g) & 1, a.status))) break;
                if (k > 0 && !(ok = mbar_wait(smem_u32(&bar_uempty[ub]), (k - 1) & 1, a.status))) break;
                tc_fence_after();
                const uint32_t d = tmem + ub * 256;
                if (g < NG) {
                    const uint32_t bhi = sb0 + RING + slot_of(g) * RB, blo = bhi + PLANE;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d, sdesc_sw128(sb0 + SDH + kk * 32), sdesc_sw128(bhi + kk * 32), IDESC_U, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d, sdesc_sw128(sb0 + SDH + kk * 32), sdesc_sw128(blo + kk * 32), IDESC_U, 1u);

                } else {
                    if (!(ok = mbar_wait(smem_u32(&bar_zrdy), 0, a.status))) break;   // normaliser tiles built
                    tc_fence_after();
                    const uint32_t zh = sb0 + RING + slot_of(ZREQ) * RB + PLANE, zl = zh + 8192;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        umma_bf16(d, sdesc_sw128(sb0 + SQH + kk * 32), sdesc_sw128(zh + kk * 32), IDESC_Z, kk > 0);
                        umma_bf16(d, sdesc_sw128(sb0 + SQH + kk * 32), sdesc_sw128(zl + kk * 32), IDESC_Z, 1u);
                    }
                }
                umma_commit(smem_u32(&bar_gdone[g & 3]));
            }
            // ---- intra-chunk: dq += (hi + lo of dSs) K over the 64-key blocks
            const int rq = NG, rk = NG + 1, rv = NG + 2;
            if (ok) ok = mbar_wait(smem_u32(&bar_uempty[0]), (uint32_t)(NG >> 1) & 1, a.status);          // U_z read
            if (ok) ok = mbar_wait(smem_u32(&bar_uempty[1]), (uint32_t)((NG - 1) >> 1) & 1, a.status);    // last U read
            if (ok) ok = mbar_wait(smem_u32(&bar_full[slot_of(rq)]), use_of(rq) & 1, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[slot_of(rk)]), use_of(rk) & 1, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[slot_of(rv)]), use_of(rv) & 1, a.status);
            tc_fence_after();
            const uint32_t SQ = sb0 + RING + slot_of(rq) * RB, SD = SQ + 16384;
            const uint32_t SK = sb0 + RING + slot_of(rk) * RB, SV = sb0 + RING + slot_of(rv) * RB;
            auto issue_sw = [&](int b) {   // s = Q K_b^T and u.Vt = dO V_b^T into buffer b & 1
                const uint32_t sw = tmem + TM_SW + (uint32_t)(b & 1) * 128;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    umma_bf16(sw, sdesc_sw128(SQ + kk * 32), sdesc_sw128(SK + b * 8192 + kk * 32), IDESC_BF_K, kk > 0);
                    umma_bf16(sw + 64, sdesc_sw128(SD + kk * 32), sdesc_sw128(SV + b * 8192 + kk * 32), IDESC_BF_K,
                              kk > 0);
                }
                umma_commit(smem_u32(&bar_sfull[b]));
            };
            if (ok && nblk > 0) issue_sw(0);
            for (int b = 0; b < nblk && ok; ++b) {
                if (abort_s) { ok = false; break; }
                if (b + 1 < nblk) {
                    if (b >= 1 && !(ok = mbar_wait(smem_u32(&bar_sfree[b - 1]), 0, a.status))) break;
                    tc_fence_after();
                    issue_sw(b + 1);
                }
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[b]), 0, a.status))) break;
                tc_fence_after();
                const uint32_t pb = tmem + TM_P + (uint32_t)(b & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t kd = sdesc_sw128_ex(SK + b * 8192 + kk * 2048, 8192, 1024);
                    umma_bf16_ts(tmem + TM_DQ, pb + kk * 8, kd, IDESC_BF_MN, (b > 0 || kk > 0) ? 1u : 0u);
                    umma_bf16_ts(tmem + TM_DQ, pb + 32 + kk * 8, kd, IDESC_BF_MN, 1u);
                }
            }
            if (ok) umma_commit(smem_u32(&bar_dqfull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;                  // tile row
        const int i = it * 128 + l;                      // chunk-local token
        const long tok = (long)c * C + i;
        const bool in = tok < a.T;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // per-chunk and per-token terms, all loaded while the tiles are on their way: the chunk-local
        // A of token threadIdx.x (C = 256 compute threads; published by the group waits' barriers),
        // this row's zeta and ucol, the operand maxima, the normaliser matrix of the state
        static_assert(C == 256, "one chunk-local A per compute thread");
        const float av = a.Aloc[bh * a.Tp + (long)c * C + threadIdx.x];
        const float ze = in ? a.zeta[bh * a.T + tok] : 0.f;
        const float uc = in ? a.ucol[bh * a.T + tok] : 0.f;
        const unsigned am_k = a.amax[bh * 4], am_v = a.amax[bh * 4 + 1];
        int kg = 0;                                      // group-wait counter
        float4 zr[4];
        z_tiles_load(a.zx + (bh * NC + c) * 4096, threadIdx.x, zr);
        bool ok = mbar_wait(smem_u32(&bar_ld), 0, a.status);
        sAv[threadIdx.x] = av;
        const float ks = pow2_scale(am_k), vs = pow2_scale(am_v);
        const float un = 1.f / (ks * ks * vs);           // exact: a power of two
        if (ok) {   // fp16 copies of the Q and dO tiles
            const int t256 = threadIdx.x;
            for (int pc = t256; pc < 1024; pc += 256) {
                tile_bf16_to_f16(early, sb0 + SQH, pc);
                tile_bf16_to_f16(early + 16384, sb0 + SDH, pc);
            }
            fence_proxy_async();
        }
        mbar_arrive(smem_u32(&bar_cvt));
        // ---- inter-chunk: dqx[m] = 2 sum_n q_i[n] (G_i + ucol_i z)[(m, n)], G_i = dO_i . S[(m, n), :],
        // for this thread's half of m (32 h .. 32 h + 31), from the block products
        // V_b[i][(m', n')] = dO_i . T_b[(m', n'), :] of the block-packed state (T_b = S on the
        // diagonal blocks, 2 S off it): block (bm, bn) adds q_i[n] V to dqx[m] (its rows) and
        // q_i[m] V to dqx[n] (its columns, the mirror (n, m)); a diagonal block holds both orders,
        // so both sums together give its 2 sum_n.  A half reads a block when either side is in its
        // range.  (S is symmetric: the backward has no initial state.)
        float dqx[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) dqx[k] = 0.f;
        const uint8_t* qrow = smem + SQH;
        auto qv = [&](int col) { return __half2float(*reinterpret_cast<const __half*>(qrow + swz_elem(l, col))); };
#pragma unroll 1
        for (int g = 0; g <= NG && ok; ++g) {
            const int ub = g & 1;
            if (!(ok = group_wait(smem_u32(&bar_gdone[g & 3]), (uint32_t)(g >> 2) & 1, a.status, warp == 0, 1, 256, gflags,
                                  kg, &abort_s)))
                break;
            if (g == ZFREE) {   // block ZFREE's products are done: its slot's upper half takes the normaliser
                const uint32_t zh = RING + slot_of(ZREQ) * RB + PLANE;
                z_tiles_store(smem + zh, smem + zh + 8192, zr, vs, threadIdx.x);
                fence_proxy_async();
                mbar_arrive(smem_u32(&bar_zrdy));
            }
            const uint32_t ub_base = tmem + lane_base + ub * 256;
            if (g < NG) {
                int bm, bn;
                tc_block_of(g, bm, bn);
                const bool side_m = (bm >> 1) == h, side_n = (bn >> 1) == h;
                if (!side_m && !side_n) {   // neither side in this half's range
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bar_uempty[ub]));
                    continue;
                }
                float qn[16], rm[16], rn[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    qn[k] = qv(16 * bn + k);
                    rm[k] = rn[k] = 0.f;
                }
#pragma unroll
                for (int mp = 0; mp < 16; ++mp) {   // columns 16 mp .. 16 mp + 15: row m' = mp, all n'
                    float v[16];
                    tmem_ld16(ub_base + 16 * mp, v);
                    if (mp == 15) {
                        tc_fence_before();
                        mbar_arrive(smem_u32(&bar_uempty[ub]));
                    }
                    const float qm = qv(16 * bm + mp);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        rm[mp] = fmaf(qn[k], v[k], rm[mp]);
                        rn[k] = fmaf(qm, v[k], rn[k]);
                    }
                }
                if (side_m) {
                    if ((bm & 1) == 0) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) dqx[k] += rm[k];
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) dqx[16 + k] += rm[k];
                    }
                }
                if (side_n) {
                    if ((bn & 1) == 0) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) dqx[k] += rn[k];
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) dqx[16 + k] += rn[k];
                    }
                }
            } else {
                float u[32];
                tmem_ld32(ub_base + h * 32, u);
                tc_fence_before();
                mbar_arrive(smem_u32(&bar_uempty[ub]));
#pragma unroll
                for (int k = 0; k < 32; ++k) dqx[k] = fmaf(2.f * uc, u[k], dqx[k]);
            }
        }
        const float Ai = sAv[i];
        // ---- intra-chunk blocks
        for (int b = 0; b < nblk && ok; ++b) {
            if (!(ok = group_wait(smem_u32(&bar_sfull[b]), 0, a.status, warp == 0, 1, 256, gflags, kg, &abort_s))) break;
            // (the P buffer's last reader, the product of block b-2, was issued before this block's
            // scores; the commit that announced them completes only after every earlier MMA of the
            // issuing thread, so the buffer is free)
            const uint32_t swb = tmem + lane_base + TM_SW + (uint32_t)(b & 1) * 128;
            const uint32_t pbb = tmem + lane_base + TM_P + (uint32_t)(b & 1) * 64;
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int cc = 2 * h + g2;
                float sv[16], wv[16];
                tmem_ld16(swb + cc * 16, sv);
                tmem_ld16(swb + 64 + cc * 16, wv);
                uint32_t ph[8], pl[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    float hi2[2], lo2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j = b * 64 + cc * 16 + 2 * k2 + u;
                        const int kx = 2 * k2 + u;
                        const float val = j <= i ? 2.f * sv[kx] * __expf(Ai - sAv[j]) * (wv[kx] + uc) : 0.f;
                        hi2[u] = __bfloat162float(__float2bfloat16_rn(val));
                        lo2[u] = val - hi2[u];
                    }
                    ph[k2] = pack_bf16x2(hi2[0], hi2[1]);
                    pl[k2] = pack_bf16x2(lo2[0], lo2[1]);
                }
                tmem_st8(pbb + cc * 8, ph);
                tmem_st8(pbb + 32 + cc * 8, pl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[b]));
            mbar_arrive(smem_u32(&bar_pfull[b]));
        }
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_dqfull), 0, a.status))) {
            tc_fence_after();
            float d0[32];
            tmem_ld32(tmem + lane_base + TM_DQ + h * 32, d0);
            if (in) {
                const float f = __expf(Ai);   // dqx already carries the factor 2
#pragma unroll
                for (int k = 0; k < 32; ++k) dqx[k] *= un;
                float g[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) g[k] = ze * (d0[k] + f * dqx[k]);
                store_row32(a.dq, (bh * a.T + tok) * 64 + h * 32, g, a.lowp != 0);
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t tc_bwd_dq(const Problem& p, const void* q, const void* k, const void* v, const void* dO, const float* Aloc,
                      const float* zeta, const float* ucol, const void* Sx, const float* zx, const unsigned* amax_f,
                      void* dq, cudaStream_t s) {
    CUtensorMap tq, td, tk, tv, ts;
    const uint64_t BH = (uint64_t)p.BH(), T = (uint64_t)p.T;
    if (!make_tmap_bf16_3d(&tq, q, BH, T, 64, 128) || !make_tmap_bf16_3d(&td, dO, BH, T, 64, 128) ||
        !make_tmap_bf16_3d(&tk, k, BH, T, 64, 256) || !make_tmap_bf16_3d(&tv, v, BH, T, 64, 256) ||
        !make_tmap_state_packed_blocks(&ts, Sx, BH * (uint64_t)p.NC))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    Args a{Aloc, zeta, ucol, zx, amax_f, dq, p.lowp_grads ? 1 : 0, status, p.T, p.NC, (int)p.Tp()};
    cudaError_t e = cudaFuncSetAttribute(tc_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(2 * p.NC, (unsigned)p.BH());
    tc_bwd_dq_kernel<<<grid, THREADS, BYTES, s>>>(tq, td, tk, tv, ts, a);
    return cudaGetLastError();
}

}  // namespace tm2
