// tm2_tc_dkdv.cu -- the key / value / A-mask gradients of the tensor-core path (bf16 inputs,
// d = dv = 64).
//
// "2Mamba2Furious", App. C / C.1: inside chunk c (chunk-local running sums A, chunk total g),
//   s_ij = q_i . k_j,  E_ij = exp(A_i - A_j) [j <= i],  W_ij = s_ij^2 E_ij,  Vt_j = [v_j, 1],
//   dL/dY_i = zeta_i u_i,  u_i = [dO_i, ucol_i]  (zeta = 1/Z, ucol = -dO.o when normalised),
//   dSs_ij = 2 s_ij E_ij zeta_i (u_i . Vt_j)          (gradient w.r.t. s_ij),
// and dS_c, dz_c the gradient w.r.t. the state at the end of the chunk (symmetric in (m, n)
// because the backward has no initial state; stored scaled by 1/Gamma_c, Gamma_c = sscale):
//   dk_j[m] = sum_i dSs_ij q_i[m] + 2 w_j Gamma_c sum_n k_j[n] ( sum_col v_j[col] dS[(m,n), col] + dz[(m,n)] )
//   dv_j    = sum_i W_ij zeta_i dO_i + w_j Gamma_c sum_n k_j[n] sum_m k_j[m] dS[(m,n), :]
//   dcumA_j = rowterm_j - Vt_j . dVt_j,      w_j = exp(g_c - A_j)
// (the row-axis sum minus the column-axis sum of the A-mask gradient; rowterm = dY.Y is 0
// when normalised; dVt_j[dv] = sum_i W_ij zeta_i ucol_i + w_j Gamma_c sum_{m,n} k_j[m] k_j[n] dz[(m,n)]).
//
// One CTA per (128-key tile, chunk, b, h).  The inter-chunk sums run first, over 16 groups of
// four state slices m = 4g .. 4g+3 (first index, in the 16-row block bm = g / 4), as one
// product per group,
//   U_g[j][(m', col)]  = sum_n k_j[n] dS[(4g+m', n), col]     (N = 256, the box MN-major),
// double-buffered in tensor memory.  The fp16 hi and residual planes of the block-packed
// gradient state come as one TMA box per plane over the run of stored blocks (bm, bm .. 3)
// (their rows (m, n), n >= 16 bm) plus one 8 KB box for each stored block (bn, bm), bn < bm,
// seen the other way round (its rows (n, m): dS is symmetric and stored as it is); all land
// as [m'][n'][col], 1 + bm boxes per plane instead of one per 16-column block.  The compute
// warps fold U_g into dvx[col] += k_j[4g+m'] U_g[j][(m', col)] (registers) and
// sum_col v_j[col] U_g[j][(m', col)] into the dk sum of key index 4g+m' (shared memory, each
// column half adding its share).  One product instead of a second, V-side chain halves the
// tensor work of this part.  A 17th product U'_z = K dzm^T (dzm[m][n] = dz[(m,n)]) adds
// the normaliser column; its tiles are built in the ring slot of the last group's residual
// plane once that group's product is done.
// The gradient state planes and normaliser states carry the reverse scan's operand scales
// ks^2 vs (exact powers of two) on top of 1/Gamma_c; the inter-chunk terms are divided by
// them together with the multiplication by Gamma_c.
// The intra-chunk part follows in the same tensor memory: per 64-query block, s^T = K Q^T and
// (u.Vt)^T = V dO^T (bf16), dSs^T and (W zeta)^T as bf16 hi + lo in tensor memory, then
// dk += dSs^T Q and dv += (W zeta)^T dO.
// Warps 0-7 compute (warp w: tensor-memory lane quadrant w % 4, column half w / 4), warp 8
// issues TMA, warp 9 the inter-chunk products and the intra-chunk scores, warps 10 and 11 the
// intra-chunk dk and dv products (one thread's tcgen05.mma instructions do not overlap, and an
// N = 64 one holds its issuer for several times its tensor-core time, so three issuers let a
// block's scores and both of its products run together).  Every mbarrier wait is bounded
// (TM2_ERR_TIMEOUT on expiry).
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"
#include "tm2_tc_tiles.cuh"

namespace tm2 {
namespace tckv {
using namespace tctile;

constexpr int C = TC_CHUNK;
constexpr int THREADS = 12 * 32;
constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_PK = 10;   // warps 10 (dk) and 11 (dv): products
static_assert(THREADS == (WARP_PK + 2) * 32, "two product warps last");
constexpr int NR = 5;                         // ring slots of 32 KB
constexpr int RB = 32768;
static_assert(NR <= 7, "a slot is reused less than four groups later (gdone ring of four)");
constexpr int NG = 16;                        // groups of four state slices
constexpr int NREQ = 2 * NG + 3;              // hi/lo plane of each group, then K|V, Q, dO (intra part)
constexpr int EARLY = NR - 1;                 // slot NR-1 first holds the K and V tiles for conversion
// shared memory
constexpr int RING = 0;
constexpr int SKH = NR * RB;                         // fp16 copy of the K tile [128][64] (A operand of U)
constexpr int SDK = SKH + 16384;                     // inter-chunk sums of dk [64 m][128 rows] fp32
constexpr int SAV = SDK + 32768;                     // A, zeta, ucol: 3 x 256 floats
// the normaliser gradient matrix (hi, lo [64][64] fp16) goes into the ring slot of group NG-1's
// lo plane, which no later request uses, once that group's products are done
constexpr int ZREQ = 2 * NG - 1;
static_assert(ZREQ + NR >= NREQ, "no later request may reuse the normaliser slot");
constexpr int SRED = SAV + 3072;                     // 128 partial sums
constexpr int BYTES = SRED + 1024 + 1024;
// tensor memory: U of group g in buffer (g & 1) at 256 (g & 1); the intra part reuses it afterwards
constexpr uint32_t TM_DK = 0, TM_DV = 64, TM_S = 128, TM_W = 192, TM_DH = 256, TM_DL = 288, TM_WH = 320, TM_WL = 352;
constexpr uint32_t TM_PARK = 384;             // inter-chunk sums parked during the intra part: 384 + 64h
constexpr uint32_t IDESC_U = idesc_f16_f32(128, 256, false, true);
constexpr uint32_t IDESC_Z = idesc_f16_f32(128, 64, false, false);
constexpr uint32_t IDESC_BF_K = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_BF_MN = idesc_bf16_f32(128, 64, false, true);

struct Args {
    const float* Aloc;    // [BH][Tp]
    const float* g;       // [BH][NC]
    const float* zeta;    // [BH][T]
    const float* ucol;    // [BH][T]
    const float* rowterm; // [BH][T]
    const float* dzx;     // [BH][NC][4096] gradient normaliser states (unscaled)
    const float* sscale;  // [BH][NC] scale of the gradient state planes
    const unsigned* amax; // [BH][4] the reverse scan's operand maxima (key, value, normaliser)
    void* dk;             // [BH][T][64] fp32, or bf16 with lowp
    void* dv;             // [BH][T][64] fp32, or bf16 with lowp
    float* dcum;          // [BH][T]
    int lowp;
    int* status;
    int T, NC, Tp;
};

// runs of 1 .. 4 consecutive packed blocks (make_tmap_state_packed_rowrun), run[nb - 1]
struct RunMaps {
    CUtensorMap run[4];
};

TM2_DEV int slot_of(int r) { return r % NR; }
TM2_DEV uint32_t use_of(int r) { return (uint32_t)(r / NR); }

}  // namespace tckv

using namespace tckv;

__global__ void __launch_bounds__(THREADS, 1) tc_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV,
                                                                 const __grid_constant__ CUtensorMap tmQ,
                                                                 const __grid_constant__ CUtensorMap tmD,
                                                                 const __grid_constant__ RunMaps rm,
                                                                 const __grid_constant__ CUtensorMap tmSt,
                                                                 const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    // gdone[g % 4]: the products of group g are done (its ring slots are free and its U buffer
    // is full): one commit per group serves the TMA producer and the compute warps
    __shared__ __align__(8) uint64_t bar_ld, bar_full[NR], bar_gdone[4], bar_cvt, bar_sfull[4], bar_pdone[4],
        bar_pfull[4], bar_uempty[2], bar_kvfull, bar_red, bar_zrdy, bar_done, bar_pend[2];
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
        for (int i = 0; i < NR; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
        }
        mbar_init(smem_u32(&bar_cvt), 256);
        for (int b = 0; b < 4; ++b) {
            mbar_init(smem_u32(&bar_sfull[b]), 1);
            mbar_init(smem_u32(&bar_pdone[b]), 2);   // dk and dv products
            mbar_init(smem_u32(&bar_pfull[b]), 256);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_gdone[i]), 1);
            mbar_init(smem_u32(&bar_gdone[i + 2]), 1);
            mbar_init(smem_u32(&bar_uempty[i]), 256);
        }
        mbar_init(smem_u32(&bar_kvfull), 2);
        mbar_init(smem_u32(&bar_red), 256);
        mbar_init(smem_u32(&bar_zrdy), 256);
        mbar_init(smem_u32(&bar_done), 1);
        mbar_init(smem_u32(&bar_pend[0]), 1);
        mbar_init(smem_u32(&bar_pend[1]), 1);
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
    const uint32_t early = sb0 + RING + EARLY * RB;   // K tile at +0, V tile at +16384

    if (warp == WARP_TMA) {
        if (lane == 0) {
            for (int i = 0; i < 4; ++i) prefetch_tmap(&rm.run[i]);
            const uint32_t lb = smem_u32(&bar_ld);
            mbar_arrive_expect_tx(lb, 2 * 16384);
            tma_load_3d(early, &tmK, lb, 0, c * C + tj * 128, (int)bh);
            tma_load_3d(early + 16384, &tmV, lb, 0, c * C + tj * 128, (int)bh);
            const int chunk_id = (int)(bh * NC + c);
            int issued = 0;
            for (int r = 0; r < NREQ && !abort_s; ++r) {
                const int sl = slot_of(r);
                const uint32_t u = use_of(r);
                // the slot's previous request belonged to group (r - NR) / 2 (fewer than four groups
                // behind, so gdone of that group cannot have moved on yet)
                if (u > 0 && !mbar_wait(smem_u32(&bar_gdone[((r - NR) >> 1) & 3]), (uint32_t)((r - NR) >> 3) & 1,
                                        a.status)) {
                    abort_s = 1;
                    break;
                }
                if (r == EARLY && !mbar_wait(smem_u32(&bar_cvt), 0, a.status)) {   // copies made: slot free
                    abort_s = 1;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_full[sl]), dst = sb0 + RING + sl * RB;
                mbar_arrive_expect_tx(fb, RB);
                if (r < 2 * NG) {
                    // the rows (m, n) of key indices m = 4 mq .. 4 mq + 3 (block row bm) for every n,
                    // landing as [m'][n'][col] with the 16-column block bn of n at 8 KB bn: the
                    // stored blocks (bm, bm .. 3) as one run (rows (m, n)), then each stored block
                    // (bn, bm), bn < bm, seen the other way round (rows (n, m))
                    const int g = r >> 1, bm = g >> 2, mq = g & 3, pc = 2 * chunk_id + (r & 1);
                    if (TM2_CHECK(tc_block_index(bm, 3) < TC_PACKED_BLOCKS && mq < 4, a.status)) {
                        tma_load_5d(dst + bm * 8192, &rm.run[3 - bm], fb, 0, 0, 4 * mq, tc_block_index(bm, bm), pc);
                        for (int bn = 0; bn < bm; ++bn)
                            tma_load_4d(dst + bn * 8192, &tmSt, fb, 0, 0, 4 * mq,
                                        TC_PACKED_BLOCKS * pc + tc_block_index(bn, bm));
                    }   // (else the request never completes: the consumer's bounded wait ends it)
                } else if (r == 2 * NG) {
                    tma_load_3d(dst, &tmK, fb, 0, c * C + tj * 128, (int)bh);
                    tma_load_3d(dst + 16384, &tmV, fb, 0, c * C + tj * 128, (int)bh);
                } else {
                    tma_load_3d(dst, r == 2 * NG + 1 ? &tmQ : &tmD, fb, 0, c * C, (int)bh);
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
            // ---- inter-chunk: U_g = K B_g (MN-major view of the group's box, hi + lo plane) into
            // buffer g & 1, then U'_z = K dzm^T
            for (int g = 0; g <= NG && ok; ++g) {
                const int ub = g & 1;
                const uint32_t k = (uint32_t)(g >> 1);
                if (abort_s) { ok = false; break; }
                if (g < NG) {
                    const int r0 = 2 * g, r1 = 2 * g + 1;
                    if (!(ok = mbar_wait(smem_u32(&bar_full[slot_of(r0)]), use_of(r0) & 1, a.status))) break;
                    if (!(ok = mbar_wait(smem_u32(&bar_full[slot_of(r1)]), use_of(r1) & 1, a.status))) break;
                }
                if (k > 0 && !(ok = mbar_wait(smem_u32(&bar_uempty[ub]), (k - 1) & 1, a.status))) break;
                tc_fence_after();
                const uint32_t d = tmem + ub * 256;
                if (g < NG) {
                    const uint32_t bhi = sb0 + RING + slot_of(2 * g) * RB, blo = sb0 + RING + slot_of(2 * g + 1) * RB;
                    // K block kk = n in 16 kk .. 16 kk + 15 at 8 KB kk ([m'][n'][col], m' slices 2 KB apart)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d, sdesc_sw128(sb0 + SKH + kk * 32), sdesc_sw128_ex(bhi + kk * 8192, 2048, 1024), IDESC_U,
                                  kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d, sdesc_sw128(sb0 + SKH + kk * 32), sdesc_sw128_ex(blo + kk * 8192, 2048, 1024), IDESC_U,
                                  1u);

                } else {
                    if (!(ok = mbar_wait(smem_u32(&bar_zrdy), 0, a.status))) break;   // normaliser tiles built
                    tc_fence_after();
                    const uint32_t zh = sb0 + RING + slot_of(ZREQ) * RB, zl = zh + 8192;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        umma_bf16(d, sdesc_sw128(sb0 + SKH + kk * 32), sdesc_sw128(zh + kk * 32), IDESC_Z, kk > 0);
                        umma_bf16(d, sdesc_sw128(sb0 + SKH + kk * 32), sdesc_sw128(zl + kk * 32), IDESC_Z, 1u);
                    }
                }
                umma_commit(smem_u32(&bar_gdone[g & 3]));
            }
            // ---- intra-chunk: dk += (dSs^T) Q, dv += (W zeta)^T dO over the 64-query blocks
            const int rkv = 2 * NG, rq = 2 * NG + 1, rd = 2 * NG + 2;
            if (ok) ok = mbar_wait(smem_u32(&bar_uempty[0]), (uint32_t)(NG >> 1) & 1, a.status);          // U'_z read
            if (ok) ok = mbar_wait(smem_u32(&bar_uempty[1]), (uint32_t)((NG - 1) >> 1) & 1, a.status);    // last U read
            if (ok) ok = mbar_wait(smem_u32(&bar_full[slot_of(rkv)]), use_of(rkv) & 1, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[slot_of(rq)]), use_of(rq) & 1, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[slot_of(rd)]), use_of(rd) & 1, a.status);
            tc_fence_after();
            const uint32_t SK = sb0 + RING + slot_of(rkv) * RB, SV = SK + 16384;
            const uint32_t SQ = sb0 + RING + slot_of(rq) * RB, SD = sb0 + RING + slot_of(rd) * RB;
            // block b + 1's scores go into S / W as soon as the compute warps have read block b's
            // (pfull[b]), while the product warps run block b's products, so that the weight step
            // of b + 1 overlaps them; pdone[b] tells the compute warps that the products of block
            // b have read the P buffers they are about to overwrite
            auto issue_sw = [&](int b) {
                const int ib = 2 * tj + b;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    umma_bf16(tmem + TM_S, sdesc_sw128(SK + kk * 32), sdesc_sw128(SQ + ib * 8192 + kk * 32), IDESC_BF_K,
                              kk > 0);
                    umma_bf16(tmem + TM_W, sdesc_sw128(SV + kk * 32), sdesc_sw128(SD + ib * 8192 + kk * 32), IDESC_BF_K,
                              kk > 0);
                }
                umma_commit(smem_u32(&bar_sfull[b]));
            };
            if (ok && nblk > 0) issue_sw(0);
            for (int b = 0; b + 1 < nblk && ok; ++b) {
                if (abort_s) { ok = false; break; }
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[b]), 0, a.status))) break;
                tc_fence_after();
                issue_sw(b + 1);
            }
            if (!ok) abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else if (warp >= WARP_PK) {
        // ---- intra-chunk products: dk += dSs^T Q (warp 10) or dv += (W zeta)^T dO (warp 11), the
        // A operand as bf16 hi + lo in tensor memory.  The accumulators share columns with the
        // inter-chunk U buffers: pfull[0] comes after the compute warps have read the last U.
        const int part = warp - WARP_PK;
        if (lane == 0) {
            const int rx = part == 0 ? 2 * NG + 1 : 2 * NG + 2;   // Q or dO (last requests: no reuse)
            bool ok = mbar_wait(smem_u32(&bar_full[slot_of(rx)]), use_of(rx) & 1, a.status);
            const uint32_t SX = sb0 + RING + slot_of(rx) * RB;
            const uint32_t acc = tmem + (part == 0 ? TM_DK : TM_DV);
            const uint32_t ph = tmem + (part == 0 ? TM_DH : TM_WH), pl = tmem + (part == 0 ? TM_DL : TM_WL);
            for (int b = 0; b < nblk && ok; ++b) {
                const int ib = 2 * tj + b;
                if (abort_s) { ok = false; break; }
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[b]), 0, a.status))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t xd = sdesc_sw128_ex(SX + ib * 8192 + kk * 2048, 8192, 1024);
                    umma_bf16_ts(acc, ph + kk * 8, xd, IDESC_BF_MN, (b > 0 || kk > 0) ? 1u : 0u);
                    umma_bf16_ts(acc, pl + kk * 8, xd, IDESC_BF_MN, 1u);
                }
                umma_commit(smem_u32(&bar_pdone[b]));
            }
            if (ok) umma_commit(smem_u32(&bar_kvfull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_pend[part]));   // none of this thread's MMAs in flight at exit
            mbar_wait(smem_u32(&bar_pend[part]), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;                  // tile row (key)
        const int j = tj * 128 + l;                      // chunk-local key index
        const long tok = (long)c * C + j;
        const bool in = tok < a.T;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        float dv64_in = 0.f;
        int kg = 0;                                      // group-wait counter
        // global reads issued before the first wait, so their latency hides under the tile loads
        const float gsc = a.sscale[bh * NC + c];
        const float gcv = a.g[bh * NC + c];
        const float rowt = in ? a.rowterm[bh * a.T + tok] : 0.f;
        const unsigned am_k = a.amax[bh * 4], am_v = a.amax[bh * 4 + 1];
        // the chunk's per-token terms, one token per compute thread (C = 256), stored once the
        // key tile has arrived and published by the group waits' barriers
        static_assert(C == 256, "one chunk token per compute thread");
        const long tok_s = (long)c * C + threadIdx.x;
        const float av_s = a.Aloc[bh * a.Tp + tok_s];
        const float ze_s = tok_s < a.T ? a.zeta[bh * a.T + tok_s] : 0.f;
        const float uc_s = tok_s < a.T ? a.ucol[bh * a.T + tok_s] : 0.f;
        float* sDK = reinterpret_cast<float*>(smem + SDK);   // [m][row]: sum_col v_j[col] U[(m, col)]
#pragma unroll
        for (int m = 0; m < 32; ++m) sDK[(32 * h + m) * 128 + l] = 0.f;
        float vj[32];   // this row's value columns 32h .. 32h + 31 (fp32)
        bool ok = mbar_wait(smem_u32(&bar_ld), 0, a.status);
        sAv[threadIdx.x] = av_s;
        sZe[threadIdx.x] = ze_s;
        sUc[threadIdx.x] = uc_s;
        if (ok) {   // fp16 copy of the key tile (the A operand of U); this row's values
            const int t256 = threadIdx.x;
            for (int pc = t256; pc < 1024; pc += 256) tile_bf16_to_f16(early, sb0 + SKH, pc);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                uint32_t x[4];
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                             : "r"(early + 16384 + swz_elem(l, 32 * h + 8 * c8)));
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    vj[8 * c8 + 2 * u] = __uint_as_float(x[u] << 16);
                    vj[8 * c8 + 2 * u + 1] = __uint_as_float(x[u] & 0xffff0000u);
                }
            }
            fence_proxy_async();
        }
        mbar_arrive(smem_u32(&bar_cvt));
        // ---- inter-chunk groups: dvx[col] += k_j[n] U[(n, col)]; sDK[n] += sum_col v_j[col] U[(n, col)]
        // (each column half adds its share; U[(m, col)] = sum_n k_j[n] dS[(m, n), col], so the
        // second sum is the dk term of key index m)
        float dvx[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) dvx[k] = 0.f;
        float dv64x = 0.f;
        float4 zr[4];
        const uint8_t* krow = smem + SKH;
#pragma unroll 1
        for (int g = 0; g <= NG && ok; ++g) {
            const int ub = g & 1;
            if (g == NG - 3) z_tiles_load(a.dzx + (bh * NC + c) * 4096, threadIdx.x, zr);   // in flight meanwhile
            if (!(ok = group_wait(smem_u32(&bar_gdone[g & 3]), (uint32_t)(g >> 2) & 1, a.status, warp == 0, 1, 256, gflags,
                                  kg, &abort_s)))
                break;
            if (g == NG - 1) {   // group NG-1's products are done: its lo slot takes the normaliser matrix
                const uint32_t zh = RING + slot_of(ZREQ) * RB;
                z_tiles_store(smem + zh, smem + zh + 8192, zr, 1.f / gsc, threadIdx.x);
                fence_proxy_async();
                mbar_arrive(smem_u32(&bar_zrdy));
            }
            const uint32_t ua = tmem + lane_base + ub * 256 + h * 32;
            if (g < NG) {
#pragma unroll 1
                for (int np = 0; np < 4; np += 2) {   // two slices per load pair (one wait for both)
                    float u0[32], u1[32];
                    tmem_ld32x2(ua + np * 64, ua + (np + 1) * 64, u0, u1);
                    if (np == 2) {
                        tc_fence_before();
                        mbar_arrive(smem_u32(&bar_uempty[ub]));
                    }
                    const float k0 = __half2float(*reinterpret_cast<const __half*>(krow + swz_elem(l, 4 * g + np)));
                    const float k1 = __half2float(*reinterpret_cast<const __half*>(krow + swz_elem(l, 4 * g + np + 1)));
                    float p0 = 0.f, p1 = 0.f;
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        dvx[k] = fmaf(k1, u1[k], fmaf(k0, u0[k], dvx[k]));
                        p0 = fmaf(vj[k], u0[k], p0);
                        p1 = fmaf(vj[k], u1[k], p1);
                    }
                    atomicAdd(&sDK[(4 * g + np) * 128 + l], p0);
                    atomicAdd(&sDK[(4 * g + np + 1) * 128 + l], p1);
                }
            } else {
                float u[32];
                tmem_ld32(ua, u);
                tc_fence_before();
                mbar_arrive(smem_u32(&bar_uempty[ub]));
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    atomicAdd(&sDK[(32 * h + k) * 128 + l], u[k]);
                    const float km = __half2float(*reinterpret_cast<const __half*>(krow + swz_elem(l, h * 32 + k)));
                    dv64x = fmaf(km, u[k], dv64x);
                }
            }
        }
        // park the inter-chunk value sums in tensor memory (outside the intra part's columns),
        // once every compute warp has read the last U (whose columns these are)
        named_bar_sync(1, 256);
        tmem_st32(tmem + lane_base + TM_PARK + h * 64 + 32, dvx);
        tmem_wait_st();
        const float Aj = sAv[j];
        // ---- intra-chunk blocks (queries i >= j)
        for (int b = 0; b < nblk && ok; ++b) {
            const int ib = 2 * tj + b;
            if (!(ok = group_wait(smem_u32(&bar_sfull[b]), 0, a.status, warp == 0, 1, 256, gflags, kg, &abort_s))) break;
            // both rounds' weights in registers while the products of block b - 1 may still read
            // the P buffers; stored once those products are done
            uint32_t dh[2][8], dl[2][8], wh[2][8], wl[2][8];
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int cc = 2 * h + g2;
                float sv[16], wv[16];
                tmem_ld16(tmem + lane_base + TM_S + cc * 16, sv);
                tmem_ld16(tmem + lane_base + TM_W + cc * 16, wv);
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
                    dh[g2][k2] = pack_bf16x2(d2h[0], d2h[1]);
                    dl[g2][k2] = pack_bf16x2(d2l[0], d2l[1]);
                    wh[g2][k2] = pack_bf16x2(w2h[0], w2h[1]);
                    wl[g2][k2] = pack_bf16x2(w2l[0], w2l[1]);
                }
            }
            if (b > 0 && !(ok = group_wait(smem_u32(&bar_pdone[b - 1]), 0, a.status, warp == 0, 1, 256, gflags, kg,
                                           &abort_s)))
                break;
            tc_fence_after();
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int cc = 2 * h + g2;
                tmem_st8(tmem + lane_base + TM_DH + cc * 8, dh[g2]);
                tmem_st8(tmem + lane_base + TM_DL + cc * 8, dl[g2]);
                tmem_st8(tmem + lane_base + TM_WH + cc * 8, wh[g2]);
                tmem_st8(tmem + lane_base + TM_WL + cc * 8, wl[g2]);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_pfull[b]));
        }
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_kvfull), 0, a.status))) {
            tc_fence_after();
            float dk0[32], dv0[32];
            tmem_ld32(tmem + lane_base + TM_DK + h * 32, dk0);
            tmem_ld32(tmem + lane_base + TM_DV + h * 32, dv0);
            tmem_ld32(tmem + lane_base + TM_PARK + h * 64 + 32, dvx);
            const float wj = __expf(gcv - Aj);
            const float ks = pow2_scale(am_k), vs = pow2_scale(am_v);
            const float gu = gsc / (ks * ks * vs);   // Gamma_c out of the planes' units (exact)
            const float fk = 2.f * wj * gu, fv = wj * gu;
            float vdot = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                dk0[k] += fk * sDK[(32 * h + k) * 128 + l];
                dv0[k] += fv * dvx[k];
                vdot = fmaf(vj[k], dv0[k], vdot);
            }
            const float part = vdot + dv64_in + fv * dv64x;   // this half's share of Vt_j . dVt_j
            if (h == 1) sRed[l] = part;
            mbar_arrive(smem_u32(&bar_red));
            ok = mbar_wait(smem_u32(&bar_red), 0, a.status);
            if (in) {
                store_row32(a.dk, (bh * a.T + tok) * 64 + h * 32, dk0, a.lowp != 0);
                store_row32(a.dv, (bh * a.T + tok) * 64 + h * 32, dv0, a.lowp != 0);
                if (h == 0 && ok) a.dcum[bh * a.T + tok] = rowt - (part + sRed[l]);
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
                        const void* dSx, const float* dzx, const float* sscale, const unsigned* amax_r, void* dk,
                        void* dv, float* dcum, cudaStream_t s) {
    CUtensorMap tk, tv, tq, td, tst;
    RunMaps rm;
    const uint64_t BH = (uint64_t)p.BH(), T = (uint64_t)p.T;
    if (!make_tmap_bf16_3d(&tk, k, BH, T, 64, 128) || !make_tmap_bf16_3d(&tv, v, BH, T, 64, 128) ||
        !make_tmap_bf16_3d(&tq, q, BH, T, 64, 256) || !make_tmap_bf16_3d(&td, dO, BH, T, 64, 256) ||
        !make_tmap_state_packed_rowrun(&rm.run[0], dSx, BH * (uint64_t)p.NC, 1) ||
        !make_tmap_state_packed_rowrun(&rm.run[1], dSx, BH * (uint64_t)p.NC, 2) ||
        !make_tmap_state_packed_rowrun(&rm.run[2], dSx, BH * (uint64_t)p.NC, 3) ||
        !make_tmap_state_packed_rowrun(&rm.run[3], dSx, BH * (uint64_t)p.NC, 4) ||
        !make_tmap_state_packed_tquads(&tst, dSx, BH * (uint64_t)p.NC))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    Args a{Aloc, g, zeta, ucol, rowterm, dzx, sscale, amax_r, dk, dv, dcum, p.lowp_grads ? 1 : 0, status, p.T, p.NC,
           (int)p.Tp()};
    cudaError_t e = cudaFuncSetAttribute(tc_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(2 * p.NC, (unsigned)p.BH());
    tc_bwd_dkdv_kernel<<<grid, THREADS, BYTES, s>>>(tk, tv, tq, td, rm, tst, a);
    return cudaGetLastError();
}

}  // namespace tm2
