// tm2_tc_e_bwd.cu -- the 2Mamba-E backward on the tensor cores (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", Sec. 6 (softmax attention with the softplus A-mask as logit bias):
//   x_ij = scale q_i . k_j + cumA_i - cumA_j (j <= i),   P_ij = exp(x_ij - lse_i),
//   dP_ij = dO_i . v_j,   dx_ij = P_ij (dP_ij - D_i),   D_i = dO_i . o_i,
//   dq_i = scale sum_j dx_ij k_j,   dk_j = scale sum_i dx_ij q_i,   dv_j = sum_i P_ij dO_i,
// and the A-mask gradient from the row sums sum_j dx_ij and column sums sum_i dx_ij
// (dcumA_t = rowsum_t - colsum_t, accumulated from the end of the sequence elsewhere).
//
// Two kernels, one CTA per 128-token tile, walking the other side in 64-token sub-blocks
// (the 128-token tiles arrive by TMA in a 4-stage ring, two sub-blocks per stage):
//  * keys (kd = true): per 64-query sub-block at or after the key tile, s^T = K Q^T and
//    dP^T = V dO^T (tcgen05.mma, M = 128, N = 64) into one of three tensor-memory buffers; the
//    compute warps form P^T and dx^T, each as bf16 hi + lo (the sums of dx over queries
//    cancel, and a long undecayed context gives a key thousands of queries of similar weight,
//    so one bf16 rounding of either would cost the 2e-2 bar), written back over the scores and
//    dP they have read; then dv += (P_hi + P_lo)^T dO and dk += (dx_hi + dx_lo)^T Q with Q, dO
//    MN-major straight from their tiles.
//  * queries (kd = false): per 64-key sub-block at or before the query tile, s = Q K^T and
//    dP = dO V^T, dx hi + lo, dq += dx K.
// With three sub-block buffers the scores of sub-block s are issued while the compute warps
// work on s - 1 and the gradient products of s - 2 drain, so the softmax step overlaps the
// tensor core (a whole 128-token block needs 256 columns for scores + dP and
// cannot be double-buffered beside the operands and accumulators).
// Instantiated with KIND = ATTN_P2 or ATTN_P1 the same kernels are the backward of the
// quadratic (C = T) form of 2Mamba and of the first-order mixer (App. C / C.1):
//   w_ij = s_ij^p e_ij, e_ij = exp(cumA_i - cumA_j),  dw_ij = zeta_i (dO_i . v_j - D_i),
//   dv_j += w_ij zeta_i dO_i,  ds_ij = p s_ij^(p-1) e_ij dw_ij,  dq_i = sum_j ds_ij k_j,
//   dk_j = sum_i ds_ij q_i,  row / column sums of w_ij dw_ij for the A-mask gradient,
// with zeta = 1/Z and D = dO . o when normalised (zeta = 1, D = 0 otherwise): P and dx of the
// softmax step become w zeta and ds.
// The per-token terms of the walked sub-blocks are staged in shared memory.  Warps 0-7
// compute (warp w: lane quadrant w % 4, half w / 4 of the sub-block's 64 tokens), warp 8
// issues TMA, warp 9 the score and dP products, warp 10 the dk (or dq) products and warp 11
// the dv products: one N = 64 instruction takes its issuing thread far longer than the tensor
// core needs for it, and instructions from different threads overlap.  Every mbarrier wait is bounded (TM2_ERR_TIMEOUT on expiry).
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {
namespace tceb {

constexpr int BT = 128;                      // tokens per tile / block
constexpr int SUB = 64;                      // walked tokens per sub-block
constexpr int NB = 3;                        // tensor-memory sub-block buffers
constexpr int THREADS = 12 * 32;
constexpr int WARP_TMA = 8, WARP_MMA = 9;   // warp 9: scores + dP; warps 10 (dk or dq), 11 (dv)
constexpr int NS = 4;                        // stages of the walked blocks (two tiles each)
constexpr int TILE = BT * 128;               // [128][64] bf16
constexpr int STAGE = 2 * TILE;
constexpr int SFIX = 0;                      // this CTA's two tiles (K, V or Q, dO)
constexpr int SSTG = 2 * TILE;
constexpr int SSC = SSTG + NS * STAGE;       // [2 buffers][3 arrays][64] per-token scalars (room for 4 x 128)
constexpr int SRED = SSC + 2 * 4 * BT * 4;   // [2 halves][128]
constexpr int SMEM_BYTES = SRED + 2 * BT * 4 + 1024;
// tensor memory: sub-block buffer u at 128 u holds the scores (columns 0-63) and dP (64-127);
// accumulators at 384 (dk or dq) and 448 (dv).  The warp of half h owns score columns
// 32 h .. +31 and dP columns 64 + 32 h .. +31 of its lanes; per 16 tokens (round q of 2) it
// reads score columns 32 h + 16 q .. +15 and dP columns 64 + 32 h + 16 q .. +15, then writes
// P hi and P lo (key tiles only) over those score columns (8 each) and dx hi and dx lo over
// those dP columns.  Column c of an operand holds tokens 2c, 2c+1 of its 16.
constexpr uint32_t TM_ACC = 384, TM_ACC2 = 448;
constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_MN = idesc_bf16_f32(128, 64, false, true);

struct Args {
    const float* cum;      // [BH][T] running sums of -softplus(a), fp32
    const float* cum_lo;   // [BH][T] their rounding residuals
    const float* lse;      // [BH][T]: lse (ATTN_E) or zeta (ATTN_P1, ATTN_P2)
    const float* Dv;       // [BH][T] dO . o (null: 0)
    void* g1;              // dk kernel: dk [BH][T][64]; dq kernel: dq (fp32, or bf16 with lowp)
    void* g2;              // dk kernel: dv [BH][T][64]; dq kernel: unused
    float* sums;           // dk kernel: column sums [BH][T]; dq kernel: row sums
    int lowp;
    int* status;
    int T, NT, BH;
    float scale;
};

}  // namespace tceb

using namespace tceb;

// The softmax-gradient step for 16 walked tokens of one row (tokens tt0 .. tt0 + 15 of the
// block): scores s, dP dp, the staged per-token terms W (log2 units) and, for the key-tile
// kernel, Dq (dO . o of each walked query).  P = 2^(scale log2e s + bias) and
// dx = P (dP - D) with bias = W - crr (key tiles: W holds the query's running sum minus its
// lse) or crr - W (query tiles: crr holds the query's, W the key's).  Masked blocks zero the
// entries outside lo <= tt < hi.  Writes P hi, P lo (key tiles), dx hi, dx lo as packed bf16
// pairs.
// For KIND = ATTN_P1 / ATTN_P2 the bias is the decay exponent alone (W and crr hold running
// sums, no lse), Zq / Zr the walked queries' / this query's zeta, and P, dx become w zeta and ds.
template <int KIND, bool kd, bool masked>
__device__ __forceinline__ void softmax_grad16(const float* s, const float* dp, const float* W, const float* Dq,
                                               const float* Zq, float crr, float Dr, float Zr, float sl2, int tt0,
                                               int lo, int hi, float& sum, uint32_t* ph, uint32_t* pl, uint32_t* dh,
                                               uint32_t* dl) {
#pragma unroll
    for (int c2 = 0; c2 < 8; ++c2) {
        float pv[2], dx[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int cc = 2 * c2 + u;
            const float bias = kd ? W[cc] - crr : crr - W[cc];
            const bool vis = !masked || (tt0 + cc >= lo && tt0 + cc < hi);
            const float Dd = kd ? Dq[cc] : Dr;
            if constexpr (KIND == ATTN_E) {
                const float P = vis ? exp2f(fmaf(sl2, s[cc], bias)) : 0.f;
                const float g = P * (dp[cc] - Dd);
                sum += g;
                pv[u] = P;
                dx[u] = g;
            } else {
                const float e = vis ? exp2f(bias) : 0.f;
                const float sv = s[cc];
                const float dw = (kd ? Zq[cc] : Zr) * (dp[cc] - Dd);
                const float w = KIND == ATTN_P2 ? sv * sv * e : sv * e;
                sum += w * dw;
                pv[u] = w * (kd ? Zq[cc] : Zr);
                dx[u] = (KIND == ATTN_P2 ? 2.f * sv * e : e) * dw;
            }
        }
        if (kd) {
            const uint32_t p2 = pack_bf16x2(pv[0], pv[1]);
            ph[c2] = p2;
            pl[c2] = pack_bf16x2(pv[0] - __uint_as_float(p2 << 16), pv[1] - __uint_as_float(p2 & 0xffff0000u));
        }
        const uint32_t h2 = pack_bf16x2(dx[0], dx[1]);
        dh[c2] = h2;
        dl[c2] = pack_bf16x2(dx[0] - __uint_as_float(h2 << 16), dx[1] - __uint_as_float(h2 & 0xffff0000u));
    }
}

// kd = true: the key-tile kernel (dk, dv, column sums); false: the query-tile kernel (dq, row sums)
template <int KIND, bool kd>
__global__ void __launch_bounds__(THREADS, 1) tc_attn_bwd_kernel(const __grid_constant__ CUtensorMap tmA,
                                                                 const __grid_constant__ CUtensorMap tmB,
                                                                 const __grid_constant__ CUtensorMap tmC,
                                                                 const __grid_constant__ CUtensorMap tmD,
                                                                 const __grid_constant__ Args a) {
    // kd: A = K, B = V (this CTA's tiles), C = Q, D = dO (walked)
    // dq: A = Q, B = dO (this CTA's tiles), C = K, D = V (walked)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_fix, bar_full[NS], bar_empty[NS], bar_sfull[NB], bar_pfull[NB], bar_bfree[NB],
        bar_accfull, bar_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int gflags[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // heaviest tiles of every head first: linear block index -> (rank of the tile's length, head)
    const long lin = (long)blockIdx.y * gridDim.x + blockIdx.x;
    const int rank = (int)(lin / a.BH);
    const long bh = lin - (long)rank * a.BH;
    const int tile = kd ? rank : a.NT - 1 - rank;
    const int nblk = kd ? a.NT - tile : tile + 1;   // walked blocks: queries at or after / keys at or before
    const int blk0 = kd ? tile : 0;
    const uint32_t sb0 = smem_u32(smem);
    constexpr int NGI = kd ? 2 : 1;                  // gradient-product issuers
    const int nsb = 2 * nblk;
    float* sSc = reinterpret_cast<float*>(smem + SSC);
    float* sRed = reinterpret_cast<float*>(smem + SRED);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_fix), 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), NGI);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(smem_u32(&bar_sfull[i]), 1);
            mbar_init(smem_u32(&bar_pfull[i]), 256);
            mbar_init(smem_u32(&bar_bfree[i]), NGI);
        }
        mbar_init(smem_u32(&bar_accfull), NGI);
        mbar_init(smem_u32(&bar_done), 1 + NGI);
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

    if (warp == WARP_TMA) {
        if (lane == 0) {
            const uint32_t fb0 = smem_u32(&bar_fix);
            mbar_arrive_expect_tx(fb0, 2 * TILE);
            tma_load_3d(sb0 + SFIX, &tmA, fb0, 0, tile * BT, (int)bh);
            tma_load_3d(sb0 + SFIX + TILE, &tmB, fb0, 0, tile * BT, (int)bh);
            int issued = 0;
            for (int c = 0; c < nblk && !abort_s; ++c) {
                const int st = c % NS;
                if (c >= NS && !mbar_wait(smem_u32(&bar_empty[st]), (uint32_t)((c / NS) - 1) & 1, a.status)) {
                    abort_s = 1;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_full[st]), dst = sb0 + SSTG + st * STAGE;
                mbar_arrive_expect_tx(fb, STAGE);
                tma_load_3d(dst, &tmC, fb, 0, (blk0 + c) * BT, (int)bh);
                tma_load_3d(dst + TILE, &tmD, fb, 0, (blk0 + c) * BT, (int)bh);
                issued = c + 1;
            }
            mbar_wait(fb0, 0, a.status);
            for (int c = issued - 1; c >= 0 && c >= issued - NS; --c)
                mbar_wait(smem_u32(&bar_full[c % NS]), (uint32_t)(c / NS) & 1, a.status);
        }
    } else if (warp == WARP_MMA) {
        // scores and dP of every walked sub-block
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&bar_fix), 0, a.status);
            tc_fence_after();
            for (int s = 0; s < nsb && ok; ++s) {
                if (abort_s) { ok = false; break; }
                const int c = s >> 1, st = c % NS, u = s % NB;
                if ((s & 1) == 0 && !(ok = mbar_wait(smem_u32(&bar_full[st]), (uint32_t)(c / NS) & 1, a.status)))
                    break;
                if (s >= NB && !(ok = mbar_wait(smem_u32(&bar_bfree[u]), (uint32_t)((s / NB) - 1) & 1, a.status)))
                    break;
                tc_fence_after();
                const uint32_t sc = sb0 + SSTG + st * STAGE + (s & 1) * (SUB * 128), sd = sc + TILE;
                const uint32_t d = tmem + 128u * (uint32_t)u;
                // (fixed tile) x (walked sub-block)^T, M = 128, N = 64, K = 64
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    umma_bf16(d, sdesc_sw128(sb0 + SFIX + kk * 32), sdesc_sw128(sc + kk * 32), IDESC_S, kk > 0);
                    umma_bf16(d + 64, sdesc_sw128(sb0 + SFIX + TILE + kk * 32), sdesc_sw128(sd + kk * 32), IDESC_S,
                              kk > 0);
                }
                umma_commit(smem_u32(&bar_sfull[u]));
            }
            if (!ok) abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else if (warp > WARP_MMA) {
        // gradient products of every sub-block once the compute warps have written P and dx:
        // part 0 accumulates dk (key tiles) or dq (query tiles), part 1 dv (key tiles only).
        // Each chain has its own issuing thread so that their instructions overlap.
        const int part = warp - WARP_MMA - 1;
        if (lane == 0 && part < NGI) {
            bool ok = true;
            for (int pz = 0; pz < nsb && ok; ++pz) {
                if (abort_s) { ok = false; break; }
                const int c = pz >> 1, st = c % NS, u = pz % NB;
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[u]), (uint32_t)(pz / NB) & 1, a.status))) break;
                tc_fence_after();
                const uint32_t sc = sb0 + SSTG + st * STAGE + (pz & 1) * (SUB * 128), sd = sc + TILE;
                const uint32_t base = tmem + 128u * (uint32_t)u;
#pragma unroll
                for (int kk = 0; kk < SUB / 16; ++kk) {   // 16 tokens: half kk / 2, round kk % 2
                    const uint32_t acc0 = (pz > 0 || kk > 0) ? 1u : 0u;
                    const uint32_t off = (kk >> 1) * 32 + (kk & 1) * 16;
                    if (part == 1) {   // dv += (P hi + lo)^T dO
                        const uint32_t opP = base + off;   // P hi, then P lo at +8
                        const uint64_t dd = sdesc_sw128_ex(sd + kk * 2048, 8192, 1024);
                        umma_bf16_ts(tmem + TM_ACC2, opP, dd, IDESC_MN, acc0);
                        umma_bf16_ts(tmem + TM_ACC2, opP + 8, dd, IDESC_MN, 1u);
                    } else {           // dk += (dx hi + lo)^T Q, or dq += (dx hi + lo) K
                        const uint32_t opH = base + 64 + off;   // dx hi, then dx lo at +8
                        const uint64_t qd = sdesc_sw128_ex(sc + kk * 2048, 8192, 1024);
                        umma_bf16_ts(tmem + TM_ACC, opH, qd, IDESC_MN, acc0);
                        umma_bf16_ts(tmem + TM_ACC, opH + 8, qd, IDESC_MN, 1u);
                    }
                }
                umma_commit(smem_u32(&bar_bfree[u]));
                if (pz & 1) umma_commit(smem_u32(&bar_empty[st]));   // both sub-blocks of the stage done
            }
            if (ok) umma_commit(smem_u32(&bar_accfull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;                  // row of this CTA's tile
        const long r = (long)tile * BT + l;              // this thread's token (key for kd, query for dq)
        const bool rin = r < a.T;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const long base = bh * a.T;
        // Decay biases in log2 units, offset by the running sum at this tile's first token so
        // the fp32 differences stay small: crr is this thread's own term (key tiles: its key's
        // offset sum; query tiles: its query's offset sum minus lse), the staged W the walked
        // tokens' (key tiles: offset sum minus lse of each query; query tiles: offset sum of
        // each key).
        constexpr float LOG2E = 1.4426950408889634f;
        const long t_ref = base + (long)tile * BT;
        const float ref = a.cum[t_ref], reflo = a.cum_lo[t_ref];
        constexpr bool E = KIND == ATTN_E;
        float crr = 0.f, Dr = 0.f, Zr = 0.f;
        if (rin) {
            const float off = (a.cum[base + r] - ref) + (a.cum_lo[base + r] - reflo);
            crr = (kd || !E) ? off * LOG2E : (off - a.lse[base + r]) * LOG2E;
            if (!kd) {
                Dr = a.Dv ? a.Dv[base + r] : 0.f;
                if (!E) Zr = a.lse[base + r];
            }
        }
        const float sl2 = a.scale * LOG2E;
        float sum = 0.f;
        int kg = 0;
        bool ok = true;
        // per-token term of walked sub-block j held by this thread: arrays W at [0, 64), D at
        // [64, 128) and (key tiles of the polynomial kinds) zeta at [128, 192) of a staging buffer
        constexpr int NARR = kd ? (E ? 2 : 3) : 1;
        const bool stager = threadIdx.x < NARR * SUB;
        const int arr = threadIdx.x >> 6, tt_st = threadIdx.x & 63;
        // the raw loads for sub-block j are issued one sub-block ahead and finished (the
        // arithmetic that needs them) only when stored, so no thread waits on their latency
        struct Raw {
            float c, cl, l;
            bool in;
        };
        auto fetch = [&](int j) {
            const long t = (long)blk0 * BT + (long)j * SUB + tt_st;
            Raw w{0.f, 0.f, 0.f, t < a.T};
            if (w.in) {
                if (arr == 1) w.l = a.Dv ? a.Dv[base + t] : 0.f;
                else if (arr == 2) w.l = a.lse[base + t];
                else {
                    w.c = a.cum[base + t];
                    w.cl = a.cum_lo[base + t];
                    if (kd && E) w.l = a.lse[base + t];
                }
            }
            return w;
        };
        auto finish = [&](const Raw& w) {
            if (!w.in) return 0.f;
            if (arr != 0) return w.l;
            const float off = (w.c - ref) + (w.cl - reflo);
            return (kd && E) ? (off - w.l) * LOG2E : off * LOG2E;
        };
        Raw nxt = stager ? fetch(0) : Raw{0.f, 0.f, 0.f, false};
        for (int sbk = 0; sbk < nsb && ok; ++sbk) {
            const int x = sbk & 1, u = sbk % NB;
            const long t0 = (long)blk0 * BT + (long)sbk * SUB;
            // the walked sub-block's terms into buffer x; the next one's loads fly meanwhile
            float* sc = sSc + x * 3 * SUB;
            if (stager && TM2_CHECK(arr * SUB + tt_st < 3 * SUB && u < NB, a.status)) {
                sc[arr * SUB + tt_st] = finish(nxt);
                if (sbk + 1 < nsb) nxt = fetch(sbk + 1);
            }
            // masks only on the diagonal block's sub-blocks and on a sub-block that runs past
            // the sequence end
            const bool masked = kd ? (sbk < 2 || t0 + SUB > a.T) : (sbk >= nsb - 2);
            const int lo = kd ? (int)(r - t0) : 0;
            const int hi = kd ? (int)min((long)SUB, (long)a.T - t0) : (int)(r - t0) + 1;
            // (the group wait's barrier also publishes the staged terms to every thread)
            if (!(ok = group_wait(smem_u32(&bar_sfull[u]), (uint32_t)(sbk / NB) & 1, a.status, warp == 0, 1, 256,
                                  gflags, kg, &abort_s)))
                break;
            const uint32_t bufc = tmem + lane_base + 128u * (uint32_t)u;
            // this warp's 32 score and 32 dP columns under one wait
            float s32[32], dp32[32];
            tmem_ld32x2(bufc + h * 32, bufc + 64 + h * 32, s32, dp32);
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4) {
                const int tt0 = h * 32 + q4 * 16;
                const float* s = s32 + 16 * q4;
                const float* dp = dp32 + 16 * q4;
                float W[16], Dq[16], Zq[16];
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    const float4 w4 = reinterpret_cast<const float4*>(sc + tt0)[v4];
                    W[4 * v4] = w4.x, W[4 * v4 + 1] = w4.y, W[4 * v4 + 2] = w4.z, W[4 * v4 + 3] = w4.w;
                    if (kd) {
                        const float4 d4 = reinterpret_cast<const float4*>(sc + SUB + tt0)[v4];
                        Dq[4 * v4] = d4.x, Dq[4 * v4 + 1] = d4.y, Dq[4 * v4 + 2] = d4.z, Dq[4 * v4 + 3] = d4.w;
                        if (!E) {
                            const float4 z4 = reinterpret_cast<const float4*>(sc + 2 * SUB + tt0)[v4];
                            Zq[4 * v4] = z4.x, Zq[4 * v4 + 1] = z4.y, Zq[4 * v4 + 2] = z4.z, Zq[4 * v4 + 3] = z4.w;
                        }
                    }
                }
                uint32_t ph[8], pl[8], dh[8], dl[8];
                if (masked)
                    softmax_grad16<KIND, kd, true>(s, dp, W, Dq, Zq, crr, Dr, Zr, sl2, tt0, lo, hi, sum, ph, pl, dh, dl);
                else
                    softmax_grad16<KIND, kd, false>(s, dp, W, Dq, Zq, crr, Dr, Zr, sl2, tt0, lo, hi, sum, ph, pl, dh, dl);
                if (kd) {   // over this round's score columns
                    tmem_st8(bufc + tt0, ph);
                    tmem_st8(bufc + tt0 + 8, pl);
                }
                tmem_st8(bufc + 64 + tt0, dh);   // over this round's dP columns
                tmem_st8(bufc + 64 + tt0 + 8, dl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_pfull[u]));
        }
        // ---- gradients of this tile's tokens; the two halves' sums combined
        if (ok) sRed[h * BT + l] = sum;
        named_bar_sync(2, 256);
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_accfull), 0, a.status))) {
            tc_fence_after();
            const float tot = sum + sRed[(1 - h) * BT + l];
            float g[32];
            tmem_ld32(tmem + lane_base + TM_ACC + h * 32, g);
            if (rin) {
#pragma unroll
                for (int u = 0; u < 32; ++u) g[u] *= a.scale;
                store_row32(a.g1, (base + r) * 64 + h * 32, g, a.lowp != 0);
                if (h == 0) a.sums[base + r] = tot;
            }
            if (kd) {
                tmem_ld32(tmem + lane_base + TM_ACC2 + h * 32, g);
                if (rin) {
                    store_row32(a.g2, (base + r) * 64 + h * 32, g, a.lowp != 0);
                }
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int KIND>
static cudaError_t launch_attn_bwd(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                                   const float* cum_lo, const float* lse_or_zeta, const float* Dvec, const void* dO,
                                   float scale, void* dq, void* dk, void* dv, float* rowsum, float* colsum,
                                   cudaStream_t s) {
    CUtensorMap tq, tk, tv, td;
    const uint64_t BH = (uint64_t)p.BH(), T = (uint64_t)p.T;
    if (!make_tmap_bf16_3d(&tq, q, BH, T, 64, BT) || !make_tmap_bf16_3d(&tk, k, BH, T, 64, BT) ||
        !make_tmap_bf16_3d(&tv, v, BH, T, 64, BT) || !make_tmap_bf16_3d(&td, dO, BH, T, 64, BT))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    const int NT = (p.T + BT - 1) / BT;
    dim3 grid((unsigned)NT, (unsigned)p.BH());
    {
        Args a{cum, cum_lo, lse_or_zeta, Dvec, dk, dv, colsum, p.lowp_grads ? 1 : 0, status, p.T, NT, (int)p.BH(),
               scale};
        cudaError_t e = cudaFuncSetAttribute(tc_attn_bwd_kernel<KIND, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SMEM_BYTES);
        if (e != cudaSuccess) return e;
        tc_attn_bwd_kernel<KIND, true><<<grid, THREADS, SMEM_BYTES, s>>>(tk, tv, tq, td, a);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    {
        Args a{cum, cum_lo, lse_or_zeta, Dvec, dq, nullptr, rowsum, p.lowp_grads ? 1 : 0, status, p.T, NT, (int)p.BH(),
               scale};
        cudaError_t e = cudaFuncSetAttribute(tc_attn_bwd_kernel<KIND, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        tc_attn_bwd_kernel<KIND, false><<<grid, THREADS, SMEM_BYTES, s>>>(tq, td, tk, tv, a);
    }
    return cudaGetLastError();
}

cudaError_t tc_e_bwd(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                     const float* cum_lo, const float* lse, const float* Dvec, const void* dO, float scale, void* dq,
                     void* dk, void* dv, float* rowsum, float* colsum, cudaStream_t s) {
    return launch_attn_bwd<ATTN_E>(p, q, k, v, cum, cum_lo, lse, Dvec, dO, scale, dq, dk, dv, rowsum, colsum, s);
}

cudaError_t tc_poly_bwd(const Problem& p, int order, const void* q, const void* k, const void* v, const float* cum,
                        const float* cum_lo, const float* zeta, const float* D, const void* dO, void* dq, void* dk,
                        void* dv, float* rowsum, float* colsum, cudaStream_t s) {
    if (order == 2)
        return launch_attn_bwd<ATTN_P2>(p, q, k, v, cum, cum_lo, zeta, D, dO, 1.f, dq, dk, dv, rowsum, colsum, s);
    if (order == 1)
        return launch_attn_bwd<ATTN_P1>(p, q, k, v, cum, cum_lo, zeta, D, dO, 1.f, dq, dk, dv, rowsum, colsum, s);
    return cudaErrorInvalidValue;
}

}  // namespace tm2
