// tm2_tc_out.cu -- the per-chunk output kernel of the tensor-core path (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", Sec. 5: w_ij = exp(cumA_i - cumA_j) (q_i . k_j)^2, o_i = N_i / Z_i with
// N_i = sum_{j<=i} w_ij v_j and Z_i = sum_{j<=i} w_ij.  Split at the chunk boundary:
//   [N_i, Z_i] = sum_{j in c, j<=i} P_ij [v_j, 1]  +  exp(A_i) sum_{m,n} q_i[m] q_i[n] [S_{c-1}, z_{c-1}][(m,n), :]
// with P_ij = (q_i . k_j)^2 exp(A_i - A_j) and S_{c-1}, z_{c-1} the state entering the chunk
// (written by the chunk-state scan as two fp16 planes, hi and residual, and fp32 z).
//
// One CTA per (128-token tile, chunk, b, h).
//  * Inter-chunk readout first, over 16 groups of four state rows m = 4g .. 4g + 3 of the
//    block-packed state (tm2_launch.h: only the 16 x 16 blocks bm <= bn, off-diagonal ones
//    doubled): U_g[i][(m', col)] = sum_{n >= 16 bm} q_i[n] T[(4g + m', n), col], bm = g / 4,
//    one tcgen05.mma of N = 256 per 16-key block bn >= bm and plane (Q exact in fp16, the four
//    rows of each block MN-major straight from their 8 KB TMA box), and the compute warps fold
//    it into fp32 registers, N_x[col] += q_i[4g + m'] U_g[i][(m', col)]; over all groups this
//    is sum_{m,n} q_i[m] q_i[n] S[(m,n), col] with 62.5% of the full state's products and
//    bytes.  A tensor-core instruction costs about the same for any N up to 256, so four rows
//    per instruction is what keeps the readout short.  A 17th product U_z = Q zm^T with zm[m][n] = z[(m,n)] gives
//    Z_x = sum_m q_i[m] U_z[i][m].  No operand is a rounded product, so the readout of nearly
//    orthogonal queries keeps its precision.
//  * Intra-chunk (causal 128 x 64 key blocks) in the same tensor memory afterwards: s = Q K^T
//    by tcgen05.mma from bf16 TMA tiles, the compute warps square it, apply the decay mask in
//    fp32, keep the row sums (Z) in fp32 and write P as two bf16 terms P_hi + P_lo (one bf16
//    term alone costs ~2^-9 relative per weight, enough to break the 2e-2 bar on
//    unnormalised outputs); both are A operands of P V (V MN-major from its tile).
//  * Epilogue: [N, Z] = intra + exp(A_i) [N_x, Z_x]; o = N / Z (or N), fp32; Z saved.  The
//    state planes hold ks^2 vs S and the normaliser state ks^2 z (the scan's operand scales,
//    exact powers of two), so N_x and Z_x are divided by those factors here.
// Warps 0-7 compute (warp w: tensor-memory lane quadrant w % 4, column half w / 4), warp 8
// issues TMA, warp 9 the MMAs.  Every mbarrier wait is bounded (TM2_ERR_TIMEOUT on expiry).
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"
#include "tm2_tc_tiles.cuh"

namespace tm2 {
namespace tcout {
using namespace tctile;

constexpr int C = TC_CHUNK;
constexpr int THREADS = 10 * 32;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
// The TMA ring is a byte ring of 24 units of 8 KB: request r takes the next size(r) units
// (wrapping to unit 0 when they would run past the end).  One request (one transaction
// barrier) carries both planes of a group, 2 (4 - bm) boxes: a CTA streams at a fixed cost
// per request plus a small cost per byte (measured: 8 KB requests 25 GB/s per SM, 32 KB
// requests 80-95 GB/s), so few large requests keep the readout short.
constexpr int UNIT = 8192;
constexpr int NUNIT = 24;
constexpr int RB = 32768;
constexpr int NG = 16;                       // groups of four state slices
constexpr int NREQ = NG + 3;                 // both planes of each group, then Q, K, V (intra part)
constexpr int EARLY_U = NUNIT - 2;           // units 22, 23 first hold the Q tile for conversion
constexpr int NGD = 16;                      // group-done barriers (a ring of 16, see the producer)
// shared memory
constexpr int RING = 0;
constexpr int SQH = NUNIT * UNIT;            // fp16 copy of the Q tile [128][64]
constexpr int SZH = SQH + 16384, SZL = SZH + 8192;   // zm hi / lo, [64][64] fp16
constexpr int SAV = SZL + 8192;              // chunk-local A, 256 floats
constexpr int SRED = SQH;                    // [2 halves][128 rows][2], over the Q copy (read by then)
constexpr int SMEM_BYTES = SAV + 1024 + 1024;
// tensor memory: U buffers at 0 and 256; the intra part reuses it after the readout: the
// intra accumulator, two score buffers and two (P hi, P lo) buffers, so that block b+1's
// scores are computed while block b's products run
constexpr uint32_t TM_Y = 0, TM_S = 64, TM_P = 192;   // score buffer x: 64 + 64x; P buffer x: 192 + 64x
constexpr uint32_t IDESC_U = idesc_f16_f32(128, 256, false, true);
constexpr uint32_t IDESC_Z = idesc_f16_f32(128, 64, false, false);
constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 64, false, true);

struct Args {
    const float* Aloc;   // [BH][Tp]
    const float* zx;     // [BH][NC][4096]
    const unsigned* amax;   // [BH][4] the forward scan's operand maxima (key, value)
    float* o;            // [BH][T][64]
    float* Z;            // [BH][T] or null
    int* status;
    int T, NC, Tp, normalize;
};

TM2_DEV int req_units(int r) { return r < NG ? 2 * (4 - (r >> 2)) : (r == NG ? 2 : 4); }

// Placement of the tile's requests in the byte ring (one thread, before the roles start): the
// first unit of each request, the latest earlier request whose units it reuses (-1: none),
// and whether it reuses the early Q tile's units (freed by the conversion).
TM2_DEV void place_requests(int8_t* off, int8_t* wait_req, int8_t* wait_cvt) {
    int8_t owner[NUNIT];
    for (int u = 0; u < NUNIT; ++u) owner[u] = (int8_t)(u >= EARLY_U ? -2 : -1);
    int at = 0;
    for (int r = 0; r < NREQ; ++r) {
        const int sz = req_units(r);
        if (at + sz > NUNIT) at = 0;
        int w = -1, cv = 0;
        for (int u = at; u < at + sz; ++u) {
            if (owner[u] == -2) cv = 1;
            else if (owner[u] > w) w = owner[u];
            owner[u] = (int8_t)r;
        }
        off[r] = (int8_t)at;
        wait_req[r] = (int8_t)w;
        wait_cvt[r] = (int8_t)cv;
        at += sz;
    }
}

}  // namespace tcout

using namespace tcout;

__global__ void __launch_bounds__(THREADS, 1) tc_chunk_out_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                  const __grid_constant__ CUtensorMap tmK,
                                                                  const __grid_constant__ CUtensorMap tmV,
                                                                  const __grid_constant__ CUtensorMap tmS,
                                                                  const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    // gdone[g % 4]: the products of group g are done (its ring slots are free and its U buffer
    // is full): one commit per group serves the TMA producer and the compute warps
    __shared__ __align__(8) uint64_t bar_ld, bar_full[NREQ], bar_cvt, bar_sfull[4], bar_sfree[4], bar_pfull[4],
        bar_gdone[NGD], bar_uempty[2], bar_yfull, bar_red, bar_done;
    __shared__ int8_t s_off[NREQ], s_wreq[NREQ], s_wcvt[NREQ];
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int gflags[2];         // group waits of the compute warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x & 1, c = blockIdx.x >> 1;
    const long bh = blockIdx.y;
    const int NC = a.NC;
    const int nblk = 2 * (t + 1);                // 64-key blocks at or before this tile
    const uint32_t sb0 = smem_u32(smem);
    float* sAv = reinterpret_cast<float*>(smem + SAV);
    float* sRed = reinterpret_cast<float*>(smem + SRED);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_ld), 1);
        for (int i = 0; i < NREQ; ++i) mbar_init(smem_u32(&bar_full[i]), 1);
        mbar_init(smem_u32(&bar_cvt), 256);
        for (int b = 0; b < 4; ++b) {
            mbar_init(smem_u32(&bar_sfull[b]), 1);
            mbar_init(smem_u32(&bar_sfree[b]), 256);
            mbar_init(smem_u32(&bar_pfull[b]), 256);
        }
        for (int i = 0; i < NGD; ++i) mbar_init(smem_u32(&bar_gdone[i]), 1);
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bar_uempty[i]), 256);
        mbar_init(smem_u32(&bar_yfull), 1);
        mbar_init(smem_u32(&bar_red), 256);
        mbar_init(smem_u32(&bar_done), 1);
        abort_s = 0;
        place_requests(s_off, s_wreq, s_wcvt);
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
    const uint32_t early = sb0 + RING + EARLY_U * UNIT;   // the Q tile, converted at the start

    if (warp == WARP_TMA) {
        if (lane == 0) {
            prefetch_tmap(&tmS);
            const uint32_t lb = smem_u32(&bar_ld);
            mbar_arrive_expect_tx(lb, 16384);
            tma_load_3d(early, &tmQ, lb, 0, c * C + t * 128, (int)bh);
            const int chunk_id = (int)(bh * NC + c);
            int issued = 0;
            for (int r = 0; r < NREQ && !abort_s; ++r) {
                // the units of the latest earlier request (group w) they reuse are free once that
                // group's products are done.  w is at most 12 groups (12 two-unit requests)
                // behind request r, and the products cannot pass group r, so the ring of 16
                // group-done barriers cannot have moved a phase past it.
                const int w = s_wreq[r];
                if (w >= 0 && !mbar_wait(smem_u32(&bar_gdone[w & (NGD - 1)]), (uint32_t)(w / NGD) & 1, a.status)) {
                    abort_s = 1;
                    break;
                }
                if (s_wcvt[r] && !mbar_wait(smem_u32(&bar_cvt), 0, a.status)) {   // copy made: units free
                    abort_s = 1;
                    break;
                }
                if (!TM2_CHECK(s_off[r] >= 0 && s_off[r] + req_units(r) <= NUNIT, a.status)) {
                    abort_s = 1;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_full[r]), dst = sb0 + RING + s_off[r] * UNIT;
                if (r < NG) {   // rows 4 mq .. 4 mq + 3 of the blocks (bm, bm .. 3), hi then lo plane
                    const int bm = r >> 2, mq = r & 3, nb = 4 - bm;
                    mbar_arrive_expect_tx(fb, (uint32_t)(2 * nb) * 8192);
                    for (int pl = 0; pl < 2; ++pl)
                        for (int j = 0; j < nb; ++j)
                            tma_load_4d(dst + (pl * nb + j) * 8192, &tmS, fb, 0, 0, 16 * tc_block_index(bm, bm + j) + 4 * mq,
                                        2 * chunk_id + pl);
                } else if (r == NG) {
                    mbar_arrive_expect_tx(fb, 16384);
                    tma_load_3d(dst, &tmQ, fb, 0, c * C + t * 128, (int)bh);
                } else {
                    mbar_arrive_expect_tx(fb, RB);
                    tma_load_3d(dst, r == NG + 1 ? &tmK : &tmV, fb, 0, c * C, (int)bh);
                }
                issued = r + 1;
            }
            // no copy may be in flight at exit
            mbar_wait(lb, 0, a.status);
            for (int r = 0; r < issued; ++r) mbar_wait(smem_u32(&bar_full[r]), 0, a.status);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&bar_cvt), 0, a.status);
            tc_fence_after();
            // ---- readout: U_g = Q [S_{4g} | .. | S_{4g+3}] (hi + lo plane), then U_z = Q zm^T
            for (int g = 0; g <= NG && ok; ++g) {
                const int ub = g & 1;
                const uint32_t k = (uint32_t)(g >> 1);
                if (abort_s) { ok = false; break; }
                if (g < NG && !(ok = mbar_wait(smem_u32(&bar_full[g]), 0, a.status))) break;
                if (k > 0 && !(ok = mbar_wait(smem_u32(&bar_uempty[ub]), (k - 1) & 1, a.status))) break;
                tc_fence_after();
                const uint32_t d = tmem + ub * 256;
                if (g < NG) {
                    // K over the key indices n >= 16 bm only: block (bm, bn) is box j = bn - bm
                    const int bm = g >> 2;
                    const uint32_t bhi = sb0 + RING + s_off[g] * UNIT, blo = bhi + (4 - bm) * 8192;
                    for (int j = 0; j < 4 - bm; ++j)
                        umma_bf16(d, sdesc_sw128(sb0 + SQH + (bm + j) * 32), sdesc_sw128_ex(bhi + j * 8192, 2048, 1024),
                                  IDESC_U, j > 0);
                    for (int j = 0; j < 4 - bm; ++j)
                        umma_bf16(d, sdesc_sw128(sb0 + SQH + (bm + j) * 32), sdesc_sw128_ex(blo + j * 8192, 2048, 1024),
                                  IDESC_U, 1u);

                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        umma_bf16(d, sdesc_sw128(sb0 + SQH + kk * 32), sdesc_sw128(sb0 + SZH + kk * 32), IDESC_Z, kk > 0);
                        umma_bf16(d, sdesc_sw128(sb0 + SQH + kk * 32), sdesc_sw128(sb0 + SZL + kk * 32), IDESC_Z, 1u);
                    }
                }
                umma_commit(smem_u32(&bar_gdone[g & (NGD - 1)]));
            }
            // ---- intra-chunk blocks (64 keys each), once the last U and U_z have been read
            const int rq = NG, rk = NG + 1, rv = NG + 2;
            if (ok) ok = mbar_wait(smem_u32(&bar_uempty[0]), (uint32_t)(NG >> 1) & 1, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_uempty[1]), (uint32_t)((NG - 1) >> 1) & 1, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[rq]), 0, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[rk]), 0, a.status);
            if (ok) ok = mbar_wait(smem_u32(&bar_full[rv]), 0, a.status);
            tc_fence_after();
            const uint32_t SQ = sb0 + RING + s_off[rq] * UNIT;
            const uint32_t SK = sb0 + RING + s_off[rk] * UNIT, SV = sb0 + RING + s_off[rv] * UNIT;
            auto issue_s = [&](int b) {   // s = Q K_b^T into score buffer b & 1
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + TM_S + (uint32_t)(b & 1) * 64, sdesc_sw128(SQ + kk * 32),
                              sdesc_sw128(SK + b * 8192 + kk * 32), IDESC_QK, kk > 0);
                umma_commit(smem_u32(&bar_sfull[b]));
            };
            if (ok && nblk > 0) issue_s(0);
            for (int b = 0; b < nblk && ok; ++b) {
                if (abort_s) { ok = false; break; }
                if (b + 1 < nblk) {
                    if (b >= 1 && !(ok = mbar_wait(smem_u32(&bar_sfree[b - 1]), 0, a.status))) break;
                    tc_fence_after();
                    issue_s(b + 1);
                }
                if (!(ok = mbar_wait(smem_u32(&bar_pfull[b]), 0, a.status))) break;
                tc_fence_after();
                const uint32_t pb = tmem + TM_P + (uint32_t)(b & 1) * 64;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t vd = sdesc_sw128_ex(SV + b * 8192 + kk * 2048, 8192, 1024);
                    umma_bf16_ts(tmem + TM_Y, pb + kk * 8, vd, IDESC_PV, (b > 0 || kk > 0) ? 1u : 0u);
                    umma_bf16_ts(tmem + TM_Y, pb + 32 + kk * 8, vd, IDESC_PV, 1u);
                }
            }
            if (ok) umma_commit(smem_u32(&bar_yfull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;              // tile row
        const int i = t * 128 + l;                   // token index inside the chunk
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        int kg = 0;                                  // group-wait counter
        // per-chunk terms, loaded while the Q tile is on its way: the chunk-local A of token
        // threadIdx.x (C = 256 compute threads; published by the group waits' barriers), the
        // operand maxima of the epilogue, and the normaliser matrix of the state
        static_assert(C == 256, "one chunk-local A per compute thread");
        const float av = a.Aloc[bh * a.Tp + (long)c * C + threadIdx.x];
        const unsigned am_k = a.amax[bh * 4], am_v = a.amax[bh * 4 + 1];
        float4 zr[4];
        z_tiles_load(a.zx + (bh * NC + c) * 4096, threadIdx.x, zr);
        bool ok = mbar_wait(smem_u32(&bar_ld), 0, a.status);
        sAv[threadIdx.x] = av;
        if (ok) {   // fp16 copy of the Q tile; the normaliser matrix of the state as hi + lo fp16
            const int t256 = threadIdx.x;
            for (int pc = t256; pc < 1024; pc += 256) tile_bf16_to_f16(early, sb0 + SQH, pc);
            z_tiles_store(smem + SZH, smem + SZL, zr, 1.f, t256);
            fence_proxy_async();
        }
        mbar_arrive(smem_u32(&bar_cvt));
        // ---- readout: nx[col] += q_i[m] U[i][(m, col)]; zxp += q_i[m'] U_z[i][m']
        float nx[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) nx[k] = 0.f;
        float zxp = 0.f, zin = 0.f;
        const uint8_t* qrow = smem + SQH;
#pragma unroll 1
        for (int g = 0; g <= NG && ok; ++g) {
            const int ub = g & 1;
            if (!(ok = group_wait(smem_u32(&bar_gdone[g & (NGD - 1)]), (uint32_t)(g / NGD) & 1, a.status, warp == 0, 1, 256, gflags,
                                  kg, &abort_s)))
                break;
            const uint32_t ua = tmem + lane_base + ub * 256 + h * 32;
            if (g < NG) {
                // two slices per load pair (one wait for both)
#pragma unroll 1
                for (int mp = 0; mp < 4; mp += 2) {
                    float u0[32], u1[32];
                    tmem_ld32x2(ua + mp * 64, ua + (mp + 1) * 64, u0, u1);
                    if (mp == 2) {
                        tc_fence_before();
                        mbar_arrive(smem_u32(&bar_uempty[ub]));
                    }
                    const float q0 = __half2float(*reinterpret_cast<const __half*>(qrow + swz_elem(l, 4 * g + mp)));
                    const float q1 = __half2float(*reinterpret_cast<const __half*>(qrow + swz_elem(l, 4 * g + mp + 1)));
#pragma unroll
                    for (int k = 0; k < 32; ++k) nx[k] = fmaf(q1, u1[k], fmaf(q0, u0[k], nx[k]));
                }
            } else {
                float u[32];
                tmem_ld32(ua, u);
                tc_fence_before();
                mbar_arrive(smem_u32(&bar_uempty[ub]));
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    zxp = fmaf(__half2float(*reinterpret_cast<const __half*>(qrow + swz_elem(l, h * 32 + k))), u[k], zxp);
            }
        }
        // ---- intra-chunk blocks; half h covers 32 of the 64 keys of a block
        const float Ai = sAv[i];
        for (int b = 0; b < nblk && ok; ++b) {
            if (!(ok = group_wait(smem_u32(&bar_sfull[b]), 0, a.status, warp == 0, 1, 256, gflags, kg, &abort_s))) break;
            // (the P buffer's last reader, the product of block b-2, was issued before this block's
            // scores; the commit that announced them completes only after every earlier MMA of the
            // issuing thread, so the buffer is free)
            const uint32_t sbb = tmem + lane_base + TM_S + (uint32_t)(b & 1) * 64;
            const uint32_t pbb = tmem + lane_base + TM_P + (uint32_t)(b & 1) * 64;
#pragma unroll
            for (int g2 = 0; g2 < 2; ++g2) {
                const int cc = 2 * h + g2;
                float s[16];
                tmem_ld16(sbb + cc * 16, s);
                uint32_t ph[8], pl[8];
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    float pv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int j = b * 64 + cc * 16 + 2 * k2 + u;
                        const float sv = s[2 * k2 + u];
                        pv[u] = j <= i ? sv * sv * __expf(Ai - sAv[j]) : 0.f;
                    }
                    const uint32_t h2 = pack_bf16x2(pv[0], pv[1]);
                    const float h0 = __uint_as_float(h2 << 16), h1 = __uint_as_float(h2 & 0xffff0000u);
                    const uint32_t l2 = pack_bf16x2(pv[0] - h0, pv[1] - h1);
                    // Z sums the weights exactly as the P V products see them (hi + rounded lo),
                    // so a row with one dominant weight gives o = v to fp32 precision
                    zin += (h0 + __uint_as_float(l2 << 16)) + (h1 + __uint_as_float(l2 & 0xffff0000u));
                    ph[k2] = h2;
                    pl[k2] = l2;
                }
                tmem_st8(pbb + cc * 8, ph);
                tmem_st8(pbb + 32 + cc * 8, pl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[b]));
            mbar_arrive(smem_u32(&bar_pfull[b]));
        }
        // ---- combine the two column halves' shares of Z, then the epilogue
        if (ok) {
            sRed[(h * 128 + l) * 2] = zin;
            sRed[(h * 128 + l) * 2 + 1] = zxp;
        }
        mbar_arrive(smem_u32(&bar_red));
        if (ok) ok = mbar_wait(smem_u32(&bar_red), 0, a.status);
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_yfull), 0, a.status))) {
            tc_fence_after();
            const float eA = __expf(Ai);
            const float ks = pow2_scale(am_k), vs = pow2_scale(am_v);
            const float uz = 1.f / (ks * ks), un = uz / vs;   // exact powers of two
            const float zi = sRed[l * 2] + sRed[(128 + l) * 2];
            const float zo = sRed[l * 2 + 1] + sRed[(128 + l) * 2 + 1];
            const float z = zi + eA * (uz * zo);
            float y[32];
            tmem_ld32(tmem + lane_base + TM_Y + h * 32, y);
#pragma unroll
            for (int k = 0; k < 32; ++k) y[k] += eA * (un * nx[k]);
            const long tok = (long)c * C + i;
            if (tok < a.T && TM2_CHECK(i >= 0 && i < C && h >= 0 && h < 2, a.status)) {
                const float inv = a.normalize ? (z != 0.f ? 1.f / z : 0.f) : 1.f;
                float4* dst = reinterpret_cast<float4*>(a.o + (bh * a.T + tok) * 64 + h * 32);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    dst[q4] = make_float4(y[4 * q4] * inv, y[4 * q4 + 1] * inv, y[4 * q4 + 2] * inv, y[4 * q4 + 3] * inv);
                if (a.Z && h == 0) a.Z[bh * a.T + tok] = z;
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t tc_chunk_out(const Problem& p, const void* q, const void* k, const void* v, const float* Aloc,
                         const void* Sx, const float* zx, const unsigned* amax, float* o, float* Z, cudaStream_t s) {
    CUtensorMap tq, tk, tv, ts;
    const uint64_t BH = (uint64_t)p.BH();
    if (!make_tmap_bf16_3d(&tq, q, BH, (uint64_t)p.T, 64, 128) || !make_tmap_bf16_3d(&tk, k, BH, (uint64_t)p.T, 64, C) ||
        !make_tmap_bf16_3d(&tv, v, BH, (uint64_t)p.T, 64, C) || !make_tmap_state_packed_quads(&ts, Sx, BH * (uint64_t)p.NC))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    Args a{Aloc, zx, amax, o, Z, status, p.T, p.NC, (int)p.Tp(), p.normalize ? 1 : 0};
    cudaError_t e = cudaFuncSetAttribute(tc_chunk_out_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(2 * p.NC, (unsigned)p.BH());
    tc_chunk_out_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(tq, tk, tv, ts, a);
    return cudaGetLastError();
}

}  // namespace tm2
