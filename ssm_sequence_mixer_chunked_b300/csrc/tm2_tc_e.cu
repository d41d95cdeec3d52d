// tm2_tc_e.cu -- the 2Mamba-E forward on the tensor cores (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", Sec. 6: causal softmax attention whose logits carry the softplus A-mask,
//   x_ij = scale q_i . k_j + cumA_i - cumA_j   (j <= i),   o_i = sum_j softmax_j(x_i.) v_j,
// with lse_i = log sum_j exp(x_ij) saved for the backward.
//
// One CTA per (128-query tile, b, h), walking the 128-key blocks at or before the tile from the
// newest (the diagonal block) to the oldest: the decay bias makes the newest keys' logits the
// largest, so the running maximum is (nearly) settled by the first block.  Per
// block: s = Q K^T by tcgen05.mma (M = N = 128, K = 64, bf16 tiles from TMA) into one of two
// tensor-memory score buffers; the compute warps (row = tensor-memory lane, half h = 64 of
// the block's keys) add the decay bias, mask, take the row maximum across both halves and
// write P = exp(x - m) as two bf16 terms, P_hi into one of two tensor-memory P buffers and
// P_lo = bf16(P - P_hi) over the score columns the writing thread has already read;
// O += P_hi V + P_lo V (P from tensor memory, V MN-major from its tile).  One bf16 rounding
// of P costs 2^-9 relative per weight, which over a long undecayed context (a -> -inf:
// thousands of keys of similar weight) puts o and the backward's dv past the 2e-2 bar;
// hi + lo carries 16 bits.  The maximum is lazy: O and the row sums are rescaled only when a
// block's maximum exceeds the one in use by more than 8 (so P <= e^8), which makes rescales
// rare.  The next block's QK^T overlaps this block's softmax, and its softmax overlaps this
// block's PV; because P_lo lives in the score buffer, the scores of block b+2 are issued once
// the products of block b have completed.  The row sums add the rounded P_hi + P_lo that the
// MMAs use, so o = O / l is exactly normalised for those weights.
// Logits are kept in log2 units (x log2 e); the decay terms are taken relative to the running
// sum at the tile's first query, so the fp32 differences stay small, and each block's key
// terms are staged once in shared memory.  Only the diagonal block is masked.
// Warps 0-7 compute (warp w: lane quadrant w % 4, key half w / 4), warp 8 issues TMA, warp 9
// the MMAs.  Every mbarrier wait is bounded (TM2_ERR_TIMEOUT on expiry).
//
// The same kernel, instantiated with KIND = ATTN_P2 or ATTN_P1, evaluates the 2Mamba mixer in
// its quadratic (C = T) form ("2Mamba2Furious", Sec. 1-2: the quadratic form costs O(T^2) but,
// with d = 64, fewer flops than the chunked form below T = 4 d^2 dv / (d + dv) = 8192; Sec. 5:
// the square on the QK product, the A-mask on the squared scores), or the first-order mixer
// with the same mask (Sec. 4, Mamba-2S: the score itself, not its square):
//   w_ij = (q_i . k_j)^p exp(cumA_i - cumA_j)  (j <= i),  N_i = sum_j w_ij v_j,  Z_i = sum_j w_ij,
// o = N / Z (normalised) or N, with Z saved.  The weights are never exponentiated scores, so
// there is no running maximum and no rescale: w = s^p 2^(crr - kw) with the decay in log2 units,
// split into bf16 hi + lo exactly as P above, Z summing the rounded weights.
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {
namespace tce {

constexpr int BQ = 128, BK = 128;
constexpr int THREADS = 10 * 32;
constexpr int WARP_TMA = 8, WARP_MMA = 9;
constexpr int NS = 4;                        // key/value stages
constexpr int TILE = BK * 128;               // [128][64] bf16
constexpr int STAGE = 2 * TILE;              // K then V
constexpr int SQ = 0;
constexpr int SSTG = TILE;                   // NS stages after the Q tile
constexpr int SMAX = SSTG + NS * STAGE;      // [2 buffers][2 halves][128] row maxima
constexpr int SSUM = SMAX + 2 * 2 * BQ * 4;  // [2 halves][128] row sums
constexpr int SFLAG = SSUM + 2 * BQ * 4;     // [2 buffers][8 warps] rescale requests
constexpr int SKW = SFLAG + 64;              // [2 buffers][128] decay terms of the block's keys
constexpr int SMEM_BYTES = SKW + 2 * BK * 4 + 1024;
constexpr uint32_t TM_S = 0;                 // score buffer x at 128 x
constexpr uint32_t TM_P = 256;               // P buffer x at 256 + 64 x (bf16 pairs)
constexpr uint32_t TM_O = 384;
constexpr float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
constexpr float LAZY = 8.f * LOG2E;          // rescale only when the maximum grows by more than e^8
constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, 64, false, true);

struct Args {
    const float* cum;    // [BH][T] inclusive running sum of -softplus(a), fp32
    const float* cum_lo; // [BH][T] its rounding residual
    float* o;            // [BH][T][64]
    float* aux;          // [BH][T]: lse (ATTN_E) or the normaliser Z (ATTN_P1, ATTN_P2)
    int* status;
    int T, NQ, BH;
    float scale;         // logit scale (ATTN_E)
    int normalize;       // o = N / Z (ATTN_P1, ATTN_P2)
};

}  // namespace tce

using namespace tce;

template <int KIND>
__global__ void __launch_bounds__(THREADS, 1) tc_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                 const __grid_constant__ CUtensorMap tmK,
                                                                 const __grid_constant__ CUtensorMap tmV,
                                                                 const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_q, bar_full[NS], bar_empty[NS], bar_sfull[2], bar_sfree[2], bar_pfull[2],
        bar_pfree[2], bar_ofull, bar_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int gflags[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // longest tiles of every head first: linear block index -> (rank of the tile's length, head)
    const long lin = (long)blockIdx.y * gridDim.x + blockIdx.x;
    const int rank = (int)(lin / a.BH);
    const long bh = lin - (long)rank * a.BH;
    const int qt = a.NQ - 1 - rank;
    const int nkb = qt + 1;                      // key blocks at or before the tile
    const uint32_t sb0 = smem_u32(smem);
    float* sMax = reinterpret_cast<float*>(smem + SMAX);
    float* sSum = reinterpret_cast<float*>(smem + SSUM);
    volatile int* sFlag = reinterpret_cast<volatile int*>(smem + SFLAG);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar_q), 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_sfull[i]), 1);
            mbar_init(smem_u32(&bar_sfree[i]), 256);
            mbar_init(smem_u32(&bar_pfull[i]), 256);
            mbar_init(smem_u32(&bar_pfree[i]), 1);
        }
        mbar_init(smem_u32(&bar_ofull), 1);
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

    if (warp == WARP_TMA) {
        if (lane == 0) {
            const uint32_t qb = smem_u32(&bar_q);
            mbar_arrive_expect_tx(qb, TILE);
            tma_load_3d(sb0 + SQ, &tmQ, qb, 0, qt * BQ, (int)bh);
            int issued = 0;
            for (int b = 0; b < nkb && !abort_s; ++b) {
                const int st = b % NS;
                if (b >= NS && !mbar_wait(smem_u32(&bar_empty[st]), (uint32_t)((b / NS) - 1) & 1, a.status)) {
                    abort_s = 1;
                    break;
                }
                const uint32_t fb = smem_u32(&bar_full[st]), dst = sb0 + SSTG + st * STAGE;
                mbar_arrive_expect_tx(fb, STAGE);
                tma_load_3d(dst, &tmK, fb, 0, (qt - b) * BK, (int)bh);          // newest block first
                tma_load_3d(dst + TILE, &tmV, fb, 0, (qt - b) * BK, (int)bh);
                issued = b + 1;
            }
            mbar_wait(qb, 0, a.status);
            for (int b = issued - 1; b >= 0 && b >= issued - NS; --b)
                mbar_wait(smem_u32(&bar_full[b % NS]), (uint32_t)(b / NS) & 1, a.status);
        }
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            bool ok = mbar_wait(smem_u32(&bar_q), 0, a.status);
            tc_fence_after();
            // s(b) = Q K_b^T, then O += P(b-1) V(b-1): block b's scores overlap block b-1's softmax
            for (int b = 0; b <= nkb && ok; ++b) {
                if (abort_s) { ok = false; break; }
                if (b < nkb) {
                    const int st = b % NS, x = b & 1;
                    if (!(ok = mbar_wait(smem_u32(&bar_full[st]), (uint32_t)(b / NS) & 1, a.status))) break;
                    if (b >= 2 && !(ok = mbar_wait(smem_u32(&bar_sfree[x]), (uint32_t)((b >> 1) - 1) & 1, a.status)))
                        break;
                    // the buffer also holds P_lo of block b-2 until that block's products complete
                    if (b >= 2 && !(ok = mbar_wait(smem_u32(&bar_pfree[x]), (uint32_t)((b >> 1) - 1) & 1, a.status)))
                        break;
                    tc_fence_after();
                    const uint32_t kb = sb0 + SSTG + st * STAGE;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem + TM_S + x * 128, sdesc_sw128(sb0 + SQ + kk * 32), sdesc_sw128(kb + kk * 32),
                                  IDESC_S, kk > 0);
                    umma_commit(smem_u32(&bar_sfull[x]));
                }
                if (b >= 1) {
                    const int c = b - 1, st = c % NS, x = c & 1;
                    if (!(ok = mbar_wait(smem_u32(&bar_pfull[x]), (uint32_t)(c >> 1) & 1, a.status))) break;
                    tc_fence_after();
                    const uint32_t vb = sb0 + SSTG + st * STAGE + TILE;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {   // keys 16 kk .. +15: half kk / 4 of the block
                        const uint64_t vd = sdesc_sw128_ex(vb + kk * 2048, 8192, 1024);
                        umma_bf16_ts(tmem + TM_O, tmem + TM_P + x * 64 + kk * 8, vd, IDESC_PV, (c > 0 || kk > 0) ? 1u : 0u);
                        umma_bf16_ts(tmem + TM_O, tmem + TM_S + x * 128 + (kk >> 2) * 64 + (kk & 3) * 8, vd, IDESC_PV, 1u);
                    }
                    umma_commit(smem_u32(&bar_pfree[x]));
                    umma_commit(smem_u32(&bar_empty[st]));
                }
            }
            if (ok) umma_commit(smem_u32(&bar_ofull));
            else abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else {
        // ---------------------------------------------------------------- compute warps
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;                  // tile row
        const long i = (long)qt * BQ + l;                // query
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const float* cumh = a.cum + bh * a.T;
        const float* cuml = a.cum_lo + bh * a.T;
        // decay terms relative to the running sum at the tile's first query, in log2 units
        const float ref = cumh[(long)qt * BQ], reflo = cuml[(long)qt * BQ];
        const float crr = i < a.T ? ((cumh[i] - ref) + (cuml[i] - reflo)) * LOG2E : 0.f;
        const float sl2 = a.scale * LOG2E;
        float* sKW = reinterpret_cast<float*>(smem + SKW);
        float m_used = -INFINITY, lsum = 0.f;
        int kg = 0;
        bool ok = true;
        // key terms: the raw running sums of block b + 1 are loaded while block b is worked on,
        // so no thread waits on their latency
        float kh = 0.f, kl = 0.f;
        bool kin = false;
        auto fetch = [&](int b) {
            const long j = (long)(qt - b) * BK + threadIdx.x;
            kin = j < a.T;
            if (kin) {
                kh = cumh[j];
                kl = cuml[j];
            }
        };
        if (threadIdx.x < BK) fetch(0);
        for (int b = 0; b < nkb && ok; ++b) {
            const int x = b & 1;
            // this block's key terms into buffer x (published by the group wait's barrier)
            if (threadIdx.x < BK) {
                sKW[x * BK + threadIdx.x] = kin ? ((kh - ref) + (kl - reflo)) * LOG2E : 0.f;
                if (b + 1 < nkb) fetch(b + 1);
            }
            if (!(ok = group_wait(smem_u32(&bar_sfull[x]), (uint32_t)(b >> 1) & 1, a.status, warp == 0, 1, 256, gflags,
                                  kg, &abort_s)))
                break;
            float s[64];
            tmem_ld32(tmem + lane_base + TM_S + x * 128 + h * 64, s);
            tmem_ld32(tmem + lane_base + TM_S + x * 128 + h * 64 + 32, s + 32);
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_sfree[x]));        // the score buffer may take block b+2
            const float4* kw4 = reinterpret_cast<const float4*>(sKW + x * BK + h * 64);
            if constexpr (KIND != ATTN_E) {
                // w = s^p 2^(crr - kw) over this thread's 64 keys; in the diagonal block key
                // h 64 + c is visible to row l when h 64 + c <= l.  P_hi into P buffer x, P_lo over
                // this thread's score columns 0-31 (its 64 scores are in registers).
#pragma unroll
                for (int r8 = 0; r8 < 4; ++r8) {
                    uint32_t ph[8], pl[8];
                    const float4 w0 = kw4[4 * r8], w1 = kw4[4 * r8 + 1], w2 = kw4[4 * r8 + 2], w3 = kw4[4 * r8 + 3];
                    const float kwv[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                                           w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        float pw[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int c = 16 * r8 + 2 * c8 + u;
                            const float sv = s[c];
                            const float e = (b > 0 || h * 64 + c <= l) ? exp2f(crr - kwv[2 * c8 + u]) : 0.f;
                            pw[u] = KIND == ATTN_P2 ? sv * sv * e : sv * e;
                        }
                        const uint32_t h2 = pack_bf16x2(pw[0], pw[1]);
                        const float h0 = __uint_as_float(h2 << 16), h1 = __uint_as_float(h2 & 0xffff0000u);
                        const uint32_t l2 = pack_bf16x2(pw[0] - h0, pw[1] - h1);
                        lsum += (h0 + __uint_as_float(l2 << 16)) + (h1 + __uint_as_float(l2 & 0xffff0000u));
                        ph[c8] = h2;
                        pl[c8] = l2;
                    }
                    tmem_st8(tmem + lane_base + TM_P + x * 64 + h * 32 + 8 * r8, ph);
                    tmem_st8(tmem + lane_base + TM_S + x * 128 + h * 64 + 8 * r8, pl);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(smem_u32(&bar_pfull[x]));
                continue;
            }
            float bmax = -INFINITY;
            if (b == 0) {   // the diagonal block: key h 64 + c is visible to row l when h 64 + c <= l
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float4 w = kw4[u];
                    const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * u + e;
                        s[c] = h * 64 + c <= l ? fmaf(sl2, s[c], crr - wv[e]) : -INFINITY;
                        bmax = fmaxf(bmax, s[c]);
                    }
                }
            } else {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float4 w = kw4[u];
                    const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int c = 4 * u + e;
                        s[c] = fmaf(sl2, s[c], crr - wv[e]);
                        bmax = fmaxf(bmax, s[c]);
                    }
                }
            }
            // row maximum over both key halves (the partner thread holds the other 64 keys), and
            // whether any row needs a rescale (one decision for the whole CTA, so that every wait
            // and every warp-wide tensor-memory access below is taken by all compute threads)
            sMax[(x * 2 + h) * BQ + l] = bmax;
            const float bm_own = bmax;
            bool need = false;
            {
                // the partner's maximum is read after the barrier; the request flag is this warp's
                const int req = __any_sync(0xffffffffu, bm_own > m_used + LAZY) ? 1 : 0;
                if (lane == 0) sFlag[x * 8 + warp] = req;
            }
            named_bar_sync(2, 256);
            bmax = fmaxf(bmax, sMax[(x * 2 + (1 - h)) * BQ + l]);
            need = bmax > m_used + LAZY;   // the same in both halves of a row
            int any = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) any |= sFlag[x * 8 + w];
            if (any) {
                const float fac = !need ? 1.f : (m_used == -INFINITY ? 0.f : exp2f(m_used - bmax));
                if (b > 0) {             // O holds blocks < b once the previous product is done
                    if (!(ok = group_wait(smem_u32(&bar_pfree[(b - 1) & 1]), (uint32_t)((b - 1) >> 1) & 1, a.status,
                                          warp == 0, 1, 256, gflags, kg, &abort_s)))
                        break;
                    float ov[32];
                    tmem_ld32(tmem + lane_base + TM_O + h * 32, ov);
#pragma unroll
                    for (int c = 0; c < 32; ++c) ov[c] *= fac;
                    tmem_st32(tmem + lane_base + TM_O + h * 32, ov);
                    tmem_wait_st();
                }
                if (need) {
                    lsum *= fac;
                    m_used = bmax;
                }
            }
            // P = exp(x - m) as P_hi (bf16) into P buffer x and P_lo = bf16(P - P_hi) over this
            // thread's score columns 0-31 (all 64 of its scores are in registers).  The P buffer's
            // last reader, the product of block b-2, was issued before the scores of block b, and
            // the commit that announced those scores completes only when every earlier MMA of the
            // issuing thread has, so it is free.
#pragma unroll
            for (int r8 = 0; r8 < 4; ++r8) {
                uint32_t ph[8], pl[8];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    const int c2 = 8 * r8 + c8;
                    const float p0 = m_used == -INFINITY ? 0.f : exp2f(s[2 * c2] - m_used);
                    const float p1 = m_used == -INFINITY ? 0.f : exp2f(s[2 * c2 + 1] - m_used);
                    const uint32_t h2 = pack_bf16x2(p0, p1);
                    const float h0 = __uint_as_float(h2 << 16), h1 = __uint_as_float(h2 & 0xffff0000u);
                    const uint32_t l2 = pack_bf16x2(p0 - h0, p1 - h1);
                    lsum += (h0 + __uint_as_float(l2 << 16)) + (h1 + __uint_as_float(l2 & 0xffff0000u));
                    ph[c8] = h2;
                    pl[c8] = l2;
                }
                tmem_st8(tmem + lane_base + TM_P + x * 64 + h * 32 + 8 * r8, ph);
                tmem_st8(tmem + lane_base + TM_S + x * 128 + h * 64 + 8 * r8, pl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_pfull[x]));
        }
        // ---- o = O / l, lse = m + log l (E) or o = N / Z, Z (the two halves' sums combined)
        if (ok) sSum[h * BQ + l] = lsum;
        named_bar_sync(2, 256);
        if (ok && !abort_s && (ok = mbar_wait(smem_u32(&bar_ofull), 0, a.status))) {
            tc_fence_after();
            const float lt = lsum + sSum[(1 - h) * BQ + l];
            float ov[32];
            tmem_ld32(tmem + lane_base + TM_O + h * 32, ov);
            if (i < a.T) {
                float inv;
                if constexpr (KIND == ATTN_E) inv = lt > 0.f ? 1.f / lt : 0.f;
                else inv = a.normalize ? (lt != 0.f ? 1.f / lt : 0.f) : 1.f;
                float4* dst = reinterpret_cast<float4*>(a.o + (bh * a.T + i) * 64 + h * 32);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    dst[u] = make_float4(ov[4 * u] * inv, ov[4 * u + 1] * inv, ov[4 * u + 2] * inv, ov[4 * u + 3] * inv);
                if (h == 0) a.aux[bh * a.T + i] = KIND == ATTN_E ? m_used * LN2 + __logf(lt) : lt;
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int KIND>
static cudaError_t launch_attn_fwd(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                                   const float* cum_lo, float scale, int normalize, float* o, float* aux,
                                   cudaStream_t s) {
    CUtensorMap tq, tk, tv;
    const uint64_t BH = (uint64_t)p.BH(), T = (uint64_t)p.T;
    if (!make_tmap_bf16_3d(&tq, q, BH, T, 64, BQ) || !make_tmap_bf16_3d(&tk, k, BH, T, 64, BK) ||
        !make_tmap_bf16_3d(&tv, v, BH, T, 64, BK))
        return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    const int NQ = (p.T + BQ - 1) / BQ;
    Args a{cum, cum_lo, o, aux, status, p.T, NQ, (int)p.BH(), scale, normalize};
    cudaError_t e = cudaFuncSetAttribute(tc_attn_fwd_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)NQ, (unsigned)p.BH());
    tc_attn_fwd_kernel<KIND><<<grid, THREADS, SMEM_BYTES, s>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

cudaError_t tc_e_fwd(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                     const float* cum_lo, float scale, float* o, float* lse, cudaStream_t s) {
    return launch_attn_fwd<ATTN_E>(p, q, k, v, cum, cum_lo, scale, 0, o, lse, s);
}

cudaError_t tc_poly_fwd(const Problem& p, int order, const void* q, const void* k, const void* v, const float* cum,
                        const float* cum_lo, float* o, float* Z, cudaStream_t s) {
    const int nrm = p.normalize ? 1 : 0;
    if (order == 2) return launch_attn_fwd<ATTN_P2>(p, q, k, v, cum, cum_lo, 1.f, nrm, o, Z, s);
    if (order == 1) return launch_attn_fwd<ATTN_P1>(p, q, k, v, cum, cum_lo, 1.f, nrm, o, Z, s);
    return cudaErrorInvalidValue;
}

}  // namespace tm2
