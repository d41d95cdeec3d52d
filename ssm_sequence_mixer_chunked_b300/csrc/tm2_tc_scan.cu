// tm2_tc_scan.cu -- the chunk-state scan of the tensor-core path (bf16 inputs, d = dv = 64).
//
// "2Mamba2Furious", Sec. 2: the second-order state has size (d^2, dv); with the running
// decay of Sec. 3-5 the state entering chunk c obeys
//     S_c = exp(g_c) S_{c-1} + sum_{j in c} w_j (k_j (x) k_j) [v_j, 1]^T,   w_j = exp(g_c - A_j),
// where A is the chunk-local running sum of -softplus(a) and g_c the chunk total; column dv
// (= 64) carries the normaliser state z.  The gradient states of the backward pass (App. C)
// obey the same recursion walked from the end,
//     dS_{c-1} = exp(g_c) dS_c + sum_{i in c} exp(A_i) zeta_i (q_i (x) q_i) [dO_i, ucol_i]^T,
// with zeta_i = 1/Z_i and ucol_i = -dO_i . o_i (normalised) or zeta = 1, ucol = 0.
//
// One CTA owns one 16 x 16 block (bm <= bn) of the (m, n) index square of one (b, h), 256 state
// rows r = 16 (m - 16 bm) + (n - 16 bn) (the block-packed layout of tm2_launch.h; the state is
// symmetric in (m, n), so 10 of the 16 blocks carry it), and walks every chunk in order.  The chunk's contribution is computed with the state rows on M,
//     H[(m,n)][col] = sum_j (key_j[m] key_j[n]) (w_j val_j[col]),
// as tcgen05.mma with M = 128 state rows (two M-blocks per CTA), N = 80 (the 64 value columns,
// the normaliser column and 15 zero rows of the operand block) and K = tokens; the key (x)
// key operand is A, built by the builder warps straight into tensor memory, and the weighted
// values are B, the operand block's rows 64-143 as the TMA brought them.  A single issuing
// thread gets about one such instruction per 120-150 SM cycles whatever N <= 128, while
// instructions of different issuing threads overlap, so each M-block has its own issuing warp
// and accumulators: 16 instructions per 64-token stage and CTA, 8 per issuer.  A commit
// (tcgen05.commit) costs its thread about as much as two of these instructions, so each
// issuer commits once per 32 tokens; that commit both frees the 32-token key-product buffer
// for the builders and, for a stage's second half, the ring slot for the TMA producer.  Shared memory
// carries only the TMA'd operand blocks (the earlier orientation, state rows on N = 256 with
// the key products staged in shared memory, was bound by shared-memory traffic at 1.2 us per
// stage; this one needs none of it), and each epilogue thread owns one whole state row, so the
// fp16 state planes go out as 128-byte rows.
//
// Precision.  Tokens whose query is nearly orthogonal to the state read it out with heavy
// cancellation, so the state must carry more than one 16-bit rounding (a single fp16
// rounding of k[m] k[n] or of the exported state puts such tokens near the 2e-2 parity
// bar).  The key (x) key operand is therefore the exact product as two fp16 terms,
// hi = fp16(k[m] k[n]) and lo = fma(k[m], k[n], -hi) (exact: bf16 inputs give 16-bit
// products), run as two MMAs; the decay weight goes into the value side (a rounding there
// only perturbs each token's contribution, which the readout then sees through non-negative
// weights).  The running state is fp32 in tensor memory and is exported as two fp16 planes
// (hi and the fp16 residual), the normaliser column as fp32.  The reverse walk scales its
// weights by 1/zmax_c (zmax_c = max over chunk c of exp(A_i) zeta_i, so they are <= 1) and
// exports slot c divided by Gamma_c = max_{c' > c} zmax_{c'} (one value per slot, the same
// in every CTA, recorded in `sscale`), so that the 1/Z factors cannot overflow fp16.
// Both walks take their key and value operands multiplied by powers of two ks, vs that bring
// the head's largest |key| and |value| into [0.5, 1) (and the reverse walk's normaliser row
// by zs, from the largest |ucol|), so the fp16 operands, the key products and the exported
// planes stay in fp16's normal range whatever the scale of the inputs (q, k, v ~ 1e-2 would
// otherwise leave the state in fp16's subnormal range).  The running state is kept in those
// units: value columns times ks^2 vs, the normaliser column times ks^2 (forward) or, after
// the reverse walk multiplies it by vs / zs, times ks^2 vs too.  S0 / z0 are brought into
// them, S_final / z_final out of them, and the readouts divide by the same exact factors.
//
// Data flow.  A pre-pass (launch_tc_scan_operands) writes one [144][64] fp16 block per
// 64-token stage: the transposed key block, the transposed weighted values, the normaliser row
// and 15 zero rows; one TMA request brings a stage into a ring slot (warp 8).  Warps 0-7 build
// the key (x) key operand of each 32 tokens (two groups of four warps taking turns; thread =
// one key index n and its state row in each M-block, hi and lo planes) into one of three
// tensor-memory buffers; warps 9 and 10 issue the MMAs of M-block 0 and 1 into accumulator
// (chunk & 1); warps 11-18 (thread = one state row, kept in registers) fold the chunk into the
// running state,
//     S_c = exp(g_c) S_{c-1} + scale H_c,
// and export it (staged in shared memory, one TMA store per plane).  An accumulator is only
// read by the fold, so the MMAs of chunk c + 1 run while chunk c is folded and exported.
// Every mbarrier wait is bounded; on expiry the status word records TM2_ERR_TIMEOUT and
// the CTA unwinds.
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {
namespace tcscan {

constexpr int C = TC_CHUNK;     // chunk length
constexpr int KS = 64;          // tokens per stage (one TMA request)
constexpr int SPC = C / KS;     // stages per chunk
constexpr int NSLOT = 8;        // ring slots, one stage each
constexpr int SLOT = TC_OPS_ROWS * 128;   // [Kt 64 rows | value^T 64 rows | normaliser row | 15 zero rows]
constexpr int NR = 256;         // state rows per CTA (two M-blocks of 128)
constexpr int NV = 80;          // accumulator columns: 64 value columns, the normaliser, 15 zero
constexpr int NACCB = 2;        // accumulator buffers per M-block (chunk it uses buffer it % NACCB)
constexpr uint32_t ACC = 80;    // accumulator of buffer b, M-block mb at column (2 b + mb) ACC
constexpr uint32_t TM_A = 2 * NACCB * ACC;   // key-product buffer x (32 tokens) at TM_A + 64 x: [mb][hi, lo]
constexpr int NAB = (512 - (int)TM_A) / 64;  // key-product buffers (5 with one accumulator buffer)
constexpr int HT = 32;          // tokens per key-product buffer
constexpr int SMEM_STG = NSLOT * SLOT;   // export staging: hi, lo planes [256 rows][128 B], 128B-swizzled
constexpr int SMEM_BYTES = SMEM_STG + 2 * 32768 + 1024;
constexpr int NBUILD = 128;     // builder threads per group (two groups: warps 0-3 first, 4-7 second half stages)
constexpr int NEPI = 256;       // epilogue threads (warps 11-18), one state row each
constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_EPI = 11;   // issuers: warps 9 (M-block 0), 10 (M-block 1)
constexpr int THREADS = 19 * 32;
constexpr uint32_t IDESC = idesc_f16_f32(128, NV, false, false);
static_assert(TC_OPS_ROWS - 64 == NV, "the operand block's rows 64.. are the N = 80 operand");
static_assert(NAB >= 3 && TM_A + 64 * NAB <= 512, "tensor memory layout");

struct Args {
    const float* g;       // [BH][NC] chunk totals
    const float* zmax;    // reverse: [BH][NC] weight scale of each chunk; forward: null
    const float* S0;      // forward: optional (BH, 4096, 64) fp32
    const float* z0;      // forward: optional (BH, 4096) fp32
    __half* Sx;           // [BH][NC][2][4096][64] fp16 planes (hi, lo), scaled by 1/sscale
    float* zx;            // [BH][NC][4096] fp32 (unscaled)
    float* sscale;        // reverse: [BH][NC] export scale per slot; forward: null (= 1)
    float* S_final;       // forward: optional (BH, 4096, 64) fp32
    float* z_final;       // forward: optional (BH, 4096) fp32
    const unsigned* amax; // [BH][4] operand maxima (fp32 bits): key, value, normaliser (reverse)
    int* status;
    int T, NC, Tp, rev;
};

// The state rows of CTA Q, block-packed (tm2_launch.h): CTA Q owns the 16 x 16 block (bm, bn),
// bm <= bn, Q = tc_block_index(bm, bn), rows r = 16 m' + n', (m, n) = (16 bm + m', 16 bn + n').
TM2_DEV void row_mn(int bm, int bn, int r, int& m, int& n) {
    m = 16 * bm + (r >> 4);
    n = 16 * bn + (r & 15);
}

TM2_DEV void ld_row_chunks4(uint32_t row_addr, int row, int c0, uint32_t* x) {   // 4 swizzled 16-byte chunks
#pragma unroll
    for (int c = 0; c < 4; ++c)
        asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(x[4 * c]), "=r"(x[4 * c + 1]), "=r"(x[4 * c + 2]), "=r"(x[4 * c + 3])
                     : "r"(row_addr + (uint32_t)(((c0 + c) ^ (row & 7)) << 4)));
}

}  // namespace tcscan

using namespace tcscan;

__global__ void __launch_bounds__(THREADS, 1) tc_state_scan_kernel(const __grid_constant__ CUtensorMap tmOps,
                                                                   const __grid_constant__ CUtensorMap tmSx,
                                                                   const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_full[NSLOT], bar_afull[NAB], bar_hsdone[NAB], bar_hfull[NACCB][2],
        bar_dfree[NACCB][2], bar_done[2];
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    __shared__ volatile int eflags[2];   // group waits of the epilogue warps
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Q = blockIdx.x;
    const long bh = blockIdx.y;
    const int NC = a.NC;
    const bool rev = a.rev != 0;
    const int nchunks = rev ? NC - 1 : NC;   // the reverse walk never needs the update of chunk 0
    const int nstages = nchunks * SPC;
    const uint32_t sbase = smem_u32(smem);

    int bm = 0, bn = 0;
    tc_block_of(Q, bm, bn);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSLOT; ++i) mbar_init(smem_u32(&bar_full[i]), 1);
        for (int i = 0; i < NAB; ++i) {
            mbar_init(smem_u32(&bar_afull[i]), NBUILD);
            mbar_init(smem_u32(&bar_hsdone[i]), 2);   // both issuers' MMAs of the half stage are done
        }
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&bar_done[i]), 1);
        for (int i = 0; i < NACCB; ++i) {
            for (int mb = 0; mb < 2; ++mb) {
                mbar_init(smem_u32(&bar_hfull[i][mb]), 1);
                mbar_init(smem_u32(&bar_dfree[i][mb]), NEPI / 2);
            }
        }
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

    auto chunk_of = [&](int it) { return rev ? NC - 1 - it : it; };

    if (warp == WARP_TMA) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmOps);
            int issued = 0;
            for (int gs = 0; gs < nstages && !abort_s; ++gs) {
                const int sl = gs % NSLOT;
                if (gs >= NSLOT) {   // the slot's previous stage: its second half stage's MMAs are done (and
                    // with them the builders' reads of it, which the issuers waited for)
                    const int ghs = 2 * (gs - NSLOT) + 1;
                    if (!mbar_wait(smem_u32(&bar_hsdone[ghs % NAB]), (uint32_t)(ghs / NAB) & 1, a.status)) {
                        abort_s = 1;
                        break;
                    }
                }
                const int stg = chunk_of(gs / SPC) * SPC + gs % SPC;   // stage index within the sequence
                const uint32_t fb = smem_u32(&bar_full[sl]);
                mbar_arrive_expect_tx(fb, SLOT);
                tma_load_3d(sbase + sl * SLOT, &tmOps, fb, 0, 0, (int)(bh * (a.Tp / KS) + stg));
                issued = gs + 1;
            }
            // no copy may be in flight at exit
            for (int gs = issued - 1; gs >= 0 && gs >= issued - NSLOT; --gs)
                mbar_wait(smem_u32(&bar_full[gs % NSLOT]), (uint32_t)(gs / NSLOT) & 1, a.status);
        }
    } else if (warp == WARP_MMA || warp == WARP_MMA + 1) {
        // ---------------------------------------------------------------- MMA issuer of M-block mb
        const int mb = warp - WARP_MMA;
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < nchunks && ok; ++it) {
                const int b = it % NACCB;
                // accumulator b was last read by the fold of chunk it - NACCB
                if (it >= NACCB &&
                    !(ok = mbar_wait(smem_u32(&bar_dfree[b][mb]), (uint32_t)((it - NACCB) / NACCB) & 1, a.status)))
                    break;
                const uint32_t d = tmem + (uint32_t)(2 * b + mb) * ACC;
                for (int s = 0; s < SPC && ok; ++s) {
                    const int gs = it * SPC + s, sl = gs % NSLOT;
                    if (abort_s) { ok = false; break; }
                    if (!(ok = mbar_wait(smem_u32(&bar_full[sl]), (uint32_t)(gs / NSLOT) & 1, a.status))) break;
                    const uint32_t bv = sbase + sl * SLOT + 64 * 128;   // rows 64-143: N = 80, K-major
                    for (int hs = 0; hs < KS / HT; ++hs) {
                        const int ghs = gs * (KS / HT) + hs, x = ghs % NAB;
                        if (!(ok = mbar_wait(smem_u32(&bar_afull[x]), (uint32_t)(ghs / NAB) & 1, a.status))) break;
                        tc_fence_after();
                        const uint32_t ah = tmem + TM_A + 64 * x + 32 * mb;
#pragma unroll
                        for (int kk = 0; kk < HT / 16; ++kk) {
                            const uint64_t bd = sdesc_sw128(bv + (2 * hs + kk) * 32);
                            umma_bf16_ts(d, ah + kk * 8, bd, IDESC, (s > 0 || hs > 0 || kk > 0) ? 1u : 0u);
                            umma_bf16_ts(d, ah + 16 + kk * 8, bd, IDESC, 1u);
                        }
                        // one commit per half stage: a commit costs the issuing thread about as
                        // much as two of these MMAs
                        umma_commit(smem_u32(&bar_hsdone[x]));
                    }
                }
                if (!ok) break;
                umma_commit(smem_u32(&bar_hfull[b][mb]));
            }
            if (!ok) abort_s = 1;
            umma_commit(smem_u32(&bar_done[mb]));
            mbar_wait(smem_u32(&bar_done[mb]), 0, a.status);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- key (x) key builders
        // group gp = warp / 4 builds the half stages hs = gp of every stage (so each group has
        // two half stages of MMA time for one build); thread: key index n, state rows (m0, n) in
        // M-block 0 and (m0 + 2, n) in M-block 1 (both at tensor-memory lane 32 (warp % 4) +
        // lane); the Kt row of n is read once, the rows of m are warp-uniform (broadcast).  A
        // column holds two consecutive tokens (the lower one in the low half), 16 columns per
        // 32 tokens; hi and lo planes.
        const int gp = warp >> 2, quad = warp & 3;
        const int r0 = quad * 32 + lane;
        int m0, m1, n;   // the key indices of rows r0 (M-block 0) and r0 + 128 (M-block 1; same n)
        row_mn(bm, bn, r0, m0, n);
        row_mn(bm, bn, r0 + 128, m1, n);
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        for (int gs = 0; gs < nstages; ++gs) {
            const int sl = gs % NSLOT;
            if (abort_s || !mbar_wait(smem_u32(&bar_full[sl]), (uint32_t)(gs / NSLOT) & 1, a.status)) {
                abort_s = 1;
                break;
            }
            const uint32_t kt = sbase + sl * SLOT;   // Kt: row x = key_j[x] over the stage's 64 tokens j
            const int hs = gp, ghs = gs * (KS / HT) + hs, x = ghs % NAB;
            if (ghs >= NAB && !mbar_wait(smem_u32(&bar_hsdone[x]), (uint32_t)(ghs / NAB - 1) & 1, a.status)) {
                abort_s = 1;
                break;
            }
            uint32_t xn[16];
            ld_row_chunks4(kt + n * 128, n, 4 * hs, xn);
#pragma unroll
            for (int mb = 0; mb < 2; ++mb) {
                const int m = mb ? m1 : m0;
                uint32_t xm[16], rh[16], rl[16];
                ld_row_chunks4(kt + m * 128, m, 4 * hs, xm);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __half2 km2 = *reinterpret_cast<const __half2*>(&xm[i]);
                    const __half2 kn2 = *reinterpret_cast<const __half2*>(&xn[i]);
                    const __half2 hi2 = __hmul2(km2, kn2);
                    const __half2 lo2 = __hfma2(km2, kn2, __hneg2(hi2));
                    rh[i] = *reinterpret_cast<const uint32_t*>(&hi2);
                    rl[i] = *reinterpret_cast<const uint32_t*>(&lo2);
                }
                const uint32_t ta = tmem + lane_base + TM_A + 64 * x + 32 * mb;
                tmem_st16(ta, rh);
                tmem_st16(ta + 16, rl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_afull[x]));
        }
    } else if (warp >= WARP_EPI) {
        // ---------------------------------------------------------------- running state (epilogue)
        // thread: state row r = 128 mb + 32 quad + lane (M-block mb = (w - 11) / 4, lane quadrant
        // w % 4), held in registers: S[0..63] the values, S[64] the normaliser.  The accumulator
        // of a chunk is only read (16 columns at a time; the group of the normaliser carries 15
        // zero columns), so the MMAs of the next chunk never wait for this fold.
        const int mb = (warp - WARP_EPI) >> 2, quad = warp & 3;
        const int r = mb * 128 + quad * 32 + lane;
        int m, n;
        row_mn(bm, bn, r, m, n);
        const long R = (long)m * 64 + n;          // the row in the full (m, n) layout
        if (!TM2_CHECK(m >= 0 && m < 64 && n >= 0 && n < 64 && r >= 0 && r < NR, a.status)) abort_s = 1;
        const long Rm = (long)n * 64 + m;         // its mirror (m, n) -> (n, m)
        // an off-diagonal block of the packed layout stands for both (m, n) and (n, m): the
        // forward exports it doubled (its readouts contract each stored row once), the reverse
        // as is (dk/dv reads each stored block in both orientations), and S0 / S_final / the
        // normaliser carry both rows
        const bool mirror = bm != bn;
        const bool twice = mirror && !rev;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        // units of the running state (see the header): forward value columns ks^2 vs, forward
        // normaliser ks^2; the reverse normaliser column is brought to ks^2 vs by vs / zs
        const float ks = pow2_scale(a.amax[bh * 4]), vs = pow2_scale(a.amax[bh * 4 + 1]);
        const float unit_v = rev ? 1.f : ks * ks * vs, unit_z = rev ? 1.f : ks * ks;
        const float zfix = rev ? vs / pow2_scale(a.amax[bh * 4 + 2]) : 1.f;
        const bool lead = warp == WARP_EPI && lane == 0;   // records sscale, issues the TMA stores
        float S[65];
        float gam = 1.f;   // reverse: running max of zmax over the chunks walked so far
#pragma unroll
        for (int i = 0; i < 65; ++i) S[i] = 0.f;
        if (!rev) {   // the initial state (forward: S0 / z0 or zero; reverse: zero); an off-diagonal
            // packed row starts from the symmetric part (S0[(m,n)] + S0[(n,m)]) / 2, which is all
            // that the readouts see; the antisymmetric rest only decays (see S_final below)
            const float f = mirror ? 0.5f : 1.f;
            if (a.S0) {
                const float4* src = reinterpret_cast<const float4*>(a.S0 + (bh * 4096 + R) * 64);
                const float4* srm = reinterpret_cast<const float4*>(a.S0 + (bh * 4096 + Rm) * 64);
#pragma unroll
                for (int q4 = 0; q4 < 16; ++q4) {
                    float4 x4 = src[q4];
                    if (mirror) {
                        const float4 y4 = srm[q4];
                        x4.x += y4.x; x4.y += y4.y; x4.z += y4.z; x4.w += y4.w;
                    }
                    S[4 * q4] = f * x4.x * unit_v; S[4 * q4 + 1] = f * x4.y * unit_v;
                    S[4 * q4 + 2] = f * x4.z * unit_v; S[4 * q4 + 3] = f * x4.w * unit_v;
                }
            }
            if (a.z0) S[64] = f * (a.z0[bh * 4096 + R] + (mirror ? a.z0[bh * 4096 + Rm] : 0.f)) * unit_z;
        }
        float dtot = 1.f;   // total decay of the walk so far (for S_final's antisymmetric part)
        // export of the state after a chunk: the values, divided by gam, as hi and residual fp16
        // planes into the swizzled staging rows (one 32 KB TMA store per plane), the normaliser
        // as fp32 straight to zx
        const uint32_t stg = sbase + SMEM_STG;
        auto export_row = [&](int slot) {
            const float inv = (twice ? 2.f : 1.f) / gam;
#pragma unroll
            for (int j = 0; j < 8; ++j) {   // 16-byte chunk j: columns 8j .. 8j + 7
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float x0 = S[8 * j + 2 * i] * inv, x1 = S[8 * j + 2 * i + 1] * inv;
                    const __half2 h2 = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(h2);
                    const __half2 l2 = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
                    hi[i] = *reinterpret_cast<const uint32_t*>(&h2);
                    lo[i] = *reinterpret_cast<const uint32_t*>(&l2);
                }
                const uint32_t off = (uint32_t)r * 128 + ((uint32_t)(j ^ (r & 7)) << 4);
                st_shared_v4(stg + off, hi[0], hi[1], hi[2], hi[3]);
                st_shared_v4(stg + 32768 + off, lo[0], lo[1], lo[2], lo[3]);
            }
            a.zx[(bh * NC + slot) * 4096 + R] = S[64];
            if (mirror) a.zx[(bh * NC + slot) * 4096 + Rm] = S[64];
            fence_proxy_async();
            named_bar_sync(2, NEPI);   // every row staged
            if (lead) {
                const int z0 = (int)((bh * NC + slot) * 2);
                tma_store_3d(&tmSx, stg, 0, Q * NR, z0);
                tma_store_3d(&tmSx, stg + 32768, 0, Q * NR, z0 + 1);
                bulk_commit_group();
            }
        };
        auto stage_begin = [&]() {   // the previous stores have read the staging rows
            if (lead) bulk_wait_read_all();
            named_bar_sync(2, NEPI);
        };
        {
            const int slot0 = rev ? NC - 1 : 0;
            if (a.sscale && lead && Q == 0) a.sscale[bh * NC + slot0] = 1.f;
            stage_begin();
            export_row(slot0);
        }
        bool ok = true;
        int kg = 0;   // group-wait counter
        for (int it = 0; it < nchunks && ok; ++it) {
            const int c = chunk_of(it), b = it % NACCB;
            const float dec = __expf(a.g[bh * NC + c]);
            const float zm = rev ? a.zmax[bh * NC + c] : 1.f;
            dtot *= dec;
            // one warp waits, the others sleep on the named barrier, and all take its outcome
            // (every epilogue thread must reach the same named barriers)
            if (!(ok = group_wait(smem_u32(&bar_hfull[b][0]), (uint32_t)(it / NACCB) & 1, a.status, warp == WARP_EPI, 2,
                                  NEPI, eflags, kg, &abort_s)))
                break;
            if (!(ok = group_wait(smem_u32(&bar_hfull[b][1]), (uint32_t)(it / NACCB) & 1, a.status, warp == WARP_EPI, 2,
                                  NEPI, eflags, kg, &abort_s)))
                break;
            // S_c = dec S_{c-1} + scale H_c
            const uint32_t cur = tmem + lane_base + (uint32_t)(2 * b + mb) * ACC;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float h[16];
                tmem_ld16(cur + 16 * k, h);
#pragma unroll
                for (int i = 0; i < 16; ++i) S[16 * k + i] = fmaf(dec, S[16 * k + i], zm * h[i]);
            }
            {
                float h[16];
                tmem_ld16(cur + 64, h);
                S[64] = fmaf(dec, S[64], zm * zfix * h[0]);
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_dfree[b][mb]));   // accumulator (b, mb) has been read
            if (rev) gam = it == 0 ? zm : fmaxf(gam, zm);
            // export the state of slot c + 1 (forward) / c - 1 (reverse)
            const int slot = rev ? c - 1 : c + 1;
            if (slot >= 0 && slot < NC) {
                if (a.sscale && lead && Q == 0) a.sscale[bh * NC + slot] = gam;
                stage_begin();
                export_row(slot);
            }
            if (!rev && it == nchunks - 1) {
                // full-layout final state; a mirrored row writes (m, n) and (n, m), each with its
                // decayed antisymmetric part of S0 restored: +-dtot (S0[(m,n)] - S0[(n,m)]) / 2
                const float iu = 1.f / unit_v;   // exact: a power of two
                if (a.S_final) {
                    float4* dst = reinterpret_cast<float4*>(a.S_final + (bh * 4096 + R) * 64);
                    float4* dsm = reinterpret_cast<float4*>(a.S_final + (bh * 4096 + Rm) * 64);
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4) {
                        float4 v4 = make_float4(S[4 * q4] * iu, S[4 * q4 + 1] * iu, S[4 * q4 + 2] * iu,
                                                S[4 * q4 + 3] * iu);
                        if (!mirror) {
                            dst[q4] = v4;
                            continue;
                        }
                        float4 d4 = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (a.S0) {
                            const float4 x4 = reinterpret_cast<const float4*>(a.S0 + (bh * 4096 + R) * 64)[q4];
                            const float4 y4 = reinterpret_cast<const float4*>(a.S0 + (bh * 4096 + Rm) * 64)[q4];
                            const float hd = 0.5f * dtot;
                            d4 = make_float4(hd * (x4.x - y4.x), hd * (x4.y - y4.y), hd * (x4.z - y4.z), hd * (x4.w - y4.w));
                        }
                        dst[q4] = make_float4(v4.x + d4.x, v4.y + d4.y, v4.z + d4.z, v4.w + d4.w);
                        dsm[q4] = make_float4(v4.x - d4.x, v4.y - d4.y, v4.z - d4.z, v4.w - d4.w);
                    }
                }
                if (a.z_final) {
                    const float zr = S[64] / unit_z;
                    float dz = 0.f;
                    if (mirror && a.z0) dz = 0.5f * dtot * (a.z0[bh * 4096 + R] - a.z0[bh * 4096 + Rm]);
                    a.z_final[bh * 4096 + R] = zr + dz;
                    if (mirror) a.z_final[bh * 4096 + Rm] = zr - dz;
                }
            }
        }
        if (lead) bulk_wait_all();
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

cudaError_t tc_state_scan(const Problem& p, const ScanIO& io, cudaStream_t s) {
    CUtensorMap tops;
    const uint64_t BH = (uint64_t)p.BH(), Tp = (uint64_t)p.Tp();
    const uint64_t dims[3] = {64, (uint64_t)TC_OPS_ROWS, BH * (Tp / KS)};
    const uint64_t strides[2] = {128, (uint64_t)TC_OPS_ROWS * 128};
    const uint32_t box[3] = {64, (uint32_t)TC_OPS_ROWS, 1};
    if (!make_tmap_f16_nd(&tops, io.ops, 3, dims, strides, box)) return cudaErrorInvalidValue;
    CUtensorMap tsx;   // the state planes as (64 columns, rows, BH x NC x 2 planes), 256-row boxes
    const uint64_t rows = (uint64_t)TC_PACKED_ROWS;   // both walks export the block-packed layout
    const uint64_t sdims[3] = {64, rows, BH * (uint64_t)p.NC * 2};
    const uint64_t sstrides[2] = {128, rows * 128};
    const uint32_t sbox[3] = {64, (uint32_t)NR, 1};
    if (!make_tmap_f16_nd(&tsx, io.Sx, 3, sdims, sstrides, sbox)) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    if (!io.amax) return cudaErrorInvalidValue;
    Args a{io.g, io.zmax, io.S0, io.z0, (__half*)io.Sx, io.zx, io.sscale, io.S_final, io.z_final, io.amax, status,
           p.T, p.NC, (int)p.Tp(), io.rev ? 1 : 0};
    cudaError_t e = cudaFuncSetAttribute(tc_state_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(TC_PACKED_BLOCKS, (unsigned)p.BH());
    tc_state_scan_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(tops, tsx, a);
    return cudaGetLastError();
}

}  // namespace tm2
