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
// One CTA owns the 256 state rows r = m*64 + n with m in {4Q .. 4Q+3} of one (b, h) and
// walks every chunk in order.  Per chunk, the local contribution of each 128-row tile is a
// dense contraction  H[(m,n), col] = sum_j key_j[m] key_j[n] (w_j val_j[col])  (M = 128 rows,
// N = 80 = 64 value columns + the normaliser column + 15 zero columns, K = chunk length),
// issued as tcgen05.mma with A (the key (x) key rows) in tensor memory and B (the weighted
// value tile, MN-major) in shared memory.
//
// Precision.  Tokens whose query is nearly orthogonal to the state read it out with heavy
// cancellation, so the state must carry more than one 16-bit rounding (a single fp16
// rounding of k[m] k[n] or of the exported state puts such tokens near the 2e-2 parity
// bar).  The A operand is therefore the exact product as two fp16 terms, hi = fp16(k[m] k[n])
// and lo = fma(k[m], k[n], -hi) (exact: bf16 inputs give 16-bit products), run as two MMAs;
// the decay weight goes into B (a rounding of the value side only perturbs each token's
// contribution, which the readout then sees through non-negative weights).  The running
// state is fp32 in the epilogue warps' registers and is exported as two fp16 planes
// (hi and the fp16 residual), the normaliser column as fp32.  The reverse walk scales its
// weights by 1/zmax_c (zmax_c = max over chunk c of exp(A_i) zeta_i, so they are <= 1) and
// exports slot c divided by Gamma_c = max_{c' > c} zmax_{c'} (one value per slot, the same
// in every CTA, recorded in `sscale`), so that the 1/Z factors cannot overflow fp16.
//
// The operands come from a pre-pass (launch_tc_scan_operands): per 64-token stage one
// [192][64] fp16 block holding the transposed key block Kt[n][j], the weighted values
// fp16(w_j val_j) and the normaliser column.  One TMA request brings two consecutive stages
// (48 KB): a TMA request costs a few hundred ns of issue time whatever its size, so large
// requests are what keeps the stream ahead of the tensor cores.  Warp roles (576 threads): warps 0-7 build the A operand
// straight from the Kt tile (warp w: tensor-memory lane quadrant w % 4, half w / 4 of the
// 64 rows of a stage); warps 8-15 fold the accumulator into the running state once per chunk
// (warp 8+e: tile e / 4, quadrant e % 4; one state row per thread) and export it; warp 16
// issues the TMA loads, warp 17 the MMAs.
// Every mbarrier wait is bounded; on expiry the status word records TM2_ERR_TIMEOUT and
// the CTA unwinds.
#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {
namespace tcscan {

constexpr int C = TC_CHUNK;     // chunk length
constexpr int KS = 64;          // tokens per stage
constexpr int SPC = C / KS;     // stages per chunk
constexpr int NP = 4;           // stage-pair buffers (one TMA request brings two stages)
constexpr int NN = 80;          // MMA N
constexpr int NG_THREADS = 256, NE_THREADS = 256;
constexpr int WARP_TMA = 16, WARP_MMA = 17;
constexpr int THREADS = 18 * 32;
constexpr int TILE = KS * 128;                // one [64][64] 16-bit tile, 128B-swizzled
constexpr int STAGE = 3 * TILE;               // Kt, then the value block and the normaliser block
constexpr int PSLOT = 2 * STAGE;              // two consecutive stages
constexpr int SMEM_BYTES = NP * PSLOT + 1024;
constexpr uint32_t TM_H = 0;                  // accumulator: tile t at t * 80
constexpr uint32_t TM_A = 160;                // A buffers: 160 + buf*128 + tile*64 + {0: hi, 32: lo}
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_f16_f32(128, NN, false, true);

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
    int* status;
    int T, NC, Tp, rev;
};

}  // namespace tcscan

using namespace tcscan;

__global__ void __launch_bounds__(THREADS, 1) tc_state_scan_kernel(const __grid_constant__ CUtensorMap tmOps,
                                                                   const __grid_constant__ Args a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_full[NP], bar_empty[NP], bar_afull[2], bar_aempty[2], bar_hfull,
        bar_hempty, bar_done;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Q = blockIdx.x;
    const long bh = blockIdx.y;
    const int NC = a.NC;
    const bool rev = a.rev != 0;
    const int nchunks = rev ? NC - 1 : NC;   // the reverse walk never needs the update of chunk 0
    const int nstages = nchunks * SPC;
    const uint32_t sbase = smem_u32(smem);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NP; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_afull[i]), NG_THREADS);
            mbar_init(smem_u32(&bar_aempty[i]), 1);
        }
        mbar_init(smem_u32(&bar_hfull), 1);
        mbar_init(smem_u32(&bar_hempty), NE_THREADS);
        mbar_init(smem_u32(&bar_done), 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), TMEM_COLS);
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
            const int npairs = nstages / 2;          // stage pairs never straddle a chunk
            int issued = 0;
            for (int pg = 0; pg < npairs && !abort_s; ++pg) {
                const int ps = pg % NP;
                if (pg >= NP && !mbar_wait(smem_u32(&bar_empty[ps]), ((pg / NP) - 1) & 1, a.status)) {
                    abort_s = 1;
                    break;
                }
                const int c = chunk_of(pg / (SPC / 2));
                const int stg = c * SPC + (pg % (SPC / 2)) * 2;   // first stage of the pair in the sequence
                const uint32_t fb = smem_u32(&bar_full[ps]);
                mbar_arrive_expect_tx(fb, PSLOT);
                tma_load_3d(sbase + ps * PSLOT, &tmOps, fb, 0, 0, (int)(bh * (a.Tp / KS) + stg));
                issued = pg + 1;
            }
            // wait for the last use of every pair buffer, so no copy is in flight at exit
            for (int pg = issued - 1; pg >= 0 && pg >= issued - NP; --pg)
                mbar_wait(smem_u32(&bar_full[pg % NP]), (pg / NP) & 1, a.status);
        }
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < nchunks && ok; ++it) {
                if (it >= 1 && !(ok = mbar_wait(smem_u32(&bar_hempty), (it - 1) & 1, a.status))) break;
                tc_fence_after();
                for (int s = 0; s < SPC; ++s) {
                    const int gs = it * SPC + s, pg = gs >> 1, ps = pg % NP, ab = gs & 1;
                    if (abort_s) { ok = false; break; }
                    if ((gs & 1) == 0 && !(ok = mbar_wait(smem_u32(&bar_full[ps]), (pg / NP) & 1, a.status))) break;
                    if (!(ok = mbar_wait(smem_u32(&bar_afull[ab]), (gs >> 1) & 1, a.status))) break;
                    tc_fence_after();
                    const uint32_t vb = sbase + ps * PSLOT + (gs & 1) * STAGE + TILE;
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int kk = 0; kk < KS / 16; ++kk) {
                            const uint64_t bd = sdesc_sw128_ex(vb + kk * 2048, TILE, 1024);
                            const uint32_t aa = tmem + TM_A + ab * 128 + t * 64 + kk * 8;
                            umma_bf16_ts(tmem + TM_H + t * 80, aa, bd, IDESC, (s > 0 || kk > 0) ? 1u : 0u);
                            umma_bf16_ts(tmem + TM_H + t * 80, aa + 32, bd, IDESC, 1u);
                        }
                    if (gs & 1) umma_commit(smem_u32(&bar_empty[ps]));
                    umma_commit(smem_u32(&bar_aempty[ab]));
                }
                if (!ok) break;
                umma_commit(smem_u32(&bar_hfull));
            }
            if (!ok) abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- A-operand builders
        const int quad = warp & 3, h = warp >> 2;
        const int l = quad * 32 + lane;              // tensor-memory lane = tile row
        const int n = l & 63, moff = l >> 6;
        for (int gs = 0; gs < nstages; ++gs) {
            const int pg = gs >> 1, ps = pg % NP, ab = gs & 1;
            if (abort_s || !mbar_wait(smem_u32(&bar_full[ps]), (pg / NP) & 1, a.status)) {
                abort_s = 1;
                break;
            }
            if (gs >= 2 && !mbar_wait(smem_u32(&bar_aempty[ab]), ((gs >> 1) - 1) & 1, a.status)) {
                abort_s = 1;
                break;
            }
            tc_fence_after();
            const uint32_t kt = sbase + ps * PSLOT + (gs & 1) * STAGE;   // Kt tile: row n = key_j[n] over j, swizzled
            // key_j[n] for this thread's 32 rows j of the stage, as fp16 pairs
            uint32_t kp[16];
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(kp[4 * v4]), "=r"(kp[4 * v4 + 1]), "=r"(kp[4 * v4 + 2]), "=r"(kp[4 * v4 + 3])
                             : "r"(kt + n * 128 + (((h * 4 + v4) ^ (n & 7)) << 4)));
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int m = 4 * Q + 2 * t + moff;   // the same for the whole warp
                uint32_t rh[16], rl[16];
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                    uint32_t xs[4];
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(xs[0]), "=r"(xs[1]), "=r"(xs[2]), "=r"(xs[3])
                                 : "r"(kt + m * 128 + (((h * 4 + v4) ^ (m & 7)) << 4)));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int p = v4 * 4 + i;
                        const __half2 km2 = *reinterpret_cast<const __half2*>(&xs[i]);
                        const __half2 kn2 = *reinterpret_cast<const __half2*>(&kp[p]);
                        const __half2 hi2 = __hmul2(km2, kn2);
                        const __half2 lo2 = __hfma2(km2, kn2, __hneg2(hi2));
                        rh[p] = *reinterpret_cast<const uint32_t*>(&hi2);
                        rl[p] = *reinterpret_cast<const uint32_t*>(&lo2);
                    }
                }
                const uint32_t ad = tmem + ((uint32_t)(quad * 32) << 16) + TM_A + ab * 128 + t * 64 + h * 16;
                tmem_st16(ad, rh);
                tmem_st16(ad + 32, rl);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_afull[ab]));
        }
    } else {
        // ---------------------------------------------------------------- running state
        const int e = warp - 8, t = e >> 2, quad = e & 3;
        const int l = quad * 32 + lane;
        const int m = 4 * Q + 2 * t + (l >> 6), n = l & 63, r = m * 64 + n;
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        float S[65];
        if (!rev && a.S0) {
            const float4* src = reinterpret_cast<const float4*>(a.S0 + (bh * 4096 + r) * 64);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 x = src[i];
                S[4 * i] = x.x; S[4 * i + 1] = x.y; S[4 * i + 2] = x.z; S[4 * i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) S[i] = 0.f;
        }
        S[64] = (!rev && a.z0) ? a.z0[bh * 4096 + r] : 0.f;
        float gam = 1.f;   // reverse: running max of zmax over the chunks walked so far
        // exports the running state as two fp16 planes (divided by gam) plus fp32 z
        auto export_state = [&](int slot) {
            const float inv = 1.f / gam;
            if (a.sscale && Q == 0 && e == 0 && lane == 0) a.sscale[bh * NC + slot] = gam;
            __half* base = a.Sx + ((bh * NC + slot) * 2) * (4096L * 64) + (long)r * 64;
            uint4* dh = reinterpret_cast<uint4*>(base);
            uint4* dl = reinterpret_cast<uint4*>(base + 4096L * 64);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t ph[4], pl[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float x0 = S[8 * i + 2 * u] * inv, x1 = S[8 * i + 2 * u + 1] * inv;
                    ph[u] = pack_f16x2(x0, x1);
                    const __half2 h2 = *reinterpret_cast<const __half2*>(&ph[u]);
                    pl[u] = pack_f16x2(x0 - __low2float(h2), x1 - __high2float(h2));
                }
                dh[i] = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                dl[i] = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            a.zx[(bh * NC + slot) * 4096 + r] = S[64];
        };
        // folds the accumulator of chunk `it` into the running state
        auto update = [&](int it, float gcv, float scl) -> bool {
            if (abort_s || !mbar_wait(smem_u32(&bar_hfull), it & 1, a.status)) return false;
            tc_fence_after();
            const float dec = __expf(gcv);
            const uint32_t hb = tmem + lane_base + TM_H + t * 80;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float hv[16];
                tmem_ld16(hb + 16 * i, hv);
#pragma unroll
                for (int k = 0; k < 16; ++k) S[16 * i + k] = fmaf(dec, S[16 * i + k], scl * hv[k]);
            }
            S[64] = fmaf(dec, S[64], scl * tmem_ld1(hb + 64));
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_hempty));
            if (rev) gam = it == 0 ? scl : fmaxf(gam, scl);
            return true;
        };
        export_state(rev ? NC - 1 : 0);
        bool ok = true;
        for (int it = 0; it < nchunks && ok; ++it) {
            const int c = chunk_of(it);
            const float gcv = a.g[bh * NC + c];                 // loaded while the chunk's MMAs run
            const float scl = rev ? a.zmax[bh * NC + c] : 1.f;
            if (!(ok = update(it, gcv, scl))) break;
            const int slot = rev ? c - 1 : c + 1;
            if (slot >= 0 && slot < NC) export_state(slot);
        }
        if (!ok) abort_s = 1;
        if (ok && !rev) {
            if (a.S_final) {
                float4* dst = reinterpret_cast<float4*>(a.S_final + (bh * 4096 + r) * 64);
#pragma unroll
                for (int i = 0; i < 16; ++i) dst[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
            }
            if (a.z_final) a.z_final[bh * 4096 + r] = S[64];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

cudaError_t tc_state_scan(const Problem& p, const ScanIO& io, cudaStream_t s) {
    CUtensorMap tops;
    const uint64_t BH = (uint64_t)p.BH(), Tp = (uint64_t)p.Tp();
    const uint64_t dims[3] = {64, (uint64_t)TC_OPS_ROWS, BH * (Tp / KS)};
    const uint64_t strides[2] = {128, (uint64_t)TC_OPS_ROWS * 128};
    const uint32_t box[3] = {64, (uint32_t)TC_OPS_ROWS, 2};
    if (!make_tmap_f16_nd(&tops, io.ops, 3, dims, strides, box)) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    Args a{io.g, io.zmax, io.S0, io.z0, (__half*)io.Sx, io.zx, io.sscale, io.S_final, io.z_final, status, p.T, p.NC,
           (int)p.Tp(), io.rev ? 1 : 0};
    cudaError_t e = cudaFuncSetAttribute(tc_state_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(16, (unsigned)p.BH());
    tc_state_scan_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(tops, a);
    return cudaGetLastError();
}

}  // namespace tm2
