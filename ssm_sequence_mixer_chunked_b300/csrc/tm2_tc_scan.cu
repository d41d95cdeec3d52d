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
// One CTA owns NR (128 or 256) state rows r = m*64 + n with m in {MP Q .. MP Q + MP - 1}
// (MP = NR / 64) of one (b, h) and walks every chunk in order.  The chunk's contribution is
// computed transposed,
//     H^T[col][(m,n)] = sum_j (w_j val_j[col]) key_j[m] key_j[n],
// as tcgen05.mma with M = 128 (the 64 value columns, the normaliser column and zero rows),
// N = NR (the CTA's state rows) and K = tokens: 8 instructions per 64-token stage.  NR = 128
// would give 32 CTAs per head (1024 at B = 2, H = 16: 6.9 waves on 148 SMs where NR = 256
// gives 3.5, i.e. 4 with a half-empty last one) and halve each stage's operand building, but
// a stage still costs its 8 instructions (0.85 us at N = 128 against 1.2 us at N = 256), so
// the walk took 0.76 ms against 0.62 ms at B = 2, H = 16, T = 8192: NR = 256 is used.
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
// Data flow.  A pre-pass (launch_tc_scan_operands) writes one [136][64] fp16 block per
// 64-token stage: the transposed key block and the transposed weighted values with the
// normaliser row (and 7 zero rows); one TMA request brings a stage into a ring slot.  Warps
// 0-7 build the key (x) key operand of a stage in shared memory (thread = one key index n and
// 16 tokens, the four state rows of that n, hi and lo planes, 128-byte swizzled K-major),
// double-buffered; warp 15 issues the MMAs into tensor-memory buffer
// (chunk & 1); warps 8, 9, 12, 13 (value columns, lane quadrants 0 and 1) and 10, 14 (the
// normaliser column, lane 64) fold the chunk into the running state,
//     S_c = exp(g_c) S_{c-1} + scale H^T_c,
// written back over H^T_c in tensor memory (so the buffer of chunk c-1 frees as soon as it
// has been read), and export it; warp 11 issues the TMA loads.
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
constexpr int NSLOT = 5;        // ring slots, one stage each
constexpr int SLOT = TC_OPS_ROWS * 128;   // [Kt 64 rows | value^T 64 rows | normaliser row | 7 zero rows]
constexpr int NR_ROWS = 256;    // state rows per CTA (128 or 256; 256 measured faster)
// key (x) key operand of a stage: hi [NR][64] then lo [NR][64]
__host__ __device__ constexpr int bbuf(int NR) { return NR * 256; }
constexpr int SB = NSLOT * SLOT;
__host__ __device__ constexpr int smem_bytes(int NR) { return SB + 2 * bbuf(NR) + 1024; }
constexpr int THREADS = 16 * 32;
constexpr int NBUILD = 256;     // builder threads (warps 0-7)
constexpr int NEPI = 192;       // epilogue threads (warps 8, 9, 10, 12, 13, 14)
constexpr int WARP_TMA = 11, WARP_MMA = 15;

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

}  // namespace tcscan

using namespace tcscan;

template <int NR>
__global__ void __launch_bounds__(THREADS, 1) tc_state_scan_kernel(const __grid_constant__ CUtensorMap tmOps,
                                                                   const __grid_constant__ Args a) {
    constexpr int MP = NR / 64;                  // key indices m per CTA
    constexpr int BBUF = bbuf(NR);
    constexpr uint32_t IDESC = idesc_f16_f32(128, NR, false, false);
    constexpr uint32_t TCOLS = 2 * NR;           // two accumulator buffers of NR columns
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    __shared__ __align__(8) uint64_t bar_full[NSLOT], bar_empty[NSLOT], bar_bfull[2], bar_bempty[2], bar_hfull[2],
        bar_dfree[2], bar_done;
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
        for (int i = 0; i < NSLOT; ++i) {
            mbar_init(smem_u32(&bar_full[i]), 1);
            mbar_init(smem_u32(&bar_empty[i]), NBUILD + 1);   // builders read Kt, the MMAs read the values
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_bfull[i]), NBUILD);
            mbar_init(smem_u32(&bar_bempty[i]), 1);
            mbar_init(smem_u32(&bar_hfull[i]), 1);
            mbar_init(smem_u32(&bar_dfree[i]), NEPI);
        }
        mbar_init(smem_u32(&bar_done), 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base_s), TCOLS);
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
                const uint32_t u = (uint32_t)(gs / NSLOT);
                if (u > 0 && !mbar_wait(smem_u32(&bar_empty[sl]), (u - 1) & 1, a.status)) {
                    abort_s = 1;
                    break;
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
    } else if (warp == WARP_MMA) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < nchunks && ok; ++it) {
                const int b = it & 1;
                if (it >= 1 && !(ok = mbar_wait(smem_u32(&bar_dfree[b]), (uint32_t)((it - 1) >> 1) & 1, a.status)))
                    break;
                for (int s = 0; s < SPC; ++s) {
                    const int gs = it * SPC + s, sl = gs % NSLOT, sb = gs & 1;
                    if (abort_s) { ok = false; break; }
                    if (!(ok = mbar_wait(smem_u32(&bar_full[sl]), (uint32_t)(gs / NSLOT) & 1, a.status))) break;
                    if (!(ok = mbar_wait(smem_u32(&bar_bfull[sb]), (uint32_t)(gs >> 1) & 1, a.status))) break;
                    tc_fence_after();
                    // value^T rows (M), K-major.  M rows 72-127 read whatever follows the slot: they
                    // only reach accumulator lanes 72-127, which nothing reads.
                    const uint32_t av = sbase + sl * SLOT + 8192;
                    const uint32_t bhi = sbase + SB + sb * BBUF, blo = bhi + NR * 128;
                    const uint32_t d = tmem + (uint32_t)b * NR;
#pragma unroll
                    for (int kk = 0; kk < KS / 16; ++kk)
                        umma_bf16(d, sdesc_sw128(av + kk * 32), sdesc_sw128(bhi + kk * 32), IDESC, (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < KS / 16; ++kk)
                        umma_bf16(d, sdesc_sw128(av + kk * 32), sdesc_sw128(blo + kk * 32), IDESC, 1u);
                    umma_commit(smem_u32(&bar_empty[sl]));
                    umma_commit(smem_u32(&bar_bempty[sb]));
                }
                if (!ok) break;
                umma_commit(smem_u32(&bar_hfull[b]));
            }
            if (!ok) abort_s = 1;
            umma_commit(smem_u32(&bar_done));
            mbar_wait(smem_u32(&bar_done), 0, a.status);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------------- key (x) key builders
        // thread: key index n = t & 63, tokens 16 * (t >> 6) .. +15, the MP state rows
        // (m' = 0..MP-1, m = MP Q + m') of that n: the Kt row of n is read once, the rows of m
        // are warp-uniform (broadcast).
        const int n = threadIdx.x & 63, kq = threadIdx.x >> 6;
        for (int gs = 0; gs < nstages; ++gs) {
            const int sl = gs % NSLOT, sb = gs & 1;
            if (abort_s || !mbar_wait(smem_u32(&bar_full[sl]), (uint32_t)(gs / NSLOT) & 1, a.status)) {
                abort_s = 1;
                break;
            }
            if (gs >= 2 && !mbar_wait(smem_u32(&bar_bempty[sb]), (uint32_t)((gs >> 1) - 1) & 1, a.status)) {
                abort_s = 1;
                break;
            }
            const uint32_t kt = sbase + sl * SLOT;   // Kt: row x = key_j[x] over the stage's 64 tokens j
            uint32_t xn[8];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2)
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(xn[4 * c2]), "=r"(xn[4 * c2 + 1]), "=r"(xn[4 * c2 + 2]), "=r"(xn[4 * c2 + 3])
                             : "r"(kt + n * 128 + (((2 * kq + c2) ^ (n & 7)) << 4)));
#pragma unroll
            for (int mp = 0; mp < MP; ++mp) {
                const int m = MP * Q + mp, r = mp * 64 + n;
                const uint32_t dhi = sbase + SB + sb * BBUF + r * 128, dlo = dhi + NR * 128;
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int k8 = 2 * kq + c2;
                    uint32_t xm[4], rh[4], rl[4];
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                                 : "=r"(xm[0]), "=r"(xm[1]), "=r"(xm[2]), "=r"(xm[3])
                                 : "r"(kt + m * 128 + ((k8 ^ (m & 7)) << 4)));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 km2 = *reinterpret_cast<const __half2*>(&xm[i]);
                        const __half2 kn2 = *reinterpret_cast<const __half2*>(&xn[4 * c2 + i]);
                        const __half2 hi2 = __hmul2(km2, kn2);
                        const __half2 lo2 = __hfma2(km2, kn2, __hneg2(hi2));
                        rh[i] = *reinterpret_cast<const uint32_t*>(&hi2);
                        rl[i] = *reinterpret_cast<const uint32_t*>(&lo2);
                    }
                    const uint32_t off = (uint32_t)((k8 ^ (r & 7)) << 4);
                    st_shared_v4(dhi + off, rh[0], rh[1], rh[2], rh[3]);
                    st_shared_v4(dlo + off, rl[0], rl[1], rl[2], rl[3]);
                }
            }
            fence_proxy_async();
            mbar_arrive(smem_u32(&bar_bfull[sb]));
            mbar_arrive(smem_u32(&bar_empty[sl]));
        }
    } else {
        // ---------------------------------------------------------------- running state (epilogue)
        // warps 8, 12: value columns 0-31; 9, 13: columns 32-63; 10, 14: the normaliser column
        // (tensor-memory lane 64 = lane 0 of the warp); e = which half of the NR state rows,
        // NK groups of 32 rows each.
        const int q = warp & 3, e = warp >= 12 ? 1 : 0;
        const bool zwarp = q == 2;
        // units of the running state (see the header): forward value columns ks^2 vs, forward
        // normaliser ks^2; the reverse normaliser column is brought to ks^2 vs by vs / zs
        const float ks = pow2_scale(a.amax[bh * 4]), vs = pow2_scale(a.amax[bh * 4 + 1]);
        const float unit = rev ? 1.f : (zwarp ? ks * ks : ks * ks * vs);
        const float zfix = (rev && zwarp) ? vs / pow2_scale(a.amax[bh * 4 + 2]) : 1.f;
        const int col = 32 * q + lane;               // value column (q < 2)
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        constexpr int NK = NR / 64;
        const long row0 = (long)Q * NR + (NR / 2) * e;   // first state row of this warp's NR / 2
        float gam = 1.f;   // reverse: running max of zmax over the chunks walked so far
        // the 32 values of rows row0 + 32k + i (i = 0..31) held by lane `src` move to lane i
        auto gather_lane = [&](const float* v, int src) {
            float out = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float t = __shfl_sync(0xffffffffu, v[i], src);
                if (lane == i) out = t;
            }
            return out;
        };
        // exports 32 rows (row0 + 32k ..) of the state held as v[i] (divided by gam)
        auto export_rows = [&](int slot, int k, const float* v) {
            const float inv = 1.f / gam;
            const long rbase = row0 + 32 * k;
            if (zwarp) {
                const float zv = gather_lane(v, 0);
                a.zx[(bh * NC + slot) * 4096 + rbase + lane] = zv;
                return;
            }
            __half* hi = a.Sx + ((bh * NC + slot) * 2) * (4096L * 64) + rbase * 64 + col;
            __half* lo = hi + 4096L * 64;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float x = v[i] * inv;
                const __half h = __float2half_rn(x);
                hi[i * 64] = h;
                lo[i * 64] = __float2half_rn(x - __half2float(h));
            }
        };
        // the initial state (forward: S0 / z0 or zero; reverse: zero), rows row0 + 32k + i
        auto initial_rows = [&](int k, float* v) {
            const long rbase = row0 + 32 * k;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
            if (rev) return;
            if (zwarp) {
                if (a.z0) {
                    const float zl = a.z0[bh * 4096 + rbase + lane] * unit;
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __shfl_sync(0xffffffffu, zl, i);
                }
            } else if (a.S0) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = a.S0[(bh * 4096 + rbase + i) * 64 + col] * unit;
            }
        };
        {
            const int slot0 = rev ? NC - 1 : 0;
            if (a.sscale && Q == 0 && warp == 8 && lane == 0) a.sscale[bh * NC + slot0] = 1.f;
            for (int k = 0; k < NK; ++k) {
                float v[32];
                initial_rows(k, v);
                export_rows(slot0, k, v);
            }
        }
        bool ok = true;
        for (int it = 0; it < nchunks && ok; ++it) {
            const int c = chunk_of(it), b = it & 1;
            const float dec = __expf(a.g[bh * NC + c]);
            const float zm = rev ? a.zmax[bh * NC + c] : 1.f;
            const float scl = zm * zfix;
            if (abort_s || !(ok = mbar_wait(smem_u32(&bar_hfull[b]), (uint32_t)(it >> 1) & 1, a.status))) break;
            tc_fence_after();
            // pass 1: S_c = dec S_{c-1} + scl H^T_c over the buffer of chunk c
            for (int k = 0; k < NK; ++k) {
                const uint32_t cur = tmem + lane_base + (uint32_t)b * NR + (NR / 2) * e + 32 * k;
                float h[32], p[32];
                tmem_ld32(cur, h);
                if (it > 0) tmem_ld32(tmem + lane_base + (uint32_t)(1 - b) * NR + (NR / 2) * e + 32 * k, p);
                else initial_rows(k, p);
#pragma unroll
                for (int i = 0; i < 32; ++i) h[i] = fmaf(dec, p[i], scl * h[i]);
                tmem_st32(cur, h);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_dfree[(it + 1) & 1]));   // the previous buffer has been read
            if (rev) gam = it == 0 ? zm : fmaxf(gam, zm);
            // pass 2: export the state of slot c + 1 (forward) / c - 1 (reverse)
            const int slot = rev ? c - 1 : c + 1;
            if (slot >= 0 && slot < NC) {
                if (a.sscale && Q == 0 && warp == 8 && lane == 0) a.sscale[bh * NC + slot] = gam;
                for (int k = 0; k < NK; ++k) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + (uint32_t)b * NR + (NR / 2) * e + 32 * k, v);
                    export_rows(slot, k, v);
                }
            }
            if (!rev && it == nchunks - 1 && (a.S_final || a.z_final)) {
                for (int k = 0; k < NK; ++k) {
                    float v[32];
                    tmem_ld32(tmem + lane_base + (uint32_t)b * NR + (NR / 2) * e + 32 * k, v);
                    const long rbase = row0 + 32 * k;
                    const float inv_unit = 1.f / unit;   // exact: a power of two
                    if (zwarp) {
                        const float zv = gather_lane(v, 0);
                        if (a.z_final) a.z_final[bh * 4096 + rbase + lane] = zv * inv_unit;
                    } else if (a.S_final) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) a.S_final[(bh * 4096 + rbase + i) * 64 + col] = v[i] * inv_unit;
                    }
                }
            }
        }
        if (!ok) abort_s = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TCOLS);
}

cudaError_t tc_state_scan(const Problem& p, const ScanIO& io, cudaStream_t s) {
    CUtensorMap tops;
    const uint64_t BH = (uint64_t)p.BH(), Tp = (uint64_t)p.Tp();
    const uint64_t dims[3] = {64, (uint64_t)TC_OPS_ROWS, BH * (Tp / KS)};
    const uint64_t strides[2] = {128, (uint64_t)TC_OPS_ROWS * 128};
    const uint32_t box[3] = {64, (uint32_t)TC_OPS_ROWS, 1};
    if (!make_tmap_f16_nd(&tops, io.ops, 3, dims, strides, box)) return cudaErrorInvalidValue;
    int* status = tc_status_ptr();
    if (!status) return cudaErrorInvalidValue;
    if (!io.amax) return cudaErrorInvalidValue;
    Args a{io.g, io.zmax, io.S0, io.z0, (__half*)io.Sx, io.zx, io.sscale, io.S_final, io.z_final, io.amax, status,
           p.T, p.NC, (int)p.Tp(), io.rev ? 1 : 0};
    constexpr int NR = NR_ROWS, SMEM = smem_bytes(NR);
    cudaError_t e = cudaFuncSetAttribute(tc_state_scan_kernel<NR>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(4096 / NR, (unsigned)p.BH());
    tc_state_scan_kernel<NR><<<grid, THREADS, SMEM, s>>>(tops, a);
    return cudaGetLastError();
}

}  // namespace tm2
