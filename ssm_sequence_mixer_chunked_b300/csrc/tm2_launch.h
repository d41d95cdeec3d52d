// tm2_launch.h -- host-side launchers of the libtm2 kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace tm2 {

// Scalar problem description shared by the launchers.
struct Problem {
    int B, H, T, d, dv, C;   // C: chunk length
    int NC;                  // number of chunks = ceil(T / C)
    int dtype;               // 0 fp32, 1 bf16
    bool normalize;
    bool tc;                 // bf16 tensor-core path (d = dv = 64, C = TC_CHUNK)
    bool lowp_grads = false; // backward: dq, dk, dv in the input type (else fp32)
    long BH() const { return (long)B * H; }
    long Tp() const { return (long)NC * C; }   // padded sequence stride of chunk-local buffers
};

// ---- K1: decay running sums ----------------------------------------------------------
// Aloc[bh][t] (t < Tp): inclusive running sum of -softplus(a) inside each chunk
// (padded positions repeat the last valid value); g[bh][c]: chunk total.
cudaError_t launch_decay(const Problem& p, const float* a, float* Aloc, float* g, cudaStream_t s);
// cum[bh][t] = global inclusive running sum (t < T), from Aloc and g, rounded to fp32; cum_lo
// (optional) its rounding residual, so that cum_i - cum_j = (hi_i - hi_j) + (lo_i - lo_j) keeps
// fp32 precision however large the sums grow.
cudaError_t launch_global_cumsum(const Problem& p, const float* Aloc, const float* g, float* cum, float* cum_lo,
                                 cudaStream_t s);
// da[bh][u] = -sigmoid(a[bh][u]) * sum_{t >= u} (row[bh][t] - col[bh][t]); col may be NULL.
cudaError_t launch_reverse_cumsum_da(const Problem& p, const float* a, const float* row,
                                     const float* col, float* da, cudaStream_t s);

// ---- SIMT (fp32 arithmetic) 2Mamba path ---------------------------------------------
// states: [BH][NC][d][dv+1][d] fp32 -- the state entering each chunk, column dv = z.
cudaError_t simt_state_scan_fwd(const Problem& p, const void* k, const void* v, const float* Aloc,
                                const float* g, const float* S0, const float* z0, float* states,
                                float* S_final, float* z_final, cudaStream_t s);
cudaError_t simt_chunk_out(const Problem& p, const void* q, const void* k, const void* v,
                           const float* Aloc, const float* states, void* o, float* Z,
                           cudaStream_t s);
// dY[bh][t][dv+1] = [dO/Z, -D/Z] (normalised) or [dO, 0]; rowterm[bh][t] = dY_t . Y_t.
cudaError_t launch_dy_prep(const Problem& p, const void* o, const float* Z, const void* dO,
                           float* dY, float* rowterm, cudaStream_t s);
// dstates: [BH][NC][d][dv+1][d], gradient w.r.t. the state at the END of each chunk.
cudaError_t simt_state_scan_bwd(const Problem& p, const void* q, const float* dY, const float* Aloc,
                                const float* g, float* dstates, cudaStream_t s);
cudaError_t simt_bwd_chunk(const Problem& p, const void* q, const void* k, const void* v,
                           const float* Aloc, const float* g, const float* dY,
                           const float* rowterm, const float* states, const float* dstates,
                           void* dq, void* dk, void* dv, float* dcum, cudaStream_t s);

// ---- bf16 tensor-core path (d = dv = 64, chunk TC_CHUNK) ------------------------------
constexpr int TC_CHUNK = 256;
// Block-packed chunk states (the forward walk's export, read by the chunk output and dq): the
// (m, n) index square of the d^2 = 4096 state rows is cut into 16 x 16 blocks and only the 10
// blocks with bm <= bn are kept, block (bm, bn) at index bm * 4 - bm (bm - 1) / 2 + (bn - bm),
// its rows ordered r = 16 (m - 16 bm) + (n - 16 bn).  The state is symmetric in (m, n) up to the
// initial state's antisymmetric part, which no readout sees.  In the forward states an
// off-diagonal block is stored doubled (it stands for (m, n) and (n, m)) and a diagonal block
// as is, so the readouts contract each stored row once:
//   sum_{m,n} x[m] x[n] S[(m,n), :] = sum_{blocks} sum_{(m,n) in block} x[m] x[n] T[(m,n), :].
// The gradient states (no initial state, exactly symmetric) are stored as they are: dk/dv reads
// each off-diagonal block in both orientations (make_tmap_state_packed_rowrun / _tquads).
// Layout [BH][NC][2 planes][TC_PACKED_ROWS][64] fp16; the normaliser states stay full.
constexpr int TC_PACKED_BLOCKS = 10;
constexpr int TC_PACKED_ROWS = TC_PACKED_BLOCKS * 256;
__host__ __device__ constexpr int tc_block_index(int bm, int bn) { return bm * 4 - bm * (bm - 1) / 2 + (bn - bm); }
__host__ __device__ inline void tc_block_of(int idx, int& bm, int& bn) {   // inverse of tc_block_index
    bm = idx < 4 ? 0 : idx < 7 ? 1 : idx < 9 ? 2 : 3;
    bn = bm + (idx - tc_block_index(bm, bm));
}
// Chunk-state scan (tm2_tc_scan.cu).  Forward (rev = false): key = k, val = v, normaliser
// column 1, weight exp(g_c - A_j); slot c = the state entering chunk c (slot 0 = S0/z0 or
// zero); S_final/z_final (optional) = the state after the last token.  Reverse (rev = true):
// key = q, val = dO, normaliser column ucol, weight exp(A_i) zeta_i; slot c = the gradient
// w.r.t. the state at the end of chunk c, scaled per (slot, CTA) by 1/sscale.
// Sx: [BH][NC][2][TC_PACKED_ROWS][64] block-packed fp16 (hi plane, residual plane; forward
// off-diagonal blocks doubled, reverse as is); zx: [BH][NC][4096] fp32 (full layout in both
// walks).
struct ScanIO {
    bool rev;
    const void* ops;       // operand blocks from launch_tc_scan_operands
    const float* g;
    const float* zmax;     // reverse only
    const float* S0;       // forward only, optional
    const float* z0;       // forward only, optional
    void* Sx;
    float* zx;
    float* sscale;         // reverse only: [BH][NC] scale of each exported slot
    float* S_final;        // forward only, optional
    float* z_final;        // forward only, optional
    const unsigned* amax;  // [BH][4] operand maxima of this walk (see launch_tc_scan_operands)
};
cudaError_t tc_state_scan(const Problem& p, const ScanIO& io, cudaStream_t s);

// Operands of the chunk-state scan (tm2_scan.cu): ops [BH][Tp/64][144][64] fp16, one block
// per 64-token stage (one TMA request each): rows 0-63 the key block transposed (row n =
// key_t[n] over the stage's tokens t), rows 64-127 the weighted values transposed (row col =
// w_t val_t[col]), row 128 = w_t zc_t, rows 129-143 zero (rows 64-143 are the walk's N = 80
// operand).  Forward: key = k, val = v,
// w = exp(g_c - A_t), zc = 1.  Reverse: key = q, val = dO, w = exp(A_t) zeta_t / zmax_c,
// zc = ucol_t.
// The key and value operands (and the reverse walk's normaliser row) are multiplied by the
// powers of two pow2_scale(amax[bh][0]), pow2_scale(amax[bh][1]) (and pow2_scale(amax[bh][2])),
// so the walk's states come out multiplied by ks^2 vs (value columns) and ks^2 zs (normaliser).
constexpr int TC_OPS_ROWS = 144;
cudaError_t launch_tc_scan_operands(const Problem& p, bool rev, const void* key, const void* val, const float* Aloc,
                                    const float* g, const float* zeta, const float* ucol, const float* zmax,
                                    const unsigned* amax, void* ops, cudaStream_t s);

// amax[bh][0], amax[bh][1] (fp32 bits) = the largest |x|, |y| of head bh of two bf16 tensors
// (BH,T,64); zero_first clears amax[BH][4] first (otherwise the maxima combine with it).
cudaError_t launch_head_absmax(const Problem& p, const void* x, const void* y, unsigned* amax, bool zero_first,
                               cudaStream_t s);

// Backward preparation: zeta = 1/Z (or 1), ucol = -dO.o (or 0), rowterm = 0 (or dO.o),
// all (BH,T) fp32, and zmax (BH,NC) = per-chunk max of exp(A_i) zeta_i.  Clears amax[BH][4]
// and sets amax[bh][2] to the largest |ucol| of the head (fp32 bits).
cudaError_t launch_tc_dy_prep(const Problem& p, const float* o, const float* Z, const void* dO, const float* Aloc,
                              float* zeta, float* ucol, float* rowterm, float* zmax, unsigned* amax, cudaStream_t s);

// Gradient kernels (tm2_tc_dq.cu, tm2_tc_dkdv.cu).  dq: Sx/zx are the forward scan's states
// (amax_f its operand maxima); dk, dv, dcum: dSx/dzx/sscale the reverse scan's (amax_r).  dq, dk,
// dv (BH,T,64) fp32, or bf16 with p.lowp_grads; dcum fp32.
cudaError_t tc_bwd_dq(const Problem& p, const void* q, const void* k, const void* v, const void* dO, const float* Aloc,
                      const float* zeta, const float* ucol, const void* Sx, const float* zx, const unsigned* amax_f,
                      void* dq, cudaStream_t s);
cudaError_t tc_bwd_dkdv(const Problem& p, const void* q, const void* k, const void* v, const void* dO,
                        const float* Aloc, const float* g, const float* zeta, const float* ucol, const float* rowterm,
                        const void* dSx, const float* dzx, const float* sscale, const unsigned* amax_r, void* dk,
                        void* dv, float* dcum, cudaStream_t s);

// Per-chunk output (intra-chunk squared masked scores and the readout of the state
// entering the chunk, slot c of Sx/zx from tc_state_scan, whose operand maxima are amax):
// o (BH,T,64) fp32, Z optional.
cudaError_t tc_chunk_out(const Problem& p, const void* q, const void* k, const void* v, const float* Aloc,
                         const void* Sx, const float* zx, const unsigned* amax, float* o, float* Z, cudaStream_t s);

// ---- decode --------------------------------------------------------------------------
// The size-2 input convolution applied inside the decode step: per tensor x in (q, k, v),
// weights (H, d, 2), optional bias (H, d), cache of the previous raw token (N, H, d) in the
// input dtype, read and then overwritten with the current token.
struct DecodeConv {
    const float* w[3];
    const float* b[3];
    void* cache[3];
};
// packed: S (N,H,d(d+1)/2,dv) and z (N,H,d(d+1)/2) symmetric-packed; conv: optional.
cudaError_t launch_decode_step(int N, int H, int d, int dv, int dtype, bool normalize, bool packed,
                               const DecodeConv* conv, const void* q, const void* k, const void* v,
                               const float* a, float* S, float* z, void* o, float* Z, cudaStream_t s);
// full (nh, d*d, cols) <-> packed (nh, d(d+1)/2, cols): pack takes the symmetric part.
cudaError_t launch_state_pack(const float* full, float* packed, long nh, int d, int cols, bool unpack,
                              cudaStream_t s);

// ---- attention-form kernels: 2Mamba-E and the quadratic (C = T) form of 2Mamba -----
// KIND of the tensor-core and CUDA-core attention-form kernels: 2Mamba-E (softmax of
// scale q.k + cumA_i - cumA_j), the first-order mixer (w = q.k exp(cumA_i - cumA_j)) and
// 2Mamba (w = (q.k)^2 exp(cumA_i - cumA_j)).
enum AttnKind { ATTN_E = 0, ATTN_P1 = 1, ATTN_P2 = 2 };

// Quadratic-form mixer of order 1 or 2 (p.normalize: o = N / Z) on the tensor cores (bf16,
// d = dv = 64) and on CUDA cores (fp32 arithmetic, any supported d): cum / cum_lo as for
// 2Mamba-E; o (BH,T,64 or dv) fp32, Z (BH,T) fp32 always written.
cudaError_t tc_poly_fwd(const Problem& p, int order, const void* q, const void* k, const void* v, const float* cum,
                        const float* cum_lo, float* o, float* Z, cudaStream_t s);
cudaError_t simt_poly_fwd(const Problem& p, int order, const void* q, const void* k, const void* v,
                          const float* cum, const float* cum_lo, void* o, float* Z, cudaStream_t s);
// Backward: zeta = 1/Z (normalised) or 1 and D = dO . o (normalised) or 0 per token (launch_poly_prep);
// rowsum / colsum the two A-mask axis sums of w_ij dw_ij, dw_ij = zeta_i (dO_i . v_j - D_i).
cudaError_t launch_poly_prep(const Problem& p, const float* o, const float* Z, const void* dO, float* D,
                             float* zeta, cudaStream_t s);
cudaError_t tc_poly_bwd(const Problem& p, int order, const void* q, const void* k, const void* v, const float* cum,
                        const float* cum_lo, const float* zeta, const float* D, const void* dO, void* dq, void* dk,
                        void* dv, float* rowsum, float* colsum, cudaStream_t s);
cudaError_t simt_poly_bwd(const Problem& p, int order, const void* q, const void* k, const void* v,
                          const float* cum, const float* cum_lo, const float* zeta, const float* D, const void* dO,
                          void* dq, void* dk, void* dv, float* rowsum, float* colsum, cudaStream_t s);

// ---- 2Mamba-E decoding over a key/value cache (tm2_e_decode.cu) ---------------------
// Kc (NH, L, d), Vc (NH, L, d) in the input dtype and cumc (NH, L, 2) fp32 hi + lo running
// sums; the token at `pos` is appended; part: NH x e_decode_max_splits(L) x (d + 2) floats.
int e_decode_splits(long NH, int pos);   // ranges of the step (at most e_decode_max_splits(L))
int e_decode_max_splits(int L);
cudaError_t launch_e_decode(long NH, int d, int dtype, int pos, int L, float scale, const void* q, const void* k,
                            const void* v, const float* a, void* Kc, void* Vc, float* cumc, float* part, float* o,
                            float* lse, cudaStream_t s);
cudaError_t launch_e_cache_fill(long NH, int T, int L, int d, int dv, int dtype, const void* k, const void* v,
                                const float* cum, const float* cum_lo, void* Kc, void* Vc, float* cumc,
                                cudaStream_t s);

// ---- the size-2 input convolution (tm2_conv.cu) ---------------------------------------
cudaError_t launch_conv2_fwd(long BH, int H, int T, int C, int dtype, const void* x, const float* w, const float* b,
                             const void* x_prev, void* y, cudaStream_t s);
cudaError_t launch_conv2_bwd(int B, int H, int T, int C, int dtype, const void* x, const float* w,
                             const void* x_prev, const void* dy, float* dx, float* dx_prev, float* dw, float* db,
                             cudaStream_t s);

// ---- 2Mamba-E ----------------------------------------------------------------------
// The forward entry points' shared steps (tm2_api.cu): argument checks (fills p; TM2_OK with
// p.BH() == 0 or T == 0 means nothing to do), the scratch size, and the launch sequence over a
// scratch area of that size (the tensor-core kernel for bf16 with d = dv = 64, the CUDA-core
// kernel otherwise), which traces its launches and records a failing launch's CUDA error for
// tm2_last_cuda_error().
int e_forward_check(const void* q, const void* k, const void* v, const float* a, const void* o, const float* lse,
                    int B, int H, int T, int d, int dv, float scale, int dtype, Problem& p);
size_t e_forward_scratch_bytes(const Problem& p);
int e_forward_run(const Problem& p, const void* q, const void* k, const void* v, const float* a, void* o, float* lse,
                  float scale, void* ws, cudaStream_t s);
// Records e as the calling thread's last CUDA error (read back by tm2_last_cuda_error()).
void record_cuda_error(cudaError_t e);
// 2Mamba-E forward on the tensor cores (tm2_tc_e.cu): bf16, d = dv = 64; cum = global running
// sum of -softplus(a) (BH, T); o (BH, T, 64) and lse (BH, T) fp32.
cudaError_t tc_e_fwd(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                     const float* cum_lo, float scale, float* o, float* lse, cudaStream_t s);
cudaError_t simt_e_fwd(const Problem& p, const void* q, const void* k, const void* v,
                       const float* cum, const float* cum_lo, float scale, void* o, float* lse, cudaStream_t s);
// Dvec[bh][t] = dO_t . o_t
cudaError_t launch_rowdot(const Problem& p, const void* o, const void* dO, float* Dvec,
                          cudaStream_t s);
// 2Mamba-E backward on the tensor cores (tm2_tc_e_bwd.cu): bf16, d = dv = 64; dq, dk, dv fp32 (bf16
// with p.lowp_grads);
// rowsum[t] = sum_j dx_tj and colsum[t] = sum_i dx_it (the A-mask gradient's two halves).
cudaError_t tc_e_bwd(const Problem& p, const void* q, const void* k, const void* v, const float* cum,
                     const float* cum_lo, const float* lse, const float* Dvec, const void* dO, float scale, void* dq,
                     void* dk, void* dv, float* rowsum, float* colsum, cudaStream_t s);
cudaError_t simt_e_bwd(const Problem& p, const void* q, const void* k, const void* v,
                       const float* cum, const float* cum_lo, const float* lse, const float* Dvec, const void* dO,
                       float scale, void* dq, void* dk, void* dv, float* rowsum, float* colsum,
                       cudaStream_t s);

}  // namespace tm2
