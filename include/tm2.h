/*
 * tm2.h -- C ABI of libtm2.so, the B300 (sm_103a) 2Mamba second-order sequence mixer.
 *
 * Method: "2Mamba2Furious: Linear in Complexity, Competitive in Accuracy"
 * (Mongaras & Larson, arXiv 2602.17363).  Per batch b and head h, with tokens
 * t = 0..T-1, q_t, k_t in R^d, v_t in R^dv and the A-mask input a_t in R:
 *
 *   l_t     = -softplus(a_t)                cumA_t = sum_{u <= t} l_u      (Sec. 3, Sec. 4)
 *   w_ij    = exp(cumA_i - cumA_j) (q_i . k_j)^2              for j <= i   (Sec. 5)
 *   N_i     = sum_{j <= i} w_ij v_j         Z_i = sum_{j <= i} w_ij
 *   o_i     = N_i / Z_i   with TM2_NORMALIZE ("softmax normalisation", Sec. 5), else N_i
 *
 * Equivalent recurrent form with the second-order state of size (d^2, dv)
 * (Sec. 2, "Softmax as a Recurrent Neural Network"; App. A):
 *   S_t = exp(l_t) S_{t-1} + (k_t (x) k_t) v_t^T,   z_t = exp(l_t) z_{t-1} + k_t (x) k_t
 *   N_t = (q_t (x) q_t)^T S_t,                      Z_t = (q_t (x) q_t)^T z_t
 *
 * 2Mamba-E (Sec. 6): o_i = sum_{j <= i} softmax_j(scale q_i . k_j + cumA_i - cumA_j) v_j.
 *
 * The boundary is the attention kernel of App. C: inputs are the post-projection,
 * post-convolution q, k, v and a; outputs are the post-attention outputs.
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise, owned by the caller,
 *    16-byte aligned (TM2_ERR_ALIGNMENT otherwise), and tensors are dense row-major:
 *    q, k, dq, dk: (B,H,T,d); v, o, dO, dv: (B,H,T,dv); a, Z, lse, da: (B,H,T).
 *  - dtype (tm2_dtype) is the element type of the inputs q, k, v and dO.  The gradients dq,
 *    dk, dv are fp32, or in dtype with TM2_GRADS_INPUT_DTYPE.  The A-mask input a, da, Z, lse
 *    and every state are fp32, and so is the forward output o: the backward takes o and forms
 *    D_i = dO_i . o_i from it, and rounding o to bf16 alone moves the normalised mixer's dq and
 *    dk by about 4e-2 of their RMS (the fp64 oracle's backward evaluated at a bf16-rounded o,
 *    B=1 H=4 T=2048 d=64), beyond the bf16 parity bar.  The arithmetic accumulates in fp32.
 *  - State layout: S is (B,H,d*d,dv) with row r = m*d + n (key feature indices m, n);
 *    z is (B,H,d*d).  The same layout serves forward (initial/final state) and decode.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *    Calls are asynchronous and never synchronise the host.  The tensor-core forward and
 *    backward also run their state walks on two high-priority streams of the library's own
 *    (created once per device), forked from `stream` and joined back into it with events
 *    (made once per host thread and device), so the call's work is ordered with respect to
 *    `stream` as if it all ran there.  The calls can be captured into a CUDA graph; a call
 *    captured before its thread has made a non-captured one runs on `stream` alone.
 *  - Argument errors are reported before anything is launched.  A launch failure
 *    returns TM2_ERR_CUDA.  Kernels whose waits are bounded record TM2_ERR_TIMEOUT in
 *    a per-device status word that tm2_poll_status() returns after the stream drains.
 *  - The library allocates no device memory: scratch comes from the caller's
 *    workspace (`ws`, `ws_bytes` >= the matching *_workspace() size, 256-byte aligned).
 *  - Supported: d = dv in {16, 32, 64}; any T >= 0 (a ragged last chunk is handled);
 *    chunk in {0 (library choice), 64, 256}.  chunk 0 picks 256 (the tensor-core path)
 *    for bf16 inputs with d = dv = 64 and 64 otherwise; 256 is accepted only where the
 *    tensor-core path applies (bf16, d = dv = 64).  Other values return
 *    TM2_ERR_UNSUPPORTED; 128 and 512 among them: the tensor-core kernels are built around
 *    256-token chunks (four 64-token stages per chunk in the state walk, two 128-token
 *    readout tiles per chunk state), and the other end of the range, one chunk of T
 *    tokens, is the quadratic form (tm2q_forward).
 *    B*H <= 65535 for the sequence entry points.
 */
#ifndef TM2_H
#define TM2_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TM2_OK = 0,
    TM2_ERR_INVALID_ARG = -1,   /* null pointer, negative size, inconsistent arguments */
    TM2_ERR_UNSUPPORTED = -2,   /* valid but not implemented (d, dv, chunk, dtype)      */
    TM2_ERR_ALIGNMENT = -3,     /* a pointer is not 16-byte aligned (workspace: 256)     */
    TM2_ERR_WORKSPACE = -4,     /* ws_bytes smaller than the *_workspace() size          */
    TM2_ERR_CUDA = -5,          /* a CUDA launch or runtime call failed                  */
    TM2_ERR_TIMEOUT = -6,       /* a bounded device wait expired (see tm2_poll_status)   */
    TM2_ERR_BOUNDS = -7         /* bounds-checked build only: a device index check failed */
} tm2_status;

typedef enum { TM2_F32 = 0, TM2_BF16 = 1 } tm2_dtype;

/* o = N / Z (the paper's "softmax normalisation", Sec. 5).  Without it o = N. */
#define TM2_NORMALIZE 1u
/* tm2_backward only: `ws` starts with the workspace of a tm2_forward call made with the same
 * q, k, v, a, shapes, chunk, dtype and TM2_NORMALIZE setting and no initial state, and not
 * modified since.  The backward then reads the decay sums and chunk states that forward
 * left there instead of recomputing them.  (Allocate max(tm2_forward_workspace,
 * tm2_backward_workspace) bytes and pass the same buffer to both calls.) */
#define TM2_REUSE_STATES 2u
/* tm2_step / tm2_step_conv: S and z are kept symmetric-packed, (N,H,d(d+1)/2,dv) and
 * (N,H,d(d+1)/2): only the rows (m, n) with m <= n, row index m*d - m(m-1)/2 + (n - m).
 * k (x) k and q (x) q are symmetric, so the readout (q (x) q)^T S sees only the symmetric part
 * of S and every update adds a symmetric term: with the off-diagonal rows weighted twice the
 * outputs are exactly those of the full state, for any initial state (tm2_state_pack keeps its
 * symmetric part), and a step moves about half the bytes ("2Mamba2Furious", Sec. 5.1: memory
 * of the squared state; Sec. 7: hidden-state size). */
#define TM2_PACKED_STATE 4u
/* Backward entry points: dq, dk, dv are written in dtype (bf16 for bf16 inputs), each the
 * round-to-nearest of the fp32 value written without the flag.  (Rounding alone can move a
 * heavy-tailed gradient tensor's max|err| / RMS past 2e-2, so the unrounded fp32 form is the
 * default.) */
#define TM2_GRADS_INPUT_DTYPE 8u

/* Library version (major*10000 + minor*100 + patch). */
int tm2_version(void);

/* Human-readable name of a tm2_status value.  Never NULL. */
const char* tm2_status_string(int status);

/* Bytes of device workspace tm2_forward needs for these arguments (0 if none).
 * Returns 0 as well for arguments tm2_forward would reject. */
size_t tm2_forward_workspace(int B, int H, int T, int d, int dv, int chunk, int dtype,
                             unsigned flags);

/*
 * 2Mamba forward (Sec. 5), chunked: decay running sums, per-chunk second-order
 * states, state passing across chunks, intra-chunk squared masked scores and the
 * inter-chunk readout of the state entering each chunk.
 *   q,k,v,a  inputs (see layout above).
 *   S0, z0   optional initial state (state before token 0), fp32; NULL = zero.
 *   o        output (B,H,T,dv) fp32.
 *   Z        optional output (B,H,T) fp32, the normaliser Z_i (tm2_backward needs it).
 *   S_final, z_final  optional outputs, the state after token T-1 (fp32).
 * Returns TM2_OK or an error status.
 */
int tm2_forward(const void* q, const void* k, const void* v, const float* a,
                const float* S0, const float* z0,
                void* o, float* Z, float* S_final, float* z_final,
                int B, int H, int T, int d, int dv, int chunk, int dtype, unsigned flags,
                void* ws, size_t ws_bytes, void* stream);

size_t tm2_backward_workspace(int B, int H, int T, int d, int dv, int chunk, int dtype,
                              unsigned flags);

/*
 * 2Mamba backward (App. C, C.1): gradients of sum(dO * o) w.r.t. q, k, v and the raw
 * A-mask input a, for a forward with no initial state.  o and Z are the forward's
 * outputs for the same inputs and flags (Z may be NULL when TM2_NORMALIZE is off).
 * o is the fp32 output of tm2_forward; dq, dk, dv fp32 (in dtype with TM2_GRADS_INPUT_DTYPE), da
 * fp32.  flags: TM2_NORMALIZE as in the forward, optionally TM2_REUSE_STATES and
 * TM2_GRADS_INPUT_DTYPE.  The A-mask gradient is the row-axis sum minus the
 * column-axis sum of w_ij * dL/dw_ij, accumulated from the end of the sequence and
 * multiplied by d(-softplus(a))/da = -sigmoid(a).
 */
int tm2_backward(const void* q, const void* k, const void* v, const float* a,
                 const void* o, const float* Z, const void* dO,
                 void* dq, void* dk, void* dv, float* da,
                 int B, int H, int T, int d, int dv_dim, int chunk, int dtype, unsigned flags,
                 void* ws, size_t ws_bytes, void* stream);

/*
 * One recurrent decode step (App. A) for N sequences x H heads, one token each:
 *   S <- exp(l) S + (k (x) k) v^T,  z <- exp(l) z + k (x) k,  y = (q (x) q)^T S,  zeta = (q (x) q)^T z
 * q, k: (N,H,d); v: (N,H,dv) in dtype; a: (N,H) fp32.
 * S: (N,H,d*d,dv) fp32, updated in place.  z: (N,H,d*d) fp32 in place, or NULL
 * (then no normaliser is tracked and TM2_NORMALIZE is rejected).
 * o: (N,H,dv) fp32, = y / zeta with TM2_NORMALIZE, else y.  Z: (N,H) fp32 zeta, or NULL.
 * No workspace.  The step is bound by HBM bandwidth: it streams S once in and once out.
 */
int tm2_step(const void* q, const void* k, const void* v, const float* a,
             float* S, float* z, void* o, float* Z,
             int N, int H, int d, int dv, int dtype, unsigned flags, void* stream);

/*
 * Quadratic (C = T, "flash") form of the mixer, order 2 (2Mamba) or 1 (the first-order mixer
 * of Mamba-2S with the same softplus A-mask).  "2Mamba2Furious", Sec. 1-2: the quadratic form
 * costs O(T^2 d) but, at d = dv = 64, fewer flops than the chunked form while
 * T < 4 d^2 dv / (d + dv) = 8192; Sec. 4 (Mamba-2S: the score q.k itself), Sec. 5 (2Mamba:
 * its square under the A-mask):
 *   w_ij = (q_i . k_j)^order exp(cumA_i - cumA_j)  (j <= i),  N_i = sum_j w_ij v_j,  Z_i = sum_j w_ij,
 *   o = N / Z with TM2_NORMALIZE, else N.
 * With order 2 the result is tm2_forward's (no initial state).  The first-order weights carry
 * the sign of q.k, so its Z can vanish; TM2_NORMALIZE is accepted for it but rarely wanted.
 * Layouts, dtypes and alignment as for tm2_forward; o (B,H,T,dv) and Z (B,H,T, optional) fp32.
 * bf16 inputs with d = dv = 64 run on the tensor cores (the 2Mamba-E kernels' skeleton with
 * the weights above), everything else on CUDA cores in fp32 arithmetic.  Any T >= 0.
 * flags: TM2_NORMALIZE (and, for the backward, TM2_GRADS_INPUT_DTYPE).
 */
size_t tm2q_forward_workspace(int B, int H, int T, int d, int dv, int order, int dtype, unsigned flags);
int tm2q_forward(const void* q, const void* k, const void* v, const float* a, void* o, float* Z,
                 int B, int H, int T, int d, int dv, int order, int dtype, unsigned flags,
                 void* ws, size_t ws_bytes, void* stream);

/*
 * Backward of tm2q_forward (App. C, C.1): gradients of sum(dO * o) w.r.t. q, k, v and the raw
 * A-mask input a, given the forward's o and Z (both may be NULL without TM2_NORMALIZE).
 * dq, dk, dv fp32 (in dtype with TM2_GRADS_INPUT_DTYPE), da fp32; da as for tm2_backward (row-axis minus column-axis sums of
 * w_ij dL/dw_ij, accumulated from the end, times -sigmoid(a)).
 */
size_t tm2q_backward_workspace(int B, int H, int T, int d, int dv, int order, int dtype, unsigned flags);
int tm2q_backward(const void* q, const void* k, const void* v, const float* a, const void* o,
                  const float* Z, const void* dO, void* dq, void* dk, void* dv, float* da,
                  int B, int H, int T, int d, int dv_dim, int order, int dtype, unsigned flags,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * tm2_step with the size-2 input convolution of Mamba-2S applied to q, k and v first
 * ("2Mamba2Furious", Sec. 3-4: window 2, no activation; App. A: inference caches the previous
 * window - 1 = 1 raw query, key and value).  Per tensor x in (q, k, v), channel c of head h:
 *   x'_t[c] = w[h][c][0] x_t[c] + w[h][c][1] x_{t-1}[c] (+ b[h][c]),
 * with x_{t-1} read from the cache (N,H,d) in dtype (zero before the first token) and x_t
 * written back to it.  wq, wk, wv: (H,d,2) fp32; bq, bk, bv: (H,d) fp32 or NULL; cq, ck, cv:
 * the caches, updated in place.  The convolved q', k', v' are fp32 (never rounded to dtype).
 * Everything else as tm2_step (flags TM2_NORMALIZE, TM2_PACKED_STATE).
 */
int tm2_step_conv(const void* q, const void* k, const void* v, const float* a,
                  const float* wq, const float* wk, const float* wv,
                  const float* bq, const float* bk, const float* bv,
                  void* cq, void* ck, void* cv,
                  float* S, float* z, void* o, float* Z,
                  int N, int H, int d, int dv, int dtype, unsigned flags, void* stream);

/*
 * Symmetric packing of NH full states S (NH,d*d,dv) / z (NH,d*d) into (NH,d(d+1)/2,dv) /
 * (NH,d(d+1)/2) (the layout of TM2_PACKED_STATE): packed row (m, n), m <= n, holds
 * (S[(m,n)] + S[(n,m)]) / 2.  tm2_state_unpack writes that symmetric full state back.
 * z / z_packed may both be NULL.  d = dv in {16, 32, 64}.
 */
int tm2_state_pack(const float* S, const float* z, float* S_packed, float* z_packed, int NH, int d, int dv,
                   void* stream);
int tm2_state_unpack(const float* S_packed, const float* z_packed, float* S, float* z, int NH, int d, int dv,
                     void* stream);

/*
 * Size-2 causal input convolution over a sequence (the training-side counterpart of
 * tm2_step_conv): x (B,H,T,C) in dtype, w (H,C,2) fp32, b (H,C) fp32 or NULL, x_prev (B,H,C)
 * in dtype or NULL (the token before t = 0; zero if NULL), y (B,H,T,C) in dtype:
 *   y_t = w[..,0] x_t + w[..,1] x_{t-1} (+ b).
 * Backward: dx (B,H,T,C), dx_prev (B,H,C, or NULL), dw (H,C,2), db (H,C, or NULL), all fp32,
 * from dy (B,H,T,C) in dtype.  C in {16, 32, 64}.  The weight gradients are reduced in
 * double-float pairs by a cluster of 8 blocks per head (deterministic, no scratch).
 */
int tm2_conv2_forward(const void* x, const float* w, const float* b, const void* x_prev, void* y,
                      int B, int H, int T, int C, int dtype, void* stream);
int tm2_conv2_backward(const void* x, const float* w, const void* x_prev, const void* dy, float* dx,
                       float* dx_prev, float* dw, float* db, int B, int H, int T, int C, int dtype,
                       void* stream);

size_t tm2e_forward_workspace(int B, int H, int T, int d, int dv, int dtype);

/*
 * 2Mamba-E forward (Sec. 6): causal softmax attention with the additive A-mask
 * cumA_i - cumA_j and logit scale `scale` (1/sqrt(d) in the paper's setting),
 * evaluated blockwise with an online running maximum.
 * o: (B,H,T,dv) fp32.  lse: (B,H,T) fp32 log-sum-exp of each row (needed by backward).
 */
int tm2e_forward(const void* q, const void* k, const void* v, const float* a,
                 void* o, float* lse,
                 int B, int H, int T, int d, int dv, float scale, int dtype,
                 void* ws, size_t ws_bytes, void* stream);

/*
 * tm2e_forward_noalloc -- the paper has no counterpart to this entry point; it exists
 * for callers that cannot allocate device memory (for example a plugin hosted by an
 * inference engine that owns and pre-plans all device memory, or a latency-critical
 * loop that must not risk cudaMalloc's implicit synchronisation).
 * It runs tm2e_forward's own checks and kernels (the tensor-core kernel for bf16 inputs with
 * d = dv = 64, the CUDA-core kernel otherwise) with the same arguments minus the workspace,
 * so its results are tm2e_forward's; its scratch is a fixed array of
 * TM2E_NOALLOC_SCRATCH_BYTES compiled into the library, held by every GPU that loads the
 * library until the process exits.
 *  - Scratch need is about 12 * B*H*T bytes (three fp32 values per token-head, plus chunk
 *    totals and padding to whole chunks); larger problems return TM2_ERR_WORKSPACE before
 *    anything is launched (B*H*T up to roughly 1.3 million token-heads fits).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *    with that device current); make that first call before any stream capture.
 *  - No cudaMalloc, cudaFree or other allocating routine is called.
 *  - All calls on a device share the array and every call overwrites what it reads, so
 *    nothing needs clearing; calls that overlap on the GPU race on it and must be
 *    serialised by the caller.
 */
#define TM2E_NOALLOC_SCRATCH_BYTES (16u << 20)
int tm2e_forward_noalloc(const void* q, const void* k, const void* v, const float* a,
                         void* o, float* lse,
                         int B, int H, int T, int d, int dv, float scale, int dtype, void* stream);

size_t tm2e_backward_workspace(int B, int H, int T, int d, int dv, int dtype);

/*
 * 2Mamba-E backward: gradients of sum(dO * o) w.r.t. q, k, v and a, given the
 * forward's o (fp32) and lse.  dq, dk, dv fp32 (in dtype with TM2_GRADS_INPUT_DTYPE, the only
 * flag), da fp32.
 */
int tm2e_backward(const void* q, const void* k, const void* v, const float* a,
                  const void* o, const float* lse, const void* dO,
                  void* dq, void* dk, void* dv, float* da,
                  int B, int H, int T, int d, int dv_dim, float scale, int dtype, unsigned flags,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * 2Mamba-E decoding over a key/value cache (Sec. 6; Sec. 1: unlike 2Mamba it needs a KV cache;
 * Sec. 2: that cache is its recurrent state, 2 N dh elements per head).  One token per
 * (sequence, head) at position `pos` (the same for the whole batch, 0 <= pos < L):
 *   cumA_pos = cumA_{pos-1} - softplus(a),   o = sum_{j <= pos} softmax_j(scale q . k_j + cumA_pos - cumA_j) v_j,
 * and k, v, cumA_pos appended to the caches.  q, k: (N,H,d); v: (N,H,dv) in dtype; a: (N,H).
 * K_cache (N,H,L,d), V_cache (N,H,L,dv) in dtype; cum_cache (N,H,L,2) fp32, the running sums
 * of -softplus(a) as hi + lo (rows < pos written by earlier steps or tm2e_fill_cache).
 * o (N,H,dv) fp32; lse (N,H) fp32 or NULL.  Workspace: tm2e_step_workspace (used from
 * pos >= 512, where the keys are split over several blocks).  The step reads the cache once:
 * it is bound by HBM bandwidth.
 */
size_t tm2e_step_workspace(int N, int H, int L, int d, int dv, int dtype);
int tm2e_step(const void* q, const void* k, const void* v, const float* a,
              void* K_cache, void* V_cache, float* cum_cache, int pos, int L,
              void* o, float* lse, int N, int H, int d, int dv, float scale, int dtype,
              void* ws, size_t ws_bytes, void* stream);
/*
 * Fills the caches with a prefill of T <= L tokens (k (B,H,T,d), v (B,H,T,dv), a (B,H,T)):
 * rows 0..T-1 of K_cache, V_cache and the running sums in cum_cache, so that decoding goes on
 * at pos = T.  Workspace: tm2e_fill_cache_workspace.
 */
size_t tm2e_fill_cache_workspace(int B, int H, int T, int d, int dv, int dtype);
int tm2e_fill_cache(const void* k, const void* v, const float* a, void* K_cache, void* V_cache,
                    float* cum_cache, int B, int H, int T, int L, int d, int dv, int dtype,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * Device status word of the current device: returns TM2_OK, or TM2_ERR_TIMEOUT if a
 * kernel's bounded wait expired since the last poll (TM2_ERR_BOUNDS in the bounds-checked
 * build if an index check failed), and clears it.  Synchronises with the device (call it
 * after the stream of interest has drained).
 *
 * Bounds-checked build (libtm2_debug.so, compiled with -DTM2_DEBUG): the tensor-core kernels
 * check the shared-memory, tensor-memory and global indices they compute before using them;
 * a failed check records TM2_ERR_BOUNDS in the status word and the access is skipped (no trap,
 * no assert).  Every call then synchronises its stream after each launch and returns a
 * non-zero status word, so a failure is reported by the call that caused it.  Calls of this
 * build cannot be captured into a CUDA graph.
 */
int tm2_poll_status(void);

/* Text of the CUDA error behind the calling thread's last TM2_ERR_CUDA ("no CUDA error" if
 * none).  Never NULL. */
const char* tm2_last_cuda_error(void);

/*
 * Self-test of the tensor-core building blocks (diagnostic; not part of the method).
 * D (128 x N, fp32) = A (128 x K, bf16, row-major) * B^T through tcgen05.mma (kind::f16)
 * into tensor memory and tcgen05.ld, i.e. the operand and accumulator conventions every
 * tensor-core kernel of the library relies on.  N in {16, 64, 80, 128, 256}; K a multiple
 * of 64, <= 512 (<= 256 with an MN-major B).  Operand forms by mode:
 *   0: A and B (N x K, row-major) loaded by TMA with 128-byte swizzle (K-major);
 *   1: A written by the threads into shared memory in the swizzled layout, B as in 0;
 *   2: one thread waits on a barrier that is never signalled, so the bounded wait expires
 *      after wait_ns nanoseconds, TM2_ERR_TIMEOUT is recorded in the status word
 *      (tm2_poll_status) and the kernel exits cleanly without touching D;
 *   3: A written by the threads into tensor memory (tcgen05.st), B as in 0;
 *   4: A as in 0, B given transposed (K x N, row-major) and consumed MN-major;
 *   5: A in tensor memory as in 3, B MN-major as in 4.
 */
int tm2_selftest_umma(const void* A, const void* B, float* D, int N, int K, int mode,
                      unsigned long long wait_ns, void* stream);

/*
 * Launch tracing (for measurement; off by default).  While enabled, every kernel an
 * entry point launches is bracketed by two CUDA events recorded on that launch's
 * stream, so per-kernel device time can be read back without a profiler.  Not
 * thread-safe: enable, call, read and disable from one host thread.
 *   tm2_trace_enable(1) clears the record list and starts recording; (0) stops.
 *   tm2_trace_count() is the number of recorded launches.
 *   tm2_trace_read(i, name, len, &ms) waits for launch i to finish and returns its
 *   kernel name (truncated to len-1 chars) and device time in milliseconds.
 */
int tm2_trace_enable(int on);
int tm2_trace_count(void);
int tm2_trace_read(int i, char* name, int name_len, float* ms);

#ifdef __cplusplus
}
#endif

#endif /* TM2_H */
