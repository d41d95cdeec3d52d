// tm2_api.cu -- the C ABI of libtm2.so (declared and documented in include/tm2.h):
// argument validation, workspace carving and the launch sequence of each entry point.
// Every launch goes on the caller's stream; nothing here allocates device memory or
// synchronises the host (except tm2_poll_status, which reads the status word).
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "tm2.h"
#include "tm2_common.cuh"
#include "tm2_launch.h"
#include "tm2_tc.h"

namespace tm2 {

struct Carve {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~(size_t)255;
        return o;
    }
};

static bool aligned16(const void* p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

// Validates the shape arguments shared by the sequence entry points and fills p.
// chunk 64 selects the fp32-arithmetic CUDA-core path, chunk TC_CHUNK the bf16 tensor-core
// path (bf16 inputs, d = dv = 64, and only where `tc_available`); chunk 0 picks the
// tensor-core path whenever it applies.
static int make_problem(int B, int H, int T, int d, int dv, int chunk, int dtype, unsigned flags,
                        Problem& p, bool tc_available = false, unsigned extra_flags = 0) {
    if (B < 0 || H < 0 || T < 0 || d <= 0 || dv <= 0) return TM2_ERR_INVALID_ARG;
    if (dtype != TM2_F32 && dtype != TM2_BF16) return TM2_ERR_UNSUPPORTED;
    if (d != dv || (d != 16 && d != 32 && d != 64)) return TM2_ERR_UNSUPPORTED;
    if (chunk != 0 && chunk != 64 && chunk != TC_CHUNK) return TM2_ERR_UNSUPPORTED;
    if ((long)B * H > 65535) return TM2_ERR_UNSUPPORTED;
    if (flags & ~(TM2_NORMALIZE | extra_flags)) return TM2_ERR_INVALID_ARG;
    const bool tc_ok = tc_available && dtype == TM2_BF16 && d == 64 && dv == 64;
    if (chunk == TC_CHUNK && !tc_ok) return TM2_ERR_UNSUPPORTED;
    p.B = B; p.H = H; p.T = T; p.d = d; p.dv = dv;
    p.tc = tc_ok && chunk != 64;
    p.C = p.tc ? TC_CHUNK : 64;
    p.NC = (T + p.C - 1) / p.C;
    p.dtype = dtype;
    p.normalize = (flags & TM2_NORMALIZE) != 0;
    p.lowp_grads = (flags & TM2_GRADS_INPUT_DTYPE) != 0;
    return TM2_OK;
}

static size_t state_floats(const Problem& p) { return (size_t)p.d * (p.dv + 1) * p.d; }

struct FwdWs { size_t Aloc, g, states, zx, amax, ops, total; };
static FwdWs plan_fwd(const Problem& p) {
    Carve c;
    FwdWs w{};
    w.Aloc = c.take(sizeof(float) * p.BH() * p.Tp());
    w.g = c.take(sizeof(float) * p.BH() * p.NC);
    if (p.tc) {   // fp16 value states [BH][NC][2][4096][64] + fp32 normaliser states [BH][NC][4096]
        w.states = c.take(2 * 2 * (size_t)p.BH() * p.NC * 4096 * 64);
        w.zx = c.take(sizeof(float) * (size_t)p.BH() * p.NC * 4096);
        w.amax = c.take(sizeof(unsigned) * 4 * (size_t)p.BH());   // operand maxima of the scan
        w.ops = c.take(6 * (size_t)p.BH() * p.Tp() * 64);   // scan operand blocks (scratch)
    } else {
        w.states = c.take(sizeof(float) * p.BH() * p.NC * state_floats(p));
    }
    w.total = c.off;
    return w;
}

struct BwdWs {
    size_t Aloc, g, states, dstates, dY, rowterm, dcum, zx, dzx, sscale, zeta, ucol, zmax, amax_f, amax_r, ops, total;
};
static BwdWs plan_bwd(const Problem& p) {
    Carve c;
    BwdWs w{};
    w.Aloc = c.take(sizeof(float) * p.BH() * p.Tp());
    w.g = c.take(sizeof(float) * p.BH() * p.NC);
    if (p.tc) {   // the prefix Aloc, g, states, zx, amax_f is laid out exactly as plan_fwd's
        const size_t planes = 2 * 2 * (size_t)p.BH() * p.NC * 4096 * 64;   // two fp16 planes per slot
        w.states = c.take(planes);
        w.zx = c.take(sizeof(float) * (size_t)p.BH() * p.NC * 4096);
        w.amax_f = c.take(sizeof(unsigned) * 4 * (size_t)p.BH());
        w.dstates = c.take(planes);
        w.dzx = c.take(sizeof(float) * (size_t)p.BH() * p.NC * 4096);
        w.sscale = c.take(sizeof(float) * (size_t)p.BH() * p.NC);
        w.zmax = c.take(sizeof(float) * (size_t)p.BH() * p.NC);
        w.zeta = c.take(sizeof(float) * p.BH() * p.T);
        w.ucol = c.take(sizeof(float) * p.BH() * p.T);
        w.rowterm = c.take(sizeof(float) * p.BH() * p.T);
        w.dcum = c.take(sizeof(float) * p.BH() * p.T);
        w.amax_r = c.take(sizeof(unsigned) * 4 * (size_t)p.BH());
        w.ops = c.take(6 * (size_t)p.BH() * p.Tp() * 64);   // scan operand blocks (scratch)
        w.total = c.off;
        return w;
    }
    w.states = c.take(sizeof(float) * p.BH() * p.NC * state_floats(p));
    w.dstates = c.take(sizeof(float) * p.BH() * p.NC * state_floats(p));
    w.dY = c.take(sizeof(float) * p.BH() * p.T * (p.dv + 1));
    w.rowterm = c.take(sizeof(float) * p.BH() * p.T);
    w.dcum = c.take(sizeof(float) * p.BH() * p.T);
    w.total = c.off;
    return w;
}

// Workspace of the quadratic-form entry points (tm2q_*): decay sums as for 2Mamba-E, a
// normaliser scratch for a NULL Z, and the backward's per-token D, zeta and axis sums.
struct QWs { size_t Aloc, g, cum, cum_lo, Zs, D, zeta, rowsum, colsum, total; };
static QWs plan_q(const Problem& p, bool backward) {
    Carve c;
    QWs w{};
    w.Aloc = c.take(sizeof(float) * p.BH() * p.Tp());
    w.g = c.take(sizeof(float) * p.BH() * p.NC);
    w.cum = c.take(sizeof(float) * p.BH() * p.T);
    w.cum_lo = c.take(sizeof(float) * p.BH() * p.T);
    if (backward) {
        w.D = c.take(sizeof(float) * p.BH() * p.T);
        w.zeta = c.take(sizeof(float) * p.BH() * p.T);
        w.rowsum = c.take(sizeof(float) * p.BH() * p.T);
        w.colsum = c.take(sizeof(float) * p.BH() * p.T);
    } else {
        w.Zs = c.take(sizeof(float) * p.BH() * p.T);
    }
    w.total = c.off;
    return w;
}

struct EWs { size_t Aloc, g, cum, cum_lo, Dvec, rowsum, colsum, total; };
static EWs plan_e(const Problem& p, bool backward) {
    Carve c;
    EWs w{};
    w.Aloc = c.take(sizeof(float) * p.BH() * p.Tp());
    w.g = c.take(sizeof(float) * p.BH() * p.NC);
    w.cum = c.take(sizeof(float) * p.BH() * p.T);
    w.cum_lo = c.take(sizeof(float) * p.BH() * p.T);
    if (backward) {
        w.Dvec = c.take(sizeof(float) * p.BH() * p.T);
        w.rowsum = c.take(sizeof(float) * p.BH() * p.T);
        w.colsum = c.take(sizeof(float) * p.BH() * p.T);
    }
    w.total = c.off;
    return w;
}

static int check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (need == 0) return TM2_OK;
    if (ws == nullptr) return TM2_ERR_WORKSPACE;
    if (ws_bytes < need) return TM2_ERR_WORKSPACE;
    if (((uintptr_t)ws & 255u) != 0) return TM2_ERR_ALIGNMENT;
    return TM2_OK;
}

static thread_local int g_last_cuda_error = 0;   // cudaError_t of the last TM2_ERR_CUDA

#define TM2_CK(call)                                                   \
    do {                                                               \
        cudaError_t e_ = (call);                                       \
        if (e_ != cudaSuccess) {                                       \
            g_last_cuda_error = (int)e_;                               \
            return TM2_ERR_CUDA;                                       \
        }                                                              \
    } while (0)

template <typename T>
static T* at(void* ws, size_t off) { return reinterpret_cast<T*>((char*)ws + off); }

// ---- launch tracing ----------------------------------------------------------------
struct TraceRec {
    const char* name;
    cudaEvent_t beg, end;
};
static bool g_trace_on = false;
static std::vector<TraceRec> g_trace;   // events are created once and reused
static size_t g_trace_n = 0;

struct TraceScope {
    TraceRec* rec = nullptr;
    cudaStream_t s;
    TraceScope(const char* name, cudaStream_t st) : s(st) {
        if (!g_trace_on) return;
        if (g_trace_n == g_trace.size()) {
            TraceRec r{name, nullptr, nullptr};
            if (cudaEventCreate(&r.beg) != cudaSuccess || cudaEventCreate(&r.end) != cudaSuccess) return;
            g_trace.push_back(r);
        }
        rec = &g_trace[g_trace_n++];
        rec->name = name;
        cudaEventRecord(rec->beg, s);
    }
    ~TraceScope() {
        if (rec) cudaEventRecord(rec->end, s);
    }
};

// High-priority streams per device (two) that take the state walks, so that readouts run beside
// them on the caller's stream: the block scheduler prefers the walks' CTAs and the readouts'
// CTAs fill the SMs a walk's last wave leaves idle.  The backward's reverse walk runs beside dq
// (which reads only the forward states); the forward splits the heads into two halves whose
// walks run concurrently, each half's chunk output following its own walk.  The streams are
// shared by the process; the fork / join events belong to the calling host thread (a call
// records and waits them in order, so calls from different threads never share one).  Both are
// made on first use; a call whose stream is being captured into a CUDA graph before they exist
// runs everything on the caller's stream in the same order (creating them is not capturable).
struct Side {
    cudaStream_t st[2];
    cudaEvent_t fork, join[2];
};
static cudaError_t side_resources(cudaStream_t caller, const Side** out) {
    static std::mutex mu;
    static cudaStream_t streams[64][2] = {};
    thread_local Side mine[64] = {};
    *out = nullptr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    Side& x = mine[dev];
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!streams[dev][0] || !x.fork) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            e = cudaStreamIsCapturing(caller, &cs);
            if (e != cudaSuccess) return e;
            if (cs != cudaStreamCaptureStatusNone) return cudaSuccess;   // one stream this time
        }
        if (!streams[dev][0]) {
            int least = 0, greatest = 0;
            e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
            if (e != cudaSuccess) return e;
            for (int i = 0; i < 2; ++i) {
                e = cudaStreamCreateWithPriority(&streams[dev][i], cudaStreamNonBlocking, greatest);
                if (e != cudaSuccess) return e;
            }
        }
        x.st[0] = streams[dev][0];
        x.st[1] = streams[dev][1];
    }
    if (!x.fork) {
        cudaEvent_t ev[3];
        for (int i = 0; i < 3; ++i) {
            e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        x.join[0] = ev[1];
        x.join[1] = ev[2];
        x.fork = ev[0];
    }
    *out = &x;
    return cudaSuccess;
}

#ifdef TM2_DEBUG
// bounds-checked build: every launch is followed by a stream synchronisation and a read of the
// device status word, so the call that broke an index check reports it
#define TM2_RUN(name, call)                          \
    do {                                             \
        {                                            \
            TraceScope ts_(name, s);                 \
            TM2_CK(call);                            \
        }                                            \
        TM2_CK(cudaStreamSynchronize(s));            \
        const int st_ = ::tm2::read_tc_status(true); \
        if (st_ != TM2_OK) return st_;               \
    } while (0)
#else
#define TM2_RUN(name, call)                  \
    do {                                     \
        TraceScope ts_(name, s);             \
        TM2_CK(call);                        \
    } while (0)
#endif

// ---- the 2Mamba-E forward, shared by tm2e_forward and tm2e_forward_noalloc ----------------
int e_forward_check(const void* q, const void* k, const void* v, const float* a, const void* o, const float* lse,
                    int B, int H, int T, int d, int dv, float scale, int dtype, Problem& p) {
    int st = make_problem(B, H, T, d, dv, 0, dtype, 0, p);
    if (st != TM2_OK) return st;
    if (!(scale == scale) || scale == 0.f) return TM2_ERR_INVALID_ARG;
    if (p.BH() == 0 || T == 0) return TM2_OK;
    if (!q || !k || !v || !a || !o || !lse) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, o, lse};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    return TM2_OK;
}

size_t e_forward_scratch_bytes(const Problem& p) { return plan_e(p, false).total; }

int e_forward_run(const Problem& p, const void* q, const void* k, const void* v, const float* a, void* o, float* lse,
                  float scale, void* ws, cudaStream_t s) {
    const EWs w = plan_e(p, false);
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    float* cum = at<float>(ws, w.cum);
    float* cum_lo = at<float>(ws, w.cum_lo);
    TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
    TM2_RUN("global_cumsum", launch_global_cumsum(p, Aloc, g, cum, cum_lo, s));
    if (p.dtype == TM2_BF16 && p.d == 64 && p.dv == 64)
        TM2_RUN("tc_e_fwd", tc_e_fwd(p, q, k, v, cum, cum_lo, scale, (float*)o, lse, s));
    else
        TM2_RUN("e_fwd", simt_e_fwd(p, q, k, v, cum, cum_lo, scale, o, lse, s));
    return TM2_OK;
}

void record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

}  // namespace tm2

using namespace tm2;

extern "C" {

int tm2_version(void) { return 100; }

const char* tm2_status_string(int status) {
    switch (status) {
        case TM2_OK: return "TM2_OK";
        case TM2_ERR_INVALID_ARG: return "TM2_ERR_INVALID_ARG: null pointer, negative size or inconsistent arguments";
        case TM2_ERR_UNSUPPORTED: return "TM2_ERR_UNSUPPORTED: shape, chunk or dtype not implemented";
        case TM2_ERR_ALIGNMENT: return "TM2_ERR_ALIGNMENT: pointer not 16-byte aligned (workspace: 256)";
        case TM2_ERR_WORKSPACE: return "TM2_ERR_WORKSPACE: workspace missing or smaller than required";
        case TM2_ERR_CUDA: return "TM2_ERR_CUDA: a CUDA launch or runtime call failed";
        case TM2_ERR_TIMEOUT: return "TM2_ERR_TIMEOUT: a bounded device wait expired";
        case TM2_ERR_BOUNDS: return "TM2_ERR_BOUNDS: a device index check failed (bounds-checked build)";
        default: return "TM2: unknown status";
    }
}

size_t tm2_forward_workspace(int B, int H, int T, int d, int dv, int chunk, int dtype,
                             unsigned flags) {
    Problem p;
    if (make_problem(B, H, T, d, dv, chunk, dtype, flags, p, true) != TM2_OK) return 0;
    return plan_fwd(p).total;
}

int tm2_forward(const void* q, const void* k, const void* v, const float* a, const float* S0,
                const float* z0, void* o, float* Z, float* S_final, float* z_final, int B, int H,
                int T, int d, int dv, int chunk, int dtype, unsigned flags, void* ws,
                size_t ws_bytes, void* stream) {
    Problem p;
    int st = make_problem(B, H, T, d, dv, chunk, dtype, flags, p, true);
    if (st != TM2_OK) return st;
    const bool work = p.BH() > 0 && T > 0;
    if (work && (!q || !k || !v || !a || !o)) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, S0, z0, o, Z, S_final, z_final};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    if (!work) {
        // no tokens: the final state is the initial state
        const size_t sb = sizeof(float) * p.BH() * d * d * dv, zb = sizeof(float) * p.BH() * d * d;
        if (S_final) TM2_CK(S0 ? cudaMemcpyAsync(S_final, S0, sb, cudaMemcpyDeviceToDevice, s)
                               : cudaMemsetAsync(S_final, 0, sb, s));
        if (z_final) TM2_CK(z0 ? cudaMemcpyAsync(z_final, z0, zb, cudaMemcpyDeviceToDevice, s)
                               : cudaMemsetAsync(z_final, 0, zb, s));
        return TM2_OK;
    }
    const FwdWs w = plan_fwd(p);
    st = check_ws(ws, ws_bytes, w.total);
    if (st != TM2_OK) return st;
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    float* states = at<float>(ws, w.states);
    TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
    if (p.tc) {
        float* zx = at<float>(ws, w.zx);
        unsigned* amax = at<unsigned>(ws, w.amax);
        void* ops = at<void>(ws, w.ops);
        TM2_RUN("head_absmax", launch_head_absmax(p, k, v, amax, true, s));
        TM2_RUN("tc_scan_operands",
                launch_tc_scan_operands(p, false, k, v, Aloc, g, nullptr, nullptr, nullptr, amax, ops, s));
        // Every walk CTA takes about the same time, so the last of its waves leaves most SMs
        // idle.  The heads are split into two halves walked concurrently on the two side
        // streams; the first half's chunk output (on the caller's stream) starts as soon as its
        // walk is done and fills the SMs the second half's walk leaves idle.
        const Side* sd = nullptr;
        TM2_CK(side_resources(s, &sd));
        const long BH = p.BH();
        const int parts = sd ? (BH >= 2 ? 2 : 1) : 1;
        const size_t T = (size_t)p.T, Tp = (size_t)p.Tp(), NC = (size_t)p.NC;
        if (sd) TM2_CK(cudaEventRecord(sd->fork, s));
        Problem pp[2];
        ScanIO io[2];
        for (int i = 0; i < parts; ++i) {
            const long lo = BH * i / parts, hi = BH * (i + 1) / parts;
            pp[i] = p;
            pp[i].B = 1;
            pp[i].H = (int)(hi - lo);
            io[i] = ScanIO{};
            io[i].rev = false;
            io[i].ops = (const char*)ops + (size_t)lo * Tp * 2 * TC_OPS_ROWS;   // [BH][Tp/64][144][64] fp16
            io[i].g = g + lo * NC;
            io[i].S0 = S0 ? S0 + lo * 4096 * 64 : nullptr;
            io[i].z0 = z0 ? z0 + lo * 4096 : nullptr;
            io[i].amax = amax + lo * 4;
            io[i].Sx = (char*)states + (size_t)lo * NC * 2 * TC_PACKED_ROWS * 64 * 2;   // packed planes
            io[i].zx = zx + lo * NC * 4096;
            io[i].S_final = S_final ? S_final + lo * 4096 * 64 : nullptr;
            io[i].z_final = z_final ? z_final + lo * 4096 : nullptr;
            if (!sd) {
                TM2_RUN("tc_state_scan_fwd", tc_state_scan(pp[i], io[i], s));
                continue;
            }
            TM2_CK(cudaStreamWaitEvent(sd->st[i], sd->fork, 0));
            {
                cudaStream_t s = sd->st[i];
                TM2_RUN("tc_state_scan_fwd", tc_state_scan(pp[i], io[i], s));
            }
            TM2_CK(cudaEventRecord(sd->join[i], sd->st[i]));
        }
        for (int i = 0; i < parts; ++i) {
            const long lo = BH * i / parts;
            const size_t tok = (size_t)lo * T;
            if (sd) TM2_CK(cudaStreamWaitEvent(s, sd->join[i], 0));
            TM2_RUN("tc_chunk_out", tc_chunk_out(pp[i], (const char*)q + tok * 64 * 2, (const char*)k + tok * 64 * 2,
                                                 (const char*)v + tok * 64 * 2, Aloc + lo * Tp, io[i].Sx, io[i].zx,
                                                 io[i].amax, (float*)o + tok * 64, Z ? Z + tok : nullptr, s));
        }
        return TM2_OK;
    }
    TM2_RUN("state_scan_fwd", simt_state_scan_fwd(p, k, v, Aloc, g, S0, z0, states, S_final, z_final, s));
    TM2_RUN("chunk_out", simt_chunk_out(p, q, k, v, Aloc, states, o, Z, s));
    return TM2_OK;
}

size_t tm2_backward_workspace(int B, int H, int T, int d, int dv, int chunk, int dtype,
                              unsigned flags) {
    Problem p;
    if (make_problem(B, H, T, d, dv, chunk, dtype, flags, p, true, TM2_REUSE_STATES | TM2_GRADS_INPUT_DTYPE) != TM2_OK)
        return 0;
    return plan_bwd(p).total;
}

int tm2_backward(const void* q, const void* k, const void* v, const float* a, const void* o,
                 const float* Z, const void* dO, void* dq, void* dk, void* dv, float* da, int B,
                 int H, int T, int d, int dv_dim, int chunk, int dtype, unsigned flags, void* ws,
                 size_t ws_bytes, void* stream) {
    Problem p;
    int st = make_problem(B, H, T, d, dv_dim, chunk, dtype, flags, p, true, TM2_REUSE_STATES | TM2_GRADS_INPUT_DTYPE);
    if (st != TM2_OK) return st;
    const bool reuse = (flags & TM2_REUSE_STATES) != 0;
    if (p.BH() == 0 || T == 0) return TM2_OK;
    if (!q || !k || !v || !a || !o || !dO || !dq || !dk || !dv || !da) return TM2_ERR_INVALID_ARG;
    if (p.normalize && !Z) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, o, Z, dO, dq, dk, dv, da};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    const BwdWs w = plan_bwd(p);
    st = check_ws(ws, ws_bytes, w.total);
    if (st != TM2_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    if (p.tc) {
        void* Sx = at<void>(ws, w.states);
        void* dSx = at<void>(ws, w.dstates);
        float* zx = at<float>(ws, w.zx);
        float* dzx = at<float>(ws, w.dzx);
        float* sscale = at<float>(ws, w.sscale);
        float* zmax = at<float>(ws, w.zmax);
        float* zeta = at<float>(ws, w.zeta);
        float* ucol = at<float>(ws, w.ucol);
        float* rowterm = at<float>(ws, w.rowterm);
        float* dcum = at<float>(ws, w.dcum);
        unsigned* amax_f = at<unsigned>(ws, w.amax_f);
        unsigned* amax_r = at<unsigned>(ws, w.amax_r);
        void* ops = at<void>(ws, w.ops);
        if (!reuse) {
            TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
            TM2_RUN("head_absmax", launch_head_absmax(p, k, v, amax_f, true, s));
            TM2_RUN("tc_scan_operands",
                    launch_tc_scan_operands(p, false, k, v, Aloc, g, nullptr, nullptr, nullptr, amax_f, ops, s));
            ScanIO f{};
            f.rev = false; f.ops = ops; f.g = g; f.Sx = Sx; f.zx = zx; f.amax = amax_f;
            TM2_RUN("tc_state_scan_fwd", tc_state_scan(p, f, s));
        }
        TM2_RUN("tc_dy_prep", launch_tc_dy_prep(p, (const float*)o, Z, dO, Aloc, zeta, ucol, rowterm, zmax, amax_r, s));
        TM2_RUN("head_absmax", launch_head_absmax(p, q, dO, amax_r, false, s));
        TM2_RUN("tc_scan_operands", launch_tc_scan_operands(p, true, q, dO, Aloc, g, zeta, ucol, zmax, amax_r, ops, s));
        ScanIO r{};
        r.rev = true; r.ops = ops; r.g = g; r.zmax = zmax; r.amax = amax_r;
        r.Sx = dSx; r.zx = dzx; r.sscale = sscale;
        // the reverse walk on a side stream, dq beside it; dk/dv waits for the walk
        const Side* sd = nullptr;
        TM2_CK(side_resources(s, &sd));
        if (sd) {
            TM2_CK(cudaEventRecord(sd->fork, s));
            TM2_CK(cudaStreamWaitEvent(sd->st[0], sd->fork, 0));
            {
                cudaStream_t s = sd->st[0];
                TM2_RUN("tc_state_scan_bwd", tc_state_scan(p, r, s));
            }
            TM2_CK(cudaEventRecord(sd->join[0], sd->st[0]));
        } else {
            TM2_RUN("tc_state_scan_bwd", tc_state_scan(p, r, s));
        }
        TM2_RUN("tc_bwd_dq", tc_bwd_dq(p, q, k, v, dO, Aloc, zeta, ucol, Sx, zx, amax_f, dq, s));
        if (sd) TM2_CK(cudaStreamWaitEvent(s, sd->join[0], 0));
        TM2_RUN("tc_bwd_dkdv", tc_bwd_dkdv(p, q, k, v, dO, Aloc, g, zeta, ucol, rowterm, dSx, dzx, sscale, amax_r,
                                           dk, dv, dcum, s));
        TM2_RUN("reverse_cumsum_da", launch_reverse_cumsum_da(p, a, dcum, nullptr, da, s));
        return TM2_OK;
    }
    float* states = at<float>(ws, w.states);
    float* dstates = at<float>(ws, w.dstates);
    float* dY = at<float>(ws, w.dY);
    float* rowterm = at<float>(ws, w.rowterm);
    float* dcum = at<float>(ws, w.dcum);
    if (!reuse) {
        TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
        TM2_RUN("state_scan_fwd", simt_state_scan_fwd(p, k, v, Aloc, g, nullptr, nullptr, states, nullptr, nullptr, s));
    }
    TM2_RUN("dy_prep", launch_dy_prep(p, o, Z, dO, dY, rowterm, s));
    TM2_RUN("state_scan_bwd", simt_state_scan_bwd(p, q, dY, Aloc, g, dstates, s));
    TM2_RUN("bwd_chunk", simt_bwd_chunk(p, q, k, v, Aloc, g, dY, rowterm, states, dstates, dq, dk, dv, dcum, s));
    TM2_RUN("reverse_cumsum_da", launch_reverse_cumsum_da(p, a, dcum, nullptr, da, s));
    return TM2_OK;
}

static int step_checks(const void* q, const void* k, const void* v, const float* a, const float* S, const float* z,
                       const void* o, const float* Z, int N, int H, int d, int dv, int dtype, unsigned flags) {
    if (N < 0 || H < 0 || d <= 0 || dv <= 0) return TM2_ERR_INVALID_ARG;
    if (dtype != TM2_F32 && dtype != TM2_BF16) return TM2_ERR_UNSUPPORTED;
    if (d != dv || (d != 16 && d != 32 && d != 64)) return TM2_ERR_UNSUPPORTED;
    if (flags & ~(TM2_NORMALIZE | TM2_PACKED_STATE)) return TM2_ERR_INVALID_ARG;
    if ((long)N * H == 0) return TM2_OK;
    if ((long)N * H > 0x7fffffffL) return TM2_ERR_UNSUPPORTED;
    if (!q || !k || !v || !a || !S || !o) return TM2_ERR_INVALID_ARG;
    if ((flags & TM2_NORMALIZE) && !z) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, S, z, o, Z};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    return TM2_OK;
}

int tm2_step(const void* q, const void* k, const void* v, const float* a, float* S, float* z,
             void* o, float* Z, int N, int H, int d, int dv, int dtype, unsigned flags,
             void* stream) {
    const int st = step_checks(q, k, v, a, S, z, o, Z, N, H, d, dv, dtype, flags);
    if (st != TM2_OK || (long)N * H == 0) return st;
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN(flags & TM2_PACKED_STATE ? "decode_step_packed" : "decode_step",
            launch_decode_step(N, H, d, dv, dtype, (flags & TM2_NORMALIZE) != 0, (flags & TM2_PACKED_STATE) != 0,
                               nullptr, q, k, v, a, S, z, o, Z, s));
    return TM2_OK;
}

int tm2_step_conv(const void* q, const void* k, const void* v, const float* a, const float* wq, const float* wk,
                  const float* wv, const float* bq, const float* bk, const float* bv, void* cq, void* ck, void* cv,
                  float* S, float* z, void* o, float* Z, int N, int H, int d, int dv, int dtype, unsigned flags,
                  void* stream) {
    int st = step_checks(q, k, v, a, S, z, o, Z, N, H, d, dv, dtype, flags);
    if (st != TM2_OK || (long)N * H == 0) return st;
    if (!wq || !wk || !wv || !cq || !ck || !cv) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {wq, wk, wv, bq, bk, bv, cq, ck, cv};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    DecodeConv c{{wq, wk, wv}, {bq, bk, bv}, {cq, ck, cv}};
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN(flags & TM2_PACKED_STATE ? "decode_step_conv_packed" : "decode_step_conv",
            launch_decode_step(N, H, d, dv, dtype, (flags & TM2_NORMALIZE) != 0, (flags & TM2_PACKED_STATE) != 0,
                               &c, q, k, v, a, S, z, o, Z, s));
    return TM2_OK;
}

static int pack_args(const float* full, const float* packed, int NH, int d, int dv) {
    if (NH < 0 || (d != 16 && d != 32 && d != 64) || dv != d) return NH < 0 ? TM2_ERR_INVALID_ARG : TM2_ERR_UNSUPPORTED;
    if (NH > 0 && (!full || !packed)) return TM2_ERR_INVALID_ARG;
    if (!aligned16(full) || !aligned16(packed)) return TM2_ERR_ALIGNMENT;
    return TM2_OK;
}

int tm2_state_pack(const float* S, const float* z, float* S_packed, float* z_packed, int NH, int d, int dv,
                   void* stream) {
    int st = pack_args(S, S_packed, NH, d, dv);
    if (st != TM2_OK) return st;
    if ((z == nullptr) != (z_packed == nullptr) || !aligned16(z) || !aligned16(z_packed)) return TM2_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN("state_pack", launch_state_pack(S, S_packed, NH, d, dv, false, s));
    if (z) TM2_RUN("state_pack", launch_state_pack(z, z_packed, NH, d, 1, false, s));
    return TM2_OK;
}

int tm2_state_unpack(const float* S_packed, const float* z_packed, float* S, float* z, int NH, int d, int dv,
                     void* stream) {
    int st = pack_args(S, S_packed, NH, d, dv);
    if (st != TM2_OK) return st;
    if ((z == nullptr) != (z_packed == nullptr) || !aligned16(z) || !aligned16(z_packed)) return TM2_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN("state_unpack", launch_state_pack(S, const_cast<float*>(S_packed), NH, d, dv, true, s));
    if (z) TM2_RUN("state_unpack", launch_state_pack(z, const_cast<float*>(z_packed), NH, d, 1, true, s));
    return TM2_OK;
}

size_t tm2e_step_workspace(int N, int H, int L, int d, int dv, int dtype) {
    if (N < 0 || H < 0 || L <= 0 || d != dv || (d != 16 && d != 32 && d != 64)) return 0;
    if (dtype != TM2_F32 && dtype != TM2_BF16) return 0;
    const size_t n = (size_t)N * H * e_decode_max_splits(L) * (dv + 2) * sizeof(float);
    return (n + 255) & ~(size_t)255;
}

int tm2e_step(const void* q, const void* k, const void* v, const float* a, void* K_cache, void* V_cache,
              float* cum_cache, int pos, int L, void* o, float* lse, int N, int H, int d, int dv, float scale,
              int dtype, void* ws, size_t ws_bytes, void* stream) {
    if (N < 0 || H < 0 || L <= 0) return TM2_ERR_INVALID_ARG;
    if (dtype != TM2_F32 && dtype != TM2_BF16) return TM2_ERR_UNSUPPORTED;
    if (d != dv || (d != 16 && d != 32 && d != 64)) return TM2_ERR_UNSUPPORTED;
    if (pos < 0 || pos >= L) return TM2_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == 0.f) return TM2_ERR_INVALID_ARG;
    const long NH = (long)N * H;
    if (NH == 0) return TM2_OK;
    if (NH > 65535L * 1024) return TM2_ERR_UNSUPPORTED;
    if (!q || !k || !v || !a || !K_cache || !V_cache || !cum_cache || !o) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, K_cache, V_cache, cum_cache, o, lse};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    const int ns = e_decode_splits(NH, pos);
    float* part = nullptr;
    if (ns > 1) {
        const int st = check_ws(ws, ws_bytes, tm2e_step_workspace(N, H, L, d, dv, dtype));
        if (st != TM2_OK) return st;
        part = (float*)ws;
    }
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN("e_decode", launch_e_decode(NH, d, dtype, pos, L, scale, q, k, v, a, K_cache, V_cache, cum_cache, part,
                                        (float*)o, lse, s));
    return TM2_OK;
}

size_t tm2e_fill_cache_workspace(int B, int H, int T, int d, int dv, int dtype) {
    return tm2e_forward_workspace(B, H, T, d, dv, dtype);
}

int tm2e_fill_cache(const void* k, const void* v, const float* a, void* K_cache, void* V_cache, float* cum_cache,
                    int B, int H, int T, int L, int d, int dv, int dtype, void* ws, size_t ws_bytes, void* stream) {
    Problem p{};
    int st = make_problem(B, H, T, d, dv, 0, dtype, 0, p);
    if (st != TM2_OK) return st;
    if (T > L) return TM2_ERR_INVALID_ARG;
    if (p.BH() == 0 || T == 0) return TM2_OK;
    if (!k || !v || !a || !K_cache || !V_cache || !cum_cache) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {k, v, a, K_cache, V_cache, cum_cache};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    const EWs w = plan_e(p, false);
    st = check_ws(ws, ws_bytes, w.total);
    if (st != TM2_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    float* cum = at<float>(ws, w.cum);
    float* cum_lo = at<float>(ws, w.cum_lo);
    TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
    TM2_RUN("global_cumsum", launch_global_cumsum(p, Aloc, g, cum, cum_lo, s));
    TM2_RUN("e_cache_fill", launch_e_cache_fill(p.BH(), T, L, d, dv, dtype, k, v, cum, cum_lo, K_cache, V_cache,
                                                cum_cache, s));
    return TM2_OK;
}

static int conv_args(int B, int H, int T, int C, int dtype) {
    if (B < 0 || H < 0 || T < 0) return TM2_ERR_INVALID_ARG;
    if (dtype != TM2_F32 && dtype != TM2_BF16) return TM2_ERR_UNSUPPORTED;
    if (C != 16 && C != 32 && C != 64) return TM2_ERR_UNSUPPORTED;
    return TM2_OK;
}

int tm2_conv2_forward(const void* x, const float* w, const float* b, const void* x_prev, void* y, int B, int H,
                      int T, int C, int dtype, void* stream) {
    int st = conv_args(B, H, T, C, dtype);
    if (st != TM2_OK) return st;
    if ((long)B * H * T == 0) return TM2_OK;
    if (!x || !w || !y) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w, b, x_prev, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return TM2_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN("conv2_fwd", launch_conv2_fwd((long)B * H, H, T, C, dtype, x, w, b, x_prev, y, s));
    return TM2_OK;
}

int tm2_conv2_backward(const void* x, const float* w, const void* x_prev, const void* dy, float* dx, float* dx_prev,
                       float* dw, float* db, int B, int H, int T, int C, int dtype, void* stream) {
    int st = conv_args(B, H, T, C, dtype);
    if (st != TM2_OK) return st;
    if ((long)B * H * T == 0) return TM2_OK;
    if (!x || !w || !dy || !dx || !dw) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {x, w, x_prev, dy, dx, dx_prev, dw, db};
    for (const void* p : ptrs)
        if (!aligned16(p)) return TM2_ERR_ALIGNMENT;
    cudaStream_t s = (cudaStream_t)stream;
    TM2_RUN("conv2_bwd", launch_conv2_bwd(B, H, T, C, dtype, x, w, x_prev, dy, dx, dx_prev, dw, db, s));
    return TM2_OK;
}

size_t tm2e_forward_workspace(int B, int H, int T, int d, int dv, int dtype) {
    Problem p;
    if (make_problem(B, H, T, d, dv, 0, dtype, 0, p) != TM2_OK) return 0;
    return plan_e(p, false).total;
}

int tm2e_forward(const void* q, const void* k, const void* v, const float* a, void* o, float* lse,
                 int B, int H, int T, int d, int dv, float scale, int dtype, void* ws,
                 size_t ws_bytes, void* stream) {
    Problem p;
    int st = tm2::e_forward_check(q, k, v, a, o, lse, B, H, T, d, dv, scale, dtype, p);
    if (st != TM2_OK || p.BH() == 0 || T == 0) return st;
    st = check_ws(ws, ws_bytes, plan_e(p, false).total);
    if (st != TM2_OK) return st;
    return tm2::e_forward_run(p, q, k, v, a, o, lse, scale, ws, (cudaStream_t)stream);
}

size_t tm2e_backward_workspace(int B, int H, int T, int d, int dv, int dtype) {
    Problem p;
    if (make_problem(B, H, T, d, dv, 0, dtype, 0, p) != TM2_OK) return 0;
    return plan_e(p, true).total;
}

int tm2e_backward(const void* q, const void* k, const void* v, const float* a, const void* o,
                  const float* lse, const void* dO, void* dq, void* dk, void* dv, float* da, int B,
                  int H, int T, int d, int dv_dim, float scale, int dtype, unsigned flags, void* ws,
                  size_t ws_bytes, void* stream) {
    Problem p;
    int st = make_problem(B, H, T, d, dv_dim, 0, dtype, flags, p, false, TM2_GRADS_INPUT_DTYPE);
    if (flags & TM2_NORMALIZE) return TM2_ERR_INVALID_ARG;
    if (st != TM2_OK) return st;
    if (!(scale == scale) || scale == 0.f) return TM2_ERR_INVALID_ARG;
    if (p.BH() == 0 || T == 0) return TM2_OK;
    if (!q || !k || !v || !a || !o || !lse || !dO || !dq || !dk || !dv || !da)
        return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, o, lse, dO, dq, dk, dv, da};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    const EWs w = plan_e(p, true);
    st = check_ws(ws, ws_bytes, w.total);
    if (st != TM2_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    float* cum = at<float>(ws, w.cum);
    float* cum_lo = at<float>(ws, w.cum_lo);
    float* Dvec = at<float>(ws, w.Dvec);
    float* rowsum = at<float>(ws, w.rowsum);
    float* colsum = at<float>(ws, w.colsum);
    TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
    TM2_RUN("global_cumsum", launch_global_cumsum(p, Aloc, g, cum, cum_lo, s));
    TM2_RUN("rowdot", launch_rowdot(p, o, dO, Dvec, s));
    if (p.dtype == TM2_BF16 && p.d == 64 && p.dv == 64)
        TM2_RUN("tc_e_bwd", tc_e_bwd(p, q, k, v, cum, cum_lo, lse, Dvec, dO, scale, dq, dk, dv, rowsum, colsum, s));
    else
        TM2_RUN("e_bwd", simt_e_bwd(p, q, k, v, cum, cum_lo, lse, Dvec, dO, scale, dq, dk, dv, rowsum, colsum, s));
    TM2_RUN("reverse_cumsum_da", launch_reverse_cumsum_da(p, a, rowsum, colsum, da, s));
    return TM2_OK;
}

static int make_q_problem(int B, int H, int T, int d, int dv, int order, int dtype, unsigned flags, Problem& p,
                          unsigned extra = 0) {
    if (order != 1 && order != 2) return TM2_ERR_UNSUPPORTED;
    return make_problem(B, H, T, d, dv, 0, dtype, flags, p, false, extra);
}

static bool q_tc(const Problem& p) { return p.dtype == TM2_BF16 && p.d == 64 && p.dv == 64; }

size_t tm2q_forward_workspace(int B, int H, int T, int d, int dv, int order, int dtype, unsigned flags) {
    Problem p{};
    if (make_q_problem(B, H, T, d, dv, order, dtype, flags, p) != TM2_OK) return 0;
    return plan_q(p, false).total;
}

int tm2q_forward(const void* q, const void* k, const void* v, const float* a, void* o, float* Z, int B, int H,
                 int T, int d, int dv, int order, int dtype, unsigned flags, void* ws, size_t ws_bytes,
                 void* stream) {
    Problem p{};
    int st = make_q_problem(B, H, T, d, dv, order, dtype, flags, p);
    if (st != TM2_OK) return st;
    if (p.BH() == 0 || T == 0) return TM2_OK;
    if (!q || !k || !v || !a || !o) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, o, Z};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    const QWs w = plan_q(p, false);
    st = check_ws(ws, ws_bytes, w.total);
    if (st != TM2_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    float* cum = at<float>(ws, w.cum);
    float* cum_lo = at<float>(ws, w.cum_lo);
    float* Zo = Z ? Z : at<float>(ws, w.Zs);
    TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
    TM2_RUN("global_cumsum", launch_global_cumsum(p, Aloc, g, cum, cum_lo, s));
    if (q_tc(p))
        TM2_RUN("tc_poly_fwd", tc_poly_fwd(p, order, q, k, v, cum, cum_lo, (float*)o, Zo, s));
    else
        TM2_RUN("poly_fwd", simt_poly_fwd(p, order, q, k, v, cum, cum_lo, o, Zo, s));
    return TM2_OK;
}

size_t tm2q_backward_workspace(int B, int H, int T, int d, int dv, int order, int dtype, unsigned flags) {
    Problem p{};
    if (make_q_problem(B, H, T, d, dv, order, dtype, flags, p, TM2_GRADS_INPUT_DTYPE) != TM2_OK) return 0;
    return plan_q(p, true).total;
}

int tm2q_backward(const void* q, const void* k, const void* v, const float* a, const void* o, const float* Z,
                  const void* dO, void* dq, void* dk, void* dv, float* da, int B, int H, int T, int d, int dv_dim,
                  int order, int dtype, unsigned flags, void* ws, size_t ws_bytes, void* stream) {
    Problem p{};
    int st = make_q_problem(B, H, T, d, dv_dim, order, dtype, flags, p, TM2_GRADS_INPUT_DTYPE);
    if (st != TM2_OK) return st;
    if (p.BH() == 0 || T == 0) return TM2_OK;
    if (!q || !k || !v || !a || !dO || !dq || !dk || !dv || !da) return TM2_ERR_INVALID_ARG;
    if (p.normalize && (!o || !Z)) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, o, Z, dO, dq, dk, dv, da};
    for (const void* x : ptrs)
        if (!aligned16(x)) return TM2_ERR_ALIGNMENT;
    const QWs w = plan_q(p, true);
    st = check_ws(ws, ws_bytes, w.total);
    if (st != TM2_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    float* Aloc = at<float>(ws, w.Aloc);
    float* g = at<float>(ws, w.g);
    float* cum = at<float>(ws, w.cum);
    float* cum_lo = at<float>(ws, w.cum_lo);
    float* D = at<float>(ws, w.D);
    float* zeta = at<float>(ws, w.zeta);
    float* rowsum = at<float>(ws, w.rowsum);
    float* colsum = at<float>(ws, w.colsum);
    TM2_RUN("decay_chunk", launch_decay(p, a, Aloc, g, s));
    TM2_RUN("global_cumsum", launch_global_cumsum(p, Aloc, g, cum, cum_lo, s));
    TM2_RUN("poly_prep", launch_poly_prep(p, (const float*)o, Z, dO, D, zeta, s));
    if (q_tc(p))
        TM2_RUN("tc_poly_bwd", tc_poly_bwd(p, order, q, k, v, cum, cum_lo, zeta, D, dO, dq, dk, dv, rowsum, colsum,
                                           s));
    else
        TM2_RUN("poly_bwd",
                simt_poly_bwd(p, order, q, k, v, cum, cum_lo, zeta, D, dO, dq, dk, dv, rowsum, colsum, s));
    TM2_RUN("reverse_cumsum_da", launch_reverse_cumsum_da(p, a, rowsum, colsum, da, s));
    return TM2_OK;
}

int tm2_trace_enable(int on) {
    g_trace_on = on != 0;
    if (g_trace_on) g_trace_n = 0;
    return TM2_OK;
}

int tm2_trace_count(void) { return (int)g_trace_n; }

int tm2_trace_read(int i, char* name, int name_len, float* ms) {
    if (i < 0 || (size_t)i >= g_trace_n || !ms) return TM2_ERR_INVALID_ARG;
    const TraceRec& r = g_trace[i];
    if (name && name_len > 0) {
        strncpy(name, r.name, (size_t)name_len - 1);
        name[name_len - 1] = 0;
    }
    if (cudaEventSynchronize(r.end) != cudaSuccess) return TM2_ERR_CUDA;
    if (cudaEventElapsedTime(ms, r.beg, r.end) != cudaSuccess) return TM2_ERR_CUDA;
    return TM2_OK;
}

int tm2_poll_status(void) { return tm2::read_tc_status(true); }

const char* tm2_last_cuda_error(void) {
    return g_last_cuda_error ? cudaGetErrorString((cudaError_t)g_last_cuda_error) : "no CUDA error";
}

}  // extern "C"
