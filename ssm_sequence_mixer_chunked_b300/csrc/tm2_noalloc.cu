// tm2_noalloc.cu -- tm2e_forward_noalloc: the 2Mamba-E forward for callers that cannot
// allocate device memory.
//
// Some hosts of this library own every byte of device memory themselves: a plugin
// inside an inference engine that plans all buffers ahead of time and forbids
// allocations once serving starts, or a latency-critical loop where cudaMalloc's
// possible implicit device synchronisation is not acceptable.  Such a caller can still
// pass its inputs and outputs, but has no way to hand over the scratch buffer that
// tm2e_forward takes as `ws`.  This entry point instead uses one fixed scratch array
// compiled into the library: a file-scope __device__ array of TM2E_NOALLOC_SCRATCH_BYTES
// (16 MiB), which every GPU that loads the library holds until the process exits.
//
// Host code cannot use the array's name as a device address, so the device address is
// looked up once per device, with that device current, by cudaGetSymbolAddress on the
// first call made on that device; later calls reuse it.  Nothing else is allocated: no
// cudaMalloc, no cudaFree, no allocating library routine.
//
// The scratch holds the chunk-local decay running sums, the chunk totals and the
// global running sums of the A-mask.  Every element a call reads is first written by
// that same call, so no part of the array needs clearing between calls.  All calls on
// a device share the one array: calls that overlap on the GPU (different streams, or
// different host threads without ordering) race on it and must be serialised by the
// caller.
#include <mutex>

#include "tm2.h"
#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

static __device__ __align__(256) unsigned char g_e_noalloc_scratch[TM2E_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[256];   // device address of g_e_noalloc_scratch, per device ordinal

static size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

}  // namespace tm2

using namespace tm2;

extern "C" int tm2e_forward_noalloc(const void* q, const void* k, const void* v, const float* a,
                                    void* o, float* lse, int B, int H, int T, int d, int dv,
                                    float scale, int dtype, void* stream) {
    if (B < 0 || H < 0 || T < 0 || d <= 0 || dv <= 0) return TM2_ERR_INVALID_ARG;
    if (dtype != TM2_F32 && dtype != TM2_BF16) return TM2_ERR_UNSUPPORTED;
    if (d != dv || (d != 16 && d != 32 && d != 64)) return TM2_ERR_UNSUPPORTED;
    if ((long)B * H > 65535) return TM2_ERR_UNSUPPORTED;
    if (!(scale == scale) || scale == 0.f) return TM2_ERR_INVALID_ARG;
    if ((long)B * H == 0 || T == 0) return TM2_OK;
    if (!q || !k || !v || !a || !o || !lse) return TM2_ERR_INVALID_ARG;
    const void* ptrs[] = {q, k, v, a, o, lse};
    for (const void* x : ptrs)
        if (((uintptr_t)x & 15u) != 0) return TM2_ERR_ALIGNMENT;

    Problem p;
    p.B = B; p.H = H; p.T = T; p.d = d; p.dv = dv;
    p.C = 64;
    p.NC = (T + p.C - 1) / p.C;
    p.dtype = dtype;
    p.normalize = false;
    // scratch: chunk-local running sums, chunk totals, global running sums and their residuals
    const size_t off_g = round256(sizeof(float) * (size_t)p.BH() * p.Tp());
    const size_t off_cum = off_g + round256(sizeof(float) * (size_t)p.BH() * p.NC);
    const size_t off_lo = off_cum + round256(sizeof(float) * (size_t)p.BH() * T);
    const size_t need = off_lo + round256(sizeof(float) * (size_t)p.BH() * T);
    if (need > (size_t)TM2E_NOALLOC_SCRATCH_BYTES) return TM2_ERR_WORKSPACE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return TM2_ERR_CUDA;
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_e_noalloc_scratch) != cudaSuccess || !addr) return TM2_ERR_CUDA;
            g_noalloc_addr[dev] = addr;
        }
        base = g_noalloc_addr[dev];
    }
    float* Aloc = reinterpret_cast<float*>((char*)base);
    float* g = reinterpret_cast<float*>((char*)base + off_g);
    float* cum = reinterpret_cast<float*>((char*)base + off_cum);
    float* cum_lo = reinterpret_cast<float*>((char*)base + off_lo);
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_decay(p, a, Aloc, g, s) != cudaSuccess) return TM2_ERR_CUDA;
    if (launch_global_cumsum(p, Aloc, g, cum, cum_lo, s) != cudaSuccess) return TM2_ERR_CUDA;
    if (simt_e_fwd(p, q, k, v, cum, cum_lo, scale, o, lse, s) != cudaSuccess) return TM2_ERR_CUDA;
    return TM2_OK;
}
