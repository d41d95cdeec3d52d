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
// Argument checks, the scratch layout and the launch sequence are tm2e_forward's own
// (e_forward_check, e_forward_scratch_bytes, e_forward_run in tm2_api.cu): the same kernels
// run on the same inputs, so the results are those of tm2e_forward.  The scratch holds the
// chunk-local decay running sums, the chunk totals and the global running sums of the A-mask
// with their rounding residuals, about 12 bytes per token-head.  Every element a call reads
// is first written by that same call, so no part of the array needs clearing between calls.
// All calls on a device share the one array: calls that overlap on the GPU (different
// streams, or different host threads without ordering) race on it and must be serialised by
// the caller.
#include <mutex>

#include "tm2.h"
#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

static __device__ __align__(256) unsigned char g_e_noalloc_scratch[TM2E_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[256];   // device address of g_e_noalloc_scratch, per device ordinal

}  // namespace tm2

using namespace tm2;

extern "C" int tm2e_forward_noalloc(const void* q, const void* k, const void* v, const float* a,
                                    void* o, float* lse, int B, int H, int T, int d, int dv,
                                    float scale, int dtype, void* stream) {
    Problem p{};
    int st = e_forward_check(q, k, v, a, o, lse, B, H, T, d, dv, scale, dtype, p);
    if (st != TM2_OK || p.BH() == 0 || T == 0) return st;
    if (e_forward_scratch_bytes(p) > (size_t)TM2E_NOALLOC_SCRATCH_BYTES) return TM2_ERR_WORKSPACE;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return TM2_ERR_CUDA;
    }
    if (dev < 0 || dev >= 256) return TM2_ERR_UNSUPPORTED;
    void* base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_e_noalloc_scratch);
            if (e != cudaSuccess || !addr) {
                record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
                return TM2_ERR_CUDA;
            }
            g_noalloc_addr[dev] = addr;
        }
        base = g_noalloc_addr[dev];
    }
    return e_forward_run(p, q, k, v, a, o, lse, scale, base, (cudaStream_t)stream);
}
