// tm2_tc.cu -- tensor-core infrastructure shared by the tcgen05 kernels: the device
// status word for bounded waits, TMA tensor-map encoding (driver entry point, no link
// dependency on libcuda), and a self-test GEMM that checks the operand/accumulator
// conventions of tm2_sm100.cuh on the device at hand.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "tm2.h"
#include "tm2_launch.h"
#include "tm2_sm100.cuh"
#include "tm2_tc.h"

namespace tm2 {

__device__ int g_tc_status = 0;

// ---- tensor maps ---------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::mutex g_encode_mu;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::lock_guard<std::mutex> lock(g_encode_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    return g_encode;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t pitch_elems, uint32_t box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t heads, uint64_t rows, uint64_t cols,
                       uint32_t box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {cols, rows, heads};
    cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_state_packed_quads(CUtensorMap* map, const void* base, uint64_t nchunks) {
    const uint64_t dims[4] = {64, 16, (uint64_t)TC_PACKED_BLOCKS * 16, 2 * nchunks};
    const uint64_t strides[3] = {128, 16 * 128, (uint64_t)TC_PACKED_ROWS * 128};
    const uint32_t box[4] = {64, 16, 4, 1};
    return make_tmap_f16_nd(map, base, 4, dims, strides, box);
}

bool make_tmap_state_packed_tquads(CUtensorMap* map, const void* base, uint64_t nchunks) {
    const uint64_t dims[4] = {64, 16, 16, (uint64_t)TC_PACKED_BLOCKS * 2 * nchunks};
    const uint64_t strides[3] = {16 * 128, 128, 256 * 128};
    const uint32_t box[4] = {64, 16, 4, 1};
    return make_tmap_f16_nd(map, base, 4, dims, strides, box);
}

bool make_tmap_state_packed_rowrun(CUtensorMap* map, const void* base, uint64_t nchunks, int nb) {
    if (nb < 1 || nb > 4) return false;
    const uint64_t dims[5] = {64, 16, 16, (uint64_t)TC_PACKED_BLOCKS, 2 * nchunks};
    const uint64_t strides[4] = {128, 16 * 128, 256 * 128, (uint64_t)TC_PACKED_ROWS * 128};
    const uint32_t box[5] = {64, 16, 4, (uint32_t)nb, 1};
    return make_tmap_f16_nd(map, base, 5, dims, strides, box);
}

bool make_tmap_state_packed_blocks(CUtensorMap* map, const void* base, uint64_t nchunks) {
    const uint64_t dims[3] = {64, (uint64_t)TC_PACKED_ROWS, 2 * nchunks};
    const uint64_t strides[2] = {128, (uint64_t)TC_PACKED_ROWS * 128};
    const uint32_t box[3] = {64, 256, 1};
    return make_tmap_f16_nd(map, base, 3, dims, strides, box);
}

bool make_tmap_f16_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                      const uint32_t* box) {
    auto enc = encoder();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i > 0) st[i - 1] = strides[i - 1];
    }
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, e,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static std::mutex g_status_mu;
static int* g_status_addr[256];

int* tc_status_ptr() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_tc_status) != cudaSuccess) return nullptr;
        g_status_addr[dev] = (int*)p;
    }
    return g_status_addr[dev];
}

int read_tc_status(bool clear) {
    int h = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&h, g_tc_status, sizeof(int)) != cudaSuccess) return TM2_ERR_CUDA;
    if (clear && h != 0 && cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int)) != cudaSuccess)
        return TM2_ERR_CUDA;
    return h;
}

// ---- self-test GEMM ------------------------------------------------------------------
// D (128 x N, fp32) = A (128 x K, bf16, row-major) * B^T, B (N x K).  Operand forms:
//   mode 0: A by TMA (K-major smem),            B K-major by TMA (B given as N x K)
//   mode 1: A written by the threads (swz128),   B K-major by TMA
//   mode 2: thread 0 waits on a barrier nothing arrives on (limit `wait_ns`), so the
//           bounded-wait path records TM2_ERR_TIMEOUT; no copy or MMA is issued.
//   mode 3: A in tensor memory (tcgen05.st),    B K-major by TMA
//   mode 4: A by TMA,                           B MN-major by TMA (B given as K x N)
//   mode 5: A in tensor memory,                 B MN-major by TMA
// MN-major B: 64-column blocks of B^T, each K rows of 128 bytes (128B swizzle), one block
// after the other; 8-row K groups are 1024 bytes apart (descriptor SBO), 64-column blocks
// K*128 bytes apart (LBO).
template <int N>
__global__ void __launch_bounds__(128) umma_selftest_kernel(const __grid_constant__ CUtensorMap tmA,
                                                            const __grid_constant__ CUtensorMap tmB,
                                                            const __nv_bfloat16* __restrict__ A, float* __restrict__ D,
                                                            int K, int mode, unsigned long long wait_ns,
                                                            int* __restrict__ status) {
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t A_TMEM_COL = 256;
    constexpr int NA = (N + 63) / 64;   // 64-column blocks of an MN-major B
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    const int KT = K / 64;
    const bool a_tma = mode == 0 || mode == 4;
    const bool a_tmem = mode == 3 || mode == 5;
    const bool b_mn = mode == 4 || mode == 5;
    uint8_t* sA = smem;                                              // KT tiles of 128 x 128 B
    uint8_t* sB = smem + (a_tmem ? 0 : KT * 16384);                  // B tiles
    __shared__ __align__(8) uint64_t bars[3];                        // tma, mma, never
    __shared__ uint32_t tmem_base_s;
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t bar_tma = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]), bar_never = smem_u32(&bars[2]);

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_never, 1);
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
    if (mode == 1) {   // thread r writes row r of A in the swizzled K-major layout
        for (int t = 0; t < KT; ++t)
            for (int c = 0; c < 8; ++c) {
                const uint4 x = *reinterpret_cast<const uint4*>(A + (size_t)tid * K + t * 64 + c * 8);
                st_shared_v4(smem_u32(sA + t * 16384) + swz128(tid, c), x.x, x.y, x.z, x.w);
            }
        fence_proxy_async();
    }
    if (a_tmem) {      // thread r writes row r of A into tensor-memory lane r
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        for (int kk = 0; kk < K / 16; ++kk) {
            const uint4* src = reinterpret_cast<const uint4*>(A + (size_t)tid * K + kk * 16);
            const uint4 x0 = src[0], x1 = src[1];
            const uint32_t r[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            tmem_st8(tmem + lane_base + A_TMEM_COL + kk * 8, r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    bool ok = true;
    if (tid == 0) {
        if (mode == 2) {
            ok = mbar_wait(bar_never, 0, status, wait_ns);
        } else {
            const uint32_t bytes = (a_tma ? KT * 16384 : 0) + (b_mn ? NA * K * 128 : KT * N * 128);
            mbar_arrive_expect_tx(bar_tma, bytes);
            if (a_tma)
                for (int t = 0; t < KT; ++t) tma_load_2d(smem_u32(sA + t * 16384), &tmA, bar_tma, t * 64, 0);
            if (b_mn) {
                for (int a = 0; a < NA; ++a)
                    for (int kb = 0; kb < K; kb += 256)
                        tma_load_2d(smem_u32(sB + a * K * 128 + kb * 128), &tmB, bar_tma, a * 64, kb);
            } else {
                for (int t = 0; t < KT; ++t) tma_load_2d(smem_u32(sB + t * N * 128), &tmB, bar_tma, t * 64, 0);
            }
            ok = mbar_wait(bar_tma, 0, status);
            if (ok) {
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, N, false, b_mn);
                for (int kk = 0; kk < K / 16; ++kk) {
                    const uint64_t bd = b_mn ? sdesc_sw128_ex(smem_u32(sB) + kk * 2048, K * 128, 1024)
                                             : sdesc_sw128(smem_u32(sB + (kk >> 2) * N * 128) + (kk & 3) * 32);
                    if (a_tmem) {
                        umma_bf16_ts(tmem, tmem + A_TMEM_COL + kk * 8, bd, idesc, kk > 0);
                    } else {
                        const uint64_t ad = sdesc_sw128(smem_u32(sA + (kk >> 2) * 16384) + (kk & 3) * 32);
                        umma_bf16(tmem, ad, bd, idesc, kk > 0);
                    }
                }
                umma_commit(bar_mma);
            }
        }
    }
    __syncthreads();
    if (mode != 2) {
        ok = mbar_wait(bar_mma, 0, status);
        tc_fence_after();
        if (ok) {
            const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
            for (int c = 0; c < N; c += 16) {
                float v[16];
                tmem_ld16(tmem + lane_base + c, v);
#pragma unroll
                for (int i = 0; i < 16; ++i) D[(size_t)tid * N + c + i] = v[i];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace tm2

using namespace tm2;

extern "C" int tm2_selftest_umma(const void* A, const void* B, float* D, int N, int K, int mode,
                                 unsigned long long wait_ns, void* stream) {
    if (K <= 0 || K % 64 != 0 || K > 512 || mode < 0 || mode > 5) return TM2_ERR_INVALID_ARG;
    const bool b_mn = mode == 4 || mode == 5, a_tmem = mode == 3 || mode == 5;
    const size_t a_bytes = a_tmem ? 0 : (size_t)(K / 64) * 16384;
    const size_t b_bytes = b_mn ? (size_t)((N + 63) / 64) * K * 128 : (size_t)(K / 64) * N * 128;
    const size_t smem = 1024 + a_bytes + b_bytes;
    if (smem > 227 * 1024) return TM2_ERR_UNSUPPORTED;
    if (!A || !B || !D) return TM2_ERR_INVALID_ARG;
    if (((uintptr_t)A & 15u) || ((uintptr_t)B & 15u) || ((uintptr_t)D & 15u)) return TM2_ERR_ALIGNMENT;
    CUtensorMap ta, tb;
    if (!make_tmap_bf16_2d(&ta, A, 128, (uint64_t)K, (uint64_t)K, 128)) return TM2_ERR_CUDA;
    if (b_mn) {   // B^T stored K x N row-major: boxes of 64 columns x min(K, 256) rows
        if (!make_tmap_bf16_2d(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)N, (uint32_t)(K < 256 ? K : 256)))
            return TM2_ERR_CUDA;
    } else if (!make_tmap_bf16_2d(&tb, B, (uint64_t)N, (uint64_t)K, (uint64_t)K, (uint32_t)N)) {
        return TM2_ERR_CUDA;
    }
    cudaStream_t s = (cudaStream_t)stream;
    int* status = tc_status_ptr();
    if (!status) return TM2_ERR_CUDA;
#define TM2_SELFTEST(NN)                                                                                   \
    case NN: {                                                                                             \
        auto kern = umma_selftest_kernel<NN>;                                                              \
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) \
            return TM2_ERR_CUDA;                                                                           \
        kern<<<1, 128, smem, s>>>(ta, tb, (const __nv_bfloat16*)A, D, K, mode, wait_ns, status);           \
        break;                                                                                             \
    }
    switch (N) {
        TM2_SELFTEST(16)
        TM2_SELFTEST(64)
        TM2_SELFTEST(80)
        TM2_SELFTEST(128)
        TM2_SELFTEST(256)
        default: return TM2_ERR_UNSUPPORTED;
    }
#undef TM2_SELFTEST
    return cudaGetLastError() == cudaSuccess ? TM2_OK : TM2_ERR_CUDA;
}
