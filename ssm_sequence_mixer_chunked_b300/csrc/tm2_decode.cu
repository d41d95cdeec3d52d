// tm2_decode.cu -- one recurrent decode step of the second-order state
// ("2Mamba2Furious", App. A: recurrent inference with a fixed-size state;
//  Sec. 2: the state has size (d^2, dv)):
//   gamma = exp(-softplus(a)),  S <- gamma S + (k (x) k) v^T,  z <- gamma z + k (x) k,
//   y = (q (x) q)^T S,  zeta = (q (x) q)^T z,  o = y / zeta (normalised) or y.
//
// The step is bound by HBM bandwidth: each (sequence, head) state of d^2 x dv fp32
// (1 MiB at d = dv = 64) is read once and written once, in place.  One 256-thread
// block per (sequence, head); a thread owns one float4 of value columns and walks
// every (256 / (dv/4))-th state row, with 8 rows' loads issued before any store so
// that each thread keeps 128 bytes in flight.  Loads and stores use the streaming
// cache hints (each byte is touched once per step).
#include <algorithm>

#include "tm2_common.cuh"
#include "tm2_launch.h"

namespace tm2 {

// Optional, selected at compile time:
//  * PACKED: the state is kept symmetric-packed, only the rows (m, n) with m <= n
//    (d(d+1)/2 of d^2; row index r = m d - m(m-1)/2 + (n - m)).  k (x) k and q (x) q are
//    symmetric, so every update adds a symmetric term and the readout sees only the symmetric
//    part of S: with the off-diagonal rows weighted 2 q_m q_n the outputs are those of the full
//    state, and the step moves about half the bytes ("2Mamba2Furious", Sec. 5.1: the squared
//    state's memory; Sec. 7: hidden-state size).
//  * CONV: the size-2 input convolution of Mamba-2S is applied to q, k, v first (Sec. 3-4:
//    window 2, no activation; App. A: inference caches the previous window - 1 = 1 raw query,
//    key and value): x'_t = w0 x_t + w1 x_{t-1} (+ b) per channel, with x_{t-1} read from and
//    x_t written to the caller's cache.
struct ConvArgs {
    const float* w[3];    // q, k, v weights (H, d, 2): [.., 0] on x_t, [.., 1] on x_{t-1}
    const float* b[3];    // biases (H, d) or null
    void* cache[3];       // previous raw q, k, v (N, H, d) in the input dtype, in/out
    int H;
};

template <int D>
struct StateRows {
    static constexpr int FULL = D * D;
    static constexpr int PACKED = D * (D + 1) / 2;
};

template <int D, int DV, typename Tin, bool PACKED, bool CONV>
__global__ void __launch_bounds__(256) decode_step_kernel(
    const Tin* __restrict__ q, const Tin* __restrict__ k, const Tin* __restrict__ v,
    const float* __restrict__ a, float* __restrict__ S, float* __restrict__ z, float* __restrict__ o,
    float* __restrict__ Zout, bool normalize, ConvArgs cv) {
    constexpr int NQ = DV / 4;        // float4 column groups per state row
    constexpr int RG = 256 / NQ;      // row groups
    constexpr int R = PACKED ? StateRows<D>::PACKED : StateRows<D>::FULL;   // state rows
    constexpr int U = 8;              // rows in flight per thread
    __shared__ float sq[D], sk[D], sv[DV];
    __shared__ uint16_t smn[PACKED ? R : 1];   // packed row -> (m << 8) | n
    __shared__ float4 sred[RG][NQ];
    __shared__ float zred[8];
    const long s = blockIdx.x;
    const int tid = threadIdx.x;
    if constexpr (CONV) {
        const int h = (int)(s % cv.H);
        const Tin* in[3] = {q, k, v};
        float* dst[3] = {sq, sk, sv};
#pragma unroll
        for (int x = 0; x < 3; ++x) {
            Tin* cache = reinterpret_cast<Tin*>(cv.cache[x]);
            for (int e = tid; e < D; e += 256) {
                const Tin cur = in[x][s * D + e];
                const float prev = to_f(cache[s * D + e]);
                const float* w = cv.w[x] + ((long)h * D + e) * 2;
                float y = fmaf(w[0], to_f(cur), w[1] * prev);
                if (cv.b[x]) y += cv.b[x][(long)h * D + e];
                dst[x][e] = y;
                cache[s * D + e] = cur;
            }
        }
    } else {
        for (int e = tid; e < D; e += 256) {
            sq[e] = to_f(q[s * D + e]);
            sk[e] = to_f(k[s * D + e]);
        }
        for (int e = tid; e < DV; e += 256) sv[e] = to_f(v[s * DV + e]);
    }
    if constexpr (PACKED) {
        for (int e = tid; e < D * D; e += 256) {
            const int m = e / D, n = e % D;
            if (n >= m) smn[m * D - m * (m - 1) / 2 + (n - m)] = (uint16_t)((m << 8) | n);
        }
    }
    const float gamma = __expf(-softplus_f(a[s]));
    __syncthreads();
    // state row r -> key indices (m, n) and the readout weight of the row
    auto row_mn = [&](int r, int& m, int& n) {
        if constexpr (PACKED) {
            const int mn = smn[r];
            m = mn >> 8;
            n = mn & 0xff;
        } else {
            m = r / D;
            n = r % D;
        }
    };

    const int cq = tid % NQ, rg = tid / NQ;
    const float4 vq = make_float4(sv[4 * cq], sv[4 * cq + 1], sv[4 * cq + 2], sv[4 * cq + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float4* Sp = reinterpret_cast<float4*>(S + s * (long)R * DV);
    for (int r0 = rg; r0 < R; r0 += RG * U) {
        float4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * RG;
            if (R % (RG * U) == 0 || r < R) x[u] = __ldcs(Sp + (long)r * NQ + cq);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int r = r0 + u * RG;
            if (R % (RG * U) != 0 && r >= R) break;
            int m, n;
            row_mn(r, m, n);
            const float kk = sk[m] * sk[n];
            const float qq = (PACKED && m != n) ? 2.f * sq[m] * sq[n] : sq[m] * sq[n];
            float4 y;
            y.x = fmaf(gamma, x[u].x, kk * vq.x);
            y.y = fmaf(gamma, x[u].y, kk * vq.y);
            y.z = fmaf(gamma, x[u].z, kk * vq.z);
            y.w = fmaf(gamma, x[u].w, kk * vq.w);
            __stcs(Sp + (long)r * NQ + cq, y);
            acc.x = fmaf(qq, y.x, acc.x);
            acc.y = fmaf(qq, y.y, acc.y);
            acc.z = fmaf(qq, y.z, acc.z);
            acc.w = fmaf(qq, y.w, acc.w);
        }
    }
    float zacc = 0.f;
    if (z) {
        float* zp = z + s * (long)R;
        for (int r = tid; r < R; r += 256) {
            int m, n;
            row_mn(r, m, n);
            const float zn = fmaf(gamma, __ldcs(zp + r), sk[m] * sk[n]);
            __stcs(zp + r, zn);
            const float qq = (PACKED && m != n) ? 2.f * sq[m] * sq[n] : sq[m] * sq[n];
            zacc = fmaf(qq, zn, zacc);
        }
    }
    sred[rg][cq] = acc;
    zacc = warp_sum(zacc);
    if ((tid & 31) == 0) zred[tid >> 5] = zacc;
    __syncthreads();
    if (tid < NQ) {
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int g2 = 0; g2 < RG; ++g2) {
            const float4 t = sred[g2][tid];
            y.x += t.x; y.y += t.y; y.z += t.z; y.w += t.w;
        }
        float ze = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) ze += zred[w];
        const float inv = (normalize && ze != 0.f) ? 1.f / ze : (normalize ? 0.f : 1.f);
        reinterpret_cast<float4*>(o + s * DV)[tid] = make_float4(y.x * inv, y.y * inv, y.z * inv, y.w * inv);
        if (tid == 0 && Zout) Zout[s] = ze;
    }
}

template <int D, typename T, bool PACKED, bool CONV>
static void decode_launch(unsigned blocks, cudaStream_t s, const void* q, const void* k, const void* v,
                          const float* a, float* S, float* z, void* o, float* Z, bool normalize, const ConvArgs& cv) {
    decode_step_kernel<D, D, T, PACKED, CONV><<<blocks, 256, 0, s>>>((const T*)q, (const T*)k, (const T*)v, a, S, z,
                                                                      (float*)o, Z, normalize, cv);
}

template <int D, typename T>
static void decode_dispatch(bool packed, bool conv, unsigned blocks, cudaStream_t s, const void* q, const void* k,
                            const void* v, const float* a, float* S, float* z, void* o, float* Z, bool normalize,
                            const ConvArgs& cv) {
    if (packed) {
        if (conv) decode_launch<D, T, true, true>(blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
        else decode_launch<D, T, true, false>(blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
    } else {
        if (conv) decode_launch<D, T, false, true>(blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
        else decode_launch<D, T, false, false>(blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
    }
}

cudaError_t launch_decode_step(int N, int H, int d, int dv, int dtype, bool normalize, bool packed,
                               const DecodeConv* conv, const void* q, const void* k, const void* v,
                               const float* a, float* S, float* z, void* o, float* Z, cudaStream_t s) {
    const unsigned blocks = (unsigned)((long)N * H);
    ConvArgs cv{};
    cv.H = H;
    if (conv) {
        for (int x = 0; x < 3; ++x) {
            cv.w[x] = conv->w[x];
            cv.b[x] = conv->b[x];
            cv.cache[x] = conv->cache[x];
        }
    }
    const bool c = conv != nullptr;
    if (dtype == 1) {
        if (d == 64) decode_dispatch<64, __nv_bfloat16>(packed, c, blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
        else if (d == 32) decode_dispatch<32, __nv_bfloat16>(packed, c, blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
        else decode_dispatch<16, __nv_bfloat16>(packed, c, blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
    } else {
        if (d == 64) decode_dispatch<64, float>(packed, c, blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
        else if (d == 32) decode_dispatch<32, float>(packed, c, blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
        else decode_dispatch<16, float>(packed, c, blocks, s, q, k, v, a, S, z, o, Z, normalize, cv);
    }
    (void)dv;
    return cudaGetLastError();
}

// Symmetric packing of full states (rows r = m d + n) and back: packed row (m, n), m <= n, is
// (S[(m,n)] + S[(n,m)]) / 2 -- the part of the state every readout (q (x) q)^T S sees; the
// unpacked state is that symmetric part.  One thread per (head, packed row, column).
__global__ void state_pack_kernel(float* __restrict__ full, float* __restrict__ packed, long nh, int d,
                                  int cols, bool unpack) {
    const int R = d * (d + 1) / 2;
    const long total = nh * (long)R * cols;
    for (long e = (long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (long)gridDim.x * blockDim.x) {
        const int c = (int)(e % cols);
        const long hr = e / cols;
        const int r = (int)(hr % R);
        const long h = hr / R;
        int m = 0, rem = r;
        while (rem >= d - m) {   // row m holds d - m packed entries
            rem -= d - m;
            ++m;
        }
        const int n = m + rem;
        const long fm = (h * d * d + (long)m * d + n) * cols + c, fn = (h * d * d + (long)n * d + m) * cols + c;
        if (unpack) {
            const float x = packed[e];
            full[fm] = x;
            full[fn] = x;
        } else {
            packed[e] = 0.5f * (full[fm] + full[fn]);
        }
    }
}

cudaError_t launch_state_pack(const float* full, float* packed, long nh, int d, int cols, bool unpack,
                              cudaStream_t s) {
    // (unpack writes `full`; the entry point passes a writable buffer on that path)
    const long total = nh * (long)(d * (d + 1) / 2) * cols;
    const unsigned blocks = (unsigned)std::min<long>((total + 255) / 256, 148L * 32);
    if (total == 0) return cudaSuccess;
    state_pack_kernel<<<blocks, 256, 0, s>>>(const_cast<float*>(full), packed, nh, d, cols, unpack);
    return cudaGetLastError();
}

}  // namespace tm2
