// softmax_rows.cu -- row-wise online softmax and log-sum-exp.
//
// Computes, for every row r of X[rows, cols],
//     LSE[r] = log sum_c exp X[r,c]            (natural log)
//     P[r,c] = exp(X[r,c] - LSE[r])
// which is the stable softmax and log-sum-exp of "从原始Softmax到在线Softmax",
// section "softmax形式推导".  The running (max, sum) pair is maintained with the
// online normaliser of "什么是 online softmax and flash attention", section
// "Online softmax", eq (3)-(7), in its pairwise form: two partial results
// (m1, s1) and (m2, s2) combine to (M, s1 e^{m1-M} + s2 e^{m2-M}), M = max.
// That form is associative, so per-thread partials merge through warp
// shuffles and shared memory in any order.
//
// Resident kernel: one CTA per row, each thread holds its slice of the row in
// registers (NV 16-byte vectors), so X is read from HBM exactly once and P is
// written once.  Loads and stores are 128-bit and coalesced (consecutive
// threads own consecutive 16-byte vectors).
// Streaming kernels: rows longer than the resident capacity are reduced with
// the per-thread online update over 16-byte vectors (one read for LSE only,
// two reads when P is also written).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fattn_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <typename T>
struct Elem;
template <>
struct Elem<float> {
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static float load1(const float* p) { return __ldg(p); }
    __device__ static void loadv(const float* p, float* f) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p));
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
};
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static float load1(const __nv_bfloat16* p) {
        const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(u) << 16);
    }
    __device__ static void loadv(const __nv_bfloat16* p, float* f) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

// Store n = kVec(TIn) consecutive outputs starting at an element index that is
// a multiple of n (so the store is naturally aligned when `vec` is true).
template <typename TOut, int n>
__device__ __forceinline__ void store_out(TOut* p, const float* f, bool vec, int valid);

template <>
__device__ __forceinline__ void store_out<float, 4>(float* p, const float* f, bool vec, int valid) {
    if (vec) {
        *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
    } else {
        for (int i = 0; i < valid; ++i) p[i] = f[i];
    }
}
template <>
__device__ __forceinline__ void store_out<float, 8>(float* p, const float* f, bool vec, int valid) {
    if (vec) {
        reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
    } else {
        for (int i = 0; i < valid; ++i) p[i] = f[i];
    }
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16, 4>(__nv_bfloat16* p, const float* f, bool vec, int valid) {
    if (vec) {
        *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
    } else {
        for (int i = 0; i < valid; ++i) p[i] = __float2bfloat16_rn(f[i]);
    }
}
template <>
__device__ __forceinline__ void store_out<__nv_bfloat16, 8>(__nv_bfloat16* p, const float* f, bool vec, int valid) {
    if (vec) {
        *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                  pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    } else {
        for (int i = 0; i < valid; ++i) p[i] = __float2bfloat16_rn(f[i]);
    }
}

// (m, s) <- (m, s) (+) (m2, s2): the pairwise online-normaliser update.
// Sums are relative to their own max; an empty partial is (-inf, 0).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == -CUDART_INF_F) return;  // both empty
    s = s * ex2((m - M) * kLog2e) + s2 * ex2((m2 - M) * kLog2e);
    m = M;
}

// Merge (m, s) across the CTA; every thread receives the row's (M, S).
template <int THREADS>
__device__ __forceinline__ void block_merge(float& m, float& s, float* sm_m, float* sm_s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
        merge_ms(m, s, m2, s2);
    }
    if constexpr (THREADS > 32) {
        constexpr int W = THREADS / 32;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane == 0) { sm_m[warp] = m; sm_s[warp] = s; }
        __syncthreads();
        m = lane < W ? sm_m[lane] : -CUDART_INF_F;
        s = lane < W ? sm_s[lane] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
            const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
            merge_ms(m, s, m2, s2);
        }
        __syncthreads();  // the scratch may be reused by the next row
    }
}

// One CTA per row (grid-strided); the row lives in registers.
template <typename TIn, typename TOut, int THREADS, int NV>
__global__ void __launch_bounds__(THREADS) softmax_rows_resident(const TIn* __restrict__ X, TOut* __restrict__ P,
                                                                 float* __restrict__ LSE, long rows, long cols,
                                                                 int vec_ok) {
    constexpr int V = Elem<TIn>::kVec;
    __shared__ float sm_m[32], sm_s[32];
    for (long row = blockIdx.x; row < rows; row += gridDim.x) {
        const TIn* x = X + row * cols;
        float v[NV][V];
        // one read of the row: 16-byte vectors, consecutive threads adjacent
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const long e0 = (long)(threadIdx.x + k * THREADS) * V;
            if (vec_ok && e0 + V <= cols) {
                Elem<TIn>::loadv(x + e0, v[k]);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) v[k][i] = (e0 + i < cols) ? Elem<TIn>::load1(x + e0 + i) : -CUDART_INF_F;
            }
        }
        // this thread's (m, s): its max, then the sum of exp relative to it
        float m = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int i = 0; i < V; ++i) m = fmaxf(m, v[k][i]);
        float s = 0.f;
        if (m != -CUDART_INF_F) {
            const float mc = m * kLog2e;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i & 3] += ex2(fmaf(v[k][i], kLog2e, -mc));
            s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        block_merge<THREADS>(m, s, sm_m, sm_s);
        // p = exp(x - M) / S = 2^(x log2e - (M log2e + log2 S))
        const float bias = fmaf(m, kLog2e, __log2f(s));
        TOut* p = P + row * cols;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const long e0 = (long)(threadIdx.x + k * THREADS) * V;
            if (e0 < cols) {
                float o[V];
#pragma unroll
                for (int i = 0; i < V; ++i) o[i] = ex2(fmaf(v[k][i], kLog2e, -bias));
                const int valid = (int)((cols - e0) < V ? (cols - e0) : V);
                store_out<TOut, V>(p + e0, o, vec_ok && valid == V, valid);
            }
        }
        if (LSE != nullptr && threadIdx.x == 0) LSE[row] = m + logf(s);
    }
}

// Per-thread online (m, s) over a strided range of 16-byte vectors of a row:
// U vectors are loaded before they are folded in, for memory-level parallelism.
template <typename TIn, int THREADS, int U>
__device__ __forceinline__ void row_online_ms(const TIn* __restrict__ x, long cols, bool vec_ok, float& m, float& s) {
    constexpr int V = Elem<TIn>::kVec;
    const long nvec = (cols + V - 1) / V;
    m = -CUDART_INF_F;
    s = 0.f;
    for (long base = threadIdx.x; base < nvec; base += (long)THREADS * U) {
        float v[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long e0 = (base + (long)u * THREADS) * V;
            if (vec_ok && e0 + V <= cols) {
                Elem<TIn>::loadv(x + e0, v[u]);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) v[u][i] = (e0 + i < cols) ? Elem<TIn>::load1(x + e0 + i) : -CUDART_INF_F;
            }
        }
        float bm = -CUDART_INF_F;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < V; ++i) bm = fmaxf(bm, v[u][i]);
        if (bm == -CUDART_INF_F) continue;
        const float mn = fmaxf(m, bm);
        const float mc = mn * kLog2e;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < V; ++i) acc += ex2(fmaf(v[u][i], kLog2e, -mc));
        s = s * ex2((m - mn) * kLog2e) + acc;  // m = -inf on the first block: 2^-inf = 0
        m = mn;
    }
}

template <typename TIn, int THREADS, int U>
__global__ void __launch_bounds__(THREADS) logsumexp_rows_stream(const TIn* __restrict__ X, float* __restrict__ LSE,
                                                                 long rows, long cols, int vec_ok) {
    __shared__ float sm_m[32], sm_s[32];
    for (long row = blockIdx.x; row < rows; row += gridDim.x) {
        float m, s;
        row_online_ms<TIn, THREADS, U>(X + row * cols, cols, vec_ok != 0, m, s);
        block_merge<THREADS>(m, s, sm_m, sm_s);
        if (threadIdx.x == 0) LSE[row] = m + logf(s);
    }
}

// Rows longer than the resident capacity: online reduction pass, then a second
// read of the row to write P.
template <typename TIn, typename TOut, int THREADS, int U>
__global__ void __launch_bounds__(THREADS) softmax_rows_stream(const TIn* __restrict__ X, TOut* __restrict__ P,
                                                               float* __restrict__ LSE, long rows, long cols,
                                                               int vec_ok) {
    constexpr int V = Elem<TIn>::kVec;
    __shared__ float sm_m[32], sm_s[32];
    for (long row = blockIdx.x; row < rows; row += gridDim.x) {
        const TIn* x = X + row * cols;
        float m, s;
        row_online_ms<TIn, THREADS, U>(x, cols, vec_ok != 0, m, s);
        block_merge<THREADS>(m, s, sm_m, sm_s);
        const float bias = fmaf(m, kLog2e, __log2f(s));
        TOut* p = P + row * cols;
        const long nvec = (cols + V - 1) / V;
        for (long vi = threadIdx.x; vi < nvec; vi += THREADS) {
            const long e0 = vi * V;
            float f[V];
            const int valid = (int)((cols - e0) < V ? (cols - e0) : V);
            if (vec_ok && valid == V) {
                Elem<TIn>::loadv(x + e0, f);
            } else {
                for (int i = 0; i < V; ++i) f[i] = i < valid ? Elem<TIn>::load1(x + e0 + i) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < V; ++i) f[i] = ex2(fmaf(f[i], kLog2e, -bias));
            store_out<TOut, V>(p + e0, f, vec_ok && valid == V, valid);
        }
        if (LSE != nullptr && threadIdx.x == 0) LSE[row] = m + logf(s);
    }
}

long grid_for_rows(long rows) {
    const long kMaxGrid = 1L << 30;
    return rows < kMaxGrid ? rows : kMaxGrid;
}

template <typename TIn, typename TOut>
cudaError_t softmax_dispatch(const TIn* X, TOut* P, float* LSE, long rows, long cols, cudaStream_t st) {
    constexpr int V = Elem<TIn>::kVec;
    const int vec_ok = (cols % V) == 0;
    const long nvec = (cols + V - 1) / V;
    const dim3 grid((unsigned)grid_for_rows(rows));
#define FA_RESIDENT(T, NVV) softmax_rows_resident<TIn, TOut, T, NVV><<<grid, T, 0, st>>>(X, P, LSE, rows, cols, vec_ok)
    if (nvec <= 32) FA_RESIDENT(32, 1);
    else if (nvec <= 64) FA_RESIDENT(32, 2);
    else if (nvec <= 128) FA_RESIDENT(32, 4);
    else if (nvec <= 256) FA_RESIDENT(32, 8);
    else if (nvec <= 512) FA_RESIDENT(64, 8);
    else if (nvec <= 1024) FA_RESIDENT(128, 8);
    else if (nvec <= 2048) FA_RESIDENT(256, 8);
    else if (nvec <= 4096) FA_RESIDENT(512, 8);
    else if (nvec <= 8192) FA_RESIDENT(1024, 8);
    else softmax_rows_stream<TIn, TOut, 512, 4><<<grid, 512, 0, st>>>(X, P, LSE, rows, cols, vec_ok);
#undef FA_RESIDENT
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t lse_dispatch(const TIn* X, float* LSE, long rows, long cols, cudaStream_t st) {
    constexpr int V = Elem<TIn>::kVec;
    const int vec_ok = (cols % V) == 0;
    const long nvec = (cols + V - 1) / V;
    const dim3 grid((unsigned)grid_for_rows(rows));
    if (nvec <= 128) logsumexp_rows_stream<TIn, 32, 4><<<grid, 32, 0, st>>>(X, LSE, rows, cols, vec_ok);
    else if (nvec <= 1024) logsumexp_rows_stream<TIn, 128, 4><<<grid, 128, 0, st>>>(X, LSE, rows, cols, vec_ok);
    else logsumexp_rows_stream<TIn, 512, 4><<<grid, 512, 0, st>>>(X, LSE, rows, cols, vec_ok);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_rows(const void* X, void* P, float* LSE, long rows, long cols, int in_bf16, int out_bf16,
                                cudaStream_t st) {
    using bf = __nv_bfloat16;
    if (in_bf16 && out_bf16)
        return softmax_dispatch((const bf*)X, (bf*)P, LSE, rows, cols, st);
    if (in_bf16)
        return softmax_dispatch((const bf*)X, (float*)P, LSE, rows, cols, st);
    if (out_bf16)
        return softmax_dispatch((const float*)X, (bf*)P, LSE, rows, cols, st);
    return softmax_dispatch((const float*)X, (float*)P, LSE, rows, cols, st);
}

cudaError_t launch_logsumexp_rows(const void* X, float* LSE, long rows, long cols, int in_bf16, cudaStream_t st) {
    if (in_bf16) return lse_dispatch((const __nv_bfloat16*)X, LSE, rows, cols, st);
    return lse_dispatch((const float*)X, LSE, rows, cols, st);
}

}  // namespace fa
