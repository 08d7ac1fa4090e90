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
// Pipelined kernel (rows of 8-64 KB whose byte length is a multiple of 16):
// persistent, one CTA per SM.  A producer warp streams whole rows into a ring
// of shared-memory stages with bulk TMA copies (mbarrier-tracked), so several
// rows are in flight per SM at all times; 16 consumer warps (one group, or
// four groups of 4 taking alternate rows when rows are 16 KB or shorter) take
// a row from shared memory into registers (128-bit loads), release the stage,
// compute exp once per element relative to their own max, merge (m, s)
// across the group and write P with 128-bit coalesced stores.  X is read from
// HBM once and P written once.
// Warp-per-row kernel (rows of whole 16-byte vectors up to 4 KB, 8 KB for
// log-sum-exp only): persistent warps, the next row loaded while the current
// one is reduced.
// Resident kernel (other row lengths up to 64K elements): one CTA per row,
// each thread holds its slice of the row in registers (NV 16-byte vectors),
// also one read and one write.
// Exponents are formed as (x - m) * log2 e, the difference first, so large
// logits keep their precision.
// Streaming kernels: rows longer than the resident capacity are reduced with
// the per-thread online update over 16-byte vectors (one read for LSE only,
// two reads when P is also written).
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>
#include <unordered_map>

#include "fattn_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2f = 0.6931471805599453f;

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

// Element-wise max of two bf16 pairs (exact: bf16 values order as their floats).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// -inf in every element of a 32-bit word: two bf16, or one fp32
template <typename T>
__host__ __device__ constexpr uint32_t neg_inf_word() {
    return sizeof(T) == 2 ? 0xFF80FF80u : 0xFF800000u;
}

// Packed fp32x2 a - b and a * b (round to nearest).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
// Max over a thread's packed slice: on bf16 pairs (exact), or on fp32 words.
template <typename TIn, int NV>
__device__ __forceinline__ float slice_max(const uint4* raw) {
    if constexpr (sizeof(TIn) == 2) {
        uint32_t mw[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
        for (int k = 1; k < NV; ++k) {
            mw[0] = bf16x2_max(mw[0], raw[k].x);
            mw[1] = bf16x2_max(mw[1], raw[k].y);
            mw[2] = bf16x2_max(mw[2], raw[k].z);
            mw[3] = bf16x2_max(mw[3], raw[k].w);
        }
        const uint32_t w = bf16x2_max(bf16x2_max(mw[0], mw[1]), bf16x2_max(mw[2], mw[3]));
        return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    } else {
        float mf[4] = {__uint_as_float(raw[0].x), __uint_as_float(raw[0].y), __uint_as_float(raw[0].z),
                       __uint_as_float(raw[0].w)};
#pragma unroll
        for (int k = 1; k < NV; ++k) {
            mf[0] = fmaxf(mf[0], __uint_as_float(raw[k].x));
            mf[1] = fmaxf(mf[1], __uint_as_float(raw[k].y));
            mf[2] = fmaxf(mf[2], __uint_as_float(raw[k].z));
            mf[3] = fmaxf(mf[3], __uint_as_float(raw[k].w));
        }
        return fmaxf(fmaxf(mf[0], mf[1]), fmaxf(mf[2], mf[3]));
    }
}

// Float pair e of a packed 16-byte vector: bf16 word e, or fp32 words 2e, 2e + 1.
template <typename TIn>
__device__ __forceinline__ float2 unpack_pair(const uint4& u, int e) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    if constexpr (sizeof(TIn) == 2) {
        return make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
    } else {
        return make_float2(__uint_as_float(w[2 * e]), __uint_as_float(w[2 * e + 1]));  // e < 2
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

// Row results of the log-sum-exp kernels: LSE (if wanted) and, for the fused
// cross-entropy, loss = LSE - x[label] (0 for a label outside [0, cols)).
template <typename TIn>
__device__ __forceinline__ void write_row_lse(const TIn* __restrict__ X, long row, long cols, float lse,
                                              float* __restrict__ LSE, const long long* __restrict__ labels,
                                              float* __restrict__ loss) {
    if (LSE != nullptr) LSE[row] = lse;
    if (loss != nullptr) {
        const long long lab = labels[row];
        loss[row] = (lab >= 0 && lab < cols) ? lse - Elem<TIn>::load1(X + row * cols + lab) : 0.f;
    }
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

// 16-byte vector vi of a row as packed words; elements past the row end (or
// the whole vector, when the row is not a whole number of vectors and this
// one is cut) are read one at a time, missing ones as -inf.
template <typename TIn>
__device__ __forceinline__ uint4 load_vec_packed(const TIn* __restrict__ x, long e0, long cols, bool vec_ok) {
    constexpr int V = Elem<TIn>::kVec;
    if (vec_ok && e0 + V <= cols) return __ldg(reinterpret_cast<const uint4*>(x + e0));
    uint32_t w[4];
    if constexpr (sizeof(TIn) == 2) {
        const unsigned short* xs = reinterpret_cast<const unsigned short*>(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = e0 + 2 * i < cols ? __ldg(xs + e0 + 2 * i) : 0xFF80u;
            const uint32_t hi = e0 + 2 * i + 1 < cols ? __ldg(xs + e0 + 2 * i + 1) : 0xFF80u;
            w[i] = lo | (hi << 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = e0 + i < cols ? __float_as_uint(__ldg(x + e0 + i)) : 0xFF800000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Block-wide max or sum of one float per thread; every thread gets the result.
template <int THREADS, bool MAX>
__device__ __forceinline__ float block_reduce(float v, float* sm) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
        v = MAX ? fmaxf(v, o) : v + o;
    }
    if constexpr (THREADS > 32) {
        constexpr int W = THREADS / 32;
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        if (lane == 0) sm[warp] = v;
        __syncthreads();
        v = lane < W ? sm[lane] : (MAX ? -CUDART_INF_F : 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v, off);
            v = MAX ? fmaxf(v, o) : v + o;
        }
        __syncthreads();  // the scratch may be reused next
    }
    return v;
}

// One CTA per row (grid-strided); the row lives in registers, packed.  Its
// max first (block-wide), then S = sum exp(x - M) (block-wide), then
// p = 2^((x - M) log2 e - log2 S) or log p = x - (M + ln S): the three passes
// of the safe softmax over registers, one read and one write of the row.
template <typename TIn, typename TOut, int THREADS, int NV, bool LOGP>
__global__ void __launch_bounds__(THREADS) softmax_rows_resident(const TIn* __restrict__ X, TOut* __restrict__ P,
                                                                 float* __restrict__ LSE, long rows, long cols,
                                                                 int vec_ok) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr int NP = V / 2;
    __shared__ float sm[32];
    for (long row = blockIdx.x; row < rows; row += gridDim.x) {
        const TIn* x = X + row * cols;
        uint4 raw[NV];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const long e0 = (long)(threadIdx.x + k * THREADS) * V;
            constexpr uint32_t ni = neg_inf_word<TIn>();
            raw[k] = e0 < cols ? load_vec_packed<TIn>(x, e0, cols, vec_ok != 0) : make_uint4(ni, ni, ni, ni);
        }
        const float M = block_reduce<THREADS, true>(slice_max<TIn, NV>(raw), sm);
        const float Mk = M == -CUDART_INF_F ? 0.f : M;  // a row of -inf only: S = 0
        const float2 mm = make_float2(Mk, Mk), kk2 = make_float2(kLog2e, kLog2e);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < NP; ++e) {
                const float2 t2 = mul2(sub2(unpack_pair<TIn>(raw[k], e), mm), kk2);
                acc = add2(acc, make_float2(ex2(t2.x), ex2(t2.y)));
            }
        const float S = block_reduce<THREADS, false>(acc.x + acc.y, sm);
        const float l2s = __log2f(S);
        const float lse_row = M + logf(S);
        TOut* p = P + row * cols;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const long e0 = (long)(threadIdx.x + k * THREADS) * V;
            if (e0 < cols) {
                float o[V];
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    const float2 x2 = unpack_pair<TIn>(raw[k], e);
                    o[2 * e] = LOGP ? x2.x - lse_row : ex2(fmaf(x2.x - Mk, kLog2e, -l2s));
                    o[2 * e + 1] = LOGP ? x2.y - lse_row : ex2(fmaf(x2.y - Mk, kLog2e, -l2s));
                }
                const int valid = (int)((cols - e0) < V ? (cols - e0) : V);
                store_out<TOut, V>(p + e0, o, vec_ok && valid == V, valid);
            }
        }
        if (LSE != nullptr && threadIdx.x == 0) LSE[row] = lse_row;
    }
}

// U strided 16-byte vectors of a row, packed (past the row end: -inf).
template <typename TIn, int THREADS, int U>
__device__ __forceinline__ void load_block_packed(const TIn* __restrict__ x, long base, long nvec, long cols,
                                                  bool vec_ok, uint4* buf) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr uint32_t ni = neg_inf_word<TIn>();
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const long vi = base + (long)u * THREADS;
        buf[u] = vi < nvec ? load_vec_packed<TIn>(x, vi * V, cols, vec_ok) : make_uint4(ni, ni, ni, ni);
    }
}

// Per-thread online (m, s) over a strided range of 16-byte vectors of a row:
// blocks of U vectors, the next block loaded while the current one is folded
// in (s <- s 2^(m - m') + sum 2^(x - m'), m' = max(m, block max)).
template <typename TIn, int THREADS, int U>
__device__ __forceinline__ void row_online_ms(const TIn* __restrict__ x, long cols, bool vec_ok, float& m, float& s) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr int NP = V / 2;
    constexpr long STEP = (long)THREADS * U;
    const long nvec = (cols + V - 1) / V;
    m = -CUDART_INF_F;
    s = 0.f;
    uint4 cur[U], nxt[U];
    long base = threadIdx.x;
    load_block_packed<TIn, THREADS, U>(x, base, nvec, cols, vec_ok, cur);
    for (; base < nvec; base += STEP) {
        load_block_packed<TIn, THREADS, U>(x, base + STEP, nvec, cols, vec_ok, nxt);
        const float bm = slice_max<TIn, U>(cur);
        if (bm != -CUDART_INF_F) {
            const float mn = fmaxf(m, bm);
            const float2 mm = make_float2(mn, mn), kk2 = make_float2(kLog2e, kLog2e);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    const float2 t2 = mul2(sub2(unpack_pair<TIn>(cur[u], e), mm), kk2);
                    acc = add2(acc, make_float2(ex2(t2.x), ex2(t2.y)));
                }
            s = s * ex2((m - mn) * kLog2e) + (acc.x + acc.y);  // m = -inf on the first block: 2^-inf = 0
            m = mn;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) cur[u] = nxt[u];
    }
}

template <typename TIn, int THREADS, int U>
__global__ void __launch_bounds__(THREADS) logsumexp_rows_stream(const TIn* __restrict__ X, float* __restrict__ LSE,
                                                                 long rows, long cols, int vec_ok,
                                                                 const long long* __restrict__ labels,
                                                                 float* __restrict__ loss) {
    __shared__ float sm_m[32], sm_s[32];
    for (long row = blockIdx.x; row < rows; row += gridDim.x) {
        float m, s;
        row_online_ms<TIn, THREADS, U>(X + row * cols, cols, vec_ok != 0, m, s);
        block_merge<THREADS>(m, s, sm_m, sm_s);
        if (threadIdx.x == 0) write_row_lse(X, row, cols, m + logf(s), LSE, labels, loss);
    }
}

// Rows longer than the resident capacity: online reduction pass, then a second
// read of the row to write P.
template <typename TIn, typename TOut, int THREADS, int U, bool LOGP>
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
        const float l2s = __log2f(s);
        const float lse_row = m + logf(s);
        TOut* p = P + row * cols;
        const long nvec = (cols + V - 1) / V;
        // second read of the row, U vectors in flight per thread
        for (long base = threadIdx.x; base < nvec; base += (long)THREADS * U) {
            uint4 raw[U];
            load_block_packed<TIn, THREADS, U>(x, base, nvec, cols, vec_ok != 0, raw);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const long vi = base + (long)u * THREADS;
                if (vi < nvec) {
                    const long e0 = vi * V;
                    float o[V];
#pragma unroll
                    for (int e = 0; e < V / 2; ++e) {
                        const float2 x2 = unpack_pair<TIn>(raw[u], e);
                        o[2 * e] = LOGP ? x2.x - lse_row : ex2(fmaf(x2.x - m, kLog2e, -l2s));
                        o[2 * e + 1] = LOGP ? x2.y - lse_row : ex2(fmaf(x2.y - m, kLog2e, -l2s));
                    }
                    const int valid = (int)((cols - e0) < V ? (cols - e0) : V);
                    store_out<TOut, V>(p + e0, o, vec_ok && valid == V, valid);
                }
            }
        }
        if (LSE != nullptr && threadIdx.x == 0) LSE[row] = m + logf(s);
    }
}


// ------------------------------------------------------------------ pipelined
constexpr int kTmaConsumers = 512;                 // 16 consumer warps
constexpr int kTmaThreads = kTmaConsumers + 32;    // + 1 producer warp
constexpr int kTmaMaxStages = 8;
constexpr uint32_t kTmaSmemBudget = 200 * 1024;
constexpr uint32_t kTmaBarBytes = 384;             // full[8], empty[8], red[8], rowq[16]
constexpr uint32_t kTmaSmemExtra = 128 /* alignment */ + kTmaBarBytes + 2 * 16 * 8 /* (m, s) slots */ + 16;
// With tail rows the barrier area also holds the row index of each item in
// the ring, after red[8]: item i's in rowq[i % kRowq].  The producer writes
// item i + kRowq's entry only once item i + kRowq - nst has been taken, and
// that item belongs to the same consumer group as item i (nst and kRowq are
// multiples of the group count) and comes after it, so a group may read its
// item's entry again until the end of that item.
constexpr int kRowq = 16;
constexpr uint32_t kTmaRowqOffset = 8u * (2 * kTmaMaxStages + 8);
static_assert(kTmaRowqOffset + 8u * kRowq <= kTmaBarBytes, "barrier area");
static_assert(kRowq > kTmaMaxStages && kRowq % 4 == 0, "row index ring");

// ------------------------------------------------------------------ tail rows
// Under full load the SMs do not stream at one rate (the row count an SM gets
// through in a fixed time varies by about +-8 %), so with a purely static
// split the slowest SM's rows set the end of the kernel.  The LSE kernel on
// rows above 16 KB and the softmax kernel on rows of 8-16 KB (where measured
// faster) therefore take their first rounds of rows statically (row
// blockIdx.x + j * gridDim.x) and the last kTailRounds rounds of 64 KB per CTA
// a chunk of rows per request from a counter, so that the faster SMs take more
// of the tail.
//
// A counter is one word of g_tail_ctr, (CTAs done << 32) | next row; it is
// zero when a launch starts.  Every CTA requests rows until the range is
// exhausted, then counts itself done; the CTA that counts gridDim.x zeroes
// the word again.  Each stream has a word of its own, so launches that share
// a word run one after another (see launch_tail).
constexpr int kTailSlots = 256;
constexpr int kTailRounds = 8;
__device__ unsigned long long g_tail_ctr[kTailSlots];

// The producer lane of the pipelined kernels with tail rows: rows into the
// ring of `nst` stages (item i's row index in rowq[i % kRowq]), then one end
// marker (row -1) per consumer group, so that every group's last item is its
// marker.  `tail`: the launch's counter (null: a static split of every row).
template <typename TIn>
__device__ __forceinline__ void produce_rows(const TIn* __restrict__ X, long rows, long cols, uint32_t base,
                                             uint32_t stage_bytes, int nst, int ng, uint32_t bar0, long long* rowq,
                                             volatile int* abort_flag, int* status,
                                             unsigned long long* __restrict__ tail) {
    const uint64_t pol = l2_policy_evict_first();  // every row is read exactly once
    const uint32_t row_bytes = (uint32_t)(cols * (long)sizeof(TIn));
    long issued = 0;
    bool live = true;
    // one item into the next stage: a row, or an end marker (r < 0)
    auto push = [&](long r) {
        if (!live) return;
        const int s = (int)(issued % nst);
        const uint32_t ph = (uint32_t)(issued / nst) & 1u;
        const uint32_t fb = bar0 + 8u * (uint32_t)s;
        if (!mbar_wait_bounded(bar0 + 8u * (uint32_t)(kTmaMaxStages + s), ph ^ 1u, abort_flag, kWaitLimitNs)) {
            *abort_flag = 1;
            atomicExch(status, kDevStatusTimeout);
            live = false;
            return;
        }
        rowq[issued % kRowq] = r;
        ++issued;
        if (r < 0) {
            mbar_arrive(fb);
            return;
        }
        mbar_expect_tx(fb, row_bytes);
        const char* src = reinterpret_cast<const char*>(X + r * cols);
        const uint32_t dst = base + (uint32_t)s * stage_bytes;
        for (uint32_t off = 0; off < row_bytes; off += 32768u) {
            const uint32_t n = row_bytes - off < 32768u ? row_bytes - off : 32768u;
            bulk_load(dst + off, src + off, n, fb, pol);
        }
    };
    const long G = gridDim.x, b = blockIdx.x;
    if (tail == nullptr) {
        for (long r = b; r < rows; r += G) push(r);
    } else {
        // a request takes c consecutive rows (about 64 KB, so that the
        // request's round trip stays below the time the rows take); static
        // rounds: all whole rounds but the last kTailRounds * c, and at least
        // the ring's depth; then chunks n of rows r0 + n c .. on request
        const long c = row_bytes >= 65536u ? 1 : 65536 / (long)row_bytes;
        const long per = rows / G;
        long ns = per - kTailRounds * c;
        if (ns < (per < nst ? per : nst)) ns = per < nst ? per : nst;
        const long r0 = ns * G, nd = (rows - r0 + c - 1) / c;
        if (nd > 0) {
            unsigned long long nxt = atomicAdd(tail, 1ull);  // one request ahead
            for (long j = 0; j < ns; ++j) push(b + j * G);
            for (;;) {
                const long n = (long)(uint32_t)nxt;
                if (n >= nd || !live) break;
                nxt = atomicAdd(tail, 1ull);
                const long e = r0 + (n + 1) * c < rows ? r0 + (n + 1) * c : rows;
                for (long r = r0 + n * c; r < e; ++r) push(r);
            }
            // (also after a timeout: the word must be zero for the next launch)
            const unsigned long long done = atomicAdd(tail, 1ull << 32);
            if ((long)(done >> 32) == G - 1) atomicExch(tail, 0ull);
        } else {
            for (long j = 0; j < ns; ++j) push(b + j * G);
        }
    }
    for (int g = 0; g < ng; ++g) push(-1);
    // drain: the copies this thread issued have landed before it exits
    for (long i = issued - nst < 0 ? 0 : issued - nst; i < issued; ++i)
        mbar_wait_bounded(bar0 + 8u * (uint32_t)(i % nst), (uint32_t)(i / nst) & 1u, nullptr, kWaitLimitNs);
}


// One CTA per SM; rows r = blockIdx.x + i * gridDim.x go through a ring of
// `nst` shared-memory stages of `stage_bytes` each.  The 16 consumer warps
// form NG groups; group g takes rows i = g, g + NG, ... (whole rows: 64 KB
// for one group of 16 warps, 32 KB for two of 8, 16 KB for four of 4), so
// that one group's cross-warp merge overlaps the others' work on shorter
// rows.  nst is a multiple of NG: stage s only ever holds rows of group
// s % NG, which consumes its stages' phases in order.
// PACKED: the slice stays packed until the exponent pass, which runs on
// fp32 pairs (faster with four or more stages in the ring; with three, at
// 64 KB rows, the unpacked form is).
// TAIL: the last rounds of rows come from the launch's counter `tail` (see
// produce_rows); the ring then carries each item's row index.
template <typename TIn, typename TOut, bool WRITE_P, int NV, bool LOGP, bool PACKED, int NG, bool TAIL>
__global__ void __launch_bounds__(kTmaThreads, 1)
softmax_rows_tma(const TIn* __restrict__ X, TOut* __restrict__ P, float* __restrict__ LSE, long rows, long cols,
                 uint32_t stage_bytes, int nst, int* status, unsigned long long* __restrict__ tail) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr int W = kTmaConsumers / 32;
    constexpr int WG = W / NG;              // warps per group
    constexpr int GT = kTmaConsumers / NG;  // threads per group
    static_assert(NG == 1 || NG == 2 || NG == 4, "consumer groups");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    uint8_t* gbase = smem_raw + (base - raw);
    // after the stages: mbarriers, then the (m, s) slots [NG][2][WG], then the abort flag
    const uint32_t bar0 = base + (uint32_t)nst * stage_bytes;
    float2* red = reinterpret_cast<float2*>(gbase + (uint32_t)nst * stage_bytes + kTmaBarBytes);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + 2 * W);
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(kTmaMaxStages + s); };
    auto red_bar = [&](int g) { return bar0 + 8u * (uint32_t)(2 * kTmaMaxStages + g); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t row_bytes = (uint32_t)(cols * (long)sizeof(TIn));
    const long nvec = cols / V;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), WG);  // released by the group that owns the stage
        }
        for (int g = 0; g < NG; ++g) mbar_init(red_bar(g), WG);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    long long* rowq = reinterpret_cast<long long*>(gbase + (uint32_t)nst * stage_bytes + kTmaRowqOffset);
    if (warp == W) {
        // ------------------------------------------------ producer
        if constexpr (TAIL) {
            if (lane == 0)
                produce_rows<TIn>(X, rows, cols, base, stage_bytes, nst, NG, bar0, rowq, abort_flag, status, tail);
            return;
        }
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();  // every row is read exactly once
            long issued = 0;
            for (long r = blockIdx.x; r < rows; r += gridDim.x, ++issued) {
                const int s = (int)(issued % nst);
                const uint32_t ph = (uint32_t)(issued / nst) & 1u;
                if (!mbar_wait_bounded(empty(s), ph ^ 1u, abort_flag, kWaitLimitNs)) {
                    *abort_flag = 1;
                    atomicExch(status, kDevStatusTimeout);
                    break;
                }
                mbar_expect_tx(full(s), row_bytes);
                const char* src = reinterpret_cast<const char*>(X + r * cols);
                const uint32_t dst = base + (uint32_t)s * stage_bytes;
                for (uint32_t off = 0; off < row_bytes; off += 32768u) {
                    const uint32_t n = row_bytes - off < 32768u ? row_bytes - off : 32768u;
                    bulk_load(dst + off, src + off, n, full(s), pol);
                }
            }
            // drain: the copies this thread issued have landed before it exits
            for (long i = issued - nst < 0 ? 0 : issued - nst; i < issued; ++i)
                mbar_wait_bounded(full((int)(i % nst)), (uint32_t)(i / nst) & 1u, nullptr, kWaitLimitNs);
        }
        return;
    }

    // ---------------------------------------------------- consumers
    const float kc = kLog2e;
    const int g = NG == 1 ? 0 : warp / WG;                              // consumer group
    const int gw = NG == 1 ? warp : warp % WG;                          // warp within the group
    const int gt = NG == 1 ? (int)threadIdx.x : (int)threadIdx.x % GT;  // thread within the group
    // item i of this CTA is the group's (i / NG)-th; static split: row
    // blockIdx.x + i * gridDim.x; with TAIL the ring holds each item's row,
    // and a row < 0 ends the group's work
    for (long i = g, r = blockIdx.x + (long)g * gridDim.x; TAIL || r < rows; i += NG, r += (long)NG * gridDim.x) {
        const int s = (int)(i % nst);
        const uint32_t ph = (uint32_t)(i / nst) & 1u;
        bool ok = mbar_wait_bounded(full(s), ph, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(status, kDevStatusTimeout);
            break;
        }
        if (TAIL && rowq[i % kRowq] < 0) break;
        // the row slice into registers, then the stage goes back to the
        // producer; v becomes exp(x - m) for this thread's max m (log p keeps
        // x itself).  A slice that is all -inf (masked logits) takes m = 0 for
        // the exponent, so every p = exp(-inf) = 0 and the sum is 0.
        const TIn* srow = reinterpret_cast<const TIn*>(gbase + (uint32_t)s * stage_bytes);
        float v[NV][V];
        float m, sum;
        if constexpr (PACKED) {
            // loaded packed; the max on the packed words (bf16 pairs: exact),
            // the exponent arguments two lanes at a time
            uint4 raw[NV];
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const long vi = gt + (long)k * GT;
                constexpr uint32_t ni = neg_inf_word<TIn>();
                raw[k] = vi < nvec ? *reinterpret_cast<const uint4*>(srow + vi * V) : make_uint4(ni, ni, ni, ni);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            m = slice_max<TIn, NV>(raw);
            const float mk = m == -CUDART_INF_F ? 0.f : m;
            const float2 mm = make_float2(mk, mk), kk2 = make_float2(kc, kc);
            float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                    float2 x2;
                    if constexpr (V == 8) {
                        x2 = make_float2(__uint_as_float(w[e / 2] << 16), __uint_as_float(w[e / 2] & 0xFFFF0000u));
                    } else {
                        x2 = make_float2(__uint_as_float(w[e]), __uint_as_float(w[e + 1]));
                    }
                    const float2 t2 = mul2(sub2(x2, mm), kk2);
                    const float2 ex = make_float2(ex2(t2.x), ex2(t2.y));
                    v[k][e] = LOGP ? x2.x : ex.x;
                    v[k][e + 1] = LOGP ? x2.y : ex.y;
                    acc[(e / 2) & 1] = add2(acc[(e / 2) & 1], ex);
                }
            }
            const float2 a2 = add2(acc[0], acc[1]);
            sum = a2.x + a2.y;
        } else {
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const long vi = gt + (long)k * GT;
                if (vi < nvec) {
                    const uint4 u = *reinterpret_cast<const uint4*>(srow + vi * V);
                    if constexpr (V == 8) {
                        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[k][2 * e] = __uint_as_float(w[e] << 16);
                            v[k][2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                        }
                    } else {
                        v[k][0] = __uint_as_float(u.x); v[k][1] = __uint_as_float(u.y);
                        v[k][2] = __uint_as_float(u.z); v[k][3] = __uint_as_float(u.w);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < V; ++e) v[k][e] = -CUDART_INF_F;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
            m = -CUDART_INF_F;
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) m = fmaxf(m, v[k][e]);
            const float mk = m == -CUDART_INF_F ? 0.f : m;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < V; ++e) {
                    const float ex = ex2((v[k][e] - mk) * kc);
                    if (WRITE_P && !LOGP) v[k][e] = ex;
                    acc[e & 3] += ex;
                }
            sum = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
        // merge (m, s): within the warp, then the group's warps through shared memory
        float M = m, S = sum;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, M, off);
            const float s2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
            merge_ms(M, S, m2, s2);
        }
        // (a bounded mbarrier exchange rather than a named barrier, so a warp
        // that gave up can never leave the others waiting forever)
        float2* slot = red + (g * 2 + ((i / NG) & 1)) * WG;
        if (lane == 0) slot[gw] = make_float2(M, S);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_bar(g));
        ok = mbar_wait_bounded(red_bar(g), (uint32_t)((i / NG) & 1), abort_flag, kWaitLimitNs);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(status, kDevStatusTimeout);
            break;
        }
        {
            const float2 a = slot[lane & (WG - 1)];
            M = a.x;
            S = a.y;
#pragma unroll
            for (int off = WG / 2; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(0xFFFFFFFFu, M, off);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
                merge_ms(M, S, m2, s2);
            }
        }
        const long row = TAIL ? (long)rowq[i % kRowq] : r;
        if (WRITE_P) {
            // p = exp(x - m) * exp(m - M) / S;  log p = x - (M + ln S)
            const float f = m == -CUDART_INF_F ? 0.f : ex2((m - M) * kc) / S;
            const float lse_row = M + logf(S);
            TOut* prow = P + row * cols;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const long vi = gt + (long)k * GT;
                if (vi < nvec) {
                    float o[V];
#pragma unroll
                    for (int e = 0; e < V; ++e) o[e] = LOGP ? v[k][e] - lse_row : v[k][e] * f;
                    store_out<TOut, V>(prow + vi * V, o, true, V);
                }
            }
        }
        if (LSE != nullptr && gt == 0) LSE[row] = M + logf(S);
    }
}


// LSE only, pipelined: the same producer as softmax_rows_tma, but the
// consumer warps form NG groups that take rows in turn, so that one group's
// merge latency overlaps the others' arithmetic.  The stage count is a
// multiple of NG, so stage s only ever holds rows of group s % NG and each
// group consumes its stages' phases in order (a group can never run a phase
// ahead on a stage another group still owns).  A group copies its row slice into registers (packed), releases the
// stage, takes the slice max on the packed values and sums one exponential
// per element relative to it.
// NG consumer groups: two of 8 warps for rows above 16 KB, eight of 2 warps
// (one stage each) for rows of 8-16 KB.  NV: 16-byte vectors per thread (the
// slots past the row end hold -inf).
// TAIL: the last rounds of rows come from the launch's counter `tail` (see
// produce_rows); the ring then carries each item's row index.
template <typename TIn, int NV, int NG, bool TAIL>
__global__ void __launch_bounds__(kTmaThreads, 1)
logsumexp_rows_tma(const TIn* __restrict__ X, float* __restrict__ LSE, long rows, long cols, uint32_t stage_bytes,
                   int nst, int* status, const long long* __restrict__ labels, float* __restrict__ loss,
                   unsigned long long* __restrict__ tail) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr int GT = kTmaConsumers / NG;     // threads per group
    constexpr int WG = GT / 32;                // warps per group
    static_assert(NG == 2 || NG == 4 || NG == 8, "consumer groups");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 127u) & ~127u;
    uint8_t* gbase = smem_raw + (base - raw);
    // after the stages: full[], empty[] (kTmaMaxStages each), red[NG]; then (m, s) slots [group][2][WG]; then the abort flag
    const uint32_t bar0 = base + (uint32_t)nst * stage_bytes;
    float2* red = reinterpret_cast<float2*>(gbase + (uint32_t)nst * stage_bytes + kTmaBarBytes);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red + NG * 2 * WG);
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(kTmaMaxStages + s); };
    auto red_bar = [&](int g) { return bar0 + 8u * (uint32_t)(2 * kTmaMaxStages + g); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t row_bytes = (uint32_t)(cols * (long)sizeof(TIn));
    const long nvec = cols / V;
    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), WG);  // released by the group that owns the stage
        }
        for (int g = 0; g < NG; ++g) mbar_init(red_bar(g), WG);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    long long* rowq = reinterpret_cast<long long*>(gbase + (uint32_t)nst * stage_bytes + kTmaRowqOffset);
    if (warp == kTmaConsumers / 32) {
        if constexpr (TAIL) {
            if (lane == 0)
                produce_rows<TIn>(X, rows, cols, base, stage_bytes, nst, NG, bar0, rowq, abort_flag, status, tail);
            return;
        }
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            long issued = 0;
            for (long r = blockIdx.x; r < rows; r += gridDim.x, ++issued) {
                const int s = (int)(issued % nst);
                const uint32_t ph = (uint32_t)(issued / nst) & 1u;
                if (!mbar_wait_bounded(empty(s), ph ^ 1u, abort_flag, kWaitLimitNs)) {
                    *abort_flag = 1;
                    atomicExch(status, kDevStatusTimeout);
                    break;
                }
                mbar_expect_tx(full(s), row_bytes);
                const char* src = reinterpret_cast<const char*>(X + r * cols);
                const uint32_t dst = base + (uint32_t)s * stage_bytes;
                for (uint32_t off = 0; off < row_bytes; off += 32768u) {
                    const uint32_t n = row_bytes - off < 32768u ? row_bytes - off : 32768u;
                    bulk_load(dst + off, src + off, n, full(s), pol);
                }
            }
            for (long i = issued - nst < 0 ? 0 : issued - nst; i < issued; ++i)
                mbar_wait_bounded(full((int)(i % nst)), (uint32_t)(i / nst) & 1u, nullptr, kWaitLimitNs);
        }
        return;
    }

    const int g = warp / WG;                        // consumer group
    const int gw = warp % WG;                       // warp within the group
    const int gt = threadIdx.x % GT;                // thread within the group
    const float2 cc = make_float2(kLog2e, kLog2e);
    long k = 0;                                     // rows this group has done
    // (static split: item i is row blockIdx.x + i * gridDim.x; with TAIL the
    // ring holds each item's row, and a row < 0 ends the group's work)
    for (long i = g; TAIL || blockIdx.x + i * (long)gridDim.x < rows; i += NG, ++k) {
        const int s = (int)(i % nst);
        const uint32_t ph = (uint32_t)(i / nst) & 1u;
        bool ok = mbar_wait_bounded(full(s), ph, abort_flag, kWaitLimitNs);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(status, kDevStatusTimeout);
            break;
        }
        if (TAIL && rowq[i % kRowq] < 0) break;
        // this thread's slice, still packed, into registers; the stage goes
        // back to the producer as soon as it is loaded
        const TIn* srow = reinterpret_cast<const TIn*>(gbase + (uint32_t)s * stage_bytes);
        uint4 raw[NV];
#pragma unroll
        for (int kk = 0; kk < NV; ++kk) {
            const long vi = gt + (long)kk * GT;
            // (past the row end: -inf, which neither the max nor the sum sees)
            constexpr uint32_t ni = neg_inf_word<TIn>();
            raw[kk] = vi < nvec ? *reinterpret_cast<const uint4*>(srow + vi * V) : make_uint4(ni, ni, ni, ni);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        // the slice max first (bf16: on the packed pairs), then one exponential
        // per element relative to it
        float m;
        if constexpr (V == 8) {
            uint32_t mw[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
            for (int kk = 1; kk < NV; ++kk) {
                mw[0] = bf16x2_max(mw[0], raw[kk].x);
                mw[1] = bf16x2_max(mw[1], raw[kk].y);
                mw[2] = bf16x2_max(mw[2], raw[kk].z);
                mw[3] = bf16x2_max(mw[3], raw[kk].w);
            }
            const uint32_t w = bf16x2_max(bf16x2_max(mw[0], mw[1]), bf16x2_max(mw[2], mw[3]));
            m = fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
        } else {
            float mf[4] = {__uint_as_float(raw[0].x), __uint_as_float(raw[0].y), __uint_as_float(raw[0].z),
                           __uint_as_float(raw[0].w)};
#pragma unroll
            for (int kk = 1; kk < NV; ++kk) {
                mf[0] = fmaxf(mf[0], __uint_as_float(raw[kk].x));
                mf[1] = fmaxf(mf[1], __uint_as_float(raw[kk].y));
                mf[2] = fmaxf(mf[2], __uint_as_float(raw[kk].z));
                mf[3] = fmaxf(mf[3], __uint_as_float(raw[kk].w));
            }
            m = fmaxf(fmaxf(mf[0], mf[1]), fmaxf(mf[2], mf[3]));
        }
        float sum = 0.f;
        if (m != -CUDART_INF_F) {
            // only the sum is kept, so the exponent is one packed FMA:
            // x log2e - m log2e (enough precision for log-sum-exp)
            const float2 nmc = make_float2(-m * kLog2e, -m * kLog2e);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int kk = 0; kk < NV; ++kk) {
                const uint32_t w[4] = {raw[kk].x, raw[kk].y, raw[kk].z, raw[kk].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float2 x2;
                    if constexpr (V == 8) {
                        x2 = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xFFFF0000u));
                    } else {
                        if (e & 1) continue;
                        x2 = make_float2(__uint_as_float(w[e]), __uint_as_float(w[e + 1]));
                    }
                    const float2 t2 = fma2(x2, cc, nmc);
                    acc[e] = add2(acc[e], make_float2(ex2(t2.x), ex2(t2.y)));
                }
            }
            const float2 a2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
            sum = a2.x + a2.y;
        }
        // warp merge in two passes: the max first (no exponentials in the
        // shuffle chain), then every lane's sum rescaled to it once and added
        float wm = m;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, off));
        float ws = wm == -CUDART_INF_F ? 0.f : sum * ex2((m - wm) * kLog2e);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xFFFFFFFFu, ws, off);
        m = wm;
        sum = ws;
        float2* slot = red + (g * 2 + (k & 1)) * WG;
        if (lane == 0) slot[gw] = make_float2(m, sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(red_bar(g));
        ok = mbar_wait_bounded(red_bar(g), (uint32_t)(k & 1), abort_flag, kWaitLimitNs);
        ok = __all_sync(0xFFFFFFFFu, ok);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(status, kDevStatusTimeout);
            break;
        }
        if (gw == 0) {
            // the same two passes over the group's WG warp results
            const float2 a = slot[lane & (WG - 1)];
            float M = a.x;
#pragma unroll
            for (int off = WG / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
            float S = M == -CUDART_INF_F ? 0.f : a.y * ex2((a.x - M) * kLog2e);
#pragma unroll
            for (int off = WG / 2; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
            if (lane == 0) {
                const long r = TAIL ? (long)rowq[i % kRowq] : blockIdx.x + i * (long)gridDim.x;
                write_row_lse(X, r, cols, M + __log2f(S) * kLn2f, LSE, labels, loss);
            }
        }
    }
}

int device_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
}

// Counter slots for the tail rows, per device: each CUDA stream (by its id,
// which a context never reuses) gets a slot of its own the first time it
// launches a pipelined kernel with tail rows, and keeps it.  Launches on one stream run one
// after another, each starting with the word its predecessor zeroed, so a
// slot never serves two launches at once.  Streams beyond kTailSlots keep the
// static split.
struct TailSlots {
    std::mutex mu;
    bool ready = false;
    unsigned long long* words = nullptr;  // device address of g_tail_ctr
    std::unordered_map<unsigned long long, int> slot_of;  // stream id -> slot
};
constexpr int kTailMaxDevices = 64;

// Run `launch(tail)` with the stream's counter when the caller wants tail rows
// (`want`), the input is at least 16 MB and the stream is not being captured
// (the replays of a captured graph could overlap launches on the stream);
// otherwise `launch(nullptr)`, a static split.  Returns the launch's error.
template <typename F>
cudaError_t launch_tail(cudaStream_t st, bool want, long rows, long row_bytes, F&& launch) {
    if (!want || rows * row_bytes < (16L << 20)) return launch(nullptr);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return launch(nullptr);
    }
    if (cs != cudaStreamCaptureStatusNone) return launch(nullptr);  // (no other query on a capturing stream)
    // (relaxed capture mode for the queries below, so that they cannot upset a
    // capture that another thread runs in global mode)
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    unsigned long long sid = 0;
    int dev = -1;
    const bool ok = cudaStreamGetId(st, &sid) == cudaSuccess && cudaGetDevice(&dev) == cudaSuccess && dev >= 0 &&
                    dev < kTailMaxDevices;
    static TailSlots slots[kTailMaxDevices];
    unsigned long long* tail = nullptr;
    if (ok) {
        TailSlots& ts = slots[dev];
        std::lock_guard<std::mutex> lock(ts.mu);
        if (!ts.ready) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_tail_ctr) == cudaSuccess) {
                ts.words = static_cast<unsigned long long*>(p);
                ts.ready = true;
            }
        }
        if (ts.ready) {
            auto it = ts.slot_of.find(sid);
            if (it != ts.slot_of.end()) {
                tail = ts.words + it->second;
            } else if ((int)ts.slot_of.size() < kTailSlots) {
                const int k = (int)ts.slot_of.size();
                ts.slot_of.emplace(sid, k);
                tail = ts.words + k;
            }
        }
    }
    (void)cudaGetLastError();  // (a failed query above is not the launch's error)
    cudaThreadExchangeStreamCaptureMode(&mode);
    return launch(tail);
}

// Launch the pipelined kernel if the row shape suits it; returns false if not.
template <typename TIn, typename TOut, bool WRITE_P, bool LOGP>
bool try_launch_tma(const TIn* X, TOut* P, float* LSE, long rows, long cols, int* status, cudaStream_t st,
                    cudaError_t* err) {
    constexpr int V = Elem<TIn>::kVec;
    const long row_bytes = cols * (long)sizeof(TIn);
    if (cols % V != 0 || row_bytes < 8192 || row_bytes > 65536 || rows < 64) return false;
    const long nvec = cols / V;
    // consumer groups: one for rows above 16 KB, four (of 4 warps) up to 16 KB
    const int ng = row_bytes > 16384 ? 1 : 4;
    const uint32_t stage = (uint32_t)((row_bytes + 127) / 128 * 128);
    // (one group: at most four stages, as measured best; four groups: two each)
    const int max_st = ng == 1 ? 4 : kTmaMaxStages;
    int nst = (int)(kTmaSmemBudget / stage);
    nst = nst > max_st ? max_st : nst;
    nst -= nst % ng;  // stage s belongs to group s % ng
    const uint32_t smem = (uint32_t)nst * stage + kTmaSmemExtra;
    const long grid = rows < device_sms() ? rows : device_sms();
    auto launch = [&](auto kern, unsigned long long* tail) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) {
            kern<<<(unsigned)grid, kTmaThreads, smem, st>>>(X, P, LSE, rows, cols, stage, nst, status, tail);
            e = cudaGetLastError();
        }
        return e;
    };
    if (ng == 4 && nvec <= 4L * (kTmaConsumers / 4)) {  // up to 8 KB
        *err = launch(softmax_rows_tma<TIn, TOut, WRITE_P, 4, LOGP, true, 4, false>, nullptr);
    } else if (ng == 4) {
        // rows of 8-16 KB: tail rows when the static rounds are at least half
        // of every CTA's rows (shorter rows, and one group of 16 warps on
        // longer ones: a static split measured as fast or faster)
        const bool tail_ok = rows / grid >= 2L * kTailRounds * (65536 / row_bytes);
        *err = launch_tail(st, tail_ok, rows, row_bytes, [&](unsigned long long* tail) {
            return tail ? launch(softmax_rows_tma<TIn, TOut, WRITE_P, 8, LOGP, true, 4, true>, tail)
                        : launch(softmax_rows_tma<TIn, TOut, WRITE_P, 8, LOGP, true, 4, false>, nullptr);
        });
    } else if (nvec <= 4L * kTmaConsumers) {  // up to 32 KB: four stages
        *err = launch(softmax_rows_tma<TIn, TOut, WRITE_P, 4, LOGP, true, 1, false>, nullptr);
    } else if (nst >= 4) {
        *err = launch(softmax_rows_tma<TIn, TOut, WRITE_P, 8, LOGP, true, 1, false>, nullptr);
    } else {
        *err = launch(softmax_rows_tma<TIn, TOut, WRITE_P, 8, LOGP, false, 1, false>, nullptr);
    }
    return true;
}


// Launch the pipelined LSE-only kernel if the row shape suits it.
template <typename TIn>
bool try_launch_lse_tma(const TIn* X, float* LSE, long rows, long cols, int* status, cudaStream_t st,
                        cudaError_t* err, const long long* labels, float* loss) {
    constexpr int V = Elem<TIn>::kVec;
    const long row_bytes = cols * (long)sizeof(TIn);
    if (cols % V != 0 || row_bytes < 8192 || row_bytes > 65536 || rows < 64) return false;
    const long nvec = cols / V;
    // consumer groups: two above 16 KB (at most four stages), eight up to 16 KB
    // (eight stages, one per group; 2.5-4 % faster than four groups of 4)
    const int ng = row_bytes > 16384 ? 2 : 8;
    const int max_st = ng == 2 ? 4 : kTmaMaxStages;
    const uint32_t stage = (uint32_t)((row_bytes + 127) / 128 * 128);
    int nst = (int)(kTmaSmemBudget / stage);
    nst = nst > max_st ? max_st : nst;
    nst -= nst % ng;  // stage s belongs to consumer group s % ng
    const uint32_t smem = (uint32_t)nst * stage + kTmaSmemExtra;
    const long grid = rows < device_sms() ? rows : device_sms();
    auto launch = [&](auto kern, unsigned long long* tail) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess) {
            kern<<<(unsigned)grid, kTmaThreads, smem, st>>>(X, LSE, rows, cols, stage, nst, status, labels, loss,
                                                             tail);
            e = cudaGetLastError();
        }
        return e;
    };
    if (ng == 8) {
        // (rows up to 16 KB: a static split measured faster)
        if (nvec <= 8L * (kTmaConsumers / 8)) *err = launch(logsumexp_rows_tma<TIn, 8, 8, false>, nullptr);
        else if (nvec <= 12L * (kTmaConsumers / 8)) *err = launch(logsumexp_rows_tma<TIn, 12, 8, false>, nullptr);
        else *err = launch(logsumexp_rows_tma<TIn, 16, 8, false>, nullptr);
        return true;
    }
    // tail rows when the static rounds are at least half of every CTA's rows
    // (fewer rounds: the requests cost more than the balance gains)
    const long chunk = row_bytes >= 65536 ? 1 : 65536 / row_bytes;
    const bool tail_ok = rows / grid >= 2L * kTailRounds * chunk;
    *err = launch_tail(st, tail_ok, rows, row_bytes, [&](unsigned long long* tail) {
        if (nvec <= 8L * (kTmaConsumers / 2))
            return tail ? launch(logsumexp_rows_tma<TIn, 8, 2, true>, tail)
                        : launch(logsumexp_rows_tma<TIn, 8, 2, false>, nullptr);
        return tail ? launch(logsumexp_rows_tma<TIn, 16, 2, true>, tail)
                    : launch(logsumexp_rows_tma<TIn, 16, 2, false>, nullptr);
    });
    return true;
}

// ------------------------------------------------------------------ warp per row
// Rows of at most 256 16-byte vectors (4 KB; 8 KB for log-sum-exp only): one
// warp per row, persistent over rows, with the next row's slice loaded while
// the current one is reduced.  The whole row is in the warp's registers, so
// the row max is known before any exponential and the sum is taken once
// against it: pass 1 the max (bf16: on the packed pairs), pass 2
// S = sum exp(x - M), pass 3 (with P) p = 2^((x - M) log2 e - log2 S) or
// log p = x - (M + ln S).
// KIND: 0 softmax (P, LSE), 1 log-softmax (log p, LSE), 2 log-sum-exp only
// (LSE and / or the fused cross-entropy loss).
constexpr int kWarpRowThreads = 256;

template <typename TIn, int NV>
__device__ __forceinline__ void warp_row_load(const TIn* __restrict__ X, long row, long rows, long cols, long nvec,
                                              int lane, uint4* buf) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr uint32_t ni = neg_inf_word<TIn>();
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const long vi = lane + 32L * k;
        buf[k] = (row < rows && vi < nvec) ? __ldg(reinterpret_cast<const uint4*>(X + row * cols + vi * V))
                                           : make_uint4(ni, ni, ni, ni);
    }
}

template <typename TIn, typename TOut, int NV, int KIND>
__global__ void __launch_bounds__(kWarpRowThreads)
softmax_rows_warp(const TIn* __restrict__ X, TOut* __restrict__ P, float* __restrict__ LSE, long rows, long cols,
                  const long long* __restrict__ labels, float* __restrict__ loss) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr int NP = V / 2;  // float pairs per vector
    const long nvec = cols / V;
    const int lane = threadIdx.x & 31;
    const long nwarps = ((long)gridDim.x * kWarpRowThreads) >> 5;
    long row = ((long)blockIdx.x * kWarpRowThreads + threadIdx.x) >> 5;
    uint4 cur[NV], nxt[NV];
    warp_row_load<TIn, NV>(X, row, rows, cols, nvec, lane, cur);
    for (; row < rows; row += nwarps) {
        warp_row_load<TIn, NV>(X, row + nwarps, rows, cols, nvec, lane, nxt);
        // pass 1: the row max
        float M = slice_max<TIn, NV>(cur);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
        // pass 2: S = sum exp(x - M)  (a row of -inf only: M taken as 0, S = 0)
        const float Mk = M == -CUDART_INF_F ? 0.f : M;
        const float2 mm = make_float2(Mk, Mk), kk2 = make_float2(kLog2e, kLog2e);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < NV; ++k)
#pragma unroll
            for (int e = 0; e < NP; ++e) {
                const float2 t2 = mul2(sub2(unpack_pair<TIn>(cur[k], e), mm), kk2);
                acc = add2(acc, make_float2(ex2(t2.x), ex2(t2.y)));
            }
        float S = acc.x + acc.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
        const float lse = M + logf(S);
        if constexpr (KIND != 2) {
            // pass 3: p (or log p), 16-byte stores
            const float l2s = __log2f(S);
            TOut* prow = P + row * cols;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const long vi = lane + 32L * k;
                if (vi < nvec) {
                    float o[V];
#pragma unroll
                    for (int e = 0; e < NP; ++e) {
                        const float2 x2 = unpack_pair<TIn>(cur[k], e);
                        if constexpr (KIND == 1) {
                            o[2 * e] = x2.x - lse;
                            o[2 * e + 1] = x2.y - lse;
                        } else {
                            o[2 * e] = ex2(fmaf(x2.x - Mk, kLog2e, -l2s));
                            o[2 * e + 1] = ex2(fmaf(x2.y - Mk, kLog2e, -l2s));
                        }
                    }
                    store_out<TOut, V>(prow + vi * V, o, true, V);
                }
            }
        }
        if (lane == 0) {
            if constexpr (KIND == 2) write_row_lse(X, row, cols, lse, LSE, labels, loss);
            else if (LSE != nullptr) LSE[row] = lse;
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) cur[k] = nxt[k];
    }
}

// Launch the warp-per-row kernel for rows of whole 16-byte vectors, at most
// 256 (512 for log-sum-exp only, which keeps no third pass).
template <typename TIn, typename TOut, int KIND>
bool try_launch_warp_rows(const TIn* X, TOut* P, float* LSE, long rows, long cols, cudaStream_t st, cudaError_t* err,
                          const long long* labels = nullptr, float* loss = nullptr) {
    constexpr int V = Elem<TIn>::kVec;
    const long nvec = cols / V;
    if (cols % V != 0 || nvec > (KIND == 2 ? 512 : 256)) return false;
    const long want = (rows + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32);
    auto launch = [&](auto kern) {
        // persistent: as many CTAs as fit on the GPU at once, or fewer for few rows
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarpRowThreads, 0);
        if (e == cudaSuccess) {
            const long cap = (long)(per_sm > 0 ? per_sm : 1) * device_sms();
            const long grid = want < cap ? want : cap;
            kern<<<(unsigned)grid, kWarpRowThreads, 0, st>>>(X, P, LSE, rows, cols, labels, loss);
            e = cudaGetLastError();
        }
        *err = e;
    };
    if (nvec <= 32) launch(softmax_rows_warp<TIn, TOut, 1, KIND>);
    else if (nvec <= 64) launch(softmax_rows_warp<TIn, TOut, 2, KIND>);
    else if (nvec <= 128) launch(softmax_rows_warp<TIn, TOut, 4, KIND>);
    else if (nvec <= 256) launch(softmax_rows_warp<TIn, TOut, 8, KIND>);
    else if constexpr (KIND == 2) launch(softmax_rows_warp<TIn, TOut, 16, KIND>);
    return true;
}

// ------------------------------------------------------------------ cluster per row
// Rows longer than one CTA's registers hold (above 64 KB): a cluster of CL
// CTAs (2 to 8) takes each row, CTA c holding the c-th of CL equal slices
// (whole multiples of 256 vectors, at most 64 KB) packed in registers (256
// threads x up to 16 vectors of 16 bytes).  Every CTA reduces its
// slice to (m, s) (slice max first, one exponential per element relative to
// it, then the pairwise online update across the CTA), stores that pair into
// a slot of every CTA of the cluster through distributed shared memory and
// arrives on each one's exchange barrier; once all CL pairs are in, every CTA
// merges them in the same order to the row's (M, S) and writes its slice of P
// (or log P) from registers.  X is read from memory once and P written once.
// Slots and exchange barriers alternate between two sets by row parity: a CTA
// reaches row k + 2 only after every CTA has arrived for row k + 1, which each
// does after reading its row-k slots.  The row loop is the same in every CTA
// of a cluster, so the two cluster-wide barriers (after set-up, before exit)
// are reached by all.  Two CTAs per SM: one reduces while the other loads.
// KIND: 0 softmax, 1 log-softmax, 2 log-sum-exp only (and / or the fused
// cross-entropy loss).
constexpr int kClThreads = 256;
constexpr int kClNV = 16;      // 16-byte vectors per thread: a 64 KB slice per CTA
constexpr int kClMaxCtas = 8;  // portable cluster size

template <typename TIn, typename TOut, int KIND>
__global__ void __launch_bounds__(kClThreads, 2)
rows_cluster(const TIn* __restrict__ X, TOut* __restrict__ P, float* __restrict__ LSE, long rows, long cols,
             int* status, const long long* __restrict__ labels, float* __restrict__ loss) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr int W = kClThreads / 32;
    __shared__ __align__(8) uint64_t xbar[2];             // exchange barriers, by row parity
    __shared__ __align__(8) float2 slots[2][kClMaxCtas];  // (m, s) of every CTA, by row parity
    __shared__ float2 wred[W];
    __shared__ int abort_flag;
    const uint32_t rank = cluster_ctarank();
    const uint32_t ncta = cluster_nctarank();
    const long cid = cluster_id_x(), ncl = num_clusters_x();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&xbar[0]), ncta);
        mbar_init(smem_u32(&xbar[1]), ncta);
        abort_flag = 0;
        fence_mbar_init();
    }
    // every CTA's barriers exist before any CTA of the cluster arrives on them
    cluster_sync_all();
    const long nvec = cols / V;
    // this CTA's vectors: [v0, v1), an equal share rounded up to whole rows of threads
    const long per = ((nvec + ncta - 1) / ncta + kClThreads - 1) / kClThreads * kClThreads;
    const long v0 = rank * per, v1 = v0 + per < nvec ? v0 + per : nvec;
    constexpr uint32_t ni = neg_inf_word<TIn>();
    const float2 cc = make_float2(kLog2e, kLog2e);
    bool ok = true;
    long k = 0;
    for (long r = cid; r < rows; r += ncl, ++k) {
        const TIn* xr = X + r * cols;
        uint4 raw[kClNV];
#pragma unroll
        for (int kk = 0; kk < kClNV; ++kk) {
            const long vi = v0 + (long)kk * kClThreads + threadIdx.x;
            raw[kk] = vi < v1 ? __ldg(reinterpret_cast<const uint4*>(xr + vi * V)) : make_uint4(ni, ni, ni, ni);
        }
        // this thread: max, then the sum of exp(x - max)
        float m = slice_max<TIn, kClNV>(raw);
        float sum = 0.f;
        if (m != -CUDART_INF_F) {
            const float2 nmc = make_float2(-m * kLog2e, -m * kLog2e);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int kk = 0; kk < kClNV; ++kk)
#pragma unroll
                for (int e = 0; e < (V == 8 ? 4 : 2); ++e) {
                    const float2 t2 = fma2(unpack_pair<TIn>(raw[kk], e), cc, nmc);
                    acc[e] = add2(acc[e], make_float2(ex2(t2.x), ex2(t2.y)));
                }
            const float2 a2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
            sum = a2.x + a2.y;
        }
        // the CTA's pair: warps by shuffles (max first, then the rescaled
        // sums), then warp 0 over the W warp results
        float wm = m;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, off));
        float ws = wm == -CUDART_INF_F ? 0.f : sum * ex2((m - wm) * kLog2e);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ws += __shfl_xor_sync(0xFFFFFFFFu, ws, off);
        if (lane == 0) wred[warp] = make_float2(wm, ws);
        __syncthreads();
        const int par = (int)(k & 1);
        if (warp == 0) {
            const float2 a = wred[lane & (W - 1)];
            float M = a.x;
#pragma unroll
            for (int off = W / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
            float S = M == -CUDART_INF_F ? 0.f : a.y * ex2((a.x - M) * kLog2e);
#pragma unroll
            for (int off = W / 2; off > 0; off >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, off);
            // lane t hands the pair to CTA t of the cluster
            if ((uint32_t)lane < ncta) {
                st_cluster_f32x2(mapa_shared(smem_u32(&slots[par][rank]), (uint32_t)lane), M, S);
                mbar_arrive_cluster(mapa_shared(smem_u32(&xbar[par]), (uint32_t)lane));
            }
        }
        ok = __syncthreads_and(mbar_wait_cluster_bounded(smem_u32(&xbar[par]), (uint32_t)(k >> 1) & 1u, &abort_flag,
                                                         kWaitLimitNs));
        if (!ok) break;
        // the row's (M, S): every CTA merges the same pairs in the same order
        float M = -CUDART_INF_F, S = 0.f;
        for (uint32_t c = 0; c < ncta; ++c) {
            const float2 q = slots[par][c];
            merge_ms(M, S, q.x, q.y);
        }
        const float lse = M + __log2f(S) * kLn2f;
        if constexpr (KIND < 2) {
            TOut* pr = P + r * cols;
            const float l2s = __log2f(S);
#pragma unroll
            for (int kk = 0; kk < kClNV; ++kk) {
                const long vi = v0 + (long)kk * kClThreads + threadIdx.x;
                if (vi >= v1) continue;
                float f[V];
#pragma unroll
                for (int e = 0; e < V / 2; ++e) {
                    const float2 x2 = unpack_pair<TIn>(raw[kk], e);
                    if (!(S > 0.f)) {
                        // a row with no finite entry: p = 0, log p = -inf (LSE = -inf)
                        f[2 * e] = f[2 * e + 1] = KIND == 1 ? -CUDART_INF_F : 0.f;
                    } else if constexpr (KIND == 1) {
                        f[2 * e] = x2.x - lse;
                        f[2 * e + 1] = x2.y - lse;
                    } else {
                        // p = 2^((x - M) log2 e - log2 S)
                        f[2 * e] = ex2(fmaf(x2.x - M, kLog2e, -l2s));
                        f[2 * e + 1] = ex2(fmaf(x2.y - M, kLog2e, -l2s));
                    }
                }
                store_out<TOut, V>(pr + vi * V, f, true, V);
            }
        }
        if (rank == 0 && threadIdx.x == 0) write_row_lse(X, r, cols, lse, LSE, labels, loss);
    }
    if (!ok && threadIdx.x == 0) {
        abort_flag = 1;
        atomicExch(status, kDevStatusTimeout);
    }
    // no CTA leaves while another CTA of the cluster may still write into its
    // shared memory
    cluster_sync_all();
}

// Launch the cluster-per-row kernel if the row shape suits it: whole 16-byte
// vectors, more than one 64 KB slice and at most kClMaxCtas of them.  For the
// log-sum-exp alone (nothing to write behind which the per-row exchange could
// hide) only when each CTA's share is nearly a full slice and the cluster has
// at most four CTAs; otherwise the streaming kernel, which keeps loads in
// flight while it reduces, measured faster.
template <typename TIn, typename TOut, int KIND>
bool try_launch_cluster(const TIn* X, TOut* P, float* LSE, long rows, long cols, int* status, cudaStream_t st,
                        cudaError_t* err, const long long* labels = nullptr, float* loss = nullptr) {
    constexpr int V = Elem<TIn>::kVec;
    constexpr long kSliceVec = (long)kClThreads * kClNV;
    if (cols % V != 0) return false;
    const long nvec = cols / V;
    if (nvec <= kSliceVec || nvec > kClMaxCtas * kSliceVec) return false;
    const int ncta = (int)((nvec + kSliceVec - 1) / kSliceVec);
    if (KIND == 2 && (ncta > 4 || (nvec + ncta - 1) / ncta < (long)(kClNV - 1) * kClThreads)) return false;
    auto kern = rows_cluster<TIn, TOut, KIND>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many clusters as fit the GPU at once (each loops over rows); the
    // occupancy query is a driver call, so its answer is kept per device and
    // cluster size
    cfg.gridDim = dim3((unsigned)ncta);
    static int active_cache[64][kClMaxCtas + 1] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *err = e;
        return true;
    }
    int active = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64) active = active_cache[dev][ncta];
    }
    if (active == 0) {
        e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
        if (e != cudaSuccess || active < 1) {
            *err = e != cudaSuccess ? e : cudaErrorLaunchOutOfResources;
            return true;
        }
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64) active_cache[dev][ncta] = active;
    }
    const long ncl = rows < active ? rows : active;
    cfg.gridDim = dim3((unsigned)(ncl * ncta));
    *err = cudaLaunchKernelEx(&cfg, kern, X, P, LSE, rows, cols, status, labels, loss);
    return true;
}

long grid_for_rows(long rows) {
    const long kMaxGrid = 1L << 30;
    return rows < kMaxGrid ? rows : kMaxGrid;
}

template <typename TIn, typename TOut, bool LOGP>
cudaError_t softmax_dispatch(const TIn* X, TOut* P, float* LSE, long rows, long cols, int* status,
                             cudaStream_t st) {
    constexpr int V = Elem<TIn>::kVec;
    cudaError_t terr;
    if (try_launch_tma<TIn, TOut, true, LOGP>(X, P, LSE, rows, cols, status, st, &terr)) return terr;
    if (try_launch_warp_rows<TIn, TOut, LOGP ? 1 : 0>(X, P, LSE, rows, cols, st, &terr)) return terr;
    if (try_launch_cluster<TIn, TOut, LOGP ? 1 : 0>(X, P, LSE, rows, cols, status, st, &terr)) return terr;
    const int vec_ok = (cols % V) == 0;
    const long nvec = (cols + V - 1) / V;
    const dim3 grid((unsigned)grid_for_rows(rows));
#define FA_RESIDENT(T, NVV) softmax_rows_resident<TIn, TOut, T, NVV, LOGP><<<grid, T, 0, st>>>(X, P, LSE, rows, cols, vec_ok)
    if (nvec <= 32) FA_RESIDENT(32, 1);
    else if (nvec <= 64) FA_RESIDENT(32, 2);
    else if (nvec <= 128) FA_RESIDENT(32, 4);
    else if (nvec <= 256) FA_RESIDENT(32, 8);
    else if (nvec <= 512) FA_RESIDENT(64, 8);
    else if (nvec <= 1024) FA_RESIDENT(128, 8);
    else if (nvec <= 2048) FA_RESIDENT(256, 8);
    else if (nvec <= 4096) FA_RESIDENT(512, 8);
    else softmax_rows_stream<TIn, TOut, 512, 8, LOGP><<<grid, 512, 0, st>>>(X, P, LSE, rows, cols, vec_ok);
#undef FA_RESIDENT
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t lse_dispatch(const TIn* X, float* LSE, long rows, long cols, int* status, cudaStream_t st,
                         const long long* labels, float* loss) {
    constexpr int V = Elem<TIn>::kVec;
    cudaError_t terr;
    if (try_launch_warp_rows<TIn, float, 2>(X, nullptr, LSE, rows, cols, st, &terr, labels, loss)) return terr;
    if (try_launch_lse_tma<TIn>(X, LSE, rows, cols, status, st, &terr, labels, loss)) return terr;
    if (try_launch_cluster<TIn, float, 2>(X, nullptr, LSE, rows, cols, status, st, &terr, labels, loss)) return terr;
    const int vec_ok = (cols % V) == 0;
    const long nvec = (cols + V - 1) / V;
    const dim3 grid((unsigned)grid_for_rows(rows));
    if (nvec <= 128) logsumexp_rows_stream<TIn, 32, 4><<<grid, 32, 0, st>>>(X, LSE, rows, cols, vec_ok, labels, loss);
    else if (nvec <= 1024) logsumexp_rows_stream<TIn, 128, 4><<<grid, 128, 0, st>>>(X, LSE, rows, cols, vec_ok, labels, loss);
    else logsumexp_rows_stream<TIn, 256, 8><<<grid, 256, 0, st>>>(X, LSE, rows, cols, vec_ok, labels, loss);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_softmax_rows(const void* X, void* P, float* LSE, long rows, long cols, int in_bf16, int out_bf16,
                                int log_out, int* status, cudaStream_t st) {
    using bf = __nv_bfloat16;
#define FA_SOFTMAX(TI, TO)                                                                            \
    return log_out ? softmax_dispatch<TI, TO, true>((const TI*)X, (TO*)P, LSE, rows, cols, status, st) \
                   : softmax_dispatch<TI, TO, false>((const TI*)X, (TO*)P, LSE, rows, cols, status, st)
    if (in_bf16 && out_bf16) { FA_SOFTMAX(bf, bf); }
    if (in_bf16) { FA_SOFTMAX(bf, float); }
    if (out_bf16) { FA_SOFTMAX(float, bf); }
    FA_SOFTMAX(float, float);
#undef FA_SOFTMAX
}

cudaError_t launch_logsumexp_rows(const void* X, float* LSE, long rows, long cols, int in_bf16,
                                  const long long* labels, float* loss, int* status, cudaStream_t st) {
    if (in_bf16) return lse_dispatch((const __nv_bfloat16*)X, LSE, rows, cols, status, st, labels, loss);
    return lse_dispatch((const float*)X, LSE, rows, cols, status, st, labels, loss);
}

}  // namespace fa
