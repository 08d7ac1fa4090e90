// attn_splitkv.cu -- merge of split-KV partial attention results.
//
// When the key tiles of a query block are split over S CTAs, split s returns
// a normalised partial output o_s (its keys only) and its log-sum-exp LSE_s.
// The partials combine exactly as the block-wise online merge of
// "从原始Softmax到在线Softmax" (section on the block-wise online softmax)
// combines normalised block results, with l_s = e^{LSE_s}:
//     LSE = log sum_s e^{LSE_s},   o = sum_s e^{LSE_s - LSE} o_s.
// A split that kept no key for a row has LSE_s = -inf and weight 0 (its o_s is
// never read).  One warp per row; lane i owns the D/32 adjacent columns
// [i D/32, (i+1) D/32), read as one 16-byte (d = 128) or 8-byte (d = 64)
// load per split, and the splits are walked sixteen at a time so their loads
// are in flight together instead of costing one memory latency each.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fattn_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplitsPerLane = 2;  // up to 64 splits: lanes hold LSE_s for s = lane and lane + 32

template <int C>
struct Vec;
template <>
struct Vec<4> {
    static __device__ __forceinline__ void load(const float* p, float* v) {
        const float4 x = *reinterpret_cast<const float4*>(p);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
};
template <>
struct Vec<2> {
    static __device__ __forceinline__ void load(const float* p, float* v) {
        const float2 x = *reinterpret_cast<const float2*>(p);
        v[0] = x.x; v[1] = x.y;
    }
};

template <int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
attn_combine_kernel(const float* __restrict__ Opart, const float* __restrict__ Lpart, void* __restrict__ O,
                    float* __restrict__ LSE, long rows, int S, int out_bf16, int N, int H, long long osb,
                    long long osh, long long osr) {
    constexpr int C = D / 32;  // adjacent columns per lane
    constexpr int kBatch = 16; // splits whose loads are in flight together
    const int lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    // every split's LSE, once: lane holds s = lane and s = lane + 32
    float ls[kMaxSplitsPerLane];
#pragma unroll
    for (int i = 0; i < kMaxSplitsPerLane; ++i) {
        const int sidx = lane + 32 * i;
        ls[i] = sidx < S ? Lpart[(long)sidx * rows + row] : -CUDART_INF_F;
    }
    // the row's maximum partial LSE and sum_s e^{LSE_s - max}
    float mx = fmaxf(ls[0], ls[1]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxSplitsPerLane; ++i)
        if (ls[i] != -CUDART_INF_F) sum += ex2((ls[i] - mx) * kLog2e);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    // every split empty (a query with no kept key): O = 0, LSE = -inf
    const float lse = sum > 0.f ? mx + logf(sum) : -CUDART_INF_F;
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    const float* base = Opart + row * D + lane * C;
    const long sstride = rows * D;  // floats between one split's partials and the next
    for (int s0 = 0; s0 < S; s0 += kBatch) {
        float v[kBatch][C];
        float w[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const int sidx = s0 + k;
            // LSE_s from the lane that holds it (uniform shuffle source)
            const float l = __shfl_sync(0xFFFFFFFFu, ((sidx >> 5) & 1) ? ls[1] : ls[0], sidx & 31);
            w[k] = (sidx < S && l != -CUDART_INF_F) ? ex2((l - lse) * kLog2e) : 0.f;
            if (w[k] != 0.f) Vec<C>::load(base + (long)sidx * sstride, v[k]);
            else {
#pragma unroll
                for (int c = 0; c < C; ++c) v[k][c] = 0.f;
            }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
#pragma unroll
            for (int c = 0; c < C; ++c) acc[c] = fmaf(w[k], v[k][c], acc[c]);
    }
    const long bh = row / N, qi = row % N;
    const long obase = (bh / H) * osb + (bh % H) * osh + qi * osr + lane * C;
    if (out_bf16) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(O) + obase;
        if constexpr (C == 4) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
        } else {
            *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0], acc[1]);
        }
    } else {
        float* dst = reinterpret_cast<float*>(O) + obase;
        if constexpr (C == 4) *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        else *reinterpret_cast<float2*>(dst) = make_float2(acc[0], acc[1]);
    }
    if (LSE != nullptr && lane == 0) LSE[row] = lse;
}

}  // namespace

cudaError_t launch_attn_combine(const AttnParams& p, cudaStream_t st) {
    const long rows = (long)p.B * p.H * p.N;
    const dim3 grid((unsigned)((rows + kRowsPerBlock - 1) / kRowsPerBlock));
    if (p.d == 64)
        attn_combine_kernel<64><<<grid, kRowsPerBlock * 32, 0, st>>>(p.Opart, p.Lpart, p.O, p.LSE, rows,
                                                                    p.num_splits, p.out_bf16, p.N, p.H, p.os[0],
                                                                    p.os[1], p.os[2]);
    else if (p.d == 128)
        attn_combine_kernel<128><<<grid, kRowsPerBlock * 32, 0, st>>>(p.Opart, p.Lpart, p.O, p.LSE, rows,
                                                                     p.num_splits, p.out_bf16, p.N, p.H, p.os[0],
                                                                     p.os[1], p.os[2]);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace fa
