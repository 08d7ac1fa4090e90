// attn_splitkv.cu -- merge of split-KV partial attention results.
//
// When the key tiles of a query block are split over S CTAs, split s returns
// a normalised partial output o_s (its keys only) and its log-sum-exp LSE_s.
// The partials combine exactly as the block-wise online merge of
// "从原始Softmax到在线Softmax" (section on the block-wise online softmax)
// combines normalised block results, with l_s = e^{LSE_s}:
//     LSE = log sum_s e^{LSE_s},   o = sum_s e^{LSE_s - LSE} o_s.
// A split that kept no key for a row has LSE_s = -inf and weight 0 (its o_s is
// never read).  One warp per row; lane i owns columns i, i + 32, ...
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fattn_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
attn_combine_kernel(const float* __restrict__ Opart, const float* __restrict__ Lpart, void* __restrict__ O,
                    float* __restrict__ LSE, long rows, int S, int out_bf16, int N, int H, long long osb,
                    long long osh, long long osr) {
    constexpr int C = D / 32;  // columns per lane
    const int lane = threadIdx.x & 31;
    const long row = (long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
    if (row >= rows) return;
    // the row's maximum partial LSE and sum_s e^{LSE_s - max}
    float mx = -CUDART_INF_F;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, Lpart[(long)s * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
    float sum = 0.f;
    for (int s = lane; s < S; s += 32) {
        const float ls = Lpart[(long)s * rows + row];
        if (ls != -CUDART_INF_F) sum += ex2((ls - mx) * kLog2e);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    // every split empty (a query with no kept key): O = 0, LSE = -inf
    const float lse = sum > 0.f ? mx + logf(sum) : -CUDART_INF_F;
    float acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = 0.f;
    for (int s = 0; s < S; ++s) {
        const float ls = Lpart[(long)s * rows + row];
        if (ls == -CUDART_INF_F) continue;
        const float w = ex2((ls - lse) * kLog2e);
        const float* o = Opart + ((long)s * rows + row) * D;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = fmaf(w, o[lane + 32 * c], acc[c]);
    }
    const long bh = row / N, qi = row % N;
    const long obase = (bh / H) * osb + (bh % H) * osh + qi * osr;
    if (out_bf16) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(O) + obase;
#pragma unroll
        for (int c = 0; c < C; ++c) dst[lane + 32 * c] = __float2bfloat16_rn(acc[c]);
    } else {
        float* dst = reinterpret_cast<float*>(O) + obase;
#pragma unroll
        for (int c = 0; c < C; ++c) dst[lane + 32 * c] = acc[c];
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
