// attn_f32.cu -- fp32 attention forward on CUDA cores.
//
// O = softmax(scale * Q K^T [+ causal mask]) V and LSE, fp32 in / fp32 out.
// Tensor cores are not used: TF32 products would not meet an fp32 accuracy
// bar.  Each query row is owned by G = D/32 adjacent threads (G = 1 for
// D <= 32); thread g of a row owns columns g, g+G, g+2G, ... so that the G
// threads of a row read adjacent shared-memory words.  Keys stream through
// shared memory in tiles of 32; per tile every row runs the block-wise online
// merge of "从原始Softmax到在线Softmax" (section on the block-wise online
// softmax):  m' = max(m, rowmax),  o~ <- e^{m-m'} o~ + sum_k e^{s_k-m'} v_k,
// l <- e^{m-m'} l + sum_k e^{s_k-m'};  o = o~ / l at the end.
// Scores are kept in base-2 units (q is pre-multiplied by scale * log2 e).
#include <math_constants.h>

#include "fattn_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kRows = 64;  // query rows per CTA
constexpr int kKeys = 32;  // keys per shared-memory tile

struct StridesF32 {
    long long q[3], k[3], v[3], o[3];  // element strides (batch, head, row)
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kRows * (D >= 32 ? D / 32 : 1))
attn_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                float* __restrict__ O, float* __restrict__ LSE, int N, int M, float qscale, int H, int coff,
                StridesF32 st) {
    constexpr int G = D >= 32 ? D / 32 : 1;  // threads per row
    constexpr int C = D / G;                 // columns per thread
    constexpr int T = kRows * G;
    __shared__ float Ks[kKeys][D];
    __shared__ float Vs[kKeys][D];

    const int tid = threadIdx.x;
    const int g = tid % G;
    const int r = tid / G;
    const long bh = blockIdx.y;
    const long hh = bh % H, bb = bh / H;
    const int i = blockIdx.x * kRows + r;  // query index
    const bool row_ok = i < N;

    const float* q_row = Q + bb * st.q[0] + hh * st.q[1] + (long)(row_ok ? i : 0) * st.q[2];
    float q[C], o[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
        q[c] = row_ok ? q_row[c * G + g] * qscale : 0.f;
        o[c] = 0.f;
    }
    float m = -CUDART_INF_F, l = 0.f;

    const float* Kh = K + bb * st.k[0] + hh * st.k[1];
    const float* Vh = V + bb * st.v[0] + hh * st.v[1];
    int kv_end = M;
    if (CAUSAL) {
        // keys kept for query i: j <= i + coff (coff = 0 top-left, M - N bottom-right)
        const int last = min(N, (int)(blockIdx.x + 1) * kRows) - 1;  // last query row of this CTA
        kv_end = (int)max(0L, min((long)M, (long)last + coff + 1));
    }
    for (int k0 = 0; k0 < kv_end; k0 += kKeys) {
        __syncthreads();
        for (int e = tid; e < kKeys * D; e += T) {
            const int kk = e / D, c = e % D;
            const bool ok = k0 + kk < M;
            Ks[kk][c] = ok ? Kh[(long)(k0 + kk) * st.k[2] + c] : 0.f;
            Vs[kk][c] = ok ? Vh[(long)(k0 + kk) * st.v[2] + c] : 0.f;
        }
        __syncthreads();
        float x[kKeys];
        float tmax = -CUDART_INF_F;
#pragma unroll
        for (int kk = 0; kk < kKeys; ++kk) {
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < C; ++c) part = fmaf(q[c], Ks[kk][c * G + g], part);
#pragma unroll
            for (int off = 1; off < G; off <<= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
            const int key = k0 + kk;
            const bool keep = key < M && (!CAUSAL || key <= i + coff);
            x[kk] = keep ? part : -CUDART_INF_F;
            tmax = fmaxf(tmax, x[kk]);
        }
        const float m_new = fmaxf(m, tmax);
        if (m_new == -CUDART_INF_F) continue;  // nothing kept yet for this row
        const float alpha = ex2(m - m_new);    // m = -inf: alpha = 0
        l *= alpha;
#pragma unroll
        for (int c = 0; c < C; ++c) o[c] *= alpha;
#pragma unroll
        for (int kk = 0; kk < kKeys; ++kk) {
            const float p = ex2(x[kk] - m_new);
            l += p;
#pragma unroll
            for (int c = 0; c < C; ++c) o[c] = fmaf(p, Vs[kk][c * G + g], o[c]);
        }
        m = m_new;
    }
    if (!row_ok) return;
    // l = 0 only for a query with no kept key: O = 0, LSE = -inf
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    float* o_row = O + bb * st.o[0] + hh * st.o[1] + (long)i * st.o[2];
#pragma unroll
    for (int c = 0; c < C; ++c) o_row[c * G + g] = o[c] * inv_l;
    if (LSE != nullptr && g == 0) LSE[bh * N + i] = l > 0.f ? (m + __log2f(l)) * kLn2 : -CUDART_INF_F;
}

template <int D>
cudaError_t launch_d(const AttnParams& p, cudaStream_t st) {
    constexpr int G = D >= 32 ? D / 32 : 1;
    const dim3 grid((p.N + kRows - 1) / kRows, p.B * p.H);
    const float qscale = p.scale * kLog2e;
    const int coff = p.causal == 2 ? p.M - p.N : 0;
    StridesF32 s;
    for (int i = 0; i < 3; ++i) {
        s.q[i] = p.qs[i]; s.k[i] = p.ks[i]; s.v[i] = p.vs[i]; s.o[i] = p.os[i];
    }
    if (p.causal)
        attn_f32_kernel<D, true><<<grid, kRows * G, 0, st>>>((const float*)p.Q, (const float*)p.K,
                                                            (const float*)p.V, (float*)p.O, p.LSE, p.N, p.M,
                                                            qscale, p.H, coff, s);
    else
        attn_f32_kernel<D, false><<<grid, kRows * G, 0, st>>>((const float*)p.Q, (const float*)p.K,
                                                             (const float*)p.V, (float*)p.O, p.LSE, p.N, p.M,
                                                             qscale, p.H, coff, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_f32(const AttnParams& p, cudaStream_t st) {
    switch (p.d) {
        case 16: return launch_d<16>(p, st);
        case 32: return launch_d<32>(p, st);
        case 64: return launch_d<64>(p, st);
        case 128: return launch_d<128>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
