// attn_f32.cu -- fp32 attention forward on CUDA cores.
//
// O = softmax(scale * Q K^T [+ causal mask]) V and LSE, fp32 in / fp32 out.
// Tensor cores are not used: TF32 products would not meet an fp32 accuracy
// bar.  A CTA takes R query rows of one (batch, head); each row is owned by G
// adjacent threads, and thread g of a row owns the 4-column chunks g, g + G,
// g + 2G, ... so that one 16-byte shared-memory load per chunk serves the G
// threads of a row from adjacent words and every row of the warp by
// broadcast.  R = 64 rows with 32 columns per thread when there are enough
// row blocks to fill the GPU; otherwise R = 16 rows with 8 columns per thread,
// four times the CTAs (a single 64 x 64 head then spreads over four SMs).
// Keys stream through shared memory in tiles of 64 (32 at d = 128); per tile every row runs
// the block-wise online merge of "从原始Softmax到在线Softmax" (section on the
// block-wise online softmax):  m' = max(m, rowmax),
// o~ <- e^{m-m'} o~ + sum_k e^{s_k-m'} v_k,  l <- e^{m-m'} l + sum_k e^{s_k-m'};
// o = o~ / l at the end.  Scores are kept in base-2 units (q is
// pre-multiplied by scale * log2 e).
#include <math_constants.h>

#include "fattn_internal.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// keys per shared-memory tile: K and V tiles take 32 KB at most
template <int D>
__host__ __device__ constexpr int keys_per_tile() {
    return D <= 64 ? 64 : 32;
}

struct StridesF32 {
    long long q[3], k[3], v[3], o[3];  // element strides (batch, head, row)
};

// threads per query row for R rows per CTA
template <int D, int R>
__host__ __device__ constexpr int threads_per_row() {
    return R == 64 ? (D >= 32 ? D / 32 : 1) : D / 8;
}

template <int D, bool CAUSAL, int R>
__global__ void __launch_bounds__(R * threads_per_row<D, R>(), 1)
attn_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K, const float* __restrict__ V,
                float* __restrict__ O, float* __restrict__ LSE, int N, int M, float qscale, int H, int coff,
                StridesF32 st) {
    constexpr int G = threads_per_row<D, R>();  // threads per row
    constexpr int NC = D / G / 4;               // 4-column chunks per thread
    constexpr int T = R * G;
    constexpr int kKeys = keys_per_tile<D>();
    static_assert(NC >= 1 && G <= 32 && (G & (G - 1)) == 0, "row split");
    __shared__ __align__(16) float Ks[kKeys][D];
    __shared__ __align__(16) float Vs[kKeys][D];

    const int tid = threadIdx.x;
    const int g = tid % G;
    const int r = tid / G;
    const long bh = blockIdx.y;
    const long hh = bh % H, bb = bh / H;
    const int i = blockIdx.x * R + r;  // query index
    const bool row_ok = i < N;

    const float* q_row = Q + bb * st.q[0] + hh * st.q[1] + (long)(row_ok ? i : 0) * st.q[2];
    float q[NC][4], o[NC][4];
#pragma unroll
    for (int v = 0; v < NC; ++v)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            q[v][e] = row_ok ? q_row[4 * (g + v * G) + e] * qscale : 0.f;
            o[v][e] = 0.f;
        }
    float m = -CUDART_INF_F, l = 0.f;

    const float* Kh = K + bb * st.k[0] + hh * st.k[1];
    const float* Vh = V + bb * st.v[0] + hh * st.v[1];
    int kv_end = M;
    if (CAUSAL) {
        // keys kept for query i: j <= i + coff (coff = 0 top-left, M - N bottom-right)
        const int last = min(N, (int)(blockIdx.x + 1) * R) - 1;  // last query row of this CTA
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
            const float4* kr = reinterpret_cast<const float4*>(Ks[kk]);
            float part = 0.f;
#pragma unroll
            for (int v = 0; v < NC; ++v) {
                const float4 kv = kr[g + v * G];
                part = fmaf(q[v][0], kv.x, part);
                part = fmaf(q[v][1], kv.y, part);
                part = fmaf(q[v][2], kv.z, part);
                part = fmaf(q[v][3], kv.w, part);
            }
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
        for (int v = 0; v < NC; ++v)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[v][e] *= alpha;
#pragma unroll
        for (int kk = 0; kk < kKeys; ++kk) {
            const float p = ex2(x[kk] - m_new);
            l += p;
            const float4* vr = reinterpret_cast<const float4*>(Vs[kk]);
#pragma unroll
            for (int v = 0; v < NC; ++v) {
                const float4 vv = vr[g + v * G];
                o[v][0] = fmaf(p, vv.x, o[v][0]);
                o[v][1] = fmaf(p, vv.y, o[v][1]);
                o[v][2] = fmaf(p, vv.z, o[v][2]);
                o[v][3] = fmaf(p, vv.w, o[v][3]);
            }
        }
        m = m_new;
    }
    if (!row_ok) return;
    // l = 0 only for a query with no kept key: O = 0, LSE = -inf
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    float* o_row = O + bb * st.o[0] + hh * st.o[1] + (long)i * st.o[2];
#pragma unroll
    for (int v = 0; v < NC; ++v)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_row[4 * (g + v * G) + e] = o[v][e] * inv_l;
    if (LSE != nullptr && g == 0) LSE[bh * N + i] = l > 0.f ? (m + __log2f(l)) * kLn2 : -CUDART_INF_F;
}

template <int D, int R>
cudaError_t launch_dr(const AttnParams& p, cudaStream_t st) {
    constexpr int T = R * threads_per_row<D, R>();
    const dim3 grid((p.N + R - 1) / R, p.B * p.H);
    const float qscale = p.scale * kLog2e;
    const int coff = p.causal == 2 ? p.M - p.N : 0;
    StridesF32 s;
    for (int i = 0; i < 3; ++i) {
        s.q[i] = p.qs[i]; s.k[i] = p.ks[i]; s.v[i] = p.vs[i]; s.o[i] = p.os[i];
    }
    if (p.causal)
        attn_f32_kernel<D, true, R><<<grid, T, 0, st>>>((const float*)p.Q, (const float*)p.K, (const float*)p.V,
                                                        (float*)p.O, p.LSE, p.N, p.M, qscale, p.H, coff, s);
    else
        attn_f32_kernel<D, false, R><<<grid, T, 0, st>>>((const float*)p.Q, (const float*)p.K, (const float*)p.V,
                                                         (float*)p.O, p.LSE, p.N, p.M, qscale, p.H, coff, s);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnParams& p, int num_sms, cudaStream_t st) {
    // 64-row blocks when they fill every SM twice over, else 16-row blocks
    const long blocks64 = (long)((p.N + 63) / 64) * p.B * p.H;
    return blocks64 >= 2L * num_sms ? launch_dr<D, 64>(p, st) : launch_dr<D, 16>(p, st);
}

}  // namespace

cudaError_t launch_attn_f32(const AttnParams& p, int num_sms, cudaStream_t st) {
    switch (p.d) {
        case 16: return launch_d<16>(p, num_sms, st);
        case 32: return launch_d<32>(p, num_sms, st);
        case 64: return launch_d<64>(p, num_sms, st);
        case 128: return launch_d<128>(p, num_sms, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fa
