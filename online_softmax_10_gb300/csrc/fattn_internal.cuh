// fattn_internal.cuh -- launchers shared between the C-ABI translation unit and
// the kernel translation units.  Not part of the public interface.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Upper bound on any single in-kernel wait before the kernel gives up and
// records a timeout (4 s of wall clock; a legitimate wait is microseconds).
constexpr uint64_t kWaitLimitNs = 4000000000ull;

// Status codes written into the per-device status word by kernels.
constexpr int kDevStatusTimeout = 5;

struct AttnParams {
    const void* Q;
    const void* K;
    const void* V;
    void* O;
    float* LSE;        // may be null
    int B, H, N, M, d;
    float scale;       // > 0
    int causal;        // 0 none, 1 top-left (j <= i), 2 bottom-right (j <= i + M - N)
    int out_bf16;      // 1: O is bf16, 0: O is fp32
    int* status;       // device status word
    int num_splits;    // > 1: key tiles split over this many CTAs (bf16 path only)
    float* Opart;      // split partial outputs, fp32 [num_splits][B*H][N][d]
    float* Lpart;      // split partial LSE, fp32 [num_splits][B*H][N]
    long long qs[3], ks[3], vs[3], os[3];  // element strides (batch, head, row); d is contiguous
};

// Row-wise kernels (softmax_rows.cu).
// log_out: write log p = x - LSE instead of p.
cudaError_t launch_softmax_rows(const void* X, void* P, float* LSE, long rows, long cols, int in_bf16,
                                int out_bf16, int log_out, int* status, cudaStream_t stream);
// LSE (may be null when loss is given); labels/loss: the fused cross-entropy
// loss[r] = LSE[r] - X[r, labels[r]] (0 outside [0, cols)), or both null.
cudaError_t launch_logsumexp_rows(const void* X, float* LSE, long rows, long cols, int in_bf16,
                                  const long long* labels, float* loss, int* status, cudaStream_t stream);

// fp32 CUDA-core attention (attn_f32.cu).  d in {16, 32, 64, 128}.
cudaError_t launch_attn_f32(const AttnParams& p, int num_sms, cudaStream_t stream);

// bf16 tensor-core attention (attn_tc.cu).  d in {64, 128}.  The three tensor
// maps describe Q [B, H, N, d], K and V [B, H, M, d] (any strides) as 4-D bf16
// tensors {d, rows, H, B} with a 64 x 128 x 1 x 1 box and 128-byte swizzle.
cudaError_t launch_attn_bf16_tc(const AttnParams& p, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                const CUtensorMap* tmV, int num_sms, cudaStream_t stream);

// Combine split partials into O and LSE (attn_splitkv.cu):
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s.
cudaError_t launch_attn_combine(const AttnParams& p, cudaStream_t stream);

// One CTA waiting on an mbarrier that never completes (attn_tc.cu).
cudaError_t launch_selftest_wait(int* status, uint64_t limit_ns, cudaStream_t stream);

}  // namespace fa
