// attn_noalloc.cu -- split-KV attention for callers that cannot allocate.
//
// fa_attn_fwd_splitkv needs a scratch buffer for the per-split partial
// results.  Some callers cannot provide one: their device memory belongs to
// another allocator (a framework's caching pool, a host application that hands
// a plugin only its inputs and outputs), or they must not call cudaMalloc /
// cudaFree at all, e.g. because cudaFree can synchronise the whole device.
// fa_attn_fwd_splitkv_noalloc serves them with a fixed scratch array that
// lives in this library's device image: a GPU holds FA_NOALLOC_SCRATCH_BYTES
// for it from the moment the library's device code is loaded there (with lazy
// module loading, the first libfattn call on that device) until the process
// exits.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "fattn.h"

namespace {

// The shared scratch.  Its name is only a host-side stand-in in host code; the
// device address is looked up per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call made with that device current and cached afterwards.
void* noalloc_scratch(int* status) {
    static void* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = FA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            *status = FA_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" int fa_attn_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                           int H, int N, int M, int d, float scale, int causal, int num_splits,
                                           int in_dtype, int out_dtype, void* stream) {
    if (B <= 0 || H <= 0 || N <= 0 || M <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
    if (num_splits < 0) return FA_ERR_INVALID_ARG;
    const int S = num_splits == 0 ? fa_attn_splitkv_num_splits(B, H, N, M, d, causal) : num_splits;
    // -1 for a split count above the library's maximum (the one limit, kept
    // where fa_attn_fwd_splitkv checks it)
    const long need = fa_attn_splitkv_workspace_bytes(B, H, N, d, S);
    if (need < 0) return FA_ERR_INVALID_ARG;
    // partials that do not fit the fixed scratch are refused, never truncated
    if (need > (long)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_INVALID_ARG;
    int status = FA_OK;
    void* scratch = noalloc_scratch(&status);
    if (scratch == nullptr) return status;
    // Every element of the partials a call reads is written by the same call
    // (splits without a kept key store LSE_s = -inf), so nothing is cleared.
    return fa_attn_fwd_splitkv(Q, K, V, O, LSE, B, H, N, M, d, scale, causal, S, scratch,
                               (long)FA_NOALLOC_SCRATCH_BYTES, in_dtype, out_dtype, stream);
}
