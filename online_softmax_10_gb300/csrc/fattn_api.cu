// fattn_api.cu -- the C ABI of libfattn (declared in include/fattn.h).
//
// Host side only: argument validation, TMA tensor-map encoding (with a small
// cache of recent maps), kernel dispatch on the caller's stream, and the per-device status word that the
// kernels' bounded waits write on a timeout.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fattn.h"
#include "fattn_internal.cuh"

// Written by kernels whose bounded waits ran out; read and cleared by
// fa_device_status().  One instance per device.
__device__ int g_fa_status;

namespace {

constexpr int kMaxDevices = 64;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }


thread_local cudaError_t t_last_cuda_error = cudaSuccess;

// FA_OK, or FA_ERR_CUDA with the runtime error remembered for fa_last_cuda_error().
int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return FA_OK;
    t_last_cuda_error = e;
    return FA_ERR_CUDA;
}

// Device address of g_fa_status on the current device (looked up once per device).
int* status_word(int* err) {
    static int* addr[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    const cudaError_t ge = cudaGetDevice(&dev);
    if (ge != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = cuda_status(ge == cudaSuccess ? cudaErrorInvalidDevice : ge);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t se = cudaGetSymbolAddress(&p, g_fa_status);
        if (se != cudaSuccess) {
            *err = cuda_status(se);
            return nullptr;
        }
        addr[dev] = static_cast<int*>(p);
    }
    return addr[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [B, H, rows, d] bf16 tensor with element strides (batch, head, row) and d
// contiguous -> 4-D tensor map {d, rows, H, B}, box 64 (d) x 128 (rows) x 1 x 1,
// 128-byte swizzle, zero fill past the last row (ragged row tails).
bool encode_bf16_4d(CUtensorMap* map, const void* ptr, long B, long H, long rows, int d, const long long* st) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    const cuuint32_t box[4] = {64, 128, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded tensor maps of recent calls.  A map depends only on (pointer,
// sizes, strides), so a hit is always the map encoding would produce; the
// cache only saves the driver call (a few microseconds per map, which matters
// for small problems).  Round-robin replacement, one lock.
struct MapKey {
    const void* ptr;
    long B, H, rows;
    int d;
    long long st[3];
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && B == o.B && H == o.H && rows == o.rows && d == o.d && st[0] == o.st[0] &&
               st[1] == o.st[1] && st[2] == o.st[2];
    }
};

class MapCache {
  public:
    bool get(const MapKey& k, CUtensorMap* out) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < kSize; ++i)
            if (used_[i] && keys_[i] == k) {
                *out = maps_[i];
                return true;
            }
        return false;
    }
    void put(const MapKey& k, const CUtensorMap& m) {
        std::lock_guard<std::mutex> lock(mu_);
        keys_[next_] = k;
        maps_[next_] = m;
        used_[next_] = true;
        next_ = (next_ + 1) % kSize;
    }

  private:
    static constexpr int kSize = 48;
    std::mutex mu_;
    MapKey keys_[kSize] = {};
    CUtensorMap maps_[kSize] = {};
    bool used_[kSize] = {};
    int next_ = 0;
};

bool encode_bf16_4d_cached(CUtensorMap* map, const void* ptr, long B, long H, long rows, int d, const long long* st) {
    static MapCache cache;
    const MapKey key{ptr, B, H, rows, d, {st[0], st[1], st[2]}};
    if (cache.get(key, map)) return true;
    if (!encode_bf16_4d(map, ptr, B, H, rows, d, st)) return false;
    cache.put(key, *map);
    return true;
}

bool mul_fits(long a, long b, long limit) { return a > 0 && b > 0 && a <= limit / b; }

int num_sms() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n;
}


// Argument checks shared by the attention entry points (nothing is enqueued).
int check_attn_args(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int M,
                    int d, float scale, int causal, int in_dtype, int out_dtype) {
    if (!Q || !K || !V || !O) return FA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || N <= 0 || M <= 0 || d <= 0) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (causal < 0 || causal > 2) return FA_ERR_INVALID_ARG;
    const long kLim = 1L << 62;
    const long bh = (long)B * H;
    if (!mul_fits(bh, (long)(N > M ? N : M), kLim) || !mul_fits(bh * (N > M ? N : M), d, kLim / 4))
        return FA_ERR_INVALID_ARG;
    if (in_dtype != FA_F32 && in_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (out_dtype != FA_F32 && out_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (bh > 65535) return FA_ERR_UNSUPPORTED;
    if (in_dtype == FA_F32) {
        if (out_dtype != FA_F32) return FA_ERR_UNSUPPORTED;
        if (d != 16 && d != 32 && d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    } else {
        if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    }
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || (LSE && !aligned16(LSE)))
        return FA_ERR_MISALIGNED;
    return FA_OK;
}

constexpr int kMaxSplits = 64;

struct Strides {
    long long q[3], k[3], v[3], o[3];  // element strides (batch, head, row)
};

Strides contiguous_strides(int H, int N, int M, int d) {
    Strides s;
    const long long qn = (long long)N * d, km = (long long)M * d;
    s.q[0] = s.o[0] = H * qn; s.q[1] = s.o[1] = qn; s.q[2] = s.o[2] = d;
    s.k[0] = s.v[0] = H * km; s.k[1] = s.v[1] = km; s.k[2] = s.v[2] = d;
    return s;
}

// Element strides that are positive and whole multiples of 16 bytes.
bool strides_ok(const long long* st, int esize) {
    for (int i = 0; i < 3; ++i)
        if (st[i] <= 0 || (st[i] * esize) % 16 != 0 || st[i] > (1LL << 40)) return false;
    return true;
}

// Launch the attention kernel(s) for validated arguments.
int attn_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int M, int d,
                const Strides& st, float scale, int causal, int S, float* opart, float* lpart, int in_dtype,
                int out_dtype, void* stream) {
    int err = FA_OK;
    int* status = status_word(&err);
    if (status == nullptr) return err;
    fa::AttnParams p{Q,      K, V,     O,     LSE, B, H, N, M, d, scale, causal, out_dtype == FA_BF16 ? 1 : 0,
                     status, S, opart, lpart, {},  {}, {}, {}};
    for (int i = 0; i < 3; ++i) {
        p.qs[i] = st.q[i]; p.ks[i] = st.k[i]; p.vs[i] = st.v[i]; p.os[i] = st.o[i];
    }
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (in_dtype == FA_F32) {
        e = fa::launch_attn_f32(p, num_sms(), cs);
    } else {
        CUtensorMap tq, tk, tv;
        if (!encode_bf16_4d_cached(&tq, Q, B, H, N, d, st.q) || !encode_bf16_4d_cached(&tk, K, B, H, M, d, st.k) ||
            !encode_bf16_4d_cached(&tv, V, B, H, M, d, st.v))
            return FA_ERR_CUDA;
        e = fa::launch_attn_bf16_tc(p, &tq, &tk, &tv, num_sms(), cs);
        if (e == cudaSuccess && S > 1) e = fa::launch_attn_combine(p, cs);
    }
    return cuda_status(e);
}

// Bytes of split workspace: partial O (fp32) then partial LSE, 256-B aligned.
long splitkv_bytes(long bh, long N, long d, long S, long* lse_offset) {
    const long obytes = S * bh * N * d * 4;
    const long off = (obytes + 255) / 256 * 256;
    if (lse_offset) *lse_offset = off;
    return off + S * bh * N * 4;
}

// Splits that fill the GPU when the (head, query block) units alone do not,
// keeping at least two key tiles per split.
int auto_splits(int B, int H, int N, int M) {
    const long units = (long)((N + 255) / 256) * B * H;
    const long sms = num_sms();
    if (sms <= 0 || units >= sms) return 1;
    long S = (sms + units - 1) / units;
    const long per = ((long)M + 127) / 128 / 2;
    if (S > per) S = per;
    if (S > kMaxSplits) S = kMaxSplits;
    return S < 1 ? 1 : (int)S;
}
}  // namespace

extern "C" {

int fa_version(void) { return FA_VERSION; }

const char* fa_last_cuda_error(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

int fa_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int M, int d,
                float scale, int causal, int in_dtype, int out_dtype, void* stream) {
    const int chk = check_attn_args(Q, K, V, O, LSE, B, H, N, M, d, scale, causal, in_dtype, out_dtype);
    if (chk != FA_OK) return chk;
    return attn_launch(Q, K, V, O, LSE, B, H, N, M, d, contiguous_strides(H, N, M, d), scale, causal, 1, nullptr,
                       nullptr, in_dtype, out_dtype, stream);
}

int fa_attn_fwd_strided(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int M,
                        int d, const long long* q_stride, const long long* k_stride, const long long* v_stride,
                        const long long* o_stride, float scale, int causal, int in_dtype, int out_dtype,
                        void* stream) {
    const int chk = check_attn_args(Q, K, V, O, LSE, B, H, N, M, d, scale, causal, in_dtype, out_dtype);
    if (chk != FA_OK) return chk;
    if (!q_stride || !k_stride || !v_stride || !o_stride) return FA_ERR_INVALID_ARG;
    const int ie = in_dtype == FA_BF16 ? 2 : 4, oe = out_dtype == FA_BF16 ? 2 : 4;
    if (!strides_ok(q_stride, ie) || !strides_ok(k_stride, ie) || !strides_ok(v_stride, ie) ||
        !strides_ok(o_stride, oe))
        return FA_ERR_MISALIGNED;
    Strides st;
    for (int i = 0; i < 3; ++i) {
        st.q[i] = q_stride[i]; st.k[i] = k_stride[i]; st.v[i] = v_stride[i]; st.o[i] = o_stride[i];
    }
    return attn_launch(Q, K, V, O, LSE, B, H, N, M, d, st, scale, causal, 1, nullptr, nullptr, in_dtype, out_dtype,
                       stream);
}

int fa_attn_splitkv_num_splits(int B, int H, int N, int M, int d, int causal) {
    (void)d;
    (void)causal;
    if (B <= 0 || H <= 0 || N <= 0 || M <= 0) return 1;
    return auto_splits(B, H, N, M);
}

long fa_attn_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits) {
    if (B <= 0 || H <= 0 || N <= 0 || d <= 0 || num_splits < 1 || num_splits > kMaxSplits) return -1;
    if (num_splits == 1) return 0;
    return splitkv_bytes((long)B * H, N, d, num_splits, nullptr);
}

int fa_attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int M,
                        int d, float scale, int causal, int num_splits, void* workspace, long workspace_bytes,
                        int in_dtype, int out_dtype, void* stream) {
    const int chk = check_attn_args(Q, K, V, O, LSE, B, H, N, M, d, scale, causal, in_dtype, out_dtype);
    if (chk != FA_OK) return chk;
    if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
    const int S = num_splits == 0 ? auto_splits(B, H, N, M) : num_splits;
    if (S == 1) return fa_attn_fwd(Q, K, V, O, LSE, B, H, N, M, d, scale, causal, in_dtype, out_dtype, stream);
    if (in_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    const long bh = (long)B * H;
    long loff = 0;
    const long need = splitkv_bytes(bh, N, d, S, &loff);
    if (workspace == nullptr || workspace_bytes < need) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_MISALIGNED;
    float* opart = static_cast<float*>(workspace);
    float* lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + loff);
    return attn_launch(Q, K, V, O, LSE, B, H, N, M, d, contiguous_strides(H, N, M, d), scale, causal, S, opart, lpart,
                       in_dtype, out_dtype, stream);
}

namespace {

int softmax_rows_impl(const void* X, void* P, float* LSE, long rows, long cols, int in_dtype, int out_dtype,
                      int log_out, void* stream) {
    if (!X || !P) return FA_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || !mul_fits(rows, cols, 1L << 60)) return FA_ERR_INVALID_ARG;
    if ((in_dtype != FA_F32 && in_dtype != FA_BF16) || (out_dtype != FA_F32 && out_dtype != FA_BF16))
        return FA_ERR_UNSUPPORTED;
    if (!aligned16(X) || !aligned16(P) || (LSE && !aligned16(LSE))) return FA_ERR_MISALIGNED;
    int err = FA_OK;
    int* status = status_word(&err);
    if (status == nullptr) return err;
    const cudaError_t e = fa::launch_softmax_rows(X, P, LSE, rows, cols, in_dtype == FA_BF16, out_dtype == FA_BF16,
                                                  log_out, status, static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

int lse_rows_impl(const void* X, const long long* labels, float* loss, float* LSE, long rows, long cols,
                  int in_dtype, void* stream) {
    if (!X || (!LSE && !loss) || (loss && !labels)) return FA_ERR_INVALID_ARG;
    if (rows <= 0 || cols <= 0 || !mul_fits(rows, cols, 1L << 60)) return FA_ERR_INVALID_ARG;
    if (in_dtype != FA_F32 && in_dtype != FA_BF16) return FA_ERR_UNSUPPORTED;
    if (!aligned16(X) || (LSE && !aligned16(LSE)) || (loss && !aligned16(loss)) || (labels && !aligned16(labels)))
        return FA_ERR_MISALIGNED;
    int err = FA_OK;
    int* status = status_word(&err);
    if (status == nullptr) return err;
    const cudaError_t e = fa::launch_logsumexp_rows(X, LSE, rows, cols, in_dtype == FA_BF16, labels, loss, status,
                                                    static_cast<cudaStream_t>(stream));
    return cuda_status(e);
}

}  // namespace

int fa_softmax_rows(const void* X, void* P, float* LSE, long rows, long cols, int in_dtype, int out_dtype,
                    void* stream) {
    return softmax_rows_impl(X, P, LSE, rows, cols, in_dtype, out_dtype, 0, stream);
}

int fa_log_softmax_rows(const void* X, void* Y, float* LSE, long rows, long cols, int in_dtype, int out_dtype,
                        void* stream) {
    return softmax_rows_impl(X, Y, LSE, rows, cols, in_dtype, out_dtype, 1, stream);
}

int fa_logsumexp_rows(const void* X, float* LSE, long rows, long cols, int in_dtype, void* stream) {
    if (!LSE) return FA_ERR_INVALID_ARG;
    return lse_rows_impl(X, nullptr, nullptr, LSE, rows, cols, in_dtype, stream);
}

int fa_cross_entropy_rows(const void* X, const long long* labels, float* loss, float* LSE, long rows, long cols,
                          int in_dtype, void* stream) {
    if (!loss || !labels) return FA_ERR_INVALID_ARG;
    return lse_rows_impl(X, labels, loss, LSE, rows, cols, in_dtype, stream);
}

int fa_device_status(void* stream, int reset) {
    int err = FA_OK;
    int* status = status_word(&err);
    if (status == nullptr) return err;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    int v = 0;
    e = cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    if (reset && v != 0) {
        const int zero = 0;
        e = cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return v == 0 ? FA_OK : v;
}

int fa_selftest_wait_timeout(int limit_us, void* stream) {
    if (limit_us < 1 || limit_us > 1000000) return FA_ERR_INVALID_ARG;
    int err = FA_OK;
    int* status = status_word(&err);
    if (status == nullptr) return err;
    const cudaError_t e = fa::launch_selftest_wait(status, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    return fa_device_status(stream, 1);
}

}  // extern "C"
