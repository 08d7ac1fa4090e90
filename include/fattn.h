/*
 * fattn.h -- C ABI of libfattn: exact attention forward with the online-softmax
 * recurrence, and row-wise online softmax / log-sum-exp, for NVIDIA GB300
 * (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor arguments are DEVICE pointers owned by the caller.  The library
 *    never allocates, frees or retains device memory, and never reads host
 *    memory through these pointers.
 *  - Every pointer must be 16-byte aligned (FA_ERR_MISALIGNED otherwise).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls are asynchronous: they validate, enqueue and return.  A
 *    launch failure is reported as FA_ERR_CUDA; nothing is synchronised.
 *  - Argument errors are detected before anything is enqueued; on any non-OK
 *    status no output has been written.
 *  - dtype codes: FA_F32 (IEEE binary32) and FA_BF16 (bfloat16).  All
 *    arithmetic inside the kernels is fp32; bf16 stores round to nearest even.
 *  - LSE is always fp32 and in natural-log units.
 *  - Device kernels never spin without a bound.  A wait that exceeds its bound
 *    makes the kernel give up, leave its outputs incomplete and record
 *    FA_ERR_DEVICE_TIMEOUT in a per-device status word that
 *    fa_device_status() returns.
 *  - Re-entrant; the only global state is per-device kernel attributes, the
 *    device status word, a cache of encoded TMA tensor maps and, for the row
 *    kernels that hand their last rows out at run time, one counter word per
 *    CUDA stream (256 per device, in the library's own device memory; the
 *    launches on a stream run in order, each leaving its word zero for the
 *    next; later streams, and launches into a stream capture, split their
 *    rows statically).
 */
#ifndef FATTN_H
#define FATTN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_dtype {
    FA_F32 = 0,
    FA_BF16 = 1
} fa_dtype;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, overflow  */
    FA_ERR_UNSUPPORTED = 2,     /* valid but not implemented (dtype, head dim) */
    FA_ERR_MISALIGNED = 3,      /* a pointer is not 16-byte aligned           */
    FA_ERR_CUDA = 4,            /* the CUDA runtime reported an error         */
    FA_ERR_DEVICE_TIMEOUT = 5   /* a kernel's bounded wait ran out            */
} fa_status;

#define FA_VERSION 100  /* 1.0.0 */

/*
 * fa_attn_fwd -- O = softmax(scale * Q K^T [+ causal mask]) V and the per-row
 * log-sum-exp of the scaled, masked scores, in one fused pass.
 *
 * Defined by: "什么是 online softmax and flash attention", section
 * "Attention的数学表达", eq (8)-(9) (shapes Q[N,K], K[M,K], V[M,K], A[N,K]
 * with K the head dimension), computed by the block-wise online merge of the
 * running max m, normaliser l and unnormalised output o~ given on
 * "从原始Softmax到在线Softmax", section on the block-wise online softmax
 * (o = o~ / l after the last key block); LSE as defined on the same page,
 * section "softmax形式推导".
 *
 *   Q    [B, H, N, d]  row-major, d fastest, dtype in_dtype
 *   K    [B, H, M, d]  row-major, dtype in_dtype
 *   V    [B, H, M, d]  row-major, dtype in_dtype
 *   O    [B, H, N, d]  row-major, dtype out_dtype (written)
 *   LSE  [B, H, N]     fp32, natural log of sum_j exp(scale * q_i . k_j) over
 *                      the keys kept for row i (written; may be NULL = skip)
 *   scale  multiplier of Q K^T: finite and > 0, usually 1/sqrt(d)
 *   causal 0: every key is kept; 1: key j is kept for query i iff j <= i
 *          (top-left aligned, also when N != M); 2: iff j <= i + (M - N)
 *          (bottom-right aligned: the last query sees every key).  A query
 *          that keeps no key (causal = 2 with N > M) gets O = 0, LSE = -inf.
 *   in_dtype / out_dtype:
 *      FA_BF16 in  -> tensor-core path, d in {64, 128}; out FA_BF16 or FA_F32
 *      FA_F32  in  -> fp32 CUDA-core path, d in {16, 32, 64, 128}; out FA_F32
 * Errors: FA_ERR_INVALID_ARG for NULL Q/K/V/O, B,H,N,M,d <= 0, a scale that is
 * not finite or not > 0, or sizes whose element count overflows;
 * FA_ERR_UNSUPPORTED for other dtype / d combinations; FA_ERR_MISALIGNED;
 * FA_ERR_CUDA.
 */
int fa_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                int B, int H, int N, int M, int d, float scale, int causal,
                int in_dtype, int out_dtype, void* stream);

/*
 * fa_attn_fwd_strided -- fa_attn_fwd on tensors with arbitrary batch, head and
 * row strides (e.g. the [B, N, H, d] layout), d contiguous in every tensor.
 *
 *   q_stride, k_stride, v_stride, o_stride: 3 element strides each, in the
 *       order (batch, head, row); positive, and each a multiple of 16 bytes.
 *       [B, H, N, d] is {H*N*d, N*d, d}; [B, N, H, d] is {N*H*d, d, H*d}.
 *   LSE stays [B, H, N] contiguous.  Everything else as fa_attn_fwd.
 * Errors: as fa_attn_fwd, plus FA_ERR_INVALID_ARG for a NULL stride array and
 * FA_ERR_MISALIGNED for a stride that breaks the 16-byte rule.
 */
int fa_attn_fwd_strided(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        int B, int H, int N, int M, int d,
                        const long long* q_stride, const long long* k_stride,
                        const long long* v_stride, const long long* o_stride,
                        float scale, int causal, int in_dtype, int out_dtype, void* stream);

/*
 * fa_attn_fwd_splitkv -- fa_attn_fwd with the key tiles of each 256-row query
 * block split over `num_splits` CTAs, for shapes with too few (batch, head,
 * query block) units to fill the GPU (few heads, short query, long keys).
 * Split s returns a normalised partial output o_s and its log-sum-exp LSE_s;
 * a second kernel merges them:
 *     LSE = log sum_s e^{LSE_s},   O = sum_s e^{LSE_s - LSE} o_s,
 * the merge of normalised block results of "从原始Softmax到在线Softmax",
 * section on the block-wise online softmax (l_s = e^{LSE_s}).
 *
 *   Q, K, V, O, LSE, B, H, N, M, d, scale, causal, in_dtype, out_dtype:
 *       as fa_attn_fwd; splitting (num_splits > 1) needs in_dtype FA_BF16.
 *   num_splits  1..64, or 0 = fa_attn_splitkv_num_splits(); 1 is fa_attn_fwd.
 *   workspace   caller-owned device scratch of at least
 *               fa_attn_splitkv_workspace_bytes(B, H, N, d, S) bytes, 256-byte
 *               aligned (fp32 partials [S][B*H][N][d], then fp32 LSE_s
 *               [S][B*H][N]); not needed (may be NULL) when S = 1.  Its
 *               contents are overwritten; calls sharing one workspace must not
 *               overlap on the GPU.
 * Errors: as fa_attn_fwd, plus FA_ERR_INVALID_ARG for num_splits outside
 * 0..64 or a missing/too small workspace, FA_ERR_MISALIGNED for a workspace
 * not 256-byte aligned, FA_ERR_UNSUPPORTED for fp32 inputs with S > 1.
 */
int fa_attn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        int B, int H, int N, int M, int d, float scale, int causal,
                        int num_splits, void* workspace, long workspace_bytes,
                        int in_dtype, int out_dtype, void* stream);

/* The split count fa_attn_fwd_splitkv uses for num_splits = 0 on the current
 * device: 1 when the (batch, head, query block) units already fill it,
 * otherwise enough splits to cover every SM, at most 64 and at least two key
 * tiles per split.  (No counterpart on the pages.) */
int fa_attn_splitkv_num_splits(int B, int H, int N, int M, int d, int causal);

/* Workspace bytes fa_attn_fwd_splitkv needs for num_splits (1..64) splits;
 * 0 for one split, -1 for invalid arguments.  (No counterpart on the pages.) */
long fa_attn_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits);

/* Size of the fixed scratch fa_attn_fwd_splitkv_noalloc uses: 32 MiB. */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * fa_attn_fwd_splitkv_noalloc -- fa_attn_fwd_splitkv for callers that cannot
 * allocate device memory: code whose device memory is owned by another
 * allocator (a framework's caching pool, a host program that hands a plugin
 * only its inputs and outputs), or code that must not call cudaMalloc or
 * cudaFree, for instance because cudaFree can synchronise the whole device.
 * Instead of a caller workspace it uses one scratch array of
 * FA_NOALLOC_SCRATCH_BYTES built into the library.  A device holds that array
 * from the moment the library's device code is loaded on it (at the latest the
 * first call of any libfattn entry point on that device; at once under eager
 * module loading) until the process exits.  It allocates nothing itself.
 * (The pages have no counterpart: this is a deployment entry point.)
 *
 *   Arguments: as fa_attn_fwd_splitkv, without workspace / workspace_bytes.
 *   Size limit: the split partials, fa_attn_splitkv_workspace_bytes(B, H, N,
 *       d, S), must fit in FA_NOALLOC_SCRATCH_BYTES; larger problems are
 *       rejected with FA_ERR_INVALID_ARG before anything is enqueued.
 *   Set-up: the first call made with a given device current looks up the
 *       scratch array's device address (cudaGetSymbolAddress) and caches it;
 *       make that first call before any stream capture.
 *   Sharing: all calls on a device use the same scratch, which keeps the last
 *       call's contents (nothing in it needs to start at zero).  Calls that
 *       overlap on the GPU (other streams, other host threads) race on it;
 *       the caller must serialise them.
 *   Failures: if a kernel's bounded wait runs out, the combine step may merge
 *       partials left by an earlier call; O and LSE are defined only when
 *       fa_device_status() returns FA_OK after the call.
 * Errors: as fa_attn_fwd_splitkv, FA_ERR_INVALID_ARG for the size limit, and
 * FA_ERR_CUDA if the scratch address cannot be looked up.
 */
int fa_attn_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                int B, int H, int N, int M, int d, float scale, int causal,
                                int num_splits, int in_dtype, int out_dtype, void* stream);

/*
 * fa_softmax_rows -- P[r, :] = softmax(X[r, :]) and LSE[r] = log sum_c exp X[r, c]
 * for every row, reading X from memory once when a row fits on chip
 * (cols <= 65536 for bf16, <= 32768 for fp32) and twice otherwise.
 *
 * Defined by: "从原始Softmax到在线Softmax", section "softmax形式推导" (stable
 * softmax, log-sum-exp), computed with the online normaliser of
 * "什么是 online softmax and flash attention", section "Online softmax",
 * eq (3)-(7), merged across threads with the pairwise form of the same update.
 *
 *   X    [rows, cols]  row-major, dtype in_dtype (FA_BF16 or FA_F32)
 *   P    [rows, cols]  row-major, dtype out_dtype (FA_BF16 or FA_F32), written;
 *                      must not be NULL and must not overlap X
 *   LSE  [rows]        fp32, written; may be NULL = skip
 * Errors: FA_ERR_INVALID_ARG for NULL X/P, rows <= 0, cols <= 0, or
 * rows*cols overflowing; FA_ERR_UNSUPPORTED for other dtypes;
 * FA_ERR_MISALIGNED; FA_ERR_CUDA.
 */
int fa_softmax_rows(const void* X, void* P, float* LSE, long rows, long cols,
                    int in_dtype, int out_dtype, void* stream);

/*
 * fa_logsumexp_rows -- LSE[r] = log sum_c exp X[r, c], one read of X.
 *
 * Defined by: "从原始Softmax到在线Softmax", section "softmax形式推导" (the
 * LSE(z) definition), computed with the online normaliser of
 * "什么是 online softmax and flash attention", section "Online softmax".
 *
 *   X    [rows, cols]  row-major, dtype in_dtype (FA_BF16 or FA_F32)
 *   LSE  [rows]        fp32, written; must not be NULL
 * Errors: as fa_softmax_rows.
 */
int fa_logsumexp_rows(const void* X, float* LSE, long rows, long cols,
                      int in_dtype, void* stream);

/*
 * fa_log_softmax_rows -- Y[r, :] = log softmax(X[r, :]) = X[r, :] - LSE[r],
 * the log-softmax identity log p_j = z_j - LSE(z) of "从原始Softmax到在线Softmax",
 * section "softmax形式推导", with LSE from the same online reduction as
 * fa_softmax_rows (one read of X when a row fits on chip).
 *
 *   X    [rows, cols]  row-major, FA_BF16 or FA_F32
 *   Y    [rows, cols]  row-major, FA_BF16 or FA_F32, written; must not overlap X
 *   LSE  [rows]        fp32, written; may be NULL
 * Errors: as fa_softmax_rows.
 */
int fa_log_softmax_rows(const void* X, void* Y, float* LSE, long rows, long cols,
                        int in_dtype, int out_dtype, void* stream);

/*
 * fa_cross_entropy_rows -- per-row cross-entropy of logits X against integer
 * labels: loss[r] = LSE(X[r, :]) - X[r, labels[r]] = -log softmax(X[r, :])[label],
 * the log-softmax-then-negative-log-likelihood of the cross_entropy_loss sketch
 * on "从原始Softmax到在线Softmax" (section "softmax实际代码实现"; worked example 2
 * gives 0.4170), fused into the log-sum-exp pass: one read of X.  The batch
 * mean of that sketch is left to the caller.
 *
 *   X       [rows, cols]  row-major logits, FA_BF16 or FA_F32
 *   labels  [rows]        int64 class indices; a label outside [0, cols)
 *                         (e.g. -100) marks an ignored row whose loss is 0
 *   loss    [rows]        fp32, written; must not be NULL
 *   LSE     [rows]        fp32, written; may be NULL
 * Errors: FA_ERR_INVALID_ARG for NULL X/labels/loss or bad sizes;
 * FA_ERR_UNSUPPORTED for other dtypes; FA_ERR_MISALIGNED; FA_ERR_CUDA.
 */
int fa_cross_entropy_rows(const void* X, const long long* labels, float* loss, float* LSE,
                          long rows, long cols, int in_dtype, void* stream);

/*
 * fa_device_status -- synchronise `stream`, then return FA_OK or the first
 * error a kernel recorded on the current device since the last reset
 * (FA_ERR_DEVICE_TIMEOUT), or FA_ERR_CUDA if the synchronisation itself
 * failed.  reset != 0 clears the recorded status.  (No counterpart on the
 * pages: this is the library's failure-detection hook.)
 */
int fa_device_status(void* stream, int reset);

/*
 * fa_selftest_wait_timeout -- launch one CTA that waits on a barrier nothing
 * ever completes, with a bound of `limit_us` microseconds (1..1000000), then
 * return fa_device_status(stream, 1).  Expected result: FA_ERR_DEVICE_TIMEOUT
 * with the CUDA context still usable.  Exercises the same bounded-wait code
 * every pipelined kernel uses.  (No counterpart on the pages.)
 */
int fa_selftest_wait_timeout(int limit_us, void* stream);

/*
 * fa_last_cuda_error -- the CUDA runtime's message for the error behind the
 * most recent FA_ERR_CUDA returned on the calling thread ("no error" if none).
 * Static storage, never NULL.  (No counterpart on the pages.)
 */
const char* fa_last_cuda_error(void);

/* Human-readable name of a status code (static storage, never NULL). */
const char* fa_status_string(int status);

/* FA_VERSION of the built library. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FATTN_H */
