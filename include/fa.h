/*
 * fa.h - C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * The operation ("用 CuTe 读懂 FlashAttention：一次 forward 的完整流程",
 * section "先固定一个例子", equation S = QK^T, P = softmax_row(sS), O = PV;
 * "CUDA 算子工程" ch. 14, section 14.1):
 *
 *   for each batch b, head h and query row i < N,
 *     O[b,h,i,:] = sum_j softmax_j(s * q_i . k_j) * v_j
 *     LSE[b,h,i] = ln sum_j exp(s * q_i . k_j)
 *   over the keys j < N, and only j <= i when `causal` is non-zero (top-left
 *   alignment, section "causal 模式在哪一步生效", Fig. 11).  LSE is the
 *   side output s*m + ln(l) of section "最后：归一化并写回 O".
 *
 * The library computes this in one kernel launch, FlashAttention-2 loop
 * order (query tiles of 128 rows, walked by one persistent CTA per SM;
 * key/value tiles streamed through shared memory; scores and weights kept
 * in tensor memory, never in HBM).
 *
 * This header needs no CUDA header: streams are passed as void*.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
#define FA_OK 0               /* success (for fa_fwd: validated and enqueued)            */
#define FA_ERR_INVALID_ARG 1  /* null pointer, non-positive size, bad dtype, bad scale    */
#define FA_ERR_UNSUPPORTED 2  /* valid request outside the compiled set (head dim d), or a
                                 split-KV request larger than the no-alloc scratch array   */
#define FA_ERR_MISALIGNED 3   /* q, k, v or o not 16-byte aligned; lse not 4-byte aligned */
#define FA_ERR_CUDA 4         /* a CUDA runtime/driver call failed (launch, encode, sync) */
#define FA_ERR_TIMEOUT 5      /* a pipeline wait inside the kernel ran out of time        */

/* Element types of q, k, v and o. */
#define FA_FP16 0             /* IEEE binary16 */
#define FA_BF16 1             /* bfloat16      */

/*
 * fa_fwd - fused scaled-dot-product attention forward with log-sum-exp.
 *
 * q, k, v : device pointers, [B, H, N, d] contiguous (row-major, d fastest),
 *           element type `dtype`.  Read only.
 * o       : device pointer, [B, H, N, d] contiguous, element type `dtype`.
 *           Written: every row i < N of every (b, h).  O is the exact softmax
 *           average of the 16-bit-rounded weights, rounded to nearest even.
 * lse     : device pointer, [B, H, N] contiguous float32.  Written: the natural
 *           log-sum-exp of the scaled scores of each row.
 * B, H, N : batch, heads, sequence length (queries = keys = N); each >= 1.
 *           B*H and N must each fit the TMA tensor map (< 2^31).
 * d       : head dimension: a multiple of 8 from 8 to 256 (else
 *           FA_ERR_UNSUPPORTED).  64, 128, 192 and 256 run kernels of exactly
 *           that width; any other d runs the next wider one, whose extra
 *           columns are zero-filled on load and never stored (same result,
 *           the time of the wider kernel).
 * scale   : the softmax scale s (for the standard definition 1/sqrt(d)); must
 *           be finite and > 0.  There is no default.
 * causal  : 0 = full attention, non-zero = key j visible to query i iff j <= i.
 * dtype   : FA_FP16 or FA_BF16.
 * stream  : cudaStream_t to enqueue on (NULL = the legacy default stream).
 *
 * Ownership: the caller owns all buffers; the library allocates no device
 * memory per call and keeps no pointer after the call returns.  q, k, v must
 * not overlap o or lse.
 * Asynchrony: the kernel is enqueued on `stream`; the return value covers
 * argument checks, tensor-map encoding and the launch itself.  Errors inside
 * the kernel (a pipeline wait that timed out) are reported by
 * fa_check_device_status().
 * Thread safety: safe to call concurrently from several host threads.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, int dtype,
           void* stream);

/*
 * fa_fwd_ex - the general form: separate query and key lengths, strided
 * tensors, three masks, optional split-KV.  Fields of fa_fwd_args:
 *   q [B, H, Nq, d], k and v [B, H, Nk, d], o [B, H, Nq, d]: 16-bit device
 *     tensors, d contiguous; *_stride = {batch, head, row} strides in
 *     elements, each a positive multiple of 8 (16 bytes, a TMA rule), e.g.
 *     {H*N*d, N*d, d} for [B, H, N, d] or {N*H*d, d, H*d} for [B, N, H, d].
 *     Base pointers 16-byte aligned (else FA_ERR_MISALIGNED).
 *   lse [B, H, Nq] fp32 with rows contiguous and lse_stride = {batch, head}.
 *   mask: FA_MASK_NONE; FA_MASK_CAUSAL_TOP_LEFT (key j visible to query i
 *     iff j <= i, section "causal 模式在哪一步生效", Fig. 11); or
 *     FA_MASK_CAUSAL_BOTTOM_RIGHT (j <= i + Nk - Nq, the alignment that
 *     section mentions for unequal lengths: the last query sees every key).
 *     A query that sees no key gets O = 0 and LSE = -inf.
 *   num_splits, workspace, workspace_bytes: as fa_fwd_splitkv (1 = none;
 *     the workspace size is fa_splitkv_workspace_size(B, H, Nq, d, splits)).
 *   scale, dtype, stream: as fa_fwd.
 * fa_fwd(...) is fa_fwd_ex with contiguous strides, Nq = Nk = N and the
 * top-left mask when `causal`.
 */
#define FA_MASK_NONE 0
#define FA_MASK_CAUSAL_TOP_LEFT 1
#define FA_MASK_CAUSAL_BOTTOM_RIGHT 2

typedef struct fa_fwd_args {
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    int B, H, Nq, Nk, d;
    long long q_stride[3];
    long long k_stride[3];
    long long v_stride[3];
    long long o_stride[3];
    long long lse_stride[2];
    float scale;
    int mask;
    int dtype;
    int num_splits;
    void* workspace;
    size_t workspace_bytes;
    void* stream;
} fa_fwd_args;

int fa_fwd_ex(const fa_fwd_args* args);

/*
 * Split-KV ("CUDA 算子工程" ch. 14, section 14.7.1): when B*H*ceil(N/256) query
 * blocks cannot fill the GPU, the key tiles of every block are divided into
 * num_splits contiguous ranges processed by separate CTAs; each writes a
 * partial O (fp32, normalised by its own weights) and partial log-sum-exps to
 * a caller-provided workspace, and a second kernel merges them:
 *   LSE = ln sum_s e^{LSE_s},  O = sum_s w_s O_s / sum_s w_s,
 * w_s being range s's sum of the 16-bit weights fed to P.V on a common scale.
 * The result matches fa_fwd within rounding.
 */
#define FA_MAX_SPLITS 32

/* Split count the library would choose for this shape on the current device:
 * 1 (fa_fwd is better) unless the query blocks fill less than half of the SMs,
 * or, with causal != 0, no more than all of them (a causal wave lasts as long
 * as its longest block); then about one wave of CTAs, with at least four key
 * tiles per range. */
int fa_splitkv_num_splits(int B, int H, int N, int d, int causal);

/* The split count fa_fwd_ex chooses for num_splits = 0 with these arguments:
 * as fa_splitkv_num_splits, with the keys per range counted from Nk (so one
 * query row against a long key sequence, as in decoding, is split). */
int fa_splitkv_num_splits_ex(const fa_fwd_args* args);

/* Workspace bytes fa_fwd_splitkv needs for num_splits >= 2 (0 otherwise, or
 * for an unsupported d).  Partial O rows are as wide as the kernel serving d. */
size_t fa_splitkv_workspace_size(int B, int H, int N, int d, int num_splits);

/*
 * fa_fwd_splitkv - fa_fwd computed in num_splits key ranges plus a merge.
 * Arguments as fa_fwd, plus:
 * num_splits      : 1 = plain fa_fwd (workspace unused), 2..FA_MAX_SPLITS =
 *                   that many ranges, 0 = fa_splitkv_num_splits().
 * workspace       : device memory owned by the caller, 256-byte aligned, at
 *                   least fa_splitkv_workspace_size() bytes; overwritten; must
 *                   not be shared by calls that may run at the same time.
 * workspace_bytes : its size (FA_ERR_INVALID_ARG if too small).
 * Both kernels are enqueued on `stream`; the library allocates nothing.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal, int dtype,
                   int num_splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_splitkv_noalloc - fa_fwd_splitkv for callers that cannot allocate
 * device memory (no counterpart on the pages: the pages do not discuss who
 * allocates the split-KV partials).  Some callers cannot call cudaMalloc: a
 * plugin whose host framework owns all device memory, or a latency-critical
 * path that cannot take cudaMalloc's implicit synchronisation.  This entry
 * point keeps the partials in a fixed array of FA_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until exit; it
 * calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments as fa_fwd_splitkv without the workspace, checked in the same
 * order as every other entry point (FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED
 * for d, FA_ERR_MISALIGNED before any size rule of the array).
 * num_splits      : 1 = plain fa_fwd (the array is not used); 2..FA_MAX_SPLITS
 *                   = that many ranges, FA_ERR_UNSUPPORTED when
 *                   fa_splitkv_workspace_size() of that count is above
 *                   FA_NOALLOC_SCRATCH_BYTES (use fa_fwd_splitkv with a
 *                   workspace instead); 0 = fa_splitkv_num_splits(), lowered
 *                   until the partials fit the array (down to 1 = fa_fwd),
 *                   so the library's own choice is never refused.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for the
 * process; make that first call before any stream capture.  cudaDeviceReset
 * unloads the library's device code, so the kept address is stale afterwards:
 * do not call this entry point after resetting a device it has run on.  All
 * calls share the one array and its contents persist from call to call; calls
 * that may overlap on the GPU race, so order them (one stream, or events).
 */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int N, int d, float scale, int causal, int dtype,
                           int num_splits, void* stream);

/*
 * fa_check_device_status - synchronise `stream`, then return and clear the
 * device-side status word: FA_OK, FA_ERR_TIMEOUT (some CTA's bounded wait
 * expired and that CTA left its outputs unwritten), or FA_ERR_CUDA if the
 * synchronisation itself failed.  The status word is shared by all launches
 * on the current device.
 */
int fa_check_device_status(void* stream);

/* fa_status_string - static, human-readable name of a status code. */
const char* fa_status_string(int status);

/* fa_version - library version as major*10000 + minor*100 + patch. */
int fa_version(void);

/*
 * fa_fwd_debug - fa_fwd with testing controls; not for production use.
 * fault_mode : 0 = none; 1 = the loader never issues the first key tile, so
 *              the tensor-core warp's wait for it must time out, set
 *              FA_ERR_TIMEOUT and let every CTA exit cleanly; 2 = the launch
 *              step reports failure instead of launching (the call returns
 *              FA_ERR_CUDA, as for a failed cudaLaunchKernel, and nothing is
 *              enqueued).
 * timeout_s  : limit of every pipeline wait, in seconds (> 0; fa_fwd uses 2 s).
 */
int fa_fwd_debug(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal, int dtype,
                 void* stream, int fault_mode, double timeout_s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
