/*
 * fa.h — C ABI of the GB300 (sm_103a) FlashAttention-style attention forward.
 *
 * Operation (non-causal scaled-dot-product attention with row log-sum-exp):
 *
 *   S = scale * Q K^T (+ mask broadcast over heads and query rows)
 *   O = softmax_row(S) V,   LSE_i = ln sum_j exp(S_ij)
 *
 * computed block by block with an online softmax (running row max m, running
 * denominator l, rescaled accumulator), so the Nq x Nk score matrix never
 * reaches device memory.  Sources:
 *  - "算子加速：注意力、编译与融合" (anrans.github.io ai-infra-handbooks, perf/kernels),
 *    section "注意力：从O(N²)显存到分块": the figure (per K/V block: S_ij = Q_i K_j^T,
 *    update m and l, O_i <- O_i e^(m_old - m) + P V_j, only O_i is written
 *    back) and the `blocked` worked example (the m / l / acc recurrence);
 *  - "FlashAttention原理与工业实战" (sheratonhq.com) §2.3: the forward kernel
 *    writes Out and a per-row Lse; §4.3: inputs must be contiguous [B,H,N,D];
 *  - "Step 3.7 Flash" (pwwt.cn) §2.3 and §3.1: scale first, then add the
 *    additive attention mask; non-causal (is_causal=False).
 *
 * All functions are thread-safe.  The library allocates no device memory.
 */
#ifndef UNET_FA_FWD_GB300_FA_H
#define UNET_FA_FWD_GB300_FA_H

#include <stddef.h>

/* The library exports these functions only; everything else is hidden. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARGUMENT = 1, /* NULL pointer, bad size, misaligned or overlapping buffer, non-finite scale */
    FA_ERR_UNSUPPORTED = 2,      /* head dimension D not in {32, 64, 128}; device not sm_103 */
    FA_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
    FA_ERR_TIMEOUT = 4,          /* a kernel wait ran past its time limit (read with fa_read_device_status) */
    FA_ERR_DEBUG_CHECK = 5       /* debug builds: a device-side bounds or schedule check failed
                                    (read with fa_read_device_status; details: fa_debug_report) */
} fa_status;

/*
 * fa_fwd — attention forward on the GPU.
 *
 *   q     device pointer, bf16 [B, H, Nq, D], contiguous row-major
 *   k, v  device pointers, bf16 [B, H, Nk, D], contiguous row-major
 *   mask  device pointer to an fp32 additive key mask [B, Nk] (0 = keep,
 *         -inf = ignore; any finite value is added to the scaled score), or
 *         NULL for no mask.  Broadcast over heads and query rows.
 *   out   device pointer, bf16 [B, H, Nq, D]: O
 *   lse   device pointer, fp32 [B, H, Nq]: natural-log row log-sum-exp of the
 *         scaled, masked scores
 *   B, H, Nq, Nk  >= 1;  D in {32, 64, 128}
 *   scale finite; multiplies Q K^T before the mask is added
 *   stream  cudaStream_t (as void*), NULL = the legacy default stream
 *
 * A row whose keys are all masked gives O = 0 and LSE = -inf.
 *
 * Ownership: the caller owns every buffer; nothing is retained after the call
 * returns (TMA descriptors are encoded per call and passed by value).  Every
 * pointer must be 16-byte aligned (a TMA requirement); out and lse must not
 * overlap q, k, v, mask or each other.
 *
 * Errors: arguments are validated before any CUDA call; an invalid call
 * returns FA_ERR_INVALID_ARGUMENT or FA_ERR_UNSUPPORTED and launches nothing.
 * FA_ERR_CUDA means a launch or set-up call failed.  FA_OK means the kernel
 * was enqueued on `stream` (the call is asynchronous); a kernel that ran out
 * of time on an internal wait records FA_ERR_TIMEOUT in the device status
 * word (see fa_read_device_status) and exits without hanging.
 */
FA_API int fa_fwd(const void* q, const void* k, const void* v, const float* mask, void* out, float* lse,
           int B, int H, int Nq, int Nk, int D, float scale, void* stream);

/* Kinds of mask fa_fwd_ex accepts. */
typedef enum {
    FA_MASK_NONE = 0,
    FA_MASK_KEY_PADDING = 1, /* fp32 [B, Nk], added to every query row (as fa_fwd's mask) */
    FA_MASK_ADDITIVE = 2,    /* fp32 [B, heads, Nq, Nk], added to each scaled score */
    FA_MASK_BOOL = 3         /* uint8 [B, heads, Nq, Nk]: nonzero keeps the pair, 0 excludes it */
} fa_mask_kind;

/* A mask for fa_fwd_ex: `data` is a contiguous device array of the kind's
 * layout; `heads` (ADDITIVE and BOOL) is 1 to broadcast over heads, or H. */
typedef struct fa_mask {
    int kind;
    const void* data;
    int heads;
} fa_mask;

/*
 * fa_fwd_ex — fa_fwd with general masks and an optional causal triangle.
 *
 * A per-(query, key) additive mask is added after the scale, like the
 * key-padding mask ("Step 3.7 Flash" §2.3, where ignored positions carry a
 * large negative); a boolean mask excludes the pairs where it is 0, i.e. it
 * is the additive mask 0 / -inf ("FlashAttention原理与工业实战" §2.1,
 * masked_fill(mask == 0, -inf)).  causal != 0 also excludes key j > query i
 * (top-left aligned: row i sees keys 0..i, the lower-triangular mask of that
 * page's §4.3 causal example); key blocks entirely above the diagonal are not
 * computed.
 *
 *   mask  NULL or kind FA_MASK_NONE: no mask; otherwise as fa_mask above.  An
 *         ADDITIVE mask must be 4-byte aligned; a mask must not overlap out or lse.
 *         Speed, not results, depends on alignment: an ADDITIVE mask whose rows
 *         start 16-byte aligned (16-byte aligned data, Nk a multiple of 4) is
 *         copied tile by tile into shared memory by TMA; a BOOL mask with
 *         16-byte aligned rows is read 16 bytes at a time; other masks are
 *         read element by element.
 *   other arguments as fa_fwd.
 *
 * Rows left with no key give O = 0, LSE = -inf.  Errors as fa_fwd, plus
 * FA_ERR_INVALID_ARGUMENT for an unknown kind, NULL data, heads not 1 or H,
 * or a misaligned or overlapping mask.
 */
FA_API int fa_fwd_ex(const void* q, const void* k, const void* v, const fa_mask* mask, int causal,
              void* out, float* lse, int B, int H, int Nq, int Nk, int D, float scale,
              void* stream);

/*
 * fa_fwd_fp8 — the forward with Q K^T in FP8 (e4m3), SageAttention-style
 * ("算子加速：注意力、编译与融合", section "SageAttention": smooth K by
 * subtracting its mean, quantise, run the low-precision product; P and V stay
 * 16-bit, as in its first version).
 *
 * A pre-pass subtracts from K its per-channel mean over the keys of each head
 * (this moves every score of row i by the same q_i . mean, so the softmax is
 * unchanged and LSE is corrected by scale * q_i . mean), then quantises Q and
 * the smoothed K to e4m3 with one scale per 128-row block (block max / 448).
 * S = Q K^T runs on the tensor cores as kind::f8f6f4 (twice the bf16 rate,
 * half the MMA instructions); the block scales are folded into the softmax's
 * exp2 multiplier; P (bf16) V (bf16) is unchanged.  Results are close to, not
 * equal to, the bf16 forward: the error budget is looser (see the tests).
 *
 *   arguments as fa_fwd (mask: fp32 key padding [B, Nk] or NULL), plus
 *   workspace  device scratch, 16-byte aligned, at least
 *              fa_fp8_workspace_bytes(B, H, Nq, Nk, D) bytes, owned by the caller
 *              and not shared with a concurrent call.
 *
 * Four kernels are enqueued on `stream` (column sums of K, their means, the
 * quantisation of K and Q, attention).  Errors as fa_fwd, plus FA_ERR_INVALID_ARGUMENT for
 * a missing, misaligned, small or overlapping workspace.
 */
FA_API int fa_fwd_fp8(const void* q, const void* k, const void* v, const float* mask, void* out,
               float* lse, int B, int H, int Nq, int Nk, int D, float scale, void* workspace,
               size_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_fp8 needs (0 for invalid sizes). */
FA_API size_t fa_fp8_workspace_bytes(int B, int H, int Nq, int Nk, int D);

/*
 * fa_fwd_split — the same forward with the key axis cut into `num_splits`
 * ranges computed by separate work units, then merged.
 *
 * Each range r yields its own normalised partial output O_r and LSE_r; the
 * merge is exact: LSE = ln sum_r e^(LSE_r), O = sum_r e^(LSE_r - LSE) O_r.
 * This is the exchange step of ring (sequence-parallel) attention in
 * "FlashAttention原理与工业实战" §6.2, here on one GPU: it fills the SMs when
 * B*H*ceil(Nq/256) work units are fewer than the SM count (few heads, short
 * query sets, long key sets).
 *
 *   q, k, v, mask, out, lse, B, H, Nq, Nk, D, scale, stream: as in fa_fwd.
 *   num_splits  >= 1 requested ranges; the library uses min(num_splits, nkv)
 *               balanced ranges of whole 128-key blocks, nkv = ceil(Nk / 128).
 *               1 behaves exactly as fa_fwd.
 *   workspace   device scratch, 16-byte aligned, at least
 *               fa_split_workspace_bytes(B, H, Nq, D, num_splits) bytes; holds
 *               fp32 partial O [ranges][B*H][Nq][D] and LSE [ranges][B*H][Nq].
 *               Owned by the caller; may be NULL when one range is used.  It
 *               must not overlap any other buffer and must not be used by
 *               another call in flight at the same time.
 *
 * Errors: as fa_fwd, plus FA_ERR_INVALID_ARGUMENT for num_splits < 1 or a
 * missing, misaligned, too small or overlapping workspace.  Two kernels are
 * enqueued on `stream` (the split forward, then the merge).
 */
FA_API int fa_fwd_split(const void* q, const void* k, const void* v, const float* mask, void* out,
                 float* lse, int B, int H, int Nq, int Nk, int D, float scale, int num_splits,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_split needs for these sizes (0 for invalid sizes). */
FA_API size_t fa_split_workspace_bytes(int B, int H, int Nq, int D, int num_splits);

/*
 * A key-range count for fa_fwd_split on a GPU with `num_sms` SMs: 1 when the
 * unsplit work units already cover every SM, else enough ranges to do so,
 * each range at least four 128-key blocks long.  Pure arithmetic; no CUDA call.
 */
FA_API int fa_split_count(int B, int H, int Nq, int Nk, int num_sms);

/*
 * fa_fwd_window — window / shifted-window attention on an img_h x img_w token
 * grid: every token attends only to the tokens of its own win_h x win_w window
 * of the grid cyclically shifted by (shift_h, shift_w) (the token at (r, c)
 * moves to ((r - shift_h) mod img_h, (c - shift_w) mod img_w)).  Computed as in
 * "Step 3.7 Flash" §3.2: the windows form a batch of
 * B * (img_h/win_h) * (img_w/win_w) attention problems of win_h*win_w tokens.
 * Here the batch is never materialised: the attention kernel reads each
 * window's rows of q, k, v from their grid positions and writes O and LSE
 * back to them.  Windows of up to 64 tokens are packed several to a batch
 * entry, each row seeing only its own window's keys.  No mask is applied
 * across the wrap-around of a shifted grid (the pages name none).
 *
 *   q, k, v, out  device bf16 [B, H, img_h*img_w, D], tokens in row-major grid order
 *   lse           device fp32 [B, H, img_h*img_w]
 *   win_h, win_w  >= 1 and dividing img_h, img_w;  shift_h, shift_w any integers
 *   workspace,    not used (fa_window_workspace_bytes returns 0); any value,
 *   workspace_bytes  NULL and 0 included, is accepted
 *   other arguments as fa_fwd
 *
 * One kernel is enqueued on `stream`.  Errors as fa_fwd, plus
 * FA_ERR_INVALID_ARGUMENT for windows that do not tile the grid or more than
 * 2^31 - 1 rows (B * H * img_h * img_w).
 */
FA_API int fa_fwd_window(const void* q, const void* k, const void* v, void* out, float* lse, int B, int H,
                  int img_h, int img_w, int D, int win_h, int win_w, int shift_h, int shift_w,
                  float scale, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes fa_fwd_window needs: 0 (kept for callers that size one). */
FA_API size_t fa_window_workspace_bytes(int B, int H, int img_h, int img_w, int D);

/* Bytes of the fixed device scratch that fa_fwd_split_noalloc uses. */
#define FA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * fa_fwd_split_noalloc — fa_fwd_split for callers that cannot allocate device
 * memory (a plugin whose host application owns every device allocation, or a
 * latency-critical path that cannot afford cudaMalloc's implicit device
 * synchronisation).  The pages have no counterpart of this entry point.
 *
 * Arguments as fa_fwd_split, without the workspace: the partial results live
 * in a fixed array of FA_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Sizes whose workspace (fa_split_workspace_bytes with the range count used)
 * exceeds FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_INVALID_ARGUMENT
 * before anything is enqueued.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before capturing
 * a stream.  All calls on a device share the one array, which keeps the last
 * call's contents: calls that overlap on the GPU (other streams, or before the
 * previous call finished) race on it and must be serialised by the caller.
 */
FA_API int fa_fwd_split_noalloc(const void* q, const void* k, const void* v, const float* mask, void* out,
                         float* lse, int B, int H, int Nq, int Nk, int D, float scale,
                         int num_splits, void* stream);

/*
 * fa_read_device_status — read, and reset to FA_OK, the status word that
 * kernels on the current device write when an internal wait times out.
 * Synchronises `stream` first.  Writes FA_OK or FA_ERR_TIMEOUT to *status.
 * Returns FA_OK, FA_ERR_INVALID_ARGUMENT (status NULL) or FA_ERR_CUDA.
 */
FA_API int fa_read_device_status(void* stream, int* status);

/*
 * fa_measure_ex2_rate — throughput of the exponential the forward takes once
 * per score (ex2.approx.ftz.f32 on the special-function unit): runs a short
 * probe kernel on `stream` (4 CTAs of 256 threads per SM, 16 independent
 * chains per thread, each CTA timed with clock64) and writes the exponentials
 * one SM completes per SM clock, bounded by its slowest CTA, to
 * *ex2_per_clock_per_sm.  The exp-bound time of a launch is then
 * B·H·Nq·Nk / (rate · SMs · clock).  ("算子加速：注意力、编译与融合",
 * section "注意力：从O(N²)显存到分块": one exponential per score in the
 * softmax.)  Diagnostic, blocking: synchronises `stream`.  Uses static device
 * storage of the library; allocates nothing.  Returns FA_OK,
 * FA_ERR_INVALID_ARGUMENT (NULL output), FA_ERR_UNSUPPORTED (more than 1024
 * SMs) or FA_ERR_CUDA.
 */
FA_API int fa_measure_ex2_rate(void* stream, double* ex2_per_clock_per_sm);

/*
 * Debug build (libfa_fwd_debug.so, compiled with FA_DEBUG; no counterpart on
 * the pages): every kernel checks its unit schedule and the index of every
 * global-memory access before using it.  A failed check skips the access,
 * records the first violation, sets FA_ERR_DEBUG_CHECK in the device status
 * word and makes its CTA drain and exit as after a wait timeout; nothing traps.
 * It stands in for a memory checker where none can run.
 *
 * fa_debug_build — 1 in the debug build, 0 in the release build.
 *
 * fa_debug_report — synchronise `stream`, copy the first recorded violation
 *   to record[8] and clear it: {check id (0 = none; 1 unit schedule, 2
 *   producer/MMA unit mismatch, 3 mask row, 4 e4m3 scale index, 5 output
 *   store), CTA, thread, value a, value b, 0, 0, number of failed checks}.
 *   The release build writes zeros.  Returns FA_OK, FA_ERR_INVALID_ARGUMENT
 *   (record NULL) or FA_ERR_CUDA.
 */
FA_API int fa_debug_build(void);
FA_API int fa_debug_report(void* stream, int* record);

/* Human-readable name of a status code (static storage; never NULL). */
FA_API const char* fa_status_string(int status);

/* Library version string, e.g. "unet_fa_fwd_gb300 0.1.0 sm_103a" (static storage). */
FA_API const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* UNET_FA_FWD_GB300_FA_H */
