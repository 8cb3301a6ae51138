/* attn.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The operation is exact scaled-dot-product attention,
 *     O   = softmax(scale * Q K^T  [+ causal mask]) V,
 *     lse = log sum_j exp(scale * q_i . k_j)       (natural log, per query row),
 * computed in one fused pass that never writes the N x N score matrix: the
 * online softmax of "Learn: The Memory Wall & FlashAttention", section 5.1
 * (running max m, running denominator l, one final O~ / l), with the
 * logsumexp L = m + log(l) of section 5.3.  Causal masking is top-left
 * aligned: key j is visible from query i iff j <= i ("4.3 FlashAttention 2 &
 * 3: Work Partitioning, Warp Specialization & FP8", "Edit 1 -- defer the
 * rescaling").  A row that sees no key would get O = 0, lse = -inf (it cannot
 * occur for the square shapes accepted here).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are caller-owned DEVICE memory on the current CUDA
 *     device.  The library allocates, frees and retains nothing; it keeps no
 *     pointer after the call returns.
 *   - Layout is [B, H, N, d] row-major, d innermost, contiguous (the layout of
 *     torch's scaled_dot_product_attention, not flash-attn's [B, N, H, d]).
 *     Queries and keys have the same length N.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Return values report argument errors and launch
 *     errors only; faults during execution surface at the caller's next
 *     synchronisation, and a pipeline wait that runs out of time is reported
 *     by attn_device_status().
 *   - Every bounded wait inside a kernel gives up after a time limit (1 s for
 *     the plain entry points), records ATTN_ERR_TIMEOUT, frees its tensor
 *     memory and returns.  A kernel held up that long (a debugger, time
 *     slicing with another context) therefore ends early: a call's outputs are
 *     defined only while attn_device_status() reports ATTN_OK.  A caller that
 *     cannot rule such delays out checks it after its results are complete.
 *   - The kernels hand out their work units dynamically from counters in the
 *     library's own device memory (64 counters used in turn, each zeroed by a
 *     memset on the caller's stream before its launch; no allocation).  Every
 *     call looks their device address up (cudaGetSymbolAddress) for the
 *     current device; the first call on a device loads the library's device
 *     code there: make one call before capturing a stream into a CUDA graph.
 *   - scale may be any finite value.  A negative scale is computed as
 *     |scale| * (q . (-k)): the score product negates its K operand, which is
 *     exact.  scale = 0 gives every visible key the same weight (O = mean of
 *     the visible V rows, lse = log of their count).
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

typedef struct CUstream_st* attn_stream_t; /* == cudaStream_t */

enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1, /* null pointer, bad size, non-finite scale, bad enum */
  ATTN_ERR_UNSUPPORTED = -2, /* head dim / dtype / device not supported */
  ATTN_ERR_ALIGNMENT = -3,   /* a tensor base address is not 16-byte aligned */
  ATTN_ERR_CUDA = -4,        /* a CUDA runtime / driver call failed (launch, encode) */
  ATTN_ERR_TIMEOUT = -5      /* a pipeline wait inside a kernel ran out of time */
};

enum attn_dtype { ATTN_BF16 = 0 };

/* Exact attention forward, bf16 operands, f32 accumulation.
 *   q, k, v : bf16 [B, H, N, d], read only.
 *   o       : bf16 [B, H, N, d], written (round to nearest even).
 *   lse     : f32 [B, H, N] logsumexp of the scaled scores, written; may be NULL.
 *   B, H, N : >= 1 (B * H < 2^31, N < 2^31).   d : 64 or 128.
 *   scale   : finite multiplier of q.k (usually 1/sqrt(d)); negative and zero
 *             values are computed exactly as the definition says.
 *   causal  : 0 or 1.   dtype : ATTN_BF16.
 * Errors: ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED (d, dtype, a device other than sm_103),
 * ATTN_ERR_ALIGNMENT (any of q, k, v, o not 16-byte aligned, lse not 4-byte aligned),
 * ATTN_ERR_CUDA. */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
             int d, float scale, int causal, int dtype, attn_stream_t stream);

/* attn_fwd generalised to grouped-query heads and a causal sliding window
 * ("4.3 FlashAttention 2 & 3", section "Calling the real kernel": KV heads
 * divide the query heads, no KV replication; Exercise 5: query i attends to
 * keys j with i - window < j <= i, blocks entirely outside the window skipped).
 *   q, o    : bf16 [B, H, N, d];  k, v : bf16 [B, H_kv, N, d]; query head h of
 *             batch b reads KV head h / (H / H_kv).  lse : f32 [B, H, N] or NULL.
 *   H_kv    : >= 1, divides H (H_kv = H: multi-head; 1: multi-query).
 *   window  : 0 for none; > 0 requires causal = 1.
 * Other arguments and errors as attn_fwd (ATTN_ERR_INVALID_ARG for a bad H_kv
 * or window). */
ATTN_API int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int H_kv, int N, int d, float scale, int causal, int window,
                         int dtype, attn_stream_t stream);

/* Split-KV attention forward: the visible key blocks of every pair of 128-row
 * query tiles are split into `num_splits` contiguous ranges, each a work unit
 * of its own, so that shapes with few (batch, head, query tile) units still
 * fill the device.  Each range writes its partial result -- O_s normalised by
 * its own denominator, and its logsumexp L_s -- to the workspace; a merge
 * kernel then computes, with M = max_s L_s,
 *     O = sum_s exp(L_s - M) O_s / sum_s exp(L_s - M),
 *     L = M + log sum_s exp(L_s - M),
 * the rule for combining two blocks' (m, l, O) states ("FlashAttention-3 & GPU
 * Kernel Optimization: Accelerating Transformer Attention", section "Online
 * softmax tiling mathematics") applied along the key axis, as in FlashDecoding
 * ("4.3 FlashAttention 2 & 3", section "Comparison, trade-offs, and when each
 * wins", paragraph on decode).  A range with no visible key has weight 0.
 *   q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window, dtype : as attn_fwd_ex.
 *   num_splits : 1 .. 64 (more ranges than key blocks leaves some empty).
 *   workspace  : caller-owned device scratch, 16-byte aligned, of at least
 *                attn_splitkv_workspace_bytes(B, H, N, d, num_splits) bytes
 *                (workspace_bytes says how large it is).  Overwritten entirely;
 *                its initial contents do not matter.  Calls that share a
 *                workspace must be ordered (the same stream, or synchronised).
 * Errors: as attn_fwd_ex; ATTN_ERR_INVALID_ARG for num_splits out of range or a
 * NULL or too small workspace; ATTN_ERR_ALIGNMENT for a workspace that is not
 * 16-byte aligned. */
ATTN_API int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int H_kv, int N, int d, float scale, int causal,
                              int window, int dtype, int num_splits, void* workspace,
                              size_t workspace_bytes, attn_stream_t stream);

/* attn_fwd_splitkv without a caller workspace and without any allocation: the
 * partial results go to one scratch array of 64 MiB (67108864 bytes) that the
 * library defines as a file-scope device variable, so it exists on every
 * device the library's code is loaded on.  The pages have no counterpart to
 * this entry point.  It is for callers that cannot call cudaMalloc: a plugin
 * running inside a host program that owns every byte of device memory through
 * its own pool (and may fail or fragment it if a library allocates behind its
 * back), or a latency-bound serving loop that must not pay cudaMalloc's implicit
 * device-wide synchronisation.  The price is 64 MiB held on every device that
 * loads the library, until the process exits.
 *   Arguments and errors: as attn_fwd_splitkv, minus the workspace;
 *   ATTN_ERR_INVALID_ARG also when attn_splitkv_workspace_bytes(B, H, N, d,
 *   num_splits) exceeds 64 MiB (nothing is launched).
 *   Nothing in the scratch needs to start at zero: every byte the merge reads
 *   is written earlier in the same call.
 *   Calls share the one array: two calls that overlap in time (different
 *   streams or host threads without ordering) race and give undefined
 *   results; order them.  Every call looks the array's device address up
 *   (cudaGetSymbolAddress with the calling device current, ATTN_ERR_CUDA if
 *   that fails); the first call on a device also loads the library's device
 *   code there, so that first call should come before any stream capture.
 *   The call makes no cudaMalloc, cudaFree or other allocating call. */
ATTN_API int attn_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int B, int H, int H_kv, int N, int d,
                                     float scale, int causal, int window, int dtype,
                                     int num_splits, attn_stream_t stream);

/* Workspace bytes attn_fwd_splitkv needs: the partial O (f32, num_splits * B *
 * H * N * d values) and the partial logsumexp (f32, num_splits * B * H * N
 * values), each rounded up to a multiple of 256 bytes; 0 for invalid arguments
 * (B, H, N < 1, d not 64 or 128, num_splits outside 1 .. 64).  Host arithmetic. */
ATTN_API size_t attn_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits);

/* A split count for attn_fwd_splitkv on a device with num_sms SMs, for the
 * shape (B, H, N, d) and causal flag the call will use: 1 if the plain
 * schedule already has at least num_sms units (pairs of 128-query tiles);
 * else the smallest S (S <= 64 and S <= ceil(N / 128), the number of 128-key
 * blocks) that minimises a time model in key blocks.  The model deals the
 * split units to the SMs in the kernel's own order, each SM taking the next
 * unit when free (a unit costs its key blocks plus 4 for its fixed work: Q
 * load, pipeline fill, epilogue), and adds for S > 1 the merge's traffic
 * (8 bytes per output element and split) at 8.8 MB per key block's time.
 * The constants were fitted to sweeps of S on the two-head 8192-token
 * workloads (non-causal and causal).  0 for invalid arguments.  Host
 * arithmetic. */
ATTN_API int attn_splitkv_default_splits(int B, int H, int N, int d, int causal, int num_sms);

/* Preparation of FP8 E4M3 operands with per-block scales and, optionally,
 * incoherent processing ("4.3 FlashAttention 2 & 3", section "Incoherent
 * processing: rotate away the outliers"; "FlashAttention-3: How Warp
 * Specialization, Asynchronous TMA Tiling, and FP8 Hardware Acceleration Scale
 * Attention on Hopper GPUs", section 4, block-wise scaling).
 *   x      : bf16 [B, H, N, d] input (Q, K or V), read only.
 *   signs  : int8 [H, d] of +1/-1, or NULL.  If given, each row x of head h is
 *            first rotated to x H_d diag(signs[h]) with H_d the orthonormal
 *            Sylvester Hadamard matrix (fast Walsh-Hadamard transform in f32);
 *            Q and K of one head must use the same signs.  V passes NULL.
 *   x8     : E4M3 output.  transpose_out == 0: [B, H, N, d].
 *            transpose_out == 1: [B, H, d, Npad] with Npad = 128 * ceil(N/128),
 *            keys contiguous, padding keys zero (the V operand layout that
 *            attn_fwd_fp8 reads).
 *   block_scale : f32 [B, H, ceil(N/128)], written: per block of 128 rows,
 *            s = amax / 448 over the (rotated) block, or 1 if the block is all
 *            zero; codes are RNE-satfinite E4M3 of x / s (f32 division).
 *   d : 128.
 * The kernel loads its tiles with bounded waits, like the attention kernels: a
 * copy that never completes sets the status word attn_device_status() reads,
 * and the outputs are then undefined.
 * Errors: as attn_fwd (ATTN_ERR_ALIGNMENT: x, x8 not 16-byte aligned, or signs
 * not 4-byte aligned). */
ATTN_API int attn_fp8_prep(const void* x, void* x8, float* block_scale, const signed char* signs, int B,
                  int H, int N, int d, int transpose_out, attn_stream_t stream);

/* Exact attention forward with E4M3 operands (f32 accumulation, f32 softmax
 * statistics, bf16 output): the FP8 forward of "FlashAttention-3: How Warp
 * Specialization, Asynchronous TMA Tiling, and FP8 Hardware Acceleration Scale
 * Attention on Hopper GPUs", section 4 (block-wise scaling: one scale per
 * block of each operand, so a score tile is s_Q * s_K * (Q8 K8^T)), with the
 * split of "4.3 FlashAttention 2 & 3", section "What stays in higher
 * precision" (operands and P in FP8; accumulators, the running max and the
 * row sums in f32).  Score tile j of query block i is
 * q_scale[i] * k_scale[j] * (Q8_i K8_j^T) * scale.  P is quantised to E4M3
 * with V's block scale folded in (p * 1.75 * v_scale[j] / max_j v_scale[j],
 * p <= 2^8 against the running reference maximum, so P' <= 448).
 *   q8, k8  : E4M3 [B, H, N, d] from attn_fp8_prep (same signs for both).
 *   v8t     : E4M3 [B, H, d, Npad] from attn_fp8_prep with transpose_out = 1.
 *   q_scale, k_scale, v_scale : f32 [B, H, ceil(N/128)] block scales.
 *   o, lse, B, H, N, scale, causal : as attn_fwd.   d : 128.
 * Errors: as attn_fwd. */
ATTN_API int attn_fwd_fp8(const void* q8, const void* k8, const void* v8t, const float* q_scale,
                 const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, attn_stream_t stream);

/* Attention backward: gradients of O = softmax(scale Q K^T [+mask]) V with
 * respect to Q, K, V, given the incoming gradient dO and the forward's O and
 * logsumexp ("4.3 FlashAttention 2 & 3", section "The backward pass:
 * recompute, and the one identity that makes it tile-able"):
 *     P = exp(scale Q K^T - L) (recomputed tile by tile, never stored),
 *     D_i = rowdot(dO_i, O_i),  dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
 *     dQ = scale dS K,  dK = scale dS^T Q.
 * With grouped KV heads, dK and dV of a KV head sum the contributions of the
 * query heads that read it.  Deterministic: dK, dV are accumulated by the
 * kernel that owns a key block, dQ by a second kernel that owns a query block
 * (no atomic adds).  P and dS enter the tensor-core products rounded to bf16;
 * accumulation is f32; outputs are rounded to bf16 (nearest even).
 *   q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, window : as attn_fwd_ex;
 *            o and lse are that call's outputs (lse is required here).
 *   dO     : bf16 [B, H, N, d], read only.
 *   dq     : bf16 [B, H, N, d], written.   dk, dv : bf16 [B, H_kv, N, d], written.
 *   workspace : caller-owned device scratch, 16-byte aligned, of at least
 *            attn_bwd_workspace_bytes(B, H, N, d) bytes (overwritten; calls
 *            sharing it must be ordered).
 * Errors: as attn_fwd_ex; ATTN_ERR_INVALID_ARG for a NULL pointer (lse
 * included) or a too small workspace; ATTN_ERR_ALIGNMENT for dO, dq, dk, dv,
 * workspace not 16-byte aligned. */
ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dO, void* dq, void* dk, void* dv, int B, int H, int H_kv, int N,
                      int d, float scale, int causal, int window, void* workspace,
                      size_t workspace_bytes, attn_stream_t stream);

/* Workspace bytes attn_bwd needs: two f32 arrays of B * H * Npad values (the
 * scaled logsumexp and D, Npad = 128 * ceil(N / 128)), each rounded up to a
 * multiple of 256 bytes; 0 for invalid arguments.  Host arithmetic. */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/* attn_fwd with an explicit status word and wait limit, for tests of the
 * failure path.  dev_status: device int, set to ATTN_ERR_TIMEOUT by a kernel
 * whose wait ran out (the caller clears it first).  timeout_ns: wait limit.
 * skip_loads: 0 for normal operation; n > 0 makes the load warp stop after n
 * K/V tiles so that consumer waits run out (the kernel then returns with the
 * status set, without faulting). */
ATTN_API int attn_fwd_debug(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int N, int d, float scale, int causal, int* dev_status,
                   unsigned long long timeout_ns, int skip_loads, attn_stream_t stream);

/* Synchronises the current device, then returns (and, if clear != 0, resets)
 * the status recorded by kernels launched through attn_fwd / attn_fwd_fp8:
 * ATTN_OK or ATTN_ERR_TIMEOUT; ATTN_ERR_CUDA if the synchronisation failed. */
ATTN_API int attn_device_status(int clear);

/* Work units (query-tile pairs of 256 rows) the persistent scheduler runs for
 * this shape, and the grid it would launch on a device with `num_sms` SMs.
 * Host-only arithmetic; lets tests check the schedule without a GPU. */
ATTN_API int attn_num_units(int B, int H, int N);
ATTN_API int attn_grid_size(int B, int H, int N, int num_sms);

/* Static description of a status code. */
ATTN_API const char* attn_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
