/*
 * attn_gb300.h -- C ABI of the GB300 (sm_103a) IO-aware attention forward library.
 *
 * The operation is scaled dot-product attention, O = softmax(scale * Q K^T) V, computed row by
 * row over the keys each query may see, together with the per-row log-sum-exp of the scaled
 * scores (CS336 Lecture 5 notes, section 6.1 for the definition; section 6.2 for the fused,
 * tiled, online-softmax forward that never writes the score matrix to HBM and keeps only m and l
 * "merged into a logsumexp"; CS336 GPU/attention notes, "Online softmax 回顾", for the merge).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  No call allocates device
 *     memory (the fused kernel uses on-chip shared and tensor memory only; the unfused
 *     comparison path uses a caller-provided workspace).  The one piece of device memory the
 *     library holds is a file-scope array of ATTN_NOALLOC_SCRATCH_BYTES (64 MiB), the scratch of
 *     attn_fwd_unfused_noalloc, which every GPU that loads the library keeps until exit.
 *   - Element types: q, k, v, o are bfloat16 (passed as void*); lse is float32;
 *     cu_seqlens is int32.
 *   - Dense layout (cu_seqlens == NULL): q, k, v, o are [B, H, N, d] contiguous, d innermost;
 *     lse is [B, H, N].
 *   - Packed variable-length layout (cu_seqlens != NULL): B is the number of sequences and N is
 *     the total token count T = cu_seqlens[B] (passed by the host, which never reads device
 *     memory); q, k, v, o are [H, T, d] and lse is [H, T].  Sequence s owns rows
 *     cu_seqlens[s] .. cu_seqlens[s+1]-1 of every head and attends only to itself.
 *     cu_seqlens must be non-decreasing with cu_seqlens[0] = 0 and cu_seqlens[B] = N; a
 *     violation is the caller's error and gives undefined output (never an out-of-bounds write
 *     outside [0, N) rows of o and lse).  Zero-length sequences are allowed and write nothing.
 *   - causal != 0 keeps key j for query i iff j <= i, positions counted from the start of each
 *     sequence.
 *   - scale multiplies the scores before the softmax (1/sqrt(d) for the usual attention); it must
 *     be finite and > 0.  lse is the natural-log log-sum-exp of the scaled scores.
 *   - d must be 64 or 128.  Pointers must be 16-byte aligned.
 *   - B, H, N >= 0; if any of them is 0 there is nothing to compute and the call returns
 *     ATTN_OK without touching the pointers.
 *   - Work is enqueued on `stream` (a cudaStream_t, 0 = legacy default stream) and runs
 *     asynchronously.  The return value covers host-side validation and the launch; a device-side
 *     failure (a pipeline wait that timed out) is reported by attn_get_last_device_error().
 *   - On any non-zero return the contents of o and lse are unspecified.
 *   - Entry points are thread-safe as long as concurrent calls use different output buffers.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,        /* a required pointer is NULL                                  */
  ATTN_ERR_HEAD_DIM = -2,    /* d is not 64 or 128                                          */
  ATTN_ERR_SHAPE = -3,       /* a negative size, or sizes whose products overflow the kernel */
  ATTN_ERR_ALIGN = -4,       /* a tensor pointer is not 16-byte aligned                     */
  ATTN_ERR_LAUNCH = -5,      /* a CUDA call failed while preparing or launching the kernel  */
  ATTN_ERR_DEVICE = -6,      /* the current device is not an sm_103 (GB300-class) GPU       */
  ATTN_ERR_SCALE = -7,       /* scale is not finite or not > 0                              */
  ATTN_ERR_WORKSPACE = -8,   /* workspace NULL, unaligned or smaller than required          */
  ATTN_ERR_UNSUPPORTED = -9, /* an argument combination this entry point does not support   */
  ATTN_ERR_SCRATCH_LIMIT = -10 /* the problem needs more than the built-in scratch (no-alloc) */
} attn_status;

/*
 * Fused forward (the hot path).  One kernel launch: each CTA keeps a 128-row tile of Q on chip,
 * streams 128-row tiles of K and V through TMA-fed shared memory, computes S = Q K^T with tcgen05
 * tensor-core MMAs into tensor memory, applies the online softmax (running row max m and sum l,
 * exp2 of log2(e)-prescaled scores, rescaling of the O accumulator) and accumulates P V on the
 * tensor cores, then writes O = acc / l in bf16 and lse = m + ln l in fp32.  The N x N score
 * matrix never reaches HBM; causal tiles above the diagonal are skipped.
 *   q, k, v : bf16 inputs (read only)          o   : bf16 output, same layout as q
 *   lse     : fp32 output                      cu_seqlens : NULL (dense) or int32[B+1] (packed;
 *                                                           a prefix sum from 0 to N, else the
 *                                                           status word reports kind 2)
 *   B, H, N, d, causal, scale : as described above; stream : cudaStream_t
 * Returns an attn_status.
 */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             const int32_t* cu_seqlens, int B, int H, int N, int d, int causal, float scale,
             void* stream);

/*
 * Grouped-query / multi-query forward (CS336 Lecture 5 notes, section 6.3: several query heads
 * share one K/V head).  As attn_fwd, except that k and v have H_kv heads and query head h reads
 * K/V head h / (H / H_kv):
 *   dense : q, o [B, H, N, d]; k, v [B, H_kv, N, d]; lse [B, H, N]
 *   packed: q, o [H, T, d];    k, v [H_kv, T, d];    lse [H, T]
 * H_kv must divide H (H_kv = H is attn_fwd; H_kv = 1 is multi-query attention), else
 * ATTN_ERR_SHAPE.  Returns an attn_status.
 */
ATTN_API int attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* cu_seqlens, int B, int H, int H_kv, int N, int d,
                          int causal, float scale, void* stream);

/*
 * Split-KV forward for problems with few query tiles (small B * H): the key/value sequence of
 * every pair of query tiles is cut into num_splits contiguous slices, each computed by its own
 * CTA (head dim 64) or cluster of two CTAs (head dim 128), so that more SMs share the work (sequence-dimension parallelism, CS336 Lecture 5 notes, section 6.3).
 * Each slice leaves its unnormalised output, its reference row maximum and its row sums in
 * `workspace`; a second kernel on `stream` merges the slices with the block merge of the CS336
 * GPU/attention notes, "Online softmax 回顾" (M = max of the slice maxima, each slice weighted by
 * exp(m_s - M), O = sum of weighted outputs / sum of weighted sums, lse = M + ln(weighted sum)).
 * Dense layout only: q, k, v, o [B, H, N, d] bf16, lse [B, H, N] fp32, as attn_fwd.
 *   num_splits : slices per query pair, at most 32 and at most the number of 128-key tiles
 *                (larger values are lowered).  <= 0 lets the library choose: the count that
 *                minimises (waves of units) x (key tiles per slice + 2), the smallest on ties,
 *                where a wave is 152 units at d = 64 and 76 (two SMs each) at d = 128.
 *                When the count is 1 this is attn_fwd and the workspace is not touched.
 *   workspace  : caller-owned device buffer of at least
 *                attn_fwd_splitkv_workspace_bytes(B, H, N, d, num_splits) bytes, 256-byte
 *                aligned, else ATTN_ERR_WORKSPACE; its contents on return are unspecified.
 * Returns an attn_status (argument checks as attn_fwd).
 */
ATTN_API int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int N, int d, int causal, float scale, int num_splits,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The slice count attn_fwd_splitkv uses for these sizes and num_splits (0 for invalid sizes or
 * a head dim other than 64 and 128).
 */
ATTN_API int attn_fwd_splitkv_slices(int B, int H, int N, int d, int num_splits);

/*
 * Workspace bytes attn_fwd_splitkv needs: with S the slice count it will use, an fp32 partial
 * output [S][B*H*N][d] followed by two fp32 planes [2][S][B*H*N] (slice max in log2 units, the
 * row sum), each region rounded up to 256 bytes.
 * Returns 0 when S is 1 (no workspace needed) or the sizes are invalid.
 */
ATTN_API size_t attn_fwd_splitkv_workspace_bytes(int B, int H, int N, int d, int num_splits);

/*
 * Backward pass (dQ, dK, dV) of the fused forward.  Nothing N x N is read or kept: S and P are
 * rebuilt tile by tile from the logsumexp the forward saved (CS336 Lecture 5 notes, section 6.2,
 * "反向传播怎么办"), and the gradients follow from the definition by the chain rule:
 * dV = P^T dO, dP = dO V^T, dS = P * (dP - D) with D_i = dO_i . O_i, dQ = scale dS K,
 * dK = scale dS^T Q.  Two kernel launches on `stream`: a row pass (D and lse * log2 e into the
 * workspace), then one grid whose first CTAs run the dK/dV pass (one CTA per 128-key tile) and
 * the rest the dQ pass (one CTA per 128-query tile); every output element is written once
 * (deterministic, no atomics).
 * Dense layout only:
 *   q, k, v, o, dout : bf16 [B, H, N, d] (o is the forward's output, dout the gradient of the loss
 *                      with respect to it)         lse : fp32 [B, H, N], the forward's lse output
 *   dq, dk, dv       : bf16 [B, H, N, d] outputs
 *   causal, scale    : as in the forward call that produced o and lse
 *   workspace        : caller-owned device buffer of at least attn_bwd_workspace_bytes(B,H,N,d)
 *                      bytes, 256-byte aligned; contents on return unspecified
 * Every tensor pointer must be 16-byte aligned (ATTN_ERR_ALIGN) and non-NULL (ATTN_ERR_NULL);
 * other checks as attn_fwd.  Returns an attn_status.
 */
ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                      int H, int N, int d, int causal, float scale, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * Backward pass of grouped-query / multi-query attention (CS336 Lecture 5 notes, section 6.3):
 * as attn_bwd, except that k, v, dk and dv have H_kv heads ([B, H_kv, N, d]) and query head h
 * reads K/V head h / (H / H_kv).  A K/V head's gradients are the sums over the query heads that
 * share it: the dK/dV pass runs one CTA per (K/V head, key tile) that visits the query tiles of
 * all of them, so the sums accumulate in tensor memory and each element is still written once.
 * H_kv must divide H, else ATTN_ERR_SHAPE.  The workspace is attn_bwd_workspace_bytes(B,H,N,d).
 */
ATTN_API int attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          int B, int H, int H_kv, int N, int d, int causal, float scale,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass on a packed batch of variable-length sequences (the layout of attn_fwd with
 * cu_seqlens): q, o, dout, dq [H, T, d]; k, v, dk, dv [H_kv, T, d]; lse [H, T]; cu_seqlens
 * int32[B + 1] on the device, B = number of sequences, T = total rows.  Sequences are independent;
 * grouped-query heads as attn_bwd_gqa (H_kv = H for multi-head).  The tile passes run one CTA per
 * (head, 128-row tile of a sequence), found by a scan of cu_seqlens; offsets are clamped into
 * [0, T].  workspace: attn_bwd_varlen_workspace_bytes(B, H, T, d) bytes, 256-byte aligned.
 * cu_seqlens NULL: ATTN_ERR_NULL.  Returns an attn_status.
 */
ATTN_API int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv,
                             const int32_t* cu_seqlens, int B, int H, int H_kv, int T, int d,
                             int causal, float scale, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Workspace bytes attn_bwd_varlen needs: two fp32 planes of H * 128 * (ceil(T/128) + B) rows,
 * each rounded up to 256 bytes.  Returns 0 for invalid sizes.
 */
ATTN_API size_t attn_bwd_varlen_workspace_bytes(int B, int H, int T, int d);

/*
 * Workspace bytes attn_bwd needs: two fp32 planes of B * H * Npad values (Npad = N rounded up to
 * 128), each rounded up to 256 bytes.  Returns 0 for invalid sizes.
 */
ATTN_API size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Per-tile E4M3 quantization (the FP8 format of CS336 Lecture 5 notes, section 3.1: 1 sign,
 * 4 exponent, 3 mantissa bits, largest magnitude 448; per-tile scaling).  For every tile of 128
 * rows of a head of the bf16 tensor x [B, H, N, d] (d = 64 or 128):
 *   scale = amax / 448 in fp32 (1 for an all-zero tile), written to scales[(b*H + h)*T + t]
 *   (T = ceil(N/128)); code = E4M3 round-to-nearest-even of x / scale rounded to nearest fp32
 *   (the IEEE quotient, which the kernel forms from the tile's reciprocal with one correction;
 *   attn_selftest_fp8_quotients checks every input), saturating at +-448, the sign bit kept for
 *   values that round to zero.
 *   transpose = 0: codes [B, H, N, d] (N*d bytes per head)
 *   transpose = 1: codes [B, H, d, Npad] with Npad = 128*T, padding codes 0 (the V operand of
 *                  attn_fwd_fp8)
 * x and codes must be 16-byte aligned, scales 4-byte aligned.  Returns an attn_status.
 */
ATTN_API int attn_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int N,
                               int d, int transpose, void* stream);

/*
 * FP8 fused forward (FlashAttention-3's FP8 path, CS336 Lecture 5 notes, section 6.3), head dim
 * 128, dense layout.  Inputs are E4M3 codes with per-tile fp32 scales as attn_quantize_fp8
 * writes them: q8, k8 [B, H, N, 128] (transpose = 0), vt8 [B, H, 128, Npad] (transpose = 1); the
 * value of an input element is code x its tile's scale.  S = Q K^T runs on kind::f8f6f4 tensor
 * cores; the probabilities enter P V as E4M3 codes of P * 48 * sv_j / max(sv) (V's tile scales
 * folded in; P <= 8 against a reference maximum that trails the row maximum by at most 3 in log2
 * units); O (bf16) and lse (fp32, natural log of the scaled scores' normaliser) as attn_fwd.
 * d other than 128: ATTN_ERR_HEAD_DIM.  Returns an attn_status.
 */
ATTN_API int attn_fwd_fp8(const void* q8, const float* sq, const void* k8, const float* sk,
                          const void* vt8, const float* sv, void* o, float* lse, int B, int H,
                          int N, int d, int causal, float scale, void* stream);

/*
 * Unfused comparison path (the "standard attention" of the pages: S written to HBM, read back for
 * the softmax, P written to HBM, read back for P V; CS336 GPU/attention notes, "Attention 为什么
 * 容易 memory-bound"; CS336 Lecture 5 notes, section 6.1).  Three kernel launches on `stream`:
 * scores (S = scale * Q K^T in fp32), row softmax (P in bf16 plus lse), and P V.  It computes the
 * same O and lse as attn_fwd and exists only as the memory-wall comparison.
 * Dense layout only (cu_seqlens must be NULL, else ATTN_ERR_UNSUPPORTED).
 *   workspace : caller-owned device buffer of at least attn_fwd_unfused_workspace_bytes(B,H,N,d)
 *               bytes, 256-byte aligned; its contents on return are unspecified.
 */
ATTN_API int attn_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse,
                     const int32_t* cu_seqlens, int B, int H, int N, int d, int causal,
                     float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes attn_fwd_unfused needs for a dense [B, H, N, d] problem: the fp32 score matrix
 * and the bf16 (unnormalised) probability matrix of every head, each row padded to a multiple of
 * 128 columns, plus one fp32 normaliser per row: about B * H * N * (6 * Npad + 4) bytes with
 * Npad = N rounded up to 128 (each region rounded up to 256 bytes).  Returns 0 for invalid sizes.
 */
ATTN_API size_t attn_fwd_unfused_workspace_bytes(int B, int H, int N, int d);

/* Size of the built-in scratch array of attn_fwd_unfused_noalloc (64 MiB per GPU). */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * The unfused comparison path without a workspace argument, for callers that cannot allocate
 * device memory.  (The reference pages have no counterpart: this is a property of this library's
 * interface, not of the method.)  Some callers cannot call cudaMalloc -- code running under a
 * memory manager that owns every device allocation, or a runtime that forbids allocation once it
 * has started -- so this entry point allocates nothing: its scratch is a file-scope device array of
 * ATTN_NOALLOC_SCRATCH_BYTES that every GPU loading this library holds until the process exits.
 *   Arguments as attn_fwd_unfused (dense layout only), without cu_seqlens and the workspace.
 *   Returns ATTN_ERR_SCRATCH_LIMIT when attn_fwd_unfused_workspace_bytes(B, H, N, d) exceeds
 *   ATTN_NOALLOC_SCRATCH_BYTES, before touching the GPU.
 *   Every call looks up the array's device address (cudaGetSymbolAddress, with the calling
 *   device current); nothing is cached, so a device reset between calls leaves no stale address.
 *   The first call in a context loads the module there; make that first call before any stream
 *   capture.
 *   All calls share the array and it keeps the last call's contents (nothing in it needs to start
 *   at zero); calls whose work overlaps on the GPU, e.g. on two streams, race on it.
 */
ATTN_API int attn_fwd_unfused_noalloc(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int H, int N, int d, int causal,
                                      float scale, void* stream);

/*
 * Device-side status of the kernels launched on `stream` since the previous call: 0 if every
 * pipeline wait completed; otherwise a code whose low byte is 1 (a wait exceeded its time limit,
 * after which the kernel drained its in-flight copies, released its tensor memory and returned;
 * bits 8..15 name the waiting role and bits 16..23 the wait site) or 2 (the cu_seqlens given to a
 * packed-batch call was not a non-decreasing prefix sum from 0 to N; the kernel computed on its
 * offsets clamped into [0, N] and read or wrote nothing outside the tensors) or 3 (a kernel's
 * shared-memory layout did not fit the dynamic shared memory it was given at a 1024-byte boundary;
 * that kernel wrote nothing and its outputs are not valid).  The first problem
 * recorded is kept.  Synchronises `stream`, then clears the status.  Returns ATTN_ERR_LAUNCH (< 0)
 * if the status cannot be read.
 */
ATTN_API int attn_get_last_device_error(void* stream);

/*
 * Diagnostic: one 128-row tensor-core product with the operand layouts and descriptors of the fused
 * kernel, written to d as fp32 row-major.  Not part of the attention path; it isolates the
 * tcgen05 operand encoding (CS336 Lecture 5 notes, section 6.2: the two matmuls of each tile pair).
 *   mode 0: d[128 x 128] = a[128 x dim] * b[128 x dim]^T   (the S = Q K^T shape)
 *   mode 1: d[128 x dim] = a[128 x 128] * b[128 x dim]     (the O += P V shape)
 *   mode 2: as mode 1 with a staged in tensor memory (the P V shape with P kept on chip)
 *   a, b : bf16 row-major device buffers (16-byte aligned); d : fp32 device buffer;
 *   dim  : 64 or 128.  Asynchronous on `stream`; returns an attn_status.
 */
ATTN_API int attn_selftest_mma(const void* a, const void* b, float* d, int mode, int dim, void* stream);

/*
 * Diagnostic: launch one warp that waits on an mbarrier nothing ever arrives on, through the same
 * bounded wait the pipeline kernels use.  After the wait limit (one second) the warp records
 * status 1 | (6 << 8) | (1 << 16) and returns, leaving the context usable; read it with
 * attn_get_last_device_error().  Exercises failure detection without faulting or hanging the GPU.
 * Returns an attn_status (the launch only).
 */
ATTN_API int attn_selftest_wait_timeout(void* stream);

/*
 * Diagnostic of attn_quantize_fp8's division: for every positive finite bf16 number amax and every
 * bf16 x with |x| <= amax (both signs, about 1.07e9 pairs), compares the E4M3 code the quantizer
 * forms for x at the tile scale amax / 448 with the code of the correctly rounded fp32 quotient
 * (the per-tile scaling of CS336 Lecture 5 notes, section 3.1), and writes the number of pairs
 * that differ to *mismatches.  mismatches: device pointer to one 8-byte-aligned 64-bit counter,
 * which the call zeroes first.  Asynchronous on `stream` (about a second of GPU time); returns an
 * attn_status (the launch only).
 */
ATTN_API int attn_selftest_fp8_quotients(unsigned long long* mismatches, void* stream);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
