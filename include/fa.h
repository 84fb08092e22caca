/*
 * fa.h — C ABI of the fused exact-attention library for NVIDIA GB300 (sm_103a).
 *
 * What is computed (FlashAttention-4 article, "Por que el enfoque estandar ya
 * no funciona": the two products S = Q K^T and O = P V with a softmax between
 * them; FlashAttention-3 page, "FlashAttention y FlashAttention-2": tiled and
 * fused so the N x N score matrix never reaches global memory).  For every
 * batch b, query head h, query row i, with kh = h / (H / Hkv):
 *
 *     s_ij  = scale * q_i . k_j                 (j visible iff !causal || j <= i)
 *     O_i   = sum_j softmax_j(s_i.) v_j,        LSE_i = ln sum_{visible j} exp(s_ij)
 *
 * and the backward pass of L = sum(dO * O):
 *
 *     dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . v_j,  D_i = dO_i . O_i,
 *     dS_ij = P_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i
 *
 * (the pages list the backward's bottlenecks, FlashAttention-4 paper summary,
 * section 2.C, but not its formulas; these follow from the forward by the chain
 * rule).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     allocates no device memory for them and keeps no reference after return.
 *   - Layouts are dense, row-major, no strides:
 *         q, o, dq, dO : bf16 [B, N, H,   d]
 *         k, v, dk, dv : bf16 [B, N, Hkv, d]
 *         lse          : fp32 [B, H, N]      (natural-log units)
 *   - Every tensor base pointer must be 16-byte aligned (tensor-memory-access
 *     copies require it).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 *     asynchronous: it validates, enqueues and returns.
 *   - Supported: d in {64, 128, 256}; N >= 1 (any length, ragged tails are
 *     masked); B, H, Hkv >= 1 with H % Hkv == 0; scale finite and > 0; B and H
 *     at most 65535; B*N*H*d below 2^40 elements (offsets are 64-bit); at most
 *     2^31 - 1 thread blocks per launch (one per 128 or 256 rows of one (batch,
 *     head)).  Larger sizes return FA_ERR_UNSUPPORTED.  Device: compute
 *     capability 10.3 (GB300).
 *   - Outputs must not alias inputs (not checked).
 *   - Errors: every argument check happens before any launch and nothing is
 *     written on error.  A launch failure returns FA_ERR_CUDA.  Faults inside a
 *     kernel surface asynchronously at the caller's next synchronisation.  Every
 *     wait inside the kernels is bounded: a wait that runs out sets a status
 *     word that fa_last_device_status() reports, and the kernel returns.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad scale, H % Hkv != 0 */
  FA_ERR_UNSUPPORTED = -2, /* head dim not in {64,128,256}, sizes beyond limits, not a GB300 */
  FA_ERR_ALIGNMENT = -3,   /* a tensor pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = -4,   /* workspace missing or smaller than fa_bwd_workspace_bytes() */
  FA_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
  FA_ERR_TIMEOUT = -6      /* a bounded wait inside a kernel ran out (reported by fa_last_device_status) */
} fa_status;

/* Forward pass.  Writes o [B,N,H,d] bf16 and lse [B,H,N] fp32 (natural log).
 * `lse` may be NULL when the caller does not need it (no backward). */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int Hkv, int N, int d, float scale, int causal, void *stream);

/* Forward pass over a packed batch of variable-length sequences.  The pages
 * only name this variant (FlashAttention-4 paper summary, section 5: varlen
 * among the attention variants the code base is meant to take up); what it
 * computes here is the plain reading: sequence b is rows
 * [cu_seqlens[b], cu_seqlens[b+1]) of every tensor, and each sequence is the
 * single-sequence problem above on its own rows (queries and keys share the
 * lengths; the causal mask is taken within the sequence, key j visible from
 * query i iff j <= i).
 *   q, o : bf16 [total, H, d];  k, v : bf16 [total, Hkv, d];
 *   lse  : fp32 [H, total] (natural log) or NULL;
 *   cu_seqlens : DEVICE int32 [B + 1], cu_seqlens[0] = 0, non-decreasing,
 *     cu_seqlens[B] = total, every length <= max_seqlen.  The table is read
 *     only on the device: lengths are clamped to [0, max_seqlen] and rows to
 *     [0, total), so a table outside this contract gives unspecified values
 *     but no out-of-bounds access.  Rows of empty sequences are not written.
 * total = 0 is valid and launches nothing.  Other rules as for fa_fwd
 * (max_seqlen takes the place of N in the size limits). */
int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                  const int *cu_seqlens, int B, int max_seqlen, int total,
                  int H, int Hkv, int d, float scale, int causal, void *stream);

/* FP8 forward with incoherent processing (FlashAttention-3 page, section 3:
 * multiply the query and key feature vectors by a random orthogonal matrix,
 * e.g. a Hadamard matrix, so outlier coordinates spread out, then quantize to
 * FP8; the orthogonal factor cancels in Q K^T).  Same inputs, outputs and rules
 * as fa_fwd, for d = 128 only (other head dims: FA_ERR_UNSUPPORTED).
 *   rot_signs : DEVICE fp32 [128] of +1/-1, the rotation M = diag(rot_signs)
 *               H_128 / sqrt(128) (H_128 the Sylvester Hadamard matrix) applied
 *               to every row of q and k; NULL means no rotation.
 *   The arithmetic: q M and k M rounded to e4m3 (round to nearest even,
 *   saturating at 448) with one fp32 scale per 128-row block of one (batch,
 *   head) mapping the block's largest magnitude to 448; v rounded to e4m3 with
 *   one scale per (batch, kv head); S = Q8 K8^T on the tensor core with fp32
 *   accumulation; P rounded to e4m3 for P V8; the row sum and LSE from the
 *   unrounded P in fp32; o written in bf16.
 *   workspace : caller-owned device memory, 256-byte aligned, of at least
 *     fa_fwd_fp8_workspace_bytes() bytes; it receives, each on a 256-byte
 *     boundary and in this order, q8 [B,N,H,128] and k8 [B,N,Hkv,128] (e4m3),
 *     vt8 [B,Hkv,128,Npad] (e4m3, keys contiguous, zero past N), the fp32
 *     scales sq [B,H,nt], sk [B,Hkv,nt], the V block maxima [B,Hkv,nt] and sv
 *     [B,Hkv] (Npad = nt * 128, nt = ceil(N / 128)).
 * Three launches on `stream`. */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int Hkv, int N, int d);
int fa_fwd_fp8(const void *q, const void *k, const void *v, const float *rot_signs, void *o, float *lse,
               int B, int H, int Hkv, int N, int d, float scale, int causal,
               void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device workspace fa_bwd needs for these sizes: two fp32 row-term
 * arrays [B,H,Npad] (D = rowsum(dO * O) and the log2-scaled LSE), Npad = N
 * rounded up to a multiple of 128, each starting on a 256-byte boundary.
 * Returns 0 for sizes fa_bwd would reject. */
size_t fa_bwd_workspace_bytes(int B, int H, int Hkv, int N, int d);

/* Backward pass.  Inputs q, k, v, o, lse from the forward, and dO [B,N,H,d].
 * Writes dq [B,N,H,d], dk and dv [B,N,Hkv,d] (bf16).  `workspace` is caller owned device
 * memory of at least fa_bwd_workspace_bytes() bytes, 256-byte aligned; its
 * contents on entry do not matter and are overwritten.  No atomics: results
 * are bitwise reproducible for the same inputs. */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dO, void *dq, void *dk, void *dv,
           int B, int H, int Hkv, int N, int d, float scale, int causal,
           void *workspace, size_t workspace_bytes, void *stream);

/* Backward pass of fa_fwd_varlen (same packed layouts and cu_seqlens table;
 * dO, dq : bf16 [total, H, d], dk, dv : bf16 [total, Hkv, d], lse from
 * fa_fwd_varlen).  Each sequence's gradients are those of its own
 * single-sequence problem.  The workspace is fa_bwd_workspace_bytes(B, H, Hkv,
 * max_seqlen, d) bytes, as for a batch of B sequences of max_seqlen rows.
 * Deterministic like fa_bwd.  total = 0 launches nothing. */
int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dO, void *dq, void *dk, void *dv, const int *cu_seqlens,
                  int B, int max_seqlen, int total, int H, int Hkv, int d, float scale, int causal,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Backward pass in one fused kernel on CTA pairs (FlashAttention-4 paper
 * summary, section 2.C: the two CTAs of a pair exchange halves of dS through
 * distributed shared memory and each adds dQ for half of the query rows), head
 * dim 128, fixed-length batches.  Same arguments and results as fa_bwd within
 * the backward tolerance, but dQ is summed over the key tiles by fp32
 * reductions in global memory, in an order that varies from run to run: the
 * result is not bitwise reproducible (fa_bwd is).  The workspace
 * (fa_bwd_fused_workspace_bytes, 256-byte aligned) holds fa_bwd's row terms
 * followed by an fp32 dQ accumulator of B*N*H*d elements.  Returns
 * FA_ERR_UNSUPPORTED for a head dim other than 128. */
size_t fa_bwd_fused_workspace_bytes(int B, int H, int Hkv, int N, int d);
int fa_bwd_fused(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dO, void *dq, void *dk, void *dv,
                 int B, int H, int Hkv, int N, int d, float scale, int causal,
                 void *workspace, size_t workspace_bytes, void *stream);

/* The three launches fa_bwd makes, for callers that schedule them separately
 * (same arguments and rules as fa_bwd; run fa_bwd_prepare first, then the
 * other two in either order, on one stream or ordered streams, with the same
 * workspace):
 *   fa_bwd_prepare: D = rowsum(dO * O) and the log2-scaled LSE into the
 *                   workspace (memory bound);
 *   fa_bwd_dkdv:    the key/value-stationary kernel: recomputes P from LSE,
 *                   writes dk and dv;
 *   fa_bwd_dq:      the query-stationary kernel: recomputes S, P and dP,
 *                   writes dq. */
int fa_bwd_prepare(const void *o, const float *lse, const void *dO, int B, int H, int Hkv, int N, int d,
                   void *workspace, size_t workspace_bytes, void *stream);
int fa_bwd_dkdv(const void *q, const void *k, const void *v, const void *dO, void *dk, void *dv,
                int B, int H, int Hkv, int N, int d, float scale, int causal,
                void *workspace, size_t workspace_bytes, void *stream);
int fa_bwd_dq(const void *q, const void *k, const void *v, const void *dO, void *dq,
              int B, int H, int Hkv, int N, int d, float scale, int causal,
              void *workspace, size_t workspace_bytes, void *stream);

/* Backward pass that allocates nothing and takes no workspace.  The pages have
 * no counterpart: this entry point exists for callers that cannot allocate
 * device memory at the time they run the backward pass (a plug-in inside a host
 * framework that owns all device memory through its own pool; a serving or
 * training loop that forbids cudaMalloc after start-up, since it synchronises
 * the device and fragments memory).  Same arguments, results and rules as
 * fa_bwd, except that the row terms fa_bwd keeps in the caller's workspace live
 * in one static device array of FA_BWD_NOALLOC_SCRATCH_BYTES bytes inside the
 * library, which every GPU that loads the library holds until the process
 * exits.
 *   - Sizes whose fa_bwd_workspace_bytes() exceeds FA_BWD_NOALLOC_SCRATCH_BYTES
 *     are rejected with FA_ERR_WORKSPACE before any launch.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture.
 *   - Every call shares the one array: calls whose kernels overlap on the GPU
 *     (different streams, or different host threads, without ordering between
 *     them) race and corrupt each other's results.  Each call re-initialises
 *     what it reads, so the contents a previous call left do not matter.
 *   - The device address is cached for the life of the process: a device
 *     reset (cudaDeviceReset, or a reset of the primary context) after the
 *     first call on that device is not supported.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine. */
#define FA_BWD_NOALLOC_SCRATCH_BYTES (64ull << 20)
/* The size of that array as the library was built (FA_BWD_NOALLOC_SCRATCH_BYTES). */
size_t fa_bwd_noalloc_scratch_bytes(void);
int fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dO, void *dq, void *dk, void *dv,
                   int B, int H, int Hkv, int N, int d, float scale, int causal, void *stream);

/* The software 2^x the kernels evaluate on the FMA pipe (FlashAttention-4
 * paper summary, section 2.B: 2^x emulated with FMA instructions, a polynomial
 * of degree 3 to 5 for the fractional part).  Range reduction x = j + f with
 * j = rint(x), |f| <= 1/2; a degree-3 minimax polynomial for 2^f; 2^j inserted
 * into the exponent.  Evaluates y[i] = 2^x[i] for n fp32 values on `stream`
 * (device pointers, 4-byte aligned).  Valid for x <= 63; x below -150 or -inf
 * gives +0.  Exposed so that its accuracy can be checked exhaustively.  The
 * kernels evaluate it either one value at a time (forward) or two at a time in
 * f32x2 arithmetic (dK/dV); this entry point computes both forms and returns
 * NaN for an element where they differ in any bit. */
int fa_exp2_poly(const float *x, float *y, long long n, void *stream);

/* Synchronises `stream`, then returns FA_OK or FA_ERR_TIMEOUT if a bounded wait
 * in any kernel of this library on the current device ran out since the last
 * call (and clears the flag).  Returns FA_ERR_CUDA if synchronisation fails. */
int fa_last_device_status(void *stream);

/* The same, and writes to *site (host pointer, may be NULL) the id of the first
 * wait that ran out since the last call, or 0.  Ids name the wait inside the
 * kernels, for diagnostics: forward 1-8 (1 Q tile loaded, 2/3 K/V tile loaded,
 * 4 P stored by the softmax warps, 5 ring slot free, 6 S computed, 7 O final,
 * 8 MMA drain); backward 11-22 (11 K/V loaded, 12 operand tile loaded, 13 ring
 * slot free, 14 S computed, 15 dP computed, 16 P stored, 17 dS stored,
 * 19 final MMA, 20 MMA drain, 21 shared-memory alignment, 22 the dQ kernel's
 * Q and dO tiles loaded; fused backward: 23 dQ partial computed, 24 S read
 * into registers, 25 dQ partial read out).  Outputs of a call in which a wait
 * ran out are unspecified. */
int fa_last_device_status_site(void *stream, int *site);

/* Test aid.  In a library built with -DFA_TEST_STALL (never the default
 * build), makes block 0 of one kernel skip one barrier arrival on every later
 * launch until called again with mode 0, so that a bounded wait runs out and
 * the kernel unwinds through its abort path (1: the forward's first P, 2: the
 * dK/dV kernels' first P, 3: the dQ kernel's first dS); build such a library
 * with a short -DFA_WAIT_LIMIT_NS.  Returns FA_ERR_INVALID_ARG for another
 * mode.  In every other build it does nothing and returns FA_ERR_UNSUPPORTED. */
int fa_debug_stall(int mode);

/* Debugging aid: how many times a warp of the forward kernels applied the
 * conditional O rescale (FlashAttention-4 paper summary, section 2.B: rescale
 * only when the running maximum moves past a threshold) since the last call on
 * this device; the counter is then reset.  Synchronizes `stream` first.
 * count: host pointer, written on FA_OK.  Returns FA_ERR_INVALID_ARG for a
 * NULL count and FA_ERR_CUDA if synchronisation or the copy fails. */
int fa_rescale_count(void *stream, unsigned *count);

/* Human-readable name of a status code (static string, never NULL). */
const char *fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
