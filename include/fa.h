/*
 * fa.h — C ABI of the fused attention forward for NVIDIA GB300 (sm_103a).
 *
 * Operation (one call = every batch and head):
 *
 *   S   = scale * Q K^T                      ("Parsing FlashAttention (2):
 *   S_ij = -inf for j > i when causal          FlashAttention-v1 forward pass",
 *   O   = softmax_row(S) V                     §1.1 and §2.1 eqs (1)-(5);
 *   LSE_i = ln sum_j exp(S_ij)                 causal mask as in "Online Softmax
 *                                              and FlashAttention", course unit 12)
 *
 * computed by the tiled online softmax of the same pages (running max m,
 * running exponent sum l, accumulator rescaled by exp(m_old - m_new)), so no
 * N x N score or probability matrix is ever written to device memory.
 * LSE_i = m_i + ln(l_i) is the single statistic that summarises (m, l) for a
 * later backward pass (page 1 §1.2(3), "recomputation").
 *
 * Conventions for every entry point:
 *  - Pointers named q, k, v, o, lse are DEVICE pointers; nothing is copied to
 *    or from the host.  The caller owns all buffers; the library allocates no
 *    device memory and keeps no per-call state.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream): they return after enqueueing and never synchronise.
 *  - Errors are reported by return code (FA_OK on success).  Arguments are
 *    validated before anything is enqueued; on error nothing is launched and
 *    the outputs are untouched.  No C++ exception crosses this boundary.
 *  - Thread-safe: concurrent calls from several host threads are allowed.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum fa_status {
  FA_OK = 0,
  FA_ERR_NULL = 1,      /* a required pointer is NULL */
  FA_ERR_SHAPE = 2,     /* B, H or N <= 0, or B*H*N*d overflows the index space */
  FA_ERR_HEAD_DIM = 3,  /* d is not a head dimension the entry point takes */
  FA_ERR_ALIGN = 4,     /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
  FA_ERR_SCALE = 5,     /* scale is NaN or infinite */
  FA_ERR_ALIAS = 6,     /* o or lse overlaps an input, or o overlaps lse */
  FA_ERR_DEVICE = 7,    /* current device is not compute capability 10.3 (sm_103a) */
  FA_ERR_LAUNCH = 8,    /* CUDA runtime / driver error while preparing or launching */
  FA_ERR_TIMEOUT = 9,   /* a kernel wait exceeded its limit (see fa_get_device_status) */
  FA_ERR_WORKSPACE = 10, /* split-KV workspace NULL or too small */
  FA_ERR_SCRATCH_LIMIT = 11, /* fa_fwd_splitkv_static: request exceeds its built-in scratch */
  FA_ERR_DTYPE = 12,    /* element type not FA_DTYPE_BF16 / FA_DTYPE_FP16 */
  FA_ERR_STRIDE = 13    /* invalid strides, or overlapping output elements */
};

/* Element types of Q, K, V and O (fa_fwd_strided). */
#define FA_DTYPE_BF16 0
#define FA_DTYPE_FP16 1

/*
 * fa_fwd — attention forward for all (batch, head) slices.
 *
 *   q, k, v : const bf16 [B][H][N][d], contiguous, 16-byte aligned (device)
 *   o       : bf16 [B][H][N][d], contiguous, 16-byte aligned (device), written
 *   lse     : fp32 [B][H][N], contiguous (device), written; natural-log units
 *             of the scaled, masked scores: LSE_i = ln sum_j exp(S_ij)
 *   B, H, N : batch, heads, sequence length (queries = keys = N), each >= 1
 *   d       : head dimension, a multiple of 16 from 16 to 128, or 256
 *   causal  : 0 = full attention, 1 = query i sees keys 0..i (square,
 *             top-left aligned)
 *   scale   : any finite float multiplying Q K^T (typically 1/sqrt(d))
 *   stream  : cudaStream_t to enqueue on
 *
 * Inputs are read, never modified; o and lse must not overlap q, k, v or each
 * other.  Arithmetic: bf16 operands, fp32 accumulation and softmax
 * statistics, bf16 probabilities in the P.V product, bf16 output rounded to
 * nearest even.
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int N,
           int d, int causal, float scale, void *stream);

/*
 * fa_fwd_strided — fa_fwd with a choice of element type and arbitrary
 * strides ("pwwt.cn FlashAttention/Triton walkthrough" §3.4 passes every
 * tensor with its batch, head and row strides; §5 lists fp16 and other head
 * dimensions among the extensions).
 *
 *   q, k, v, o : [B][H][N][d] tensors of `dtype` elements (device, base
 *                16-byte aligned); element (b, h, n, c) of tensor X lives at
 *                X + b*X_strides[0] + h*X_strides[1] + n*X_strides[2] + c
 *   *_strides  : 3 int64 element strides (batch, head, row), each a
 *                non-negative multiple of 8 below 2^38; NULL = contiguous
 *                [B][H][N][d].  Columns are always contiguous.  Distinct
 *                elements of o must not overlap (FA_ERR_STRIDE).
 *   lse        : fp32 [B][H][N], contiguous (device), written
 *   dtype      : FA_DTYPE_BF16 or FA_DTYPE_FP16 (the P.V operand P takes the
 *                same type; accumulation and statistics are fp32)
 *   other arguments and the result as for fa_fwd.
 */
int fa_fwd_strided(const void *q, const int64_t *q_strides, const void *k,
                   const int64_t *k_strides, const void *v, const int64_t *v_strides, void *o,
                   const int64_t *o_strides, float *lse, int dtype, int B, int H, int N, int d,
                   int causal, float scale, void *stream);

/*
 * fa_fwd_host — the forward of fa_fwd for inputs and outputs in HOST
 * memory, the one entry point that copies: on `stream` it queues the copies
 * of q, k, v into the caller's device workspace (one cudaMemcpyAsync each),
 * the forward kernel, and the copies of O and LSE back.  The pages' method
 * has no counterpart; it is the end-to-end path of a caller whose tensors
 * live on the host.
 *
 *   q_host, k_host, v_host : const [B][H][N][d] elements of `dtype`
 *                            (FA_DTYPE_BF16 / FA_DTYPE_FP16), contiguous, host
 *   o_host                 : [B][H][N][d] of `dtype`, host, written
 *   lse_host               : fp32 [B][H][N], host, written
 *   d, causal, scale       : as for fa_fwd_strided
 *   workspace              : device memory of at least
 *                            fa_fwd_host_workspace_bytes() bytes, 256-byte
 *                            aligned, owned by the caller (Q, K, V, O and LSE
 *                            staged there, overwritten)
 * Page-locked host memory lets the copies run asynchronously at full
 * bandwidth; pageable memory works, with the driver's staging.  The host
 * outputs hold the result once `stream` has been synchronised; the host
 * inputs must stay unchanged until then.  Host outputs must not overlap a
 * host input or each other (FA_ERR_ALIAS).  Everything fa_fwd would reject
 * is rejected before any copy is queued; FA_ERR_WORKSPACE when the
 * workspace is missing or small.
 */
int fa_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host,
                float *lse_host, int dtype, int B, int H, int N, int d, int causal, float scale,
                void *workspace, size_t workspace_bytes, void *stream);

/* Device workspace bytes fa_fwd_host needs (0 on invalid arguments). */
size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_fwd_splitkv — attention of a short block of queries against a long key
 * sequence (decode), split over the keys.
 *
 * Same operation as fa_fwd with Nq queries and Nk keys; causal masking is
 * aligned to the end of the keys: query i (0 <= i < Nq) sees keys
 * 0 .. Nk - Nq + i (for Nq == Nk this is fa_fwd's rule).  The keys are cut
 * into contiguous ranges, each range's attention (a normalised output and its
 * log-sum-exp) is computed, and the ranges are merged with the block-merge
 * identity ("Parsing FlashAttention (2)" eq. (20); "Online Softmax and
 * FlashAttention", course unit 12):
 *     LSE = ln sum_s e^(LSE_s),   O = sum_s e^(LSE_s - LSE) O_s.
 * With at most 8 ranges the ranges of a (batch, head) run as one thread-block
 * cluster and merge on chip (one launch, workspace untouched); otherwise the
 * partials go through `workspace` and a second launch merges them.
 *
 *   q         : const bf16 [B][H][Nq][d] (device, 16-byte aligned)
 *   k, v      : const bf16 [B][H][Nk][d] (device, 16-byte aligned)
 *   o         : bf16 [B][H][Nq][d] (device), written
 *   lse       : fp32 [B][H][Nq] (device), written (natural log)
 *   Nq        : 1 .. 16 queries;  Nk >= 1 keys (causal needs Nq <= Nk)
 *   d         : 64 or 128;  B*H <= 65535
 *   num_splits: key ranges, 0 = the library's choice for the current device
 *               (the most ranges whose CTAs, two per multiprocessor, all run
 *               at once), else 1 .. 256; the count used may be lower (at
 *               least 64 keys per range)
 *   workspace : device scratch of at least fa_fwd_splitkv_workspace_bytes()
 *               bytes (16-byte aligned), owned by the caller, overwritten;
 *               must not overlap any other argument.  Calls that share a
 *               workspace must be ordered (same stream) or they race.
 * Returns FA_OK or an FA_ERR_* code (FA_ERR_WORKSPACE when the workspace is
 * missing or too small); validates before enqueueing; asynchronous.
 */
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                   int Nq, int Nk, int d, int causal, float scale, int num_splits,
                   void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace fa_fwd_splitkv needs for these arguments on the current
 * device (0 on invalid arguments or without a usable device when
 * num_splits == 0). */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);

/* Number of key ranges fa_fwd_splitkv uses for these arguments (0 on invalid
 * arguments or without a usable device when num_splits == 0). */
int fa_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * fa_fwd_splitkv_host — fa_fwd_splitkv for inputs and outputs in HOST memory:
 * on `stream` it queues the copies of q, k, v into the caller's device
 * workspace (one cudaMemcpyAsync each), the split-KV launch(es), and the
 * copies of O and LSE back.  The pages' method has no counterpart; it is the
 * end-to-end path of a decode caller whose tensors live on the host.
 *
 *   q_host, k_host, v_host, o_host, lse_host : as fa_fwd_splitkv's device
 *       tensors (bf16 [B][H][Nq|Nk][d], fp32 [B][H][Nq]), contiguous, host
 *   B .. num_splits : as for fa_fwd_splitkv
 *   workspace : device memory of at least fa_fwd_splitkv_host_workspace_bytes()
 *       bytes, 256-byte aligned, owned by the caller (Q, K, V, O, LSE and the
 *       split partials staged there, overwritten)
 * Host outputs must not overlap a host input or each other (FA_ERR_ALIAS).
 * Everything fa_fwd_splitkv would reject is rejected before any copy is
 * queued; FA_ERR_WORKSPACE when the workspace is missing or small.  The host
 * outputs hold the result once `stream` has been synchronised; the host
 * inputs must stay unchanged until then.
 */
int fa_fwd_splitkv_host(const void *q_host, const void *k_host, const void *v_host, void *o_host,
                        float *lse_host, int B, int H, int Nq, int Nk, int d, int causal,
                        float scale, int num_splits, void *workspace, size_t workspace_bytes,
                        void *stream);

/* Device workspace bytes fa_fwd_splitkv_host needs on the current device (0
 * on invalid arguments or without a usable device when num_splits == 0). */
size_t fa_fwd_splitkv_host_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * fa_fwd_splitkv_static — fa_fwd_splitkv for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a library service.
 *
 * Some callers cannot call cudaMalloc or any allocator: code whose device
 * memory all belongs to a pool or arena it does not control, code that must
 * not risk the implicit synchronisation or the failure of an allocation in
 * the middle of its work, and plug-ins whose host hands them no allocator.
 * This entry point takes the same inputs and outputs as fa_fwd_splitkv but
 * no workspace: its scratch (the per-range partial outputs and
 * log-sum-exps) lives in a device array built into the library, of
 * fa_fwd_splitkv_static_scratch_bytes() bytes (8 MiB), which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or allocating library routine.
 *
 * Arguments, layout, results and arithmetic are those of fa_fwd_splitkv
 * (num_splits included), without workspace and workspace_bytes.  A request
 * whose scratch would exceed the array (about splits * B * H * Nq * (4d + 4)
 * bytes; fa_fwd_splitkv_workspace_bytes() gives the exact figure) is
 * rejected with FA_ERR_SCRATCH_LIMIT before anything is enqueued.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current, and again after the device's context
 * has been replaced, e.g. by cudaDeviceReset); make that first call before
 * any stream capture.  Every call on a device shares the one array, which keeps the
 * last call's contents (nothing in it needs to start at zero); calls whose
 * kernels overlap on the GPU, e.g. on two unordered streams or from two
 * host threads, race on it and give undefined results: order them on one
 * stream.  Returns FA_OK or an FA_ERR_* code; asynchronous.
 */
int fa_fwd_splitkv_static(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int H, int Nq, int Nk, int d, int causal, float scale, int num_splits,
                          void *stream);

/* Size in bytes of fa_fwd_splitkv_static's built-in scratch array. */
size_t fa_fwd_splitkv_static_scratch_bytes(void);

/*
 * fa_bwd — gradients of the attention forward: the backward pass by
 * recomputation for which "Parsing FlashAttention (2)" §1 and "Online
 * Softmax and FlashAttention" keep the row statistics (here LSE).
 *
 * With s = scale * Q K^T (+ causal mask), P = exp(s - LSE), D_i =
 * rowsum(dO_i * O_i):  dV = P^T dO,  dS = P * (dO V^T - D),
 * dQ = scale * dS K,  dK = scale * dS^T Q  (the gradients of sum(dO * O)).
 *
 *   q, k, v, o, dout : const bf16 [B][H][N][d] (device, contiguous, 16-byte
 *                      aligned); o and lse as written by fa_fwd for the same
 *                      q, k, v, causal and scale
 *   lse              : const fp32 [B][H][N] (device, 4-byte aligned)
 *   dq, dk, dv       : bf16 [B][H][N][d] (device), written
 *   d                : a multiple of 16 from 16 to 128 (computed in 64- or
 *                      128-wide tiles whose extra columns are zeros and are
 *                      never stored);  causal, scale as for fa_fwd
 *   workspace        : device scratch of at least fa_bwd_workspace_bytes()
 *                      bytes (16-byte aligned), owned by the caller,
 *                      overwritten (D and LSE * log2(e) per query row)
 * Outputs and workspace must not overlap an input or each other.  Three
 * kernel launches on `stream` (a pre-pass, the dK/dV pass, the dQ pass), no
 * atomics: the result is deterministic.  Returns FA_OK or an FA_ERR_* code
 * (FA_ERR_WORKSPACE when the workspace is missing or small); validates
 * before enqueueing; asynchronous.
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int B, int H, int N, int d,
           int causal, float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * fa_bwd_ex — fa_bwd for either element type: q, k, v, o, dout, dq, dk, dv
 * all hold `dtype` elements (FA_DTYPE_BF16 or FA_DTYPE_FP16: IEEE binary16
 * bit patterns), the MMAs run on that type (P and dS rounded to it, as the
 * forward rounds P) with fp32 accumulation; lse, the workspace and every
 * other argument as for fa_bwd, which is fa_bwd_ex with FA_DTYPE_BF16.
 * Returns FA_ERR_DTYPE for any other dtype, else as fa_bwd.
 */
int fa_bwd_ex(const void *q, const void *k, const void *v, const void *o, const float *lse,
              const void *dout, void *dq, void *dk, void *dv, int dtype, int B, int H, int N,
              int d, int causal, float scale, void *workspace, size_t workspace_bytes,
              void *stream);

/*
 * fa_bwd_strided — fa_bwd_ex with every [B][H][N][d] tensor at its own
 * strides, as fa_fwd_strided takes them ("pwwt.cn FlashAttention/Triton
 * walkthrough" §3.4 passes every tensor with its batch, head and row strides).
 *
 *   q, k, v, o, dout    : const [B][H][N][d] `dtype` tensors (device, base
 *                         16-byte aligned); element (b, h, n, c) of tensor X
 *                         lives at X + b*X_strides[0] + h*X_strides[1] +
 *                         n*X_strides[2] + c
 *   dq, dk, dv          : [B][H][N][d] `dtype` tensors (device, base 16-byte
 *                         aligned), written at their strides
 *   *_strides           : 3 int64 element strides (batch, head, row), each a
 *                         non-negative multiple of 8 below 2^38; NULL =
 *                         contiguous.  Columns are always contiguous.
 *                         Distinct elements of dq, dk or dv must not overlap
 *                         (FA_ERR_STRIDE); inputs may share elements.
 *   lse, workspace, dtype, B .. scale, stream : as for fa_bwd_ex
 * The address span of each output (first to one past the last element) and
 * the workspace must overlap no input's span and no other output's
 * (FA_ERR_ALIAS).  fa_bwd_ex is this call with every stride NULL.  Returns
 * FA_OK or an FA_ERR_* code; validates before enqueueing; asynchronous.
 */
int fa_bwd_strided(const void *q, const int64_t *q_strides, const void *k,
                   const int64_t *k_strides, const void *v, const int64_t *v_strides,
                   const void *o, const int64_t *o_strides, const float *lse, const void *dout,
                   const int64_t *dout_strides, void *dq, const int64_t *dq_strides, void *dk,
                   const int64_t *dk_strides, void *dv, const int64_t *dv_strides, int dtype,
                   int B, int H, int N, int d, int causal, float scale, void *workspace,
                   size_t workspace_bytes, void *stream);

/* Workspace bytes fa_bwd, fa_bwd_ex and fa_bwd_strided need (0 on invalid
 * arguments). */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_bwd_host — fa_bwd_ex for inputs and outputs in HOST memory: on `stream`
 * it queues the copies of q, k, v, o, lse and dout into the caller's device
 * workspace (one cudaMemcpyAsync each), the three backward launches, and the
 * copies of dq, dk, dv back.  The pages' method has no counterpart; it is
 * the end-to-end path of a caller whose tensors live on the host.
 *
 *   q_host .. dout_host : as fa_bwd_ex's device inputs (`dtype` [B][H][N][d],
 *                         fp32 lse [B][H][N]), contiguous, host
 *   dq_host, dk_host, dv_host : `dtype` [B][H][N][d], host, written
 *   dtype .. scale      : as for fa_bwd_ex
 *   workspace           : device memory of at least fa_bwd_host_workspace_bytes()
 *                         bytes, 256-byte aligned, owned by the caller (the
 *                         nine tensors and the backward's workspace staged
 *                         there, overwritten)
 * Host outputs must not overlap a host input or each other (FA_ERR_ALIAS).
 * Everything fa_bwd_ex would reject is rejected before any copy is queued;
 * FA_ERR_WORKSPACE when the workspace is missing or small.  The host outputs
 * hold the result once `stream` has been synchronised; the host inputs must
 * stay unchanged until then.
 */
int fa_bwd_host(const void *q_host, const void *k_host, const void *v_host, const void *o_host,
                const float *lse_host, const void *dout_host, void *dq_host, void *dk_host,
                void *dv_host, int dtype, int B, int H, int N, int d, int causal, float scale,
                void *workspace, size_t workspace_bytes, void *stream);

/* Device workspace bytes fa_bwd_host needs (0 on invalid arguments). */
size_t fa_bwd_host_workspace_bytes(int B, int H, int N, int d);

/*
 * fa_fwd_order_ablation — the attention forward of fa_fwd in one of the two
 * loop orders the pages compare, for measuring their HBM traffic and time
 * side by side (a measurement instrument; fa_fwd is the production path).
 *
 *   order 1: "Parsing FlashAttention (2): FlashAttention-v1 forward pass" §4
 *            Algorithm 1 — per (batch, head), K/V tiles outer and query tiles
 *            inner; every step reads Q_i and the running O_i, m_i, l_i from
 *            the workspace in HBM and writes them back (normalised update,
 *            eq. (37)); one CTA per (batch, head).
 *   order 2: "Online Softmax and FlashAttention" (course unit 12) — query
 *            tiles outer with Q_i and the accumulator on chip, K/V tiles
 *            streamed, O written once; one CTA per (batch, head, query tile).
 * Both run the same 64 x 64 tile code on warp-level tensor-core MMAs.
 *
 *   q, k, v, o, lse, B, H, N, causal, scale : as for fa_fwd (contiguous bf16)
 *   d          : 64 or 128
 *   workspace  : at least fa_fwd_order_ablation_workspace_bytes() bytes of
 *                device memory (16-byte aligned), owned by the caller,
 *                overwritten (order 1: the running fp32 O, m, l of every row)
 * Returns FA_OK or an FA_ERR_* code; validates before enqueueing; async.
 */
int fa_fwd_order_ablation(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                          int H, int N, int d, int causal, float scale, int order,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of fa_fwd_order_ablation (0 on invalid arguments). */
size_t fa_fwd_order_ablation_workspace_bytes(int B, int H, int N, int d, int order);

/* Human-readable text for a return code (static storage, never NULL). */
const char *fa_strerror(int code);

/*
 * Device status word of the kernels on the current device: a bit set of
 * FA_DEVICE_STATUS_* values, sticky until fa_clear_device_status().  Reading
 * it synchronises the current device (it copies one word to the host).
 * Returns FA_OK or FA_ERR_LAUNCH; *status must not be NULL (FA_ERR_NULL).
 */
#define FA_DEVICE_STATUS_TIMEOUT 1u
/* Set only by the guarded build of the library (libfa_guarded.so, the same
 * sources compiled with FA_GUARDED=1): a TMA tile origin, TMEM column range,
 * shared-memory destination or global store failed its bounds check; the
 * access was skipped (outputs undefined, no fault).  Never set by libfa.so. */
#define FA_DEVICE_STATUS_BOUNDS 2u
int fa_get_device_status(unsigned int *status);
int fa_clear_device_status(void);

/*
 * Upper bound, in nanoseconds, on any single wait inside the kernels
 * (default 1e9).  A wait that exceeds it sets FA_DEVICE_STATUS_TIMEOUT, the
 * kernel abandons its work (outputs undefined), frees its on-chip resources
 * and exits.  0 restores the default.  Applies to later calls, process-wide.
 */
int fa_set_wait_limit_ns(unsigned long long ns);

/*
 * Test hook: a bit set of FA_INJECT_* faults applied by later calls,
 * process-wide (0 = none, the default).  FA_INJECT_SKIP_FIRST_V_LOAD makes
 * every CTA skip one streamed-tile copy — the first V tile of fa_fwd /
 * fa_fwd_strided / fa_fwd_host (every head dimension), the first K/V tile of
 * the split-KV pass, the first streamed stage of each fa_bwd pass — so a wait
 * runs out and the call ends with FA_DEVICE_STATUS_TIMEOUT set.  No GPU
 * fault is involved: the kernels drain what they issued, free TMEM and exit.
 * For tests of the failure path only.
 */
#define FA_INJECT_SKIP_FIRST_V_LOAD 1u
int fa_set_fault_injection(unsigned int flags);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
