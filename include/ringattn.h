/*
 * ringattn.h -- C ABI of libringattn.so: ring-order blockwise attention on one
 * GB300 GPU (sm_103a).
 *
 * Pages this interface implements (title and section only):
 *   [FT] "Ring Attention如何让大模型突破百万Token上下文：从环形通信到计算重叠的技术突围"
 *        (answer.freetools.me)
 *   [CH] "Ring Attention with Blockwise Transformers for Near Infinite Context",
 *        reading notes on arXiv 2310.01889 (papers.chlience.com)
 *   [AQ] "Ring Attention" explainer (aiqz.cc)
 *
 * Common conventions
 * ------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    never frees or retains them; it allocates no device memory on any call
 *    (the backward takes a caller-sized workspace).
 *  - Q, K, V, O, dO, dQ, dK, dV are dense row-major [B, H, S, D] in *storage
 *    order*.  The sequence is cut into N equal blocks of c = S / N rows, one per
 *    virtual ring host ([CH] §5.2).  Layout RA_CONTIGUOUS: storage row p holds
 *    token p.  Layout RA_STRIPED: storage row p = i*c + r holds token r*N + i,
 *    i.e. token t lives on block t mod N ([FT] "因果掩码的负载均衡挑战").
 *  - LSE is float32 [B, H, S], storage order: LSE = ln sum_k exp(q.k / sqrt(D))
 *    over the keys the row sees (natural log, scaled-score units).
 *  - dtype RA_BF16: 16-bit bfloat16 tensors, float32 accumulation, outputs
 *    rounded to nearest even.  dtype RA_F32: float32 tensors throughout.
 *  - Causal masking is per token (key token <= query token, [AQ] §工程实现);
 *    with the contiguous layout whole KV blocks j > i are skipped.
 *  - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream).  Argument errors are detected on the host before any
 *    launch and return synchronously; output contents are then unchanged.
 *    After a launched call fails, output contents are unspecified.
 *  - Return value: an ra_status.  ra_last_error() gives a message for the most
 *    recent non-OK status of the calling thread.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RA_API __attribute__((visibility("default")))
#else
#define RA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_ARG = 1,          /* bad pointer, size, alignment or enum value   */
  RA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement  */
  RA_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed  */
  RA_ERR_TIMEOUT = 4       /* a bounded device-side wait ran out           */
} ra_status;

typedef enum {
  RA_F32 = 0,
  RA_BF16 = 1,
  RA_F32_BF16 = 2   /* ra_merge only: float32 state O_a, bf16 partial O_b */
} ra_dtype;
typedef enum { RA_CONTIGUOUS = 0, RA_STRIPED = 1 } ra_layout;

/*
 * ra_fwd -- forward pass: O = softmax(Q K^T / sqrt(D)) V and its LSE.
 *
 * Each query block i sweeps the KV blocks in ring order j = i, i-1, ... mod N
 * ([FT] "Ring Attention的核心洞察" step 3; [AQ] §环状拓扑) and folds every
 * score tile S_ij = Q_i K_j^T / sqrt(D) into per-row online-softmax state
 * (running max m, denominator l, unnormalised numerator O) ([AQ] §分块注意力,
 * the m / l / O update equations; [FT] "Online Softmax").  At the end
 * O <- O / l and LSE <- m + ln l.
 *
 *   Q, K, V : [B,H,S,D] of `dtype`, 16-byte aligned.
 *   O       : [B,H,S,D] of `dtype` (output), 16-byte aligned.
 *   LSE     : [B,H,S] float32 (output), 4-byte aligned.
 *   B, H, S, D, N : B,H >= 1; S >= 1 with S % N == 0; N >= 1.
 *                   RA_BF16 requires D == 128.  RA_F32 requires D % 4 == 0
 *                   and D <= 128.  Any block length c = S/N is accepted
 *                   (a partial last tile is masked).
 *   causal  : 0 or 1.   layout : ra_layout.   dtype : ra_dtype.
 *   stream  : cudaStream_t.
 * Errors: RA_ERR_ARG (null pointer, misalignment, S % N != 0, sizes <= 0,
 * bad enum, B*H*S*D overflowing int64, or B*H or S beyond 2^31-1),
 * RA_ERR_UNSUPPORTED (D outside the list above), RA_ERR_CUDA.
 */
RA_API int ra_fwd(const void* Q, const void* K, const void* V,
           int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
           int causal, int layout, int dtype,
           void* O, float* LSE, void* stream);

/*
 * ra_fwd_step -- one step of one ring host: query block i against KV block j.
 *
 * The per-host operation of a multi-device ring ([CH] §5.2: each host keeps
 * Q_i and, every round, attends it to the K_j, V_j it currently holds while
 * forwarding them; [FT] "Ring Attention的核心洞察" steps 3-4).  Returns the
 * partial state over block j's keys only: O normalised over those keys and
 * LSE = ln sum over them; rows that see none of them get O = 0, LSE = -inf.
 * Chaining the N steps of a host with ra_merge gives that host's rows of
 * ra_fwd.  The mask uses the true token positions of blocks i and j under
 * `layout` (contiguous causal j > i: all masked, no kernel runs).
 *
 *   Q_i, K_j, V_j : [B,H,c,D] of `dtype` (the blocks, not the whole sequence).
 *   O : [B,H,c,D] of `dtype` (output);  LSE : [B,H,c] float32 (output).
 *   N : ring size; i, j : block indices in [0, N).  Other arguments and errors
 *   as for ra_fwd (with S = c and one block).
 */
RA_API int ra_fwd_step(const void* Q_i, const void* K_j, const void* V_j,
           int64_t B, int64_t H, int64_t c, int64_t D,
           int64_t N, int64_t i, int64_t j,
           int causal, int layout, int dtype,
           void* O, float* LSE, void* stream);

/*
 * ra_fwd_step_fold -- ra_fwd_step that folds its partial state into the
 * host's running state instead of returning it ([CH] §5.2, one host and one
 * round; the fold is the LogSumExp merge of [FT] "Online Softmax").  Per row:
 *     lse = M + ln(e^{lse_acc-M} + e^{lse_j-M}),  M = max(lse_acc, lse_j);
 *     O_acc <- e^{lse_acc-lse} O_acc + e^{lse_j-lse} O_j,  LSE_acc <- lse,
 * where (O_j, lse_j) is what ra_fwd_step would return.  It happens in the
 * forward kernel's epilogue, one thread per row, so a round is one launch and
 * the partial never leaves the chip in bf16.  Start a host's state at
 * LSE_acc = -inf (such rows are empty: O_acc is not read there) and fold the
 * N rounds in any order; the result is that host's rows of ra_fwd in float32.
 * Rows that see none of block j's keys are left unchanged, and a contiguous
 * causal round j > i launches nothing.
 *
 *   Q_i, K_j, V_j : [B,H,c,128] bf16 (dtype must be RA_BF16).
 *   O_acc : [B,H,c,128] float32, 16-byte aligned (in/out);
 *   LSE_acc : [B,H,c] float32 (in/out).  Other arguments as ra_fwd_step.
 * Errors: RA_ERR_ARG (null pointer, misalignment, indices, sizes),
 * RA_ERR_UNSUPPORTED (dtype other than bf16, D != 128), RA_ERR_CUDA.
 */
RA_API int ra_fwd_step_fold(const void* Q_i, const void* K_j, const void* V_j, int64_t B, int64_t H, int64_t c,
                            int64_t D, int64_t N, int64_t i, int64_t j, int causal, int layout, int dtype,
                            float* O_acc, float* LSE_acc, void* stream);

/*
 * ra_merge -- LogSumExp merge of two partial states over disjoint key sets,
 * in place into (O_a, lse_a)  ([FT] "Online Softmax": l = l1 e^{m1-m} +
 * l2 e^{m2-m} and its log-space form).  Per row:
 *     M = max(lse_a, lse_b);  lse = M + ln(e^{lse_a-M} + e^{lse_b-M});
 *     O_a <- e^{lse_a-lse} O_a + e^{lse_b-lse} O_b.
 * Both lse -inf (no key seen on either side): lse = -inf and O = 0.
 *
 *   O_a : [rows, D] of `dtype` (in/out);   lse_a : [rows] float32 (in/out)
 *   O_b : [rows, D] of `dtype` (in);       lse_b : [rows] float32 (in)
 *   dtype RA_F32_BF16: O_a float32, O_b bf16 -- a ring host keeps its running
 *   output in float32 across the rounds and folds each round's bf16 partial
 *   (from ra_fwd_step) into it, so the output is rounded once, not per round.
 *   rows >= 0 (0 is a no-op), D in 1..1024.  Pointers 4-byte aligned (O_* of
 *   bf16 may be 2-byte aligned).  O_a and O_b must not overlap unless equal.
 * Errors: RA_ERR_ARG, RA_ERR_CUDA.
 */
RA_API int ra_merge(void* O_a, float* lse_a, const void* O_b, const float* lse_b,
             int64_t rows, int64_t D, int dtype, void* stream);

/*
 * ra_bwd_workspace_bytes -- size of the caller-allocated workspace ra_bwd
 * needs for these sizes: per query row -D_vec = -rowsum(dO * O) and
 * -LSE * log2(e) (stored negated), each per 128-row query tile of every block
 * ([B,H,N,ceil(S/N/128),128] float32, 8 bytes per padded row in all), each
 * part 256-byte aligned.  Returns 0 on bad sizes (as ra_bwd would reject
 * them).
 */
RA_API size_t ra_bwd_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N);

/*
 * ra_bwd -- backward pass from the saved output and LSE.
 *
 * The pages state only that the backward re-sweeps the KV blocks along the
 * ring to accumulate dQ, dK, dV from the saved softmax state ([CH] §5.2, last
 * paragraph).  This computes the gradient of the forward's definition:
 *     P = exp(Q K^T / sqrt(D) - LSE) on visible entries (0 elsewhere),
 *     dV = P^T dO,  dP = dO V^T,  D_vec = rowsum(dO * O),
 *     dS = P * (dP - D_vec),  dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D).
 * Each KV tile sweeps the query blocks that see it in ring order (dK, dV);
 * each query tile sweeps the KV blocks in the forward's ring order (dQ).
 * No atomics: every output element is written once, so results are
 * bit-reproducible.
 *
 *   Q, K, V, O, dO : [B,H,S,D] inputs;  LSE [B,H,S] float32 input (as ra_fwd
 *   wrote it).  dQ, dK, dV : [B,H,S,D] outputs of `dtype`.  16-byte aligned.
 *   workspace : device memory of at least ra_bwd_workspace_bytes(B,H,S,D,N)
 *   bytes, 256-byte aligned; its contents on entry do not matter.  Calls that
 *   share a workspace must not overlap on the GPU.
 *   Sizes, causal, layout as for ra_fwd; RA_BF16 with D == 128 only.
 * Errors: RA_ERR_ARG (also: workspace too small), RA_ERR_UNSUPPORTED,
 * RA_ERR_CUDA.
 */
RA_API int ra_bwd(const void* Q, const void* K, const void* V, const void* O,
           const float* LSE, const void* dO,
           void* dQ, void* dK, void* dV,
           int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
           int causal, int layout, int dtype,
           void* workspace, size_t ws_bytes, void* stream);

/*
 * ra_bwd_step -- one host and one ring round of the backward: the gradient
 * contributions of query block i against KV block j, ADDED into float32
 * accumulators.  In a multi-host ring ([CH] §5.2: the backward, like the
 * forward, sweeps the KV blocks around the ring), host i keeps dQ_i and the
 * accumulators dK_j, dV_j travel with K_j, V_j; after N rounds each has
 * collected every query block's share and returns to its owner.
 *     P = exp(Q_i K_j^T / sqrt(D) - LSE_i) on the pair's visible entries,
 *     dV_j += P^T dO_i,  dS = P * (dO_i V_j^T - rowsum(dO_i * O_i)),
 *     dQ_i += dS K_j / sqrt(D),  dK_j += dS^T Q_i / sqrt(D).
 * LSE_i and O_i are block i's FINAL forward results (not a partial state).
 * Masking as in ra_fwd_step: diag-type pairs mask by true token position, a
 * contiguous causal pair j > i adds nothing (no kernel runs).
 *
 *   Q_i, O_i, dO_i : [B,H,c,D] bf16;  LSE_i [B,H,c] float32;
 *   K_j, V_j : [B,H,c,D] bf16;  dQ_i, dK_j, dV_j : [B,H,c,D] float32
 *   accumulators (read and written).  All 16-byte aligned (LSE 4-byte).
 *   B, H, c, N >= 1;  0 <= i, j < N;  D == 128;  dtype RA_BF16.
 *   workspace : at least ra_bwd_workspace_bytes(B,H,c,D,1) bytes, 256-byte
 *   aligned.
 * Errors: RA_ERR_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA.
 */
RA_API int ra_bwd_step(const void* Q_i, const void* K_j, const void* V_j, const void* O_i,
           const float* LSE_i, const void* dO_i,
           float* dQ_i, float* dK_j, float* dV_j,
           int64_t B, int64_t H, int64_t c, int64_t D, int64_t N, int64_t i, int64_t j,
           int causal, int layout, int dtype,
           void* workspace, size_t ws_bytes, void* stream);

/*
 * ra_bwd_noalloc -- ra_bwd for callers that cannot allocate device memory.
 *
 * No passage of the pages corresponds to this entry point: it exists for
 * callers that cannot hand ra_bwd a workspace, e.g. code running inside a host
 * framework that owns all device memory through its own pool and forbids side
 * allocations, or a latency-critical path that must not call cudaMalloc
 * (which can synchronise the device).  It computes exactly what ra_bwd
 * computes, with the same arguments minus the workspace, and allocates
 * nothing: the workspace is a fixed 48 MiB device array inside the library,
 * which every GPU that loads the library holds until the process exits.
 *
 *   Arguments, results and errors as for ra_bwd.  Sizes whose
 *   ra_bwd_workspace_bytes(B,H,S,D,N) exceeds 48 MiB (50331648 bytes) are
 *   rejected with RA_ERR_ARG and a message saying so; about 6 million query
 *   rows B*H*S fit (e.g. 32 heads of 131072 tokens need 32 MiB).
 *   The first call on each device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   All calls share the one array and leave their intermediate values in it;
 *   every value a call reads is first written by that same call.  Calls whose
 *   executions overlap on the GPU (different streams, or different host
 *   threads, on the same device) race on the array and give wrong results:
 *   serialise them.
 */
RA_API int ra_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
           const float* LSE, const void* dO,
           void* dQ, void* dK, void* dV,
           int64_t B, int64_t H, int64_t S, int64_t D, int64_t N,
           int causal, int layout, int dtype, void* stream);

/*
 * Ring decode ([CH] §5.6: at inference the query has length 1 and the long KV
 * cache is spread along the ring; [AQ] "超长序列推理与 KV Cache 分发": every
 * card keeps one segment of the cache; [FT] "局限与未来": split-KV decode).
 *
 * ra_decode -- attention of ONE new query token per (b, h) over its whole KV
 * cache: O = sum_t e^{s_t - LSE} V_t, s_t = q.K_t / sqrt(D), LSE = ln sum_t
 * e^{s_t}.  The cache's last row is the new token's own key/value, so every
 * cached key is visible (no mask).  The S cache rows are cut into N ring
 * blocks, block j = rows [j*c, min((j+1)*c, S)), c = ceil(S/N) (trailing
 * blocks may be short or empty); each block's partial state is computed from
 * that block alone and the partials are folded with the LogSumExp merge of
 * ra_merge.  Called with N = 1 on one block's segment, ra_decode is the
 * per-host step of a ring: its (O, LSE) chain through ra_merge.
 *
 *   q       : [B,H,D] bf16, 16-byte aligned.
 *   K, V    : [B,H,S,D] bf16 caches, 16-byte aligned.
 *   O       : [B,H,D] bf16 (output), 2-byte aligned.
 *   LSE     : [B,H] float32 (output), 4-byte aligned.
 *   B, H, S, N : >= 1 (N > S allowed: the extra blocks are empty).
 *   D       : 128.   dtype : RA_BF16.
 *   workspace, ws_bytes : caller-owned device memory, 256-byte aligned, of at
 *             least ra_decode_workspace_bytes(B, H, S, D, N) bytes (per-chunk
 *             partial states; contents on entry are ignored).
 * Errors: RA_ERR_ARG (null pointer, misalignment, sizes, workspace too small),
 * RA_ERR_UNSUPPORTED (dtype other than RA_BF16, D != 128), RA_ERR_CUDA.
 */
RA_API size_t ra_decode_workspace_bytes(int64_t B, int64_t H, int64_t S, int64_t D, int64_t N);
RA_API int ra_decode(const void* q, const void* K, const void* V,
                     int64_t B, int64_t H, int64_t S, int64_t D, int64_t N, int dtype,
                     void* O, float* LSE, void* workspace, size_t ws_bytes, void* stream);

/*
 * ra_ffn -- blockwise gated feedforward ([CH] §5.2: the feedforward acts on
 * each host's own block only and runs blockwise; §5.3: its largest activation
 * is bounded per block; the experiments use LLaMA-style models, whose
 * feedforward is the gated one):
 *     Y = (silu(X W1^T) * (X W3^T)) W2^T,   silu(a) = a / (1 + e^-a).
 * The T rows of X are processed `block_rows` at a time; the f-wide
 * intermediate of one block (bf16, in `workspace`) is the only intermediate.
 * Per block: one tensor-core GEMM with the gate/up pairing fused into its
 * epilogue, then one for the down projection.
 *
 *   X, Y    : [T, h] bf16 (input, output), 16-byte aligned.
 *   W1, W3  : [f, h] bf16; W2 : [h, f] bf16 (the (out, in) layout of a linear
 *             layer), 16-byte aligned.
 *   T, block_rows >= 1;  h a multiple of 256;  f a multiple of 128.
 *   dtype   : RA_BF16.
 *   workspace, ws_bytes : at least ra_ffn_workspace_bytes(T, h, f, block_rows)
 *             bytes (the block's intermediate, min(block_rows, T) * f bf16,
 *             then one 4-byte tile counter per launch), 256-byte aligned; its
 *             contents on entry do not matter.  Calls sharing a workspace
 *             must not overlap on the GPU.
 * Errors: RA_ERR_ARG (null pointer, sizes, alignment, workspace too small),
 * RA_ERR_UNSUPPORTED (dtype), RA_ERR_CUDA.
 */
RA_API size_t ra_ffn_workspace_bytes(int64_t T, int64_t h, int64_t f, int64_t block_rows);
RA_API int ra_ffn(const void* X, const void* W1, const void* W3, const void* W2, void* Y,
                  int64_t T, int64_t h, int64_t f, int64_t block_rows, int dtype,
                  void* workspace, size_t ws_bytes, void* stream);

/*
 * ra_set_timing_buffer -- per-virtual-host time accounting for later bf16
 * ra_fwd calls from any thread (process-wide setting; NULL disables).
 * `dev_buf` is a caller-owned device array of n uint64 that the caller zeroes;
 * a call with ring size N needs n >= N*N.  Entry [i*N + s] accumulates the
 * nanoseconds (%globaltimer) that the kernel's CTAs spent on query block i's
 * rows while processing ring step s (KV block (i - s) mod N).  This is the
 * per-virtual-device time of [FT] "因果掩码的负载均衡挑战".
 * Errors: RA_ERR_ARG (n < 1 with a non-NULL buffer).
 */
RA_API int ra_set_timing_buffer(uint64_t* dev_buf, size_t n);

/*
 * Kernel timing (opt-in measurement aid).  ra_set_kernel_timing(1) makes every
 * later ra_fwd / ra_bwd / ra_decode / ra_ffn call, from any thread, record CUDA events on its own
 * stream immediately before and after each kernel it launches; 0 turns it off
 * and drops unread records.  ra_kernel_times() waits for the recorded events,
 * writes one record per timed kernel (oldest call first) and releases them:
 *   call RA_CALL_FWD: kernel 0 = the forward kernel (bf16 on one CTA per SM,
 *                     or float32), kernel 1 = the bf16 forward on SM pairs
 *                     (see ra_set_fwd_kernel);
 *   call RA_CALL_BWD: kernel 0 = preprocess (D_vec, LSE*log2e),
 *                     kernel 1 = dK/dV kernel, kernel 2 = dQ kernel.
 *   call RA_CALL_DECODE: kernel 0 = per-chunk partials, kernel 1 = combine;
 *   call RA_CALL_FFN: kernel 2b = gated up projection of block b, 2b+1 = its
 *                     down projection (calls of more than 8 blocks run untimed).
 * `ms` is the event-to-event time in milliseconds; `sm_mhz` as described below.  *count receives the number
 * of records; if it exceeds `capacity`, the first `capacity` are written, the
 * rest are dropped and RA_ERR_ARG is returned.  The library creates (and keeps
 * for reuse) the events; no device memory is allocated.
 */
typedef enum { RA_CALL_FWD = 0, RA_CALL_BWD = 1, RA_CALL_DECODE = 2, RA_CALL_FFN = 3 } ra_call_kind;
typedef struct {
  int call;     /* ra_call_kind */
  int kernel;   /* index inside the call, see above */
  float ms;     /* duration, or -1 if it could not be measured */
  float sm_mhz; /* tensor-core kernels (bf16 forward, dK/dV, dQ): the SM clock
                   the kernel ran at, from its first CTA's cycle counter over
                   its own lifetime against the global nanosecond timer
                   (kept for up to 256 such kernels between two reads; -1
                   beyond that); -1 for the other kernels */
} ra_kernel_time;
RA_API int ra_set_kernel_timing(int enable);
RA_API int ra_kernel_times(ra_kernel_time* out, int capacity, int* count);

/*
 * ra_set_fwd_kernel -- which kernel the bf16 forward (ra_fwd, ra_fwd_step,
 * ra_fwd_step_fold) launches; a process-wide setting that applies to calls
 * made after it returns, from any thread, on any device.  Both kernels compute
 * the method's forward ("Ring Attention" explainer, aiqz.cc, §分块注意力: the
 * same tiles, the same online-softmax update, in the same order) and give
 * bit-identical results; they differ in how the GPU's SMs share the work:
 *   RA_FWD_SINGLE (the default): one CTA per SM, work units of 256 query rows;
 *   RA_FWD_PAIR: 2-CTA clusters on SM pairs, whose tensor-core MMAs span both
 *                SMs (M = 256) so that each SM loads only half of every K and
 *                V tile; work units of 512 query rows.  A call fails with
 *                RA_ERR_UNSUPPORTED if the device cannot hold one such cluster.
 * Returns RA_ERR_ARG for any other `kind`.  The float32 path is unaffected.
 */
typedef enum { RA_FWD_SINGLE = 0, RA_FWD_PAIR = 1 } ra_fwd_kernel;
RA_API int ra_set_fwd_kernel(int kind);

/*
 * ra_set_wait_test -- test aid for the bounded waits (no counterpart on the
 * pages).  ra_set_wait_test(1) makes the NEXT bf16 ra_fwd call (from any
 * thread) withhold the first query tile of every CTA, so no data for it ever
 * arrives: the kernel's waits run out after their 2-second limit, each CTA
 * abandons its work, releases its resources and returns, and the following
 * ra_check_device_status() returns RA_ERR_TIMEOUT.  That call's outputs are
 * unspecified; the device and the library stay usable.  The switch clears
 * itself once used; ra_set_wait_test(0) clears it unused.
 */
RA_API int ra_set_wait_test(int enable);

/*
 * ra_check_device_status -- synchronise `stream`, then read and clear the
 * library's device-side status word.  Returns RA_ERR_TIMEOUT if any kernel
 * launched since the previous check gave up a bounded wait (the kernel then
 * returned early and its outputs are unspecified), else RA_OK or RA_ERR_CUDA.
 */
RA_API int ra_check_device_status(void* stream);

/*
 * ra_read_checks -- report of the bounds-checked build (no counterpart on the
 * pages; it stands in for a memory checker).  libringattn_checked.so is built
 * from the same sources with every global-memory index of the epilogues and
 * of the merge, preprocess, decode and float32 kernels, and every TMA box
 * start coordinate, checked against the extent of the tensor it addresses.
 * A failed check skips that access (a skipped TMA copy makes its waiters time
 * out, so the call also reports RA_ERR_TIMEOUT) and is counted here.
 * Synchronises `stream`, copies the current device's record into *out and
 * clears it.  events[0]: rows of the bf16 forward whose running maximum jumped
 * past the rescale threshold after keys had been folded in (their O was
 * rescaled); events[1]: rescale passes over O (one per warp and tile);
 * events[2]: TMA boxes checked; events[3]: other accesses checked.
 * violations: accesses found out of bounds; first_site / first_index /
 * first_extent: where the first one was (site codes name kernel and access;
 * a TMA index packs z<<40 | y<<16 | x).
 * Errors: RA_ERR_UNSUPPORTED from the default build (libringattn.so), which
 * checks nothing; RA_ERR_ARG (null out); RA_ERR_CUDA.
 */
typedef struct {
  uint64_t events[8];
  uint32_t violations;
  uint32_t first_site;
  int64_t first_index;
  int64_t first_extent;
} ra_check_report;
RA_API int ra_read_checks(ra_check_report* out, void* stream);

/* Message for the calling thread's most recent non-OK status ("" if none). */
RA_API const char* ra_last_error(void);

/* Library version string, e.g. "ringattn 0.2 sm_103a" ("... checked" for the
 * bounds-checked build). */
RA_API const char* ra_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RINGATTN_H */
