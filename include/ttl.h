/*
 * ttl.h -- C ABI of the tensor-parallel transformer-block library (GB300, sm_103a).
 *
 * One process drives one GPU.  The t tensor-parallel "ranks" of the method are t
 * logical shards held as separate device buffers on that GPU, and every collective
 * of the method (all-reduce, reduce-scatter, all-gather) is an on-device kernel over
 * those buffers.  There are no inter-GPU collectives.
 *
 * Conventions for every entry point:
 *  - Matrices are row-major.  `ttl_bf16` is IEEE bfloat16 storage; fp32 is IEEE binary32.
 *  - Every data pointer is a DEVICE pointer owned by the caller.  The library does not
 *    allocate device memory; where it needs scratch it asks for a caller-provided
 *    workspace whose size a *_workspace_size() function reports.
 *  - A shard set is a HOST array of t (or g) device pointers, one per shard; each shard
 *    may be its own allocation.  The host array only needs to live for the call.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream); `event` arguments are
 *    cudaEvent_t.  Every call is asynchronous on its stream unless it says otherwise.
 *  - Device pointers and leading dimensions must be 16-byte aligned (TMA and 128-bit
 *    accesses); violations return TTL_ERR_ALIGN before anything is launched.
 *  - Return value: TTL_OK or an error code; ttl_last_error() then describes the failure
 *    (thread-local).  Argument errors are detected on the host before any launch.
 *    Errors found by a kernel (a bounded wait that timed out, an out-of-range CE target)
 *    are recorded in a per-device status word that ttl_device_status() reads.
 *  - Weights cross the boundary in math orientation [in, out] (the pages' "weight
 *    [k, n]"), except the LM head, which is [V, h] (vocab rows).
 *
 * Sources (web pages on Megatron-style tensor parallelism):
 *  [TPSP] "v4:Tensor Parallel 与 Sequence Parallel"
 *  [COMM] "TP 的 communication:一层几次?每次多少数据?"
 *  [GTP]  "Generalized Tensor Parallelism(GTP)是什么?"
 */
#ifndef TTL_H_
#define TTL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ttl_bf16;

/* Status codes. */
#define TTL_OK 0
#define TTL_ERR_ARG 1         /* null pointer, negative size, bad enum value           */
#define TTL_ERR_SHAPE 2       /* shape not divisible as the method requires            */
#define TTL_ERR_ALIGN 3       /* pointer or leading dimension not 16-byte aligned      */
#define TTL_ERR_CUDA 4        /* a CUDA runtime/driver call failed                     */
#define TTL_ERR_TIMEOUT 5     /* a bounded device-side wait ran out                    */
#define TTL_ERR_DEVICE 6      /* a kernel found invalid data (e.g. CE target >= V)     */
#define TTL_ERR_UNSUPPORTED 7 /* no sm_103a device, or a size beyond a stated maximum  */

#define TTL_MAX_SHARDS 16     /* largest t (and g) accepted                             */

#define TTL_ACT_GELU_TANH 0   /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))         */
#define TTL_ACT_SWIGLU 1      /* SiLU(x Wg) * (x Wu), no bias                            */

/* ------------------------------------------------------------------ housekeeping */

/* Human-readable description of the last error returned on this thread. */
const char* ttl_last_error(void);

/* Library ABI version (major * 100 + minor). */
int ttl_version(void);

/* Synchronises `stream`, then reads and clears the current device's status word.
 * *status_out receives TTL_OK or the first error a kernel recorded since the last call.
 * Returns TTL_OK unless the synchronisation itself failed. */
int ttl_device_status(void* stream, int* status_out);

/* Failure-path self test: launches one CTA that waits on an mbarrier nobody arrives on,
 * with a wall-clock limit of `timeout_us` microseconds (1 .. 10^6).  The wait gives up,
 * records TTL_ERR_TIMEOUT in the status word and the kernel returns normally, so the
 * context stays usable.  Synchronous; returns what ttl_device_status() would report. */
int ttl_selftest_wait_timeout(int64_t timeout_us, void* stream);

/* ------------------------------------------------------------------ launch tracing */

/* Kernel kinds reported by the tracer. */
#define TTL_K_GEMM 0        /* tcgen05 grouped GEMM (any epilogue)            */
#define TTL_K_REDUCE 1      /* shard reduce-scatter / all-reduce              */
#define TTL_K_GATHER 2      /* shard all-gather                               */
#define TTL_K_GTP_GATHER 3  /* GTP shard -> slot gather                       */
#define TTL_K_FINALIZE 4    /* GTP main_grad += staging                       */
#define TTL_K_CE_STATS 5    /* CE per-shard max / sum-exp / target logit      */
#define TTL_K_CE_SMALL 6    /* CE combine and mean                            */
#define TTL_K_CE_DLOGITS 7  /* CE dlogits                                     */
#define TTL_K_OTHER 8       /* column sums, zero fills                        */
#define TTL_K_EMBED 9       /* vocab-parallel embedding lookup / gradient     */
#define TTL_K_SOFTMAX 10    /* attention row softmax / softmax backward       */
#define TTL_K_ATTN_CORE 11  /* fused attention cores (scores, softmax, P V)  */

/* Starts (on != 0) or stops tracing on this process.  While on, every kernel launch the
 * library makes is bracketed by a pair of CUDA events recorded on the launch stream, and
 * the launch's algorithmic FLOPs and HBM bytes are noted.  Starting clears old records;
 * at most `capacity` launches are kept (1 .. 1<<20).  Events are created by this call. */
int ttl_trace_enable(int on, int capacity);

/* Synchronises on the recorded events and copies up to `max` records: kind, elapsed
 * milliseconds, FLOPs and bytes per launch.  *count receives the number recorded. */
int ttl_trace_read(int max, int* kind, float* ms, double* flops, double* bytes, int* count);

/* ------------------------------------------------------------------ GEMM core */

/* D[M,N] = op(A)[M,K] . op(B)[K,N] on the tcgen05 tensor cores, fp32 accumulation.
 * A is stored [M,K] (a_kmajor = 1) or [K,M] (a_kmajor = 0); B is stored [N,K]
 * (b_kmajor = 1) or [K,N] (b_kmajor = 0); lda/ldb/ldd are the row strides in elements.
 * D is bf16 (d_fp32 = 0) or fp32 (d_fp32 = 1).  M, N, K >= 0; N, K and the strides
 * multiples of 8.  This is the plain building block; the TP entry points below fuse
 * their activations and reductions around the same kernel.  [TPSP] "TP 的数学". */
int ttl_gemm(int64_t M, int64_t N, int64_t K, const ttl_bf16* A, int64_t lda, int a_kmajor,
             const ttl_bf16* B, int64_t ldb, int b_kmajor, void* D, int64_t ldd, int d_fp32,
             void* stream);

/* ------------------------------------------------------------------ partial-sum reduction */

/* The t buffers are full-shape partial sums [rows, cols] bf16 (cols a multiple of 8, t
 * dividing rows).  Buffer r owns token slab r = rows [r*rows/t, (r+1)*rows/t).
 * Sums are taken in fp32 in buffer order 0..t-1 and rounded once to bf16 (round to
 * nearest even); `bias` (nullable, bf16 [cols]) is the row-parallel bias, added once to
 * the sum before rounding.  [COMM] "Ring all-reduce" and Fig. 2; [TPSP] "SP". */

/* Reduce-scatter in place: slab r of buffer r <- sum over all buffers' slab r.
 * Other slabs are not written. */
int ttl_shard_reduce_scatter(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, const ttl_bf16* bias,
                             void* stream);

/* All-gather in place: slab r of buffer r is copied (bit-exact) into every other buffer. */
int ttl_shard_all_gather(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, void* stream);

/* All-reduce = reduce-scatter + all-gather, fused into one pass: every buffer ends with
 * the same bits the two phases would give.  Having no slabs to own, it accepts any number of
 * rows (t need not divide rows). */
int ttl_shard_all_reduce(int t, int64_t rows, int64_t cols, ttl_bf16* const* bufs, const ttl_bf16* bias,
                         void* stream);

/* ------------------------------------------------------------------ TP MLP block */

/* Forward of the MLP block  f -> column fc1 -> activation -> row fc2 -> g.
 * [TPSP] "MLP:先 column,再 row" and the f/g pseudocode.
 *   X        [T,h]            input, full on every shard (f forward is the identity)
 *   A[i]     [h,f/t]          fc1 column shard i (SwiGLU: the gate weight)
 *   A_up[i]  [h,f/t]          SwiGLU up weight shard (NULL for GeLU)
 *   B[i]     [f/t,h]          fc2 row shard i
 *   b1[i]    [f/t]            optional column bias shard (GeLU only; NULL = none)
 *   b2       [h]              optional row bias, added once after the sum (NULL = none)
 *   U_save[i][T,f/t]          out: pre-activation (SwiGLU: the gate pre-activation G_i)
 *   V_save[i][T,f/t]          out: SwiGLU up pre-activation V_i (NULL for GeLU)
 *   Hact[i]  [T,f/t]          out: activation, the row layer's input
 *   Z[i]     [T,h]            out: first the partial H_i B_i, then (g forward) the
 *                             all-reduced Z in every buffer
 * t in 1..TTL_MAX_SHARDS must divide f.  All bf16. */
int ttl_tp_mlp_fwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* X,
                   const ttl_bf16* const* A, const ttl_bf16* const* A_up, const ttl_bf16* const* B,
                   const ttl_bf16* const* b1, const ttl_bf16* b2, ttl_bf16* const* U_save,
                   ttl_bf16* const* V_save, ttl_bf16* const* Hact, ttl_bf16* const* Z, void* stream);

/* Workspace bytes ttl_tp_mlp_bwd needs: the per-shard activation gradients
 * (GeLU: dU_i; SwiGLU: dG_i and dV_i), t x T x f/t bf16 each, 256-byte aligned. */
size_t ttl_tp_mlp_bwd_workspace_size(int t, int act, int64_t T, int64_t h, int64_t f);

/* Backward of the MLP block.  g backward is the identity (dY full on every shard);
 * row fc2 backward is local; f backward all-reduces dX.  [TPSP] table
 * "Column 和 Row 各在哪里通信", table "完整流程:column parallel,t = 3", bias question.
 *   dY [T,h]; X, A, A_up, B, U_save, V_save, Hact as saved by ttl_tp_mlp_fwd
 *   dA[i]    [h,f/t]   out  (SwiGLU: dWg_i)      dA_up[i] [h,f/t] out (SwiGLU: dWu_i)
 *   dB[i]    [f/t,h]   out                       db1[i]   [f/t]   out, optional (GeLU)
 *   db2      [h]       out, optional (the row bias gradient, once)
 *   dX[i]    [T,h]     out: partial dU_i A_i^T, then the all-reduced dX in every buffer
 *   ws       workspace of ttl_tp_mlp_bwd_workspace_size() bytes */
int ttl_tp_mlp_bwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* X, const ttl_bf16* dY,
                   const ttl_bf16* const* A, const ttl_bf16* const* A_up, const ttl_bf16* const* B,
                   const ttl_bf16* const* U_save, const ttl_bf16* const* V_save, const ttl_bf16* const* Hact,
                   ttl_bf16* const* dA, ttl_bf16* const* dA_up, ttl_bf16* const* dB, ttl_bf16* const* db1,
                   ttl_bf16* db2, ttl_bf16* const* dX, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ sequence-parallel MLP block */

/* The MLP block with sequence parallelism ([TPSP] "SP"): its input and output are t token
 * slabs of T/t rows (slab r = rows [r T/t, (r+1) T/t)), held by shard r.  The all-gather
 * before fc1 and the reduce-scatter after fc2 run inside the GEMMs: fc1 reads X slab by slab
 * through one tensor map per slab, and output slab r is one accumulator over the t shards'
 * H_i[slab r] B_i, so no full-shape partial sum is written.  The shard sums are taken in
 * fp32 inside that accumulator (the literal block rounds each partial to bf16 first).
 *   X_slabs[r] [T/t,h]; A, A_up, B, U_save, V_save, Hact as for ttl_tp_mlp_fwd (full T rows)
 *   Z_slabs[r] [T/t,h] out: slab r of the block output
 * t | T, T/t a multiple of 128, no biases. */
int ttl_sp_mlp_fwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* const* X_slabs,
                   const ttl_bf16* const* A, const ttl_bf16* const* A_up, const ttl_bf16* const* B,
                   ttl_bf16* const* U_save, ttl_bf16* const* V_save, ttl_bf16* const* Hact,
                   ttl_bf16* const* Z_slabs, void* stream);

/* Workspace bytes of ttl_sp_mlp_bwd (the same per-shard activation gradients as the TP block). */
size_t ttl_sp_mlp_bwd_workspace_size(int t, int act, int64_t T, int64_t h, int64_t f);

/* Backward of ttl_sp_mlp_fwd: dZ_slabs[r] [T/t,h] in, dX_slabs[r] [T/t,h] out.  The
 * all-gather of dZ (the reduce-scatter's backward) is folded into the dgrad's operand loads
 * and the weight gradients' K segments; the reduce-scatter of the dX partials (the
 * all-gather's backward) into the dX GEMM's K loop over shards.  dA, dA_up, dB as for
 * ttl_tp_mlp_bwd.  SwiGLU needs 2t <= 16. */
int ttl_sp_mlp_bwd(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* const* X_slabs,
                   const ttl_bf16* const* dZ_slabs, const ttl_bf16* const* A, const ttl_bf16* const* A_up,
                   const ttl_bf16* const* B, const ttl_bf16* const* U_save, const ttl_bf16* const* V_save,
                   const ttl_bf16* const* Hact, ttl_bf16* const* dA, ttl_bf16* const* dA_up, ttl_bf16* const* dB,
                   ttl_bf16* const* dX_slabs, void* ws, size_t ws_bytes, void* stream);

/* Size of the library's own scratch area used by ttl_tp_mlp_bwd_static_ws: 16 MiB. */
#define TTL_STATIC_WS_BYTES (16u << 20)

/* ttl_tp_mlp_bwd without a workspace argument, for callers that cannot allocate device
 * memory: for example a program whose device memory is all owned by another allocator that
 * forbids further cudaMalloc, or a latency-critical loop that must not pay for cudaMalloc and
 * its implicit device-wide synchronisation.  The pages have no counterpart to this entry
 * point; it exists only for such callers.
 *   Arguments and results are those of ttl_tp_mlp_bwd (minus ws / ws_bytes).  The scratch is
 *   a fixed TTL_STATIC_WS_BYTES array inside the library, present on every GPU that loads the
 *   library until the process exits.  A shape whose ttl_tp_mlp_bwd_workspace_size() exceeds
 *   it is rejected with TTL_ERR_UNSUPPORTED before anything runs.
 *   No device memory is allocated or freed.  The scratch used is the current device's, so
 *   the current device must be the one that holds every pointer argument and the stream.
 *   The first call on each device looks up the scratch's device address with that device
 *   current and keeps it for the life of the process; make that first call before any stream
 *   capture, and do not call this entry point again on a device after cudaDeviceReset (the
 *   kept address would be stale).
 *   All calls share the one scratch array, and it keeps whatever the last call left in it
 *   (nothing in it needs to start at zero: every element is written before it is read).
 *   Calls that overlap on the GPU (e.g. on two streams at once) race on it and give wrong
 *   results: order them on one stream or with events. */
int ttl_tp_mlp_bwd_static_ws(int t, int act, int64_t T, int64_t h, int64_t f, const ttl_bf16* X,
                             const ttl_bf16* dY, const ttl_bf16* const* A, const ttl_bf16* const* A_up,
                             const ttl_bf16* const* B, const ttl_bf16* const* U_save,
                             const ttl_bf16* const* V_save, const ttl_bf16* const* Hact, ttl_bf16* const* dA,
                             ttl_bf16* const* dA_up, ttl_bf16* const* dB, ttl_bf16* const* db1, ttl_bf16* db2,
                             ttl_bf16* const* dX, void* stream);

/* ------------------------------------------------------------------ GTP_remat weight path */

/* [GTP] concepts "GTP_remat", "Prefetch chain", "Deferred finalize", Fig. 1 and the list
 * "all-gather 和 weight gradient 怎么藏在计算后面".  A TP slice W [K,N] is held as g
 * row shards shards[j] = W[j*K/g : (j+1)*K/g, :] ([K/g, N] bf16, separate allocations);
 * g in 1..TTL_MAX_SHARDS divides K. */

/* Gather the g shards into `slot` [K,N] (bit-exact row concatenation) on `stream`
 * (typically a side stream), then record `done_event` on it if non-NULL. */
int ttl_gtp_gather(int g, int64_t K, int64_t N, const ttl_bf16* const* shards, ttl_bf16* slot, void* stream,
                   void* done_event);

/* The layer GEMM on the TP slice.  transpose_w = 0:  Y[M,N]  = X[M,K] . W
 *                                   transpose_w = 1:  Y[M,K]  = X[M,N] . W^T (dgrad)
 * If `slot` is non-NULL the GEMM reads the gathered slot (after making `stream` wait on
 * `slot_ready_event` if that is non-NULL); if `slot` is NULL the gather is folded into
 * the GEMM's operand loads, which read the shards directly (no slot needed). */
int ttl_gtp_gather_gemm(int g, int64_t M, int64_t K, int64_t N, const ttl_bf16* X,
                        const ttl_bf16* const* shards, const ttl_bf16* slot, void* slot_ready_event,
                        ttl_bf16* Y, int transpose_w, void* stream);

/* The finalize step alone: main_grad[j] += staging[j] (fp32, g shards of [K/g,N]) on `stream`.
 * [GTP] concept "Deferred finalize": the merge into main_grad runs one backward layer after
 * the layer's weight gradient.  A caller that wants it off the compute stream (the chain
 * helper does) passes staging_prev = NULL to ttl_gtp_wgrad_rs_finalize and issues this on
 * another stream after an event recorded behind that layer's weight-gradient call. */
int ttl_gtp_finalize(int g, int64_t K, int64_t N, const float* const* staging, float* const* main_grad,
                     void* stream);

/* Weight gradient of one layer, reduce-scattered into shards, with deferred finalize.
 *   staging_cur[j] [K/g,N] fp32 <- rows of X^T dY for shard j (the sum over the g token
 *                  groups' partials, folded into the GEMM's token contraction)
 *   staging_prev / main_grad_prev (both NULL or both set): finalize of the layer handled
 *                  one backward step earlier, main_grad_prev[j] += staging_prev[j]
 *   sync = 1:      also finalize this layer now, main_grad_cur[j] += staging_cur[j]
 *                  (the last backward layer: nothing follows it)
 *   X [M,K] bf16, dY [M,N] bf16; g divides K.
 * Both finalizes run inside the weight-gradient GEMM's epilogue, element by element beside
 * the tile it writes (one fp32 addition per element, as a separate pass would do), so they
 * add no launch to the critical path.  staging_prev may be staging_cur itself (one staging
 * set reused by every layer): each element of it is read before it is overwritten. */
int ttl_gtp_wgrad_rs_finalize(int g, int64_t M, int64_t K, int64_t N, const ttl_bf16* X, const ttl_bf16* dY,
                              float* const* staging_cur, const float* const* staging_prev,
                              float* const* main_grad_prev, int sync, float* const* main_grad_cur,
                              void* stream);

/* ------------------------------------------------------------------ vocab-parallel CE */

#define TTL_CE_FP32_DLOGITS 1  /* also write fp32 dlogits in place over `logits`  */
#define TTL_CE_FORWARD_ONLY 2  /* stop after the loss (no dlogits, no dH)         */

/* Column-parallel LM head + cross-entropy from three numbers per token.
 * [TPSP] "Embedding 和 LM head:按 vocab 切".  Shard i owns ids [i V/t, (i+1) V/t).
 *   H [T,h] bf16; W[i] [V/t,h] bf16; target [T] int64 in [0,V)
 *   logits[i]  [T,V/t] fp32   scratch: Z_i = H W_i^T (dlogits if TTL_CE_FP32_DLOGITS)
 *   dlogits[i] [T,V/t] bf16   out: (softmax - onehot) / T
 *   stats      [(3t+2) T] fp32 out: rows 3i, 3i+1, 3i+2 = shard i's max, sum exp(z - max),
 *              target logit (0 if not owned); row 3t = log-sum-exp; row 3t+1 = loss per token
 *   loss       [1] fp32 out: mean over the T tokens
 *   dH         [T,h] bf16 out: sum_i dlogits_i W_i
 *   ws         optional workspace of ttl_vocab_parallel_ce_workspace_size() bytes.  With it,
 *              the LM-head GEMM's epilogue computes each row's max and sum of exponentials
 *              tile by tile while it writes the logits, so the statistics never re-read the
 *              fp32 logits, and one launch merges them, combines the shards and takes the
 *              mean; with ws = NULL separate passes scan the logits, combine, and average.
 *              Same results up to fp32 rounding order.
 * t in 1..TTL_MAX_SHARDS divides V; V/t a multiple of 8.  A target outside [0,V) sets
 * TTL_ERR_DEVICE in the status word and that token's loss to NaN. */
int ttl_vocab_parallel_ce(int t, int64_t T, int64_t h, int64_t V, const ttl_bf16* H, const ttl_bf16* const* W,
                          const int64_t* target, float* const* logits, ttl_bf16* const* dlogits, float* stats,
                          float* loss, ttl_bf16* dH, void* ws, size_t ws_bytes, int flags, void* stream);

/* Bytes of the optional ttl_vocab_parallel_ce workspace: per token, 8 bytes for each 128-wide
 * half of a 256-wide column tile of every vocab shard, plus 4, each part rounded up to 256
 * bytes, plus 256 for a completion counter; 0 for invalid arguments. */
size_t ttl_vocab_parallel_ce_workspace_size(int t, int64_t T, int64_t h, int64_t V);

/* ------------------------------------------------------------------ vocab-parallel embedding */

/* Embedding lookup with the table split by vocabulary rows.  [TPSP] "Embedding 和 LM head:按
 * vocab 切": a shard outputs 0 for tokens whose id it does not own and the all-reduce of the
 * t outputs gives every token its own row.  Shard i owns ids [i V/t, (i+1) V/t).
 *   ids    [T] int64 in [0,V)   E[i] [V/t,h] bf16   out[i] [T,h] bf16 (every buffer ends
 *   with the looked-up rows)
 *   literal = 1: masked per-shard lookups, then the on-device all-reduce of the t buffers;
 *   literal = 0: one pass that copies each token's row from its owning shard into all t
 *                buffers (the same bits, without the all-reduce's traffic).
 * An id outside [0,V) sets TTL_ERR_DEVICE in the status word and gives a zero row. */
int ttl_vocab_parallel_embedding_fwd(int t, int64_t T, int64_t h, int64_t V, const int64_t* ids,
                                     const ttl_bf16* const* E, ttl_bf16* const* out, int literal, void* stream);

/* Backward: the all-reduce's backward is the identity, so shard i accumulates
 *   dE[i][id - i V/t] += dY[tok]   for every token whose id it owns
 * into fp32 dE[i] [V/t,h] (zero it first for a fresh gradient).  Tokens sharing an id are
 * summed with atomic adds, so the fp32 summation order is not fixed. */
int ttl_vocab_parallel_embedding_bwd(int t, int64_t T, int64_t h, int64_t V, const int64_t* ids,
                                     const ttl_bf16* dY, float* const* dE, void* stream);

/* ------------------------------------------------------------------ TP attention block */

/* Attention split by heads ([TPSP] "Attention:按 head 切"; [COMM] Fig. 1): shard i holds
 * query heads [i n_q/t, (i+1) n_q/t) and KV heads [i n_kv/t, (i+1) n_kv/t) (grouped-query
 * attention: query head j reads KV head j / (n_q / n_kv)); W_Q, W_K, W_V are column-parallel
 * by head, each shard computes its heads' attention alone, W_O is row-parallel and g
 * all-reduces the t partials.  The attention is causal scaled dot-product attention with
 * scale 1/sqrt(d) over one sequence of T tokens (no rotary embedding, no biases).  Matrices
 * are row-major bf16, head-major columns (head c at columns [c d, (c+1) d)).
 *   X [T,h]; Wq[i] [h, n_q/t d]; Wk[i], Wv[i] [h, n_kv/t d]; Wo[i] [n_q/t d, h]
 *   Q_save[i] [T, n_q/t d], K_save[i], V_save[i] [T, n_kv/t d], O_save[i] [T, n_q/t d]  out
 *   P_save[i] [n_q/t, T, T] out: the probabilities, head-major; row q is written for keys
 *             j < min(T, round_up(q+1, 128)) (zeros above the diagonal), the rest is untouched
 *   Y[i] [T,h] out: partial O_i Wo_i, then the all-reduced block output in every buffer
 *   ws   unused: ttl_tp_attn_fwd_workspace_size() returns 0 and ws may be null.  The scores
 *        and the softmax statistics stay on chip: one fused kernel per 128-query tile computes
 *        the scores twice in tensor memory (exact row statistics, then the probabilities, which
 *        feed P V from tensor memory)
 * t | n_q, t | n_kv, n_kv | n_q, d = 64 or 128, T and h multiples of 8.  Errors:
 * TTL_ERR_ARG (null or short arguments), TTL_ERR_SHAPE, TTL_ERR_ALIGN (pointers not 16-byte
 * aligned); nothing is launched when the call returns an error. */
size_t ttl_tp_attn_fwd_workspace_size(int t, int64_t T, int n_q, int n_kv, int d);
int ttl_tp_attn_fwd(int t, int64_t T, int64_t h, int n_q, int n_kv, int d, const ttl_bf16* X,
                    const ttl_bf16* const* Wq, const ttl_bf16* const* Wk, const ttl_bf16* const* Wv,
                    const ttl_bf16* const* Wo, ttl_bf16* const* Q_save, ttl_bf16* const* K_save,
                    ttl_bf16* const* V_save, ttl_bf16* const* P_save, ttl_bf16* const* O_save,
                    ttl_bf16* const* Y, void* ws, size_t ws_bytes, void* stream);

/* Backward of ttl_tp_attn_fwd: g backward is the identity (dY full on every shard), the heads'
 * attention backward is local (dS = P (dP - rowsum(dO O)) / sqrt(d), the KV gradients summed
 * over each group's query heads), f backward all-reduces dX.
 *   dY [T,h]; X, W*, *_save as given to / written by ttl_tp_attn_fwd
 *   dWq[i], dWk[i], dWv[i], dWo[i] out, shaped like the weights
 *   dX[i] [T,h] out: partial, then the all-reduced dX in every buffer
 *   ws   workspace of ttl_tp_attn_bwd_workspace_size() bytes: rowsum(dO O) per query row, then
 *        per shard dO, dQ, dK, dV.  The score gradients dS never reach memory: a kernel per
 *        query tile (dQ) and one per key tile (dK, dV) each recompute dP = dO V^T in tensor
 *        memory and dS from the saved P
 * T = 0 writes zero weight gradients (token-sized pointers may then be null). */
size_t ttl_tp_attn_bwd_workspace_size(int t, int64_t T, int n_q, int n_kv, int d);
int ttl_tp_attn_bwd(int t, int64_t T, int64_t h, int n_q, int n_kv, int d, const ttl_bf16* X,
                    const ttl_bf16* dY, const ttl_bf16* const* Wq, const ttl_bf16* const* Wk,
                    const ttl_bf16* const* Wv, const ttl_bf16* const* Wo, const ttl_bf16* const* Q_save,
                    const ttl_bf16* const* K_save, const ttl_bf16* const* V_save,
                    const ttl_bf16* const* P_save, const ttl_bf16* const* O_save, ttl_bf16* const* dWq,
                    ttl_bf16* const* dWk, ttl_bf16* const* dWv, ttl_bf16* const* dWo, ttl_bf16* const* dX,
                    void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TTL_H_ */
