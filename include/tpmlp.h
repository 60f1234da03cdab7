/*
 * tpmlp.h -- C ABI of the t-sharded Megatron tensor-parallel MLP block on one
 * GB300 (sm_103a).
 *
 * The block (row convention, all matrices row-major):
 *   GeLU  : A_i = X W1_i,  H_i = GeLU(A_i),                    Y = sum_i H_i W2_i
 *   SwiGLU: G_i = X W1_i,  U_i = X W3_i,  H_i = U_i * Swish(G_i), Y = sum_i H_i W2_i
 * with X [T x d], W1_i / W3_i [d x d_i] (column shard i of W1 / W3),
 * W2_i [d_i x d] (row shard i of W2), H_i [T x d_i], Y [T x d] and
 * sum_i d_i = d_ff.
 *   - Column split of W1 and the identity GeLU(X [W11, W12]) =
 *     [GeLU(X W11), GeLU(X W12)]; row split of W2 and the partial-sum identity
 *     [H1, H2][W21; W22] = H1 W21 + H2 W22; the SwiGLU split: "Parallelism"
 *     tag page of Jiang Yi's homepage, post "megatron-lm", Method / FFN.
 *   - f is the identity forward and a sum (all-reduce) backward; g is a sum
 *     forward and the identity backward: same page, the f/g operator table;
 *     "Tensor parallelism" (brunomaga.github.io), Megatron_f / Megatron_g;
 *     "AI Training Network Primer" ch. 3, section 3.4, Fig. 3.4 and 3.6.
 * Optional biases (any may be NULL): b1_i [d_i] (SwiGLU also b3_i [d_i]) are
 * added to X W1_i (X W3_i) before the activation; b2 [d] is added to Y once,
 * after the g-sum, not once per shard ("Tensor parallelism",
 * brunomaga.github.io, Megatron_FeedForward: fc2 has no bias, fc2_bias is
 * added after the all-reduce).  Their gradients are sums over tokens:
 * db2 = sum_r dY[r, :], db1_i = sum_r dA_i[r, :] (SwiGLU dG_i), db3_i =
 * sum_r dU_i[r, :]; they cost one extra, HBM-bound launch per backward phase
 * that asks for them.
 * On one GPU the t shards sit side by side in HBM and both sums are
 * accumulations in the kernels' fp32 accumulators: the g-sum inside the
 * row-parallel GEMM's K loop, the f-sum inside the dX GEMM's K loop.  There
 * is no collective.
 *
 * Conventions shared by every entry point
 *   - Pointers named X, W*, H, Y, dY, dX, dW*, saved, dact, workspace are
 *     DEVICE pointers owned by the caller; the library never allocates,
 *     frees or retains them.  Arrays of pointers (const void* const* W1 ...)
 *     are HOST arrays of t device pointers, read during the call only.
 *   - Every tensor is a dense row-major 2-D array of the plan's dtype, its
 *     start 16-byte aligned; with bf16, d and every d_i must be multiples of 8
 *     (16-byte rows for the tensor-memory-access engine), with fp32 of 4.
 *   - Calls are asynchronous on the given stream (0 = the legacy default
 *     stream).  Argument errors are reported synchronously before anything
 *     is launched.  A device-side watchdog (a bounded wait inside the
 *     kernels) records TPMLP_ERR_DEVICE_TIMEOUT in the workspace's status
 *     word instead of hanging; tpmlp_check() reads and clears it.
 *   - Outputs are overwritten, never accumulated into.  Results are
 *     deterministic: every reduction has a fixed order, with no atomics
 *     on data (see tpmlp_plan_set_stream_k for the one dependence on the
 *     device's SM count).
 *   - Thread safety: a plan is immutable after creation and may be used from
 *     several threads; calls that share a workspace must be ordered on the
 *     device (same stream or events).
 */
#ifndef TPMLP_H_
#define TPMLP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TPMLP_API __attribute__((visibility("default")))
#else
#define TPMLP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tpmlp_stream_t; /* == cudaStream_t */

typedef enum {
  TPMLP_OK = 0,
  TPMLP_ERR_INVALID_ARG = 1,     /* NULL pointer, bad enum value, NULL plan */
  TPMLP_ERR_SHAPE = 2,           /* T < 0, d < 1, t < 1 or > TPMLP_MAX_SHARDS, some d_i < 1 */
  TPMLP_ERR_ALIGNMENT = 3,       /* a pointer not 16-byte aligned, d or d_i not a multiple of 8 (bf16) / 4 (fp32) */
  TPMLP_ERR_UNSUPPORTED = 4,     /* device is not sm_103 (GB300) or a size beyond the kernels' limits */
  TPMLP_ERR_CUDA = 5,            /* a CUDA runtime/driver call failed; see tpmlp_last_cuda_error() */
  TPMLP_ERR_DEVICE_TIMEOUT = 6,  /* a kernel's bounded wait expired (reported by tpmlp_check) */
  TPMLP_ERR_NOT_IMPLEMENTED = 7
} tpmlp_status;

typedef enum { TPMLP_ACT_GELU = 0, TPMLP_ACT_SWIGLU = 1 } tpmlp_act;
typedef enum { TPMLP_BF16 = 0, TPMLP_FP32 = 1 } tpmlp_dtype;

#define TPMLP_MAX_SHARDS 16

/* Problem description.  d_i points to t shard widths (host memory, copied
 * by tpmlp_plan_create).  Shard i covers hidden units [o_i, o_i + d_i) with
 * o_i = d_0 + ... + d_{i-1}; widths may differ (the pages allow
 * d_1 + d_2 = d_ff with d_1 != d_2).                                          */
typedef struct {
  int64_t T;           /* tokens (b * s); may be 0 */
  int64_t d;           /* hidden size */
  int32_t t;           /* number of shards, 1 .. TPMLP_MAX_SHARDS */
  const int64_t* d_i;  /* t widths, sum = d_ff */
  tpmlp_act act;
  tpmlp_dtype dtype;   /* storage dtype of every tensor; accumulation is fp32 */
} tpmlp_desc;

typedef struct tpmlp_plan tpmlp_plan;

/* Validate desc and build a plan (host memory only).  On error *out is NULL. */
TPMLP_API tpmlp_status tpmlp_plan_create(const tpmlp_desc* desc, tpmlp_plan** out);
/* Free a plan (NULL is a no-op). */
TPMLP_API void tpmlp_plan_destroy(tpmlp_plan* plan);

/* Bytes of device workspace every call needs.  fp32 plans: a 256-byte block
 * holding the device status word.  bf16 plans: that block, then the ticket
 * counters and fp32 partial accumulators of the stream-K schedules (16 KB +
 * 160 x 256 KB, about 42 MB; see tpmlp_plan_set_stream_k).  The caller allocates it once,
 * zero-filled, and passes it to every call of this plan; calls that share it
 * must be ordered on the device.                                             */
TPMLP_API size_t tpmlp_workspace_size(const tpmlp_plan* plan);

/* Forward.  Inputs X [T x d]; W1[i], W3[i] (SwiGLU only; pass NULL for GeLU)
 * [d x d_i]; W2[i] [d_i x d]; optional biases b1[i], b3[i] (SwiGLU) [d_i] and
 * b2 [d] (NULL for none; b1 and b3 are arrays of t device pointers).
 * Outputs: Y [T x d]; H[i] [T x d_i]; saved =
 * the pre-activations kept for backward: GeLU t pointers A_i [T x d_i];
 * SwiGLU 2t pointers, G_0..G_{t-1} then U_0..U_{t-1}, each [T x d_i].
 * Two kernels run: the column-parallel GEMM with the activation fused into
 * its epilogue (f forward = identity: X is read by every shard), then the
 * row-parallel GEMM whose K loop walks shard 0..t-1 into one fp32
 * accumulator (the g-sum).                                                    */
TPMLP_API tpmlp_status tpmlp_forward(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                     const void* const* W3, const void* const* W2, const void* const* b1,
                                     const void* const* b3, const void* b2, void* Y, void* const* saved,
                                     void* const* H, void* workspace, tpmlp_stream_t stream);

/* Backward.  Inputs: X, W1, W3, W2 as in forward; saved and H as written by
 * tpmlp_forward; dY [T x d].  Outputs: dact = per-shard activation gradients
 * (GeLU t pointers dA_i; SwiGLU 2t pointers dG_0..dG_{t-1}, dU_0..dU_{t-1},
 * each [T x d_i]), dX [T x d], dW1[i], dW3[i] (SwiGLU only, else NULL)
 * [d x d_i], dW2[i] [d_i x d], and optionally the bias gradients db1[i],
 * db3[i] [d_i] and db2 [d] (NULL: not computed).
 * g backward is the identity (every shard reads the same dY).  Two kernels
 * run: (1) dH_i = dY W2_i^T with act' fused (writes dact) together with
 * dW2_i = H_i^T dY; (2) dX = sum_i dA_i W1_i^T (SwiGLU: + dU_i W3_i^T) with
 * the f-sum in one fp32 accumulator, together with dW1_i = X^T dA_i
 * (dW3_i = X^T dU_i).  With T = 0 the weight gradients are zero-filled.       */
TPMLP_API tpmlp_status tpmlp_backward(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                      const void* const* W3, const void* const* W2, const void* const* saved,
                                      const void* const* H, const void* dY, void* const* dact, void* dX,
                                      void* const* dW1, void* const* dW3, void* const* dW2, void* const* db1,
                                      void* const* db3, void* db2, void* workspace, tpmlp_stream_t stream);

/* Backward with recomputation: the same arguments and results as
 * tpmlp_backward, except that H is not read: the contents of H[i] may have
 * been discarded after tpmlp_forward (only X and the pre-activations in
 * saved must survive), and H[i] is used as scratch that ends up holding the
 * recomputed H_i = act(saved_i).  The first launch computes dact and writes
 * H_i from the saved pre-activations it already reads for act' (GeLU: A_i;
 * SwiGLU: U_i * Swish(G_i)); the second computes dX (the f-sum), dW1, dW3 and
 * dW2 = H_i^T dY.  This trades nothing in FLOPs for not keeping H between the
 * passes ("AI Training Network Primer" ch. 3, section 3.1, and the
 * "Parallelism" page's GPipe post: activation recomputation saves memory by
 * recomputing what the backward pass needs from what was kept).  Because H is
 * recomputed from the bf16 pre-activation rather than from the fp32
 * accumulator, dW2 may differ from tpmlp_backward's in the last bits.       */
TPMLP_API tpmlp_status tpmlp_backward_recompute(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                                const void* const* W3, const void* const* W2,
                                                const void* const* saved, void* const* H, const void* dY,
                                                void* const* dact, void* dX, void* const* dW1, void* const* dW3,
                                                void* const* dW2, void* const* db1, void* const* db3, void* db2,
                                                void* workspace, tpmlp_stream_t stream);

/* The two launches of tpmlp_forward, callable one at a time (same arguments
 * and layouts; each is exactly one kernel launch):
 *   tpmlp_forward_column: saved and H from X, W1 (and W3), b1 (and b3).
 *   tpmlp_forward_row:    Y = sum_i H_i W2_i + b2 (the g-sum in the accumulator). */
TPMLP_API tpmlp_status tpmlp_forward_column(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                            const void* const* W3, const void* const* b1, const void* const* b3,
                                            void* const* saved, void* const* H, void* workspace,
                                            tpmlp_stream_t stream);
TPMLP_API tpmlp_status tpmlp_forward_row(const tpmlp_plan* plan, const void* const* W2, const void* b2,
                                         void* const* H, void* Y, void* workspace, tpmlp_stream_t stream);

/* tpmlp_forward_row without a workspace argument, for callers that cannot
 * allocate device memory: code handed only its input and output buffers by a
 * host framework that owns the device allocator (a plugin or an operator
 * inside someone else's runtime), or a latency-bound caller that must not
 * call cudaMalloc because it synchronises the whole device.  The pages have
 * no counterpart: it is an interface variant, not a step of the method.
 *
 * Same arguments, layouts and result as tpmlp_forward_row with b2 = NULL
 * (one launch of the row-parallel GEMM whose K loop carries the g-sum).  Its only scratch, the
 * device status word, lives in a library-owned static device array of
 * 256 bytes (held by every GPU that loads the library until the process
 * exits); the call allocates and frees nothing.  The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress) with the device
 * current.  The address is
 * kept for the life of the process: after a cudaDeviceReset, which destroys
 * the device's context and the array with it, the kept address is stale, and
 * this entry point must not be called again in that process.  Each call clears
 * the status word on the stream, launches, then waits for the stream and
 * reports the kernel's status itself (TPMLP_ERR_DEVICE_TIMEOUT if a bounded
 * wait expired), so it blocks until its kernel has finished.  All calls on a
 * device share the array: calls that overlap on the GPU (other streams, other
 * host threads) race on the status word.  It never uses the stream-K tail
 * (whose flags and partial sums need the full workspace), so its results are
 * those of tpmlp_forward_row with TPMLP_STREAM_K_OFF.                       */
TPMLP_API tpmlp_status tpmlp_forward_row_noalloc(const tpmlp_plan* plan, const void* const* W2, void* const* H,
                                                 void* Y, tpmlp_stream_t stream);

/* The two launches of tpmlp_backward, callable one at a time:
 *   tpmlp_backward_dgrad: dact from dY, W2 and saved (act' fused), and dW2
 *                         from H and dY; db2 (optional) from dY.
 *   tpmlp_backward_fsum:  dX = sum_i dact_i W1_i^T (+ dU_i W3_i^T) (the
 *                         f-sum in the accumulator), dW1 and dW3 from X and
 *                         dact; db1, db3 (optional) from dact.  Must follow
 *                         tpmlp_backward_dgrad.
 * Each is one GEMM launch, plus one column-sum launch when bias gradients are
 * requested.                                                                 */
TPMLP_API tpmlp_status tpmlp_backward_dgrad(const tpmlp_plan* plan, const void* const* W2, const void* const* saved,
                                            const void* const* H, const void* dY, void* const* dact,
                                            void* const* dW2, void* db2, void* workspace, tpmlp_stream_t stream);
TPMLP_API tpmlp_status tpmlp_backward_fsum(const tpmlp_plan* plan, const void* X, const void* const* W1,
                                           const void* const* W3, const void* const* dact, void* dX,
                                           void* const* dW1, void* const* dW3, void* const* db1, void* const* db3,
                                           void* workspace, tpmlp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Sequence-parallel layout ("AI Training Network Primer" ch. 3, section 3.4,
 * Fig. 3.7): each rank of the TP group keeps a stripe of the tokens; an
 * all-gather rebuilds the full X before the block, and a reduce-scatter after
 * it sums the shards' partial outputs and gives each rank its own stripe of
 * Y; the backward pass mirrors it (all-gather of the dY stripes,
 * reduce-scatter of the partial dX).  On one GPU both collectives are layout:
 * the kernels read X and dY directly from the stripe buffers (the g- and
 * f-sums stay in the accumulators) and write each stripe's rows of Y and dX
 * into that stripe's buffer.  The activations (saved, H, dact) and all
 * weight and bias gradients keep their full layouts.
 *
 * tpmlp_plan_set_sequence_stripes: stripe j holds stripe_rows[j] >= 0
 * consecutive tokens, in token order; the rows sum to the plan's T; every
 * stripe but the first starts at a multiple of 128 tokens (no tensor-memory-
 * access box crosses a stripe).  Copied into the plan; may not be changed
 * while another call uses the plan.
 * Stripe arguments are HOST arrays of nstripes DEVICE pointers, each a dense
 * row-major [stripe_rows[j] x d] array (16-byte aligned; NULL allowed for an
 * empty stripe).  Otherwise the arguments, results and launches are those of
 * tpmlp_forward / tpmlp_backward (no recompute variant); db2 sums dY over all
 * stripes.  Without stripes set on the plan the calls fail with
 * TPMLP_ERR_INVALID_ARG.                                                      */
TPMLP_API tpmlp_status tpmlp_plan_set_sequence_stripes(tpmlp_plan* plan, int32_t nstripes,
                                                       const int64_t* stripe_rows);
TPMLP_API tpmlp_status tpmlp_forward_sp(const tpmlp_plan* plan, const void* const* X_stripes, const void* const* W1,
                                        const void* const* W3, const void* const* W2, const void* const* b1,
                                        const void* const* b3, const void* b2, void* const* Y_stripes,
                                        void* const* saved, void* const* H, void* workspace, tpmlp_stream_t stream);
TPMLP_API tpmlp_status tpmlp_backward_sp(const tpmlp_plan* plan, const void* const* X_stripes,
                                         const void* const* W1, const void* const* W3, const void* const* W2,
                                         const void* const* saved, const void* const* H,
                                         const void* const* dY_stripes, void* const* dact, void* const* dX_stripes,
                                         void* const* dW1, void* const* dW3, void* const* dW2, void* const* db1,
                                         void* const* db3, void* db2, void* workspace, tpmlp_stream_t stream);

/* ---------------------------------------------------------------------------
 * Attention projections of the tensor-parallel self-attention block.
 *
 * Q/K/V are column-parallel (split by heads: shard i owns a subset of the
 * heads) and the output projection is row-parallel with the g-sum; the f
 * operator sums the shards' input gradients in backward ("Parallelism" tag
 * page of Jiang Yi's homepage, post "megatron-lm", Method / Attention:
 * W_Q = [W_Q1, ..., W_Qh], O = [o_1, ..., o_h] W_O; "Tensor parallelism"
 * (brunomaga.github.io), Megatron_MHA: one column-parallel QKV linear of
 * width 3 x (local heads x head size) whose output is split into q, k, v, and a
 * row-parallel output projection followed by Megatron_g; "AI Training
 * Network Primer" ch. 3, section 3.4, Fig. 3.5: with grouped-query attention
 * a shard owns 16 query heads and one key/value head).  The attention core
 * (scores, mask, softmax, the product with V) runs between these calls and is
 * not part of this library.  Neither projection has a bias (Megatron_MHA
 * builds both linears with bias=False).
 *
 * Per shard i, with dq_i = its query heads x head size, dkv_i = its key/value
 * heads x head size (dkv_i = dq_i without grouped-query attention) and
 * n_i = dq_i + 2 dkv_i:
 *   Wqkv[i] [d x n_i]  = [WQ_i | WK_i | WV_i]  (columns 0..dq_i-1 are WQ_i,
 *                        then dkv_i columns of WK_i, then dkv_i of WV_i)
 *   QKV[i]  [T x n_i]  = X Wqkv[i]             (= [Q_i | K_i | V_i])
 *   O[i]    [T x dq_i]   the attention core's output for the shard's heads
 *   WO[i]   [dq_i x d]   row shard i of the output projection
 *   Z       [T x d]    = sum_i O_i WO_i         (g: summed in the accumulator)
 * Backward, from dZ [T x d] and the core's dQKV[i] [T x n_i] =
 * [dQ_i | dK_i | dV_i]:
 *   dO[i]    = dZ WO_i^T              dWO[i]   = O_i^T dZ
 *   dX       = sum_i dQKV_i Wqkv_i^T  (f: summed in the accumulator)
 *   dWqkv[i] = X^T dQKV_i
 * Every call is one kernel launch; layouts, ownership, alignment, streams and
 * errors follow the conventions above (dq_i and dkv_i play the role of d_i).
 * The plan is an attention plan (tpmlp_attn_plan_create); passing it to an
 * MLP entry point, or an MLP plan here, is TPMLP_ERR_INVALID_ARG.  With T = 0
 * the weight gradients are zero-filled.                                       */
typedef struct {
  int64_t T;             /* tokens (b * s); may be 0 */
  int64_t d;             /* hidden size */
  int32_t t;             /* number of shards, 1 .. TPMLP_MAX_SHARDS */
  const int64_t* dq_i;   /* t query widths (host memory, copied) */
  const int64_t* dkv_i;  /* t key/value widths (host memory, copied) */
  tpmlp_dtype dtype;
} tpmlp_attn_desc;

/* Validate desc and build an attention plan (destroy with tpmlp_plan_destroy;
 * its workspace size is tpmlp_workspace_size's).                              */
TPMLP_API tpmlp_status tpmlp_attn_plan_create(const tpmlp_attn_desc* desc, tpmlp_plan** out);
/* QKV[i] = X Wqkv[i] for every shard (f forward is the identity). */
TPMLP_API tpmlp_status tpmlp_attn_qkv_forward(const tpmlp_plan* plan, const void* X, const void* const* Wqkv,
                                              void* const* QKV, void* workspace, tpmlp_stream_t stream);
/* Z = sum_i O[i] WO[i], the g-sum inside one fp32 accumulator. */
TPMLP_API tpmlp_status tpmlp_attn_out_forward(const tpmlp_plan* plan, const void* const* WO, const void* const* O,
                                              void* Z, void* workspace, tpmlp_stream_t stream);
/* dO[i] = dZ WO[i]^T and dWO[i] = O[i]^T dZ (g backward is the identity). */
TPMLP_API tpmlp_status tpmlp_attn_out_backward(const tpmlp_plan* plan, const void* const* WO, const void* const* O,
                                               const void* dZ, void* const* dO, void* const* dWO, void* workspace,
                                               tpmlp_stream_t stream);
/* dX = sum_i dQKV[i] Wqkv[i]^T (the f-sum) and dWqkv[i] = X^T dQKV[i]. */
TPMLP_API tpmlp_status tpmlp_attn_qkv_backward(const tpmlp_plan* plan, const void* X, const void* const* Wqkv,
                                               const void* const* dQKV, void* dX, void* const* dWqkv,
                                               void* workspace, tpmlp_stream_t stream);

/* Watchdog controls, for testing the failure path without faulting a GPU.
 * Neither may run while another call uses the plan.
 *   tpmlp_plan_set_timeout: bound, in milliseconds (>= 1), of every wait
 *     inside this plan's kernels (default 2000; the environment variable
 *     TPMLP_WAIT_TIMEOUT_MS sets the default of new plans).
 *   tpmlp_plan_set_stall_injection: with enable != 0 the tensor-core kernels
 *     of this plan load nothing, so the first wait of their MMA issuer is
 *     never satisfied and runs out after the timeout; the kernel then records
 *     TPMLP_ERR_DEVICE_TIMEOUT in the status word, every role leaves its loop,
 *     the CTAs free their TMEM and exit, and the CUDA context stays usable.
 *     Outputs are undefined while it is enabled.  The fp32 path has no waits
 *     and ignores it.  enable == 2 instead delays every part of a split
 *     stream-K tile but its first (see tpmlp_plan_set_stream_k) by 20 ms, as
 *     if their CTA pairs ran late: another part than the first then finishes
 *     the tile; results and status must be those of a run without it.      */
TPMLP_API tpmlp_status tpmlp_plan_set_timeout(tpmlp_plan* plan, uint32_t timeout_ms);
TPMLP_API tpmlp_status tpmlp_plan_set_stall_injection(tpmlp_plan* plan, int enable);

/* Stream-K schedules of the bf16 (tensor-core) launches.  A launch deals its
 * 256 x 256 tiles to the resident CTA pairs round robin; when the tile count
 * is not a multiple of the pairs, the last wave leaves pairs idle, and when
 * a launch mixes long-K weight-gradient tiles (K = T) with short ones, the
 * pairs that draw a long tile finish late.  A stream-K schedule cuts the K
 * blocks of some tiles into ranges, one per pair: every part of a split tile
 * leaves its fp32 accumulator in the workspace and takes a ticket; the part
 * that takes the last ticket adds all parts in K order and finishes the
 * tile.  No pair waits for another, so the schedule makes no assumption about
 * which pairs are resident or when they run (other kernels may share the
 * GPU).  The fixed order keeps results deterministic for a given device, but
 * they differ in rounding from the unsplit K sum (within the fp32
 * accumulation bound) and depend on the pair count, i.e. on the device's SM
 * count.
 *   TPMLP_STREAM_K_AUTO (default): per launch, the last partial wave of
 *     equal-depth tiles is split, when that shortens a pair's work by at
 *     least 2 % and 16 K blocks of 128 after charging each extra part its
 *     read-back;
 *   TPMLP_STREAM_K_ALWAYS: the last wave of every launch whose last wave has
 *     at most pairs / 2 tiles, with as many parts as fit (tests);
 *   TPMLP_STREAM_K_BALANCE: the launch's long-K weight-gradient tiles are
 *     placed last and their K blocks spread over the pairs so that every pair
 *     ends with the same estimated work (a launch without such tiles spreads
 *     all of its tiles); a range of K blocks may then end inside one tile,
 *     cover whole tiles and start inside another;
 *   TPMLP_STREAM_K_OFF: plain round robin.
 * tpmlp_forward_row_noalloc never uses it.  Not while another call uses the
 * plan.                                                                      */
#define TPMLP_STREAM_K_OFF 0
#define TPMLP_STREAM_K_AUTO 1
#define TPMLP_STREAM_K_ALWAYS 2
#define TPMLP_STREAM_K_BALANCE 3
TPMLP_API tpmlp_status tpmlp_plan_set_stream_k(tpmlp_plan* plan, int mode);

/* Synchronise the stream, read the workspace's status word and clear it.
 * Returns TPMLP_OK, TPMLP_ERR_DEVICE_TIMEOUT, or TPMLP_ERR_CUDA.               */
TPMLP_API tpmlp_status tpmlp_check(const tpmlp_plan* plan, void* workspace, tpmlp_stream_t stream);

/* Human-readable name of a status code (static string). */
TPMLP_API const char* tpmlp_status_string(tpmlp_status status);
/* The last CUDA error code seen by this thread (0 if none), for TPMLP_ERR_CUDA. */
TPMLP_API int tpmlp_last_cuda_error(void);
/* Description of the last failure on this thread (argument, CUDA or tensor
 * map error; empty string after a successful call).  Static storage per
 * thread, valid until the next call on the same thread.                      */
TPMLP_API const char* tpmlp_last_error(void);
/* ABI version: 100 * major + minor (1.01: optional biases; 1.02: attention
 * projections; 1.03: sequence-parallel layout; 1.04: stream-K tail, larger
 * bf16 workspace; 1.05: tpmlp_last_split_tiles, tpmlp_eval_activation, a
 * 16 KB counter block in the bf16 workspace). */
TPMLP_API int tpmlp_version(void);

/* Kernel launches the last compute call (tpmlp_forward, tpmlp_backward, a
 * phase or an attention entry point) on this thread made (for accounting; 0
 * before the first call).                                                    */
TPMLP_API int tpmlp_last_launch_count(void);

/* Diagnostics of the stream-K schedules (see tpmlp_plan_set_stream_k), for
 * tests that must know which output tiles were computed in parts.
 * launch_kind names a launch of the block:
 *   0 the column-parallel GEMM (tpmlp_forward_column), 1 the row-parallel
 *   GEMM with the g-sum (tpmlp_forward_row), 2 the dgrad launch
 *   (tpmlp_backward_dgrad), 3 the f-sum launch (tpmlp_backward_fsum),
 *   4..7 the attention projections' QKV forward, output forward, output
 *   backward and QKV backward.
 * Returns how many tiles the last launch of that kind made on this thread
 * split into parts (0 if none, or no such launch yet; -1 for an unknown
 * kind) and writes the first min(count, cap) of them to tiles (host memory,
 * may be NULL) as quadruples: the problem's index in its launch, the tile's
 * first output row, its first output column, and the device address of the
 * problem's first output (Y, dX, the pre-activation, dA, dG, dW1, dW2 ... as
 * the caller passed it; 0 for a token-striped output), which identifies the
 * tensor the tile belongs to.                                                */
TPMLP_API int tpmlp_last_split_tiles(int launch_kind, int64_t* tiles, int cap);

/* The activation forms of the kernels' epilogues, evaluated on plain fp32
 * device arrays of n elements (x = the pre-activation A or the gate G, y =
 * the up projection U, dh = the incoming gradient dH), so that they can be
 * checked against a reference over any set of inputs.  The bf16 tensor-core
 * epilogues compute Phi from the rational approximation of erf given as
 * formula 7.1.26 in Abramowitz & Stegun (absolute error at most 1.5e-7) and
 * the sigmoid from the fast exponential and reciprocal; the fp32 path calls
 * erff and expf.  The GeLU forms are those of GeLU(a) = a Phi(a) and
 * GeLU'(a) = Phi(a) + a phi(a); Swish is g sigmoid(g) ("Parallelism" tag page
 * of Jiang Yi's homepage, post "megatron-lm", Method / FFN and the SwiGLU
 * listing; "Tensor parallelism", brunomaga.github.io, Megatron_FeedForward's
 * F.gelu).  Outputs (device, fp32, n elements; unused ones may be NULL):
 *   TPMLP_ACT_EVAL_GELU        out0 = GeLU(x)                       (bf16 column epilogue)
 *   TPMLP_ACT_EVAL_GELU_BWD    out0 = dh GeLU'(x)                   (bf16 dgrad epilogue)
 *   TPMLP_ACT_EVAL_GELU_BWD_H  out0 = dh GeLU'(x), out1 = GeLU(x)   (same, with H recomputed)
 *   TPMLP_ACT_EVAL_SWIGLU      out0 = y Swish(x)                    (bf16 column epilogue)
 *   TPMLP_ACT_EVAL_SWIGLU_BWD  out0 = dG = dh y Swish'(x), out1 = dU = dh Swish(x)
 *   TPMLP_ACT_EVAL_SWIGLU_BWD_H  the same and out2 = y Swish(x)     (H recomputed)
 *   TPMLP_ACT_EVAL_FP32_GELU   out0 = GeLU(x), out1 = dh GeLU'(x)   (fp32 path)
 *   TPMLP_ACT_EVAL_FP32_SWIGLU out0 = y Swish(x), out1 = dG, out2 = dU (fp32 path)
 * Inputs an entry does not read may be NULL.  Asynchronous on the stream;
 * one kernel launch.  Errors: TPMLP_ERR_INVALID_ARG (unknown fn, n < 0, a
 * needed pointer NULL), TPMLP_ERR_ALIGNMENT (a pointer not 4-byte aligned),
 * TPMLP_ERR_UNSUPPORTED (not sm_103), TPMLP_ERR_CUDA.                        */
#define TPMLP_ACT_EVAL_GELU 0
#define TPMLP_ACT_EVAL_GELU_BWD 1
#define TPMLP_ACT_EVAL_GELU_BWD_H 2
#define TPMLP_ACT_EVAL_SWIGLU 3
#define TPMLP_ACT_EVAL_SWIGLU_BWD 4
#define TPMLP_ACT_EVAL_SWIGLU_BWD_H 5
#define TPMLP_ACT_EVAL_FP32_GELU 6
#define TPMLP_ACT_EVAL_FP32_SWIGLU 7
TPMLP_API tpmlp_status tpmlp_eval_activation(int fn, const float* x, const float* y, const float* dh, float* out0,
                                             float* out1, float* out2, int64_t n, tpmlp_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* TPMLP_H_ */
