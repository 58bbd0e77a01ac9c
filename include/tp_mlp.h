/*
 * tp_mlp.h - C ABI of libtpmlp.so, the tensor-parallel transformer MLP on
 * one GB300 (sm_103a).
 *
 * The method (Megatron-style tensor parallelism):
 *   - the first linear layer is column-parallel: W1 is split along its output
 *     dimension into T column blocks W1_i, X is replicated, Y_i = act(X W1_i)
 *     ("Tensor Parallelism in Action: Megatron-LM Matrix Splitting", section
 *     1, "Column Parallel (W1)"; "Slice the matrix itself", section
 *     "Column-Parallel & Row-Parallel GEMMs");
 *   - the activation needs no exchange because it is elementwise
 *     ("Tensor Parallelism in Action", section 2, question 2);
 *   - the second linear layer is row-parallel: W2 is split along its input
 *     dimension into T row blocks W2_i, giving partial products
 *     Z_i = Y_i W2_i ("Tensor Parallelism in Action", section 1, "Row
 *     Parallel (W2)");
 *   - one all-reduce-sum completes it, Z = sum_i Z_i ("Slice the matrix
 *     itself", section "Mathematical formulation - row-parallel matrix
 *     multiplication summation"; "Tensor parallelism" guide, section
 *     "Concept").
 * Here all T shards are partitions on ONE GPU and the all-reduce-sum is
 * arithmetic in device memory (or in the tensor-core accumulator): there is
 * no collective and nothing crosses GPUs.
 *
 * Conventions for every call:
 *   - Every call returns a tp_status_t (or a size); none aborts or throws.
 *   - Matrices are row-major.  The pages' convention Y = X W is used, so W1 is
 *     [H x F] (in x out) and W2 is [F x H].
 *   - Pointers are DEVICE pointers unless the name ends in _host / host_dst.
 *     Device pointers must be 16-byte aligned.  The caller owns every buffer
 *     it passes; the library owns only what a tp_shards_t holds and its own
 *     per-device status word.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued on it and the call returns without waiting, except where a
 *     call says otherwise.  Argument errors are returned synchronously;
 *     device-side errors (a wait that ran out, a failed device check) are
 *     reported by tp_last_device_status().
 *   - The calling thread's current CUDA device is used; it must be sm_103
 *     (GB300) or the call returns TP_ERR_ARCH.
 *   - Shapes are int64_t.  T (shards) is 1..64.
 */
#ifndef TP_MLP_H
#define TP_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TP_ABI_VERSION 1

/* Exported symbols of libtpmlp.so (the library hides everything else). */
#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

typedef enum {
    TP_OK = 0,
    TP_ERR_ARG = 1,          /* null pointer, bad size, misaligned pointer, bad enum */
    TP_ERR_INDIVISIBLE = 2,  /* F % T != 0 or n_heads % T != 0 (shards must be equal) */
    TP_ERR_DTYPE = 3,        /* element type not supported for this call */
    TP_ERR_ARCH = 4,         /* current device is not sm_103 */
    TP_ERR_OOM = 5,          /* device or host allocation failed */
    TP_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed */
    TP_ERR_TIMEOUT = 7,      /* a device-side wait ran past its limit (kernel returned early) */
    TP_ERR_DEVICE_CHECK = 8, /* a device-side check failed */
    TP_ERR_UNSUPPORTED = 9,  /* shape outside what the kernels tile (see each call) */
    TP_ERR_WORKSPACE = 10    /* workspace smaller than the *_workspace_bytes() figure */
} tp_status_t;

typedef enum {
    TP_ACT_GELU_ERF = 0,  /* GeLU(y) = 0.5 y (1 + erf(y / sqrt 2)) */
    TP_ACT_SWIGLU = 1,    /* h = SiLU(X Wg) * (X Wu), SiLU(g) = g / (1 + exp(-g)) */
    TP_ACT_IDENTITY = 2   /* no activation */
} tp_act_t;

typedef enum {
    TP_F32 = 0,   /* float32 in, float32 FMA (CUDA cores), float32 out */
    TP_BF16 = 1   /* bfloat16 in, float32 accumulate (tensor cores), float32 out */
} tp_dtype_t;

typedef enum {
    TP_VAR_AUTO = 0,      /* the library picks per shape */
    TP_VAR_PARTIALS = 1,  /* row-parallel GEMM writes T float32 partials, then the shard-sum */
    TP_VAR_TMEM_ACC = 2   /* one accumulator sums all shards' K ranges; partials never reach memory */
} tp_variant_t;

/* Opaque, library-owned sharded weights. */
typedef struct tp_shards *tp_shards_t;

/* Human-readable name of a status; never NULL. */
TP_API const char *tp_status_str(tp_status_t s);

/* TP_ABI_VERSION of the loaded library. */
TP_API int tp_abi_version(void);

/*
 * tp_shard_weights - the shard layout (column blocks of W1, row blocks of W2).
 * Pages: "Tensor Parallelism in Action", section 1 (W1 = [W1_1 | W1_2],
 * W2 = [W2_1; W2_2]); "Slice the matrix itself" ("First linear layer
 * (Gate/Up) is split column-wise ... Second linear layer (Down) is split
 * row-wise").
 *
 *   W1   [H x F] (GELU_ERF, IDENTITY) or [H x 2F] = [Wg | Wu] (SWIGLU, gate
 *        first), element type dt.
 *   W2   [F x H], element type dt.
 *   Shard i holds columns [i F/T, (i+1) F/T) of W1 (for SWIGLU the SAME
 *   columns of Wg and of Wu) and rows [i F/T, (i+1) F/T) of W2.  The copies
 *   are bit-exact; the device layout is K-major (each shard's W1_i and W2_i
 *   stored transposed, [out x in]) for the tensor-core GEMMs, and for TP_BF16
 *   cut into k-tiles of 64 columns (each tile holding the 64 K values of every
 *   row contiguously).  tp_shard_get returns the logical shard.
 *   W1 and W2 are only read; the caller may free them once `stream` has
 *   reached the end of this call's work.
 *   Errors: F % T != 0 -> TP_ERR_INDIVISIBLE; for TP_BF16, H % 128 != 0 or
 *   F/T % 128 != 0 -> TP_ERR_UNSUPPORTED (the tensor-core tiles are 128
 *   rows by 64 K); SWIGLU with F/T % 128 != 0 -> TP_ERR_UNSUPPORTED;
 *   allocation -> TP_ERR_OOM.
 *   *out receives a handle to free with tp_shards_destroy().
 */
TP_API tp_status_t tp_shard_weights(const void *W1, const void *W2, int64_t H, int64_t F, int T,
                             tp_act_t act, tp_dtype_t dt, void *stream, tp_shards_t *out);

/*
 * tp_shard_weights_qkv - head-sharded attention projections ("Tensor
 * parallelism" guide, section "Walking through a transformer block": shard
 * heads across ranks; the output projection is row-parallel and ends in an
 * all-reduce, "Slice the matrix itself", section "All-Reduce Synchronization").
 *
 *   Wqkv [H x 3H] = [Wq | Wk | Wv], head h in columns [h hd, (h+1) hd) of
 *        each; bfloat16.
 *   Wo   [H x H], input rows grouped by head the same way; bfloat16.
 *   Shard i holds heads [i nh/T, (i+1) nh/T): those columns of Wq, Wk and
 *   Wv (3 W columns, W = nh/T * hd) and those W rows of Wo.
 *   Errors: n_heads * head_dim != H -> TP_ERR_ARG; n_heads % T != 0 ->
 *   TP_ERR_INDIVISIBLE; H % 128, W % 64 or 3W % 128 != 0 ->
 *   TP_ERR_UNSUPPORTED.
 */
TP_API tp_status_t tp_shard_weights_qkv(const void *Wqkv, const void *Wo, int64_t H, int n_heads,
                                 int head_dim, int T, void *stream, tp_shards_t *out);

/*
 * tp_shard_get - copy the LOGICAL shard i to host memory, row-major, for
 * bit-exact layout checks.  Synchronous (waits for the device).
 *   MLP shards: which = 0 -> W1_i (Wg_i for SWIGLU) [H x F/T];
 *               which = 1 -> Wu_i [H x F/T] (SWIGLU only);
 *               which = 2 -> W2_i [F/T x H].
 *   QKV shards: which = 0 -> Wqkv_i [H x 3W] (= [Wq_i | Wk_i | Wv_i]);
 *               which = 2 -> Wo_i [W x H].
 *   host_dst must hold that many elements of the shards' element type.
 */
TP_API tp_status_t tp_shard_get(tp_shards_t s, int i, int which, void *host_dst);

/* Shape of a handle: any pointer may be NULL.  kind: 0 = MLP, 1 = QKV. */
TP_API tp_status_t tp_shard_info(tp_shards_t s, int *kind, int64_t *H, int64_t *F, int *T,
                          int *act, int *dtype);

/* Free a handle and its device buffers (synchronises the device first). */
TP_API void tp_shards_destroy(tp_shards_t s);

/*
 * tp_mlp_workspace_bytes - device workspace tp_mlp_forward needs for M
 * tokens and variant v: Y (T x M x F/T, element type of the shards) plus,
 * for the partials variant and for decode, the float32 partials.
 */
TP_API size_t tp_mlp_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v);

/*
 * tp_mlp_forward - Z = sum_i act(X W1_i) W2_i for all T shards on this GPU.
 *   X  [M x H] device, element type of the shards (replicated input).
 *   Z  [M x H] float32 device, written in full (caller-owned).
 *   act must be the activation the shards were made for (GELU_ERF and
 *   IDENTITY are interchangeable for non-SwiGLU shards).
 *   workspace: device buffer of at least tp_mlp_workspace_bytes(s, M, v)
 *   bytes, or NULL to let the library allocate it stream-ordered
 *   (cudaMallocAsync/cudaFreeAsync on `stream`).
 *   Steps (bf16): column-parallel GEMM with the activation fused into its
 *   epilogue, Y_i stored as bfloat16; row-parallel GEMM; the all-reduce-sum
 *   (shard-sum kernel over float32 partials in ascending shard order, or the
 *   tensor-memory accumulator over all shards' K ranges).  M <= 16 uses the
 *   memory-bound decode kernels (weights as the 128-row MMA operand).
 *   M == 0 is a no-op.  Asynchronous on `stream`.
 */
TP_API tp_status_t tp_mlp_forward(tp_shards_t s, const void *X, int64_t M, tp_act_t act,
                           tp_variant_t v, float *Z, void *workspace, size_t ws_bytes,
                           void *stream);

/*
 * tp_colpar_forward - the column-parallel layer alone (step 1 of
 * tp_mlp_forward): Y_i = act(X W1_i) for every shard i ("Tensor Parallelism
 * in Action", section 1, "Column Parallel (W1)": no exchange after it).
 *   X  [M x H] device, element type of the shards.
 *   Y  [T x M x F/T] device out, element type of the shards: shard i's
 *      block Y_i is contiguous (the rank-local layout).
 *   workspace: tp_colpar_workspace_bytes(s, M) bytes (0 except for the
 *   decode shapes, M <= 16), or NULL to allocate stream-ordered.
 *   Asynchronous on `stream`.
 */
TP_API size_t tp_colpar_workspace_bytes(tp_shards_t s, int64_t M);
TP_API tp_status_t tp_colpar_forward(tp_shards_t s, const void *X, int64_t M, tp_act_t act,
                                     void *Y, void *workspace, size_t ws_bytes, void *stream);

/*
 * tp_rowpar_forward - the row-parallel layer and its all-reduce-sum (steps 2
 * and 3 of tp_mlp_forward): Z = sum_i Y_i W2_i ("Tensor Parallelism in
 * Action", section 1, "Row Parallel (W2)" and "Output Combination").
 *   Y  [T x M x F/T] device, as tp_colpar_forward writes it.
 *   Z  [M x H] float32 device out.
 *   workspace: tp_rowpar_workspace_bytes(s, M, v) bytes (the float32
 *   partials when the plan uses them), or NULL to allocate stream-ordered.
 *   Asynchronous on `stream`.
 */
TP_API size_t tp_rowpar_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v);
TP_API tp_status_t tp_rowpar_forward(tp_shards_t s, const void *Y, int64_t M, tp_variant_t v,
                                     float *Z, void *workspace, size_t ws_bytes, void *stream);

/*
 * tp_mlp_forward_noalloc - tp_mlp_forward (variant AUTO) that allocates no
 * memory at all.  The pages have no counterpart to this call: it exists for
 * callers that cannot allocate device memory while they run the MLP, such as
 * a decode loop captured into a CUDA graph or driven by a real-time
 * scheduler that forbids allocator calls (cudaMalloc can synchronise the
 * device and take unbounded time), or a host runtime that hands out all
 * device memory itself and has none to lend as workspace.
 *   Its scratch is a fixed 16 MiB device array inside the library, which
 *   every GPU that loads the library holds until the process exits.  The
 *   call runs the AUTO plan when its workspace (tp_mlp_workspace_bytes(s,
 *   M, TP_VAR_AUTO)) fits in 16 MiB; that size depends on the GPU's SM
 *   count, because the AUTO plan splits K to fill the SMs.  Where it does
 *   not fit, the call refits the plan to the scratch: no float32 partials of
 *   the second layer (all shards summed in one TMEM accumulator, as
 *   TP_VAR_TMEM_ACC) and, for decode, as many first-layer split-K slots as
 *   fit.  Only a call whose Y ([T x M x F/T]) and one set of first-layer
 *   partials alone exceed 16 MiB is rejected, with TP_ERR_WORKSPACE.  The
 *   memory-bound decode shapes (M <= 16 tokens) of an H = 8192, F = 28672,
 *   T = 8 MLP fit on any SM count.
 *   The first call on a device looks up the scratch's device address
 *   (cudaGetSymbolAddress) and keeps it for the life of the process; make
 *   that first call before any stream capture.  cudaDeviceReset() is not
 *   supported afterwards (the address, like the library's other per-device
 *   state, would be stale).
 *   `s` must have been made on the current device (else TP_ERR_ARG: making a
 *   handle creates the device state this call needs, so a handle from
 *   another device is the only way to reach it without that state), and
 *   X, Z are as for tp_mlp_forward.
 *   All calls share the one scratch array and it keeps the last call's
 *   contents; every byte a call reads from it is written earlier in the same
 *   call, so nothing needs clearing.  Calls that overlap on the GPU (on
 *   different streams, or from several threads without ordering) race on the
 *   scratch and give wrong results: order them on one stream.
 */
TP_API tp_status_t tp_mlp_forward_noalloc(tp_shards_t s, const void *X, int64_t M, tp_act_t act,
                                          float *Z, void *stream);

/* Device workspace tp_mlp_forward_host needs: X and Z staging plus
 * tp_mlp_workspace_bytes(). */
TP_API size_t tp_mlp_host_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v);

/*
 * tp_mlp_forward_host - the same computation from HOST buffers: copies
 * X_host ([M x H], element type of the shards) to the device, runs
 * tp_mlp_forward and copies Z back to Z_host ([M x H] float32), all on
 * `stream`.  Pinned host memory makes the copies asynchronous; the call
 * returns once the work is enqueued (synchronise `stream` before reading
 * Z_host).  workspace as above, sized by tp_mlp_host_workspace_bytes().
 */
TP_API tp_status_t tp_mlp_forward_host(tp_shards_t s, const void *X_host, int64_t M, tp_act_t act,
                                tp_variant_t v, float *Z_host, void *workspace,
                                size_t ws_bytes, void *stream);

/*
 * Training: the forward pass that keeps what the backward pass needs, and
 * the backward pass.  The pages say the tensor-parallel all-reduces run "on
 * every single layer forward/backward pass" ("Slice the matrix itself",
 * section "Strict NVLink Domain Constraint") and that each layer contract
 * fixes "which gradient path communicates" (the duoan.github.io post on
 * ColumnParallelLinear / RowParallelLinear).  With P = X W1 (the
 * pre-activation), Hh = act(P) and the upstream gradient dZ:
 *   dH_i = dZ W2_i^T, dP_i = dH_i * act'(P_i)   (per shard, no exchange)
 *   dW2_i = Hh_i^T dZ, dW1_i = X^T dP_i          (per shard, local)
 *   dX = sum_i dP_i W1_i^T                      (the backward all-reduce-sum)
 * bfloat16 shards only.
 *
 * tp_shards_enable_backward - give a handle the weights in the caller's
 *   layout (W1 [H x F] or [H x 2F], W2 [F x H], the same matrices that were
 *   sharded), which the backward GEMMs read K-major.  The handle keeps
 *   copies (device memory: one more set of weights).
 *
 * tp_mlp_forward_train - tp_mlp_forward that also keeps, for the backward
 *   pass, Hsave = act(X W1_i) as [T x M x F/T] bfloat16 (it is also the
 *   row-parallel layer's input) and Psave = the pre-activations: GeLU
 *   [T x M x F/T], SwiGLU [2 x T x M x F/T] (gate, then up); unused (may be
 *   NULL) for IDENTITY.  Always uses the tensor-core prefill tiles, any M.
 *   workspace: tp_mlp_train_workspace_bytes(s, M, v) bytes or NULL.
 *
 * tp_mlp_backward - from X [M x H], Hsave, Psave and dZ [M x H] (bfloat16,
 *   device), writes dX [M x H], dW1 [H x F] (SwiGLU [H x 2F] = [dWg | dWu])
 *   and dW2 [F x H], float32, in the caller's weight layout.  Requires
 *   tp_shards_enable_backward.  v chooses how dX's sum over shards is done
 *   (TMEM accumulation, or float32 partials + shard-sum).  workspace:
 *   tp_mlp_backward_workspace_bytes(s, M, v) bytes or NULL.  Asynchronous.
 */
TP_API tp_status_t tp_shards_enable_backward(tp_shards_t s, const void *W1, const void *W2,
                                             void *stream);
TP_API size_t tp_mlp_train_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v);
TP_API tp_status_t tp_mlp_forward_train(tp_shards_t s, const void *X, int64_t M, tp_act_t act,
                                        tp_variant_t v, float *Z, void *Hsave, void *Psave,
                                        void *workspace, size_t ws_bytes, void *stream);
TP_API size_t tp_mlp_backward_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v);
TP_API tp_status_t tp_mlp_backward(tp_shards_t s, const void *X, const void *Hsave,
                                   const void *Psave, const void *dZ, int64_t M, tp_variant_t v,
                                   float *dX, float *dW1, float *dW2, void *workspace,
                                   size_t ws_bytes, void *stream);

/* Device workspace tp_attn_proj_forward needs (float32 partials for the
 * partials variant; 0 for the accumulator variant). */
TP_API size_t tp_attn_proj_workspace_bytes(tp_shards_t s, int64_t M, tp_variant_t v);

/*
 * tp_attn_proj_forward - the head-sharded attention projections.
 *   X   [M x H] bfloat16 (replicated input).
 *   QKV [T x M x 3W] bfloat16 out: QKV_i = X Wqkv_i = [Q_i | K_i | V_i], each
 *       shard's block contiguous (rank-local layout).  May be NULL to skip.
 *   A   [M x H] bfloat16: the attention output, heads side by side (A_i =
 *       the W columns of shard i's heads).  May be NULL (with Z) to skip.
 *   Z   [M x H] float32 out: Z = sum_i A_i Wo_i (row-parallel + all-reduce).
 *   Asynchronous on `stream`.
 */
TP_API tp_status_t tp_attn_proj_forward(tp_shards_t s, const void *X, const void *A, int64_t M,
                                 tp_variant_t v, void *QKV, float *Z, void *workspace,
                                 size_t ws_bytes, void *stream);

/*
 * tp_block_forward - one tensor-parallel transformer block on this GPU:
 * head-sharded attention, then the MLP, each ending in its all-reduce-sum
 * ("Slice the matrix itself", section "All-Reduce Synchronization": two
 * all-reduces per layer, after the attention's and after the MLP's
 * row-parallel projection; "Tensor parallelism" guide, section "Walking
 * through a transformer block": heads sharded across ranks, the two
 * all-reduces on the attention and MLP residual paths).
 *   attn: a handle from tp_shard_weights_qkv with head_dim 128 (other head
 *         dims -> TP_ERR_UNSUPPORTED);
 *   mlp:  a bfloat16 handle from tp_shard_weights with the same H and T.
 *   X [M x H] bfloat16.  Per token r and head h (heads in shard order):
 *     o_h = sum_{j <= r} softmax_j(q_h . k_jh / sqrt(head_dim)) v_jh
 *     (causal != 0; all keys j < M when causal == 0),
 *     h = X + sum_i O_i Wo_i, out = h + sum_i act(h W1_i) W2_i.
 *   No normalisation layers (the pages name none).  Q, K, V, the
 *   probabilities, O and the MLP input h are rounded to bfloat16 on the way;
 *   scores, sums and outputs are float32.  The attention core is the one of
 *   tp_attention_forward (scores never reach memory).
 *   out [M x H] float32; h_out [M x H] float32 or NULL: the residual stream
 *   after the attention all-reduce.  workspace: tp_block_workspace_bytes()
 *   bytes or NULL.  Asynchronous.
 */
TP_API size_t tp_block_workspace_bytes(tp_shards_t attn, tp_shards_t mlp, int64_t M, tp_variant_t v);
TP_API tp_status_t tp_block_forward(tp_shards_t attn, tp_shards_t mlp, const void *X, int64_t M,
                                    int causal, tp_variant_t v, float *out, float *h_out,
                                    void *workspace, size_t ws_bytes, void *stream);

/*
 * tp_attention_forward - the attention core of the block for a set of heads
 * ("Tensor parallelism" guide, section "Walking through a transformer
 * block": heads are sharded across ranks, so each head's attention runs
 * where its shard lives, with no communication).  For every head h and
 * token r < M:
 *   O[r][h hd + d] = sum_j softmax_j(q_rh . k_jh / sqrt(hd)) v_jh[d]
 * over keys j <= r (causal != 0) or all j < M (causal == 0); scores and
 * probabilities stay on chip (one fused kernel per call).  The probabilities
 * are rounded to bfloat16 for the P V product and the sums are float32.
 *   Q, K, V: bfloat16, head-major [n_heads][M][head_dim], device, 16-byte
 *            aligned (the layout tp_block_forward's QKV projection writes).
 *   head_dim must be 128 (else TP_ERR_UNSUPPORTED).
 *   O: bfloat16 [M][ldo] out, head h in columns [h hd, (h+1) hd);
 *      ldo >= n_heads hd and a multiple of 8; 16-byte aligned; must not
 *      overlap Q, K or V (TP_ERR_ARG).
 *   workspace, ws_bytes: unused (the call needs no scratch);
 *      tp_attention_workspace_bytes returns 0.
 *   M == 0 is a no-op.  Asynchronous on `stream`.
 */
TP_API size_t tp_attention_workspace_bytes(int64_t M, int n_heads, int head_dim);
TP_API tp_status_t tp_attention_forward(const void *Q, const void *K, const void *V, int64_t M,
                                        int n_heads, int head_dim, int causal, void *O, int64_t ldo,
                                        void *workspace, size_t ws_bytes, void *stream);

/*
 * tp_partial_sum - the all-reduce-sum arithmetic on one GPU ("Slice the
 * matrix itself", section "Mathematical formulation": Y = sum_i X_i W_i, then
 * All-Reduce-Sum).
 *   Zi  host array of T device pointers, each to n float32 values.
 *   Z   n float32 out: Z[k] = ((Zi[0][k] + Zi[1][k]) + ...) + Zi[T-1][k],
 *       float32, shards in ascending order (deterministic, no atomics).
 *       Z may be Zi[0] (in place); any other overlap is an error.
 *   n == 0 is a no-op.  Asynchronous on `stream`.
 */
TP_API tp_status_t tp_partial_sum(const float *const *Zi, int T, int64_t n, float *Z, void *stream);

/*
 * The other collectives of tensor parallelism, on one GPU ("Tensor
 * Parallelism in Action", section 2, question 3: AllReduce, AllGather,
 * ReduceScatter; the ring all-reduce's 2 (T - 1) / T * H * B bytes in the
 * "Tensor parallelism" guide, section "Walking through a transformer block",
 * are its reduce-scatter half plus its all-gather half).
 *
 * tp_reduce_scatter - rank i keeps block i of the sum: with nb = n / T,
 *   out[i][k] = ((Zi[0][i nb + k] + Zi[1][i nb + k]) + ...) + Zi[T-1][i nb + k],
 *   float32, ranks in ascending order.  Zi: T device pointers to n floats;
 *   out: T device pointers to nb floats each, overlapping neither each other
 *   nor any Zi.  n % T != 0 -> TP_ERR_INDIVISIBLE.  Asynchronous on `stream`.
 *
 * tp_all_gather - out = parts[0] | parts[1] | ... | parts[T-1], each part
 *   n_per elements of elem_bytes bytes, in rank order.  A part that already
 *   sits at its place in `out` (the in-place form) is left as it is; any
 *   other overlap -> TP_ERR_ARG.  Asynchronous on `stream`.
 *
 * tp_partial_sum_bf16 - the all-reduce-sum of tp_partial_sum, rounded once
 *   to bfloat16 (nearest, ties to even): Z is n bfloat16 values and must not
 *   overlap the inputs.  Asynchronous on `stream`.
 */
TP_API tp_status_t tp_reduce_scatter(const float *const *Zi, int T, int64_t n, float *const *out,
                                     void *stream);
TP_API tp_status_t tp_all_gather(const void *const *parts, int T, int64_t n_per, int elem_bytes,
                                 void *out, void *stream);
TP_API tp_status_t tp_partial_sum_bf16(const float *const *Zi, int T, int64_t n, void *Z, void *stream);

/*
 * tp_last_device_status - synchronise `stream`, then return and clear the
 * current device's status word: TP_OK, TP_ERR_TIMEOUT (a kernel's bounded
 * wait ran out and it returned early; its outputs are undefined) or
 * TP_ERR_DEVICE_CHECK.  The word collects every kernel of this library on
 * the device since the last call.  A CUDA error from the stream is returned
 * as TP_ERR_CUDA.
 */
TP_API tp_status_t tp_last_device_status(void *stream);

/*
 * tp_set_machine_balance - the exchange rate, in dense bf16 tensor-core flop
 * per byte of HBM traffic, that the AUTO planners (tp_mlp_forward,
 * tp_attn_proj_forward, tp_block_forward and their workspace queries) use to
 * weigh the row-parallel GEMM's work against the float32 partials that
 * variant A writes and the shard-sum reads (the pages' "partial sums"
 * completed by the all-reduce, "Slice the matrix itself", section
 * "Mathematical formulation").  The default comes from the device's own
 * figures: 8192 flop per SM per clock at the peak SM clock, against two
 * transfers of the memory bus width per memory clock.  A caller that has
 * measured both rates passes their ratio; 0 restores the default.  Negative,
 * NaN or absurd values (> 1e6) -> TP_ERR_ARG.  Process-wide; affects plans
 * made after the call (workspace sizes included).
 */
TP_API tp_status_t tp_set_machine_balance(double flop_per_byte);

/*
 * tp_set_rowpar_schedule - how the row-parallel GEMM with one TMEM accumulator
 * over all shards (the all-reduce-sum inside the accumulator, "Slice the
 * matrix itself", section "Mathematical formulation") lays its output tiles
 * over the GPU's CTA pairs.  1 (default): where it pays, each 256-row block of
 * the output is cut into tiles of 288..480 columns (near-equal widths, two
 * MMAs per k-step into two accumulators) run in one or two rounds of the
 * pairs, instead of 256-column tiles in more rounds (at M = 2048, H = 4096 on
 * a 152-SM GB300: one round of 480- and 448-column tiles against two rounds
 * of 256; at M = 4096, two rounds against four).  Applies to the MLP's
 * second layer, the training backward's dX, the attention output
 * projection and the block's row-parallel layers; a tile's epilogue is
 * exposed once per round, so a layer that also adds a residual takes the
 * wide tiles only where its K is long enough (in the block at M = 4096: the
 * MLP's down-projection, not the output projection).  0: always 256-column
 * tiles.  Both sum every output element over the same K order in one
 * accumulator, so they give identical results.  Other values -> TP_ERR_ARG.
 * Process-wide; affects calls made after it (workspace sizes do not depend on
 * it).
 */
TP_API tp_status_t tp_set_rowpar_schedule(int wide);

/*
 * tp_rowpar_tiles - the tiles tp_mlp_forward's row-parallel GEMM would use
 * for M tokens with variant v on the current device and schedule (see
 * tp_set_rowpar_schedule).  out[3] (host memory): the widest tile's columns,
 * the number of such tiles per 256-row block, and the tiles per block (the
 * others 32 columns narrower), or three zeros where the call takes any other
 * form (256-column tiles, float32 partials, the decode or CUDA-core path).
 * A query only: nothing is launched.  NULL or foreign handle, M <= 0 or a bad
 * variant -> TP_ERR_ARG.
 */
TP_API tp_status_t tp_rowpar_tiles(tp_shards_t s, int64_t M, tp_variant_t v, int32_t *out);

/*
 * tp_set_wait_limit_ns - limit on every device-side wait (default 2 s) in
 * kernels launched after this call, process-wide.  0 restores the default.
 * A limit below 1 ms is a test limit: the tensor-core kernels then first
 * wait on a barrier that nothing ever completes, so their waits run out on
 * purpose and the timeout path (abort, let issued copies and MMAs finish,
 * release tensor memory, return) is exercised; the call's results are
 * undefined and tp_last_device_status() reports TP_ERR_TIMEOUT.  Nothing
 * faults or hangs.
 */
TP_API tp_status_t tp_set_wait_limit_ns(uint64_t ns);

/*
 * tp_inject_alloc_failures - failure injection for tests (the pages have no
 * counterpart): the next `count` device allocations this library makes
 * (workspaces it allocates itself, shard buffers, scratch of tp_shard_get)
 * fail as if the device were out of memory.  The calls that needed them
 * return TP_ERR_OOM and leave nothing allocated behind; later calls work
 * again.  0 cancels pending failures; count < 0 -> TP_ERR_ARG.  Process-wide;
 * no CUDA call is made.
 */
TP_API tp_status_t tp_inject_alloc_failures(int count);

#ifdef __cplusplus
}
#endif

#endif /* TP_MLP_H */
