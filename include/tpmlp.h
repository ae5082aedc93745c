/*
 * tpmlp.h -- C ABI of libtpmlp, the GB300 (sm_103a) tensor-parallel linear block.
 *
 * The method (Megatron-style tensor parallelism):
 *   column-parallel linear   Y_i = X W_i, W split by column, X replicated
 *                            [张量并行 notes (cloudchewie), §并行化矩阵乘法运算, 列并行;
 *                             Infra: Tensor Parallel (pufanyi), Column-wise TP]
 *   per-shard activation     H_i = GELU(Y_i) or A_i = SiLU(X Wg_i) * (X Wu_i), no communication
 *                            [张量并行 notes, §MLP 层的并行化; 20260402-parallelism, §1 TP]
 *   row-parallel linear      Z_i = H_i W2_i, W split by row
 *                            [张量并行 notes, §并行化矩阵乘法运算, 行并行; Infra: Tensor Parallel, Row-wise TP]
 *   shard sum                Z = sum_i Z_i  (the all-reduce; here an on-device reduction)
 *   backward                 dW_i = X^T dY_i, dX = sum_i dY_i W_i^T (column shards);
 *                            dW_i = X_i^T dY, dX_i = dY W_i^T (row shards)
 *                            [Infra: Tensor Parallel, Column-wise / Row-wise TP backward]
 * All N shards run as virtual ranks on ONE GPU: shard i's work is a contiguous
 * slab of one kernel's tile space, and the sum over shards is done on the device
 * either by a separate reduction of per-shard fp32 partials (TP_REDUCE_BUFFERS)
 * or by folding every shard's K-slice into one on-chip accumulator in shard
 * order (TP_REDUCE_SPLITK).
 *
 * Conventions for every entry point
 *   - Tensors are dense and row-major. X is (M, h) with M = b*s tokens (the pages'
 *     X:(b, s, h)); a weight W is (h, h') = (in, out) so that Y = X W (the pages'
 *     W:(h, h')) [张量并行 notes, §基本思想]. The linear entry points also take
 *     (out, in) weights (tp_wlayout).
 *   - Column shard i of a weight = columns [i*h'/N, (i+1)*h'/N); row shard i = rows
 *     [i*h/N, (i+1)*h/N). Shards are blocks of one allocation, in shard order.
 *   - Element types: TP_BF16 (bf16 storage, fp32 accumulation, tensor cores) or
 *     TP_F32 (fp32 storage and arithmetic on CUDA cores, no TF32).
 *   - Pointers named as device buffers must be device memory (or managed memory);
 *     the caller owns every buffer. The library never allocates device memory:
 *     scratch comes from the caller's workspace `ws` (size from tp_workspace_size).
 *     All device buffers must be 16-byte aligned.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream). Argument errors are returned before anything is launched, and then
 *     no output has been written.
 *   - bf16 shape rules: h, h'/N and every output width are multiples of 64; M >= 0 is
 *     arbitrary (M = 0 returns TP_OK and launches nothing). fp32: any positive sizes
 *     with h' divisible by N.
 *   - A device wait that exceeds its time limit (tp_set_wait_timeout_ns) makes the
 *     kernel stop and record TP_ERR_TIMEOUT in a per-device status word, read (and
 *     cleared) by tp_check_status. Kernels never trap.
 *   - Thread safety: calls may come from several host threads; tp_last_error is
 *     per thread.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TP_API __attribute__((visibility("default")))
#else
#define TP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define TPMLP_VERSION 2

typedef enum tp_status {
  TP_OK = 0,
  TP_ERR_INVALID_ARG = 1, /* null pointer, non-positive N, negative size, unknown enum   */
  TP_ERR_SHAPE = 2,       /* divisibility or tile rule broken (h' % N, heads % N, ...)   */
  TP_ERR_DTYPE = 3,       /* element type not supported by this call                    */
  TP_ERR_ALIGNMENT = 4,   /* a device buffer is not 16-byte aligned                     */
  TP_ERR_WORKSPACE = 5,   /* workspace missing or smaller than tp_workspace_size        */
  TP_ERR_CUDA = 6,        /* a CUDA call failed; tp_last_error() has the detail          */
  TP_ERR_TIMEOUT = 7,     /* a bounded device wait expired (reported by tp_check_status) */
  TP_ERR_UNSUPPORTED = 8  /* no sm_103 device, or a feature not built                    */
} tp_status;

typedef enum tp_dtype { TP_F32 = 0, TP_BF16 = 1 } tp_dtype;

typedef enum tp_act {
  TP_ACT_NONE = 0,   /* plain linear                                                      */
  TP_ACT_GELU = 1,   /* exact erf GELU: x * 1/2 [1 + erf(x / sqrt 2)]
                        [张量并行 notes, §MLP 层的并行化, GELU formula]                        */
  TP_ACT_SWIGLU = 2  /* SiLU(X Wg) * (X Wu); the pages name W_gate/W_up
                        [20260402-parallelism, §1 TP]; SiLU(x) = x / (1 + e^-x)            */
} tp_act;

typedef enum tp_reduce {
  TP_REDUCE_BUFFERS = 0, /* each shard writes fp32 partials P[i] (M x n) to the workspace;
                            a coalesced HBM kernel sums them in shard order 0..N-1        */
  TP_REDUCE_SPLITK = 1   /* the K-slices of all shards are folded into one on-chip fp32
                            accumulator, shard 0 first; no partial buffers               */
} tp_reduce;

/*
 * Storage order of the weights of the linear entry points (tp_col_linear, tp_row_linear,
 * tp_mlp_fwd, tp_mlp_bwd). The pages write Y = X W with W:(h, h') [张量并行 notes,
 * §基本思想; Infra: Tensor Parallel]; the Megatron listing keeps each shard's weight as
 * (out, in) for F.linear, Y = X W^T [Megatron-LM 分布式大模型训练实战 04, 核心实现,
 * ColumnParallelLinear / RowParallelLinear].
 *   TP_W_IN_OUT: a weight is stored (in, out) row-major, the pages' W itself. A column
 *                shard is a column block of the stored matrix, a row shard a row block.
 *   TP_W_OUT_IN: a weight is stored (out, in) row-major, i.e. W^T. A column shard
 *                (out features [i out/N, (i+1) out/N)) is then a ROW block of the stored
 *                matrix, and a row shard (in features [i in/N, (i+1) in/N)) a COLUMN
 *                block; weight gradients are written in the same (out, in) order.
 * Either way the tensor cores read the stored matrix in place (K-major or MN-major
 * operand), with no transpose copy.
 */
typedef enum tp_wlayout { TP_W_IN_OUT = 0, TP_W_OUT_IN = 1 } tp_wlayout;

typedef enum tp_op {
  TP_OP_COL_LINEAR = 0,
  TP_OP_ROW_LINEAR = 1,
  TP_OP_MLP_FWD = 2,
  TP_OP_MLP_BWD = 3,
  TP_OP_ATTN_PROJ_FWD = 4,
  TP_OP_ATTN_PROJ_BWD = 5,
  TP_OP_LAYERNORM_BWD = 6,
  TP_OP_LAYER_FWD = 7,
  TP_OP_LAYER_BWD = 8,
  TP_OP_SP_MLP_FWD = 9,
  TP_OP_SP_MLP_BWD = 10
} tp_op;

/* Weights of the pre-LN transformer layer (tp_layer_fwd / tp_layer_bwd). */
typedef struct tp_layer_weights {
  const void* Wqkv;     /* (h, 3h) = [W_q | W_k | W_v], head t at columns t*d of each block */
  const void* Wo;       /* (h, h), row block i = shard i's heads                            */
  const void* W1;       /* (h, f), column-split                                              */
  const void* W2;       /* (f, h), row-split                                                 */
  const float* gamma1;  /* (h) LN1 scale and shift, fp32                                     */
  const float* beta1;
  const float* gamma2;  /* (h) LN2                                                           */
  const float* beta2;
} tp_layer_weights;

/* State the layer's forward saves for its backward (all written by tp_layer_fwd). */
typedef struct tp_layer_saved {
  void* xn1;     /* (M, h) LN1(x)                       */
  float* mean1;  /* (M) LN1 row mean, fp32              */
  float* rstd1;  /* (M) LN1 row 1/sqrt(var + eps)       */
  void* qkv;     /* (M, 3h)                             */
  void* o;       /* (M, h) attention output, heads concatenated */
  float* lse;    /* (b, n_heads, s) softmax log-sum-exp */
  void* x1;      /* (M, h) x + attention block          */
  void* xn2;     /* (M, h) LN2(x1)                      */
  float* mean2;
  float* rstd2;
  void* y;       /* (M, f) MLP pre-activation           */
  void* hh;      /* (M, f) GELU(y)                      */
} tp_layer_saved;

/* Parameter gradients written by tp_layer_bwd. */
typedef struct tp_layer_grads {
  void* dWqkv;  /* (h, 3h) */
  void* dWo;    /* (h, h)  */
  void* dW1;    /* (h, f)  */
  void* dW2;    /* (f, h)  */
  float* dgamma1;
  float* dbeta1;
  float* dgamma2;
  float* dbeta2;
} tp_layer_grads;

/* The small tensor-parallel GPT: embedding (vocabulary-parallel, shared with the output
 * layer), `layers` pre-LN layers, final LayerNorm, output layer, cross-entropy. */
typedef struct tp_gpt_config {
  int64_t vocab;   /* v, divisible by N */
  int64_t hidden;  /* h */
  int64_t heads;   /* attention heads (head_dim = h / heads in {16, 32, 64}) */
  int64_t ffn;     /* f */
  int64_t layers;
  int64_t batch;   /* b */
  int64_t seq;     /* s; token rows M = b*s, the s rows of one sequence consecutive */
  int32_t shards;  /* N */
} tp_gpt_config;

typedef struct tp_gpt_weights {
  const void* E;                   /* (vocab, h): embedding, and the output layer's weight */
  const float* gammaf;             /* (h) final LayerNorm */
  const float* betaf;
  const tp_layer_weights* layers;  /* `layers` entries */
} tp_gpt_weights;

typedef struct tp_gpt_grads {
  void* dE;                        /* (vocab, h): output layer's gradient + embedding's */
  float* dgammaf;
  float* dbetaf;
  const tp_layer_grads* layers;    /* `layers` entries */
} tp_gpt_grads;

/* ------------------------------------------------------------------ utilities */

/* Library version (TPMLP_VERSION). */
TP_API int tp_version(void);

/* Static string naming a status code; never NULL. */
TP_API const char* tp_status_string(tp_status s);

/* Detail of the last failing call made by this host thread ("" if none). */
TP_API const char* tp_last_error(void);

/* Synchronise `stream`, then read and clear the current device's sticky status
 * word. Returns TP_ERR_TIMEOUT if any kernel since the last check stopped on an
 * expired wait, TP_ERR_CUDA if the synchronisation failed, else TP_OK. */
TP_API tp_status tp_check_status(void* stream);

/* Time limit of every bounded device wait, in nanoseconds (default 4e9). Applies
 * to launches made after the call, from any thread. 0 restores the default. */
TP_API void tp_set_wait_timeout_ns(uint64_t ns);

/* Large GEMM tiles (M >= 256 rows, 256 columns) run on CTA pairs (two SMs sharing one
 * 256 x 256 tile through tcgen05 pair MMAs) when enabled (default 1), except on
 * problems so small that narrower one-CTA tiles spread them over more SMs; 0 restricts
 * every GEMM to the one-CTA kernel; 2 runs the pair kernel for every GEMM it can take,
 * small ones included (to test it on small shapes). Any other value is treated as 1.
 * Results agree within rounding in every mode; this switch exists to compare the
 * kernels. Applies to launches made after it. */
TP_API void tp_set_gemm_pair_mode(int enable);

/* Width of the CTA-pair tiles: 1 (default) uses 256 x 512 tiles -- two pair MMAs per
 * K step into one 128 x 512 accumulator per CTA, 3/4 of the operand bytes per FLOP of
 * 256 x 256 -- where the output width is whole 512-column tiles (256 for the paired
 * gate/up form), K is long beside the bytes the epilogue writes, and there are at
 * least four tiles per SM pair or the wide tiles need enough fewer waves of the SM
 * pairs; 0 keeps 256 x 256 tiles; 2 takes the wide tiles for every pair-kernel GEMM
 * (to test that form on small shapes). Results agree within rounding in every mode.
 * Applies to launches made after the call; any other value is treated as 1. */
TP_API void tp_set_gemm_wide_mode(int mode);

/* Number of kernel launches this library has made in this process (all threads). */
TP_API uint64_t tp_launch_count(void);

/* Bytes of workspace `op` needs for these sizes (0 if none). For TP_OP_ROW_LINEAR,
 * h is the reduced width k and f the output width n. For the attention and
 * LayerNorm ops, M = b*s and h the hidden width (f is ignored). For the layer ops,
 * f is the MLP width. Returns 0 on invalid arguments. */
TP_API size_t tp_workspace_size(tp_op op, int64_t M, int64_t h, int64_t f, int32_t N,
                         tp_dtype dtype, tp_act act, tp_reduce mode);

/*
 * Plain GEMM on the library's engine (tensor cores for bf16, CUDA cores for fp32):
 *   C (M, N) = A B, fp32 accumulation, C row-major with element type `dtype`.
 *   A is (M, K) row-major, or -- when a_trans != 0 -- stored as its transpose (K, M);
 *   B is (K, N) row-major, or -- when b_trans != 0 -- stored as its transpose (N, K).
 * This is the building block of every layer below (the transposed forms are how the
 * backward reads X^T, H^T and W^T in place, with no transpose copies).
 * bf16 rule: the stored row widths (K or M for A, N or K for B) and N are multiples of 8.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_SHAPE, TP_ERR_ALIGNMENT, TP_ERR_CUDA.
 */
TP_API tp_status tp_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         int a_trans, int b_trans, tp_dtype dtype, void* stream);

/* ------------------------------------------------------------------ layers */

/*
 * Column-parallel linear with the per-shard activation fused into its epilogue.
 * [张量并行 notes, §并行化矩阵乘法运算, 列并行; Infra: Tensor Parallel, Column-wise TP]
 *
 *   X    (M, h)  device, read        replicated input (every shard reads all of it)
 *   W    (h, f)  device, read        column shard i = columns [i f/N, (i+1) f/N)
 *   W_up (h, f)  device, read        SwiGLU only (the up projection), else NULL
 *   Y    (M, f)  device, written     pre-activation X W (gate for SwiGLU); NULL = not kept
 *   Y_up (M, f)  device, written     SwiGLU only: X W_up; NULL = not kept
 *   out  (M, f)  device, written     act(Y): Y itself (NONE), GELU(Y), or SiLU(Y) * Y_up;
 *                                    shard i's output is column block i (the all-gather
 *                                    is this layout, no copy)
 *   w_layout                         TP_W_IN_OUT: W, W_up as above; TP_W_OUT_IN: W, W_up
 *                                    stored (f, h), shard i = row block i (the
 *                                    Megatron listing's ColumnParallelLinear weight)
 * Errors: TP_ERR_INVALID_ARG (null X/W/out, N < 1, SwiGLU without W_up, unknown
 *         w_layout), TP_ERR_SHAPE (f % N, bf16 tile rules), TP_ERR_ALIGNMENT, TP_ERR_CUDA.
 */
TP_API tp_status tp_col_linear(const void* X, const void* W, const void* W_up,
                        void* Y, void* Y_up, void* out,
                        int64_t M, int64_t h, int64_t f, int32_t N,
                        tp_dtype dtype, tp_act act, tp_wlayout w_layout, void* stream);

/*
 * Row-parallel linear followed by the shard sum (the all-reduce stand-in).
 * [张量并行 notes, §并行化矩阵乘法运算, 行并行; Infra: Tensor Parallel, Row-wise TP]
 *
 *   Xs       (M, k) device, read     column block i = shard i's input X_i
 *   W        (k, n) device, read     row block i = W_i
 *   residual (M, n) device, read     added after the sum; NULL = none
 *   out      (M, n) device, written  sum_i X_i W_i (+ residual), element type `dtype`
 *   ws, ws_bytes                     TP_REDUCE_BUFFERS needs N*M*n*4 bytes
 *                                    (tp_workspace_size(TP_OP_ROW_LINEAR, M, k, n, ...))
 *   w_layout                         TP_W_IN_OUT: W as above; TP_W_OUT_IN: W stored
 *                                    (n, k), W_i = column block i (the Megatron
 *                                    listing's RowParallelLinear weight)
 * Errors: as tp_col_linear, plus TP_ERR_WORKSPACE.
 */
TP_API tp_status tp_row_linear(const void* Xs, const void* W, const void* residual, void* out,
                        int64_t M, int64_t k, int64_t n, int32_t N,
                        tp_dtype dtype, tp_reduce mode, void* ws, size_t ws_bytes,
                        tp_wlayout w_layout, void* stream);

/*
 * The shard sum on its own: out = sum_{i=0}^{N-1} partials[i] (+ residual), in
 * that order, fp32 arithmetic. [张量并行 notes, §MLP 层的并行化, g forward: all-reduce
 * adds Z_1 and Z_2 into Z]
 *
 *   partials (N, M, n) fp32 device, read
 *   residual (M, n) device, element type out_dtype, read; NULL = none
 *   out      (M, n) device, written, element type out_dtype
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_ALIGNMENT, TP_ERR_CUDA. Any n >= 1.
 */
TP_API tp_status tp_shard_reduce(const float* partials, const void* residual, void* out,
                          int32_t N, int64_t M, int64_t n, tp_dtype out_dtype,
                          void* stream);

/*
 * The shard sum followed by LayerNorm, fused into one pass over the partials:
 *   x = sum_{i=0}^{N-1} partials[i] (+ residual), shards in that order in fp32, rounded
 *       to dtype and written to sum_out (the residual stream after the all-reduce);
 *   y = gamma * (x - mean) * rstd + beta over the full width h of the ROUNDED x,
 *       biased variance, rstd = 1 / sqrt(var + eps).
 * The all-reduce has to finish before LayerNorm because its statistics need the
 * whole hidden width [张量并行 notes, §相关分析, the forward bottleneck before LN];
 * here the sum is normalised while it is still on chip.
 *
 *   partials (N, M, h) fp32 read;  residual (M, h) dtype read or NULL
 *   gamma, beta (h) fp32 read;  sum_out (M, h) dtype written or NULL
 *   y (M, h) dtype written;  mean, rstd (M) fp32 written or NULL
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_DTYPE, TP_ERR_SHAPE (h % 8, h > 16384),
 * TP_ERR_ALIGNMENT (every buffer 16-byte aligned), TP_ERR_CUDA.
 */
TP_API tp_status tp_shard_reduce_ln(const float* partials, const void* residual,
                                    const float* gamma, const float* beta, void* sum_out,
                                    void* y, float* mean, float* rstd, int32_t N, int64_t M,
                                    int64_t h, float eps, tp_dtype dtype, void* stream);

/*
 * Row-parallel linear whose shard sum feeds LayerNorm:
 *   sum_out = sum_i Xs_i W_i (+ residual),  y = LN(sum_out; gamma, beta, eps)
 * with the operands, shard split and modes of tp_row_linear and the LN of
 * tp_shard_reduce_ln. TP_REDUCE_BUFFERS writes fp32 partials and normalises them in
 * the fused reduction; TP_REDUCE_SPLITK folds the sum in the GEMM and then runs LN.
 *   sum_out (M, n) written (required);  y (M, n) written;  mean, rstd (M) or NULL
 *   ws: tp_workspace_size(TP_OP_ROW_LINEAR, M, k, n, N, dtype, TP_ACT_NONE, mode).
 * Errors: as tp_row_linear, plus TP_ERR_SHAPE for n % 8 or n > 16384.
 */
TP_API tp_status tp_row_linear_ln(const void* Xs, const void* W, const void* residual,
                                  const float* gamma, const float* beta, void* sum_out, void* y,
                                  float* mean, float* rstd, int64_t M, int64_t k, int64_t n,
                                  int32_t N, float eps, tp_dtype dtype, tp_reduce mode, void* ws,
                                  size_t ws_bytes, void* stream);

/*
 * Tensor-parallel MLP forward: Z = sum_i act(X W1_i) W2_i (+ residual).
 * [张量并行 notes, §MLP 层的并行化, column-then-row formula; Infra: Tensor Parallel, MLP;
 *  20260402-parallelism, §1 TP (W_gate/W_up by column, second layer by row)]
 *
 *   X     (M, h) read;  W1 (h, f) read;  W1_up (h, f) read (SwiGLU only, else NULL)
 *   W2    (f, h) read;  residual (M, h) read or NULL
 *   Y     (M, f) written: GELU -> X W1; SwiGLU -> gate X W1. NULL = not kept.
 *   Y_up  (M, f) written: SwiGLU -> up X W1_up. NULL = not kept.
 *   H     (M, f) written: GELU(Y) or SiLU(Y) * Y_up, the row-parallel input.
 *                NULL = kept in the workspace instead.
 *   Z     (M, h) written.
 *   act   TP_ACT_GELU or TP_ACT_SWIGLU.  mode: the shard sum variant.
 *   w_layout  TP_W_IN_OUT as above; TP_W_OUT_IN: W1, W1_up stored (f, h) and W2 stored
 *             (h, f), the Megatron listing's (out, in) weights.
 * For bf16 and M <= 64 (decode) a weight-streaming kernel family is used.
 * Errors: as tp_row_linear.
 */
TP_API tp_status tp_mlp_fwd(const void* X, const void* W1, const void* W1_up, const void* W2,
                     const void* residual, void* Y, void* Y_up, void* H, void* Z,
                     int64_t M, int64_t h, int64_t f, int32_t N,
                     tp_dtype dtype, tp_act act, tp_reduce mode,
                     void* ws, size_t ws_bytes, tp_wlayout w_layout, void* stream);

/*
 * Tensor-parallel MLP backward. g-backward is the identity (every shard reads all
 * of dZ) and f-backward is the shard sum of dX [张量并行 notes, §MLP 层的并行化,
 * g/f backward]; per shard [Infra: Tensor Parallel, Column-wise / Row-wise TP]:
 *   GELU:   dY_i = (dZ W2_i^T) * GELU'(Y_i), dW2_i = H_i^T dZ, dW1_i = X^T dY_i,
 *           dX = sum_i dY_i W1_i^T
 *   SwiGLU: dA_i = dZ W2_i^T; dG_i = dA_i * U_i * s (1 + G_i (1 - s)), s = sigmoid(G_i);
 *           dU_i = dA_i * SiLU(G_i); dW2_i = A_i^T dZ; dW1_i = X^T dG_i;
 *           dW1up_i = X^T dU_i; dX = sum_i (dG_i W1_i^T + dU_i W1up_i^T)
 *
 *   X, W1, W1_up, W2       as in tp_mlp_fwd (read)
 *   Y, Y_up, H             the forward's saved Y (gate), Y_up (up, SwiGLU) and H (read)
 *   dZ    (M, h) read
 *   dX    (M, h) written;  dW1 (h, f), dW1_up (h, f, SwiGLU), dW2 (f, h) written
 *   ws    dY (or dG and dU) plus, for TP_REDUCE_BUFFERS, N*M*h fp32 partials
 *   w_layout  as tp_mlp_fwd; with TP_W_OUT_IN the gradients are written (out, in)
 *             like their weights: dW1, dW1_up (f, h) = dY^T X, dU^T X and dW2 (h, f) =
 *             dZ^T H.
 * With TP_REDUCE_BUFFERS the dX GEMM runs before the weight-gradient GEMMs and the
 * shard sum of its partials runs on a side stream beside them (they do not read dX);
 * the call is still one ordered unit on `stream`.
 * Errors: as tp_row_linear.
 */
TP_API tp_status tp_mlp_bwd(const void* X, const void* W1, const void* W1_up, const void* W2,
                     const void* Y, const void* Y_up, const void* H, const void* dZ,
                     void* dX, void* dW1, void* dW1_up, void* dW2,
                     int64_t M, int64_t h, int64_t f, int32_t N,
                     tp_dtype dtype, tp_act act, tp_reduce mode,
                     void* ws, size_t ws_bytes, tp_wlayout w_layout, void* stream);

/*
 * Row-parallel linear + shard sum with per-shard partial buffers, allocating
 * nothing. (The pages have no counterpart: this is a deployment variant.)
 *
 * Same computation, arguments and errors as tp_row_linear with
 * mode = TP_REDUCE_BUFFERS, but the N*M*n fp32 partials live in a fixed 32 MiB
 * device array inside the library instead of a caller workspace. For callers that
 * cannot allocate device memory -- e.g. code running in a host process whose
 * device memory is owned by that process's own pool allocator, or under a fixed
 * memory budget -- and so can neither call cudaMalloc nor supply a workspace.
 * No cudaMalloc, cudaFree or allocating library routine is called.
 *   - Sizes with N*M*n*4 > 32 MiB are rejected with TP_ERR_WORKSPACE (nothing launched).
 *   - Every device that loads the library holds the 32 MiB until the process exits.
 *   - The first call on each device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream capture.
 *     The cached address does not survive cudaDeviceReset (the reset discards the
 *     array, which may come back elsewhere): do not call this entry point on a
 *     device after resetting it in the same process.
 *   - All calls share the one array: calls that overlap on the GPU (e.g. on two
 *     streams at once) race. Nothing in it needs to start at zero: every partial
 *     that is read is written first by the same call.
 */
TP_API tp_status tp_row_linear_noalloc(const void* Xs, const void* W, const void* residual,
                                       void* out, int64_t M, int64_t k, int64_t n, int32_t N,
                                       tp_dtype dtype, void* stream);

/* ------------------------------------------------------------------ attention block */

/*
 * LayerNorm over the full hidden width: y = gamma * (x - mu) / sqrt(var + eps) + beta,
 * biased variance. [张量并行 notes, §相关分析: LN needs the complete activation, so
 * it runs replicated after the shard sum]
 *   x (M, h) read; gamma, beta (h) fp32 read; y (M, h) written;
 *   mean, rstd (M) fp32 written (NULL = not kept). eps: the pages leave it open; the
 *   layer entry points use 1e-5.
 */
TP_API tp_status tp_layernorm_fwd(const void* x, const float* gamma, const float* beta, void* y,
                                  float* mean, float* rstd, int64_t M, int64_t h, float eps,
                                  tp_dtype dtype, void* stream);

/*
 * LayerNorm backward with an optional residual gradient added:
 *   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat)),  g = dy * gamma
 *   dgamma = sum_rows dy * xhat, dbeta = sum_rows dy (fp32, deterministic order; the
 *   rows are replicated on every rank, so they need no all-reduce [张量并行 notes, §相关分析])
 * dres may be NULL; dgamma/dbeta may be NULL (then no workspace is needed).
 */
TP_API tp_status tp_layernorm_bwd(const void* x, const float* gamma, const float* mean,
                                  const float* rstd, const void* dy, const void* dres, void* dx,
                                  float* dgamma, float* dbeta, int64_t M, int64_t h,
                                  tp_dtype dtype, void* ws, size_t ws_bytes, void* stream);

/*
 * Head-sharded attention block, forward: out = x + sum_i O_i W_o,i with
 *   xn = LN(x; gamma, beta), QKV = xn W_qkv, O_t = softmax(Q_t K_t^T / sqrt(d)) V_t.
 * Shard i owns heads [i*H/N, (i+1)*H/N): its columns of W_q, W_k, W_v (column-parallel)
 * and row block i of W_o (row-parallel); no gather of heads is needed, the shard
 * outputs are summed [张量并行 notes, §Multi-Head Attention 的并行化; Infra: Tensor
 * Parallel, attention; 20260402-parallelism, §1 TP]. n_heads % N == 0 and N <= n_heads
 * [Infra: Tensor Parallel, attention, the Megatron check]; head_dim = h / n_heads
 * in {16, 32, 64}. Softmax scale 1/sqrt(d); causal != 0 masks keys after the query.
 *   x (b*s, h) read (rows of one sequence consecutive); gamma, beta (h) fp32;
 *   Wqkv (h, 3h) = [W_q | W_k | W_v]; Wo (h, h)
 *   saved for the backward (written): xn (M, h), mean, rstd (M) fp32, qkv (M, 3h),
 *   o (M, h), lse (b, n_heads, s) fp32;  out (M, h) written.
 *   ws: TP_REDUCE_BUFFERS needs N*M*h*4 bytes.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_SHAPE (h % heads, heads % N, head_dim, bf16: (h/N) % 64),
 *         TP_ERR_ALIGNMENT, TP_ERR_WORKSPACE, TP_ERR_CUDA.
 */
TP_API tp_status tp_attn_proj_fwd(const void* x, const float* gamma, const float* beta,
                                  const void* Wqkv, const void* Wo, void* xn, float* mean,
                                  float* rstd, void* qkv, void* o, float* lse, void* out,
                                  int64_t b, int64_t s, int64_t h, int32_t n_heads, int32_t N,
                                  int causal, tp_dtype dtype, tp_reduce mode, void* ws,
                                  size_t ws_bytes, void* stream);

/*
 * Attention block backward (dout = d out). dWo_i = O_i^T dout, dO_i = dout W_o,i^T,
 * per head dV = P^T dO, dS = P * (dO V^T - rowsum(dO * O)), dQ = dS K/sqrt(d),
 * dK = dS^T Q/sqrt(d); dW_qkv = xn^T dQKV; f-backward dxn = sum_i dQKV_i W_qkv,i^T;
 * dx = dout + LN'(dxn) (the residual branch).
 *   inputs: the forward's x, gamma, Wqkv, Wo and saved xn, mean, rstd, qkv, o, lse
 *   outputs: dx (M, h), dgamma, dbeta (h) fp32, dWqkv (h, 3h), dWo (h, h)
 *   ws: tp_workspace_size(TP_OP_ATTN_PROJ_BWD, b*s, h, 0, N, dtype, 0, mode)
 */
TP_API tp_status tp_attn_proj_bwd(const void* x, const float* gamma, const void* Wqkv,
                                  const void* Wo, const void* xn, const float* mean,
                                  const float* rstd, const void* qkv, const void* o,
                                  const float* lse, const void* dout, void* dx, float* dgamma,
                                  float* dbeta, void* dWqkv, void* dWo, int64_t b, int64_t s,
                                  int64_t h, int32_t n_heads, int32_t N, int causal,
                                  tp_dtype dtype, tp_reduce mode, void* ws, size_t ws_bytes,
                                  void* stream);

/*
 * Grouped-query attention under head sharding [张量并行 notes, §相关分析, GQA]: H =
 * n_heads query heads share Hkv = n_kv_heads key/value heads, query head t using
 * key/value head t / (H / Hkv). N shards (H % N == 0): when N <= Hkv (Hkv % N == 0)
 * shard i owns H/N query heads and Hkv/N key/value heads; when N > Hkv (N % Hkv == 0)
 * it owns H/N query heads of one group and a replica of that group's key/value head,
 * and the replicas' weight gradients are all-reduced so the copies stay equal.
 * head_dim = h / H in {16, 32, 64}; W_o is (H head_dim = h, h).
 *
 * Sharded QKV weight Wqkv (h, W), W = tp_gqa_qkv_cols(...): shard i's block of
 * S = W / N columns is [W_q of its query heads | W_k of its key/value heads | W_v of
 * the same] (the per-rank layout of the Megatron-LM 实战 04 listing's column-parallel
 * QKV); tp_gqa_pack_qkv builds it from the full W_q (h, H d), W_k, W_v (h, Hkv d).
 * qkv (M, W) is laid out the same way. bf16 also needs S % 64 == 0 and (h / N) % 64 == 0.
 */
TP_API int64_t tp_gqa_qkv_cols(int64_t h, int32_t n_heads, int32_t n_kv_heads, int32_t N);
TP_API size_t tp_gqa_workspace_size(int fwd, int64_t M, int64_t h, int32_t n_heads,
                                    int32_t n_kv_heads, int32_t N, tp_dtype dtype,
                                    tp_reduce mode);
TP_API tp_status tp_gqa_pack_qkv(const void* Wq, const void* Wk, const void* Wv, void* Wqkv,
                                 int64_t h, int32_t n_heads, int32_t n_kv_heads, int32_t N,
                                 tp_dtype dtype, void* stream);
/* The attention core alone on the sharded qkv (M, W): O (M, h) and lse (b, n_heads, s);
 * backward: dqkv (M, W) from dO, each key/value head's gradient summing the query heads
 * of its block that use it (a replica's share; tp_gqa_attn_proj_bwd adds the replicas).
 * Every element of dqkv's M rows is written. The backward's ws is optional scratch of at
 * least tp_gqa_attention_bwd_workspace_size(b, s, n_heads) bytes, 16-byte aligned: with
 * it, bf16 at head_dim 64 runs on the tensor cores (the per-row (lse, D = rowsum(dO * O))
 * pairs are kept there); with ws == NULL every case runs on the CUDA cores. A ws that is
 * given but too small is TP_ERR_WORKSPACE, one not 16-byte aligned TP_ERR_ALIGNMENT. */
TP_API size_t tp_gqa_attention_bwd_workspace_size(int64_t b, int64_t s, int32_t n_heads);
TP_API tp_status tp_gqa_attention_fwd(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                                      int64_t h, int32_t n_heads, int32_t n_kv_heads, int32_t N,
                                      int causal, tp_dtype dtype, void* stream);
TP_API tp_status tp_gqa_attention_bwd(const void* qkv, const void* o, const float* lse,
                                      const void* dO, void* dqkv, int64_t b, int64_t s, int64_t h,
                                      int32_t n_heads, int32_t n_kv_heads, int32_t N, int causal,
                                      tp_dtype dtype, void* ws, size_t ws_bytes, void* stream);
/* out = x + sum_i O_i W_o,i, O from LN(x) and the sharded Wqkv; saved state as
 * tp_attn_proj_fwd with qkv (M, W) and lse (b, n_heads, s). */
TP_API tp_status tp_gqa_attn_proj_fwd(const void* x, const float* gamma, const float* beta,
                                      const void* Wqkv, const void* Wo, void* xn, float* mean,
                                      float* rstd, void* qkv, void* o, float* lse, void* out,
                                      int64_t b, int64_t s, int64_t h, int32_t n_heads,
                                      int32_t n_kv_heads, int32_t N, int causal, tp_dtype dtype,
                                      tp_reduce mode, void* ws, size_t ws_bytes, void* stream);
/* Backward: dWqkv (h, W) in the sharded layout, each replicated key/value head's
 * columns holding the sum over its replicas; dx includes the residual's dout. */
TP_API tp_status tp_gqa_attn_proj_bwd(const void* x, const float* gamma, const void* Wqkv,
                                      const void* Wo, const void* xn, const float* mean,
                                      const float* rstd, const void* qkv, const void* o,
                                      const float* lse, const void* dout, void* dx,
                                      float* dgamma, float* dbeta, void* dWqkv, void* dWo,
                                      int64_t b, int64_t s, int64_t h, int32_t n_heads,
                                      int32_t n_kv_heads, int32_t N, int causal, tp_dtype dtype,
                                      tp_reduce mode, void* ws, size_t ws_bytes, void* stream);

/*
 * Sequence-parallel pre-LN MLP sub-block, out = x + MLP(LN(x))
 * [20260402-parallelism, §5 Sequence Parallelism]. The rows are split over the N
 * ranks of the tensor-parallel group along the sequence: rank r holds rows
 * [r M/N, (r+1) M/N) of x, xn, mean, rstd, out and dx (M % N == 0; sequence-major
 * rows, so each rank's piece is one contiguous block). Forward: LN on each rank's
 * rows; all-gather of xn (the ranks' blocks are adjacent in one buffer, so the
 * gather is the buffer itself); the tensor-parallel MLP of tp_mlp_fwd; the sum
 * after the row-parallel GEMM is a reduce-scatter: rank r receives its rows of
 * sum_i Z_i and adds its residual rows x_r. The two collectives move the same
 * bytes as the all-reduce they replace.
 *   x (M, h) read;  gamma, beta (h) fp32 read;  W1, W1_up, W2 as tp_mlp_fwd
 *   xn (M, h), mean, rstd (M) fp32 written (saved for the backward)
 *   Y, Y_up, H as tp_mlp_fwd (H required here);  out (M, h) written
 *   ws: tp_workspace_size(TP_OP_SP_MLP_FWD, M, h, f, N, dtype, act, mode)
 * Errors: as tp_mlp_fwd, plus TP_ERR_SHAPE when M % N != 0.
 */
TP_API tp_status tp_sp_mlp_fwd(const void* x, const float* gamma, const float* beta,
                               const void* W1, const void* W1_up, const void* W2, void* xn,
                               float* mean, float* rstd, void* Y, void* Y_up, void* H, void* out,
                               int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dtype,
                               tp_act act, tp_reduce mode, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * Backward of tp_sp_mlp_fwd. dout's rank blocks are all-gathered (every shard reads
 * all of it); the MLP's input gradient is reduce-scattered, so rank r gets its rows
 * of sum_i dX_i; LN backward runs on each rank's rows and adds the residual's dout_r.
 * Each rank's LN parameters see only that rank's rows, so the per-rank gradients
 * differ: dgamma_ranks[r] / dbeta_ranks[r] (N, h) fp32 are each rank's sums (NULL =
 * not kept) and dgamma / dbeta (h) fp32 their sum over the ranks in rank order (the
 * all-reduce sequence parallelism adds for the LN parameters).
 *   dx (M, h) written;  dW1, dW1_up, dW2 as tp_mlp_bwd
 *   ws: tp_workspace_size(TP_OP_SP_MLP_BWD, M, h, f, N, dtype, act, mode)
 * Errors: as tp_mlp_bwd, plus TP_ERR_SHAPE when M % N != 0.
 */
TP_API tp_status tp_sp_mlp_bwd(const void* x, const float* gamma, const void* W1,
                               const void* W1_up, const void* W2, const void* xn,
                               const float* mean, const float* rstd, const void* Y,
                               const void* Y_up, const void* H, const void* dout, void* dx,
                               float* dgamma, float* dbeta, float* dgamma_ranks,
                               float* dbeta_ranks, void* dW1, void* dW1_up, void* dW2, int64_t M,
                               int64_t h, int64_t f, int32_t N, tp_dtype dtype, tp_act act,
                               tp_reduce mode, void* ws, size_t ws_bytes, void* stream);

/*
 * Pre-LN transformer layer with the tensor-parallel attention block and GELU MLP
 * [Megatron-LM 实战 04 张量并行实现, 核心实现, TPTransformerLayer]:
 *   x1 = x + Attn(LN1(x)),  out = x1 + MLP(LN2(x1)).
 * tp_layer_fwd fills every field of *saved; tp_layer_bwd reads them and writes dx and
 * every field of *grads. Sizes: M = b*s tokens, h hidden, f MLP width, n_heads, N shards.
 * The shard sum after W_o and LN2 run as one pass (tp_row_linear_ln), so h <= 16384.
 * ws: tp_workspace_size(TP_OP_LAYER_FWD / TP_OP_LAYER_BWD, b*s, h, f, N, dtype, 0, mode).
 * Errors: those of tp_attn_proj_fwd / _bwd and tp_mlp_fwd / _bwd.
 */
TP_API tp_status tp_layer_fwd(const void* x, const tp_layer_weights* w, const tp_layer_saved* saved,
                              void* out, int64_t b, int64_t s, int64_t h, int64_t f,
                              int32_t n_heads, int32_t N, int causal, tp_dtype dtype,
                              tp_reduce mode, void* ws, size_t ws_bytes, void* stream);

TP_API tp_status tp_layer_bwd(const void* x, const tp_layer_weights* w,
                              const tp_layer_saved* saved, const void* dout, void* dx,
                              const tp_layer_grads* grads, int64_t b, int64_t s, int64_t h,
                              int64_t f, int32_t n_heads, int32_t N, int causal, tp_dtype dtype,
                              tp_reduce mode, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ vocabulary-parallel
 * embedding, cross-entropy, the small GPT and its optimiser. Shard i of the vocabulary
 * owns rows [i v/N, (i+1) v/N) of E and the same columns of the logits. Token ids and
 * targets are int32 device arrays; ids or targets outside [0, v) give a zero embedding
 * row and a zero loss / gradient row (the mean still divides by M). */

/* x[t] = sum_i (E_i[ids[t]] if shard i owns ids[t], else 0): every shard looks up the ids
 * it owns and the all-reduce adds the results [张量并行 notes, §嵌入层的并行化, input].
 *   ids (M) int32;  E (vocab, h) read;  x (M, h) written.
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_SHAPE (vocab % N), TP_ERR_DTYPE, TP_ERR_ALIGNMENT. */
TP_API tp_status tp_vocab_embed_fwd(const int32_t* ids, const void* E, void* x, int64_t M,
                                    int64_t vocab, int64_t h, int32_t N, tp_dtype dtype,
                                    void* stream);

/* dE[v] (+)= sum over tokens t with ids[t] == v of dx[t], in token order (shard i fills
 * its own rows). accumulate != 0 adds to dE (e.g. to the output layer's gradient of a
 * shared embedding: grad_total = grad_in + grad_out [张量并行 notes, §嵌入层的并行化]);
 * 0 overwrites it. */
TP_API tp_status tp_vocab_embed_bwd(const int32_t* ids, const void* dx, void* dE, int64_t M,
                                    int64_t vocab, int64_t h, int32_t N, int accumulate,
                                    tp_dtype dtype, void* stream);

/* Cross-entropy of logits (M, vocab) against targets (M), vocabulary-parallel
 * [张量并行 notes, §损失计算层的并行化]: m = all-reduce(max) of the shards' row maxima,
 * S = all-reduce(sum) of the shards' sums of exp(l - m), the target's shard adds
 * log S + m - l_target to its loss, and the loss is the sum of the N shard losses / M.
 *   lse (M) fp32 written (m + log S, for the backward); row_loss (M) fp32 written;
 *   shard_loss (N) fp32 written or NULL; loss (1) fp32 device written (the mean). */
TP_API tp_status tp_vocab_ce_fwd(const void* logits, const int32_t* targets, float* lse,
                                 float* row_loss, float* shard_loss, float* loss, int64_t M,
                                 int64_t vocab, int32_t N, tp_dtype dtype, void* stream);

/* dlogits = scale * (softmax(logits) - one_hot(targets)), from lse; dlogits may be the
 * logits buffer itself (in place). scale = 1/M for the mean loss. */
TP_API tp_status tp_vocab_ce_bwd(const void* logits, const int32_t* targets, const float* lse,
                                 void* dlogits, int64_t M, int64_t vocab, int32_t N,
                                 float scale, tp_dtype dtype, void* stream);

/* AdamW with decoupled weight decay over n fp32 values, step >= 1 (bias corrections
 * 1 - beta^step): p <- p (1 - lr wd); m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
 * p <- p - lr (m / bc1) / (sqrt(v / bc2) + eps). The listing of the Megatron-LM 实战 04
 * page trains its GPT with AdamW; the paper has no kernel for it. m, v start at 0. */
TP_API tp_status tp_adamw_step(float* p, const float* g, float* m, float* v, int64_t n,
                               int64_t step, float lr, float beta1, float beta2, float eps,
                               float weight_decay, void* stream);

/* The device-side bookkeeping of one training step, for a loop whose steps replay from a
 * CUDA graph (a graph cannot take a new host argument per replay): *step (one int32 in
 * device memory, 0 before the first step) advances by one, and when loss and loss_hist
 * are given (both or neither), loss_hist[(*step - 1) % hist_len] = *loss. Enqueue it after
 * the step's loss is written and before tp_adamw_step_device. (The pages' training loop,
 * Megatron-LM 实战 04, 训练入口, keeps its step count and losses on the host.)
 * Errors: TP_ERR_INVALID_ARG, TP_ERR_ALIGNMENT (4-byte), TP_ERR_CUDA. */
TP_API tp_status tp_train_step_advance(int32_t* step, const float* loss, float* loss_hist,
                                       int64_t hist_len, void* stream);

/* tp_adamw_step with the step count read from device memory (*step >= 1, the counter that
 * tp_train_step_advance keeps) instead of a host argument; the same arithmetic, with the
 * bias corrections 1 - beta^step formed in fp32 on the device (the host entry point forms
 * them in double: results may differ in the last bits). p, g, m, v and step must be 4-byte
 * aligned. */
TP_API tp_status tp_adamw_step_device(float* p, const float* g, float* m, float* v, int64_t n,
                                      const int32_t* step, float lr, float beta1, float beta2,
                                      float eps, float weight_decay, void* stream);

/* Bytes of workspace tp_gpt_fwd_bwd needs (0 on invalid arguments). */
TP_API size_t tp_gpt_workspace_size(const tp_gpt_config* cfg, tp_dtype dtype, tp_reduce mode);

/* Loss and every gradient of the small GPT [Megatron-LM 实战 04 张量并行实现, 核心实现,
 * SmallGPT]: embedding (vocabulary-parallel), the layers of tp_layer_fwd, final LN,
 * output layer x_f E^T (column-parallel over the vocabulary), vocabulary-parallel
 * cross-entropy (mean over the M rows); then the backward: the output layer's input
 * gradient is summed over the vocabulary shards, its weight gradient written to dE, the
 * layers' backward, and the embedding's gradient added to dE. fp32 only (the listing
 * trains in fp32).
 *   ids, targets (b*s) int32;  loss (1) fp32 device written.
 * Errors: those of the parts; TP_ERR_DTYPE for bf16; TP_ERR_SHAPE (vocab % N, heads). */
TP_API tp_status tp_gpt_fwd_bwd(const tp_gpt_config* cfg, const tp_gpt_weights* w,
                                const tp_gpt_grads* g, const int32_t* ids,
                                const int32_t* targets, float* loss, tp_dtype dtype,
                                tp_reduce mode, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------ testing */

/* Failure injection for tests. While enabled (non-zero), every launch of a kernel with
 * bounded barrier waits -- the tensor-core GEMMs (CTA-pair, one-CTA and decode
 * configurations) and the tensor-core attention forward, dQ and dK/dV kernels --
 * makes its MMA thread first wait on a barrier that nothing arrives on, so the
 * bounded wait expires; the kernel then stops cleanly (its copies and MMAs drained,
 * TMEM freed) and tp_check_status reports TP_ERR_TIMEOUT. Nothing faults on the
 * device. Off by default; outputs of launches made while it is on are undefined. */
TP_API void tp_debug_inject_wait_fault(int enable);

#ifdef __cplusplus
}
#endif
#endif /* TPMLP_H */
