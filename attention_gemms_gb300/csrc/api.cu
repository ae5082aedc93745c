// C ABI of libtpmlp: argument validation, workspace carving and the composition
// of the tensor-parallel linear block out of GEMM / reduction launches.
#include <cuda_runtime.h>

#include <initializer_list>
#include <mutex>
#include <string>

#include "internal.h"

namespace tp {

tp_status check_device();
void set_debug_hang(int v);
void set_pair_mode(int v);
void set_wide_mode(int v);

namespace {
bool al16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }
}  // namespace

tp_status need(bool cond, tp_status s, const char* msg) { return cond ? TP_OK : fail(s, msg); }

tp_status check_aligned(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (p && !al16(p)) return fail(TP_ERR_ALIGNMENT, "device buffers must be 16-byte aligned");
  return TP_OK;
}

tp_status check_dtype(tp_dtype dt) {
  return need(dt == TP_BF16 || dt == TP_F32, TP_ERR_DTYPE, "dtype must be TP_BF16 or TP_F32");
}

// Extents of buffers that can exist in device memory: every extent below 2^31, a
// matrix below 2^40 elements, at most 65536 shards. Sizes past these limits are
// rejected before any byte count is formed, so N * rows * cols * 4 and the workspace
// sums built from such products cannot wrap around in 64 bits.
bool extents_ok(int64_t rows, int64_t cols, int64_t N) {
  constexpr int64_t kMaxExtent = int64_t(1) << 31, kMaxElems = int64_t(1) << 40;
  return rows >= 0 && cols >= 0 && rows < kMaxExtent && cols < kMaxExtent && N >= 1 &&
         N <= 65536 && rows * cols < kMaxElems;
}
tp_status check_extents(int64_t rows, int64_t cols, int64_t N) {
  return need(extents_ok(rows, cols, N), TP_ERR_SHAPE,
              "sizes too large (an extent >= 2^31, a matrix >= 2^40 elements or N > 65536)");
}

// bf16 tile rules: reduced widths and per-shard widths are whole 64-column blocks
tp_status check_mlp_shape(int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt) {
  TP_TRY(need(N >= 1, TP_ERR_INVALID_ARG, "shard count N must be >= 1"));
  TP_TRY(need(M >= 0 && h >= 1 && f >= 1, TP_ERR_INVALID_ARG, "sizes must be positive (M >= 0)"));
  TP_TRY(check_extents(M, h, N));
  TP_TRY(check_extents(M, f, N));
  TP_TRY(check_extents(h, f, 1));
  TP_TRY(need(f % N == 0, TP_ERR_SHAPE, "h' (f) must be divisible by the shard count N"));
  if (dt == TP_BF16) {
    TP_TRY(need(h % 64 == 0, TP_ERR_SHAPE, "bf16 path: h must be a multiple of 64"));
    TP_TRY(need((f / N) % 64 == 0, TP_ERR_SHAPE, "bf16 path: h'/N must be a multiple of 64"));
  }
  return TP_OK;
}

// fp32 shard partials of variant A; saturates at 2^62 bytes (no wrap-around) for sizes
// that check_extents would reject
size_t partial_bytes(int64_t M, int64_t n, int32_t N, tp_reduce mode) {
  if (mode != TP_REDUCE_BUFFERS || M <= 0 || n <= 0 || N <= 0) return 0;
  constexpr size_t kCap = size_t(1) << 62;
  const size_t rows = static_cast<size_t>(M), cols = static_cast<size_t>(n);
  if (cols > kCap / rows) return kCap;
  const size_t elems = rows * cols;
  if (elems > kCap / (sizeof(float) * static_cast<size_t>(N))) return kCap;
  return elems * static_cast<size_t>(N) * sizeof(float);
}

// A weight of the linear map from `in` to `out` features as the B operand B(k, n) of
// D = A B (k over `in`, n over `out`): stored (in, out) it is read MN-major, stored
// (out, in) K-major -- in place either way.
void weight_operand(GemmDesc& d, int s, const void* W, int64_t in, int64_t out, bool w_out_in) {
  if (w_out_in) {
    d.B[s] = {W, out, in, in};
    d.b_mn = false;
  } else {
    d.B[s] = {W, in, out, out};
    d.b_mn = true;
  }
}

// The transpose W^T of such a weight as the B operand (k over `out`, n over `in`), for
// the backward's dH = dZ W^T: stored (in, out) it is read K-major, stored (out, in)
// MN-major.
void weight_t_operand(GemmDesc& d, int s, const void* W, int64_t in, int64_t out, bool w_out_in) {
  if (w_out_in) {
    d.B[s] = {W, out, in, in};
    d.b_mn = true;
  } else {
    d.B[s] = {W, in, out, out};
    d.b_mn = false;
  }
}

tp_status col_impl(const void* X, const void* W, const void* Wu, void* Y, void* Yu, void* out,
                   int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt, tp_act act,
                   cudaStream_t st, bool w_out_in) {
  GemmDesc d;
  d.dtype = dt;
  d.M = M;
  d.N = f;
  d.K = h;
  d.A[0] = {X, M, h, h};
  weight_operand(d, 0, W, h, f, w_out_in);
  d.ldo = f;
  d.shards = N;
  d.shard_axis = 1;
  if (act == TP_ACT_NONE) {
    d.epi = EPI_STORE;
    d.out[0] = out;
    d.out_f32 = dt == TP_F32;
  } else if (act == TP_ACT_GELU) {
    d.epi = EPI_GELU;
    d.out[0] = Y;
    d.out[1] = out;
  } else {
    d.paired = true;
    weight_operand(d, 1, Wu, h, f, w_out_in);
    d.epi = EPI_SWIGLU;
    d.out[0] = Y;
    d.out[1] = Yu;
    d.out[2] = out;
  }
  return launch_gemm(d, st);
}

// out = sum_i Xs_i W_i (+ residual): variant A (partials + reduce) or B (split-K fold)
tp_status row_impl(const void* Xs, const void* W, const void* residual, void* out, int64_t M,
                   int64_t k, int64_t n, int32_t N, tp_dtype dt, tp_reduce mode, void* ws,
                   cudaStream_t st, bool w_out_in) {
  GemmDesc d;
  d.dtype = dt;
  d.M = M;
  d.N = n;
  d.A[0] = {Xs, M, k, k};
  weight_operand(d, 0, W, k, n, w_out_in);
  d.ldo = n;
  d.epi = EPI_STORE;
  if (mode == TP_REDUCE_SPLITK) {
    d.K = k;
    d.in[0] = residual;
    d.out[0] = out;
    d.out_f32 = dt == TP_F32;
    return launch_gemm(d, st);
  }
  d.K = k / N;
  d.groups = N;
  d.out[0] = ws;
  d.out_f32 = true;
  d.out_group_stride = M * n;
  // Many rows: two row blocks, each a GEMM writing its rows of every shard's partial and
  // a shard sum of those rows; the first block's sum (HBM-bound) runs on a side stream
  // beside the second block's GEMM (tensor-bound), so only the second sum is exposed.
  const int64_t half = M >= 2048 ? (M / 2 + 255) / 256 * 256 : 0;  // whole 256-row tiles
  if (half > 0 && half < M) {
    const size_t elt = elem_size(dt);
    float* P = static_cast<float*>(ws);
    GemmDesc d0 = d;
    d0.M = half;
    TP_TRY(launch_gemm(d0, st));
    SideBranch first(st);
    const bool beside = first.stream() != st;
    TP_TRY(launch_shard_reduce(P, residual, out, N, half, n, dt, first.stream(), beside ? 2 : 8,
                               M * n));
    GemmDesc d1 = d;
    d1.M = M - half;
    d1.A[0] = {static_cast<const char*>(Xs) + half * k * elt, M - half, k, k};
    d1.out[0] = P + half * n;
    TP_TRY(launch_gemm(d1, st));
    TP_TRY(launch_shard_reduce(P + half * n,
                               residual ? static_cast<const char*>(residual) + half * n * elt : nullptr,
                               static_cast<char*>(out) + half * n * elt, N, M - half, n, dt, st, 8,
                               M * n));
    return first.join();
  }
  TP_TRY(launch_gemm(d, st));
  return launch_shard_reduce(static_cast<const float*>(ws), residual, out, N, M, n, dt, st);
}

// sum_out = sum_i Xs_i W_i (+ residual), y = LN(sum_out): variant A fuses the LN into
// the reduction of the partials; variant B folds the sum in the GEMM, then runs LN
tp_status row_ln_impl(const void* Xs, const void* W, const void* residual, const float* gamma,
                      const float* beta, void* sum_out, void* y, float* mean, float* rstd,
                      int64_t M, int64_t k, int64_t n, int32_t N, float eps, tp_dtype dt,
                      tp_reduce mode, void* ws, cudaStream_t st) {
  if (mode == TP_REDUCE_SPLITK) {
    TP_TRY(row_impl(Xs, W, residual, sum_out, M, k, n, N, dt, mode, ws, st));
    return launch_layernorm_fwd(sum_out, gamma, beta, y, mean, rstd, M, n, eps, dt, st);
  }
  GemmDesc d;
  d.dtype = dt;
  d.M = M;
  d.N = n;
  d.K = k / N;
  d.groups = N;
  d.A[0] = {Xs, M, k, k};
  d.B[0] = {W, k, n, n};
  d.b_mn = true;
  d.ldo = n;
  d.epi = EPI_STORE;
  d.out[0] = ws;
  d.out_f32 = true;
  d.out_group_stride = M * n;
  TP_TRY(launch_gemm(d, st));
  return launch_shard_reduce_ln(static_cast<const float*>(ws), residual, gamma, beta, sum_out, y,
                                mean, rstd, N, M, n, eps, dt, st);
}

// The GEMM of dX = sum_i sum_s dA_s,i B_s,i^T over nseg operand pairs (dY with W1, or
// dG/dU with Wg/Wu): split-K writes dX itself into `dst`; buffers writes the N fp32
// partials (M x h each) into `dst`
tp_status dx_gemm(const void* const* dA, const void* const* Wt, int nseg, void* dst, int64_t M,
                  int64_t h, int64_t f, int32_t N, tp_dtype dt, tp_reduce mode, cudaStream_t st,
                  bool w_out_in) {
  GemmDesc d;
  d.dtype = dt;
  d.M = M;
  d.N = h;
  d.nseg = nseg;
  for (int s = 0; s < nseg; ++s) {
    d.A[s] = {dA[s], M, f, f};                       // dY (M, f), K-major
    weight_t_operand(d, s, Wt[s], h, f, w_out_in);   // W1^T as B(k = f, n = h)
  }
  d.ldo = h;
  d.epi = EPI_STORE;
  d.out[0] = dst;
  if (mode == TP_REDUCE_SPLITK) {
    d.K = f;
    d.out_f32 = dt == TP_F32;
    return launch_gemm(d, st);
  }
  d.K = f / N;
  d.groups = N;
  d.out_f32 = true;
  d.out_group_stride = M * h;
  return launch_gemm(d, st);
}

}  // namespace tp

using namespace tp;

extern "C" {

void tp_debug_inject_wait_fault(int enable) { set_debug_hang(enable); }

void tp_set_gemm_pair_mode(int enable) { set_pair_mode(enable == 0 || enable == 2 ? enable : 1); }

void tp_set_gemm_wide_mode(int mode) { set_wide_mode(mode == 0 || mode == 2 ? mode : 1); }

size_t tp_workspace_size(tp_op op, int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dtype,
                         tp_act act, tp_reduce mode) {
  if (N < 1 || M < 0 || h < 1 || (f < 1 && op != TP_OP_ATTN_PROJ_FWD && op != TP_OP_ATTN_PROJ_BWD &&
                                   op != TP_OP_LAYERNORM_BWD))
    return 0;
  if (dtype != TP_BF16 && dtype != TP_F32) return 0;
  // sizes the entry points reject (check_extents) need no workspace either
  if (!extents_ok(M, 3 * h, N) || !extents_ok(M, f, N) || !extents_ok(h, f, 1)) return 0;
  const size_t elt = elem_size(dtype);
  switch (op) {
    case TP_OP_COL_LINEAR: return 0;
    case TP_OP_ROW_LINEAR: return partial_bytes(M, f, N, mode);
    case TP_OP_MLP_FWD:
      return align_up(static_cast<size_t>(M) * f * elt, 256) + partial_bytes(M, h, N, mode);
    case TP_OP_MLP_BWD:
      return (act == TP_ACT_SWIGLU ? 2 : 1) * align_up(static_cast<size_t>(M) * f * elt, 256) +
             partial_bytes(M, h, N, mode);
    case TP_OP_ATTN_PROJ_FWD: return attn_workspace_size(true, M, h, N, dtype, mode);
    case TP_OP_ATTN_PROJ_BWD: return attn_workspace_size(false, M, h, N, dtype, mode);
    case TP_OP_LAYERNORM_BWD: return layernorm_bwd_ws_bytes(M, h);
    case TP_OP_LAYER_FWD: return layer_workspace_size(true, M, h, f, N, dtype, mode);
    case TP_OP_LAYER_BWD: return layer_workspace_size(false, M, h, f, N, dtype, mode);
    case TP_OP_SP_MLP_FWD: return sp_mlp_workspace_size(true, M, h, f, N, dtype, act, mode);
    case TP_OP_SP_MLP_BWD: return sp_mlp_workspace_size(false, M, h, f, N, dtype, act, mode);
    default: return 0;
  }
}

tp_status tp_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                  int a_trans, int b_trans, tp_dtype dtype, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(A && B && C, TP_ERR_INVALID_ARG, "A, B and C are required"));
  TP_TRY(need(M >= 0 && N >= 0 && K >= 1, TP_ERR_INVALID_ARG, "need M, N >= 0 and K >= 1"));
  if (dtype == TP_BF16) {
    TP_TRY(need(N % 8 == 0 && (a_trans ? M : K) % 8 == 0 && (b_trans ? K : N) % 8 == 0,
                TP_ERR_SHAPE, "bf16 path: N and the stored row widths must be multiples of 8"));
  }
  TP_TRY(check_aligned({A, B, C}));
  if (M == 0 || N == 0) return TP_OK;
  TP_TRY(check_device());
  GemmDesc d;
  d.dtype = dtype;
  d.M = M;
  d.N = N;
  d.K = K;
  d.a_mn = a_trans != 0;
  d.b_mn = b_trans == 0;
  d.A[0] = a_trans ? Operand{A, K, M, M} : Operand{A, M, K, K};
  d.B[0] = b_trans ? Operand{B, N, K, K} : Operand{B, K, N, N};
  d.ldo = N;
  d.epi = EPI_STORE;
  d.out[0] = C;
  d.out_f32 = dtype == TP_F32;
  return launch_gemm(d, static_cast<cudaStream_t>(stream));
}

tp_status check_wlayout(tp_wlayout wl) {
  return need(wl == TP_W_IN_OUT || wl == TP_W_OUT_IN, TP_ERR_INVALID_ARG,
              "w_layout must be TP_W_IN_OUT or TP_W_OUT_IN");
}

tp_status tp_col_linear(const void* X, const void* W, const void* W_up, void* Y, void* Y_up,
                        void* out, int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dtype,
                        tp_act act, tp_wlayout w_layout, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(check_wlayout(w_layout));
  TP_TRY(need(act >= TP_ACT_NONE && act <= TP_ACT_SWIGLU, TP_ERR_INVALID_ARG, "unknown act"));
  TP_TRY(need(X && W && out, TP_ERR_INVALID_ARG, "X, W and out are required"));
  TP_TRY(need(act != TP_ACT_SWIGLU || W_up, TP_ERR_INVALID_ARG, "SwiGLU needs W_up"));
  TP_TRY(check_mlp_shape(M, h, f, N, dtype));
  TP_TRY(check_aligned({X, W, W_up, Y, Y_up, out}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return col_impl(X, W, W_up, Y, Y_up, out, M, h, f, N, dtype, act,
                  static_cast<cudaStream_t>(stream), w_layout == TP_W_OUT_IN);
}

tp_status tp_row_linear(const void* Xs, const void* W, const void* residual, void* out, int64_t M,
                        int64_t k, int64_t n, int32_t N, tp_dtype dtype, tp_reduce mode, void* ws,
                        size_t ws_bytes, tp_wlayout w_layout, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(check_wlayout(w_layout));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(Xs && W && out, TP_ERR_INVALID_ARG, "Xs, W and out are required"));
  TP_TRY(need(N >= 1, TP_ERR_INVALID_ARG, "shard count N must be >= 1"));
  TP_TRY(need(M >= 0 && k >= 1 && n >= 1, TP_ERR_INVALID_ARG, "sizes must be positive (M >= 0)"));
  TP_TRY(check_extents(M, n, N));
  TP_TRY(check_extents(M, k, 1));
  TP_TRY(check_extents(k, n, 1));
  TP_TRY(need(k % N == 0, TP_ERR_SHAPE, "k must be divisible by the shard count N"));
  if (dtype == TP_BF16) {
    TP_TRY(need((k / N) % 64 == 0, TP_ERR_SHAPE, "bf16 path: k/N must be a multiple of 64"));
    TP_TRY(need(n % 64 == 0, TP_ERR_SHAPE, "bf16 path: n must be a multiple of 64"));
  }
  TP_TRY(check_aligned({Xs, W, residual, out, ws}));
  if (M == 0) return TP_OK;
  const size_t need_ws = partial_bytes(M, n, N, mode);
  TP_TRY(need(ws_bytes >= need_ws && (need_ws == 0 || ws), TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  return row_impl(Xs, W, residual, out, M, k, n, N, dtype, mode, ws,
                  static_cast<cudaStream_t>(stream), w_layout == TP_W_OUT_IN);
}

tp_status tp_shard_reduce(const float* partials, const void* residual, void* out, int32_t N,
                          int64_t M, int64_t n, tp_dtype out_dtype, void* stream) {
  TP_TRY(check_dtype(out_dtype));
  TP_TRY(need(partials && out, TP_ERR_INVALID_ARG, "partials and out are required"));
  TP_TRY(need(N >= 1 && M >= 0 && n >= 1, TP_ERR_INVALID_ARG, "need N >= 1, M >= 0, n >= 1"));
  TP_TRY(check_extents(M, n, N));
  TP_TRY(check_aligned({partials, residual, out}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_shard_reduce(partials, residual, out, N, M, n, out_dtype,
                             static_cast<cudaStream_t>(stream));
}

tp_status tp_shard_reduce_ln(const float* partials, const void* residual, const float* gamma,
                             const float* beta, void* sum_out, void* y, float* mean, float* rstd,
                             int32_t N, int64_t M, int64_t h, float eps, tp_dtype dtype,
                             void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(partials && gamma && beta && y, TP_ERR_INVALID_ARG,
              "partials, gamma, beta and y are required"));
  TP_TRY(need(N >= 1 && M >= 0 && h >= 1 && eps >= 0.0f, TP_ERR_INVALID_ARG,
              "need N >= 1, M >= 0, h >= 1, eps >= 0"));
  TP_TRY(check_extents(M, h, N));
  TP_TRY(need(h % 8 == 0 && h <= kReduceLnMaxH, TP_ERR_SHAPE,
              "fused reduce + LayerNorm: h must be a multiple of 8 and at most 16384"));
  TP_TRY(check_aligned({partials, residual, gamma, beta, sum_out, y, mean, rstd}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_shard_reduce_ln(partials, residual, gamma, beta, sum_out, y, mean, rstd, N, M, h,
                                eps, dtype, static_cast<cudaStream_t>(stream));
}

tp_status tp_row_linear_ln(const void* Xs, const void* W, const void* residual,
                           const float* gamma, const float* beta, void* sum_out, void* y,
                           float* mean, float* rstd, int64_t M, int64_t k, int64_t n, int32_t N,
                           float eps, tp_dtype dtype, tp_reduce mode, void* ws, size_t ws_bytes,
                           void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(Xs && W && gamma && beta && sum_out && y, TP_ERR_INVALID_ARG,
              "Xs, W, gamma, beta, sum_out and y are required"));
  TP_TRY(need(N >= 1, TP_ERR_INVALID_ARG, "shard count N must be >= 1"));
  TP_TRY(need(M >= 0 && k >= 1 && n >= 1 && eps >= 0.0f, TP_ERR_INVALID_ARG,
              "sizes must be positive (M >= 0) and eps >= 0"));
  TP_TRY(check_extents(M, n, N));
  TP_TRY(check_extents(M, k, 1));
  TP_TRY(check_extents(k, n, 1));
  TP_TRY(need(k % N == 0, TP_ERR_SHAPE, "k must be divisible by the shard count N"));
  TP_TRY(need(n % 8 == 0 && n <= kReduceLnMaxH, TP_ERR_SHAPE,
              "fused reduce + LayerNorm: n must be a multiple of 8 and at most 16384"));
  if (dtype == TP_BF16) {
    TP_TRY(need((k / N) % 64 == 0, TP_ERR_SHAPE, "bf16 path: k/N must be a multiple of 64"));
    TP_TRY(need(n % 64 == 0, TP_ERR_SHAPE, "bf16 path: n must be a multiple of 64"));
  }
  TP_TRY(check_aligned({Xs, W, residual, gamma, beta, sum_out, y, mean, rstd, ws}));
  if (M == 0) return TP_OK;
  const size_t need_ws = partial_bytes(M, n, N, mode);
  TP_TRY(need(ws_bytes >= need_ws && (need_ws == 0 || ws), TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  return row_ln_impl(Xs, W, residual, gamma, beta, sum_out, y, mean, rstd, M, k, n, N, eps, dtype,
                     mode, ws, static_cast<cudaStream_t>(stream));
}

tp_status tp_mlp_fwd(const void* X, const void* W1, const void* W1_up, const void* W2,
                     const void* residual, void* Y, void* Y_up, void* H, void* Z, int64_t M,
                     int64_t h, int64_t f, int32_t N, tp_dtype dtype, tp_act act, tp_reduce mode,
                     void* ws, size_t ws_bytes, tp_wlayout w_layout, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(check_wlayout(w_layout));
  TP_TRY(need(act == TP_ACT_GELU || act == TP_ACT_SWIGLU, TP_ERR_INVALID_ARG,
              "MLP act must be TP_ACT_GELU or TP_ACT_SWIGLU"));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(X && W1 && W2 && Z, TP_ERR_INVALID_ARG, "X, W1, W2 and Z are required"));
  TP_TRY(need(act != TP_ACT_SWIGLU || W1_up, TP_ERR_INVALID_ARG, "SwiGLU needs W1_up"));
  TP_TRY(check_mlp_shape(M, h, f, N, dtype));
  TP_TRY(check_aligned({X, W1, W1_up, W2, residual, Y, Y_up, H, Z, ws}));
  if (M == 0) return TP_OK;
  const size_t h_bytes = H ? 0 : align_up(static_cast<size_t>(M) * f * elem_size(dtype), 256);
  const size_t need_ws = h_bytes + partial_bytes(M, h, N, mode);
  TP_TRY(need(ws_bytes >= need_ws && (need_ws == 0 || ws), TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* Hb = H ? H : ws;
  void* parts = static_cast<char*>(ws) + h_bytes;
  const bool wt = w_layout == TP_W_OUT_IN;
  TP_TRY(col_impl(X, W1, W1_up, Y, Y_up, Hb, M, h, f, N, dtype, act, st, wt));
  return row_impl(Hb, W2, residual, Z, M, f, h, N, dtype, mode, parts, st, wt);
}

tp_status tp_mlp_bwd(const void* X, const void* W1, const void* W1_up, const void* W2,
                     const void* Y, const void* Y_up, const void* H, const void* dZ, void* dX,
                     void* dW1, void* dW1_up, void* dW2, int64_t M, int64_t h, int64_t f,
                     int32_t N, tp_dtype dtype, tp_act act, tp_reduce mode, void* ws,
                     size_t ws_bytes, tp_wlayout w_layout, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(check_wlayout(w_layout));
  TP_TRY(need(act == TP_ACT_GELU || act == TP_ACT_SWIGLU, TP_ERR_INVALID_ARG,
              "MLP act must be TP_ACT_GELU or TP_ACT_SWIGLU"));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  const bool sw = act == TP_ACT_SWIGLU;
  TP_TRY(need(X && W1 && W2 && Y && H && dZ && dX && dW1 && dW2, TP_ERR_INVALID_ARG,
              "X, W1, W2, Y, H, dZ, dX, dW1 and dW2 are required"));
  TP_TRY(need(!sw || (W1_up && Y_up && dW1_up), TP_ERR_INVALID_ARG,
              "SwiGLU needs W1_up, Y_up and dW1_up"));
  TP_TRY(check_mlp_shape(M, h, f, N, dtype));
  TP_TRY(check_aligned({X, W1, W1_up, W2, Y, Y_up, H, dZ, dX, dW1, dW1_up, dW2, ws}));
  if (M == 0) return TP_OK;
  const size_t elt = elem_size(dtype);
  const size_t g_one = align_up(static_cast<size_t>(M) * f * elt, 256);
  const size_t g_bytes = (sw ? 2 : 1) * g_one;
  const size_t need_ws = g_bytes + partial_bytes(M, h, N, mode);
  TP_TRY(need(ws_bytes >= need_ws && ws, TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool wt = w_layout == TP_W_OUT_IN;
  void* dY = ws;  // GELU: dY; SwiGLU: dG then dU
  void* dU = static_cast<char*>(ws) + g_one;
  void* parts = static_cast<char*>(ws) + g_bytes;

  // 1. g-backward is the identity: every shard reads all of dZ.
  //    dH_i = dZ W2_i^T with the activation derivative fused (row-parallel dX_i = dY W_i^T)
  {
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = f;
    d.K = h;
    d.A[0] = {dZ, M, h, h};
    weight_t_operand(d, 0, W2, f, h, wt);  // W2^T as B(k = h, n = f)
    d.ldo = f;
    d.shards = N;
    d.shard_axis = 1;
    if (sw) {
      d.epi = EPI_DSWIGLU;
      d.in[0] = Y;
      d.in[1] = Y_up;
      d.out[0] = dY;
      d.out[1] = dU;
    } else {
      d.epi = EPI_DGELU;
      d.in[0] = Y;
      d.out[0] = dY;
    }
    TP_TRY(launch_gemm(d, st));
  }
  // 2. dW2_i = H_i^T dZ (row-parallel weight gradient; shard i = row block i of the
  //    (f, h) gradient), or in (out, in) storage dW2_i^T = dZ^T H_i (column block i)
  auto dw2 = [&]() -> tp_status {
    GemmDesc d;
    d.dtype = dtype;
    d.K = M;
    d.a_mn = true;
    d.b_mn = true;
    d.epi = EPI_STORE;
    d.out[0] = dW2;
    d.out_f32 = dtype == TP_F32;
    d.shards = N;
    if (wt) {
      d.M = h;
      d.N = f;
      d.A[0] = {dZ, M, h, h};
      d.B[0] = {H, M, f, f};
      d.ldo = f;
      d.shard_axis = 1;
    } else {
      d.M = f;
      d.N = h;
      d.A[0] = {H, M, f, f};
      d.B[0] = {dZ, M, h, h};
      d.ldo = h;
      d.shard_axis = 0;
    }
    return launch_gemm(d, st);
  };
  // 3. dW1_i = X^T dY_i (column-parallel weight gradient; shard i = column block i), or
  //    in (out, in) storage dW1_i^T = dY_i^T X (row block i); SwiGLU also dW1up from dU
  auto dw1 = [&]() -> tp_status {
    GemmDesc d;
    d.dtype = dtype;
    d.K = M;
    d.a_mn = true;
    d.b_mn = true;
    d.shards = N;
    if (wt) {  // one GEMM per projection: the gate's and the up's gradients are row blocks
      d.M = f;
      d.N = h;
      d.B[0] = {X, M, h, h};
      d.ldo = h;
      d.shard_axis = 0;
      d.epi = EPI_STORE;
      d.out_f32 = dtype == TP_F32;
      d.A[0] = {dY, M, f, f};
      d.out[0] = dW1;
      TP_TRY(launch_gemm(d, st));
      if (!sw) return TP_OK;
      d.A[0] = {dU, M, f, f};
      d.out[0] = dW1_up;
      return launch_gemm(d, st);
    }
    d.M = h;
    d.N = f;
    d.A[0] = {X, M, h, h};
    d.B[0] = {dY, M, f, f};
    d.ldo = f;
    d.shard_axis = 1;
    if (sw) {
      d.paired = true;
      d.B[1] = {dU, M, f, f};
      d.epi = EPI_PAIR;
      d.out[0] = dW1;
      d.out[1] = dW1_up;
    } else {
      d.epi = EPI_STORE;
      d.out[0] = dW1;
      d.out_f32 = dtype == TP_F32;
    }
    return launch_gemm(d, st);
  };
  // 4. f-backward: dX = sum_i dY_i W1_i^T (SwiGLU: + dU_i W1up_i^T)
  const void* dA[2] = {dY, dU};
  const void* Wt[2] = {W1, W1_up};
  const int nseg = sw ? 2 : 1;
  if (mode == TP_REDUCE_SPLITK) {
    TP_TRY(dw2());
    TP_TRY(dw1());
    return dx_gemm(dA, Wt, nseg, dX, M, h, f, N, dtype, mode, st, wt);
  }
  // Per-shard partials: dX's GEMM comes first, and the shard sum of its partials (the
  // all-reduce stand-in, HBM-bound) runs on a side stream beside the two weight-gradient
  // GEMMs (tensor-core-bound), which do not read dX. A grid of two reduce CTAs per SM
  // leaves every SM room for the GEMM's persistent CTA.
  TP_TRY(dx_gemm(dA, Wt, nseg, parts, M, h, f, N, dtype, mode, st, wt));
  SideBranch sum(st);
  const bool beside = sum.stream() != st;
  TP_TRY(launch_shard_reduce(static_cast<const float*>(parts), nullptr, dX, N, M, h, dtype,
                             sum.stream(), beside ? 2 : 8));
  TP_TRY(dw2());
  TP_TRY(dw1());
  return sum.join();
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation variant
//
// tp_row_linear_noalloc: the row-parallel linear with per-shard partial buffers
// (TP_REDUCE_BUFFERS), for callers that cannot allocate device memory -- for
// example a library loaded into a host process whose device memory is owned by
// its own pool allocator, or which runs under a fixed device-memory budget, so it
// can neither call cudaMalloc itself nor hand this library a workspace. The fp32
// partials live in the fixed array below instead of a caller workspace.

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB, held by every device that loads the library

__device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device. In host code the
// symbol's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, called with that device current; it is looked up once per
// device and cached (a cudaDeviceReset of the device invalidates the cached address).
tp_status noalloc_scratch(void** out) {
  int dev = 0;
  TP_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(TP_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    TP_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TP_OK;
}

}  // namespace

extern "C" tp_status tp_row_linear_noalloc(const void* Xs, const void* W, const void* residual,
                                           void* out, int64_t M, int64_t k, int64_t n, int32_t N,
                                           tp_dtype dtype, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(Xs && W && out, TP_ERR_INVALID_ARG, "Xs, W and out are required"));
  TP_TRY(need(N >= 1, TP_ERR_INVALID_ARG, "shard count N must be >= 1"));
  TP_TRY(need(M >= 0 && k >= 1 && n >= 1, TP_ERR_INVALID_ARG, "sizes must be positive (M >= 0)"));
  TP_TRY(check_extents(M, n, N));
  TP_TRY(check_extents(M, k, 1));
  TP_TRY(check_extents(k, n, 1));
  TP_TRY(need(k % N == 0, TP_ERR_SHAPE, "k must be divisible by the shard count N"));
  if (dtype == TP_BF16) {
    TP_TRY(need((k / N) % 64 == 0, TP_ERR_SHAPE, "bf16 path: k/N must be a multiple of 64"));
    TP_TRY(need(n % 64 == 0, TP_ERR_SHAPE, "bf16 path: n must be a multiple of 64"));
  }
  TP_TRY(check_aligned({Xs, W, residual, out}));
  if (M == 0) return TP_OK;
  const size_t need_bytes = partial_bytes(M, n, N, TP_REDUCE_BUFFERS);
  TP_TRY(need(need_bytes <= kNoAllocScratchBytes, TP_ERR_WORKSPACE,
              "N*M*n*4 bytes of partials exceed the fixed 32 MiB scratch of tp_row_linear_noalloc"));
  TP_TRY(check_device());
  void* scratch = nullptr;
  TP_TRY(noalloc_scratch(&scratch));
  // every partial element the reduction reads is written first by the GEMM, so the
  // previous call's contents need no clearing
  return row_impl(Xs, W, residual, out, M, k, n, N, dtype, TP_REDUCE_BUFFERS, scratch,
                  static_cast<cudaStream_t>(stream));
}

