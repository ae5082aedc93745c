// C ABI of the sequence-parallel pre-LN MLP sub-block: the LN / residual region split
// over the ranks along the sequence, the all-reduce after the row-parallel GEMM split
// into reduce-scatter + all-gather [20260402-parallelism, §5 Sequence Parallelism].
//
// All ranks are virtual ranks of one GPU, and each rank's rows are one contiguous
// block of the same buffer, in rank order. So the all-gather of the ranks' LN outputs
// (forward) and of dout (backward) is the buffer itself, and the reduce-scatter is the
// shard sum, of which each rank owns its rows (the split-K fold or the fp32-partials
// reduction, with the residual rows added in the same pass). What is rank-specific is
// the LN parameter gradient: each rank's gamma / beta see only its rows, so their
// gradients are summed per rank and then over the ranks.
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace tp {
namespace {

tp_status check_sp(int64_t M, int32_t N, tp_act act, tp_reduce mode, tp_dtype dt) {
  TP_TRY(check_dtype(dt));
  TP_TRY(need(act == TP_ACT_GELU || act == TP_ACT_SWIGLU, TP_ERR_INVALID_ARG,
              "MLP act must be TP_ACT_GELU or TP_ACT_SWIGLU"));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(N >= 1 && M >= 0, TP_ERR_INVALID_ARG, "need N >= 1 and M >= 0"));
  return need(M % N == 0, TP_ERR_SHAPE,
              "sequence parallelism: the rows M must split evenly over the N ranks");
}

size_t a256(size_t x) { return align_up(x, 256); }

size_t mlp_fwd_ws(int64_t M, int64_t h, int32_t N, tp_reduce mode) {
  return partial_bytes(M, h, N, mode);  // H is a caller buffer here
}

size_t mlp_bwd_ws(int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt, tp_act act,
                  tp_reduce mode) {
  return (act == TP_ACT_SWIGLU ? 2 : 1) * a256(static_cast<size_t>(M) * f * elem_size(dt)) +
         partial_bytes(M, h, N, mode);
}

}  // namespace

size_t sp_mlp_workspace_size(bool fwd, int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt,
                             tp_act act, tp_reduce mode) {
  if (M % N) return 0;
  if (fwd) return mlp_fwd_ws(M, h, N, mode);
  // dxn (the reduce-scattered MLP input gradient), then the MLP backward's scratch,
  // reused afterwards for the per-rank LN parameter partials
  return a256(static_cast<size_t>(M) * h * elem_size(dt)) +
         std::max(mlp_bwd_ws(M, h, f, N, dt, act, mode), layernorm_bwd_ws_bytes(M, h, N));
}

}  // namespace tp

using namespace tp;

extern "C" {

tp_status tp_sp_mlp_fwd(const void* x, const float* gamma, const float* beta, const void* W1,
                        const void* W1_up, const void* W2, void* xn, float* mean, float* rstd,
                        void* Y, void* Y_up, void* H, void* out, int64_t M, int64_t h, int64_t f,
                        int32_t N, tp_dtype dtype, tp_act act, tp_reduce mode, void* ws,
                        size_t ws_bytes, void* stream) {
  TP_TRY(check_sp(M, N, act, mode, dtype));
  TP_TRY(need(x && gamma && beta && xn && mean && rstd && H && out, TP_ERR_INVALID_ARG,
              "x, gamma, beta, xn, mean, rstd, H and out are required"));
  TP_TRY(check_aligned({x, gamma, beta, xn, mean, rstd}));
  TP_TRY(check_mlp_shape(M, h, f, N, dtype));
  if (M == 0) return TP_OK;
  TP_TRY(need(ws_bytes >= mlp_fwd_ws(M, h, N, mode) && (mode == TP_REDUCE_SPLITK || ws),
              TP_ERR_WORKSPACE, "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  // LN on each rank's rows (rows are independent: one launch covers every rank)
  TP_TRY(launch_layernorm_fwd(x, gamma, beta, xn, mean, rstd, M, h, 1e-5f, dtype,
                              static_cast<cudaStream_t>(stream)));
  // all-gather = the adjacent rank blocks of xn; the TP MLP; reduce-scatter + x_r
  return tp_mlp_fwd(xn, W1, W1_up, W2, x, Y, Y_up, H, out, M, h, f, N, dtype, act, mode, ws,
                    ws_bytes, TP_W_IN_OUT, stream);
}

tp_status tp_sp_mlp_bwd(const void* x, const float* gamma, const void* W1, const void* W1_up,
                        const void* W2, const void* xn, const float* mean, const float* rstd,
                        const void* Y, const void* Y_up, const void* H, const void* dout,
                        void* dx, float* dgamma, float* dbeta, float* dgamma_ranks,
                        float* dbeta_ranks, void* dW1, void* dW1_up, void* dW2, int64_t M,
                        int64_t h, int64_t f, int32_t N, tp_dtype dtype, tp_act act,
                        tp_reduce mode, void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_sp(M, N, act, mode, dtype));
  TP_TRY(need(x && gamma && xn && mean && rstd && dout && dx && dgamma && dbeta,
              TP_ERR_INVALID_ARG, "x, gamma, xn, mean, rstd, dout, dx, dgamma and dbeta are required"));
  TP_TRY(check_aligned({x, gamma, xn, mean, rstd, dout, dx, dgamma, dbeta, dgamma_ranks,
                        dbeta_ranks, ws}));
  TP_TRY(check_mlp_shape(M, h, f, N, dtype));
  if (M == 0) return TP_OK;
  const size_t need_ws = sp_mlp_workspace_size(false, M, h, f, N, dtype, act, mode);
  TP_TRY(need(ws_bytes >= need_ws && ws, TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  char* p = static_cast<char*>(ws);
  void* dxn = p;
  char* rest = p + a256(static_cast<size_t>(M) * h * elem_size(dtype));
  const size_t rest_bytes = ws_bytes - (rest - p);
  // all-gather of dout (the buffer itself) -> MLP backward -> reduce-scatter of dX
  TP_TRY(tp_mlp_bwd(xn, W1, W1_up, W2, Y, Y_up, H, dout, dxn, dW1, dW1_up, dW2, M, h, f, N,
                    dtype, act, mode, rest, rest_bytes, TP_W_IN_OUT, stream));
  // LN backward on each rank's rows + the residual's dout_r; LN parameter gradients
  // per rank, then summed over the ranks
  return launch_layernorm_bwd_ranks(x, gamma, mean, rstd, dxn, dout, dx, dgamma, dbeta,
                                    dgamma_ranks, dbeta_ranks, M, h, N, rest, dtype,
                                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"
