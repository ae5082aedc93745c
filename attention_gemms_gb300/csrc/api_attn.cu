// C ABI of the head-sharded attention block, LayerNorm and the pre-LN transformer
// layer built from them and from the tensor-parallel MLP.
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace tp {
namespace {

tp_status check_attn_shape(int64_t b, int64_t s, int64_t h, int32_t heads, int32_t N,
                           tp_dtype dt) {
  TP_TRY(need(b >= 0 && s >= 0 && h >= 1 && heads >= 1 && N >= 1, TP_ERR_INVALID_ARG,
              "need b, s >= 0 and h, n_heads, N >= 1"));
  TP_TRY(need(b < (int64_t(1) << 31) && s < (int64_t(1) << 31), TP_ERR_SHAPE, "b or s too large"));
  TP_TRY(check_extents(b * s, 3 * h, N));
  TP_TRY(need(h % heads == 0, TP_ERR_SHAPE, "h must be divisible by n_heads"));
  // heads are split across shards: TP degree <= heads and heads % N == 0
  TP_TRY(need(heads % N == 0, TP_ERR_SHAPE, "n_heads must be divisible by the shard count N"));
  const int64_t d = h / heads;
  TP_TRY(need(d == 16 || d == 32 || d == 64, TP_ERR_SHAPE, "head_dim must be 16, 32 or 64"));
  if (dt == TP_BF16)
    TP_TRY(need((h / N) % 64 == 0, TP_ERR_SHAPE, "bf16 path: h/N must be a multiple of 64"));
  return TP_OK;
}

size_t a256(size_t x) { return align_up(x, 256); }

// dO | dQKV | dxn | shard partials | LN scratch | attention (lse, D) pairs: 8 bytes per
// (row, head), at most h / 16 heads (head_dim >= 16)
size_t attn_bwd_ws(int64_t M, int64_t h, int32_t N, tp_dtype dt, tp_reduce mode) {
  const size_t e = elem_size(dt);
  return a256(M * h * e) + a256(M * 3 * h * e) + a256(M * h * e) +
         a256(partial_bytes(M, h, N, mode)) + a256(layernorm_bwd_ws_bytes(M, h)) +
         a256(attention_bwd_tc_ws_bytes(M, 1, static_cast<int>(h / 16)));
}

// QKV = xn W_qkv (all shards' columns; shard i owns its heads' columns of W_q, W_k, W_v)
tp_status qkv_fwd(const void* xn, const void* Wqkv, void* qkv, int64_t M, int64_t h, tp_dtype dt,
                  cudaStream_t st) {
  GemmDesc d;
  d.dtype = dt;
  d.M = M;
  d.N = 3 * h;
  d.K = h;
  d.A[0] = {xn, M, h, h};
  d.B[0] = {Wqkv, h, 3 * h, 3 * h};
  d.b_mn = true;
  d.ldo = 3 * h;
  d.epi = EPI_STORE;
  d.out[0] = qkv;
  d.out_f32 = dt == TP_F32;
  return launch_gemm(d, st);
}

}  // namespace

size_t attn_workspace_size(bool fwd, int64_t M, int64_t h, int32_t N, tp_dtype dt,
                           tp_reduce mode) {
  return fwd ? partial_bytes(M, h, N, mode) : attn_bwd_ws(M, h, N, dt, mode);
}

size_t layer_workspace_size(bool fwd, int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt,
                            tp_reduce mode) {
  const size_t e = elem_size(dt);
  if (fwd) return partial_bytes(M, h, N, mode);
  const size_t mlp = a256(M * f * e) + partial_bytes(M, h, N, mode);
  const size_t rest = std::max(std::max(mlp, a256(layernorm_bwd_ws_bytes(M, h))),
                               attn_bwd_ws(M, h, N, dt, mode));
  return 2 * a256(M * h * e) + rest;
}

// Validation and the part of the attention block before W_o: LN1, QKV, attention.
tp_status attn_core_fwd(const void* x, const float* gamma, const float* beta, const void* Wqkv,
                        const void* Wo, void* xn, float* mean, float* rstd, void* qkv, void* o,
                        float* lse, void* out, int64_t b, int64_t s, int64_t h, int32_t n_heads,
                        int32_t N, int causal, tp_dtype dtype, tp_reduce mode, void* ws,
                        size_t ws_bytes, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(x && gamma && beta && Wqkv && Wo && xn && mean && rstd && qkv && o && lse && out,
              TP_ERR_INVALID_ARG, "all tensors of tp_attn_proj_fwd are required"));
  TP_TRY(check_attn_shape(b, s, h, n_heads, N, dtype));
  TP_TRY(check_aligned({x, gamma, beta, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, ws}));
  const int64_t M = b * s;
  if (M == 0) return TP_OK;
  const size_t need_ws = partial_bytes(M, h, N, mode);
  TP_TRY(need(ws_bytes >= need_ws && (need_ws == 0 || ws), TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // LN needs the whole hidden width: every shard holds the full x (replicated)
  TP_TRY(launch_layernorm_fwd(x, gamma, beta, xn, mean, rstd, M, h, 1e-5f, dtype, st));
  TP_TRY(qkv_fwd(xn, Wqkv, qkv, M, h, dtype, st));
  return launch_attention_fwd(qkv, o, lse, b, s, h, n_heads, causal, dtype, st);
}

}  // namespace tp

using namespace tp;

extern "C" {

tp_status tp_layernorm_fwd(const void* x, const float* gamma, const float* beta, void* y,
                           float* mean, float* rstd, int64_t M, int64_t h, float eps,
                           tp_dtype dtype, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(x && gamma && beta && y, TP_ERR_INVALID_ARG, "x, gamma, beta and y are required"));
  TP_TRY(need(M >= 0 && h >= 1 && eps >= 0.0f, TP_ERR_INVALID_ARG, "need M >= 0, h >= 1, eps >= 0"));
  TP_TRY(check_aligned({x, gamma, beta, y, mean, rstd}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_layernorm_fwd(x, gamma, beta, y, mean, rstd, M, h, eps, dtype,
                              static_cast<cudaStream_t>(stream));
}

tp_status tp_layernorm_bwd(const void* x, const float* gamma, const float* mean,
                           const float* rstd, const void* dy, const void* dres, void* dx,
                           float* dgamma, float* dbeta, int64_t M, int64_t h, tp_dtype dtype,
                           void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(x && gamma && mean && rstd && dy && dx, TP_ERR_INVALID_ARG,
              "x, gamma, mean, rstd, dy and dx are required"));
  TP_TRY(need(M >= 0 && h >= 1, TP_ERR_INVALID_ARG, "need M >= 0, h >= 1"));
  TP_TRY(check_aligned({x, gamma, mean, rstd, dy, dres, dx, dgamma, dbeta, ws}));
  if (M == 0) return TP_OK;
  const size_t need_ws = (dgamma || dbeta) ? layernorm_bwd_ws_bytes(M, h) : 0;
  TP_TRY(need(ws_bytes >= need_ws && (need_ws == 0 || ws), TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  return launch_layernorm_bwd(x, gamma, mean, rstd, dy, dres, dx, dgamma, dbeta, M, h, ws, dtype,
                              static_cast<cudaStream_t>(stream));
}

tp_status tp_attn_proj_fwd(const void* x, const float* gamma, const float* beta, const void* Wqkv,
                           const void* Wo, void* xn, float* mean, float* rstd, void* qkv, void* o,
                           float* lse, void* out, int64_t b, int64_t s, int64_t h,
                           int32_t n_heads, int32_t N, int causal, tp_dtype dtype, tp_reduce mode,
                           void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(attn_core_fwd(x, gamma, beta, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, b, s, h,
                       n_heads, N, causal, dtype, mode, ws, ws_bytes, stream));
  if (b * s == 0) return TP_OK;
  // shard i's O_i feeds row block i of W_o directly (no gather); sum + residual
  return row_impl(o, Wo, x, out, b * s, h, h, N, dtype, mode, ws,
                  static_cast<cudaStream_t>(stream));
}

tp_status tp_attn_proj_bwd(const void* x, const float* gamma, const void* Wqkv, const void* Wo,
                           const void* xn, const float* mean, const float* rstd, const void* qkv,
                           const void* o, const float* lse, const void* dout, void* dx,
                           float* dgamma, float* dbeta, void* dWqkv, void* dWo, int64_t b,
                           int64_t s, int64_t h, int32_t n_heads, int32_t N, int causal,
                           tp_dtype dtype, tp_reduce mode, void* ws, size_t ws_bytes,
                           void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(x && gamma && Wqkv && Wo && xn && mean && rstd && qkv && o && lse && dout && dx &&
                  dgamma && dbeta && dWqkv && dWo,
              TP_ERR_INVALID_ARG, "all tensors of tp_attn_proj_bwd are required"));
  TP_TRY(check_attn_shape(b, s, h, n_heads, N, dtype));
  TP_TRY(check_aligned({x, gamma, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dgamma,
                        dbeta, dWqkv, dWo, ws}));
  const int64_t M = b * s;
  if (M == 0) return TP_OK;
  TP_TRY(need(ws_bytes >= attn_bwd_ws(M, h, N, dtype, mode) && ws, TP_ERR_WORKSPACE,
              "workspace smaller than tp_workspace_size"));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dtype);
  char* w = static_cast<char*>(ws);
  void* dO = w;
  w += a256(M * h * e);
  void* dqkv = w;
  w += a256(M * 3 * h * e);
  void* dxn = w;
  w += a256(M * h * e);
  void* parts = w;
  w += a256(partial_bytes(M, h, N, mode));
  void* lnws = w;
  w += a256(layernorm_bwd_ws_bytes(M, h));
  void* ldws = w;
  // The weight gradients are off the critical path: dW_o runs on a side stream beside
  // dO and the attention backward, dW_qkv beside dx_n and the LayerNorm backward.
  SideBranch br(st);

  // dWo_i = O_i^T dout (row-parallel weight gradient; row block i of W_o)
  {
    GemmDesc d;
    d.dtype = dtype;
    d.M = h;
    d.N = h;
    d.K = M;
    d.A[0] = {o, M, h, h};
    d.a_mn = true;
    d.B[0] = {dout, M, h, h};
    d.b_mn = true;
    d.ldo = h;
    d.epi = EPI_STORE;
    d.out[0] = dWo;
    d.out_f32 = dtype == TP_F32;
    d.shards = N;
    d.shard_axis = 0;
    TP_TRY(launch_gemm(d, br.stream()));
  }
  // dO_i = dout W_o,i^T (g-backward is the identity: every shard reads all of dout)
  {
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = h;
    d.K = h;
    d.A[0] = {dout, M, h, h};
    d.B[0] = {Wo, h, h, h};  // W_o (h, h) read as B(k = out, n = in): K-major
    d.ldo = h;
    d.epi = EPI_STORE;
    d.out[0] = dO;
    d.out_f32 = dtype == TP_F32;
    d.shards = N;
    d.shard_axis = 1;
    TP_TRY(launch_gemm(d, st));
  }
  TP_TRY(launch_attention_bwd(qkv, o, lse, dO, dqkv, ldws, b, s, h, n_heads, causal, dtype, st));
  // dW_qkv = xn^T dQKV (column-parallel weight gradient), once dQKV is complete
  TP_TRY(br.fork());
  {
    GemmDesc d;
    d.dtype = dtype;
    d.M = h;
    d.N = 3 * h;
    d.K = M;
    d.A[0] = {xn, M, h, h};
    d.a_mn = true;
    d.B[0] = {dqkv, M, 3 * h, 3 * h};
    d.b_mn = true;
    d.ldo = 3 * h;
    d.epi = EPI_STORE;
    d.out[0] = dWqkv;
    d.out_f32 = dtype == TP_F32;
    TP_TRY(launch_gemm(d, br.stream()));
  }
  // f-backward: dxn = sum_i dQKV_i W_qkv,i^T. Shard i's K range is its heads' columns
  // of the Q, K and V blocks: three K segments at offsets 0, h, 2h.
  {
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = h;
    d.ldo = h;
    d.epi = EPI_STORE;
    if (mode == TP_REDUCE_SPLITK) {
      d.K = 3 * h;
      d.A[0] = {dqkv, M, 3 * h, 3 * h};
      d.B[0] = {Wqkv, h, 3 * h, 3 * h};
      d.out[0] = dxn;
      d.out_f32 = dtype == TP_F32;
      TP_TRY(launch_gemm(d, st));
    } else {
      d.K = h / N;
      d.groups = N;
      d.nseg = 3;
      for (int sg = 0; sg < 3; ++sg) {
        d.A[sg] = {dqkv, M, 3 * h, 3 * h};
        d.B[sg] = {Wqkv, h, 3 * h, 3 * h};
        d.seg_k0[sg] = sg * h;
      }
      d.out[0] = parts;
      d.out_f32 = true;
      d.out_group_stride = M * h;
      TP_TRY(launch_gemm(d, st));
      TP_TRY(launch_shard_reduce(static_cast<const float*>(parts), nullptr, dxn, N, M, h, dtype,
                                 st));
    }
  }
  // LN backward plus the residual branch: dx = dout + LN'(dxn)
  TP_TRY(launch_layernorm_bwd(x, gamma, mean, rstd, dxn, dout, dx, dgamma, dbeta, M, h, lnws,
                              dtype, st));
  return br.join();
}

tp_status tp_layer_fwd(const void* x, const tp_layer_weights* w, const tp_layer_saved* sv,
                       void* out, int64_t b, int64_t s, int64_t h, int64_t f, int32_t n_heads,
                       int32_t N, int causal, tp_dtype dtype, tp_reduce mode, void* ws,
                       size_t ws_bytes, void* stream) {
  TP_TRY(need(w && sv, TP_ERR_INVALID_ARG, "weights and saved-state structs are required"));
  TP_TRY(need(sv->x1 && sv->xn2 && sv->mean2 && sv->rstd2 && sv->y && sv->hh, TP_ERR_INVALID_ARG,
              "saved x1, xn2, mean2, rstd2, y and hh are required"));
  TP_TRY(need(ws_bytes >= layer_workspace_size(true, b * s, h, f, N, dtype, mode) ||
                  b * s == 0,
              TP_ERR_WORKSPACE, "workspace smaller than tp_workspace_size"));
  // x1 = x + sum_i O_i W_o,i  with O from LN1(x); then xn2 = LN2(x1). The sum and
  // LN2 run as one pass over the shard partials (buffers mode) or the split-K GEMM
  // followed by LN2.
  TP_TRY(need(w->gamma2 && w->beta2, TP_ERR_INVALID_ARG, "gamma2 and beta2 are required"));
  TP_TRY(need(h % 8 == 0 && h <= kReduceLnMaxH, TP_ERR_SHAPE,
              "layer: h must be a multiple of 8 and at most 16384"));
  TP_TRY(check_aligned({w->gamma2, w->beta2, sv->x1, sv->xn2, sv->mean2, sv->rstd2}));
  TP_TRY(attn_core_fwd(x, w->gamma1, w->beta1, w->Wqkv, w->Wo, sv->xn1, sv->mean1, sv->rstd1,
                       sv->qkv, sv->o, sv->lse, sv->x1, b, s, h, n_heads, N, causal, dtype, mode,
                       ws, ws_bytes, stream));
  if (b * s > 0)
    TP_TRY(row_ln_impl(sv->o, w->Wo, x, w->gamma2, w->beta2, sv->x1, sv->xn2, sv->mean2,
                       sv->rstd2, b * s, h, h, N, 1e-5f, dtype, mode, ws,
                       static_cast<cudaStream_t>(stream)));
  // out = x1 + sum_i GELU(xn2 W1_i) W2_i
  return tp_mlp_fwd(sv->xn2, w->W1, nullptr, w->W2, sv->x1, sv->y, nullptr, sv->hh, out, b * s,
                    h, f, N, dtype, TP_ACT_GELU, mode, ws, ws_bytes, TP_W_IN_OUT, stream);
}

tp_status tp_layer_bwd(const void* x, const tp_layer_weights* w, const tp_layer_saved* sv,
                       const void* dout, void* dx, const tp_layer_grads* g, int64_t b, int64_t s,
                       int64_t h, int64_t f, int32_t n_heads, int32_t N, int causal,
                       tp_dtype dtype, tp_reduce mode, void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(w && sv && g, TP_ERR_INVALID_ARG, "weights, saved-state and grads structs are required"));
  TP_TRY(need(dout && dx && g->dgamma2 && g->dbeta2, TP_ERR_INVALID_ARG,
              "dout, dx, dgamma2 and dbeta2 are required"));
  TP_TRY(need(b >= 0 && s >= 0 && h >= 1 && f >= 1, TP_ERR_INVALID_ARG, "sizes must be positive"));
  const int64_t M = b * s;
  if (M == 0) return TP_OK;
  const size_t need_ws = layer_workspace_size(false, M, h, f, N, dtype, mode);
  TP_TRY(need(ws_bytes >= need_ws && ws, TP_ERR_WORKSPACE, "workspace smaller than tp_workspace_size"));
  TP_TRY(check_aligned({ws}));
  const size_t e = elem_size(dtype);
  char* p = static_cast<char*>(ws);
  void* dxn2 = p;
  void* dx1 = p + a256(M * h * e);
  char* rest = p + 2 * a256(M * h * e);
  const size_t rest_bytes = ws_bytes - 2 * a256(M * h * e);
  TP_TRY(tp_mlp_bwd(sv->xn2, w->W1, nullptr, w->W2, sv->y, nullptr, sv->hh, dout, dxn2, g->dW1,
                    nullptr, g->dW2, M, h, f, N, dtype, TP_ACT_GELU, mode, rest, rest_bytes,
                    TP_W_IN_OUT, stream));
  TP_TRY(tp_layernorm_bwd(sv->x1, w->gamma2, sv->mean2, sv->rstd2, dxn2, dout, dx1, g->dgamma2,
                          g->dbeta2, M, h, dtype, rest, rest_bytes, stream));
  return tp_attn_proj_bwd(x, w->gamma1, w->Wqkv, w->Wo, sv->xn1, sv->mean1, sv->rstd1, sv->qkv,
                          sv->o, sv->lse, dx1, dx, g->dgamma1, g->dbeta1, g->dWqkv, g->dWo, b, s,
                          h, n_heads, N, causal, dtype, mode, rest, rest_bytes, stream);
}

}  // extern "C"
