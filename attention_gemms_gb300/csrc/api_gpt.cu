// C ABI of the vocabulary-parallel embedding / cross-entropy, AdamW, and the small GPT
// composed from them and the tensor-parallel layer
// [Megatron-LM 实战 04 张量并行实现, 核心实现, SmallGPT; 张量并行 notes, §嵌入层的并行化,
//  §损失计算层的并行化].
#include <cuda_runtime.h>

#include <cmath>
#include <vector>

#include "internal.h"

namespace tp {
namespace {

size_t a256(size_t x) { return align_up(x, 256); }

tp_status check_vocab(int64_t M, int64_t v, int64_t h, int32_t N, tp_dtype dt) {
  TP_TRY(check_dtype(dt));
  TP_TRY(need(N >= 1 && M >= 0 && v >= 1 && h >= 1, TP_ERR_INVALID_ARG,
              "need N >= 1, M >= 0, vocab >= 1, h >= 1"));
  return need(v % N == 0, TP_ERR_SHAPE, "the vocabulary size must be divisible by N");
}

// Carving of the GPT workspace: every block 256-byte aligned.
struct GptLayout {
  size_t xs, saved, xf, meanf, rstdf, logits, lse, rows, dxf, dxa, dxb, scratch, total;
  size_t per_layer;            // bytes of one layer's saved state
  size_t off[12];              // offsets of the 12 saved tensors within a layer block
  size_t scratch_bytes;
};

GptLayout gpt_layout(const tp_gpt_config& c, tp_dtype dt, tp_reduce mode) {
  GptLayout L{};
  const int64_t M = c.batch * c.seq, h = c.hidden, f = c.ffn, v = c.vocab;
  const size_t e = elem_size(dt), mh = a256(M * h * e);
  // xn1, mean1, rstd1, qkv, o, lse, x1, xn2, mean2, rstd2, y, hh
  const size_t sizes[12] = {mh, a256(M * 4), a256(M * 4), a256(M * 3 * h * e), mh,
                            a256(c.batch * c.heads * c.seq * 4), mh, mh, a256(M * 4),
                            a256(M * 4), a256(M * f * e), a256(M * f * e)};
  size_t o = 0;
  for (int i = 0; i < 12; ++i) {
    L.off[i] = o;
    o += sizes[i];
  }
  L.per_layer = o;
  size_t p = 0;
  L.xs = p;      p += (c.layers + 1) * mh;
  L.saved = p;   p += c.layers * L.per_layer;
  L.xf = p;      p += mh;
  L.meanf = p;   p += a256(M * 4);
  L.rstdf = p;   p += a256(M * 4);
  L.logits = p;  p += a256(M * v * e);
  L.lse = p;     p += a256(M * 4);
  L.rows = p;    p += a256(M * 4);
  L.dxf = p;     p += mh;
  L.dxa = p;     p += mh;
  L.dxb = p;     p += mh;
  L.scratch = p;
  size_t sc = std::max(layer_workspace_size(true, M, h, f, c.shards, dt, mode),
                       layer_workspace_size(false, M, h, f, c.shards, dt, mode));
  sc = std::max(sc, partial_bytes(M, h, c.shards, mode));   // output layer's dx shard sum
  sc = std::max(sc, layernorm_bwd_ws_bytes(M, h));
  L.scratch_bytes = a256(sc);
  L.total = p + L.scratch_bytes;
  return L;
}

tp_status check_gpt(const tp_gpt_config* c, tp_dtype dt) {
  TP_TRY(need(c != nullptr, TP_ERR_INVALID_ARG, "config is required"));
  TP_TRY(need(dt == TP_F32, TP_ERR_DTYPE, "the GPT step runs in fp32 (the listing's precision)"));
  TP_TRY(need(c->vocab >= 1 && c->hidden >= 1 && c->heads >= 1 && c->ffn >= 1 &&
                  c->layers >= 0 && c->batch >= 0 && c->seq >= 0 && c->shards >= 1,
              TP_ERR_INVALID_ARG, "invalid GPT configuration"));
  TP_TRY(need(c->vocab % c->shards == 0, TP_ERR_SHAPE,
              "the vocabulary size must be divisible by N"));
  return TP_OK;
}

}  // namespace
}  // namespace tp

using namespace tp;

extern "C" {

tp_status tp_vocab_embed_fwd(const int32_t* ids, const void* E, void* x, int64_t M, int64_t vocab,
                             int64_t h, int32_t N, tp_dtype dtype, void* stream) {
  TP_TRY(check_vocab(M, vocab, h, N, dtype));
  TP_TRY(need(ids && E && x, TP_ERR_INVALID_ARG, "ids, E and x are required"));
  TP_TRY(check_aligned({E, x}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_vocab_embed_fwd(ids, E, x, M, vocab, h, N, dtype,
                                static_cast<cudaStream_t>(stream));
}

tp_status tp_vocab_embed_bwd(const int32_t* ids, const void* dx, void* dE, int64_t M,
                             int64_t vocab, int64_t h, int32_t N, int accumulate, tp_dtype dtype,
                             void* stream) {
  TP_TRY(check_vocab(M, vocab, h, N, dtype));
  TP_TRY(need(dE && (M == 0 || (ids && dx)), TP_ERR_INVALID_ARG, "ids, dx and dE are required"));
  TP_TRY(check_aligned({dx, dE}));
  TP_TRY(check_device());
  return launch_vocab_embed_bwd(ids, dx, dE, M, vocab, h, accumulate != 0, dtype,
                                static_cast<cudaStream_t>(stream));
}

tp_status tp_vocab_ce_fwd(const void* logits, const int32_t* targets, float* lse, float* row_loss,
                          float* shard_loss, float* loss, int64_t M, int64_t vocab, int32_t N,
                          tp_dtype dtype, void* stream) {
  TP_TRY(check_vocab(M, vocab, 1, N, dtype));
  TP_TRY(need(logits && targets && lse && row_loss && loss, TP_ERR_INVALID_ARG,
              "logits, targets, lse, row_loss and loss are required"));
  TP_TRY(check_aligned({logits, lse, row_loss, shard_loss, loss}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_vocab_ce_fwd(logits, targets, lse, row_loss, shard_loss, loss, M, vocab, N, dtype,
                             static_cast<cudaStream_t>(stream));
}

tp_status tp_vocab_ce_bwd(const void* logits, const int32_t* targets, const float* lse,
                          void* dlogits, int64_t M, int64_t vocab, int32_t N, float scale,
                          tp_dtype dtype, void* stream) {
  TP_TRY(check_vocab(M, vocab, 1, N, dtype));
  TP_TRY(need(logits && targets && lse && dlogits, TP_ERR_INVALID_ARG,
              "logits, targets, lse and dlogits are required"));
  TP_TRY(check_aligned({logits, lse, dlogits}));
  if (M == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_vocab_ce_bwd(logits, targets, lse, dlogits, M, vocab, scale, dtype,
                             static_cast<cudaStream_t>(stream));
}

tp_status tp_adamw_step(float* p, const float* g, float* m, float* v, int64_t n, int64_t step,
                        float lr, float beta1, float beta2, float eps, float weight_decay,
                        void* stream) {
  TP_TRY(need(p && g && m && v, TP_ERR_INVALID_ARG, "p, g, m and v are required"));
  TP_TRY(need(n >= 0 && step >= 1, TP_ERR_INVALID_ARG, "need n >= 0 and step >= 1"));
  TP_TRY(need(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f && eps > 0.0f,
              TP_ERR_INVALID_ARG, "need 0 <= beta < 1 and eps > 0"));
  if (n == 0) return TP_OK;
  TP_TRY(check_device());
  const float bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta1), static_cast<double>(step)));
  const float bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta2), static_cast<double>(step)));
  return launch_adamw(p, g, m, v, n, lr, beta1, beta2, eps, weight_decay, bc1, bc2,
                      static_cast<cudaStream_t>(stream));
}

tp_status tp_train_step_advance(int32_t* step, const float* loss, float* loss_hist,
                                int64_t hist_len, void* stream) {
  TP_TRY(need(step != nullptr, TP_ERR_INVALID_ARG, "step is required"));
  TP_TRY(need((loss == nullptr) == (loss_hist == nullptr), TP_ERR_INVALID_ARG,
              "loss and loss_hist go together"));
  TP_TRY(need(!loss_hist || hist_len >= 1, TP_ERR_INVALID_ARG, "hist_len must be >= 1"));
  for (const void* q : {static_cast<const void*>(step), static_cast<const void*>(loss),
                        static_cast<const void*>(loss_hist)})
    TP_TRY(need(reinterpret_cast<uintptr_t>(q) % 4 == 0, TP_ERR_ALIGNMENT,
                "step, loss and loss_hist must be 4-byte aligned"));
  TP_TRY(check_device());
  return launch_step_advance(step, loss, loss_hist, hist_len, static_cast<cudaStream_t>(stream));
}

tp_status tp_adamw_step_device(float* p, const float* g, float* m, float* v, int64_t n,
                               const int32_t* step, float lr, float beta1, float beta2, float eps,
                               float weight_decay, void* stream) {
  TP_TRY(need(p && g && m && v && step, TP_ERR_INVALID_ARG, "p, g, m, v and step are required"));
  TP_TRY(need(n >= 0, TP_ERR_INVALID_ARG, "need n >= 0"));
  TP_TRY(need(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f && eps > 0.0f,
              TP_ERR_INVALID_ARG, "need 0 <= beta < 1 and eps > 0"));
  for (const void* q : {static_cast<const void*>(p), static_cast<const void*>(g),
                        static_cast<const void*>(m), static_cast<const void*>(v),
                        static_cast<const void*>(step)})
    TP_TRY(need(reinterpret_cast<uintptr_t>(q) % 4 == 0, TP_ERR_ALIGNMENT,
                "p, g, m, v and step must be 4-byte aligned"));
  if (n == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_adamw_dev(p, g, m, v, n, step, lr, beta1, beta2, eps, weight_decay,
                          static_cast<cudaStream_t>(stream));
}

size_t tp_gpt_workspace_size(const tp_gpt_config* cfg, tp_dtype dtype, tp_reduce mode) {
  if (!cfg || dtype != TP_F32 || cfg->shards < 1 || cfg->vocab % cfg->shards) return 0;
  return gpt_layout(*cfg, dtype, mode).total;
}

tp_status tp_gpt_fwd_bwd(const tp_gpt_config* cfg, const tp_gpt_weights* w, const tp_gpt_grads* g,
                         const int32_t* ids, const int32_t* targets, float* loss, tp_dtype dtype,
                         tp_reduce mode, void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_gpt(cfg, dtype));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(w && g && w->E && w->gammaf && w->betaf && g->dE && g->dgammaf && g->dbetaf &&
                  (cfg->layers == 0 || (w->layers && g->layers)),
              TP_ERR_INVALID_ARG, "weights, gradients and their tensors are required"));
  TP_TRY(need(ids && targets && loss, TP_ERR_INVALID_ARG, "ids, targets and loss are required"));
  const tp_gpt_config& c = *cfg;
  const int64_t M = c.batch * c.seq, h = c.hidden, f = c.ffn, v = c.vocab;
  const int32_t N = c.shards;
  if (M == 0) return TP_OK;
  const GptLayout L = gpt_layout(c, dtype, mode);
  TP_TRY(need(ws && ws_bytes >= L.total, TP_ERR_WORKSPACE,
              "workspace smaller than tp_gpt_workspace_size"));
  TP_TRY(check_aligned({ws, w->E, g->dE}));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(ws);
  const size_t mh = a256(M * h * elem_size(dtype));
  auto xs = [&](int64_t l) { return static_cast<void*>(base + L.xs + l * mh); };
  std::vector<tp_layer_saved> sv(c.layers);
  for (int64_t l = 0; l < c.layers; ++l) {
    char* q = base + L.saved + l * L.per_layer;
    sv[l] = tp_layer_saved{q + L.off[0], reinterpret_cast<float*>(q + L.off[1]),
                           reinterpret_cast<float*>(q + L.off[2]), q + L.off[3], q + L.off[4],
                           reinterpret_cast<float*>(q + L.off[5]), q + L.off[6], q + L.off[7],
                           reinterpret_cast<float*>(q + L.off[8]),
                           reinterpret_cast<float*>(q + L.off[9]), q + L.off[10], q + L.off[11]};
  }
  void* xf = base + L.xf;
  float* meanf = reinterpret_cast<float*>(base + L.meanf);
  float* rstdf = reinterpret_cast<float*>(base + L.rstdf);
  void* logits = base + L.logits;
  float* lse = reinterpret_cast<float*>(base + L.lse);
  float* rows = reinterpret_cast<float*>(base + L.rows);
  void* dxf = base + L.dxf;
  void* dxa = base + L.dxa;
  void* dxb = base + L.dxb;
  void* scratch = base + L.scratch;
  const size_t sb = L.scratch_bytes;

  // ---- forward
  TP_TRY(tp_vocab_embed_fwd(ids, w->E, xs(0), M, v, h, N, dtype, stream));
  for (int64_t l = 0; l < c.layers; ++l)
    TP_TRY(tp_layer_fwd(xs(l), &w->layers[l], &sv[l], xs(l + 1), c.batch, c.seq, h, f,
                        static_cast<int32_t>(c.heads), N, 0, dtype, mode, scratch, sb, stream));
  TP_TRY(launch_layernorm_fwd(xs(c.layers), w->gammaf, w->betaf, xf, meanf, rstdf, M, h, 1e-5f,
                              dtype, st));
  {  // output layer, column-parallel over the vocabulary: logits_i = x_f E_i^T
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = v;
    d.K = h;
    d.A[0] = {xf, M, h, h};
    d.B[0] = {w->E, v, h, h};  // E (v, h) read as B(k = h, n = v): K-major
    d.ldo = v;
    d.shards = N;
    d.shard_axis = 1;
    d.epi = EPI_STORE;
    d.out[0] = logits;
    d.out_f32 = dtype == TP_F32;
    TP_TRY(launch_gemm(d, st));
  }
  TP_TRY(launch_vocab_ce_fwd(logits, targets, lse, rows, nullptr, loss, M, v, N, dtype, st));

  // ---- backward
  TP_TRY(launch_vocab_ce_bwd(logits, targets, lse, logits, M, v, 1.0f / static_cast<float>(M),
                             dtype, st));
  // dx_f = sum_i dlogits_i E_i: the output layer's input gradient, summed over the shards
  TP_TRY(row_impl(logits, w->E, nullptr, dxf, M, v, h, N, dtype, mode, scratch, st));
  {  // dE = dlogits^T x_f (shard i: its rows of dE)
    GemmDesc d;
    d.dtype = dtype;
    d.M = v;
    d.N = h;
    d.K = M;
    d.a_mn = true;
    d.A[0] = {logits, M, v, v};  // dlogits (M, v) read as A(m = v, k = M): MN-major
    d.B[0] = {xf, M, h, h};      // x_f (M, h) = B(k = M, n = h)
    d.b_mn = true;
    d.ldo = h;
    d.epi = EPI_STORE;
    d.out[0] = g->dE;
    d.out_f32 = dtype == TP_F32;
    TP_TRY(launch_gemm(d, st));
  }
  TP_TRY(launch_layernorm_bwd(xs(c.layers), w->gammaf, meanf, rstdf, dxf, nullptr, dxa,
                              g->dgammaf, g->dbetaf, M, h, scratch, dtype, st));
  void* cur = dxa;
  void* nxt = dxb;
  for (int64_t l = c.layers - 1; l >= 0; --l) {
    TP_TRY(tp_layer_bwd(xs(l), &w->layers[l], &sv[l], cur, nxt, &g->layers[l], c.batch, c.seq,
                        h, f, static_cast<int32_t>(c.heads), N, 0, dtype, mode, scratch, sb,
                        stream));
    std::swap(cur, nxt);
  }
  // the embedding's gradient added to the output layer's (shared weight)
  return launch_vocab_embed_bwd(ids, cur, g->dE, M, v, h, true, dtype, st);
}

}  // extern "C"
