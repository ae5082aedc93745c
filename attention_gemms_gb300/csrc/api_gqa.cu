// C ABI of the head-sharded grouped-query attention block [张量并行 notes, §相关分析:
// the tensor-parallel degree may reach the number of query heads when key/value heads
// are fewer, provided the key/value heads stay consistent across the shards].
//
// Sharded weight layout (the per-rank column-parallel QKV of the Megatron-LM 实战 04
// page, whose output is reshaped to [3, heads_per_rank, head_dim]): shard i owns one
// block of S = (hq + 2 hkv) d columns, [W_q of its hq query heads | W_k of its hkv
// key/value heads | W_v of the same], blocks in shard order. hq = H / N; hkv = Hkv / N
// when N <= Hkv, else 1 and each key/value head has r = N / Hkv replicas (one per shard
// of its group). Every shard's block has the same width, so the column-parallel
// projection, the row-parallel input gradient (N K-groups of S columns) and the weight
// gradient are plain engine GEMMs. After the weight gradient the replicas of each
// key/value head add their copies (in replica order) and all take the sum: the
// all-reduce that keeps the copies equal.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace tp {
namespace {

size_t a256(size_t x) { return align_up(x, 256); }

struct Gqa {
  int hq, hkv, r;   // per shard; replication factor
  int64_t d, S, W;  // head dim, block width, all blocks' width
};

tp_status gqa_shape(int64_t h, int32_t H, int32_t Hkv, int32_t N, tp_dtype dt, Gqa* g) {
  TP_TRY(need(h >= 1 && H >= 1 && Hkv >= 1 && N >= 1, TP_ERR_INVALID_ARG,
              "need h, n_heads, n_kv_heads, N >= 1"));
  TP_TRY(need(h % H == 0, TP_ERR_SHAPE, "h must be divisible by n_heads"));
  TP_TRY(need(H % Hkv == 0, TP_ERR_SHAPE, "n_heads must be divisible by n_kv_heads"));
  TP_TRY(need(H % N == 0, TP_ERR_SHAPE, "n_heads must be divisible by N (N <= n_heads)"));
  TP_TRY(need(N <= Hkv ? Hkv % N == 0 : N % Hkv == 0, TP_ERR_SHAPE,
              "N must divide n_kv_heads, or be a multiple of it (replicated key/value heads)"));
  g->d = h / H;
  TP_TRY(need(g->d == 16 || g->d == 32 || g->d == 64, TP_ERR_SHAPE,
              "head_dim must be 16, 32 or 64"));
  g->hq = H / N;
  g->hkv = N <= Hkv ? Hkv / N : 1;
  g->r = N <= Hkv ? 1 : N / Hkv;
  g->S = static_cast<int64_t>(g->hq + 2 * g->hkv) * g->d;
  g->W = N * g->S;
  if (dt == TP_BF16) {
    TP_TRY(need(g->S % 64 == 0, TP_ERR_SHAPE,
                "bf16 path: each shard's QKV block ((hq + 2 hkv) * head_dim) must be a multiple of 64"));
    TP_TRY(need((h / N) % 64 == 0, TP_ERR_SHAPE, "bf16 path: h/N must be a multiple of 64"));
  }
  return TP_OK;
}

template <typename T>
__global__ void gqa_pack_kernel(const T* __restrict__ Wq, const T* __restrict__ Wk,
                                const T* __restrict__ Wv, T* __restrict__ Wsh, int64_t h, int H,
                                int Hkv, int hq, int hkv, int r, int d, int64_t S, int64_t W) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t n = h * W;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = e / W, col = e - row * W;
    const int64_t i = col / S, c = col - i * S;
    T v;
    if (c < static_cast<int64_t>(hq) * d) {
      v = Wq[row * H * d + i * hq * d + c];
    } else {
      const int64_t ck = c - static_cast<int64_t>(hq) * d;
      const bool is_k = ck < static_cast<int64_t>(hkv) * d;
      const int64_t cc = is_k ? ck : ck - static_cast<int64_t>(hkv) * d;
      const int64_t head = (r == 1 ? i * hkv : i / r) + cc / d;
      v = (is_k ? Wk : Wv)[row * Hkv * d + head * d + cc % d];
    }
    Wsh[e] = v;
  }
}

// the replicas of each key/value head (shards j r .. j r + r - 1) sum their K and V
// gradient columns in replica order and all store the sum
template <typename T>
__global__ void gqa_replica_sum_kernel(T* __restrict__ dW, int64_t h, int Hkv, int hq, int r,
                                       int d, int64_t S, int64_t W) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t per_row = static_cast<int64_t>(Hkv) * 2 * d;
  const int64_t n = h * per_row;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = e / per_row, k = e - row * per_row;
    const int64_t j = k / (2 * d), kk = k - j * 2 * d;  // kk < d: K, else V (hkv = 1 per block)
    const int64_t off = static_cast<int64_t>(hq) * d + kk;
    float sum = 0.0f;
    for (int q = 0; q < r; ++q) {
      const T* p = dW + row * W + (j * r + q) * S + off;
      sum += static_cast<float>(*p);
    }
    for (int q = 0; q < r; ++q) dW[row * W + (j * r + q) * S + off] = static_cast<T>(sum);
  }
}

// The same sum moving 16 bytes (8 bf16 or 4 fp32 columns) per access: d, S and W are
// multiples of 16 columns and dW is 16-byte aligned, so every vector is aligned.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4& r, float (&f)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  } else {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
}
template <typename T>
__device__ __forceinline__ uint4 pack16(const float (&f)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 2) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&t);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
}

template <typename T>
__global__ void gqa_replica_sum_vec_kernel(T* __restrict__ dW, int64_t h, int Hkv, int hq, int r,
                                           int d, int64_t S, int64_t W) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  constexpr int E = 16 / sizeof(T);
  const int dv = d / E;
  const int64_t per_row = static_cast<int64_t>(Hkv) * 2 * dv;
  const int64_t n = h * per_row;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = e / per_row, k = e - row * per_row;
    const int64_t j = k / (2 * dv), kk = (k - j * 2 * dv) * E;  // kk < d: K, else V
    const int64_t off = static_cast<int64_t>(hq) * d + kk;
    float sum[E];
#pragma unroll
    for (int i = 0; i < E; ++i) sum[i] = 0.0f;
    for (int q = 0; q < r; ++q) {
      float f[E];
      unpack16<T>(*reinterpret_cast<const uint4*>(dW + row * W + (j * r + q) * S + off), f);
#pragma unroll
      for (int i = 0; i < E; ++i) sum[i] += f[i];
    }
    const uint4 v = pack16<T>(sum);
    for (int q = 0; q < r; ++q) *reinterpret_cast<uint4*>(dW + row * W + (j * r + q) * S + off) = v;
  }
}

unsigned grid_for(int64_t n) {
  return static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256,
                                                                     8ll * device_sm_count())));
}

size_t fwd_ws(int64_t M, int64_t h, int32_t N, tp_reduce mode) { return partial_bytes(M, h, N, mode); }

size_t bwd_ws(int64_t M, int64_t h, const Gqa& g, int32_t N, tp_dtype dt, tp_reduce mode) {
  const size_t e = elem_size(dt);
  return a256(M * h * e) + a256(M * g.W * e) + a256(M * h * e) +
         a256(partial_bytes(M, h, N, mode)) + a256(layernorm_bwd_ws_bytes(M, h)) +
         a256(attention_bwd_tc_ws_bytes(M, 1, static_cast<int>(h / g.d)));
}

}  // namespace
}  // namespace tp

using namespace tp;

extern "C" {

int64_t tp_gqa_qkv_cols(int64_t h, int32_t n_heads, int32_t n_kv_heads, int32_t N) {
  Gqa g;
  if (gqa_shape(h, n_heads, n_kv_heads, N, TP_F32, &g) != TP_OK) return 0;
  return g.W;
}

size_t tp_gqa_workspace_size(int fwd, int64_t M, int64_t h, int32_t n_heads, int32_t n_kv_heads,
                             int32_t N, tp_dtype dtype, tp_reduce mode) {
  Gqa g;
  if (M < 0 || (dtype != TP_BF16 && dtype != TP_F32) ||
      gqa_shape(h, n_heads, n_kv_heads, N, dtype, &g) != TP_OK)
    return 0;
  return fwd ? fwd_ws(M, h, N, mode) : bwd_ws(M, h, g, N, dtype, mode);
}

tp_status tp_gqa_pack_qkv(const void* Wq, const void* Wk, const void* Wv, void* Wqkv, int64_t h,
                          int32_t n_heads, int32_t n_kv_heads, int32_t N, tp_dtype dtype,
                          void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(Wq && Wk && Wv && Wqkv, TP_ERR_INVALID_ARG, "Wq, Wk, Wv and Wqkv are required"));
  Gqa g;
  TP_TRY(gqa_shape(h, n_heads, n_kv_heads, N, dtype, &g));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = grid_for(h * g.W);
  if (dtype == TP_BF16)
    TP_CUDA_TRY(launch_kernel(gqa_pack_kernel<__nv_bfloat16>, grid, 256, 0, st,
        static_cast<const __nv_bfloat16*>(Wq), static_cast<const __nv_bfloat16*>(Wk),
        static_cast<const __nv_bfloat16*>(Wv), static_cast<__nv_bfloat16*>(Wqkv), h, n_heads,
        n_kv_heads, g.hq, g.hkv, g.r, static_cast<int>(g.d), g.S, g.W));
  else
    TP_CUDA_TRY(launch_kernel(gqa_pack_kernel<float>, grid, 256, 0, st,
        static_cast<const float*>(Wq), static_cast<const float*>(Wk),
        static_cast<const float*>(Wv), static_cast<float*>(Wqkv), h, n_heads, n_kv_heads, g.hq,
        g.hkv, g.r, static_cast<int>(g.d), g.S, g.W));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

tp_status tp_gqa_attention_fwd(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                               int64_t h, int32_t n_heads, int32_t n_kv_heads, int32_t N,
                               int causal, tp_dtype dtype, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(qkv && o && lse, TP_ERR_INVALID_ARG, "qkv, o and lse are required"));
  TP_TRY(need(b >= 0 && s >= 0, TP_ERR_INVALID_ARG, "need b, s >= 0"));
  Gqa g;
  TP_TRY(gqa_shape(h, n_heads, n_kv_heads, N, TP_F32, &g));
  if (b * s == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_gqa_attention_fwd(qkv, o, lse, b, s, n_heads, n_kv_heads, N,
                                  static_cast<int>(g.d), causal, dtype,
                                  static_cast<cudaStream_t>(stream));
}

size_t tp_gqa_attention_bwd_workspace_size(int64_t b, int64_t s, int32_t n_heads) {
  if (b < 0 || s < 0 || n_heads < 1) return 0;
  return std::max<size_t>(attention_bwd_tc_ws_bytes(b, s, n_heads), 256);
}

tp_status tp_gqa_attention_bwd(const void* qkv, const void* o, const float* lse, const void* dO,
                               void* dqkv, int64_t b, int64_t s, int64_t h, int32_t n_heads,
                               int32_t n_kv_heads, int32_t N, int causal, tp_dtype dtype,
                               void* ws, size_t ws_bytes, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(qkv && o && lse && dO && dqkv, TP_ERR_INVALID_ARG,
              "qkv, o, lse, dO and dqkv are required"));
  TP_TRY(need(b >= 0 && s >= 0, TP_ERR_INVALID_ARG, "need b, s >= 0"));
  Gqa g;
  TP_TRY(gqa_shape(h, n_heads, n_kv_heads, N, TP_F32, &g));
  if (ws) {
    TP_TRY(need(ws_bytes >= tp_gqa_attention_bwd_workspace_size(b, s, n_heads), TP_ERR_WORKSPACE,
                "workspace smaller than tp_gqa_attention_bwd_workspace_size"));
    TP_TRY(need(reinterpret_cast<uintptr_t>(ws) % 16 == 0, TP_ERR_ALIGNMENT,
                "workspace must be 16-byte aligned"));
  }
  if (b * s == 0) return TP_OK;
  TP_TRY(check_device());
  return launch_gqa_attention_bwd(qkv, o, lse, dO, dqkv, ws, b, s, n_heads, n_kv_heads, N,
                                  static_cast<int>(g.d), causal, dtype,
                                  static_cast<cudaStream_t>(stream));
}

tp_status tp_gqa_attn_proj_fwd(const void* x, const float* gamma, const float* beta,
                               const void* Wqkv, const void* Wo, void* xn, float* mean,
                               float* rstd, void* qkv, void* o, float* lse, void* out, int64_t b,
                               int64_t s, int64_t h, int32_t n_heads, int32_t n_kv_heads,
                               int32_t N, int causal, tp_dtype dtype, tp_reduce mode, void* ws,
                               size_t ws_bytes, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(x && gamma && beta && Wqkv && Wo && xn && mean && rstd && qkv && o && lse && out,
              TP_ERR_INVALID_ARG, "all tensors of tp_gqa_attn_proj_fwd are required"));
  TP_TRY(need(b >= 0 && s >= 0, TP_ERR_INVALID_ARG, "need b, s >= 0"));
  Gqa g;
  TP_TRY(gqa_shape(h, n_heads, n_kv_heads, N, dtype, &g));
  TP_TRY(check_aligned({x, gamma, beta, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, out, ws}));
  const int64_t M = b * s;
  if (M == 0) return TP_OK;
  TP_TRY(need(ws_bytes >= fwd_ws(M, h, N, mode) && (mode == TP_REDUCE_SPLITK || ws),
              TP_ERR_WORKSPACE, "workspace smaller than tp_gqa_workspace_size"));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TP_TRY(launch_layernorm_fwd(x, gamma, beta, xn, mean, rstd, M, h, 1e-5f, dtype, st));
  {  // column-parallel projection: shard i's block of S columns
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = g.W;
    d.K = h;
    d.A[0] = {xn, M, h, h};
    d.B[0] = {Wqkv, h, g.W, g.W};
    d.b_mn = true;
    d.ldo = g.W;
    d.shards = N;
    d.shard_axis = 1;
    d.epi = EPI_STORE;
    d.out[0] = qkv;
    d.out_f32 = dtype == TP_F32;
    TP_TRY(launch_gemm(d, st));
  }
  TP_TRY(launch_gqa_attention_fwd(qkv, o, lse, b, s, n_heads, n_kv_heads, N,
                                  static_cast<int>(g.d), causal, dtype, st));
  // shard i's O_i (its query heads) feeds row block i of W_o; sum + residual
  return row_impl(o, Wo, x, out, M, h, h, N, dtype, mode, ws, st);
}

tp_status tp_gqa_attn_proj_bwd(const void* x, const float* gamma, const void* Wqkv,
                               const void* Wo, const void* xn, const float* mean,
                               const float* rstd, const void* qkv, const void* o,
                               const float* lse, const void* dout, void* dx, float* dgamma,
                               float* dbeta, void* dWqkv, void* dWo, int64_t b, int64_t s,
                               int64_t h, int32_t n_heads, int32_t n_kv_heads, int32_t N,
                               int causal, tp_dtype dtype, tp_reduce mode, void* ws,
                               size_t ws_bytes, void* stream) {
  TP_TRY(check_dtype(dtype));
  TP_TRY(need(mode == TP_REDUCE_BUFFERS || mode == TP_REDUCE_SPLITK, TP_ERR_INVALID_ARG,
              "unknown reduce mode"));
  TP_TRY(need(x && gamma && Wqkv && Wo && xn && mean && rstd && qkv && o && lse && dout && dx &&
                  dgamma && dbeta && dWqkv && dWo,
              TP_ERR_INVALID_ARG, "all tensors of tp_gqa_attn_proj_bwd are required"));
  TP_TRY(need(b >= 0 && s >= 0, TP_ERR_INVALID_ARG, "need b, s >= 0"));
  Gqa g;
  TP_TRY(gqa_shape(h, n_heads, n_kv_heads, N, dtype, &g));
  TP_TRY(check_aligned({x, gamma, Wqkv, Wo, xn, mean, rstd, qkv, o, lse, dout, dx, dgamma,
                        dbeta, dWqkv, dWo, ws}));
  const int64_t M = b * s;
  if (M == 0) return TP_OK;
  TP_TRY(need(ws && ws_bytes >= bwd_ws(M, h, g, N, dtype, mode), TP_ERR_WORKSPACE,
              "workspace smaller than tp_gqa_workspace_size"));
  TP_TRY(check_device());
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t e = elem_size(dtype);
  char* w = static_cast<char*>(ws);
  void* dO = w;
  w += a256(M * h * e);
  void* dqkv = w;
  w += a256(M * g.W * e);
  void* dxn = w;
  w += a256(M * h * e);
  void* parts = w;
  w += a256(partial_bytes(M, h, N, mode));
  void* lnws = w;
  w += a256(layernorm_bwd_ws_bytes(M, h));
  void* ldws = w;  // attention (lse, D) pairs
  // The weight gradients are off the critical path: dW_o runs on a side stream beside
  // dO and the attention backward, dW_qkv and the replicas' sum beside dx_n and the
  // LayerNorm backward.
  SideBranch br(st);
  {  // dW_o,i = O_i^T dout
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
  {  // dO_i = dout W_o,i^T (every shard reads all of dout)
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = h;
    d.K = h;
    d.A[0] = {dout, M, h, h};
    d.B[0] = {Wo, h, h, h};
    d.ldo = h;
    d.epi = EPI_STORE;
    d.out[0] = dO;
    d.out_f32 = dtype == TP_F32;
    d.shards = N;
    d.shard_axis = 1;
    TP_TRY(launch_gemm(d, st));
  }
  TP_TRY(launch_gqa_attention_bwd(qkv, o, lse, dO, dqkv, ldws, b, s, n_heads, n_kv_heads, N,
                                  static_cast<int>(g.d), causal, dtype, st));
  TP_TRY(br.fork());  // dQKV is complete
  {  // dWqkv = xn^T dQKV (each block: its shard's gradient, replicas' partial K/V)
    GemmDesc d;
    d.dtype = dtype;
    d.M = h;
    d.N = g.W;
    d.K = M;
    d.A[0] = {xn, M, h, h};
    d.a_mn = true;
    d.B[0] = {dqkv, M, g.W, g.W};
    d.b_mn = true;
    d.ldo = g.W;
    d.epi = EPI_STORE;
    d.out[0] = dWqkv;
    d.out_f32 = dtype == TP_F32;
    TP_TRY(launch_gemm(d, br.stream()));
  }
  if (g.r > 1) {  // all-reduce among each key/value head's replicas
    // d, S and W are multiples of 16 columns (head_dim 16, 32 or 64) and dWqkv is
    // 16-byte aligned: the vector kernel applies whenever W's rows are 16-byte multiples
    const int64_t E = 16 / static_cast<int64_t>(elem_size(dtype));
    const bool vec = g.d % E == 0 && g.S % E == 0 && g.W % E == 0;
    const unsigned grid = grid_for(h * n_kv_heads * 2 * g.d / (vec ? E : 1));
    if (dtype == TP_BF16 && vec)
      TP_CUDA_TRY(launch_kernel(gqa_replica_sum_vec_kernel<__nv_bfloat16>, grid, 256, 0, br.stream(),
          static_cast<__nv_bfloat16*>(dWqkv), h, n_kv_heads, g.hq, g.r, static_cast<int>(g.d),
          g.S, g.W));
    else if (dtype == TP_BF16)
      TP_CUDA_TRY(launch_kernel(gqa_replica_sum_kernel<__nv_bfloat16>, grid, 256, 0, br.stream(),
          static_cast<__nv_bfloat16*>(dWqkv), h, n_kv_heads, g.hq, g.r, static_cast<int>(g.d),
          g.S, g.W));
    else if (vec)
      TP_CUDA_TRY(launch_kernel(gqa_replica_sum_vec_kernel<float>, grid, 256, 0, br.stream(),
          static_cast<float*>(dWqkv), h, n_kv_heads, g.hq, g.r, static_cast<int>(g.d), g.S, g.W));
    else
      TP_CUDA_TRY(launch_kernel(gqa_replica_sum_kernel<float>, grid, 256, 0, br.stream(),
          static_cast<float*>(dWqkv), h, n_kv_heads, g.hq, g.r, static_cast<int>(g.d), g.S, g.W));
    count_launch();
    TP_CUDA_TRY(cudaGetLastError());
  }
  {  // f-backward: dxn = sum_i dQKV_i Wqkv_i^T (shard i: one K-group of S columns)
    GemmDesc d;
    d.dtype = dtype;
    d.M = M;
    d.N = h;
    d.A[0] = {dqkv, M, g.W, g.W};
    d.B[0] = {Wqkv, h, g.W, g.W};  // Wqkv (h, W) read as B(k = W, n = h): K-major
    d.ldo = h;
    d.epi = EPI_STORE;
    if (mode == TP_REDUCE_SPLITK) {
      d.K = g.W;
      d.out[0] = dxn;
      d.out_f32 = dtype == TP_F32;
      TP_TRY(launch_gemm(d, st));
    } else {
      d.K = g.S;
      d.groups = N;
      d.out[0] = parts;
      d.out_f32 = true;
      d.out_group_stride = M * h;
      TP_TRY(launch_gemm(d, st));
      TP_TRY(launch_shard_reduce(static_cast<const float*>(parts), nullptr, dxn, N, M, h, dtype,
                                 st));
    }
  }
  TP_TRY(launch_layernorm_bwd(x, gamma, mean, rstd, dxn, dout, dx, dgamma, dbeta, M, h, lnws,
                              dtype, st));
  return br.join();
}

}  // extern "C"
