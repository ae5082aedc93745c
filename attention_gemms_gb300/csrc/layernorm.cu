// LayerNorm over the full hidden width, forward and backward, with the residual
// add of the backward fused in:
//   y  = gamma * (x - mu) * rstd + beta,  rstd = 1 / sqrt(var + eps), biased variance
//   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat)),  g = dy * gamma
//   dgamma = sum_rows dy * xhat,  dbeta = sum_rows dy
// (LN formula of the 张量并行 notes, §相关分析; the statistics need the whole hidden
// width, which is why the shard sum precedes it.)
// Row kernels use one warp per row; the parameter gradients are column sums taken
// in a fixed order (per-chunk partials, then a second pass over the chunks), so
// results are deterministic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace tp {
namespace {

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

constexpr int kRowWarps = 8;  // rows per CTA in the row kernels

template <typename T>
__global__ void __launch_bounds__(32 * kRowWarps) ln_fwd_kernel(const T* __restrict__ x,
                                                                const float* __restrict__ gamma,
                                                                const float* __restrict__ beta,
                                                                T* __restrict__ y, float* mean,
                                                                float* rstd, int64_t M, int h,
                                                                float eps) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const T* xr = x + row * h;
  float s = 0.0f;
  for (int c = lane; c < h; c += 32) s += ld(xr, c);
  const float mu = warp_sum(s) / h;
  float v = 0.0f;
  for (int c = lane; c < h; c += 32) {
    const float d = ld(xr, c) - mu;
    v += d * d;
  }
  const float rs = 1.0f / sqrtf(warp_sum(v) / h + eps);
  T* yr = y + row * h;
  for (int c = lane; c < h; c += 32) st(yr, c, gamma[c] * ((ld(xr, c) - mu) * rs) + beta[c]);
  if (lane == 0) {
    if (mean) mean[row] = mu;
    if (rstd) rstd[row] = rs;
  }
}

template <typename T>
__global__ void __launch_bounds__(32 * kRowWarps) ln_bwd_dx_kernel(
    const T* __restrict__ x, const float* __restrict__ gamma, const float* __restrict__ mean,
    const float* __restrict__ rstd, const T* __restrict__ dy, const T* __restrict__ dres,
    T* __restrict__ dx, int64_t M, int h) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float mu = mean[row], rs = rstd[row];
  const T* xr = x + row * h;
  const T* dyr = dy + row * h;
  float s1 = 0.0f, s2 = 0.0f;
  for (int c = lane; c < h; c += 32) {
    const float g = ld(dyr, c) * gamma[c];
    s1 += g;
    s2 += g * (ld(xr, c) - mu) * rs;
  }
  s1 = warp_sum(s1) / h;
  s2 = warp_sum(s2) / h;
  for (int c = lane; c < h; c += 32) {
    const float xh = (ld(xr, c) - mu) * rs;
    float v = rs * (ld(dyr, c) * gamma[c] - s1 - xh * s2);
    if (dres) v += ld(dres + row * h, c);
    st(dx + row * h, c, v);
  }
}

constexpr int kColThreads = 256;
constexpr int kRowsPerChunk = 64;

// partial[chunk][0:h] = sum over the chunk's rows of dy * xhat, partial[chunk][h:2h] = of dy.
// Rows are grouped by rank (rank r owns rows [r * rank_rows, (r + 1) * rank_rows), one
// rank when the LN input is replicated) and each rank's rows are cut into cpr chunks
// of at most kRowsPerChunk rows; chunk index = r * cpr + c.
template <typename T>
__global__ void __launch_bounds__(kColThreads) ln_bwd_param_partial_kernel(
    const T* __restrict__ x, const float* __restrict__ mean, const float* __restrict__ rstd,
    const T* __restrict__ dy, float* __restrict__ partial, int64_t M, int h, int64_t rank_rows,
    int cpr) {
  const int c = blockIdx.x * kColThreads + threadIdx.x;
  const int rank = blockIdx.y / cpr, chunk = blockIdx.y - rank * cpr;
  const int64_t rank_end = min(M, (rank + 1) * rank_rows);
  const int64_t r0 = rank * rank_rows + static_cast<int64_t>(chunk) * kRowsPerChunk;
  if (c >= h) return;
  float sg = 0.0f, sb = 0.0f;
  const int64_t r1 = min(rank_end, r0 + kRowsPerChunk);
  for (int64_t r = r0; r < r1; ++r) {
    const float d = ld(dy + r * h, c);
    sg += d * (ld(x + r * h, c) - mean[r]) * rstd[r];
    sb += d;
  }
  partial[blockIdx.y * 2ll * h + c] = sg;
  partial[blockIdx.y * 2ll * h + h + c] = sb;
}

// per rank: the sum of its chunks in order (written to dgamma_ranks / dbeta_ranks
// (ranks, h) when given); then the sum over the ranks in rank order
__global__ void __launch_bounds__(kColThreads) ln_bwd_param_final_kernel(
    const float* __restrict__ partial, int ranks, int cpr, int h, float* dgamma, float* dbeta,
    float* dgamma_ranks, float* dbeta_ranks) {
  const int c = blockIdx.x * kColThreads + threadIdx.x;
  if (c >= h) return;
  float tg = 0.0f, tb = 0.0f;
  for (int r = 0; r < ranks; ++r) {
    float sg = 0.0f, sb = 0.0f;
    for (int k = r * cpr; k < (r + 1) * cpr; ++k) {
      sg += partial[k * 2ll * h + c];
      sb += partial[k * 2ll * h + h + c];
    }
    if (dgamma_ranks) dgamma_ranks[static_cast<int64_t>(r) * h + c] = sg;
    if (dbeta_ranks) dbeta_ranks[static_cast<int64_t>(r) * h + c] = sb;
    tg += sg;
    tb += sb;
  }
  if (dgamma) dgamma[c] = tg;
  if (dbeta) dbeta[c] = tb;
}

template <typename T>
tp_status fwd_t(const void* x, const float* gamma, const float* beta, void* y, float* mean,
                float* rstd, int64_t M, int h, float eps, cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>((M + kRowWarps - 1) / kRowWarps);
  ln_fwd_kernel<T><<<blocks, 32 * kRowWarps, 0, st>>>(static_cast<const T*>(x), gamma, beta,
                                                       static_cast<T*>(y), mean, rstd, M, h, eps);
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

template <typename T>
tp_status bwd_t(const void* x, const float* gamma, const float* mean, const float* rstd,
                const void* dy, const void* dres, void* dx, float* dgamma, float* dbeta,
                float* dgamma_ranks, float* dbeta_ranks, int64_t M, int h, int ranks, float* ws,
                cudaStream_t st) {
  const unsigned rblocks = static_cast<unsigned>((M + kRowWarps - 1) / kRowWarps);
  ln_bwd_dx_kernel<T><<<rblocks, 32 * kRowWarps, 0, st>>>(
      static_cast<const T*>(x), gamma, mean, rstd, static_cast<const T*>(dy),
      static_cast<const T*>(dres), static_cast<T*>(dx), M, h);
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  if (!dgamma && !dbeta && !dgamma_ranks && !dbeta_ranks) return TP_OK;
  const int64_t rank_rows = M / ranks;
  const int cpr = static_cast<int>((rank_rows + kRowsPerChunk - 1) / kRowsPerChunk);
  const dim3 g1((h + kColThreads - 1) / kColThreads, ranks * cpr);
  ln_bwd_param_partial_kernel<T><<<g1, kColThreads, 0, st>>>(
      static_cast<const T*>(x), mean, rstd, static_cast<const T*>(dy), ws, M, h, rank_rows, cpr);
  ln_bwd_param_final_kernel<<<(h + kColThreads - 1) / kColThreads, kColThreads, 0, st>>>(
      ws, ranks, cpr, h, dgamma, dbeta, dgamma_ranks, dbeta_ranks);
  count_launch(2);
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

}  // namespace

size_t layernorm_bwd_ws_bytes(int64_t M, int64_t h, int ranks) {
  if (ranks < 1 || M % ranks) return 0;
  const int64_t cpr = (M / ranks + kRowsPerChunk - 1) / kRowsPerChunk;
  return static_cast<size_t>(ranks * cpr) * 2 * h * sizeof(float);
}

tp_status launch_layernorm_fwd(const void* x, const float* gamma, const float* beta, void* y,
                               float* mean, float* rstd, int64_t M, int64_t h, float eps,
                               tp_dtype dt, cudaStream_t st) {
  if (M <= 0) return TP_OK;
  if (h > (1 << 24) || M / kRowWarps > 2147483647ll) return fail(TP_ERR_SHAPE, "LN too large");
  return dt == TP_BF16
             ? fwd_t<__nv_bfloat16>(x, gamma, beta, y, mean, rstd, M, static_cast<int>(h), eps, st)
             : fwd_t<float>(x, gamma, beta, y, mean, rstd, M, static_cast<int>(h), eps, st);
}

tp_status launch_layernorm_bwd(const void* x, const float* gamma, const float* mean,
                               const float* rstd, const void* dy, const void* dres, void* dx,
                               float* dgamma, float* dbeta, int64_t M, int64_t h, void* ws,
                               tp_dtype dt, cudaStream_t st) {
  return launch_layernorm_bwd_ranks(x, gamma, mean, rstd, dy, dres, dx, dgamma, dbeta, nullptr,
                                    nullptr, M, h, 1, ws, dt, st);
}

tp_status launch_layernorm_bwd_ranks(const void* x, const float* gamma, const float* mean,
                                     const float* rstd, const void* dy, const void* dres,
                                     void* dx, float* dgamma, float* dbeta, float* dgamma_ranks,
                                     float* dbeta_ranks, int64_t M, int64_t h, int ranks,
                                     void* ws, tp_dtype dt, cudaStream_t st) {
  if (M <= 0) return TP_OK;
  if (ranks < 1 || M % ranks) return fail(TP_ERR_SHAPE, "LN rows must split evenly over the ranks");
  const int64_t cpr = (M / ranks + kRowsPerChunk - 1) / kRowsPerChunk;
  if (h > (1 << 24) || ranks * cpr > 65535) return fail(TP_ERR_SHAPE, "LN too large");
  float* w = static_cast<float*>(ws);
  const int hh = static_cast<int>(h);
  return dt == TP_BF16 ? bwd_t<__nv_bfloat16>(x, gamma, mean, rstd, dy, dres, dx, dgamma, dbeta,
                                              dgamma_ranks, dbeta_ranks, M, hh, ranks, w, st)
                       : bwd_t<float>(x, gamma, mean, rstd, dy, dres, dx, dgamma, dbeta,
                                      dgamma_ranks, dbeta_ranks, M, hh, ranks, w, st);
}

}  // namespace tp
