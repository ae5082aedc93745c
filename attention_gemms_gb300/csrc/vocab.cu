// Vocabulary-parallel embedding and cross-entropy, and the AdamW update.
//
// Shard i of the vocabulary owns rows [i v/N, (i+1) v/N) of the word embedding E (v, h)
// and the same columns of the logits (the output layer shares E).
//  * Embedding [张量并行 notes, §嵌入层的并行化]: every shard looks the ids up in its
//    block, returning a zero row for ids it does not own, and the all-reduce adds the
//    shards' results. One warp per token visits the shards in order.
//  * Its gradient: shard i adds dx[t] to row id_t of its block for the tokens it owns.
//    One CTA per vocabulary row scans the ids in token order, so the sums are
//    deterministic (no atomics).
//  * Cross-entropy [张量并行 notes, §损失计算层的并行化]: the shards' row maxima are
//    combined (all-reduce max), then the shards' sums of exp(l - m) (all-reduce sum),
//    so the logits are never gathered; the shard owning a row's target contributes
//    log S + m - l_target, each shard sums its rows, and the N shard sums are added.
//    With 8-aligned shards one warp per row reads the row once: each lane keeps a
//    running (max, sum of exp) per shard, re-based when the max grows, and the shards'
//    (m_i, s_i) are combined exactly as the two all-reduces do. Otherwise one CTA per
//    row makes two plain passes (max, then sum of exp(l - m)).
//  * The gradient softmax - one_hot, scaled, needs only m + log S per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "internal.h"

namespace tp {
namespace {

__device__ __forceinline__ float ldv(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ldv(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void stv(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void stv(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

constexpr int kThreads = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// block-wide reductions over kThreads threads; every thread gets the result
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) r += red[w];
  return r;
}

// ------------------------------------------------------------------ embedding

template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_embed_fwd_kernel(
    const int32_t* __restrict__ ids, const T* __restrict__ E, T* __restrict__ x, int64_t M,
    int64_t v, int h, int N) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const int64_t id = ids[row], vs = v / N;
  for (int c = lane; c < h; c += 32) {
    float acc = 0.0f;  // the all-reduce of the shards' masked lookups, shard 0 first
    for (int i = 0; i < N; ++i) {
      const int64_t lo = i * vs;
      acc += (id >= lo && id < lo + vs) ? ldv(E, id * h + c) : 0.0f;
    }
    stv(x, row * h + c, acc);
  }
}

constexpr int kIdTile = 1024;

template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_embed_bwd_kernel(
    const int32_t* __restrict__ ids, const T* __restrict__ dx, T* __restrict__ dE, int64_t M,
    int h, int accumulate) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  __shared__ int32_t tile[kIdTile];
  const int64_t vrow = blockIdx.x;  // a vocabulary row lies in exactly one shard's block
  for (int c0 = 0; c0 < h; c0 += kThreads) {
    const int c = c0 + threadIdx.x;
    float acc = (accumulate && c < h) ? ldv(dE, vrow * h + c) : 0.0f;
    for (int64_t t0 = 0; t0 < M; t0 += kIdTile) {
      const int n = static_cast<int>(min(static_cast<int64_t>(kIdTile), M - t0));
      __syncthreads();
      for (int j = threadIdx.x; j < n; j += kThreads) tile[j] = ids[t0 + j];
      __syncthreads();
      if (c < h)
        for (int j = 0; j < n; ++j)
          if (tile[j] == vrow) acc += ldv(dx, (t0 + j) * h + c);  // tokens in order
    }
    if (c < h) stv(dE, vrow * h + c, acc);
  }
}

// ------------------------------------------------------------------ cross-entropy

template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_ce_fwd_kernel(
    const T* __restrict__ logits, const int32_t* __restrict__ targets, float* __restrict__ lse,
    float* __restrict__ row_loss, int64_t v, int N) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  __shared__ float red[kThreads / 32];
  const int64_t row = blockIdx.x;
  const T* L = logits + row * v;
  const int64_t vs = v / N;
  // all-reduce (max) of the shards' row maxima
  float m = -INFINITY;
  for (int i = 0; i < N; ++i) {
    float mi = -INFINITY;
    for (int64_t c = i * vs + threadIdx.x; c < (i + 1) * vs; c += kThreads) mi = fmaxf(mi, ldv(L, c));
    m = fmaxf(m, block_max(mi, red));
  }
  // all-reduce (sum) of the shards' sums of exp(l - m), shard 0 first
  float S = 0.0f;
  for (int i = 0; i < N; ++i) {
    float si = 0.0f;
    for (int64_t c = i * vs + threadIdx.x; c < (i + 1) * vs; c += kThreads) si += expf(ldv(L, c) - m);
    S += block_sum(si, red);
  }
  if (threadIdx.x == 0) {
    const float l = m + logf(S);
    const int64_t t = targets[row];
    lse[row] = l;
    row_loss[row] = (t >= 0 && t < v) ? l - ldv(L, t) : 0.0f;  // the owning shard's term
  }
}

// 8 consecutive values as fp32 (16-byte aligned)
__device__ __forceinline__ void ld8(const __nv_bfloat16* p, float* v) {
  const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void ld8(const float* p, float* v) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void st8(__nv_bfloat16* p, const float* v) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  __stcs(reinterpret_cast<uint4*>(p), u);
}
__device__ __forceinline__ void st8(float* p, const float* v) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
}

// The vectorised kernels work in base 2: with y = x log2(e), exp(x - m) = 2^(y - m2),
// m2 = m log2(e), one multiply-add and one exp2 per logit; lse = (m2 + log2 S) ln 2.
constexpr float kLog2e = 1.4426950408889634f;  // log2(e)
constexpr float kLn2 = 0.6931471805599453f;    // ln(2)

// 2^x on the special-function unit (PTX ex2.approx.ftz: relative error about 2^-22,
// results below 2^-126 flushed to zero, which only drops terms that cannot move a sum
// that already holds 2^0 = 1 from the row maximum); 2^-inf = 0
__device__ __forceinline__ float ex2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (m2, s) running maximum (base-2 scaled) and sum of 2^(y - m2), updated with 8 logits
// (the maximum is taken on the raw logits and scaled once: rounding is monotonic, so
// it equals the maximum of the scaled logits; each exponent is one fused multiply-add)
__device__ __forceinline__ void online8(float& m2, float& s, const float* x) {
  float mx = x[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) mx = fmaxf(mx, x[k]);
  mx *= kLog2e;
  if (mx > m2) {
    s *= ex2_sfu(m2 - mx);  // m2 = -inf at first: s = 0 stays 0
    m2 = mx;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) s += ex2_sfu(fmaf(x[k], kLog2e, -m2));
}

// (m2, s) pairs combined: max of the two, sums re-based to it
__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  s = (m == -INFINITY ? 0.0f : s * ex2_sfu(m - mm)) + (m2 == -INFINITY ? 0.0f : s2 * ex2_sfu(m2 - mm));
  m = mm;
}

constexpr int kVecMaxShards = 8;

// Vectorised forward (v/N a multiple of 8, N <= 8): one warp per row, one read of the
// row, no barriers. For each shard the lanes keep running (max, sum of exponentials)
// over their 8-column chunks and combine them with shuffles into the shard's
// (m_i, s_i); the shards are then combined as the pages' two all-reduces:
// m = max_i m_i, S = sum_i s_i 2^(m_i - m) in shard order (each shard's sum of
// exp(l - m), re-based to the global maximum).
template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_ce_fwd_vec_kernel(
    const T* __restrict__ logits, const int32_t* __restrict__ targets, float* __restrict__ lse,
    float* __restrict__ row_loss, int64_t M, int64_t v, int N) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const T* L = logits + row * v;
  const int64_t vs8 = v / N / 8;
  float mi[kVecMaxShards], si[kVecMaxShards];
#pragma unroll
  for (int i = 0; i < kVecMaxShards; ++i) {
    mi[i] = -INFINITY;
    si[i] = 0.0f;
    if (i < N) {
      float m = -INFINITY, sm = 0.0f;
      int64_t c8 = i * vs8 + lane;
      const int64_t e8 = (i + 1) * vs8;
      for (; c8 + 96 < e8; c8 += 128) {  // four chunks in flight per lane
        float x0[8], x1[8], x2[8], x3[8];
        ld8(L + c8 * 8, x0);
        ld8(L + (c8 + 32) * 8, x1);
        ld8(L + (c8 + 64) * 8, x2);
        ld8(L + (c8 + 96) * 8, x3);
        online8(m, sm, x0);
        online8(m, sm, x1);
        online8(m, sm, x2);
        online8(m, sm, x3);
      }
      for (; c8 < e8; c8 += 32) {
        float x0[8];
        ld8(L + c8 * 8, x0);
        online8(m, sm, x0);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        combine(m, sm, __shfl_xor_sync(0xFFFFFFFFu, m, o), __shfl_xor_sync(0xFFFFFFFFu, sm, o));
      mi[i] = m;
      si[i] = sm;
    }
  }
  if (lane == 0) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kVecMaxShards; ++i)
      if (i < N) m = fmaxf(m, mi[i]);  // all-reduce (max)
    float S = 0.0f;
#pragma unroll
    for (int i = 0; i < kVecMaxShards; ++i)
      if (i < N) S += si[i] * exp2f(mi[i] - m);  // all-reduce (sum)
    const float l = (m + log2f(S)) * kLn2;
    const int64_t t = targets[row];
    lse[row] = l;
    row_loss[row] = (t >= 0 && t < v) ? l - ldv(L, t) : 0.0f;
  }
}

// Vectorised gradient (v a multiple of 8): 8 columns per thread per step, streamed
template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_ce_bwd_vec_kernel(
    const T* logits, const int32_t* __restrict__ targets, const float* __restrict__ lse,
    T* dlogits, int64_t v, float scale) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const float l2 = lse[row] * kLog2e;
  const int64_t t = targets[row];
  const T* L = logits + row * v;
  T* D = dlogits + row * v;
  const int64_t n8 = v / 8;
  for (int64_t c8 = threadIdx.x; c8 < n8; c8 += kThreads) {
    float x[8];
    ld8(L + c8 * 8, x);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float p = exp2f(fmaf(x[k], kLog2e, -l2));  // exp(x - lse)
      if (c8 * 8 + k == t) p -= 1.0f;
      x[k] = p * scale;
    }
    st8(D + c8 * 8, x);  // may overwrite the logits in place (same elements)
  }
}

// shard i's loss = the sum of its rows' terms (rows whose target it owns); the loss is
// the sum over the shards (in order) divided by M. One CTA, fixed reduction order.
__global__ void __launch_bounds__(1024) vocab_ce_loss_kernel(
    const float* __restrict__ row_loss, const int32_t* __restrict__ targets,
    float* __restrict__ shard_loss, float* __restrict__ loss, int64_t M, int64_t v, int N) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  __shared__ float red[32];
  const int64_t vs = v / N;
  float total = 0.0f;
  for (int i = 0; i < N; ++i) {
    float s = 0.0f;
    for (int64_t r = threadIdx.x; r < M; r += 1024) {
      const int64_t t = targets[r];
      if (t >= i * vs && t < (i + 1) * vs) s += row_loss[r];
    }
    s = warp_sum(s);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
      float si = 0.0f;
      for (int w = 0; w < 32; ++w) si += red[w];
      if (shard_loss) shard_loss[i] = si;
      total += si;
    }
  }
  if (threadIdx.x == 0) loss[0] = total / static_cast<float>(M);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) vocab_ce_bwd_kernel(
    const T* logits, const int32_t* __restrict__ targets, const float* __restrict__ lse,
    T* dlogits, int64_t v, float scale) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t row = blockIdx.x;
  const float l = lse[row];
  const int64_t t = targets[row];
  for (int64_t c = threadIdx.x; c < v; c += kThreads) {
    float p = expf(ldv(logits, row * v + c) - l);
    if (c == t) p -= 1.0f;
    stv(dlogits, row * v + c, p * scale);  // may overwrite the logits in place
  }
}

// ------------------------------------------------------------------ AdamW

__global__ void __launch_bounds__(kThreads) adamw_kernel(
    float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
    float* __restrict__ v, int64_t n, float lr, float b1, float b2, float eps, float wd,
    float bc1, float bc2) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float gi = g[i];
    const float mi = b1 * m[i] + (1.0f - b1) * gi;
    const float vi = b2 * v[i] + (1.0f - b2) * gi * gi;
    m[i] = mi;
    v[i] = vi;
    const float pi = p[i] * (1.0f - lr * wd);
    p[i] = pi - lr * (mi / bc1) / (sqrtf(vi / bc2) + eps);
  }
}

// The same update with the step count read from device memory: thread 0 of every CTA
// forms the bias corrections 1 - beta^step for the CTA (fp32 powf: double precision
// costs every CTA microseconds on this part's FP64 units), so the launch has no
// per-step argument and can replay from a CUDA graph.
__global__ void __launch_bounds__(kThreads) adamw_dev_kernel(
    float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
    float* __restrict__ v, int64_t n, const int32_t* __restrict__ step, float lr, float b1,
    float b2, float eps, float wd) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  __shared__ float bc[2];
  if (threadIdx.x == 0) {
    const float t = static_cast<float>(*step);
    bc[0] = 1.0f - powf(b1, t);
    bc[1] = 1.0f - powf(b2, t);
  }
  __syncthreads();
  const float bc1 = bc[0], bc2 = bc[1];
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += stride) {
    const float gi = g[i];
    const float mi = b1 * m[i] + (1.0f - b1) * gi;
    const float vi = b2 * v[i] + (1.0f - b2) * gi * gi;
    m[i] = mi;
    v[i] = vi;
    const float pi = p[i] * (1.0f - lr * wd);
    p[i] = pi - lr * (mi / bc1) / (sqrtf(vi / bc2) + eps);
  }
}

// One step of a training loop's device-side bookkeeping: the step counter advances by
// one, and the step's loss goes to its slot of the loss history.
__global__ void step_advance_kernel(int32_t* step, const float* loss, float* hist,
                                    int64_t hist_len) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int32_t t = *step + 1;
  *step = t;
  if (loss && hist) hist[static_cast<int64_t>(t - 1) % hist_len] = *loss;
}

template <typename T>
tp_status embed_fwd_t(const int32_t* ids, const void* E, void* x, int64_t M, int64_t v, int h,
                      int N, cudaStream_t st) {
  const int64_t blocks = (M + kThreads / 32 - 1) / (kThreads / 32);
  TP_CUDA_TRY(launch_kernel(vocab_embed_fwd_kernel<T>, static_cast<unsigned>(blocks), kThreads, 0, st,
      ids, static_cast<const T*>(E), static_cast<T*>(x), M, v, h, N));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

}  // namespace

tp_status launch_vocab_embed_fwd(const int32_t* ids, const void* E, void* x, int64_t M, int64_t v,
                                 int64_t h, int N, tp_dtype dt, cudaStream_t st) {
  if (M <= 0) return TP_OK;
  if (M / (kThreads / 32) > 2147483647ll || h > (1 << 30)) return fail(TP_ERR_SHAPE, "embedding too large");
  return dt == TP_BF16 ? embed_fwd_t<__nv_bfloat16>(ids, E, x, M, v, static_cast<int>(h), N, st)
                       : embed_fwd_t<float>(ids, E, x, M, v, static_cast<int>(h), N, st);
}

tp_status launch_vocab_embed_bwd(const int32_t* ids, const void* dx, void* dE, int64_t M,
                                 int64_t v, int64_t h, bool accumulate, tp_dtype dt,
                                 cudaStream_t st) {
  if (v <= 0) return TP_OK;
  if (v > 2147483647ll || h > (1 << 30)) return fail(TP_ERR_SHAPE, "embedding too large");
  const int hh = static_cast<int>(h);
  if (dt == TP_BF16)
    TP_CUDA_TRY(launch_kernel(vocab_embed_bwd_kernel<__nv_bfloat16>, static_cast<unsigned>(v), kThreads, 0, st,
        ids, static_cast<const __nv_bfloat16*>(dx), static_cast<__nv_bfloat16*>(dE), M, hh,
        accumulate ? 1 : 0));
  else
    TP_CUDA_TRY(launch_kernel(vocab_embed_bwd_kernel<float>, static_cast<unsigned>(v), kThreads, 0, st,
        ids, static_cast<const float*>(dx), static_cast<float*>(dE), M, hh, accumulate ? 1 : 0));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

tp_status launch_vocab_ce_fwd(const void* logits, const int32_t* targets, float* lse,
                              float* row_loss, float* shard_loss, float* loss, int64_t M,
                              int64_t v, int N, tp_dtype dt, cudaStream_t st) {
  if (M <= 0) return TP_OK;
  if (M > 2147483647ll) return fail(TP_ERR_SHAPE, "too many rows for one launch");
  const unsigned g = static_cast<unsigned>(M);
  const bool vec = (v / N) % 8 == 0 && N <= kVecMaxShards &&
                   reinterpret_cast<uintptr_t>(logits) % 16 == 0;
  const unsigned gw = static_cast<unsigned>((M + kThreads / 32 - 1) / (kThreads / 32));
  if (dt == TP_BF16) {
    const auto* L = static_cast<const __nv_bfloat16*>(logits);
    if (vec) TP_CUDA_TRY(launch_kernel(vocab_ce_fwd_vec_kernel<__nv_bfloat16>, gw, kThreads, 0, st, L, targets, lse, row_loss, M, v, N));
    else TP_CUDA_TRY(launch_kernel(vocab_ce_fwd_kernel<__nv_bfloat16>, g, kThreads, 0, st, L, targets, lse, row_loss, v, N));
  } else {
    const auto* L = static_cast<const float*>(logits);
    if (vec) TP_CUDA_TRY(launch_kernel(vocab_ce_fwd_vec_kernel<float>, gw, kThreads, 0, st, L, targets, lse, row_loss, M, v, N));
    else TP_CUDA_TRY(launch_kernel(vocab_ce_fwd_kernel<float>, g, kThreads, 0, st, L, targets, lse, row_loss, v, N));
  }
  TP_CUDA_TRY(launch_kernel(vocab_ce_loss_kernel, 1, 1024, 0, st, row_loss, targets, shard_loss, loss, M, v, N));
  count_launch(2);
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

tp_status launch_vocab_ce_bwd(const void* logits, const int32_t* targets, const float* lse,
                              void* dlogits, int64_t M, int64_t v, float scale, tp_dtype dt,
                              cudaStream_t st) {
  if (M <= 0) return TP_OK;
  if (M > 2147483647ll) return fail(TP_ERR_SHAPE, "too many rows for one launch");
  const unsigned g = static_cast<unsigned>(M);
  const bool vec = v % 8 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(dlogits) % 16 == 0;
  if (dt == TP_BF16) {
    const auto* L = static_cast<const __nv_bfloat16*>(logits);
    auto* D = static_cast<__nv_bfloat16*>(dlogits);
    if (vec) TP_CUDA_TRY(launch_kernel(vocab_ce_bwd_vec_kernel<__nv_bfloat16>, g, kThreads, 0, st, L, targets, lse, D, v, scale));
    else TP_CUDA_TRY(launch_kernel(vocab_ce_bwd_kernel<__nv_bfloat16>, g, kThreads, 0, st, L, targets, lse, D, v, scale));
  } else {
    const auto* L = static_cast<const float*>(logits);
    auto* D = static_cast<float*>(dlogits);
    if (vec) TP_CUDA_TRY(launch_kernel(vocab_ce_bwd_vec_kernel<float>, g, kThreads, 0, st, L, targets, lse, D, v, scale));
    else TP_CUDA_TRY(launch_kernel(vocab_ce_bwd_kernel<float>, g, kThreads, 0, st, L, targets, lse, D, v, scale));
  }
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

tp_status launch_adamw(float* p, const float* g, float* m, float* v, int64_t n, float lr,
                       float b1, float b2, float eps, float wd, float bc1, float bc2,
                       cudaStream_t st) {
  if (n <= 0) return TP_OK;
  const int64_t blocks = std::min<int64_t>((n + kThreads - 1) / kThreads, 8ll * device_sm_count());
  TP_CUDA_TRY(launch_kernel(adamw_kernel, static_cast<unsigned>(blocks), kThreads, 0, st, p, g, m, v, n, lr, b1, b2,
                                                                    eps, wd, bc1, bc2));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

tp_status launch_adamw_dev(float* p, const float* g, float* m, float* v, int64_t n,
                           const int32_t* step, float lr, float b1, float b2, float eps, float wd,
                           cudaStream_t st) {
  if (n <= 0) return TP_OK;
  const int64_t blocks = std::min<int64_t>((n + kThreads - 1) / kThreads, 8ll * device_sm_count());
  TP_CUDA_TRY(launch_kernel(adamw_dev_kernel, static_cast<unsigned>(blocks), kThreads, 0, st, p, g, m, v, n, step, lr,
                                                                        b1, b2, eps, wd));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

tp_status launch_step_advance(int32_t* step, const float* loss, float* hist, int64_t hist_len,
                              cudaStream_t st) {
  TP_CUDA_TRY(launch_kernel(step_advance_kernel, 1, 1, 0, st, step, loss, hist, hist_len));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

}  // namespace tp
