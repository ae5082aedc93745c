// The shard sum that stands in for the all-reduce: out = sum_{i<N} P[i] (+ residual),
// shards added in order 0..N-1 in fp32. HBM-bound: every thread owns 8 consecutive
// elements, reads them from each partial with two 128-bit streaming loads (four
// shards' loads are issued before they are added, to keep bytes in flight) and
// writes 8 outputs with one 128-bit (bf16) or two (fp32) stores. Grid-stride over
// a grid of a few CTAs per SM.
//
// The fused variant adds the LayerNorm that must follow the sum (its statistics need
// the whole hidden width [张量并行 notes, §相关分析]): a group of 1..8 warps owns one
// row, keeps the row's sum on chip (8 elements per thread per 128-bit chunk),
// rounds it to the output type, takes mean and biased variance of the rounded values
// with warp shuffles and a shared-memory step, and writes the sum and the normalised
// row in the same pass, so the sum is never read back from HBM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace tp {
namespace {

__device__ __forceinline__ void add4(float* s, float4 v) {
  s[0] += v.x;
  s[1] += v.y;
  s[2] += v.z;
  s[3] += v.w;
}

__device__ __forceinline__ void load_res8(const __nv_bfloat16* R, int64_t e, float* r) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(R + e));
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[2 * i] = __uint_as_float(w[i] << 16);
    r[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load_res8(const float* R, int64_t e, float* r) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(R + e));
  const float4 b = __ldg(reinterpret_cast<const float4*>(R + e) + 1);
  r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
  r[4] = b.x; r[5] = b.y; r[6] = b.z; r[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* O, int64_t e, const float* s) {
  uint4 u;
  uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(s[2 * i], s[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(O + e) = u;
}
__device__ __forceinline__ void store8(float* O, int64_t e, const float* s) {
  reinterpret_cast<float4*>(O + e)[0] = make_float4(s[0], s[1], s[2], s[3]);
  reinterpret_cast<float4*>(O + e)[1] = make_float4(s[4], s[5], s[6], s[7]);
}

template <typename OutT>
__global__ void __launch_bounds__(256) shard_reduce_vec8(const float* __restrict__ P,
                                                         const OutT* __restrict__ R,
                                                         OutT* __restrict__ O, int N,
                                                         int64_t items, int64_t E) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < items;
       it += stride) {
    const int64_t e = it * 8;
    const float4* p0 = reinterpret_cast<const float4*>(P + e);
    float s[8];
    {
      const float4 a = __ldcs(p0), b = __ldcs(p0 + 1);
      s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
      s[4] = b.x; s[5] = b.y; s[6] = b.z; s[7] = b.w;
    }
    int i = 1;
    for (; i + 3 < N; i += 4) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4* q = reinterpret_cast<const float4*>(P + (i + j) * E + e);
        v[2 * j] = __ldcs(q);
        v[2 * j + 1] = __ldcs(q + 1);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        add4(s, v[2 * j]);
        add4(s + 4, v[2 * j + 1]);
      }
    }
    for (; i < N; ++i) {
      const float4* q = reinterpret_cast<const float4*>(P + i * E + e);
      add4(s, __ldcs(q));
      add4(s + 4, __ldcs(q + 1));
    }
    if (R) {
      float r[8];
      load_res8(R, e, r);
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] += r[k];
    }
    store8(O, e, s);
  }
}

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float& o, float v) { o = v; }
__device__ __forceinline__ void from_f(__nv_bfloat16& o, float v) { o = __float2bfloat16_rn(v); }

template <typename OutT>
__global__ void __launch_bounds__(256) shard_reduce_scalar(const float* __restrict__ P,
                                                           const OutT* __restrict__ R,
                                                           OutT* __restrict__ O, int N,
                                                           int64_t E, int64_t gs) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < E;
       e += stride) {
    float s = P[e];
    for (int i = 1; i < N; ++i) s += P[i * gs + e];
    if (R) s += to_f(R[e]);
    from_f(O[e], s);
  }
}

// E elements of each partial (shard i's at P + i gs) summed into O
template <typename OutT>
tp_status run(const float* P, const void* R, void* O, int N, int64_t E, int64_t gs,
              int blocks_per_sm, cudaStream_t st) {
  const bool vec = (E % 8 == 0) && (gs % 8 == 0) && (reinterpret_cast<uintptr_t>(P) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(O) % 16 == 0) &&
                   (R == nullptr || reinterpret_cast<uintptr_t>(R) % 16 == 0);
  const int64_t work = vec ? E / 8 : E;
  const int64_t blocks =
      std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(blocks_per_sm) * device_sm_count());
  if (vec)
    TP_CUDA_TRY(launch_kernel(shard_reduce_vec8<OutT>, static_cast<unsigned>(blocks), 256, 0, st,
        P, static_cast<const OutT*>(R), static_cast<OutT*>(O), N, work, gs));
  else
    TP_CUDA_TRY(launch_kernel(shard_reduce_scalar<OutT>, static_cast<unsigned>(blocks), 256, 0, st,
        P, static_cast<const OutT*>(R), static_cast<OutT*>(O), N, E, gs));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}


__device__ __forceinline__ float round_to(float v, const __nv_bfloat16*) {
  return __bfloat162float(__float2bfloat16_rn(v));
}
__device__ __forceinline__ float round_to(float v, const float*) { return v; }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// sum over the wpr warps of a row group; wpr is uniform over the CTA, so every
// thread reaches the barrier
__device__ __forceinline__ float group_sum(float v, float* red, int warp, int grp, int wpr) {
  v = warp_sum(v);
  if (wpr == 1) return v;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < wpr; ++w) t += red[grp * wpr + w];
  return t;
}

// One row per group of wpr warps (8 / wpr rows per CTA); thread t of the group owns
// the 8-element chunks t, t + G, ..., of the row (G = 32 wpr threads). The rounded sum
// of a thread's chunks waits in shared memory (slot [2 it + half][G] for its it-th
// chunk, read back only by the same thread, so no barrier is needed for it) rather
// than in registers: at ~40 registers a thread six CTAs fit on an SM, which keeps
// enough partial bytes in flight while other CTAs reduce and write.
#ifndef TP_RLN_UNROLL
#define TP_RLN_UNROLL 4  // shards whose loads are issued together
#endif
#ifndef TP_RLN_MINB
#define TP_RLN_MINB 1    // CTAs per SM the register allocation must allow
#endif
constexpr int kRlnUnroll = TP_RLN_UNROLL;

template <typename T>
__global__ void __launch_bounds__(256, TP_RLN_MINB) shard_reduce_ln_kernel(
    const float* __restrict__ P, const T* __restrict__ R, const float* __restrict__ gamma,
    const float* __restrict__ beta, T* __restrict__ S, T* __restrict__ Y, float* __restrict__ mean,
    float* __restrict__ rstd, int N, int64_t M, int h, float eps, int wpr, int iters) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  extern __shared__ float4 rowbuf[];
  __shared__ float red[2][8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / wpr, tig = (warp - grp * wpr) * 32 + lane, G = wpr * 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (8 / wpr) + grp;
  const bool live = row < M;
  const int64_t E = M * static_cast<int64_t>(h), base = row * h;
  float4* mine = rowbuf + static_cast<int64_t>(grp) * iters * 2 * G + tig;
  float s1 = 0.0f;
  if (live) {
    for (int it = 0; it < iters; ++it) {
      const int c = (it * G + tig) * 8;
      if (c >= h) break;
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = 0.0f;
#pragma unroll kRlnUnroll
      for (int i = 0; i < N; ++i) {
        const float4* q = reinterpret_cast<const float4*>(P + i * E + base + c);
        add4(v, __ldcs(q));
        add4(v + 4, __ldcs(q + 1));
      }
      if (R) {
        float r[8];
        load_res8(R, base + c, r);
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] += r[k];
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[k] = round_to(v[k], R);  // the stored sum is what LN normalises
        s1 += v[k];
      }
      mine[(2 * it) * G] = make_float4(v[0], v[1], v[2], v[3]);
      mine[(2 * it + 1) * G] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  const float mu = group_sum(s1, red[0], warp, grp, wpr) / h;
  float s2 = 0.0f;
  if (live) {
    for (int it = 0; it < iters; ++it) {
      if ((it * G + tig) * 8 >= h) break;
      const float4 a = mine[(2 * it) * G], b = mine[(2 * it + 1) * G];
      const float d[8] = {a.x - mu, a.y - mu, a.z - mu, a.w - mu,
                          b.x - mu, b.y - mu, b.z - mu, b.w - mu};
#pragma unroll
      for (int k = 0; k < 8; ++k) s2 += d[k] * d[k];
    }
  }
  const float rs = 1.0f / sqrtf(group_sum(s2, red[1], warp, grp, wpr) / h + eps);
  if (!live) return;
  for (int it = 0; it < iters; ++it) {
    const int c = (it * G + tig) * 8;
    if (c >= h) break;
    const float4 a = mine[(2 * it) * G], b = mine[(2 * it + 1) * G];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (S) store8(S, base + c, v);
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma + c));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma + c) + 1);
    const float4 b0 = __ldg(reinterpret_cast<const float4*>(beta + c));
    const float4 b1 = __ldg(reinterpret_cast<const float4*>(beta + c) + 1);
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    float y[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = g[k] * ((v[k] - mu) * rs) + bb[k];
    store8(Y, base + c, y);
  }
  if (tig == 0) {
    if (mean) mean[row] = mu;
    if (rstd) rstd[row] = rs;
  }
}

template <typename T>
tp_status run_ln(const float* P, const void* R, const float* gamma, const float* beta, void* S,
                 void* Y, float* mean, float* rstd, int N, int64_t M, int h, float eps,
                 cudaStream_t st) {
  const int chunks = h / 8;
  int G = 32;
  while (G < chunks && G < 256) G *= 2;
  const int wpr = G / 32, rows = 8 / wpr, iters = (chunks + G - 1) / G;
  const size_t smem = static_cast<size_t>(rows) * iters * 2 * G * sizeof(float4);
  static std::atomic<uint64_t> attr_set{0};  // per device; h <= 16384: at most 64 KB
  if (needs_setup(attr_set)) {
    TP_CUDA_TRY(cudaFuncSetAttribute(shard_reduce_ln_kernel<T>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024));
    mark_device(attr_set);
  }
  const int64_t blocks = (M + rows - 1) / rows;
  if (blocks > 2147483647ll) return fail(TP_ERR_SHAPE, "too many rows for one launch");
  TP_CUDA_TRY(launch_kernel(shard_reduce_ln_kernel<T>, static_cast<unsigned>(blocks), 256, smem, st,
      P, static_cast<const T*>(R), gamma, beta, static_cast<T*>(S), static_cast<T*>(Y), mean,
      rstd, N, M, h, eps, wpr, iters));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

}  // namespace

tp_status launch_shard_reduce(const float* P, const void* residual, void* out, int N, int64_t M,
                              int64_t n, tp_dtype out_dtype, cudaStream_t st, int blocks_per_sm,
                              int64_t group_stride) {
  const int64_t E = M * n;
  if (E <= 0) return TP_OK;
  const int64_t gs = group_stride > 0 ? group_stride : E;
  blocks_per_sm = std::max(1, std::min(blocks_per_sm, 8));
  return out_dtype == TP_BF16 ? run<__nv_bfloat16>(P, residual, out, N, E, gs, blocks_per_sm, st)
                              : run<float>(P, residual, out, N, E, gs, blocks_per_sm, st);
}

tp_status launch_shard_reduce_ln(const float* P, const void* residual, const float* gamma,
                                 const float* beta, void* sum_out, void* y, float* mean,
                                 float* rstd, int N, int64_t M, int64_t h, float eps,
                                 tp_dtype dt, cudaStream_t st) {
  if (M <= 0) return TP_OK;
  const int hh = static_cast<int>(h);
  return dt == TP_BF16
             ? run_ln<__nv_bfloat16>(P, residual, gamma, beta, sum_out, y, mean, rstd, N, M, hh, eps, st)
             : run_ln<float>(P, residual, gamma, beta, sum_out, y, mean, rstd, N, M, hh, eps, st);
}

}  // namespace tp
