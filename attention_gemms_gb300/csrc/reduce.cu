// The shard sum that stands in for the all-reduce: out = sum_{i<N} P[i] (+ residual),
// shards added in order 0..N-1 in fp32. HBM-bound: every thread owns 8 consecutive
// elements, reads them from each partial with two 128-bit streaming loads (four
// shards' loads are issued before they are added, to keep bytes in flight) and
// writes 8 outputs with one 128-bit (bf16) or two (fp32) stores. Grid-stride over
// a grid of a few CTAs per SM.
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
                                                           int64_t E) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < E;
       e += stride) {
    float s = P[e];
    for (int i = 1; i < N; ++i) s += P[i * E + e];
    if (R) s += to_f(R[e]);
    from_f(O[e], s);
  }
}

template <typename OutT>
tp_status run(const float* P, const void* R, void* O, int N, int64_t E, cudaStream_t st) {
  const bool vec = (E % 8 == 0) && (reinterpret_cast<uintptr_t>(P) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(O) % 16 == 0) &&
                   (R == nullptr || reinterpret_cast<uintptr_t>(R) % 16 == 0);
  const int64_t work = vec ? E / 8 : E;
  const int64_t blocks = std::min<int64_t>((work + 255) / 256, 8ll * device_sm_count());
  if (vec)
    shard_reduce_vec8<OutT><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        P, static_cast<const OutT*>(R), static_cast<OutT*>(O), N, work, E);
  else
    shard_reduce_scalar<OutT><<<static_cast<unsigned>(blocks), 256, 0, st>>>(
        P, static_cast<const OutT*>(R), static_cast<OutT*>(O), N, E);
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

}  // namespace

tp_status launch_shard_reduce(const float* P, const void* residual, void* out, int N, int64_t M,
                              int64_t n, tp_dtype out_dtype, cudaStream_t st) {
  const int64_t E = M * n;
  if (E <= 0) return TP_OK;
  return out_dtype == TP_BF16 ? run<__nv_bfloat16>(P, residual, out, N, E, st)
                              : run<float>(P, residual, out, N, E, st);
}

}  // namespace tp
