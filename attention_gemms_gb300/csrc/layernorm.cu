// LayerNorm over the full hidden width, forward and backward, with the residual
// add of the backward fused in:
//   y  = gamma * (x - mu) * rstd + beta,  rstd = 1 / sqrt(var + eps), biased variance
//   dx = dres + rstd * (g - mean(g) - xhat * mean(g * xhat)),  g = dy * gamma
//   dgamma = sum_rows dy * xhat,  dbeta = sum_rows dy
// (LN formula of the 张量并行 notes, §相关分析; the statistics need the whole hidden
// width, which is why the shard sum precedes it.)
// Row kernels use one warp per row; the parameter gradients are column sums taken
// in a fixed order (per-chunk partials, then a second pass over the chunks), so
// results are deterministic. When a row is a whole number of 16-byte vectors
// (h * sizeof(T) % 16 == 0, every buffer 16-byte aligned) the kernels move 16 bytes
// per lane and access; the row's later passes hit L1 / L2, so x and dy are read from
// DRAM once. Other widths take the scalar kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

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
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
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
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
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

// 16 bytes of T as floats
template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
  using Raw = float4;
  __device__ static void unpack(const Raw& r, float (&f)[4]) {
    f[0] = r.x;
    f[1] = r.y;
    f[2] = r.z;
    f[3] = r.w;
  }
  __device__ static Raw pack(const float (&f)[4]) { return make_float4(f[0], f[1], f[2], f[3]); }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  using Raw = uint4;
  __device__ static void unpack(const Raw& r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ static Raw pack(const float (&f)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<const uint32_t*>(&t);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};
// N consecutive fp32 parameters starting at a multiple of N
template <int N>
__device__ __forceinline__ void ld_params(const float* __restrict__ p, int64_t v, float (&f)[N]) {
  const float4* p4 = reinterpret_cast<const float4*>(p) + v * (N / 4);
#pragma unroll
  for (int k = 0; k < N / 4; ++k) {
    const float4 t = __ldg(p4 + k);
    f[4 * k] = t.x;
    f[4 * k + 1] = t.y;
    f[4 * k + 2] = t.z;
    f[4 * k + 3] = t.w;
  }
}

template <typename T>
__global__ void __launch_bounds__(32 * kRowWarps) ln_fwd_vec_kernel(
    const T* __restrict__ x, const float* __restrict__ gamma, const float* __restrict__ beta,
    T* __restrict__ y, float* mean, float* rstd, int64_t M, int h, float eps) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using V = Vec<T>;
  constexpr int E = V::N;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const int nv = h / E;
  const typename V::Raw* xr = reinterpret_cast<const typename V::Raw*>(x + row * h);
  float s = 0.0f;
#pragma unroll 8
  for (int v = lane; v < nv; v += 32) {
    float f[E];
    V::unpack(xr[v], f);
#pragma unroll
    for (int e = 0; e < E; ++e) s += f[e];
  }
  const float mu = warp_sum(s) / h;
  float q = 0.0f;
#pragma unroll 4
  for (int v = lane; v < nv; v += 32) {
    float f[E];
    V::unpack(xr[v], f);
#pragma unroll
    for (int e = 0; e < E; ++e) q += (f[e] - mu) * (f[e] - mu);
  }
  const float rs = 1.0f / sqrtf(warp_sum(q) / h + eps);
  typename V::Raw* yr = reinterpret_cast<typename V::Raw*>(y + row * h);
#pragma unroll 4
  for (int v = lane; v < nv; v += 32) {
    float f[E], g[E], b[E];
    V::unpack(xr[v], f);
    ld_params<E>(gamma, v, g);
    ld_params<E>(beta, v, b);
#pragma unroll
    for (int e = 0; e < E; ++e) f[e] = g[e] * ((f[e] - mu) * rs) + b[e];
    yr[v] = V::pack(f);
  }
  if (lane == 0) {
    if (mean) mean[row] = mu;
    if (rstd) rstd[row] = rs;
  }
}

template <typename T>
__global__ void __launch_bounds__(32 * kRowWarps) ln_bwd_dx_vec_kernel(
    const T* __restrict__ x, const float* __restrict__ gamma, const float* __restrict__ mean,
    const float* __restrict__ rstd, const T* __restrict__ dy, const T* __restrict__ dres,
    T* __restrict__ dx, int64_t M, int h) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using V = Vec<T>;
  constexpr int E = V::N;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const float mu = mean[row], rs = rstd[row];
  const int nv = h / E;
  const typename V::Raw* xr = reinterpret_cast<const typename V::Raw*>(x + row * h);
  const typename V::Raw* dyr = reinterpret_cast<const typename V::Raw*>(dy + row * h);
  float s1 = 0.0f, s2 = 0.0f;
#pragma unroll 8
  for (int v = lane; v < nv; v += 32) {
    float a[E], d[E], g[E];
    V::unpack(xr[v], a);
    V::unpack(dyr[v], d);
    ld_params<E>(gamma, v, g);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float gg = d[e] * g[e];
      s1 += gg;
      s2 += gg * (a[e] - mu) * rs;
    }
  }
  s1 = warp_sum(s1) / h;
  s2 = warp_sum(s2) / h;
  const typename V::Raw* rr = dres ? reinterpret_cast<const typename V::Raw*>(dres + row * h) : nullptr;
  typename V::Raw* out = reinterpret_cast<typename V::Raw*>(dx + row * h);
#pragma unroll 4
  for (int v = lane; v < nv; v += 32) {
    float a[E], d[E], g[E], r[E];
    V::unpack(xr[v], a);
    V::unpack(dyr[v], d);
    ld_params<E>(gamma, v, g);
    if (rr) {
      V::unpack(rr[v], r);
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) r[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float xh = (a[e] - mu) * rs;
      a[e] = rs * (d[e] * g[e] - s1 - xh * s2) + r[e];
    }
    out[v] = V::pack(a);
  }
}

constexpr int kColThreads = 256;
constexpr int kRowsPerChunk = 64;

// The parameter-gradient partials of one chunk of rows, vectorised: lane j of every
// warp owns the 16-byte column vector blockIdx.x * 32 + j; warp w sums rows
// w, w + 8, ... of the chunk in order, then the eight warps' sums are added in warp
// order (fixed, so deterministic). Same chunking and output as the scalar kernel below.
template <typename T>
__global__ void __launch_bounds__(32 * kRowWarps) ln_bwd_param_partial_vec_kernel(
    const T* __restrict__ x, const float* __restrict__ mean, const float* __restrict__ rstd,
    const T* __restrict__ dy, float* __restrict__ partial, int64_t M, int h, int64_t rank_rows,
    int cpr) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using V = Vec<T>;
  constexpr int E = V::N;
  __shared__ float red[kRowWarps][32][2 * E + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = blockIdx.x * 32 + lane, nv = h / E;
  const int rank = blockIdx.y / cpr, chunk = blockIdx.y - rank * cpr;
  const int64_t rank_end = min(M, (rank + 1) * rank_rows);
  const int64_t r0 = rank * rank_rows + static_cast<int64_t>(chunk) * kRowsPerChunk;
  const int64_t r1 = min(rank_end, r0 + kRowsPerChunk);
  float sg[E], sb[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = sb[e] = 0.0f;
  if (v < nv) {
#pragma unroll 8
    for (int64_t r = r0 + warp; r < r1; r += kRowWarps) {
      float a[E], d[E];
      V::unpack(reinterpret_cast<const typename V::Raw*>(x + r * h)[v], a);
      V::unpack(reinterpret_cast<const typename V::Raw*>(dy + r * h)[v], d);
      const float mu = mean[r], rs = rstd[r];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sg[e] += d[e] * (a[e] - mu) * rs;
        sb[e] += d[e];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    red[warp][lane][e] = sg[e];
    red[warp][lane][E + e] = sb[e];
  }
  __syncthreads();
  // thread (warp w, lane j): output element w of the 2E values of column vector j
  for (int k = warp; k < 2 * E; k += kRowWarps) {
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kRowWarps; ++w) t += red[w][lane][k];
    if (v < nv) {
      const int e = k < E ? k : k - E;
      partial[blockIdx.y * 2ll * h + (k < E ? 0 : h) + static_cast<int64_t>(v) * E + e] = t;
    }
  }
}

// The partials and their final sum in one launch, for the replicated LN (one rank) with
// at most kClusterChunks chunks of at most kRowsPerChunk rows, or kMaxClusterChunks where
// the device places such clusters (larger inputs keep the partial and final kernels,
// whose grid has more CTAs): the CTAs of a cluster (1 x chunks) take the chunks of
// one block of 32 column vectors, each keeps its chunk's sums in shared memory, and
// after a cluster barrier CTA c adds up its share of the block's 2E x 32 outputs over
// the cluster's CTAs in chunk order (distributed shared memory) and writes dgamma and
// dbeta. A fixed order, so deterministic; no workspace and no second launch.
constexpr int kClusterChunks = 8;      // portable cluster size
constexpr int kMaxClusterChunks = 16;  // with the non-portable opt-in, where it can be placed

template <typename T>
__global__ void __launch_bounds__(32 * kRowWarps) ln_bwd_param_cluster_vec_kernel(
    const T* __restrict__ x, const float* __restrict__ mean, const float* __restrict__ rstd,
    const T* __restrict__ dy, float* __restrict__ dgamma, float* __restrict__ dbeta, int64_t M,
    int h, int64_t rows_per_chunk) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using V = Vec<T>;
  constexpr int E = V::N;
  __shared__ float red[kRowWarps][32][2 * E + 1];
  __shared__ float tot[2 * E][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = blockIdx.x * 32 + lane, nv = h / E;
  const int chunk = static_cast<int>(cluster_ctarank()), chunks = gridDim.y;
  const int64_t r0 = static_cast<int64_t>(chunk) * rows_per_chunk;
  const int64_t r1 = min(M, r0 + rows_per_chunk);
  float sg[E], sb[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sg[e] = sb[e] = 0.0f;
  if (v < nv) {
#pragma unroll 8
    for (int64_t r = r0 + warp; r < r1; r += kRowWarps) {
      float a[E], d[E];
      V::unpack(reinterpret_cast<const typename V::Raw*>(x + r * h)[v], a);
      V::unpack(reinterpret_cast<const typename V::Raw*>(dy + r * h)[v], d);
      const float mu = mean[r], rs = rstd[r];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        sg[e] += d[e] * (a[e] - mu) * rs;
        sb[e] += d[e];
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) {
    red[warp][lane][e] = sg[e];
    red[warp][lane][E + e] = sb[e];
  }
  __syncthreads();
  for (int k = warp; k < 2 * E; k += kRowWarps) {  // the chunk's sums, warps in order
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kRowWarps; ++w) t += red[w][lane][k];
    tot[k][lane] = t;
  }
  cluster_sync_all();  // every chunk's sums are in its CTA's shared memory
  const int per = (2 * E * 32 + chunks - 1) / chunks;
  for (int o = chunk * per + static_cast<int>(threadIdx.x); o < min(2 * E * 32, (chunk + 1) * per);
       o += blockDim.x) {
    const int k = o / 32, j = o % 32;
    const uint32_t addr = smem_u32(&tot[k][j]);
    float t = 0.0f;
    for (int q = 0; q < chunks; ++q) t += ld_cluster_f32(mapa_shared(addr, static_cast<uint32_t>(q)));
    const int vv = blockIdx.x * 32 + j;
    if (vv < nv) {
      const int e = k < E ? k : k - E;
      float* dst = k < E ? dgamma : dbeta;
      if (dst) dst[static_cast<int64_t>(vv) * E + e] = t;
    }
  }
  cluster_sync_all();  // no CTA leaves while another still reads its sums
}

// partial[chunk][0:h] = sum over the chunk's rows of dy * xhat, partial[chunk][h:2h] = of dy.
// Rows are grouped by rank (rank r owns rows [r * rank_rows, (r + 1) * rank_rows), one
// rank when the LN input is replicated) and each rank's rows are cut into cpr chunks
// of at most kRowsPerChunk rows; chunk index = r * cpr + c.
template <typename T>
__global__ void __launch_bounds__(kColThreads) ln_bwd_param_partial_kernel(
    const T* __restrict__ x, const float* __restrict__ mean, const float* __restrict__ rstd,
    const T* __restrict__ dy, float* __restrict__ partial, int64_t M, int h, int64_t rank_rows,
    int cpr) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
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

constexpr int kFinalCols = 64, kFinalGroups = 4;  // columns per CTA, chunk groups per column

// per rank: the sum of its chunks (written to dgamma_ranks / dbeta_ranks (ranks, h)
// when given); then the sum over the ranks in rank order. A rank's chunks are split
// into kFinalGroups consecutive groups summed in parallel, each in chunk order, and
// the group sums are added in group order: a fixed order, so results are deterministic.
__global__ void __launch_bounds__(kFinalCols * kFinalGroups) ln_bwd_param_final_kernel(
    const float* __restrict__ partial, int ranks, int cpr, int h, float* dgamma, float* dbeta,
    float* dgamma_ranks, float* dbeta_ranks) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  __shared__ float red[kFinalGroups][2][kFinalCols];
  const int cl = threadIdx.x % kFinalCols, q = threadIdx.x / kFinalCols;
  const int c = blockIdx.x * kFinalCols + cl;
  const int per = (cpr + kFinalGroups - 1) / kFinalGroups;
  float tg = 0.0f, tb = 0.0f;
  for (int r = 0; r < ranks; ++r) {
    const int k0 = r * cpr + q * per, k1 = min((r + 1) * cpr, k0 + per);
    float sg = 0.0f, sb = 0.0f;
    if (c < h) {
#pragma unroll 8
      for (int k = k0; k < k1; ++k) {
        sg += partial[k * 2ll * h + c];
        sb += partial[k * 2ll * h + h + c];
      }
    }
    red[q][0][cl] = sg;
    red[q][1][cl] = sb;
    __syncthreads();
    if (q == 0 && c < h) {
      float g = 0.0f, b = 0.0f;
#pragma unroll
      for (int i = 0; i < kFinalGroups; ++i) {
        g += red[i][0][cl];
        b += red[i][1][cl];
      }
      if (dgamma_ranks) dgamma_ranks[static_cast<int64_t>(r) * h + c] = g;
      if (dbeta_ranks) dbeta_ranks[static_cast<int64_t>(r) * h + c] = b;
      tg += g;
      tb += b;
    }
    __syncthreads();
  }
  if (q == 0 && c < h) {
    if (dgamma) dgamma[c] = tg;
    if (dbeta) dbeta[c] = tb;
  }
}

// Whether the device places clusters of `chunks` CTAs of the parameter-sum kernel (16
// needs the non-portable opt-in): asked once per device, before the first such launch.
template <typename T>
bool cluster_fits(int chunks) {
  static std::atomic<int> known[64];  // 0 unknown, 1 fits, 2 does not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (known[dev].load() != 0) return known[dev].load() == 1;
  auto kern = ln_bwd_param_cluster_vec_kernel<T>;
  bool fits = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
              cudaSuccess;
  if (fits) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(chunks);
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(1, static_cast<unsigned>(chunks), 1);
    cfg.blockDim = dim3(32 * kRowWarps, 1, 1);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    fits = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
  }
  if (!fits) cudaGetLastError();  // the query's own error, not a launch's
  known[dev].store(fits ? 1 : 2);
  return fits;
}

// whole 16-byte vectors per row (the buffers themselves are 16-byte aligned)
template <typename T>
bool vec_rows(int h) {
  return (static_cast<int64_t>(h) * sizeof(T)) % 16 == 0;
}

template <typename T>
tp_status fwd_t(const void* x, const float* gamma, const float* beta, void* y, float* mean,
                float* rstd, int64_t M, int h, float eps, cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>((M + kRowWarps - 1) / kRowWarps);
  if (vec_rows<T>(h))
    TP_CUDA_TRY(launch_kernel(ln_fwd_vec_kernel<T>, blocks, 32 * kRowWarps, 0, st,
        static_cast<const T*>(x), gamma, beta, static_cast<T*>(y), mean, rstd, M, h, eps));
  else
    TP_CUDA_TRY(launch_kernel(ln_fwd_kernel<T>, blocks, 32 * kRowWarps, 0, st, static_cast<const T*>(x), gamma, beta,
                                                         static_cast<T*>(y), mean, rstd, M, h, eps));
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
  const bool vec = vec_rows<T>(h);
  if (vec)
    TP_CUDA_TRY(launch_kernel(ln_bwd_dx_vec_kernel<T>, rblocks, 32 * kRowWarps, 0, st,
        static_cast<const T*>(x), gamma, mean, rstd, static_cast<const T*>(dy),
        static_cast<const T*>(dres), static_cast<T*>(dx), M, h));
  else
    TP_CUDA_TRY(launch_kernel(ln_bwd_dx_kernel<T>, rblocks, 32 * kRowWarps, 0, st,
        static_cast<const T*>(x), gamma, mean, rstd, static_cast<const T*>(dy),
        static_cast<const T*>(dres), static_cast<T*>(dx), M, h));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  if (!dgamma && !dbeta && !dgamma_ranks && !dbeta_ranks) return TP_OK;
  const int64_t want_chunks = (M + kRowsPerChunk - 1) / kRowsPerChunk;
  if (vec && ranks == 1 && !dgamma_ranks && !dbeta_ranks &&
      (want_chunks <= kClusterChunks ||
       (want_chunks <= kMaxClusterChunks && cluster_fits<T>(kMaxClusterChunks)))) {
    const int chunks = static_cast<int>(
        want_chunks <= kClusterChunks ? std::max<int64_t>(1, want_chunks) : kMaxClusterChunks);
    const int64_t rows_per_chunk = (M + chunks - 1) / chunks;
    constexpr int cols = 32 * Vec<T>::N;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(chunks);
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>((h + cols - 1) / cols), static_cast<unsigned>(chunks), 1);
    cfg.blockDim = dim3(32 * kRowWarps, 1, 1);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    TP_CUDA_TRY(cudaLaunchKernelEx(&cfg, ln_bwd_param_cluster_vec_kernel<T>,
                                   static_cast<const T*>(x), mean, rstd, static_cast<const T*>(dy),
                                   dgamma, dbeta, M, h, rows_per_chunk));
    count_launch();
    return TP_OK;
  }
  const int64_t rank_rows = M / ranks;
  const int cpr = static_cast<int>((rank_rows + kRowsPerChunk - 1) / kRowsPerChunk);
  if (vec) {
    constexpr int cols = 32 * Vec<T>::N;  // columns per CTA
    const dim3 g1((h + cols - 1) / cols, ranks * cpr);
    TP_CUDA_TRY(launch_kernel(ln_bwd_param_partial_vec_kernel<T>, g1, 32 * kRowWarps, 0, st,
        static_cast<const T*>(x), mean, rstd, static_cast<const T*>(dy), ws, M, h, rank_rows, cpr));
  } else {
    const dim3 g1((h + kColThreads - 1) / kColThreads, ranks * cpr);
    TP_CUDA_TRY(launch_kernel(ln_bwd_param_partial_kernel<T>, g1, kColThreads, 0, st,
        static_cast<const T*>(x), mean, rstd, static_cast<const T*>(dy), ws, M, h, rank_rows, cpr));
  }
  TP_CUDA_TRY(launch_kernel(ln_bwd_param_final_kernel, (h + kFinalCols - 1) / kFinalCols, kFinalCols * kFinalGroups, 0, st,
      ws, ranks, cpr, h, dgamma, dbeta, dgamma_ranks, dbeta_ranks));
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
