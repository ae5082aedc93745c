// Decode GEMV for one token (the kernel is written for up to 4): out[t, n] = sum_k X[t, k] W[k, n] with W (K x N)
// row-major, streamed from HBM once. Memory-bound (arithmetic intensity ~ T FLOP per
// weight byte [20260402-parallelism, Decode 阶段, 线性层]), so CUDA cores suffice and
// the kernel is about keeping bytes in flight:
//   * a CTA owns a strip of 64 output columns (128 bytes of every weight row) and a
//     K range (the whole K, or one shard's K slice for the row-parallel partials);
//   * lane l of warp w reads 16 bytes (8 columns) of rows k = 4 w + l / 8 (mod 32),
//     four (paired gate/up) or eight rows per thread per step, with non-allocating
//     128-bit loads;
//   * the four row groups of a warp are summed with warp shuffles, the eight warps
//     through shared memory in a fixed order, then the epilogue runs (SwiGLU of the
//     gate/up pair, GELU, plain store, or the fp32 shard partial).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "epi_math.cuh"
#include "internal.h"

namespace tp {
namespace {

constexpr int kStrip = 64;
constexpr int kWarps = 8;

struct GemvParams {
  const __nv_bfloat16* X;   // (T, K) row-major, ld = ldx
  const __nv_bfloat16* W;   // (K, N), ld = ldw
  const __nv_bfloat16* Wu;  // second weight (SwiGLU up), same layout
  int64_t ldx, ldw, N, K, kg;
  void* out0;
  void* out1;
  void* out2;
  int64_t ldo, group_stride;
};

__device__ __forceinline__ uint4 ld_stream(const __nv_bfloat16* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void unpack(uint4 r, float* v) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void st_bf16(void* base, int64_t i, float v) {
  reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

template <int T, int EPI, bool PAIRED>
__global__ void __launch_bounds__(32 * kWarps) gemv_kernel(const GemvParams p) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  // rows in flight per thread: the paired (gate/up) kernel streams two weights
  constexpr int kUnroll = PAIRED ? 4 : 8;
  __shared__ float red[PAIRED ? 2 : 1][kWarps][T][kStrip];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rsub = lane >> 3, c8 = (lane & 7) * 8;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * kStrip;
  const int g = blockIdx.y;
  const int64_t kb = g * p.kg, ke = min(p.K, kb + p.kg);
  const bool col_ok = n0 + c8 < p.N;  // N % 8 == 0: all 8 columns valid or none
  float acc[T][8], acc2[PAIRED ? T : 1][8];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[t][j] = 0.0f;
      if constexpr (PAIRED) acc2[t][j] = 0.0f;
    }
  const __nv_bfloat16* wcol = p.W + n0 + c8;
  const __nv_bfloat16* ucol = PAIRED ? p.Wu + n0 + c8 : nullptr;
  int64_t k = kb + warp * 4 + rsub;
  // main loop: kUnroll rows per thread in flight (plus their up-projection rows)
  for (; k + 32 * (kUnroll - 1) < ke; k += 32 * kUnroll) {
    uint4 wv[kUnroll], uv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      wv[u] = col_ok ? ld_stream(wcol + (k + 32 * u) * p.ldw) : make_uint4(0, 0, 0, 0);
      if constexpr (PAIRED)
        uv[u] = col_ok ? ld_stream(ucol + (k + 32 * u) * p.ldw) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float wf[8], uf[8];
      unpack(wv[u], wf);
      if constexpr (PAIRED) unpack(uv[u], uf);
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const float xv = __bfloat162float(__ldg(p.X + t * p.ldx + k + 32 * u));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[t][j] = fmaf(xv, wf[j], acc[t][j]);
          if constexpr (PAIRED) acc2[t][j] = fmaf(xv, uf[j], acc2[t][j]);
        }
      }
    }
  }
  for (; k < ke; k += 32) {  // tail rows
    float wf[8], uf[8];
    unpack(col_ok ? ld_stream(wcol + k * p.ldw) : make_uint4(0, 0, 0, 0), wf);
    if constexpr (PAIRED) unpack(col_ok ? ld_stream(ucol + k * p.ldw) : make_uint4(0, 0, 0, 0), uf);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const float xv = __bfloat162float(__ldg(p.X + t * p.ldx + k));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc[t][j] = fmaf(xv, wf[j], acc[t][j]);
        if constexpr (PAIRED) acc2[t][j] = fmaf(xv, uf[j], acc2[t][j]);
      }
    }
  }
  // the four row groups of the warp (lanes l, l^8, l^16, l^24 share columns)
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float v = acc[t][j];
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
      if (rsub == 0) red[0][warp][t][c8 + j] = v;
      if constexpr (PAIRED) {
        float u = acc2[t][j];
        u += __shfl_xor_sync(0xFFFFFFFFu, u, 8);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, 16);
        if (rsub == 0) red[1][warp][t][c8 + j] = u;
      }
    }
  __syncthreads();
  // epilogue: thread -> (t, column) of the strip; warps summed in order 0..7
  for (int e = threadIdx.x; e < T * kStrip; e += 32 * kWarps) {
    const int t = e / kStrip, cc = e % kStrip;
    const int64_t n = n0 + cc;
    if (n >= p.N) continue;
    float a = 0.0f, b = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      a += red[0][w][t][cc];
      if constexpr (PAIRED) b += red[1][w][t][cc];
    }
    const int64_t i = t * p.ldo + n;
    if constexpr (EPI == EPI_SWIGLU) {
      if (p.out0) st_bf16(p.out0, i, a);
      if (p.out1) st_bf16(p.out1, i, b);
      st_bf16(p.out2, i, silu_sfu(a) * b);
    } else if constexpr (EPI == EPI_GELU) {
      if (p.out0) st_bf16(p.out0, i, a);
      st_bf16(p.out1, i, gelu_f(a));
    } else {  // EPI_STORE: fp32 partial of K group g, or the bf16 output
      if (p.group_stride >= 0)
        reinterpret_cast<float*>(p.out0)[g * p.group_stride + i] = a;
      else
        st_bf16(p.out0, i, a);
    }
  }
}

template <int T>
tp_status launch_t(int epi, bool paired, const GemvParams& p, dim3 grid, cudaStream_t st) {
  if (epi == EPI_SWIGLU && paired) TP_CUDA_TRY(launch_kernel(gemv_kernel<T, EPI_SWIGLU, true>, grid, 32 * kWarps, 0, st, p));
  else if (epi == EPI_GELU) TP_CUDA_TRY(launch_kernel(gemv_kernel<T, EPI_GELU, false>, grid, 32 * kWarps, 0, st, p));
  else if (epi == EPI_STORE) TP_CUDA_TRY(launch_kernel(gemv_kernel<T, EPI_STORE, false>, grid, 32 * kWarps, 0, st, p));
  else return fail(TP_ERR_INVALID_ARG, "GEMV epilogue not supported");
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

}  // namespace

// Whether a GEMM is a decode-sized (M <= 4) bf16 problem this kernel handles: K-major
// X, MN-major W (as the column- and row-parallel linears store them), one K segment;
// every other problem goes to the tensor-core engine.
bool gemv_eligible(const GemmDesc& d) {
  // one token: at two or more the register cost of the per-token accumulators cuts the
  // CTAs per SM, and with them the bytes in flight, below the tensor-core path's
  if (d.dtype != TP_BF16 || d.M != 1 || d.a_mn || !d.b_mn || d.nseg != 1) return false;
  if (d.epi == EPI_SWIGLU) { if (!d.paired) return false; }
  else if (d.epi == EPI_GELU || d.epi == EPI_STORE) { if (d.paired) return false; }
  else return false;
  if (d.epi == EPI_STORE && d.in[0]) return false;  // residual handled by the engine
  if (d.epi == EPI_STORE && !d.out_f32 && d.groups != 1) return false;
  // enough 64-column strips to occupy every SM twice (e.g. not a split-K fold of a
  // narrow output, which would leave most SMs idle)
  if ((d.N + kStrip - 1) / kStrip * d.groups < 2 * device_sm_count()) return false;
  if (d.N % 8 || d.B[0].ld % 8 || (d.paired && d.B[1].ld != d.B[0].ld)) return false;
  return true;
}

tp_status launch_gemv(const GemmDesc& d, cudaStream_t st) {
  GemvParams p{};
  p.X = static_cast<const __nv_bfloat16*>(d.A[0].ptr);
  p.W = static_cast<const __nv_bfloat16*>(d.B[0].ptr);
  p.Wu = d.paired ? static_cast<const __nv_bfloat16*>(d.B[1].ptr) : nullptr;
  p.ldx = d.A[0].ld;
  p.ldw = d.B[0].ld;
  p.N = d.N;
  p.K = d.groups * d.K;
  p.kg = d.K;
  p.out0 = d.out[0];
  p.out1 = d.out[1];
  p.out2 = d.out[2];
  p.ldo = d.ldo;
  p.group_stride = (d.epi == EPI_STORE && d.out_f32) ? d.out_group_stride : -1;
  if (d.epi == EPI_STORE && d.out_f32 && d.groups == 1) p.group_stride = 0;
  const int64_t gx = (d.N + kStrip - 1) / kStrip;
  if (gx > 2147483647ll || d.groups > 65535) return fail(TP_ERR_SHAPE, "GEMV grid too large");
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(d.groups));
  switch (d.M) {
    case 1: return launch_t<1>(d.epi, d.paired, p, grid, st);
    case 2: return launch_t<2>(d.epi, d.paired, p, grid, st);
    case 3: return launch_t<3>(d.epi, d.paired, p, grid, st);
    default: return launch_t<4>(d.epi, d.paired, p, grid, st);
  }
}

}  // namespace tp
