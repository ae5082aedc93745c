// fp32 GEMM engine on CUDA cores (FFMA, no TF32: TF32's 10-bit mantissa would not
// hold the fp32 path to 1e-5). Same problem descriptor and epilogues as the
// tensor-core engine; 64 x 64 output tile per CTA, 4 x 4 per thread, K in steps of 32.
// Each thread gathers a whole K step of A and B into registers before storing it to
// shared memory, and the next step's loads are issued before the current step's FMAs,
// so one load latency per step is hidden behind the arithmetic instead of several
// being paid in a row (the small fp32 GEMMs are latency-bound).
// When the output has few tiles (fewer than half the SMs), the K steps of a tile are
// split over the CTAs of a thread-block cluster (2, 4 or 8): each CTA accumulates its
// share, parks the partial tile in shared memory, and after a cluster barrier CTA r
// sums row slice r of the tile over the cluster's CTAs in rank order (distributed
// shared memory) and runs the epilogue on it. The order of the sum is fixed, so the
// result is deterministic; no workspace is needed.
#include <cuda_runtime.h>

#include <atomic>

#include <algorithm>

#include "epi_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int TM = 64, TN = 64, TK = 32;
constexpr int kPer = TM * TK / 256;  // elements of A (and of each B) per thread per K step

struct SimtParams {
  const float* A[3];
  const float* B[3];
  int64_t lda[3], ldb[3], k0[3];
  int64_t M, N, K;
  int a_mn, b_mn, nseg, paired;
  float* out0;
  float* out1;
  float* out2;
  const float* in0;
  const float* in1;
  int64_t ldo, out_group_stride;
  int split;  // CTAs of a cluster sharing one output tile's K steps (1: no split)
};


template <int EPI>
__device__ __forceinline__ void epi1(const SimtParams& p, int g, int64_t r, int64_t c, float a,
                                     float b) {
  const int64_t i = r * p.ldo + c;
  if constexpr (EPI == EPI_STORE) {
    p.out0[g * p.out_group_stride + i] = a + (p.in0 ? p.in0[i] : 0.0f);
  } else if constexpr (EPI == EPI_GELU) {
    if (p.out0) p.out0[i] = a;
    p.out1[i] = gelu_f(a);
  } else if constexpr (EPI == EPI_SWIGLU) {
    if (p.out0) p.out0[i] = a;
    if (p.out1) p.out1[i] = b;
    p.out2[i] = silu_f(a) * b;
  } else if constexpr (EPI == EPI_DGELU) {
    p.out0[i] = a * gelu_prime_f(p.in0[i]);
  } else if constexpr (EPI == EPI_DSWIGLU) {
    float du;
    p.out0[i] = dswiglu_f(a, p.in0[i], p.in1[i], du);
    p.out1[i] = du;
  } else if constexpr (EPI == EPI_PAIR) {
    p.out0[i] = a;
    p.out1[i] = b;
  }
}

template <int EPI, bool PAIRED>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const SimtParams p) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  constexpr int NB = PAIRED ? 2 : 1;
  // A and B staging; reused for the partial tile of a split (unpaired only: TM x TN fits)
  constexpr int kFloats = TK * (TM + 4) + NB * TK * (TN + 4);
  static_assert(PAIRED || kFloats >= TM * TN, "partial tile must fit the staging buffers");
  __shared__ __align__(16) float sm[kFloats];
  auto As = reinterpret_cast<float(*)[TM + 4]>(sm);
  auto Bs = reinterpret_cast<float(*)[TK][TN + 4]>(sm + TK * (TM + 4));
  const int split = p.split;
  const int rank = split > 1 ? static_cast<int>(cluster_ctarank()) : 0;  // blockIdx.x % split
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * TM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x / split) * TN;
  const int g = blockIdx.z;
  float acc[4][4] = {}, acc2[4][4] = {};
  float ra[kPer], rb[NB][kPer];
  // element e of a step: consecutive threads walk the contiguous storage dimension
  auto a_idx = [&](int e, int& mm, int& kk) {
    mm = p.a_mn ? e % TM : e / TK;
    kk = p.a_mn ? e / TM : e % TK;
  };
  auto b_idx = [&](int e, int& nn, int& kk) {
    nn = p.b_mn ? e % TN : e / TK;
    kk = p.b_mn ? e / TN : e % TK;
  };
  auto load = [&](int s, int64_t k0) {  // one K step of segment s: global -> registers
    const float* A = p.A[s];
    const int64_t lda = p.lda[s];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      int mm, kk;
      a_idx(threadIdx.x + i * 256, mm, kk);
      const int64_t gm = m0 + mm, lk = k0 + kk, gk = p.k0[s] + g * p.K + lk;
      ra[i] = (gm < p.M && lk < p.K) ? (p.a_mn ? A[gk * lda + gm] : A[gm * lda + gk]) : 0.0f;
    }
#pragma unroll
    for (int h = 0; h < NB; ++h) {
      const float* B = p.B[PAIRED ? h : s];
      const int64_t ldb = p.ldb[PAIRED ? h : s];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        int nn, kk;
        b_idx(threadIdx.x + i * 256, nn, kk);
        const int64_t gn = n0 + nn, lk = k0 + kk, gk = p.k0[s] + g * p.K + lk;
        rb[h][i] = (gn < p.N && lk < p.K) ? (p.b_mn ? B[gk * ldb + gn] : B[gn * ldb + gk]) : 0.0f;
      }
    }
  };
  const int64_t steps = (p.K + TK - 1) / TK, total = steps * p.nseg;
  const int64_t per = (total + split - 1) / split;  // this CTA's K steps: [it0, it1)
  const int64_t it0 = rank * per, it1 = it0 + per < total ? it0 + per : total;
  if (it0 < it1) load(static_cast<int>(it0 / steps), (it0 % steps) * TK);
  for (int64_t it = it0; it < it1; ++it) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {  // registers -> shared (the previous step's reads ended
      int mm, kk;                     // at the __syncthreads below)
      a_idx(threadIdx.x + i * 256, mm, kk);
      As[kk][mm] = ra[i];
#pragma unroll
      for (int h = 0; h < NB; ++h) {
        int nn, kb;
        b_idx(threadIdx.x + i * 256, nn, kb);
        Bs[h][kb][nn] = rb[h][i];
      }
    }
    __syncthreads();
    if (it + 1 < it1) {  // the next step's loads fly while this step's FMAs run
      const int64_t nx = it + 1;
      load(static_cast<int>(nx / steps), (nx % steps) * TK);
    }
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[0][kk][tx * 4 + i];
        if constexpr (PAIRED) b2[i] = Bs[NB - 1][kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if constexpr (PAIRED) acc2[i][j] = fmaf(a[i], b2[j], acc2[i][j]);
        }
    }
    __syncthreads();
  }
  if (split == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t r = m0 + ty * 4 + i, c = n0 + tx * 4 + j;
        if (r < p.M && c < p.N) epi1<EPI>(p, g, r, c, acc[i][j], acc2[i][j]);
      }
    return;
  }
  if constexpr (!PAIRED) {  // split K (the host splits unpaired problems only)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sm[(ty * 4 + i) * TN + tx * 4 + j] = acc[i][j];
    cluster_sync_all();  // every CTA's partial tile is in its shared memory
    const int rows = TM / split;
    for (int e = threadIdx.x; e < rows * TN; e += 256) {
      const int rr = rank * rows + e / TN, cc = e % TN;
      const uint32_t off = smem_u32(sm + rr * TN + cc);
      float v = 0.0f;
      for (int q = 0; q < split; ++q) v += ld_cluster_f32(mapa_shared(off, static_cast<uint32_t>(q)));
      const int64_t r = m0 + rr, c = n0 + cc;
      if (r < p.M && c < p.N) epi1<EPI>(p, g, r, c, v, 0.0f);
    }
    cluster_sync_all();  // no CTA leaves while another still reads its tile
  }
}

// Whether the device can place a cluster of `split` CTAs of this kernel: asked once per
// device and cluster size (cudaOccupancyMaxActiveClusters), before the first launch.
template <int EPI, bool PAIRED>
bool cluster_fits(int split) {
  static std::atomic<int> known[64][4];  // 0 unknown, 1 fits, 2 does not
  const int slot = split == 2 ? 0 : split == 4 ? 1 : split == 8 ? 2 : 3;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
  if (dev >= 0 && known[dev][slot].load() != 0) return known[dev][slot].load() == 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const bool fits = cudaOccupancyMaxActiveClusters(&n, gemm_simt_kernel<EPI, PAIRED>, &cfg) ==
                        cudaSuccess && n > 0;
  if (!fits) cudaGetLastError();  // the query's own error, not a launch's
  if (dev >= 0) known[dev][slot].store(fits ? 1 : 2);
  return fits;
}

template <int EPI, bool PAIRED>
cudaError_t launch_k(const SimtParams& p, dim3 grid, cudaStream_t st) {
  if (p.split == 1 || !cluster_fits<EPI, PAIRED>(p.split)) {
    // unsplit: one CTA per tile (also when the device cannot place the cluster)
    SimtParams q = p;
    q.split = 1;
    return launch_kernel(gemm_simt_kernel<EPI, PAIRED>, grid, 256, 0, st, q);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(p.split);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid.x * static_cast<unsigned>(p.split), grid.y, grid.z);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_simt_kernel<EPI, PAIRED>, p);
}

}  // namespace

tp_status launch_gemm_simt(const GemmDesc& d, cudaStream_t st) {
  if (d.M <= 0 || d.N <= 0 || d.K <= 0) return TP_OK;
  SimtParams p{};
  if (d.nseg < 1 || d.nseg > 3) return fail(TP_ERR_INVALID_ARG, "1 to 3 K segments");
  for (int s = 0; s < 3; ++s) {
    const int sa = s < d.nseg ? s : 0;
    const int sb = s < (d.paired ? 2 : d.nseg) ? s : 0;
    p.k0[s] = d.seg_k0[s];
    p.A[s] = static_cast<const float*>(d.A[sa].ptr);
    p.lda[s] = d.A[sa].ld;
    p.B[s] = static_cast<const float*>(d.B[sb].ptr);
    p.ldb[s] = d.B[sb].ld;
  }
  p.M = d.M;
  p.N = d.N;
  p.K = d.K;
  p.a_mn = d.a_mn;
  p.b_mn = d.b_mn;
  p.nseg = d.nseg;
  p.paired = d.paired;
  p.out0 = static_cast<float*>(d.out[0]);
  p.out1 = static_cast<float*>(d.out[1]);
  p.out2 = static_cast<float*>(d.out[2]);
  p.in0 = static_cast<const float*>(d.in[0]);
  p.in1 = static_cast<const float*>(d.in[1]);
  p.ldo = d.ldo;
  p.out_group_stride = d.out_group_stride;
  const int64_t gx = (d.N + TN - 1) / TN, gy = (d.M + TM - 1) / TM;
  if (gx > 2147483647ll || gy > 65535 || d.groups > 65535)
    return fail(TP_ERR_SHAPE, "fp32 GEMM grid too large");
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(d.groups));
  const bool pr = d.paired;
  // split K over a cluster while the tiles (times the split) stay within half the SMs
  // and every CTA keeps at least one K step: at these sizes a K step is a global-load
  // latency, so fewer steps per CTA is a shorter launch
  const int64_t tiles = gx * gy * d.groups, ksteps = (d.K + TK - 1) / TK * d.nseg;
  p.split = 1;
  while (!pr && p.split < 8 && tiles * p.split * 4 <= device_sm_count() &&
         ksteps >= 2 * p.split)
    p.split *= 2;
  cudaError_t e = cudaSuccess;
  switch (d.epi) {
    case EPI_STORE: e = launch_k<EPI_STORE, false>(p, grid, st); break;
    case EPI_GELU: e = launch_k<EPI_GELU, false>(p, grid, st); break;
    case EPI_SWIGLU:
      if (!pr) return fail(TP_ERR_INVALID_ARG, "SwiGLU epilogue needs a paired problem");
      e = launch_k<EPI_SWIGLU, true>(p, grid, st);
      break;
    case EPI_DGELU: e = launch_k<EPI_DGELU, false>(p, grid, st); break;
    case EPI_DSWIGLU: e = launch_k<EPI_DSWIGLU, false>(p, grid, st); break;
    case EPI_PAIR:
      if (!pr) return fail(TP_ERR_INVALID_ARG, "pair epilogue needs a paired problem");
      e = launch_k<EPI_PAIR, true>(p, grid, st);
      break;
    default: return fail(TP_ERR_INVALID_ARG, "unknown epilogue");
  }
  count_launch();
  TP_CUDA_TRY(e);
  return TP_OK;
}

}  // namespace tp
