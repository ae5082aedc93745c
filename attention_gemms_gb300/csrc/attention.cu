// Per-head softmax attention of the head-sharded attention block, forward and
// backward. Heads are independent [张量并行 notes, §Multi-Head Attention 的并行化], so
// shard i's heads (a contiguous range of grid.y) never exchange data with other
// shards. A head map places the heads in the qkv rows (M = b*s rows):
//  * multi-head layout: W_qkv = [W_q | W_k | W_v], head t of Q, K, V at columns t*d,
//    h + t*d, 2h + t*d;
//  * grouped-query layout (per-shard blocks): shard i's columns are one block of S =
//    (hq + 2 hkv) d columns, [its hq query heads | its hkv key/value heads (K) | (V)];
//    local query head tl uses local key/value head tl / g. With fewer key/value heads
//    than shards, each block holds its own copy of its group's key/value head.
// o (M, H d), head t at t*d; lse (b, H, s) the log-sum-exp of each score row.
//   forward:  O = softmax(Q K^T / sqrt(d)) V        [Megatron-LM 实战 04, TPAttention]
//   backward: P = exp(S - lse), Dr = rowsum(dO * O), dV = P^T dO, dP = dO V^T,
//             dS = P * (dP - Dr), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d)
// At the page-2 layer's sizes (s = 128, d = 16) this is a few MFLOP per head, so
// these kernels use CUDA cores: four lanes per query row (forward, dQ) or key row
// (dK, dV), which split the head dimensions and the streamed rows between them; 64
// rows per CTA, the other operand streamed through shared memory in blocks of 64
// rows; softmax statistics in fp32. bf16 at head_dim 64 runs on the tensor cores
// (attention_tc.cu).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace tp {
namespace {

constexpr int RB = 64;  // rows per CTA and per shared-memory block
#ifndef TP_ATTN_TC
#define TP_ATTN_TC 1  // bf16, head_dim 64: the tensor-core kernels of attention_tc.cu
#endif

// Where query head t (0 <= t < H) and its key/value head sit in a qkv row.
struct HeadMap {
  int64_t ldq;     // row stride of qkv
  int64_t S;       // columns per shard block (0 for the multi-head layout)
  int64_t KO, VO;  // offsets of the K and V heads within a block
  int hq;          // query heads per block
  int g;           // query heads per key/value head within a block
  int hkv;         // key/value heads per block
  int H;           // query heads in total
  int64_t ldo;     // row stride of o and dO (H * d)
};

template <int D>
__device__ __forceinline__ int64_t qcol(const HeadMap& m, int t) {
  const int i = t / m.hq;
  return i * m.S + static_cast<int64_t>(t - i * m.hq) * D;
}
template <int D>
__device__ __forceinline__ int64_t kcol(const HeadMap& m, int t) {
  const int i = t / m.hq;
  return i * m.S + m.KO + static_cast<int64_t>((t - i * m.hq) / m.g) * D;
}
template <int D>
__device__ __forceinline__ int64_t vcol(const HeadMap& m, int t) {
  const int i = t / m.hq;
  return i * m.S + m.VO + static_cast<int64_t>((t - i * m.hq) / m.g) * D;
}

__device__ __forceinline__ float ld(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

// Each query (or key) row is handled by four adjacent lanes: P = D / 16 of them split
// the head dimensions (lane `part` owns dimensions part, part + P, part + 2P, ...,
// interleaved so the P lanes of a row read consecutive shared-memory words) and
// KS = 4 / P of them split the other operand's rows (lane `ks` takes rows ks, ks + KS,
// ...), each keeping its own partial state that the KS lanes merge at the end. Partial
// dot products are summed over the P lanes with xor-shuffles. Every lane runs every
// shuffle: all lanes of a warp run the same number of loop steps, and rows past the end
// and masked entries are handled by masking values, never by skipping the loop body.
constexpr int DP = 16;  // head dimensions per lane
constexpr int LPR = 4;  // lanes per row
// Shared-memory rows hold each lane's 16 dimensions contiguously, padded to 20 floats:
// a lane reads them with four 128-bit loads, and the P lanes of a row (offsets 0, 80,
// 160, 240 bytes) hit different banks.
constexpr int DPAD = DP + 4;

__device__ __forceinline__ void lds16(const float* src, float* v) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float4 t = reinterpret_cast<const float4*>(src)[u];
    v[4 * u] = t.x;
    v[4 * u + 1] = t.y;
    v[4 * u + 2] = t.z;
    v[4 * u + 3] = t.w;
  }
}

// sum over the lanes whose index differs in bits [lo, hi) (xor-shuffle tree)
template <int LO, int HI>
__device__ __forceinline__ float lane_sum(float v) {
#pragma unroll
  for (int o = LO; o < HI; o <<= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
template <int P>
__device__ __forceinline__ float row_sum(float v) {
  return lane_sum<1, P>(v);
}

template <int D>
struct Lanes {
  static constexpr int P = D / DP, KS = LPR / P;  // dimension lanes, row-split lanes
  int r, part, ks;
  __device__ explicit Lanes(int tid) : r(tid / LPR), part((tid % LPR) % P), ks((tid % LPR) / P) {}
};

template <typename T, int D>
__global__ void __launch_bounds__(RB * LPR) attn_fwd_kernel(
    const T* __restrict__ qkv, T* __restrict__ o, float* __restrict__ lse, int s,
    const HeadMap hm, float scale, int causal) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using Ln = Lanes<D>;
  constexpr int P = Ln::P, KS = Ln::KS;
  __shared__ __align__(16) float Ks[RB][P][DPAD];
  __shared__ __align__(16) float Vs[RB][P][DPAD];
  const int b = blockIdx.z, t = blockIdx.y;
  const Ln L(threadIdx.x);
  const int r = L.r, part = L.part, ks = L.ks;
  const int qi = blockIdx.x * RB + r;
  const int64_t ldq = hm.ldq, qc = qcol<D>(hm, t), kc = kcol<D>(hm, t), vc = vcol<D>(hm, t);
  const T* base = qkv + static_cast<int64_t>(b) * s * ldq;
  const bool valid = qi < s;
  float q[DP], acc[DP];
#pragma unroll
  for (int k = 0; k < DP; ++k) {
    q[k] = valid ? ld(base + qi * ldq, qc + part + P * k) * scale : 0.0f;
    acc[k] = 0.0f;
  }
  float m = -INFINITY, l = 0.0f;
  const int kend = causal ? min(s, static_cast<int>(blockIdx.x + 1) * RB) : s;
  for (int k0 = 0; k0 < kend; k0 += RB) {
    __syncthreads();
    const int kj = k0 + r;  // this row's key; the KS lanes of a part load slices of it
#pragma unroll
    for (int k = ks * (DP / KS); k < (ks + 1) * (DP / KS); ++k) {
      Ks[r][part][k] = kj < s ? ld(base + kj * ldq, kc + part + P * k) : 0.0f;
      Vs[r][part][k] = kj < s ? ld(base + kj * ldq, vc + part + P * k) : 0.0f;
    }
    __syncthreads();
    for (int j0 = 0; j0 < RB; j0 += 32) {
      float sc[32 / KS];
      float mb = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < 32 / KS; ++jj) {
        const int j = j0 + jj * KS + ks;
        float kv[DP];
        lds16(&Ks[j][part][0], kv);
        float v = 0.0f;
#pragma unroll
        for (int k = 0; k < DP; ++k) v = fmaf(q[k], kv[k], v);
        v = row_sum<P>(v);
        const int key = k0 + j;
        if (!valid || key >= s || (causal && key > qi)) v = -INFINITY;
        sc[jj] = v;
        mb = fmaxf(mb, v);
      }
      const float mn = fmaxf(m, mb);
      if (mn == -INFINITY) continue;  // every key of this lane so far masked (no shuffles below)
      const float corr = expf(m - mn);
      l *= corr;
#pragma unroll
      for (int k = 0; k < DP; ++k) acc[k] *= corr;
#pragma unroll
      for (int jj = 0; jj < 32 / KS; ++jj) {
        const float p = expf(sc[jj] - mn);
        l += p;
        float vv[DP];
        lds16(&Vs[j0 + jj * KS + ks][part][0], vv);
#pragma unroll
        for (int k = 0; k < DP; ++k) acc[k] = fmaf(p, vv[k], acc[k]);
      }
      m = mn;
    }
  }
  // merge the KS lanes' (max, sum, output) states (symmetric: every lane ends equal)
#pragma unroll
  for (int off = P; off < LPR; off <<= 1) {
    const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    const float lo = __shfl_xor_sync(0xFFFFFFFFu, l, off);
    const float mn = fmaxf(m, mo);
    const float a = m == -INFINITY ? 0.0f : expf(m - mn);
    const float c = mo == -INFINITY ? 0.0f : expf(mo - mn);
    l = l * a + lo * c;
#pragma unroll
    for (int k = 0; k < DP; ++k) {
      const float ao = __shfl_xor_sync(0xFFFFFFFFu, acc[k], off);
      acc[k] = acc[k] * a + ao * c;
    }
    m = mn;
  }
  if (!valid || ks != 0) return;
  const float inv = 1.0f / l;
  T* orow = o + (static_cast<int64_t>(b) * s + qi) * hm.ldo + t * D;
#pragma unroll
  for (int k = 0; k < DP; ++k) st(orow, part + P * k, acc[k] * inv);
  if (part == 0) lse[(static_cast<int64_t>(b) * hm.H + t) * s + qi] = m + logf(l);
}

// dK, dV: four lanes per key row of one key/value head (grid.y runs over the blocks'
// key/value heads, replicas included); the query rows of every query head of the block
// that uses it are streamed through shared memory, so the head's gradient sums their
// contributions; the KS lanes of a part take every KS-th query and sum at the end.
template <typename T, int D>
__global__ void __launch_bounds__(RB * LPR) attn_bwd_dkdv_kernel(
    const T* __restrict__ qkv, const T* __restrict__ o, const float* __restrict__ lse,
    const T* __restrict__ dO, T* __restrict__ dqkv, int s, const HeadMap hm, float scale,
    int causal) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using Ln = Lanes<D>;
  constexpr int P = Ln::P, KS = Ln::KS;
  __shared__ __align__(16) float Qs[RB][P][DPAD];
  __shared__ __align__(16) float dOs[RB][P][DPAD];
  __shared__ float Ls[RB], Ds[RB];
  const int b = blockIdx.z, u = blockIdx.y;
  const int blk = u / hm.hkv, kvl = u - blk * hm.hkv;
  const Ln L(threadIdx.x);
  const int r = L.r, part = L.part, ks = L.ks;
  const int kj = blockIdx.x * RB + r;
  const int64_t ldq = hm.ldq;
  const int64_t kc = blk * hm.S + hm.KO + static_cast<int64_t>(kvl) * D;
  const int64_t vc = blk * hm.S + hm.VO + static_cast<int64_t>(kvl) * D;
  const T* base = qkv + static_cast<int64_t>(b) * s * ldq;
  const T* obase = o + static_cast<int64_t>(b) * s * hm.ldo;
  const T* dobase = dO + static_cast<int64_t>(b) * s * hm.ldo;
  const bool valid = kj < s;
  float k[DP], v[DP], dk[DP], dv[DP];
#pragma unroll
  for (int c = 0; c < DP; ++c) {
    k[c] = valid ? ld(base + kj * ldq, kc + part + P * c) : 0.0f;
    v[c] = valid ? ld(base + kj * ldq, vc + part + P * c) : 0.0f;
    dk[c] = 0.0f;
    dv[c] = 0.0f;
  }
  const int qstart = causal ? static_cast<int>(blockIdx.x) * RB : 0;
  for (int tl = kvl * hm.g; tl < (kvl + 1) * hm.g; ++tl) {  // the block's query heads of this group
    const int t = blk * hm.hq + tl;
    const int64_t qc = blk * hm.S + static_cast<int64_t>(tl) * D;
    const float* lrow = lse + (static_cast<int64_t>(b) * hm.H + t) * s;
    for (int q0 = qstart; q0 < s; q0 += RB) {
      __syncthreads();
      const int qi = q0 + r;  // this row's query; the KS lanes of a part load slices of it
      float dsum = 0.0f;
#pragma unroll
      for (int c = ks * (DP / KS); c < (ks + 1) * (DP / KS); ++c) {
        const int dd = part + P * c;
        const float qv = qi < s ? ld(base + qi * ldq, qc + dd) : 0.0f;
        const float dov = qi < s ? ld(dobase + qi * hm.ldo, t * D + dd) : 0.0f;
        const float ov = qi < s ? ld(obase + qi * hm.ldo, t * D + dd) : 0.0f;
        Qs[r][part][c] = qv;
        dOs[r][part][c] = dov;
        dsum = fmaf(dov, ov, dsum);
      }
      dsum = lane_sum<1, LPR>(dsum);  // over every dimension slice of the row
      if (part == 0 && ks == 0) {
        Ls[r] = qi < s ? lrow[qi] : 0.0f;
        Ds[r] = dsum;
      }
      __syncthreads();
      const int iend = min(RB, s - q0);
      for (int i0 = 0; i0 < iend; i0 += KS) {  // the same step count on every lane
        const int i = i0 + ks;
        const bool in = i < iend;
        const int ii = in ? i : 0;
        float qv[DP], dov[DP];
        lds16(&Qs[ii][part][0], qv);
        lds16(&dOs[ii][part][0], dov);
        float sc = 0.0f, dp = 0.0f;
#pragma unroll
        for (int c = 0; c < DP; ++c) {
          sc = fmaf(qv[c], k[c], sc);
          dp = fmaf(dov[c], v[c], dp);
        }
        sc = row_sum<P>(sc);
        dp = row_sum<P>(dp);
        const bool live = in && valid && !(causal && kj > q0 + i);
        const float pr = live ? expf(sc * scale - Ls[ii]) : 0.0f;
        const float ds = pr * (dp - Ds[ii]) * scale;
#pragma unroll
        for (int c = 0; c < DP; ++c) {
          dv[c] = fmaf(pr, dov[c], dv[c]);
          dk[c] = fmaf(ds, qv[c], dk[c]);
        }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < DP; ++c) {  // the KS lanes' partial sums (a fixed xor tree)
    dk[c] = lane_sum<P, LPR>(dk[c]);
    dv[c] = lane_sum<P, LPR>(dv[c]);
  }
  if (!valid || ks != 0) return;
  T* row = dqkv + (static_cast<int64_t>(b) * s + kj) * ldq;
#pragma unroll
  for (int c = 0; c < DP; ++c) {
    st(row, kc + part + P * c, dk[c]);
    st(row, vc + part + P * c, dv[c]);
  }
}

// dQ: four lanes per query row; key rows streamed through shared memory, every KS-th
// key to each of a part's KS lanes
template <typename T, int D>
__global__ void __launch_bounds__(RB * LPR) attn_bwd_dq_kernel(
    const T* __restrict__ qkv, const T* __restrict__ o, const float* __restrict__ lse,
    const T* __restrict__ dO, T* __restrict__ dqkv, int s, const HeadMap hm, float scale,
    int causal) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  using Ln = Lanes<D>;
  constexpr int P = Ln::P, KS = Ln::KS;
  __shared__ __align__(16) float Ks[RB][P][DPAD];
  __shared__ __align__(16) float Vs[RB][P][DPAD];
  const int b = blockIdx.z, t = blockIdx.y;
  const Ln L(threadIdx.x);
  const int r = L.r, part = L.part, ks = L.ks;
  const int qi = blockIdx.x * RB + r;
  const int64_t ldq = hm.ldq, qc = qcol<D>(hm, t), kc = kcol<D>(hm, t), vc = vcol<D>(hm, t);
  const T* base = qkv + static_cast<int64_t>(b) * s * ldq;
  const bool valid = qi < s;
  float q[DP], dov[DP], dq[DP];
  float dsum = 0.0f, Lq = 0.0f;
  {
    const T* orow = o + (static_cast<int64_t>(b) * s + (valid ? qi : 0)) * hm.ldo + t * D;
    const T* dorow = dO + (static_cast<int64_t>(b) * s + (valid ? qi : 0)) * hm.ldo + t * D;
#pragma unroll
    for (int c = 0; c < DP; ++c) {
      const int dd = part + P * c;
      q[c] = valid ? ld(base + qi * ldq, qc + dd) : 0.0f;
      dov[c] = valid ? ld(dorow, dd) : 0.0f;
      dsum = fmaf(dov[c], valid ? ld(orow, dd) : 0.0f, dsum);
      dq[c] = 0.0f;
    }
    dsum = row_sum<P>(dsum);
    Lq = valid ? lse[(static_cast<int64_t>(b) * hm.H + t) * s + qi] : 0.0f;
  }
  const int kend = causal ? min(s, static_cast<int>(blockIdx.x + 1) * RB) : s;
  for (int k0 = 0; k0 < kend; k0 += RB) {
    __syncthreads();
    const int kj = k0 + r;
#pragma unroll
    for (int c = ks * (DP / KS); c < (ks + 1) * (DP / KS); ++c) {
      Ks[r][part][c] = kj < s ? ld(base + kj * ldq, kc + part + P * c) : 0.0f;
      Vs[r][part][c] = kj < s ? ld(base + kj * ldq, vc + part + P * c) : 0.0f;
    }
    __syncthreads();
    const int jend = min(RB, s - k0);
    for (int j0 = 0; j0 < jend; j0 += KS) {  // the same step count on every lane
      const int j = j0 + ks;
      const bool in = j < jend;
      const int jj = in ? j : 0;
      float kv[DP], vv[DP];
      lds16(&Ks[jj][part][0], kv);
      lds16(&Vs[jj][part][0], vv);
      float sc = 0.0f, dp = 0.0f;
#pragma unroll
      for (int c = 0; c < DP; ++c) {
        sc = fmaf(q[c], kv[c], sc);
        dp = fmaf(dov[c], vv[c], dp);
      }
      sc = row_sum<P>(sc);
      dp = row_sum<P>(dp);
      const bool live = in && valid && !(causal && k0 + j > qi);
      const float pr = live ? expf(sc * scale - Lq) : 0.0f;
      const float ds = pr * (dp - dsum) * scale;
#pragma unroll
      for (int c = 0; c < DP; ++c) dq[c] = fmaf(ds, kv[c], dq[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < DP; ++c) dq[c] = lane_sum<P, LPR>(dq[c]);  // the KS lanes' partials
  if (!valid || ks != 0) return;
  T* row = dqkv + (static_cast<int64_t>(b) * s + qi) * ldq;
#pragma unroll
  for (int c = 0; c < DP; ++c) st(row, qc + part + P * c, dq[c]);
}

template <typename T, int D>
tp_status run_fwd(const void* qkv, void* o, float* lse, int b, int s, const HeadMap& hm,
                  int causal, cudaStream_t st) {
  const dim3 grid((s + RB - 1) / RB, hm.H, b);
  TP_CUDA_TRY(launch_kernel(attn_fwd_kernel<T, D>, grid, RB * LPR, 0, st, static_cast<const T*>(qkv), static_cast<T*>(o), lse,
                                              s, hm, 1.0f / sqrtf(static_cast<float>(D)), causal));
  count_launch();
  TP_CUDA_TRY(cudaGetLastError());
  return TP_OK;
}

template <typename T, int D>
tp_status run_bwd(const void* qkv, const void* o, const float* lse, const void* dO, void* dqkv,
                  int b, int s, const HeadMap& hm, int kv_heads, int causal, cudaStream_t st) {
  const float scale = 1.0f / sqrtf(static_cast<float>(D));
  // dQ and dK/dV read the same inputs and write disjoint columns of dqkv: dQ runs on a
  // side stream beside dK/dV (the grids are small at these sizes)
  SideBranch br(st, 1);
  const cudaError_t e1 = launch_kernel(
      attn_bwd_dq_kernel<T, D>, dim3((s + RB - 1) / RB, hm.H, b), RB * LPR, 0, br.stream(),
      static_cast<const T*>(qkv), static_cast<const T*>(o), lse, static_cast<const T*>(dO),
      static_cast<T*>(dqkv), s, hm, scale, causal);
  const cudaError_t e2 = launch_kernel(
      attn_bwd_dkdv_kernel<T, D>, dim3((s + RB - 1) / RB, kv_heads, b), RB * LPR, 0, st,
      static_cast<const T*>(qkv), static_cast<const T*>(o), lse, static_cast<const T*>(dO),
      static_cast<T*>(dqkv), s, hm, scale, causal);
  count_launch(2);
  TP_TRY(br.join());
  if (e1 != cudaSuccess) return cuda_fail(e1, "attn_bwd_dq_kernel launch");
  TP_CUDA_TRY(e2);
  return TP_OK;
}

template <typename T>
tp_status fwd_d(const void* qkv, void* o, float* lse, int b, int s, const HeadMap& hm, int d,
                int causal, cudaStream_t st) {
  switch (d) {
    case 16: return run_fwd<T, 16>(qkv, o, lse, b, s, hm, causal, st);
    case 32: return run_fwd<T, 32>(qkv, o, lse, b, s, hm, causal, st);
    case 64: return run_fwd<T, 64>(qkv, o, lse, b, s, hm, causal, st);
  }
  return fail(TP_ERR_SHAPE, "head_dim must be 16, 32 or 64");
}

template <typename T>
tp_status bwd_d(const void* qkv, const void* o, const float* lse, const void* dO, void* dqkv,
                int b, int s, const HeadMap& hm, int kv_heads, int d, int causal,
                cudaStream_t st) {
  switch (d) {
    case 16: return run_bwd<T, 16>(qkv, o, lse, dO, dqkv, b, s, hm, kv_heads, causal, st);
    case 32: return run_bwd<T, 32>(qkv, o, lse, dO, dqkv, b, s, hm, kv_heads, causal, st);
    case 64: return run_bwd<T, 64>(qkv, o, lse, dO, dqkv, b, s, hm, kv_heads, causal, st);
  }
  return fail(TP_ERR_SHAPE, "head_dim must be 16, 32 or 64");
}

HeadMap mha_map(int64_t h, int heads) {
  HeadMap m{};
  m.ldq = 3 * h;
  m.S = 0;  // one block: head t at t*d, h + t*d, 2h + t*d
  m.KO = h;
  m.VO = 2 * h;
  m.hq = heads;
  m.g = 1;
  m.hkv = heads;
  m.H = heads;
  m.ldo = h;
  return m;
}

HeadMap gqa_map(int heads, int kv_heads, int N, int d) {
  const int hq = heads / N, hkv = kv_heads >= N ? kv_heads / N : 1;
  HeadMap m{};
  m.S = static_cast<int64_t>(hq + 2 * hkv) * d;
  m.ldq = N * m.S;
  m.KO = static_cast<int64_t>(hq) * d;
  m.VO = static_cast<int64_t>(hq + hkv) * d;
  m.hq = hq;
  m.g = hq / hkv;
  m.hkv = hkv;
  m.H = heads;
  m.ldo = static_cast<int64_t>(heads) * d;
  return m;
}

tp_status check_sizes(int64_t b, int64_t s, int heads) {
  if (b > 65535 || heads > 65535 || s > (1 << 24)) return fail(TP_ERR_SHAPE, "attention sizes out of range");
  return TP_OK;
}

}  // namespace

tp_status launch_attention_fwd(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                               int64_t h, int heads, int causal, tp_dtype dt, cudaStream_t st) {
  if (b <= 0 || s <= 0) return TP_OK;
  TP_TRY(check_sizes(b, s, heads));
  if (h > (1 << 20)) return fail(TP_ERR_SHAPE, "attention sizes out of range");
  const HeadMap m = mha_map(h, heads);
  const int d = static_cast<int>(h / heads), bi = static_cast<int>(b), si = static_cast<int>(s);
  if (TP_ATTN_TC && attention_tc_eligible(dt, d, m.ldq, qkv, o, m.ldo))
    return launch_attention_fwd_tc(qkv, o, lse, b, s, heads, m.hq, m.g, m.S, m.KO, m.VO, m.ldq,
                                   m.ldo, causal, st);
  return dt == TP_BF16 ? fwd_d<__nv_bfloat16>(qkv, o, lse, bi, si, m, d, causal, st)
                       : fwd_d<float>(qkv, o, lse, bi, si, m, d, causal, st);
}

tp_status launch_attention_bwd(const void* qkv, const void* o, const float* lse, const void* dO,
                               void* dqkv, void* ldws, int64_t b, int64_t s, int64_t h, int heads,
                               int causal, tp_dtype dt, cudaStream_t st) {
  if (b <= 0 || s <= 0) return TP_OK;
  TP_TRY(check_sizes(b, s, heads));
  if (h > (1 << 20)) return fail(TP_ERR_SHAPE, "attention sizes out of range");
  const HeadMap m = mha_map(h, heads);
  const int d = static_cast<int>(h / heads), bi = static_cast<int>(b), si = static_cast<int>(s);
  if (TP_ATTN_TC && ldws && attention_bwd_tc_eligible(dt, d, m.ldq, qkv, o, dO, dqkv, m.ldo))
    return launch_attention_bwd_tc(qkv, o, lse, dO, dqkv, ldws, b, s, heads, m.hq, m.g, m.hkv,
                                   heads, m.S, m.KO, m.VO, m.ldq, m.ldo, causal, st);
  return dt == TP_BF16
             ? bwd_d<__nv_bfloat16>(qkv, o, lse, dO, dqkv, bi, si, m, heads, d, causal, st)
             : bwd_d<float>(qkv, o, lse, dO, dqkv, bi, si, m, heads, d, causal, st);
}

tp_status launch_gqa_attention_fwd(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                                   int heads, int kv_heads, int N, int d, int causal, tp_dtype dt,
                                   cudaStream_t st) {
  if (b <= 0 || s <= 0) return TP_OK;
  TP_TRY(check_sizes(b, s, heads));
  const HeadMap m = gqa_map(heads, kv_heads, N, d);
  const int bi = static_cast<int>(b), si = static_cast<int>(s);
  if (TP_ATTN_TC && attention_tc_eligible(dt, d, m.ldq, qkv, o, m.ldo))
    return launch_attention_fwd_tc(qkv, o, lse, b, s, heads, m.hq, m.g, m.S, m.KO, m.VO, m.ldq,
                                   m.ldo, causal, st);
  return dt == TP_BF16 ? fwd_d<__nv_bfloat16>(qkv, o, lse, bi, si, m, d, causal, st)
                       : fwd_d<float>(qkv, o, lse, bi, si, m, d, causal, st);
}

tp_status launch_gqa_attention_bwd(const void* qkv, const void* o, const float* lse,
                                   const void* dO, void* dqkv, void* ldws, int64_t b, int64_t s,
                                   int heads, int kv_heads, int N, int d, int causal, tp_dtype dt,
                                   cudaStream_t st) {
  if (b <= 0 || s <= 0) return TP_OK;
  TP_TRY(check_sizes(b, s, heads));
  const HeadMap m = gqa_map(heads, kv_heads, N, d);
  const int bi = static_cast<int>(b), si = static_cast<int>(s), kvg = N * m.hkv;
  if (TP_ATTN_TC && ldws && attention_bwd_tc_eligible(dt, d, m.ldq, qkv, o, dO, dqkv, m.ldo))
    return launch_attention_bwd_tc(qkv, o, lse, dO, dqkv, ldws, b, s, heads, m.hq, m.g, m.hkv,
                                   kvg, m.S, m.KO, m.VO, m.ldq, m.ldo, causal, st);
  return dt == TP_BF16
             ? bwd_d<__nv_bfloat16>(qkv, o, lse, dO, dqkv, bi, si, m, kvg, d, causal, st)
             : bwd_d<float>(qkv, o, lse, dO, dqkv, bi, si, m, kvg, d, causal, st);
}

}  // namespace tp
