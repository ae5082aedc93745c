// Tensor-core GEMM engine for sm_103a: TMA -> shared-memory ring -> tcgen05.mma
// (bf16 in, fp32 accumulate in TMEM) -> fused epilogue from TMEM.
//
// One persistent CTA per SM, 6 warps with fixed roles:
//   warp 0      TMA producer (one lane): fills a STAGES-deep ring of A/B tiles
//   warp 1      MMA issuer (one lane) and TMEM owner: 128 x BN x 16 MMAs into one
//               of two TMEM accumulators (double buffer), commits to mbarriers
//   warps 2-5   epilogue: tcgen05.ld of the accumulator (each warp owns 32 TMEM
//               lanes = 32 rows), activation / gradient / residual math, stores
// The tile space is enumerated shard by shard (each virtual rank's slab in turn),
// and inside a slab in groups of 16 M-tiles so that concurrently running CTAs
// share operand tiles through L2.
//
// Large GEMMs run on the CTA-pair kernel further down (gemm_tc2_kernel): two CTAs of a
// cluster share 256 x 256 tiles through cta_group::2 MMAs, or 256 x 512 tiles with one
// 128 x 512 accumulator per CTA, and stage the epilogue's outputs in shared memory for
// TMA stores.
//
// Every mbarrier wait is bounded by a time limit; on expiry the CTA records
// TP_ERR_TIMEOUT in the device status word, waits for its own copies and MMAs
// in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>

#include "epi_math.cuh"
#include "internal.h"
#include "ptx.cuh"

// GELU and GELU' of the bf16 epilogues: the SFU forms (1), or erff / expf (0)
#ifndef TP_GELU_SFU
#define TP_GELU_SFU 1
#endif
#if TP_GELU_SFU
#define TP_GELU gelu_sfu
#define TP_GELU_PRIME gelu_prime_sfu
#else
#define TP_GELU gelu_f
#define TP_GELU_PRIME gelu_prime_f
#endif

namespace tp {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kThreads = 192;
#ifndef TP_GROUP_M
#define TP_GROUP_M 16
#endif
#ifndef TP_PAIR_STAGES
#define TP_PAIR_STAGES 6
#endif
#ifndef TP_MN_3D
#define TP_MN_3D 1
#endif
// tcgen05.fence::after_thread_sync after every full-stage wait of the MMA thread
// (copies and MMAs are both async-proxy operations ordered by the mbarrier itself,
// so the fence is only required once per tile, after the accumulator handoff)
#ifndef TP_KLOOP_FENCE
#define TP_KLOOP_FENCE 0
#endif
constexpr bool kMn3d = TP_MN_3D != 0;
constexpr int kGroupM = TP_GROUP_M;
constexpr uint64_t kDrainTimeoutNs = 1000000000ull;

// DEC: decode-sized problems (M <= 64 rows): only the first a_rows (<= 64) rows of
// each A tile are loaded; the MMA still computes 128 rows, the rest of which read
// whatever shared memory follows and are never stored (row m of D depends on row m
// of A only). The smaller stages let two CTAs share an SM.
// decode configuration: two CTAs per SM of 4 stages each keep more weight bytes in
// flight than one CTA of 8 (the copies one producer thread keeps outstanding are
// the limit at these sizes)
#ifndef TP_DEC_STAGES
#define TP_DEC_STAGES 4
#endif
#ifndef TP_DEC_CTAS_PER_SM
#define TP_DEC_CTAS_PER_SM 2
#endif
template <int BN, bool DEC = false>
struct TcCfg {
  static constexpr int STAGES = DEC ? TP_DEC_STAGES : (BN == 256 ? 4 : 6);
  static constexpr int A_BYTES = DEC ? 64 * BK * 2 : BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TMEM_COLS = 2 * BN;
  static constexpr int NBARS = 2 * STAGES + 6;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + NBARS * 8 + 16;
};

struct TcParams {  // CUtensorMap members carry their own 128-byte alignment
  CUtensorMap tmA[3];
  CUtensorMap tmB[3];
  CUtensorMap tmO[3];  // pair kernel, tma_out: maps of out0..out2 for TMA stores
  int64_t M, N, K;  // N counts logical output columns
  int a_mn, b_mn, nseg, paired, groups;
  int a3d, b3d;  // MN-major operand maps are 3-D (x: 64 columns, y: k, z: 64-column chunk)
  int a_rows;    // rows of A loaded per tile by the decode configuration
  int seg_k0[3];
  int tiles_m, tiles_n, kb_per_seg;
  int shards, shard_axis;
  void* out0;
  void* out1;
  void* out2;
  const void* in0;
  const void* in1;
  int64_t ldo;
  int out_f32;
  int st32;  // outputs 32-byte aligned with a pitch of 32-byte multiples: 256-bit stores
  int ld32;  // epilogue inputs likewise: 256-bit loads
  int64_t out_group_stride;
  int tma_out;  // pair kernel: the epilogue stages outputs in shared memory, TMA stores them
  int* status;
  uint64_t timeout_ns;
  int debug_hang;
};

// Optional wait-cycle counters (compile with -DTP_GEMM_STATS; off in normal builds):
// per CTA, [0] producer waiting for a free stage, [1] MMA waiting for data,
// [2] MMA waiting for a free accumulator, [3] epilogue waiting for an accumulator,
// [4] epilogue busy, [5] MMA thread lifetime, [6] tiles, [7] producer lifetime.
#ifdef TP_GEMM_STATS
__device__ unsigned long long g_gemm_stats[1024][16];
#define TP_STAT(i, v) atomicAdd(&g_gemm_stats[blockIdx.x][i], static_cast<unsigned long long>(v))
#define TP_CLK() clock64()
#else
#define TP_STAT(i, v) ((void)(v))
#define TP_CLK() 0ll
#endif

struct TileCoord {
  int g, mt, nt;
};

__device__ __forceinline__ TileCoord tile_coord(const TcParams& p, int t) {
  const int tm = p.tiles_m, tn = p.tiles_n;
  int g = 0;
  if (p.groups > 1) {
    g = t / (tm * tn);
    t -= g * tm * tn;
  }
  int slab_m = tm, slab_n = tn, s = 0;
  if (p.shards > 1) {
    if (p.shard_axis == 0) slab_m = tm / p.shards;
    else slab_n = tn / p.shards;
    s = t / (slab_m * slab_n);
    t -= s * slab_m * slab_n;
  }
  const int grp = t / (kGroupM * slab_n);
  const int first_m = grp * kGroupM;
  const int gm = min(slab_m - first_m, kGroupM);
  const int r = t - grp * kGroupM * slab_n;
  int mt = first_m + r % gm;
  int nt = r / gm;
  if (p.shards > 1) {
    if (p.shard_axis == 0) mt += s * slab_m;
    else nt += s * slab_n;
  }
  return {g, mt, nt};
}

__device__ __forceinline__ void record_timeout(int* status) {
  atomicCAS(status, 0, static_cast<int>(TP_ERR_TIMEOUT));
  atomicAdd(status + 1, 1);
}

// ---- bf16 pack / unpack of 8 values (16 bytes)
__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 r;
  uint32_t* w = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&b);
  }
  return r;
}
__device__ __forceinline__ void unpack8(uint4 r, float* v) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void st8(void* base, int64_t idx, const float* v) {
  *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + idx) = pack8(v);
}
__device__ __forceinline__ void ld8(const void* base, int64_t idx, float* v) {
  unpack8(__ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + idx)), v);
}

// Inputs an epilogue reads (residual / saved activations), 8 columns at a time
template <int EPI>
struct EpiInputs {
  static constexpr int n = EPI == EPI_DSWIGLU ? 2 : (EPI == EPI_DGELU || EPI == EPI_STORE ? 1 : 0);
};

// Epilogue of 8 consecutive output columns of one row. a: accumulator values,
// b: the paired half (gate/up second operand) when the problem is paired. pre0/pre1:
// the 16 bytes of in0/in1 at this position when `preloaded` (else loaded here).
template <int EPI>
__device__ __forceinline__ void epi8(const TcParams& p, int g, int64_t row, int64_t col,
                                     const float* a, const float* b, bool preloaded = false,
                                     uint4 pre0 = uint4{}, uint4 pre1 = uint4{}) {
  const int64_t idx = row * p.ldo + col;
  float v[8], w[8];
  auto in8 = [&](const void* base, const uint4& pre, float* dst) {
    if (preloaded) unpack8(pre, dst);
    else ld8(base, idx, dst);
  };
  if constexpr (EPI == EPI_STORE) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = a[i];
    if (p.in0) {
      in8(p.in0, pre0, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += w[i];
    }
    if (p.out_f32) {
      float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out0) +
                                            g * p.out_group_stride + idx);
      o[0] = make_float4(v[0], v[1], v[2], v[3]);
      o[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      st8(p.out0, idx, v);
    }
  } else if constexpr (EPI == EPI_GELU) {
    if (p.out0) st8(p.out0, idx, a);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = TP_GELU(a[i]);
    st8(p.out1, idx, v);
  } else if constexpr (EPI == EPI_SWIGLU) {
    if (p.out0) st8(p.out0, idx, a);
    if (p.out1) st8(p.out1, idx, b);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = silu_sfu(a[i]) * b[i];
    st8(p.out2, idx, v);
  } else if constexpr (EPI == EPI_DGELU) {
    in8(p.in0, pre0, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = a[i] * TP_GELU_PRIME(w[i]);
    st8(p.out0, idx, v);
  } else if constexpr (EPI == EPI_DSWIGLU) {
    float gg[8], uu[8], du[8];
    in8(p.in0, pre0, gg);
    in8(p.in1, pre1, uu);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = dswiglu_sfu(a[i], gg[i], uu[i], du[i]);
    st8(p.out0, idx, v);
    st8(p.out1, idx, du);
  } else if constexpr (EPI == EPI_PAIR) {
    st8(p.out0, idx, a);
    st8(p.out1, idx, b);
  }
}

// ---- 32 bytes (16 bf16) of an epilogue input in one non-coherent 256-bit load
__device__ __forceinline__ void ld_b256(const void* ptr, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                 "=r"(hi.z), "=r"(hi.w)
               : "l"(ptr));
}

// ---- 16 consecutive columns: one 256-bit store per output when the host found the
// outputs 32-byte aligned (st32), else two 128-bit stores
__device__ __forceinline__ void st_b256(void* ptr, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st16(void* base, int64_t idx, const float* v, bool wide) {
  __nv_bfloat16* ptr = reinterpret_cast<__nv_bfloat16*>(base) + idx;
  if (wide) {
    const uint4 lo = pack8(v), hi = pack8(v + 8);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    st_b256(ptr, w);
  } else {
    reinterpret_cast<uint4*>(ptr)[0] = pack8(v);
    reinterpret_cast<uint4*>(ptr)[1] = pack8(v + 8);
  }
}
__device__ __forceinline__ void st16_f32(float* ptr, const float* v, bool wide) {
  if (wide) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(v[i]);
    st_b256(ptr, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(v[8 + i]);
    st_b256(ptr + 8, w);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      reinterpret_cast<float4*>(ptr)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}
__device__ __forceinline__ void in16(const void* base, int64_t idx, float* v, bool pre, uint4 x0,
                                     uint4 x1) {
  if (pre) {
    unpack8(x0, v);
    unpack8(x1, v + 8);
  } else {
    ld8(base, idx, v);
    ld8(base, idx + 8, v + 8);
  }
}

// The epilogue of epi8 over 16 consecutive columns of one row (same arithmetic).
template <int EPI>
__device__ __forceinline__ void epi16(const TcParams& p, int g, int64_t row, int64_t col,
                                      const float* a, const float* b, bool pre, uint4 i0a,
                                      uint4 i0b, uint4 i1a, uint4 i1b) {
  const int64_t idx = row * p.ldo + col;
  const bool wide = p.st32 != 0;
  float v[16], w[16];
  if constexpr (EPI == EPI_STORE) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = a[i];
    if (p.in0) {
      in16(p.in0, idx, w, pre, i0a, i0b);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] += w[i];
    }
    if (p.out_f32)
      st16_f32(reinterpret_cast<float*>(p.out0) + g * p.out_group_stride + idx, v, wide);
    else
      st16(p.out0, idx, v, wide);
  } else if constexpr (EPI == EPI_GELU) {
    if (p.out0) st16(p.out0, idx, a, wide);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = TP_GELU(a[i]);
    st16(p.out1, idx, v, wide);
  } else if constexpr (EPI == EPI_SWIGLU) {
    if (p.out0) st16(p.out0, idx, a, wide);
    if (p.out1) st16(p.out1, idx, b, wide);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = silu_sfu(a[i]) * b[i];
    st16(p.out2, idx, v, wide);
  } else if constexpr (EPI == EPI_DGELU) {
    in16(p.in0, idx, w, pre, i0a, i0b);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = a[i] * TP_GELU_PRIME(w[i]);
    st16(p.out0, idx, v, wide);
  } else if constexpr (EPI == EPI_DSWIGLU) {
    float uu[16], du[16];
    in16(p.in0, idx, w, pre, i0a, i0b);
    in16(p.in1, idx, uu, pre, i1a, i1b);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = dswiglu_sfu(a[i], w[i], uu[i], du[i]);
    st16(p.out0, idx, v, wide);
    st16(p.out1, idx, du, wide);
  } else if constexpr (EPI == EPI_PAIR) {
    st16(p.out0, idx, a, wide);
    st16(p.out1, idx, b, wide);
  }
}

// ---- pair-kernel epilogue through shared memory: a warp's 32 rows x 32 columns of
// one output go to a 2 KB staging box (row r from lane r, 64 bytes, its 16-byte
// granules permuted by the 64-byte swizzle the output map names -- which also keeps
// the 32 lanes' writes free of bank conflicts) and leave by one TMA store, instead of
// 32 scattered 32-byte stores per instruction. Each warp owns two boxes and reuses
// one once the store issued from it two outputs ago has read it.
struct EpiStager {
  uint32_t base;  // this warp's two boxes (shared::cta address)
  uint32_t k;     // the box the next output goes to
  int lane;
  __device__ __forceinline__ uint32_t box(uint32_t i) const { return base + i * 2048u; }
  __device__ __forceinline__ uint32_t at(uint32_t i, int q) const {
    return box(i) + lane * 64 + 16 * (q ^ ((lane >> 1) & 3));
  }
  // wait until at most `free_boxes` earlier stores still read this warp's boxes
  template <int N>
  __device__ __forceinline__ void acquire() {
    if (lane == 0) bulk_wait_read<N>();
    __syncwarp();
  }
  __device__ __forceinline__ void store(uint32_t i, const CUtensorMap* m, int x, int y, int z) {
    if (lane == 0) {
      tma_store_3d(m, box(i), x, y, z);
      bulk_commit();
    }
  }
  __device__ __forceinline__ void publish() {  // the lanes' box writes, visible to TMA
    fence_proxy_async_smem();
    __syncwarp();
  }
};

__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}

// 32 bf16 values val(0..31) of this lane's row, stored as one box at (x, y)
template <class F>
__device__ __forceinline__ void stage_bf16(EpiStager& st, const CUtensorMap* m, int x, int y,
                                           F&& val) {
  st.acquire<1>();
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(st.at(st.k, q), bf2(val(8 * q), val(8 * q + 1)), bf2(val(8 * q + 2), val(8 * q + 3)),
                 bf2(val(8 * q + 4), val(8 * q + 5)), bf2(val(8 * q + 6), val(8 * q + 7)));
  st.publish();
  st.store(st.k, m, x, y, 0);
  st.k ^= 1u;
}

// 32 fp32 values as two boxes of 16 columns: (x, y, z) and (x + 16, y, z)
template <class F>
__device__ __forceinline__ void stage_f32(EpiStager& st, const CUtensorMap* m, int x, int y, int z,
                                          F&& val) {
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    st.acquire<1>();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = 16 * hf + 4 * q;
      st_shared_v4(st.at(st.k, q), __float_as_uint(val(j)), __float_as_uint(val(j + 1)),
                   __float_as_uint(val(j + 2)), __float_as_uint(val(j + 3)));
    }
    st.publish();
    st.store(st.k, m, x + 16 * hf, y, z);
    st.k ^= 1u;
  }
}

// element j (0..31) of 32 bf16 inputs preloaded as four 16-byte words
__device__ __forceinline__ float in_at(const uint4* pin, int j) {
  const uint4 v = pin[j >> 3];
  const int w = (j & 7) >> 1;
  const uint32_t u = w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w;
  return __uint_as_float((j & 1) ? (u & 0xFFFF0000u) : (u << 16));
}

// The epilogue of one 32-column chunk of the warp's 32 rows (same arithmetic as
// epi16), outputs staged and TMA-stored; rows >= M and columns >= N of a box are not
// written by the store.
template <int EPI>
__device__ __forceinline__ void epi_chunk_tma(const TcParams& p, EpiStager& st, int g, int x, int y,
                                              const uint32_t* ra, const uint32_t* rb,
                                              const uint4* pin0, const uint4* pin1, bool has0) {
  auto A = [&](int j) { return __uint_as_float(ra[j]); };
  auto B = [&](int j) { return __uint_as_float(rb[j]); };
  if constexpr (EPI == EPI_STORE) {
    auto v = [&](int j) { return has0 ? A(j) + in_at(pin0, j) : A(j); };
    if (p.out_f32) stage_f32(st, &p.tmO[0], x, y, g, v);
    else stage_bf16(st, &p.tmO[0], x, y, v);
  } else if constexpr (EPI == EPI_GELU) {
    if (p.out0) stage_bf16(st, &p.tmO[0], x, y, A);
    stage_bf16(st, &p.tmO[1], x, y, [&](int j) { return TP_GELU(A(j)); });
  } else if constexpr (EPI == EPI_SWIGLU) {
    if (p.out0) stage_bf16(st, &p.tmO[0], x, y, A);
    if (p.out1) stage_bf16(st, &p.tmO[1], x, y, B);
    stage_bf16(st, &p.tmO[2], x, y, [&](int j) { return silu_sfu(A(j)) * B(j); });
  } else if constexpr (EPI == EPI_DGELU) {
    stage_bf16(st, &p.tmO[0], x, y, [&](int j) { return A(j) * TP_GELU_PRIME(in_at(pin0, j)); });
  } else if constexpr (EPI == EPI_DSWIGLU) {
    // dG and dU share the gate's sigmoid: both boxes are filled in one pass
    st.acquire<0>();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float dg[8], du[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dg[i] = dswiglu_sfu(A(8 * q + i), in_at(pin0, 8 * q + i), in_at(pin1, 8 * q + i), du[i]);
      st_shared_v4(st.at(st.k, q), bf2(dg[0], dg[1]), bf2(dg[2], dg[3]), bf2(dg[4], dg[5]),
                   bf2(dg[6], dg[7]));
      st_shared_v4(st.at(st.k ^ 1u, q), bf2(du[0], du[1]), bf2(du[2], du[3]), bf2(du[4], du[5]),
                   bf2(du[6], du[7]));
    }
    st.publish();
    st.store(st.k, &p.tmO[0], x, y, 0);
    st.store(st.k ^ 1u, &p.tmO[1], x, y, 0);  // the older of the two groups is box k's
  } else if constexpr (EPI == EPI_PAIR) {
    stage_bf16(st, &p.tmO[0], x, y, A);
    stage_bf16(st, &p.tmO[1], x, y, B);
  }
}

template <int BN, int EPI, bool DEC>
__global__ void __launch_bounds__(kThreads, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<BN, DEC>;
  constexpr int S = C::STAGES;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
#ifdef TP_GEMM_STATS
  __shared__ volatile long long issue_clk[8], commit_clk[8];
#endif

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  const uint32_t never_bar = bar0 + 8u * (2 * S + 5);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(drain_bar, 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA[0]);
    tma_prefetch_desc(&p.tmB[0]);
    for (int s = 1; s < p.nseg; ++s) {
      tma_prefetch_desc(&p.tmA[s]);
      tma_prefetch_desc(&p.tmB[s]);
    }
    if (p.paired) tma_prefetch_desc(&p.tmB[1]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // the set-up above overlaps the previous kernel; operands and outputs are touched after
  pdl_wait();
  pdl_trigger();

  const int ntiles = p.tiles_m * p.tiles_n * p.groups;
  const int nkb = p.nseg * p.kb_per_seg;
  const int bn_logical = p.paired ? BN / 2 : BN;
  uint32_t issued = 0;      // producer: loads issued
  bool mma_issued = false;  // MMA thread: any MMA issued

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      const uint32_t stage_tx =
          DEC ? static_cast<uint32_t>(p.a_rows * BK * 2 + C::B_BYTES) : C::STAGE_BYTES;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      [[maybe_unused]] const long long t_start = TP_CLK();
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        const TileCoord tc = tile_coord(p, t);
        const int m0 = tc.mt * BM;
        const int n0 = tc.nt * bn_logical;
        for (int kb = 0; kb < nkb; ++kb) {
          [[maybe_unused]] const long long tw = TP_CLK();
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          TP_STAT(0, TP_CLK() - tw);
          const int seg = kb / p.kb_per_seg;
          const int k0 = p.seg_k0[seg] + static_cast<int>(tc.g * p.K) + (kb - seg * p.kb_per_seg) * BK;
          const uint32_t a_dst = sbase + stage * C::STAGE_BYTES;
          const uint32_t b_dst = a_dst + C::A_BYTES;
#ifdef TP_GEMM_STATS
          {
            const long long now = clock64();
            if (issued >= static_cast<uint32_t>(S)) TP_STAT(9, now - commit_clk[stage]);
            issue_clk[stage] = now;
          }
#endif
          mbar_arrive_expect_tx(full_bar(stage), stage_tx);
          if (p.a_mn && p.a3d) {
            tma_load_3d(a_dst, &p.tmA[seg], full_bar(stage), 0, k0, m0 / 64);
          } else if (p.a_mn) {
            tma_load_2d(a_dst, &p.tmA[seg], full_bar(stage), m0, k0);
            tma_load_2d(a_dst + 8192, &p.tmA[seg], full_bar(stage), m0 + 64, k0);
          } else {
            tma_load_2d(a_dst, &p.tmA[seg], full_bar(stage), k0, m0);
          }
          if (p.paired && !p.b_mn) {
            // K-major halves ((out, in) weights): BN/2 gate rows, then BN/2 up rows
            tma_load_2d(b_dst, &p.tmB[0], full_bar(stage), k0, n0);
            tma_load_2d(b_dst + (BN / 2) * 128, &p.tmB[1], full_bar(stage), k0, n0);
          } else if (p.paired) {
            constexpr int HALF = BN / 128;  // 64-wide boxes per half
            if (p.b3d) {
              tma_load_3d(b_dst, &p.tmB[0], full_bar(stage), 0, k0, n0 / 64);
              tma_load_3d(b_dst + HALF * 8192, &p.tmB[1], full_bar(stage), 0, k0, n0 / 64);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) {
                const int half = j / HALF;
                tma_load_2d(b_dst + j * 8192, &p.tmB[half], full_bar(stage), n0 + 64 * (j % HALF),
                            k0);
              }
            }
          } else if (p.b_mn && p.b3d) {
            tma_load_3d(b_dst, &p.tmB[seg], full_bar(stage), 0, k0, n0 / 64);
          } else if (p.b_mn) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b_dst + j * 8192, &p.tmB[seg], full_bar(stage), n0 + 64 * j, k0);
          } else {
            tma_load_2d(b_dst, &p.tmB[seg], full_bar(stage), k0, n0);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      TP_STAT(7, TP_CLK() - t_start);
      if (!ok) record_timeout(p.status);
    }
    __syncwarp();  // reconverge before the block-wide (aligned) barriers below
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, BN, p.a_mn, p.b_mn);
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u, b_kstep = p.b_mn ? 2048u : 32u;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      if (p.debug_hang) ok = mbar_wait(never_bar, 0, p.timeout_ns, abort_flag);
      [[maybe_unused]] const long long t_start = TP_CLK();
      for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
        [[maybe_unused]] long long tw = TP_CLK();
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        TP_STAT(2, TP_CLK() - tw);
        TP_STAT(6, 1);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          tw = TP_CLK();
          if (!mbar_wait(full_bar(stage), phase, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          TP_STAT(1, TP_CLK() - tw);
#ifdef TP_GEMM_STATS
          TP_STAT(8, clock64() - issue_clk[stage]);
          TP_STAT(10, 1);
#endif
          if (TP_KLOOP_FENCE) tc_fence_after();
          const uint32_t a_addr = sbase + stage * C::STAGE_BYTES;
          const uint32_t b_addr = a_addr + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = sw128_desc(a_addr + kk * a_kstep, a_lbo, 1024u);
            const uint64_t bd = sw128_desc(b_addr + kk * b_kstep, b_lbo, 1024u);
            mma_bf16_ss(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_issued = true;
          mma_commit(empty_bar(stage));
#ifdef TP_GEMM_STATS
          commit_clk[stage] = clock64();
#endif
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      TP_STAT(5, TP_CLK() - t_start);
      if (!ok) record_timeout(p.status);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lanes [32*quad, 32*quad + 32)
    uint32_t acc = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const TileCoord tc = tile_coord(p, t);
      int ok = 1;
      [[maybe_unused]] const long long tw = TP_CLK();
      if (lane == 0) ok = mbar_wait(tfull_bar(acc), acc_phase, p.timeout_ns, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      [[maybe_unused]] const long long tb = TP_CLK();
      if (warp == 2 && lane == 0) TP_STAT(3, tb - tw);
      if (!ok) {
        if (lane == 0) record_timeout(p.status);
        break;
      }
      tc_fence_after();
      const int64_t row = static_cast<int64_t>(tc.mt) * BM + quad * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      const int64_t col_base = static_cast<int64_t>(tc.nt) * bn_logical;
      for (int c = 0; c < bn_logical / 32; ++c) {
        uint32_t ra[32], rb[32];
        tmem_ld32(t_row + c * 32, ra);
        if (p.paired) tmem_ld32(t_row + BN / 2 + c * 32, rb);
        tmem_ld_wait();
        if (row < p.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t col = col_base + c * 32 + q * 8;
            if (col < p.N) {
              float a[8], b[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                a[i] = __uint_as_float(ra[q * 8 + i]);
                b[i] = __uint_as_float(rb[q * 8 + i]);
              }
              epi8<EPI>(p, tc.g, row, col, a, b);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (warp == 2 && lane == 0) TP_STAT(4, TP_CLK() - tb);
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (*abort_flag) {
    volatile int no_abort = 0;
    if (warp == 0) {
      if (lane == 0) {
        // wait for every copy this CTA issued: the last load into stage s
        for (int s = 0; s < S; ++s) {
          if (issued > static_cast<uint32_t>(s)) {
            const uint32_t last = ((issued - 1u - s) / S) * S + s;
            mbar_wait(full_bar(s), (last / S) & 1u, kDrainTimeoutNs, &no_abort);
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0 && mma_issued) {
        mma_commit(drain_bar);
        mbar_wait(drain_bar, 0, kDrainTimeoutNs, &no_abort);
      }
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// Same roles as gemm_tc_kernel, but two CTAs of a cluster share one 256 x 256 tile
// through tcgen05.mma.cta_group::2: CTA r of the pair stages A rows [128 r, 128 r + 128)
// and B columns [128 r, 128 r + 128) of the tile (32 KB per 64-deep K block instead
// of 48 KB for 128 x 256 on one CTA), and holds D rows [128 r, 128 r + 128) in its
// TMEM. The even CTA issues the MMAs; its commits arrive on the barriers of both
// CTAs (multicast). Both CTAs' copies of a stage complete on the even CTA's "full"
// barrier (pair form of the TMA load), whose producer expects both halves' bytes;
// the odd CTA's epilogue warps report "accumulator drained" to the even CTA with
// remote arrives. At exit both CTAs wait for the pair's last MMAs, then for each
// other, before freeing TMEM.

#ifndef TP_PAIR_DUAL
#define TP_PAIR_DUAL 1
#endif
// TP_PAIR_DUAL: a second producer warp (warp 6) issues the B copies while warp 0 issues A
#ifndef TP_PAIR_EPI_WARPS
#define TP_PAIR_EPI_WARPS 4
#endif
// TP_PAIR_EPI_WARPS = 8: a second set of four epilogue warps (after the producer warps)
// drains the other half of each accumulator tile's columns, halving the epilogue time
static_assert(TP_PAIR_EPI_WARPS == 4 || TP_PAIR_EPI_WARPS == 8, "4 or 8 epilogue warps");
constexpr int kEpiHi0 = TP_PAIR_DUAL ? 7 : 6;  // first warp of the second epilogue set
constexpr uint64_t kPairDrainNs = 20000000ull;

// Wide form (WN = 2): the pair computes a 256 x 512 tile -- two N = 256 MMAs per K
// step into one 128 x 512 fp32 accumulator per CTA, all 512 TMEM columns. A stage
// holds A 128 x 64 and two B halves of 128 x 64 per CTA (48 KB), four stages deep.
// Per FLOP it moves 3/4 of the operand bytes of the 256 x 256 tile from L2 into
// shared memory, which is what bounds the narrow form's issue rate. With a single
// accumulator the epilogue drains the first 256 columns, hands them back
// (tempty 0) and then drains the second half (tempty 1); meanwhile the next tile's
// first stages already run their first-half MMAs.
#ifndef TP_WIDE_STAGES
#define TP_WIDE_STAGES 4
#endif
template <int WN>
struct PairCfg {
  static constexpr int EPI_WARPS = WN == 2 ? 8 : TP_PAIR_EPI_WARPS;
  static constexpr int THREADS = 32 * (kEpiHi0 + (EPI_WARPS == 8 ? 4 : 0));
  static constexpr int STAGES = WN == 2 ? TP_WIDE_STAGES : TP_PAIR_STAGES;
  static constexpr int B_HALF_BYTES = 128 * BK * 2;                // 128 x 64 bf16
  static constexpr int STAGE_BYTES = (1 + WN) * B_HALF_BYTES;      // A + WN B halves
  static constexpr int NACC = WN == 2 ? 1 : 2;                     // TMEM accumulators
  static constexpr int NBARS = 2 * STAGES + 7;
  // epilogue staging: two 2 KB boxes (32 rows x 64 bytes) per epilogue warp
  static constexpr int STAGING_BYTES = EPI_WARPS * 2 * 2048;
  static constexpr int SMEM = STAGES * STAGE_BYTES + STAGING_BYTES + 1024 + NBARS * 8 + 16;
};
static_assert(PairCfg<2>::SMEM <= 232448 && PairCfg<1>::SMEM <= 232448, "shared memory per CTA");

template <int EPI, int WN>
__global__ void __launch_bounds__(PairCfg<WN>::THREADS, 1)
    gemm_tc2_kernel(const __grid_constant__ TcParams p) {
  using C = PairCfg<WN>;
  constexpr int S = C::STAGES;
  constexpr int A_BYTES = 128 * BK * 2;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* staging = smem + S * C::STAGE_BYTES;  // 1024-byte aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::STAGING_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
#ifdef TP_GEMM_STATS
  __shared__ volatile long long issue_clk[S], commit_clk[S];
#endif

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  const uint32_t exit_bar = bar0 + 8u * (2 * S + 5);
  const uint32_t never_bar = bar0 + 8u * (2 * S + 6);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);  // even CTA: its producer's expect-tx; odd CTA: unused
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), leader ? 2 * C::EPI_WARPS : 1);  // epilogue warps of both CTAs
    }
    mbar_init(drain_bar, 1);
    mbar_init(exit_bar, 1);
    mbar_init(never_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmA[0]);
    tma_prefetch_desc(&p.tmB[0]);
    for (int s = 1; s < p.nseg; ++s) {
      tma_prefetch_desc(&p.tmA[s]);
      tma_prefetch_desc(&p.tmB[s]);
    }
    if (p.paired) tma_prefetch_desc(&p.tmB[1]);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // the set-up above overlaps the previous kernel; operands and outputs are touched after
  pdl_wait();
  pdl_trigger();

  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int ntiles = p.tiles_m * p.tiles_n * p.groups;
  const int nkb = p.nseg * p.kb_per_seg;
  const int bn_logical = p.paired ? 128 : 256;
  uint32_t issued = 0;

  if (warp == 0 || (TP_PAIR_DUAL && warp == 6)) {
    const bool load_a = warp == 0;
    const bool load_b = !TP_PAIR_DUAL || warp == 6;
    if (lane == 0) {
      // ------------------------------------------------------------ producer (both CTAs)
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      [[maybe_unused]] const long long t_start = TP_CLK();
      const uint32_t lead_full0 = mapa_shared(full_bar(0), 0);
      for (int t = pair; t < ntiles && ok; t += npairs) {
        const TileCoord tc = tile_coord(p, t);
        const int m0 = tc.mt * 256 + static_cast<int>(rank) * 128;
        const int n0 = tc.nt * bn_logical * WN;
        for (int kb = 0; kb < nkb; ++kb) {
          [[maybe_unused]] const long long tw = TP_CLK();
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          TP_STAT(0, TP_CLK() - tw);
          const int seg = kb / p.kb_per_seg;
          const int k0 =
              p.seg_k0[seg] + static_cast<int>(tc.g * p.K) + (kb - seg * p.kb_per_seg) * BK;
          const uint32_t a_dst = sbase + stage * C::STAGE_BYTES;
          const uint32_t b_dst = a_dst + A_BYTES;
          const uint32_t fb = lead_full0 + 8u * stage;  // the even CTA's barrier
#ifdef TP_GEMM_STATS
          if (leader) {
            const long long now = clock64();
            if (issued >= static_cast<uint32_t>(S)) TP_STAT(9, now - commit_clk[stage]);
            issue_clk[stage] = now;
          }
#endif
          if (leader && load_a) mbar_arrive_expect_tx(full_bar(stage), 2 * C::STAGE_BYTES);
          if (!load_a) {
          } else if (p.a_mn && p.a3d) {
            tma_load_3d_pair(a_dst, &p.tmA[seg], fb, 0, k0, m0 / 64);
          } else if (p.a_mn) {
            tma_load_2d_pair(a_dst, &p.tmA[seg], fb, m0, k0);
            tma_load_2d_pair(a_dst + 8192, &p.tmA[seg], fb, m0 + 64, k0);
          } else {
            tma_load_2d_pair(a_dst, &p.tmA[seg], fb, k0, m0);
          }
          // B: WN halves of the tile's MMA width, each split between the two CTAs
#pragma unroll
          for (int h = 0; h < WN; ++h) {
            const uint32_t bh = b_dst + h * C::B_HALF_BYTES;
            if (!load_b) {
            } else if (p.paired && !p.b_mn) {
              // K-major ((out, in) weights): even CTA 128 gate rows, odd CTA the same up rows
              tma_load_2d_pair(bh, &p.tmB[rank], fb, k0, n0 + h * 128);
            } else if (p.paired) {
              // even CTA: 128 gate columns, odd CTA: the same 128 up columns
              const int nb = n0 + h * 128;
              if (p.b3d) {
                tma_load_3d_pair(bh, &p.tmB[rank], fb, 0, k0, nb / 64);
              } else {
                tma_load_2d_pair(bh, &p.tmB[rank], fb, nb, k0);
                tma_load_2d_pair(bh + 8192, &p.tmB[rank], fb, nb + 64, k0);
              }
            } else if (p.b_mn) {
              const int nb = n0 + h * 256 + static_cast<int>(rank) * 128;
              if (p.b3d) {
                tma_load_3d_pair(bh, &p.tmB[seg], fb, 0, k0, nb / 64);
              } else {
                tma_load_2d_pair(bh, &p.tmB[seg], fb, nb, k0);
                tma_load_2d_pair(bh + 8192, &p.tmB[seg], fb, nb + 64, k0);
              }
            } else {
              tma_load_2d_pair(bh, &p.tmB[seg], fb, k0,
                               n0 + h * 256 + static_cast<int>(rank) * 128);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      TP_STAT(7, TP_CLK() - t_start);
      if (!ok) record_timeout(p.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------------ pair MMA issuer
      const uint32_t idesc = idesc_bf16_f32(256, 256, p.a_mn, p.b_mn);
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, b_lbo = p.b_mn ? 8192u : 16u;
      const uint32_t a_kstep = p.a_mn ? 2048u : 32u, b_kstep = p.b_mn ? 2048u : 32u;
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      if (p.debug_hang) ok = mbar_wait(never_bar, 0, p.timeout_ns, abort_flag);
      [[maybe_unused]] const long long t_start = TP_CLK();
      // the MMAs of one stage for the tile halves [h0, h1), K block kb of the tile
      auto issue = [&](uint32_t d_tmem, int h0, int h1, int kb) {
        const uint32_t a_addr = sbase + stage * C::STAGE_BYTES;
        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = sw128_desc(a_addr + kk * a_kstep, a_lbo, 1024u);
#pragma unroll
          for (int h = 0; h < WN; ++h) {
            if (h < h0 || h >= h1) continue;
            const uint64_t bd =
                sw128_desc(b_addr + h * C::B_HALF_BYTES + kk * b_kstep, b_lbo, 1024u);
            mma_bf16_ss_pair(d_tmem + h * 256, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
        }
      };
      auto wait_full = [&]() {
        [[maybe_unused]] const long long tw = TP_CLK();
        if (!mbar_wait(full_bar(stage), phase, p.timeout_ns, abort_flag)) return false;
        TP_STAT(1, TP_CLK() - tw);
#ifdef TP_GEMM_STATS
        TP_STAT(8, clock64() - issue_clk[stage]);
        TP_STAT(10, 1);
#endif
        if (TP_KLOOP_FENCE) tc_fence_after();
        return true;
      };
      auto release = [&]() {
        mma_commit_pair(empty_bar(stage), 0x3);
#ifdef TP_GEMM_STATS
        commit_clk[stage] = clock64();
#endif
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      };
      for (int t = pair; t < ntiles && ok; t += npairs) {
        [[maybe_unused]] long long tw = TP_CLK();
        // narrow: accumulator `acc` drained; wide: the first half of the accumulator
        if (!mbar_wait(tempty_bar(WN == 2 ? 0 : acc), acc_phase ^ 1u, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        TP_STAT(2, TP_CLK() - tw);
        TP_STAT(6, 1);
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        int kb = 0;
        if constexpr (WN == 2) {
          // the first stages' first-half MMAs run while the epilogue drains the second
          // half of the previous tile; then the same stages' second-half MMAs
          const int pre = min(S, nkb);
          const uint32_t stage0 = stage, phase0 = phase;
          for (int j = 0; j < pre && ok; ++j) {
            ok = wait_full();
            if (!ok) break;
            issue(d_tmem, 0, 1, j);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (pre == nkb) mma_commit_pair(tfull_bar(0), 0x3);  // the first half is complete
          if (!mbar_wait(tempty_bar(1), acc_phase ^ 1u, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          stage = stage0;
          phase = phase0;
          for (int j = 0; j < pre; ++j) {
            issue(d_tmem, 1, 2, j);
            release();
          }
          kb = pre;
        }
        // wide: the last `post` stages run their first-half MMAs first, so that the first
        // half of the accumulator is complete (tfull 0) and drains while their second-half
        // MMAs run (tfull 1)
        const int post = WN == 2 ? min(S, nkb - kb) : 0;
        for (; kb < nkb - post; ++kb) {
          if (!wait_full()) {
            ok = false;
            break;
          }
          issue(d_tmem, 0, WN, kb);
          release();
        }
        if (!ok) break;
        if constexpr (WN == 2) {
          if (post > 0) {
            const uint32_t stage0 = stage, phase0 = phase;
            for (int j = 0; j < post && ok; ++j) {
              ok = wait_full();
              if (!ok) break;
              issue(d_tmem, 0, 1, kb + j);
              if (++stage == S) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            mma_commit_pair(tfull_bar(0), 0x3);
            stage = stage0;
            phase = phase0;
            for (int j = 0; j < post; ++j) {
              issue(d_tmem, 1, 2, kb + j);
              release();
            }
            kb += post;
          }
          mma_commit_pair(tfull_bar(1), 0x3);
        } else {
          mma_commit_pair(tfull_bar(acc), 0x3);
        }
        if (C::NACC == 2) {
          acc ^= 1u;
          if (acc == 0) acc_phase ^= 1u;
        } else {
          acc_phase ^= 1u;
        }
      }
      TP_STAT(5, TP_CLK() - t_start);
      if (!ok) record_timeout(p.status);
    }
    __syncwarp();
  } else if ((warp >= 2 && warp < 6) || warp >= kEpiHi0) {
    // -------------------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;  // a warp reaches the TMEM lanes of quarter warp % 4
    const int nchunk = bn_logical / 32;
    // with eight epilogue warps each set drains half of every accumulator half's chunks
    constexpr int kEW = C::EPI_WARPS;
    const int c_lo = kEW == 8 && warp >= kEpiHi0 ? nchunk / 2 : 0;
    const int c_hi = kEW == 8 && warp < 6 ? nchunk / 2 : nchunk;
    const uint32_t remote_tempty0 = mapa_shared(tempty_bar(0), 0);
    const int epi_slot = warp < 6 ? warp - 2 : warp - kEpiHi0 + 4;
    EpiStager stg{smem_u32(staging) + static_cast<uint32_t>(epi_slot) * 4096u, 0u, lane};
    uint32_t acc = 0, acc_phase = 0;
    for (int t = pair; t < ntiles; t += npairs) {
      const TileCoord tc = tile_coord(p, t);
      int ok = 1;
      [[maybe_unused]] const long long tw = TP_CLK();
      // narrow: the whole accumulator; wide: each half is waited for below
      if (lane == 0 && WN == 1)
        ok = mbar_wait(tfull_bar(acc), acc_phase, p.timeout_ns, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      [[maybe_unused]] const long long tb = TP_CLK();
      if (warp == 2 && lane == 0) TP_STAT(3, tb - tw);
      if (!ok) {
        if (lane == 0) record_timeout(p.status);
        break;
      }
      tc_fence_after();
      const int64_t row =
          static_cast<int64_t>(tc.mt) * 256 + static_cast<int>(rank) * 128 + quad * 32 + lane;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * 256;
      for (int h = 0; h < WN && ok; ++h) {
        if (WN == 2) {
          if (lane == 0) ok = mbar_wait(tfull_bar(h), acc_phase, p.timeout_ns, abort_flag) ? 1 : 0;
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) {
            if (lane == 0) record_timeout(p.status);
            break;
          }
          tc_fence_after();
        }
        const int64_t col_base = (static_cast<int64_t>(tc.nt) * WN + h) * bn_logical;
        const uint32_t t_half = t_row + h * 256;
        for (int c = c_lo; c < c_hi; ++c) {
          uint32_t ra[32], rb[32];
          tmem_ld32(t_half + c * 32, ra);
          if (p.paired) tmem_ld32(t_half + 128 + c * 32, rb);
          // the chunk's epilogue inputs are requested together, while the TMEM load runs
          constexpr int kIn = EpiInputs<EPI>::n;
          uint4 pin0[4] = {}, pin1[4] = {};
          const bool has0 = kIn >= 1 && p.in0 != nullptr;
          if (kIn > 0 && row < p.M) {
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              const int64_t col = col_base + c * 32 + qq * 16;
              const int64_t idx = row * p.ldo + col;
              const __nv_bfloat16* i0 = reinterpret_cast<const __nv_bfloat16*>(p.in0) + idx;
              const __nv_bfloat16* i1 = reinterpret_cast<const __nv_bfloat16*>(p.in1) + idx;
              if (p.ld32 && col + 16 <= p.N) {  // a whole 32-byte sector per load
                if (has0) ld_b256(i0, pin0[2 * qq], pin0[2 * qq + 1]);
                if (kIn == 2) ld_b256(i1, pin1[2 * qq], pin1[2 * qq + 1]);
              } else {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                  if (col + 8 * hh < p.N) {
                    if (has0) pin0[2 * qq + hh] = __ldg(reinterpret_cast<const uint4*>(i0 + 8 * hh));
                    if (kIn == 2) pin1[2 * qq + hh] = __ldg(reinterpret_cast<const uint4*>(i1 + 8 * hh));
                  }
                }
              }
            }
          }
          tmem_ld_wait();
          if (p.tma_out) {
            const int64_t x = col_base + c * 32, y = row - lane;  // the warp's first row
            if (y < p.M && x < p.N)
              epi_chunk_tma<EPI>(p, stg, tc.g, static_cast<int>(x), static_cast<int>(y), ra, rb,
                                 pin0, pin1, kIn > 0 && has0);
          } else if (row < p.M) {
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {  // 16 columns at a time
              const int64_t col = col_base + c * 32 + qq * 16;
              float a[16], b[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                a[i] = __uint_as_float(ra[qq * 16 + i]);
                b[i] = __uint_as_float(rb[qq * 16 + i]);
              }
              if (col + 16 <= p.N)
                epi16<EPI>(p, tc.g, row, col, a, b, kIn > 0 && has0, pin0[2 * qq], pin0[2 * qq + 1],
                           pin1[2 * qq], pin1[2 * qq + 1]);
              else if (col < p.N)  // N % 8 == 0: the last 8 columns
                epi8<EPI>(p, tc.g, row, col, a, b, kIn > 0 && has0, pin0[2 * qq], pin1[2 * qq]);
            }
          }
        }
        // wide tile: this half of the accumulator is free for the next tile's MMAs
        if (WN == 2) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(tempty_bar(h));
            else mbar_arrive_remote(remote_tempty0 + 8u * h);
          }
        }
      }
      if (!ok) break;
      if (warp == 2 && lane == 0) TP_STAT(4, TP_CLK() - tb);
      if (C::NACC == 2) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(tempty_bar(acc));
          else mbar_arrive_remote(remote_tempty0 + 8u * acc);
        }
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      } else {
        acc_phase ^= 1u;
      }
    }
    // the staged stores have read shared memory and written their outputs before exit
    if (p.tma_out) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  volatile int no_abort = 0;
  // after an abort, the even CTA waits (bounded) for the copies of both CTAs, whose
  // completions land on its barriers; the odd CTA stays until the exit handshake
  if (*abort_flag && warp == 0 && leader) {
    if (lane == 0) {
      for (int s = 0; s < S; ++s) {
        if (issued > static_cast<uint32_t>(s)) {
          const uint32_t last = ((issued - 1u - s) / S) * S + s;
          mbar_wait(full_bar(s), (last / S) & 1u, kPairDrainNs, &no_abort);
        }
      }
    }
    __syncwarp();
  }
  if (warp == 1) {
    // every MMA of the pair has completed once the even CTA's final commit arrives
    if (lane == 0) {
      if (leader) mma_commit_pair(drain_bar, 0x3);
      mbar_wait(drain_bar, 0, kPairDrainNs, &no_abort);
    }
    __syncwarp();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // neither CTA leaves while the other may still signal its barriers or read its smem
    mbar_arrive_remote(mapa_shared(exit_bar, rank ^ 1u));
    mbar_wait(exit_bar, 0, kPairDrainNs, &no_abort);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 2-D bf16 map over a row-major tensor, 128-byte swizzle, zero fill out of bounds.
tp_status make_map(CUtensorMap* m, const Operand& op, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  if (reinterpret_cast<uintptr_t>(op.ptr) % 16 != 0 || (op.ld * 2) % 16 != 0)
    return fail(TP_ERR_ALIGNMENT, "TMA operand base/pitch not 16-byte aligned");
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(op.cols), static_cast<cuuint64_t>(op.rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(op.ld) * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(op.ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")");
  return TP_OK;
}

// 3-D view of an MN-major operand for loading `chunks` 64-column chunks at once:
// dims (64, rows, cols / 64), strides (ld * 2, 128) bytes, box (64, 64, chunks).
tp_status make_map_3d(CUtensorMap* m, const Operand& op, uint32_t chunks) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  if (reinterpret_cast<uintptr_t>(op.ptr) % 16 != 0 || (op.ld * 2) % 16 != 0 || op.cols % 64 != 0)
    return fail(TP_ERR_ALIGNMENT, "3-D TMA operand not 16-byte aligned or ragged");
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(op.rows),
                              static_cast<cuuint64_t>(op.cols / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(op.ld) * 2, 128};
  const cuuint32_t box[3] = {64, 64, chunks};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(op.ptr), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (code " + std::to_string(r) + ")");
  return TP_OK;
}

// Store map of an output for the pair kernel's staged epilogue: 3-D (columns, rows,
// groups), box 32 rows x 64 bytes (32 bf16 or 16 fp32 columns) x 1, 64-byte swizzle
// (the staging boxes' layout). Groups stride `gstride` elements (fp32 partials).
tp_status make_out_map(CUtensorMap* m, void* ptr, bool f32, int64_t N, int64_t M, int64_t ldo,
                       int64_t groups, int64_t gstride) {
  EncodeTiledFn enc = get_encoder();
  if (!enc) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  const int64_t esz = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M),
                              static_cast<cuuint64_t>(groups)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldo * esz),
                                 static_cast<cuuint64_t>(gstride * esz)};
  const cuuint32_t box[3] = {f32 ? 16u : 32u, 32u, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (code " + std::to_string(r) + ")");
  return TP_OK;
}

template <int BN, int EPI, bool DEC>
tp_status launch_bn_epi(const TcParams& prm, int grid, cudaStream_t st) {
  auto kern = gemm_tc_kernel<BN, EPI, DEC>;
  static std::atomic<uint64_t> attr_set{0};  // per instantiation and device
  if (needs_setup(attr_set)) {
    TP_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     TcCfg<BN, DEC>::SMEM_BYTES));
    mark_device(attr_set);
  }
  TP_CUDA_TRY(launch_kernel(kern, grid, kThreads, TcCfg<BN, DEC>::SMEM_BYTES, st, prm));
  count_launch();
  return TP_OK;
}

template <int BN, bool DEC>
tp_status launch_bn(int epi, const TcParams& prm, int grid, cudaStream_t st) {
  switch (epi) {
    case EPI_STORE: return launch_bn_epi<BN, EPI_STORE, DEC>(prm, grid, st);
    case EPI_GELU: return launch_bn_epi<BN, EPI_GELU, DEC>(prm, grid, st);
    case EPI_SWIGLU: return launch_bn_epi<BN, EPI_SWIGLU, DEC>(prm, grid, st);
    case EPI_DGELU: return launch_bn_epi<BN, EPI_DGELU, DEC>(prm, grid, st);
    case EPI_DSWIGLU: return launch_bn_epi<BN, EPI_DSWIGLU, DEC>(prm, grid, st);
    case EPI_PAIR: return launch_bn_epi<BN, EPI_PAIR, DEC>(prm, grid, st);
  }
  return fail(TP_ERR_INVALID_ARG, "unknown epilogue");
}

template <int EPI, int WN>
tp_status launch_pair_epi(const TcParams& prm, int64_t ntiles, cudaStream_t st) {
  auto kern = gemm_tc2_kernel<EPI, WN>;
  constexpr int kSmem = PairCfg<WN>::SMEM;
  static std::atomic<int> max_pairs_dev[64];  // per instantiation and device (0: unknown)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = -1;
  int max_pairs = dev >= 0 ? max_pairs_dev[dev].load() : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(PairCfg<WN>::THREADS, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query below takes the cluster shape only
  if (max_pairs == 0) {
    TP_CUDA_TRY(
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem));
    cfg.gridDim = dim3(2 * static_cast<unsigned>(device_sm_count() / 2), 1, 1);
    int n = 0;
    TP_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
    if (n <= 0) return fail(TP_ERR_CUDA, "no CTA pair of the GEMM kernel fits on the device");
    max_pairs = n;
    if (dev >= 0) max_pairs_dev[dev].store(n);
  }
  const int pairs = static_cast<int>(std::min<int64_t>(ntiles, max_pairs));
  cfg.gridDim = dim3(2 * static_cast<unsigned>(pairs), 1, 1);
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  TP_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, prm));
  count_launch();
  return TP_OK;
}

template <int WN>
tp_status launch_pair_wn(int epi, const TcParams& prm, int64_t ntiles, cudaStream_t st) {
  switch (epi) {
    case EPI_STORE: return launch_pair_epi<EPI_STORE, WN>(prm, ntiles, st);
    case EPI_GELU: return launch_pair_epi<EPI_GELU, WN>(prm, ntiles, st);
    case EPI_SWIGLU: return launch_pair_epi<EPI_SWIGLU, WN>(prm, ntiles, st);
    case EPI_DGELU: return launch_pair_epi<EPI_DGELU, WN>(prm, ntiles, st);
    case EPI_DSWIGLU: return launch_pair_epi<EPI_DSWIGLU, WN>(prm, ntiles, st);
    case EPI_PAIR: return launch_pair_epi<EPI_PAIR, WN>(prm, ntiles, st);
  }
  return fail(TP_ERR_INVALID_ARG, "unknown epilogue");
}

tp_status launch_pair(int epi, bool wide, const TcParams& prm, int64_t ntiles, cudaStream_t st) {
  return wide ? launch_pair_wn<2>(epi, prm, ntiles, st) : launch_pair_wn<1>(epi, prm, ntiles, st);
}

std::atomic<int> g_debug_hang{0};
// 1: CTA-pair kernel for large problems, 0: one-CTA kernel only, 2: the pair kernel for
// every GEMM it can run (at least 256 rows and 256 TMEM columns), small ones included
std::atomic<int> g_pair_mode{1};
// 256 x 512 pair tiles: 0 never, 1 where the width is whole wide tiles and there are
// at least four per SM pair, 2 whenever the pair kernel runs (tests of the wide form)
std::atomic<int> g_wide_mode{1};

}  // namespace

void set_debug_hang(int v) { g_debug_hang.store(v); }
int debug_hang_flag() { return g_debug_hang.load(); }
void set_pair_mode(int v) { g_pair_mode.store(v); }
void set_wide_mode(int v) { g_wide_mode.store(v); }

// bytes the epilogue writes per output element (logical column) of a row
#ifndef TP_TMA_STORE
#define TP_TMA_STORE 1  // 0: the pair kernel's epilogue stores straight from registers
#endif
#ifndef TP_WIDE_K_PER_BYTE
#define TP_WIDE_K_PER_BYTE 1024
#endif
int epi_out_bytes(const GemmDesc& d) {
  int n = 0;
  for (void* o : d.out) n += o != nullptr;
  return std::max(n, 1) * (d.out_f32 ? 4 : 2);
}

tp_status launch_gemm_tc(const GemmDesc& d, cudaStream_t st) {
  if (d.M <= 0 || d.N <= 0 || d.K <= 0) return TP_OK;
  if (d.paired && d.nseg != 1) return fail(TP_ERR_INVALID_ARG, "paired GEMM needs one K segment");
  if (d.N % 8 != 0) return fail(TP_ERR_SHAPE, "GEMM output width must be a multiple of 8");
  if (d.groups > 1 && d.K % BK != 0)
    return fail(TP_ERR_SHAPE, "per-shard K must be a multiple of 64");
  if (d.nseg < 1 || d.nseg > 3) return fail(TP_ERR_INVALID_ARG, "1 to 3 K segments");
  for (int s = 0; s < d.nseg; ++s)
    if (d.seg_k0[s] % BK != 0 || d.seg_k0[s] > (1ll << 30))
      return fail(TP_ERR_SHAPE, "K segment offsets must be multiples of 64");
  const int epi = d.epi;
  // tile width in TMEM columns: 256 unless the problem is narrow, or has so few rows
  // (decode: M <= 64 tokens, one M-tile) that 128-wide tiles are needed to give
  // every SM its share of the weight stream
  const int64_t n_tmem = d.paired ? 2 * d.N : d.N;
  int BN = (n_tmem >= 256 && d.M > 64) ? 256 : 128;
  // 256 x 256 tiles on CTA pairs once there are at least 256 rows
  bool pair = BN == 256 && d.M >= 256 && g_pair_mode.load() != 0;
  // small problems (a handful of tiles, e.g. M = 1024 tokens at h = 128): narrower
  // one-CTA tiles, down to 128 x 64, while that leaves at most half the SMs busy, so
  // more SMs share the operand loads and the epilogue (unpaired, not the decode form)
  if (!d.paired && d.M > 64 && g_pair_mode.load() != 2) {
    const int64_t sms = device_sm_count();
    auto ctas = [&](int64_t tm, int64_t bn) {
      return (d.M + tm - 1) / tm * ((d.N + bn - 1) / bn) * d.groups;
    };
    if (pair && 2 * ctas(256, 256) * 2 <= sms) pair = false;
    while (!pair && BN > 64 && 2 * ctas(BM, BN) <= sms) BN /= 2;
  }
  const int bn_logical = d.paired ? BN / 2 : BN;
  const int tile_m = pair ? 256 : BM;
  // pair tiles twice as wide (256 x 512): 3/4 of the operand bytes per FLOP, but one
  // accumulator, so most of each tile's epilogue is not hidden behind MMAs: taken
  // where the width is whole wide tiles, the tile's K is long beside the bytes its
  // epilogue writes per output element, and either there are at least four wide tiles
  // per SM pair or the wide tiles need so many fewer waves of the 76 pairs that a wave
  // of them (2 narrow tiles' work at ~10 % more per cycle) still ends first
  // (2048 x 4096 x 2048: 64 wide tiles in one wave, not 128 narrow ones in two)
  bool wide = false;
  if (pair) {
    const int64_t ww = 2 * bn_logical;
    const int64_t rows = (d.M + 255) / 256 * d.groups;
    const int64_t wtiles = rows * ((d.N + ww - 1) / ww);
    const int64_t ntiles = rows * ((d.N + bn_logical - 1) / bn_logical);
    const int64_t pairs_n = std::max<int64_t>(device_sm_count() / 2, 1);
    auto waves = [&](int64_t t) { return (t + pairs_n - 1) / pairs_n; };
    const bool many = wtiles >= 4 * pairs_n || 18 * waves(wtiles) < 10 * waves(ntiles);
    const int64_t k_tile = static_cast<int64_t>(d.nseg) * d.K;
    const int mode = g_wide_mode.load();
    wide = mode == 2 || (mode == 1 && d.N % ww == 0 && many &&
                         k_tile >= static_cast<int64_t>(TP_WIDE_K_PER_BYTE) * epi_out_bytes(d));
  }
  const int tile_w = bn_logical * (wide ? 2 : 1);  // logical output columns of a tile
  // decode configuration: at most 64 K-major rows of A
  const bool dec = !pair && BN == 128 && !d.a_mn && d.M <= 64;
  const int a_rows = dec ? static_cast<int>((d.M + 7) / 8 * 8) : BM;

  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  const int nb = d.paired ? 2 : d.nseg;
  // MN-major operands whose rows are whole 64-column chunks use one 3-D load per stage
  bool a3d = kMn3d && d.a_mn, b3d = kMn3d && d.b_mn;
  for (int s = 0; s < d.nseg; ++s) a3d = a3d && d.A[s].cols % 64 == 0;
  for (int s = 0; s < nb; ++s) b3d = b3d && d.B[s].cols % 64 == 0;
  // B chunks per load: the pair kernel's column half (2), or the whole (half) tile
  const uint32_t b_chunks = pair ? 2u : static_cast<uint32_t>(d.paired ? BN / 128 : BN / 64);
  for (int s = 0; s < d.nseg; ++s) {
    if (a3d) TP_TRY(make_map_3d(&prm.tmA[s], d.A[s], 2));
    else if (d.a_mn) TP_TRY(make_map(&prm.tmA[s], d.A[s], 64, 64));
    else TP_TRY(make_map(&prm.tmA[s], d.A[s], 64, static_cast<uint32_t>(a_rows)));
  }
  for (int s = 0; s < nb; ++s) {
    if (b3d) TP_TRY(make_map_3d(&prm.tmB[s], d.B[s], b_chunks));
    else if (d.b_mn) TP_TRY(make_map(&prm.tmB[s], d.B[s], 64, 64));
    else TP_TRY(make_map(&prm.tmB[s], d.B[s], 64,
                         static_cast<uint32_t>(pair ? 128 : (d.paired ? BN / 2 : BN))));
  }
  prm.a3d = a3d;
  prm.b3d = b3d;
  prm.a_rows = a_rows;
  for (int s = d.nseg; s < 3; ++s) prm.tmA[s] = prm.tmA[0];
  for (int s = nb; s < 3; ++s) prm.tmB[s] = prm.tmB[0];
  for (int s = 0; s < 3; ++s) prm.seg_k0[s] = static_cast<int>(d.seg_k0[s]);
  prm.M = d.M;
  prm.N = d.N;
  prm.K = d.K;
  prm.a_mn = d.a_mn;
  prm.b_mn = d.b_mn;
  prm.nseg = d.nseg;
  prm.paired = d.paired;
  prm.groups = d.groups;
  prm.tiles_m = static_cast<int>((d.M + tile_m - 1) / tile_m);
  prm.tiles_n = static_cast<int>((d.N + tile_w - 1) / tile_w);
  prm.kb_per_seg = static_cast<int>((d.K + BK - 1) / BK);
  prm.shards = 1;
  prm.shard_axis = d.shard_axis;
  if (d.shards > 1) {
    const int along = d.shard_axis == 0 ? prm.tiles_m : prm.tiles_n;
    if (along % d.shards == 0) prm.shards = d.shards;
  }
  prm.out0 = d.out[0];
  prm.out1 = d.out[1];
  prm.out2 = d.out[2];
  prm.in0 = d.in[0];
  prm.in1 = d.in[1];
  prm.ldo = d.ldo;
  prm.out_f32 = d.out_f32;
  prm.out_group_stride = d.out_group_stride;
  {
    const int64_t esz = d.out_f32 ? 4 : 2;
    bool ok = (d.ldo * esz) % 32 == 0 && (!d.out_f32 || (d.out_group_stride * 4) % 32 == 0);
    for (void* o : d.out) ok = ok && reinterpret_cast<uintptr_t>(o) % 32 == 0;
    prm.st32 = ok ? 1 : 0;
    bool ok_in = (d.ldo * 2) % 32 == 0;
    for (const void* i : d.in) ok_in = ok_in && reinterpret_cast<uintptr_t>(i) % 32 == 0;
    prm.ld32 = ok_in ? 1 : 0;
  }
  // pair kernel: outputs staged in shared memory and TMA-stored, where every output's
  // base, pitch and group stride are 16-byte multiples, and there are at least two
  // tiles per SM pair: with one tile per pair the epilogue is the launch's tail, and
  // the staging round trips lengthen it (the 2048^3 GEMM: 898 against 987 TFLOP/s)
  prm.tma_out = 0;
  const int64_t pair_tiles =
      static_cast<int64_t>(prm.tiles_m) * prm.tiles_n * prm.groups;  // set above
  if (pair && TP_TMA_STORE && pair_tiles >= device_sm_count()) {
    const int64_t esz = d.out_f32 ? 4 : 2;
    const int64_t groups = d.out_f32 && d.groups > 1 ? d.groups : 1;
    const int64_t gstride = groups > 1 ? d.out_group_stride : d.ldo * d.M;
    bool ok = (d.ldo * esz) % 16 == 0 && (gstride * esz) % 16 == 0 && gstride > 0;
    for (void* o : d.out) ok = ok && reinterpret_cast<uintptr_t>(o) % 16 == 0;
    if (ok) {
      for (int o = 0; o < 3; ++o)
        if (d.out[o]) TP_TRY(make_out_map(&prm.tmO[o], d.out[o], d.out_f32, d.N, d.M, d.ldo, groups, gstride));
      prm.tma_out = 1;
    }
  }
  prm.status = device_status_word();
  if (!prm.status) return fail(TP_ERR_CUDA, "device status word unavailable");
  prm.timeout_ns = wait_timeout_ns();
  prm.debug_hang = g_debug_hang.load();

  const int64_t ntiles = static_cast<int64_t>(prm.tiles_m) * prm.tiles_n * prm.groups;
  if (ntiles > (1ll << 30)) return fail(TP_ERR_SHAPE, "problem too large");
  if (pair) return launch_pair(epi, wide, prm, ntiles, st);
  const int grid = static_cast<int>(
      std::min<int64_t>(ntiles, static_cast<int64_t>(device_sm_count()) * (dec ? TP_DEC_CTAS_PER_SM : 1)));
  if (dec) return launch_bn<128, true>(epi, prm, grid, st);
  if (BN == 64) return launch_bn<64, false>(epi, prm, grid, st);
  return BN == 256 ? launch_bn<256, false>(epi, prm, grid, st)
                   : launch_bn<128, false>(epi, prm, grid, st);
}

}  // namespace tp

#ifdef TP_GEMM_STATS
// Instrumented builds only: copy out and clear the wait-cycle counters.
extern "C" TP_API int tp_debug_gemm_stats(unsigned long long* out, int ctas) {
  if (ctas > 1024) ctas = 1024;
  if (cudaMemcpyFromSymbol(out, tp::g_gemm_stats, sizeof(unsigned long long) * 16 * ctas) !=
      cudaSuccess)
    return 1;
  static unsigned long long zero[1024][16];
  return cudaMemcpyToSymbol(tp::g_gemm_stats, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
#endif
