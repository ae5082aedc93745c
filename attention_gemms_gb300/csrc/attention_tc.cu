// Tensor-core attention, head_dim 64, bf16, forward and backward, with the head map of
// the CUDA-core kernels (multi-head layout or grouped-query per-shard blocks). Same
// outputs: O (bf16) and lse (fp32, natural log); dqkv (bf16).
//
// Forward: O = softmax(Q K^T / sqrt(d)) V. One CTA per (128 query rows, NH query heads),
// NH = 2 when a key/value head's query heads come in pairs (they share every K/V block),
// else 1; keys in blocks of 64; two CTAs per SM, so one CTA's softmax overlaps the
// other's MMAs (128-key blocks with one CTA per SM took 1.5x longer):
//   the TMA warp (one lane) loads the NH Q tiles once and K, V blocks into two stages
//     straight from the qkv rows (128-byte swizzle, 64 columns = one head);
//   the MMA warp (one lane) owns TMEM (per head S: 64 columns, O: 64) and issues
//     S = Q K^T (M 128, N 64, K 64) and O += P V (M 128, N 64, K 64), serving the
//     heads in turn;
//   four softmax warps per head, one thread per query row, read a block's scores from
//     TMEM once, keep the running maximum (moved lazily) and sum (base 2), write
//     P = 2^(s - m) as bf16 into shared memory in the swizzled K-major layout the MMA
//     reads, and rescale O in TMEM when the maximum moves.
// Ordering: P and the O rescale wait for the head's previous P V (o_done); once the
// softmax warps hand over P (p_full) -- after reading the current S -- the next block's
// S is issued ahead of this block's P V; a K/V stage is refilled after every head's P V
// of it completes (kv_empty).
// Backward (below): a D / lse pair kernel, then dK/dV and dQ kernels that recompute S
// and dP in TMEM.
// Every wait is bounded; on a timeout the CTA records TP_ERR_TIMEOUT, stops issuing,
// waits (bounded) for its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace tp {
namespace {

constexpr int kQ = 128;                   // query rows per CTA = TMEM lanes
constexpr int kKB = 64;                   // keys per block
constexpr int kQTile = kQ * 64 * 2;       // Q: 128 rows x 64 dims, bf16: 16 KB
constexpr int kKVTile = kKB * 64 * 2;     // a K or V block: 64 keys x 64 dims: 8 KB
// Forward layout for NH query heads per CTA (1, or 2 heads sharing a key/value head):
// Q tiles | K/V stages | P tiles | barriers. TMEM: S of head h at 64 h, O at 64 NH + 64 h.
template <int NH>
struct FwdLayout {
  static constexpr int kOffQ = 0;                      // head h: kOffQ + h kQTile
  static constexpr int kOffKV = NH * kQTile;           // stage st: K at kOffKV + 2 st kKVTile, V after
  static constexpr int kOffP = kOffKV + 4 * kKVTile;   // head h: 128 rows x 64 keys (one swizzle atom)
  static constexpr int kOffBar = kOffP + NH * kQ * kKB * 2;
  static constexpr int kSmem = kOffBar + 16 * 8 + 16 + 1024;  // + alignment slack
  static constexpr int kThreads = (4 * NH + 2) * 32;  // 4 softmax warps per head, TMA, MMA
  static constexpr uint32_t kTmemCols = 128 * NH;
};
#ifndef TP_ATTN_CTAS
#define TP_ATTN_CTAS 2  // CTAs per SM the register allocation must allow (3 spills)
#endif
constexpr int kCtasPerSm = TP_ATTN_CTAS;
constexpr uint64_t kDrainNs = 20000000ull;

struct AttnTcParams {
  CUtensorMap tm;       // qkv: (b*s rows, ldq columns), box 64 x 128, 128-byte swizzle (Q)
  CUtensorMap tmkv;     // the same tensor, box 64 x 64 (K, V blocks)
  void* o;              // (b*s, ldo) bf16
  float* lse;           // (b, H, s)
  int s, H, hq, g;      // sequence, query heads, query heads per block, per key/value head
  int64_t S, KO, VO, ldo;
  float scale_log2;     // log2(e) / sqrt(64)
  int causal;
  int* status;
  uint64_t timeout_ns;
  int debug_hang;       // test hook: the MMA thread first waits on a barrier nothing arrives on
};

__device__ __forceinline__ void record_timeout_attn(int* status) {
  atomicCAS(status, 0, static_cast<int>(TP_ERR_TIMEOUT));
  atomicAdd(status + 1, 1);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// generic-proxy shared-memory writes (P) made visible to the tensor cores' async proxy
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x on the special-function unit (PTX ex2.approx.ftz: relative error about 2^-22,
// subnormal results flushed to zero); P is rounded to bf16 right after
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 32 fp32 values times `mul` as bf16 to global memory (16-byte aligned)
__device__ __forceinline__ void st_row_bf16(__nv_bfloat16* dst, const uint32_t* v, float mul) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 w;
    w.x = pack_bf16x2(__uint_as_float(v[8 * u]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
    w.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
    w.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
    w.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
    reinterpret_cast<uint4*>(dst)[u] = w;
  }
}

template <int NH>
__global__ void __launch_bounds__(FwdLayout<NH>::kThreads, kCtasPerSm) attn_fwd_tc_kernel(const __grid_constant__ AttnTcParams p) {
  using Lay = FwdLayout<NH>;
  constexpr int kProd = 4 * NH, kMma = 4 * NH + 1;  // warp roles
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0, drain = bar0 + 8 * 11, never = bar0 + 8 * 12;
  auto kv_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (3 + st); };
  auto s_full = [&](int h) { return bar0 + 8u * (5 + h); };
  auto p_full = [&](int h) { return bar0 + 8u * (7 + h); };
  auto o_done = [&](int h) { return bar0 + 8u * (9 + h); };
  auto s_free = [&](int h) { return bar0 + 8u * (13 + h); };  // slot 12: the test hook's

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, t0 = blockIdx.y * NH, q0 = blockIdx.x * kQ;  // heads t0 .. t0 + NH - 1
  const int blk = t0 / p.hq, tl0 = t0 - blk * p.hq;                     // same key/value head
  auto qcol_of = [&](int h) {
    return static_cast<int>(blk * p.S + static_cast<int64_t>(tl0 + h) * 64);
  };
  const int kc = static_cast<int>(blk * p.S + p.KO + static_cast<int64_t>(tl0 / p.g) * 64);
  const int vc = static_cast<int>(blk * p.S + p.VO + static_cast<int64_t>(tl0 / p.g) * 64);
  const int row0 = b * p.s;
  const int kend = p.causal ? min(p.s, q0 + kQ) : p.s;
  const int nkb = (kend + kKB - 1) / kKB;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(kv_full(st), 1);
      mbar_init(kv_empty(st), 1);
    }
    for (int h = 0; h < NH; ++h) {
      mbar_init(s_full(h), 1);
      mbar_init(p_full(h), 4);  // one arrive per softmax warp of the head
      mbar_init(s_free(h), 4);  // likewise, once a warp has read the head's S out of TMEM
      mbar_init(o_done(h), 1);
    }
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMma) {
    tmem_alloc(smem_u32(tmem_slot), Lay::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();  // the set-up above overlaps the previous kernel
  pdl_trigger();
  auto tS = [&](int h) { return tmem + 64u * h; };
  auto tO = [&](int h) { return tmem + 64u * NH + 64u * h; };
  int issued_kv = 0;  // producer: K/V blocks issued

  if (warp == kProd) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(q_full, NH * kQTile);
      for (int h = 0; h < NH; ++h)
        tma_load_2d(sb + Lay::kOffQ + h * kQTile, &p.tm, q_full, qcol_of(h), row0 + q0);
      for (int j = 0; j < nkb; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(kv_empty(st), ((j >> 1) - 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t dst = sb + Lay::kOffKV + st * 2 * kKVTile;
        mbar_arrive_expect_tx(kv_full(st), 2 * kKVTile);
        tma_load_2d(dst, &p.tmkv, kv_full(st), kc, row0 + j * kKB);
        tma_load_2d(dst + kKVTile, &p.tmkv, kv_full(st), vc, row0 + j * kKB);
        ++issued_kv;
      }
      if (!ok) record_timeout_attn(p.status);
    }
    __syncwarp();
  } else if (warp == kMma) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kKB, 0, 0);  // Q, K both K-major
      const uint32_t id_o = idesc_bf16_f32(128, 64, 0, 1);   // P K-major, V MN-major
      bool ok = mbar_wait(q_full, 0, p.timeout_ns, abort_flag);
      if (ok && p.debug_hang) ok = mbar_wait(never, 0, p.timeout_ns, abort_flag);
      // S_h = Q_h K^T of key block j (the block's K/V stage must have landed)
      auto issue_s = [&](int j, int h) -> bool {
        const int st = j & 1;
        if (!mbar_wait(kv_full(st), (j >> 1) & 1, p.timeout_ns, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kaddr = sb + Lay::kOffKV + st * 2 * kKVTile;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tS(h), sw128_desc(sb + Lay::kOffQ + h * kQTile + kk * 32, 16u, 1024u),
                      sw128_desc(kaddr + kk * 32, 16u, 1024u), id_s, kk > 0 ? 1u : 0u);
        mma_commit(s_full(h));
        return true;
      };
      for (int h = 0; h < NH && ok; ++h) ok = issue_s(0, h);
      for (int j = 0; j < nkb && ok; ++j) {
        const int st = j & 1;
        const uint32_t vaddr = sb + Lay::kOffKV + st * 2 * kKVTile + kKVTile;
        // the heads in turn: while one head's softmax runs, the other's MMAs do
        for (int h = 0; h < NH && ok; ++h) {
          // S_h(j) has been read out of TMEM: the next block's scores are issued while
          // the softmax warps still form P_h(j), and go ahead of P V
          if (!mbar_wait(s_free(h), j & 1, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (j + 1 < nkb && !issue_s(j + 1, h)) {
            ok = false;
            break;
          }
          if (!mbar_wait(p_full(h), j & 1, p.timeout_ns, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kKB / 16; ++kk)
            mma_bf16_ss(tO(h), sw128_desc(sb + Lay::kOffP + h * (kQ * kKB * 2) + kk * 32, 16u, 1024u),
                        sw128_desc(vaddr + kk * 2048, 8192u, 1024u), id_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(o_done(h));
        }
        if (ok) mma_commit(kv_empty(st));  // after every head's P V of block j
      }
      if (!ok) record_timeout_attn(p.status);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax (4 warps per head)
    const int hh = warp >> 2, quarter = warp & 3;
    const int t = t0 + hh;
    const int r = quarter * 32 + lane;  // query row within the tile = TMEM lane
    const int qi = q0 + r;
    const uint32_t lanes = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t sP = sb + Lay::kOffP + hh * (kQ * kKB * 2);
    float m2 = -INFINITY, l = 0.0f;
    bool ok = true;
    // every lane polls the barrier (one warp-wide instruction per poll), so the warp does
    // not split into a waiting lane and 31 lanes parked at a shuffle; the lanes agree on
    // the outcome before any warp-wide TMEM access
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(bar, parity, p.timeout_ns, abort_flag);
      return __all_sync(0xFFFFFFFFu, w) != 0;
    };
    for (int j = 0; j < nkb; ++j) {
      if (!wait_all(s_full(hh), j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = j * kKB;
      uint32_t v[kKB];  // the row's 64 scores, read once
      tmem_ld32(tS(hh) + lanes, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld32(tS(hh) + lanes + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(hh));
      // the block's row maximum (masked keys: beyond the sequence, or after the query)
      const bool full = k0 + kKB <= p.s && !(p.causal && k0 + kKB - 1 > qi);
      float mb = -INFINITY;
      if (full) {
#pragma unroll
        for (int i = 0; i < kKB; ++i) mb = fmaxf(mb, __uint_as_float(v[i]));
        mb *= p.scale_log2;
      } else {
#pragma unroll
        for (int i = 0; i < kKB; ++i) {
          const int key = k0 + i;
          const bool live = key < p.s && !(p.causal && key > qi);
          if (!live) v[i] = __float_as_uint(-INFINITY);
          mb = fmaxf(mb, __uint_as_float(v[i]));
        }
        mb *= p.scale_log2;
      }
      // Lazy rescaling: the running maximum m2 moves only when the block's maximum
      // exceeds it by more than 8 (a factor 256 in P, harmless in bf16 and the fp32
      // sums); otherwise P = 2^(s - m2) with the stale m2 and O needs no rescale.
      // O / l and the log-sum-exp use the same m2, so the result does not change.
      const bool move = mb > m2 + 8.0f;
      const float m_new = move ? mb : m2;
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      const float corr = move ? ex2_approx(m2 - m_use) : 1.0f;  // 0 on the first block
      // P may be overwritten and O rescaled once the previous block's P V is complete
      if (j > 0 && !wait_all(o_done(hh), (j - 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P = 2^(s - m) as bf16 into the swizzled K-major P tile (128-byte rows)
      float sum = 0.0f;
#pragma unroll
      for (int i = 0; i < kKB; ++i) {
        const float e = ex2_approx(fmaf(__uint_as_float(v[i]), p.scale_log2, -m_use));
        sum += e;
        v[i] = __float_as_uint(e);
      }
#pragma unroll
      for (int ch = 0; ch < kKB / 8; ++ch) {  // 8 keys = 16 bytes per store
        const uint32_t addr = sP + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
        const uint32_t* q8 = v + 8 * ch;
        st_shared_v4(addr,
                     pack_bf16x2(__uint_as_float(q8[0]), __uint_as_float(q8[1])),
                     pack_bf16x2(__uint_as_float(q8[2]), __uint_as_float(q8[3])),
                     pack_bf16x2(__uint_as_float(q8[4]), __uint_as_float(q8[5])),
                     pack_bf16x2(__uint_as_float(q8[6]), __uint_as_float(q8[7])));
      }
      l = l * corr + sum;
      m2 = m_new;
      if (j > 0 && __any_sync(0xFFFFFFFFu, move)) {  // O *= corr (a warp-wide TMEM access)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(tO(hh) + lanes + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(tO(hh) + lanes + c * 32, o);
        }
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(hh));
    }
    if (ok && wait_all(o_done(hh), (nkb - 1) & 1)) {
      tc_fence_after();
      const float inv = 1.0f / l;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) +
                            (static_cast<int64_t>(row0) + qi) * p.ldo + static_cast<int64_t>(t) * 64;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(tO(hh) + lanes + c * 32, o);
        tmem_ld_wait();
        if (qi < p.s) st_row_bf16(orow + c * 32, o, inv);
      }
      if (qi < p.s)
        p.lse[(static_cast<int64_t>(b) * p.H + t) * p.s + qi] = (m2 + log2f(l)) * 0.6931471805599453f;
    } else if (lane == 0) {
      record_timeout_attn(p.status);
    }
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (*abort_flag) {
    volatile int no_abort = 0;
    if (warp == kProd && lane == 0) {  // the copies this CTA issued have landed
      mbar_wait(q_full, 0, kDrainNs, &no_abort);
      for (int st = 0; st < 2; ++st) {
        const int n = issued_kv > st ? (issued_kv - 1 - st) / 2 : -1;  // last block on stage st
        if (n >= 0) mbar_wait(kv_full(st), n & 1, kDrainNs, &no_abort);
      }
    }
    if (warp == kMma && lane == 0) {  // and the MMAs it issued have completed
      mma_commit(drain);
      mbar_wait(drain, 0, kDrainNs, &no_abort);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMma) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

// ---------------------------------------------------------------------- backward
//
// dP = dO V^T, P = exp(S / sqrt(d) - lse), dS = P * (dP - D) / sqrt(d), D = rowsum(dO * O);
// dQ = dS K (one CTA per 128 query rows), dK = dS^T Q and dV = P^T dO (one CTA per 128
// key rows of a key/value head, looping over 64-query blocks of every query head of its
// group). The Q / dO / K tiles in shared memory serve as K-major operands of S and dP and
// as MN-major operands of the gradient products (the same 128-byte-swizzled rows read
// along the other dimension).

constexpr int kBwdQKVTile = 128 * 64 * 2;  // 16 KB
constexpr int kBwdBlk = 64 * 64 * 2;       // 8 KB: a 64-row block
// dQ: Q, dO, three K/V stages, dS; dK/dV: K, V, two Q/dO stages, P^T, dS^T, and a
// per-warp table of the 64 (lse, D) pairs of the current query block. + barriers + slack
constexpr int kKvStagesDq = 3;
constexpr int kBwdSmemDq = (3 + kKvStagesDq) * kBwdQKVTile + 256 + 1024;
constexpr int kBwdSmemKv = 6 * kBwdQKVTile + 256 + 8 * 32 * 8 + 1024;

struct AttnBwdParams {
  CUtensorMap tq128, tq64;    // qkv, boxes 64 x 128 and 64 x 64
  CUtensorMap tdo128, tdo64;  // dO, the same boxes
  const float2* ld;           // (b, H, s): (lse log2(e), D)
  void* dqkv;
  int64_t ldq;
  int s, H, hq, g, hkv;
  int64_t S, KO, VO;
  float scale_log2, scale;
  int causal;
  int* status;
  uint64_t timeout_ns;
  int debug_hang;  // test hook, as in the forward's parameters
};

// ld[b, t, q] = (lse log2(e), D) with D = the sum over the head's 64 columns of dO * O;
// eight lanes per (row, head), 16 bytes of O and of dO each
__global__ void __launch_bounds__(256) attn_bwd_dsum_kernel(const __nv_bfloat16* __restrict__ O,
                                                            const __nv_bfloat16* __restrict__ dO,
                                                            const float* __restrict__ lse,
                                                            float2* __restrict__ ld, int64_t rows,
                                                            int s, int H, int64_t ldo) {
  pdl_wait();  // the previous kernel's results are complete and visible
  pdl_trigger();
  const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t w = gt >> 3;
  const int sub = static_cast<int>(gt & 7);
  const bool live = w < rows * H;  // the whole group of eight agrees
  const int64_t row = live ? w / H : 0;
  const int t = live ? static_cast<int>(w - row * H) : 0;
  float acc = 0.0f;
  if (live) {
    const uint4 o4 = *reinterpret_cast<const uint4*>(O + row * ldo + t * 64 + sub * 8);
    const uint4 d4 = *reinterpret_cast<const uint4*>(dO + row * ldo + t * 64 + sub * 8);
    const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, dw[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[i]));
      const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[i]));
      acc = fmaf(a.x, c.x, fmaf(a.y, c.y, acc));
    }
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  if (live && sub == 0) {
    const int64_t b = row / s, q = row - b * s, i = (b * H + t) * s + q;
    ld[i] = make_float2(lse[i] * 1.4426950408889634f, acc);
  }
}


constexpr int kThreadsBwd = 320;  // warps 0-7 element-wise, 8 TMA, 9 MMA

// Element-wise warps of the backward kernels: warp w reads TMEM lanes 32 (w % 4) ..
// + 31 (one row each) and the w / 4-th 32-column half of every 64-column block.
struct BwdLane {
  int quarter, half, r;
  uint32_t lanes;
  __device__ explicit BwdLane(int warp, int lane)
      : quarter(warp & 3), half(warp >> 2), r((warp & 3) * 32 + lane),
        lanes(static_cast<uint32_t>((warp & 3) * 32) << 16) {}
};

// 32 bf16 values, packed in pairs (16 words), of row r into the swizzled tile at column
// half c (16-byte chunks 4c .. 4c + 3)
__device__ __forceinline__ void st_tile_packed(uint32_t tile, int r, int c, const uint32_t* w) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int ch = c * 4 + u;
    const uint32_t addr = tile + (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
    st_shared_v4(addr, w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
  }
}

// dQ: one CTA per (128 query rows, query head); keys in blocks of 64.
// MMA order per block j: [S(j + 1), dP(j + 1)] then dQ(j) += dS(j) K(j), so the
// element-wise warps work on block j + 1 while dQ(j) runs.
__global__ void __launch_bounds__(kThreadsBwd, 2) attn_bwd_dq_tc_kernel(const __grid_constant__ AttnBwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  // Q (16 KB) | dO (16 KB) | K/V stages (K 8 KB, V 8 KB each) | dS (16 KB) | barriers.
  // Three stages: a stage is released once dQ of its key block completes, which comes
  // just before S of the block after next is wanted; the third stage lets its load start
  // a block earlier
  constexpr int NS = kKvStagesDq;
  const uint32_t sQ = sb, sdO = sb + kBwdQKVTile, sKV = sb + 2 * kBwdQKVTile,
                 sdS = sb + (2 + NS) * kBwdQKVTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (3 + NS) * kBwdQKVTile);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  // barriers: qd_full | kv_full[NS] | kv_empty[NS] | s_full p_full o_done drain never s_free
  constexpr int kB = 1 + 2 * NS;
  static_assert(kB + 6 <= 16, "barriers overlap the TMEM slot");
  const uint32_t qd_full = bar0, s_full = bar0 + 8 * kB, p_full = bar0 + 8 * (kB + 1),
                 o_done = bar0 + 8 * (kB + 2), drain = bar0 + 8 * (kB + 3),
                 never = bar0 + 8 * (kB + 4), s_free = bar0 + 8 * (kB + 5);
  auto kv_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (1 + NS + st); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, t = blockIdx.y, q0 = blockIdx.x * 128;
  const int blk = t / p.hq, tl = t - blk * p.hq;
  const int qc = static_cast<int>(blk * p.S + static_cast<int64_t>(tl) * 64);
  const int kc = static_cast<int>(blk * p.S + p.KO + static_cast<int64_t>(tl / p.g) * 64);
  const int vc = static_cast<int>(blk * p.S + p.VO + static_cast<int64_t>(tl / p.g) * 64);
  const int row0 = b * p.s;
  const int kend = p.causal ? min(p.s, q0 + 128) : p.s;
  const int nkb = (kend + 63) / 64;

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    for (int st = 0; st < NS; ++st) {
      mbar_init(kv_full(st), 1);
      mbar_init(kv_empty(st), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 8);  // one arrive per element-wise warp
    mbar_init(s_free, 8);  // likewise, once a warp has read S and dP out of TMEM
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();  // the set-up above overlaps the previous kernel
  pdl_trigger();
  const uint32_t tS = tmem, tdP = tmem + 64, tdQ = tmem + 128;
  int issued = 0;

  if (warp == 8) {
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(qd_full, 2 * kBwdQKVTile);
      tma_load_2d(sQ, &p.tq128, qd_full, qc, row0 + q0);
      tma_load_2d(sdO, &p.tdo128, qd_full, t * 64, row0 + q0);
      for (int j = 0; j < nkb; ++j) {
        const int st = j % NS;
        if (j >= NS && !mbar_wait(kv_empty(st), (j / NS - 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t dst = sKV + st * 2 * kBwdBlk;
        mbar_arrive_expect_tx(kv_full(st), 2 * kBwdBlk);
        tma_load_2d(dst, &p.tq64, kv_full(st), kc, row0 + j * 64);
        tma_load_2d(dst + kBwdBlk, &p.tq64, kv_full(st), vc, row0 + j * 64);
        ++issued;
      }
      if (!ok) record_timeout_attn(p.status);
    }
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t id_g = idesc_bf16_f32(128, 64, 0, 1);
      bool ok = mbar_wait(qd_full, 0, p.timeout_ns, abort_flag);
      if (ok && p.debug_hang) ok = mbar_wait(never, 0, p.timeout_ns, abort_flag);
      auto issue_s = [&](int j) -> bool {  // S = Q K^T and dP = dO V^T of key block j
        const int st = j % NS;
        if (!mbar_wait(kv_full(st), (j / NS) & 1, p.timeout_ns, abort_flag)) return false;
        tc_fence_after();
        const uint32_t k = sKV + st * 2 * kBwdBlk, v = k + kBwdBlk;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tS, sw128_desc(sQ + kk * 32, 16u, 1024u), sw128_desc(k + kk * 32, 16u, 1024u),
                      id_s, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tdP, sw128_desc(sdO + kk * 32, 16u, 1024u), sw128_desc(v + kk * 32, 16u, 1024u),
                      id_s, kk > 0 ? 1u : 0u);
        mma_commit(s_full);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkb && ok; ++j) {
        // S and dP of block j have been read out of TMEM: the next block's are issued
        // while the element-wise warps still form dS of block j
        if (!mbar_wait(s_free, j & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (j + 1 < nkb && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(p_full, j & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = j % NS;
        const uint32_t k = sKV + st * 2 * kBwdBlk;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dQ += dS K (K read MN-major: rows = keys)
          mma_bf16_ss(tdQ, sw128_desc(sdS + kk * 32, 16u, 1024u),
                      sw128_desc(k + kk * 2048, 8192u, 1024u), id_g, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(o_done);
        mma_commit(kv_empty(st));
      }
      if (!ok) record_timeout_attn(p.status);
    }
    __syncwarp();
  } else {
    const BwdLane L(warp, lane);
    const int qi = q0 + L.r;
    const bool valid = qi < p.s;
    const float2 ld = valid ? p.ld[(static_cast<int64_t>(b) * p.H + t) * p.s + qi]
                            : make_float2(0.0f, 0.0f);
    const float lse2 = ld.x, Dq = ld.y;
    bool ok = true;
    // every lane polls the barrier (one warp-wide instruction per poll), so the warp does
    // not split into a waiting lane and 31 lanes parked at a shuffle; the lanes agree on
    // the outcome before any warp-wide TMEM access
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(bar, parity, p.timeout_ns, abort_flag);
      return __all_sync(0xFFFFFFFFu, w) != 0;
    };
    for (int j = 0; j < nkb; ++j) {
      if (!wait_all(s_full, j & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[32], pv[32];
      tmem_ld32(tS + L.lanes + L.half * 32, sv);
      tmem_ld32(tdP + L.lanes + L.half * 32, pv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      const int k0 = j * 64 + L.half * 32;
      uint32_t dk[16];  // P (dP - D) as packed bf16 pairs; 1 / sqrt(d) applied to dQ at the end
      if (valid && k0 + 32 <= p.s && !(p.causal && k0 + 31 > qi)) {
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          dk[i >> 1] = pack_bf16x2(
              ex2_approx(fmaf(__uint_as_float(sv[i]), p.scale_log2, -lse2)) *
                  (__uint_as_float(pv[i]) - Dq),
              ex2_approx(fmaf(__uint_as_float(sv[i + 1]), p.scale_log2, -lse2)) *
                  (__uint_as_float(pv[i + 1]) - Dq));
      } else {  // keys beyond the sequence or after the query, rows beyond the sequence
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = k0 + i + e;
            const bool live = valid && key < p.s && !(p.causal && key > qi);
            const float pr =
                live ? ex2_approx(fmaf(__uint_as_float(sv[i + e]), p.scale_log2, -lse2)) : 0.0f;
            ds[e] = pr * (__uint_as_float(pv[i + e]) - Dq);
          }
          dk[i >> 1] = pack_bf16x2(ds[0], ds[1]);
        }
      }
      // the dS tile is free once the previous block's dQ MMA has completed
      if (j > 0 && !wait_all(o_done, (j - 1) & 1)) {
        ok = false;
        break;
      }
      st_tile_packed(sdS, L.r, L.half, dk);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && wait_all(o_done, (nkb - 1) & 1)) {
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tdQ + L.lanes + L.half * 32, v);
      tmem_ld_wait();
      if (valid)
        st_row_bf16(static_cast<__nv_bfloat16*>(p.dqkv) + (static_cast<int64_t>(row0) + qi) * p.ldq +
                        qc + L.half * 32,
                    v, p.scale);
    } else if (lane == 0) {
      record_timeout_attn(p.status);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    volatile int no_abort = 0;
    if (warp == 8 && lane == 0) {
      mbar_wait(qd_full, 0, kDrainNs, &no_abort);
      for (int st = 0; st < NS; ++st) {
        const int n = issued > st ? (issued - 1 - st) / NS : -1;
        if (n >= 0) mbar_wait(kv_full(st), n & 1, kDrainNs, &no_abort);
      }
    }
    if (warp == 9 && lane == 0) {
      mma_commit(drain);
      mbar_wait(drain, 0, kDrainNs, &no_abort);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// dK, dV: one CTA per (128 key rows, key/value head of a block); work items = (query
// head of the group, 64-query block). MMA order per item w: [S^T(w + 1), dP^T(w + 1)]
// then dV += P^T(w) dO(w), dK += dS^T(w) Q(w).
__global__ void __launch_bounds__(kThreadsBwd, 2) attn_bwd_dkdv_tc_kernel(const __grid_constant__ AttnBwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  // K (16 KB) | V (16 KB) | Q0 dO0 Q1 dO1 (8 KB each) | P^T (16 KB) | dS^T (16 KB) | barriers
  const uint32_t sK = sb, sV = sb + kBwdQKVTile, sQD = sb + 2 * kBwdQKVTile,
                 sPT = sb + 4 * kBwdQKVTile, sdST = sb + 5 * kBwdQKVTile;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * kBwdQKVTile);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float2* ldtab = reinterpret_cast<float2*>(smem + 6 * kBwdQKVTile + 256);  // [8 warps][32]
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t kv_full = bar0, s_full = bar0 + 8 * 5, p_full = bar0 + 8 * 6,
                 o_done = bar0 + 8 * 7, drain = bar0 + 8 * 8, never = bar0 + 8 * 9,
                 s_free = bar0 + 8 * 10;
  auto qd_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto qd_empty = [&](int st) { return bar0 + 8u * (3 + st); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, u = blockIdx.y, k0 = blockIdx.x * 128;
  const int blk = u / p.hkv, kvl = u - blk * p.hkv;
  const int kc = static_cast<int>(blk * p.S + p.KO + static_cast<int64_t>(kvl) * 64);
  const int vc = static_cast<int>(blk * p.S + p.VO + static_cast<int64_t>(kvl) * 64);
  const int row0 = b * p.s;
  const int qb0 = p.causal ? k0 / 64 : 0;      // earlier queries see none of these keys
  const int nqb = (p.s + 63) / 64 - qb0;
  const int nw = p.g * nqb;                    // (query head of the group, query block)

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int st = 0; st < 2; ++st) {
      mbar_init(qd_full(st), 1);
      mbar_init(qd_empty(st), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 8);
    mbar_init(s_free, 8);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  pdl_wait();  // the set-up above overlaps the previous kernel
  pdl_trigger();
  const uint32_t tST = tmem, tdPT = tmem + 64, tdV = tmem + 128, tdK = tmem + 192;
  auto head_of = [&](int w) { return blk * p.hq + kvl * p.g + w / nqb; };
  int issued = 0;

  if (warp == 8) {
    if (lane == 0) {
      bool ok = true;
      mbar_arrive_expect_tx(kv_full, 2 * kBwdQKVTile);
      tma_load_2d(sK, &p.tq128, kv_full, kc, row0 + k0);
      tma_load_2d(sV, &p.tq128, kv_full, vc, row0 + k0);
      for (int w = 0; w < nw; ++w) {
        const int st = w & 1;
        if (w >= 2 && !mbar_wait(qd_empty(st), ((w >> 1) - 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        const int t = head_of(w), tl = t - blk * p.hq, qb = qb0 + w % nqb;
        const int qc = static_cast<int>(blk * p.S + static_cast<int64_t>(tl) * 64);
        const uint32_t dst = sQD + st * 2 * kBwdBlk;
        mbar_arrive_expect_tx(qd_full(st), 2 * kBwdBlk);
        tma_load_2d(dst, &p.tq64, qd_full(st), qc, row0 + qb * 64);
        tma_load_2d(dst + kBwdBlk, &p.tdo64, qd_full(st), t * 64, row0 + qb * 64);
        ++issued;
      }
      if (!ok) record_timeout_attn(p.status);
    }
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t id_g = idesc_bf16_f32(128, 64, 0, 1);
      bool ok = mbar_wait(kv_full, 0, p.timeout_ns, abort_flag);
      if (ok && p.debug_hang) ok = mbar_wait(never, 0, p.timeout_ns, abort_flag);
      auto issue_s = [&](int w) -> bool {  // S^T = K Q^T and dP^T = V dO^T of item w
        const int st = w & 1;
        if (!mbar_wait(qd_full(st), (w >> 1) & 1, p.timeout_ns, abort_flag)) return false;
        tc_fence_after();
        const uint32_t q = sQD + st * 2 * kBwdBlk, d = q + kBwdBlk;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tST, sw128_desc(sK + kk * 32, 16u, 1024u), sw128_desc(q + kk * 32, 16u, 1024u),
                      id_s, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tdPT, sw128_desc(sV + kk * 32, 16u, 1024u), sw128_desc(d + kk * 32, 16u, 1024u),
                      id_s, kk > 0 ? 1u : 0u);
        mma_commit(s_full);
        return true;
      };
      if (ok && nw > 0) ok = issue_s(0);
      for (int w = 0; w < nw && ok; ++w) {
        // S^T and dP^T of item w have been read out of TMEM: the next item's are issued
        // while the element-wise warps still form P^T and dS^T of item w
        if (!mbar_wait(s_free, w & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (w + 1 < nw && !issue_s(w + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(p_full, w & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = w & 1;
        const uint32_t q = sQD + st * 2 * kBwdBlk, d = q + kBwdBlk;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dV += P^T dO (dO read MN-major: rows = queries)
          mma_bf16_ss(tdV, sw128_desc(sPT + kk * 32, 16u, 1024u),
                      sw128_desc(d + kk * 2048, 8192u, 1024u), id_g, (w > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // dK += dS^T Q
          mma_bf16_ss(tdK, sw128_desc(sdST + kk * 32, 16u, 1024u),
                      sw128_desc(q + kk * 2048, 8192u, 1024u), id_g, (w > 0 || kk > 0) ? 1u : 0u);
        mma_commit(o_done);
        mma_commit(qd_empty(st));
      }
      if (!ok) record_timeout_attn(p.status);
    }
    __syncwarp();
  } else {
    const BwdLane L(warp, lane);
    const int kj = k0 + L.r;
    const bool valid = kj < p.s;
    bool ok = true;
    // every lane polls the barrier (one warp-wide instruction per poll), so the warp does
    // not split into a waiting lane and 31 lanes parked at a shuffle; the lanes agree on
    // the outcome before any warp-wide TMEM access
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = mbar_wait(bar, parity, p.timeout_ns, abort_flag);
      return __all_sync(0xFFFFFFFFu, w) != 0;
    };
    float2* tab = ldtab + warp * 32;
    const float4* tab4 = reinterpret_cast<const float4*>(tab);
    // the (lse, D) pair of this lane's query in item w (this warp's 32 queries); loaded
    // one item ahead so the global load's latency overlaps the current item
    auto ld_pair = [&](int w) -> float2 {
      const int q = (qb0 + w % nqb) * 64 + L.half * 32 + lane;
      return q < p.s ? p.ld[(static_cast<int64_t>(b) * p.H + head_of(w)) * p.s + q]
                     : make_float2(0.0f, 0.0f);
    };
    float2 ld_next = nw > 0 ? ld_pair(0) : make_float2(0.0f, 0.0f);
    for (int w = 0; w < nw; ++w) {
      if (!wait_all(s_full, w & 1)) {
        ok = false;
        break;
      }
      const int qh = (qb0 + w % nqb) * 64 + L.half * 32;  // this warp's 32 queries
      tab[lane] = ld_next;  // the previous item's reads of the table ended at its __syncwarp
      __syncwarp();
      if (w + 1 < nw) ld_next = ld_pair(w + 1);
      tc_fence_after();
      uint32_t sv[32], pv[32];
      tmem_ld32(tST + L.lanes + L.half * 32, sv);
      tmem_ld32(tdPT + L.lanes + L.half * 32, pv);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      // P^T and P^T (dP^T - D) as packed bf16 pairs; 1 / sqrt(d) applied to dK at the end
      uint32_t pk[16], dk[16];
      // bit c set: query qh + c sees this lane's key (it is in the sequence, the key row
      // is, and, causal, the key does not come after it); one loop for full and masked
      // items (two specialised loops exceed the register budget of two 320-thread CTAs
      // per SM), so the test per entry is one bit of this word
      const int hi = valid ? min(p.s - qh, 32) : 0;
      const int lo = p.causal ? max(kj - qh, 0) : 0;
      const uint32_t live_bits =
          hi <= lo ? 0u : ((hi - lo == 32 ? 0xFFFFFFFFu : ((1u << (hi - lo)) - 1u)) << lo);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float4 l4 = tab4[i >> 1];  // (lse, D) of queries qh + i, qh + i + 1
        float pr[2], ds[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float l2 = e ? l4.z : l4.x, dq = e ? l4.w : l4.y;
          const float x = fmaf(__uint_as_float(sv[i + e]), p.scale_log2, -l2);
          pr[e] = ex2_approx((live_bits & (1u << (i + e))) ? x : -INFINITY);  // 2^-inf = 0
          ds[e] = pr[e] * (__uint_as_float(pv[i + e]) - dq);
        }
        pk[i >> 1] = pack_bf16x2(pr[0], pr[1]);
        dk[i >> 1] = pack_bf16x2(ds[0], ds[1]);
      }
      // the P^T and dS^T tiles are free once the previous item's dV, dK MMAs completed
      if (w > 0 && !wait_all(o_done, (w - 1) & 1)) {
        ok = false;
        break;
      }
      st_tile_packed(sPT, L.r, L.half, pk);
      st_tile_packed(sdST, L.r, L.half, dk);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && (nw == 0 || wait_all(o_done, (nw - 1) & 1))) {
      tc_fence_after();
      __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.dqkv) + (static_cast<int64_t>(row0) + kj) * p.ldq;
      uint32_t v[32];
      if (nw > 0) {
        tmem_ld32(tdV + L.lanes + L.half * 32, v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      if (valid) st_row_bf16(drow + vc + L.half * 32, v, 1.0f);
      if (nw > 0) {
        tmem_ld32(tdK + L.lanes + L.half * 32, v);
        tmem_ld_wait();
      }
      if (valid) st_row_bf16(drow + kc + L.half * 32, v, p.scale);
    } else if (lane == 0) {
      record_timeout_attn(p.status);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    volatile int no_abort = 0;
    if (warp == 8 && lane == 0) {
      mbar_wait(kv_full, 0, kDrainNs, &no_abort);
      for (int st = 0; st < 2; ++st) {
        const int n = issued > st ? (issued - 1 - st) / 2 : -1;
        if (n >= 0) mbar_wait(qd_full(st), n & 1, kDrainNs, &no_abort);
      }
    }
    if (warp == 9 && lane == 0) {
      mma_commit(drain);
      mbar_wait(drain, 0, kDrainNs, &no_abort);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                             CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                             CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}

}  // namespace

// Whether the tensor-core forward takes this problem: bf16, head_dim 64, and a qkv
// row pitch TMA can address.
bool attention_tc_eligible(tp_dtype dt, int d, int64_t ldq, const void* qkv, const void* o,
                           int64_t ldo) {
  return dt == TP_BF16 && d == 64 && (ldq * 2) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(qkv) % 16 == 0 && reinterpret_cast<uintptr_t>(o) % 16 == 0 &&
         (ldo * 2) % 16 == 0;
}

tp_status launch_attention_fwd_tc(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                                  int heads, int hq, int g, int64_t S, int64_t KO, int64_t VO,
                                  int64_t ldq, int64_t ldo, int causal, cudaStream_t st) {
  if (b <= 0 || s <= 0) return TP_OK;
  if (b * s > 2147483647ll || ldq > 2147483647ll) return fail(TP_ERR_SHAPE, "attention too large");
  EncodeFn enc = encoder();
  if (!enc) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  AttnTcParams p{};
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(ldq), static_cast<cuuint64_t>(b * s)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldq) * 2};
  const cuuint32_t estr[2] = {1, 1};
  for (int m = 0; m < 2; ++m) {
    const cuuint32_t box[2] = {64, m == 0 ? static_cast<cuuint32_t>(kQ) : static_cast<cuuint32_t>(kKB)};
    const CUresult r = enc(m == 0 ? &p.tm : &p.tmkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                           const_cast<void*>(qkv), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")");
  }
  p.o = o;
  p.lse = lse;
  p.s = static_cast<int>(s);
  p.H = heads;
  p.hq = hq;
  p.g = g;
  p.S = S;
  p.KO = KO;
  p.VO = VO;
  p.ldo = ldo;
  p.scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  p.causal = causal;
  p.status = device_status_word();
  if (!p.status) return fail(TP_ERR_CUDA, "device status word unavailable");
  p.timeout_ns = wait_timeout_ns();
  p.debug_hang = debug_hang_flag();
  static std::atomic<uint64_t> attr_set{0};
  if (needs_setup(attr_set)) {
    TP_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_tc_kernel<1>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     FwdLayout<1>::kSmem));
    TP_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_tc_kernel<2>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     FwdLayout<2>::kSmem));
    mark_device(attr_set);
  }
  // two query heads per CTA when a key/value head's query heads come in pairs (the
  // pair shares every K/V block, and one head's softmax overlaps the other's MMAs)
  const int nh = g % 2 == 0 ? 2 : 1;
  const dim3 grid(static_cast<unsigned>((s + kQ - 1) / kQ), static_cast<unsigned>(heads / nh),
                  static_cast<unsigned>(b));
  if (nh == 2)
    TP_CUDA_TRY(launch_kernel(attn_fwd_tc_kernel<2>, grid, FwdLayout<2>::kThreads,
                              FwdLayout<2>::kSmem, st, p));
  else
    TP_CUDA_TRY(launch_kernel(attn_fwd_tc_kernel<1>, grid, FwdLayout<1>::kThreads,
                              FwdLayout<1>::kSmem, st, p));
  count_launch();
  return TP_OK;
}

bool attention_bwd_tc_eligible(tp_dtype dt, int d, int64_t ldq, const void* qkv, const void* o,
                               const void* dO, const void* dqkv, int64_t ldo) {
  return attention_tc_eligible(dt, d, ldq, qkv, o, ldo) &&
         reinterpret_cast<uintptr_t>(dO) % 16 == 0 && reinterpret_cast<uintptr_t>(dqkv) % 16 == 0;
}

size_t attention_bwd_tc_ws_bytes(int64_t b, int64_t s, int heads) {
  return static_cast<size_t>(b) * s * heads * sizeof(float2);
}

tp_status launch_attention_bwd_tc(const void* qkv, const void* o, const float* lse, const void* dO,
                                  void* dqkv, void* ldws, int64_t b, int64_t s, int heads, int hq,
                                  int g, int hkv, int kv_total, int64_t S, int64_t KO, int64_t VO,
                                  int64_t ldq, int64_t ldo, int causal, cudaStream_t st) {
  if (b <= 0 || s <= 0) return TP_OK;
  if (b * s > 2147483647ll || ldq > 2147483647ll) return fail(TP_ERR_SHAPE, "attention too large");
  if (!ldws || reinterpret_cast<uintptr_t>(ldws) % 16 != 0)
    return fail(TP_ERR_INVALID_ARG, "attention backward workspace missing or misaligned");
  EncodeFn enc = encoder();
  if (!enc) return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  AttnBwdParams p{};
  auto encode = [&](CUtensorMap* m, const void* ptr, int64_t cols, uint32_t box_rows) -> tp_status {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(b * s)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return fail(TP_ERR_CUDA, "cuTensorMapEncodeTiled failed (code " + std::to_string(r) + ")");
    return TP_OK;
  };
  TP_TRY(encode(&p.tq128, qkv, ldq, 128));
  TP_TRY(encode(&p.tq64, qkv, ldq, 64));
  TP_TRY(encode(&p.tdo128, dO, ldo, 128));
  TP_TRY(encode(&p.tdo64, dO, ldo, 64));
  p.ld = static_cast<const float2*>(ldws);
  p.dqkv = dqkv;
  p.ldq = ldq;
  p.s = static_cast<int>(s);
  p.H = heads;
  p.hq = hq;
  p.g = g;
  p.hkv = hkv;
  p.S = S;
  p.KO = KO;
  p.VO = VO;
  p.scale_log2 = 1.4426950408889634f / 8.0f;  // log2(e) / sqrt(64)
  p.scale = 0.125f;                           // 1 / sqrt(64)
  p.causal = causal;
  p.status = device_status_word();
  if (!p.status) return fail(TP_ERR_CUDA, "device status word unavailable");
  p.timeout_ns = wait_timeout_ns();
  p.debug_hang = debug_hang_flag();
  static std::atomic<uint64_t> attr_set{0};
  if (needs_setup(attr_set)) {
    TP_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dq_tc_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmemDq));
    TP_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dkdv_tc_kernel,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmemKv));
    mark_device(attr_set);
  }
  const int64_t pairs = b * s * heads;
  TP_CUDA_TRY(launch_kernel(attn_bwd_dsum_kernel, static_cast<unsigned>((pairs * 8 + 255) / 256),
                            256, 0, st, static_cast<const __nv_bfloat16*>(o),
                            static_cast<const __nv_bfloat16*>(dO), lse, static_cast<float2*>(ldws),
                            b * s, static_cast<int>(s), heads, ldo));
  const unsigned tiles = static_cast<unsigned>((s + 127) / 128);
  // dQ and dK/dV are independent: dQ runs on a side stream beside dK/dV, whose grid
  // (one CTA per 128 key rows of a key/value head) often leaves CTA slots free
  SideBranch br(st, 1);
  const cudaError_t e1 = launch_kernel(
      attn_bwd_dq_tc_kernel, dim3(tiles, static_cast<unsigned>(heads), static_cast<unsigned>(b)),
      kThreadsBwd, kBwdSmemDq, br.stream(), p);
  const cudaError_t e2 = launch_kernel(
      attn_bwd_dkdv_tc_kernel,
      dim3(tiles, static_cast<unsigned>(kv_total), static_cast<unsigned>(b)), kThreadsBwd,
      kBwdSmemKv, st, p);
  count_launch(3);
  TP_TRY(br.join());
  if (e1 != cudaSuccess) return cuda_fail(e1, "attn_bwd_dq_tc_kernel launch");
  TP_CUDA_TRY(e2);
  return TP_OK;
}

}  // namespace tp
