// Internal interfaces of libtpmlp: the GEMM problem descriptor shared by the
// tensor-core (tcgen05) and CUDA-core engines, epilogue kinds, launchers and
// error plumbing. Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <cstddef>
#include <cstdint>
#include <initializer_list>
#include <string>
#include <utility>

#include "../../include/tpmlp.h"

namespace tp {

// ------------------------------------------------------------------ errors

void set_error(const std::string& msg);  // thread-local detail for tp_last_error
tp_status fail(tp_status s, const std::string& msg);
tp_status cuda_fail(cudaError_t e, const char* what);

#define TP_CUDA_TRY(expr)                                   \
  do {                                                      \
    cudaError_t _e = (expr);                                \
    if (_e != cudaSuccess) return ::tp::cuda_fail(_e, #expr); \
  } while (0)

#define TP_TRY(expr)                    \
  do {                                  \
    tp_status _s = (expr);              \
    if (_s != TP_OK) return _s;         \
  } while (0)

// per-device sticky status word (device address) and the wait limit
int* device_status_word();             // for the current device; nullptr on failure
uint64_t wait_timeout_ns();
int device_sm_count();                 // current device
// One-time per-device set-up (kernel attributes): true when `done` has no mark for the
// current device; mark_device(done) records it. The set-up is idempotent, so two
// threads racing only repeat it. Devices beyond 63 are set up on every call.
inline uint64_t device_bit() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  return 1ull << dev;
}
inline bool needs_setup(const std::atomic<uint64_t>& done) {
  const uint64_t b = device_bit();
  return b == 0 || (done.load(std::memory_order_acquire) & b) == 0;
}
inline void mark_device(std::atomic<uint64_t>& done) { done.fetch_or(device_bit()); }
void count_launch(int n = 1);
// test hook (tp_debug_inject_wait_fault): kernels launched while it is set make their
// MMA thread wait on a barrier nothing arrives on, so the bounded wait runs out
int debug_hang_flag();

// An independent branch of one library call on a per-device side stream: the
// constructor forks it off `main` (an event recorded on `main`, waited for by the side
// stream), fork() re-forks it at a later point of `main`, join() makes `main` wait for
// everything enqueued on stream() (the destructor joins when the caller did not). A
// recursive mutex per device is held from construction to the join, so branches of
// concurrent calls do not interleave on the shared stream (a nested branch on the same
// thread shares it and only adds ordering). While `main` is being captured into a
// graph before the side stream exists, or if it cannot be created, stream() is `main`
// and the branch runs in order. Slots are separate side streams, for branches that may
// nest (the attention backward's inside the attention block's).
class SideBranch {
 public:
  static constexpr int kSlots = 2;
  explicit SideBranch(cudaStream_t main, int slot = 0);
  ~SideBranch();
  SideBranch(const SideBranch&) = delete;
  SideBranch& operator=(const SideBranch&) = delete;
  cudaStream_t stream() const;
  tp_status fork();
  tp_status join();

 private:
  cudaStream_t main_;
  void* side_ = nullptr;
  std::unique_lock<std::recursive_mutex> lock_;
};

// ------------------------------------------------------------------ launches
//
// Programmatic dependent launch: every kernel of the library is launched (launch_kernel)
// so that its CTAs may start while the kernel before it on the stream is finishing. A
// kernel calls pdl_wait() before its first access to global memory -- everything the
// earlier kernels of the stream wrote is then complete and visible, and nothing they
// still read is overwritten -- and pdl_trigger() right after, which lets the next
// kernel's CTAs start their own set-up (barrier init, TMEM allocation, tensor-map
// prefetch) in turn. The next kernel launches only once every CTA of this one has
// passed its trigger, so a waiting CTA never holds resources an earlier kernel's CTA
// still needs. Without the attribute (the environment variable TP_NO_PDL=1) the
// instructions return at once and the stream serialises the kernels as usual.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ GEMM problem

// Epilogue applied to each accumulator tile.
enum EpiKind : int {
  EPI_STORE = 0,    // out[0] = acc (+ in[0] residual)
  EPI_GELU = 1,     // out[0] = acc (pre-activation, optional), out[1] = GELU(acc)
  EPI_SWIGLU = 2,   // paired: out[0] = g (optional), out[1] = u (optional), out[2] = SiLU(g) u
  EPI_DGELU = 3,    // out[0] = acc * GELU'(in[0])
  EPI_DSWIGLU = 4,  // a = acc, g = in[0], u = in[1]: out[0] = dG, out[1] = dU
  EPI_PAIR = 5,     // paired: out[0] = first half, out[1] = second half
  EPI_COUNT = 6
};

// A 2-D row-major tensor in storage order.
struct Operand {
  const void* ptr = nullptr;
  int64_t rows = 0, cols = 0;  // storage extents
  int64_t ld = 0;              // row pitch, elements
};

// D (M x N) = sum_{s < nseg} sum_k A_s(m, k0_s + k) B_s(k0_s + k, n), per K-group g:
//   A(m, k) is A.ptr[m * ld + k] (K-major) or A.ptr[k * ld + m] (a_mn: MN-major),
//   B(k, n) is B.ptr[n * ld + k] (K-major) or B.ptr[k * ld + n] (b_mn: MN-major);
//   segment s starts at K offset seg_k0[s]; group g reads k in [g*K, (g+1)*K) of
//   every segment and writes its output g*out_group_stride elements further (the
//   per-shard partial buffers of the shard sum).
// paired: B[0] feeds the first half of every tile's columns and B[1] the second;
//   logical column n of the output takes B[0](., n) and B[1](., n) (gate/up).
struct GemmDesc {
  int64_t M = 0, N = 0, K = 0;
  bool a_mn = false, b_mn = false;
  int nseg = 1;  // <= 3
  Operand A[3], B[3];
  int64_t seg_k0[3] = {0, 0, 0};
  bool paired = false;
  int groups = 1;
  int shards = 1;      // tile order: `shards` equal slabs along shard_axis, slab-major
  int shard_axis = 1;  // 0 = M, 1 = N
  int epi = EPI_STORE;
  void* out[3] = {nullptr, nullptr, nullptr};
  const void* in[2] = {nullptr, nullptr};
  int64_t ldo = 0;     // row pitch of outputs and of in[] (elements)
  bool out_f32 = false;  // EPI_STORE: fp32 output (partials), else the element type
  int64_t out_group_stride = 0;
  tp_dtype dtype = TP_BF16;
};

tp_status launch_gemm_tc(const GemmDesc& d, cudaStream_t st);    // bf16, tcgen05
bool gemv_eligible(const GemmDesc& d);                             // bf16, M <= 4
tp_status launch_gemv(const GemmDesc& d, cudaStream_t st);
tp_status launch_gemm_simt(const GemmDesc& d, cudaStream_t st);  // fp32, CUDA cores
// blocks_per_sm: CTAs of 256 threads per SM of the grid-stride grid (8 saturates HBM
// alone; 2 leaves room on every SM for a persistent GEMM CTA running beside it).
// group_stride: elements from one shard's partial to the next (0: M * n), so that a
// block of rows of larger partial buffers can be summed on its own
tp_status launch_shard_reduce(const float* P, const void* residual, void* out, int N,
                              int64_t M, int64_t n, tp_dtype out_dtype, cudaStream_t st,
                              int blocks_per_sm = 8, int64_t group_stride = 0);
// sum + residual, rounded to dt, then LayerNorm of the rounded row: h % 8 == 0,
// h <= kReduceLnMaxH, 16-byte aligned buffers
constexpr int64_t kReduceLnMaxH = 16384;
tp_status launch_shard_reduce_ln(const float* P, const void* residual, const float* gamma,
                                 const float* beta, void* sum_out, void* y, float* mean,
                                 float* rstd, int N, int64_t M, int64_t h, float eps,
                                 tp_dtype dt, cudaStream_t st);

inline tp_status launch_gemm(const GemmDesc& d, cudaStream_t st) {
  if (d.dtype != TP_BF16) return launch_gemm_simt(d, st);
  return gemv_eligible(d) ? launch_gemv(d, st) : launch_gemm_tc(d, st);
}

// ------------------------------------------------------------------ other kernels

tp_status launch_layernorm_fwd(const void* x, const float* gamma, const float* beta, void* y,
                               float* mean, float* rstd, int64_t M, int64_t h, float eps,
                               tp_dtype dt, cudaStream_t st);
tp_status launch_layernorm_bwd(const void* x, const float* gamma, const float* mean,
                               const float* rstd, const void* dy, const void* dres, void* dx,
                               float* dgamma, float* dbeta, int64_t M, int64_t h, void* ws,
                               tp_dtype dt, cudaStream_t st);
// LN backward whose parameter gradients are also kept per rank: rank r owns rows
// [r M / ranks, (r + 1) M / ranks) (M % ranks == 0); dgamma = sum over ranks in order
tp_status launch_layernorm_bwd_ranks(const void* x, const float* gamma, const float* mean,
                                     const float* rstd, const void* dy, const void* dres,
                                     void* dx, float* dgamma, float* dbeta, float* dgamma_ranks,
                                     float* dbeta_ranks, int64_t M, int64_t h, int ranks,
                                     void* ws, tp_dtype dt, cudaStream_t st);
size_t layernorm_bwd_ws_bytes(int64_t M, int64_t h, int ranks = 1);
size_t attn_workspace_size(bool fwd, int64_t M, int64_t h, int32_t N, tp_dtype dt,
                           tp_reduce mode);
size_t layer_workspace_size(bool fwd, int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt,
                            tp_reduce mode);
tp_status launch_attention_fwd(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                               int64_t h, int heads, int causal, tp_dtype dt, cudaStream_t st);
// ldws: nullable scratch of attention_bwd_tc_ws_bytes(b, s, heads) bytes (16-byte aligned);
// with it, bf16 head_dim 64 takes the tensor-core backward, without it the CUDA-core one
tp_status launch_attention_bwd(const void* qkv, const void* o, const float* lse, const void* dO,
                               void* dqkv, void* ldws, int64_t b, int64_t s, int64_t h, int heads,
                               int causal, tp_dtype dt, cudaStream_t st);
// grouped-query layout (per-shard blocks [Q heads | K heads | V heads], key/value heads
// replicated per block when kv_heads < N); o (M, heads * d)
tp_status launch_gqa_attention_fwd(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                                   int heads, int kv_heads, int N, int d, int causal, tp_dtype dt,
                                   cudaStream_t st);
// tensor-core forward (attention_tc.cu): bf16, head_dim 64
bool attention_tc_eligible(tp_dtype dt, int d, int64_t ldq, const void* qkv, const void* o,
                           int64_t ldo);
tp_status launch_attention_fwd_tc(const void* qkv, void* o, float* lse, int64_t b, int64_t s,
                                  int heads, int hq, int g, int64_t S, int64_t KO, int64_t VO,
                                  int64_t ldq, int64_t ldo, int causal, cudaStream_t st);
// tensor-core backward: (lse, D) pairs into ldws, then dK/dV and dQ
bool attention_bwd_tc_eligible(tp_dtype dt, int d, int64_t ldq, const void* qkv, const void* o,
                               const void* dO, const void* dqkv, int64_t ldo);
size_t attention_bwd_tc_ws_bytes(int64_t b, int64_t s, int heads);
tp_status launch_attention_bwd_tc(const void* qkv, const void* o, const float* lse, const void* dO,
                                  void* dqkv, void* ldws, int64_t b, int64_t s, int heads, int hq,
                                  int g, int hkv, int kv_total, int64_t S, int64_t KO, int64_t VO,
                                  int64_t ldq, int64_t ldo, int causal, cudaStream_t st);
tp_status launch_gqa_attention_bwd(const void* qkv, const void* o, const float* lse,
                                   const void* dO, void* dqkv, void* ldws, int64_t b, int64_t s,
                                   int heads, int kv_heads, int N, int d, int causal, tp_dtype dt,
                                   cudaStream_t st);

// vocabulary-parallel embedding / cross-entropy and AdamW (vocab.cu)
tp_status launch_vocab_embed_fwd(const int32_t* ids, const void* E, void* x, int64_t M, int64_t v,
                                 int64_t h, int N, tp_dtype dt, cudaStream_t st);
tp_status launch_vocab_embed_bwd(const int32_t* ids, const void* dx, void* dE, int64_t M,
                                 int64_t v, int64_t h, bool accumulate, tp_dtype dt,
                                 cudaStream_t st);
tp_status launch_vocab_ce_fwd(const void* logits, const int32_t* targets, float* lse,
                              float* row_loss, float* shard_loss, float* loss, int64_t M,
                              int64_t v, int N, tp_dtype dt, cudaStream_t st);
tp_status launch_vocab_ce_bwd(const void* logits, const int32_t* targets, const float* lse,
                              void* dlogits, int64_t M, int64_t v, float scale, tp_dtype dt,
                              cudaStream_t st);
tp_status launch_adamw(float* p, const float* g, float* m, float* v, int64_t n, float lr,
                       float b1, float b2, float eps, float wd, float bc1, float bc2,
                       cudaStream_t st);
// AdamW whose step count (for the bias corrections) is read from device memory
tp_status launch_adamw_dev(float* p, const float* g, float* m, float* v, int64_t n,
                           const int32_t* step, float lr, float b1, float b2, float eps, float wd,
                           cudaStream_t st);
// *step += 1; hist[(*step - 1) % hist_len] = *loss (when loss and hist are given)
tp_status launch_step_advance(int32_t* step, const float* loss, float* hist, int64_t hist_len,
                              cudaStream_t st);

// ------------------------------------------------------------------ API helpers (api.cu)

tp_status need(bool cond, tp_status s, const char* msg);
tp_status check_aligned(std::initializer_list<const void*> ptrs);
tp_status check_dtype(tp_dtype dt);
tp_status check_device();
size_t partial_bytes(int64_t M, int64_t n, int32_t N, tp_reduce mode);
bool extents_ok(int64_t rows, int64_t cols, int64_t N);  // see check_extents
tp_status check_extents(int64_t rows, int64_t cols, int64_t N);
tp_status check_mlp_shape(int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt);
size_t sp_mlp_workspace_size(bool fwd, int64_t M, int64_t h, int64_t f, int32_t N, tp_dtype dt,
                             tp_act act, tp_reduce mode);
// w_out_in: W stored (n, k) (TP_W_OUT_IN) instead of (k, n)
tp_status row_impl(const void* Xs, const void* W, const void* residual, void* out, int64_t M,
                   int64_t k, int64_t n, int32_t N, tp_dtype dt, tp_reduce mode, void* ws,
                   cudaStream_t st, bool w_out_in = false);
tp_status row_ln_impl(const void* Xs, const void* W, const void* residual, const float* gamma,
                      const float* beta, void* sum_out, void* y, float* mean, float* rstd,
                      int64_t M, int64_t k, int64_t n, int32_t N, float eps, tp_dtype dt,
                      tp_reduce mode, void* ws, cudaStream_t st);
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t elem_size(tp_dtype t) { return t == TP_BF16 ? 2 : 4; }

}  // namespace tp
