// Runtime plumbing of libtpmlp: thread-local error detail, the per-device sticky
// status word that bounded device waits report into, the wait limit, SM counts,
// the launch counter and the per-device side stream of SideBranch.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <mutex>
#include <string>

#include "internal.h"

namespace tp {

// status[0]: first error code recorded by a kernel; status[1]: how many CTAs gave up.
__device__ int g_tp_status[4];

namespace {
thread_local std::string t_err;
std::atomic<uint64_t> g_timeout_ns{0};
std::atomic<uint64_t> g_launches{0};
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

struct Side {
  std::recursive_mutex mu;  // held from a branch's fork to its join (nesting allowed)
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ready = false, failed = false;
};
Side g_side[kMaxDevices][SideBranch::kSlots];
}  // namespace

SideBranch::SideBranch(cudaStream_t main, int slot) : main_(main) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || slot < 0 ||
      slot >= kSlots)
    return;
  Side& sd = g_side[dev][slot];
  std::unique_lock<std::recursive_mutex> lk(sd.mu);
  if (!sd.ready) {
    // created outside stream capture only; while the caller's stream is being captured
    // (or after a failed creation) the branch runs on the caller's stream
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (sd.failed || cudaStreamIsCapturing(main, &cs) != cudaSuccess ||
        cs != cudaStreamCaptureStatusNone)
      return;
    if (cudaStreamCreateWithFlags(&sd.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) {
      sd.failed = true;
      cudaGetLastError();
      return;
    }
    sd.ready = true;
  }
  side_ = &sd;
  lock_ = std::move(lk);
  if (fork() != TP_OK) {  // a failed fork: run on the caller's stream instead
    side_ = nullptr;
    lock_ = std::unique_lock<std::recursive_mutex>();
  }
}

cudaStream_t SideBranch::stream() const {
  return side_ ? static_cast<Side*>(side_)->stream : main_;
}

tp_status SideBranch::fork() {
  if (!side_) return TP_OK;
  Side& sd = *static_cast<Side*>(side_);
  TP_CUDA_TRY(cudaEventRecord(sd.fork, main_));
  TP_CUDA_TRY(cudaStreamWaitEvent(sd.stream, sd.fork, 0));
  return TP_OK;
}

tp_status SideBranch::join() {
  if (!side_) return TP_OK;
  Side& sd = *static_cast<Side*>(side_);
  side_ = nullptr;
  const cudaError_t a = cudaEventRecord(sd.join, sd.stream);
  const cudaError_t b = a == cudaSuccess ? cudaStreamWaitEvent(main_, sd.join, 0) : a;
  lock_ = std::unique_lock<std::recursive_mutex>();
  if (b != cudaSuccess) return cuda_fail(b, "joining the side stream");
  return TP_OK;
}

SideBranch::~SideBranch() {
  if (side_) join();
}

void set_error(const std::string& msg) { t_err = msg; }

tp_status fail(tp_status s, const std::string& msg) {
  t_err = std::string(tp_status_string(s)) + ": " + msg;
  return s;
}

tp_status cuda_fail(cudaError_t e, const char* what) {
  t_err = std::string("TP_ERR_CUDA: ") + what + ": " + cudaGetErrorString(e);
  return TP_ERR_CUDA;
}

int* device_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_tp_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

uint64_t wait_timeout_ns() {
  const uint64_t v = g_timeout_ns.load();
  return v ? v : kDefaultTimeoutNs;
}

void count_launch(int n) { g_launches.fetch_add(static_cast<uint64_t>(n)); }

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("TP_NO_PDL");
    return !(e && e[0] == '1');
  }();
  return on;
}

// The kernels are built for sm_103a only.
tp_status check_device() {
  int dev = 0, maj = 0, min = 0;
  TP_CUDA_TRY(cudaGetDevice(&dev));
  TP_CUDA_TRY(cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev));
  TP_CUDA_TRY(cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev));
  if (maj != 10 || min != 3)
    return fail(TP_ERR_UNSUPPORTED, "device is sm_" + std::to_string(maj) + std::to_string(min) +
                                        "; this library is built for sm_103a");
  return TP_OK;
}

}  // namespace tp

extern "C" {

int tp_version(void) { return TPMLP_VERSION; }

const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_INVALID_ARG: return "TP_ERR_INVALID_ARG";
    case TP_ERR_SHAPE: return "TP_ERR_SHAPE";
    case TP_ERR_DTYPE: return "TP_ERR_DTYPE";
    case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT";
    case TP_ERR_WORKSPACE: return "TP_ERR_WORKSPACE";
    case TP_ERR_CUDA: return "TP_ERR_CUDA";
    case TP_ERR_TIMEOUT: return "TP_ERR_TIMEOUT";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED";
  }
  return "TP_ERR_UNKNOWN";
}

const char* tp_last_error(void) { return tp::t_err.c_str(); }

void tp_set_wait_timeout_ns(uint64_t ns) { tp::g_timeout_ns.store(ns); }

uint64_t tp_launch_count(void) { return tp::g_launches.load(); }

tp_status tp_check_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TP_CUDA_TRY(cudaStreamSynchronize(st));
  int* d = tp::device_status_word();
  if (!d) return tp::fail(TP_ERR_CUDA, "device status word unavailable");
  int h[4] = {0, 0, 0, 0};
  TP_CUDA_TRY(cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost));
  if (h[0] == 0) return TP_OK;
  const int zero[4] = {0, 0, 0, 0};
  TP_CUDA_TRY(cudaMemcpy(d, zero, sizeof(zero), cudaMemcpyHostToDevice));
  return tp::fail(static_cast<tp_status>(h[0]),
                  "a bounded device wait expired in " + std::to_string(h[1]) + " CTA role(s)");
}

}  // extern "C"
