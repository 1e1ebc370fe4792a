// Host plumbing of libkvc: status strings, the device error word, the launch
// counter, parameter checks, workspace sizing and the RoPE table.
#include <atomic>
#include <cstddef>
#include <cmath>
#include <mutex>

#include "kvc_common.cuh"
#include "kvc_internal.h"

#include <cstddef>
static_assert(sizeof(kvc_params) == 144, "kvc_params layout");
static_assert(offsetof(kvc_params, salient_extract) == 136, "kvc_params layout");
static_assert(offsetof(kvc_params, tree_cuts) == 128, "kvc_params layout");
static_assert(offsetof(kvc_params, head_full_frac) == 120, "kvc_params layout");
static_assert(offsetof(kvc_params, packed_rows) == 112, "kvc_params layout");
static_assert(offsetof(kvc_params, total_ctx) == 104, "kvc_params layout");
static_assert(offsetof(kvc_params, budget_ratio) == 64, "kvc_params layout");
static_assert(offsetof(kvc_params, decode_reserve) == 96, "kvc_params layout");

// Device error word: first device-detected error code since the last read.
__device__ int32_t g_kvc_err_word;

namespace kvc {

static std::atomic<int64_t> g_launches{0};
static std::mutex g_err_mu;
static int32_t* g_err_ptr[256];

void count_launch(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

static std::atomic<uint64_t> g_wait_ns{kWaitNs};
static std::atomic<int> g_withhold{0};
uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int withhold_copies() { return g_withhold.load(std::memory_order_relaxed); }

// Last CUDA runtime error seen by any call (diagnostics for KVC_ECUDA).
std::atomic<int> g_last_cuda_error{0};
int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return KVC_OK;
  g_last_cuda_error.store((int)e, std::memory_order_relaxed);
  return KVC_ECUDA;
}

static int g_sms[256];
int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
  std::lock_guard<std::mutex> g(g_err_mu);
  if (g_sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

int32_t* err_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> g(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_kvc_err_word) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int32_t*>(ptr);
  }
  return g_err_ptr[dev];
}

int check_params(const kvc_params* p) {
  if (!p) return KVC_EINVAL;
  if (p->B < 1 || p->L < 1 || p->H < 1) return KVC_EINVAL;
  if (!(p->G == 1 || p->G == 2 || p->G == 4 || p->G == 8)) return KVC_EINVAL;
  if (!(p->d == 64 || p->d == 128)) return KVC_EINVAL;
  if (p->P < 1 || p->G * p->P > 256) return KVC_EINVAL;
  if (p->W < p->P) return KVC_EINVAL;
  if (!(p->dtype == KVC_F32 || p->dtype == KVC_BF16)) return KVC_EINVAL;
  if (p->n_max < p->W + 16 || p->S_max < 1) return KVC_EINVAL;
  if (p->decode_reserve < 0 || p->total_ctx < 0 || p->packed_rows < 0) return KVC_EINVAL;
  if (!(p->head_full_frac >= 0.0 && p->head_full_frac <= 1.0)) return KVC_EINVAL;
  return KVC_OK;
}

}  // namespace kvc

extern "C" {

const char* kvc_last_cuda_error(void) {
  const int e = kvc::g_last_cuda_error.load(std::memory_order_relaxed);
  return e == 0 ? "none" : cudaGetErrorString((cudaError_t)e);
}

const char* kvc_status_string(int s) {
  switch (s) {
    case KVC_OK: return "ok";
    case KVC_EINVAL: return "invalid argument";
    case KVC_EBUDGET: return "budget smaller than the recent window";
    case KVC_ECAPACITY: return "append past the reserved capacity";
    case KVC_ECUDA: return "CUDA runtime error";
    case KVC_ETIMEOUT: return "bounded device wait timed out";
    case KVC_EWORKSPACE: return "workspace missing or too small";
    case KVC_EDEVICE: return "device-side check failed";
    case KVC_ESCRATCH: return "problem too large for the allocation-free entry point's scratch";
    default: return "unknown status";
  }
}

int kvc_device_error(void* stream, int32_t* code) {
  if (!code) return KVC_EINVAL;
  int32_t* w = kvc::err_word();
  if (!w) return KVC_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, w, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(w, 0, sizeof(int32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return KVC_ECUDA;
  *code = h;
  return KVC_OK;
}

int64_t kvc_launch_count(void) { return kvc::g_launches.load(); }

int kvc_set_wait_limit(uint64_t first_wait_ns, int32_t withhold_copies) {
  if (first_wait_ns < 1000 || first_wait_ns > kvc::kWaitNs) return KVC_EINVAL;
  kvc::g_wait_ns.store(first_wait_ns, std::memory_order_relaxed);
  kvc::g_withhold.store(withhold_copies ? 1 : 0, std::memory_order_relaxed);
  return KVC_OK;
}

size_t kvc_workspace_bytes(int which, const kvc_params* p) {
  if (kvc::check_params(p) != KVC_OK) return 0;
  switch (which) {
    case KVC_WS_SCORE: return kvc::score_workspace_bytes(p);
    case KVC_WS_SELECT: return kvc::select_workspace_bytes(p);
    case KVC_WS_PACK: return kvc::pack_workspace_bytes(p);
    case KVC_WS_DECODE: return kvc::decode_workspace_bytes(p);
    case KVC_WS_PARTITION: return kvc::partition_workspace_bytes(p);
    default: return 0;
  }
}

}  // extern "C"

// ---------------------------------------------------------------- RoPE table
__global__ void rope_table_kernel(int half, double base, int64_t n_half, float* cos_tab,
                                  float* sin_tab) {
  int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t total = n_half * half;
  if (idx >= total) return;
  int64_t e = idx / half;
  int j = (int)(idx - e * half);
  double theta = pow(base, -2.0 * (double)j / (double)(2 * half));
  double ang = 0.5 * (double)e * theta;
  double s, c;
  sincos(ang, &s, &c);
  cos_tab[idx] = (float)c;
  sin_tab[idx] = (float)s;
}

extern "C" int kvc_rope_table(int32_t d, float base, int64_t n_half, float* cos_tab,
                              float* sin_tab, void* stream) {
  if (!(d == 64 || d == 128) || n_half < 1 || !cos_tab || !sin_tab || !(base > 1.0f))
    return KVC_EINVAL;
  int half = d / 2;
  int64_t total = n_half * half;
  int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 0x7fffffff) return KVC_EINVAL;
  rope_table_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      half, (double)base, n_half, cos_tab, sin_tab);
  kvc::count_launch();
  return kvc::cuda_status(cudaGetLastError());
}
