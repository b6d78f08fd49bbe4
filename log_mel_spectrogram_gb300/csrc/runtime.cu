// runtime.cu -- host-side services shared by the entry points: status
// strings, per-thread CUDA error record, per-device facts, kernel attribute
// setup, per-launch tokens and the workspace error-word readback.
#include <atomic>
#include <chrono>
#include <cstdlib>
#include <mutex>
#include <random>
#include <set>
#include <utility>
#include <vector>

#include "internal.h"

namespace lm {

namespace {
thread_local int g_last_cuda_error = 0;
std::mutex g_mu;
std::vector<DeviceInfo> g_devices;            // indexed by device ordinal
std::set<std::pair<const void *, int>> g_smem_set;  // (kernel, device) already configured
}  // namespace

lm_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  (void)cudaGetLastError();  // clear the sticky-free error state of the runtime
  return LM_ERR_CUDA;
}

lm_status current_device_info(DeviceInfo *info) {
  int dev = 0;
  LM_CUDA_TRY(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < static_cast<int>(g_devices.size()) && g_devices[dev].device == dev) {
      *info = g_devices[dev];
      return LM_OK;
    }
  }
  DeviceInfo d;
  d.device = dev;
  LM_CUDA_TRY(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
  LM_CUDA_TRY(cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev >= static_cast<int>(g_devices.size())) g_devices.resize(dev + 1);
  g_devices[dev] = d;
  *info = d;
  return LM_OK;
}

lm_status ensure_smem_attribute(const void *kernel, int bytes) {
  int dev = 0;
  LM_CUDA_TRY(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_set.count({kernel, dev})) return LM_OK;
  }
  DeviceInfo d;
  if (lm_status st = current_device_info(&d); st != LM_OK) return st;
  if (bytes > d.max_smem_optin) return LM_ERR_UNSUPPORTED;
  // Opt into the device maximum once, so any smaller request also fits.
  LM_CUDA_TRY(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem_optin));
  std::lock_guard<std::mutex> lk(g_mu);
  g_smem_set.insert({kernel, dev});
  return LM_OK;
}

const char *env_or(const char *name, const char *fallback) {
  const char *v = std::getenv(name);
  return (v && *v) ? v : fallback;
}

uint64_t call_token(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (cs != cudaStreamCaptureStatusNone) return 0;
  static std::atomic<uint64_t> counter{[] {
    std::random_device rd;
    const uint64_t r = (static_cast<uint64_t>(rd()) << 32) ^ rd();
    return r ^ static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count());
  }()};
  uint64_t t = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  if (t == 0) t = counter.fetch_add(1, std::memory_order_relaxed) + 1;  // 0 means "no token"
  return t;
}

}  // namespace lm

extern "C" const char *lm_status_string(int status) {
  switch (status) {
    case LM_OK: return "LM_OK";
    case LM_ERR_INVALID_ARG: return "LM_ERR_INVALID_ARG: null pointer or invalid size";
    case LM_ERR_UNSUPPORTED: return "LM_ERR_UNSUPPORTED: request outside the supported range";
    case LM_ERR_MISALIGNED: return "LM_ERR_MISALIGNED: pointer lacks the required alignment";
    case LM_ERR_CUDA: return "LM_ERR_CUDA: a CUDA runtime call failed";
    case LM_ERR_OUT_OF_MEMORY: return "LM_ERR_OUT_OF_MEMORY: plan tables could not be allocated";
    case LM_ERR_DEVICE_FAULT: return "LM_ERR_DEVICE_FAULT: a kernel's bounded wait ran out";
    case LM_ERR_WORKSPACE: return "LM_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown lm_status";
  }
}

extern "C" int lm_last_cuda_error(void) { return lm::g_last_cuda_error; }

extern "C" int lm_version(void) { return 100; }

extern "C" lm_status lm_workspace_error(const void *workspace, size_t workspace_bytes, uint32_t *device_error,
                                        lm_stream_t stream) {
  if (!workspace || !device_error) return LM_ERR_INVALID_ARG;
  if (workspace_bytes < lm::kWorkspaceHeaderBytes) return LM_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  LM_CUDA_TRY(cudaStreamSynchronize(s));
  uint32_t v = 0;
  LM_CUDA_TRY(cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost));
  *device_error = v;
  return v ? LM_ERR_DEVICE_FAULT : LM_OK;
}
