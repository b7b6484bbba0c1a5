// Status strings, workspace initialisation, device status word, process-wide settings of libdominotree.
#include <atomic>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "dt_internal.cuh"

namespace dt {
namespace {
std::atomic<uint64_t> g_barrier_timeout_ns{2000000000ull};
std::atomic<int> g_lookahead{0};
std::atomic<int> g_topm_cluster{1};
}
uint64_t barrier_timeout_ns() { return g_barrier_timeout_ns.load(std::memory_order_relaxed); }
int lookahead_setting() { return g_lookahead.load(std::memory_order_relaxed); }
bool topm_cluster_setting() { return g_topm_cluster.load(std::memory_order_relaxed) != 0; }

namespace {
std::mutex g_cache_mu;
std::vector<DeviceInfo> g_devices;
struct SmemSetting {
  int dev;
  const void* fn;
  size_t bytes;
};
std::vector<SmemSetting> g_smem;
}  // namespace

cudaError_t current_device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    for (const DeviceInfo& d : g_devices)
      if (d.dev == dev) {
        *out = d;
        return cudaSuccess;
      }
  }
  DeviceInfo d{dev, 0, 0, 0, 0};
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cluster, cudaDevAttrClusterLaunch, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  g_devices.push_back(d);
  *out = d;
  return cudaSuccess;
}

cudaError_t ensure_dynamic_smem(const void* fn, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  SmemSetting* have = nullptr;
  for (SmemSetting& sset : g_smem)
    if (sset.dev == dev && sset.fn == fn) have = &sset;
  if (have && have->bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  if (have) have->bytes = bytes;
  else g_smem.push_back(SmemSetting{dev, fn, bytes});
  return cudaSuccess;
}
}  // namespace dt

extern "C" const char* dt_status_string(dt_status s) {
  switch (s) {
    case DT_OK: return "ok";
    case DT_ERR_INVALID_ARG: return "invalid argument";
    case DT_ERR_UNSUPPORTED: return "outside the supported envelope";
    case DT_ERR_CUDA: return "CUDA runtime error";
    case DT_ERR_TIMEOUT: return "grid-barrier wait ran out of its time budget";
    case DT_ERR_NUMERIC: return "NaN among the logits";
  }
  return "unknown status";
}

extern "C" int dt_abi_version(void) { return DT_ABI_VERSION; }

extern "C" void dt_set_barrier_timeout_ns(uint64_t ns) {
  dt::g_barrier_timeout_ns.store(ns, std::memory_order_relaxed);
}

extern "C" dt_status dt_set_lookahead(int k) {
  if (k < 0 || k > DT_MAX_LOOKAHEAD) return DT_ERR_INVALID_ARG;
  dt::g_lookahead.store(k, std::memory_order_relaxed);
  return DT_OK;
}

extern "C" dt_status dt_set_topm_cluster(int enable) {
  if (enable != 0 && enable != 1) return DT_ERR_INVALID_ARG;
  dt::g_topm_cluster.store(enable, std::memory_order_relaxed);
  return DT_OK;
}

extern "C" dt_status dt_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace || workspace_bytes < sizeof(dt::WsHeader) || !dt::aligned16(workspace)) return DT_ERR_INVALID_ARG;
  return dt::cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, stream));
}

extern "C" dt_status dt_get_error(void* workspace, cudaStream_t stream) {
  if (!workspace || !dt::aligned16(workspace)) return DT_ERR_INVALID_ARG;
  unsigned status = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&status, workspace, sizeof status, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return DT_ERR_CUDA;
  if (status != 0) {  // clear the status word (the abort word stays until the workspace is re-initialised)
    e = cudaMemsetAsync(workspace, 0, sizeof status, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return DT_ERR_CUDA;
  }
  return static_cast<dt_status>(status);
}

extern "C" dt_status dt_build_stats_read(void* workspace, dt_build_stats* out, cudaStream_t stream) {
  if (!workspace || !out || !dt::aligned16(workspace)) return DT_ERR_INVALID_ARG;
  dt::WsHeader h{};
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&h, workspace, sizeof h, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return DT_ERR_CUDA;
  out->launch_ns = h.stat_launch_ns;
  out->gather_ns = h.stat_gather_ns;
  out->gather_bytes = h.stat_gather_bytes;
  out->waves = static_cast<int32_t>(h.stat_waves);
  out->expansions = static_cast<int32_t>(h.stat_expansions);
  return DT_OK;
}
