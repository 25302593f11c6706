// Host helpers of libmtphead.so: cached device attributes and the kernel launch with
// programmatic stream serialization.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {
std::atomic<unsigned long long> g_stage_wait_ns{kWaitLimitNs};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices] = {};
std::set<std::pair<int, const void*>> g_smem_set;  // (device, kernel) with max smem raised
}  // namespace

unsigned long long stage_wait_ns() { return g_stage_wait_ns.load(std::memory_order_relaxed); }

unsigned long long set_stage_wait_ns(unsigned long long ns) {
  return g_stage_wait_ns.exchange(ns, std::memory_order_relaxed);
}

TmapEncodeFn tensor_map_encoder() {
  static std::once_flag once;
  static TmapEncodeFn fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<TmapEncodeFn>(p);
  });
  return fn;
}

cudaError_t device_info(DeviceInfo* info) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_have[dev]) {
    DeviceInfo d{};
    err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    d.smem_optin -= kSmemReserve;  // room for the kernels' static shared variables
    g_info[dev] = d;
    g_have[dev] = true;
  }
  *info = g_info[dev];
  return cudaSuccess;
}

cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    const auto key = std::make_pair(dev, kernel);
    if (g_smem_set.find(key) == g_smem_set.end()) {
      if (!g_have[dev]) return cudaErrorNotReady;  // device_info() runs first
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g_info[dev].smem_optin);
      if (err != cudaSuccess) return err;
      g_smem_set.insert(key);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kernel, args);
}

}  // namespace mtp
