// Per-device facts the launchers need, looked up once per device and cached (host side).
// Every launch runs on the calling thread's current device, so each cache is keyed by
// that device; a process driving several GPUs gets each GPU's own values.
#include <map>
#include <mutex>
#include <utility>

#include "internal.h"

namespace dcp {

namespace {
std::mutex g_mu;
std::map<int, int> g_sms;                                   // device -> SM count
std::map<std::pair<int, const void*>, size_t> g_smem;       // (device, kernel) -> limit set
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) return it->second;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 2)
    sms = 148;
  g_sms[dev] = sms;
  return sms;
}

cudaError_t raise_smem_limit(const void* kernel, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  const auto key = std::make_pair(dev, kernel);
  auto it = g_smem.find(key);
  if (it != g_smem.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  g_smem[key] = bytes;
  return cudaSuccess;
}

}  // namespace dcp
