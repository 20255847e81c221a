// Status strings, the device error word, and cached per-device facts.
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace moe {

// The library's device error word (one per device that loads the library). Kernels
// OR MOE_DEVERR_* bits into it through a pointer passed as a parameter.
__device__ uint32_t g_device_error;

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_ready[kMaxDevices];
std::mutex g_mu;
}  // namespace

int current_device(DeviceInfo* out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  if (dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ready[dev]) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    if (d.cc_major != 10 || d.cc_minor != 3) return MOE_ERR_UNSUPPORTED;  // built for sm_103a only
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    d.error_word = static_cast<uint32_t*>(p);
    g_info[dev] = d;
    g_ready[dev] = true;
  }
  *out = g_info[dev];
  return MOE_OK;
}

int prefer_max_shared(const void* func) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  static std::mutex mu;
  static std::vector<std::pair<int, const void*>> done;
  std::lock_guard<std::mutex> lock(mu);
  for (const auto& d : done)
    if (d.first == dev && d.second == func) return MOE_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
      cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  done.emplace_back(dev, func);
  return MOE_OK;
}

}  // namespace moe

extern "C" const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MOE_ERR_ALIGNMENT: return "misaligned pointer";
    case MOE_ERR_CAPACITY: return "size beyond capacity";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_UNSUPPORTED: return "no supported (sm_103) CUDA device";
    case MOE_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

extern "C" int moe_version(void) { return 100; }

extern "C" int moe_device_error(uint32_t* bits, int clear) {
  moe::DeviceInfo d;
  int st = moe::current_device(&d);
  if (st != MOE_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, d.error_word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (bits) *bits = v;
  if (clear) {
    uint32_t z = 0;
    if (cudaMemcpy(d.error_word, &z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
