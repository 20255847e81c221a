// Router logits without a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they compute the
// router logits: an engine that hands all device memory to its own pool at start-up
// and forbids allocations afterwards, or a plug-in that is only given input and output
// buffers. For them this entry point runs the same tensor-core split-K kernels as
// moe_router_logits, with the split-K partials kept in a fixed array that the library
// itself reserves in device memory (on every GPU that loads the library, until exit).
//
// The array is read only after the GEMM has overwritten every element that is read
// (each split writes its full tile), so nothing in it needs to start at zero. All
// calls on a device share it: calls whose kernels overlap on the GPU race.
#include <mutex>

#include "router.cuh"

namespace moe {
namespace {

constexpr size_t kScratchBytes = MOE_ROUTER_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
float* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the array on the current device: looked up once per device (with
// that device current) on the first call, then cached.
int scratch_address(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_router_logits_noalloc(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E,
                                         moe_stream_t stream) {
  using namespace moe;
  if (T < 1 || E < 1 || H < 8 || H % 8 != 0) return MOE_ERR_INVALID_ARGUMENT;
  if ((long long)T * E > (1LL << 40)) return MOE_ERR_CAPACITY;  // as moe_router_logits
  if (!x || !w || !logits) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(logits, 4)) return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  // the kernel moe_router_logits picks for a handful of tokens needs no scratch
  if (T <= kAutoGemvMaxTokens) return launch_router_gemv(x, w, logits, T, H, E, as_cuda(stream));
  const TcPlan p = tc_plan(T, H, E, dev.sm_count);
  const size_t need = tc_workspace(p, T, E);
  if (need > kScratchBytes) return MOE_ERR_CAPACITY;
  float* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  return launch_router_tc(x, w, logits, T, H, E, p, scratch, dev.error_word, as_cuda(stream));
}
