// Router logits: the C ABI and the choice between the two kernel families.
#include "router.cuh"

namespace moe {
namespace {

constexpr int kAlgoAuto = 0, kAlgoSimt = 1, kAlgoTc = 2;

// A handful of tokens: the CUDA-core GEMV (one pass over the gate, no split-K);
// otherwise the tensor cores.
int pick(int algo, int T) {
  if (algo != kAlgoAuto) return algo;
  return T <= kAutoGemvMaxTokens ? kAlgoSimt : kAlgoTc;
}

size_t workspace_for(int T, int H, int E, int sm_count) {
  int S = 1, kc = 0;
  simt_plan(T, H, E, sm_count, &S, &kc);
  const size_t simt = S > 1 ? (size_t)S * T * E * sizeof(float) : 0;
  const size_t tc = tc_workspace(tc_plan(T, H, E, sm_count), T, E);
  return simt > tc ? simt : tc;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_router_logits_workspace(int T, int H, int E) {
  moe::DeviceInfo dev;
  if (T < 1 || H < 8 || E < 1 || moe::current_device(&dev) != MOE_OK) return 0;
  return moe::workspace_for(T, H, E, dev.sm_count);
}

extern "C" int moe_router_logits_ex(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E,
                                    void* workspace, size_t workspace_bytes, int algo, moe_stream_t stream) {
  using namespace moe;
  if (T < 1 || E < 1 || H < 8 || H % 8 != 0) return MOE_ERR_INVALID_ARGUMENT;
  if (algo < kAlgoAuto || algo > kAlgoTc) return MOE_ERR_INVALID_ARGUMENT;
  if ((long long)T * E > (1LL << 40)) return MOE_ERR_CAPACITY;
  if (!x || !w || !logits) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(logits, 4)) return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const size_t need = workspace_for(T, H, E, dev.sm_count);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16))) return MOE_ERR_WORKSPACE;
  float* part = static_cast<float*>(workspace);
  cudaStream_t s = as_cuda(stream);
  if (pick(algo, T) == kAlgoSimt) {
    if (T <= kGemvMaxTokens) return launch_router_gemv(x, w, logits, T, H, E, s);
    int S = 1, kc = 0;
    simt_plan(T, H, E, dev.sm_count, &S, &kc);
    return launch_router_simt(x, w, logits, T, H, E, S, kc, part, s);
  }
  return launch_router_tc(x, w, logits, T, H, E, tc_plan(T, H, E, dev.sm_count), part, dev.error_word, s);
}

extern "C" int moe_router_logits(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E,
                                 void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  return moe_router_logits_ex(x, w, logits, T, H, E, workspace, workspace_bytes, 0, stream);
}

extern "C" size_t moe_front_projection_workspace(int T, int H, int E, int L) {
  moe::DeviceInfo dev;
  if (T < 1 || H < 8 || E < 1 || L < 1 || moe::current_device(&dev) != MOE_OK) return 0;
  return moe::front_workspace(moe::front_plan(T, H, E, L, dev.sm_count), T, E, L);
}

extern "C" int moe_front_projection(const uint16_t* x, const uint16_t* w_router, const uint16_t* w_down, float* logits,
                                    uint16_t* latent, int T, int H, int E, int L, void* workspace,
                                    size_t workspace_bytes, moe_stream_t stream) {
  using namespace moe;
  if (T < 1 || E < 1 || L < 1 || H < 8 || H % 8 != 0) return MOE_ERR_INVALID_ARGUMENT;
  if ((long long)T * (E > L ? E : L) > (1LL << 40) || (long long)E + L >= (1LL << 24)) return MOE_ERR_CAPACITY;
  if (!x || !w_router || !w_down || !logits || !latent) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(w_down, 16) || !aligned(logits, 4) || !aligned(latent, 2))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const TcPlan p = front_plan(T, H, E, L, dev.sm_count);
  const size_t need = front_workspace(p, T, E, L);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16))) return MOE_ERR_WORKSPACE;
  return launch_front_tc(x, w_router, w_down, logits, latent, T, H, E, L, p, static_cast<float*>(workspace),
                         dev.error_word, as_cuda(stream));
}
