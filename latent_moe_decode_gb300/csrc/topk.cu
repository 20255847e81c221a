// Sigmoid + e_score_correction_bias top-K with renormalised weights.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer,
// EpMoeLayer.topk (one group, sigmoid scoring, correction bias, renormalize, scale);
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideRoute docstring
// (an exact top-16 with renormalised weights) and WideScratch (ids int32, weights BF16).
//
// Selection key c_e = sigmoid(logit_e) + bias_e; order (c descending, expert index
// ascending); weights are the unbiased scores over their slot-order FP32 sum.
//
// GB300 design: one warp per token for E <= 1024 (four tokens per CTA of 128 threads),
// no CTA barrier. Lane l holds the experts 128 j + 4 l + i (i < 4), so each 16-byte load
// instruction of the warp reads 512 contiguous bytes of the logits row. Selection runs
// in two tiers. Every expert first gets an approximate key (1/2 + tanh(x/2)/2 with the
// hardware's approximate tanh: one MUFU operation, within 2^-11 of the specified sigmoid
// over all inputs). The K-th largest of the 32 lane maxima is a lower bound of the K-th
// largest key (K different lanes hold a key at least that large), found by every lane
// counting the lane maxima above and at least its own (independent shuffles; a bitonic
// sort's 15 dependent exchanges measured 0.1-0.16 us slower a call). Every expert whose approximate key is within a margin of that
// bound (about 23 of 896 for the decode batches) is a candidate -- the margin covers
// twice the approximation error, so the exact top K are among them. Only the candidates
// get the specified sigmoid and their exact keys; up to 64 are ranked by shuffles (each
// candidate counts the candidates whose (key, ~expert) orders before its own:
// independent comparisons), more (heavy ties) by exact keys for all and K rounds of a
// warp argmax. The result is that of the exact keys, bit for bit. (Eight tokens a CTA
// measured slower: 5.6 against 5.1-5.4 us a call at T = 1020, 8.4 against 7.8 at 4096.)
// For 1024 < E <= 4096, or rows that are not 16-byte aligned, one CTA of 4 warps takes
// a token (topk.cuh).
#include "topk.cuh"

namespace moe {
namespace {

using namespace topk_impl;

template <int NJ, bool WARP>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  route_block<NJ, WARP, false>(a, blockIdx.x);
}

// The kernel's dynamic shared memory limit is always set to the largest pad (the cap of
// two), never lowered, so that calls from several host threads with different pads
// cannot race on it.
template <typename Kern>
int launch_capped(Kern kern, dim3 grid, dim3 block, cudaStream_t s, const TopkArgs& a, const DeviceInfo& dev) {
  const void* k = reinterpret_cast<const void*>(kern);
  const size_t pad = cta_cap_pad(k, grid.x, dev), most = cta_cap_pad(k, 2LL * dev.sm_count, dev);
  if (most > 0 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_pdl(kern, grid, block, pad <= most ? pad : 0, s, a);
}

}  // namespace
}  // namespace moe


extern "C" int moe_topk_route(const float* logits, const float* bias, int T, int E, int K,
                              int renormalize, float scale, int32_t* ids, float* weights,
                              uint16_t* weights_bf16, moe_stream_t stream) {
  using namespace moe;
  using namespace moe::topk_impl;
  if (T < 0 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARGUMENT;
  if (E > MOE_MAX_EXPERTS || K > MOE_MAX_TOPK) return MOE_ERR_CAPACITY;
  if (T == 0) return MOE_OK;
  if (!logits || !ids) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(logits, 4) || (bias && !aligned(bias, 4)) || !aligned(ids, 4) || (weights && !aligned(weights, 4)) ||
      (weights_bf16 && !aligned(weights_bf16, 2)))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  TopkArgs a{logits, bias, T, E, K, renormalize ? 1 : 0, scale, ids, weights, weights_bf16};
  const bool warp = use_warp_body(E, logits, bias);
  const dim3 grid((unsigned)route_blocks(T, warp)), block(kThreads);
  cudaStream_t s = as_cuda(stream);
  if (E > kWarpMaxE) return launch_pdl(topk_kernel<32, false>, grid, block, 0, s, a);
  switch ((E + 127) / 128) {  // experts per thread (CTA body) or per lane / 4 (warp body)
#define MOE_TOPK_CASE(N) \
  case N: return warp ? launch_capped(topk_kernel<N, true>, grid, block, s, a, dev) : launch_pdl(topk_kernel<N, false>, grid, block, 0, s, a);
    MOE_TOPK_CASE(1)
    MOE_TOPK_CASE(2)
    MOE_TOPK_CASE(3)
    MOE_TOPK_CASE(4)
    MOE_TOPK_CASE(5)
    MOE_TOPK_CASE(6)
    MOE_TOPK_CASE(7)
    MOE_TOPK_CASE(8)
#undef MOE_TOPK_CASE
  }
  return MOE_ERR_CAPACITY;
}
