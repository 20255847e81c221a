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
// GB300 design: one CTA of 4 warps per token. Thread i holds the experts i + 128 j
// (j < NJ), so each load instruction of a warp reads 128 contiguous bytes of the
// logits row. Selection runs in two tiers. Every expert first gets an approximate key
// (the hardware's approximate exp2 and reciprocal: within 1.79e-7 of the specified
// sigmoid over all inputs). The K-th largest of the 128 thread maxima is a lower bound
// of the K-th largest key (K different threads hold a key at least that large): each
// warp sorts its 32 maxima with a bitonic network over shuffles, and two rounds of
// bitonic merging of the four sorted lists give the top 32 of all 128. Every expert
// whose approximate key is within a margin of that bound (about 17 of 896 for random
// scores) is a candidate -- the margin covers twice the approximation error, so the
// exact top K are among them. Only the candidates get the specified sigmoid and their
// exact keys; up to 32 are ranked by one warp (each lane counts the candidates whose
// (key, ~expert) orders before its own: 32 independent comparisons), 32 < count <= 64
// by counting over shared memory, more (heavy ties) by exact keys for all and K rounds
// of argmax. The result is that of the exact keys, bit for bit.
#include "topk.cuh"

namespace moe {
namespace {

using namespace topk_impl;

template <int NJ>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkArgs a) {
  topk_token<NJ>(a, blockIdx.x);
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
  dim3 grid(T), block(kThreads);
  cudaStream_t s = as_cuda(stream);
  switch ((E + 127) / 128) {
    case 1: return launch_pdl(topk_kernel<1>, grid, block, 0, s, a);
    case 2: return launch_pdl(topk_kernel<2>, grid, block, 0, s, a);
    case 3: return launch_pdl(topk_kernel<3>, grid, block, 0, s, a);
    case 4: return launch_pdl(topk_kernel<4>, grid, block, 0, s, a);
    case 5: return launch_pdl(topk_kernel<5>, grid, block, 0, s, a);
    case 6: return launch_pdl(topk_kernel<6>, grid, block, 0, s, a);
    case 7: return launch_pdl(topk_kernel<7>, grid, block, 0, s, a);
    case 8: return launch_pdl(topk_kernel<8>, grid, block, 0, s, a);
  }
  return MOE_ERR_CAPACITY;
}
