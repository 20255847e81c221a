// The routing-and-combine step as one call: the four launches of the chain, in order,
// on the caller's stream. The router is launched the ordinary way (it starts once its
// predecessor has completed) and signals its dependents after that; the later kernels
// use programmatic dependent launch and wait for their predecessor only before reading
// what the chain wrote -- the MXFP8 CTAs (a step input) not at all, Finalize only at
// its end, so it streams its rows while the lists kernel runs.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideMoE.run
// (router -> route -> Finalize on one stream) and ...moe.ep.layer, EpMoeLayer.__call__.
#include "common.cuh"

extern "C" size_t moe_route_finalize_workspace(int T, int H, int E, int K) {
  return moe_router_logits_workspace(T, H, E) + moe_build_routing_lists_workspace(T, K, E);
}

extern "C" int moe_route_finalize(const uint16_t* x, const uint16_t* w, const float* bias, const uint16_t* latent,
                                  const uint16_t* rows, int T, int H, int L, int E, int K, int renormalize,
                                  float scale, float* logits, int32_t* ids, float* weights, uint16_t* weights_bf16,
                                  int32_t* offsets, int32_t* pairs, uint8_t* q, uint8_t* scales, uint16_t* out,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (T < 1 || K < 1 || !weights_bf16) return MOE_ERR_INVALID_ARGUMENT;
  const size_t rws = moe_router_logits_workspace(T, H, E);
  const size_t lws = moe_build_routing_lists_workspace(T, K, E);
  if (workspace_bytes < rws + lws || (rws + lws > 0 && !workspace)) return MOE_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int st = moe_router_logits(x, w, logits, T, H, E, ws, rws, stream);
  if (st != MOE_OK) return st;
  // the latent is an input of the step, complete before the router started: the
  // quantisation CTAs run beside the router instead of after it
  st = moe::route_quantize(logits, bias, T, E, K, renormalize, scale, ids, weights, weights_bf16, latent, T, L, q,
                           scales, true, moe::as_cuda(stream));
  if (st != MOE_OK) return st;
  st = moe_build_routing_lists(ids, T, K, E, offsets, pairs, lws ? ws + rws : nullptr, lws, stream);
  if (st != MOE_OK) return st;
  // Finalize reads only the step's rows and top-K's weights, both complete once the lists
  // kernel has passed its own wait (it signals its dependents only then): Finalize runs
  // beside the lists instead of after them.
  return moe::finalize(rows, (int64_t)T * K, nullptr, weights_bf16, MOE_DTYPE_BF16, nullptr, 1.0f, T, K, L, out, true,
                       moe::as_cuda(stream));
}
