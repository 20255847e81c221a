// The routing-and-combine step as one call: three launches on the caller's stream --
// the router, whose epilogue warps quantise the latent to MXFP8 while its mainloop runs;
// top-K; Finalize with the routing lists. The later kernels use programmatic dependent
// launch and execute griddepcontrol.wait before they read anything an earlier kernel
// of the step wrote. Reads of the step's own inputs may come first: Finalize issues its
// first row copies before its wait (and reads top-K's weights only after it).
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideMoE.run
// (router -> route -> Finalize on one stream) and ...moe.ep.layer, EpMoeLayer.__call__.
#include "router.cuh"

namespace {
size_t align256(size_t n) { return (n + 255) / 256 * 256; }

// the router's partials [S][T][E] (or its cluster workspace, if larger)
size_t router_part_bytes(int T, int H, int E) {
  moe::DeviceInfo dev;
  if (T < 1 || H < 8 || E < 1 || moe::current_device(&dev) != MOE_OK) return 0;
  const size_t a = moe_router_logits_workspace(T, H, E), b = moe::router_partials_bytes(T, H, E, dev.sm_count);
  return align256(a > b ? a : b);
}

// the routing CTAs' slot map [ceil(E/32)][nb][32] words (nb = ceil(T/4) blocks of 4
// tokens) and its below counts [ceil(E/32)][nb rounded up to 16] bytes
size_t smap_bytes(int T, int E) { return align256((size_t)(E + 31) / 32 * ((T + 3) / 4) * 32 * 4); }
size_t map_bytes(int T, int E) {
  if (T < 1 || E < 1) return 0;
  return smap_bytes(T, E) + align256((size_t)(E + 31) / 32 * (((T + 3) / 4 + 15) / 16 * 16));
}
}  // namespace

extern "C" size_t moe_route_finalize_workspace(int T, int H, int E, int K) {
  return router_part_bytes(T, H, E) + map_bytes(T, E) + moe_build_routing_lists_workspace(T, K, E);
}

extern "C" int moe_route_finalize(const uint16_t* x, const uint16_t* w, const float* bias, const uint16_t* latent,
                                  const uint16_t* rows, int T, int H, int L, int E, int K, int renormalize,
                                  float scale, float* logits, int32_t* ids, float* weights, uint16_t* weights_bf16,
                                  int32_t* offsets, int32_t* pairs, uint8_t* q, uint8_t* scales, uint16_t* out,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  using namespace moe;
  if (T < 1 || K < 1 || !weights_bf16) return MOE_ERR_INVALID_ARGUMENT;
  if (E < 1 || H < 8 || H % 8 != 0 || (long long)T * E > (1LL << 40)) return MOE_ERR_INVALID_ARGUMENT;
  if (E > MOE_MAX_EXPERTS || K > MOE_MAX_TOPK || K > E) return K > E ? MOE_ERR_INVALID_ARGUMENT : MOE_ERR_CAPACITY;
  if (!x || !w || !logits || !ids || !offsets || !pairs || !rows || !out) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(logits, 4)) return MOE_ERR_ALIGNMENT;
  if (!aligned(rows, 16) || !aligned(out, 16) || !aligned(ids, 4) || !aligned(offsets, 4) || !aligned(pairs, 4))
    return MOE_ERR_ALIGNMENT;
  if (L < 32 || L % 32 != 0 || !latent || !q || !scales) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(latent, 16) || !aligned(q, 8) || !aligned(scales, 8) || (weights && !aligned(weights, 4)) ||
      !aligned(weights_bf16, 2) || (bias && !aligned(bias, 4)))
    return MOE_ERR_ALIGNMENT;
  const size_t rws = router_part_bytes(T, H, E), mws = map_bytes(T, E);
  const size_t lws = moe_build_routing_lists_workspace(T, K, E);
  if (workspace_bytes < rws + mws + lws || !workspace) return MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 16)) return MOE_ERR_WORKSPACE;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // The router stores its split-K partials and the top-K launch sums them (in split
  // order, as the router's own reduction would: the same logits, bit for bit), so the
  // router skips its on-chip exchange; with one split it writes the logits itself.
  // The router's epilogue warps, idle while its mainloop runs, also quantise the latent
  // (a step input) to MXFP8; the few-token GEMV router leaves that to the top-K launch.
  int S = 1;
  bool quantised = false;
  float* part = reinterpret_cast<float*>(ws);
  LatentQuant lq;
  lq.x = latent;
  lq.nchunks = (long long)T * (L / 8);
  lq.q = q;
  lq.scales = scales;
  st = launch_router_partials(x, w, logits, T, H, E, dev.sm_count, part, dev.error_word, as_cuda(stream), &S, &lq,
                              &quantised);
  if (st != MOE_OK) return st;
  // The routing CTAs come first in the grid and the quantisation CTAs after them (as in
  // the public call): measured, quantisation CTAs dispatched first to run beside the
  // router could only use the SMs it leaves idle and delayed the routing CTAs by 1.4 to
  // 2.8 us a step. The routing CTAs also write a slot map from which the Finalize launch
  // builds the routing lists in CTAs of its own, beside its row stream (Finalize does not
  // read the lists); where the warp-per-token body does not apply, the lists kernel runs
  // between the two.
  const float* pp = S > 1 ? part : nullptr;
  const bool map = route_uses_warp_body(E, logits, bias, pp, S) && finalize_lists_fit(T, K);
  uint32_t* smap = reinterpret_cast<uint32_t*>(ws + rws);
  uint8_t* below = ws + rws + smap_bytes(T, E);
  st = route_quantize(logits, bias, T, E, K, renormalize, scale, ids, weights, weights_bf16, latent, quantised ? 0 : T, L, q, scales,
                      false, as_cuda(stream), pp, S, map ? smap : nullptr, map ? below : nullptr);
  if (st != MOE_OK) return st;
  // Finalize starts its row copies (a step input) before its wait and reads top-K's
  // weights after it.
  if (map) return finalize_with_lists(rows, weights_bf16, T, K, L, out, smap, below, E, offsets, pairs, as_cuda(stream));
  st = moe_build_routing_lists(ids, T, K, E, offsets, pairs, lws ? ws + rws + mws : nullptr, lws, stream);
  if (st != MOE_OK) return st;
  return finalize(rows, (int64_t)T * K, nullptr, weights_bf16, MOE_DTYPE_BF16, nullptr, 1.0f, T, K, L, out, true,
                  as_cuda(stream));
}
