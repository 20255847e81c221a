// Sigmoid + bias top-K and MXFP8 quantisation of the latent rows in one launch.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideRoute
// (the top-K CTAs and the latent-quantisation CTAs of a batch share one grid).
//
// GB300 design: the two jobs share nothing, so in one grid the quantisation CTAs
// stream the latent through HBM on the SMs the routing CTAs leave free, instead of
// running after them. The routing CTAs run the top-K selection (topk.cuh: four tokens
// per CTA, one per warp, at E <= 1024) and come first in the grid; Q CTAs each quantise
// a 16 KB span of the latent (mxfp8.cuh), one bulk copy per CTA. (With latent_ready the
// order is reversed and the quantisation CTAs skip the wait, to run beside a preceding
// kernel; the one-call step measured that slower: beside its router only the SMs the
// router leaves idle could take them, and they delayed the routing CTAs.) Both bodies are
// the ones the separate calls use, so the results are identical to moe_topk_route
// followed by mxfp8_quantize_rows.
#include "mxfp8.cuh"
#include "topk.cuh"

namespace moe {
namespace {

using namespace topk_impl;
constexpr int kQuantUnroll = 8;  // 128 threads x 8 chunks = 16 KB per quantisation CTA

template <int NJ, bool WARP, bool PART>
__global__ void __launch_bounds__(kThreads) route_quant_kernel(const TopkArgs a, const uint16_t* __restrict__ x,
                                                               long long nchunks, uint8_t* __restrict__ q,
                                                               uint8_t* __restrict__ scales, uint32_t* err, int qblocks,
                                                               int rblocks, int quant_wait) {
  // Blocks are dispatched in index order. When the quantisation CTAs need not wait they
  // come first and take the SMs that are free while the preceding kernel still runs;
  // otherwise the routing CTAs (the longer ones) come first.
  const int b = (int)blockIdx.x;
  if (quant_wait) {
    if (b < rblocks) route_block<NJ, WARP, PART>(a, b);
    else mxfp8_impl::mxfp8_block<kThreads, kQuantUnroll>(x, nchunks, q, scales, err, (long long)(b - rblocks), true);
  } else {
    if (b < qblocks) mxfp8_impl::mxfp8_block<kThreads, kQuantUnroll>(x, nchunks, q, scales, err, (long long)b, false);
    else route_block<NJ, WARP, PART>(a, b - qblocks);
  }
}

}  // namespace
}  // namespace moe

namespace moe {

bool route_uses_warp_body(int E, const float* logits, const float* bias, const float* part, int S) {
  using namespace topk_impl;
  // (with partials, the warp body also stores the logits as float4)
  return use_warp_body(E, part ? static_cast<const void*>(part) : logits, bias, part ? S : 0) &&
         (!part || aligned(logits, 16));
}

int route_quantize(const float* logits, const float* bias, int T, int E, int K, int renormalize, float scale,
                   int32_t* ids, float* weights, uint16_t* weights_bf16, const uint16_t* latent, int rows, int cols,
                   uint8_t* q, uint8_t* scales, bool latent_ready, cudaStream_t s, const float* part, int S,
                   uint32_t* smap, uint8_t* below) {
  using namespace moe::topk_impl;
  if (T < 1 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARGUMENT;
  if (E > MOE_MAX_EXPERTS || K > MOE_MAX_TOPK) return MOE_ERR_CAPACITY;
  if (rows < 0 || cols < 32 || cols % 32 != 0) return MOE_ERR_INVALID_ARGUMENT;
  if (!logits || !ids || (rows > 0 && (!latent || !q || !scales))) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(logits, 4) || (bias && !aligned(bias, 4)) || !aligned(ids, 4) || (weights && !aligned(weights, 4)) ||
      (weights_bf16 && !aligned(weights_bf16, 2)))
    return MOE_ERR_ALIGNMENT;
  if (rows > 0 && (!aligned(latent, 16) || !aligned(q, 8) || !aligned(scales, 8))) return MOE_ERR_ALIGNMENT;
  const long long nchunks = (long long)rows * (cols / 8);
  const long long per = (long long)kThreads * kQuantUnroll;
  const long long qblocks = (nchunks + per - 1) / per;
  // (with partials, the warp body also stores the logits as float4)
  const bool warp = route_uses_warp_body(E, logits, bias, part, S);
  if (smap && (!warp || !below || !aligned(below, 16))) return MOE_ERR_INVALID_ARGUMENT;
  const long long rblocks = route_blocks(T, warp);
  if (rblocks + qblocks > (1LL << 31) - 1) return MOE_ERR_CAPACITY;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  TopkArgs a{logits, bias, T, E, K, renormalize ? 1 : 0, scale, ids, weights, weights_bf16};
  if (part) {
    if (S < 1 || !aligned(part, 4)) return MOE_ERR_INVALID_ARGUMENT;
    a.part = part;
    a.S = S;
    a.logits_out = const_cast<float*>(logits);
    a.discard = (E % 32 == 0 && aligned(part, 128)) ? 1 : 0;
  }
  a.smap = smap;
  a.below = below;
  const dim3 grid((unsigned)(rblocks + qblocks)), block(kThreads);
  const int qb = (int)qblocks, rb = (int)rblocks, qw = latent_ready ? 0 : 1;
  // With partials and no more CTAs than SMs, an SM may hold at most two of them (unused
  // dynamic shared memory): placed as the router's CTAs leave, they otherwise gathered
  // on the SMs freed first (measured, the one-call step at T = 256: 22.9 against 23.5 us;
  // at T = 1020, 255 CTAs, the cap measured 0.3 us slower and is not taken). The limit
  // is that pad for every call, so that calls from several threads do not race on it.
  const bool capped = part && grid.x <= (unsigned)dev.sm_count;
#define MOE_RQ_LAUNCH(NJ, W)                                                                                      \
  if (part) {                                                                                                     \
    auto kern = route_quant_kernel<NJ, W, true>;                                                                  \
    const size_t most = cta_cap_pad(reinterpret_cast<const void*>(kern), dev.sm_count, dev);                      \
    if (most > 0 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) !=        \
                        cudaSuccess)                                                                              \
      return MOE_ERR_CUDA;                                                                                        \
    return launch_pdl(kern, grid, block, capped ? most : 0, s, a, latent, nchunks, q, scales, dev.error_word, qb, \
                      rb, qw);                                                                                    \
  }                                                                                                               \
  return launch_pdl(route_quant_kernel<NJ, W, false>, grid, block, 0, s, a, latent, nchunks, q, scales,           \
                    dev.error_word, qb, rb, qw);
  if (E > kWarpMaxE) {
    MOE_RQ_LAUNCH(32, false)
  }
  switch ((E + 127) / 128) {  // experts per thread (CTA body) or per lane / 4 (warp body)
#define MOE_RQ_CASE(N)          \
  case N:                       \
    if (warp) {                 \
      MOE_RQ_LAUNCH(N, true)    \
    } else {                    \
      MOE_RQ_LAUNCH(N, false)   \
    }
    MOE_RQ_CASE(1)
    MOE_RQ_CASE(2)
    MOE_RQ_CASE(3)
    MOE_RQ_CASE(4)
    MOE_RQ_CASE(5)
    MOE_RQ_CASE(6)
    MOE_RQ_CASE(7)
    MOE_RQ_CASE(8)
#undef MOE_RQ_CASE
  }
#undef MOE_RQ_LAUNCH
  return MOE_ERR_CAPACITY;
}

}  // namespace moe

extern "C" int moe_topk_route_quantize(const float* logits, const float* bias, int T, int E, int K, int renormalize,
                                       float scale, int32_t* ids, float* weights, uint16_t* weights_bf16,
                                       const uint16_t* latent, int rows, int cols, uint8_t* q, uint8_t* scales,
                                       moe_stream_t stream) {
  return moe::route_quantize(logits, bias, T, E, K, renormalize, scale, ids, weights, weights_bf16, latent, rows, cols,
                             q, scales, false, moe::as_cuda(stream));
}
