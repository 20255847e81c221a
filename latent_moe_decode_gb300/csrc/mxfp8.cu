// MXFP8 (OCP Microscaling) quantisation of BF16 rows.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide (module
// docstring: MXFP8 activations; WideRoute: a token's MXFP8 plan row is written from
// its BF16 latent) and ...moe.ep.layer (module docstring: the latent in MXFP8). The
// pages fix no more than "MXFP8"; the OCP MX v1.0 reading is: per block of 32
// consecutive elements, scale exponent se = floor(log2 amax) - 8 (8 = emax of E4M3)
// clamped to [-127, 127] and stored as the E8M0 byte se + 127; elements E4M3(v / 2^se),
// round to nearest even, saturating to +-448.
//
// GB300 design: an HBM stream (2 bytes in, 1 + 1/32 bytes out per element). A thread
// owns a 16-byte chunk (8 elements), four consecutive lanes a 32-element block: the
// block maximum is two xor-shuffles away. amax is taken on the BF16 magnitude bits
// (their integer order is the value order), so floor(log2 amax) is read from the
// exponent field. v * 2^-se is one exact FP32 multiply (or underflows far below half
// the smallest E4M3 subnormal); cvt.rn.satfinite.e4m3x2.f32 rounds two at a time. A
// warp writes its 8 elements' bytes per lane (256 contiguous bytes) and its 8 scale
// bytes as one 8-byte store. The input is one contiguous span: each CTA stages its
// 16 KB piece with a single bulk (TMA) copy onto an mbarrier, so every CTA's whole
// input is in flight at once; threads then read their chunks from shared memory
// (consecutive lanes, consecutive 16 bytes: conflict-free).
#include "mxfp8.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

template <bool CEIL, bool TILED>
__global__ void __launch_bounds__(kThreads) mxfp8_kernel(const uint16_t* __restrict__ x, long long nchunks,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                                                         uint32_t* err, int rows, int nsc, int ct) {
  mxfp8_impl::mxfp8_block<kThreads, kUnroll, CEIL, TILED>(x, nchunks, q, scales, err, blockIdx.x, true, nsc, ct);
  if (TILED) mxfp8_impl::tcgen05_scale_padding(scales, rows, nsc, ct);
}

int quantize(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales, int scale_rule, bool tiled,
             cudaStream_t stream) {
  if (rows < 0 || cols < 32 || cols % 32 != 0) return MOE_ERR_INVALID_ARGUMENT;
  if (scale_rule != MXFP8_SCALE_FLOOR && scale_rule != MXFP8_SCALE_CEIL) return MOE_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !scales) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(scales, tiled ? 16 : 8)) return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const long long nchunks = (long long)rows * (cols / 8);
  const long long per = (long long)kThreads * kUnroll;
  const long long blocks = (nchunks + per - 1) / per;
  if (blocks > (1LL << 31) - 1) return MOE_ERR_CAPACITY;
  const int nsc = cols / 32, ct = (nsc + 3) / 4;
  const bool ceil = scale_rule == MXFP8_SCALE_CEIL;
  auto kern = tiled ? (ceil ? mxfp8_kernel<true, true> : mxfp8_kernel<false, true>)
                    : (ceil ? mxfp8_kernel<true, false> : mxfp8_kernel<false, false>);
  return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), 0, stream, x, nchunks, q, scales, dev.error_word,
                    rows, nsc, ct);
}

}  // namespace
}  // namespace moe


extern "C" int mxfp8_quantize_rows_ex(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales,
                                      int scale_rule, moe_stream_t stream) {
  return moe::quantize(x, rows, cols, q, scales, scale_rule, false, moe::as_cuda(stream));
}

extern "C" int mxfp8_quantize_rows(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales,
                                   moe_stream_t stream) {
  return mxfp8_quantize_rows_ex(x, rows, cols, q, scales, MXFP8_SCALE_FLOOR, stream);
}

extern "C" size_t mxfp8_tcgen05_scales_bytes(int rows, int cols) {
  if (rows < 0 || cols < 32 || cols % 32 != 0) return 0;
  return (size_t)((rows + 127) / 128) * (size_t)((cols / 32 + 3) / 4) * 512;
}

extern "C" int mxfp8_quantize_rows_tcgen05(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales,
                                           int scale_rule, moe_stream_t stream) {
  return moe::quantize(x, rows, cols, q, scales, scale_rule, true, moe::as_cuda(stream));
}
