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
// bytes as one 8-byte store. The input is one contiguous span: CTAs of 512 threads
// (up to three per SM) take contiguous runs of 16 KB stages and keep four bulk (TMA)
// copies in flight on mbarriers; threads read their chunks from shared memory
// (consecutive lanes, consecutive 16 bytes: conflict-free). (Small CTAs of one 16 KB
// span each left a few SMs with more of a call's CTAs than others -- back-to-back calls
// place them while earlier calls' still run -- and measured 5.9-6.1 us a call at
// T = 1020; the 64 KB of stages per CTA caps every SM at three.)
#include "mxfp8.cuh"

namespace moe {
namespace {

constexpr int kThreads = 512;
constexpr int kStageChunks = 1024;  // 16 KB of input per stage (a multiple of 32 chunks)
constexpr int kStages = 4;          // 64 KB of stages per CTA

// Up to three CTAs per SM (their stages' shared memory admits no more): CTA b takes a
// contiguous run of whole stages of the input, keeps up to kStages bulk copies of it in
// flight on mbarriers, converts each stage as it lands (512 threads, two warp groups of
// 32 chunks per warp) and refills the buffer. (Measured back to back: one CTA per SM
// 5.0 us a call at T = 1020 and 14.4 at 4096, two 6.5 / 12.0, three 4.1 / 11.4.)
// Before its wait the CTA asks L2 for its whole run (a hint), so the DRAM fetch
// overlaps the preceding kernel's end.
template <bool CEIL, bool TILED>
__global__ void __launch_bounds__(kThreads) mxfp8_kernel(const uint16_t* __restrict__ x, long long nchunks,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                                                         uint32_t* err, int rows, int nsc, int ct) {
  extern __shared__ __align__(128) uint4 stage[];  // [kStages][kStageChunks]
  __shared__ __align__(8) uint64_t bar_mem[kStages];
  const int lane = threadIdx.x & 31;
  const long long nst = (nchunks + kStageChunks - 1) / kStageChunks;
  const long long s0 = (long long)blockIdx.x * nst / gridDim.x, s1 = ((long long)blockIdx.x + 1) * nst / gridDim.x;
  const int n = (int)(s1 - s0);  // this CTA's stages
  auto bar = [&](int b) { return smem_u32(&bar_mem[b]); };
  auto span = [&](int i) { return (int)min((long long)kStageChunks, nchunks - (s0 + i) * kStageChunks); };
  if (threadIdx.x == 0) {
    for (int b = 0; b < kStages; ++b) mbar_init(bar(b), 1);
    mbar_fence_init();
  }
  __syncthreads();  // the barriers are initialised before any thread waits on them
  grid_launch_dependents();
  if (threadIdx.x == 0 && n > 0)  // (its first kStages stages)
    prefetch_l2(x + s0 * kStageChunks * 8,
                (uint32_t)((min(min(s1, s0 + kStages) * kStageChunks, nchunks) - s0 * kStageChunks) * 16));
  grid_wait();
  const uint64_t pol = policy_evict_first();
  auto issue = [&](int i) {
    const int b = i % kStages;
    mbar_expect_tx(bar(b), (uint32_t)span(i) * 16u);
    bulk_g2s(smem_u32(stage + (size_t)b * kStageChunks), x + (s0 + i) * kStageChunks * 8, (uint32_t)span(i) * 16u,
             bar(b), pol);
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < n && i < kStages; ++i) issue(i);
  for (int i = 0; i < n; ++i) {
    const int b = i % kStages;
    if (!__syncthreads_and(mbar_wait(bar(b), (uint32_t)(i / kStages) & 1u, err))) {
      // (a stage never landed: error set; the copies still in flight are waited for,
      // each with the same bound, before the CTA leaves)
      for (int j = i + 1; j < n && j < i + kStages; ++j) mbar_wait(bar(j % kStages), (uint32_t)(j / kStages) & 1u, err);
      break;
    }
    const long long c0 = (s0 + i) * kStageChunks;
    const int nch = span(i);
#pragma unroll
    for (int u = 0; u < kStageChunks / kThreads; ++u) {
      const int wl = u * kThreads + (threadIdx.x & ~31);  // this warp's first chunk in the stage
      if (wl >= nch) break;                                // warp-uniform
      const uint4 v = wl + lane < nch ? stage[(size_t)b * kStageChunks + wl + lane] : make_uint4(0, 0, 0, 0);
      mxfp8_impl::convert_warp<CEIL, TILED>(v, c0 + wl, nchunks, q, scales, nsc, ct);
    }
    __syncthreads();  // every thread is done with buffer b
    if (threadIdx.x == 0 && i + kStages < n) issue(i + kStages);
  }
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
  const long long nst = (nchunks + kStageChunks - 1) / kStageChunks;
  const long long blocks = nst < 3LL * dev.sm_count ? nst : 3LL * dev.sm_count;
  const int nsc = cols / 32, ct = (nsc + 3) / 4;
  const bool ceil = scale_rule == MXFP8_SCALE_CEIL;
  auto kern = tiled ? (ceil ? mxfp8_kernel<true, true> : mxfp8_kernel<false, true>)
                    : (ceil ? mxfp8_kernel<true, false> : mxfp8_kernel<false, false>);
  constexpr size_t smem = (size_t)kStages * kStageChunks * 16;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_pdl(kern, dim3((unsigned)blocks), dim3(kThreads), smem, stream, x, nchunks, q, scales, dev.error_word,
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
