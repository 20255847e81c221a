// MXFP8 (OCP Microscaling) quantisation of BF16 rows.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide (module
// docstring: "MXFP8 activations"; WideRoute: a token's MXFP8 plan row is written from
// its BF16 latent) and ...moe.ep.layer (module docstring: "the MXFP8 latent"). The
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
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kThreads) mxfp8_kernel(const uint16_t* __restrict__ x, long long nchunks,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ scales,
                                                         uint32_t* err) {
  __shared__ __align__(128) uint4 stage[kThreads * kUnroll];
  __shared__ __align__(8) uint64_t bar_mem;
  const int lane = threadIdx.x & 31;
  const long long cta0 = (long long)blockIdx.x * kThreads * kUnroll;  // first chunk of this CTA
  const int nch = (int)min((long long)kThreads * kUnroll, nchunks - cta0);
  const uint32_t bar = smem_u32(&bar_mem);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  __syncthreads();  // the barrier is initialised before any thread waits on it
  grid_launch_dependents();
  grid_wait();
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar, (uint32_t)nch * 16u);
    bulk_g2s(smem_u32(stage), x + cta0 * 8, (uint32_t)nch * 16u, bar, policy_evict_first());
  }
  const bool ok = __all_sync(kFull, mbar_wait(bar, 0, err));
  if (!ok) return;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int wl = u * kThreads + (threadIdx.x & ~31);  // this warp's first chunk in the CTA
    if (wl >= nch) break;                                // warp-uniform
    const int cl = wl + lane;
    const uint4 v = cl < nch ? stage[cl] : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
    m = max(m, __shfl_xor_sync(kFull, m, 1));
    m = max(m, __shfl_xor_sync(kFull, m, 2));
    uint32_t sbyte;
    uint2 codes;
    if (m >= 0x7F80u) {  // an infinity or NaN in the block
      sbyte = 0xFFu;
      codes = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
    } else {
      int se = -127;
      if (m != 0u) {
        const int ex = (int)(m >> 7);
        const int fl = ex ? ex - 127 : (31 - __clz((int)(m & 0x7Fu))) - 133;
        se = min(max(fl - 8, -127), 127);
      }
      sbyte = (uint32_t)(se + 127);
      const float mult = __int_as_float((127 - se) << 23);  // 2^-se, a normal FP32
      uint32_t p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = e4m3x2(__fmul_rn(bf16_lo(w[j]), mult), __fmul_rn(bf16_hi(w[j]), mult));
      codes = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
    }
    const long long c = cta0 + cl;
    if (cl < nch) *reinterpret_cast<uint2*>(q + c * 8) = codes;
    // scale bytes of the warp's 8 blocks (held by lanes 0, 4, ..., 28)
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = __shfl_sync(kFull, sbyte, 4 * i);
    const long long blk0 = (cta0 + wl) >> 2;
    if (lane == 0) {
      if (wl + 32 <= nch) {
        *reinterpret_cast<uint2*>(scales + blk0) =
            make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
      } else {
        const int nb = (nch - wl) >> 2;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < nb) scales[blk0 + i] = (uint8_t)b[i];
      }
    }
  }
}

}  // namespace
}  // namespace moe

extern "C" int mxfp8_quantize_rows(const uint16_t* x, int rows, int cols, uint8_t* q, uint8_t* scales,
                                   moe_stream_t stream) {
  using namespace moe;
  if (rows < 0 || cols < 32 || cols % 32 != 0) return MOE_ERR_INVALID_ARGUMENT;
  if (rows == 0) return MOE_OK;
  if (!x || !q || !scales) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(x, 16) || !aligned(q, 8) || !aligned(scales, 8)) return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const long long nchunks = (long long)rows * (cols / 8);
  const long long per = (long long)kThreads * kUnroll;
  const long long blocks = (nchunks + per - 1) / per;
  if (blocks > (1LL << 31) - 1) return MOE_ERR_CAPACITY;
  return launch_pdl(mxfp8_kernel, dim3((unsigned)blocks), dim3(kThreads), 0, as_cuda(stream), x, nchunks, q, scales,
                    dev.error_word);
}
