// MXFP8 (OCP MX) quantisation of a flat BF16 span: the per-CTA body shared by the
// quantisation kernel and the fused top-K + MXFP8 launch.
#pragma once

#include "common.cuh"

namespace moe {
namespace mxfp8_impl {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Byte offset of scale (row r, scale column c) in the tcgen05 block-scaling layout:
// 128 x 4 tiles of 512 bytes in row-tile-major order (ct column tiles per row tile);
// inside a tile, 32 lines of 16 bytes, line l holding rows l, l + 32, l + 64, l + 96.
__device__ __forceinline__ size_t tcgen05_scale_offset(int r, int c, int ct) {
  return ((size_t)(r >> 7) * ct + (size_t)(c >> 2)) * 512 + 16 * (r & 31) + 4 * ((r >> 5) & 3) + (c & 3);
}

// One warp's 32 consecutive chunks [c0, c0 + 32) of the flat input (c0 a multiple of
// 32; lane l holds chunk c0 + l, its 16 bytes in v; chunks at or past nchunks are
// neither read nor stored): the E4M3 codes, and the 8 blocks' scale bytes. CEIL: the
// round-up scale rule (the smallest power of two X with amax / X <= 448) instead of the
// OCP floor rule. TILED: scales in the tcgen05 tile layout (nsc scale columns per row,
// ct column tiles) instead of row-major.
template <bool CEIL, bool TILED>
__device__ __forceinline__ void convert_warp(uint4 v, long long c0, long long nchunks, uint8_t* __restrict__ q,
                                             uint8_t* __restrict__ scales, int nsc, int ct) {
  const int lane = threadIdx.x & 31;
  const long long c = c0 + lane;
  const bool valid = c < nchunks;
  if (!valid) v = make_uint4(0, 0, 0, 0);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  m = max(m, __shfl_xor_sync(kFullMask, m, 1));
  m = max(m, __shfl_xor_sync(kFullMask, m, 2));
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
      int up = 0;  // amax / 2^fl > 1.75 (448 = 1.75 * 2^8): one step up keeps amax / X <= 448
      if (CEIL) {
        const uint32_t man = ex ? (m & 0x7Fu) | 0x80u : (m & 0x7Fu);  // amax = man * 2^(fl - msb)
        const int msb = ex ? 7 : 31 - __clz((int)man);
        up = 4u * man > (7u << msb) ? 1 : 0;
      }
      se = min(max(fl - 8 + up, -127), 127);
    }
    sbyte = (uint32_t)(se + 127);
    const float mult = __int_as_float((127 - se) << 23);  // 2^-se, a normal FP32
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) p[j] = e4m3x2(__fmul_rn(bf16_lo(w[j]), mult), __fmul_rn(bf16_hi(w[j]), mult));
    codes = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
  }
  if (valid) *reinterpret_cast<uint2*>(q + c * 8) = codes;
  if constexpr (TILED) {
    // the first lane of each block writes its scale byte at its tile position
    if ((lane & 3) == 0 && valid) {
      const long long blk = c >> 2;  // = row * nsc + scale column
      const int r = (int)(blk / nsc);
      scales[tcgen05_scale_offset(r, (int)(blk - (long long)r * nsc), ct)] = (uint8_t)sbyte;
    }
  } else {
    // scale bytes of the warp's 8 blocks (held by lanes 0, 4, ..., 28)
    uint32_t b[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) b[i] = __shfl_sync(kFullMask, sbyte, 4 * i);
    const long long blk0 = c0 >> 2;
    if (lane == 0) {
      if (c0 + 32 <= nchunks) {
        *reinterpret_cast<uint2*>(scales + blk0) = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                                                              b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
      } else {
        const int nb = (int)((nchunks - c0) >> 2);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < nb) scales[blk0 + i] = (uint8_t)b[i];
      }
    }
  }
}

// One CTA's 16-byte chunks [block * THREADS * UNROLL, ...) of the flat input. With
// wait = false the CTA does not wait for the preceding kernel (the caller knows the
// input was complete before that kernel started).
template <int THREADS, int UNROLL, bool CEIL = false, bool TILED = false>
__device__ __forceinline__ void mxfp8_block(const uint16_t* __restrict__ x, long long nchunks, uint8_t* __restrict__ q,
                                            uint8_t* __restrict__ scales, uint32_t* err, long long block,
                                            bool wait = true, int nsc = 0, int ct = 0) {
  constexpr int kThreads = THREADS, kUnroll = UNROLL;
  __shared__ __align__(128) uint4 stage[kThreads * kUnroll];
  __shared__ __align__(8) uint64_t bar_mem;
  const int lane = threadIdx.x & 31;
  const long long cta0 = block * kThreads * kUnroll;  // first chunk of this CTA
  const int nch = (int)min((long long)kThreads * kUnroll, nchunks - cta0);
  const uint32_t bar = smem_u32(&bar_mem);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_fence_init();
  }
  __syncthreads();  // the barrier is initialised before any thread waits on it
  grid_launch_dependents();
  if (wait) {
    // the span's DRAM fetch overlaps the preceding kernel's end (a hint only)
    if (threadIdx.x == 0) prefetch_l2(x + cta0 * 8, (uint32_t)nch * 16u);
    grid_wait();
  }
  if (threadIdx.x == 0) {
    mbar_expect_tx(bar, (uint32_t)nch * 16u);
    bulk_g2s(smem_u32(stage), x + cta0 * 8, (uint32_t)nch * 16u, bar, policy_evict_first());
  }
  const bool ok = __all_sync(kFullMask, mbar_wait(bar, 0, err));
  if (!ok) return;
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int wl = u * kThreads + (threadIdx.x & ~31);  // this warp's first chunk in the CTA
    if (wl >= nch) break;                                // warp-uniform
    const uint4 v = wl + lane < nch ? stage[wl + lane] : make_uint4(0, 0, 0, 0);
    convert_warp<CEIL, TILED>(v, cta0 + wl, nchunks, q, scales, nsc, ct);
  }
}

// The padding bytes of the tcgen05 scale layout (rows past `rows` up to the row
// tile, scale columns past nsc up to the column tile) set to 0, by every thread of
// the grid in turn.
__device__ __forceinline__ void tcgen05_scale_padding(uint8_t* __restrict__ scales, int rows, int nsc, int ct) {
  const int cw = 4 * ct, rt_rows = (rows + 127) / 128 * 128;
  const long long colpad = (long long)rows * (cw - nsc);
  const long long total = colpad + (long long)(rt_rows - rows) * cw;
  for (long long p = (long long)blockIdx.x * blockDim.x + threadIdx.x; p < total; p += (long long)gridDim.x * blockDim.x) {
    int r, c;
    if (p < colpad) {
      r = (int)(p / (cw - nsc));
      c = nsc + (int)(p - (long long)r * (cw - nsc));
    } else {
      const long long q2 = p - colpad;
      r = rows + (int)(q2 / cw);
      c = (int)(q2 - (long long)(r - rows) * cw);
    }
    scales[tcgen05_scale_offset(r, c, ct)] = 0;
  }
}

}  // namespace mxfp8_impl
}  // namespace moe
