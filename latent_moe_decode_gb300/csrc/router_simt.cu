// Router logits on the CUDA cores (small token counts) and the split-K reduce.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer,
// EpMoeLayer (the FP32-output split-K router projection of the [896, 7168] BF16 gate:
// split 4 for up to 32 tokens, 64-row weight tiles, split-K partials reduced in FP32) and
// EpMoeLayer.stock_order (mm(x, gate^T) with an FP32 output).
//
// GB300 design: at a handful of tokens the router is one pass over the 12.8 MB weight,
// HBM-bound on the CUDA cores. A CTA of 8 warps owns 16 experts (2 per warp) x 16
// tokens x one K chunk; the chunk of the 16 hidden rows is staged in shared memory and
// every lane streams 16-byte weight fragments (a warp reads 512 contiguous bytes of an
// expert row per load). A lane accumulates <= 128 products per output in FP32, then the
// 32 lane partials of the warp's 32 outputs are combined by a transposing butterfly
// (31 shuffles), after which lane l holds output l. Split-K partials go to the
// workspace and a second kernel sums them in split order (deterministic).
// For at most 8 tokens the GEMV form below takes over: no split-K and no second kernel.
#include "router.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xFFFFFFFFu;

__global__ void __launch_bounds__(kThreads) router_simt_kernel(const uint16_t* __restrict__ x,
                                                               const uint16_t* __restrict__ w, float* __restrict__ out,
                                                               int T, int H, int E, int kc) {
  extern __shared__ uint4 xs[];  // [16 tokens][kc / 8]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.y * 16;
  const int e0 = blockIdx.x * 16 + 2 * warp;
  const int s = blockIdx.z;
  const int kb = s * kc;
  const int len8 = (min(H, kb + kc) - kb) / 8;
  const int row8 = kc / 8;
  grid_wait();
  grid_launch_dependents();  // after the wait: dependents may rely on all before the router
  for (int i = threadIdx.x; i < 16 * len8; i += kThreads) {
    const int tt = i / len8, kk = i - tt * len8;
    xs[tt * row8 + kk] = (t0 + tt < T) ? ld_nc16(x + (size_t)(t0 + tt) * H + kb + kk * 8) : make_uint4(0, 0, 0, 0);
  }
  __syncthreads();

  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.f;
  const uint16_t* wa = w + (size_t)min(e0, E - 1) * H + kb;
  const uint16_t* wb = w + (size_t)min(e0 + 1, E - 1) * H + kb;
  for (int kk = lane; kk < len8; kk += 32) {
    const uint4 va = ld_nc16(wa + kk * 8), vb = ld_nc16(wb + kk * 8);
    const uint32_t a4[4] = {va.x, va.y, va.z, va.w}, b4[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      const uint4 xv = xs[tt * row8 + kk];
      const uint32_t x4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[tt] = __fmaf_rn(bf16_lo(a4[j]), bf16_lo(x4[j]), acc[tt]);
        acc[tt] = __fmaf_rn(bf16_hi(a4[j]), bf16_hi(x4[j]), acc[tt]);
        acc[16 + tt] = __fmaf_rn(bf16_lo(b4[j]), bf16_lo(x4[j]), acc[16 + tt]);
        acc[16 + tt] = __fmaf_rn(bf16_hi(b4[j]), bf16_hi(x4[j]), acc[16 + tt]);
      }
    }
  }
  // transposing butterfly: afterwards lane l holds the warp total of output l
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? acc[i] : acc[i + off];
      const float keep = upper ? acc[i + off] : acc[i];
      acc[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
    }
  }
  const int e = e0 + (lane >> 4), t = t0 + (lane & 15);
  if (e < E && t < T) out[((size_t)s * T + t) * E + e] = acc[0];
}

// GEMV form for T <= 8 tokens (TT: the tokens rounded up to 1, 2, 3, 4 or 8): the 12.8 MB
// gate is one HBM stream and the tokens' rows are small, so no K is split and no
// partials leave the CTA. A CTA of kGemvWarps warps owns kGemvRows expert rows over the
// whole hidden dimension; the 16-byte fragments f of a row are dealt to warps in runs
// of 32 (warp (f / 32) % kGemvWarps, lane f % 32), so every load instruction of a warp
// reads 512 contiguous bytes of a gate row. A lane accumulates its products (at most
// H / 224 fragments x 8 = 32 at H = 7168) per output in FP32 in hidden order, each
// warp's 32 lane sums are combined by a fixed shuffle tree, and the warps' sums in warp
// order: deterministic. The CTA first asks L2 to prefetch its gate rows (weights may be
// read before the wait for the preceding kernel only as a prefetch) so the stream
// starts while the preceding kernel finishes.
constexpr int kGemvWarps = 7;
// Expert rows per CTA and CTAs per SM, by the rounded token count (measured back to back
// over cold inputs at E = 896, H = 7168): 3 rows, two CTAs per SM, at 1, 2 and 3 tokens
// (3.6 / 4.1 / 5.0 us; 2 rows and three per SM: 4.0 / 4.7 / 5.3-5.6); 2 rows, three per SM,
// at 4 (5.3 us; 3 rows: 6.0); 6 rows, one CTA per SM, at 8. The tokens' rows are re-read from L2 by
// every CTA, so fewer, wider CTAs read them fewer times, until too few CTAs are resident
// to keep the gate's stream in flight.
template <int TT>
constexpr int gemv_rows() { return TT == 8 ? 6 : (TT == 4 ? 2 : 3); }
template <int TT>
constexpr int gemv_ctas_per_sm() { return TT == 8 ? 1 : (TT == 4 ? 3 : 2); }

template <int TT, int kGemvRows = gemv_rows<TT>()>
__global__ void __launch_bounds__(kGemvWarps * 32, gemv_ctas_per_sm<TT>()) router_gemv_kernel(const uint16_t* __restrict__ x,
                                                                      const uint16_t* __restrict__ w,
                                                                      float* __restrict__ out, int T, int H, int E) {
  __shared__ float red[kGemvWarps][kGemvRows * TT];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e0 = blockIdx.x * kGemvRows;
  const int F = H / 8;                                           // 16-byte fragments per row
  const int NI = (F + 32 * kGemvWarps - 1) / (32 * kGemvWarps);  // fragments per lane
  const uint16_t* wr[kGemvRows];
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r) wr[r] = w + (size_t)min(e0 + r, E - 1) * H;
  for (int i = 0; i < NI; ++i) {
    const int f = lane + 32 * (warp + kGemvWarps * i);
    if (f < F)
#pragma unroll
      for (int r = 0; r < kGemvRows; ++r) asm volatile("prefetch.global.L2 [%0];" ::"l"(wr[r] + f * 8));
  }
  grid_launch_dependents();
  grid_wait();
  float acc[kGemvRows][TT];
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
    for (int t = 0; t < TT; ++t) acc[r][t] = 0.f;
  // NU fragments per lane at a time: all their loads first (addresses clamped into the
  // row, contributions past the row dropped), then the products in hidden order
  constexpr int NU = TT <= 4 ? 4 : 2;
  for (int i0 = 0; i0 < NI; i0 += NU) {
    uint4 wv[NU][kGemvRows], xv[NU][TT];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int f = min(lane + 32 * (warp + kGemvWarps * (i0 + u)), F - 1);
#pragma unroll
      for (int r = 0; r < kGemvRows; ++r) wv[u][r] = ld_nc16(wr[r] + f * 8);
#pragma unroll
      for (int t = 0; t < TT; ++t) xv[u][t] = ld_nc16(x + (size_t)min(t, T - 1) * H + f * 8);
    }
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int f = lane + 32 * (warp + kGemvWarps * (i0 + u));
      if (i0 + u >= NI || f >= F) continue;
#pragma unroll
      for (int r = 0; r < kGemvRows; ++r) {
        const uint32_t a4[4] = {wv[u][r].x, wv[u][r].y, wv[u][r].z, wv[u][r].w};
#pragma unroll
        for (int t = 0; t < TT; ++t) {
          const uint32_t b4[4] = {xv[u][t].x, xv[u][t].y, xv[u][t].z, xv[u][t].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[r][t] = __fmaf_rn(bf16_lo(a4[j]), bf16_lo(b4[j]), acc[r][t]);
            acc[r][t] = __fmaf_rn(bf16_hi(a4[j]), bf16_hi(b4[j]), acc[r][t]);
          }
        }
      }
    }
  }
  // the warp's sum of each output: a fixed xor tree over the lanes
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r)
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float v = acc[r][t];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
      if (lane == 0) red[warp][r * TT + t] = v;
    }
  __syncthreads();
  if (threadIdx.x < kGemvRows * TT) {
    const int r = threadIdx.x / TT, t = threadIdx.x - r * TT, e = e0 + r;
    float v = red[0][threadIdx.x];
#pragma unroll
    for (int q = 1; q < kGemvWarps; ++q) v = __fadd_rn(v, red[q][threadIdx.x]);
    if (t < T && e < E) out[(size_t)t * E + e] = v;
  }
}

__global__ void __launch_bounds__(256) router_reduce_kernel(const float* __restrict__ part, int S, long long n,
                                                            float* __restrict__ logits) {
  grid_wait();
  grid_launch_dependents();  // after the wait: dependents may rely on all before the router
  for (long long i = (long long)blockIdx.x * 256 + threadIdx.x; i < n; i += (long long)gridDim.x * 256) {
    float v = part[i];
    for (int s = 1; s < S; ++s) v = __fadd_rn(v, part[(size_t)s * n + i]);
    logits[i] = v;
  }
}

}  // namespace

// Splits of the SIMT path: per-lane chains of at most 128 products (kc <= 4096) and
// enough CTAs to cover the SMs twice.
void simt_plan(int T, int H, int E, int sm_count, int* S, int* kc) {
  const long long tiles = (long long)((E + 15) / 16) * ((T + 15) / 16);
  int s = (int)((2LL * sm_count + tiles - 1) / tiles);
  s = max(s, (H + 4095) / 4096);
  s = min(s, max(1, H / 256));
  int k = (H + s - 1) / s;
  k = (k + 255) / 256 * 256;
  *S = (H + k - 1) / k;
  *kc = k;
}

int launch_router_simt(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, int S, int kc,
                       float* part, cudaStream_t stream) {
  const size_t smem = (size_t)16 * kc * 2;
  // (the limit is the largest staging any plan uses -- kc <= 4096 -- the same for every
  // call: calls from several host threads never lower it under one another)
  if (kc > 4096) return MOE_ERR_INVALID_ARGUMENT;
  if (cudaFuncSetAttribute(router_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16 * 4096 * 2) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  dim3 grid((E + 15) / 16, (T + 15) / 16, S);
  int st = launch_pdl(router_simt_kernel, grid, dim3(kThreads), smem, stream, x, w, S == 1 ? logits : part, T, H, E, kc);
  if (st != MOE_OK || S == 1) return st;
  return launch_router_reduce(part, S, T, E, logits, stream);
}

template <int TT>
int launch_gemv(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, cudaStream_t stream) {
  const dim3 grid((E + gemv_rows<TT>() - 1) / gemv_rows<TT>()), block(kGemvWarps * 32);
  return launch_pdl(router_gemv_kernel<TT>, grid, block, 0, stream, x, w, logits, T, H, E);
}

int launch_router_gemv(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, cudaStream_t stream) {
  if (T <= 1) return launch_gemv<1>(x, w, logits, T, H, E, stream);
  if (T <= 2) return launch_gemv<2>(x, w, logits, T, H, E, stream);
  if (T <= 3) return launch_gemv<3>(x, w, logits, T, H, E, stream);
  if (T <= 4) return launch_gemv<4>(x, w, logits, T, H, E, stream);
  if (T <= kGemvMaxTokens) return launch_gemv<8>(x, w, logits, T, H, E, stream);
  return MOE_ERR_INVALID_ARGUMENT;
}

int launch_router_reduce(const float* part, int S, int T, int E, float* logits, cudaStream_t stream) {
  const long long n = (long long)T * E;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(router_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, part, S, n, logits);
}

}  // namespace moe
