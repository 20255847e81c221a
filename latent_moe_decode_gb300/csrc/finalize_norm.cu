// Finalize with the RMSNorm epilogue: the routed latent of a token (the weighted
// top-K sum of its expert rows, rounded once to BF16) and its RMS-normalised copy.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer,
// EpMoeLayer.forward / stock_order (routed = the experts' weighted sum, then
// rms_norm(normed, routed, w["norm"], eps = 1e-5) before the up projection), and
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, module docstring
// and WideMoE.tail (the latent all-reduce with the RMSNorm fused; on one GPU there is
// no all-reduce and the norm becomes Finalize's epilogue). The routed sum follows the
// wide page's Finalize (FP32 fma over k in order, one BF16 rounding) with the options
// of the GLM finalize page's kernel (gathered rows, -1 skipped, BF16 or FP32 weights
// times routed_scaling_factor).
//
// Per token t, with x[c] the BF16 routed value as FP32:
//   ss = sum_c x[c]^2           (FP32; each thread's 8 columns in order, then a
//                                fixed shuffle tree over the warp and over the warps)
//   r  = rsqrt_rn(ss / H + eps) (correctly rounded divide, add and reciprocal root)
//   out[t, c] = bf16_rn((x[c] * r) * g[c])
//
// GB300 design: one CTA per token, H/8 threads, each owning one 16-byte fragment (8
// columns) of every row, as the wide page's Finalize. A thread copies all its row
// fragments of a chunk of up to KC rows (cp.async, L1 bypassed, L2 evict-first) into
// its own shared-memory slots before it waits and sums them, so a CTA keeps up to
// 112 KB in flight; at H = 3584, K = 16 that is the whole token and two CTAs fit on an
// SM, so one CTA's loads are in flight while the other reduces and stores (for more
// tokens than one wave of that, three CTAs per SM with chunks of ten rows). Slots are
// private to their thread; the CTA meets at two barriers: after its weights and row
// indices are staged, and in the sum of squares.
#include "common.cuh"
#include <type_traits>

namespace moe {
namespace {

constexpr int kMaxThreads = 1024;                  // H <= 8192
// Row staging per CTA: two CTAs per SM ((228 KB - 2 x 1 KB reserved) / 2, less static:
// a token's 16 rows of 3584 in one chunk) while the tokens fit in one wave of them,
// else three per SM (ten rows a chunk; the last wave of CTAs less empty: measured at
// T = 1020 24.1 against 26.8 us, at T = 4096 79.3 against 85.5 us; at T = 256 the two-CTA
// form is faster, 8.1 against 9.4 us)
constexpr uint32_t kSlotBytes2 = 115712 - 512;
constexpr uint32_t kSlotBytes3 = 76544;

struct NormArgs {
  const uint16_t* rows;
  long long n_rows;
  const int32_t* row_index;  // [T, K] or nullptr
  const void* weights;       // [T, K] FP32 or BF16
  float scale;
  const uint16_t* gamma;     // [H]
  float eps;
  int T, K, H, KC;
  uint16_t* routed;          // [T, H] or nullptr
  uint16_t* out;             // [T, H]
  uint32_t* err;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}

template <bool GATHER, bool BF16W>
__global__ void __launch_bounds__(kMaxThreads) finalize_norm_kernel(const NormArgs a) {
  extern __shared__ __align__(16) uint4 slots[];  // [KC][H/8]
  __shared__ float warp_ss[32];
  __shared__ float w_sm[MOE_MAX_TOPK];    // the token's weights, times routed_scaling_factor
  __shared__ int32_t r_sm[MOE_MAX_TOPK];  // its row indices (-1: skipped)
  const int t = blockIdx.x, tid = threadIdx.x, nthr = blockDim.x;
  const int col = tid * 8;
  const size_t H = (size_t)a.H;
  grid_launch_dependents();
  grid_wait();  // rows, weights and indices may come from the preceding kernel
  const uint64_t pol = policy_evict_first();
  const uint32_t base = smem_u32(slots) + (uint32_t)tid * 16u;
  using WRaw = typename std::conditional<BF16W, uint16_t, float>::type;
  if (tid < a.K) {  // one load per weight and index for the whole CTA
    const size_t ix = (size_t)t * a.K + tid;
    long long r = GATHER ? (long long)__ldg(a.row_index + ix) : (long long)ix;
    if (GATHER && (r < -1 || r >= a.n_rows)) {
      set_error(a.err, MOE_DEVERR_ROW_INDEX);
      r = -1;
    }
    float w;
    if constexpr (BF16W) w = bf16_to_f32(__ldg(static_cast<const WRaw*>(a.weights) + ix));
    else w = __ldg(static_cast<const WRaw*>(a.weights) + ix);
    if (a.scale != 1.0f) w = __fmul_rn(w, a.scale);
    w_sm[tid] = w;
    r_sm[tid] = (int32_t)r;
  }
  __syncthreads();

  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
  for (int k0 = 0; k0 < a.K; k0 += a.KC) {
    const int kc = a.K - k0 < a.KC ? a.K - k0 : a.KC;
    for (int j = 0; j < kc; ++j) {
      const int r = r_sm[k0 + j];
      if (r != -1) cp_async16(base + (uint32_t)(j * nthr * 16), a.rows + (size_t)r * H + col, pol);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    for (int j = 0; j < kc; ++j) {
      if (r_sm[k0 + j] == -1) continue;  // a -1 row: its term is skipped
      const float w = w_sm[k0 + j];
      const uint4 v = slots[(size_t)j * nthr + tid];
      const uint32_t q4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __fmaf_rn(w, bf16_lo(q4[q]), acc[2 * q]);
        acc[2 * q + 1] = __fmaf_rn(w, bf16_hi(q4[q]), acc[2 * q + 1]);
      }
    }
  }
  // the routed latent: one BF16 rounding
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  if (a.routed) st16(a.routed + (size_t)t * H + col, o);
  const uint32_t p4[4] = {o.x, o.y, o.z, o.w};
  float x[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[2 * q] = bf16_lo(p4[q]);
    x[2 * q + 1] = bf16_hi(p4[q]);
  }
  // sum of squares: this thread's columns in order, then the warp, then the warps
  float ss = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) ss = __fmaf_rn(x[q], x[q], ss);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xFFFFFFFFu, ss, d));
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
  if (lane == 0) warp_ss[warp] = ss;
  __syncthreads();
  float tot = lane < nwarps ? warp_ss[lane] : 0.0f;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) tot = __fadd_rn(tot, __shfl_xor_sync(0xFFFFFFFFu, tot, d));
  const float r = __frsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)a.H), a.eps));
  const uint4 g = *reinterpret_cast<const uint4*>(a.gamma + col);
  const uint32_t g4[4] = {g.x, g.y, g.z, g.w};
  float y[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    y[2 * q] = __fmul_rn(__fmul_rn(x[2 * q], r), bf16_lo(g4[q]));
    y[2 * q + 1] = __fmul_rn(__fmul_rn(x[2 * q + 1], r), bf16_hi(g4[q]));
  }
  uint4 n;
  n.x = pack_bf16x2(y[0], y[1]);
  n.y = pack_bf16x2(y[2], y[3]);
  n.z = pack_bf16x2(y[4], y[5]);
  n.w = pack_bf16x2(y[6], y[7]);
  st16(a.out + (size_t)t * H + col, n);
}

template <bool G, bool B>
int launch(const NormArgs& a, cudaStream_t s) {
  auto kern = finalize_norm_kernel<G, B>;
  const size_t smem = (size_t)a.KC * (a.H / 8) * 16;
  // (the limit is the largest staging any call uses, the same for every call: calls from
  // several host threads never lower it under one another)
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSlotBytes2) != cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_pdl(kern, dim3((unsigned)a.T), dim3((unsigned)(a.H / 8)), smem, s, a);
}

}  // namespace
}  // namespace moe

extern "C" int moe_finalize_rmsnorm(const uint16_t* rows, int64_t n_rows, const int32_t* row_index,
                                    const void* weights, int weights_dtype, float routed_scaling_factor,
                                    const uint16_t* norm_weight, float eps, int T, int K, int H, uint16_t* routed,
                                    uint16_t* out, moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || K < 1 || K > MOE_MAX_TOPK || H < 256 || H % 256 != 0 || n_rows < 0 || !(eps >= 0.0f))
    return MOE_ERR_INVALID_ARGUMENT;
  if (weights_dtype != MOE_DTYPE_F32 && weights_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARGUMENT;
  if (H > 8 * kMaxThreads || T > 0x7FFFFFFF) return MOE_ERR_CAPACITY;
  if (T == 0) return MOE_OK;
  if (!rows || !weights || !norm_weight || !out) return MOE_ERR_INVALID_ARGUMENT;
  if (!row_index && n_rows < (long long)T * K) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(rows, 16) || !aligned(out, 16) || !aligned(norm_weight, 16) || (routed && !aligned(routed, 16)))
    return MOE_ERR_ALIGNMENT;
  if (!aligned(weights, weights_dtype == MOE_DTYPE_F32 ? 4 : 2) || (row_index && !aligned(row_index, 4)))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const int row_bytes = (H / 8) * 16;
  const uint32_t slot_bytes = (long long)T > 2LL * dev.sm_count ? kSlotBytes3 : kSlotBytes2;
  int KC = (int)(slot_bytes / (uint32_t)row_bytes);
  KC = KC < 1 ? 1 : (KC > K ? K : KC);
  NormArgs a{rows, (long long)n_rows, row_index, weights, routed_scaling_factor, norm_weight, eps, T, K, H, KC,
             routed, out, dev.error_word};
  cudaStream_t s = as_cuda(stream);
  const bool g = row_index != nullptr, b = weights_dtype == MOE_DTYPE_BF16;
  if (g) return b ? launch<true, true>(a, s) : launch<true, false>(a, s);
  return b ? launch<false, true>(a, s) : launch<false, false>(a, s);
}
