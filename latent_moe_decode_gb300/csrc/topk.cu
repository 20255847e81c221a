// Sigmoid + e_score_correction_bias top-K with renormalised weights.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer,
// EpMoeLayer.topk (one group, sigmoid scoring, correction bias, renormalize, scale);
// vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideRoute docstring
// ("exact top16 and renormalized weights") and WideScratch (ids int32, weights BF16).
//
// Selection key c_e = sigmoid(logit_e) + bias_e; order (c descending, expert index
// ascending); weights are the unbiased scores over their slot-order FP32 sum.
//
// GB300 design: one warp per token. Lane l holds the experts 128 j + 4 l + m (j < NJ,
// m < 4), loaded as float4, so every load instruction of the warp reads 512
// contiguous bytes. Selection does not run K serial argmax rounds: the K-th largest
// of the 32 lane maxima (found with a 15-step bitonic network over shuffles) is a
// lower bound of the K-th largest key, because K different lanes hold a key at least
// that large. The few candidates at or above that bound are compacted into shared
// memory and ranked by counting (key greater, or equal with a lower index); the
// candidate of rank k takes slot k. When more than 64 candidates pass the bound
// (heavy ties) the warp falls back to K rounds of warp argmax (redux.sync).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kListCap = 64;
constexpr unsigned kFull = 0xFFFFFFFFu;

// --- the specified sigmoid -------------------------------------------------------
// exp(y) = 2^n exp(r), n = rint(y log2 e), r = y - n ln2 with ln2 split into a high
// part whose low 12 significand bits are zero (so n * LN2_HI is exact) and a low part
// (Cody & Waite, 1980); exp(r) by the degree-7 Taylor polynomial in Horner form with
// fused multiply-adds; 2^n applied as two exact power-of-two products.
constexpr double kLn2 = 0.693147180559945309417232121458;
constexpr float kLog2e = (float)(1.0 / kLn2);
constexpr float kLn2Hi = 0.693115234375f;  // (float)ln2 = 0x3F317218 with the low 12 bits cleared
constexpr float kLn2Lo = (float)(kLn2 - 0.693115234375);
constexpr float kC0 = 1.0f, kC1 = 1.0f, kC2 = (float)(1.0 / 2.0), kC3 = (float)(1.0 / 6.0),
                kC4 = (float)(1.0 / 24.0), kC5 = (float)(1.0 / 120.0), kC6 = (float)(1.0 / 720.0),
                kC7 = (float)(1.0 / 5040.0);

__device__ __forceinline__ float round_half_even(float x) {
  float r;
  asm("cvt.rni.f32.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float spec_exp(float y) {  // -17.5 < y < 88.5
  const float n = round_half_even(__fmul_rn(y, kLog2e));
  float r = __fmaf_rn(-n, kLn2Hi, y);
  r = __fmaf_rn(-n, kLn2Lo, r);
  float p = kC7;
  p = __fmaf_rn(p, r, kC6);
  p = __fmaf_rn(p, r, kC5);
  p = __fmaf_rn(p, r, kC4);
  p = __fmaf_rn(p, r, kC3);
  p = __fmaf_rn(p, r, kC2);
  p = __fmaf_rn(p, r, kC1);
  p = __fmaf_rn(p, r, kC0);
  const int ni = (int)n;
  const int a = ni / 2, b = ni - a;
  p = __fmul_rn(p, __int_as_float((a + 127) << 23));
  p = __fmul_rn(p, __int_as_float((b + 127) << 23));
  return p;
}

// sigma(x) = 1 / (1 + exp(-x)), correctly rounded reciprocal; 1 for x >= 17.5,
// 0 for x <= -88.5, NaN for NaN.
__device__ __forceinline__ float spec_sigmoid(float x) {
  if (x != x) return x;
  if (x >= 17.5f) return 1.0f;
  if (x <= -88.5f) return 0.0f;
  const float e = spec_exp(-x);
  return __frcp_rn(__fadd_rn(1.0f, e));
}

// Monotone 32-bit key of an FP32 value: larger value -> larger key, -0 == +0,
// NaN -> 1 (below every number); 0 is reserved for "no candidate".
__device__ __forceinline__ uint32_t order_key(float c) {
  if (c != c) return 1u;
  uint32_t b = __float_as_uint(c);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct TopkArgs {
  const float* logits;
  const float* bias;
  int T, E, K, renorm;
  float scale;
  int32_t* ids;
  float* weights;
  uint16_t* weights_bf16;
  int vec;  // logits rows and bias may be read as float4
};

struct WarpSmem {
  uint32_t key[kListCap];
  int32_t e[kListCap];
  float s[kListCap];
  int32_t slot_id[MOE_MAX_TOPK];
  float slot_s[MOE_MAX_TOPK];
};

template <int NJ>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) topk_kernel(const TopkArgs a) {
  __shared__ WarpSmem smem_all[kWarpsPerBlock];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int t = blockIdx.x * kWarpsPerBlock + wib;
  WarpSmem& sm = smem_all[wib];
  grid_launch_dependents();
  grid_wait();
  if (t >= a.T) return;
  const int E = a.E, K = a.K;
  const float* lg = a.logits + (size_t)t * E;

  // 1) scores and keys of this lane's candidates
  uint32_t key[NJ * 4];
  float s[NJ * 4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e0 = 128 * j + 4 * lane;
    float x[4], b[4] = {0.f, 0.f, 0.f, 0.f};
    if (a.vec && e0 < E) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(lg + e0));
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
      if (a.bias) {
        const float4 bb = __ldg(reinterpret_cast<const float4*>(a.bias + e0));
        b[0] = bb.x; b[1] = bb.y; b[2] = bb.z; b[3] = bb.w;
      }
    } else {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        x[m] = (e0 + m < E) ? __ldg(lg + e0 + m) : 0.f;
        if (a.bias && e0 + m < E) b[m] = __ldg(a.bias + e0 + m);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int i = 4 * j + m;
      const float sv = spec_sigmoid(x[m]);
      const float c = a.bias ? __fadd_rn(sv, b[m]) : sv;
      s[i] = sv;
      key[i] = (e0 + m < E) ? order_key(c) : 0u;
    }
  }

  // 2) bound: the K-th largest lane maximum
  uint32_t lmax = 0;
#pragma unroll
  for (int i = 0; i < NJ * 4; ++i) lmax = max(lmax, key[i]);
  uint32_t v = lmax;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, v, j);
      const bool ascending = (lane & k) == 0;
      const bool keep_min = ((lane & j) == 0) == ascending;
      v = keep_min ? min(v, o) : max(v, o);
    }
  }
  const uint32_t bound = __shfl_sync(kFull, v, 32 - K);  // ascending: K-th largest

  // 3) candidates at or above the bound
  uint32_t flags = 0;
#pragma unroll
  for (int i = 0; i < NJ * 4; ++i)
    if (key[i] != 0u && key[i] >= bound) flags |= 1u << i;
  const int mine = __popc(flags);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(kFull, incl, 31);

  if (total <= kListCap) {
    int pos = incl - mine;
#pragma unroll
    for (int i = 0; i < NJ * 4; ++i) {
      if (flags & (1u << i)) {
        sm.key[pos] = key[i];
        sm.e[pos] = 128 * (i >> 2) + 4 * lane + (i & 3);
        sm.s[pos] = s[i];
        ++pos;
      }
    }
    __syncwarp();
    for (int item = lane; item < total; item += 32) {
      const uint32_t ki = sm.key[item];
      const int ei = sm.e[item];
      int rank = 0;
      for (int q = 0; q < total; ++q) {
        const uint32_t kq = sm.key[q];
        rank += (kq > ki) || (kq == ki && sm.e[q] < ei);
      }
      if (rank < K) {
        sm.slot_id[rank] = ei;
        sm.slot_s[rank] = sm.s[item];
      }
    }
  } else {
    // heavy ties: K rounds of warp argmax over (key desc, expert asc)
    for (int k = 0; k < K; ++k) {
      uint32_t bk = 0;
      int be = 0x7FFFFFFF;
      float bs = 0.f;
#pragma unroll
      for (int i = 0; i < NJ * 4; ++i) {
        if (key[i] > bk) {  // ascending expert order within the lane: first max wins
          bk = key[i];
          be = 128 * (i >> 2) + 4 * lane + (i & 3);
          bs = s[i];
        }
      }
      const uint32_t wk = __reduce_max_sync(kFull, bk);
      const int we = (int)__reduce_min_sync(kFull, bk == wk ? (uint32_t)be : 0x7FFFFFFFu);
      const float ws = __shfl_sync(kFull, bs, (we & 127) >> 2);
      if (lane == 0) {
        sm.slot_id[k] = we;
        sm.slot_s[k] = ws;
      }
#pragma unroll
      for (int i = 0; i < NJ * 4; ++i)
        if (128 * (i >> 2) + 4 * lane + (i & 3) == we) key[i] = 0u;
    }
  }
  __syncwarp();

  // 4) weights: unbiased scores over their slot-order FP32 sum
  float S = 0.f;
  for (int k = 0; k < K; ++k) S = __fadd_rn(S, sm.slot_s[k]);
  if (lane < K) {
    const float sv = sm.slot_s[lane];
    float w = a.renorm ? (S == 0.f ? 0.f : __fdiv_rn(sv, S)) : sv;
    if (a.scale != 1.0f) w = __fmul_rn(w, a.scale);
    const size_t o = (size_t)t * K + lane;
    a.ids[o] = sm.slot_id[lane];
    if (a.weights) a.weights[o] = w;
    if (a.weights_bf16) a.weights_bf16[o] = f32_to_bf16(w);
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_topk_route(const float* logits, const float* bias, int T, int E, int K,
                              int renormalize, float scale, int32_t* ids, float* weights,
                              uint16_t* weights_bf16, moe_stream_t stream) {
  using namespace moe;
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
  const int vec = (E % 4 == 0) && aligned(logits, 16) && (!bias || aligned(bias, 16));
  TopkArgs a{logits, bias, T, E, K, renormalize ? 1 : 0, scale, ids, weights, weights_bf16, vec};
  dim3 grid((T + kWarpsPerBlock - 1) / kWarpsPerBlock), block(kWarpsPerBlock * 32);
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
