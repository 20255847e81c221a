// Sigmoid + bias top-K: the per-token selection shared by the top-K kernel and the
// fused top-K + MXFP8 launch.
#pragma once

#include "common.cuh"

namespace moe {
namespace topk_impl {


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
// 0 for x <= -88.5, NaN for NaN (special cases selected, not branched).
__device__ __forceinline__ float spec_sigmoid(float x) {
  const bool hi = x >= 17.5f, lo = x <= -88.5f;
  const float e = spec_exp((hi || lo) ? 0.0f : -x);
  const float r = __frcp_rn(__fadd_rn(1.0f, e));
  return hi ? 1.0f : (lo ? 0.0f : r);
}

// A fast sigmoid used only to find the candidates: 1 / (1 + 2^(-x log2 e)) with the
// hardware's approximate exp2 and reciprocal. Over all 2^32 inputs it differs from
// spec_sigmoid by at most 1.79e-7 (< 2^-22.4; measured exhaustively on the GPU and
// pinned by a test) and agrees on NaN.
constexpr float kApproxErr = 2.384185791e-7f;  // 2^-22: the bound the margin below assumes
__device__ __forceinline__ float approx_sigmoid(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(__fmul_rn(-x, kLog2e)));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.0f, e)));
  return r;
}

// Monotone 32-bit key of an FP32 value: larger value -> larger key, -0 == +0,
// NaN -> 1 (below every number); 0 is reserved for "no candidate".
__device__ __forceinline__ uint32_t order_key(float c) {
  if (c != c) return 1u;
  uint32_t b = __float_as_uint(c);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// The FP32 value of an order key (the inverse of order_key for keys >= 2).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

struct TopkArgs {
  const float* logits;
  const float* bias;
  int T, E, K, renorm;
  float scale;
  int32_t* ids;
  float* weights;
  uint16_t* weights_bf16;
  // Optional: the router's split-K partials [S][T][E] instead of logits. Each token's
  // logits are then their sum in split order (as the router's own reduction), written
  // to logits_out; the partial lines read are invalidated in L2 when discard is set.
  const float* part = nullptr;
  int S = 0;
  float* logits_out = nullptr;
  int discard = 0;
};

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;

// One token's selection, run by a CTA of kThreads threads. PART: the logits are summed
// from the router's split-K partials (a.part) and written (a.logits_out); a separate
// instantiation, so the plain selection keeps its register count (and occupancy).
template <int NJ, bool PART = false>
__device__ __forceinline__ void topk_token(const TopkArgs& a, const int t) {
  __shared__ uint32_t s_top[kWarps][32];
  __shared__ int s_cnt[kWarps];
  __shared__ uint32_t l_key[kListCap];
  __shared__ int32_t l_e[kListCap];
  __shared__ float l_s[kListCap];
  __shared__ int32_t slot_id[MOE_MAX_TOPK];
  __shared__ float slot_s[MOE_MAX_TOPK];
  __shared__ uint32_t r_key[kWarps];
  __shared__ int32_t r_e[kWarps];
  __shared__ float r_s[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E, K = a.K;
  grid_launch_dependents();
  grid_wait();
  const float* lg = a.logits + (size_t)t * E;

  // 1) approximate keys of this thread's experts tid + 128 j
  uint32_t key[NJ];
  float x[NJ], b[NJ];
  if constexpr (PART) {
    // the logits: the S partials summed in split order, 4 splits' loads in flight at once
    constexpr int kSG = 4;
    for (int s0 = 0; s0 < a.S; s0 += kSG) {
      float p[kSG][NJ];
#pragma unroll
      for (int i = 0; i < kSG; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int e = tid + 128 * j;
          p[i][j] = (s0 + i < a.S && e < E) ? __ldcg(a.part + ((size_t)(s0 + i) * a.T + t) * E + e) : 0.f;
        }
#pragma unroll
      for (int i = 0; i < kSG; ++i)
        if (s0 + i < a.S)
#pragma unroll
          for (int j = 0; j < NJ; ++j) x[j] = s0 + i == 0 ? p[i][j] : __fadd_rn(x[j], p[i][j]);
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = tid + 128 * j;
      if (e < E) a.logits_out[(size_t)t * E + e] = x[j];
    }
    __syncwarp();  // every lane's loads are consumed before their lines are invalidated
    if (a.discard) {  // whole 128-byte lines of this warp's experts (E % 32 == 0, aligned)
      for (int l = lane; l < a.S * NJ; l += 32) {
        const int s = l / NJ, j = l - s * NJ;
        const int e0 = 32 * warp + 128 * j;
        if (e0 < E)
          asm volatile("discard.global.L2 [%0], 128;" ::"l"(a.part + ((size_t)s * a.T + t) * E + e0) : "memory");
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = tid + 128 * j;
      x[j] = e < E ? __ldg(lg + e) : 0.f;
    }
  }
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = tid + 128 * j;
    b[j] = (a.bias && e < E) ? __ldg(a.bias + e) : 0.f;
  }
  uint32_t tmax = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = tid + 128 * j;
    const float sv = approx_sigmoid(x[j]);
    const float c = a.bias ? __fadd_rn(sv, b[j]) : sv;
    key[j] = e < E ? order_key(c) : 0u;
    tmax = max(tmax, key[j]);
  }

  // 2) bound: the K-th largest of the 128 thread maxima
  uint32_t v = tmax;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, v, j);
      const bool descending = (lane & k) == 0;
      const bool keep_max = ((lane & j) == 0) == descending;
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  s_top[warp][lane] = v;  // descending: lane l holds the warp's (l+1)-th largest
  __syncthreads();
  // top 32 of the union of two descending lists: max(a[l], b[31-l]) is bitonic;
  // five half-cleaner steps sort it descending
  auto merge = [&](uint32_t x, uint32_t y) {
    uint32_t m = max(x, y);
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, m, j);
      m = (lane & j) == 0 ? max(m, o) : min(m, o);
    }
    return m;
  };
  const uint32_t m01 = merge(s_top[0][lane], s_top[1][31 - lane]);
  const uint32_t m23 = merge(s_top[2][lane], s_top[3][31 - lane]);
  const uint32_t top = merge(m01, __shfl_sync(kFull, m23, 31 - lane));
  const uint32_t bound = __shfl_sync(kFull, top, K - 1);
  // K experts (one in each of K threads) have an approximate key >= bound, so the exact
  // K-th largest key is >= bound - err, and every exact top-K expert has an approximate
  // key >= bound - 2 err, err = |approximate - exact key| <= 2^-22 + a few ulps of the
  // key. The margin 2^-19 (1 + |bound|) covers that; a bound that is not a finite
  // number takes every expert.
  uint32_t thr = 1u;
  if (bound >= 2u) {
    const float f = key_value(bound);
    const float g = __fsub_rn(f, 0x1p-19f * (1.0f + fabsf(f)));
    if (isfinite(g)) thr = order_key(g);
  }

  // 3) candidates at or above the threshold, compacted in thread order
  uint32_t flags = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (key[j] != 0u && key[j] >= thr) flags |= 1u << j;
  const int mine = __popc(flags);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_cnt[warp] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    before += w < warp ? s_cnt[w] : 0;
    total += s_cnt[w];
  }

  // exact key and score of candidate expert e (logit xv, bias bv)
  auto exact = [&](float xv, float bv, float* sc) {
    const float sv = spec_sigmoid(xv);
    *sc = sv;
    return order_key(a.bias ? __fadd_rn(sv, bv) : sv);
  };
  if (total <= 32) {
    // compact, then one warp computes the exact keys and sorts (key desc, expert asc):
    // lane k holds slot k
    int pos = before + incl - mine;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (flags & (1u << j)) {
        l_e[pos] = tid + 128 * j;
        l_s[pos] = x[j];
        l_key[pos] = __float_as_uint(b[j]);
        ++pos;
      }
    }
    __syncthreads();
    if (warp != 0) return;
    unsigned long long c = 0;  // (key << 32) | ~expert; 0 = empty
    float cs = 0.f;
    if (lane < total) {
      const uint32_t k = exact(l_s[lane], __uint_as_float(l_key[lane]), &cs);
      c = ((unsigned long long)k << 32) | (0xFFFFFFFFu - (uint32_t)l_e[lane]);
    }
    // slot of each candidate = how many candidates order before it (keys distinct with the
    // expert in the low word): 32 independent comparisons instead of a sorting network
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) rank += __shfl_sync(kFull, c, j) > c;
    if (lane < total && rank < K) {
      slot_id[rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)(c & 0xFFFFFFFFull));
      slot_s[rank] = cs;
    }
    __syncwarp();
    // weights: unbiased scores over their slot-order FP32 sum (all loads first, then the
    // sum in order)
    float sc[MOE_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k) sc[k] = k < K ? slot_s[k] : 0.f;
    float S = 0.f;
#pragma unroll
    for (int k = 0; k < MOE_MAX_TOPK; ++k)
      if (k < K) S = __fadd_rn(S, sc[k]);
    if (lane < K) {
      const float sv = slot_s[lane];
      float w = a.renorm ? (S == 0.f ? 0.f : __fdiv_rn(sv, S)) : sv;
      if (a.scale != 1.0f) w = __fmul_rn(w, a.scale);
      const size_t o = (size_t)t * K + lane;
      a.ids[o] = slot_id[lane];
      if (a.weights) a.weights[o] = w;
      if (a.weights_bf16) a.weights_bf16[o] = f32_to_bf16(w);
    }
    return;
  }
  if (total <= kListCap) {
    int pos = before + incl - mine;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (flags & (1u << j)) {
        float sc;
        l_key[pos] = exact(x[j], b[j], &sc);
        l_e[pos] = tid + 128 * j;
        l_s[pos] = sc;
        ++pos;
      }
    }
    __syncthreads();
    if (tid < total) {
      const uint32_t ki = l_key[tid];
      const int ei = l_e[tid];
      int rank = 0;
      for (int q = 0; q < total; ++q) {
        const uint32_t kq = l_key[q];
        rank += (kq > ki) || (kq == ki && l_e[q] < ei);
      }
      if (rank < K) {
        slot_id[rank] = ei;
        slot_s[rank] = l_s[tid];
      }
    }
  } else {
    // heavy ties: exact keys of all experts, then K rounds of argmax over (key desc,
    // expert asc)
    float s[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const uint32_t kx = exact(x[j], b[j], &s[j]);
      key[j] = tid + 128 * j < E ? kx : 0u;
    }
    for (int k = 0; k < K; ++k) {
      uint32_t bk = 0;
      int be = 0x7FFFFFFF;
      float bs = 0.f;
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        if (key[j] > bk) {  // ascending expert order within the thread: first max wins
          bk = key[j];
          be = tid + 128 * j;
          bs = s[j];
        }
      }
      const uint32_t wk = __reduce_max_sync(kFull, bk);
      const int we = (int)__reduce_min_sync(kFull, bk == wk ? (uint32_t)be : 0x7FFFFFFFu);
      const float ws = __shfl_sync(kFull, bs, we & 31);  // expert e lives in thread e % 128
      if (lane == 0) {
        r_key[warp] = wk;
        r_e[warp] = we;
        r_s[warp] = ws;
      }
      __syncthreads();
      uint32_t gk = 0;
      int ge = 0x7FFFFFFF;
      float gs = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (r_key[w] > gk || (r_key[w] == gk && r_e[w] < ge)) {
          gk = r_key[w];
          ge = r_e[w];
          gs = r_s[w];
        }
      }
      if (tid == 0) {
        slot_id[k] = ge;
        slot_s[k] = gs;
      }
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (tid + 128 * j == ge) key[j] = 0u;
      __syncthreads();
    }
  }
  __syncthreads();

  // 4) weights: unbiased scores over their slot-order FP32 sum
  if (tid < K) {
    float S = 0.f;
    for (int k = 0; k < K; ++k) S = __fadd_rn(S, slot_s[k]);
    const float sv = slot_s[tid];
    float w = a.renorm ? (S == 0.f ? 0.f : __fdiv_rn(sv, S)) : sv;
    if (a.scale != 1.0f) w = __fmul_rn(w, a.scale);
    const size_t o = (size_t)t * K + tid;
    a.ids[o] = slot_id[tid];
    if (a.weights) a.weights[o] = w;
    if (a.weights_bf16) a.weights_bf16[o] = f32_to_bf16(w);
  }
}

}  // namespace topk_impl
}  // namespace moe
