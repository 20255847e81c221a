// Sigmoid + bias top-K: the per-token selection shared by the top-K kernel and the
// fused top-K + MXFP8 launch. Two bodies: one warp per token for E <= 1024 (the decode
// shapes: 28 experts per lane at E = 896, no CTA barrier), and one CTA of 4 warps per
// token for 1024 < E <= 4096.
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

// A fast sigmoid used only to find the candidates: 1/2 + tanh(x/2)/2 with the
// hardware's approximate tanh (one MUFU operation). Over all 2^32 inputs it stays
// within kApproxErr of spec_sigmoid (measured exhaustively on the GPU and pinned by a
// test) and agrees on NaN.
constexpr float kApproxErr = 0x1p-11f;
__device__ __forceinline__ float approx_sigmoid(float x) {
  float th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(__fmul_rn(0.5f, x)));
  return __fmaf_rn(0.5f, th, 0.5f);
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
  // Optional (warp body): each 4-token routing CTA b also writes, for the routing lists
  // that the one-call step builds in its Finalize launch, the slot map (range-major:
  // word smap[r][b][j] for expert e = 32 r + j; byte i: the slot of e in token 4b + i,
  // 0xFF when that token did not pick e) and below[r][b] (its pairs with an expert
  // below 32 r; rows of ceil(nb / 16) * 16 bytes, nb = ceil(T / 4)).
  uint32_t* smap = nullptr;
  uint8_t* below = nullptr;
};

constexpr int kThreads = 128;  // both bodies: CTAs of 4 warps
constexpr int kWarps = kThreads / 32;
constexpr int kWarpMaxE = 1024;     // the warp body's experts (32 per lane at most)
constexpr int kMaxPartSplits = 8;  // split-K partials the warp body sums (wide token tiles split at most 8 ways)

// The logits of this thread's experts e = e_first + e_stride * j (j < NJ; a warp's 32
// lanes cover one 128-byte line per j). PART: the sum in split order of the router's S
// partials (two splits' loads in flight at a time), written to a.logits_out, and the
// lines read invalidated in L2 when a.discard is set (E % 32 == 0, aligned workspace).
template <int NJ, bool PART>
__device__ __forceinline__ void load_logits(const TopkArgs& a, int t, int e_first, int e_stride, float (&x)[NJ]) {
  const int E = a.E;
  if constexpr (PART) {
    for (int s0 = 0; s0 < a.S; s0 += 2) {
      const float* r0 = a.part + ((size_t)s0 * a.T + t) * E;
      const float* r1 = r0 + (size_t)a.T * E;
      const bool two = s0 + 1 < a.S;
      float p0[NJ], p1[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int e = e_first + e_stride * j;
        p0[j] = e < E ? __ldcg(r0 + e) : 0.f;
        p1[j] = (two && e < E) ? __ldcg(r1 + e) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        x[j] = s0 == 0 ? p0[j] : __fadd_rn(x[j], p0[j]);
        if (two) x[j] = __fadd_rn(x[j], p1[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = e_first + e_stride * j;
      if (e < E) a.logits_out[(size_t)t * E + e] = x[j];
    }
    __syncwarp();  // every lane's loads are consumed before their lines are invalidated
    if (a.discard) {
      const int lane = threadIdx.x & 31, w0 = e_first - lane;  // the warp's first expert
      for (int l = lane; l < a.S * NJ; l += 32) {
        const int s = l / NJ, j = l - s * NJ;
        const int e0 = w0 + e_stride * j;
        if (e0 < E)
          asm volatile("discard.global.L2 [%0], 128;" ::"l"(a.part + ((size_t)s * a.T + t) * E + e0) : "memory");
      }
    }
  } else {
    const float* lg = a.logits + (size_t)t * E;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = e_first + e_stride * j;
      x[j] = e < E ? __ldg(lg + e) : 0.f;
    }
  }
}

// Descending bitonic sort of one value per lane over the warp (shuffles): lane l ends
// with the (l+1)-th largest.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t v) {
  const int lane = threadIdx.x & 31;
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
  return v;
}

// Candidate threshold from a bound on approximate keys. K experts have an approximate
// key >= bound, so the exact K-th largest key is >= bound - err, and every exact
// top-K expert has an approximate key >= bound - 2 err, where err (|approximate -
// exact key|) is at most kApproxErr plus an ulp or two of the key. The margin
// 2 kApproxErr + 2^-21 (1 + |bound|) covers that; a bound that is not a finite number
// takes every expert.
__device__ __forceinline__ uint32_t candidate_threshold(uint32_t bound) {
  if (bound < 2u) return 1u;
  const float f = key_value(bound);
  const float g = __fsub_rn(f, 2.0f * kApproxErr + 0x1p-21f * (1.0f + fabsf(f)));
  return isfinite(g) ? order_key(g) : 1u;
}

// (exact key << 32) | ~expert: one integer order for "key descending, expert ascending".
__device__ __forceinline__ unsigned long long rank_key(uint32_t key, int e) {
  return ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

// The exact key and score of an expert with logit xv and bias bv.
__device__ __forceinline__ uint32_t exact_key(const TopkArgs& a, float xv, float bv, float* sc) {
  const float sv = spec_sigmoid(xv);
  *sc = sv;
  return order_key(a.bias ? __fadd_rn(sv, bv) : sv);
}

// Outputs of token t from its slots (slot order): by lanes 0..K-1 of one warp. The
// weights are the unbiased scores over their FP32 sum taken in slot order.
__device__ __forceinline__ void write_slots(const TopkArgs& a, int t, const int32_t* slot_id, const float* slot_s) {
  const int lane = threadIdx.x & 31;
  if (lane >= a.K) return;
  float S = 0.f;
  for (int k = 0; k < a.K; ++k) S = __fadd_rn(S, slot_s[k]);
  const float sv = slot_s[lane];
  float w = a.renorm ? (S == 0.f ? 0.f : __fdiv_rn(sv, S)) : sv;
  if (a.scale != 1.0f) w = __fmul_rn(w, a.scale);
  const size_t o = (size_t)t * a.K + lane;
  a.ids[o] = slot_id[lane];
  if (a.weights) a.weights[o] = w;
  if (a.weights_bf16) a.weights_bf16[o] = f32_to_bf16(w);
}

// ---------------------------------------------------------------------------------
// One warp per token (E <= kWarpMaxE, E % 4 == 0, 16-byte aligned rows). Lane l holds
// the experts 128 j + 4 l + i (j < NJ4, i < 4): one 16-byte load per j, so a load
// instruction of the warp reads 512 contiguous bytes of the logits row.
struct __align__(16) WarpScratch {  // (16: the logits row is stored as float4)
  float x[kWarpMaxE];  // the token's logits (exact keys of the candidates read them here)
  int32_t e[64];       // candidates (at most 64 take the ranking paths)
  int32_t slot_id[MOE_MAX_TOPK];
  float slot_s[MOE_MAX_TOPK];
};

// The token's logits in the float4 layout (PART: summed from the split-K partials in
// split order, two splits' loads in flight, written to a.logits_out, the lines read
// invalidated in L2 when a.discard is set).
template <int NJ4, bool PART>
__device__ __forceinline__ void load_logits4(const TopkArgs& a, int t, float4 (&x)[NJ4]) {
  const int lane = threadIdx.x & 31, E = a.E;
  if constexpr (PART) {
    // group j: every split's float4 loaded at once (up to kMaxPartSplits), then summed
    // in split order; the groups are independent, so several are in flight together
    const float* base = a.part + (size_t)t * E + 4 * lane;
    const size_t sstride = (size_t)a.T * E;
#pragma unroll
    for (int j = 0; j < NJ4; ++j) {
      const bool in = 128 * j + 4 * lane < E;
      float4 p[kMaxPartSplits];
#pragma unroll
      for (int q = 0; q < kMaxPartSplits; ++q)
        p[q] = (in && q < a.S) ? __ldcg(reinterpret_cast<const float4*>(base + q * sstride + 128 * j))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
      x[j] = p[0];
#pragma unroll
      for (int q = 1; q < kMaxPartSplits; ++q) {
        if (q < a.S) {
          x[j].x = __fadd_rn(x[j].x, p[q].x), x[j].y = __fadd_rn(x[j].y, p[q].y);
          x[j].z = __fadd_rn(x[j].z, p[q].z), x[j].w = __fadd_rn(x[j].w, p[q].w);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < NJ4; ++j) {
      const int e = 128 * j + 4 * lane;
      if (e < E) *reinterpret_cast<float4*>(a.logits_out + (size_t)t * E + e) = x[j];
    }
    __syncwarp();  // every lane's loads are consumed before their lines are invalidated
    if (a.discard) {  // the warp's 512 bytes per (split, j): four 128-byte lines
      for (int l = lane; l < a.S * NJ4 * 4; l += 32) {
        const int s = l / (NJ4 * 4), r = l - s * NJ4 * 4, e0 = 128 * (r >> 2) + 32 * (r & 3);
        if (e0 < E)
          asm volatile("discard.global.L2 [%0], 128;" ::"l"(a.part + ((size_t)s * a.T + t) * E + e0) : "memory");
      }
    }
  } else {
    const float* lg = a.logits + (size_t)t * E;
#pragma unroll
    for (int j = 0; j < NJ4; ++j) {
      const int e = 128 * j + 4 * lane;
      x[j] = e < E ? __ldg(reinterpret_cast<const float4*>(lg + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// The warp body's rare path -- heavy ties, NaN or infinite keys (fewer than K or more
// than 64 candidates, or no finite bound): exact keys of all experts (lane l: experts
// l + 32 i, from the logits row staged in shared memory), then K rounds of a warp argmax
// over (key descending, expert ascending). Out of line and not unrolled, so that its code
// does not crowd the instruction cache of the common path.
static __device__ __noinline__ void select_all_exact(const TopkArgs& a, const float* xrow, int32_t* slot_id, float* slot_s) {
  const int lane = threadIdx.x & 31, E = a.E, n = (E + 31) / 32;
  uint32_t key[kWarpMaxE / 32];
  float sc[kWarpMaxE / 32];
#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    const int e = 32 * i + lane;
    key[i] = e < E ? exact_key(a, xrow[e], a.bias ? __ldg(a.bias + e) : 0.f, &sc[i]) : 0u;
  }
#pragma unroll 1
  for (int k = 0; k < a.K; ++k) {
    uint32_t bk = 0;
    int bi = -1;
#pragma unroll 1
    for (int i = 0; i < n; ++i)
      if (key[i] > bk) {  // ascending expert order within the lane: the first maximum wins
        bk = key[i];
        bi = i;
      }
    const uint32_t wk = __reduce_max_sync(kFull, bk);
    const int we = (int)__reduce_min_sync(kFull, (bk == wk && bi >= 0) ? (uint32_t)(32 * bi + lane) : 0x7FFFFFFFu);
    const float wsv = __shfl_sync(kFull, bi >= 0 ? sc[bi] : 0.f, we & 31);  // expert e lives in lane e % 32
    if (lane == 0) {
      slot_id[k] = we;
      slot_s[k] = wsv;
    }
    if ((we & 31) == lane) key[we >> 5] = 0u;
  }
}

template <int NJ4, bool PART>
__device__ __forceinline__ void topk_token_warp(const TopkArgs& a, const int t, WarpScratch& ws) {
  static_assert(4 * NJ4 <= 32, "one flag bit per expert of a lane");
  constexpr int NJ = 4 * NJ4;
  const int lane = threadIdx.x & 31;
  const int E = a.E, K = a.K;
  float4 x4[NJ4], b4[NJ4];
  // the bias first: its loads overlap the logits' (with partials, the loads' write-back
  // and L2 invalidation would otherwise order it after them: measured 0.7 us a step at
  // T = 1020)
#pragma unroll
  for (int j = 0; j < NJ4; ++j) {
    const int e = 128 * j + 4 * lane;
    b4[j] = (a.bias && e < E) ? __ldg(reinterpret_cast<const float4*>(a.bias + e)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  load_logits4<NJ4, PART>(a, t, x4);
#pragma unroll
  for (int j = 0; j < NJ4; ++j) {
    const int e = 128 * j + 4 * lane;
    if (e < E) *reinterpret_cast<float4*>(&ws.x[e]) = x4[j];  // the row, for the candidates' exact keys
  }
  // 1) approximate keys as floats (NaN never a candidate); the lane maximum, as a tree
  //    (fmaxf ignores NaN; all NaN gives NaN, taken as -inf below)
  float c[NJ], mx[NJ];
#pragma unroll
  for (int j = 0; j < NJ4; ++j) {
    const float xs[4] = {x4[j].x, x4[j].y, x4[j].z, x4[j].w}, bs[4] = {b4[j].x, b4[j].y, b4[j].z, b4[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float sv = approx_sigmoid(xs[i]);
      c[4 * j + i] = 128 * j + 4 * lane < E ? (a.bias ? __fadd_rn(sv, bs[i]) : sv) : -INFINITY;
      mx[4 * j + i] = c[4 * j + i];
    }
  }
#pragma unroll
  for (int w = NJ; w > 1; w = (w + 1) / 2) {
#pragma unroll
    for (int i = 0; i < w / 2; ++i) mx[i] = fmaxf(mx[2 * i], mx[2 * i + 1]);
    if (w & 1) mx[w / 2] = mx[w - 1];
  }
  const float m = mx[0];
  // 2) bound: the K-th largest of the 32 lane maxima (-inf for a lane without a number).
  //    Each lane counts the maxima above its own and those at least its own (independent
  //    shuffles, no chain of dependent exchanges); a lane with fewer than K above and at
  //    least K at or above holds that value.
  const float v = m != m ? -INFINITY : m;
  int gt0 = 0, gt1 = 0, ge0 = 0, ge1 = 0;  // (two counters each: shorter add chains)
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float o0 = __shfl_sync(kFull, v, i), o1 = __shfl_sync(kFull, v, i + 1);
    gt0 += o0 > v;
    ge0 += o0 >= v;
    gt1 += o1 > v;
    ge1 += o1 >= v;
  }
  const unsigned holds = __ballot_sync(kFull, gt0 + gt1 < K && ge0 + ge1 >= K);
  const float B = __shfl_sync(kFull, v, __ffs(holds) - 1);
  // every exact top-K expert has an approximate key within 2 err of the bound (err =
  // kApproxErr plus an ulp or two of the key); a bound that is not a finite number
  // sends the token to the all-exact path
  const float thr = __fsub_rn(B, 2.0f * kApproxErr + 0x1p-21f * (1.0f + fabsf(B)));
  // 3) candidates: counted, and compacted in lane order (their expert ids)
  uint32_t flags = 0;
#pragma unroll
  for (int j = 0; j < NJ; ++j) flags |= (c[j] >= thr ? 1u : 0u) << j;
  const int mine = __popc(flags);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(kFull, incl, 31);
  if (isfinite(thr) && total >= K && total <= 64) {
    int pos = incl - mine;
    for (uint32_t f = flags; f != 0u; f &= f - 1u) {  // (a lane's few candidates, ascending)
      const int j = __ffs(f) - 1;
      ws.e[pos++] = 128 * (j >> 2) + 4 * lane + (j & 3);
    }
    __syncwarp();
    // 4) exact keys of the candidates (lane i: candidates i and i + 32); a candidate's
    //    slot is the number of candidates ordering before it (keys made distinct by the
    //    expert in the low word): independent comparisons over shuffles
    unsigned long long c0 = 0, c1 = 0;
    float s0 = 0.f, s1 = 0.f;
    if (lane < total) {
      const int e = ws.e[lane];
      c0 = rank_key(exact_key(a, ws.x[e], a.bias ? __ldg(a.bias + e) : 0.f, &s0), e);
    }
    if (lane + 32 < total) {
      const int e = ws.e[lane + 32];
      c1 = rank_key(exact_key(a, ws.x[e], a.bias ? __ldg(a.bias + e) : 0.f, &s1), e);
    }
    int r0 = 0, r1 = 0;
    if (total <= 32) {  // (lanes past `total` hold no candidate: key 0, ordering below all)
#pragma unroll 4
      for (int i = 0; i < total; ++i) r0 += __shfl_sync(kFull, c0, i) > c0;
    } else {
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        const unsigned long long o0 = __shfl_sync(kFull, c0, i), o1 = __shfl_sync(kFull, c1, i);
        r0 += (o0 > c0) + (o1 > c0);
        r1 += (o0 > c1) + (o1 > c1);
      }
    }
    if (lane < total && r0 < K) {
      ws.slot_id[r0] = (int32_t)(0xFFFFFFFFu - (uint32_t)c0);
      ws.slot_s[r0] = s0;
    }
    if (lane + 32 < total && r1 < K) {
      ws.slot_id[r1] = (int32_t)(0xFFFFFFFFu - (uint32_t)c1);
      ws.slot_s[r1] = s1;
    }
  } else {
    select_all_exact(a, ws.x, ws.slot_id, ws.slot_s);
  }
  __syncwarp();
  // 5) weights
  write_slots(a, t, ws.slot_id, ws.slot_s);
}

// ---------------------------------------------------------------------------------
// One CTA of kThreads threads per token (small batches, and any E <= 32 * kThreads).
// Thread i holds the experts i + 128 j. The bound is the K-th largest of the 128 thread maxima
// (each warp sorts its 32, two rounds of bitonic merges give the top 32 of all 128);
// up to 32 candidates are ranked by warp 0 over shuffles, up to 64 by counting over
// shared memory, more (heavy ties) by exact keys for all and K rounds of argmax.
template <int NJ, bool PART = false>
__device__ __forceinline__ void topk_token_cta(const TopkArgs& a, const int t) {
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

  // 1) approximate keys of this thread's experts tid + 128 j
  uint32_t key[NJ];
  float x[NJ], b[NJ];
  load_logits<NJ, PART>(a, t, tid, 128, x);
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
  s_top[warp][lane] = warp_sort_desc(tmax);  // descending: lane l holds the warp's (l+1)-th largest
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
  const uint32_t thr = candidate_threshold(__shfl_sync(kFull, top, K - 1));

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

  if (total <= 32) {
    // compact, then one warp computes the exact keys and ranks them
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
    unsigned long long c = 0;  // rank_key; 0 = empty
    float cs = 0.f;
    if (lane < total) c = rank_key(exact_key(a, l_s[lane], __uint_as_float(l_key[lane]), &cs), l_e[lane]);
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) rank += __shfl_sync(kFull, c, j) > c;
    if (lane < total && rank < K) {
      slot_id[rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)(c & 0xFFFFFFFFull));
      slot_s[rank] = cs;
    }
    __syncwarp();
    write_slots(a, t, slot_id, slot_s);
    return;
  }
  if (total <= kListCap) {
    int pos = before + incl - mine;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (flags & (1u << j)) {
        float sc;
        l_key[pos] = exact_key(a, x[j], b[j], &sc);
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
      const uint32_t kx = exact_key(a, x[j], b[j], &s[j]);
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
  if (warp == 0) write_slots(a, t, slot_id, slot_s);
}

// The routing part of a launch: CTA `blk` of the routing CTAs. Warp body (NJ = experts
// per lane / 4): its 4 warps take tokens 4 blk .. 4 blk + 3; CTA body (NJ = experts
// per thread): token blk. Waits for the preceding kernel (which writes the logits or
// partials) before reading.
template <int NJ, bool WARP, bool PART>
__device__ __forceinline__ void route_block(const TopkArgs& a, int blk) {
  __shared__ uint32_t s_map[WARP ? kWarpMaxE : 1];
  grid_launch_dependents();
  if (!PART && (a.E & 3) == 0) {
    // the logits rows' DRAM fetch overlaps the preceding kernel's end (a hint only)
    const int t = WARP ? blk * kWarps + (int)(threadIdx.x >> 5) : blk;
    if ((threadIdx.x & (WARP ? 31 : 127)) == 0 && t < a.T && aligned(a.logits, 16))
      prefetch_l2(a.logits + (size_t)t * a.E, (uint32_t)a.E * 4u);
  }
  if (WARP && a.smap)  // cleared before the wait (experts past E up to the range end stay absent)
    for (int i = threadIdx.x; i < (a.E + 31) / 32 * 32; i += kThreads) s_map[i] = 0xFFFFFFFFu;
  grid_wait();
  if constexpr (WARP) {
    __shared__ WarpScratch ws[kWarps];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = blk * kWarps + warp;
    if (t < a.T) topk_token_warp<NJ, PART>(a, t, ws[warp]);
    if (a.smap) {
      __syncthreads();  // the map is cleared and every token's slots are known
      // byte `warp` of expert e's word: this token's slot of e (a token's experts are
      // distinct, so every byte has one writer)
      if (t < a.T && lane < a.K) reinterpret_cast<uint8_t*>(s_map)[4 * ws[warp].slot_id[lane] + warp] = (uint8_t)lane;
      __syncthreads();
      const int nr = (a.E + 31) / 32, nb = (a.T + 3) / 4, nbp = (nb + 15) / 16 * 16;
      if (warp == 0) {
        // this block's pairs below each range (nr <= 32 here: E <= kWarpMaxE): a scan of
        // the per-range counts (slot bytes are below 0x80, absent ones 0xFF)
        // (lane l reads word 32 i + l of range i: conflict-free; a warp sum per range)
        int c = 0;
        for (int i = 0; i < nr; ++i) {
          const int v = __reduce_add_sync(kFull, __popc(~s_map[32 * i + lane] & 0x80808080u));
          if (lane == i) c = v;
        }
        int inc = c;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int y = __shfl_up_sync(kFull, inc, d);
          if (lane >= d) inc += y;
        }
        if (lane < nr) a.below[(size_t)lane * nbp + blk] = (uint8_t)(inc - c);
      }
      for (int i = threadIdx.x; i < nr * 32; i += kThreads) a.smap[((size_t)(i >> 5) * nb + blk) * 32 + (i & 31)] = s_map[i];
    }
  } else {
    topk_token_cta<NJ, PART>(a, blk);
  }
}

// Routing CTAs for T tokens.
__host__ __device__ constexpr int route_blocks(int T, bool warp) { return warp ? (T + kWarps - 1) / kWarps : T; }

// Which body routes a launch: the warp body (measured faster at every batch size, 1 to
// 4096 tokens) wherever its float4 layout applies -- E <= kWarpMaxE, E % 4 == 0,
// 16-byte aligned rows and bias, at most kMaxPartSplits partials -- else the CTA body.
inline bool use_warp_body(int E, const void* rows, const float* bias, int S = 0) {
  return E <= kWarpMaxE && E % 4 == 0 && aligned(rows, 16) && (!bias || aligned(bias, 16)) && S <= kMaxPartSplits;
}

// Dynamic shared memory (never touched) that lets an SM hold no more than the fewest
// CTAs per SM one wave of `blocks` CTAs needs: back-to-back calls place a call's CTAs
// while earlier calls' still hold the SMs, and uncapped some SMs took up to seven of
// one call's CTAs, which then set its time (T = 1020: 5.9 us a call uncapped, 4.2
// capped at two per SM; a cap below one wave's need measured slower, 13.5 us at T =
// 4096 with two). 0 when no cap is needed.
inline size_t cta_cap_pad(const void* kern, long long blocks, const DeviceInfo& dev) {
  long long cap = (blocks + dev.sm_count - 1) / dev.sm_count;
  if (cap < 2) cap = 2;  // (room for the next call's CTA beside this one's)
  cudaFuncAttributes fa;
  if (cap < 1 || dev.smem_per_sm <= 0 || cudaFuncGetAttributes(&fa, kern) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const long long fixed = (long long)fa.sharedSizeBytes + dev.smem_reserved;  // per CTA
  const long long natural = dev.smem_per_sm / (fixed > 0 ? fixed : 1);     // (by shared memory alone)
  if (cap >= natural || cap >= 8) return 0;
  long long pad = dev.smem_per_sm / cap - fixed;
  pad = pad / 1024 * 1024 - 1024;  // (round down, and a margin below the cap's limit)
  return pad > 0 ? (size_t)pad : 0;
}

}  // namespace topk_impl
}  // namespace moe
