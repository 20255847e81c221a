// Router logits: the two kernel families and their launch plans.
#pragma once

#include "common.cuh"

namespace moe {

// CUDA-core split-K path (small token counts).
void simt_plan(int T, int H, int E, int sm_count, int* S, int* kc);
int launch_router_simt(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, int S, int kc,
                       float* part, cudaStream_t stream);

// CUDA-core GEMV for T <= kGemvMaxTokens: no split-K, no workspace, one launch.
constexpr int kGemvMaxTokens = 8;
// The automatic choice (moe_router_logits, the one-call step) runs the GEMV only up to
// this many tokens: its token count is rounded up to 1, 2, 3, 4 or 8, and from 5 tokens the
// tcgen05 plan of one 16-token tile is faster (measured back to back over cold inputs:
// 5.7 against 6.9 us at T = 4, 7.6 against 6.8 at T = 6, 7.8 against 6.8 at T = 8).
constexpr int kAutoGemvMaxTokens = 4;
int launch_router_gemv(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, cudaStream_t stream);

// The one-call step's MXFP8 of the latent (mxfp8_quantize_rows, OCP floor rule,
// row-major scales), done by the tensor-core router's epilogue warps while its mainloop
// runs: the flat input of nchunks 16-byte chunks (16-byte aligned), q (8-byte aligned),
// scales (8-byte aligned).
struct LatentQuant {
  const uint16_t* x = nullptr;
  long long nchunks = 0;
  uint8_t* q = nullptr;
  uint8_t* scales = nullptr;
};

// Tensor-core (tcgen05) split-K path.
struct TcPlan {
  int bn;    // token tile: 16, 32, 64, 128 or 256
  int S;     // K splits
  int n_kb;  // 64-wide K blocks
  bool cluster;  // the S splits of a tile form a cluster and reduce in one kernel (partials through L2)
  bool pair = false;  // CTA pairs (cta_group::2 MMAs over 256 weight rows); S pairs per cluster
};
// Split-K workspace a plan needs (bytes): the partials [S][T][E] of the two-kernel
// reduction, or, for a cluster plan, every tile's S partial tiles [BN][128].
inline size_t tc_workspace(const TcPlan& p, int T, int E) {
  if (p.S <= 1) return 0;
  if (!p.cluster) return (size_t)p.S * T * E * sizeof(float);
  size_t m_tiles = (size_t)((E + 127) / 128);
  if (p.pair) m_tiles = (m_tiles + 1) / 2 * 2;  // pairs of 128-row tiles (the last may be padding)
  const size_t tiles = m_tiles * ((T + p.bn - 1) / p.bn);
  return tiles * p.S * p.bn * 128 * sizeof(float);
}
TcPlan tc_plan(int T, int H, int E, int sm_count);         // single CTAs or CTA pairs
TcPlan tc_plan_single(int T, int H, int E, int sm_count);  // single CTAs only
int launch_router_tc(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, const TcPlan& p,
                     float* part, uint32_t* err, cudaStream_t stream, const LatentQuant* lq = nullptr);

// The front projection: router logits (FP32 [T, E]) and the latent down projection
// (BF16 [T, L], one rounding of the FP32 sum) in one tensor-core launch over x. The
// plan's splits are reduced on chip (cluster plan) or there are none.
TcPlan front_plan(int T, int H, int E, int L, int sm_count);
size_t front_workspace(const TcPlan& p, int T, int E, int L);
int launch_front_tc(const uint16_t* x, const uint16_t* w, const uint16_t* w2, float* logits, uint16_t* latent, int T,
                    int H, int E, int L, const TcPlan& p, float* part, uint32_t* err, cudaStream_t stream);

// The tensor-core router's split-K partials [S][T][E] without their reduction (the
// consumer sums them in split order; S == 1: logits written directly). *S_out = S.
// With lq, the launch also quantises the latent when it runs the tensor-core kernel
// (*quantised = true; false for the few-token GEMV, which leaves it to the caller).
int launch_router_partials(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, int sm_count,
                           float* part, uint32_t* err, cudaStream_t stream, int* S_out,
                           const LatentQuant* lq = nullptr, bool* quantised = nullptr);
size_t router_partials_bytes(int T, int H, int E, int sm_count);

// logits = sum over s of part[s] (split order), part [S][T][E].
int launch_router_reduce(const float* part, int S, int T, int E, float* logits, cudaStream_t stream);

}  // namespace moe
