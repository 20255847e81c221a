// Router logits: the two kernel families and their launch plans.
#pragma once

#include "common.cuh"

namespace moe {

// CUDA-core split-K path (small token counts).
void simt_plan(int T, int H, int E, int sm_count, int* S, int* kc);
int launch_router_simt(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, int S, int kc,
                       float* part, cudaStream_t stream);

// Tensor-core (tcgen05) split-K path.
struct TcPlan {
  int bn;    // token tile: 16, 32, 64, 128 or 256
  int S;     // K splits
  int n_kb;  // 64-wide K blocks
  bool cluster;  // splits reduced on chip through distributed shared memory (no workspace)
};
// Split-K workspace a plan needs (bytes).
inline size_t tc_workspace(const TcPlan& p, int T, int E) {
  return (p.S > 1 && !p.cluster) ? (size_t)p.S * T * E * sizeof(float) : 0;
}
TcPlan tc_plan(int T, int H, int E, int sm_count);
int launch_router_tc(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, const TcPlan& p,
                     float* part, uint32_t* err, cudaStream_t stream);

// logits = sum over s of part[s] (split order), part [S][T][E].
int launch_router_reduce(const float* part, int S, int T, int E, float* logits, cudaStream_t stream);

}  // namespace moe
