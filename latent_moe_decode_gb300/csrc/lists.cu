// Per-expert routing lists: a deterministic counting sort of the (token, slot) pairs.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideRoute
// (docstring and kernel): each of token t's pairs is appended to its expert's list as
// the code t*K + k -- the expanded-row index Finalize reads. The pages append with a
// relaxed atomic counter, so their list order is arbitrary; here every list is in
// ascending token order and stored as CSR (offsets = exclusive prefix sum of counts).
//
// GB300 design: one CTA of 32 warps per chunk of 1024 tokens; lane l of warp w owns
// token 32 w + l. For each slot k the warp groups equal expert ids with match.any; the
// group's lowest lane ORs the group's lane mask into M[w][e] in shared memory (one
// writer per word per step, so no atomics). Then per expert: P[w][e] = the tokens of
// warps before w that chose e (prefix of popc(M)), counts = popc sums, offsets = a
// block scan over experts, and a pair lands at
//   offsets[e] + (pairs of earlier chunks) + P[w][e] + popc(M[w][e] & lanes below l).
// Up to 1024 tokens need one launch; beyond, a counting launch writes per-chunk counts
// to the workspace and a placing launch adds the earlier chunks' counts.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kChunk = 1024;  // tokens per CTA (32 warps x 32 lanes)
constexpr unsigned kFull = 0xFFFFFFFFu;

enum Mode { kSingle = 0, kCount = 1, kPlace = 2 };

struct ListArgs {
  const int32_t* ids;
  int T, K, E;
  int32_t* offsets;
  int32_t* pairs;
  int32_t* counts;  // [nchunks][E] workspace (kCount / kPlace)
  int nchunks;
  uint32_t* err;
};

size_t smem_bytes(int E) { return (size_t)32 * E * 4 + (size_t)32 * E * 2 + (size_t)(E + 1) * 4 + 32 * 4; }

// Exclusive scan of one value per thread over a 1024-thread block; *total gets the sum.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int ws = warp_sums[lane];
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += y;
    }
    warp_sums[lane] = wi - ws;  // exclusive warp offsets
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_sums[w] + incl - v;
  __syncthreads();
  return r;
}

// KMAX: compile-time bound on K (16 or 32), the size of the per-thread id array.
template <int MODE, int KMAX>
__global__ void __launch_bounds__(1024) lists_kernel(const ListArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int E = a.E, K = a.K;
  uint32_t* M = reinterpret_cast<uint32_t*>(smem);           // [32][E] lane masks
  uint16_t* P = reinterpret_cast<uint16_t*>(M + 32 * E);     // [32][E] warp prefixes
  int32_t* base = reinterpret_cast<int32_t*>(P + 32 * E);    // [E + 1]
  int32_t* warp_sums = base + E + 1;                         // [32]
  __shared__ int total_sh;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int chunk = blockIdx.x;

  grid_launch_dependents();
  grid_wait();
  for (int i = tid; i < 32 * E; i += kChunk) M[i] = 0u;

  const int t = chunk * kChunk + tid;
  const bool live = t < a.T;
  int my_e[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    int e = -1;
    if (live && k < K) {
      e = __ldg(a.ids + (size_t)t * K + k);
      if (e < 0 || e >= E) {
        set_error(a.err, MOE_DEVERR_EXPERT_ID);
        e = -1;
      }
    }
    my_e[k] = e;
  }
  __syncthreads();
  uint32_t* Mw = M + w * E;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {  // uniform across the block
      const unsigned g = __match_any_sync(kFull, my_e[k]);
      if (my_e[k] >= 0 && lane == __ffs(g) - 1) Mw[my_e[k]] |= g;
      __syncwarp();
    }
  }
  __syncthreads();

  // per expert: warp prefixes and this chunk's count
  int cnt = 0;
  const int e_own = tid;  // E <= 1024: one expert per thread
  if (e_own < E) {
    int run = 0;
    for (int ww = 0; ww < 32; ++ww) {
      P[ww * E + e_own] = (uint16_t)run;
      run += __popc(M[ww * E + e_own]);
    }
    cnt = run;
  }
  if (MODE == kCount) {
    if (e_own < E) a.counts[(size_t)chunk * E + e_own] = cnt;
    return;
  }
  int pre = 0, all = cnt;
  if (MODE == kPlace && e_own < E) {
    all = 0;
    for (int c = 0; c < a.nchunks; ++c) {
      const int v = a.counts[(size_t)c * E + e_own];
      all += v;
      if (c < chunk) pre += v;
    }
  }
  const int excl = block_exclusive_scan(e_own < E ? all : 0, warp_sums, &total_sh);
  if (e_own < E) {
    base[e_own] = excl + pre;
    if (chunk == 0) a.offsets[e_own] = excl;
  }
  if (chunk == 0 && tid == 0) a.offsets[E] = total_sh;
  __syncthreads();

  if (live) {
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (k < K && my_e[k] >= 0) {
        const int e = my_e[k];
        const int pos = base[e] + P[w * E + e] + __popc(Mw[e] & below);
        a.pairs[pos] = t * K + k;
      }
    }
  }
}

template <int KMAX>
int launch_all(const ListArgs& a, size_t smem, cudaStream_t s) {
  if (a.nchunks == 1) {
    if (cudaFuncSetAttribute(lists_kernel<kSingle, KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    return launch_pdl(lists_kernel<kSingle, KMAX>, dim3(1), dim3(kChunk), smem, s, a);
  }
  if (cudaFuncSetAttribute(lists_kernel<kCount, KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(lists_kernel<kPlace, KMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int st = launch_pdl(lists_kernel<kCount, KMAX>, dim3(a.nchunks), dim3(kChunk), smem, s, a);
  if (st != MOE_OK) return st;
  return launch_pdl(lists_kernel<kPlace, KMAX>, dim3(a.nchunks), dim3(kChunk), smem, s, a);
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_build_routing_lists_workspace(int T, int K, int E) {
  if (T <= moe::kChunk || E < 1) return 0;
  (void)K;
  const size_t nchunks = ((size_t)T + moe::kChunk - 1) / moe::kChunk;
  return nchunks * (size_t)E * sizeof(int32_t);
}

extern "C" int moe_build_routing_lists(const int32_t* ids, int T, int K, int E, int32_t* offsets,
                                       int32_t* pairs, void* workspace, size_t workspace_bytes,
                                       moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || K < 1 || E < 1) return MOE_ERR_INVALID_ARGUMENT;
  if (K > MOE_MAX_TOPK || E > MOE_MAX_EXPERTS) return MOE_ERR_CAPACITY;
  if ((long long)T * K > (1LL << 31) - 1) return MOE_ERR_CAPACITY;
  if (!offsets || (T > 0 && (!ids || !pairs))) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(offsets, 4) || (ids && !aligned(ids, 4)) || (pairs && !aligned(pairs, 4))) return MOE_ERR_ALIGNMENT;
  const size_t need = moe_build_routing_lists_workspace(T, K, E);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 4))) return MOE_ERR_WORKSPACE;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const int nchunks = T <= kChunk ? 1 : (T + kChunk - 1) / kChunk;
  ListArgs a{ids, T, K, E, offsets, pairs, static_cast<int32_t*>(workspace), nchunks, dev.error_word};
  const size_t smem = smem_bytes(E);
  cudaStream_t s = as_cuda(stream);
  return K <= 16 ? launch_all<16>(a, smem, s) : launch_all<MOE_MAX_TOPK>(a, smem, s);
}
