// Per-expert routing lists: a deterministic, atomics-free counting sort.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, WideRoute
// (docstring and kernel): each of token t's pairs is appended to its expert's list as
// the code t*K + k -- the expanded-row index Finalize reads. The pages append with a
// relaxed atomic counter, so their list order is arbitrary; here every list is in
// ascending token order and stored as CSR (offsets = exclusive prefix sum of counts).
//
// GB300 design: the pair code of ids[t, k] is its flat index i = t*K + k, so for an
// expert e
//   offsets[e]             = #{ i : 0 <= ids[i] < e }
//   pairs[offsets[e] + r]  = the r-th i (ascending) with ids[i] == e
// i.e. an order-preserving filter of the flat id array (T*K*4 bytes, L2-resident).
// One thread-block cluster of kCluster CTAs per range of 32 experts; CTA c of a cluster
// owns the c-th chunk of the ids, and each of its 16 warps a contiguous part of that,
// walked in steps of 32 (lane l reads id step*32 + l: every load a coalesced 128
// bytes; all steps of a part in flight at once -- one L2 round trip, since round trips,
// not arithmetic, set this kernel's time). Pass 1 counts, per (warp, owned expert), the
// matches -- each step's matching lanes grouped by expert (__match_any_sync), the
// group's lowest lane writing its size to a per-warp table, lane j summing expert j's
// column, so every shared-memory cell has one writer and no atomic is used -- and, per
// lane, the ids below the range; the owned slot of each loaded id (or "none") stays in
// registers, a byte an id. Warp j scans expert j's counts over the warps (shuffles)
// into each warp's start within the CTA's share. The CTAs then exchange their per-expert totals and
// below-counts through distributed shared memory (after a cluster barrier), so each
// knows where its share of every list starts, and CTA 0 writes the range's offsets.
// Pass 2 places a block of 16 steps without a serial chain: the ranks inside every step
// come from __match_any_sync at once (no step waits on another), a per-warp table turns
// the steps' group sizes into per-step starts, and every match is then written in
// parallel -- lists in ascending index order. No workspace and no atomics (shared or
// global): the counts and placements come from warp votes and single-writer tables.
#include "lists.cuh"

namespace moe {
namespace {

using namespace lists_impl;
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kCluster = 8;  // CTAs sharing one expert range, one chunk of the ids each

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// An int from the same shared-memory variable of CTA `rank` of the cluster.
__device__ __forceinline__ int ld_cluster(const int* local, uint32_t rank) {
  uint32_t remote;
  int v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

__global__ void __launch_bounds__(kThreads) lists_kernel(const ListArgs a) {
  __shared__ int s_cnt[kWarps][kMaxEpc + 1];  // count, then start within the CTA's share, per (warp, expert)
  __shared__ __align__(16) uint16_t s_tab[kWarps][kBatch][kMaxEpc];
  __shared__ int s_below[kWarps];
  __shared__ int s_tot[kMaxEpc + 1];   // this CTA's matches per owned expert; [kMaxEpc]: its ids below
  __shared__ int s_base[kMaxEpc + 1];  // offsets of the owned experts
  __shared__ int s_start[kMaxEpc];     // where this CTA's share of each owned expert's list starts
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t crank = cluster_rank();
  Scan sc;
  sc.e_lo = blockIdx.y * a.epc;
  sc.nexp = min(a.epc, a.E - sc.e_lo);
  sc.n = a.n;
#pragma unroll
  for (int h = 0; h < kHeld / 4; ++h) sc.held[h] = kFull;
  // CTA c of the cluster owns the flat ids [c0, c1); warp w of it [r0, r1) (multiples of 32)
  const int chunk = (int)(((long long)a.n + kCluster * 32 - 1) / (kCluster * 32)) * 32;
  const int c0 = (int)min((long long)a.n, (long long)crank * chunk), c1 = min(a.n, c0 + chunk);
  const int per = (chunk / 32 + kWarps - 1) / kWarps * 32;
  const int r0 = min(c1, c0 + warp * per), r1 = min(c1, r0 + per);
  static_assert(kMaxEpc == 32 && kWarps == 16, "one lane per owned expert; two expert columns per warp");
  static_assert(kHeld == kBatch && kBatch % 4 == 0, "held steps are one pass-2 block");

  // this CTA's ids: their DRAM fetch overlaps the preceding kernel's end (a hint only)
  if (threadIdx.x == 0 && c1 - c0 >= 4 && ((reinterpret_cast<uintptr_t>(a.ids + c0) & 15) == 0))
    prefetch_l2(a.ids + c0, (uint32_t)((c1 - c0) & ~3) * 4u);
  grid_wait();
  grid_launch_dependents();  // after the wait: dependents may rely on all before the lists

  // pass 1: lane j counts this warp's matches of owned expert j
  int* cnt = s_cnt[warp];
  uint16_t(*tab)[kMaxEpc] = s_tab[warp];
  const bool check = blockIdx.y == 0;  // the first expert range's cluster checks every id once
  const int count = check ? count_all<true>(a, sc, r0, r1, lane, tab) : count_all<false>(a, sc, r0, r1, lane, tab);
  cnt[lane] = count;
  if (check && __any_sync(kFull, sc.bad) && lane == 0) set_error(a.err, MOE_DEVERR_EXPERT_ID);
  const int below = __reduce_add_sync(kFull, sc.below);
  if (lane == 0) s_below[warp] = below;
  __syncthreads();

  // expert j's counts over the warps -> each warp's start within this CTA's share
  // (lanes 0-15 scan column `warp`, lanes 16-31 column `warp + 16`; lane & 15 = warp)
  {
    const int j = warp + (lane & 16), w = lane & 15;
    const int c = s_cnt[w][j];
    int inc = c;
#pragma unroll
    for (int d = 1; d < 16; d <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, d, 16);
      if (w >= d) inc += y;
    }
    s_cnt[w][j] = inc - c;  // the cell this thread alone read
    if (w == 15) s_tot[j] = inc;
    if (warp == 0 && lane == 0) {
      int b = 0;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) b += s_below[ww];
      s_tot[kMaxEpc] = b;
    }
  }
  cluster_sync_all();  // every CTA's totals are written and visible to the cluster

  // warp 0 gathers the cluster's totals (lane j = expert e_lo + j; zero past nexp)
  if (warp == 0) {
    int pre = 0, all = 0, base = 0;
#pragma unroll
    for (uint32_t r = 0; r < (uint32_t)kCluster; ++r) {
      const int v = ld_cluster(&s_tot[lane], r);
      pre += r < crank ? v : 0;
      all += v;
      base += ld_cluster(&s_tot[kMaxEpc], r);
    }
    int inc = all;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, d);
      if (lane >= d) inc += y;
    }
    s_base[lane] = base + inc - all;
    s_start[lane] = base + inc - all + pre;
    if (lane == 31) s_base[32] = base + inc;
  }
  cluster_arrive();  // this CTA reads no other CTA's shared memory from here on
  __syncthreads();
  if (crank == 0 && (threadIdx.x < sc.nexp || (threadIdx.x == sc.nexp && sc.e_lo + sc.nexp == a.E)))
    a.offsets[sc.e_lo + threadIdx.x] = s_base[threadIdx.x];

  // pass 2
  place_all(a, sc, r0, r1, lane, tab, cnt, s_start);
  cluster_wait();  // no CTA exits while another may still read its shared memory
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_build_routing_lists_workspace(int T, int K, int E) {
  (void)T;
  (void)K;
  (void)E;
  return 0;
}

extern "C" int moe_build_routing_lists(const int32_t* ids, int T, int K, int E, int32_t* offsets,
                                       int32_t* pairs, void* workspace, size_t workspace_bytes,
                                       moe_stream_t stream) {
  using namespace moe;
  (void)workspace;
  (void)workspace_bytes;
  if (T < 0 || K < 1 || E < 1) return MOE_ERR_INVALID_ARGUMENT;
  if (K > MOE_MAX_TOPK || E > MOE_MAX_EXPERTS) return MOE_ERR_CAPACITY;
  if ((long long)T * K > (1LL << 31) - 1) return MOE_ERR_CAPACITY;
  if (!offsets || (T > 0 && (!ids || !pairs))) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(offsets, 4) || (ids && !aligned(ids, 4)) || (pairs && !aligned(pairs, 4))) return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  const int epc = kMaxEpc;
  ListArgs a{ids, T * K, E, epc, offsets, pairs, dev.error_word};
  auto kern = lists_kernel;
  if (prefer_max_shared(reinterpret_cast<const void*>(kern)) != MOE_OK) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster, (E + epc - 1) / epc);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = as_cuda(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
