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
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kCluster = 8;  // CTAs sharing one expert range, one chunk of the ids each
constexpr int kMaxEpc = 32;  // experts per CTA
constexpr int kBatch = 16;   // steps (32 ids each) in flight per warp
constexpr int kHeld = 16;    // steps whose owned slots stay in registers
constexpr unsigned kFull = 0xFFFFFFFFu;

struct ListArgs {
  const int32_t* ids;
  int n;  // T * K
  int E, epc;
  int32_t* offsets;
  int32_t* pairs;
  uint32_t* err;
};

struct Scan {
  int e_lo, nexp, n;
  int below = 0;
  bool bad = false;
  uint32_t held[kHeld / 4];  // byte s%4 of held[s/4]: owned slot of step s's id, 0xFF = none
};

// Pass 1 over kBatch steps from flat id b0 (+ lane); CHECK also flags ids outside [0, E).
// Within each step the lanes holding an owned expert are grouped by it
// (__match_any_sync) and the group's lowest lane writes the group size to
// tab[step][expert] -- one writer per cell, no atomics; lane j then adds column j (its
// expert) to its count.
template <bool CHECK, bool HOLD>
__device__ __forceinline__ void count_batch(const ListArgs& a, Scan& sc, int b0, int r1, int lane,
                                            uint16_t (*tab)[kMaxEpc], int& count, int step0) {
  int v[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int i = b0 + 32 * u + lane;
    v[u] = i < r1 ? __ldg(a.ids + i) : -1;  // -1: never below e_lo, never owned
    if (CHECK && i < r1 && (unsigned)v[u] >= (unsigned)a.E) sc.bad = true;
  }
#pragma unroll
  for (int u = 0; u < kBatch; ++u) tab[u][lane] = 0;
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    sc.below += (unsigned)v[u] < (unsigned)sc.e_lo;
    const unsigned jv = (unsigned)(v[u] - sc.e_lo);
    const bool m = jv < (unsigned)sc.nexp;
    const unsigned bal = __ballot_sync(kFull, m);
    if (m) {
      const unsigned peers = __match_any_sync(bal, jv);
      if ((peers & ((1u << lane) - 1u)) == 0) tab[u][jv] = (uint16_t)__popc(peers);
      if (HOLD) {
        const int st = step0 + u;
        sc.held[st / 4] &= ~((~jv & 0xFFu) << (8 * (st % 4)));
      }
    }
  }
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kBatch; ++u) count += tab[u][lane];
  __syncwarp();
}

// Pass 2 for one block of up to kBatch steps of a warp: the ids i0 + 32*st + lane, with
// owned slots in the bytes of slot[] (0xFF = none). (1) Within each step, the matching
// lanes are grouped by expert (__match_any_sync); a lane's rank is the count of its
// group's lanes below it, and the group's lowest lane records the group size in
// tab[st][expert]. The steps do not depend on one another. (2) Lane j turns column j
// of tab into exclusive prefixes over the steps. (3) Every match is written at
// base[expert] + run[expert] + tab[st][expert] + rank; lane j then advances run[j].
__device__ __forceinline__ void place_block(const ListArgs& a, const uint32_t (&slot)[kBatch / 4], int i0, int nsteps,
                                            int nexp, int lane, uint16_t (*tab)[kMaxEpc], int* run, const int* base) {
#pragma unroll
  for (int st = 0; st < kBatch; ++st) tab[st][lane] = 0;
  __syncwarp();
  uint32_t rk[kBatch / 4] = {};
#pragma unroll
  for (int st = 0; st < kBatch; ++st) {
    if (st >= nsteps) break;  // warp-uniform
    const unsigned jv = (slot[st / 4] >> (8 * (st % 4))) & 0xFFu;
    const bool m = jv < (unsigned)nexp;
    const unsigned bal = __ballot_sync(kFull, m);
    if (m) {
      const unsigned peers = __match_any_sync(bal, jv);
      const unsigned r = __popc(peers & ((1u << lane) - 1u));
      rk[st / 4] |= r << (8 * (st % 4));
      if (r == 0) tab[st][jv] = (uint16_t)__popc(peers);
    }
  }
  __syncwarp();
  int total = 0;
#pragma unroll
  for (int st = 0; st < kBatch; ++st) {
    const int c = tab[st][lane];
    tab[st][lane] = (uint16_t)total;
    total += c;
  }
  __syncwarp();
#pragma unroll
  for (int st = 0; st < kBatch; ++st) {
    if (st >= nsteps) break;  // warp-uniform
    const unsigned jv = (slot[st / 4] >> (8 * (st % 4))) & 0xFFu;
    if (jv < (unsigned)nexp) {
      const int r = (int)((rk[st / 4] >> (8 * (st % 4))) & 0xFFu);
      a.pairs[base[jv] + run[jv] + tab[st][jv] + r] = i0 + 32 * st + lane;
    }
  }
  __syncwarp();
  run[lane] += total;
  __syncwarp();
}

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

  grid_wait();
  grid_launch_dependents();  // after the wait: dependents may rely on all before the lists

  // pass 1: lane j counts this warp's matches of owned expert j
  int* cnt = s_cnt[warp];
  uint16_t(*tab)[kMaxEpc] = s_tab[warp];
  int count = 0;
  const bool check = blockIdx.y == 0;  // the first expert range's cluster checks every id once
  if (r0 < r1) {
    if (check) count_batch<true, true>(a, sc, r0, r1, lane, tab, count, 0);
    else count_batch<false, true>(a, sc, r0, r1, lane, tab, count, 0);
  }
  for (int b0 = r0 + 32 * kHeld; b0 < r1; b0 += 32 * kBatch) {
    if (check) count_batch<true, false>(a, sc, b0, r1, lane, tab, count, 0);
    else count_batch<false, false>(a, sc, b0, r1, lane, tab, count, 0);
  }
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
  if (r0 < r1) place_block(a, sc.held, r0, min(kBatch, (r1 - r0 + 31) / 32), sc.nexp, lane, tab, cnt, s_start);
  for (int b0 = r0 + 32 * kHeld; b0 < r1; b0 += 32 * kBatch) {
    uint32_t slot[kBatch / 4];
#pragma unroll
    for (int h = 0; h < kBatch / 4; ++h) slot[h] = kFull;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = b0 + 32 * u + lane;
      const unsigned jv = (unsigned)((i < r1 ? __ldg(a.ids + i) : -1) - sc.e_lo);
      if (jv < (unsigned)sc.nexp) slot[u / 4] &= ~((~jv & 0xFFu) << (8 * (u % 4)));
    }
    place_block(a, slot, b0, min(kBatch, (r1 - b0 + 31) / 32), sc.nexp, lane, tab, cnt, s_start);
  }
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
