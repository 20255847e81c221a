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
// i.e. an order-preserving filter of the flat id array. That array is small (T*K*4
// bytes, L2-resident), so every CTA scans all of it and owns a range of experts: no
// cross-CTA scan, no workspace, no global atomics. Inside a CTA the 16 warps split the
// ids into contiguous ranges, loaded 1024 at a time (8 int4 per lane in flight; the
// first batch stays in registers for pass 2). Pass 1 counts, per warp, the ids below
// the CTA's first expert and (shared-memory atomics: counts do not depend on order)
// the matches of each owned expert; the CTA then knows where each warp's run of each
// expert starts. Pass 2 ballots which lanes hold a match -- most steps have none -- and
// writes those few in lane order, so every list stays in ascending index order.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxEpc = 32;      // experts per CTA
constexpr int kTargetCtas = 32;  // CTAs per launch (E / kMaxEpc at most 32 for E <= 1024)
constexpr int kBatch = 8;   // int4 loads in flight per lane (1024 ids per warp per batch)
constexpr unsigned kFull = 0xFFFFFFFFu;

struct ListArgs {
  const int32_t* ids;
  long long n;  // T * K
  int E, epc;
  int32_t* offsets;
  int32_t* pairs;
  uint32_t* err;
  int vec;  // ids may be read as int4
};

// ids i0..i0+3; entries at or past `end` read as -1 (never below e_lo, never a match)
__device__ __forceinline__ int4 load4(const ListArgs& a, long long i0, long long end) {
  if (a.vec && i0 + 3 < end) return __ldg(reinterpret_cast<const int4*>(a.ids + i0));
  int4 v;
  v.x = i0 < end ? __ldg(a.ids + i0) : -1;
  v.y = i0 + 1 < end ? __ldg(a.ids + i0 + 1) : -1;
  v.z = i0 + 2 < end ? __ldg(a.ids + i0 + 2) : -1;
  v.w = i0 + 3 < end ? __ldg(a.ids + i0 + 3) : -1;
  return v;
}

__global__ void __launch_bounds__(kThreads) lists_kernel(const ListArgs a) {
  __shared__ int s_below[kWarps];
  __shared__ int s_cnt[kWarps][kMaxEpc];
  __shared__ int s_run[kWarps][kMaxEpc];
  __shared__ int s_base[kMaxEpc + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e_lo = blockIdx.x * a.epc;
  const int nexp = min(a.epc, a.E - e_lo);
  // warp w scans flat ids [r0, r1): 128 per step, 4 per lane, lanes in order
  const long long per = ((a.n + kWarps - 1) / kWarps + 127) / 128 * 128;
  const long long r0 = min(a.n, (long long)warp * per), r1 = min(a.n, r0 + per);
  static_assert(kWarps * kMaxEpc == kThreads, "one counter per thread");
  s_cnt[threadIdx.x / kMaxEpc][threadIdx.x % kMaxEpc] = 0;
  __syncthreads();

  grid_launch_dependents();
  grid_wait();

  // pass 1 (the first batch of ids stays in registers for pass 2)
  int below = 0;
  bool bad = false;
  int4 held[kBatch];
  for (long long b0 = r0; b0 < r1; b0 += kBatch * 128) {
    int4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) v[u] = load4(a, b0 + 128 * u + 4 * lane, r1);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        below += (unsigned)q[m] < (unsigned)e_lo;
        const unsigned jv = (unsigned)(q[m] - e_lo);
        if (jv < (unsigned)nexp) atomicAdd(&s_cnt[warp][jv], 1);
        bad |= (unsigned)q[m] >= (unsigned)a.E && b0 + 128 * u + 4 * lane + m < r1;
      }
      if (b0 == r0) held[u] = v[u];
    }
  }
  if (blockIdx.x == 0 && __any_sync(kFull, bad) && lane == 0) set_error(a.err, MOE_DEVERR_EXPERT_ID);
  below = __reduce_add_sync(kFull, below);
  if (lane == 0) s_below[warp] = below;
  __syncthreads();

  // offsets of the owned experts, and where each warp's run of each expert starts
  if (threadIdx.x == 0) {
    int base = 0;
    for (int w = 0; w < kWarps; ++w) base += s_below[w];
    for (int j = 0; j < nexp; ++j) {
      s_base[j] = base;
      for (int w = 0; w < kWarps; ++w) base += s_cnt[w][j];
    }
    s_base[nexp] = base;
  }
  __syncthreads();
  {
    const int w = threadIdx.x / kMaxEpc, j = threadIdx.x % kMaxEpc;
    if (j < nexp) {
      int start = s_base[j];
      for (int ww = 0; ww < w; ++ww) start += s_cnt[ww][j];
      s_run[w][j] = start;
    }
  }
  if (threadIdx.x < nexp || (threadIdx.x == nexp && e_lo + nexp == a.E)) a.offsets[e_lo + threadIdx.x] = s_base[threadIdx.x];
  __syncthreads();

  // pass 2: the few matches, in lane order
  int* run = s_run[warp];
  for (long long b0 = r0; b0 < r1; b0 += kBatch * 128) {
    int4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) v[u] = (b0 == r0) ? held[u] : load4(a, b0 + 128 * u + 4 * lane, r1);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const long long b = b0 + 128 * u;
      if (b >= r1) break;  // warp-uniform
      const int q[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      unsigned m4 = 0;
#pragma unroll
      for (int m = 0; m < 4; ++m) m4 |= ((unsigned)(q[m] - e_lo) < (unsigned)nexp) ? (1u << m) : 0u;
      unsigned any = __ballot_sync(kFull, m4 != 0);
      while (any) {
        const int l = __ffs(any) - 1;
        any &= any - 1;
        if (lane == l) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if (m4 & (1u << m)) {
              const int jv = q[m] - e_lo;
              a.pairs[run[jv]++] = (int32_t)(b + 4 * lane + m);
            }
          }
        }
        __syncwarp();
      }
    }
  }
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
  // The time is set by each CTA's scan of all ids, not by the CTA count, so few CTAs
  // (about 32) do: the rest of the GPU stays free for work running beside the lists.
  int epc = (E + kTargetCtas - 1) / kTargetCtas;
  epc = epc < 1 ? 1 : (epc > kMaxEpc ? kMaxEpc : epc);
  const long long n = (long long)T * K;
  ListArgs a{ids, n, E, epc, offsets, pairs, dev.error_word, (K % 4 == 0 && aligned(ids, 16)) ? 1 : 0};
  return launch_pdl(lists_kernel, dim3((E + epc - 1) / epc), dim3(kThreads), 0, as_cuda(stream), a);
}
