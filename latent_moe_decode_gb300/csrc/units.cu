// Unit windows of the routing lists: the work plan of a grouped expert engine that
// streams each touched expert's weights once per `window` of its tokens.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, module
// docstring (the wide grouped engine takes its work units from the routing lists,
// reading each expert that has tokens once for every 8 of them).
//
// For each expert e with n_e = offsets[e+1] - offsets[e] listed pairs there are
// ceil(n_e / W) units; unit j of e covers list positions offsets[e] + jW ..
// min(offsets[e] + (j+1)W, offsets[e+1]). Units are numbered by expert, then j;
// unit_offsets is the exclusive prefix sum of the per-expert unit counts.
//
// GB300 design: one CTA of 1024 threads (E <= 1024 experts, one per thread) reads the
// offsets (at most 4 KB), scans the unit counts (warp shuffles, then one warp over the
// 32 warp totals), and then every thread writes units u = tid, tid + 1024, ... (each
// finds its expert by binary search over the scanned counts in shared memory), so the
// writes are coalesced and a heavy expert's units are spread over all threads.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads, 1)
    units_kernel(const int32_t* __restrict__ offsets, int E, int W, int32_t* __restrict__ unit_offsets,
                 int32_t* __restrict__ unit_expert, int32_t* __restrict__ unit_start, int32_t* __restrict__ unit_len,
                 int max_units, uint32_t* err) {
  __shared__ int32_t uoff[kThreads + 1];  // exclusive unit prefix per expert
  __shared__ int32_t woff[kThreads + 1];  // list offsets
  __shared__ int32_t wsum[32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  grid_wait();
  grid_launch_dependents();
  int n = 0, o = 0;
  if (e < E) {
    o = offsets[e];
    n = offsets[e + 1] - o;
  }
  const int u = n > 0 ? (n + W - 1) / W : 0;
  int incl = u;  // inclusive scan within the warp
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane], sc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xFFFFFFFFu, sc, d);
      if (lane >= d) sc += x;
    }
    wsum[lane] = sc - v;  // exclusive over warps
  }
  __syncthreads();
  const int excl = wsum[warp] + incl - u;
  if (e < E) {
    uoff[e] = excl;
    woff[e] = o;
  }
  if (e == E - 1) {  // (thread E - 1 alone writes entry E)
    uoff[E] = excl + u;
    woff[E] = o + n;
  }
  __syncthreads();
  if (e < E) unit_offsets[e] = uoff[e];
  if (e == 0) unit_offsets[E] = uoff[E];
  const int total = uoff[E];
  if (e == 0 && total > max_units) set_error(err, MOE_DEVERR_CAPACITY);  // not within the capacity bound
  const int lim = total < max_units ? total : max_units;
  for (int i = e; i < lim; i += kThreads) {
    int lo = 0, hi = E - 1;  // the expert x with uoff[x] <= i < uoff[x + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (uoff[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    const int j = i - uoff[lo];
    const int start = woff[lo] + j * W;
    const int end = woff[lo + 1];
    unit_expert[i] = lo;
    unit_start[i] = start;
    unit_len[i] = end - start < W ? end - start : W;
  }
}

}  // namespace
}  // namespace moe

extern "C" int moe_unit_windows_capacity(int T, int K, int E, int window) {
  if (T < 0 || K < 1 || E < 1 || window < 1) return -1;
  const long long pairs = (long long)T * K;
  long long cap = (pairs + window - 1) / window + E;  // each expert adds at most one partial unit
  if (cap > pairs) cap = pairs;
  return cap > 0x7FFFFFFF ? -1 : (int)cap;
}

extern "C" int moe_build_unit_windows(const int32_t* offsets, int E, int window, int32_t* unit_offsets,
                                      int32_t* unit_expert, int32_t* unit_start, int32_t* unit_len, int max_units,
                                      moe_stream_t stream) {
  using namespace moe;
  if (E < 1 || window < 1 || max_units < 0) return MOE_ERR_INVALID_ARGUMENT;
  if (E > MOE_MAX_EXPERTS) return MOE_ERR_CAPACITY;
  if (!offsets || !unit_offsets || (max_units > 0 && (!unit_expert || !unit_start || !unit_len)))
    return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(offsets, 4) || !aligned(unit_offsets, 4) || !aligned(unit_expert, 4) || !aligned(unit_start, 4) ||
      !aligned(unit_len, 4))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  const int st = current_device(&dev);
  if (st != MOE_OK) return st;
  return launch_pdl(units_kernel, dim3(1), dim3(kThreads), 0, as_cuda(stream), offsets, E, window, unit_offsets,
                    unit_expert, unit_start, unit_len, max_units, dev.error_word);
}
