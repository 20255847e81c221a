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
// GB300 design: one CTA of 1024 threads (E <= 4096 experts, up to four consecutive
// experts per thread) reads the offsets (at most 16 KB), scans the unit counts (each
// thread's own experts, warp shuffles, then one warp over the 32 warp totals), and then
// every thread writes units u = tid, tid + 1024, ... (each finds its expert by binary
// search over the scanned counts in shared memory), so the writes are coalesced and a
// heavy expert's units are spread over all threads.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kPer = MOE_MAX_EXPERTS / kThreads;  // experts per thread

__global__ void __launch_bounds__(kThreads, 1)
    units_kernel(const int32_t* __restrict__ offsets, int E, int W, int32_t* __restrict__ unit_offsets,
                 int32_t* __restrict__ unit_expert, int32_t* __restrict__ unit_start, int32_t* __restrict__ unit_len,
                 int max_units, uint32_t* err) {
  __shared__ int32_t uoff[MOE_MAX_EXPERTS + 1];  // exclusive unit prefix per expert
  __shared__ int32_t woff[MOE_MAX_EXPERTS + 1];  // list offsets
  __shared__ int32_t wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_wait();
  grid_launch_dependents();
  // this thread's experts e0 .. e0 + kPer - 1 (those below E)
  const int e0 = tid * kPer;
  int o[kPer + 1], u[kPer], mine = 0;
#pragma unroll
  for (int i = 0; i <= kPer; ++i) o[i] = e0 + i <= E ? offsets[e0 + i] : 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int n = e0 + i < E ? o[i + 1] - o[i] : 0;
    u[i] = n > 0 ? (n + W - 1) / W : 0;
    mine += u[i];
  }
  int incl = mine;  // inclusive scan of the thread totals within the warp
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
  int excl = wsum[warp] + incl - mine;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = e0 + i;
    if (e < E) {
      uoff[e] = excl;
      woff[e] = o[i];
      excl += u[i];
      if (e == E - 1) {  // (the thread holding expert E - 1 alone writes entry E)
        uoff[E] = excl;
        woff[E] = o[i + 1];
      }
    }
  }
  __syncthreads();
  for (int e = tid; e <= E; e += kThreads) unit_offsets[e] = uoff[e];
  const int total = uoff[E];
  if (tid == 0 && total > max_units) set_error(err, MOE_DEVERR_CAPACITY);  // not within the capacity bound
  const int lim = total < max_units ? total : max_units;
  for (int i = tid; i < lim; i += kThreads) {
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
