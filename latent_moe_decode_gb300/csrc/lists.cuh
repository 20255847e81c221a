// Per-expert routing lists: the per-warp counting and placing steps shared by the
// cluster kernel of moe_build_routing_lists (lists.cu) and the one-CTA-per-range form
// that the one-call step runs inside its Finalize launch (finalize.cu).
//
// The pair code of ids[t, k] is its flat index i = t*K + k, so for an expert e
//   offsets[e]             = #{ i : 0 <= ids[i] < e }
//   pairs[offsets[e] + r]  = the r-th i (ascending) with ids[i] == e
// i.e. an order-preserving filter of the flat id array. A CTA owns a range of 32
// experts (one per lane); its warps walk the ids in steps of 32 (lane l reads id
// step*32 + l: one coalesced 128-byte load per step). Counting and placing use warp
// votes and single-writer tables only: no atomics.
#pragma once

#include "common.cuh"

namespace moe {
namespace lists_impl {

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

// Pass 2 over the ids [r0, r1) of a warp whose first kHeld steps' owned slots are in
// sc.held: every match written at base[expert] + run[expert] + its rank in the warp's
// id order (run[j]: where this warp's share of expert j's list starts, advanced here).
__device__ __forceinline__ void place_all(const ListArgs& a, const Scan& sc, int r0, int r1, int lane,
                                          uint16_t (*tab)[kMaxEpc], int* run, const int* base) {
  if (r0 < r1) place_block(a, sc.held, r0, min(kBatch, (r1 - r0 + 31) / 32), sc.nexp, lane, tab, run, base);
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
    place_block(a, slot, b0, min(kBatch, (r1 - b0 + 31) / 32), sc.nexp, lane, tab, run, base);
  }
}

// Pass 1 over the ids [r0, r1) of a warp: lane j's count of owned expert j (returned),
// sc.below (this lane's ids below the range) and sc.held filled; CHECK flags ids outside
// [0, E) in sc.bad.
template <bool CHECK>
__device__ __forceinline__ int count_all(const ListArgs& a, Scan& sc, int r0, int r1, int lane,
                                         uint16_t (*tab)[kMaxEpc]) {
  int count = 0;
  if (r0 < r1) count_batch<CHECK, true>(a, sc, r0, r1, lane, tab, count, 0);
  for (int b0 = r0 + 32 * kHeld; b0 < r1; b0 += 32 * kBatch) count_batch<CHECK, false>(a, sc, b0, r1, lane, tab, count, 0);
  return count;
}

// Shared memory of the one-CTA-per-range form (W warps).
template <int W>
struct RangeSmem {
  int cnt[W][kMaxEpc];                    // per (warp, expert): count, then the warp's start in the list
  __align__(16) uint16_t tab[W][kBatch][kMaxEpc];
  int below[W];
  int start[kMaxEpc];                     // where each owned expert's list starts (its offset)
};

// One CTA of W warps builds the lists of expert range `range` (32 experts) from all
// the ids, with no other CTA involved: warp w scans the w-th contiguous part of the ids
// (in steps of 32), the warps' counts are scanned per expert, the ids below the range
// give the base, and the CTA writes its offsets and places its pairs. Every thread of
// the CTA calls this; the CTA must already have waited for the ids.
template <int W>
__device__ __forceinline__ void lists_range_cta(const ListArgs& a, int range, RangeSmem<W>& sm) {
  static_assert(W >= 1 && W <= 32, "one warp per part of the ids");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Scan sc;
  sc.e_lo = range * kMaxEpc;
  sc.nexp = min(kMaxEpc, a.E - sc.e_lo);
  sc.n = a.n;
#pragma unroll
  for (int h = 0; h < kHeld / 4; ++h) sc.held[h] = kFull;
  const int per = ((a.n + 31) / 32 + W - 1) / W * 32;
  const int r0 = min(a.n, warp * per), r1 = min(a.n, r0 + per);
  const int count = range == 0 ? count_all<true>(a, sc, r0, r1, lane, sm.tab[warp])
                               : count_all<false>(a, sc, r0, r1, lane, sm.tab[warp]);
  sm.cnt[warp][lane] = count;
  if (range == 0 && __any_sync(kFull, sc.bad) && lane == 0) set_error(a.err, MOE_DEVERR_EXPERT_ID);
  const int below = __reduce_add_sync(kFull, sc.below);
  if (lane == 0) sm.below[warp] = below;
  __syncthreads();
  if (warp == 0) {
    // lane j: expert e_lo + j's count over the warps -> each warp's start, the offsets
    int b = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) b += sm.below[w];
    int wstart[W];
#pragma unroll
    for (int w = 0; w < W; ++w) {
      wstart[w] = tot;
      tot += sm.cnt[w][lane];
    }
    int inc = tot;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, d);
      if (lane >= d) inc += y;
    }
    const int off = b + inc - tot;  // offsets[e_lo + lane]
    sm.start[lane] = off;
#pragma unroll
    for (int w = 0; w < W; ++w) sm.cnt[w][lane] = wstart[w];
    if (lane < sc.nexp) a.offsets[sc.e_lo + lane] = off;
    if (lane == sc.nexp - 1 && sc.e_lo + sc.nexp == a.E) a.offsets[a.E] = off + tot;
  }
  __syncthreads();
  place_all(a, sc, r0, r1, lane, sm.tab[warp], sm.cnt[warp], sm.start);
}

// ---------------------------------------------------------------------------------
// The one-call step's lists from the routing CTAs' slot map (TopkArgs::smap): for every
// 4-token block b and expert e, the four tokens' slots of e (0xFF when absent), stored
// range-major (smap[r][b][j], e = 32 r + j), so a range's map is contiguous and expert
// e's list is the present bytes of its column in (b, byte) order -- token order --
// with pair codes (4b + i) * K + slot. One CTA of W warps builds the lists of one range
// of 32 experts (lane = expert): the pairs below the range are the sum of one row of
// `below` (written by the routing CTAs); warp w takes a contiguous share of the blocks;
// pass 1 counts each expert's pairs in the share, the shares' counts are scanned per
// expert and the range's totals over the experts, and pass 2 writes every pair in
// order. No atomics.
struct MapArgs {
  const uint32_t* smap;  // [ceil(E / 32)][nb][32]
  const uint8_t* below;  // [ceil(E / 32)][nbp]
  int T, K, E;
  int32_t* offsets;
  int32_t* pairs;
};

template <int W>
struct MapSmem {
  int base[W];
  __align__(16) uint32_t words[1];  // [chunk blocks][32]: the range's map, staged; then the
                                    // per-(chunk, warp, expert) counts (bytes past the struct's end)
};

// Chunks of `chunk` blocks that cover a range's map of nb blocks.
__host__ __device__ constexpr int map_chunks(int nb, int chunk) { return (nb + chunk - 1) / chunk; }

// Shared memory the lists role needs to stage `chunk` blocks of a range's map of nb
// blocks at a time, with its per-(chunk, warp, expert) counts.
template <int W>
__host__ __device__ constexpr size_t map_smem_bytes(int nb, int chunk) {
  return sizeof(MapSmem<W>) + (size_t)chunk * 32 * 4 + (size_t)map_chunks(nb, chunk) * W * 32 * 4;
}

// The largest chunk (blocks) whose map_smem_bytes fits in `bytes`, or 0.
template <int W>
inline int map_chunk_for(int nb, size_t bytes) {
  for (int chunk = nb; chunk >= 1;) {
    if (map_smem_bytes<W>(nb, chunk) <= bytes) return chunk;
    const size_t fixed = sizeof(MapSmem<W>) + (size_t)map_chunks(nb, chunk) * W * 32 * 4;
    if (fixed >= bytes) return 0;
    const int fit = (int)((bytes - fixed) / (32 * 4));
    chunk = fit < chunk ? fit : chunk - 1;
  }
  return 0;
}

__device__ __forceinline__ void cp_async16_ca(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}

// Stage blocks [c0, c1) of the range's map: every 16-byte copy requested at once (one
// round trip however busy the memory system is), then awaited.
template <int W>
__device__ __forceinline__ void stage_map(const uint32_t* rmap, int c0, int c1, uint32_t* words) {
  __syncthreads();  // the previous chunk's words are no longer read
  const uint4* src = reinterpret_cast<const uint4*>(rmap + (size_t)c0 * 32);
  uint4* dst = reinterpret_cast<uint4*>(words);
  for (int i = threadIdx.x; i < (c1 - c0) * 8; i += W * 32) cp_async16_ca(dst + i, src + i);
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  __syncthreads();
}

// chunk: the blocks of the range's map staged at a time (the CTA's shared memory holds
// map_smem_bytes<W>(nb, chunk)). Pass 1 stages every chunk in turn and counts, per
// (chunk, warp, expert), the pairs of the warp's share of the chunk; warp 0 then turns
// the counts into the offsets and every (chunk, warp)'s start in each list; pass 2
// places the pairs chunk by chunk, the chunk still staged first (with one chunk -- T up
// to about 2000 at 16 KB of stages per warp -- the map is read once).
template <int W>
__device__ __forceinline__ void lists_from_map(const MapArgs& m, int range, MapSmem<W>& sm, int chunk) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = (m.T + 3) / 4, nbp = (nb + 15) / 16 * 16, nch = map_chunks(nb, chunk);
  const int e = range * kMaxEpc + lane;
  const uint32_t* rmap = m.smap + (size_t)range * nb * 32;
  int* ccnt = reinterpret_cast<int*>(sm.words + (size_t)chunk * 32);  // [nch][W][32]
  // the pairs below the range: one row of nbp bytes (zero past nb)
  int lower = 0;
  const uint8_t* brow = m.below + (size_t)range * nbp;
  for (int i = threadIdx.x * 16; i < nbp; i += W * 32 * 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(brow + i);
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int by = 0; by < 4; ++by)
        if (i + 4 * j + by < nb) lower += (q[j] >> (8 * by)) & 0xFFu;
  }
  lower = __reduce_add_sync(kFull, lower);
  if (lane == 0) sm.base[warp] = lower;
  // pass 1: expert e's pairs in this warp's share of each chunk
  for (int ci = 0; ci < nch; ++ci) {
    const int c0 = ci * chunk, c1 = min(nb, c0 + chunk);
    stage_map<W>(rmap, c0, c1, sm.words);
    const int per = (c1 - c0 + W - 1) / W, b0 = min(c1, c0 + warp * per), b1 = min(c1, b0 + per);
    int c = 0;
    for (int b = b0; b < b1; ++b) c += __popc(~sm.words[(b - c0) * 32 + lane] & 0x80808080u);
    ccnt[(ci * W + warp) * 32 + lane] = c;
  }
  __syncthreads();
  if (warp == 0) {
    int tot = 0, base = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) base += sm.base[w];
    for (int i = 0; i < nch * W; ++i) tot += ccnt[i * 32 + lane];
    int inc = tot;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, d);
      if (lane >= d) inc += y;
    }
    int run = base + inc - tot;  // offsets[e]
    if (e < m.E) m.offsets[e] = run;
    if (e == m.E - 1) m.offsets[m.E] = run + tot;
    for (int i = 0; i < nch * W; ++i) {  // (chunk, warp) order = token order
      const int v = ccnt[i * 32 + lane];
      ccnt[i * 32 + lane] = run;
      run += v;
    }
  }
  __syncthreads();
  // pass 2: expert e's pairs in this warp's share of each chunk, in token order (the
  // starts are known, so the chunk still staged goes first)
  for (int k = 0; k < nch; ++k) {
    const int ci = nch - 1 - k;
    const int c0 = ci * chunk, c1 = min(nb, c0 + chunk);
    if (k > 0) stage_map<W>(rmap, c0, c1, sm.words);
    const int per = (c1 - c0 + W - 1) / W, b0 = min(c1, c0 + warp * per), b1 = min(c1, b0 + per);
    int pos = ccnt[(ci * W + warp) * 32 + lane];
    for (int b = b0; b < b1; ++b) {
      const uint32_t wv = sm.words[(b - c0) * 32 + lane];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t slot = (wv >> (8 * i)) & 0xFFu;
        if (slot != 0xFFu) m.pairs[pos++] = (4 * b + i) * m.K + (int)slot;
      }
    }
  }
}

}  // namespace lists_impl
}  // namespace moe
