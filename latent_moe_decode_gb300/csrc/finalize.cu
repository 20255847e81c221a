// Finalize: the routing-weighted top-K sum of the experts' rows.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, class
// Finalize (out[t] = sum_k w[t,k] * rows[16t+k], FP32, k in order, fma, one BF16
// rounding; every row load of a thread in flight before the math), and
// vllm.models.glm5next.nvidia.specialized_decode.cutedsl.finalize_publish,
// _QuadFinalizePublishDeviceKernel (weights BF16 or FP32, times routed_scaling_factor
// when it is not 1, zero for a -1 permuted index whose row is skipped; the
// shared-expert row added once in FP32 after all k).
//
// GB300 design: a pure HBM stream (T*K rows of H BF16 in, T rows out). The unit of
// work is one 16-byte fragment (8 columns) of one token, numbered flat over (token,
// fragment) so that a warp covers 512 contiguous bytes of each row. The grid is
// persistent (as many CTAs as fit: three per SM at K = 16) and thread i of the grid
// takes the fragments i, i + G, i + 2G, ... (G threads in the grid). Each thread runs
// its own ring of kStages shared-memory stages: it issues the asynchronous 16-byte
// copies (cp.async, bypassing L1, evict-first in L2) of all K row fragments of the
// next item, and loads that item's K weights into registers, before it waits for and
// sums the current one (FP32 fma chain in k order, one 16-byte store). HBM thus always
// has the next items in flight and the stream does not drain between waves of CTAs;
// the weights, loaded one item ahead, never add their latency to an item. Slots are private to their thread ([stage][k]
// [thread]: conflict-free), so no CTA barrier is needed. Two stages and three CTAs per
// SM keep more bytes in flight than three stages and two CTAs (the shared memory of
// an SM holds six items either way).
// When the rows are an input complete before the preceding kernel started (the
// one-call step: the preceding kernels make only the weights), the first two items'
// row copies are issued before griddepcontrol.wait and their weights are read after
// it, so the first 30 MB of rows stream in while the preceding kernel finishes.
#include <type_traits>

#include "lists.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;

struct FinArgs {
  const uint16_t* rows;
  long long n_rows;
  const int32_t* row_index;  // [T, K] or nullptr
  const void* weights;       // [T, K] FP32 or BF16
  const uint16_t* shared;    // [T, H] or nullptr
  float scale;
  int T, K, H;
  uint16_t* out;
  uint32_t* err;
  // 1: wait for the preceding kernel before reading anything; 0: the rows (and the
  // shared rows) were complete before the preceding kernel started, so the first row
  // copies are issued before the wait, and the weights (and indices) after it
  int wait_all;
  // LISTS instantiations: the first n_list CTAs build the routing lists from the
  // routing CTAs' slot map (one 32-expert range each) instead of summing rows
  lists_impl::MapArgs lm;
  int n_list;
  int map_chunk;  // blocks of the slot map a lists CTA stages at a time
  // GATHER: each lane takes `group` consecutive 32-fragment runs of one token in turn
  // (its row indices and weights then load once per group); 1 when the fragments of a
  // token are not a multiple of 32 * group
  int group;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kStages = 2;

// The lists role of a LISTS launch, kept out of line: inlined, its code changed how the
// compiler scheduled Finalize's loop (more registers), which cost the row stream 7 us
// at T = 1020.
__device__ __noinline__ void build_lists(const lists_impl::MapArgs& m, int range, uint4* smem, int chunk) {
  lists_impl::lists_from_map<kThreads / 32>(m, range, *reinterpret_cast<lists_impl::MapSmem<kThreads / 32>*>(smem),
                                            chunk);
}

// KT: compile-time K (0 = runtime K, up to MOE_MAX_TOPK). LISTS: the launch also builds
// the routing lists (the one-call step): its first a.n_list CTAs do that, beside the
// row stream, and the others run Finalize.
template <int KT, bool GATHER, bool BF16W, bool SHARED, bool LISTS = false>
__global__ void __launch_bounds__(kThreads) finalize_kernel(const FinArgs a) {
  extern __shared__ __align__(16) uint4 slots[];  // [kStages][K (+1 shared)][kThreads]
  int cta = (int)blockIdx.x, ncta = (int)gridDim.x;
  if constexpr (LISTS) {
    if (cta < a.n_list) {
      grid_launch_dependents();
      grid_wait();  // the slot map comes from the preceding kernel
      build_lists(a.lm, cta, slots, a.map_chunk);
      return;
    }
    cta -= a.n_list;
    ncta -= a.n_list;
  }
  constexpr int KM = KT ? KT : MOE_MAX_TOPK;
  const int K = KT ? KT : a.K;
  const int frags = a.H >> 3;
  const long long total = (long long)a.T * frags;
  const long long stride = (long long)ncta * kThreads;
  const long long f0 = (long long)cta * kThreads + threadIdx.x;
  const size_t H = (size_t)a.H;
  grid_launch_dependents();
  // indices choose the rows to copy: with a gather, everything waits
  const bool early = !a.wait_all && !GATHER;
  if (!early && threadIdx.x < 32) {
    // The CTA's first fragments (at most two tokens' worth): the row
    // spans (without a gather), the shared-row spans, and the tokens' indices and weights
    // are asked of L2 before the wait, so their DRAM fetch overlaps the preceding
    // kernel's end (hints only: nothing is read into registers or shared memory).
    const int lane = threadIdx.x;
    const long long span = GATHER ? (long long)kThreads * a.group : kThreads;  // the CTA's first fragments
    const long long lo = (long long)cta * span, hi = min(lo + span, total);
    for (long long f = lo; f < hi;) {
      const int t = (int)(f / frags);
      const long long end = min(hi, (long long)(t + 1) * frags);
      const size_t col = (size_t)(f - (long long)t * frags) * 8;
      const uint32_t bytes = (uint32_t)(end - f) * 16u;
      if (!GATHER)
        for (int k = lane; k < K; k += 32) prefetch_l2(a.rows + ((size_t)t * K + k) * a.H + col, bytes);
      if (SHARED && lane == 0) prefetch_l2(a.shared + (size_t)t * a.H + col, bytes);
      if (GATHER && lane == 1) asm volatile("prefetch.global.L2 [%0];" ::"l"(a.row_index + (size_t)t * K));
      if (lane == 2) asm volatile("prefetch.global.L2 [%0];" ::"l"(static_cast<const char*>(a.weights) + (size_t)t * K * (BF16W ? 2 : 4)));
      f = end;
    }
  }
  if (!early) grid_wait();
  const uint64_t pol = policy_evict_first();
  const uint32_t base = smem_u32(slots) + threadIdx.x * 16u;
  const int SL = K + (SHARED ? 1 : 0);  // slots per stage: K rows, then the shared row
  const uint32_t stage_bytes = (uint32_t)SL * kThreads * 16u;

  // Copies of fragment fi's K row fragments (and its shared-row fragment) into stage
  // st, as one commit group (empty past the end), and, with weights, its K raw weights
  // into wraw[st]; returns the mask of rows not skipped.
  using WRaw = typename std::conditional<BF16W, uint16_t, float>::type;
  WRaw wraw[kStages][KM];
  // GATHER: the row indices and raw weights of the token last issued (a lane's next
  // items are of the same token while its group lasts)
  int ctok = -1;
  int cidx[GATHER ? KM : 1];  // (a row index is an int32; -1 for a skipped or out-of-range one)
  WRaw cw[GATHER ? KM : 1];
  auto issue = [&](int st, long long fi, bool weights) -> uint32_t {
    uint32_t m = 0;
    if (fi < total) {
      const int t = (int)(fi / frags);
      const int col = (int)(fi - (long long)t * frags) * 8;
      if constexpr (GATHER) {
        if (t != ctok) {
          ctok = t;
#pragma unroll
          for (int k = 0; k < KM; ++k) {
            if (KT || k < K) {
              const size_t ix = (size_t)t * K + k;
              int r = __ldg(a.row_index + ix);
              if (r < -1 || (long long)r >= a.n_rows) {
                set_error(a.err, MOE_DEVERR_ROW_INDEX);
                r = -1;
              }
              cidx[k] = r;
              cw[k] = __ldg(static_cast<const WRaw*>(a.weights) + ix);
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < KM; ++k) {
        if (KT || k < K) {
          const size_t ix = (size_t)t * K + k;
          const long long r = GATHER ? cidx[GATHER ? k : 0] : (long long)ix;
          if (weights) wraw[st][k] = GATHER ? cw[GATHER ? k : 0] : __ldg(static_cast<const WRaw*>(a.weights) + ix);
          if (r != -1) {
            m |= 1u << k;
            cp_async16(base + (uint32_t)st * stage_bytes + (uint32_t)(k * kThreads * 16), a.rows + (size_t)r * H + col,
                       pol);
          }
        }
      }
      if (SHARED)
        cp_async16(base + (uint32_t)st * stage_bytes + (uint32_t)(K * kThreads * 16), a.shared + (size_t)t * H + col, pol);
    }
    cp_async_commit();
    return m;
  };
  auto load_weights = [&](int st, long long fi) {
    if (fi < total) {
      const int t = (int)(fi / frags);
#pragma unroll
      for (int k = 0; k < KM; ++k)
        if (KT || k < K) wraw[st][k] = __ldg(static_cast<const WRaw*>(a.weights) + (size_t)t * K + k);
    }
  };

  // Each iteration issues the item one ahead, then waits for and sums the current one.
  // When the rows are ready early, the first two items' rows are issued before the
  // wait (the first iteration then issues nothing) and their weights read after it.
  uint32_t mask[kStages];
  static_assert(kStages == 2, "the early prologue issues exactly the first two items");
  if (early) {
    mask[0] = issue(0, f0, false);
    mask[1] = issue(1, f0 + stride, false);
    grid_wait();  // the weights may come from the preceding kernel
    load_weights(0, f0);
    load_weights(1, f0 + stride);
  } else if constexpr (!GATHER) {
    mask[0] = issue(0, f0, true);
  } else {  // the first item of the gather order below: run 0 of group 0
    mask[0] = issue(0, ((long long)cta * (kThreads / 32) + (threadIdx.x >> 5)) * 32LL * a.group + (threadIdx.x & 31), true);
  }
  // sum item fi (waiting for its stage s) and store its 8 outputs
  auto consume = [&](int s, long long fi) {
    const int t = (int)(fi / frags);
    const int col = (int)(fi - (long long)t * frags) * 8;
    // the weights, loaded at issue, times routed_scaling_factor
    float w[KM];
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      float wk = 0.0f;
      if (KT || k < K) {
        if constexpr (BF16W) wk = bf16_to_f32(wraw[s][k]); else wk = wraw[s][k];
        if (a.scale != 1.0f) wk = __fmul_rn(wk, a.scale);
      }
      w[k] = wk;
    }
    cp_async_wait<kStages - 1>();
    // FP32 fma over k in order
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    const uint4* sl = slots + (size_t)s * SL * kThreads + threadIdx.x;
#pragma unroll
    for (int k = 0; k < KM; ++k) {
      if (!((mask[s] >> k) & 1u)) continue;
      const uint4 v = sl[k * kThreads];
      const uint32_t q4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __fmaf_rn(w[k], bf16_lo(q4[q]), acc[2 * q]);
        acc[2 * q + 1] = __fmaf_rn(w[k], bf16_hi(q4[q]), acc[2 * q + 1]);
      }
    }
    if (SHARED) {
      const uint4 sh = sl[K * kThreads];
      const uint32_t q4[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        acc[2 * q] = __fadd_rn(acc[2 * q], bf16_lo(q4[q]));
        acc[2 * q + 1] = __fadd_rn(acc[2 * q + 1], bf16_hi(q4[q]));
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    st16(a.out + (size_t)t * H + col, o);
  };
  bool ahead = early;  // the item one ahead is already issued
  if constexpr (!GATHER) {
    for (long long f = f0; f < total; f += kStages * stride) {
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        const long long fi = f + s * stride;
        constexpr int kAhead = kStages - 1;
        const int sn = (s + kAhead) % kStages;
        if (!ahead) mask[sn] = issue(sn, fi + kAhead * stride, true);
        ahead = false;
        if (fi >= total) break;
        consume(s, fi);
      }
    }
  } else {
    // item q of this lane: run (q mod group) of its warp's group number q / group, each
    // group 32 * group consecutive fragments of one token (one warp: 512 contiguous bytes
    // of every row per item)
    const long long wg = (long long)cta * (kThreads / 32) + (threadIdx.x >> 5), wtot = (long long)ncta * (kThreads / 32);
    const int lane = threadIdx.x & 31, R = a.group;
    auto item = [&](long long q) { return (wg + (q / R) * wtot) * 32LL * R + lane + 32LL * (q % R); };
    for (long long q = 0;; q += kStages) {
      bool end = false;
#pragma unroll
      for (int s = 0; s < kStages; ++s) {
        const long long fi = item(q + s);
        constexpr int kAhead = kStages - 1;
        const int sn = (s + kAhead) % kStages;
        mask[sn] = issue(sn, item(q + s + kAhead), true);
        if (fi >= total) {
          end = true;
          break;
        }
        consume(s, fi);
      }
      if (end) break;
    }
  }
  cp_async_wait<0>();
}

template <int KT, bool G, bool B, bool S, bool LISTS = false>
int launch_one(FinArgs a, int sm_count, cudaStream_t s) {
  size_t smem = (size_t)kStages * ((KT ? KT : a.K) + (S ? 1 : 0)) * kThreads * 16;
  if (LISTS) {
    // the lists CTAs stage their range's map in the shared memory Finalize's stages
    // use: all of it when it fits (one round trip), else chunks of what fits
    a.map_chunk = lists_impl::map_chunk_for<kThreads / 32>((a.T + 3) / 4, smem);
    if (a.map_chunk < 1) return MOE_ERR_CAPACITY;
  }
  auto kern = finalize_kernel<KT, G, B, S, LISTS>;
  // (the limit is the instantiation's largest need, the same for every call: calls from
  // several host threads never lower it under one another)
  constexpr size_t most = (size_t)kStages * ((KT ? KT : MOE_MAX_TOPK) + (S ? 1 : 0)) * kThreads * 16;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most) != cudaSuccess)
    return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm < 1)
    return MOE_ERR_CUDA;
  const long long threads = (long long)a.T * (a.H / 8);
  const long long need = (threads + kThreads - 1) / kThreads;
  // persistent: every CTA resident at once (the list CTAs included). A LISTS launch
  // follows the top-K launch closely (programmatic dependent launch): its CTAs are placed
  // while some top-K CTAs still hold room on their SMs, and a CTA that found no room
  // then started only when another CTA of this launch ended -- a full share late. So it
  // leaves a fifth of the SM count in slots unclaimed (measured at T = 1020: 44.1 us a
  // step against 48.3 with every slot taken and 46.2 with Finalize launched only after
  // the top-K CTAs end; 16 and 32 unclaimed slots measured the same, at T = 256, 1020
  // and 4096).
  long long room = (long long)sm_count * per_sm - (LISTS ? a.n_list + sm_count / 5 : 0);
  if (room < 1) room = 1;
  const long long grid = (need < room ? need : room) + (LISTS ? a.n_list : 0);
  return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, a);
}

template <int KT>
int launch_variant(const FinArgs& a, bool gather, bool bf16w, bool shared, int sm_count, cudaStream_t s) {
#define MOE_FIN_CASE(G, B, S) \
  if (gather == G && bf16w == B && shared == S) return launch_one<KT, G, B, S>(a, sm_count, s);
  MOE_FIN_CASE(false, false, false)
  MOE_FIN_CASE(false, false, true)
  MOE_FIN_CASE(false, true, false)
  MOE_FIN_CASE(false, true, true)
  MOE_FIN_CASE(true, false, false)
  MOE_FIN_CASE(true, false, true)
  MOE_FIN_CASE(true, true, false)
  MOE_FIN_CASE(true, true, true)
#undef MOE_FIN_CASE
  return MOE_ERR_INVALID_ARGUMENT;
}

}  // namespace
}  // namespace moe

namespace moe {

int finalize(const uint16_t* rows, int64_t n_rows, const int32_t* row_index, const void* weights, int weights_dtype,
             const uint16_t* shared, float routed_scaling_factor, int T, int K, int H, uint16_t* out,
             bool rows_ready, cudaStream_t s) {
  if (T < 0 || K < 1 || K > MOE_MAX_TOPK || H < 8 || H % 8 != 0 || n_rows < 0)
    return MOE_ERR_INVALID_ARGUMENT;
  if (weights_dtype != MOE_DTYPE_F32 && weights_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARGUMENT;
  if ((long long)T * (H / 8) > (1LL << 31) * (long long)kThreads - 1) return MOE_ERR_CAPACITY;
  if (T == 0) return MOE_OK;
  if (!rows || !weights || !out) return MOE_ERR_INVALID_ARGUMENT;
  if (!row_index && n_rows < (long long)T * K) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(rows, 16) || !aligned(out, 16) || (shared && !aligned(shared, 16))) return MOE_ERR_ALIGNMENT;
  if (!aligned(weights, weights_dtype == MOE_DTYPE_F32 ? 4 : 2) || (row_index && !aligned(row_index, 4)))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;

  FinArgs a{rows, (long long)n_rows, row_index, weights, shared, routed_scaling_factor, T, K, H, out, dev.error_word,
            rows_ready ? 0 : 1};
  const bool gather = row_index != nullptr, bf16w = weights_dtype == MOE_DTYPE_BF16, sh = shared != nullptr;
  const int frags = H / 8;
  a.group = frags % 128 == 0 ? 4 : (frags % 64 == 0 ? 2 : 1);
  if (K == 16) return launch_variant<16>(a, gather, bf16w, sh, dev.sm_count, s);
  if (K == 8) return launch_variant<8>(a, gather, bf16w, sh, dev.sm_count, s);
  return launch_variant<0>(a, gather, bf16w, sh, dev.sm_count, s);
}

// Whether the lists CTAs of finalize_with_lists have room for a range's map in chunks
// (with their per-chunk counts) in the shared memory of Finalize's stages: T up to
// 65280 at K = 16, 16256 at K = 8.
bool finalize_lists_fit(int T, int K) {
  if (T < 1 || K < 1 || K > MOE_MAX_TOPK) return false;
  const size_t smem = (size_t)kStages * K * kThreads * 16;
  return lists_impl::map_chunk_for<kThreads / 32>((T + 3) / 4, smem) >= 1;
}

// Finalize of the one-call step (rows t*K + k, BF16 weights; rows ready before the
// preceding kernel started) with the routing lists built by the same launch from the
// routing CTAs' slot map.
int finalize_with_lists(const uint16_t* rows, const uint16_t* weights_bf16, int T, int K, int H, uint16_t* out,
                        const uint32_t* smap, const uint8_t* below, int E, int32_t* offsets, int32_t* pairs,
                        cudaStream_t s) {
  if (T < 1 || K < 1 || K > MOE_MAX_TOPK || H < 8 || H % 8 != 0 || E < 1 || E > MOE_MAX_EXPERTS)
    return MOE_ERR_INVALID_ARGUMENT;
  if ((long long)T * K > (1LL << 31) - 1 || (long long)T * (H / 8) > (1LL << 31) * (long long)kThreads - 1)
    return MOE_ERR_CAPACITY;
  if (!rows || !weights_bf16 || !out || !smap || !below || !offsets || !pairs) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(rows, 16) || !aligned(out, 16) || !aligned(weights_bf16, 2) || !aligned(smap, 4) || !aligned(below, 16) ||
      !aligned(offsets, 4) || !aligned(pairs, 4))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;
  FinArgs a{rows, (long long)T * K, nullptr, weights_bf16, nullptr, 1.0f, T, K, H, out, dev.error_word, 0};
  a.lm = lists_impl::MapArgs{smap, below, T, K, E, offsets, pairs};
  a.n_list = (E + lists_impl::kMaxEpc - 1) / lists_impl::kMaxEpc;
  if (K == 16) return launch_one<16, false, true, false, true>(a, dev.sm_count, s);
  if (K == 8) return launch_one<8, false, true, false, true>(a, dev.sm_count, s);
  return launch_one<0, false, true, false, true>(a, dev.sm_count, s);
}

}  // namespace moe

extern "C" int moe_finalize(const uint16_t* rows, int64_t n_rows, const int32_t* row_index,
                            const void* weights, int weights_dtype, const uint16_t* shared,
                            float routed_scaling_factor, int T, int K, int H, uint16_t* out,
                            moe_stream_t stream) {
  return moe::finalize(rows, n_rows, row_index, weights, weights_dtype, shared, routed_scaling_factor, T, K, H, out,
                       false, moe::as_cuda(stream));
}
