// Finalize: the routing-weighted top-K sum of the experts' rows.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, class
// Finalize (out[t] = sum_k w[t,k] * rows[16t+k], FP32, k in order, fma, one BF16
// rounding; every row load of a thread in flight before the math), and
// vllm.models.glm5next.nvidia.specialized_decode.cutedsl.finalize_publish,
// _QuadFinalizePublishDeviceKernel (the token's indices and weights staged first;
// weights BF16 or FP32, times routed_scaling_factor when it is not 1, zero for a -1
// permuted index whose row is skipped; the shared-expert row added once in FP32 after
// all k).
//
// GB300 design: a pure HBM stream (T*K rows of H BF16 in, T rows out), run as a
// persistent, pipelined kernel. An item is one token's 64-fragment (512-column)
// segment. In each CTA a producer warp walks the CTA's items: lane k reads row index k
// (and applies the -1 / range test) and issues the bulk (TMA) copy of that 1 KB row
// segment into a 4-stage shared-memory ring, all completing on the stage's full
// mbarrier; so up to 4 items' rows (68 KB for K = 16) are in flight per CTA and ~200
// KB per SM, independent of how the compiler schedules registers. Two consumer warps
// (one thread per 16-byte fragment) load the item's weights while its copies fly, wait
// on the full barrier, read their fragment of every row from shared memory (row-major
// by k: conflict-free), run the FP32 fma chain in k order, store 16 bytes, and release
// the stage on its empty barrier. Row copies are marked evict-first in L2; every wait
// is bounded.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kCF = 64;                   // fragments (8 columns) per item: one per consumer thread
constexpr int kConsumerWarps = kCF / 32;  // 2
constexpr int kThreads = 32 + kCF;        // producer warp + consumers
constexpr int kStages = 4;

struct FinArgs {
  const uint16_t* rows;
  long long n_rows;
  const int32_t* row_index;  // [T, K] or nullptr
  const void* weights;       // [T, K] FP32 or BF16
  const uint16_t* shared;    // [T, H] or nullptr
  float scale;
  int T, K, H;
  int cpt;  // items per token
  uint16_t* out;
  uint32_t* err;
};

size_t smem_bytes(int K, bool shared) {
  return kStages * (size_t)(K + (shared ? 1 : 0)) * kCF * 16 + 2 * kStages * 8 + (size_t)kStages * MOE_MAX_TOPK * 8;
}

// KT: compile-time K (0 = runtime K).
template <int KT, bool GATHER, bool BF16W, bool SHARED>
__global__ void __launch_bounds__(kThreads) finalize_kernel(const FinArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int K = KT ? KT : a.K;
  const uint32_t sbytes = (uint32_t)((K + (SHARED ? 1 : 0)) * kCF * 16);
  const uint32_t ring = smem_u32(smem);
  const uint32_t bars = ring + kStages * sbytes;  // full[kStages], empty[kStages]
  long long* s_row = reinterpret_cast<long long*>(smem + kStages * sbytes + 2 * kStages * 8);  // [kStages][32]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int frags = a.H >> 3;
  const long long n_items = (long long)a.T * a.cpt;
  const size_t H = (size_t)a.H;

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(bars + 8u * st, 1);                           // full: the producer's arrive + the bytes
      mbar_init(bars + 8u * (kStages + st), kConsumerWarps);  // empty: one arrive per consumer warp
    }
    mbar_fence_init();
  }
  __syncthreads();  // barriers initialised before any wait
  grid_launch_dependents();
  grid_wait();  // rows, weights and indices may come from the preceding kernel

  if (warp == 0) {  // producer
    const uint64_t pol = policy_evict_first();
    long long j = 0;
    for (long long i = blockIdx.x; i < n_items; i += gridDim.x, ++j) {
      const int st = (int)(j % kStages);
      const uint32_t ph = (uint32_t)(j / kStages) & 1u;
      if (!mbar_wait(bars + 8u * (kStages + st), ph ^ 1u, a.err)) break;
      const int t = (int)(i / a.cpt);
      const int f0 = (int)(i - (long long)t * a.cpt) * kCF;
      const uint32_t bytes = (uint32_t)min(kCF, frags - f0) * 16u;
      long long r = -1;
      if (lane < K) {
        const size_t ix = (size_t)t * K + lane;
        r = GATHER ? (long long)__ldg(a.row_index + ix) : (long long)ix;
        if (GATHER && (r < -1 || r >= a.n_rows)) {
          set_error(a.err, MOE_DEVERR_ROW_INDEX);
          r = -1;
        }
        s_row[st * MOE_MAX_TOPK + lane] = r;
      }
      const uint32_t used = (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, lane < K && r != -1)) + (SHARED ? 1u : 0u);
      __syncwarp();  // the indices are written before the arrive that publishes them
      const uint32_t full = bars + 8u * st, dst = ring + (uint32_t)st * sbytes;
      if (lane == 0) mbar_expect_tx(full, used * bytes);
      __syncwarp();
      if (lane < K && r != -1)
        bulk_g2s(dst + (uint32_t)(lane * kCF * 16), a.rows + (size_t)r * H + (size_t)f0 * 8, bytes, full, pol);
      if (SHARED && lane == 0)
        bulk_g2s(dst + (uint32_t)(K * kCF * 16), a.shared + (size_t)t * H + (size_t)f0 * 8, bytes, full, pol);
    }
    return;
  }

  // consumers
  const int c = tid - 32;
  long long j = 0;
  for (long long i = blockIdx.x; i < n_items; i += gridDim.x, ++j) {
    const int st = (int)(j % kStages);
    const uint32_t ph = (uint32_t)(j / kStages) & 1u;
    const int t = (int)(i / a.cpt);
    const int f0 = (int)(i - (long long)t * a.cpt) * kCF;
    const int nf = min(kCF, frags - f0);
    // the item's weights, loaded while its rows are in flight
    float w[KT ? KT : MOE_MAX_TOPK];
#pragma unroll
    for (int k = 0; k < (KT ? KT : MOE_MAX_TOPK); ++k) {
      float wk = 0.0f;
      if (KT || k < K) {
        const size_t ix = (size_t)t * K + k;
        wk = BF16W ? bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.weights) + ix))
                   : __ldg(static_cast<const float*>(a.weights) + ix);
        if (a.scale != 1.0f) wk = __fmul_rn(wk, a.scale);
      }
      w[k] = wk;
    }
    if (!mbar_wait(bars + 8u * st, ph, a.err)) break;
    if (c < nf) {
      const uint4* frag = reinterpret_cast<const uint4*>(smem + (size_t)st * sbytes) + c;
      const long long* rs = s_row + st * MOE_MAX_TOPK;
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
      for (int k = 0; k < (KT ? KT : MOE_MAX_TOPK); ++k) {
        if (!KT && k >= K) break;
        if (rs[k] == -1) continue;
        const uint4 v = frag[k * kCF];
        const uint32_t q4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = __fmaf_rn(w[k], bf16_lo(q4[q]), acc[2 * q]);
          acc[2 * q + 1] = __fmaf_rn(w[k], bf16_hi(q4[q]), acc[2 * q + 1]);
        }
      }
      if (SHARED) {
        const uint4 v = frag[K * kCF];
        const uint32_t q4[4] = {v.x, v.y, v.z, v.w};
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
      st16(a.out + (size_t)t * H + (size_t)(f0 + c) * 8, o);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8u * (kStages + st));
  }
}

template <int KT, bool G, bool B, bool S>
int launch_one(const FinArgs& a, int sm_count, cudaStream_t s) {
  const size_t smem = smem_bytes(a.K, S);
  auto kern = finalize_kernel<KT, G, B, S>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm < 1)
    return MOE_ERR_CUDA;
  const long long items = (long long)a.T * a.cpt;
  const long long want = (long long)sm_count * per_sm;
  const unsigned grid = (unsigned)(items < want ? items : want);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
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

extern "C" int moe_finalize(const uint16_t* rows, int64_t n_rows, const int32_t* row_index,
                            const void* weights, int weights_dtype, const uint16_t* shared,
                            float routed_scaling_factor, int T, int K, int H, uint16_t* out,
                            moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || K < 1 || K > MOE_MAX_TOPK || H < 8 || H % 8 != 0 || n_rows < 0)
    return MOE_ERR_INVALID_ARGUMENT;
  if (weights_dtype != MOE_DTYPE_F32 && weights_dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARGUMENT;
  const int cpt = (H / 8 + kCF - 1) / kCF;
  if ((long long)T * cpt > (1LL << 40)) return MOE_ERR_CAPACITY;
  if (T == 0) return MOE_OK;
  if (!rows || !weights || !out) return MOE_ERR_INVALID_ARGUMENT;
  if (!row_index && n_rows < (long long)T * K) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned(rows, 16) || !aligned(out, 16) || (shared && !aligned(shared, 16))) return MOE_ERR_ALIGNMENT;
  if (!aligned(weights, weights_dtype == MOE_DTYPE_F32 ? 4 : 2) || (row_index && !aligned(row_index, 4)))
    return MOE_ERR_ALIGNMENT;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != MOE_OK) return st;

  FinArgs a{rows, (long long)n_rows, row_index, weights, shared, routed_scaling_factor, T, K, H, cpt, out, dev.error_word};
  const bool gather = row_index != nullptr, bf16w = weights_dtype == MOE_DTYPE_BF16, sh = shared != nullptr;
  cudaStream_t s = as_cuda(stream);
  if (K == 16) return launch_variant<16>(a, gather, bf16w, sh, dev.sm_count, s);
  if (K == 8) return launch_variant<8>(a, gather, bf16w, sh, dev.sm_count, s);
  return launch_variant<0>(a, gather, bf16w, sh, dev.sm_count, s);
}
