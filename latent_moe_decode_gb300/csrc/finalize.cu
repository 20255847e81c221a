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
// GB300 design: a pure HBM stream (T*K rows of H BF16 in, T rows out). One thread owns
// one 16-byte fragment (8 columns) of one token; the grid is flat over (token,
// fragment), so a warp covers 512 contiguous bytes of each row. The thread issues the
// asynchronous 16-byte copies (cp.async, bypassing L1, evict-first in L2) of all of its
// K row fragments into its own shared-memory slots before it touches any of them, so
// all K loads are in flight at once whatever registers the compiler allocates
// (16 x 16 B per thread, ~220 KB per SM at 7 CTAs of 128 threads). It loads the
// weights while they fly, waits for its own copies only, then runs the FP32 fma chain
// in k order from shared memory (slot [k][thread]: conflict-free) and stores 16 bytes.
#include "common.cuh"

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
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// KT: compile-time K (0 = runtime K, up to MOE_MAX_TOPK).
template <int KT, bool GATHER, bool BF16W, bool SHARED>
__global__ void __launch_bounds__(kThreads) finalize_kernel(const FinArgs a) {
  extern __shared__ __align__(16) uint4 slots[];  // [K][kThreads]
  constexpr int KM = KT ? KT : MOE_MAX_TOPK;
  const int K = KT ? KT : a.K;
  const int frags = a.H >> 3;
  const long long f = (long long)blockIdx.x * kThreads + threadIdx.x;
  grid_launch_dependents();
  grid_wait();  // rows, weights and indices may come from the preceding kernel
  if (f >= (long long)a.T * frags) return;
  const int t = (int)(f / frags);
  const int col = (int)(f - (long long)t * frags) * 8;
  const size_t H = (size_t)a.H;
  const uint64_t pol = policy_evict_first();
  const uint32_t base = smem_u32(slots) + threadIdx.x * 16u;

  // 1) every row copy in flight
  bool use[KM];
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    use[k] = false;
    if (KT || k < K) {
      const size_t ix = (size_t)t * K + k;
      long long r = GATHER ? (long long)__ldg(a.row_index + ix) : (long long)ix;
      if (GATHER && (r < -1 || r >= a.n_rows)) {
        set_error(a.err, MOE_DEVERR_ROW_INDEX);
        r = -1;
      }
      use[k] = r != -1;
      if (use[k]) cp_async16(base + (uint32_t)(k * kThreads * 16), a.rows + (size_t)r * H + col, pol);
    }
  }
  uint4 sh = make_uint4(0, 0, 0, 0);
  if (SHARED) sh = ld_stream16(a.shared + (size_t)t * H + col, pol);
  // 2) the weights while the rows fly
  float w[KM];
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    float wk = 0.0f;
    if (KT || k < K) {
      const size_t ix = (size_t)t * K + k;
      wk = BF16W ? bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.weights) + ix))
                 : __ldg(static_cast<const float*>(a.weights) + ix);
      if (a.scale != 1.0f) wk = __fmul_rn(wk, a.scale);
    }
    w[k] = wk;
  }
  cp_async_wait_all();
  // 3) FP32 fma over k in order
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    if (!use[k]) continue;
    const uint4 v = slots[k * kThreads + threadIdx.x];
    const uint32_t q4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] = __fmaf_rn(w[k], bf16_lo(q4[q]), acc[2 * q]);
      acc[2 * q + 1] = __fmaf_rn(w[k], bf16_hi(q4[q]), acc[2 * q + 1]);
    }
  }
  if (SHARED) {
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
}

template <int KT, bool G, bool B, bool S>
int launch_one(const FinArgs& a, cudaStream_t s) {
  const size_t smem = (size_t)(KT ? KT : a.K) * kThreads * 16;
  auto kern = finalize_kernel<KT, G, B, S>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return MOE_ERR_CUDA;
  const long long threads = (long long)a.T * (a.H / 8);
  return launch_pdl(kern, dim3((unsigned)((threads + kThreads - 1) / kThreads)), dim3(kThreads), smem, s, a);
}

template <int KT>
int launch_variant(const FinArgs& a, bool gather, bool bf16w, bool shared, cudaStream_t s) {
#define MOE_FIN_CASE(G, B, S) \
  if (gather == G && bf16w == B && shared == S) return launch_one<KT, G, B, S>(a, s);
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

  FinArgs a{rows, (long long)n_rows, row_index, weights, shared, routed_scaling_factor, T, K, H, out, dev.error_word};
  const bool gather = row_index != nullptr, bf16w = weights_dtype == MOE_DTYPE_BF16, sh = shared != nullptr;
  cudaStream_t s = as_cuda(stream);
  if (K == 16) return launch_variant<16>(a, gather, bf16w, sh, s);
  if (K == 8) return launch_variant<8>(a, gather, bf16w, sh, s);
  return launch_variant<0>(a, gather, bf16w, sh, s);
}
