// Finalize: the routing-weighted top-K sum of the experts' rows.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide, class
// Finalize (out[t] = sum_k w[t,k] * rows[16t+k], FP32, k in order, fma, one BF16
// rounding; every row load of a thread in flight before the math), and
// vllm.models.glm5next.nvidia.specialized_decode.cutedsl.finalize_publish,
// _QuadFinalizePublishDeviceKernel (weights BF16 or FP32, times routed_scaling_factor
// when it is not 1, -1 permuted indices skipped, the shared-expert row added once in
// FP32 after all k).
//
// GB300 design: the kernel is a pure HBM stream (T*K rows of H BF16 in, T rows out).
// One thread owns 8 consecutive columns (one 16-byte fragment) of one token and issues
// the 16-byte loads of all of its K rows (a chunk of up to 16) before its first FMA,
// so each thread keeps up to 256 bytes in flight. The grid is flat over
// (token, fragment): a warp reads 512 contiguous bytes of a row per load instruction.
// Row loads are marked read-once (no L1 allocation, evict-first in L2).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kFinThreads = 128;

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

// KC: loads in flight per chunk. EXACT: K == KC (one chunk, no bounds on k).
template <int KC, bool EXACT, bool GATHER, bool BF16W, bool SHARED>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(const FinArgs a) {
  const int frags = a.H >> 3;
  const long long f = (long long)blockIdx.x * kFinThreads + threadIdx.x;
  grid_launch_dependents();
  grid_wait();  // rows, weights and indices may come from the preceding kernel
  if (f >= (long long)a.T * frags) return;
  const int t = (int)(f / frags);
  const int col = (int)(f - (long long)t * frags) * 8;
  const uint64_t pol = policy_evict_first();
  const size_t H = (size_t)a.H;

  uint4 sh = make_uint4(0, 0, 0, 0);
  if (SHARED) sh = ld_stream16(a.shared + (size_t)t * H + col, pol);

  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;

  const int K = EXACT ? KC : a.K;
  for (int k0 = 0; k0 < K; k0 += KC) {
    uint4 v[KC];
    bool use[KC];
    // 1) every row load of the chunk in flight first
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      const int k = k0 + i;
      const bool in = EXACT || k < K;
      long long r = (long long)t * K + k;
      if (GATHER) {
        r = in ? (long long)__ldg(a.row_index + (size_t)t * K + k) : -1;
        if (r < -1 || r >= a.n_rows) {
          set_error(a.err, MOE_DEVERR_ROW_INDEX);
          r = -1;
        }
      }
      use[i] = in && r != -1;
      v[i] = use[i] ? ld_stream16(a.rows + (size_t)r * H + col, pol) : make_uint4(0, 0, 0, 0);
    }
    // 2) the chunk's weights (times the routing scale when it is not 1)
    float w[KC];
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      const int k = k0 + i;
      float wk = 0.0f;
      if (EXACT || k < K) {
        const size_t wi = (size_t)t * K + k;
        wk = BF16W ? bf16_to_f32(__ldg(static_cast<const uint16_t*>(a.weights) + wi))
                   : __ldg(static_cast<const float*>(a.weights) + wi);
        if (a.scale != 1.0f) wk = __fmul_rn(wk, a.scale);
      }
      w[i] = wk;
    }
    // 3) FP32 fma over k in order
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      if (!use[i]) continue;
      const uint32_t q[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[2 * j] = __fmaf_rn(w[i], bf16_lo(q[j]), acc[2 * j]);
        acc[2 * j + 1] = __fmaf_rn(w[i], bf16_hi(q[j]), acc[2 * j + 1]);
      }
    }
  }
  if (SHARED) {
    const uint32_t q[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] = __fadd_rn(acc[2 * j], bf16_lo(q[j]));
      acc[2 * j + 1] = __fadd_rn(acc[2 * j + 1], bf16_hi(q[j]));
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  st16(a.out + (size_t)t * H + col, o);
}

template <int KC, bool EXACT>
int launch_variant(const FinArgs& a, bool gather, bool bf16w, bool shared, dim3 grid, cudaStream_t s) {
#define MOE_FIN_CASE(G, B, S) \
  if (gather == G && bf16w == B && shared == S) \
    return launch_pdl(finalize_kernel<KC, EXACT, G, B, S>, grid, dim3(kFinThreads), 0, s, a);
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
  if ((long long)T * (H / 8) > (1LL << 31) - 1) return MOE_ERR_CAPACITY;
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
  const long long threads = (long long)T * (H / 8);
  dim3 grid((unsigned)((threads + kFinThreads - 1) / kFinThreads));
  const bool gather = row_index != nullptr, bf16w = weights_dtype == MOE_DTYPE_BF16, sh = shared != nullptr;
  cudaStream_t s = as_cuda(stream);
  if (K == 16) return launch_variant<16, true>(a, gather, bf16w, sh, grid, s);
  if (K == 8) return launch_variant<8, true>(a, gather, bf16w, sh, grid, s);
  return launch_variant<8, false>(a, gather, bf16w, sh, grid, s);
}
