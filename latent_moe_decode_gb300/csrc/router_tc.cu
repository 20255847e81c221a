// Router logits on the 5th-generation tensor cores (tcgen05), split-K.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer,
// EpMoeLayer (the FP32-output split-K router projection of the [896, 7168] BF16 gate,
// "split-K reduces in FP32") and front_tactic (64-row weight tiles, a token tile of the
// next size in {8, 16, 32, 64, 128} at or above the batch, the deepest pipeline that
// fits in about 200 KiB of shared memory, 256-byte K steps).
//
// GB300 design: logits^T = W x^T, i.e. the MMA's M dimension runs over experts and its
// N dimension over tokens, so a decode batch of 8..256 tokens is one N tile and the
// gate is the streamed operand. One CTA (4 warps) computes a 128-expert x BN-token
// tile over a range of 64-wide K blocks:
//   - warp 0, one lane: TMA producer. Each stage is a 128x64 BF16 gate tile and a
//     BNx64 BF16 token tile, both 128-byte swizzled (K-major), landed on a full
//     mbarrier with a transaction count;
//   - warp 1, one lane: issues 4 tcgen05.mma (kind::f16, BF16 x BF16 -> FP32, M=128,
//     N=BN, K=16) per stage into a TMEM accumulator and releases the stage with
//     tcgen05.commit on its empty mbarrier;
//   - all 4 warps: read the accumulator back with tcgen05.ld (warp w owns TMEM lanes
//     32w..32w+31 = 32 experts) and store FP32 rows; lanes hold consecutive experts, so
//     every store instruction writes 128 contiguous bytes.
// Split-K partials [S][T][E] are summed by the reduce kernel in split order.
// Every mbarrier wait is bounded by the global timer; on expiry the kernel sets
// MOE_DEVERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies in flight,
// frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "router.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;              // experts per CTA (TMEM lanes)
constexpr int kBK = 64;               // K elements per stage (128 bytes: one swizzle span)
constexpr int kThreads = 128;         // 4 warps

template <int BN>
struct Cfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = (200 * 1024) / kStageBytes < 8 ? (200 * 1024) / kStageBytes : 8;
  static constexpr int kTmemCols = BN < 32 ? 32 : BN;
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 256;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor: K-major tile of 128-byte rows, 128-byte swizzle,
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;             // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;             // descriptor version of the sm_100 family
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// Instruction descriptor: BF16 x BF16 -> FP32, both K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t instr_desc(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x, float* out,
                     int T, int E, int n_kb, int S, uint32_t* err) {
  using C = Cfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x, nt = blockIdx.y, mt = blockIdx.z;
  const int kb0 = (int)(((long long)s * n_kb) / S), kb1 = (int)(((long long)(s + 1) * n_kb) / S);
  const int nkb = kb1 - kb0;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;  // 1024-aligned for the 128-byte swizzle
  const uint32_t bar0 = base + C::kStages * C::kStageBytes;     // full[kStages], empty[kStages], accum, tmem slot
  auto full = [&](int i) { return bar0 + 8u * i; };
  auto empty = [&](int i) { return bar0 + 8u * (C::kStages + i); };
  const uint32_t accum = bar0 + 8u * (2 * C::kStages);
  const uint32_t slot = accum + 8u;
  uint32_t* slot_ptr = reinterpret_cast<uint32_t*>(smem_raw + (slot - smem_u32(smem_raw)));

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(accum, 1);
    mbar_fence_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *slot_ptr;

  grid_launch_dependents();
  grid_wait();  // x (and the gate) may be written by the preceding kernel

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        if (!mbar_wait(empty(st), ph ^ 1u, err)) break;
        const uint32_t a_dst = base + st * C::kStageBytes;
        mbar_expect_tx(full(st), C::kStageBytes);
        tma_load_2d(a_dst, &tm_w, (kb0 + i) * kBK, mt * kBM, full(st));
        tma_load_2d(a_dst + C::kABytes, &tm_x, (kb0 + i) * kBK, nt * BN, full(st));
        ++issued;
      }
      // our copies still in flight land before the CTA may exit
      const int first = issued > C::kStages ? issued - C::kStages : 0;
      for (int i = first; i < issued; ++i) mbar_wait(full(i % C::kStages), (uint32_t)(i / C::kStages) & 1u, err);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {  // MMA issuer
      constexpr uint32_t idesc = instr_desc(BN);
      for (int i = 0; i < nkb; ++i) {
        const int st = i % C::kStages;
        if (!mbar_wait(full(st), (uint32_t)(i / C::kStages) & 1u, err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = base + st * C::kStageBytes;
        const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16(tmem, sw128_desc(a_addr + 32u * k), sw128_desc(b_addr + 32u * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
        mma_commit(empty(st));
      }
      mma_commit(accum);
    }
    __syncwarp();
  }

  // epilogue: TMEM lane = expert row, column = token
  const bool done = __all_sync(0xFFFFFFFFu, mbar_wait(accum, 0, err));  // warp-uniform for tcgen05.ld
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (done) {
    const int e = mt * kBM + warp * 32 + lane;
    float* dst = out + (size_t)s * T * E;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
      if (e < E) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = nt * BN + c0 + j;
          if (t < T) dst[(size_t)t * E + e] = __uint_as_float(v[j]);
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D BF16 tensor [rows, cols] (cols contiguous), box of 64 columns x box_rows rows,
// 128-byte swizzle; out-of-range rows and columns read as zero.
bool make_map(CUtensorMap* m, const void* ptr, int rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
int launch_bn(const uint16_t* x, const uint16_t* w, float* dst, int T, int H, int E, const TcPlan& p, uint32_t* err,
              cudaStream_t stream) {
  CUtensorMap tm_w, tm_x;
  if (!make_map(&tm_w, w, E, H, kBM) || !make_map(&tm_x, x, T, H, BN)) return MOE_ERR_CUDA;
  if (cudaFuncSetAttribute(router_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<BN>::kSmem) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  dim3 grid(p.S, (T + BN - 1) / BN, (E + kBM - 1) / kBM);
  return launch_pdl(router_tc_kernel<BN>, grid, dim3(kThreads), Cfg<BN>::kSmem, stream, tm_w, tm_x, dst, T, E, p.n_kb,
                    p.S, err);
}

}  // namespace

TcPlan tc_plan(int T, int H, int E, int sm_count) {
  TcPlan p;
  p.bn = 256;
  for (int b : {16, 32, 64, 128, 256})
    if (b >= T) {
      p.bn = b;
      break;
    }
  p.n_kb = (H + kBK - 1) / kBK;
  const int tiles = ((E + kBM - 1) / kBM) * ((T + p.bn - 1) / p.bn);
  int s = sm_count / (tiles > 0 ? tiles : 1);
  s = s < 1 ? 1 : s;
  s = s > 32 ? 32 : s;
  if (s > p.n_kb / 2) s = p.n_kb / 2 > 0 ? p.n_kb / 2 : 1;
  p.S = s;
  return p;
}

int launch_router_tc(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, const TcPlan& p,
                     float* part, uint32_t* err, cudaStream_t stream) {
  float* dst = p.S == 1 ? logits : part;
  int st;
  switch (p.bn) {
    case 16: st = launch_bn<16>(x, w, dst, T, H, E, p, err, stream); break;
    case 32: st = launch_bn<32>(x, w, dst, T, H, E, p, err, stream); break;
    case 64: st = launch_bn<64>(x, w, dst, T, H, E, p, err, stream); break;
    case 128: st = launch_bn<128>(x, w, dst, T, H, E, p, err, stream); break;
    default: st = launch_bn<256>(x, w, dst, T, H, E, p, err, stream); break;
  }
  if (st != MOE_OK || p.S == 1) return st;
  return launch_router_reduce(part, p.S, T, E, logits, stream);
}

}  // namespace moe
