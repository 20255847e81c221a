// Shared device/host helpers of the sm_103a routing-and-combine kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_decode.h"

namespace moe {

// ---------------------------------------------------------------------------
// Host side: per-device facts, the device error word, PDL launches.

struct DeviceInfo {
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int smem_per_sm = 0;        // shared memory an SM holds (bytes)
  int smem_reserved = 0;      // shared memory the system reserves per CTA (bytes)
  uint32_t* error_word = nullptr;  // device address of the library's error word
};

// Facts about the current device, cached per device. Returns MOE_OK or an error.
int current_device(DeviceInfo* out);

// Every kernel of the library runs with the largest shared-memory carveout (once per
// kernel and device). The kernels of one step then share one SM configuration: an SM
// need not drain to switch its L1/shared split between them, so a kernel can start
// beside, or (programmatic dependent launch) right behind, the previous one.
int prefer_max_shared(const void* func);

// Sigmoid top-K and MXFP8 of the latent in one launch (moe_topk_route_quantize). With
// latent_ready the quantisation CTAs do not wait for the preceding kernel: only for a
// latent complete before that kernel started, and a preceding kernel that signals its
// dependents after its own wait (the router kernels do). With part != nullptr the
// logits are not read but made: the sum in split order of the router's S partials
// part [S][T][E], written to `logits` (which is then an output). With smap (warp body
// only) the routing CTAs also write the slot map and the below counts of TopkArgs.
int route_quantize(const float* logits, const float* bias, int T, int E, int K, int renormalize, float scale,
                   int32_t* ids, float* weights, uint16_t* weights_bf16, const uint16_t* latent, int rows, int cols,
                   uint8_t* q, uint8_t* scales, bool latent_ready, cudaStream_t s, const float* part = nullptr,
                   int S = 0, uint32_t* smap = nullptr, uint8_t* below = nullptr);

// Finalize (moe_finalize). With rows_ready (no row_index) the first row copies are
// issued before the kernel waits for its predecessor, and everything else (weights) is
// read after the wait: only when the rows (and shared rows) were complete before the
// preceding kernel started.
int finalize(const uint16_t* rows, int64_t n_rows, const int32_t* row_index, const void* weights, int weights_dtype,
             const uint16_t* shared, float routed_scaling_factor, int T, int K, int H, uint16_t* out,
             bool rows_ready, cudaStream_t s);

// Finalize of the one-call step (rows t*K + k with BF16 weights, the rows complete
// before the preceding kernel started) whose launch also builds the routing lists, in
// CTAs of its own beside the row stream, from the slot map the routing CTAs wrote
// (route_quantize with smap).
bool finalize_lists_fit(int T, int K);
int finalize_with_lists(const uint16_t* rows, const uint16_t* weights_bf16, int T, int K, int H, uint16_t* out,
                        const uint32_t* smap, const uint8_t* below, int E, int32_t* offsets, int32_t* pairs,
                        cudaStream_t s);

// Whether route_quantize runs the warp-per-token body for these arguments (the body
// that can write the slot map).
bool route_uses_warp_body(int E, const float* logits, const float* bias, const float* part, int S);

inline cudaStream_t as_cuda(moe_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

__host__ __device__ inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Launch `kernel` on `stream` with programmatic stream serialization allowed, so it
// may start while its predecessor is still running; every kernel of this library
// executes griddepcontrol.wait before it touches data a predecessor may write.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args&&... args) {
  if (prefer_max_shared(reinterpret_cast<const void*>(kernel)) != MOE_OK) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Device side.

// Wait until the preceding kernel in the stream has completed and its writes are
// visible (a no-op when launched without a programmatic dependency).
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to begin launching.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void set_error(uint32_t* word, uint32_t bit) {
  if (word) atomicOr(word, bit);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// Two FP32 -> packed BF16 pair (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// L2 cache policy for data read exactly once (evict first).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 16-byte streaming load: no L1 allocation, L2 line marked evict-first.
__device__ __forceinline__ uint4 ld_stream16(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---------------------------------------------------------------------------
// mbarriers and bulk (TMA) copies.

constexpr uint64_t kWaitTimeoutNs = 1000000000ull;  // every mbarrier wait gives up after 1 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with parity `parity`; false, with MOE_DEVERR_TIMEOUT set,
// after kWaitTimeoutNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer() - t0 > kWaitTimeoutNs) {
      set_error(err, MOE_DEVERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Ask L2 to fetch `bytes` (a multiple of 16) from global address src (16-byte
// aligned). A hint with no effect on results: safe before griddepcontrol.wait even for
// data the preceding kernel writes (L2 is where writes and reads meet; nothing lands in
// registers or shared memory).
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this CTA's shared memory, completing on `bar`; the L2 line gets `policy`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

}  // namespace moe
