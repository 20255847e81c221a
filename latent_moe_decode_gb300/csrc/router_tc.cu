// Router logits on the 5th-generation tensor cores (tcgen05), split-K.
//
// Source: vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer,
// EpMoeLayer (the FP32-output split-K router projection of the [896, 7168] BF16 gate,
// its split-K partials reduced in FP32) and front_tactic (64-row weight tiles, a token tile of the
// next size in {8, 16, 32, 64, 128} at or above the batch, the deepest pipeline that
// fits in about 200 KiB of shared memory, 256-byte K steps).
//
// GB300 design: logits^T = W x^T, i.e. the MMA's M dimension runs over experts and its
// N dimension over tokens, so a decode batch of 8..256 tokens is one N tile and the
// gate is the streamed operand. One CTA (16 warps) computes a 128-expert x BN-token
// tile over a range of 64-wide K blocks:
//   - warp 0, one lane: TMA producer. Each stage is a 128x64 BF16 gate tile and a
//     BNx64 BF16 token tile, both 128-byte swizzled (K-major), landed on a full
//     mbarrier with a transaction count;
//   - warp 1, one lane: issues 4 tcgen05.mma (kind::f16, BF16 x BF16 -> FP32, M=128,
//     N=BN, K=16) per stage into a TMEM accumulator and releases the stage with
//     tcgen05.commit on its empty mbarrier;
//   - all 16 warps: read the accumulator back with tcgen05.ld (warp w reaches TMEM lanes
//     32(w%4)..32(w%4)+31 = 32 experts; the four warpgroups take turns on 16-column
//     chunks) and store FP32 rows; lanes hold consecutive experts, so every store
//     instruction writes 128 contiguous bytes. The epilogue is latency-bound, hence the
//     many warps although the mainloop needs two threads.
// Split-K: when the S split CTAs of a tile fit as one thread-block cluster (S <= 8 for
// wide token tiles; up to a non-portable 16 for tiles of 64 tokens or fewer, so that
// more SMs stream the gate; all clusters co-resident), the reduction happens in the
// same kernel: the CTAs write partials from TMEM to the caller's workspace (128
// contiguous bytes per warp store, L2-resident), a cluster barrier orders those writes
// before the reads, and the tile's outputs are summed over the S partials in split
// order -- wide tiles by owners of 16-column x 32-row units (their own partial
// straight from TMEM), narrow tiles column by column over all the cluster's warps --
// written as final logits (lanes = consecutive experts: 128 contiguous bytes per
// store), and the workspace lines read are invalidated in L2 (discard.global.L2), so
// the scratch never costs an HBM write-back. Otherwise the partials [S][T][E] go to
// the workspace and a second kernel sums them in split order.
// Variants of the same kernel: PAIR, two CTAs on two SMs running one M = 256 MMA
// (cta_group::2) over their 128-row tiles, each staging half the token rows (for wide
// batches: a third fewer bytes per SM for the same MMA work); FRONT, a second weight
// (the latent down projection) whose tiles follow the router's and store BF16 rows (the
// front projection); and the step's partials mode (no cluster, S > 1: the partials
// [S][T][E] are summed by the top-K launch of the one-call step).
// Every mbarrier wait is bounded by the global timer; on expiry the kernel sets
// MOE_DEVERR_TIMEOUT, stops issuing work, waits (bounded) for its own copies in flight,
// frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mxfp8.cuh"
#include "router.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;              // experts per CTA (TMEM lanes)
constexpr int kBK = 64;               // K elements per stage (128 bytes: one swizzle span)
constexpr int kThreads = 512;         // 16 warps: two lanes run the mainloop, all sixteen the epilogue
constexpr int kGroups = kThreads / 128;  // warpgroups: each reaches all 128 TMEM lanes
constexpr int kMaxSplits = 16;           // splits of a cluster plan (16: a non-portable cluster)

// PAIR: two CTAs (one SM each) run one M = 256 MMA (cta_group::2); each stages its
// own 128 weight rows and half of the BN token rows.
template <int BN, bool PAIR = false>
struct Cfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kBBytes = kBRows * kBK * 2;
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

// The same for a CTA pair: `bar` is a shared::cluster address that may lie in the
// peer CTA (the pair's leader counts both CTAs' bytes on one barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Shared::cluster address of the same shared-memory offset in cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
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

// Instruction descriptor: BF16 x BF16 -> FP32, both K-major, M = m (128, or 256 for a
// CTA pair), N = n.
__host__ __device__ constexpr uint32_t instr_desc(int n, int m = kBM) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// CTA pair: M = 256 over both CTAs' weight rows, N = BN over both CTAs' token rows;
// issued by the leader, each CTA's TMEM receives its 128 rows.
__device__ __forceinline__ void mma_bf16_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc));
}

// CTA pair: arrive on the barrier at this shared-memory offset in every CTA of `mask`
// (cluster ranks) once the leader's MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The reduction's units are the (16-column chunk, 32-row quarter) blocks of a tile,
// numbered 4 * chunk + quarter; split r of S owns the units [first(r), first(r + 1)).
// (A quarter is what one warp reads from TMEM.)
__host__ __device__ constexpr int unit_first(int r, int units, int S) { return (r * units) / S; }

// Output of one logit (or latent) value: expert tiles (mt < mt1) store FP32 logits
// [T, E]; with FRONT, the tiles past them are rows of the second weight and store the
// latent [T, L] rounded once to BF16 (round to nearest even).
template <bool FRONT>
__device__ __forceinline__ void store_out(float* out, uint16_t* out2, int t, int mt, int mt1, int row, int E, int L,
                                          float v) {
  if (!FRONT || mt < mt1) {
    const int e = mt * kBM + row;
    if (e < E) out[(size_t)t * E + e] = v;
  } else {
    const int l = (mt - mt1) * kBM + row;
    if (l < L) out2[(size_t)t * L + l] = f32_to_bf16(v);
  }
}

// This CTA's share of the latent's MXFP8 (OCP floor rule, row-major scales), by warps 2
// and up: the CTAs of the grid take equal runs of 32-chunk groups, a warp a group at a
// time (lane = chunk), four groups' loads in flight per warp.
__device__ __forceinline__ void quantise_share(const uint16_t* __restrict__ lat, long long nchunks,
                                               uint8_t* __restrict__ q, uint8_t* __restrict__ sc) {
  const int lane = threadIdx.x & 31, qw = (threadIdx.x >> 5) - 2;
  constexpr int kQuantWarps = kThreads / 32 - 2, kU = 4;
  const long long nct = (long long)gridDim.x * gridDim.y * gridDim.z;
  const long long b = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
  const long long groups = (nchunks + 31) / 32;
  const long long g0 = b * groups / nct, g1 = (b + 1) * groups / nct;
  for (long long g = g0 + qw; g < g1; g += (long long)kQuantWarps * kU) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long c = (g + (long long)u * kQuantWarps) * 32 + lane;
      v[u] = (g + (long long)u * kQuantWarps < g1 && c < nchunks) ? __ldg(reinterpret_cast<const uint4*>(lat) + c)
                                                                    : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const long long gu = g + (long long)u * kQuantWarps;
      if (gu < g1) mxfp8_impl::convert_warp<false, false>(v[u], gu * 32, nchunks, q, sc, 0, 0);
    }
  }
}

// CLUSTER: the S split CTAs of a tile form one cluster and reduce in this kernel.
// FRONT: the tiles mt >= mt1 stream a second weight (tm_w2, the latent down
// projection) and write BF16 rows of `out2`: one launch for both GEMMs that read x.
// PAIR: CTAs 2s and 2s + 1 of a cluster are a pair that computes 256 weight rows x BN
// tokens with cta_group::2 MMAs (blockIdx.z counts pairs of 128-row tiles). Each CTA
// loads its 128 weight rows and BN/2 token rows; both CTAs' copies complete on the
// leader's (even CTA's) full barrier, the leader issues the MMAs, and its commits
// arrive on the empty and accumulator barriers of both CTAs. A pair reads half the
// token bytes per SM of two single CTAs for the same MMA work.
template <int BN, bool CLUSTER, bool FRONT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_w2, float* out, uint16_t* out2, float* part, int T, int E,
                     int L, int mt1, int n_kb, int S, int discard, int late, uint32_t* err,
                     const uint16_t* __restrict__ lat, long long lat_chunks, uint8_t* __restrict__ lq,
                     uint8_t* __restrict__ lsc) {
  using C = Cfg<BN, PAIR>;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = PAIR ? (int)(blockIdx.x & 1u) : 0;  // pair half (cluster rank parity)
  const int s = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x, nt = blockIdx.y;
  const int mt = PAIR ? 2 * (int)blockIdx.z + h : (int)blockIdx.z;  // this CTA's 128-row tile
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
    if (FRONT) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w2)) : "memory");
  }
  if (warp == 2) {
    if constexpr (PAIR) {  // one warp of each CTA of the pair, collectively
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(C::kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(C::kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  if constexpr (PAIR)
    cluster_sync();  // the peer's barriers are initialised before any copy may complete on them
  else
    __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *slot_ptr;

  grid_wait();  // x (and the weights) may be written by the preceding kernel
  // after the wait (dependents may rely on all before this kernel); with `late`, only
  // once the CTA's outputs are written
  if (!late) grid_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {  // TMA producer
      const CUtensorMap* wmap = (FRONT && mt >= mt1) ? &tm_w2 : &tm_w;
      const int wrow = ((FRONT && mt >= mt1) ? mt - mt1 : mt) * kBM;
      const int xrow = nt * BN + h * C::kBRows;
      // a pair's copies complete on the leader's barrier, which expects both CTAs' bytes
      const uint32_t lead = PAIR ? (cluster_rank() & ~1u) : 0u;
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % C::kStages;
        const uint32_t ph = (uint32_t)(i / C::kStages) & 1u;
        if (!mbar_wait(empty(st), ph ^ 1u, err)) break;
        const uint32_t a_dst = base + st * C::kStageBytes;
        if constexpr (PAIR) {
          const uint32_t fb = map_rank(full(st), lead);
          if (h == 0) mbar_expect_tx(full(st), 2 * C::kStageBytes);
          tma_load_2d_pair(a_dst, wmap, (kb0 + i) * kBK, wrow, fb);
          tma_load_2d_pair(a_dst + C::kABytes, &tm_x, (kb0 + i) * kBK, xrow, fb);
        } else {
          mbar_expect_tx(full(st), C::kStageBytes);
          tma_load_2d(a_dst, wmap, (kb0 + i) * kBK, wrow, full(st));
          tma_load_2d(a_dst + C::kABytes, &tm_x, (kb0 + i) * kBK, xrow, full(st));
        }
        ++issued;
      }
      // our copies still in flight land before the CTA may exit (a pair's peer: its
      // copies complete on the leader's barriers, which the leader's MMA waits for)
      if (h == 0) {
        const int first = issued > C::kStages ? issued - C::kStages : 0;
        for (int i = first; i < issued; ++i) mbar_wait(full(i % C::kStages), (uint32_t)(i / C::kStages) & 1u, err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && h == 0) {  // MMA issuer (a pair's leader)
      constexpr uint32_t idesc = instr_desc(BN, PAIR ? 2 * kBM : kBM);
      const uint16_t pair_mask = PAIR ? (uint16_t)(3u << (cluster_rank() & ~1u)) : (uint16_t)0;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % C::kStages;
        if (!mbar_wait(full(st), (uint32_t)(i / C::kStages) & 1u, err)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = base + st * C::kStageBytes;
        const uint32_t b_addr = a_addr + C::kABytes;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          if constexpr (PAIR)
            mma_bf16_pair(tmem, sw128_desc(a_addr + 32u * k), sw128_desc(b_addr + 32u * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
          else
            mma_bf16(tmem, sw128_desc(a_addr + 32u * k), sw128_desc(b_addr + 32u * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
        }
        if constexpr (PAIR)
          mma_commit_pair(empty(st), pair_mask);
        else
          mma_commit(empty(st));
      }
      if constexpr (PAIR)
        mma_commit_pair(accum, pair_mask);
      else
        mma_commit(accum);
    }
    __syncwarp();
  }
  // While warps 0 and 1 stream and multiply, the other warps quantise this CTA's share
  // of the latent (the one-call step's MXFP8; its chunks are a step input)
  if (lat != nullptr && warp >= 2) quantise_share(lat, lat_chunks, lq, lsc);
  // epilogue: TMEM lane = expert row, column = token
  const bool done = __all_sync(0xFFFFFFFFu, mbar_wait(accum, 0, err));  // warp-uniform for tcgen05.ld
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const int wg = warp >> 2;                                    // warpgroup: its 16-column chunks
  const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // this warp's 32 TMEM lanes
  const int row = (warp & 3) * 32 + lane;                           // = expert row within the tile
  if constexpr (CLUSTER) {
    // Wide tiles: split s owns the units [first(s), first(s + 1)) of the tile (16
    // columns x 32 rows each). Every warp writes the units of its rows that other splits
    // own from TMEM to its slot of the workspace ([column][128 rows] FP32: every store
    // instruction of a warp writes 128 contiguous bytes; 18 MB at T = 1020, resident in
    // L2). After a cluster barrier (release / acquire at cluster scope) each owner warp
    // reads its units of the other S - 1 partials (a split's 16 loads at once), sums
    // them per column in split order with its own partial (read from TMEM) and writes
    // the logits; it then invalidates the workspace lines it read in L2
    // (discard.global.L2), so the scratch is never written back to HBM. (Measured
    // slower: every split's loads in flight at once, and row-contiguous 16-byte slots,
    // which touch twice the L2 sectors.) Narrow tiles reduce by columns (below).
    constexpr int nch = BN / 16;
    const int q4 = warp & 3;  // this warp's 32-row quarter
    const int my0 = unit_first(s, 4 * nch, S), my1 = unit_first(s + 1, 4 * nch, S);
    auto mine = [&](int ch) { return 4 * ch + q4 >= my0 && 4 * ch + q4 < my1; };
    const size_t tile = (size_t)mt * gridDim.y + nt;  // (a pair's two CTAs: two tiles)
    float* slot = part + (tile * S + s) * (size_t)BN * kBM;
    // a pair's padding half (rows past both weights) computes zeros no one stores: its
    // splits skip the exchange (still meeting at the cluster barrier)
    const bool live = mt < mt1 + (FRONT ? (L + kBM - 1) / kBM : 0);
    if constexpr (BN <= 64) {
      // Narrow tiles (few columns, many splits): every split writes its whole partial;
      // after the cluster barrier each (column, 32-row quarter) of the tile is one item,
      // dealt to the cluster's warps in turn, whose lanes load that column's S values
      // (all in flight: one round trip), sum them in split order and store.
      if (done && live) {
#pragma unroll 1
        for (int ch = wg; ch < nch; ch += kGroups) {
          uint32_t v[16];
          tmem_ld16(tl + (uint32_t)(16 * ch), v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(slot + (size_t)(16 * ch + j) * kBM + row, __uint_as_float(v[j]));
        }
      }
      cluster_sync();  // every split's partial is written and visible to the cluster
      if (done && live) {
        const int nwarps = S * (kThreads / 32);
#pragma unroll 1
        for (int it = s * (kThreads / 32) + warp; it < 4 * BN; it += nwarps) {
          const int c = it >> 2, r = (it & 3) * 32 + lane;  // column, row
          const float* src = part + (tile * S * BN + c) * (size_t)kBM + r;  // split 0
          float pv[kMaxSplits];
#pragma unroll
          for (int q = 0; q < kMaxSplits; ++q)
            if (q < S) pv[q] = __ldcg(src + (size_t)q * BN * kBM);
          float acc = pv[0];
#pragma unroll
          for (int q = 1; q < kMaxSplits; ++q)  // split order
            if (q < S) acc = __fadd_rn(acc, pv[q]);
          __syncwarp();  // every lane's loads are consumed before their lines are invalidated
          if (discard && lane < S)  // split `lane`'s line of this column and quarter
            asm volatile("discard.global.L2 [%0], 128;" ::"l"(src - r + (it & 3) * 32 + (size_t)lane * BN * kBM)
                         : "memory");
          const int t = nt * BN + c;
          if (t < T) store_out<FRONT>(out, out2, t, mt, mt1, r, E, L, acc);
        }
      }
    } else {  // wide tiles: owners of units
      if (done && live) {
#pragma unroll 1
        for (int ch = wg; ch < nch; ch += kGroups) {
          if (mine(ch)) continue;
          uint32_t v[16];
          tmem_ld16(tl + (uint32_t)(16 * ch), v);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(slot + (size_t)(16 * ch + j) * kBM + row, __uint_as_float(v[j]));
        }
      }
      cluster_sync();  // every split's partial chunks are written and visible to the cluster
      if (done && live) {
#pragma unroll 1
        for (int ch = my0 / 4 + wg; ch < (my1 + 3) / 4; ch += kGroups) {
          if (!mine(ch)) continue;  // (warp-uniform)
          uint32_t v[16];
          tmem_ld16(tl + (uint32_t)(16 * ch), v);
          tmem_wait_ld();
          float acc[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {  // split order (S <= 8 here); a split's 16 columns loaded at once
            if (q >= S) break;
            float p[16];
            if (q == s) {
#pragma unroll
              for (int j = 0; j < 16; ++j) p[j] = __uint_as_float(v[j]);
            } else {
              const float* src = part + ((tile * S + q) * (size_t)BN + 16 * ch) * kBM + row;
#pragma unroll
              for (int j = 0; j < 16; ++j) p[j] = __ldcg(src + (size_t)j * kBM);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = q == 0 ? p[j] : __fadd_rn(acc[j], p[j]);
          }
          __syncwarp();  // every lane's loads are consumed before their lines are invalidated
          if (discard && lane < 16) {  // (a workspace aligned to 128 bytes: whole lines)
            for (int q = 0; q < S; ++q) {
              if (q == s) continue;
              const float* line = part + ((tile * S + q) * (size_t)BN + 16 * ch + lane) * kBM + (warp & 3) * 32;
              asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
            }
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = nt * BN + 16 * ch + j;
            if (t < T) store_out<FRONT>(out, out2, t, mt, mt1, row, E, L, acc[j]);
          }
        }
      }
    }
  } else if (done) {
    // the logits (S == 1), or split s's partial of part [S][T][E] for a consumer that sums
    // them (the routing step's top-K launch; FRONT plans have S == 1)
    float* dst = out + (size_t)s * T * E;
#pragma unroll 1
    for (int c0 = 16 * wg; c0 < BN; c0 += 16 * kGroups) {
      uint32_t v[16];
      tmem_ld16(tl + (uint32_t)c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int t = nt * BN + c0 + j;
        if (t < T) store_out<FRONT>(dst, out2, t, mt, mt1, row, E, L, __uint_as_float(v[j]));
      }
    }
  }
  if (late) grid_launch_dependents();
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  if constexpr (PAIR) {
    cluster_sync();  // neither CTA of a pair leaves while the other may still touch its shared memory
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
  } else {
    __syncthreads();
    if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
  }
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

// w2 / out2 / L: the second weight of a front launch (FRONT), else unused.
// late: the CTAs let the dependent grid launch only once their outputs are written
// (else right after their wait).
template <int BN, bool CLUSTER, bool FRONT, bool PAIR>
int launch_bn(const uint16_t* x, const uint16_t* w, const uint16_t* w2, float* dst, uint16_t* out2, float* part, int T,
              int H, int E, int L, const TcPlan& p, uint32_t* err, cudaStream_t stream, bool late = false,
              const LatentQuant* lq = nullptr) {
  using C = Cfg<BN, PAIR>;
  CUtensorMap tm_w, tm_x, tm_w2;
  if (!make_map(&tm_w, w, E, H, kBM) || !make_map(&tm_x, x, T, H, C::kBRows)) return MOE_ERR_CUDA;
  if (FRONT ? !make_map(&tm_w2, w2, L, H, kBM) : false) return MOE_ERR_CUDA;
  if (!FRONT) tm_w2 = tm_w;
  const int mt1 = (E + kBM - 1) / kBM;
  const int m_tiles = mt1 + (FRONT ? (L + kBM - 1) / kBM : 0);
  auto kern = router_tc_kernel<BN, CLUSTER, FRONT, PAIR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (prefer_max_shared(reinterpret_cast<const void*>(kern)) != MOE_OK) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = PAIR ? dim3(2 * p.S, (T + BN - 1) / BN, (m_tiles + 1) / 2) : dim3(p.S, (T + BN - 1) / BN, m_tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  // Programmatic dependent launch only for the cluster plans of token tiles up to 128
  // (T <= 256), whose launch then starts as the preceding kernel's CTAs leave (measured:
  // the step 1 us faster at T = 64 and 256; the call alone at T = 16 / 64 / 256 6.7 /
  // 7.4 / 11.0 us instead of 9.9 / 10.1 / 14.2). The 256-token tiles (T = 1020: the public
  // call's 5-CTA clusters, the step's partials plan) are launched the ordinary way: early,
  // their CTAs (a whole SM's shared memory each) only contended with the preceding kernel
  // (measured slower: the call alone 22.8 instead of 19 us).
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (CLUSTER || PAIR) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = PAIR ? (CLUSTER ? 2 * p.S : 2) : (CLUSTER ? p.S : 1);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (CLUSTER && !FRONT && BN <= 128) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if ((CLUSTER || PAIR) && attr[0].val.clusterDim.x > 8 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return MOE_ERR_CUDA;
  const int discard = (reinterpret_cast<uintptr_t>(part) & 127u) == 0 ? 1 : 0;
  const LatentQuant none;
  const LatentQuant& l = lq ? *lq : none;
  return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, tm_w2, dst, out2, part, T, E, L, mt1, p.n_kb, p.S, discard,
                            late ? 1 : 0, err, l.x, l.nchunks, l.q, l.scales) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// Clusters of S CTAs (split CTAs of one tile, or pairs of them) that can be resident
// at once.
template <int BN, bool PAIR = false>
int max_clusters(int S) {
  static int cache[kMaxSplits + 1] = {0};
  if (S < 2 || S > kMaxSplits) return 0;
  if (cache[S]) return cache[S];
  auto kern = router_tc_kernel<BN, true, false, PAIR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<BN, PAIR>::kSmem) !=
          cudaSuccess ||
      (S > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S, 64, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<BN, PAIR>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[S] = n > 0 ? n : -1;
  return n;
}

int max_clusters_bn(int bn, int S) {
  switch (bn) {
    case 16: return max_clusters<16>(S);
    case 32: return max_clusters<32>(S);
    case 64: return max_clusters<64>(S);
    case 128: return max_clusters<128>(S);
    default: return max_clusters<256>(S);
  }
}

int max_pair_clusters_bn(int bn, int n_ctas) {
  switch (bn) {
    case 32: return max_clusters<32, true>(n_ctas);
    case 64: return max_clusters<64, true>(n_ctas);
    case 128: return max_clusters<128, true>(n_ctas);
    default: return max_clusters<256, true>(n_ctas);
  }
}

}  // namespace

namespace {
// CTA pairs over pairs of 128-row tiles: S pairs of a tile per cluster (at most 4: the
// portable 8 CTAs), or no split.
TcPlan pair_plan(int T, int H, int m_tiles, int sm_count) {
  TcPlan p;
  p.pair = true;
  p.bn = 256;
  for (int b : {32, 64, 128, 256})  // (a pair's MMA takes N >= 32)
    if (b >= T) {
      p.bn = b;
      break;
    }
  p.n_kb = (H + kBK - 1) / kBK;
  const int pairs = (m_tiles + 1) / 2;
  const int tiles = pairs * ((T + p.bn - 1) / p.bn);  // pair tiles
  int s = sm_count / (2 * (tiles > 0 ? tiles : 1));
  s = s < 1 ? 1 : s;
  if (s > 4) s = 4;
  if (s > p.n_kb / 2) s = p.n_kb / 2 > 0 ? p.n_kb / 2 : 1;
  p.S = 1;
  p.cluster = false;
  for (int c = s; c >= 2; --c) {
    if (max_pair_clusters_bn(p.bn, 2 * c) >= tiles) {
      p.S = c;
      p.cluster = true;
      break;
    }
  }
  return p;
}

int plan_ctas(const TcPlan& p, int T, int m_tiles) {
  const int n = (T + p.bn - 1) / p.bn;
  return p.pair ? 2 * p.S * ((m_tiles + 1) / 2) * n : p.S * m_tiles * n;
}
}  // namespace

// Single CTAs (M = 128) or CTA pairs (M = 256): pairs stage a third less per K block
// for the same MMA work, so they are taken for token tiles of 128 or more whenever they
// keep at least as many SMs busy.
TcPlan tc_plan(int T, int H, int E, int sm_count) {
  const TcPlan single = tc_plan_single(T, H, E, sm_count);
  if (single.bn < 128) return single;
  const int m_tiles = (E + kBM - 1) / kBM;
  const TcPlan pair = pair_plan(T, H, m_tiles, sm_count);
  return plan_ctas(pair, T, m_tiles) >= plan_ctas(single, T, m_tiles) ? pair : single;
}

namespace {
// The split-K plan for one token tile width bn.
TcPlan plan_for_bn(int bn, int T, int H, int E, int sm_count) {
  TcPlan p;
  p.bn = bn;
  p.n_kb = (H + kBK - 1) / kBK;
  const int tiles = ((E + kBM - 1) / kBM) * ((T + p.bn - 1) / p.bn);
  int s = sm_count / (tiles > 0 ? tiles : 1);
  s = s < 1 ? 1 : s;
  s = s > 32 ? 32 : s;
  if (s > p.n_kb / 2) s = p.n_kb / 2 > 0 ? p.n_kb / 2 : 1;
  // at most one cluster of splits: the on-chip reduction in one kernel beats more
  // splits reduced through a workspace by a second kernel. Narrow token tiles (BN <= 64,
  // a few tiles) go up to a non-portable cluster of 16 so that more SMs stream the
  // weight; wider tiles stay within the portable 8 (their exchange grows with S).
  const int cap = p.bn <= 64 ? kMaxSplits : 8;
  if (s > cap) s = cap;
  p.S = s;
  p.cluster = false;
  if (s >= 2) {
    // the largest cluster of splits whose clusters are all resident at once
    for (int c = s; c >= 2; --c) {
      if (max_clusters_bn(p.bn, c) >= tiles) {
        p.S = c;
        p.cluster = true;
        break;
      }
    }
  }
  return p;
}
}  // namespace

// The token tile is the narrowest of 16 .. 256 that covers T; when its plan would keep
// fewer than 70 % of the SMs busy (few tiles, splits capped), narrower tiles are tried
// (more tiles, each with less to exchange), down to 64 columns.
TcPlan tc_plan_single(int T, int H, int E, int sm_count) {
  int bn = 256;
  for (int b : {16, 32, 64, 128, 256})
    if (b >= T) {
      bn = b;
      break;
    }
  const int m_tiles = (E + kBM - 1) / kBM;
  auto ctas = [&](const TcPlan& q) { return q.S * m_tiles * ((T + q.bn - 1) / q.bn); };
  TcPlan best = plan_for_bn(bn, T, H, E, sm_count);
  for (int b = bn / 2; b >= 64 && 10 * ctas(best) < 7 * sm_count; b /= 2) {
    const TcPlan q = plan_for_bn(b, T, H, E, sm_count);
    if (ctas(q) > ctas(best)) best = q;
  }
  return best;
}

int launch_router_tc(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, const TcPlan& p,
                     float* part, uint32_t* err, cudaStream_t stream, const LatentQuant* lq) {
  const bool direct = p.S == 1 || p.cluster;
  float* dst = direct ? logits : part;
  int st;
#define MOE_TC_CASE(B)                                                                                         \
  case B:                                                                                                       \
    st = p.cluster ? launch_bn<B, true, false, false>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, false, lq) \
                   : launch_bn<B, false, false, false>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, false, lq); \
    break;
#define MOE_TC_PAIR_CASE(B)                                                                                    \
  case B:                                                                                                       \
    st = p.cluster ? launch_bn<B, true, false, true>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, false, lq) \
                   : launch_bn<B, false, false, true>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, false, lq); \
    break;
  if (p.pair) {
    if (p.S > 1 && !p.cluster) return MOE_ERR_INVALID_ARGUMENT;
    switch (p.bn) {
      MOE_TC_PAIR_CASE(128)
      MOE_TC_PAIR_CASE(256)
      default: return MOE_ERR_INVALID_ARGUMENT;
    }
  } else {
    switch (p.bn) {
      MOE_TC_CASE(16)
      MOE_TC_CASE(32)
      MOE_TC_CASE(64)
      MOE_TC_CASE(128)
      MOE_TC_CASE(256)
      default: return MOE_ERR_INVALID_ARGUMENT;
    }
  }
#undef MOE_TC_CASE
#undef MOE_TC_PAIR_CASE
  if (st != MOE_OK || direct) return st;
  return launch_router_reduce(part, p.S, T, E, logits, stream);
}

// The front launch runs CTA pairs over pairs of 128-row tiles (both weights' tiles in
// one sequence: a pair may hold the last router tile and the first latent tile). Its
// splits are reduced only on chip: a cluster of S pairs, or no split.
// The router's split-K partials without their reduction: the plan of tc_plan with the
// splits not reduced on chip; each split CTA stores its FP32 partial to part [S][T][E]
// and the consumer sums them in split order (moe_route_finalize: the top-K launch), which
// gives the same sums as the cluster reduction, bit for bit. Only for wide token tiles,
// whose on-chip exchange is the expensive one (5-6 us at T = 1020); narrow tiles (64
// columns or fewer, up to 16 splits) keep their one-round-trip column reduction, which
// costs less than 16 partials read by the consumer. Then, as with one split, the logits
// are written to `logits` directly and *S_out = 1; otherwise *S_out = S.
int launch_router_partials(const uint16_t* x, const uint16_t* w, float* logits, int T, int H, int E, int sm_count,
                           float* part, uint32_t* err, cudaStream_t stream, int* S_out, const LatentQuant* lq,
                           bool* quantised) {
  if (quantised) *quantised = false;
  if (T <= kAutoGemvMaxTokens) {  // what moe_router_logits runs for a handful of tokens
    *S_out = 1;
    return launch_router_gemv(x, w, logits, T, H, E, stream);
  }
  if (quantised) *quantised = lq != nullptr;
  TcPlan p = tc_plan(T, H, E, sm_count);
  if (p.S == 1 || p.bn <= 64) {
    *S_out = 1;
    return launch_router_tc(x, w, logits, T, H, E, p, part, err, stream, lq);
  }
  *S_out = p.S;
  float* dst = p.S > 1 ? part : logits;
  p.cluster = false;
  int st = MOE_ERR_INVALID_ARGUMENT;
  // The partials' consumer (the step's top-K launch) is launched only once every CTA has
  // written its partial: dispatched earlier, its CTAs crowded onto the few SMs this
  // launch leaves free (measured: the step 1.6 us faster at T = 256, 0.6 at T = 1020).
  const bool late = p.S > 1;
#define MOE_TC_PART_CASE(B)                                                                                     \
  case B:                                                                                                        \
    st = p.pair ? launch_bn<B, false, false, true>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, late, lq) \
                : launch_bn<B, false, false, false>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, late, lq); \
    break;
  switch (p.bn) {
    case 16:
      st = launch_bn<16, false, false, false>(x, w, nullptr, dst, nullptr, part, T, H, E, 0, p, err, stream, late, lq);
      break;
    MOE_TC_PART_CASE(32)
    MOE_TC_PART_CASE(64)
    MOE_TC_PART_CASE(128)
    MOE_TC_PART_CASE(256)
    default: break;
  }
#undef MOE_TC_PART_CASE
  return st;
}

size_t router_partials_bytes(int T, int H, int E, int sm_count) {
  if (T <= kAutoGemvMaxTokens) return 0;
  const TcPlan p = tc_plan(T, H, E, sm_count);
  return (p.S > 1 && p.bn > 64) ? (size_t)p.S * T * E * sizeof(float) : 0;
}

// Both weights' 128-row tiles in one sequence, on CTA pairs or single CTAs, whichever
// keeps more SMs busy (at small T pairs need 8-CTA clusters of which too few fit at
// once; single CTAs split K over up to 16). Splits are reduced only on chip.
TcPlan front_plan(int T, int H, int E, int L, int sm_count) {
  const int m_tiles = (E + kBM - 1) / kBM + (L + kBM - 1) / kBM;
  const TcPlan pair = pair_plan(T, H, m_tiles, sm_count);
  TcPlan single = tc_plan_single(T, H, m_tiles * kBM, sm_count);
  if (single.S > 1 && !single.cluster) single.S = 1;
  return plan_ctas(pair, T, m_tiles) >= plan_ctas(single, T, m_tiles) ? pair : single;
}

size_t front_workspace(const TcPlan& p, int T, int E, int L) {
  return tc_workspace(p, T, ((E + kBM - 1) / kBM + (L + kBM - 1) / kBM) * kBM);  // (pairs: rounded to even)
}

int launch_front_tc(const uint16_t* x, const uint16_t* w, const uint16_t* w2, float* logits, uint16_t* latent, int T,
                    int H, int E, int L, const TcPlan& p, float* part, uint32_t* err, cudaStream_t stream) {
  if (p.S > 1 && !p.cluster) return MOE_ERR_INVALID_ARGUMENT;
#define MOE_TC_CASE(B, PR)                                                                                     \
  case B:                                                                                                       \
    return p.cluster ? launch_bn<B, true, true, PR>(x, w, w2, logits, latent, part, T, H, E, L, p, err, stream) \
                     : launch_bn<B, false, true, PR>(x, w, w2, logits, latent, part, T, H, E, L, p, err, stream);
  if (p.pair) {
    switch (p.bn) {
      MOE_TC_CASE(32, true)
      MOE_TC_CASE(64, true)
      MOE_TC_CASE(128, true)
      MOE_TC_CASE(256, true)
      default: return MOE_ERR_INVALID_ARGUMENT;
    }
  }
  switch (p.bn) {
    MOE_TC_CASE(16, false)
    MOE_TC_CASE(32, false)
    MOE_TC_CASE(64, false)
    MOE_TC_CASE(128, false)
    MOE_TC_CASE(256, false)
    default: return MOE_ERR_INVALID_ARGUMENT;
  }
#undef MOE_TC_CASE
}

}  // namespace moe
