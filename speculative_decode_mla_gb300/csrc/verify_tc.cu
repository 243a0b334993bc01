// tcgen05 split-KV tree-verify kernel for sm_103a.
//
// One work unit = (sequence b, 128-row tile of its T*H query rows, KV chunk s).
// A unit runs on a cluster of two CTAs (one per SM) that split the value
// dimensions: CTA rank r owns value dims [256r, 256r + 256) and RoPE dims
// [512 + 32r, 512 + 32r + 32) of every 576-dim latent row. Per 64-position tile:
//
//   producer warps 0-3  gather: slot = slot_table[b][t] (page_size=1), then 16-byte
//                       cp.async of this CTA's 512 value bytes and the 128-byte RoPE
//                       block of row kv[slot] into a 128B-swizzled (UMMA K-major)
//                       smem stage; 4 stages.
//   MMA warp 4          S_r = Q_r K_r^T over the CTA's 288 contraction dims
//                       (tcgen05.mma kind::f16, A = Q from TMEM, B = K from smem,
//                       fp32 accumulate in TMEM); then O_r += P V_r (A = P from TMEM,
//                       B = the same smem stage read MN-major, N = 256).
//   softmax warps 5-8   one thread per query row: read S_r from TMEM, swap partial
//                       scores with the partner CTA through distributed shared memory
//                       (st.async with a byte count on the partner's mbarrier; two
//                       buffers), S = S_0 + S_1 (the same bits on both CTAs), apply the
//                       ancestor bitmask on tree positions, online softmax in the exp2
//                       domain (O is rescaled only when the running max grows by more
//                       than 2^8), write P (bf16) to TMEM.
//   exchange warp 9     tells the partner when this CTA has read a score buffer.
//   epilogue            O_r / l goes through 128B-swizzled smem to TMA tensor stores
//                       (rows past the sequence are clipped by the tensor map); lse to
//                       the split workspace. The combine kernel merges the splits.
//
// Every wait is bounded (about 2 s); on timeout the kernel stops issuing work,
// drains what it started, reports MLA_CHECK_TIMEOUT in dev_status when given,
// writes NaN lse for its rows so the result is visibly invalid, and exits.
#include <cuda.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kRows = 128;              // query rows per tile (MMA M)
constexpr int kKeys = 64;               // positions per KV tile (S MMA N)
constexpr int kStages = 4;
// The producer marks tile t ready kLag tiles after issuing it (once its own copies have landed).
// kLag must stay below kStages - 1: the slot it waits for is freed by a PV that needs tile t - kStages + 1.
constexpr int kLag = 2;
constexpr int kBlockBytes = kKeys * 128;            // 64 rows x 128 B (one 64-dim block)
constexpr int kStageBytes = 5 * kBlockBytes;        // 4 value blocks + the RoPE block
constexpr int kXBytes = kRows * kKeys * 4;          // one partial-score exchange buffer
constexpr int kSmemX = kStages * kStageBytes;       // two exchange buffers follow the stages
constexpr int kSmemBar = kSmemX + 2 * kXBytes;
constexpr int kSmemBytes = kSmemBar + 512 + 1024;   // barriers, TMEM slot, tree parents + alignment slack
constexpr int kEpiBoxBytes = kRows * 128;           // one 32-column fp32 box of O (reuses the stages)

constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kSoftmaxWarp0 = 5;
constexpr int kExchangeWarp = 9;
constexpr int kThreads = 10 * 32;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQ = 352;

// barrier indices (8 bytes each)
constexpr int kBarKvFull = 0, kBarKvEmpty = 4, kBarQFull = 8, kBarSFull = 9, kBarSEmpty = 10, kBarPFull = 11,
              kBarPEmpty = 12, kBarXFull = 13 /*2*/, kBarXEmpty = 15 /*2*/, kBarXRead = 17 /*2*/, kBarDrain = 19,
              kBarEpi = 20, kNumBars = 21;

constexpr long long kTimeoutCycles = 4000000000ll;  // ~2 s at 2 GHz

// Optional event timeline (built only with -DMLA_TC_TRACE): %globaltimer stamps of pipeline
// events, kTraceSlots per CTA, into a buffer registered with mla_tc_trace_set.
constexpr int kTraceSlots = 160;  // 8 fixed events, then 6 per tile for the first 24 tiles, then 4 at the end
static_assert(kTraceSlots >= 8 + 6 * 24 + 4, "trace slots");
#ifdef MLA_TC_TRACE
}  // namespace
__device__ unsigned long long* g_mla_trace;
namespace {
__device__ __forceinline__ void trace_event(int slot) {
  if (g_mla_trace != nullptr && slot < kTraceSlots) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    g_mla_trace[(size_t)blockIdx.x * kTraceSlots + slot] = t;
  }
}
#define TRACE(slot) trace_event(slot)
#else
#define TRACE(slot) ((void)0)
#endif

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when another role aborted or the wait timed out (then it aborts).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         bool cluster_scope = false) {
  const long long start = clock64();
  while (true) {
    if (cluster_scope ? mbar_test_cluster(bar, parity) : mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - start > kTimeoutCycles) {
      *abort_flag = 1;
      return false;
    }
  }
}
// The same wait taken by every lane of a warp; the result is uniform across the warp.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          bool cluster_scope = false) {
  const bool ok = wait_bar(bar, parity, abort_flag, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t cta) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(cta));
  return r;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 2^x on the MUFU unit (flushes subnormal results to zero; P below 2^-126 is dropped).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// UMMA shared-memory descriptor, 128-byte swizzle (layout type 2), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= 2ull << 61;
  return d;
}
// Instruction descriptor for kind::f16: bf16 A and B, fp32 D, M x N, B K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t instr_desc(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

#define TMEM_LD16(addr, r)                                                                                       \
  asm volatile(                                                                                                  \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];" \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),       \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])   \
      : "r"(addr))
#define TMEM_ST16(addr, r)                                                                                        \
  asm volatile(                                                                                                   \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" \
      ::"r"(addr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),     \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])            \
      : "memory")
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------ the kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const VerifyArgs a, const __grid_constant__ CUtensorMap tmap_o) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t bar0 = base + kSmemBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemBar + 8 * kNumBars);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  int32_t* s_parent = reinterpret_cast<int32_t*>(smem + kSmemBar + 8 * kNumBars + 8);  // up to 64 entries

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) TRACE(0);
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const uint32_t peer = rank ^ 1u;

  // which unit
  const int unit = blockIdx.x >> 1;
  const int s = unit % a.splits;
  const int bt = unit / a.splits;
  const int tile_idx = bt % a.row_tiles;
  const int b = bt / a.row_tiles;
  const int R = a.T * a.H;
  const int row0 = tile_idx * kRows;
  const int32_t L = load_len(a, b);
  const int64_t N = (int64_t)L + a.T;
  const int64_t t0 = (int64_t)s * a.chunk;
  const int64_t t1 = min(N, t0 + a.chunk);
  if (t0 >= t1) {  // nothing of this sequence falls in this chunk: an empty partial
    if (rank == 0 && threadIdx.x < kRows && row0 + (int)threadIdx.x < R)
      a.part_lse[(int64_t)s * a.rows + (int64_t)b * R + row0 + threadIdx.x] = -INFINITY;
    return;
  }
  const int ntiles = (int)((t1 - t0 + kKeys - 1) / kKeys);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKvFull + i), kProducerWarps * 32);
      mbar_init(bar(kBarKvEmpty + i), 1);
    }
    mbar_init(bar(kBarQFull), 4);
    mbar_init(bar(kBarSFull), 1);
    mbar_init(bar(kBarSEmpty), 4);
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarPEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarXFull + i), 1);   // armed locally with the exchange's byte count
      mbar_init(bar(kBarXEmpty + i), 1);  // one remote arrive per use from the partner
      mbar_init(bar(kBarXRead + i), 4);   // the four softmax warps have read the buffer
    }
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarEpi), 4);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_arrive_expect_tx(bar(kBarXFull + 0), kXBytes);  // first use of each exchange buffer
    mbar_arrive_expect_tx(bar(kBarXFull + 1), kXBytes);
  }
  if (threadIdx.x < a.T) {  // tree parents of this sequence, validated, into shared memory
    int p = a.tree_parent[(int64_t)b * a.T + threadIdx.x];
    if (p < -1 || p >= (int)threadIdx.x) {
      report(a.dev_status, a.debug, MLA_CHECK_BAD_PARENT);
      p = -1;
    }
    s_parent[threadIdx.x] = p;
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // barrier inits visible to the partner before any remote operation
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) TRACE(1);

  if (warp < kProducerWarps) {
    // ---------------------------------------------------------------- producer: page_size=1 gather
    const int key_base = warp * 16;
    const char* kvb = reinterpret_cast<const char*>(a.kv);
    // slot entries are fetched one tile ahead so their latency hides behind the copies
    const int32_t* tab = a.slot_table + (int64_t)b * a.stride;
    auto fetch = [&](int t) -> int32_t {
      const int64_t pos = t0 + (int64_t)t * kKeys + key_base + (lane & 15);
      return pos < t1 ? tab[pos] : 0;  // positions past the end read row 0 (masked later)
    };
    int32_t slot_next = fetch(0);
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int stage = t % kStages;
      if (t >= kStages && !wait_warp(bar(kBarKvEmpty + stage), ((t / kStages) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      int32_t slot = slot_next;
      if (t + 1 < ntiles) slot_next = fetch(t + 1);
      if (slot < 0 || (int64_t)slot >= a.num_slots) {
        report(a.dev_status, a.debug, MLA_CHECK_BAD_SLOT);
        slot = slot < 0 ? 0 : (int32_t)(a.num_slots - 1);
      }
      const uint32_t sbase = base + stage * kStageBytes;
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {  // this CTA's 512 value bytes of one row per instruction
        const int key = key_base + k;
        const int64_t sl = __shfl_sync(0xffffffffu, slot, k);
        const char* src = kvb + sl * (kDK * 2) + rank * 512 + lane * 16;
        const uint32_t dst =
            sbase + (lane >> 3) * kBlockBytes + key * 128 + ((((uint32_t)lane & 7u) ^ ((uint32_t)key & 7u)) << 4);
        cp_async16(dst, src);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // the 128-byte RoPE block of four rows per instruction
        const int kk = k * 4 + (lane >> 3);
        const int key = key_base + kk;
        const int64_t sl = __shfl_sync(0xffffffffu, slot, kk);
        const char* src = kvb + sl * (kDK * 2) + 1024 + (lane & 7) * 16;
        const uint32_t dst =
            sbase + 4 * kBlockBytes + key * 128 + ((((uint32_t)lane & 7u) ^ ((uint32_t)key & 7u)) << 4);
        cp_async16(dst, src);
      }
      cp_async_commit();
      if (t == 0 && threadIdx.x == 0) TRACE(2);
      if (t >= kLag) {
        cp_async_wait<kLag>();
        fence_proxy_async();
        mbar_arrive(bar(kBarKvFull + (t - kLag) % kStages));
        if (t == kLag && threadIdx.x == 0) TRACE(3);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    if (ok) {
      for (int t = max(0, ntiles - kLag); t < ntiles; ++t) mbar_arrive(bar(kBarKvFull + t % kStages));
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = instr_desc(kRows, kKeys, 0);
      constexpr uint32_t idesc_pv = instr_desc(kRows, 256, 1);
      bool ok = wait_bar(bar(kBarQFull), 0, abort_flag);
      TRACE(4);
      tc_fence_after();
      auto issue_pv = [&](int t) -> bool {
        if (!wait_bar(bar(kBarPFull), t & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t sbase = base + (t % kStages) * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 16 positions per step; V read MN-major from the same stage
          const uint64_t bd = smem_desc(sbase + kk * 2048, kBlockBytes, 1024);
          mma_tmem_a(tmem + kColO, tmem + kColP + kk * 8, bd, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(kBarKvEmpty + t % kStages));
        mma_commit(bar(kBarPEmpty));
        return true;
      };
      for (int t = 0; t < ntiles && ok; ++t) {
        const int stage = t % kStages;
        if (!wait_bar(bar(kBarKvFull + stage), (t / kStages) & 1, abort_flag)) { ok = false; break; }
        if (t == 0) TRACE(5);
        if (t > 0 && !wait_bar(bar(kBarSEmpty), (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sbase = base + stage * kStageBytes;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = smem_desc(sbase + j * kBlockBytes + kk * 32, 16, 1024);
            mma_tmem_a(tmem + kColS, tmem + kColQ + j * 32 + kk * 8, bd, idesc_s, (j | kk) ? 1u : 0u);
          }
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {  // this CTA's half of the RoPE dims
          const uint64_t bd = smem_desc(sbase + 4 * kBlockBytes + (rank * 2 + kk) * 32, 16, 1024);
          mma_tmem_a(tmem + kColS, tmem + kColQ + 128 + kk * 8, bd, idesc_s, 1u);
        }
        mma_commit(bar(kBarSFull));
        if (t > 0 && !issue_pv(t - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(ntiles - 1);
      // drain: every MMA issued so far has completed once this barrier flips
      mma_commit(bar(kBarDrain));
      const long long st = clock64();
      while (!mbar_test(bar(kBarDrain), 0) && clock64() - st < kTimeoutCycles) {
      }
    }
    __syncwarp();
  } else if (warp == kExchangeWarp) {
    // ---------------------------------------------------------------- score-buffer release to the partner
    if (lane == 0) {
      const uint32_t xempty_remote0 = map_to_cta(bar(kBarXEmpty), peer);
      for (int t = 0; t < ntiles; ++t) {
        if (!wait_bar(bar(kBarXRead + (t & 1)), (t >> 1) & 1, abort_flag)) break;
        mbar_arrive_remote(xempty_remote0 + 8u * (uint32_t)(t & 1));
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warps, one thread per row
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const int local_row = row0 + r;
    const bool valid = local_row < R;
    const int64_t grow = (int64_t)b * R + local_row;
    const int node = valid ? local_row / a.H : 0;

    // Q -> TMEM: this CTA's 256 value dims then its 32 RoPE dims, two bf16 per column.
    // All 36 loads are issued before the first TMEM store so their latencies overlap.
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(a.q + (valid ? grow : 0) * kDK);
      uint32_t v[144];
#pragma unroll
      for (int chunk = 0; chunk < 36; ++chunk) {  // 16-byte chunks: 0..31 value, 32..35 RoPE
        const int src = chunk < 32 ? rank * 32 + chunk : 64 + rank * 4 + (chunk - 32);
        const uint4 x = valid ? __ldg(qrow + src) : make_uint4(0, 0, 0, 0);
        v[chunk * 4 + 0] = x.x;
        v[chunk * 4 + 1] = x.y;
        v[chunk * 4 + 2] = x.z;
        v[chunk * 4 + 3] = x.w;
      }
#pragma unroll
      for (int c = 0; c < 9; ++c) TMEM_ST16(lane_addr + kColQ + c * 16, (v + c * 16));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarQFull));
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE(6);
    }

    // anc*(node) from the parents in shared memory: bit j set iff j is node or one of its ancestors
    uint64_t anc = ~0ull;
    if (valid) {
      anc = 0;
      for (int j = node, step = 0; j >= 0 && step < kMaxNodes; j = s_parent[j], ++step) anc |= 1ull << j;
    }

    const uint32_t x_remote0 = map_to_cta(base + kSmemX, peer);
    const uint32_t xfull_remote0 = map_to_cta(bar(kBarXFull), peer);
    // l_run sums the exact exponentials (for lse); l_bf sums the bf16-rounded P the MMA
    // multiplies with (for normalising O, so a constant value column comes out as exactly 1)
    float m_run = -INFINITY, l_run = 0.f, l_bf = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int xb = t & 1;
      if (!wait_warp(bar(kBarSFull), t & 1, abort_flag)) { ok = false; break; }
      if (warp == kSoftmaxWarp0 && lane == 0 && t < 24) TRACE(8 + 6 * t);
      tc_fence_after();
      float sc[kKeys];
      {
        uint32_t* su = reinterpret_cast<uint32_t*>(sc);
#pragma unroll
        for (int c = 0; c < 4; ++c) TMEM_LD16(lane_addr + kColS + c * 16, (su + c * 16));
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty));
      if (warp == kSoftmaxWarp0 && lane == 0 && t < 24) TRACE(9 + 6 * t);

      // swap partial scores with the partner: asynchronous remote stores into its buffer xb,
      // each landing with a byte count on the partner's x_full[xb]
      if (t >= 2 && !wait_warp(bar(kBarXEmpty + xb), ((t - 2) >> 1) & 1, abort_flag, true)) { ok = false; break; }
      const uint32_t xr = x_remote0 + (uint32_t)(xb * kXBytes);
      const uint32_t xf = xfull_remote0 + 8u * (uint32_t)xb;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        asm volatile(
            "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                xr + (j * kRows + r) * 16),
            "f"(sc[4 * j]), "f"(sc[4 * j + 1]), "f"(sc[4 * j + 2]), "f"(sc[4 * j + 3]), "r"(xf)
            : "memory");
      }
      if (warp == kSoftmaxWarp0 && lane == 0 && t < 24) TRACE(10 + 6 * t);
      if (!wait_warp(bar(kBarXFull + xb), (t >> 1) & 1, abort_flag, true)) { ok = false; break; }
      if (warp == kSoftmaxWarp0 && lane == 0) {
        if (t < 24) TRACE(11 + 6 * t);
        mbar_arrive_expect_tx(bar(kBarXFull + xb), kXBytes);  // arm this buffer's next use
      }
      const float4* xbuf = reinterpret_cast<const float4*>(smem + kSmemX + xb * kXBytes);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 o = xbuf[j * kRows + r];
        sc[4 * j] += o.x;
        sc[4 * j + 1] += o.y;
        sc[4 * j + 2] += o.z;
        sc[4 * j + 3] += o.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarXRead + xb));  // the exchange warp releases it to the partner

      // tree positions (tail tiles only) and positions past the end are masked
      const int64_t p0 = t0 + (int64_t)t * kKeys;
      if (p0 + kKeys > L) {
#pragma unroll
        for (int k = 0; k < kKeys; ++k) {
          const int64_t p = p0 + k;
          const bool vis = p < L || (p < N && ((anc >> (p - L)) & 1ull));
          if (!vis) sc[k] = -INFINITY;
        }
      }
      float mt = sc[0];
#pragma unroll
      for (int k = 1; k < kKeys; ++k) mt = fmaxf(mt, sc[k]);
      const float m_new = fmaxf(m_run, mt * a.scale_log2);  // softmax_scale > 0
      bool rescale = false;
      float alpha = 1.f;
      if (m_new > m_run + 8.f) {  // also the first visible tile (m_run = -inf)
        alpha = ex2(m_run - m_new);
        l_run *= alpha;
        l_bf *= alpha;
        m_run = m_new;
        rescale = t > 0;
      }
      const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
      uint32_t pk[kKeys / 2];
      float lsum = 0.f, lbf = 0.f;
#pragma unroll
      for (int k = 0; k < kKeys; k += 2) {
        const float e0 = ex2(fmaf(sc[k], a.scale_log2, neg_m));
        const float e1 = ex2(fmaf(sc[k + 1], a.scale_log2, neg_m));
        const uint32_t pr = pack_bf16(e0, e1);
        lsum += e0 + e1;
        lbf += __uint_as_float(pr << 16) + __uint_as_float(pr & 0xffff0000u);
        pk[k / 2] = pr;
      }
      l_run += lsum;
      l_bf += lbf;

      // P -> TMEM once PV of the previous tile has finished with it (and with O)
      if (warp == kSoftmaxWarp0 && lane == 0 && t < 24) TRACE(12 + 6 * t);
      if (t > 0) {
        if (!wait_warp(bar(kBarPEmpty), (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
      // tcgen05.ld/st are warp-collective: the whole warp rescales when any of its rows
      // must, and rows that need no rescale multiply by exactly 1.
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < 16; ++c) {
          uint32_t o[16];
          TMEM_LD16(lane_addr + kColO + c * 16, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 16; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * f);
          TMEM_ST16(lane_addr + kColO + c * 16, o);
        }
      }
      TMEM_ST16(lane_addr + kColP, pk);
      TMEM_ST16(lane_addr + kColP + 16, (pk + 16));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
      if (warp == kSoftmaxWarp0 && lane == 0 && t < 24) TRACE(13 + 6 * t);
    }

    // epilogue: O_r / l through 128B-swizzled smem boxes (the stage buffers are idle now)
    // to TMA tensor stores; lse to the workspace
    if (ok) ok = wait_warp(bar(kBarPEmpty), (ntiles - 1) & 1, abort_flag);
    if (warp == kSoftmaxWarp0 && lane == 0) TRACE(kTraceSlots - 4);
    if (ok) {
      tc_fence_after();
      const float inv = l_bf > 0.f ? 1.f / l_bf : 0.f;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {  // box c holds columns [32c, 32c + 32) of this CTA's half
        uint32_t o[32];
        TMEM_LD16(lane_addr + kColO + c * 32, o);
        TMEM_LD16(lane_addr + kColO + c * 32 + 16, (o + 16));
        tmem_wait_ld();
        float4* box = reinterpret_cast<float4*>(smem + c * kEpiBoxBytes + r * 128);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          box[u ^ (r & 7)] = make_float4(__uint_as_float(o[4 * u]) * inv, __uint_as_float(o[4 * u + 1]) * inv,
                                         __uint_as_float(o[4 * u + 2]) * inv, __uint_as_float(o[4 * u + 3]) * inv);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarEpi));
      if (warp == kSoftmaxWarp0) {
        ok = wait_warp(bar(kBarEpi), 0, abort_flag);
        if (ok && lane == 0) {
          const int z = s * a.B + b;
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            asm volatile(
                "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(&tmap_o),
                "r"((int)rank * 256 + c * 32), "r"(row0), "r"(z), "r"(base + c * kEpiBoxBytes)
                : "memory");
          }
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
          asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
        __syncwarp();
      }
      if (valid && rank == 0)
        a.part_lse[(int64_t)s * a.rows + grow] =
            l_run > 0.f ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE(kTraceSlots - 3);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    report(a.dev_status, 1, MLA_CHECK_TIMEOUT);
    if (rank == 0 && threadIdx.x < kRows && row0 + (int)threadIdx.x < R)
      a.part_lse[(int64_t)s * a.rows + (int64_t)b * R + row0 + threadIdx.x] = __int_as_float(0x7fc00000);
  }
  tc_fence_after();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  cluster_sync();  // neither CTA leaves while the partner may still write into its shared memory
  if (threadIdx.x == 0) TRACE(kTraceSlots - 2);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

int tc_kernel_supported() { return encode_tiled() != nullptr ? 1 : 0; }

#ifdef MLA_TC_TRACE
extern "C" int mla_tc_trace_set(void* buffer) {
  return cudaMemcpyToSymbol(g_mla_trace, &buffer, sizeof buffer) == cudaSuccess ? 0 : -4;
}
#endif

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream) {
  static bool configured[64] = {};  // the smem opt-in is set once per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const int64_t units = (int64_t)a.B * a.row_tiles * a.splits;
  if (units * 2 > 0x7fffffff) return cudaErrorInvalidConfiguration;
  // The split partials viewed as [splits * B][R][512] fp32; a store box is 32 columns x 128 rows,
  // so rows past a sequence's R rows fall outside dimension 1 and are not written.
  const int R = a.T * a.H;
  CUtensorMap tmap;
  const cuuint64_t dims[3] = {(cuuint64_t)kDLatent, (cuuint64_t)R, (cuuint64_t)a.splits * (cuuint64_t)a.B};
  const cuuint64_t strides[2] = {(cuuint64_t)kDLatent * 4, (cuuint64_t)R * kDLatent * 4};
  const cuuint32_t box[3] = {32, (cuuint32_t)kRows, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return cudaErrorNotSupported;
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.part_o, dims, strides, box, elem,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  verify_tc_kernel<<<dim3((unsigned)(units * 2)), kThreads, kSmemBytes, stream>>>(a, tmap);
  return cudaGetLastError();
}

}  // namespace mla
