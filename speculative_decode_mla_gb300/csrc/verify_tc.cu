// tcgen05 split-KV tree-verify kernel for sm_103a.
//
// One work unit = (sequence b, 128-row tile of its T*H query rows, KV chunk s).
// A unit runs on a cluster of two CTAs (one per SM) that split the value
// dimensions: CTA rank r owns value dims [256r, 256r + 256) and RoPE dims
// [512 + 32r, 512 + 32r + 32) of every 576-dim latent row. Per 64-position tile:
//
//   producer warps 0-3  gather: slot = slot_table[b][t] (page_size=1), then 16-byte
//                       cp.async of this CTA's 512 value bytes (128B-swizzled, UMMA K-major)
//                       and its 64 RoPE bytes (64B-swizzled) of row kv[slot] into a smem
//                       stage. Warp p takes rows 16p..16p+15 of every tile and the tiles go
//                       out in order; a stage's barrier fires when its copies land
//                       (cp.async.mbarrier.arrive.noinc), so no producer waits on its own
//                       copies. One producer per warp scheduler keeps the issue load even.
//   S issuer warp 4     S_r(t) = Q_r K_r^T over the CTA's 288 contraction dims into TMEM score
//                       buffer t % 2 (tcgen05.mma kind::f16, fp32 accumulate; A = Q's value
//                       dims 0..223 from TMEM, its value dims 224..255 and 32 RoPE dims from
//                       shared memory, B = K from the stage) once the tile has landed and the
//                       softmax and the sender have read S_r(t-2), so a tile's scores are
//                       computed while the previous tile's are still being read and exchanged.
//   PV issuer warp 5    O_r += P(t) V_r(t) (A = P from shared memory, B = the same stage read
//                       MN-major, N = 256), then l += P(t) 1 (N = 16 against a ones matrix:
//                       the row sums of the bf16 weights, in TMEM); its completion frees the
//                       stage.
//   sender warps 11-14  as soon as S_r(t) is in TMEM, push it to the partner CTA through
//                       distributed shared memory (st.async with a byte count on the
//                       partner's mbarrier; two receive buffers per CTA), as 16-bit codes on a
//                       per-row power-of-two grid that the partner decodes exactly in one fma
//                       (each partial off by at most half the grid step).
//   softmax warps 7-10  one thread per query row: read S_r(t) from TMEM, add the partner's
//                       partial (S = S_0 + S_1), apply the ancestor bitmask on tree
//                       positions, online softmax in the exp2 domain (O is rescaled only
//                       when the running max grows by more than 2^8), write P (bf16) to
//                       shared memory (128B-swizzled, the PV MMA's K-major A operand).
//   release warp 6      tells the partner when this CTA has read a receive buffer.
//   epilogue            O_r / l (fp16, l the tensor cores' row sum of the same bf16 weights)
//                       goes through 128B-swizzled smem to TMA tensor stores (rows past the
//                       sequence are clipped by the tensor map); lse (from the fp32 sum of the
//                       unrounded exponentials) to the split workspace. The combine kernel,
//                       launched as a programmatic dependent, merges the splits.
//
// TMEM (512 columns): O [0, 256), two S buffers [256, 384), l [384, 400), Q [400, 512).
// A batch of 2..64 sequences takes its units longest first (lpt_unit), from the lengths.
//
// Every wait is bounded (about 2 s); on timeout the kernel stops issuing work,
// drains what it started, reports MLA_CHECK_TIMEOUT in dev_status when given,
// writes NaN lse for its rows so the result is visibly invalid, and exits.
#include <cuda.h>
#include <cuda_fp16.h>
#include <string.h>

#include <atomic>

#include "common.cuh"

namespace mla {
namespace {

constexpr int kRows = 128;              // query rows per tile (MMA M)
constexpr int kKeys = 64;               // positions per KV tile (S MMA N)
constexpr int kStages = 4;              // KV stages in shared memory
constexpr int kBlockBytes = kKeys * 128;            // 64 rows x 128 B (one 64-dim block, 128B swizzle)
constexpr int kRopeBytes = kKeys * 64;              // 64 rows x 64 B: this CTA's 32 RoPE dims, 64B swizzle
constexpr int kStageBytes = 4 * kBlockBytes + kRopeBytes;  // 4 value blocks + the RoPE half
constexpr int kXCodeBytes = kRows * kKeys * 2;      // 16-bit codes of the partial scores of one tile
constexpr int kXBytes = kXCodeBytes + kRows * 8;    // + each row's grid (top, step)
constexpr int kSmemP = kStages * kStageBytes;       // P (bf16, 128 rows x 64 positions, 128B swizzle)
constexpr int kSmemQR = kSmemP + kRows * 128;       // the CTA's 32 RoPE dims of Q (128 rows x 64 B, 64B swizzle)
constexpr int kSmemX = kSmemQR + kRows * 64;        // two exchange buffers
constexpr int kSmemQV = kSmemX + 2 * kXBytes;       // Q's value dims 224..255 of this CTA (the same layout as QR)
constexpr int kSmemOnes = kSmemQV + kRows * 64;     // 16 x 64 bf16 ones: the B operand of the row sums of P
constexpr int kSmemBar = kSmemOnes + 16 * 128;
constexpr int kSmemBytes = kSmemBar + 512 + 1024;   // barriers, TMEM slot, tree parents + alignment slack
constexpr int kEpiBoxBytes = kRows * 128;           // one 64-column fp16 box of O (reuses the stages)
static_assert(kStageBytes % 1024 == 0 && kSmemP % 1024 == 0 && kSmemQR % 1024 == 0 && kSmemX % 16 == 0 &&
                  kXBytes % 16 == 0 && kSmemQV % 512 == 0 && kSmemOnes % 1024 == 0,
              "stage, P, Q, exchange and ones alignment");
static_assert(kSmemBytes <= 232448, "shared memory");

constexpr int kProducerWarps = 4;  // warps 0..3, one per scheduler; warp p gathers rows 16p..16p+15 of each tile
constexpr int kSIssueWarp = 4;      // issues S = Q K^T; allocates and frees TMEM
constexpr int kPVIssueWarp = 5;     // issues O += P V
constexpr int kReleaseWarp = 6;     // tells the partner when a receive buffer has been read
constexpr int kSoftmaxWarp0 = 7;    // warps 7..10: TMEM lane quarters 3, 0, 1, 2
constexpr int kSenderWarp0 = 11;    // warps 11..14: TMEM lane quarters 3, 0, 1, 2
constexpr int kThreads = 15 * 32;
constexpr int kParentThread0 = kSIssueWarp * 32;  // threads reading the tree parents (T <= 64: warps 4-5)

constexpr uint32_t kTmemCols = 512;
// O 256, two S buffers of 64, the row sums of P (16 identical columns), Q's value dims 0..223 (112)
constexpr uint32_t kColO = 0, kColS = 256, kColL = 384, kColQ = 400;
constexpr int kQTmemSteps = 14;  // K-steps of 16 value dims whose A operand is in TMEM

// barrier indices (8 bytes each)
constexpr int kBarKvFull = 0, kBarKvEmpty = kStages, kBarQFull = 2 * kStages, kBarSFull = kBarQFull + 1 /*2*/,
              kBarSEmpty = kBarQFull + 3 /*2*/, kBarPFull = kBarQFull + 5, kBarPEmpty = kBarQFull + 6,
              kBarXFull = kBarQFull + 7 /*2*/, kBarXEmpty = kBarQFull + 9 /*2*/, kBarXRead = kBarQFull + 11 /*2*/,
              kBarDrainS = kBarQFull + 13, kBarDrainP = kBarQFull + 14, kNumBars = kBarQFull + 15;
static_assert(8 * kNumBars + 8 + 4 * kMaxNodes <= 512, "barrier area");

constexpr long long kTimeoutCycles = 4000000000ll;  // ~2 s at 2 GHz

// Optional event timeline (built only with -DMLA_TC_TRACE): %globaltimer stamps of pipeline
// events, kTraceSlots per CTA, into a buffer registered with mla_tc_trace_set.
// 8 fixed events, then 13 per tile for the first 18 tiles (softmax, sender, producer, MMA), then 4 at
// the end
constexpr int kTraceSlots = 256;
constexpr int kTraceTiles = 18;
static_assert(kTraceSlots >= 8 + 13 * kTraceTiles + 4, "trace slots");
#ifdef MLA_TC_TRACE
}  // namespace
__device__ unsigned long long* g_mla_trace;
namespace {
// The buffer pointer is read once per thread at kernel start (trace_buf), so an event costs a
// timer read and a store, not a global load on the path being timed.
__device__ __forceinline__ void trace_event(unsigned long long* buf, int slot) {
  if (buf != nullptr && slot < kTraceSlots) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    buf[(size_t)blockIdx.x * kTraceSlots + slot] = t;
  }
}
#define TRACE(slot) trace_event(trace_buf, slot)
#else
#define TRACE(slot) ((void)0)
#endif
#define TRACE_TILE(t, k) \
  if ((t) < kTraceTiles) TRACE(8 + 13 * (t) + (k))

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
      "{ .reg .pred p; mbarrier.try_wait.parity.relaxed.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false when another role aborted or the wait timed out (then it aborts).
// cluster_scope: the phase is completed from the partner CTA (st.async bytes, remote arrive), a
// release at cluster scope; it is polled relaxed and, once seen, acquired by one fence restricted
// to shared::cluster memory, which is cheaper than an acquiring poll.
// A probe of an mbarrier costs over a hundred cycles even when the phase has completed, and
// reading the clock costs some too: the first probe goes out before the clock is read.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         bool cluster_scope = false) {
  if (cluster_scope) {
    if (mbar_test_cluster(bar, parity)) {
      asm volatile("fence.acquire.sync_restrict::shared::cluster.cluster;" ::: "memory");
      return true;
    }
  } else if (mbar_test(bar, parity)) {
    return true;
  }
  const long long start = clock64();
  while (true) {
    if (cluster_scope) {
      if (mbar_test_cluster(bar, parity)) {
        asm volatile("fence.acquire.sync_restrict::shared::cluster.cluster;" ::: "memory");
        return true;
      }
    } else if (mbar_test(bar, parity)) {
      return true;
    }
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
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
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

// UMMA shared-memory descriptor, descriptor version 1; layout 2 = 128-byte swizzle, 4 = 64-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout = 2) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= (uint64_t)layout << 61;
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
__device__ __forceinline__ void mma_smem_a(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Three-input maximum (one instruction on this architecture; max is exact in any order).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Largest of a tile's kKeys scores, as eight interleaved chains of three-input maxima.
__device__ __forceinline__ float max_of_keys(const float* x) {
  static_assert(kKeys == 64, "chains of 8 + 3 x 16 + 8");
  float m[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    m[u] = max3(x[u], x[8 + u], x[16 + u]);
    m[u] = max3(m[u], x[24 + u], x[32 + u]);
    m[u] = max3(m[u], x[40 + u], x[48 + u]);
    m[u] = fmaxf(m[u], x[56 + u]);
  }
  return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}
// Largest of the negated scores (the negated smallest score).
__device__ __forceinline__ float max_of_neg_keys(const float* x) {
  float m[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    m[u] = max3(-x[u], -x[8 + u], -x[16 + u]);
    m[u] = max3(m[u], -x[24 + u], -x[32 + u]);
    m[u] = max3(m[u], -x[40 + u], -x[48 + u]);
    m[u] = fmaxf(m[u], -x[56 + u]);
  }
  return max3(max3(m[0], m[1], m[2]), max3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}
// Two fp32 lanes per instruction (the packed f32x2 forms); each lane rounds exactly as fmaf / +.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n.reg .b64 ra, rb, rc, rd;\n"
      "mov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\nmov.b64 rc, {%6, %7};\n"
      "fma.rn.f32x2 rd, ra, rb, rc;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n.reg .b64 ra, rb, rd;\n"
      "mov.b64 ra, {%2, %3};\nmov.b64 rb, {%4, %5};\n"
      "add.rn.f32x2 rd, ra, rb;\nmov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint32_t* v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
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

// Inclusive prefix sum over the 64 values v0 (sequences 0..31, one per lane) and v1 (32..63).
__device__ __forceinline__ void warp_scan64(int v0, int v1, int lane, int& inc0, int& inc1) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int u0 = __shfl_up_sync(0xffffffffu, v0, d), u1 = __shfl_up_sync(0xffffffffu, v1, d);
    if (lane >= d) {
      v0 += u0;
      v1 += u1;
    }
  }
  inc0 = v0;
  inc1 = v1 + __shfl_sync(0xffffffffu, v0, 31);
}
// The first sequence whose inclusive prefix exceeds idx (-1 if none), and that prefix.
__device__ __forceinline__ int first_above(int inc0, int inc1, int idx, int& inc_at) {
  uint32_t m = __ballot_sync(0xffffffffu, inc0 > idx);
  if (m) {
    const int l = __ffs(m) - 1;
    inc_at = __shfl_sync(0xffffffffu, inc0, l);
    return l;
  }
  m = __ballot_sync(0xffffffffu, inc1 > idx);
  const int l = m ? __ffs(m) - 1 : 0;
  inc_at = __shfl_sync(0xffffffffu, inc1, l);
  return m ? 32 + l : -1;
}
// Longest-first order of the work units of a batch of 2..64 sequences of different lengths, for
// unit idx in [0, B x splits): every sequence's full chunks first (sequence by sequence), then
// the partial last chunks from the longest down (equal lengths by sequence), then the (sequence,
// split) pairs past a sequence's end, which only mark their partial empty. Clusters start in index
// order, so the long units start first and the short ones fill the gaps at the end. Every lane of
// the warp calls it; the result (sequence, split) is uniform across the warp.
__device__ __forceinline__ void lpt_unit(const VerifyArgs& a, int idx, int lane, int& b_out, int& s_out) {
  int full[2], part[2], nsp[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int bb = lane + 32 * i;
    const int64_t n = bb < a.B ? (int64_t)load_len(a, bb) + load_tree_size(a, bb) : 0;
    full[i] = (int)(n / a.chunk);
    part[i] = (int)(n % a.chunk);
    nsp[i] = full[i] + (part[i] > 0);
  }
  int inc0, inc1, at;
  // 1. full chunks
  warp_scan64(full[0], full[1], lane, inc0, inc1);
  const int nfull = __shfl_sync(0xffffffffu, inc1, 31);
  if (idx < nfull) {
    const int bb = first_above(inc0, inc1, idx, at);
    b_out = bb;
    s_out = idx - (at - __shfl_sync(0xffffffffu, (bb >> 5) ? full[1] : full[0], bb & 31));
    return;
  }
  idx -= nfull;
  // 2. partial chunks, longest first: the one whose rank among the partial chunks is idx
  const int npart = __popc(__ballot_sync(0xffffffffu, part[0] > 0)) + __popc(__ballot_sync(0xffffffffu, part[1] > 0));
  if (idx < npart) {
    int rank[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
        const int pj = __shfl_sync(0xffffffffu, part[h], j);
        const int bj = 32 * h + j;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int bi = lane + 32 * i;
          rank[i] += (pj > part[i] || (pj == part[i] && bj < bi)) && pj > 0;
        }
      }
    }
    const uint32_t m0 = __ballot_sync(0xffffffffu, part[0] > 0 && rank[0] == idx);
    const uint32_t m1 = __ballot_sync(0xffffffffu, part[1] > 0 && rank[1] == idx);
    const int bb = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
    b_out = bb;
    s_out = __shfl_sync(0xffffffffu, (bb >> 5) ? full[1] : full[0], bb & 31);
    return;
  }
  idx -= npart;
  // 3. splits past each sequence's end
  warp_scan64(lane < a.B ? a.splits - nsp[0] : 0, lane + 32 < a.B ? a.splits - nsp[1] : 0, lane, inc0, inc1);
  const int bb = first_above(inc0, inc1, idx, at);
  const int bsafe = bb < 0 ? 0 : bb;  // (idx < B x splits always finds one)
  const int emp = a.splits - __shfl_sync(0xffffffffu, (bsafe >> 5) ? nsp[1] : nsp[0], bsafe & 31);
  b_out = bsafe;
  s_out = a.splits - emp + (idx - (at - emp));
}

// ------------------------------------------------------------------ the kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    verify_tc_kernel(const VerifyArgs a, const __grid_constant__ CUtensorMap tmap_o,
                     const __grid_constant__ CUtensorMap tmap_kv, const __grid_constant__ CUtensorMap tmap_rope) {
  extern __shared__ uint8_t smem_raw[];
#ifdef MLA_TC_TRACE
  unsigned long long* const trace_buf = g_mla_trace;
#endif
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
  // Let the dependent combine grid be scheduled early; it waits for this grid's results anyway.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const uint32_t peer = rank ^ 1u;

  // which unit
  // which unit: (split, row tile, sequence) from the index, or, for a batch in longest-first
  // order, the row tile from the index and the (sequence, split) from the lengths after the wait
  const int unit = blockIdx.x >> 1;
  int s, tile_idx, b;
  if (a.lpt) {
    tile_idx = unit % a.row_tiles;
    s = b = 0;
  } else {
    s = unit % a.splits;
    const int bt = unit / a.splits;
    tile_idx = bt % a.row_tiles;
    b = bt / a.row_tiles;
  }
  const int R = a.T * a.H;
  const int row0 = tile_idx * kRows;
  // Launched as a programmatic dependent: everything above read no global memory; from here on
  // the inputs may have been written by the kernel before this one in the stream. With
  // MLA_FLAG_PREFIX_STABLE the producer warps may read the prefix (length, slots, rows) first and
  // wait just before anything else (see the producer section).
  const bool producer = warp < kProducerWarps;
  const bool early_ok = a.early_prefix && producer;  // (never with the longest-first order)
  if (!early_ok) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (a.lpt) lpt_unit(a, unit / a.row_tiles, lane, b, s);
  const int64_t t0 = (int64_t)s * a.chunk;

  // The reads the set-up waits on are issued together, before anything waits on one: the slots
  // of the first kStages tiles (producer warp), the prefix length and the tree parents. The query
  // rows are read after the set-up, so they do not delay it.
  const int32_t* tab = a.hybrid ? nullptr : a.slot_table + (int64_t)b * a.stride;
  int32_t sr[kStages];  // producer warp p, lane l: slot of row 16p + (l & 15) of each of the next kStages tiles
  if (producer && !a.hybrid) {  // (hybrid addressing computes them once the prefix length is known)
    const int64_t pre_end = min(t0 + (int64_t)a.chunk, (int64_t)a.stride);  // stays inside this row
#pragma unroll
    for (int j = 0; j < kStages; ++j) {
      const int64_t pos = t0 + (int64_t)j * kKeys + warp * 16 + (lane & 15);
      sr[j] = pos < pre_end ? tab[pos] : 0;
    }
  }
  const int32_t L_raw = a.seq_lens[b];
  // the tree parents are read by warps 4-5 (never early), and T <= 64
  const int pidx = (int)threadIdx.x - kParentThread0;
  const int32_t par_raw = (pidx >= 0 && pidx < a.T) ? a.tree_parent[(int64_t)b * a.T + pidx] : -1;

  int32_t L = L_raw;
  if (L < 0 || L > a.max_seq_len) {
    report(a.dev_status, a.debug, MLA_CHECK_BAD_LENGTH);
    L = L < 0 ? 0 : a.max_seq_len;
  }
  // Early prefix tiles: the chunk's first (up to kStages) tiles that lie wholly inside the prefix.
  // A producer warp with some issues them before waiting; otherwise it waits here.
  int early_tiles = 0;
  if (early_ok) {
    if (t0 < L) early_tiles = (int)min((int64_t)kStages, (min((int64_t)L, t0 + (int64_t)a.chunk) - t0) / kKeys);
    if (early_tiles == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  // this sequence's tree (T unless trees are ragged); read after the wait
  int32_t Tb = early_tiles > 0 ? a.T : load_tree_size(a, b);
  int64_t N = (int64_t)L + Tb;
  int64_t t1 = min(N, t0 + a.chunk);
  if (t0 >= t1) {  // nothing of this sequence falls in this chunk: an empty partial (both CTAs agree;
                   // never taken by an early producer, whose chunk starts inside the prefix)
    if (rank == 0 && threadIdx.x < kRows && row0 + (int)threadIdx.x < R)
      a.part_lse[(int64_t)s * a.rows + (int64_t)b * R + row0 + threadIdx.x] = -INFINITY;
    return;
  }
  int ntiles = (int)((t1 - t0 + kKeys - 1) / kKeys);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kBarKvFull + i), 32 * kProducerWarps);  // one asynchronous arrive per producer lane
      mbar_init(bar(kBarKvEmpty + i), 1);
    }
    mbar_init(bar(kBarQFull), 8);  // the softmax and the sender warps each stored their Q chunks
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSEmpty + i), 8);  // the softmax and the sender warps have both read S buffer i
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarXFull + i), 1);   // armed locally with the exchange's byte count
      mbar_init(bar(kBarXEmpty + i), 1);  // one remote arrive from the partner's release warp per use
      mbar_init(bar(kBarXRead + i), 4);   // the four softmax warps have read the buffer
    }
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarPEmpty), 1);
    mbar_init(bar(kBarDrainS), 1);
    mbar_init(bar(kBarDrainP), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_arrive_expect_tx(bar(kBarXFull + 0), kXBytes);  // first use of each exchange buffer
    mbar_arrive_expect_tx(bar(kBarXFull + 1), kXBytes);
  }
  if (pidx >= 0 && pidx < a.T) {  // tree parents of this sequence, validated, into shared memory
    int p = par_raw;
    if (pidx >= Tb) {
      p = -1;  // a padding node of a smaller tree
    } else if (p < -1 || p >= pidx) {
      report(a.dev_status, a.debug, MLA_CHECK_BAD_PARENT);
      p = -1;
    }
    s_parent[pidx] = p;
  }
  if (warp == kSIssueWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // The producer warps only signal that the barriers and parents they wrote are ready (named
  // barrier 1, and their arrival on the cluster barrier) and start the KV stream at once; they
  // need neither TMEM nor the partner, and complete their cluster-barrier phase after their last
  // copy. Named barrier 2 makes thread 0's barrier inits visible to the other producer warps.
  uint32_t tmem = 0;
  if (producer) {
    asm volatile("bar.sync 2, %0;" ::"n"(32 * kProducerWarps) : "memory");
    asm volatile("bar.arrive 1, %0;" ::"n"(kThreads) : "memory");
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  } else {
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
    tc_fence_after();
    cluster_sync();  // barrier inits visible to the partner before any remote operation
    tmem = *tmem_slot;
  }
  if (threadIdx.x == 0) TRACE(1);

  if (warp >= kSoftmaxWarp0) {
    // Q: chunk c < 28 of the CTA's 32 value chunks (8 dims each) at TMEM column kColQ + 4c (two
    // bf16 per column), chunks 28-31 and its 4 RoPE chunks in shared memory; the softmax warps
    // store chunks 0-19, the sender warps chunks 20-35.
    const bool q_sender = warp >= kSenderWarp0;
    const int q_row = (warp & 3) * 32 + lane;  // tile row = TMEM lane of this thread
    const int q_c0 = q_sender ? 20 : 0, q_n = q_sender ? 16 : 20;
    const bool qvalid = row0 + q_row < R && (row0 + q_row) / a.H < Tb;
    const uint4* qrow = reinterpret_cast<const uint4*>(a.q + (qvalid ? (int64_t)b * R + row0 + q_row : 0) * kDK);
    uint32_t qv[80];
    // two chunks (one 32-byte sector) per load, not kept in L1: each row is read once, and
    // 16-byte pieces of 128 rows per warp would otherwise cycle through L1 eight times
#pragma unroll
    for (int i = 0; i < 20; i += 2) {
      const int chunk = q_c0 + i;  // even; a pair never straddles the value/RoPE boundary
#pragma unroll
      for (int k = 0; k < 8; ++k) qv[i * 4 + k] = 0u;
      if (qvalid && i < q_n) {
        const int src = chunk < 32 ? (int)rank * 32 + chunk : 64 + (int)rank * 4 + (chunk - 32);
        asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(qv[i * 4 + 0]), "=r"(qv[i * 4 + 1]), "=r"(qv[i * 4 + 2]), "=r"(qv[i * 4 + 3]),
                       "=r"(qv[i * 4 + 4]), "=r"(qv[i * 4 + 5]), "=r"(qv[i * 4 + 6]), "=r"(qv[i * 4 + 7])
                     : "l"(qrow + src));
      }
    }
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    if (!q_sender) {
#pragma unroll
      for (int c = 0; c < 5; ++c) TMEM_ST16(lane_addr + kColQ + c * 16, (qv + c * 16));
      // the ones operand of the row sums of P (bf16 1.0; 2 KB, 16 bytes per thread of warps 7-10)
      reinterpret_cast<uint4*>(smem + kSmemOnes)[q_row] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
      fence_proxy_async();  // generic-proxy stores, read by the MMA (async proxy)
    } else {
#pragma unroll
      for (int c = 0; c < 2; ++c) TMEM_ST16(lane_addr + kColQ + 80 + c * 16, (qv + c * 16));
      // value chunks 28-31 and RoPE chunks 32-35: row q_row of the 64B-swizzled K-major A operands
      // of their K-steps
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t off = q_row * 64 + (((uint32_t)c ^ (((uint32_t)q_row >> 1) & 3u)) << 4);
        st_shared_v4(base + kSmemQV + off, qv + 32 + 4 * c);
        st_shared_v4(base + kSmemQR + off, qv + 48 + 4 * c);
      }
      fence_proxy_async();  // generic-proxy stores, read by the MMA (async proxy)
    }
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(kBarQFull));
    if (warp == kSoftmaxWarp0 && lane == 0) TRACE(6);
  }

  if (producer) {
    // ---------------------------------------------------------------- producers: page_size=1 gather
    // Every producer warp issues its 16 rows of each tile, tile by tile in order, so across the
    // GPU the first tiles' rows are requested first. No wait on their own copies:
    // cp.async.mbarrier.arrive.noinc makes each lane's arrival on the stage's barrier fire once
    // that lane's copies so far have landed.
    const char* kvb = reinterpret_cast<const char*>(a.kv);
    const int row_base = warp * 16;
    // The slot of lane l's row (16p + (l & 15)) at position pos; positions past the end read row 0
    // (they are masked later).
    auto slot_at = [&](int64_t pos) -> int32_t { return pos < t1 ? (int32_t)slot_of(a, b, L, pos) : 0; };
    int64_t pbase = 0;  // hybrid addressing: slot of prefix position 0
    if (a.hybrid) {
      pbase = a.prefix_base[b];
      if (pbase < 0 || pbase + L > a.num_slots) {
        report(a.dev_status, a.debug, MLA_CHECK_BAD_SLOT);
        pbase = pbase < 0 ? 0 : a.num_slots - 1;  // in range; the TMA path is not used then
      }
    }
    const bool prefix_tiles_by_tma = a.hybrid && pbase + L <= a.num_slots && pbase + L < 0x7fffffffll;

    // Tile t into stage j; sl_own is the slot of this lane's row of the tile.
    auto issue_tile = [&](int t, int j, int32_t sl_own) {
      const uint32_t sbase = base + j * kStageBytes;
      const int64_t p0 = t0 + (int64_t)t * kKeys;
      if (prefix_tiles_by_tma && p0 + kKeys <= L) {
        // Hybrid addressing, a tile wholly inside the contiguous prefix: rows pbase + p0 ... + 63
        // by 2-D TMA boxes that land in the same swizzled layouts (4 value blocks of 64 columns,
        // then this CTA's 32 RoPE columns). One lane arms the stage with the byte count; every
        // other producer lane arrives plainly, so the stage completes when the bytes land.
        if (warp == 0 && lane == 0) {
          const uint32_t full = bar(kBarKvFull + j);
          mbar_arrive_expect_tx(full, kStageBytes);
          const int y = (int)(pbase + p0);
#pragma unroll
          for (int vb = 0; vb < 4; ++vb)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                "%3}], [%4];" ::"r"(sbase + vb * kBlockBytes),
                "l"(&tmap_kv), "r"((int)rank * 256 + vb * 64), "r"(y), "r"(full)
                : "memory");
          asm volatile(
              "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
              "%3}], [%4];" ::"r"(sbase + 4 * kBlockBytes),
              "l"(&tmap_rope), "r"(kDLatent + (int)rank * 32), "r"(y), "r"(full)
              : "memory");
        } else {
          mbar_arrive(bar(kBarKvFull + j));
        }
        return;
      }
      if (sl_own < 0 || (int64_t)sl_own >= a.num_slots) {
        report(a.dev_status, a.debug, MLA_CHECK_BAD_SLOT);
        sl_own = sl_own < 0 ? 0 : (int32_t)min((int64_t)sl_own, a.num_slots - 1);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {  // this CTA's 512 value bytes of one row per instruction
        const int row = row_base + k;
        const int64_t sl = __shfl_sync(0xffffffffu, sl_own, k);
        const char* src = kvb + sl * (kDK * 2) + rank * 512 + lane * 16;
        const uint32_t dst =
            sbase + (lane >> 3) * kBlockBytes + row * 128 + ((((uint32_t)lane & 7u) ^ ((uint32_t)row & 7u)) << 4);
        cp_async16(dst, src);
      }
#pragma unroll
      for (int g = 0; g < 2; ++g) {  // this CTA's 64 RoPE bytes of eight rows per instruction
        const int kr = g * 8 + (lane >> 2);
        const int row = row_base + kr;
        const int64_t sl = __shfl_sync(0xffffffffu, sl_own, kr);
        const char* src = kvb + sl * (kDK * 2) + 1024 + rank * 64 + (lane & 3) * 16;
        const uint32_t dst = sbase + 4 * kBlockBytes + row * 64 +
                             ((((uint32_t)lane & 3u) ^ (((uint32_t)row >> 1) & 3u)) << 4);
        cp_async16(dst, src);
      }
      asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar(kBarKvFull + j)) : "memory");
    };

    if (early_tiles > 0) {
      // MLA_FLAG_PREFIX_STABLE: the first tiles lie wholly inside the prefix, whose length, slots
      // and rows the preceding kernel does not write; they go out now, before that kernel has
      // finished. Everything else (tree size, tree slots, later tiles) waits for it.
#pragma unroll
      for (int j = 0; j < kStages; ++j) {
        if (j < early_tiles) {
          const int64_t pos = t0 + (int64_t)j * kKeys + row_base + (lane & 15);  // < L
          issue_tile(j, j, (int32_t)slot_of(a, b, L, pos));
          if (warp == 0 && lane == 0) TRACE_TILE(j, 6);
        }
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      Tb = load_tree_size(a, b);
      N = (int64_t)L + Tb;
      t1 = min(N, t0 + a.chunk);
      ntiles = (int)((t1 - t0 + kKeys - 1) / kKeys);
    }
    // sr[j]: the slot for the next tile that uses stage j (tile j, or tile j + kStages when
    // tile j already went out early). Slots prefetched before the wait are read again here when
    // the early path was allowed (tree entries may have been rewritten by the preceding kernel).
    const bool fresh_slots = a.hybrid || early_ok;
#pragma unroll
    for (int j = 0; j < kStages; ++j) {
      const int64_t pos = t0 + (int64_t)(j < early_tiles ? j + kStages : j) * kKeys + row_base + (lane & 15);
      if (fresh_slots) sr[j] = slot_at(pos);
      else if (pos >= t1) sr[j] = 0;
    }
    bool ok = true;
    for (int tb = 0; tb < ntiles && ok; tb += kStages) {
#pragma unroll
      for (int j = 0; j < kStages; ++j) {
        const int t = tb + j;
        if (t >= ntiles) break;
        if (t < early_tiles) continue;
        if (t >= kStages && !wait_warp(bar(kBarKvEmpty + j), ((t / kStages) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int32_t sl_own = sr[j];
        {  // the slot of this lane's row of tile t + kStages, needed once this stage comes round again
          const int64_t pn = t0 + (int64_t)(t + kStages) * kKeys + row_base + (lane & 15);
          sr[j] = fresh_slots ? slot_at(pn) : (pn < t1 ? tab[pn] : 0);
        }
        issue_tile(t, j, sl_own);
        if (warp == 0 && lane == 0) TRACE_TILE(t, 6);  // tile t's copies issued (warp 0)
      }
    }
    cp_async_wait_all();  // no copy may still be in flight when the CTA exits
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // this warp's setup phase
  } else if (warp == kSIssueWarp) {
    // ---------------------------------------------------------------- S issuer (one thread)
    // S(t) = Q_r K_r^T over the CTA's 288 contraction dims into S buffer t % 2 (A = Q, B = K from
    // the stage) once tile t has landed and both readers are done with S(t-2) in that buffer.
    if (lane == 0) {
      constexpr uint32_t idesc_s = instr_desc(kRows, kKeys, 0);
      bool ok = wait_bar(bar(kBarQFull), 0, abort_flag);
      TRACE(4);
      for (int t = 0; t < ntiles && ok; ++t) {
        const int sb = t & 1;  // S buffer of tile t
        ok = wait_bar(bar(kBarKvFull + t % kStages), (t / kStages) & 1, abort_flag);
        if (ok && t >= 2) ok = wait_bar(bar(kBarSEmpty + sb), ((t >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        if (t == 0) TRACE(5);
        // the stage was written by cp.async (generic proxy) and is read by the MMA (async proxy)
        fence_proxy_async();
        tc_fence_after();
        const uint32_t sbase = base + (t % kStages) * kStageBytes;
        const uint32_t dS = tmem + kColS + (uint32_t)(sb * kKeys);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t bd = smem_desc(sbase + (i >> 2) * kBlockBytes + (i & 3) * 32, 16, 1024);
          if (i < kQTmemSteps)
            mma_tmem_a(dS, tmem + kColQ + i * 8, bd, idesc_s, i ? 1u : 0u);
          else  // value dims 224..255 (64B-swizzled, 512 B per 8 rows)
            mma_smem_a(dS, smem_desc(base + kSmemQV + (i - kQTmemSteps) * 32, 16, 512, 4), bd, idesc_s, 1u);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {  // this CTA's half of the RoPE dims (64B-swizzled, 512 B per 8 rows)
          const uint64_t ad = smem_desc(base + kSmemQR + kk * 32, 16, 512, 4);
          const uint64_t bd = smem_desc(sbase + 4 * kBlockBytes + kk * 32, 16, 512, 4);
          mma_smem_a(dS, ad, bd, idesc_s, 1u);
        }
        mma_commit(bar(kBarSFull + sb));
        TRACE_TILE(t, 8);  // S(t) issued
      }
      // drain: every MMA this thread issued has completed once this barrier flips
      mma_commit(bar(kBarDrainS));
      const long long st = clock64();
      while (!mbar_test(bar(kBarDrainS), 0) && clock64() - st < kTimeoutCycles) {
      }
    }
    __syncwarp();
  } else if (warp == kPVIssueWarp) {
    // ---------------------------------------------------------------- PV issuer (one thread)
    // O_r += P(t) V_r(t) once the softmax has written P(t); its completion frees the KV stage
    // and the P columns.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = instr_desc(kRows, 256, 1);
      constexpr uint32_t idesc_l = instr_desc(kRows, 16, 0);
      bool ok = true;
      for (int t = 0; t < ntiles && ok; ++t) {
        ok = wait_bar(bar(kBarPFull), t & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sbase = base + (t % kStages) * kStageBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 16 positions per step; V read MN-major from the same stage
          const uint64_t ad = smem_desc(base + kSmemP + kk * 32, 16, 1024);
          const uint64_t bd = smem_desc(sbase + kk * 2048, kBlockBytes, 1024);
          mma_smem_a(tmem + kColO, ad, bd, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // the row sums of P: B = 16 columns of ones
          mma_smem_a(tmem + kColL, smem_desc(base + kSmemP + kk * 32, 16, 1024),
                     smem_desc(base + kSmemOnes + kk * 32, 16, 1024), idesc_l, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(kBarKvEmpty + t % kStages));
        mma_commit(bar(kBarPEmpty));
        TRACE_TILE(t, 9);  // PV(t) issued
      }
      mma_commit(bar(kBarDrainP));
      const long long st = clock64();
      while (!mbar_test(bar(kBarDrainP), 0) && clock64() - st < kTimeoutCycles) {
      }
    }
    __syncwarp();
  } else if (warp == kReleaseWarp) {
    // ---------------------------------------------------------------- receive-buffer release to the partner
    // (kept off the softmax warps: a cluster-scope release arrive is slow)
    if (lane == 0) {
      const uint32_t xempty_remote0 = map_to_cta(bar(kBarXEmpty), peer);
      for (int t = 0; t < ntiles; ++t) {
        if (!wait_bar(bar(kBarXRead + (t & 1)), (t >> 1) & 1, abort_flag)) break;
        mbar_arrive_remote(xempty_remote0 + 8u * (uint32_t)(t & 1));
      }
    }
    __syncwarp();
  } else if (warp >= kSenderWarp0) {
    // ---------------------------------------------------------------- sender warps: S_r to the partner
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const int local_row = row0 + r;
    uint64_t anc = ~0ull;  // anc*(node): the tree positions this row can see
    if (local_row < R && local_row / a.H < Tb) {
      anc = 0;
      for (int j = local_row / a.H, step = 0; j >= 0 && step < kMaxNodes; j = s_parent[j], ++step) anc |= 1ull << j;
    }
    const uint32_t x_remote0 = map_to_cta(base + kSmemX, peer);
    const uint32_t xfull_remote0 = map_to_cta(bar(kBarXFull), peer);
    for (int t = 0; t < ntiles; ++t) {
      const int xb = t & 1;
      if (!wait_warp(bar(kBarSFull + xb), (t >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      uint32_t su[kKeys];
#pragma unroll
      for (int c = 0; c < 4; ++c) TMEM_LD16(lane_addr + kColS + xb * kKeys + c * 16, (su + c * 16));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + xb));
      // The partial goes to the partner as 16-bit codes on a per-row fixed-point grid. Over the
      // keys the row can see in this tile, hi and lo are the largest and smallest partials; s is
      // the smallest power of two with (hi - lo) / s <= 65534 and |hi| / s <= 2^22, n = ceil(hi / s),
      // and a key's code is round(n - p / s), in [0, 65535]. The partner reads back
      // n s - code s, exactly, so each partial it sees is off by at most s / 2. Positions past
      // the end and tree positions the row cannot see stay out of the range; their codes are
      // meaningless and they are masked later.
      const float* sv = reinterpret_cast<const float*>(su);
      float hi = -INFINITY, lo = INFINITY;
      const int64_t p0 = t0 + (int64_t)t * kKeys;
      if (p0 + kKeys <= L) {
        hi = max_of_keys(sv);
        lo = -max_of_neg_keys(sv);
      } else {
#pragma unroll
        for (int k = 0; k < kKeys; ++k) {
          const int64_t p = p0 + k;
          if (p < L || (p < N && ((anc >> (p - L)) & 1ull))) {
            hi = fmaxf(hi, sv[k]);
            lo = fminf(lo, sv[k]);
          }
        }
      }
      if (!(hi >= lo)) hi = lo = 0.f;  // nothing visible (or a padding row)
      const float span = fmaxf(fmaxf((hi - lo) * (1.f / 65534.f), fabsf(hi) * 2.38418579e-7f), 7.8886091e-31f);
      const uint32_t xbits = __float_as_uint(span);
      const uint32_t sbits = ((xbits & 0x7FFFFFu) ? xbits + 0x800000u : xbits) & 0x7F800000u;  // s, >= 2^-100
      const float inv_step = __uint_as_float(0x7F000000u - sbits);                                // 1 / s
      // 2^23 + n: an integer below 2^24, so exact, as is top = (2^23 + n) s
      const float base = ceilf(hi * inv_step) + 8388608.f;
      uint32_t hv[kKeys / 2];
#pragma unroll
      for (int k = 0; k < kKeys; k += 2) {
        // 2^23 + n - p / s rounded once to fp32 lands on the integer 2^23 + code, whose low 16
        // mantissa bits are the code
        const float2 cc = fma2(make_float2(sv[k], sv[k + 1]), make_float2(-inv_step, -inv_step), make_float2(base, base));
        const float c0 = cc.x, c1 = cc.y;
        hv[k / 2] = __byte_perm(__float_as_uint(c0), __float_as_uint(c1), 0x5410);
      }
      const float top = base * __uint_as_float(sbits);
      // the partner's buffer xb is free once it has read what this CTA sent there two tiles ago
      if (t >= 2 && !wait_warp(bar(kBarXEmpty + xb), ((t - 2) >> 1) & 1, abort_flag, true)) break;
      const uint32_t xr = x_remote0 + (uint32_t)(xb * kXBytes);
      const uint32_t xf = xfull_remote0 + 8u * (uint32_t)xb;
#pragma unroll
      for (int j = 0; j < kKeys / 8; ++j) {  // 16-byte chunk j of row r holds keys 8j .. 8j + 7
        asm volatile(
            "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                xr + (j * kRows + r) * 16),
            "r"(hv[4 * j]), "r"(hv[4 * j + 1]), "r"(hv[4 * j + 2]), "r"(hv[4 * j + 3]), "r"(xf)
            : "memory");
      }
      asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
                       xr + kXCodeBytes + r * 8),
                   "r"(__float_as_uint(top)), "r"(sbits), "r"(xf)
                   : "memory");
      if (warp == kSenderWarp0 && lane == 0) TRACE_TILE(t, 2);
    }
  } else {
    // ---------------------------------------------------------------- softmax warps, one thread per row
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const int local_row = row0 + r;
    const bool valid = local_row < R && local_row / a.H < Tb;  // not past R, not a padding node
    const int64_t grow = (int64_t)b * R + local_row;
    const int node = valid ? local_row / a.H : 0;

    // anc*(node) from the parents in shared memory: bit j set iff j is node or one of its ancestors
    uint64_t anc = ~0ull;
    if (valid) {
      anc = 0;
      for (int j = node, step = 0; j >= 0 && step < kMaxNodes; j = s_parent[j], ++step) anc |= 1ull << j;
    }

    // l_run sums the exponentials in fp32 (it gives lse). O is normalised by the tensor cores' own
    // row sums of the bf16 weights (TMEM columns kColL, a PV product with a ones matrix), so O / l
    // is a convex combination of the values with exactly the weights used for them.
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t) {
      const int xb = t & 1;
      if (!wait_warp(bar(kBarSFull + xb), (t >> 1) & 1, abort_flag)) { ok = false; break; }
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE_TILE(t, 0);
      tc_fence_after();
      float sc[kKeys];
      {
        uint32_t* su = reinterpret_cast<uint32_t*>(sc);
#pragma unroll
        for (int c = 0; c < 4; ++c) TMEM_LD16(lane_addr + kColS + xb * kKeys + c * 16, (su + c * 16));
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarSEmpty + xb));
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE_TILE(t, 1);

      if (!wait_warp(bar(kBarXFull + xb), (t >> 1) & 1, abort_flag, true)) { ok = false; break; }
      if (warp == kSoftmaxWarp0 && lane == 0) {
        TRACE_TILE(t, 3);
        mbar_arrive_expect_tx(bar(kBarXFull + xb), kXBytes);  // arm this buffer's next use
      }
      // S = own partial + partner's partial (raw scores; the exp2-domain scale is applied in the
      // exponent). A code's bits placed over the exponent of 2^23 read as c = 2^23 + code, and the
      // partner's partial n s - code s is top - c s, exact in one fma (every term is an integer
      // multiple of the power of two s, below 2^24 s in magnitude).
      {
        const uint8_t* xbuf = smem + kSmemX + xb * kXBytes;
        const uint2 hs = reinterpret_cast<const uint2*>(xbuf + kXCodeBytes)[r];
        const float top = __uint_as_float(hs.x), step = __uint_as_float(hs.y);
#pragma unroll
        for (int j = 0; j < kKeys / 8; ++j) {
          const uint4 w = reinterpret_cast<const uint4*>(xbuf)[j * kRows + r];
          const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float c0 = __uint_as_float(__byte_perm(wv[u], 0x4B000000u, 0x7610));
            const float c1 = __uint_as_float(__byte_perm(wv[u], 0x4B000000u, 0x7632));
            const int k = 8 * j + 2 * u;
            const float2 v = fma2(make_float2(c0, c1), make_float2(-step, -step), make_float2(top, top));
            const float2 t2 = add2(make_float2(sc[k], sc[k + 1]), v);
            sc[k] = t2.x;
            sc[k + 1] = t2.y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarXRead + xb));  // the release warp lets the partner refill it
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE_TILE(t, 7);

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
      const float mt = max_of_keys(sc) * a.scale_log2;  // exp2 domain (softmax_scale > 0)
      const float m_new = fmaxf(m_run, mt);
      bool rescale = false;
      float alpha = 1.f;
      if (m_new > m_run + 8.f) {  // also the first visible tile (m_run = -inf)
        alpha = ex2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
        rescale = t > 0;
      }
      const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
      uint32_t pk[kKeys / 2];
      float lsum0 = 0.f, lsum1 = 0.f;  // two partial sums: shorter dependency chains
#pragma unroll
      for (int k = 0; k < kKeys; k += 2) {
        const float2 x = fma2(make_float2(sc[k], sc[k + 1]), make_float2(a.scale_log2, a.scale_log2),
                              make_float2(neg_m, neg_m));
        const float e0 = ex2(x.x);
        const float e1 = ex2(x.y);
        pk[k / 2] = pack_bf16(e0, e1);
        const float2 ls = add2(make_float2(lsum0, lsum1), make_float2(e0, e1));
        lsum0 = ls.x;
        lsum1 = ls.y;
      }
      l_run += lsum0 + lsum1;

      // P -> shared memory once PV of the previous tile has finished with it (and with O)
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE_TILE(t, 4);
      if (t > 0) {
        if (!wait_warp(bar(kBarPEmpty), (t - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
      // tcgen05.ld/st are warp-collective: the whole warp rescales when any of its rows
      // must, and rows that need no rescale multiply by exactly 1.
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c <= 16; ++c) {  // O's 16 column blocks, then the row sums of P
          const uint32_t col = c < 16 ? kColO + c * 16 : kColL;
          uint32_t o[16];
          TMEM_LD16(lane_addr + col, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 16; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * f);
          TMEM_ST16(lane_addr + col, o);
        }
      }
      // P -> shared memory, the K-major A operand of the PV MMA: row r as eight 16-byte
      // chunks of 8 positions, 128B-swizzled
#pragma unroll
      for (int c = 0; c < 8; ++c)
        st_shared_v4(base + kSmemP + r * 128 + (((uint32_t)c ^ ((uint32_t)r & 7u)) << 4), pk + 4 * c);
      fence_proxy_async();  // generic-proxy stores, read by the MMA (async proxy)
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
      if (warp == kSoftmaxWarp0 && lane == 0) TRACE_TILE(t, 5);
    }

    // epilogue: O_r / l through 128B-swizzled smem boxes (the stage buffers are idle now)
    // to TMA tensor stores; lse to the workspace
    if (ok) ok = wait_warp(bar(kBarPEmpty), (ntiles - 1) & 1, abort_flag);
    if (warp == kSoftmaxWarp0 && lane == 0) TRACE(kTraceSlots - 4);
    if (ok) {
      tc_fence_after();
      uint32_t lr[16];
      TMEM_LD16(lane_addr + kColL, lr);
      tmem_wait_ld();
      const float l_round = __uint_as_float(lr[0]);
      const float inv = l_round > 0.f ? 1.f / l_round : 0.f;
      const int z = s * a.B + b;
      // Each warp owns its 32 rows (its TMEM lane quarter) of every box and stores them itself, so
      // the TMA store of box c overlaps the TMEM reads and conversion of box c + 1.
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {  // box c holds columns [64c, 64c + 64) of this CTA's half, fp16
        uint32_t o[64];
#pragma unroll
        for (int u = 0; u < 4; ++u) TMEM_LD16(lane_addr + kColO + c * 64 + u * 16, (o + u * 16));
        tmem_wait_ld();
        uint4* box = reinterpret_cast<uint4*>(smem + c * kEpiBoxBytes + r * 128);
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // 16-byte chunk u = 8 columns, at position u ^ (r & 7)
          uint32_t w[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const __half2 h = __floats2half2_rn(__uint_as_float(o[8 * u + 2 * k]) * inv,
                                                __uint_as_float(o[8 * u + 2 * k + 1]) * inv);
            w[k] = *reinterpret_cast<const uint32_t*>(&h);
          }
          box[u ^ (r & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          asm volatile(
              "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(&tmap_o),
              "r"((int)rank * 256 + c * 64), "r"(row0 + q4 * 32), "r"(z),
              "r"(base + c * kEpiBoxBytes + q4 * 32 * 128)
              : "memory");
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
      }
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      __syncwarp();
      if (local_row < R && rank == 0)  // padding rows of a smaller tree carry no weight
        a.part_lse[(int64_t)s * a.rows + grow] =
            (valid && l_run > 0.f) ? (m_run + log2f(l_run)) * 0.6931471805599453f : -INFINITY;
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
  if (warp == kSIssueWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  cluster_sync();  // neither CTA leaves while the partner may still write into its shared memory
  if (threadIdx.x == 0) TRACE(kTraceSlots - 2);
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
  // Looked up once per process; the initialiser of a function-local static runs in one thread
  // while concurrent first callers wait for it.
  static const EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

int tc_kernel_supported() { return tensor_map_encoder() != nullptr ? 1 : 0; }

#ifdef MLA_TC_TRACE
extern "C" int mla_tc_trace_set(void* buffer) {
  return cudaMemcpyToSymbol(g_mla_trace, &buffer, sizeof buffer) == cudaSuccess ? 0 : -4;
}
#endif

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream) {
  // the smem opt-in is set once per device (threads racing on the first call may both set it;
  // setting it twice is harmless)
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  const int64_t units = (int64_t)a.B * a.row_tiles * a.splits;
  if (units * 2 > 0x7fffffff) return cudaErrorInvalidConfiguration;
  // The split partials viewed as [splits * B][R][512] fp16; a store box is 64 columns x 32 rows
  // (one softmax warp's rows), so rows past a sequence's R rows fall outside dimension 1 and are
  // not written.
  const int R = a.T * a.H;
  CUtensorMap tmap;
  const cuuint64_t dims[3] = {(cuuint64_t)kDLatent, (cuuint64_t)R, (cuuint64_t)a.splits * (cuuint64_t)a.B};
  const cuuint64_t strides[2] = {(cuuint64_t)kDLatent * 2, (cuuint64_t)R * kDLatent * 2};
  const cuuint32_t box[3] = {64, 32, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  if (enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, a.part_o, dims, strides, box, elem,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  // Hybrid addressing: the pool as a 2-D tensor [num_slots][576] bf16 for the contiguous-prefix
  // tiles; boxes of 64 rows x 64 columns (128B swizzle) and 64 rows x 32 RoPE columns (64B swizzle).
  CUtensorMap tmap_kv, tmap_rope;
  memset(&tmap_kv, 0, sizeof tmap_kv);
  memset(&tmap_rope, 0, sizeof tmap_rope);
  if (a.hybrid) {
    const cuuint64_t kdims[2] = {(cuuint64_t)kDK, (cuuint64_t)a.num_slots};
    const cuuint64_t kstrides[1] = {(cuuint64_t)kDK * 2};
    const cuuint32_t kbox[2] = {64, (cuuint32_t)kKeys}, rbox[2] = {32, (cuuint32_t)kKeys}, kelem[2] = {1, 1};
    if (enc(&tmap_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(a.kv), kdims, kstrides, kbox,
            kelem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        enc(&tmap_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(a.kv), kdims, kstrides, rbox,
            kelem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // Programmatic dependent launch: the CTAs may be scheduled while the previous kernel in the
  // stream drains; they wait for its results (griddepcontrol.wait) before the first global read.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * 2));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, verify_tc_kernel, a, tmap, tmap_kv, tmap_rope);
}

}  // namespace mla
