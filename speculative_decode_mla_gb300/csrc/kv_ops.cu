// KV-pool steps on either side of tree verification (declared in include/mla_kv_ops.h):
// tree-KV append (scatter the new nodes' rows to their slots), accept-commit (move the
// accepted path's slots behind the prefix) and Tier-0 compaction (copy each sequence's
// rows into one contiguous range of a destination pool).
//
// Append and compaction are row copies: 72 chunks of 16 bytes per 1152-byte latent row,
// loads issued before stores so each thread keeps several in flight. Compaction gives a
// CTA 32 consecutive positions of one sequence, so its stores cover one contiguous
// 36 KB range of the destination. Accept-commit is one small CTA per sequence.
#include "mla_kv_ops.h"

#include "common.cuh"

namespace mla {
namespace {

constexpr int kChunks = kDK * 2 / 16;  // 16-byte chunks per latent row (72)
constexpr int kCompactRows = 32;       // positions per compaction CTA
constexpr int kCompactThreads = 256;
constexpr int kCompactPerThread = kCompactRows * kChunks / kCompactThreads;  // 9
static_assert(kCompactRows * kChunks % kCompactThreads == 0, "compaction tiling");

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Prefix length of sequence b clamped to [0, max_seq_len]; *ok is false when it had to be clamped.
__device__ __forceinline__ int32_t clamp_len(const int32_t* seq_lens, int64_t b, int32_t max_seq_len,
                                             int32_t debug, int32_t* dev_status, bool* ok) {
  int32_t L = seq_lens[b];
  *ok = L >= 0 && L <= max_seq_len;
  if (!*ok) {
    report(dev_status, debug, MLA_CHECK_BAD_LENGTH);
    L = L < 0 ? 0 : max_seq_len;
  }
  return L;
}

// One warp per tree node: pool[slot_table[b][L_b + j]] = tree_kv[b*T + j].
__global__ void __launch_bounds__(256) tree_append_kernel(uint4* __restrict__ pool, int64_t num_slots,
                                                          const uint4* __restrict__ tree_kv,
                                                          const int32_t* __restrict__ slot_table,
                                                          const int32_t* __restrict__ seq_lens, int32_t B,
                                                          int32_t T, int32_t stride, int32_t max_seq_len,
                                                          int32_t debug, int32_t* dev_status) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (int64_t)B * T) return;
  const int64_t b = row / T;
  const int j = (int)(row % T);
  bool len_ok;
  const int32_t L = clamp_len(seq_lens, b, max_seq_len, debug, dev_status, &len_ok);
  const int64_t slot = slot_table[b * stride + L + j];
  if (slot < 0 || slot >= num_slots) {
    if (lane == 0) report(dev_status, debug, MLA_CHECK_BAD_SLOT);
    return;
  }
  const uint4* src = tree_kv + row * kChunks;
  uint4* dst = pool + slot * kChunks;
  uint4 v[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int c = lane + 32 * i;
    if (c < kChunks) v[i] = ld_stream(src + c);
  }
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int c = lane + 32 * i;
    if (c < kChunks) dst[c] = v[i];
  }
}

// One CTA of 64 threads per sequence: validate the accepted path, then rewrite the tree block
// of the slot table (accepted slots first, in path order, then the rejected ones in node order).
__global__ void __launch_bounds__(64) accept_commit_kernel(int32_t* __restrict__ slot_table,
                                                           int32_t* __restrict__ seq_lens,
                                                           const int32_t* __restrict__ tree_parent,
                                                           const int32_t* __restrict__ accepted,
                                                           const int32_t* __restrict__ num_accepted,
                                                           int32_t T, int32_t stride, int32_t max_seq_len,
                                                           int32_t debug, int32_t* dev_status) {
  __shared__ int32_t s_slot[kMaxNodes], s_par[kMaxNodes], s_acc[kMaxNodes], s_pos[kMaxNodes];
  __shared__ int32_t s_L, s_n, s_ok;
  const int64_t b = blockIdx.x;
  const int j = threadIdx.x;
  if (j == 0) {
    bool len_ok;
    s_L = clamp_len(seq_lens, b, max_seq_len, debug, dev_status, &len_ok);
    s_n = num_accepted[b];
    s_ok = len_ok ? 1 : 0;
  }
  __syncthreads();
  const int32_t L = s_L;
  if (j < T) {
    s_slot[j] = slot_table[b * stride + L + j];
    s_par[j] = tree_parent[b * T + j];
    s_acc[j] = accepted[b * T + j];
    s_pos[j] = -1;
  }
  __syncthreads();
  if (j == 0 && s_ok) {
    const int32_t n = s_n;
    bool ok = n >= 0 && n <= T;
    if (!ok) report(dev_status, debug, MLA_CHECK_BAD_LENGTH);
    if (ok && (int64_t)L + n > max_seq_len) {
      report(dev_status, debug, MLA_CHECK_BAD_LENGTH);
      ok = false;
    }
    for (int k = 0; ok && k < n; ++k) {  // a root-first path: each node's parent is the one before it
      const int32_t a = s_acc[k];
      if (a < 0 || a >= T || s_pos[a] != -1 || s_par[a] != (k == 0 ? -1 : s_acc[k - 1])) {
        report(dev_status, debug, MLA_CHECK_BAD_PARENT);
        ok = false;
      } else {
        s_pos[a] = k;
      }
    }
    if (ok) {
      int32_t rank = n;
      for (int i = 0; i < T; ++i)
        if (s_pos[i] == -1) s_pos[i] = rank++;
    }
    s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  if (!s_ok) return;
  if (j < T) slot_table[b * stride + L + s_pos[j]] = s_slot[j];
  if (j == 0) seq_lens[b] = L + s_n;
}

// CTA (x, y): positions [32x, 32x + 32) of sequence b0 + y.
__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(
    const uint4* __restrict__ src, int64_t src_slots, uint4* __restrict__ dst, int64_t dst_slots,
    const int32_t* slot_table, int32_t* new_table, const int32_t* __restrict__ seq_lens,
    const int64_t* __restrict__ dst_base, int32_t b0, int32_t T, int32_t stride, int32_t max_seq_len,
    int32_t debug, int32_t* dev_status) {
  __shared__ int64_t s_src[kCompactRows], s_dst[kCompactRows];
  const int64_t b = (int64_t)b0 + blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kCompactRows;
  bool len_ok;
  const int32_t L = clamp_len(seq_lens, b, max_seq_len, threadIdx.x == 0 ? debug : 0, dev_status, &len_ok);
  const int64_t n = (int64_t)L + T;
  if (t0 >= n) return;
  if (threadIdx.x < kCompactRows) {
    const int64_t t = t0 + threadIdx.x;
    int64_t sl = -1, d = -1;
    if (t < n) {
      sl = slot_table[b * stride + t];  // read before new_table (possibly the same array) is rewritten
      d = dst_base[b] + t;
      if (sl < 0 || sl >= src_slots || d < 0 || d >= dst_slots) {
        report(dev_status, debug, MLA_CHECK_BAD_SLOT);
        sl = -1;
      } else if (new_table) {
        new_table[b * stride + t] = (int32_t)d;
      }
    }
    s_src[threadIdx.x] = sl;
    s_dst[threadIdx.x] = d;
  }
  __syncthreads();
  uint4 v[kCompactPerThread];
#pragma unroll
  for (int i = 0; i < kCompactPerThread; ++i) {
    const int c = threadIdx.x + i * kCompactThreads;
    const int64_t sl = s_src[c / kChunks];
    if (sl >= 0) v[i] = ld_stream(src + sl * kChunks + c % kChunks);
  }
#pragma unroll
  for (int i = 0; i < kCompactPerThread; ++i) {
    const int c = threadIdx.x + i * kCompactThreads;
    const int r = c / kChunks;
    if (s_src[r] >= 0) dst[s_dst[r] * kChunks + c % kChunks] = v[i];
  }
}

int check_common(const int32_t* slot_table, const int32_t* seq_lens, int32_t num_seqs, int32_t num_nodes,
                 int32_t stride, int32_t max_seq_len) {
  if (!slot_table || !seq_lens || !aligned(slot_table, 4) || !aligned(seq_lens, 4)) return MLA_ERR_INVALID_ARGUMENT;
  if (num_seqs < 1 || num_nodes < 1 || num_nodes > kMaxNodes || max_seq_len < 0) return MLA_ERR_INVALID_ARGUMENT;
  if ((int64_t)stride < (int64_t)max_seq_len + num_nodes) return MLA_ERR_INVALID_ARGUMENT;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_tree_kv_append(void* pool, int64_t num_slots, const void* tree_kv, const int32_t* slot_table,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t num_nodes, int32_t stride,
                                  int32_t max_seq_len, int32_t debug, int32_t* dev_status, mla_stream_t stream) {
  int rc = check_common(slot_table, seq_lens, num_seqs, num_nodes, stride, max_seq_len);
  if (rc) return rc;
  if (!pool || !tree_kv || !aligned(pool, 16) || !aligned(tree_kv, 16) || num_slots < 1) return MLA_ERR_INVALID_ARGUMENT;
  if (debug && !dev_status) return MLA_ERR_INVALID_ARGUMENT;
  const int64_t rows = (int64_t)num_seqs * num_nodes;
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffff) return MLA_ERR_INVALID_ARGUMENT;
  tree_append_kernel<<<(unsigned)blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(pool), num_slots, static_cast<const uint4*>(tree_kv), slot_table, seq_lens, num_seqs,
      num_nodes, stride, max_seq_len, debug, dev_status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" int mla_tree_accept_commit(int32_t* slot_table, int32_t* seq_lens, const int32_t* tree_parent,
                                      const int32_t* accepted, const int32_t* num_accepted, int32_t num_seqs,
                                      int32_t num_nodes, int32_t stride, int32_t max_seq_len, int32_t debug,
                                      int32_t* dev_status, mla_stream_t stream) {
  int rc = check_common(slot_table, seq_lens, num_seqs, num_nodes, stride, max_seq_len);
  if (rc) return rc;
  if (!tree_parent || !accepted || !num_accepted || !aligned(tree_parent, 4) || !aligned(accepted, 4) ||
      !aligned(num_accepted, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  if (debug && !dev_status) return MLA_ERR_INVALID_ARGUMENT;
  accept_commit_kernel<<<(unsigned)num_seqs, 64, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      slot_table, seq_lens, tree_parent, accepted, num_accepted, num_nodes, stride, max_seq_len, debug, dev_status);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" int mla_kv_compact(const void* src_pool, int64_t src_slots, void* dst_pool, int64_t dst_slots,
                              const int32_t* slot_table, int32_t* new_slot_table, const int32_t* seq_lens,
                              const int64_t* dst_base, int32_t num_seqs, int32_t num_nodes, int32_t stride,
                              int32_t max_seq_len, int32_t debug, int32_t* dev_status, mla_stream_t stream) {
  int rc = check_common(slot_table, seq_lens, num_seqs, num_nodes, stride, max_seq_len);
  if (rc) return rc;
  if (!src_pool || !dst_pool || !dst_base || !aligned(src_pool, 16) || !aligned(dst_pool, 16) ||
      !aligned(dst_base, 8) || (new_slot_table && !aligned(new_slot_table, 4)))
    return MLA_ERR_INVALID_ARGUMENT;
  if (src_slots < 1 || dst_slots < 1 || dst_slots > 0x7fffffff) return MLA_ERR_INVALID_ARGUMENT;
  if (debug && !dev_status) return MLA_ERR_INVALID_ARGUMENT;
  const int64_t chunks = ((int64_t)max_seq_len + num_nodes + kCompactRows - 1) / kCompactRows;
  if (chunks > 0x7fffffff) return MLA_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int32_t b0 = 0; b0 < num_seqs; b0 += 65535) {  // grid.y is at most 65535
    const int32_t nb = num_seqs - b0 < 65535 ? num_seqs - b0 : 65535;
    kv_compact_kernel<<<dim3((unsigned)chunks, (unsigned)nb), kCompactThreads, 0, s>>>(
        static_cast<const uint4*>(src_pool), src_slots, static_cast<uint4*>(dst_pool), dst_slots, slot_table,
        new_slot_table, seq_lens, dst_base, b0, num_nodes, stride, max_seq_len, debug, dev_status);
    if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
