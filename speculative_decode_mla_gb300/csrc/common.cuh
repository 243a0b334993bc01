// Shared definitions of the tree-verify MLA attention library (host + device).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_verify.h"

namespace mla {

constexpr int kDLatent = 512;            // value width (latent dims)
constexpr int kDRope = 64;               // RoPE dims appended to each key row
constexpr int kDK = kDLatent + kDRope;   // 576 bf16 = 1152 bytes per latent row
constexpr int kTileTokens = 64;          // KV positions per tile; chunks are multiples of it
constexpr int kMaxNodes = 64;            // tree nodes per sequence (one u64 ancestor mask)
constexpr int kLptMaxSeqs = 64;          // longest-first unit order: up to two sequences per lane

// Everything a kernel needs, by value (a kernel parameter).
struct VerifyArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;
  const int32_t* slot_table;    // [B][stride]; unused when hybrid
  const int64_t* prefix_base;   // hybrid addressing: prefix position t of sequence b is slot prefix_base[b] + t
  const int32_t* tree_slots;    // hybrid addressing: tree node j of sequence b is slot tree_slots[b*T + j]
  const int32_t* tree_sizes;    // ragged trees: sequence b has tree_sizes[b] nodes (1..T); nullptr = T each
  const int32_t* seq_lens;
  const int32_t* tree_parent;
  __half* part_o;     // [splits][rows][512] fp16, each split normalised over its own part
  float* part_lse;    // [splits][rows]
  int32_t* dev_status;
  int64_t num_slots;
  int64_t rows;       // B*T*H
  int32_t B, T, H, stride, max_seq_len;
  int32_t chunk, splits, row_tiles, rows_per_tile;
  int32_t debug;
  int32_t hybrid;     // 1: prefix_base / tree_slots addressing, 0: slot_table
  int32_t early_prefix;  // MLA_FLAG_PREFIX_STABLE: the prefix may be gathered before the preceding kernel ends
  int32_t lpt;        // tcgen05 kernel, 2 <= B <= 64: work units in longest-first order (from the lengths)
  float scale;        // softmax scale
  float scale_log2;   // softmax scale * log2(e)
};

// Host-side launchers (each returns a cudaError_t from the launch).
cudaError_t launch_verify_simt(const VerifyArgs& a, cudaStream_t stream);
cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream);
// part_dtype: MLA_DTYPE_F32 or MLA_DTYPE_F16. With `dependent`, the launch may start while the
// preceding kernel on the stream finishes (programmatic dependent launch); the kernel waits
// for that kernel's results before reading the partials.
cudaError_t launch_combine(int32_t splits, int64_t rows, int32_t d_v, const void* part_o, int32_t part_dtype,
                           const float* part_lse, void* out, float* lse, int32_t out_dtype, bool dependent,
                           cudaStream_t stream);
int tc_kernel_supported();
// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point (no link to
// libcuda); nullptr when the driver does not provide it.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Device helpers ------------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int debug, int bit) {
  if (debug && status) atomicOr(status, bit);
}

// Prefix length of sequence b, clamped into [0, max_seq_len].
__device__ __forceinline__ int32_t load_len(const VerifyArgs& a, int b) {
  int32_t L = a.seq_lens[b];
  if (L < 0 || L > a.max_seq_len) {
    report(a.dev_status, a.debug, MLA_CHECK_BAD_LENGTH);
    L = L < 0 ? 0 : a.max_seq_len;
  }
  return L;
}

// Number of tree nodes of sequence b (T unless trees are ragged), clamped into [1, T].
__device__ __forceinline__ int32_t load_tree_size(const VerifyArgs& a, int b) {
  if (!a.tree_sizes) return a.T;
  int32_t n = a.tree_sizes[b];
  if (n < 1 || n > a.T) {
    report(a.dev_status, a.debug, MLA_CHECK_BAD_LENGTH);
    n = n < 1 ? 1 : a.T;
  }
  return n;
}

// Ancestor-or-self bit set of node i (bit j set iff j == i or j is an ancestor of i).
// A parent outside [-1, i) is treated as -1 (reported under debug checks).
__device__ __forceinline__ uint64_t ancestor_mask(const VerifyArgs& a, int b, int i) {
  const int32_t* par = a.tree_parent + (int64_t)b * a.T;
  uint64_t m = 0;
  int j = i;
  for (int step = 0; step < kMaxNodes && j >= 0; ++step) {
    m |= 1ull << j;
    int p = par[j];
    if (p < -1 || p >= j) {
      report(a.dev_status, a.debug, MLA_CHECK_BAD_PARENT);
      p = -1;
    }
    j = p;
  }
  return m;
}

// Slot of logical position t of sequence b (prefix length L): the slot table's entry, or with
// hybrid addressing the contiguous prefix base + t for t < L and the tree node's own slot after.
__device__ __forceinline__ int64_t slot_of(const VerifyArgs& a, int b, int32_t L, int64_t t) {
  if (!a.hybrid) return a.slot_table[(int64_t)b * a.stride + t];
  return t < L ? a.prefix_base[b] + t : (int64_t)a.tree_slots[(int64_t)b * a.T + (t - L)];
}

// Physical slot of position t of sequence b (prefix length L), clamped into [0, num_slots).
__device__ __forceinline__ int64_t load_slot(const VerifyArgs& a, int b, int32_t L, int64_t t) {
  int64_t s = slot_of(a, b, L, t);
  if (s < 0 || s >= a.num_slots) {
    report(a.dev_status, a.debug, MLA_CHECK_BAD_SLOT);
    s = s < 0 ? 0 : a.num_slots - 1;
  }
  return s;
}

}  // namespace mla
