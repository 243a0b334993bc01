// C ABI of the tree-verify MLA attention library: argument checks, the split
// planner and kernel dispatch. Declared in include/mla_verify.h.
#include <math.h>
#include <string.h>

#include "common.cuh"

namespace mla {
namespace {

constexpr int64_t kMaxSlots = (1ll << 31) - 1;
constexpr int kTcRowsPerTile = 128;   // query rows of one tcgen05 row tile (MMA M)
constexpr int kSimtRowsPerTile = 8;   // one warp per row, 8 warps per CTA
constexpr int kMaxSplits = 65535;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int check_desc(const mla_verify_desc* d) {
  if (!d) return MLA_ERR_INVALID_ARGUMENT;
  if (d->d_latent != kDLatent || d->d_rope != kDRope) return MLA_ERR_UNSUPPORTED;
  if (d->num_nodes < 1 || d->num_nodes > kMaxNodes) return MLA_ERR_UNSUPPORTED;
  if (d->num_seqs < 1 || d->num_heads < 1 || d->max_seq_len < 0) return MLA_ERR_INVALID_ARGUMENT;
  if (d->num_slots < 1 || d->num_slots > kMaxSlots) return MLA_ERR_INVALID_ARGUMENT;
  if ((int64_t)d->slot_table_stride < (int64_t)d->max_seq_len + d->num_nodes) return MLA_ERR_INVALID_ARGUMENT;
  if (!isfinite(d->softmax_scale) || !(d->softmax_scale > 0.f)) return MLA_ERR_INVALID_ARGUMENT;
  if (d->out_dtype != MLA_DTYPE_BF16 && d->out_dtype != MLA_DTYPE_F32) return MLA_ERR_INVALID_ARGUMENT;
  if (d->flags & ~(MLA_FLAG_DEBUG_CHECKS | MLA_FLAG_SIMT | MLA_FLAG_PREFIX_STABLE)) return MLA_ERR_INVALID_ARGUMENT;
  if (d->num_splits < 0 || d->num_splits > kMaxSplits || d->total_tokens_hint < 0) return MLA_ERR_INVALID_ARGUMENT;
  const int64_t rows = (int64_t)d->num_seqs * d->num_nodes * d->num_heads;
  if (rows > (1ll << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if ((int64_t)d->num_seqs * d->slot_table_stride > (1ll << 40)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_verify_plan(const mla_verify_desc* d, int32_t num_sms, mla_verify_plan_t* plan) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!plan || num_sms < 1) return MLA_ERR_INVALID_ARGUMENT;
  mla_verify_plan_t p;
  memset(&p, 0, sizeof p);
  const bool simt = (d->flags & MLA_FLAG_SIMT) != 0;
  p.kernel = simt ? 1 : 0;
  p.rows_per_tile = simt ? kSimtRowsPerTile : kTcRowsPerTile;
  const int64_t R = (int64_t)d->num_nodes * d->num_heads;
  p.row_tiles = (int32_t)cdiv(R, p.rows_per_tile);
  const int64_t max_n = (int64_t)d->max_seq_len + d->num_nodes;
  const int64_t max_tiles = cdiv(max_n, kTileTokens);
  const int64_t uniform_total = (int64_t)d->num_seqs * max_n;
  const int64_t total = d->total_tokens_hint > 0 ? d->total_tokens_hint : uniform_total;
  const bool ragged = total < uniform_total;
  // Work units are (sequence, row tile, chunk). A tcgen05 unit runs on a pair of
  // CTAs (one per SM); SIMT units are small CTAs, several per SM.
  const int64_t slots = simt ? (int64_t)num_sms * 8 : (int64_t)(num_sms / 2 > 0 ? num_sms / 2 : 1);
  int64_t best_tiles = 1;
  if (d->num_splits > 0) {
    best_tiles = cdiv(max_tiles, d->num_splits);
  } else if (ragged && !simt && d->num_seqs <= kLptMaxSeqs) {
    // A batch of different lengths whose units run longest first: the chunk is the clusters'
    // even share of all tiles, so the full chunks never outnumber the cluster slots, and the
    // shorter last chunks fill the slots as they free.
    const int64_t share = cdiv(cdiv(total, kTileTokens) * p.row_tiles, slots);
    best_tiles = share < 1 ? 1 : (share > max_tiles ? max_tiles : share);
    if (cdiv(max_tiles, best_tiles) > kMaxSplits) best_tiles = cdiv(max_tiles, kMaxSplits);
  } else {
    // Pick the chunk (in 64-token tiles) that minimises the estimated makespan:
    // waves of units x (tiles per chunk + a fixed per-unit cost of ~4 tiles for the
    // query load, pipeline fill and partial write-back), plus the combine's
    // re-read of the partials (~0.5 tile-equivalents per split per row tile).
    double best = 1e300;
    for (int64_t ct = 1; ct <= max_tiles; ++ct) {
      const int64_t splits = cdiv(max_tiles, ct);
      if (splits > kMaxSplits) continue;
      int64_t units;
      if (ragged) units = p.row_tiles * (cdiv(total, ct * kTileTokens) + d->num_seqs / 2);
      else units = (int64_t)d->num_seqs * p.row_tiles * splits;
      const double waves = (double)cdiv(units, slots);
      const double cost = waves * (double)(ct + 4) + 0.5 * (double)splits * p.row_tiles * d->num_seqs / slots;
      if (cost < best - 1e-9) {
        best = cost;
        best_tiles = ct;
      }
    }
  }
  p.chunk_tokens = (int32_t)(best_tiles * kTileTokens);
  p.num_splits = (int32_t)cdiv(max_n, p.chunk_tokens);
  const int64_t units = (int64_t)d->num_seqs * p.row_tiles * p.num_splits;
  p.ctas = (int32_t)(simt ? units : 2 * units);
  const int64_t rows = (int64_t)d->num_seqs * R;
  const int64_t o_bytes = (int64_t)p.num_splits * rows * kDLatent * 2;  // fp16 partials
  const int64_t l_bytes = (int64_t)p.num_splits * rows * 4;
  p.workspace_bytes = cdiv(o_bytes, 256) * 256 + cdiv(l_bytes, 256) * 256;
  *plan = p;
  return MLA_OK;
}

namespace {
int current_sms(int32_t* sms) {
  int dev = 0, n = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_NO_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return MLA_ERR_NO_DEVICE;
  if (major != 10) return MLA_ERR_NO_DEVICE;
  *sms = n;
  return MLA_OK;
}
}  // namespace

extern "C" int mla_verify_workspace_size(const mla_verify_desc* d, size_t* bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARGUMENT;
  int rc = check_desc(d);
  if (rc) return rc;
  int32_t sms = 0;
  rc = current_sms(&sms);
  if (rc) return rc;
  mla_verify_plan_t p;
  rc = mla_verify_plan(d, sms, &p);
  if (rc) return rc;
  *bytes = (size_t)p.workspace_bytes;
  return MLA_OK;
}

namespace {
// Checks, plans and launches the split (attention) kernel; *partials receive the workspace
// layout. Shared by mla_verify_attn and mla_verify_attn_partials.
int run_splits(const mla_verify_desc* d, const void* q, const void* kv_pool, const int32_t* slot_table,
               const int32_t* seq_lens, const int32_t* tree_parent, void* workspace, size_t workspace_bytes,
               int32_t* dev_status, cudaStream_t s, mla_verify_plan_t* plan_out, VerifyArgs* args_out,
               const int64_t* prefix_base = nullptr, const int32_t* tree_slots = nullptr,
               const int32_t* tree_sizes = nullptr) {
  const bool hybrid = prefix_base != nullptr;
  int rc = check_desc(d);
  if (rc) return rc;
  if (!q || !kv_pool || !seq_lens || !tree_parent || !workspace) return MLA_ERR_INVALID_ARGUMENT;
  if (hybrid ? (!tree_slots || !aligned(prefix_base, 8) || !aligned(tree_slots, 4))
             : (!slot_table || !aligned(slot_table, 4)))
    return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(kv_pool, 16) || !aligned(workspace, 256) || !aligned(seq_lens, 4) ||
      !aligned(tree_parent, 4) || !aligned(tree_sizes, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  const bool debug = (d->flags & MLA_FLAG_DEBUG_CHECKS) != 0;
  if (debug && !dev_status) return MLA_ERR_INVALID_ARGUMENT;
  int32_t sms = 0;
  rc = current_sms(&sms);
  if (rc) return rc;
  mla_verify_plan_t p;
  rc = mla_verify_plan(d, sms, &p);
  if (rc) return rc;
  if (workspace_bytes < (size_t)p.workspace_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (p.kernel == 0 && !tc_kernel_supported()) return MLA_ERR_UNSUPPORTED;

  const int64_t rows = (int64_t)d->num_seqs * d->num_nodes * d->num_heads;
  VerifyArgs a;
  memset(&a, 0, sizeof a);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.kv = static_cast<const __nv_bfloat16*>(kv_pool);
  a.slot_table = hybrid ? nullptr : slot_table;
  a.prefix_base = prefix_base;
  a.tree_slots = tree_slots;
  a.tree_sizes = tree_sizes;
  a.hybrid = hybrid ? 1 : 0;
  a.early_prefix = (d->flags & MLA_FLAG_PREFIX_STABLE) ? 1 : 0;
  // Several sequences: the tcgen05 kernel orders its units longest first from the lengths it
  // reads after the programmatic-launch wait (so not with the early prefix gather).
  a.lpt = (p.kernel == 0 && d->num_seqs >= 2 && d->num_seqs <= kLptMaxSeqs && !a.early_prefix) ? 1 : 0;
  a.seq_lens = seq_lens;
  a.tree_parent = tree_parent;
  a.part_o = static_cast<__half*>(workspace);
  const int64_t o_bytes = (int64_t)p.num_splits * rows * kDLatent * 2;
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + cdiv(o_bytes, 256) * 256);
  a.dev_status = dev_status;
  a.num_slots = d->num_slots;
  a.rows = rows;
  a.B = d->num_seqs;
  a.T = d->num_nodes;
  a.H = d->num_heads;
  a.stride = d->slot_table_stride;
  a.max_seq_len = d->max_seq_len;
  a.chunk = p.chunk_tokens;
  a.splits = p.num_splits;
  a.row_tiles = p.row_tiles;
  a.rows_per_tile = p.rows_per_tile;
  a.debug = debug ? 1 : 0;
  a.scale = d->softmax_scale;
  a.scale_log2 = d->softmax_scale * 1.4426950408889634f;

  if (debug && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess) return MLA_ERR_CUDA;
  cudaError_t e = p.kernel == 1 ? launch_verify_simt(a, s) : launch_verify_tc(a, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  *plan_out = p;
  *args_out = a;
  return MLA_OK;
}

// With debug checks: wait for the stream and turn a non-zero device status into an error.
int finish_debug(const mla_verify_desc* d, int32_t* dev_status, cudaStream_t s) {
  if (!(d->flags & MLA_FLAG_DEBUG_CHECKS)) return MLA_OK;
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, dev_status, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  return h != 0 ? MLA_ERR_DEVICE_CHECK : MLA_OK;
}
}  // namespace

extern "C" int mla_verify_attn(const mla_verify_desc* d, const void* q, const void* kv_pool,
                               const int32_t* slot_table, const int32_t* seq_lens, const int32_t* tree_parent,
                               void* out, float* lse, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, mla_stream_t stream) {
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) {
    const int rc = check_desc(d);
    return rc ? rc : MLA_ERR_INVALID_ARGUMENT;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mla_verify_plan_t p;
  VerifyArgs a;
  int rc = run_splits(d, q, kv_pool, slot_table, seq_lens, tree_parent, workspace, workspace_bytes, dev_status, s,
                      &p, &a);
  if (rc) return rc;
  cudaError_t e = launch_combine(p.num_splits, a.rows, kDLatent, a.part_o, MLA_DTYPE_F16, a.part_lse, out, lse,
                                 d->out_dtype, /*dependent=*/true, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return finish_debug(d, dev_status, s);
}

extern "C" int mla_verify_attn_partials(const mla_verify_desc* d, const void* q, const void* kv_pool,
                                        const int32_t* slot_table, const int32_t* seq_lens,
                                        const int32_t* tree_parent, void* workspace, size_t workspace_bytes,
                                        int32_t* dev_status, mla_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mla_verify_plan_t p;
  VerifyArgs a;
  int rc = run_splits(d, q, kv_pool, slot_table, seq_lens, tree_parent, workspace, workspace_bytes, dev_status, s,
                      &p, &a);
  if (rc) return rc;
  return finish_debug(d, dev_status, s);
}

extern "C" int mla_verify_attn_hybrid(const mla_verify_desc* d, const void* q, const void* kv_pool,
                                      const int64_t* prefix_base, const int32_t* tree_slots, const int32_t* seq_lens,
                                      const int32_t* tree_parent, void* out, float* lse, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, mla_stream_t stream) {
  if (!d) return MLA_ERR_INVALID_ARGUMENT;
  if (!prefix_base) return MLA_ERR_INVALID_ARGUMENT;
  mla_verify_desc dh = *d;  // there is no slot table: its stride only has to pass the shared checks
  dh.slot_table_stride = (int32_t)((int64_t)d->max_seq_len + d->num_nodes > 0x7fffffff
                                       ? 0x7fffffff
                                       : (int64_t)d->max_seq_len + d->num_nodes);
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) {
    const int rc = check_desc(&dh);
    return rc ? rc : MLA_ERR_INVALID_ARGUMENT;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mla_verify_plan_t p;
  VerifyArgs a;
  int rc = run_splits(&dh, q, kv_pool, nullptr, seq_lens, tree_parent, workspace, workspace_bytes, dev_status, s,
                      &p, &a, prefix_base, tree_slots);
  if (rc) return rc;
  cudaError_t e = launch_combine(p.num_splits, a.rows, kDLatent, a.part_o, MLA_DTYPE_F16, a.part_lse, out, lse,
                                 d->out_dtype, /*dependent=*/true, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return finish_debug(d, dev_status, s);
}

extern "C" int mla_verify_attn_ragged(const mla_verify_desc* d, const void* q, const void* kv_pool,
                                      const int32_t* slot_table, const int32_t* seq_lens, const int32_t* tree_sizes,
                                      const int32_t* tree_parent, void* out, float* lse, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, mla_stream_t stream) {
  if (!tree_sizes) {
    const int rc = check_desc(d);
    return rc ? rc : MLA_ERR_INVALID_ARGUMENT;
  }
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) {
    const int rc = check_desc(d);
    return rc ? rc : MLA_ERR_INVALID_ARGUMENT;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  mla_verify_plan_t p;
  VerifyArgs a;
  int rc = run_splits(d, q, kv_pool, slot_table, seq_lens, tree_parent, workspace, workspace_bytes, dev_status, s,
                      &p, &a, nullptr, nullptr, tree_sizes);
  if (rc) return rc;
  cudaError_t e = launch_combine(p.num_splits, a.rows, kDLatent, a.part_o, MLA_DTYPE_F16, a.part_lse, out, lse,
                                 d->out_dtype, /*dependent=*/true, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  return finish_debug(d, dev_status, s);
}

extern "C" int mla_verify_combine(int32_t num_splits, int64_t rows, int32_t d_v, const void* part_o,
                                  int32_t part_dtype, const float* part_lse, void* out, float* lse,
                                  int32_t out_dtype, mla_stream_t stream) {
  if (part_dtype != MLA_DTYPE_F32 && part_dtype != MLA_DTYPE_F16) return MLA_ERR_INVALID_ARGUMENT;
  if (num_splits < 1 || rows < 0 || d_v < 4 || d_v % 4 != 0 || d_v > 1024) return MLA_ERR_INVALID_ARGUMENT;
  if (rows > (1ll << 31) - 1) return MLA_ERR_UNSUPPORTED;
  if (out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_F32) return MLA_ERR_INVALID_ARGUMENT;
  if (rows > 0 && (!part_o || !part_lse || !out)) return MLA_ERR_INVALID_ARGUMENT;
  if (!aligned(part_o, 16) || !aligned(out, 16) || !aligned(part_lse, 4) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARGUMENT;
  cudaError_t e = launch_combine(num_splits, rows, d_v, part_o, part_dtype, part_lse, out, lse, out_dtype,
                                 /*dependent=*/false, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" const char* mla_verify_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported shape or configuration";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA runtime or launch error";
    case MLA_ERR_DEVICE_CHECK: return "device-side input check failed (see dev_status bits)";
    case MLA_ERR_NO_DEVICE: return "no usable sm_103 device is current";
    default: return "unknown status";
  }
}
