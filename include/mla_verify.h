/*
 * mla_verify.h -- C ABI of the tree-verify MLA attention library (sm_103a).
 *
 * The operation. One verify step of DDTree speculative decoding checks a draft
 * tree of T nodes per sequence against the target model's whole KV cache in one
 * forward pass ("The Moment of Certainty", The Final Piece: the verify block
 * carries a custom tree mask; page_size=1 because accepted tree nodes are not
 * contiguous). For MLA the cache holds one compressed latent row per token
 * ("Diagnosing Latency-Bound Decode", The Technical Depth) and, with page_size=1,
 * every token is reached through its own slot (The Reasoning, Step 4). The
 * prefix needs no mask and can be streamed; only the small tree block takes the
 * visibility bitmask ("The Moment of Certainty", The Path Forward; "The GPU That
 * Wasn't There", The Native Engine Thesis).
 *
 * For sequence b with prefix length L_b, node i < T and head h, the query row
 *   q[(b*T + i)*H + h][0:576]          (512 latent dims, then 64 RoPE dims)
 * attends to the visible positions
 *   V(b, i) = { t < L_b }  U  { L_b + j : j = i or j an ancestor of i },
 * where position t's key row is kv_pool[slot_table[b*stride + t]][0:576] and its
 * value row is the first 512 dims of that same row (absorbed MLA form). With
 * s_t = softmax_scale * <q, k_t>:
 *   out[row][0:512] = sum_t softmax(s)_t * v_t,   lse[row] = ln sum_t exp(s_t).
 * The tree nodes' own latent rows live in the pool too, at
 * slot_table[b*stride + L_b + j] (the caller writes them before the call).
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device (or managed) addresses on the
 *    current device; pointers marked "host" are host addresses.
 *  - The caller owns every buffer, workspace included. mla_verify_attn and
 *    mla_verify_combine allocate nothing, never synchronise the stream (unless
 *    MLA_FLAG_DEBUG_CHECKS is set) and only enqueue kernels on `stream`
 *    (0 = the legacy default stream), so they may be captured in a CUDA graph.
 *  - Return value: MLA_OK (0) or a negative MLA_ERR_* code; nothing is launched
 *    when a host-side check fails. Outputs are then left untouched.
 *  - Inputs are never written. out, lse and workspace must not alias inputs or
 *    each other.
 */
#ifndef MLA_VERIFY_H
#define MLA_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *mla_stream_t;

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARGUMENT = -1,  /* null pointer, bad size, misaligned buffer, bad field */
  MLA_ERR_UNSUPPORTED = -2,       /* d_latent != 512, d_rope != 64, T outside 1..64, ... */
  MLA_ERR_WORKSPACE_TOO_SMALL = -3,
  MLA_ERR_CUDA = -4,              /* a CUDA runtime call or a launch failed */
  MLA_ERR_DEVICE_CHECK = -5,      /* MLA_FLAG_DEBUG_CHECKS found a bad slot, parent or length */
  MLA_ERR_NO_DEVICE = -6          /* no usable sm_103 device is current */
};

/* Element types. out: BF16 or F32. Split partials (mla_verify_combine's part_o): F32 or F16. */
enum mla_dtype { MLA_DTYPE_BF16 = 0, MLA_DTYPE_F32 = 1, MLA_DTYPE_F16 = 2 };

enum mla_flags {
  /* Check every slot, parent and prefix length on the device, write the findings
   * to dev_status, synchronise the stream and return MLA_ERR_DEVICE_CHECK when
   * something was wrong. Without this flag bad values are clamped into range on
   * the device (no fault, no report). Not capturable in a CUDA graph. */
  MLA_FLAG_DEBUG_CHECKS = 1 << 0,
  /* Run the plain SIMT reference kernel (fp32 FMA, no tensor cores) instead of
   * the tcgen05 kernel. Same partial layout and combine; for tests and debugging. */
  MLA_FLAG_SIMT = 1 << 1,
  /* A promise from the caller: the kernel enqueued just before this call on the
   * stream does not write seq_lens, the prefix part of the slot table (entries
   * [0, L_b)), prefix_base, or the prefix rows of kv_pool. The tcgen05 kernel is
   * launched as a programmatic dependent of that kernel; with this flag its
   * gather starts on the first prefix tiles before that kernel has finished
   * (everything else -- q, the tree, tree sizes and slots -- is still read only
   * after it). Typical use: consecutive layers of one decode step, whose
   * prefixes were written by earlier steps. Results are identical with or
   * without the flag when the promise holds. */
  MLA_FLAG_PREFIX_STABLE = 1 << 2
};

/* Bits the device checks may set in *dev_status. */
enum mla_device_check {
  MLA_CHECK_BAD_SLOT = 1 << 0,    /* slot_table entry outside [0, num_slots) */
  MLA_CHECK_BAD_PARENT = 1 << 1,  /* tree_parent[i] outside [-1, i) */
  MLA_CHECK_BAD_LENGTH = 1 << 2,  /* seq_lens[b] outside [0, max_seq_len] */
  MLA_CHECK_TIMEOUT = 1 << 3      /* a bounded wait inside a kernel gave up */
};

/* Shapes of one call. Every field is host-visible, so the launch plan is a pure
 * function of this struct (graph-capture safe). */
typedef struct mla_verify_desc {
  int32_t num_seqs;           /* B >= 1 */
  int32_t num_nodes;          /* T, tree nodes per sequence, 1..64 (same for every sequence) */
  int32_t num_heads;          /* H >= 1 */
  int32_t d_latent;           /* must be 512 (value width) */
  int32_t d_rope;             /* must be 64 (key row = d_latent + d_rope = 576) */
  int32_t slot_table_stride;  /* int32 entries per sequence row of slot_table; >= max_seq_len + T */
  int64_t num_slots;          /* rows in kv_pool, 1 .. 2^31 - 1 */
  int32_t max_seq_len;        /* host-known upper bound of every seq_lens[b] */
  float softmax_scale;        /* finite and > 0; 1/sqrt(192) for the absorbed MLA head */
  int32_t out_dtype;          /* MLA_DTYPE_BF16 (default) or MLA_DTYPE_F32 */
  int32_t flags;              /* MLA_FLAG_* */
  int32_t num_splits;         /* 0: planner decides; > 0: force this many KV splits */
  int64_t total_tokens_hint;  /* 0, or a host-known estimate of sum_b (L_b + T), to size splits */
} mla_verify_desc;

/* The launch plan chosen for a desc (for introspection and tests). */
typedef struct mla_verify_plan_t {
  int32_t kernel;         /* 0: tcgen05 kernel, 1: SIMT reference kernel */
  int32_t num_splits;     /* KV partitions per (sequence, row tile); partial slots per row */
  int32_t chunk_tokens;   /* positions per partition, a multiple of 64 (the KV tile) */
  int32_t row_tiles;      /* row tiles per sequence */
  int32_t rows_per_tile;  /* query rows per tile */
  int32_t ctas;           /* CTAs launched by the attention kernel */
  int64_t workspace_bytes;
} mla_verify_plan_t;

/*
 * mla_verify_plan -- the split plan for `desc` on a GPU with `num_sms` SMs.
 * Pure host function (no CUDA call; callable without a GPU). The KV range of
 * every sequence is cut into chunks of chunk_tokens positions (multiples of the
 * 64-position KV tile) so that the (sequence, row tile, chunk) units fill all SMs at
 * batch 1 (split-KV / flash-decoding; the pages' batch-1 verify had "low
 * parallelism", "The Moment of Certainty", Message 12190: The Synthesis).
 * For a batch of 2..64 sequences the tcgen05 kernel takes its units longest first;
 * when total_tokens_hint is below B x (max_seq_len + T) (lengths differ), the
 * chunk is the cluster slots' even share of all tiles. The hint only sizes the
 * plan: any lengths give correct results.
 * Returns MLA_OK or MLA_ERR_INVALID_ARGUMENT / MLA_ERR_UNSUPPORTED.
 */
int mla_verify_plan(const mla_verify_desc *desc, int32_t num_sms, mla_verify_plan_t *plan);

/*
 * mla_verify_workspace_size -- device workspace bytes mla_verify_attn needs for
 * `desc` on the current device (queries its SM count). *bytes receives the size.
 * Layout (owned by the library, opaque to the caller): partial outputs
 * float16 [num_splits][B*T*H][512] (each normalised over its own part, so
 * |o| <= max |v|), then partial lse float32 [num_splits][B*T*H] at the next
 * 256-byte boundary. Returns MLA_OK, MLA_ERR_INVALID_ARGUMENT, MLA_ERR_UNSUPPORTED
 * or MLA_ERR_NO_DEVICE.
 */
int mla_verify_workspace_size(const mla_verify_desc *desc, size_t *bytes);

/*
 * mla_verify_attn -- tree-verify attention (the operation above).
 *   q           device bf16 [B*T][H][576], 16-byte aligned; row (b*T+i)*H+h.
 *   kv_pool     device bf16 [num_slots][576] (1152-byte rows), 16-byte aligned.
 *   slot_table  device int32 [B][slot_table_stride]; entries [0, L_b + T) of row b
 *               are read: prefix slots, then the T tree nodes' slots.
 *   seq_lens    device int32 [B], prefix lengths L_b (tree excluded), <= max_seq_len.
 *   tree_parent device int32 [B][T]; parent[i] in [-1, i) (topological order);
 *               -1 attaches node i to the prefix only (node 0's parent is -1).
 *   out         device [B*T][H][512], bf16 or float32 per desc->out_dtype, 16-byte aligned.
 *   lse         device float32 [B*T][H], natural log, scale included.
 *   workspace   device, >= mla_verify_workspace_size bytes, 256-byte aligned.
 *   dev_status  device int32 or NULL; with MLA_FLAG_DEBUG_CHECKS it must be
 *               non-NULL and receives the OR of MLA_CHECK_* bits (zeroed first).
 *   stream      the stream every kernel is enqueued on.
 * The result does not depend on which physical slots hold the rows: the same
 * logical inputs give bit-identical outputs under any slot permutation.
 */
int mla_verify_attn(const mla_verify_desc *desc, const void *q, const void *kv_pool,
                    const int32_t *slot_table, const int32_t *seq_lens, const int32_t *tree_parent,
                    void *out, float *lse, void *workspace, size_t workspace_bytes,
                    int32_t *dev_status, mla_stream_t stream);

/*
 * mla_verify_attn_partials -- the split stage of mla_verify_attn alone: every
 * (sequence, row tile, chunk) partial of the plan is written to `workspace`,
 * and no combine is launched. With plan = mla_verify_plan(desc, SM count of the
 * current device) and rows = B*T*H, the workspace then holds
 *   part_o   float16 [plan.num_splits][rows][512] at workspace, and
 *   part_lse float32 [plan.num_splits][rows] at the next 256-byte boundary after it,
 * and mla_verify_combine(plan.num_splits, rows, 512, part_o, MLA_DTYPE_F16,
 * part_lse, out, lse, desc->out_dtype, stream) then returns exactly what
 * mla_verify_attn returns for the same inputs. Use it to time or schedule the two
 * stages separately. Arguments, checks and return codes are those of
 * mla_verify_attn without out and lse.
 */
int mla_verify_attn_partials(const mla_verify_desc *desc, const void *q, const void *kv_pool,
                             const int32_t *slot_table, const int32_t *seq_lens, const int32_t *tree_parent,
                             void *workspace, size_t workspace_bytes, int32_t *dev_status,
                             mla_stream_t stream);

/*
 * mla_verify_attn_hybrid -- mla_verify_attn with hybrid addressing: each
 * sequence's prefix is one contiguous range of the pool (base + length) and
 * only the tree tail is addressed per token (page_size=1) -- the variant the
 * pages propose ("Diagnosing Latency-Bound Decode", Broader Implications and
 * Output; "The Moment of Certainty", The Path Forward), e.g. after
 * mla_kv_compact has made the prefix contiguous.
 *   prefix_base device int64 [B]: prefix position t < L_b is slot prefix_base[b] + t;
 *               [prefix_base[b], prefix_base[b] + L_b) must lie in [0, num_slots).
 *   tree_slots  device int32 [B][T]: tree node j of sequence b is slot tree_slots[b][j].
 * There is no slot table: desc->slot_table_stride is ignored. Everything else
 * (arguments, workspace, checks, return codes) is as for mla_verify_attn, and
 * the result is bit-identical to mla_verify_attn over the slot table
 * slot_table[b][t] = prefix_base[b] + t (t < L_b), tree_slots[b][t - L_b] (t >= L_b).
 * Tiles of 64 positions wholly inside the prefix are loaded as 2-D TMA tiles.
 */
int mla_verify_attn_hybrid(const mla_verify_desc *desc, const void *q, const void *kv_pool,
                           const int64_t *prefix_base, const int32_t *tree_slots, const int32_t *seq_lens,
                           const int32_t *tree_parent, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, mla_stream_t stream);

/*
 * mla_verify_attn_ragged -- mla_verify_attn for a batch whose trees differ in
 * size (batched verify with a ragged T per sequence; the pages' drafter builds
 * trees of varying size, "The Moment of Doubt", Input). desc->num_nodes is the
 * largest tree, T_max, and every buffer keeps the mla_verify_attn layout for it;
 * sequence b has T_b = tree_sizes[b] (1 <= T_b <= T_max) nodes:
 *   tree_sizes  device int32 [B].
 *   slot_table  row b holds the prefix, then the T_b tree nodes' slots at [L_b, L_b + T_b).
 *   tree_parent row b: entries [0, T_b) as for mla_verify_attn; the rest are ignored.
 *   q, out, lse rows of nodes j >= T_b are padding: q is not read, out is 0 and lse is -inf.
 * A tree size outside [1, T_max] is clamped (MLA_CHECK_BAD_LENGTH under debug checks).
 * Everything else is as for mla_verify_attn; with every T_b = T_max the result is
 * bit-identical to it.
 */
int mla_verify_attn_ragged(const mla_verify_desc *desc, const void *q, const void *kv_pool,
                           const int32_t *slot_table, const int32_t *seq_lens, const int32_t *tree_sizes,
                           const int32_t *tree_parent, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, int32_t *dev_status, mla_stream_t stream);

/*
 * mla_verify_combine -- LSE-weighted merge of split partials (flash-decoding
 * combine). For each row r:
 *   lse[r] = ln sum_s exp(part_lse[s][r]);  out[r] = sum_s exp(part_lse[s][r] - lse[r]) * part_o[s][r]
 * Partials with part_lse = -inf carry no weight (and their part_o is not read);
 * a row whose partials are all -inf gets lse = -inf and out = 0.
 *   part_o   device [num_splits][rows][d_v], float32 or float16 per part_dtype, each
 *            normalised over its own part; 16-byte aligned.
 *   part_lse device float32 [num_splits][rows].
 *   out      device [rows][d_v], bf16 or float32 per out_dtype, 16-byte aligned.
 *   lse      device float32 [rows] or NULL.
 * d_v must be a positive multiple of 4. This is also the seam for a split of
 * the KV range across GPUs: each GPU's (o, lse) pair is one partial.
 */
int mla_verify_combine(int32_t num_splits, int64_t rows, int32_t d_v, const void *part_o,
                       int32_t part_dtype, const float *part_lse, void *out, float *lse,
                       int32_t out_dtype, mla_stream_t stream);

/*
 * mla_verify_attn_noalloc -- mla_verify_attn for callers that cannot allocate
 * device memory. The pages have no counterpart: this is a library convenience.
 *
 * Some callers cannot provide the workspace mla_verify_attn asks for: a plugin
 * whose host framework hands it only the input and output device pointers and
 * no allocator; a serving process that has already reserved nearly all device
 * memory for its KV pool, so a cudaMalloc would fail; a latency-critical decode
 * loop that cannot afford cudaMalloc/cudaFree, which may synchronise the device.
 * This entry point takes the same arguments as mla_verify_attn minus the
 * workspace, and uses instead a scratch array of MLA_VERIFY_NOALLOC_SCRATCH_BYTES
 * that the library itself holds in device memory (a file-scope __device__
 * array: every GPU on which the library's module is loaded keeps those bytes
 * until the process exits). It calls no allocation routine of any kind.
 *
 * - Set-up: the first call on each device (with that device current) looks up
 *   the array's device address once and caches it. Make that first call before
 *   any stream capture begins on that device. The cached address is kept for
 *   the life of the process, so resetting a device (cudaDeviceReset) after the
 *   first call on it is not supported.
 * - Limit: when the plan for `desc` on the current device needs more than
 *   MLA_VERIFY_NOALLOC_SCRATCH_BYTES of workspace (see
 *   mla_verify_workspace_size), the call returns MLA_ERR_WORKSPACE_TOO_SMALL and
 *   launches nothing.
 * - Sharing: every call on a device uses the same array, and the array keeps
 *   the previous call's contents. Nothing in it needs to start at zero (each
 *   call writes every partial it reads), but two calls whose kernels overlap in
 *   time on the GPU (different streams without ordering between them) race on
 *   the array and corrupt each other's results. Order such calls on one stream
 *   or with events. Calls ordered on one stream are safe back to back, also
 *   with MLA_FLAG_PREFIX_STABLE: that flag lets a call read its prefix inputs
 *   early, but its writes to the array (the split partials) still come after
 *   it has waited for the preceding call's combine to finish.
 * Other arguments, return codes and behaviour are those of mla_verify_attn.
 */
#define MLA_VERIFY_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB */
int mla_verify_attn_noalloc(const mla_verify_desc *desc, const void *q, const void *kv_pool,
                            const int32_t *slot_table, const int32_t *seq_lens, const int32_t *tree_parent,
                            void *out, float *lse, int32_t *dev_status, mla_stream_t stream);

/* A static, human-readable description of a status code. */
const char *mla_verify_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MLA_VERIFY_H */
