/*
 * mla_kv_ops.h -- the KV-pool steps on either side of tree verification for
 * DDTree speculative decoding over a page_size=1 MLA latent pool.
 *
 * Same pool, slot-table and sequence conventions as mla_verify.h: the pool is
 * bf16 [slots][576] (1152-byte rows); slot_table is int32 [num_seqs][stride];
 * sequence b has a prefix of L_b = seq_lens[b] tokens at slot_table[b][0, L_b)
 * and its T = num_nodes tree nodes at slot_table[b][L_b, L_b + T); a seq_lens
 * entry outside [0, max_seq_len] is clamped (and reported under `debug`).
 *
 * All functions enqueue on `stream`, allocate nothing, never synchronise and
 * are graph-capturable. They return MLA_OK, MLA_ERR_INVALID_ARGUMENT (null or
 * misaligned pointer, bad size) or MLA_ERR_CUDA (launch failure). With a
 * non-NULL dev_status and debug != 0, device-side checks OR MLA_CHECK_* bits
 * into *dev_status (which the caller zeroes); offending entries are skipped,
 * never dereferenced.
 */
#ifndef MLA_KV_OPS_H
#define MLA_KV_OPS_H

#include <stddef.h>
#include <stdint.h>

#include "mla_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_tree_kv_append -- write the tree nodes' latent rows into the slots the
 * slot table gives them, before verification (the tree KV lives in the pool:
 * "The Moment of Certainty", The Final Piece, on accepted nodes being scattered
 * across the cache):
 *   for b < num_seqs, j < num_nodes:
 *     pool[slot_table[b][L_b + j]] = tree_kv[b * num_nodes + j]
 *   pool     device bf16 [num_slots][576], 16-byte aligned (written).
 *   tree_kv  device bf16 [num_seqs * num_nodes][576], 16-byte aligned.
 * A slot outside [0, num_slots) is skipped (MLA_CHECK_BAD_SLOT under debug).
 * Two nodes sharing a slot leave one of the two rows there (unspecified which).
 */
int mla_tree_kv_append(void *pool, int64_t num_slots, const void *tree_kv, const int32_t *slot_table,
                       const int32_t *seq_lens, int32_t num_seqs, int32_t num_nodes, int32_t stride,
                       int32_t max_seq_len, int32_t debug, int32_t *dev_status, mla_stream_t stream);

/*
 * mla_tree_accept_commit -- after verification, make the accepted path part of
 * the prefix (accepted nodes are non-contiguous in the verify block: "The
 * Moment of Certainty", The Final Piece). For each sequence b with
 * n = num_accepted[b] and path a = accepted[b][0, n) (node indices, root first):
 *   slot_table[b][L_b + k]     = old slot of node a[k]          for k < n
 *   slot_table[b][L_b + n + i] = old slot of the i-th rejected node, in node order
 *   seq_lens[b]                = L_b + n
 * so the tree block stays a permutation of its old slots (the rejected nodes'
 * slots can be reused by the next tree). The path is validated: 0 <= n <= T,
 * parent[a[0]] == -1 and parent[a[k]] == a[k-1]; an invalid path leaves the
 * sequence unchanged (MLA_CHECK_BAD_PARENT under debug), as does a prefix
 * length that would exceed max_seq_len (MLA_CHECK_BAD_LENGTH).
 *   slot_table   device int32 [num_seqs][stride] (updated in place).
 *   seq_lens     device int32 [num_seqs] (updated in place).
 *   tree_parent  device int32 [num_seqs][num_nodes], as for mla_verify_attn.
 *   accepted     device int32 [num_seqs][num_nodes]; entries past n are ignored.
 *   num_accepted device int32 [num_seqs].
 * num_nodes must be in [1, 64] and stride >= max_seq_len + num_nodes.
 */
int mla_tree_accept_commit(int32_t *slot_table, int32_t *seq_lens, const int32_t *tree_parent,
                           const int32_t *accepted, const int32_t *num_accepted, int32_t num_seqs,
                           int32_t num_nodes, int32_t stride, int32_t max_seq_len, int32_t debug,
                           int32_t *dev_status, mla_stream_t stream);

/*
 * mla_kv_compact -- Tier-0 KV defragmentation: keep each request's KV
 * contiguous in the pool ("The Moment of Reckoning (User Challenge...)",
 * Output, item 4). Copies each sequence's visible rows, in logical order, into
 * one contiguous range of a destination pool and points the slot table there:
 *   for b < num_seqs, t < n_b = L_b + num_nodes:
 *     dst_pool[dst_base[b] + t] = src_pool[slot_table[b][t]]
 *     new_slot_table[b][t]      = dst_base[b] + t     (when new_slot_table != NULL)
 *   src_pool        device bf16 [src_slots][576]; dst_pool device bf16 [dst_slots][576];
 *                   both 16-byte aligned; they must not overlap.
 *   dst_base        device int64 [num_seqs]: first destination slot of each sequence;
 *                   [dst_base[b], dst_base[b] + n_b) must lie in [0, dst_slots) and the
 *                   ranges of different sequences must not overlap.
 *   new_slot_table  device int32 [num_seqs][stride] or NULL; it may be slot_table itself
 *                   (each entry is read before it is rewritten). dst_slots <= 2^31 - 1.
 * A source slot outside [0, src_slots) or a destination row outside [0, dst_slots)
 * is skipped (MLA_CHECK_BAD_SLOT under debug). After it, mla_verify_attn over
 * (dst_pool, new_slot_table) returns exactly what it returned over
 * (src_pool, slot_table).
 */
int mla_kv_compact(const void *src_pool, int64_t src_slots, void *dst_pool, int64_t dst_slots,
                   const int32_t *slot_table, int32_t *new_slot_table, const int32_t *seq_lens,
                   const int64_t *dst_base, int32_t num_seqs, int32_t num_nodes, int32_t stride,
                   int32_t max_seq_len, int32_t debug, int32_t *dev_status, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_KV_OPS_H */
