"""Pins of the KV-pool step oracles (tree-KV append, accept-commit, Tier-0 compaction) on the CPU.

Each definition in ``oracle/__init__.py`` is checked against something other than itself: the
float64 attention oracle (whose own pins live in test_oracle_pins.py), or structural facts that
a mistake would break (rows land where the table says, nothing is lost, order is path order).
"""
import numpy as np
import pytest

import oracle
from speculative_decode_mla_gb300 import workloads as W

SCALE = W.SOFTMAX_SCALE


@pytest.fixture(scope="module", autouse=True)
def built():
    oracle.build()


def rows_of(p, b, nodes):
    """Global query rows (all heads) of the given nodes of sequence b."""
    return [(b * p.T + i) * p.H + h for i in nodes for h in range(p.H)]


# ------------------------------------------------------------------ compaction
def test_compaction_preserves_attention_bitwise():
    p = W.custom_problem([300, 41, 777], 7, 3, seed=51, pool_slack=100)
    n = p.seq_lens.astype(np.int64) + p.T
    base = np.array([5, 5 + int(n[0]) + 9, 5 + int(n[0]) + 9 + int(n[1]) + 1], dtype=np.int64)
    dst_slots = int(base[-1] + n[-1] + 3)
    dst, table = oracle.kv_compact(p.kv, p.slot_table, p.seq_lens, p.T, base, dst_slots)
    o0, l0 = oracle.verify_problem(p, SCALE)
    o1, l1 = oracle.verify(p.seq_lens, table, p.tree_parent, p.q, dst, num_heads=p.H, scale=SCALE)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_compaction_makes_each_sequence_contiguous_and_touches_nothing_else():
    p = W.custom_problem([100, 0, 64], 5, 2, seed=52, pool_slack=10)
    n = p.seq_lens.astype(np.int64) + p.T
    base = np.array([0, int(n[0]) + 4, int(n[0]) + int(n[1]) + 10], dtype=np.int64)
    dst_slots = int(base[-1] + n[-1] + 6)
    dst, table = oracle.kv_compact(p.kv, p.slot_table, p.seq_lens, p.T, base, dst_slots)
    used = np.zeros(dst_slots, dtype=bool)
    for b in range(p.B):
        rng = np.arange(base[b], base[b] + n[b])
        assert np.array_equal(table[b, :n[b]], rng)                     # contiguous, in logical order
        assert np.array_equal(table[b, n[b]:], p.slot_table[b, n[b]:])  # beyond N_b: untouched
        for t in range(n[b]):
            assert np.array_equal(dst[base[b] + t], p.kv[p.slot_table[b, t]])
        used[rng] = True
    assert not dst[~used].any()


# ------------------------------------------------------------------ tree-KV append
def test_append_then_verify_equals_verify_with_rows_in_place():
    p = W.custom_problem([200, 33], 6, 4, seed=53, pool_slack=20)
    tree_kv = np.stack([p.kv[p.slot_table[b, p.seq_lens[b] + j]] for b in range(p.B) for j in range(p.T)])
    holed = p.kv.copy()
    for b in range(p.B):
        holed[p.slot_table[b, p.seq_lens[b]:p.seq_lens[b] + p.T]] = 0  # the tree rows are not there yet
    filled = oracle.tree_kv_append(holed, tree_kv, p.slot_table, p.seq_lens, p.T)
    assert np.array_equal(filled, p.kv)
    o0, l0 = oracle.verify_problem(p, SCALE)
    o1, l1 = oracle.verify(p.seq_lens, p.slot_table, p.tree_parent, p.q, filled, num_heads=p.H, scale=SCALE)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


# ------------------------------------------------------------------ accept-commit
def commit(p, accepted, n):
    acc = np.full((p.B, p.T), -1, dtype=np.int32)
    for b, path in enumerate(accepted):
        acc[b, :len(path)] = path
    return oracle.tree_accept_commit(p.slot_table, p.seq_lens, p.tree_parent, acc, np.array(n, dtype=np.int32),
                                     max_seq_len=p.max_seq_len + p.T)


def some_path(parent, leaf):
    path = []
    while leaf >= 0:
        path.append(leaf)
        leaf = int(parent[leaf])
    return path[::-1]


def test_commit_of_a_chain_accepting_everything_keeps_the_table():
    p = W.custom_problem([50], 8, 2, tree="chain", seed=54)
    table, lens, ok = commit(p, [list(range(8))], [8])
    assert ok.all() and lens[0] == 58 and np.array_equal(table, p.slot_table)


def test_commit_puts_the_path_behind_the_prefix_and_loses_no_slot():
    p = W.custom_problem([120, 7], 12, 2, seed=55)
    paths = [some_path(p.tree_parent[0], 11), some_path(p.tree_parent[1], 9)]
    table, lens, ok = commit(p, paths, [len(x) for x in paths])
    assert ok.all()
    for b, path in enumerate(paths):
        L, n = int(p.seq_lens[b]), len(path)
        assert lens[b] == L + n
        assert np.array_equal(table[b, :L], p.slot_table[b, :L])          # the prefix is untouched
        for k, node in enumerate(path):                                   # path order, root first
            assert table[b, L + k] == p.slot_table[b, L + node]
        rejected = [j for j in range(p.T) if j not in path]
        assert list(table[b, L + n:L + p.T]) == [int(p.slot_table[b, L + j]) for j in rejected]
        assert sorted(table[b, L:L + p.T]) == sorted(p.slot_table[b, L:L + p.T])


def test_committed_path_attends_causally_like_it_did_in_the_tree():
    """Node a_k saw the prefix and a_0..a_k in the tree; after the commit those are positions < L + k + 1,
    so re-verifying the accepted nodes as a chain over the old prefix gives the same attention."""
    p = W.custom_problem([90], 10, 3, seed=56)
    path = some_path(p.tree_parent[0], 9)
    n = len(path)
    table, lens, ok = commit(p, [path], [n])
    assert ok.all()
    before, lb = oracle.verify_problem(p, SCALE, rows=rows_of(p, 0, path))
    L = int(p.seq_lens[0])
    chain_table = table[:, :L + n].copy()
    q_path = p.q.reshape(p.T, p.H, -1)[path]
    after, la = oracle.verify(p.seq_lens, chain_table, np.array([[-1] + list(range(n - 1))], dtype=np.int32),
                              q_path, p.kv, num_heads=p.H, scale=SCALE)
    assert np.array_equal(before, after) and np.array_equal(lb, la)


@pytest.mark.parametrize("case", ["wrong_parent", "repeat", "too_many", "not_from_root", "past_max"])
def test_invalid_paths_leave_the_sequence_unchanged(case):
    p = W.custom_problem([40], 6, 1, tree="chain", seed=57)
    path, n, max_len = [0, 1, 2], 3, p.max_seq_len + p.T
    if case == "wrong_parent":
        path = [0, 2, 1]
    elif case == "repeat":
        path = [0, 0]
        n = 2
    elif case == "too_many":
        n = 7
    elif case == "not_from_root":
        path = [1, 2]
        n = 2
    acc = np.full((1, p.T), -1, dtype=np.int32)
    acc[0, :len(path)] = path
    if case == "past_max":
        max_len = int(p.seq_lens[0]) + 2
    table, lens, ok = oracle.tree_accept_commit(p.slot_table, p.seq_lens, p.tree_parent, acc,
                                                np.array([n], dtype=np.int32), max_len)
    assert not ok.any() and np.array_equal(table, p.slot_table) and np.array_equal(lens, p.seq_lens)
