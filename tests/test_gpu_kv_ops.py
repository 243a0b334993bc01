"""GPU parity of the KV-pool steps (include/mla_kv_ops.h) against their numpy oracles, through the C ABI.

All three are integer / copy work, so the bar is bit-exact. Integration: verify attention over the
compacted pool is bit-identical to verify over the original one.
"""
import numpy as np
import pytest

import oracle
from _helpers import device_problem, to_dev
from speculative_decode_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decode_mla_gb300 import _build
    _build.build()
    oracle.build()


def bf16(a):
    import torch
    return to_dev(a.view(np.int16)).view(torch.bfloat16)


def host_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_tree_kv_append_bitwise():
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([300, 0, 77, 1024], 11, 2, seed=61, pool_slack=50, stride_pad=11)
    rng = np.random.default_rng(0)
    tree_kv = rng.integers(0, 1 << 16, size=(p.B * p.T, W.D_K), dtype=np.uint16)
    want = oracle.tree_kv_append(p.kv, tree_kv, p.slot_table, p.seq_lens, p.T)
    pool = bf16(p.kv.copy())
    m.tree_kv_append(pool, bf16(tree_kv), to_dev(p.slot_table), to_dev(p.seq_lens), max_seq_len=p.max_seq_len)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(pool), want)


def test_tree_kv_append_reports_and_skips_a_bad_slot():
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([40], 4, 1, seed=62, pool_slack=4, stride_pad=4)
    table = p.slot_table.copy()
    table[0, 40 + 2] = p.num_slots + 5  # node 2's slot is out of range
    tree_kv = np.full((p.T, W.D_K), 0x3F80, dtype=np.uint16)
    pool = bf16(p.kv.copy())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.tree_kv_append(pool, bf16(tree_kv), to_dev(table), to_dev(p.seq_lens), max_seq_len=p.max_seq_len,
                     debug=True, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & m.CHECK_BAD_SLOT
    got = host_bits(pool)
    for j in (0, 1, 3):
        assert (got[table[0, 40 + j]] == 0x3F80).all()
    keep = np.ones(p.num_slots, dtype=bool)
    keep[[table[0, 40 + j] for j in (0, 1, 3)]] = False
    assert np.array_equal(got[keep], p.kv[keep])


def random_paths(p, rng, invalid_every=0):
    acc = np.full((p.B, p.T), -1, dtype=np.int32)
    n = np.zeros(p.B, dtype=np.int32)
    for b in range(p.B):
        leaf = int(rng.integers(0, p.T))
        path = []
        while leaf >= 0:
            path.append(leaf)
            leaf = int(p.tree_parent[b, leaf])
        path = path[::-1][:int(rng.integers(0, len(path) + 1))]
        if invalid_every and b % invalid_every == 1 and len(path) >= 2:
            path[0], path[1] = path[1], path[0]
        acc[b, :len(path)] = path
        n[b] = len(path)
    return acc, n


@pytest.mark.parametrize("T", [1, 9, 64])
def test_tree_accept_commit_bitwise(T):
    import torch
    import speculative_decode_mla_gb300 as m
    lens = [0, 5, 300, 64, 1000, 17, 2048, 3]
    p = W.custom_problem(lens, T, 1, seed=63 + T, stride_pad=T)
    rng = np.random.default_rng(T)
    acc, n = random_paths(p, rng, invalid_every=3)
    max_len = p.max_seq_len + T
    want_t, want_l, valid = oracle.tree_accept_commit(p.slot_table, p.seq_lens, p.tree_parent, acc, n, max_len)
    st_d, sl_d = to_dev(p.slot_table), to_dev(p.seq_lens)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.tree_accept_commit(st_d, sl_d, to_dev(p.tree_parent), to_dev(acc), to_dev(n), max_seq_len=max_len,
                         debug=True, dev_status=status)
    torch.cuda.synchronize()
    assert np.array_equal(st_d.cpu().numpy(), want_t)
    assert np.array_equal(sl_d.cpu().numpy(), want_l)
    assert bool(status.item() & m.CHECK_BAD_PARENT) == (not valid.all())


def test_commit_then_verify_matches_the_oracle():
    """Accept a path, then verify a fresh tree on top of the new prefix: GPU and oracle agree."""
    import torch
    import speculative_decode_mla_gb300 as m
    from _helpers import TOL_LSE_ABS, TOL_MAX_ABS, TOL_REL_L2
    p = W.custom_problem([700, 90], 8, 4, seed=64, stride_pad=8)
    rng = np.random.default_rng(3)
    acc, n = random_paths(p, rng)
    max_len = p.max_seq_len + p.T
    st_d, sl_d = to_dev(p.slot_table), to_dev(p.seq_lens)
    m.tree_accept_commit(st_d, sl_d, to_dev(p.tree_parent), to_dev(acc), to_dev(n), max_seq_len=max_len)
    table, lens, _ = oracle.tree_accept_commit(p.slot_table, p.seq_lens, p.tree_parent, acc, n, max_len)
    # the next tree: the rejected nodes' slots come first in the block, the rest are unused slots
    new_table = table.copy()
    spare = iter(range(p.num_slots, p.num_slots + 64))
    kv = np.concatenate([p.kv, W.normal_bf16(99, 64 * W.D_K).reshape(64, W.D_K)])
    for b in range(p.B):
        for j in range(p.T):
            if lens[b] + j >= table.shape[1] or j >= p.T - n[b]:
                new_table[b, lens[b] + j] = next(spare)
    st_d.copy_(to_dev(new_table))
    o, l = m.verify(bf16(p.q), bf16(kv), st_d, sl_d, to_dev(p.tree_parent), max_seq_len=max_len,
                    out_dtype=m.MLA_DTYPE_F32)
    torch.cuda.synchronize()
    ro, rl = oracle.verify(lens, new_table, p.tree_parent, p.q, kv, num_heads=p.H, scale=W.SOFTMAX_SCALE)
    got = o.cpu().numpy().reshape(ro.shape).astype(np.float64)
    assert np.abs(got - ro).max() <= TOL_MAX_ABS
    assert np.linalg.norm(got - ro) / np.linalg.norm(ro) <= TOL_REL_L2
    assert np.abs(l.cpu().numpy().reshape(-1) - rl).max() <= TOL_LSE_ABS


@pytest.mark.parametrize("in_place", [False, True])
def test_kv_compact_bitwise_and_verify_unchanged(in_place):
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([5000, 0, 130, 2047], 9, 13, seed=65, pool_slack=333, stride_pad=9)
    N = p.seq_lens.astype(np.int64) + p.T
    base = np.concatenate([[7], 7 + np.cumsum(N[:-1] + 3)]).astype(np.int64)
    dst_slots = int(base[-1] + N[-1] + 5)
    want_dst, want_t = oracle.kv_compact(p.kv, p.slot_table, p.seq_lens, p.T, base, dst_slots)
    q, kv, st, sl, tp = device_problem(p)
    ref_o, ref_l = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len + p.T)
    dst = torch.zeros((dst_slots, W.D_K), dtype=torch.bfloat16, device="cuda")
    new_t = st if in_place else torch.full_like(st, -7)
    m.kv_compact(kv, dst, st, sl, to_dev(base), num_nodes=p.T, max_seq_len=p.max_seq_len + p.T,
                 new_slot_table=new_t)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(dst), want_dst)
    nt = new_t.cpu().numpy()
    for b in range(p.B):
        assert np.array_equal(nt[b, :N[b]], want_t[b, :N[b]])
    o, l = m.verify(q, dst, new_t, sl, tp, max_seq_len=p.max_seq_len + p.T)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(l, ref_l)


def test_kv_compact_64k_pool():
    """The 64k workload's pool (151 MB, random slots) compacted: sampled rows and verify bit-identical."""
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.make_problem("64k")
    q, kv, st, sl, tp = device_problem(p)
    ref_o, ref_l = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len)
    N = int(p.seq_lens[0]) + p.T
    dst = torch.empty((N + 128, W.D_K), dtype=torch.bfloat16, device="cuda")
    new_t = torch.full_like(st, -1)
    m.kv_compact(kv, dst, st, sl, to_dev(np.array([64], dtype=np.int64)), num_nodes=p.T,
                 max_seq_len=p.max_seq_len, new_slot_table=new_t)
    torch.cuda.synchronize()
    assert np.array_equal(new_t.cpu().numpy()[0, :N], np.arange(64, 64 + N))
    idx = np.random.default_rng(1).choice(N, size=500, replace=False)
    got = host_bits(dst[torch.from_numpy(64 + idx).cuda()])
    assert np.array_equal(got, p.kv[p.slot_table[0, idx]])
    o, l = m.verify(q, dst, new_t, sl, tp, max_seq_len=p.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(l, ref_l)
