"""GPU: verify attention with hybrid addressing (contiguous prefix + per-node tree slots).

The bar: bit-identical to mla_verify_attn over the equivalent slot table (same kernels, same
tile arithmetic; prefix tiles arrive by 2-D TMA instead of the row gather), and within the
parity tolerances of the float64 oracle.
"""
import numpy as np
import pytest

import oracle
from _helpers import assert_close, device_problem, to_dev
from speculative_decode_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCALE = W.SOFTMAX_SCALE


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decode_mla_gb300 import _build
    _build.build()
    oracle.build()


def flags(kernel):
    import speculative_decode_mla_gb300 as m
    return m.MLA_FLAG_SIMT if kernel == "simt" else 0


def hybrid_layout(lens, T, num_slots, seed):
    """Non-overlapping contiguous prefix ranges at random bases, tree nodes at random other slots;
    returns (prefix_base int64 [B], tree_slots int32 [B, T], the equivalent slot table [B, max L + T])."""
    rng = np.random.default_rng(seed)
    B = len(lens)
    free = np.ones(num_slots, dtype=bool)
    base = np.zeros(B, dtype=np.int64)
    cursor = int(rng.integers(0, 50))
    for b in range(B):
        base[b] = cursor
        free[cursor:cursor + lens[b]] = False
        cursor += lens[b] + int(rng.integers(0, 70))
    assert cursor <= num_slots
    spare = rng.permutation(np.flatnonzero(free))
    tree = spare[:B * T].reshape(B, T).astype(np.int32)
    stride = max(lens) + T
    table = np.zeros((B, stride), dtype=np.int32)
    for b in range(B):
        table[b, :lens[b]] = base[b] + np.arange(lens[b])
        table[b, lens[b]:lens[b] + T] = tree[b]
    return base, tree, table


SHAPES = [
    ([0], 1, 1),
    ([63, 64, 65], 4, 3),
    ([1000, 4097, 128], 9, 13),
    ([2048], 64, 2),
]


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"L{s[0]}-T{s[1]}-H{s[2]}" for s in SHAPES])
def test_hybrid_is_bit_identical_to_the_slot_table_path(kernel, shape):
    import torch
    import speculative_decode_mla_gb300 as m
    lens, T, H = shape
    num_slots = sum(lens) + 80 * len(lens) + T * len(lens) + 64
    p = W.custom_problem(lens, T, H, seed=71 + T, pool_slack=num_slots - (sum(lens) + T * len(lens)))
    base, tree, table = hybrid_layout(lens, T, p.num_slots, seed=T + H)
    q, kv, _, sl, tp = device_problem(p)
    ref_o, ref_l = m.verify(q, kv, to_dev(table), sl, tp, max_seq_len=max(lens), flags=flags(kernel))
    o, l = m.verify_hybrid(q, kv, to_dev(base), to_dev(tree), sl, tp, max_seq_len=max(lens), flags=flags(kernel))
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(l, ref_l)
    ro, rl = oracle.verify(p.seq_lens, table, p.tree_parent, p.q, p.kv, num_heads=H, scale=SCALE)
    assert_close(o.float().cpu().numpy().reshape(ro.shape).astype(np.float64), l.cpu().numpy().reshape(-1), ro, rl,
                 f"hybrid {shape}")


def test_hybrid_64k_after_compaction():
    """The 64k pool compacted to one contiguous prefix: the hybrid call (TMA prefix tiles) is
    bit-identical to the slot-table call over the compacted table."""
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.make_problem("64k")
    q, kv, st, sl, tp = device_problem(p)
    L = int(p.seq_lens[0])
    N = L + p.T
    dst = torch.empty((N + 64, W.D_K), dtype=torch.bfloat16, device="cuda")
    new_t = torch.full_like(st, -1)
    m.kv_compact(kv, dst, st, sl, to_dev(np.array([32], dtype=np.int64)), num_nodes=p.T,
                 max_seq_len=p.max_seq_len, new_slot_table=new_t)
    ref_o, ref_l = m.verify(q, dst, new_t, sl, tp, max_seq_len=p.max_seq_len)
    tree = new_t[:, L:L + p.T].contiguous()
    o, l = m.verify_hybrid(q, dst, to_dev(np.array([32], dtype=np.int64)), tree, sl, tp, max_seq_len=p.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(l, ref_l)


def test_hybrid_reports_a_prefix_range_outside_the_pool():
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([300], 4, 2, seed=75, pool_slack=10)
    q, kv, _, sl, tp = device_problem(p)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = to_dev(np.array([p.num_slots - 100], dtype=np.int64))  # 300 prefix rows cannot fit
    tree = to_dev(np.arange(4, dtype=np.int32).reshape(1, 4))
    desc = m.make_desc(1, 4, 2, p.num_slots, 304, 300, flags=m.MLA_FLAG_DEBUG_CHECKS)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty((4, 2, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((4, 2), dtype=torch.float32, device="cuda")
    rc = m.verify_attn_hybrid_raw(desc, q.data_ptr(), kv.data_ptr(), base.data_ptr(), tree.data_ptr(), sl.data_ptr(),
                                  tp.data_ptr(), out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
                                  status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == -5  # MLA_ERR_DEVICE_CHECK
    assert status.item() & m.CHECK_BAD_SLOT
