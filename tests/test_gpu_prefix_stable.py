"""GPU: MLA_FLAG_PREFIX_STABLE (the gather of the first prefix tiles may start before the preceding
kernel on the stream has finished). Results must be bit-identical to calls without the flag, also
when the preceding kernel writes the tree rows the call reads (tree-KV append just before it)."""
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


SHAPES = [([0, 64, 65, 1000], 4, 3), ([5000, 130, 2047], 9, 13), ([200], 64, 2)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"L{s[0]}-T{s[1]}-H{s[2]}" for s in SHAPES])
@pytest.mark.parametrize("splits", [0, 3, 40])
def test_flag_gives_bit_identical_results(shape, splits):
    import torch
    import speculative_decode_mla_gb300 as m
    lens, T, H = shape
    p = W.custom_problem(lens, T, H, seed=91 + T, pool_slack=17)
    q, kv, st, sl, tp = device_problem(p)
    o1, l1 = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, num_splits=splits)
    o2, l2 = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, num_splits=splits,
                      flags=m.MLA_FLAG_PREFIX_STABLE)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_flag_after_a_kernel_that_writes_the_tree_rows():
    """tree-KV append immediately before a flagged verify on the same stream (no sync): the tree
    rows must be read after the append, the prefix may be read before it finishes."""
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([3000, 700], 16, 8, seed=92, pool_slack=30)
    q, kv, st, sl, tp = device_problem(p)
    ref_o, ref_l = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len)
    torch.cuda.synchronize()
    tree_rows = torch.stack([kv[int(p.slot_table[b, p.seq_lens[b] + j])]
                             for b in range(p.B) for j in range(p.T)]).contiguous()
    for rep in range(3):
        holed = kv.clone()
        for b in range(p.B):
            idx = torch.from_numpy(p.slot_table[b, p.seq_lens[b]:p.seq_lens[b] + p.T].astype(np.int64)).cuda()
            holed[idx] = 0
        torch.cuda.synchronize()
        m.tree_kv_append(holed, tree_rows, st, sl, max_seq_len=p.max_seq_len)
        o, l = m.verify(q, holed, st, sl, tp, max_seq_len=p.max_seq_len, flags=m.MLA_FLAG_PREFIX_STABLE)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16)) and torch.equal(l, ref_l)


def test_flag_with_hybrid_and_ragged():
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([4097, 100], 9, 4, seed=93, pool_slack=64)
    q, kv, st, sl, tp = device_problem(p)
    sizes = to_dev(np.array([9, 3], dtype=np.int32))
    o1, l1 = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, tree_sizes=sizes)
    o2, l2 = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, tree_sizes=sizes,
                      flags=m.MLA_FLAG_PREFIX_STABLE)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
