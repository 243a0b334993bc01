"""GPU: batched verify with a ragged tree size per sequence (mla_verify_attn_ragged).

Definition used as the reference: each sequence is verified on its own, with its own T_b nodes,
by the float64 oracle; padding rows (nodes j >= T_b) must come out as out = 0, lse = -inf.
"""
import numpy as np
import pytest

import oracle
from _helpers import assert_close, device_problem, to_dev
from speculative_decode_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCALE = W.SOFTMAX_SCALE
KERNELS = ["tc", "simt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decode_mla_gb300 import _build
    _build.build()
    oracle.build()


def flags(kernel, debug=False):
    import speculative_decode_mla_gb300 as m
    return (m.MLA_FLAG_SIMT if kernel == "simt" else 0) | (m.MLA_FLAG_DEBUG_CHECKS if debug else 0)


def ragged_reference(p, sizes):
    """(out [B*T*H, 512], lse) with each sequence verified alone on its first T_b nodes."""
    T, H = p.T, p.H
    out = np.zeros((p.B * T * H, 512))
    lse = np.full(p.B * T * H, -np.inf)
    for b in range(p.B):
        tb = int(sizes[b])
        q_b = p.q.reshape(p.B, T, H, -1)[b, :tb]
        o, l = oracle.verify(p.seq_lens[b:b + 1], p.slot_table[b:b + 1], p.tree_parent[b:b + 1, :tb], q_b, p.kv,
                             num_heads=H, scale=SCALE)
        out[b * T * H:b * T * H + tb * H] = o
        lse[b * T * H:b * T * H + tb * H] = l
    return out, lse


@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged_batch_matches_per_sequence_oracle(kernel):
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([3000, 130, 0, 2047, 64, 900], 16, 8, seed=81, pool_slack=40)
    sizes = np.array([16, 1, 5, 9, 16, 2], dtype=np.int32)
    q, kv, st, sl, tp = device_problem(p)
    o, l = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, flags=flags(kernel), tree_sizes=to_dev(sizes),
                    out_dtype=m.MLA_DTYPE_F32)
    torch.cuda.synchronize()
    got_o = o.cpu().numpy().reshape(-1, 512).astype(np.float64)
    got_l = l.cpu().numpy().reshape(-1)
    ro, rl = ragged_reference(p, sizes)
    valid = np.isfinite(rl)
    assert_close(got_o[valid], got_l[valid], ro[valid], rl[valid], "ragged")
    assert not got_o[~valid].any() and np.isneginf(got_l[~valid]).all()


@pytest.mark.parametrize("kernel", KERNELS)
def test_ragged_with_full_sizes_is_bit_identical_to_the_uniform_call(kernel):
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([500, 77, 4097], 9, 13, seed=82, pool_slack=5)
    q, kv, st, sl, tp = device_problem(p)
    o1, l1 = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, flags=flags(kernel))
    o2, l2 = m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, flags=flags(kernel),
                      tree_sizes=to_dev(np.full(p.B, p.T, dtype=np.int32)))
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_ragged_reports_a_tree_size_out_of_range():
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([100, 30], 4, 2, seed=83)
    q, kv, st, sl, tp = device_problem(p)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MLAError) as ei:
        m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, flags=flags("tc", debug=True),
                 tree_sizes=to_dev(np.array([4, 9], dtype=np.int32)), dev_status=status)
    assert ei.value.status == -5 and status.item() & m.CHECK_BAD_LENGTH
