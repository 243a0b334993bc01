"""GPU parity of a multi-layer verify step captured as one CUDA graph and replayed.

The pages' decode runs graph-captured ("The Moment of Doubt", Input), and their native
verify engine was built to be capture-safe ("The GPU That Wasn't There", The Native
Engine Thesis). Here eight layers, each with its own latent pool and query and one
shared slot table, run as one graph: a tree-KV append writes the tree nodes' rows into
the first layer's pool, then eight verify calls follow back to back on one stream,
each chained to the one before it by programmatic dependent launch. The graph is
replayed twice, and every layer's out and lse is compared with the oracle after each
replay (and bit for bit with eager calls and between replays), once without and once
with MLA_FLAG_PREFIX_STABLE. That flag lets a call gather its first prefix tiles before
the preceding kernel (the append, or the previous layer's combine) has finished, which
is where a misplaced wait would show only under replay.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from _helpers import assert_close, bf16_dev, to_dev
from speculative_decode_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCALE = W.SOFTMAX_SCALE
LAYERS = 8


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decode_mla_gb300 import _build
    _build.build()
    oracle.build()


def layer_problems(lens, T, H, seed):
    """One problem per layer: shared lengths, tree and slot table; each layer its own q and pool."""
    p0 = W.custom_problem(lens, T, H, seed=seed, pool_slack=41)
    cid = p0.cfg.config_id
    out = []
    for layer in range(LAYERS):
        qs, ks = W.tensor_seed(cid, layer, W.STREAM_Q), W.tensor_seed(cid, layer, W.STREAM_KV)
        q = W.normal_bf16(qs, p0.q.size).reshape(p0.q.shape)
        kv = W.normal_bf16(ks, p0.kv.size).reshape(p0.kv.shape)
        out.append(dataclasses.replace(p0, q=q, kv=kv, q_seed=qs, kv_seed=ks))
    return out


@pytest.mark.parametrize("prefix_stable", [False, True], ids=["plain", "prefix_stable"])
def test_graph_replay_matches_oracle(prefix_stable):
    import torch
    import speculative_decode_mla_gb300 as m
    probs = layer_problems([12000, 3000], 16, 8, seed=71)
    p0 = probs[0]
    flags = m.MLA_FLAG_PREFIX_STABLE if prefix_stable else 0
    st, sl, tp = to_dev(p0.slot_table), to_dev(p0.seq_lens), to_dev(p0.tree_parent)
    pools = [bf16_dev(p.kv) for p in probs]
    qs = [bf16_dev(p.q) for p in probs]
    # the tree nodes' rows of layer 0, appended inside the graph; their slots start out zeroed
    tree_slots = np.concatenate([p0.slot_table[b, p0.seq_lens[b]:p0.seq_lens[b] + p0.T] for b in range(p0.B)])
    tree_idx = torch.from_numpy(tree_slots.astype(np.int64)).cuda()
    tree_kv = pools[0][tree_idx].clone()

    desc = m.make_desc(p0.B, p0.T, p0.H, p0.num_slots, p0.stride, p0.max_seq_len, flags=flags)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((p0.B * p0.T, p0.H, 512), dtype=torch.bfloat16, device="cuda") for _ in range(LAYERS)]
    lses = [torch.empty((p0.B * p0.T, p0.H), dtype=torch.float32, device="cuda") for _ in range(LAYERS)]

    def step():  # on the current stream (the capture stream while capturing)
        sp = torch.cuda.current_stream().cuda_stream
        m.tree_kv_append(pools[0], tree_kv, st, sl, max_seq_len=p0.max_seq_len)
        for layer in range(LAYERS):
            rc = m.verify_attn_raw(desc, qs[layer].data_ptr(), pools[layer].data_ptr(), st.data_ptr(),
                                   sl.data_ptr(), tp.data_ptr(), outs[layer].data_ptr(), lses[layer].data_ptr(),
                                   ws.data_ptr(), ws.numel(), 0, sp)
            assert rc == 0, m.status_string(rc)

    def reset():  # the replay must rewrite the tree rows and every output
        pools[0][tree_idx] = 0
        for o, l in zip(outs, lses):
            o.fill_(float("nan"))
            l.fill_(float("nan"))

    # eager reference (same calls, no graph)
    reset()
    step()
    torch.cuda.synchronize()
    eager = [(o.clone(), l.clone()) for o, l in zip(outs, lses)]

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()

    ref = [oracle.verify_problem(p, SCALE) for p in probs]
    replays = []
    for rep in range(2):
        reset()
        g.replay()
        torch.cuda.synchronize()
        got = [(o.clone(), l.clone()) for o, l in zip(outs, lses)]
        replays.append(got)
        for layer, ((o, l), (ro, rl)) in enumerate(zip(got, ref)):
            oo = o.float().cpu().numpy().reshape(p0.rows, 512).astype(np.float64)
            assert_close(oo, l.cpu().numpy().reshape(-1), ro, rl, f"replay {rep} layer {layer}")
            eo, el = eager[layer]
            assert torch.equal(o.view(torch.int16), eo.view(torch.int16)) and torch.equal(l, el), \
                f"replay {rep} layer {layer} differs from the eager call"
    for (a, al), (b, bl) in zip(*replays):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and torch.equal(al, bl)
