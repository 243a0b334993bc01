"""GPU parity: the library's kernels against the float64 oracle, through the C ABI.

Bar (written here, per element / per tensor): max-abs error <= 1e-2 and relative L2
error <= 5e-3 on out (bf16 inputs, fp32 accumulation, bf16 output); |lse| error <= 1e-3.
Full-size configs are checked on rows sampled across every node, head and sequence.
"""
import numpy as np
import pytest

import oracle
from _helpers import assert_close, bf16_dev, device_problem, errors, run, to_dev
from speculative_decode_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCALE = W.SOFTMAX_SCALE


def kernels():
    import speculative_decode_mla_gb300 as m
    return {"simt": m.MLA_FLAG_SIMT, "tc": 0}


KERNELS = ["tc", "simt"]


@pytest.fixture(scope="module", autouse=True)
def built():
    from speculative_decode_mla_gb300 import _build
    _build.build()
    oracle.build()


def flags_of(name, debug=False):
    import speculative_decode_mla_gb300 as m
    return kernels()[name] | (m.MLA_FLAG_DEBUG_CHECKS if debug else 0)


def sample_rows(p, per_seq=8, seed=0):
    """Rows checked against the oracle on the full-size configs, stratified so that every part of
    the kernel's row layout is compared: in every sequence, one row from each 32-row lane quarter
    of each 128-row tile (the tensor-core kernel's TMEM lane groups), all heads of the first and
    of the last node, and ``per_seq`` more drawn at random."""
    rng = np.random.default_rng(seed)
    R = p.T * p.H
    rows = []
    for b in range(p.B):
        pick = set(rng.choice(R, size=min(per_seq, R), replace=False).tolist())
        for q0 in range(0, R, 32):  # each lane quarter of each row tile
            pick.add(int(rng.integers(q0, min(q0 + 32, R))))
        pick |= set(range(min(p.H, R))) | set(range(R - p.H, R))
        rows += [b * R + r for r in sorted(pick)]
    return np.array(rows, dtype=np.int64)


def test_sample_rows_cover_every_lane_quarter():
    for name in ("wide", "185k", "batched"):
        p = W.make_problem(name, with_kv=False)
        R = p.T * p.H
        rows = sample_rows(p, per_seq=4)
        for b in range(p.B):
            local = rows[(rows >= b * R) & (rows < (b + 1) * R)] - b * R
            assert set(np.unique(local // 32)) == set(range((R + 31) // 32))
            assert set(range(p.H)) <= set(local) and set(range(R - p.H, R)) <= set(local)


# ------------------------------------------------------------------ named configs
@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny(kernel):
    p = W.make_problem("tiny")
    o, l = run(p, flags_of(kernel))
    ro, rl = oracle.verify_problem(p, SCALE)
    assert_close(o, l, ro, rl, "tiny")


@pytest.mark.parametrize("kernel", KERNELS)
def test_64k_all_rows(kernel):
    p = W.make_problem("64k")
    o, l = run(p, flags_of(kernel))
    ro, rl = oracle.verify_problem(p, SCALE)
    assert_close(o, l, ro, rl, "64k")


@pytest.mark.parametrize("kernel", KERNELS)
def test_batched_sampled_rows(kernel):
    p = W.make_problem("batched")
    o, l = run(p, flags_of(kernel), total_tokens_hint=int((p.seq_lens + p.T).sum()))
    rows = sample_rows(p, per_seq=6)
    ro, rl = oracle.verify_problem(p, SCALE, rows=rows)
    assert_close(o[rows], l[rows], ro, rl, "batched")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("cfg", ["wide", "wide_identity"])
def test_wide_sampled_rows(kernel, cfg):
    p = W.make_problem(cfg)
    o, l = run(p, flags_of(kernel))
    rows = sample_rows(p, per_seq=16)
    ro, rl = oracle.verify_problem(p, SCALE, rows=rows)
    assert_close(o[rows], l[rows], ro, rl, cfg)


@pytest.mark.parametrize("kernel", KERNELS)
def test_185k_61_layers_sampled(kernel):
    """61 device-drawn pools (about 13 GB) and one shared slot table; layers 0, 30, 60 checked."""
    import torch
    import speculative_decode_mla_gb300 as m
    cfg = W.CONFIGS["185k"]
    p0 = W.make_problem(cfg, layer=0, with_kv=False)
    st, sl, tp = to_dev(p0.slot_table), to_dev(p0.seq_lens), to_dev(p0.tree_parent)
    pool = torch.empty((cfg.layers, p0.num_slots, W.D_K), dtype=torch.bfloat16, device="cuda")
    qs = torch.empty((cfg.layers, p0.B * p0.T, p0.H, W.D_K), dtype=torch.bfloat16, device="cuda")
    for layer in range(cfg.layers):
        m.fill_normal_bf16(pool[layer], W.tensor_seed(cfg.config_id, layer, W.STREAM_KV))
        m.fill_normal_bf16(qs[layer], W.tensor_seed(cfg.config_id, layer, W.STREAM_Q))
    outs = []
    for layer in range(cfg.layers):
        o, l = m.verify(qs[layer], pool[layer], st, sl, tp, max_seq_len=p0.max_seq_len, flags=flags_of(kernel))
        outs.append((o, l))
    torch.cuda.synchronize()
    for layer in (0, 30, 60):
        p = W.make_problem(cfg, layer=layer)
        o = outs[layer][0].float().cpu().numpy().reshape(p.rows, 512).astype(np.float64)
        l = outs[layer][1].cpu().numpy().reshape(-1)
        rows = sample_rows(p, per_seq=10, seed=layer)
        ro, rl = oracle.verify_problem(p, SCALE, rows=rows)
        assert_close(o[rows], l[rows], ro, rl, f"185k layer {layer}")
    del pool, qs


# ------------------------------------------------------------------ shapes and edge cases
SHAPES = [
    ([0], 1, 1, "random"),          # single visible key
    ([0], 5, 3, "chain"),           # no prefix, tree only
    ([1], 1, 16, "random"),
    ([63], 1, 2, "random"),         # one tile exactly (63 + 1)
    ([64], 1, 2, "random"),         # tree crosses the tile edge
    ([130, 7, 1000], 8, 16, "random"),  # ragged batch, 128 rows per sequence
    ([333], 64, 2, "random"),       # T at its maximum
    ([77, 300], 3, 5, "star"),      # rows per sequence not a multiple of 8 / 128
    ([2000], 16, 8, "chain"),       # chain tree: causal tail
    ([5000, 4500, 6000], 9, 13, "random"),  # several tiles and a ragged tail per sequence
    ([3000, 700, 5000], 16, 16, "random"),  # several sequences of two row tiles each, longest first
    ([(i * 53) % 700 for i in range(64)], 3, 4, "random"),  # 64 sequences: the longest-first unit order
    ([(i * 97) % 900 for i in range(70)], 2, 2, "random"),  # 70 sequences: units in index order
]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{len(s[0])}-L{max(s[0])}-T{s[1]}-H{s[2]}-{s[3]}" for s in SHAPES])
def test_shapes(kernel, shape):
    lens, T, H, tree = shape
    p = W.custom_problem(lens, T, H, tree=tree, seed=len(lens) * 100 + T + H, pool_slack=37, stride_pad=5)
    o, l = run(p, flags_of(kernel))
    ro, rl = oracle.verify_problem(p, SCALE)
    assert_close(o, l, ro, rl, str(shape))


@pytest.mark.parametrize("kernel", KERNELS)
def test_single_key_returns_value_exactly(kernel):
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([0], 1, 4, seed=3)
    o, l = run(p, flags_of(kernel), out_dtype=m.MLA_DTYPE_F32)
    v = W.bf16_bits_to_f32(p.kv[p.slot_table[0, 0]])[:512].astype(np.float64)
    for h in range(4):
        assert np.array_equal(o[h], v)
    ro, rl = oracle.verify_problem(p, SCALE)
    assert np.abs(l - rl).max() < 1e-4


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits", [1, 2, 7, 33])
def test_split_count_changes_only_rounding(kernel, splits):
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([3000], 16, 8, seed=21)
    ref_o, ref_l = run(p, flags_of(kernel), out_dtype=m.MLA_DTYPE_F32, num_splits=1)
    o, l = run(p, flags_of(kernel), out_dtype=m.MLA_DTYPE_F32, num_splits=splits)
    # SIMT: fp32 reordering plus the fp16 rounding of each split's partial; the tensor-core path
    # also re-rounds its bf16 P with each split's own running max
    tol = 1e-3 if kernel == "simt" else 3e-3  # both also round each split's partial to fp16
    assert np.abs(o - ref_o).max() <= tol
    assert np.abs(l - ref_l).max() <= 1e-5
    ro, rl = oracle.verify_problem(p, SCALE)
    assert_close(o, l, ro, rl, f"splits={splits}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_slot_permutation_is_bit_identical(kernel):
    p = W.custom_problem([2500, 700], 12, 6, seed=22, pool_slack=100)
    o1, l1 = run(p, flags_of(kernel))
    rng = np.random.default_rng(1)
    perm = rng.permutation(p.num_slots)
    p.kv = p.kv[perm]
    p.slot_table = np.argsort(perm)[p.slot_table].astype(np.int32)
    o2, l2 = run(p, flags_of(kernel))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("kernel", KERNELS)
def test_constant_value_column_is_one(kernel):
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([4000], 16, 8, seed=23)
    one = W.f32_to_bf16_bits(np.ones(1, np.float32))[0]
    p.kv[:, 5] = one
    p.kv[:, 300] = one
    o, _ = run(p, flags_of(kernel), out_dtype=m.MLA_DTYPE_F32)
    # Both kernels normalise O by the sum of the very weights the PV product used, so a constant
    # column is 1 up to accumulation rounding: SIMT sums in fp32 (~1e-6). The tensor-core path adds
    # (i) its fp32 accumulation of ~N = 4000 terms, at most N * 2^-24 ~ 2.4e-4 relative, and
    # (ii) the fp16 rounding of each split's normalised partial, at most 2^-11 ~ 4.9e-4 near 1.0;
    # (i) + (ii) ~ 7.3e-4 sets the bar at 1e-3.
    tol = 1e-5 if kernel == "simt" else 1e-3
    assert np.abs(o[:, 5] - 1).max() < tol and np.abs(o[:, 300] - 1).max() < tol


@pytest.mark.parametrize("kernel", KERNELS)
def test_zero_query_gives_mean(kernel):
    p = W.custom_problem([1500], 8, 4, seed=24)
    p.q[:] = 0
    o, l = run(p, flags_of(kernel))
    ro, rl = oracle.verify_problem(p, SCALE)
    assert_close(o, l, ro, rl, "q=0")


@pytest.mark.parametrize("kernel", KERNELS)
def test_f32_output_is_tighter(kernel):
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([6000], 16, 8, seed=25)
    o, l = run(p, flags_of(kernel), out_dtype=m.MLA_DTYPE_F32)
    ro, rl = oracle.verify_problem(p, SCALE)
    err, rel, lerr = errors(o, l, ro, rl)
    assert rel <= 4e-3 and err <= 5e-3 and lerr <= 1e-3


# ------------------------------------------------------------------ device checks and errors
@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fault", ["slot", "parent", "length"])
def test_debug_checks_report_bad_inputs(kernel, fault):
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([200], 6, 2, seed=26)
    q, kv, st, sl, tp = device_problem(p)
    expect = {"slot": m.CHECK_BAD_SLOT, "parent": m.CHECK_BAD_PARENT, "length": m.CHECK_BAD_LENGTH}[fault]
    if fault == "slot":
        st[0, 17] = p.num_slots + 5
    elif fault == "parent":
        tp[0, 3] = 4
    else:
        sl[0] = 250  # above max_seq_len
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MLAError) as ei:
        m.verify(q, kv, st, sl, tp, max_seq_len=200, flags=flags_of(kernel, debug=True), dev_status=status)
    assert ei.value.status == -5
    assert int(status.item()) & expect
    # without debug checks the bad value is clamped: the call succeeds and nothing faults
    out, _ = m.verify(q, kv, st, sl, tp, max_seq_len=200, flags=flags_of(kernel))
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("kernel", KERNELS)
def test_debug_checks_clean_inputs_pass(kernel):
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([500], 8, 4, seed=27)
    status = torch.full((1,), 123, dtype=torch.int32, device="cuda")
    dev = device_problem(p)
    m.verify(*dev, max_seq_len=p.max_seq_len, flags=flags_of(kernel, debug=True), dev_status=status)
    assert int(status.item()) == 0


def test_workspace_too_small_is_rejected():
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([500], 8, 4, seed=28)
    dev = device_problem(p)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(m.MLAError) as ei:
        m.verify(*dev, max_seq_len=p.max_seq_len, workspace=ws)
    assert ei.value.status == -3


# ------------------------------------------------------------------ combine entry point
def test_combine_entry_point_matches_oracle_combine():
    """Partials of disjoint position windows (as a cross-GPU split would make) merged on the GPU."""
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([900, 40], 8, 4, seed=29)
    cuts = [0, 100, 101, 500, 940, 10 ** 9]
    parts = [oracle.verify_problem(p, SCALE, pos_begin=a, pos_end=b) for a, b in zip(cuts[:-1], cuts[1:])]
    po = np.stack([x[0] for x in parts])
    pl = np.stack([x[1] for x in parts])
    ro, rl = oracle.combine(po, pl)
    o, l = m.combine(torch.from_numpy(po.astype(np.float32)).cuda(), torch.from_numpy(pl.astype(np.float32)).cuda(),
                     out_dtype=m.MLA_DTYPE_F32)
    oh, lh = m.combine(torch.from_numpy(po.astype(np.float16)).cuda(), torch.from_numpy(pl.astype(np.float32)).cuda(),
                       out_dtype=m.MLA_DTYPE_F32)
    torch.cuda.synchronize()
    assert np.abs(o.cpu().numpy() - ro).max() < 1e-5
    # fp16 partials (the library's own split workspace format): 11-bit mantissa on |o| <= max|v|
    assert np.abs(oh.cpu().numpy() - ro).max() < 4e-3 * np.abs(po).max()
    assert np.array_equal(lh.cpu().numpy(), l.cpu().numpy())
    finite = np.isfinite(rl)
    assert np.abs(l.cpu().numpy()[finite] - rl[finite]).max() < 1e-5
    full_o, full_l = oracle.verify_problem(p, SCALE)
    assert_close(o.cpu().numpy().astype(np.float64), l.cpu().numpy(), full_o, full_l, "combine")


@pytest.mark.parametrize("dtype", ["f16", "f32"])
def test_combine_many_rows_same_bits_as_few_rows(dtype):
    """From 2048 (row, 128-column) items on, the combine runs one warp per item instead of one CTA
    per row; it folds the splits in the same order, so a row's result carries the same bits
    whichever kernel ran it. Checked on seeded partials with empty splits (lse = -inf) at the end
    of some rows, as a batch of sequences of different lengths leaves them, and against the
    oracle's combine."""
    import torch
    import speculative_decode_mla_gb300 as m
    rng = np.random.default_rng(83)
    splits, rows, d_v = 11, 700, 512  # 700 x 4 column blocks = 2800 items: the per-warp kernel
    po = rng.standard_normal((splits, rows, d_v)).astype(np.float32)
    pl = (rng.standard_normal((splits, rows)) * 3.0).astype(np.float32)
    nsp = rng.integers(1, splits + 1, size=rows)  # row r has splits [0, nsp[r]) with positions
    pl[np.arange(splits)[:, None] >= nsp[None, :]] = -np.inf
    pt = np.float16 if dtype == "f16" else np.float32
    big_o, big_l = m.combine(torch.from_numpy(po.astype(pt)).cuda(), torch.from_numpy(pl).cuda(),
                             out_dtype=m.MLA_DTYPE_F32)
    few = 100  # 400 items: one CTA per row
    sm_o, sm_l = m.combine(torch.from_numpy(np.ascontiguousarray(po[:, :few].astype(pt))).cuda(),
                           torch.from_numpy(np.ascontiguousarray(pl[:, :few])).cuda(), out_dtype=m.MLA_DTYPE_F32)
    torch.cuda.synchronize()
    assert np.array_equal(big_o.cpu().numpy()[:few], sm_o.cpu().numpy())
    assert np.array_equal(big_l.cpu().numpy()[:few], sm_l.cpu().numpy())
    ro, rl = oracle.combine(po.astype(pt).astype(np.float64), pl.astype(np.float64))
    assert np.abs(big_o.cpu().numpy() - ro).max() < 1e-5 * max(1.0, np.abs(po).max())
    assert np.abs(big_l.cpu().numpy() - rl).max() < 1e-5 * max(1.0, np.abs(rl).max())


@pytest.mark.parametrize("kernel", KERNELS)
def test_partials_then_combine_equals_attn(kernel):
    """mla_verify_attn_partials + mla_verify_combine on its workspace is bit-identical to mla_verify_attn."""
    import torch
    import speculative_decode_mla_gb300 as m
    p = W.custom_problem([5000, 130, 2047], 9, 13, seed=31, pool_slack=19)
    q, kv, st, sl, tp = device_problem(p)
    desc = m.make_desc(p.B, p.T, p.H, p.num_slots, p.stride, p.max_seq_len, flags=flags_of(kernel))
    plan = m.plan(desc, torch.cuda.get_device_properties(0).multi_processor_count)
    ws = torch.empty(m.workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty((p.B * p.T, p.H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.B * p.T, p.H), dtype=torch.float32, device="cuda")
    sp = torch.cuda.current_stream().cuda_stream
    assert m.verify_attn_raw(desc, q.data_ptr(), kv.data_ptr(), st.data_ptr(), sl.data_ptr(), tp.data_ptr(),
                             out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp) == 0
    ref_o, ref_l = out.clone(), lse.clone()
    ws.fill_(0xAB)  # partials must be fully rewritten
    assert m.verify_attn_partials_raw(desc, q.data_ptr(), kv.data_ptr(), st.data_ptr(), sl.data_ptr(),
                                      tp.data_ptr(), ws.data_ptr(), ws.numel(), 0, sp) == 0
    part_o, part_l = m.partials_views(ws, plan, p.rows)
    o2, l2 = m.combine(part_o, part_l, out_dtype=m.MLA_DTYPE_BF16)
    torch.cuda.synchronize()
    assert torch.equal(o2.view(torch.int16), ref_o.view(p.rows, 512).view(torch.int16))
    assert torch.equal(l2.view(-1), ref_l.view(-1))
    ro, rl = oracle.verify_problem(p, SCALE)
    assert_close(o2.float().cpu().numpy().astype(np.float64), l2.cpu().numpy().reshape(-1), ro, rl, "partials")


# ------------------------------------------------------------------ input generator
def test_device_generator_matches_host_bitwise():
    import torch
    import speculative_decode_mla_gb300 as m
    for seed, n, start in [(1, 1000, 0), (W.tensor_seed(2, 60, 1), 4099, 12345), (2 ** 63 + 5, 77, 3)]:
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        m.fill_normal_bf16(t, seed, start)
        got = t.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, W.normal_bf16(seed, n, start=start))
