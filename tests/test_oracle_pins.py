"""Pins of the float64 oracle against things other than itself (CPU only).

Each pin is chosen so that a plausible mistake anywhere in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a wrong mask) fails at least
one of them; ``test_planted_mistakes_are_caught`` compiles such mistakes into the
oracle and checks exactly that.
"""
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from speculative_decode_mla_gb300.workloads import (
    SOFTMAX_SCALE, bf16_bits_to_f32, custom_problem, f32_to_bf16_bits)

SCALE = SOFTMAX_SCALE


# ---------------------------------------------------------------- independent brute force
def ancestor_closure(parent):
    """Reflexive-transitive closure of the child->parent relation by boolean matrix powers.

    Written independently of the oracle's bitmask recursion: R[i, j] = 1 iff j is i or an
    ancestor of i, from repeated squaring of (I + A) where A[i, parent[i]] = 1.
    """
    T = len(parent)
    A = np.eye(T, dtype=np.int64)
    for i, p in enumerate(parent):
        if p >= 0:
            A[i, p] = 1
    R = A.copy()
    for _ in range(int(np.ceil(np.log2(max(T, 2)))) + 1):
        R = ((R @ R) > 0).astype(np.int64)
    return R.astype(bool)


def brute_force(p, scale=SCALE):
    """Dense score matrix [rows, N] and a dense visibility matrix built from positions."""
    outs, lses = [], []
    for b in range(p.B):
        L = int(p.seq_lens[b])
        N = L + p.T
        R = ancestor_closure(p.tree_parent[b])
        vis = np.zeros((p.T, N), dtype=bool)
        vis[:, :L] = True
        vis[:, L:] = R
        K = bf16_bits_to_f32(p.kv[p.slot_table[b, :N]]).astype(np.float64)  # [N, 576]
        Q = bf16_bits_to_f32(p.q[b * p.T:(b + 1) * p.T]).astype(np.float64)  # [T, H, 576]
        S = scale * np.einsum("thd,nd->thn", Q, K)
        S = np.where(vis[:, None, :], S, -np.inf)
        lse = logsumexp(S, axis=-1)
        W = np.exp(S - lse[..., None])
        outs.append(np.einsum("thn,nd->thd", W, K[:, :512]).reshape(-1, 512))
        lses.append(lse.reshape(-1))
    return np.concatenate(outs), np.concatenate(lses)


def causal_reference(qrows, keys, scale=SCALE):
    """Plain causal attention of the last len(qrows) positions of a sequence of keys."""
    N, T = len(keys), len(qrows)
    S = scale * (qrows @ keys.T)  # [T, N]
    pos = np.arange(N)[None, :]
    me = (N - T + np.arange(T))[:, None]
    S = np.where(pos <= me, S, -np.inf)
    lse = logsumexp(S, axis=-1)
    return np.exp(S - lse[:, None]) @ keys[:, :512], lse


def close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    return np.max(np.abs(a - b)) <= tol * max(1.0, np.max(np.abs(b)))


# ---------------------------------------------------------------- pins
def test_ancestor_masks_hand_example():
    # parents  -1, 0, 0, 1, 3  : node 4 -> 3 -> 1 -> 0
    m = oracle.ancestor_masks(np.array([-1, 0, 0, 1, 3]))
    assert list(m) == [0b1, 0b11, 0b101, 0b1011, 0b11011]


def test_ancestor_masks_match_closure():
    rng = np.random.default_rng(3)
    for T in (1, 2, 7, 33, 64):
        parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, T)], dtype=np.int32)
        m = oracle.ancestor_masks(parent)
        R = ancestor_closure(parent)
        for i in range(T):
            assert [(int(m[i]) >> j) & 1 for j in range(T)] == list(R[i].astype(int))


def test_bad_tree_rejected():
    with pytest.raises(ValueError):
        oracle.ancestor_masks(np.array([-1, 1]))  # parent[i] must be < i
    with pytest.raises(ValueError):
        oracle.ancestor_masks(np.array([-1, -2]))


@pytest.mark.parametrize("lens,T,H,tree", [([5], 4, 2, "random"), ([0, 3, 17], 6, 3, "random"),
                                           ([9, 1], 8, 1, "chain"), ([4], 5, 2, "star"),
                                           ([31], 64, 1, "random")])
def test_brute_force(lens, T, H, tree):
    p = custom_problem(lens, T, H, tree=tree, seed=len(lens) + T, pool_slack=7)
    out, lse = oracle.verify_problem(p, SCALE)
    bo, bl = brute_force(p)
    assert close(out, bo) and close(lse, bl)


def test_slot_permutation_bit_identical():
    p = custom_problem([40, 13], 9, 4, seed=11, pool_slack=20)
    out, lse = oracle.verify_problem(p, SCALE)
    rng = np.random.default_rng(5)
    perm = rng.permutation(p.num_slots)  # new_slot -> old_slot
    inv = np.argsort(perm)
    p.kv = p.kv[perm]
    p.slot_table = inv[p.slot_table].astype(np.int32)
    out2, lse2 = oracle.verify_problem(p, SCALE)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_chain_tree_equals_causal():
    p = custom_problem([23], 8, 3, tree="chain", seed=4)
    out, lse = oracle.verify_problem(p, SCALE)
    N = 23 + 8
    keys = bf16_bits_to_f32(p.kv[p.slot_table[0, :N]]).astype(np.float64)
    q = bf16_bits_to_f32(p.q).astype(np.float64)  # [T, H, 576]
    for h in range(3):
        co, cl = causal_reference(q[:, h, :], keys)
        assert close(out.reshape(8, 3, 512)[:, h], co) and close(lse.reshape(8, 3)[:, h], cl)


def test_star_tree_equals_single_token_decode():
    p = custom_problem([12], 5, 2, tree="star", seed=6)
    out, lse = oracle.verify_problem(p, SCALE)
    keys = bf16_bits_to_f32(p.kv[p.slot_table[0, :17]]).astype(np.float64)
    q = bf16_bits_to_f32(p.q).astype(np.float64)
    for i in range(5):
        sub = np.concatenate([keys[:12], keys[12 + i:13 + i]])  # prefix + the node itself
        for h in range(2):
            s = SCALE * sub @ q[i, h]
            w = np.exp(s - logsumexp(s))
            assert close(out[i * 2 + h], w @ sub[:, :512]) and close(lse[i * 2 + h], logsumexp(s))


def test_single_key_returns_its_value_exactly():
    p = custom_problem([0], 1, 4, seed=8, pool_slack=3)
    out, lse = oracle.verify_problem(p, SCALE)
    k = bf16_bits_to_f32(p.kv[p.slot_table[0, 0]]).astype(np.float64)
    for h in range(4):
        assert np.array_equal(out[h], k[:512])  # weight exactly 1
        qh = bf16_bits_to_f32(p.q[0, h]).astype(np.float64)
        assert abs(lse[h] - SCALE * float(qh @ k)) <= 1e-12 * max(1, abs(lse[h]))


def test_weights_sum_to_one_and_mask_is_exact():
    p = custom_problem([30], 12, 2, seed=9)
    masks = oracle.ancestor_masks(p.tree_parent[0])
    for row in range(0, 24, 5):
        w = oracle.row_weights(p.seq_lens, p.slot_table, p.tree_parent, p.q, p.kv, row, num_heads=2,
                               scale=SCALE)
        assert abs(w.sum() - 1.0) < 1e-12
        i = row // 2
        for j in range(12):
            assert (w[30 + j] > 0) == bool((int(masks[i]) >> j) & 1)
        assert np.all(w[:30] > 0)


def test_zero_query_gives_mean_of_visible_values():
    p = custom_problem([10], 6, 2, seed=10)
    p.q[:] = 0
    out, lse = oracle.verify_problem(p, SCALE)
    R = ancestor_closure(p.tree_parent[0])
    keys = bf16_bits_to_f32(p.kv[p.slot_table[0, :16]]).astype(np.float64)
    for i in range(6):
        vis = np.concatenate([np.ones(10, bool), R[i]])
        for h in range(2):
            assert close(out[i * 2 + h], keys[vis, :512].mean(axis=0))
            assert abs(lse[i * 2 + h] - np.log(vis.sum())) < 1e-12


def test_constant_value_column_gives_one():
    p = custom_problem([50], 7, 3, seed=12)
    p.kv[:, 77] = f32_to_bf16_bits(np.ones(1, np.float32))[0]
    out, _ = oracle.verify_problem(p, SCALE)
    assert np.max(np.abs(out[:, 77] - 1.0)) < 1e-12


def test_combine_of_position_chunks_equals_whole():
    p = custom_problem([57, 20], 10, 2, seed=13)
    out, lse = oracle.verify_problem(p, SCALE)
    cuts = [0, 7, 8, 30, 31, 59, 64, 67, 2 ** 40]  # includes chunks with nothing visible for some rows
    parts = [oracle.verify_problem(p, SCALE, pos_begin=a, pos_end=b) for a, b in zip(cuts[:-1], cuts[1:])]
    po = np.stack([x[0] for x in parts])
    pl = np.stack([x[1] for x in parts])
    assert np.isneginf(pl).any()
    co, cl = oracle.combine(po, pl)
    assert close(co, out) and close(cl, lse)


def test_combine_closed_form():
    # two parts with lse ln 1 and ln 3 carry weights 1/4 and 3/4; lse = ln 4
    po = np.array([[[1.0, 0.0]], [[0.0, 2.0]]])
    pl = np.log(np.array([[1.0], [3.0]]))
    o, l = oracle.combine(po, pl)
    assert np.allclose(o, [[0.25, 1.5]], atol=1e-15, rtol=0) and abs(l[0] - np.log(4.0)) < 1e-15
    o, l = oracle.combine(np.zeros((2, 1, 2)), np.full((2, 1), -np.inf))
    assert np.isneginf(l[0]) and not o.any()


def test_sampled_rows_match_full_run():
    p = custom_problem([33, 8, 70], 4, 3, seed=14)
    out, lse = oracle.verify_problem(p, SCALE)
    rows = [35, 0, 17, 12]
    o2, l2 = oracle.verify_problem(p, SCALE, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


def test_out_of_range_slot_rejected():
    p = custom_problem([5], 2, 1, seed=15)
    p.slot_table[0, 3] = p.num_slots
    with pytest.raises(ValueError):
        oracle.verify_problem(p, SCALE)


def test_page_figures_pin_the_byte_model():
    """The pages' 4.5 GB and ~13 GB per step fit a 1152-byte latent row per token per layer."""
    from speculative_decode_mla_gb300.workloads import D_K
    fig = {}
    with open(os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                fig[k] = float(v)
    row_bytes = D_K * 2
    gb64 = fig["layers"] * fig["ctx_64k_tokens"] * row_bytes / 1e9
    gb185 = fig["layers"] * fig["ctx_185k_tokens"] * row_bytes / 1e9
    assert abs(gb64 - fig["kv_gb_per_step_64k"]) / fig["kv_gb_per_step_64k"] < 0.05
    assert abs(gb185 - fig["kv_gb_per_step_185k"]) / fig["kv_gb_per_step_185k"] < 0.05
    eff = fig["kv_gb_per_step_64k"] / (fig["step_ms_64k"] / 1e3)
    assert abs(eff - fig["eff_gbs_64k"]) < 0.1
    assert abs(100 * eff / (fig["peak_tbs"] * 1e3) - fig["frac_of_peak_pct_64k"]) < 0.01
    assert abs(fig["kv_gb_per_step_64k"] / fig["peak_tbs"] - fig["floor_ms_64k"]) < 0.01
    assert abs(fig["peak_tbs"] * 1e3 / eff - fig["shortfall_x"]) < 2


MUTANT_PROBLEMS = [([6, 0], 7, 3, "random"), ([4], 3, 2, "chain")]


def _pins_pass():
    """The cheap pins, run against whatever oracle library is active."""
    for lens, T, H, tree in MUTANT_PROBLEMS:
        p = custom_problem(lens, T, H, tree=tree, seed=T, pool_slack=2)
        out, lse = oracle.verify_problem(p, SCALE)
        bo, bl = brute_force(p)
        if not (close(out, bo) and close(lse, bl)):
            return False
    p = custom_problem([0], 1, 2, seed=8)
    out, _ = oracle.verify_problem(p, SCALE)
    k = bf16_bits_to_f32(p.kv[p.slot_table[0, 0]]).astype(np.float64)
    return bool(np.array_equal(out[0], k[:512]))


@pytest.mark.parametrize("mutation", range(1, 8))
def test_planted_mistakes_are_caught(mutation, tmp_path):
    lib = oracle.build_mutant(mutation, str(tmp_path))
    with oracle.use_library(lib):
        assert not _pins_pass(), f"planted mistake {mutation} went unnoticed"


def test_unmutated_oracle_passes_same_pins():
    assert _pins_pass()
