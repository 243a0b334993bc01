"""The seeded input generators (CPU): published SplitMix64 vectors, determinism, structure."""
import os

import numpy as np

from speculative_decode_mla_gb300 import workloads as W


def test_splitmix64_published_vectors():
    path = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_vectors.txt")
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            i, h = line.split()
            assert W.splitmix64_scalar(0, int(i)) == int(h, 16)
            assert int(W.splitmix64(0, np.array([int(i)], dtype=np.uint64))[0]) == int(h, 16)


def test_normal_generator_moments_and_bounds():
    x = W.bf16_bits_to_f32(W.normal_bf16(123, 1 << 20))
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert np.abs(x).max() <= 3.47


def test_normal_generator_is_counter_based():
    a = W.normal_bf16(99, 1000)
    b = W.normal_bf16(99, 600, start=400)
    assert np.array_equal(a[400:], b)
    assert np.array_equal(W.normal_bf16(99, 1000, chunk=7), a)


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -9], dtype=np.float32)
    r = W.bf16_bits_to_f32(W.f32_to_bf16_bits(f))
    assert list(r) == [1.0, 1.0, 1.0 + 4 * 2 ** -8, -2.5, 1.0]


def test_trees_are_topological():
    for s in range(20):
        p = W.random_tree(s, 64)
        assert p[0] == -1 and all(0 <= p[i] < i for i in range(1, 64))


def test_slot_table_is_injective_and_in_range():
    p = W.make_problem("batched", with_kv=False)
    used = np.concatenate([p.slot_table[b, : p.seq_lens[b] + p.T] for b in range(p.B)])
    assert len(np.unique(used)) == len(used) and used.min() >= 0 and used.max() < p.num_slots
    assert p.seq_lens.min() >= 1024 and p.seq_lens.max() < 32768
    assert p.rows == 32 * 8 * 16


def test_identity_table():
    cfg = W.CONFIGS["wide_identity"]
    t = W.make_slot_table(cfg, np.array([10], np.int32), 100, 80)
    assert np.array_equal(t[0, :74], np.arange(74))


def test_config_shapes_match_the_workloads():
    c = W.CONFIGS
    assert (c["64k"].prefix_len, c["64k"].num_nodes, c["64k"].num_heads) == (65536, 16, 8)
    assert (c["185k"].prefix_len, c["185k"].num_nodes, c["185k"].layers) == (184320, 32, 61)
    assert (c["wide"].num_heads, c["wide"].num_nodes) == (64, 64)
    assert W.kv_bytes_per_layer_step([65536], 16) == (65536 + 16) * 1156
