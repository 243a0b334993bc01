"""Seeded synthetic workloads for tree-verify MLA attention.

This module is the one piece shared by the oracle side and the CUDA side: it
draws inputs and nothing else. It holds none of the method's arithmetic (no
scores, no softmax, no masking); it only produces the tensors a verify call
consumes, with the shapes and structure of the long-context DDTree decode the
pages diagnose (one sequence at 64k-185k context, a small draft tree, a
page_size=1 latent pool whose token order is scattered over physical slots).

Generators (all counter-based, so any element can be drawn on its own, on the
host here or on the device by the library's fill kernel):

* ``splitmix64(seed, i)``: the SplitMix64 output function (Steele, Lea and
  Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) applied
  to the counter state ``seed + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64``.
* ``normal_bf16``: an Irwin-Hall approximation of N(0, 1). The four 16-bit
  fields of one 64-bit draw are summed, centred (mean 131070) and multiplied in
  float32 by the float32 constant 0x37DDB3D7 (= sqrt(3)/65536 rounded to
  float32), then rounded to bf16 with round-to-nearest-even. Every step is
  exact integer work or one correctly rounded float32 multiply, so the host and
  the device produce the same bits. The tails stop at +-3.46 sigma.
* slot permutations: pool slots sorted by a SplitMix64 key (a uniform random
  permutation); tree parents: ``parent[0] = -1`` and, for ``i >= 1``,
  ``parent[i] = (hi32(h) * i) >> 32``, uniform in ``[0, i)``.

Everything here is host-side numpy; the device fill entry point mirrors
``normal_bf16`` for the pools that are too large to draw on the host.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1
NORMAL_SCALE_BITS = 0x37DDB3D7  # float32(sqrt(3) / 65536)
NORMAL_SCALE = np.array([NORMAL_SCALE_BITS], dtype=np.uint32).view(np.float32)[0]

STREAM_Q, STREAM_KV, STREAM_SLOTS, STREAM_TREE, STREAM_LENS = 0, 1, 2, 3, 4

D_LATENT = 512
D_ROPE = 64
D_K = D_LATENT + D_ROPE
D_V = D_LATENT
SOFTMAX_SCALE = float(1.0 / np.sqrt(192.0))


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, idx: np.ndarray) -> np.ndarray:
    """SplitMix64 output for counters ``idx`` (uint64 array) under ``seed``."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & MASK64) + (idx + np.uint64(1)) * np.uint64(GAMMA)
        return _mix(z)


def splitmix64_scalar(seed: int, i: int) -> int:
    z = (seed + (i + 1) * GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def tensor_seed(config_id: int, layer: int, stream: int) -> int:
    """Seed of one tensor: base ``0x5EED0000 + 16*config + layer``, hashed with the stream id."""
    base = 0x5EED0000 + 16 * config_id + layer
    return splitmix64_scalar(base, stream)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round-to-nearest-even), returned as uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, n: int, start: int = 0, chunk: int = 1 << 23) -> np.ndarray:
    """``n`` bf16 draws (uint16 bits) of the Irwin-Hall N(0,1) stream, counters ``start..start+n``."""
    out = np.empty(n, dtype=np.uint16)
    for c0 in range(0, n, chunk):
        c1 = min(n, c0 + chunk)
        h = splitmix64(seed, np.arange(start + c0, start + c1, dtype=np.uint64))
        m = np.uint64(0xFFFF)
        s = (h & m) + ((h >> np.uint64(16)) & m) + ((h >> np.uint64(32)) & m) + (h >> np.uint64(48))
        xi = s.astype(np.int64) - 131070
        x = xi.astype(np.float32) * NORMAL_SCALE
        out[c0:c1] = f32_to_bf16_bits(x)
    return out


def random_permutation(seed: int, n: int) -> np.ndarray:
    keys = splitmix64(seed, np.arange(n, dtype=np.uint64))
    return np.argsort(keys, kind="stable").astype(np.int32)


def random_tree(seed: int, T: int) -> np.ndarray:
    """``parent[0] = -1``; ``parent[i]`` uniform in ``[0, i)`` (topological order)."""
    h = splitmix64(seed, np.arange(T, dtype=np.uint64))
    i = np.arange(T, dtype=np.uint64)
    p = ((h >> np.uint64(32)) * i) >> np.uint64(32)
    p = p.astype(np.int64)
    p[0] = -1
    return p.astype(np.int32)


def chain_tree(T: int) -> np.ndarray:
    return (np.arange(T, dtype=np.int32) - 1).astype(np.int32)


def star_tree(T: int) -> np.ndarray:
    return np.full(T, -1, dtype=np.int32)


def log_uniform_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    h = splitmix64(seed, np.arange(n, dtype=np.uint64))
    u = (h >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    L = np.floor(lo * np.exp(u * np.log(hi / lo))).astype(np.int64)
    return np.clip(L, lo, hi - 1).astype(np.int32)


@dataclasses.dataclass
class Config:
    """One verify workload. ``seq_lens`` are prefix lengths (the tree is extra)."""

    name: str
    config_id: int
    num_seqs: int
    num_nodes: int
    num_heads: int
    tree: str  # "chain" | "random"
    lens: str  # "fixed" | "log_uniform"
    prefix_len: int = 0
    len_lo: int = 0
    len_hi: int = 0
    pool_slots: int = 0  # 0 = exactly sum of visible tokens
    layers: int = 1
    identity_table: bool = False


CONFIGS = {
    "tiny": Config("tiny", 0, 1, 8, 8, "chain", "fixed", prefix_len=1024, pool_slots=4096),
    "64k": Config("64k", 1, 1, 16, 8, "random", "fixed", prefix_len=65536, pool_slots=131072),
    "185k": Config("185k", 2, 1, 32, 8, "random", "fixed", prefix_len=184320, pool_slots=184352, layers=61),
    "batched": Config("batched", 3, 32, 8, 16, "random", "log_uniform", len_lo=1024, len_hi=32768),
    "wide": Config("wide", 4, 1, 64, 64, "random", "fixed", prefix_len=131072, pool_slots=131136),
    "wide_identity": Config("wide_identity", 4, 1, 64, 64, "random", "fixed", prefix_len=131072,
                            pool_slots=131136, identity_table=True),
}


@dataclasses.dataclass
class Problem:
    """Host copies of one verify call's inputs (bf16 tensors as uint16 bits)."""

    cfg: Config
    seq_lens: np.ndarray  # int32 [B] prefix lengths
    tree_parent: np.ndarray  # int32 [B, T]
    slot_table: np.ndarray  # int32 [B, stride]
    q: np.ndarray  # uint16 [B*T, H, 576]
    kv: Optional[np.ndarray]  # uint16 [num_slots, 576] (None when drawn on the device)
    num_slots: int
    kv_seed: int
    q_seed: int

    @property
    def B(self):
        return self.cfg.num_seqs

    @property
    def T(self):
        return self.cfg.num_nodes

    @property
    def H(self):
        return self.cfg.num_heads

    @property
    def stride(self):
        return self.slot_table.shape[1]

    @property
    def rows(self):
        return self.B * self.T * self.H

    @property
    def max_seq_len(self):
        return int(self.seq_lens.max())


def make_lengths(cfg: Config) -> np.ndarray:
    if cfg.lens == "fixed":
        return np.full(cfg.num_seqs, cfg.prefix_len, dtype=np.int32)
    return log_uniform_lengths(tensor_seed(cfg.config_id, 0, STREAM_LENS), cfg.num_seqs, cfg.len_lo, cfg.len_hi)


def make_trees(cfg: Config) -> np.ndarray:
    T = cfg.num_nodes
    if cfg.tree == "chain":
        return np.stack([chain_tree(T)] * cfg.num_seqs)
    seed = tensor_seed(cfg.config_id, 0, STREAM_TREE)
    return np.stack([random_tree(splitmix64_scalar(seed, b), T) for b in range(cfg.num_seqs)])


def make_slot_table(cfg: Config, seq_lens: np.ndarray, num_slots: int, stride: int) -> np.ndarray:
    """Token ``t`` of sequence ``b`` lives at slot ``table[b, t]`` (page_size=1).

    Sequences take consecutive ranges of one random permutation of the pool,
    so their slots are interleaved at random. Entries past ``N_b`` stay 0.
    """
    N = seq_lens.astype(np.int64) + cfg.num_nodes
    table = np.zeros((cfg.num_seqs, stride), dtype=np.int32)
    if cfg.identity_table:
        perm = np.arange(num_slots, dtype=np.int32)
    else:
        perm = random_permutation(tensor_seed(cfg.config_id, 0, STREAM_SLOTS), num_slots)
    off = 0
    for b in range(cfg.num_seqs):
        table[b, : N[b]] = perm[off: off + N[b]]
        off += int(N[b])
    return table


def make_problem(cfg: Config | str, layer: int = 0, with_kv: bool = True,
                 stride_pad: int = 0) -> Problem:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    seq_lens = make_lengths(cfg)
    N = seq_lens.astype(np.int64) + cfg.num_nodes
    num_slots = cfg.pool_slots or int(N.sum())
    assert num_slots >= int(N.sum())
    stride = int(N.max()) + stride_pad
    table = make_slot_table(cfg, seq_lens, num_slots, stride)
    trees = make_trees(cfg)
    q_seed = tensor_seed(cfg.config_id, layer, STREAM_Q)
    kv_seed = tensor_seed(cfg.config_id, layer, STREAM_KV)
    rows = cfg.num_seqs * cfg.num_nodes * cfg.num_heads
    q = normal_bf16(q_seed, rows * D_K).reshape(cfg.num_seqs * cfg.num_nodes, cfg.num_heads, D_K)
    kv = normal_bf16(kv_seed, num_slots * D_K).reshape(num_slots, D_K) if with_kv else None
    return Problem(cfg, seq_lens, trees, table, q, kv, num_slots, kv_seed, q_seed)


def custom_problem(seq_lens: List[int], T: int, H: int, *, tree: str = "random", seed: int = 1,
                   pool_slack: int = 0, identity: bool = False, stride_pad: int = 0) -> Problem:
    """A small problem of any shape (parity and edge cases), same recipe as the named configs."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = len(seq_lens)
    cfg = Config(f"custom{seed}", 8 + seed, B, T, H, tree, "fixed", identity_table=identity)
    N = seq_lens.astype(np.int64) + T
    num_slots = int(N.sum()) + pool_slack
    stride = int(N.max()) + stride_pad
    table = make_slot_table(cfg, seq_lens, num_slots, stride)
    if tree == "chain":
        trees = np.stack([chain_tree(T)] * B)
    elif tree == "star":
        trees = np.stack([star_tree(T)] * B)
    else:
        s = tensor_seed(cfg.config_id, 0, STREAM_TREE)
        trees = np.stack([random_tree(splitmix64_scalar(s, b), T) for b in range(B)])
    q_seed = tensor_seed(cfg.config_id, 0, STREAM_Q)
    kv_seed = tensor_seed(cfg.config_id, 0, STREAM_KV)
    q = normal_bf16(q_seed, B * T * H * D_K).reshape(B * T, H, D_K)
    kv = normal_bf16(kv_seed, num_slots * D_K).reshape(num_slots, D_K)
    return Problem(cfg, seq_lens, trees, table, q, kv, num_slots, kv_seed, q_seed)


def kv_bytes_per_layer_step(seq_lens, T: int) -> int:
    """Algorithmic KV bytes of one layer-step: each visible token's 1152-B row plus its 4-B slot entry."""
    N = np.asarray(seq_lens, dtype=np.int64) + T
    return int(N.sum()) * (D_K * 2 + 4)


def algorithmic_bytes(seq_lens, T: int, H: int) -> int:
    """KV + slot bytes plus each row's q (1152 B), out (1024 B bf16) and lse (4 B)."""
    rows = len(seq_lens) * T * H
    return kv_bytes_per_layer_step(seq_lens, T) + rows * (D_K * 2 + D_V * 2 + 4)


def algorithmic_flops(seq_lens, T: int, H: int) -> int:
    """2 * rows * (576 + 512) per visible token (masked tree work excluded)."""
    N = np.asarray(seq_lens, dtype=np.int64) + T
    return int(2 * T * H * (D_K + D_V) * N.sum())
