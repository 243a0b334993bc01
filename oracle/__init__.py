"""Float64 CPU oracle for tree-verify MLA attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers. The library's product path
never imports this package, and this package imports nothing from the library.

The arithmetic lives in ``mla_oracle.c`` (plain loops, float64, OpenMP over
rows); this module compiles it with gcc and marshals numpy arrays through
ctypes. See the C file's header for the definition it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "libmla_oracle.so")
_lib = None

ERRORS = {0: "ok", -1: "invalid argument", -2: "tree parent out of order", -3: "slot out of range",
          -4: "out of memory"}


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags: the same source builds on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def build_mutant(mutation: int, out_dir: str) -> str:
    """Compile a planted-mistake build (``-DORACLE_MUTATION=n``) into ``out_dir``; for the pin tests."""
    path = os.path.join(out_dir, f"libmla_oracle_mut{mutation}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", f"-DORACLE_MUTATION={mutation}",
                    "-o", path, _SRC, "-lm"], check=True)
    return path


def _declare(lib):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_verify.argtypes = [i32, i32, i32, i32, i32, P, P, i64, P, P, P, i64, f64, P, i64,
                                  i64, i64, P, P, i32]
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_row_weights.argtypes = [i32, i32, i32, i32, i32, P, P, i64, P, P, P, i64, f64, i64, P]
    lib.oracle_row_weights.restype = ctypes.c_int
    lib.oracle_combine.argtypes = [i32, i64, i32, P, P, P, P]
    lib.oracle_combine.restype = ctypes.c_int
    lib.oracle_ancestor_masks.argtypes = [i32, P, P]
    lib.oracle_ancestor_masks.restype = ctypes.c_int
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


_active = None  # a planted-mistake library installed by the pin tests, else None


class use_library:
    """Context manager: route every oracle call through the library at ``path`` (pin tests only)."""

    def __init__(self, path: str):
        self.lib = _declare(ctypes.CDLL(path))

    def __enter__(self):
        global _active
        self.prev, _active = _active, self.lib
        return self

    def __exit__(self, *exc):
        global _active
        _active = self.prev


def _load():
    global _lib
    if _active is not None:
        return _active
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        _lib = _declare(lib)
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle error {rc}: {ERRORS.get(rc, 'unknown')}")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def ancestor_masks(parent: np.ndarray) -> np.ndarray:
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    out = np.zeros(len(parent), dtype=np.uint64)
    _check(_load().oracle_ancestor_masks(len(parent), _ptr(parent), _ptr(out)))
    return out


def verify(seq_lens, slot_table, tree_parent, q, kv, *, num_heads: int, scale: float,
           d_latent: int = 512, d_rope: int = 64, rows: Optional[Sequence[int]] = None,
           pos_begin: int = 0, pos_end: int = 2 ** 62, num_threads: int = 0):
    """Exact attention in float64. Returns (out [rows, d_latent], lse [rows]).

    ``q``: uint16 bf16 bits [B*T, H, d_latent + d_rope]; ``kv``: uint16 [num_slots, d_latent + d_rope];
    ``slot_table``: int32 [B, stride]; ``tree_parent``: int32 [B, T]; ``seq_lens``: int32 [B] prefix lengths.
    ``rows``: global row ids ``(b*T + i)*H + h`` (default all, in order).
    """
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    slot_table = np.ascontiguousarray(slot_table, dtype=np.int32)
    tree_parent = np.ascontiguousarray(tree_parent, dtype=np.int32)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kv = np.ascontiguousarray(kv, dtype=np.uint16)
    B = len(seq_lens)
    T = tree_parent.shape[-1]
    H = num_heads
    dk = d_latent + d_rope
    assert q.size == B * T * H * dk and kv.shape[-1] == dk
    assert tree_parent.shape == (B, T) and slot_table.shape[0] == B
    if rows is None:
        rows_arr = None
        n = B * T * H
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = len(rows_arr)
    out = np.zeros((n, d_latent), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    _check(_load().oracle_verify(B, T, H, d_latent, d_rope, _ptr(seq_lens), _ptr(slot_table),
                                 slot_table.shape[1], _ptr(tree_parent), _ptr(q), _ptr(kv),
                                 kv.shape[0], float(scale),
                                 _ptr(rows_arr) if rows_arr is not None else None, n,
                                 int(pos_begin), int(pos_end), _ptr(out), _ptr(lse), int(num_threads)))
    return out, lse


def row_weights(seq_lens, slot_table, tree_parent, q, kv, row: int, *, num_heads: int, scale: float,
                d_latent: int = 512, d_rope: int = 64) -> np.ndarray:
    """Softmax weights of one row over logical positions 0..N_b-1 (0 where not visible)."""
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    slot_table = np.ascontiguousarray(slot_table, dtype=np.int32)
    tree_parent = np.ascontiguousarray(tree_parent, dtype=np.int32)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kv = np.ascontiguousarray(kv, dtype=np.uint16)
    B, T = tree_parent.shape
    b = row // num_heads // T
    w = np.zeros(int(seq_lens[b]) + T, dtype=np.float64)
    _check(_load().oracle_row_weights(B, T, num_heads, d_latent, d_rope, _ptr(seq_lens), _ptr(slot_table),
                                      slot_table.shape[1], _ptr(tree_parent), _ptr(q), _ptr(kv),
                                      kv.shape[0], float(scale), int(row), _ptr(w)))
    return w


def combine(part_o: np.ndarray, part_lse: np.ndarray):
    """Merge partials [S, rows, d_v] / [S, rows] into (out [rows, d_v], lse [rows]), float64."""
    part_o = np.ascontiguousarray(part_o, dtype=np.float64)
    part_lse = np.ascontiguousarray(part_lse, dtype=np.float64)
    S, rows, d_v = part_o.shape
    out = np.zeros((rows, d_v), dtype=np.float64)
    lse = np.zeros(rows, dtype=np.float64)
    _check(_load().oracle_combine(S, rows, d_v, _ptr(part_o), _ptr(part_lse), _ptr(out), _ptr(lse)))
    return out, lse


def verify_problem(p, scale: float, rows=None, **kw):
    """``verify`` on a seeded problem object (fields seq_lens, slot_table, tree_parent, q, kv, H)."""
    return verify(p.seq_lens, p.slot_table, p.tree_parent, p.q, p.kv, num_heads=p.H, scale=scale,
                  rows=rows, **kw)


# ---------------------------------------------------------------------------------------------
# KV-pool steps around verification (plain numpy, the definitions written out). They follow
# "The Moment of Certainty", The Final Piece (the tree nodes' rows live at their own slots,
# and accepted nodes are scattered, so accepting a path rewrites the slot table) and "The Moment
# of Reckoning (User Challenge...)", Output, item 4 (Tier-0 defragmentation keeps each request's
# KV contiguous in the pool).

def tree_kv_append(pool: np.ndarray, tree_kv: np.ndarray, slot_table: np.ndarray, seq_lens: np.ndarray,
                   num_nodes: int) -> np.ndarray:
    """pool[slot_table[b][L_b + j]] = tree_kv[b*T + j]; returns the new pool (the input is not modified)."""
    out = pool.copy()
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        for j in range(num_nodes):
            out[int(slot_table[b, L + j])] = tree_kv[b * num_nodes + j]
    return out


def tree_accept_commit(slot_table: np.ndarray, seq_lens: np.ndarray, tree_parent: np.ndarray,
                       accepted: np.ndarray, num_accepted: np.ndarray, max_seq_len: int):
    """Accepted path first (in path order) behind the prefix, then the rejected nodes in node order;
    seq_lens += n. An invalid path (not root-first along parent links, n outside [0, T], or a prefix
    longer than max_seq_len) leaves the sequence unchanged. Returns (table, lens, valid per sequence)."""
    table = slot_table.copy()
    lens = seq_lens.copy()
    T = tree_parent.shape[1]
    valid = np.zeros(len(seq_lens), dtype=bool)
    for b in range(len(seq_lens)):
        L, n = int(seq_lens[b]), int(num_accepted[b])
        if not (0 <= L <= max_seq_len and 0 <= n <= T and L + n <= max_seq_len):
            continue
        path = [int(a) for a in accepted[b, :n]]
        ok = all(0 <= a < T for a in path) and len(set(path)) == n
        if ok:
            for k, a in enumerate(path):
                if int(tree_parent[b, a]) != (path[k - 1] if k else -1):
                    ok = False
        if not ok:
            continue
        old = [int(x) for x in slot_table[b, L:L + T]]
        order = path + [j for j in range(T) if j not in path]
        for pos, node in enumerate(order):
            table[b, L + pos] = old[node]
        lens[b] = L + n
        valid[b] = True
    return table, lens, valid


def kv_compact(src_pool: np.ndarray, slot_table: np.ndarray, seq_lens: np.ndarray, num_nodes: int,
               dst_base: np.ndarray, dst_slots: int):
    """dst[dst_base[b] + t] = src[slot_table[b][t]] and new_table[b][t] = dst_base[b] + t for
    t < L_b + T; rows of dst outside every range stay zero. Returns (dst, new_table)."""
    dst = np.zeros((dst_slots,) + src_pool.shape[1:], dtype=src_pool.dtype)
    table = slot_table.copy()
    for b in range(len(seq_lens)):
        for t in range(int(seq_lens[b]) + num_nodes):
            d = int(dst_base[b]) + t
            dst[d] = src_pool[int(slot_table[b, t])]
            table[b, t] = d
    return dst, table
