"""The C-ABI library on the CPU: it loads, exports every declared symbol, plans, and rejects bad input.

No compute call is made here (no GPU); every check below returns before any CUDA call.
"""
import ctypes
import glob
import os
import re

import pytest

import speculative_decode_mla_gb300 as m
from speculative_decode_mla_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return m.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for mt in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                              src, flags=re.M):
            names.add(mt.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "mla_verify_attn" in names and "mla_verify_combine" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/*.h but not exported"


def test_library_links_no_oracle_code():
    syms = os.popen(f"nm -D --defined-only {m.LIB_PATH}").read()
    assert "oracle_" not in syms


def desc(**kw):
    base = dict(num_seqs=1, num_nodes=16, num_heads=8, num_slots=131072, slot_table_stride=65552,
                max_seq_len=65536)
    base.update(kw)
    return m.make_desc(base.pop("num_seqs"), base.pop("num_nodes"), base.pop("num_heads"), base.pop("num_slots"),
                       base.pop("slot_table_stride"), base.pop("max_seq_len"), **base)


def test_plan_64k_fills_the_gpu(lib):
    p = m.plan(desc(flags=0), 152)
    assert p.kernel == 0 and p.rows_per_tile == 128 and p.row_tiles == 1
    assert p.chunk_tokens % 64 == 0  # whole 64-position KV tiles
    assert p.num_splits * p.chunk_tokens >= 65552 > (p.num_splits - 1) * p.chunk_tokens
    assert 60 <= p.num_splits <= 76 and p.ctas == 2 * p.num_splits
    assert p.workspace_bytes >= p.num_splits * 128 * 512 * 2 + p.num_splits * 128 * 4


def test_plan_forced_splits_and_simt(lib):
    p = m.plan(desc(num_splits=5, flags=m.MLA_FLAG_SIMT), 152)
    assert p.kernel == 1 and p.num_splits == 5 and p.rows_per_tile == 8 and p.row_tiles == 16
    p = m.plan(desc(num_splits=1, flags=0), 152)
    assert p.num_splits == 1 and p.chunk_tokens >= 65552


def test_plan_is_deterministic_and_pure(lib):
    a = m.plan(desc(flags=0, num_heads=64, num_nodes=64, max_seq_len=131072, slot_table_stride=131136), 152)
    b = m.plan(desc(flags=0, num_heads=64, num_nodes=64, max_seq_len=131072, slot_table_stride=131136), 152)
    assert bytes(a) == bytes(b) and a.row_tiles == 32


def test_plan_ragged_hint_uses_more_splits(lib):
    d0 = desc(num_seqs=32, num_nodes=8, num_heads=16, max_seq_len=32767, slot_table_stride=32775, flags=0)
    d1 = desc(num_seqs=32, num_nodes=8, num_heads=16, max_seq_len=32767, slot_table_stride=32775, flags=0,
              total_tokens_hint=300000)
    assert m.plan(d1, 152).chunk_tokens <= m.plan(d0, 152).chunk_tokens


@pytest.mark.parametrize("total", [20000, 300000, 1000000])
def test_plan_ragged_full_chunks_fit_one_wave(lib, total):
    """A ragged batch (2..64 sequences, lengths summed in the hint): however the lengths fall, its
    full chunks number at most total / chunk, and the chunk is the clusters' even share of all
    tiles, so they never outnumber the 76 cluster slots of a 152-SM part."""
    d = desc(num_seqs=32, num_nodes=8, num_heads=16, max_seq_len=32767, slot_table_stride=32775, flags=0,
             total_tokens_hint=total)
    p = m.plan(d, 152)
    tiles = -(-total // 64)
    assert p.chunk_tokens == max(1, -(-tiles // 76)) * 64
    assert total // p.chunk_tokens <= 76
    assert p.num_splits * p.chunk_tokens >= 32767 + 8


@pytest.mark.parametrize("bad", [dict(num_nodes=0), dict(num_nodes=65), dict(num_heads=0), dict(num_seqs=0),
                                 dict(slot_table_stride=100), dict(num_slots=0), dict(max_seq_len=-1),
                                 dict(softmax_scale=float("nan")), dict(out_dtype=7), dict(flags=1 << 9),
                                 dict(num_splits=-2)])
def test_plan_rejects_bad_desc(lib, bad):
    d = desc(**bad)
    out = m.Plan()
    rc = lib.mla_verify_plan(ctypes.byref(d), 152, ctypes.byref(out))
    assert rc in (-1, -2)


def test_unsupported_dims(lib):
    d = desc()
    d.d_latent = 256
    assert lib.mla_verify_plan(ctypes.byref(d), 152, ctypes.byref(m.Plan())) == -2


def test_attn_rejects_null_and_misaligned_pointers(lib):
    d = desc()
    fake = 1 << 20
    args = [fake] * 5 + [fake, fake, fake]
    assert m.verify_attn_raw(d, 0, *args[1:5], *args[5:], 1 << 30, 0, 0) == -1
    assert m.verify_attn_raw(d, fake + 2, *args[1:5], *args[5:], 1 << 30, 0, 0) == -1  # q not 16-B aligned
    dd = desc(flags=m.MLA_FLAG_DEBUG_CHECKS)
    assert m.verify_attn_raw(dd, *args, 1 << 30, 0, 0) == -1  # debug checks need dev_status


def test_partials_rejects_null_and_misaligned_pointers(lib):
    d = desc()
    fake = 1 << 20
    f = m.verify_attn_partials_raw
    assert f(d, 0, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -1         # null q
    assert f(d, fake, fake, fake, fake, fake, 0, 1 << 30, 0, 0) == -1         # null workspace
    assert f(d, fake, fake, fake, fake, fake, fake + 16, 1 << 30, 0, 0) == -1  # workspace not 256-B aligned
    assert f(desc(flags=m.MLA_FLAG_DEBUG_CHECKS), fake, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -1
    assert f(desc(num_nodes=0), fake, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -2


def test_hybrid_rejects_null_and_misaligned_pointers(lib):
    d = desc(slot_table_stride=0)  # ignored by the hybrid call
    fake = 1 << 20
    f = m.verify_attn_hybrid_raw
    assert f(d, fake, fake, 0, fake, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -1      # no prefix_base
    assert f(d, fake, fake, fake, 0, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -1      # no tree_slots
    assert f(d, fake, fake, fake + 4, fake, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -1  # base not 8-B aligned
    assert f(d, fake, fake, fake, fake, fake, fake, 0, fake, fake, 1 << 30, 0, 0) == -1      # no out
    assert f(desc(num_nodes=65), fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -2


def test_ragged_rejects_null_and_misaligned_tree_sizes(lib):
    d = desc()
    fake = 1 << 20
    f = m.verify_attn_ragged_raw
    assert f(d, fake, fake, fake, fake, 0, fake, fake, fake, fake, 1 << 30, 0, 0) == -1      # no tree_sizes
    assert f(d, fake, fake, fake, fake, fake + 2, fake, fake, fake, fake, 1 << 30, 0, 0) == -1  # misaligned
    assert f(desc(num_nodes=65), fake, fake, fake, fake, fake, fake, fake, fake, fake, 1 << 30, 0, 0) == -2


def test_combine_rejects_bad_args(lib):
    f = lib.mla_verify_combine
    assert f(0, 4, 512, 16, 1, 16, 16, 16, 0, None) == -1      # no splits
    assert f(2, 4, 510, 16, 1, 16, 16, 16, 0, None) == -1      # d_v not a multiple of 4
    assert f(2, 4, 512, 16, 1, 16, 16, 16, 5, None) == -1      # bad output dtype
    assert f(2, 4, 512, 16, 0, 16, 16, 16, 0, None) == -1      # partials must be f32 or f16
    assert f(2, 4, 512, 0, 1, 16, 16, 16, 0, None) == -1       # null partials


def test_status_strings(lib):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert m.status_string(s) and m.status_string(s) != "unknown status"
    assert m.status_string(-99) == "unknown status"


def test_fill_rejects_bad_args(lib):
    assert lib.mla_fill_normal_bf16(None, 10, 1, 0, None) == -1
    assert lib.mla_fill_normal_bf16(16, -1, 1, 0, None) == -1
    assert lib.mla_fill_normal_bf16(None, 0, 1, 0, None) == 0
