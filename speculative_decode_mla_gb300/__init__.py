"""Tree-verify MLA attention over a page_size=1 latent KV pool, on one GB300 (sm_103a).

A thin ctypes binding of the C ABI in ``include/mla_verify.h`` (``libmla_verify.so``,
built in-tree by ``_build.build()``). Every step of the computation runs in the
library's CUDA kernels; this module only marshals arguments. PyTorch provides
device memory and streams. There is no CPU fallback: if the library is missing
or no sm_103 device is present, calls raise.

    out, lse = verify(q, kv_pool, slot_table, seq_lens, tree_parent, max_seq_len=L)
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_verify.so")

MLA_OK = 0
MLA_DTYPE_BF16, MLA_DTYPE_F32, MLA_DTYPE_F16 = 0, 1, 2
MLA_FLAG_DEBUG_CHECKS, MLA_FLAG_SIMT, MLA_FLAG_PREFIX_STABLE = 1, 2, 4
CHECK_BAD_SLOT, CHECK_BAD_PARENT, CHECK_BAD_LENGTH, CHECK_TIMEOUT = 1, 2, 4, 8
D_LATENT, D_ROPE = 512, 64
DEFAULT_SCALE = 1.0 / math.sqrt(192.0)

# The kernel a default call runs (the tcgen05 kernel): flags used unless a call overrides them.
DEFAULT_FLAGS = 0


class Desc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_nodes", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("d_latent", ctypes.c_int32), ("d_rope", ctypes.c_int32), ("slot_table_stride", ctypes.c_int32),
                ("num_slots", ctypes.c_int64), ("max_seq_len", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("out_dtype", ctypes.c_int32), ("flags", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("total_tokens_hint", ctypes.c_int64)]


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("num_splits", ctypes.c_int32), ("chunk_tokens", ctypes.c_int32),
                ("row_tiles", ctypes.c_int32), ("rows_per_tile", ctypes.c_int32), ("ctas", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64)]


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def load_library(path: str = LIB_PATH):
    """Load (once) the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: run __graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.mla_verify_plan.argtypes = [ctypes.POINTER(Desc), i32, ctypes.POINTER(Plan)]
    lib.mla_verify_workspace_size.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(ctypes.c_size_t)]
    lib.mla_verify_attn.argtypes = [ctypes.POINTER(Desc), P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
    lib.mla_verify_attn_partials.argtypes = [ctypes.POINTER(Desc), P, P, P, P, P, P, ctypes.c_size_t, P, P]
    lib.mla_verify_attn_hybrid.argtypes = [ctypes.POINTER(Desc), P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
    lib.mla_verify_attn_ragged.argtypes = [ctypes.POINTER(Desc), P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
    lib.mla_verify_combine.argtypes = [i32, i64, i32, P, i32, P, P, P, i32, P]
    lib.mla_verify_status_string.argtypes = [ctypes.c_int]
    lib.mla_verify_status_string.restype = ctypes.c_char_p
    lib.mla_fill_normal_bf16.argtypes = [P, i64, ctypes.c_uint64, ctypes.c_uint64, P]
    lib.mla_tree_kv_append.argtypes = [P, i64, P, P, P, i32, i32, i32, i32, i32, P, P]
    lib.mla_tree_accept_commit.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, P, P]
    lib.mla_kv_compact.argtypes = [P, i64, P, i64, P, P, P, P, i32, i32, i32, i32, i32, P, P]
    for f in ("mla_verify_plan", "mla_verify_workspace_size", "mla_verify_attn", "mla_verify_attn_partials",
              "mla_verify_attn_hybrid", "mla_verify_attn_ragged",
              "mla_verify_combine", "mla_fill_normal_bf16", "mla_tree_kv_append", "mla_tree_accept_commit",
              "mla_kv_compact"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().mla_verify_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != MLA_OK:
        raise MLAError(rc, what)


def make_desc(num_seqs, num_nodes, num_heads, num_slots, slot_table_stride, max_seq_len, *,
              softmax_scale: float = DEFAULT_SCALE, out_dtype: int = MLA_DTYPE_BF16,
              flags: Optional[int] = None, num_splits: int = 0, total_tokens_hint: int = 0) -> Desc:
    return Desc(int(num_seqs), int(num_nodes), int(num_heads), D_LATENT, D_ROPE, int(slot_table_stride),
                int(num_slots), int(max_seq_len), float(softmax_scale), int(out_dtype),
                DEFAULT_FLAGS if flags is None else int(flags), int(num_splits), int(total_tokens_hint))


def plan(desc: Desc, num_sms: int) -> Plan:
    p = Plan()
    _check(load_library().mla_verify_plan(ctypes.byref(desc), int(num_sms), ctypes.byref(p)), "mla_verify_plan")
    return p


def workspace_size(desc: Desc) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().mla_verify_workspace_size(ctypes.byref(desc), ctypes.byref(n)),
           "mla_verify_workspace_size")
    return int(n.value)


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def verify_attn_raw(desc: Desc, q: int, kv_pool: int, slot_table: int, seq_lens: int, tree_parent: int,
                    out: int, lse: int, workspace: int, workspace_bytes: int, dev_status: int, stream: int) -> int:
    """Direct C-ABI call with integer device pointers; returns the status code."""
    return load_library().mla_verify_attn(ctypes.byref(desc), q, kv_pool, slot_table, seq_lens, tree_parent, out,
                                          lse, workspace, int(workspace_bytes), dev_status or None, stream or None)


def verify_attn_hybrid_raw(desc: Desc, q: int, kv_pool: int, prefix_base: int, tree_slots: int, seq_lens: int,
                           tree_parent: int, out: int, lse: int, workspace: int, workspace_bytes: int, dev_status: int,
                           stream: int) -> int:
    """Direct C-ABI call of the hybrid-addressing verify (contiguous prefix + per-node tree slots)."""
    return load_library().mla_verify_attn_hybrid(ctypes.byref(desc), q, kv_pool, prefix_base, tree_slots, seq_lens,
                                                 tree_parent, out, lse, workspace, int(workspace_bytes),
                                                 dev_status or None, stream or None)


def verify_hybrid(q, kv_pool, prefix_base, tree_slots, seq_lens, tree_parent, *, max_seq_len: int,
                  softmax_scale: float = DEFAULT_SCALE, out_dtype: int = MLA_DTYPE_BF16, flags: Optional[int] = None,
                  num_splits: int = 0, dev_status=None, stream=None):
    """Tree-verify attention with hybrid addressing: prefix position t of sequence b is slot
    prefix_base[b] + t (int64 [B]); tree node j is slot tree_slots[b, j] (int32 [B, T])."""
    import torch
    B, T = tree_parent.shape
    H = q.shape[1]
    desc = make_desc(B, T, H, kv_pool.shape[0], max_seq_len + T, max_seq_len, softmax_scale=softmax_scale,
                     out_dtype=out_dtype, flags=DEFAULT_FLAGS if flags is None else flags, num_splits=num_splits)
    ws = torch.empty(workspace_size(desc), dtype=torch.uint8, device=q.device)
    out = torch.empty((B * T, H, 512), device=q.device,
                      dtype=torch.bfloat16 if out_dtype == MLA_DTYPE_BF16 else torch.float32)
    lse = torch.empty((B * T, H), dtype=torch.float32, device=q.device)
    rc = verify_attn_hybrid_raw(desc, q.data_ptr(), kv_pool.data_ptr(), prefix_base.data_ptr(), tree_slots.data_ptr(),
                                seq_lens.data_ptr(), tree_parent.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                ws.data_ptr(), ws.numel(), _ptr_or_none(dev_status), _stream_ptr(stream))
    _check(rc, "mla_verify_attn_hybrid")
    return out, lse


def verify_attn_ragged_raw(desc: Desc, q: int, kv_pool: int, slot_table: int, seq_lens: int, tree_sizes: int,
                           tree_parent: int, out: int, lse: int, workspace: int, workspace_bytes: int, dev_status: int,
                           stream: int) -> int:
    """Direct C-ABI call of the ragged-tree verify (tree_sizes int32 [B], T_b <= desc.num_nodes)."""
    return load_library().mla_verify_attn_ragged(ctypes.byref(desc), q, kv_pool, slot_table, seq_lens, tree_sizes,
                                                 tree_parent, out, lse, workspace, int(workspace_bytes),
                                                 dev_status or None, stream or None)


def verify_attn_partials_raw(desc: Desc, q: int, kv_pool: int, slot_table: int, seq_lens: int, tree_parent: int,
                             workspace: int, workspace_bytes: int, dev_status: int, stream: int) -> int:
    """Direct C-ABI call of the split stage alone (partials into the workspace); returns the status code."""
    return load_library().mla_verify_attn_partials(ctypes.byref(desc), q, kv_pool, slot_table, seq_lens, tree_parent,
                                                   workspace, int(workspace_bytes), dev_status or None, stream or None)


def partials_views(workspace, plan: Plan, rows: int):
    """(part_o fp16 [splits, rows, 512], part_lse fp32 [splits, rows]) views of a uint8 workspace tensor."""
    import torch
    o_bytes = plan.num_splits * rows * 512 * 2
    l_off = (o_bytes + 255) // 256 * 256
    part_o = workspace[:o_bytes].view(torch.float16).view(plan.num_splits, rows, 512)
    part_l = workspace[l_off:l_off + plan.num_splits * rows * 4].view(torch.float32).view(plan.num_splits, rows)
    return part_o, part_l


def verify(q, kv_pool, slot_table, seq_lens, tree_parent, *, max_seq_len: int,
           softmax_scale: float = DEFAULT_SCALE, out_dtype: int = MLA_DTYPE_BF16, flags: Optional[int] = None,
           num_splits: int = 0, total_tokens_hint: int = 0, out=None, lse=None, workspace=None,
           dev_status=None, stream=None, tree_sizes=None):
    """Tree-verify attention on torch CUDA tensors (see ``include/mla_verify.h``).

    q: bf16 [B*T, H, 576]; kv_pool: bf16 [num_slots, 576]; slot_table: int32 [B, stride];
    seq_lens: int32 [B]; tree_parent: int32 [B, T]. Returns (out [B*T, H, 512], lse [B*T, H]).
    Buffers may be passed in to avoid allocation (out, lse, workspace as a uint8 tensor).
    tree_sizes (int32 [B], each in 1..T) selects the ragged-tree call (mla_verify_attn_ragged).
    """
    import torch
    B, T = tree_parent.shape
    H = q.shape[1]
    desc = make_desc(B, T, H, kv_pool.shape[0], slot_table.shape[1], max_seq_len, softmax_scale=softmax_scale,
                     out_dtype=out_dtype, flags=flags, num_splits=num_splits, total_tokens_hint=total_tokens_hint)
    for t in (q, kv_pool, slot_table, seq_lens, tree_parent):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("inputs must be contiguous CUDA tensors")
    dev = q.device
    if out is None:
        out = torch.empty((B * T, H, D_LATENT), device=dev,
                          dtype=torch.bfloat16 if out_dtype == MLA_DTYPE_BF16 else torch.float32)
    if lse is None:
        lse = torch.empty((B * T, H), device=dev, dtype=torch.float32)
    if workspace is None:
        workspace = torch.empty(workspace_size(desc), device=dev, dtype=torch.uint8)
    if tree_sizes is not None:
        rc = verify_attn_ragged_raw(desc, q.data_ptr(), kv_pool.data_ptr(), slot_table.data_ptr(),
                                    seq_lens.data_ptr(), tree_sizes.data_ptr(), tree_parent.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                    dev_status.data_ptr() if dev_status is not None else 0, _stream_ptr(stream))
        _check(rc, "mla_verify_attn_ragged")
        return out, lse
    rc = verify_attn_raw(desc, q.data_ptr(), kv_pool.data_ptr(), slot_table.data_ptr(), seq_lens.data_ptr(),
                         tree_parent.data_ptr(), out.data_ptr(), lse.data_ptr(), workspace.data_ptr(),
                         workspace.numel(), dev_status.data_ptr() if dev_status is not None else 0,
                         _stream_ptr(stream))
    _check(rc, "mla_verify_attn")
    return out, lse


def combine(part_o, part_lse, *, out_dtype: int = MLA_DTYPE_BF16, out=None, lse=None, stream=None):
    """LSE-weighted merge of partials: part_o f32 or f16 [S, rows, d_v], part_lse f32 [S, rows]."""
    import torch
    S, rows, d_v = part_o.shape
    if out is None:
        out = torch.empty((rows, d_v), device=part_o.device,
                          dtype=torch.bfloat16 if out_dtype == MLA_DTYPE_BF16 else torch.float32)
    if lse is None:
        lse = torch.empty((rows,), device=part_o.device, dtype=torch.float32)
    part_dtype = MLA_DTYPE_F16 if part_o.dtype == torch.float16 else MLA_DTYPE_F32
    if part_o.dtype not in (torch.float16, torch.float32):
        raise ValueError("part_o must be float32 or float16")
    rc = load_library().mla_verify_combine(S, rows, d_v, part_o.data_ptr(), part_dtype, part_lse.data_ptr(),
                                           out.data_ptr(), lse.data_ptr(), out_dtype, _stream_ptr(stream))
    _check(rc, "mla_verify_combine")
    return out, lse


def tree_kv_append(pool, tree_kv, slot_table, seq_lens, *, max_seq_len: int, debug: bool = False,
                   dev_status=None, stream=None):
    """Write the tree nodes' rows into their slots (``include/mla_kv_ops.h``). pool bf16 [slots, 576],
    tree_kv bf16 [B*T, 576], slot_table int32 [B, stride], seq_lens int32 [B]. In place on pool."""
    B = seq_lens.shape[0]
    T = tree_kv.shape[0] // B
    rc = load_library().mla_tree_kv_append(pool.data_ptr(), pool.shape[0], tree_kv.data_ptr(), slot_table.data_ptr(),
                                           seq_lens.data_ptr(), B, T, slot_table.shape[1], max_seq_len, int(debug),
                                           _ptr_or_none(dev_status), _stream_ptr(stream))
    _check(rc, "mla_tree_kv_append")
    return pool


def tree_accept_commit(slot_table, seq_lens, tree_parent, accepted, num_accepted, *, max_seq_len: int,
                       debug: bool = False, dev_status=None, stream=None):
    """Move the accepted path's slots behind the prefix and advance seq_lens (in place)."""
    B, T = tree_parent.shape
    rc = load_library().mla_tree_accept_commit(slot_table.data_ptr(), seq_lens.data_ptr(), tree_parent.data_ptr(),
                                               accepted.data_ptr(), num_accepted.data_ptr(), B, T,
                                               slot_table.shape[1], max_seq_len, int(debug),
                                               _ptr_or_none(dev_status), _stream_ptr(stream))
    _check(rc, "mla_tree_accept_commit")
    return slot_table, seq_lens


def kv_compact(src_pool, dst_pool, slot_table, seq_lens, dst_base, *, num_nodes: int, max_seq_len: int,
               new_slot_table=None, debug: bool = False, dev_status=None, stream=None):
    """Tier-0 compaction: copy each sequence's rows into dst_pool[dst_base[b]:] and rewrite new_slot_table."""
    rc = load_library().mla_kv_compact(src_pool.data_ptr(), src_pool.shape[0], dst_pool.data_ptr(), dst_pool.shape[0],
                                       slot_table.data_ptr(), _ptr_or_none(new_slot_table), seq_lens.data_ptr(),
                                       dst_base.data_ptr(), seq_lens.shape[0], num_nodes, slot_table.shape[1],
                                       max_seq_len, int(debug), _ptr_or_none(dev_status), _stream_ptr(stream))
    _check(rc, "mla_kv_compact")
    return dst_pool, new_slot_table


def _ptr_or_none(t):
    return None if t is None else t.data_ptr()


def fill_normal_bf16(dst, seed: int, start: int = 0, stream=None):
    """Draw the seeded synthetic bf16 stream into a CUDA tensor in place (``include/mla_workload.h``)."""
    rc = load_library().mla_fill_normal_bf16(dst.data_ptr(), dst.numel(), seed & ((1 << 64) - 1), start,
                                             _stream_ptr(stream))
    _check(rc, "mla_fill_normal_bf16")
    return dst
