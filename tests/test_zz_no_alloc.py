"""mla_verify_attn_noalloc: the verify call for callers that cannot allocate device memory.

Some callers of this library have no way to obtain a workspace: a plugin that its
host framework hands only input and output device pointers, a serving process that
has reserved nearly all device memory for its KV pool, a decode loop that cannot
afford a device-synchronising cudaMalloc. For them the library keeps its own fixed
32 MiB scratch array in device memory and takes no workspace argument.

These tests call that entry point through the C ABI and check, on several calls in
a row (each reusing the scratch the previous one left behind), that its output
matches the workspace-taking entry point bit for bit, and so within the parity
tolerances used by the other GPU tests. The file name sorts last so a stop-at-first-failure run has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from _helpers import TOL_LSE_ABS, TOL_MAX_ABS, TOL_REL_L2, device_problem
from speculative_decode_mla_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    import speculative_decode_mla_gb300 as m
    from speculative_decode_mla_gb300 import _build
    _build.build()
    lib = m.load_library()
    f = lib.mla_verify_attn_noalloc
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(m.Desc), P, P, P, P, P, P, P, P, P]
    f.restype = ctypes.c_int
    return lib


def _call_noalloc(lib, p, dev, flags=0):
    import torch
    import speculative_decode_mla_gb300 as m
    q, kv, st, sl, tp = dev
    desc = m.make_desc(p.B, p.T, p.H, p.num_slots, p.stride, p.max_seq_len, flags=flags)
    out = torch.full((p.B * p.T, p.H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((p.B * p.T, p.H), float("nan"), dtype=torch.float32, device="cuda")
    rc = lib.mla_verify_attn_noalloc(ctypes.byref(desc), q.data_ptr(), kv.data_ptr(), st.data_ptr(), sl.data_ptr(),
                                     tp.data_ptr(), out.data_ptr(), lse.data_ptr(), None,
                                     torch.cuda.current_stream().cuda_stream)
    return rc, out, lse


def _call_with_workspace(p, dev, flags=0):
    import speculative_decode_mla_gb300 as m
    q, kv, st, sl, tp = dev
    return m.verify(q, kv, st, sl, tp, max_seq_len=p.max_seq_len, flags=flags)


def _compare(a_out, a_lse, b_out, b_lse):
    a = a_out.float().cpu().numpy().astype(np.float64)
    b = b_out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(a).all()
    err = np.abs(a - b).max()
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    lerr = np.abs(a_lse.cpu().numpy() - b_lse.cpu().numpy()).max()
    assert err <= TOL_MAX_ABS and rel <= TOL_REL_L2 and lerr <= TOL_LSE_ABS, (err, rel, lerr)


def _bits_equal(a, b):
    import torch
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def _assert_bit_identical(out, lse, ref_out, ref_lse):
    assert _bits_equal(out, ref_out) and _bits_equal(lse, ref_lse)


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(lib):
    """Calls in a row share the scratch and find the previous call's partials there. Both entry
    points run the same plan and kernels, so their results must agree bit for bit (and with the
    parity tolerances). The small problem runs both before and after the large one, so a partial
    that the second small call failed to rewrite would be read back from the large call's data."""
    import torch
    import speculative_decode_mla_gb300 as m
    small = W.custom_problem([3000, 517, 9000], 9, 13, seed=41, pool_slack=11)
    large = W.make_problem("64k")
    for p, flags in ((small, 0), (large, 0), (small, 0), (small, m.MLA_FLAG_PREFIX_STABLE),
                     (large, m.MLA_FLAG_PREFIX_STABLE)):
        dev = device_problem(p)
        rc, out, lse = _call_noalloc(lib, p, dev, flags)
        assert rc == 0, f"mla_verify_attn_noalloc returned {rc}"
        ref_out, ref_lse = _call_with_workspace(p, dev, flags)
        torch.cuda.synchronize()
        _compare(out, lse, ref_out, ref_lse)
        _assert_bit_identical(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    import torch
    import speculative_decode_mla_gb300 as m
    # 16 sequences of 64 nodes x 64 heads over 131k positions need more than 32 MiB of partials
    desc = m.make_desc(16, 64, 64, 1 << 24, 131072 + 64, 131072)
    assert m.workspace_size(desc) > SCRATCH_BYTES
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    fake = out.data_ptr()
    rc = lib.mla_verify_attn_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake, fake, None,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == -3  # MLA_ERR_WORKSPACE_TOO_SMALL, nothing launched
    torch.cuda.synchronize()
    assert not out.any()
