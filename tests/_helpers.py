"""Shared test helpers: move seeded problems to the device, run the library, compare with the oracle."""
import numpy as np

TOL_MAX_ABS = 1e-2     # GPU vs oracle, per element of out
TOL_REL_L2 = 5e-3      # GPU vs oracle, relative L2 over the whole out tensor
TOL_LSE_ABS = 1e-3     # lse, natural log


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.view(dtype)


def bf16_dev(bits):
    import torch
    return to_dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def device_problem(p):
    """(q, kv, slot_table, seq_lens, tree_parent) as CUDA tensors."""
    return (bf16_dev(p.q), bf16_dev(p.kv), to_dev(p.slot_table), to_dev(p.seq_lens), to_dev(p.tree_parent))


def run(p, flags=None, dev=None, **kw):
    import speculative_decode_mla_gb300 as m
    import torch
    q, kv, st, sl, tp = dev if dev is not None else device_problem(p)
    out, lse = m.verify(q, kv, st, sl, tp, max_seq_len=kw.pop("max_seq_len", p.max_seq_len), flags=flags, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().reshape(p.rows, 512).astype(np.float64), lse.cpu().numpy().reshape(-1)


def errors(got_o, got_l, ref_o, ref_l):
    err = float(np.abs(got_o - ref_o).max())
    rel = float(np.linalg.norm(got_o - ref_o) / max(np.linalg.norm(ref_o), 1e-300))
    lerr = float(np.abs(got_l - ref_l).max())
    return err, rel, lerr


def assert_close(got_o, got_l, ref_o, ref_l, what=""):
    err, rel, lerr = errors(got_o, got_l, ref_o, ref_l)
    assert err <= TOL_MAX_ABS and rel <= TOL_REL_L2 and lerr <= TOL_LSE_ABS, \
        f"{what}: max_abs={err:.3e} rel_l2={rel:.3e} lse_abs={lerr:.3e}"
    return err, rel, lerr
