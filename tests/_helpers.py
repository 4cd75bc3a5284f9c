"""Shared helpers of the GPU parity tests (comparison rule, tensor moves).

Comparison rule for floating point, per element:
    |gpu - oracle| <= abs + rel * scale
    outputs y:  scale = max(|oracle|, cond), cond = sum_n |C_n h_n| + |D x|
                (the oracle's condition scale: the size of the terms whose
                sum is y, so that cancellation in that sum does not fake a
                failure; for the gated delta rule sum_k |S_pk q_k|)
    states:     scale = |oracle|
fp32 inputs: rel 1e-5, abs 1e-6.  bf16 inputs: rel 2e-2, and an abs floor of
1e-2 * rms(oracle) over the compared tensor.  Two GPU results compared with
each other (each carrying its own rounding against the exact value) use
twice the bound (``pair=True``).
"""
import numpy as np

import synth

REL = {synth.F32: 1e-5, synth.BF16: 2e-2}
ABS_F32 = 1e-6
ABS_BF16_RMS = 1e-2


def tol(dtype_code):
    return REL[dtype_code]


def check_close(gpu, ref, dtype_code, what="", positions_axis=None, pair=False, cond=None):
    """Assert the comparison rule (``cond`` given: an output, else a state);
    on failure report the worst elements and the maximum error per position
    along ``positions_axis``."""
    rel = REL[dtype_code]
    g = np.asarray(gpu, np.float64)
    o = np.asarray(ref, np.float64)
    assert g.shape == o.shape, (what, g.shape, o.shape)
    if o.size == 0:
        return
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    abs_ = ABS_BF16_RMS * np.sqrt(np.mean(o * o)) if dtype_code == synth.BF16 else ABS_F32
    if pair:
        rel, abs_ = 2 * rel, 2 * abs_
    if cond is not None:
        c = np.asarray(cond, np.float64)
        assert c.shape == o.shape, (what, "cond", c.shape, o.shape)
        scale = np.maximum(np.abs(o), c)
    else:
        scale = np.abs(o)
    err = np.abs(g - o)
    bound = abs_ + rel * scale
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = [f"{what}: {bad.sum()} of {o.size} elements out of tolerance (rel {rel}, abs {abs_:.3e}, "
               f"{'condition scale' if cond is not None else 'element'} scale)"]
        for i in idx:
            t = tuple(int(v) for v in i)
            msg.append(f"  at {t}: gpu {g[t]!r} oracle {o[t]!r} err {err[t]:.3e} bound {bound[t]:.3e}")
        if positions_axis is not None:
            ax = tuple(a for a in range(o.ndim) if a != positions_axis)
            per = (err / np.maximum(bound, 1e-300)).max(axis=ax)
            msg.append(f"  worst err/bound by position: {np.array2string(per[:64], precision=2)}")
        raise AssertionError("\n".join(msg))


def to_device(a, dtype_code, device="cuda"):
    """numpy input (fp32, or uint16 bf16 patterns) -> torch tensor on the GPU."""
    import torch
    if dtype_code == synth.BF16:
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device)


def to_host(t):
    """GPU tensor (fp32 or bf16) -> fp64 numpy."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def empty_like_out(shape, dtype_code, device="cuda"):
    import torch
    return torch.empty(shape, dtype=torch.bfloat16 if dtype_code == synth.BF16 else torch.float32, device=device)
