"""Shared helpers of the GPU parity tests (comparison rule, tensor moves).

Comparison rule for floating point, per element:
    |gpu - oracle| <= abs + rel * max(|oracle|, rms(oracle))
where rms is taken over the compared tensor, so that an element that is
small only because of cancellation is judged against the tensor's scale.
fp32 inputs: rel 1e-5, abs 1e-6.  bf16 inputs: rel 2e-2, abs 0.
Two GPU results compared with each other (each carrying its own rounding
against the exact value) use twice the bound (``pair=True``).
"""
import numpy as np

import synth

TOL = {synth.F32: (1e-5, 1e-6), synth.BF16: (2e-2, 0.0)}


def tol(dtype_code):
    return TOL[dtype_code]


def check_close(gpu, ref, dtype_code, what="", positions_axis=None, pair=False):
    """Assert the comparison rule; on failure report the worst elements and
    the maximum error per position along ``positions_axis``."""
    rel, abs_ = tol(dtype_code)
    if pair:
        rel, abs_ = 2 * rel, 2 * abs_
    g = np.asarray(gpu, np.float64)
    o = np.asarray(ref, np.float64)
    assert g.shape == o.shape, (what, g.shape, o.shape)
    if o.size == 0:
        return
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    scale = np.maximum(np.abs(o), np.sqrt(np.mean(o * o)))
    err = np.abs(g - o)
    bound = abs_ + rel * scale
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        msg = [f"{what}: {bad.sum()} of {o.size} elements out of tolerance (rel {rel}, abs {abs_})"]
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
