"""GPU parity of the batched decode step against the CPU oracle."""
import numpy as np
import pytest

import oracle
import synth
from tests._helpers import check_close, empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 2000


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _pool(m, H, P, N, G, dt_in, dt_dt, n_slots, init, mode=0, W=16, T1=1):
    import torch
    cfg = m.make_config(H, P, N, G, dt_in, dt_dt, mode, W, T1)
    t = torch.from_numpy(np.ascontiguousarray(init, np.float32)).cuda() if init is not None else None
    return m.ssm_state_init(cfg, n_slots, t)


def _step_inputs(seed, step, batch, H, P, G, N, dt_in, dt_dt):
    x, dt, B, C = synth.batch_tokens(seed, step, batch, 1, H, P, G, N, dt_in, dt_dt)
    return x[:, 0], dt[:, 0], B[:, 0], C[:, 0]


@pytest.mark.parametrize("H,P,N,G,dt_in,dt_dt", [
    (2, 16, 16, 1, synth.F32, synth.F32),      # tiny fp32 shape
    (4, 20, 32, 2, synth.F32, synth.F32),      # headdim not a multiple of the warp's rows
    (3, 8, 64, 3, synth.F32, synth.BF16),      # one head per group, bf16 dt
    (8, 64, 128, 4, synth.BF16, synth.F32),    # Mamba-2 head shape, bf16 inputs
    (2, 64, 256, 1, synth.F32, synth.F32),     # widest dstate
])
def test_decode_matches_oracle(H, P, N, G, dt_in, dt_dt):
    import torch
    m = _mod()
    n_slots, slots, steps = 7, [5, 0, 3], 6
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(n_slots)])
    pool = _pool(m, H, P, N, G, dt_in, dt_dt, n_slots, init)
    opool = oracle.OraclePool(H, P, N, G, n_slots, A, D, init_state=init.astype(np.float64))
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    try:
        for s in range(steps):
            x, dt, B, C = _step_inputs(SEED, s, len(slots), H, P, G, N, dt_in, dt_dt)
            y = empty_like_out((len(slots), H, P), dt_in)
            st = m.ssm_decode_step(pool, slots, to_device(x, dt_in), to_device(dt, dt_dt), to_device(B, dt_in),
                                   to_device(C, dt_in), Ad, Dd, y)
            assert st == m.SSM_OK
            _, yo = opool.decode(slots, synth.widen(x, dt_in), synth.widen(dt, dt_dt), synth.widen(B, dt_in),
                                 synth.widen(C, dt_in))
            check_close(to_host(y), yo, dt_in, f"y step {s}", cond=opool.last_cond)
        got = torch.empty((n_slots, H, P, N), dtype=torch.float32, device="cuda")
        assert m.ssm_state_gather(pool, list(range(n_slots)), got) == m.SSM_OK
        check_close(to_host(got), opool.state, dt_in, "state")
        for s in range(n_slots):
            st, meta = m.ssm_slot_info(pool, s)
            assert st == m.SSM_OK and meta.position == (steps if s in slots else 0)
        st, flags = m.ssm_pool_status(pool)
        assert st == m.SSM_OK and flags == 0
        assert m.ssm_last_path(pool) == "decode"
    finally:
        m.ssm_state_destroy(pool)


@pytest.mark.parametrize("dt_in,dt_dt", [(synth.F32, synth.F32), (synth.BF16, synth.F32), (synth.BF16, synth.BF16)])
def test_decode_from_host_buffers_equals_device_path(dt_in, dt_dt):
    """ssm_decode_steps_host over n steps (inputs and outputs in page-locked
    host memory) gives bit for bit the outputs and states of n ssm_decode_step
    calls on the same rows, and follows the oracle; a later call with a larger
    batch regrows the staging; pageable host memory is refused and changes
    nothing."""
    import torch
    m = _mod()
    H, P, N, G, n_slots = 8, 64, 128, 4, 7
    A, D = synth.head_params(SEED + 1, H)
    init = np.stack([synth.init_state(SEED + 1, s, H, P, N) for s in range(n_slots)])
    pd = _pool(m, H, P, N, G, dt_in, dt_dt, n_slots, init)
    ph = _pool(m, H, P, N, G, dt_in, dt_dt, n_slots, init)
    opool = oracle.OraclePool(H, P, N, G, n_slots, A, D, init_state=init.astype(np.float64))
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    side = torch.cuda.Stream()
    try:
        for call, (slots, steps) in enumerate((([5, 0, 3], 5), ([1, 2, 4, 6, 5, 0, 3], 3))):
            R = len(slots)
            rows = [_step_inputs(SEED + 1, 10 * call + t, R, H, P, G, N, dt_in, dt_dt) for t in range(steps)]
            host = [torch.stack([to_device(r[i], code, "cpu") for r in rows]).pin_memory()
                    for i, code in enumerate((dt_in, dt_dt, dt_in, dt_in))]
            y_host = empty_like_out((steps, R, H, P), dt_in, "cpu").pin_memory()
            if call == 1:  # pageable buffers: refused before anything is queued
                st = m.ssm_decode_steps_host(ph, slots, steps, *(h.clone() for h in host), Ad, Dd, y_host.clone())
                assert st == m.SSM_ERR_INVALID_ARG
            with torch.cuda.stream(side):
                st = m.ssm_decode_steps_host(ph, slots, steps, *host, Ad, Dd, y_host, stream=side)
            assert st == m.SSM_OK
            side.synchronize()
            for t, (x, dt, B, C) in enumerate(rows):
                y = empty_like_out((R, H, P), dt_in)
                assert m.ssm_decode_step(pd, slots, to_device(x, dt_in), to_device(dt, dt_dt), to_device(B, dt_in),
                                         to_device(C, dt_in), Ad, Dd, y) == m.SSM_OK
                assert torch.equal(y.cpu(), y_host[t]), f"call {call} step {t}: host path differs"
                _, yo = opool.decode(slots, synth.widen(x, dt_in), synth.widen(dt, dt_dt), synth.widen(B, dt_in),
                                     synth.widen(C, dt_in))
                check_close(to_host(y_host[t]), yo, dt_in, f"host path y call {call} step {t}", cond=opool.last_cond)
        gd = torch.empty((n_slots, H, P, N), device="cuda")
        gh = torch.empty_like(gd)
        assert m.ssm_state_gather(pd, list(range(n_slots)), gd) == m.SSM_OK
        assert m.ssm_state_gather(ph, list(range(n_slots)), gh) == m.SSM_OK
        assert torch.equal(gd, gh)
        for s in range(n_slots):
            assert m.ssm_slot_info(ph, s)[1].position == m.ssm_slot_info(pd, s)[1].position
        assert m.ssm_pool_status(ph) == (m.SSM_OK, 0)
    finally:
        m.ssm_state_destroy(pd)
        m.ssm_state_destroy(ph)


def test_decode_nemotron_shape_full_batch_sampled():
    """Batched decode, Nemotron-shaped (H=128, P=64, N=128, G=8), batch 256,
    64 successive steps, bf16 x/B/C, fp32 dt and N(0, 0.1) fp32 state; the
    oracle follows three requests (all heads) through all 64 steps."""
    import torch
    m = _mod()
    H, P, N, G, R, steps = 128, 64, 128, 8, 256, 64
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)])
    pool = _pool(m, H, P, N, G, synth.BF16, synth.F32, R, init)
    sample = [0, 97, 255]
    ost = init[sample].astype(np.float64)
    del init
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    slots = list(range(R))
    try:
        for s in range(steps):
            x, dt, B, C = _step_inputs(SEED, s, R, H, P, G, N, synth.BF16, synth.F32)
            y = empty_like_out((R, H, P), synth.BF16)
            st = m.ssm_decode_step(pool, slots, to_device(x, synth.BF16), to_device(dt, synth.F32),
                                   to_device(B, synth.BF16), to_device(C, synth.BF16), Ad, Dd, y)
            assert st == m.SSM_OK
            yo, yc = oracle.decode_step(ost, synth.widen(x[sample], synth.BF16), synth.widen(dt[sample], synth.F32),
                                        synth.widen(B[sample], synth.BF16), synth.widen(C[sample], synth.BF16), A, D,
                                        want_cond=True)
            check_close(to_host(y[sample]), yo, synth.BF16, f"y step {s}", cond=yc)
        got = torch.empty((len(sample), H, P, N), dtype=torch.float32, device="cuda")
        assert m.ssm_state_gather(pool, sample, got) == m.SSM_OK
        check_close(to_host(got), ost, synth.BF16, "state after 64 steps")
        # fp32 state arithmetic: far inside the bf16 bound
        err = np.abs(to_host(got) - ost).max() / np.abs(ost).max()
        assert err < 1e-5, err
        st, meta = m.ssm_slot_info(pool, 255)
        assert meta.position == steps
    finally:
        m.ssm_state_destroy(pool)
