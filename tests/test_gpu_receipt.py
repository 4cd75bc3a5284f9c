"""Checkpoint receipt on the GPU: a slot checkpointed as receipt + blob and
restored elsewhere continues exactly as the uninterrupted slot does (bit for
bit: the recurrence is deterministic), and every incompatible resume is
refused with the slot untouched (Mamba Streaming State That Survives
Chunking, Make reset, checkpoint, and cancellation observable; the
SSM.PREFIX state-store page, Validation: state hydration with zero drift)."""
import numpy as np
import pytest

import synth
from tests._helpers import empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 7000


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _pool(m, H, P, N, G, dt_in, mode, n_slots, W=8, T1=5):
    import torch
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(n_slots)])
    cfg = m.make_config(H, P, N, G, dt_in, synth.F32, mode, W, T1)
    return m.ssm_state_init(cfg, n_slots, torch.from_numpy(init).cuda())


def _states(m, pool, slots, H, P, N):
    import torch
    got = torch.empty((len(slots), H, P, N), dtype=torch.float32, device="cuda")
    assert m.ssm_state_gather(pool, slots, got) == m.SSM_OK
    return to_host(got)


def _decode(m, pool, slots, step, H, P, N, G, dt_in, A, D):
    x, dt, B, C = synth.batch_tokens(SEED, step, 1, 1, H, P, G, N, dt_in, synth.F32)
    # the same token for every slot named
    rep = lambda a: np.repeat(a[:, 0], len(slots), axis=0)
    y = empty_like_out((len(slots), H, P), dt_in)
    assert m.ssm_decode_step(pool, slots, to_device(rep(x), dt_in), to_device(rep(dt), synth.F32),
                             to_device(rep(B), dt_in), to_device(rep(C), dt_in), A, D, y) == m.SSM_OK
    return to_host(y)


def _verify_commit(m, pool, slots, step, T1, H, P, N, G, dt_in, A, D, acc):
    import torch
    x, dt, B, C = synth.batch_tokens(SEED, 100 + step, 1, T1, H, P, G, N, dt_in, synth.F32)
    rep = lambda a: np.repeat(a, len(slots), axis=0)
    y = empty_like_out((len(slots), T1, H, P), dt_in)
    assert m.ssm_verify_replay(pool, slots, T1, to_device(rep(x), dt_in), to_device(rep(dt), synth.F32),
                               to_device(rep(B), dt_in), to_device(rep(C), dt_in), A, D, y) == m.SSM_OK
    a = torch.full((len(slots),), acc, dtype=torch.int32, device="cuda")
    assert m.ssm_state_commit(pool, slots, a, False, A) == m.SSM_OK
    return to_host(y)


@pytest.mark.parametrize("mode,dt_in,shape", [
    (0, synth.F32, (4, 16, 32, 2)),       # copy pool, decode in place
    (1, synth.BF16, (4, 64, 128, 2)),     # replay pool: verify + commit (tensor-core paths)
])
def test_hydration_is_bit_exact(mode, dt_in, shape):
    import torch
    m = _mod()
    H, P, N, G = shape
    A, D = synth.head_params(SEED, H)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    T1 = 5
    pool = _pool(m, H, P, N, G, dt_in, mode, 4, T1=T1)
    other = _pool(m, H, P, N, G, dt_in, mode, 2, T1=T1)
    ident = m.stream_identity(0xABCDEF, 3, 9, 7)
    try:
        step = (lambda p, sl, s: _decode(m, p, sl, s, H, P, N, G, dt_in, Ad, Dd)) if mode == 0 else \
               (lambda p, sl, s: _verify_commit(m, p, sl, s, T1, H, P, N, G, dt_in, Ad, Dd, 2))
        for s in range(5):
            step(pool, [0], s)
        before = m.ssm_slot_info(pool, 0)[1]
        st, blob = m.ssm_state_checkpoint_receipt(pool, 0, ident, Ad)
        assert st == m.SSM_OK and len(blob) == m.ssm_receipt_bytes(H, P, N)
        st, r, _ = m.ssm_receipt_decode(blob)
        assert st == m.SSM_OK and r.position == before.position and r.next_chunk == before.next_chunk
        assert (r.nheads, r.headdim, r.dstate, r.ngroups, r.input_dtype) == (H, P, N, G, dt_in)
        epoch1 = m.ssm_slot_info(pool, 1)[1].epoch
        assert m.ssm_state_restore_receipt(pool, 1, blob, ident) == m.SSM_OK
        assert m.ssm_state_restore_receipt(other, 0, blob, ident) == m.SSM_OK
        meta1 = m.ssm_slot_info(pool, 1)[1]
        assert meta1.position == before.position and meta1.next_chunk == before.next_chunk
        assert meta1.epoch == epoch1 + 1 and meta1.log_len == 0 and meta1.flags == 0
        s0 = _states(m, pool, [0, 1], H, P, N)
        assert np.array_equal(s0[0], s0[1])
        # continue the original and both restored copies with the same tokens
        for s in range(5, 12):
            ya = step(pool, [0, 1], s)
            yb = step(other, [0], s)
            assert np.array_equal(ya[0], ya[1]) and np.array_equal(ya[0], yb[0]), s
        sa = _states(m, pool, [0, 1], H, P, N)
        sb = _states(m, other, [0], H, P, N)
        assert np.abs(sa[0] - sa[1]).max() == 0.0 and np.abs(sa[0] - sb[0]).max() == 0.0
        assert m.ssm_pool_status(pool)[1] == 0 and m.ssm_pool_status(other)[1] == 0
    finally:
        m.ssm_state_destroy(pool)
        m.ssm_state_destroy(other)


def test_incompatible_resume_is_refused():
    import torch
    m = _mod()
    H, P, N, G = 4, 16, 32, 2
    A, D = synth.head_params(SEED, H)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    pool = _pool(m, H, P, N, G, synth.F32, 0, 3)
    pools = [_pool(m, H + 2, P, N, G, synth.F32, 0, 1),      # other dimensions
             _pool(m, H, P, N, G + 2, synth.F32, 0, 1),      # other group count
             _pool(m, H, P, N, G, synth.BF16, 0, 1)]         # other input precision
    ident = m.stream_identity(41, 42, 43, 3)
    try:
        for s in range(3):
            _decode(m, pool, [0], s, H, P, N, G, synth.F32, Ad, Dd)
        st, blob = m.ssm_state_checkpoint_receipt(pool, 0, ident, Ad)
        assert st == m.SSM_OK
        keep = _states(m, pool, [2], H, P, N)
        meta_keep = m.ssm_slot_info(pool, 2)[1]
        wrong = [m.stream_identity(40, 42, 43, 3), m.stream_identity(41, 41, 43, 3),
                 m.stream_identity(41, 42, 44, 3), m.stream_identity(41, 42, 43, 4)]
        for w in wrong:
            assert m.ssm_state_restore_receipt(pool, 2, blob, w) == m.SSM_ERR_SCHEMA
        bad = bytearray(blob)
        bad[-1] ^= 1
        assert m.ssm_state_restore_receipt(pool, 2, bytes(bad), ident) == m.SSM_ERR_SCHEMA
        assert m.ssm_state_restore_receipt(pool, 2, blob[:-4], ident) == m.SSM_ERR_SCHEMA
        assert np.array_equal(_states(m, pool, [2], H, P, N), keep)            # nothing changed
        meta = m.ssm_slot_info(pool, 2)[1]
        assert (meta.position, meta.next_chunk, meta.epoch) == \
            (meta_keep.position, meta_keep.next_chunk, meta_keep.epoch)
        for q in pools:
            assert m.ssm_state_restore_receipt(q, 0, blob, ident) == m.SSM_ERR_SCHEMA
        assert m.ssm_state_restore_receipt(pool, 2, blob, ident) == m.SSM_OK  # the right one is taken
    finally:
        m.ssm_state_destroy(pool)
        for q in pools:
            m.ssm_state_destroy(q)
