"""Checkpoint / restore and the slot lifecycle on the GPU (Mamba Streaming
State That Survives Chunking, Make reset, checkpoint, and cancellation
observable; SSM.PREFIX recurrent-state companion, Validation: a restored
state continues bit for bit like the uninterrupted stream)."""
import numpy as np
import pytest

import synth
from tests._helpers import empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 5000


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _decode(m, pool, slots, s, H, P, G, N, A, D, dt_in=synth.BF16):
    x, dt, B, C = synth.batch_tokens(SEED, s, len(slots), 1, H, P, G, N, dt_in, synth.F32)
    y = empty_like_out((len(slots), H, P), dt_in)
    st = m.ssm_decode_step(pool, slots, to_device(x[:, 0], dt_in), to_device(dt[:, 0], synth.F32),
                           to_device(B[:, 0], dt_in), to_device(C[:, 0], dt_in), A, D, y)
    assert st == m.SSM_OK
    return to_host(y)


@pytest.mark.parametrize("mode", [0, 1])
def test_checkpoint_restore_is_bit_exact(mode):
    """Decode 40 tokens, checkpoint, restore into another slot, decode 40 more
    on both: outputs and states identical (max-abs-diff 0)."""
    import torch
    m = _mod()
    H, P, N, G = 8, 64, 128, 2
    A, D = synth.head_params(SEED, H)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    pool = m.ssm_state_init(m.make_config(H, P, N, G, synth.BF16, synth.F32, mode, 8, 1), 4)
    try:
        for s in range(40):
            _decode(m, pool, [0], s, H, P, G, N, Ad, Dd)
        st, host, meta = m.ssm_state_checkpoint(pool, 0, Ad)
        assert st == m.SSM_OK and meta.position == 40 and meta.log_len == 0
        assert m.ssm_state_restore(pool, 2, host, meta) == m.SSM_OK
        _, meta2 = m.ssm_slot_info(pool, 2)
        assert meta2.position == 40 and meta2.next_chunk == meta.next_chunk and meta2.epoch == meta.epoch
        for s in range(40, 80):
            y0 = _decode(m, pool, [0], s, H, P, G, N, Ad, Dd)
            y2 = _decode(m, pool, [2], s, H, P, G, N, Ad, Dd)
            assert np.array_equal(y0, y2)
        got = torch.empty((2, H, P, N), dtype=torch.float32, device="cuda")
        m.ssm_state_gather(pool, [0, 2], got)
        g = to_host(got)
        assert np.array_equal(g[0], g[1])
        # a state of the wrong size is refused, not padded or truncated
        assert m.ssm_state_restore(pool, 3, host[:, :, :64], meta) == m.SSM_ERR_SCHEMA
    finally:
        m.ssm_state_destroy(pool)


def test_replay_pool_refuses_in_place_update_with_pending_log():
    import torch
    m = _mod()
    H, P, N, G = 2, 16, 16, 1
    A, D = synth.head_params(SEED, H)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    pool = m.ssm_state_init(m.make_config(H, P, N, G, synth.F32, synth.F32, 1, 8, 3), 2)
    try:
        x, dt, B, C = synth.batch_tokens(SEED, 0, 1, 3, H, P, G, N)
        y = empty_like_out((1, 3, H, P), synth.F32)
        assert m.ssm_verify_replay(pool, [0], 3, to_device(x, 0), to_device(dt, 0), to_device(B, 0),
                                   to_device(C, 0), Ad, Dd, y) == m.SSM_OK
        acc = torch.tensor([1], dtype=torch.int32, device="cuda")
        assert m.ssm_state_commit(pool, [0], acc, False, Ad) == m.SSM_OK
        assert m.ssm_slot_info(pool, 0)[1].log_len == 2
        _decode(m, pool, [0], 5, H, P, G, N, Ad, Dd, dt_in=synth.F32)   # refused on the device
        st, flags = m.ssm_pool_status(pool, clear=True)
        assert flags & m.SSM_FLAG_LOG_NOT_EMPTY
        assert m.ssm_slot_info(pool, 0)[1].flags & 1
        # checkpoint of a poisoned slot is refused; reset brings it back
        assert m.ssm_state_checkpoint(pool, 0, Ad)[0] == m.SSM_ERR_INVALID_STATE
        assert m.ssm_state_reset(pool, [0]) == m.SSM_OK
        _decode(m, pool, [0], 6, H, P, G, N, Ad, Dd, dt_in=synth.F32)
        assert m.ssm_pool_status(pool)[1] == 0
        assert m.ssm_slot_info(pool, 0)[1].position == 1
    finally:
        m.ssm_state_destroy(pool)


def test_pool_memory_accounting():
    m = _mod()
    H, P, N, G, S = 128, 64, 128, 8, 4
    pc = m.ssm_state_init(m.make_config(H, P, N, G, synth.BF16, synth.F32, 0, 16, 9), S)
    pr = m.ssm_state_init(m.make_config(H, P, N, G, synth.BF16, synth.F32, 1, 16, 9), S)
    try:
        state = S * H * P * N * 4
        assert m.ssm_pool_bytes(pc) >= state * (1 + 2 * 9)        # base + double-buffered snapshots
        log_entry = H * P * 2 + H * 4 + G * N * 2                  # x, dt, B of one token
        logs = S * (16 - 1 + 9) * log_entry
        staging = H * P * N * 4                                    # one slot, for checkpoints
        cb_w = -(-(16 - 1 + 9) // 4) * 4
        scratch = S * (9 * G * cb_w + 9 * H * cb_w + 12 * H + 9 * G * N) * 4  # per request: C.B, W, decay, C
        assert state + logs <= m.ssm_pool_bytes(pr) <= state + logs + staging + scratch + (1 << 20)
    finally:
        m.ssm_state_destroy(pc)
        m.ssm_state_destroy(pr)
