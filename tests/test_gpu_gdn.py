"""Gated delta rule on the GPU against the fp64 oracle (Why Speculative
Decoding Slows Hybrid Mamba Models, When the layer is a different kind of
recurrence: Gated DeltaNet unrolls as a decay plus a sum, so the same replay
applies).  In-place decode, replay verify from checkpoint + log, commit with
appends and folds, the error paths, and sampled requests at the benchmark's
size.  Tolerances as for the Mamba-2 path: fp32 inputs rel 1e-5 / abs 1e-6,
bf16 inputs rel 2e-2."""
import numpy as np
import pytest

import synth
from oracle import gdn as og
from tests._helpers import check_close, to_device, to_host

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 8100


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _wide(parts, dt_in):
    codes = (dt_in, dt_in, dt_in, synth.F32, synth.F32)
    return tuple(synth.widen(a, c) for a, c in zip(parts, codes))


def _dev(parts, dt_in):
    codes = (dt_in, dt_in, dt_in, synth.F32, synth.F32)
    return tuple(to_device(a, c) for a, c in zip(parts, codes))


def _out(shape, dt_in):
    import torch
    return torch.empty(shape, dtype=torch.bfloat16 if dt_in == synth.BF16 else torch.float32, device="cuda")


def _pools(m, H, G, dk, dv, dt_in, n_slots, W, T1):
    import torch
    init = np.stack([synth.gdn_init_state(SEED, s, H, dv, dk) for s in range(n_slots)])
    pool = m.ssm_gdn_init(m.make_gdn_config(H, G, dk, dv, dt_in, W, T1), n_slots, torch.from_numpy(init).cuda())
    opool = og.GdnOraclePool(H, G, dk, dv, n_slots, W=W, max_tokens=T1, init_state=init.astype(np.float64))
    return pool, opool


def _states(m, pool, slots):
    import torch
    got = torch.empty((len(slots), pool.H, pool.dv, pool.dk), dtype=torch.float32, device="cuda")
    assert m.ssm_gdn_gather(pool, slots, got) == m.SSM_OK
    return to_host(got)


@pytest.mark.parametrize("dt_in,H,G,dk,dv", [
    (synth.F32, 4, 2, 64, 36),
    (synth.F32, 2, 1, 128, 128),
    (synth.BF16, 8, 4, 128, 128),
    (synth.BF16, 4, 4, 64, 64),
])
def test_decode_matches_oracle(dt_in, H, G, dk, dv):
    m = _mod()
    slots = [6, 1, 3, 0]
    pool, opool = _pools(m, H, G, dk, dv, dt_in, 8, 8, 4)
    try:
        for s in range(6):
            parts = synth.gdn_batch_tokens(SEED, s, len(slots), 1, H, G, dk, dv, dt_in)
            one = tuple(a[:, 0] for a in parts)
            y = _out((len(slots), H, dv), dt_in)
            assert m.ssm_gdn_decode_step(pool, slots, *_dev(one, dt_in), y) == m.SSM_OK
            yo = opool.decode(slots, *_wide(one, dt_in))
            check_close(to_host(y), yo, dt_in, f"y step {s}", cond=opool.last_cond)
        check_close(_states(m, pool, slots), opool.state[slots], dt_in, "states")
        for sl in slots:
            st, pos, ll, fl = m.ssm_gdn_slot_info(pool, sl)
            assert (st, pos, ll, fl) == (m.SSM_OK, 6, 0, 0)
        assert m.ssm_gdn_status(pool)[1] == 0
    finally:
        m.ssm_gdn_destroy(pool)


def _run_verify(m, dt_in, H, G, dk, dv, W, T1, p, steps, slots, n_slots=8, force_at=()):
    import torch
    pool, opool = _pools(m, H, G, dk, dv, dt_in, n_slots, W, T1)
    acc = synth.accept_counts(SEED + 1, steps, len(slots), T1 - 1, p)
    folds = 0
    for s in range(steps):
        parts = synth.gdn_batch_tokens(SEED, 100 + s, len(slots), T1, H, G, dk, dv, dt_in)
        y = _out((len(slots), T1, H, dv), dt_in)
        assert m.ssm_gdn_verify_replay(pool, slots, T1, *_dev(parts, dt_in), y) == m.SSM_OK
        # bf16 pools with 128 x 128 heads take the checkpoint product on the tensor cores
        tc = dt_in == synth.BF16 and dk == 128 and dv == 128 and 4 <= T1 <= 32
        assert m.ssm_gdn_last_path(pool) == ("gdn_verify_tc" if tc else "gdn_verify")
        yo = opool.verify(slots, *_wide(parts, dt_in))
        check_close(to_host(y), yo, dt_in, f"y step {s}", positions_axis=1, cond=opool.last_cond)
        a = torch.from_numpy(np.ascontiguousarray(acc[s], dtype=np.int32)).cuda()
        ff = s in force_at
        assert m.ssm_gdn_commit(pool, slots, a, ff) == m.SSM_OK
        # bf16 pools with 128 x 128 heads and logs of at most 32 tokens fold on the tensor cores
        fold_tc = dt_in == synth.BF16 and dk == 128 and dv == 128 and W - 1 + T1 <= 32
        assert m.ssm_gdn_last_commit_path(pool) == ("gdn_fold_tc" if fold_tc else "gdn_fold")
        folds += len(opool.commit(slots, acc[s], force_fold=ff))
        for sl in slots:
            st, pos, ll, fl = m.ssm_gdn_slot_info(pool, sl)
            assert st == m.SSM_OK and ll == opool.log_len(sl) and pos == opool.position[sl] and fl == 0, (s, sl)
    return pool, opool, folds


@pytest.mark.parametrize("dt_in,H,G,dk,dv,W,T1,p", [
    (synth.F32, 4, 2, 64, 36, 8, 4, 0.7),
    (synth.F32, 2, 2, 128, 64, 16, 9, 0.8),
    (synth.BF16, 8, 4, 128, 128, 16, 9, 0.8),
    (synth.BF16, 4, 2, 128, 128, 8, 5, 0.6),
    (synth.BF16, 4, 1, 64, 128, 32, 17, 0.9),
    (synth.F32, 4, 2, 128, 128, 8, 5, 0.7),
    (synth.BF16, 2, 1, 128, 128, 32, 17, 0.9),
    (synth.BF16, 4, 2, 128, 128, 16, 17, 0.95),
])
def test_replay_verify_and_commit_match_oracle(dt_in, H, G, dk, dv, W, T1, p):
    m = _mod()
    slots = [5, 0, 7, 2, 3]
    pool, opool, folds = _run_verify(m, dt_in, H, G, dk, dv, W, T1, p, steps=8, slots=slots, force_at=(5,))
    try:
        assert folds > 0
        # a forced fold applies every log: the checkpoints then hold the full states
        import torch
        assert m.ssm_gdn_verify_replay(pool, slots, 1, *_dev(synth.gdn_batch_tokens(SEED, 999, len(slots), 1, H, G,
                                                                                        dk, dv, dt_in), dt_in),
                                       _out((len(slots), 1, H, dv), dt_in)) == m.SSM_OK
        opool.verify(slots, *_wide(synth.gdn_batch_tokens(SEED, 999, len(slots), 1, H, G, dk, dv, dt_in), dt_in))
        zero = torch.zeros(len(slots), dtype=torch.int32, device="cuda")
        assert m.ssm_gdn_commit(pool, slots, zero, True) == m.SSM_OK
        opool.commit(slots, np.zeros(len(slots), np.int32), force_fold=True)
        check_close(_states(m, pool, slots), opool.state[slots], dt_in, "states after a forced fold")
        assert m.ssm_gdn_status(pool)[1] == 0
    finally:
        m.ssm_gdn_destroy(pool)


def test_replay_pool_used_for_decode_agrees_with_decode():
    """One token a step through verify + commit (window 16) against decode in place."""
    import torch
    m = _mod()
    H, G, dk, dv, dt_in = 4, 2, 128, 128, synth.F32
    slots = [1, 4, 2]
    rp, _ = _pools(m, H, G, dk, dv, dt_in, 6, 16, 1)
    dp, _ = _pools(m, H, G, dk, dv, dt_in, 6, 16, 1)
    zero = torch.zeros(len(slots), dtype=torch.int32, device="cuda")
    try:
        for s in range(20):
            parts = synth.gdn_batch_tokens(SEED, 300 + s, len(slots), 1, H, G, dk, dv, dt_in)
            yr = _out((len(slots), 1, H, dv), dt_in)
            yd = _out((len(slots), H, dv), dt_in)
            assert m.ssm_gdn_verify_replay(rp, slots, 1, *_dev(parts, dt_in), yr) == m.SSM_OK
            assert m.ssm_gdn_commit(rp, slots, zero) == m.SSM_OK
            assert m.ssm_gdn_decode_step(dp, slots, *_dev(tuple(a[:, 0] for a in parts), dt_in), yd) == m.SSM_OK
            check_close(to_host(yr)[:, 0], to_host(yd), dt_in, f"step {s}", pair=True)
        assert m.ssm_gdn_slot_info(rp, 1)[2] == 20 % 16  # one fold at the 16th token
    finally:
        m.ssm_gdn_destroy(rp)
        m.ssm_gdn_destroy(dp)


@pytest.mark.parametrize("which,dk,dv", [(w, 64, 64) for w in ("q", "k", "v", "g", "beta")] +
                         [("k", 128, 128), ("beta", 128, 128)])
def test_nonfinite_input_poisons_only_its_request(which, dk, dv):
    """dk = dv = 128 (bf16) runs the tensor-core streaming kernel, whose gate drops the poisoned request."""
    import torch
    m = _mod()
    H, G, dt_in, T1 = 4, 2, synth.BF16, (4 if dk == 128 else 3)
    slots = [0, 1, 2]
    pool, opool = _pools(m, H, G, dk, dv, dt_in, 4, 8, T1)
    try:
        parts = list(synth.gdn_batch_tokens(SEED, 400, 3, T1, H, G, dk, dv, dt_in))
        idx = ("q", "k", "v", "g", "beta").index(which)
        bad = parts[idx].copy()
        bad[1, 1].flat[0] = 0x7FC0 if bad.dtype == np.uint16 else np.nan
        parts[idx] = bad
        y = _out((3, T1, H, dv), dt_in)
        assert m.ssm_gdn_verify_replay(pool, slots, T1, *_dev(tuple(parts), dt_in), y) == m.SSM_OK
        assert m.ssm_gdn_last_path(pool) == ("gdn_verify_tc" if dk == 128 else "gdn_verify")
        st, flags = m.ssm_gdn_status(pool, clear=True)
        assert flags & m.SSM_FLAG_NONFINITE_INPUT
        assert m.ssm_gdn_slot_info(pool, 1)[3] & 1 and m.ssm_gdn_slot_info(pool, 0)[3] == 0
        good = [0, 2]
        yo = opool.verify(good, *(a[good] for a in _wide(tuple(parts), dt_in)))
        check_close(to_host(y[good]), yo, dt_in, "the other requests", cond=opool.last_cond)
        assert m.ssm_gdn_commit(pool, slots, torch.zeros(3, dtype=torch.int32, device="cuda")) == m.SSM_OK
        assert m.ssm_gdn_slot_info(pool, 1)[1] == 0 and m.ssm_gdn_slot_info(pool, 0)[1] == 1
        assert m.ssm_gdn_reset(pool, [1]) == m.SSM_OK
        assert m.ssm_gdn_slot_info(pool, 1)[1:] == (0, 0, 0)
        assert not _states(m, pool, [1]).any()
    finally:
        m.ssm_gdn_destroy(pool)


def test_bad_accept_and_misuse():
    import torch
    m = _mod()
    H, G, dk, dv, dt_in, T1 = 2, 1, 64, 64, synth.F32, 3
    pool, _ = _pools(m, H, G, dk, dv, dt_in, 4, 8, T1)
    try:
        parts = _dev(synth.gdn_batch_tokens(SEED, 500, 2, T1, H, G, dk, dv, dt_in), dt_in)
        y = _out((2, T1, H, dv), dt_in)
        # commit before any verify, duplicate slots, too many tokens: refused on the host
        acc = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
        assert m.ssm_gdn_commit(pool, [0, 1], acc) == m.SSM_ERR_INVALID_STATE
        assert m.ssm_gdn_verify_replay(pool, [0, 0], T1, *parts, y) == m.SSM_ERR_INVALID_ARG
        assert m.ssm_gdn_verify_replay(pool, [0, 1], T1, *parts, y) == m.SSM_OK
        assert m.ssm_gdn_commit(pool, [0, 1], acc) == m.SSM_OK      # accept 5 > n_tok - 1
        st, flags = m.ssm_gdn_status(pool)
        assert flags & m.SSM_FLAG_BAD_ACCEPT
        assert m.ssm_gdn_slot_info(pool, 1)[3] & 1 and m.ssm_gdn_slot_info(pool, 0)[1] == 1
    finally:
        m.ssm_gdn_destroy(pool)


def test_full_size_sampled_requests():
    """Replay verify + commit at the benchmark's shape (256 requests, 32 value
    heads, 16 key heads, 128 x 128, bf16, window 16, 8 drafts) on the
    tensor-core streaming kernel; sampled requests checked against the oracle
    step by step."""
    import torch
    m = _mod()
    H, G, dk, dv, dt_in, W, T1, R = 32, 16, 128, 128, synth.BF16, 16, 9, 256
    sample = [0, 17, 142, 255]
    init = np.stack([synth.gdn_init_state(SEED, s, H, dv, dk) for s in range(R)])
    pool = m.ssm_gdn_init(m.make_gdn_config(H, G, dk, dv, dt_in, W, T1), R, torch.from_numpy(init).cuda())
    opool = og.GdnOraclePool(H, G, dk, dv, len(sample), W=W, max_tokens=T1, init_state=init[sample].astype(np.float64))
    acc = synth.accept_counts(SEED + 2, 6, R, T1 - 1, 0.8)
    try:
        slots = list(range(R))
        for s in range(6):
            parts = synth.gdn_batch_tokens(SEED, 600 + s, R, T1, H, G, dk, dv, dt_in)
            y = _out((R, T1, H, dv), dt_in)
            assert m.ssm_gdn_verify_replay(pool, slots, T1, *_dev(parts, dt_in), y) == m.SSM_OK
            assert m.ssm_gdn_last_path(pool) == "gdn_verify_tc"
            yo = opool.verify(list(range(len(sample))), *(a[sample] for a in _wide(parts, dt_in)))
            check_close(to_host(y)[sample], yo, dt_in, f"sampled y step {s}", positions_axis=1, cond=opool.last_cond)
            assert m.ssm_gdn_commit(pool, slots, torch.from_numpy(acc[s]).cuda()) == m.SSM_OK
            assert m.ssm_gdn_last_commit_path(pool) == "gdn_fold_tc"
            opool.commit(list(range(len(sample))), acc[s][sample])
        assert m.ssm_gdn_status(pool)[1] == 0
        check_close(_states(m, pool, sample), opool.state, dt_in, "sampled checkpoints")
    finally:
        m.ssm_gdn_destroy(pool)
