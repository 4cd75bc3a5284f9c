"""GPU parity of replay pools that fold a full log in the next verify
(SSM_FOLD_IN_VERIFY) against the oracle's fold-in-verify rule: outputs,
checkpoints, log lengths and positions, the moves of kept tokens at the
commit (overlapping ones included), a forced fold, a checkpoint read and a
second verify between a verify and its commit, a poisoned request with a
full log, and the speculative-verify workload at batch 512."""
import numpy as np
import pytest

import oracle
import synth
from tests._helpers import check_close, empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 3500
BF, F32 = synth.BF16, synth.F32


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _dev(x, dt, B, C):
    return to_device(x, BF), to_device(dt, F32), to_device(B, BF), to_device(C, BF)


def _wide(x, dt, B, C):
    return synth.widen(x, BF), synth.widen(dt, F32), synth.widen(B, BF), synth.widen(C, BF)


def _pools(m, H, P, N, G, R, W, T1, init):
    import torch
    init_t = torch.from_numpy(np.ascontiguousarray(init, np.float32)).cuda()
    cfg = m.make_config(H, P, N, G, BF, F32, m.SSM_MODE_REPLAY, W, T1, fold=m.SSM_FOLD_IN_VERIFY)
    pool = m.ssm_state_init(cfg, R, init_t)
    return pool


def _log_lens(m, pool, R):
    return np.array([m.ssm_slot_info(pool, s)[1].log_len for s in range(R)])


@pytest.mark.parametrize("W,T1,p", [(4, 5, 0.7), (8, 9, 0.8), (16, 9, 0.8), (32, 9, 0.9), (3, 17, 0.9)])
def test_fold_in_verify_matches_oracle(W, T1, p):
    """Every step: outputs against the oracle, then every slot's log length
    right after the verify (a full log folded: 0) and after the commit, and
    positions; at the end the stored checkpoints.  W = 4 with 5 step tokens
    moves kept tokens over rows they overlap; W = 32 folds with K = 48;
    17 step tokens take 32 output columns."""
    import torch
    m = _mod()
    H, P, N, G, R = 8, 64, 128, 2, 6
    T = T1 - 1
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)])
    pool = _pools(m, H, P, N, G, R, W, T1, init)
    opool = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, max_tokens=T1,
                              init_state=init.astype(np.float64), fold_in_verify=True)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    steps = max(8, int(3 * W / oracle.expected_tokens_kept(p, T)) + 2)
    acc_all = synth.accept_counts(SEED + W, steps, R, T, p)
    slots = [4, 0, 5, 2, 1, 3]
    folds = 0
    try:
        for s in range(steps):
            x, dt, B, C = synth.batch_tokens(SEED, s, R, T1, H, P, G, N, BF, F32)
            full = opool.log_len[slots] >= W
            folds += int(full.sum())
            y = empty_like_out((R, T1, H, P), BF)
            assert m.ssm_verify_replay(pool, slots, T1, *_dev(x, dt, B, C), Ad, Dd, y) == m.SSM_OK
            assert m.ssm_last_path(pool) == "verify_replay_tc_fold"
            _, yo = opool.verify(slots, *_wide(x, dt, B, C))
            check_close(to_host(y), yo, BF, f"y step {s}", positions_axis=1, cond=opool.last_cond)
            np.testing.assert_array_equal(_log_lens(m, pool, R), opool.log_len, err_msg=f"log after verify {s}")
            acc = acc_all[s]
            assert m.ssm_state_commit(pool, slots, torch.from_numpy(acc).cuda(), False, Ad) == m.SSM_OK
            assert m.ssm_last_path(pool) == "commit_replay_append"
            opool.commit(slots, acc)
            np.testing.assert_array_equal(_log_lens(m, pool, R), opool.log_len, err_msg=f"log after commit {s}")
        assert folds >= 2, "the window filled too rarely"
        for sl in range(R):
            assert m.ssm_slot_info(pool, sl)[1].position == opool.position[sl]
        got = torch.empty((R, H, P, N), device="cuda")
        assert m.ssm_state_gather(pool, list(range(R)), got) == m.SSM_OK
        check_close(to_host(got), opool.state, BF, "checkpoints")
        assert m.ssm_pool_status(pool) == (m.SSM_OK, 0)
    finally:
        m.ssm_state_destroy(pool)


def test_fold_in_verify_checkpoint_reverify_force_fold_and_decode():
    """Between a verify that folded and its commit: a checkpoint read (the
    log is already in the checkpoint), a second verify in place of the first,
    and the commit that moves the kept tokens; then a forced fold at the
    commit empties the log so that a decode step may run."""
    import torch
    m = _mod()
    H, P, N, G, R, W, T1 = 4, 64, 128, 2, 3, 4, 5
    T = T1 - 1
    A, D = synth.head_params(SEED + 1, H)
    init = np.stack([synth.init_state(SEED + 1, s, H, P, N) for s in range(R)])
    pool = _pools(m, H, P, N, G, R, W, T1, init)
    opool = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, max_tokens=T1,
                              init_state=init.astype(np.float64), fold_in_verify=True)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    slots = [0, 1, 2]
    step = [0]

    def verify():
        x, dt, B, C = synth.batch_tokens(SEED + 1, step[0], R, T1, H, P, G, N, BF, F32)
        step[0] += 1
        y = empty_like_out((R, T1, H, P), BF)
        assert m.ssm_verify_replay(pool, slots, T1, *_dev(x, dt, B, C), Ad, Dd, y) == m.SSM_OK
        _, yo = opool.verify(slots, *_wide(x, dt, B, C))
        check_close(to_host(y), yo, BF, f"y step {step[0]}", positions_axis=1, cond=opool.last_cond)

    def commit(acc, force=False):
        assert m.ssm_state_commit(pool, slots, torch.tensor(acc, dtype=torch.int32, device="cuda"), force,
                                  Ad) == m.SSM_OK
        opool.commit(slots, acc, force_fold=force)
        np.testing.assert_array_equal(_log_lens(m, pool, R), opool.log_len)

    try:
        verify()
        commit([T, T, 1])  # logs of 5, 5 and 2 tokens: the first two are full
        assert list(opool.log_len) == [5, 5, 2]
        verify()           # folds slots 0 and 1
        # a checkpoint read between the verify and its commit: slot 0 is folded already, slot 2 folds now
        for sl in (0, 2):
            st, buf, meta = m.ssm_state_checkpoint(pool, sl, Ad)
            assert st == m.SSM_OK and meta.log_len == 0
            opool.flush([sl])
            check_close(buf.astype(np.float64), opool.state[sl], BF, f"checkpoint of slot {sl}")
        verify()           # a second verify in place of the first (nothing left to fold)
        commit([2, 0, 4])  # kept tokens move to the start of the emptied logs
        verify()
        commit([1, 1, 1], force=True)
        assert list(opool.log_len) == [0, 0, 0]
        # the logs are empty: a decode step runs and matches the oracle
        x, dt, B, C = (a[:, 0] for a in synth.batch_tokens(SEED + 1, 99, R, 1, H, P, G, N, BF, F32))
        y = empty_like_out((R, H, P), BF)
        assert m.ssm_decode_step(pool, slots, *_dev(x, dt, B, C), Ad, Dd, y) == m.SSM_OK
        _, yo = opool.decode(slots, *_wide(x, dt, B, C))
        check_close(to_host(y), yo, BF, "decode after a forced fold", cond=opool.last_cond)
        got = torch.empty((R, H, P, N), device="cuda")
        assert m.ssm_state_gather(pool, slots, got) == m.SSM_OK
        check_close(to_host(got), opool.state, BF, "states")
        assert m.ssm_pool_status(pool) == (m.SSM_OK, 0)
    finally:
        m.ssm_state_destroy(pool)


def test_fold_in_verify_poisoned_full_log_writes_nothing():
    """A NaN in the step of a request whose log is full: the request is
    flagged and poisoned, its checkpoint, log and outputs stay as they were;
    the other requests (one folding, one not) match the oracle."""
    import torch
    m = _mod()
    H, P, N, G, R, W, T1 = 4, 64, 128, 2, 3, 4, 5
    T = T1 - 1
    A, D = synth.head_params(SEED + 2, H)
    init = np.stack([synth.init_state(SEED + 2, s, H, P, N) for s in range(R)])
    pool = _pools(m, H, P, N, G, R, W, T1, init)
    opool = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, max_tokens=T1,
                              init_state=init.astype(np.float64), fold_in_verify=True)
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    slots = [0, 1, 2]
    try:
        x, dt, B, C = synth.batch_tokens(SEED + 2, 0, R, T1, H, P, G, N, BF, F32)
        y = empty_like_out((R, T1, H, P), BF)
        assert m.ssm_verify_replay(pool, slots, T1, *_dev(x, dt, B, C), Ad, Dd, y) == m.SSM_OK
        opool.verify(slots, *_wide(x, dt, B, C))
        acc = [T, T, 0]
        assert m.ssm_state_commit(pool, slots, torch.tensor(acc, dtype=torch.int32, device="cuda"), False,
                                  Ad) == m.SSM_OK
        opool.commit(slots, acc)
        before = torch.empty((R, H, P, N), device="cuda")
        m.ssm_state_gather(pool, slots, before)
        x, dt, B, C = synth.batch_tokens(SEED + 2, 1, R, T1, H, P, G, N, BF, F32)
        x = x.copy()
        x[0, 2, 1, 5] = np.uint16(0x7FC0)  # NaN in request 0's step, whose log is full
        y = torch.zeros((R, T1, H, P), dtype=torch.bfloat16, device="cuda")
        assert m.ssm_verify_replay(pool, slots, T1, *_dev(x, dt, B, C), Ad, Dd, y) == m.SSM_OK
        st, flags = m.ssm_pool_status(pool, clear=True)
        assert flags & m.SSM_FLAG_NONFINITE_INPUT
        _, meta0 = m.ssm_slot_info(pool, 0)
        assert meta0.flags & 1 and meta0.log_len == 5
        assert torch.count_nonzero(y[0]) == 0
        _, yo = opool.verify([1, 2], *_wide(x[1:], dt[1:], B[1:], C[1:]))
        check_close(to_host(y[1:]), yo, BF, "the other requests", positions_axis=1, cond=opool.last_cond)
        after = torch.empty_like(before)
        m.ssm_state_gather(pool, slots, after)
        assert torch.equal(after[0], before[0])
        check_close(to_host(after[1:]), opool.state[1:], BF, "the other checkpoints")
    finally:
        m.ssm_state_destroy(pool)


@pytest.mark.parametrize("T,p,W", [(8, 0.8, 16), (4, 0.6, 8), (8, 0.6, 32), (4, 0.8, 32)])
def test_fold_in_verify_full_batch_sampled(T, p, W):
    """The speculative-verify workload at batch 512 (Nemotron-shaped heads,
    bf16 token inputs, fp32 state) on a fold-in-verify pool: three requests
    followed by the oracle (outputs every step, checkpoints at the end), and
    every slot's position and log length against the oracle's rule."""
    import torch
    m = _mod()
    H, P, N, G, R = 128, 64, 128, 8, 512
    steps = {8: 6, 16: 8, 32: 14}[W]
    T1 = T + 1
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)])
    init_t = torch.from_numpy(init).cuda()
    sample = [0, 211, 511]
    osample = oracle.OraclePool(H, P, N, G, len(sample), A, D, mode=1, W=W, max_tokens=T1,
                                init_state=init[sample].astype(np.float64), fold_in_verify=True)
    del init
    meta_rule = oracle.OraclePool(1, 1, 16, 1, R, np.zeros(1), np.zeros(1), mode=1, W=W, max_tokens=T1,
                                  fold_in_verify=True)
    pool = m.ssm_state_init(m.make_config(H, P, N, G, BF, F32, 1, W, T1, fold=m.SSM_FOLD_IN_VERIFY), R, init_t)
    del init_t
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    acc_all = synth.accept_counts(SEED, steps, R, T, p)
    slots = list(range(R))
    n_folds = 0
    try:
        for s in range(steps):
            x, dt, B, C = synth.batch_tokens(SEED, s, R, T1, H, P, G, N, BF, F32)
            y = empty_like_out((R, T1, H, P), BF)
            assert m.ssm_verify_replay(pool, slots, T1, *_dev(x, dt, B, C), Ad, Dd, y) == m.SSM_OK
            assert m.ssm_last_path(pool) == "verify_replay_tc_fold"
            assert m.ssm_state_commit(pool, slots, torch.from_numpy(acc_all[s]).cuda(), False, Ad) == m.SSM_OK
            assert m.ssm_last_path(pool) == "commit_replay_append"
            _, yo = osample.verify(list(range(len(sample))), *_wide(x[sample], dt[sample], B[sample], C[sample]))
            osample.commit(list(range(len(sample))), acc_all[s][sample])
            check_close(to_host(y[sample]), yo, BF, f"y step {s}", positions_axis=1, cond=osample.last_cond)
            z = np.zeros((R, T1, 1, 1))
            n_folds += int(np.sum(meta_rule.log_len >= W))
            meta_rule.verify(slots, z, np.zeros((R, T1, 1)), np.zeros((R, T1, 1, 16)), np.zeros((R, T1, 1, 16)))
            meta_rule.commit(slots, acc_all[s])
        assert n_folds > 0, "the window never filled"
        torch.cuda.synchronize()
        assert m.ssm_pool_status(pool) == (m.SSM_OK, 0)
        for sl in slots[::37] + [R - 1]:
            _, meta = m.ssm_slot_info(pool, sl)
            assert meta.position == meta_rule.position[sl] and meta.log_len == meta_rule.log_len[sl]
        got = torch.empty((len(sample), H, P, N), dtype=torch.float32, device="cuda")
        m.ssm_state_gather(pool, sample, got)
        check_close(to_host(got), osample.state, BF, "checkpoints")
    finally:
        m.ssm_state_destroy(pool)
