"""GPU parity of speculative verify (state copies and ReplaySSM replay) and of
the commit (pointer move, log append, fold) against the CPU oracle.  Index
state (positions, log lengths, fold decisions) must match bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from tests._helpers import check_close, empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 3000


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _dev_inputs(x, dt, B, C, dt_in, dt_dt):
    return to_device(x, dt_in), to_device(dt, dt_dt), to_device(B, dt_in), to_device(C, dt_in)


def _wide(x, dt, B, C, dt_in, dt_dt):
    return synth.widen(x, dt_in), synth.widen(dt, dt_dt), synth.widen(B, dt_in), synth.widen(C, dt_in)


def _run_small(mode, W, T, p, steps, H=4, P=16, N=32, G=2, dt_in=synth.F32, n_tok_pattern=None, force_last=True,
               expect_path=None, y_round_mismatch=None, expect_commit_path=None):
    import torch
    m = _mod()
    n_slots, slots = 8, [6, 1, 3, 0, 7]
    R = len(slots)
    T1 = T + 1
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(n_slots)])
    cfg = m.make_config(H, P, N, G, dt_in, synth.F32, mode, W, T1)
    pool = m.ssm_state_init(cfg, n_slots, torch.from_numpy(init).cuda())
    opool = oracle.OraclePool(H, P, N, G, n_slots, A, D, mode=mode, W=W, max_tokens=T1,
                              init_state=init.astype(np.float64))
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    acc_all = synth.accept_counts(SEED, steps, R, T, p)
    verify = m.ssm_verify_copy if mode == m.SSM_MODE_COPY else m.ssm_verify_replay
    ys, conds = [], []
    try:
        for s in range(steps):
            nt = T1 if n_tok_pattern is None else n_tok_pattern[s % len(n_tok_pattern)]
            acc = np.minimum(acc_all[s], nt - 1).astype(np.int32)
            x, dt, B, C = synth.batch_tokens(SEED, s, R, nt, H, P, G, N, dt_in, synth.F32)
            y = empty_like_out((R, nt, H, P), dt_in)
            assert verify(pool, slots, nt, *_dev_inputs(x, dt, B, C, dt_in, synth.F32), Ad, Dd, y) == m.SSM_OK
            if expect_path is not None:
                assert m.ssm_last_path(pool) == expect_path
            _, yo = opool.verify(slots, *_wide(x, dt, B, C, dt_in, synth.F32))
            check_close(to_host(y), yo, dt_in, f"y step {s}", positions_axis=1, cond=opool.last_cond)
            if y_round_mismatch is not None:  # share of outputs that differ from the oracle rounded to bf16
                g = np.asarray(to_host(y), np.float64)
                o16 = synth.bf16_to_f32(synth.f32_to_bf16(np.asarray(yo, np.float32))).astype(np.float64)
                frac = float(np.mean(g != o16))
                assert frac <= y_round_mismatch, (s, frac, y_round_mismatch)
            ys.append(to_host(y))
            conds.append(opool.last_cond)
            force = force_last and s == steps - 1
            assert m.ssm_state_commit(pool, slots, torch.from_numpy(acc).cuda(), force, Ad) == m.SSM_OK
            if expect_commit_path is not None:
                assert m.ssm_last_path(pool) == expect_commit_path
            _, folded = opool.commit(slots, acc, force_fold=force)
            for sl in range(n_slots):
                st, meta = m.ssm_slot_info(pool, sl)
                assert st == m.SSM_OK
                assert meta.position == opool.position[sl], (s, sl)
                assert meta.log_len == opool.log_len[sl], (s, sl)
                assert meta.flags == 0
        got = torch.empty((n_slots, H, P, N), dtype=torch.float32, device="cuda")
        assert m.ssm_state_gather(pool, list(range(n_slots)), got) == m.SSM_OK
        check_close(to_host(got), opool.state, dt_in, "state")
        st, flags = m.ssm_pool_status(pool)
        assert st == m.SSM_OK and flags == 0
        return pool, opool, (ys, conds), (A, D)
    except BaseException:
        m.ssm_state_destroy(pool)
        raise


@pytest.mark.parametrize("T,p", [(4, 0.6), (3, 0.9)])
def test_copy_verify_matches_oracle(T, p):
    m = _mod()
    pool, _, _, _ = _run_small(m.SSM_MODE_COPY, 16, T, p, steps=7)
    m.ssm_state_destroy(pool)


@pytest.mark.parametrize("W,T,p", [(3, 4, 0.6), (8, 4, 0.8), (16, 2, 0.5), (1, 3, 0.7)])
def test_replay_verify_matches_oracle(W, T, p):
    m = _mod()
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, W, T, p, steps=9)
    m.ssm_state_destroy(pool)


def test_replay_kernel_choice():
    """Pools take the tensor-map verify (group coefficient + streaming
    kernels); an odd headdim (21, which neither the tensor-map nor the
    bulk-copy kernel takes) runs the one-CTA-per-head kernel and the
    unpipelined fold.  The bulk-copy kernel serves ssm_verify_replay_static
    (test_zz_no_alloc).  All match the oracle."""
    m = _mod()
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, 4, 3, 0.7, steps=6, expect_path="verify_replay_tma")
    m.ssm_state_destroy(pool)
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, 4, 3, 0.7, steps=6, P=21, expect_path="verify_replay")
    m.ssm_state_destroy(pool)


@pytest.mark.parametrize("dt_in,T,W,path", [
    (synth.F32, 8, 16, "verify_replay_tc"),   # fp32 inputs: C split too (three MMAs per K step)
    (synth.BF16, 8, 16, "verify_replay_tc"),
    (synth.BF16, 19, 8, "verify_replay_tc"),  # 20 step tokens: 32 MMA columns
    (synth.F32, 19, 8, "verify_replay_tc"),
])
def test_replay_tensor_core_verify(dt_in, T, W, path):
    """Heads of 64 rows in pairs run C_j . h_c on the tensor cores with the
    checkpoint split into hi and lo (tf32 for fp32 inputs, with C split too;
    bf16 for bf16 inputs); at fp32 inputs the oracle's 1e-5 tolerance checks
    that the splits keep fp32 accuracy."""
    m = _mod()
    fold = "commit_replay_fold_tc" if dt_in == synth.BF16 else "commit_replay_fold_pipe"
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, W, T, 0.7, steps=6, H=4, P=64, N=128, G=2, dt_in=dt_in,
                               expect_path=path, expect_commit_path=fold)
    m.ssm_state_destroy(pool)


@pytest.mark.parametrize("dt_in,T,W,fold", [
    (synth.BF16, 8, 32, "commit_replay_fold_tc"),    # log capacity 40: the fold's K = 48
    (synth.F32, 8, 32, "commit_replay_fold_pipe"),
    (synth.BF16, 4, 32, "commit_replay_fold_tc"),    # capacity 36
    (synth.BF16, 19, 40, "commit_replay_fold_tc"),   # capacity 59: K = 64, 32 MMA columns
])
def test_replay_tensor_core_wide_window(dt_in, T, W, fold):
    """Windows whose log holds more than 32 tokens (W - 1 + T + 1 > 32) stay on
    the tensor-core verify and, for bf16 pools, the tensor-core fold; 16 steps
    so the log fills and folds at least once before the final forced fold."""
    m = _mod()
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, W, T, 0.7, steps=16, H=4, P=64, N=128, G=2, dt_in=dt_in,
                               expect_path="verify_replay_tc", expect_commit_path=fold)
    m.ssm_state_destroy(pool)


@pytest.mark.parametrize("T,W", [(8, 16), (19, 8)])
def test_replay_tensor_core_bf16_product_keeps_fp32_grade(T, W):
    """bf16 inputs run C_j . h_c as kind::f16 MMAs with the fp32 checkpoint
    split into bf16 hi and lo (16 significant bits, |v - hi - lo| <= 2^-17 |v|).
    Then y equals the fp64 oracle rounded to bf16 for all but 1 % of the
    outputs: only fp32 rounding right at a bf16 tie can flip one (measured:
    0.02-0.04 %).  With the lo term dropped the product is off by about 2^-9
    of its size and 6-11 % of the outputs round the other way."""
    m = _mod()
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, W, T, 0.7, steps=6, H=4, P=64, N=128, G=2, dt_in=synth.BF16,
                               expect_path="verify_replay_tc", y_round_mismatch=0.01)
    m.ssm_state_destroy(pool)


def test_replay_tensor_core_mixed_token_counts():
    m = _mod()
    pool, _, _, _ = _run_small(m.SSM_MODE_REPLAY, 8, 8, 0.6, steps=8, H=8, P=64, N=128, G=2, dt_in=synth.BF16,
                               n_tok_pattern=[9, 3, 1, 7], expect_path="verify_replay_tc")
    m.ssm_state_destroy(pool)


def test_replay_mixed_token_counts_and_checkpoint_fold():
    import torch
    m = _mod()
    pool, opool, _, (A, D) = _run_small(m.SSM_MODE_REPLAY, 8, 4, 0.7, steps=6, n_tok_pattern=[5, 2, 3, 1],
                                        force_last=False)
    try:
        Ad = torch.from_numpy(A).cuda()
        for sl in (6, 1):
            st, host, meta = m.ssm_state_checkpoint(pool, sl, Ad)
            assert st == m.SSM_OK and meta.log_len == 0
            opool.flush([sl])
            check_close(host.astype(np.float64), opool.state[sl], synth.F32, f"checkpoint {sl}")
            assert meta.position == opool.position[sl]
    finally:
        m.ssm_state_destroy(pool)


def test_copy_and_replay_agree_on_gpu():
    """Same inputs and accept counts through both flavours: outputs agree and,
    after a final forced fold, so do the states (The Fix: the same math)."""
    import torch
    m = _mod()
    pc, _, (yc, cc), _ = _run_small(m.SSM_MODE_COPY, 16, 4, 0.7, steps=8)
    pr, _, (yr, _), _ = _run_small(m.SSM_MODE_REPLAY, 4, 4, 0.7, steps=8)
    try:
        for a, b, c in zip(yc, yr, cc):
            check_close(b, a, synth.F32, "replay vs copy y", pair=True, cond=c)
        sc = torch.empty((8, 4, 16, 32), dtype=torch.float32, device="cuda")
        sr = torch.empty_like(sc)
        m.ssm_state_gather(pc, list(range(8)), sc)
        m.ssm_state_gather(pr, list(range(8)), sr)
        check_close(to_host(sr), to_host(sc), synth.F32, "replay vs copy state", pair=True)
    finally:
        m.ssm_state_destroy(pc)
        m.ssm_state_destroy(pr)


def test_verify_host_side_errors():
    import torch
    m = _mod()
    H, P, N, G = 2, 16, 16, 1
    cfg = m.make_config(H, P, N, G, 0, 0, m.SSM_MODE_COPY, 4, 3)
    pool = m.ssm_state_init(cfg, 4)
    try:
        A = torch.full((H,), -1.0, device="cuda")
        acc = torch.zeros(2, dtype=torch.int32, device="cuda")
        # commit with no verify since the last reset
        assert m.ssm_state_commit(pool, [0, 1], acc, False, A) == m.SSM_ERR_INVALID_STATE
        x = torch.zeros((2, 3, H, P), device="cuda")
        dt = torch.zeros((2, 3, H), device="cuda")
        B = torch.zeros((2, 3, G, N), device="cuda")
        y = torch.empty_like(x)
        # duplicate slot, slot out of range, too many tokens, wrong flavour
        assert m.ssm_verify_copy(pool, [1, 1], 3, x, dt, B, B, A, A, y) == m.SSM_ERR_INVALID_ARG
        assert m.ssm_verify_copy(pool, [1, 4], 3, x, dt, B, B, A, A, y) == m.SSM_ERR_INVALID_ARG
        x4 = torch.zeros((2, 4, H, P), device="cuda")
        sl_arr, sl_ptr = m._binding._host_i32([0, 1])
        assert m._binding._lib.ssm_verify_copy(pool.handle, 2, 4, sl_ptr,
                                               x4.data_ptr(), dt.data_ptr(), B.data_ptr(), B.data_ptr(),
                                               A.data_ptr(), A.data_ptr(), x4.data_ptr(), None) == m.SSM_ERR_INVALID_ARG
        del sl_arr
        assert m.ssm_verify_replay(pool, [0, 1], 3, x, dt, B, B, A, A, y) == m.SSM_ERR_INVALID_ARG
        # a released slot refuses work until reset
        assert m.ssm_state_release(pool, [1]) == m.SSM_OK
        assert m.ssm_verify_copy(pool, [0, 1], 3, x, dt, B, B, A, A, y) == m.SSM_ERR_INVALID_STATE
        assert m.ssm_state_reset(pool, [1]) == m.SSM_OK
        assert m.ssm_verify_copy(pool, [0, 1], 3, x, dt, B, B, A, A, y) == m.SSM_OK
        # accept outside [0, n_tok - 1] is flagged on the device and the slot skipped
        bad = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
        assert m.ssm_state_commit(pool, [0, 1], bad, False, A) == m.SSM_OK
        st, flags = m.ssm_pool_status(pool, clear=True)
        assert flags & m.SSM_FLAG_BAD_ACCEPT
        assert m.ssm_slot_info(pool, 0)[1].position == 2 and m.ssm_slot_info(pool, 0)[1].flags == 0
        assert m.ssm_slot_info(pool, 1)[1].position == 0 and m.ssm_slot_info(pool, 1)[1].flags & 1
    finally:
        m.ssm_state_destroy(pool)


@pytest.mark.parametrize("T,p,W", [(T, p, W) for T in (4, 8) for p in (0.6, 0.8) for W in (8, 16, 32)])
def test_config3_full_batch_sampled(T, p, W):
    """Speculative verify at batch 512 with Nemotron-shaped heads, bf16 token
    inputs, fp32 state, at every (T, p, W) point of the workload: copy and
    replay flavours on the same inputs and accept counts; three requests
    followed by the oracle; every slot's position and log length checked
    against the oracle's commit rule.  Replay runs the tensor-core verify and
    fold at every window (a log of up to 40 tokens at W = 32); enough steps
    that the window fills (W = 32 needs about 32 / E[1 + accept] steps)."""
    import torch
    m = _mod()
    H, P, N, G, R = 128, 64, 128, 8, 512
    steps = {8: 6, 16: 8, 32: 14}[W]
    T1 = T + 1
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(R)])
    init_t = torch.from_numpy(init).cuda()
    sample = [0, 211, 511]
    osample = {md: oracle.OraclePool(H, P, N, G, len(sample), A, D, mode=md, W=W, max_tokens=T1,
                                     init_state=init[sample].astype(np.float64)) for md in (0, 1)}
    del init
    # the commit rule on every slot, tracked by the oracle pool at unit size
    meta_rule = oracle.OraclePool(1, 1, 16, 1, R, np.zeros(1), np.zeros(1), mode=1, W=W, max_tokens=T1)
    pools = {md: m.ssm_state_init(m.make_config(H, P, N, G, synth.BF16, synth.F32, md, W, T1), R, init_t)
             for md in (0, 1)}
    del init_t
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    acc_all = synth.accept_counts(SEED, steps, R, T, p)
    slots = list(range(R))
    n_folds = 0
    try:
        for s in range(steps):
            x, dt, B, C = synth.batch_tokens(SEED, s, R, T1, H, P, G, N, synth.BF16, synth.F32)
            dev = _dev_inputs(x, dt, B, C, synth.BF16, synth.F32)
            acc = torch.from_numpy(acc_all[s]).cuda()
            ys = {}
            for md, fn in ((0, m.ssm_verify_copy), (1, m.ssm_verify_replay)):
                y = empty_like_out((R, T1, H, P), synth.BF16)
                assert fn(pools[md], slots, T1, *dev, Ad, Dd, y) == m.SSM_OK
                assert m.ssm_last_path(pools[md]) == ("verify_copy" if md == 0 else "verify_replay_tc")
                assert m.ssm_state_commit(pools[md], slots, acc, False, Ad) == m.SSM_OK
                assert m.ssm_last_path(pools[md]) == ("commit_copy" if md == 0 else "commit_replay_fold_tc")
                ys[md] = y
                _, yo = osample[md].verify(list(range(len(sample))),
                                           *_wide(x[sample], dt[sample], B[sample], C[sample], synth.BF16, synth.F32))
                osample[md].commit(list(range(len(sample))), acc_all[s][sample])
                check_close(to_host(y[sample]), yo, synth.BF16, f"mode {md} y step {s}", positions_axis=1,
                            cond=osample[md].last_cond)
            check_close(to_host(ys[1]), to_host(ys[0]), synth.BF16, f"replay vs copy step {s}", pair=True)
            z = np.zeros((R, T1, 1, 1))
            meta_rule.verify(slots, z, np.zeros((R, T1, 1)), np.zeros((R, T1, 1, 16)), np.zeros((R, T1, 1, 16)))
            _, folded = meta_rule.commit(slots, acc_all[s])
            n_folds += int(folded.sum())
        assert n_folds > 0, "the window never filled"
        torch.cuda.synchronize()
        for md in (0, 1):
            st, flags = m.ssm_pool_status(pools[md])
            assert st == m.SSM_OK and flags == 0
            for sl in slots[::37] + [R - 1]:
                _, meta = m.ssm_slot_info(pools[md], sl)
                assert meta.position == meta_rule.position[sl]
                if md == 1:
                    assert meta.log_len == meta_rule.log_len[sl]
            got = torch.empty((len(sample), H, P, N), dtype=torch.float32, device="cuda")
            m.ssm_state_gather(pools[md], sample, got)
            check_close(to_host(got), osample[md].state, synth.BF16, f"mode {md} state")
    finally:
        for pl in pools.values():
            m.ssm_state_destroy(pl)


@pytest.mark.parametrize("mode,where", [(1, "x"), (1, "B"), (1, "C"), (1, "dt"), (0, "x"), (0, "B")])
def test_nonfinite_verify_input_poisons_only_its_request(mode, where):
    """A NaN or Inf in one request's step inputs (bf16 x / B / C, fp32 dt)
    flags SSM_FLAG_NONFINITE_INPUT and poisons that request's slot; its commit
    is refused on the device (position and log left as they were); the other
    requests' outputs, commits and later steps match the oracle."""
    import torch
    m = _mod()
    H, P, N, G, T, W = 4, 64, 128, 2, 4, 8
    T1 = T + 1
    slots = [0, 1, 2]
    A, D = synth.head_params(SEED, H)
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(3)])
    pool = m.ssm_state_init(m.make_config(H, P, N, G, synth.BF16, synth.F32, mode, W, T1), 3,
                            torch.from_numpy(init).cuda())
    opool = oracle.OraclePool(H, P, N, G, 3, A, D, mode=mode, W=W, max_tokens=T1, init_state=init.astype(np.float64))
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    verify = m.ssm_verify_copy if mode == m.SSM_MODE_COPY else m.ssm_verify_replay
    nan16, inf16 = np.uint16(0x7FC0), np.uint16(0x7F80)
    try:
        for s in range(4):
            live = slots if s < 2 else [0, 2]
            x, dt, B, C = synth.batch_tokens(SEED + 5, s, len(live), T1, H, P, G, N, synth.BF16, synth.F32)
            if s == 1:  # request 1 of this step
                if where == "x":
                    x[1, 2, 3, 5] = inf16
                elif where == "B":
                    B[1, 0, 1, 7] = nan16
                elif where == "C":
                    C[1, 4, 0, 9] = inf16
                else:
                    dt[1, 3, 2] = np.nan
            y = empty_like_out((len(live), T1, H, P), synth.BF16)
            assert verify(pool, live, T1, *_dev_inputs(x, dt, B, C, synth.BF16, synth.F32), Ad, Dd, y) == m.SSM_OK
            good = [i for i, sl in enumerate(live) if not (s == 1 and sl == 1)]
            gsl = [live[i] for i in good]
            _, yo = opool.verify(gsl, *[synth.widen(a[good], d) for a, d in
                                        ((x, synth.BF16), (dt, synth.F32), (B, synth.BF16), (C, synth.BF16))])
            check_close(to_host(y)[good], yo, synth.BF16, f"y step {s}", positions_axis=1, cond=opool.last_cond)
            acc = np.full(len(live), 2, np.int32)
            if s == 1:
                before = m.ssm_slot_info(pool, 1)[1]
            assert m.ssm_state_commit(pool, live, torch.from_numpy(acc).cuda(), False, Ad) == m.SSM_OK
            opool.commit(gsl, acc[good])
            st, flags = m.ssm_pool_status(pool, clear=True)
            if s == 1:
                assert flags & m.SSM_FLAG_NONFINITE_INPUT, flags
                meta = m.ssm_slot_info(pool, 1)[1]
                assert meta.flags & 1
                assert (meta.position, meta.log_len) == (before.position, before.log_len)
            else:
                assert flags == 0, (s, flags)
            for sl in (0, 2):
                meta = m.ssm_slot_info(pool, sl)[1]
                assert meta.position == opool.position[sl] and meta.log_len == opool.log_len[sl] and meta.flags == 0
        got = torch.empty((3, H, P, N), dtype=torch.float32, device="cuda")
        assert m.ssm_state_gather(pool, [0, 1, 2], got) == m.SSM_OK
        check_close(to_host(got)[[0, 2]], opool.state[[0, 2]], synth.BF16, "healthy states")
    finally:
        m.ssm_state_destroy(pool)


def test_bounded_wait_runs_out_and_the_pool_recovers():
    """Failure path of the tensor-core replay verify, made on the host: the
    next verify withholds one CTA's per-item loads
    (ssm_debug_stall_next_verify), so the waits on them run out (each bounded,
    about a second) and that CTA's roles leave through their abort paths.  The
    call returns, SSM_FLAG_TIMEOUT is raised (and nothing else), and the same
    step verified again, then committed, matches the oracle."""
    import time

    import torch
    m = _mod()
    H, P, N, G, R, T1, W = 4, 64, 128, 2, 4, 5, 8
    A, D = synth.head_params(SEED + 5, H)
    init = np.stack([synth.init_state(SEED + 5, s, H, P, N) for s in range(R)])
    pool = m.ssm_state_init(m.make_config(H, P, N, G, synth.BF16, synth.F32, m.SSM_MODE_REPLAY, W, T1), R,
                            torch.from_numpy(init).cuda())
    opool = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, max_tokens=T1,
                              init_state=init.astype(np.float64))
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    slots = list(range(R))
    try:
        x, dt, B, C = synth.batch_tokens(SEED + 5, 0, R, T1, H, P, G, N, synth.BF16, synth.F32)
        dev = _dev_inputs(x, dt, B, C, synth.BF16, synth.F32)
        y = empty_like_out((R, T1, H, P), synth.BF16)
        assert m.ssm_debug_stall_next_verify(pool) == m.SSM_OK
        t0 = time.monotonic()
        assert m.ssm_verify_replay(pool, slots, T1, *dev, Ad, Dd, y) == m.SSM_OK
        assert m.ssm_last_path(pool) == "verify_replay_tc"
        st, flags = m.ssm_pool_status(pool, clear=True)
        assert st == m.SSM_OK and flags == m.SSM_FLAG_TIMEOUT, flags
        assert time.monotonic() - t0 < 60
        for sl in slots:  # a pool-wide flag: no slot is poisoned
            assert m.ssm_slot_info(pool, sl)[1].flags == 0
        # the same step again, then its commit, as if the failed call had not happened
        y = empty_like_out((R, T1, H, P), synth.BF16)
        assert m.ssm_verify_replay(pool, slots, T1, *dev, Ad, Dd, y) == m.SSM_OK
        _, yo = opool.verify(slots, *_wide(x, dt, B, C, synth.BF16, synth.F32))
        check_close(to_host(y), yo, synth.BF16, "y after the timeout", positions_axis=1, cond=opool.last_cond)
        acc = np.array([2, 0, 4, 1], np.int32)
        assert m.ssm_state_commit(pool, slots, torch.from_numpy(acc).cuda(), False, Ad) == m.SSM_OK
        opool.commit(slots, acc)
        x, dt, B, C = synth.batch_tokens(SEED + 5, 1, R, T1, H, P, G, N, synth.BF16, synth.F32)
        assert m.ssm_verify_replay(pool, slots, T1, *_dev_inputs(x, dt, B, C, synth.BF16, synth.F32), Ad, Dd,
                                   y) == m.SSM_OK
        _, yo = opool.verify(slots, *_wide(x, dt, B, C, synth.BF16, synth.F32))
        check_close(to_host(y), yo, synth.BF16, "the next step", positions_axis=1, cond=opool.last_cond)
        assert m.ssm_pool_status(pool) == (m.SSM_OK, 0)
    finally:
        m.ssm_state_destroy(pool)
