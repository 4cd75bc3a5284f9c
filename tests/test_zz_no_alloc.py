"""The replay verify entry point that allocates nothing, against the pool's.

Some callers cannot call cudaMalloc: a serving engine whose caching
allocator owns all device memory, or a plugin that is handed only the
buffers its host runtime manages.  They cannot create a pool, so
ssm_verify_replay_static gives them the replay verify on buffers they own,
with its scratch taken from an array built into the library.  This test
runs the same verify steps through a pool (ssm_verify_replay plus
ssm_state_commit) and through the static entry point on caller-owned
checkpoint and log buffers, and compares the outputs of two calls in a row.
It lives in its own file, collected after every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from tests._helpers import check_close, empty_like_out, to_device, to_host

pytestmark = pytest.mark.gpu


def test_static_scratch_replay_matches_pool_entry_point():
    import torch

    import hybrid_serving_mamba_gb300 as m
    H, P, N, G, R, T1, W = 16, 64, 128, 4, 6, 5, 8
    BF, F = synth.BF16, synth.F32
    seed = synth.BASE_SEED + 7000
    A, D = synth.head_params(seed, H)
    init = np.stack([synth.init_state(seed, s, H, P, N) for s in range(R)])
    Ad, Dd = torch.from_numpy(A).cuda(), torch.from_numpy(D).cuda()
    init_t = torch.from_numpy(init).cuda()
    slots = list(range(R))
    acc1 = np.array([0, 1, 2, 0, 1, 2], np.int32)   # log after step 0: 1..3 tokens
    acc2 = np.array([1, 0, 2, 1, 0, 1], np.int32)   # log after step 1: 3..6 tokens, below W: no fold
    steps = [synth.batch_tokens(seed, s, R, T1, H, P, G, N, BF, F) for s in range(3)]
    dev = [tuple(to_device(a, code) for a, code in zip(st, (BF, F, BF, BF))) for st in steps]

    # the pool path: verify, commit (append), verify, commit (append), verify
    pool = m.ssm_state_init(m.make_config(H, P, N, G, BF, F, m.SSM_MODE_REPLAY, W, T1), R, init_t)
    try:
        y_pool = []
        for s, acc in ((0, acc1), (1, acc2), (2, None)):
            y = empty_like_out((R, T1, H, P), BF)
            assert m.ssm_verify_replay(pool, slots, T1, *dev[s], Ad, Dd, y) == m.SSM_OK
            y_pool.append(y)
            if acc is not None:
                assert m.ssm_state_commit(pool, slots, torch.from_numpy(acc).cuda(), False, Ad) == m.SSM_OK
        assert m.ssm_pool_status(pool)[1] == 0
    finally:
        m.ssm_state_destroy(pool)

    # the caller's own checkpoint and log, holding the tokens kept at step 0
    Wc = W - 1 + T1
    ckpt = init_t.clone()
    log_x = torch.zeros((R, Wc, H, P), dtype=torch.bfloat16, device="cuda")
    log_dt = torch.zeros((R, Wc, H), device="cuda")
    log_B = torch.zeros((R, Wc, G, N), dtype=torch.bfloat16, device="cuda")
    x0, dt0, B0, _ = dev[0]
    for r in range(R):
        c = int(acc1[r]) + 1
        log_x[r, :c] = x0[r, :c]
        log_dt[r, :c] = dt0[r, :c]
        log_B[r, :c] = B0[r, :c]
    log_len = torch.from_numpy(acc1 + 1).cuda()
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")

    # two calls in a row; each call stages its step after the log, so
    # appending the kept tokens is log_len += c
    for call, s in enumerate((1, 2)):
        y = empty_like_out((R, T1, H, P), BF)
        st = m.ssm_verify_replay_static(R, T1, H, P, N, G, W, BF, F, ckpt, log_x, log_dt, log_B, log_len,
                                        *dev[s], Ad, Dd, y, flags)
        assert st == m.SSM_OK
        # the bulk-copy pipelined kernel (the tensor-map kernels need the pool's larger scratch)
        assert m.ssm_last_path(None) == "verify_replay_pipe"
        torch.cuda.synchronize()
        check_close(to_host(y), to_host(y_pool[s]), BF, f"static call {call} (verify step {s})", positions_axis=1,
                    pair=True)
        if s == 1:
            log_len += torch.from_numpy(acc2 + 1).cuda()
    assert int(flags.item()) == 0
    assert torch.equal(ckpt, init_t)   # the checkpoint is read only

    # requests beyond the built-in scratch are refused before any work; each limit on its own
    lib = m.library()
    p = ctypes.c_void_p(ckpt.data_ptr())
    ptrs = [p] * 13  # ckpt .. y; flags and the stream follow
    # the batch limit alone (everything else in range, the scratch need small)
    assert lib.ssm_verify_replay_static(1025, 1, 8, 64, 128, 1, 1, BF, F, *ptrs, p, None) == m.SSM_ERR_INVALID_ARG
    # the scratch size alone: batch 1024, G 8, 9 tokens, Wc4 = 24 -> 1,769,472 floats > 1,047,552
    assert lib.ssm_verify_replay_static(1024, 9, 64, 64, 128, 8, 16, BF, F, *ptrs, p, None) == m.SSM_ERR_INVALID_ARG
    assert 1024 * 8 * 9 * 24 > m.SSM_STATIC_SCRATCH_FLOATS >= 1024 * 8 * 1 * 4


def test_static_scratch_replay_at_serving_batch():
    """At batch 512 with Nemotron-shaped heads, 8 drafts and window 16 (the
    speculative verify workload) the static entry point runs the persistent
    bulk-copy kernel over the whole GPU and gives the outputs of the pool's
    verify on the same checkpoints and empty logs, on two calls in a row."""
    import torch

    import hybrid_serving_mamba_gb300 as m
    H, P, N, G, R, T1, W = 128, 64, 128, 8, 512, 9, 16  # scratch: 512 * 8 * 9 * 24 floats
    BF, F = synth.BF16, synth.F32
    seed = synth.BASE_SEED + 7100
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    A = -torch.exp(torch.rand(H, generator=gen, device="cuda") * 1.5)
    D = torch.randn(H, generator=gen, device="cuda")
    ckpt = (torch.randn((R, H, P, N), generator=gen, device="cuda") * 0.1).contiguous()
    x = torch.randn((R, T1, H, P), generator=gen, device="cuda").bfloat16()
    dt = torch.nn.functional.softplus(torch.randn((R, T1, H), generator=gen, device="cuda") * 0.5 - 2.0)
    B = torch.randn((R, T1, G, N), generator=gen, device="cuda").bfloat16()
    C = torch.randn((R, T1, G, N), generator=gen, device="cuda").bfloat16()
    pool = m.ssm_state_init(m.make_config(H, P, N, G, BF, F, m.SSM_MODE_REPLAY, W, T1), R, ckpt)
    try:
        y_pool = torch.empty((R, T1, H, P), dtype=torch.bfloat16, device="cuda")
        assert m.ssm_verify_replay(pool, list(range(R)), T1, x, dt, B, C, A, D, y_pool) == m.SSM_OK
    finally:
        m.ssm_state_destroy(pool)
    Wc = W - 1 + T1
    log_x = torch.zeros((R, Wc, H, P), dtype=torch.bfloat16, device="cuda")
    log_dt = torch.zeros((R, Wc, H), device="cuda")
    log_B = torch.zeros((R, Wc, G, N), dtype=torch.bfloat16, device="cuda")
    log_len = torch.zeros(R, dtype=torch.int32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        y = torch.empty_like(y_pool)
        assert m.ssm_verify_replay_static(R, T1, H, P, N, G, W, BF, F, ckpt, log_x, log_dt, log_B, log_len,
                                          x, dt, B, C, A, D, y, flags) == m.SSM_OK
        assert m.ssm_last_path(None) == "verify_replay_pipe"
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        check_close(to_host(y), to_host(y_pool), BF, f"static call {call} at batch {R}", pair=True)
