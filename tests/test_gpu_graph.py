"""CUDA-graph capture of the decode and verify loops: a graph of library calls,
replayed with new inputs copied into its fixed buffers, gives bit for bit the
outputs, states and positions of the same calls made one by one (Mamba
Streaming State That Survives Chunking, Separate Mamba-2 algebra from kernel
behavior: graph-capture overhead is one of the costs to measure, so the
captured path has to be the same computation).

The captured calls are the decode step, the replay verify with its commit
(folds included, the window filling during the run) and the copy verify with
its commit.  Host-side checks run once, at capture; everything a replay
changes lives on the device."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

SEED = synth.BASE_SEED + 7600


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def _dev(a, code):
    from tests._helpers import to_device
    return to_device(a, code)


def _pool(m, shape, dt_in, mode, n_slots, W, T1):
    import torch
    H, P, N, G = shape
    init = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(n_slots)])
    cfg = m.make_config(H, P, N, G, dt_in, synth.F32, mode, W, T1)
    return m.ssm_state_init(cfg, n_slots, torch.from_numpy(init).cuda())


def _states(m, pool, slots, shape):
    import torch
    H, P, N, _ = shape
    got = torch.empty((len(slots), H, P, N), dtype=torch.float32, device="cuda")
    assert m.ssm_state_gather(pool, slots, got) == m.SSM_OK
    torch.cuda.synchronize()
    return got.cpu()


def _positions(m, pool, slots):
    return [m.ssm_slot_info(pool, s)[1].position for s in slots]


@pytest.mark.parametrize("dt_in,shape", [
    (synth.BF16, (8, 64, 128, 2)),
    (synth.F32, (4, 16, 32, 2)),
])
def test_decode_graph_matches_eager(dt_in, shape):
    """One graph per decode step (replayed with each step's inputs), and one
    graph holding a loop of four steps, against the same steps eagerly."""
    import torch
    m = _mod()
    H, P, N, G = shape
    A, D = (torch.from_numpy(v).cuda() for v in synth.head_params(SEED, H))
    slots = [5, 0, 3, 6, 1]
    R, steps = len(slots), 8
    toks = [synth.batch_tokens(SEED, s, R, 1, H, P, G, N, dt_in, synth.F32) for s in range(steps)]
    toks = [tuple(_dev(a[:, 0], c) for a, c in zip(t, (dt_in, synth.F32, dt_in, dt_in))) for t in toks]
    tdt = torch.bfloat16 if dt_in == synth.BF16 else torch.float32
    eager = _pool(m, shape, dt_in, m.SSM_MODE_COPY, 8, 8, 1)
    one = _pool(m, shape, dt_in, m.SSM_MODE_COPY, 8, 8, 1)
    loop = _pool(m, shape, dt_in, m.SSM_MODE_COPY, 8, 8, 1)
    warm = _pool(m, shape, dt_in, m.SSM_MODE_COPY, 8, 8, 1)
    try:
        # first calls (one-time attribute setting) happen outside the capture
        y0 = torch.empty((R, H, P), dtype=tdt, device="cuda")
        assert m.ssm_decode_step(warm, slots, *toks[0], A, D, y0) == m.SSM_OK
        torch.cuda.synchronize()

        static = [torch.empty_like(t) for t in toks[0]]
        ys = torch.empty((R, H, P), dtype=tdt, device="cuda")
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1):
            assert m.ssm_decode_step(one, slots, *static, A, D, ys) == m.SSM_OK
        K = 4
        static_loop = [torch.stack([toks[s][i] for s in range(K)]).clone() for i in range(4)]
        yl = torch.empty((K, R, H, P), dtype=tdt, device="cuda")
        g4 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g4):
            for s in range(K):
                assert m.ssm_decode_step(loop, slots, *(t[s] for t in static_loop), A, D, yl[s]) == m.SSM_OK

        ye = []
        for s in range(steps):
            y = torch.empty((R, H, P), dtype=tdt, device="cuda")
            assert m.ssm_decode_step(eager, slots, *toks[s], A, D, y) == m.SSM_OK
            ye.append(y)
        for s in range(steps):
            for dst, src in zip(static, toks[s]):
                dst.copy_(src)
            g1.replay()
            torch.cuda.synchronize()
            assert torch.equal(ys, ye[s]), f"step {s}: graph output differs from eager"
        for rep in range(steps // K):
            for i in range(4):
                static_loop[i].copy_(torch.stack([toks[rep * K + s][i] for s in range(K)]))
            g4.replay()
            torch.cuda.synchronize()
            for s in range(K):
                assert torch.equal(yl[s], ye[rep * K + s]), f"loop graph step {rep * K + s}"
        se = _states(m, eager, slots, shape)
        assert torch.equal(_states(m, one, slots, shape), se)
        assert torch.equal(_states(m, loop, slots, shape), se)
        assert _positions(m, one, slots) == _positions(m, eager, slots) == [steps] * R
        assert _positions(m, loop, slots) == [steps] * R
        for p in (eager, one, loop):
            assert m.ssm_pool_status(p)[1] == 0
    finally:
        for p in (eager, one, loop, warm):
            m.ssm_state_destroy(p)


@pytest.mark.parametrize("mode,dt_in,shape,W,T1", [
    (1, synth.BF16, (8, 64, 128, 2), 8, 5),    # replay: tensor-core verify and fold
    (1, synth.F32, (4, 16, 32, 2), 8, 4),      # replay: CUDA-core verify and fold
    (0, synth.BF16, (4, 64, 128, 2), 8, 5),    # copy verify, pointer-move commit
])
def test_verify_commit_graph_matches_eager(mode, dt_in, shape, W, T1):
    """verify + commit captured as one graph and replayed with each step's
    drafts and accept counts (device int32), the window filling and folding
    during the run, against the same calls eagerly."""
    import torch
    m = _mod()
    H, P, N, G = shape
    A, D = (torch.from_numpy(v).cuda() for v in synth.head_params(SEED + 1, H))
    slots = [2, 7, 4, 0, 5, 1]
    R, steps = len(slots), 10
    acc = synth.accept_counts(SEED, steps, R, T1 - 1, 0.7)
    toks = [synth.batch_tokens(SEED, 50 + s, R, T1, H, P, G, N, dt_in, synth.F32) for s in range(steps)]
    toks = [tuple(_dev(a, c) for a, c in zip(t, (dt_in, synth.F32, dt_in, dt_in))) for t in toks]
    accs = [torch.from_numpy(np.ascontiguousarray(acc[s], dtype=np.int32)).cuda() for s in range(steps)]
    tdt = torch.bfloat16 if dt_in == synth.BF16 else torch.float32
    eager = _pool(m, shape, dt_in, mode, 8, W, T1)
    graph = _pool(m, shape, dt_in, mode, 8, W, T1)
    warm = _pool(m, shape, dt_in, mode, 8, W, T1)
    verify = m.ssm_verify_replay if mode == m.SSM_MODE_REPLAY else m.ssm_verify_copy
    try:
        y0 = torch.empty((R, T1, H, P), dtype=tdt, device="cuda")
        for s in range(3):  # first calls of every kernel the run will use, folds included
            assert verify(warm, slots, T1, *toks[s], A, D, y0) == m.SSM_OK
            assert m.ssm_state_commit(warm, slots, accs[s], s == 2, A) == m.SSM_OK
        torch.cuda.synchronize()

        static = [torch.empty_like(t) for t in toks[0]]
        sacc = torch.empty_like(accs[0])
        ys = torch.empty((R, T1, H, P), dtype=tdt, device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            assert verify(graph, slots, T1, *static, A, D, ys) == m.SSM_OK
            assert m.ssm_state_commit(graph, slots, sacc, False, A) == m.SSM_OK

        folds = 0
        for s in range(steps):
            ye = torch.empty((R, T1, H, P), dtype=tdt, device="cuda")
            assert verify(eager, slots, T1, *toks[s], A, D, ye) == m.SSM_OK
            assert m.ssm_state_commit(eager, slots, accs[s], False, A) == m.SSM_OK
            for dst, src in zip(static, toks[s]):
                dst.copy_(src)
            sacc.copy_(accs[s])
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(ys, ye), f"step {s}: graph outputs differ from eager"
            if mode == m.SSM_MODE_REPLAY:
                le = [m.ssm_slot_info(eager, x)[1].log_len for x in slots]
                lg = [m.ssm_slot_info(graph, x)[1].log_len for x in slots]
                assert le == lg, (s, le, lg)
                folds += sum(1 for v in le if v == 0)
        assert torch.equal(_states(m, graph, slots, shape), _states(m, eager, slots, shape))
        want = [int(steps + acc[:, i].sum()) for i in range(R)]
        assert _positions(m, graph, slots) == _positions(m, eager, slots) == want
        if mode == m.SSM_MODE_REPLAY:
            assert folds > 0, "the run never folded: the window does not fill"
        for p in (eager, graph):
            assert m.ssm_pool_status(p)[1] == 0
    finally:
        for p in (eager, graph, warm):
            m.ssm_state_destroy(p)
