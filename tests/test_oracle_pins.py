"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test fixes the oracle against something independent: a library routine
the recurrence reduces to (scipy.signal.lfilter, numpy.cumsum), a closed form
written out separately (the unrolled sum, the matrix "dual" form of Mamba-2),
the page's own scalar toy and printed numbers (tests/golden), and the
properties the pages require (chunk equivalence, reset independence, replay
exactness, declared ordering errors).
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.signal import lfilter

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            try:
                rows.append([float(v) for v in parts])
            except ValueError:
                out[parts[0]] = [float(v) for v in parts[1:]]
    return out, rows


def _toy_pool():
    """The Mamba-2 recurrence reduced to the page's scalar toy."""
    g, _ = _read_golden("page1_toy.txt")
    decay = g["decay"][0]
    A = np.array([math.log(decay)])
    return oracle.OraclePool(1, 1, 1, 1, n_slots=2, A=A, D=np.zeros(1)), g


def _toy_chunks(tokens):
    t = np.asarray(tokens, np.float64).reshape(-1, 1, 1)
    L = t.shape[0]
    return (t, np.ones((L, 1)), np.ones((L, 1, 1)), np.ones((L, 1, 1)))


def _scan_partition(pool, slot, x, dt, B, C, parts, reset_before=()):
    ys = []
    seq = 0
    for i, L in enumerate(parts):
        if i in reset_before:
            pool.reset([slot])
            seq = 0
        a = sum(parts[:i])
        st, y = pool.scan_chunk([slot], [seq], [(x[a:a + L], dt[a:a + L], B[a:a + L], C[a:a + L])])
        assert st == oracle.OK
        seq += 1
        ys.append(y[0])
    return np.concatenate(ys, axis=0)


# ---------------------------------------------------------------------------
# the page's scalar toy

def test_toy_matches_lfilter_and_page_properties():
    pool, g = _toy_pool()
    tok = g["tokens"]
    x, dt, B, C = _toy_chunks(tok)
    full = _scan_partition(pool, 0, x, dt, B, C, [len(tok)])[:, 0, 0]
    # library routine: y[n] = x[n] + decay * y[n-1]
    ref = lfilter([1.0], [1.0, -g["decay"][0]], np.asarray(tok))
    np.testing.assert_allclose(full, ref, rtol=1e-14, atol=0)
    st_full = pool.state[0].copy()
    assert pool.position[0] == len(tok)                     # position == token count

    pool.reset([0])
    parts = [int(v) for v in g["partition"]]
    chunked = _scan_partition(pool, 0, x, dt, B, C, parts)[:, 0, 0]
    assert np.array_equal(chunked, full)                    # chunked output == full
    assert np.array_equal(pool.state[0], st_full)           # chunked state == full

    pool.reset([0])
    lead_empty = _scan_partition(pool, 0, x, dt, B, C, [0, len(tok)])[:, 0, 0]
    assert np.array_equal(lead_empty, full)                 # leading empty chunk == full

    pool.reset([0])
    rp = [int(v) for v in g["reset_partition"]]
    with_reset = _scan_partition(pool, 0, x, dt, B, C, rp, reset_before=(1,))[:, 0, 0]
    assert not np.array_equal(with_reset, full)             # reset separates

    pool.reset([0])
    xs = np.concatenate([x[3:], x[:3]])
    swapped = _scan_partition(pool, 0, xs, dt, B, C, [6, 3])[:, 0, 0]
    assert not np.array_equal(swapped, full)                # swapped chunks differ

    pool.reset([0])
    bad = (np.array([[[1.0]], [[np.nan]]]), np.ones((2, 1)), np.ones((2, 1, 1)), np.ones((2, 1, 1)))
    st, _ = pool.scan_chunk([0], [0], [bad])
    assert st == oracle.ERR_INVALID_CHUNK                   # malformed input refused
    assert pool.position[0] == 0 and pool.next_chunk[0] == 0 and pool.state[0, 0, 0, 0] == 0

    rt = g["repeat_tokens"]
    xa, dta, Ba, Ca = _toy_chunks(rt)
    pool.reset([0, 1])
    a = _scan_partition(pool, 0, xa, dta, Ba, Ca, [int(v) for v in g["repeat_a"]])
    b = _scan_partition(pool, 1, xa, dta, Ba, Ca, [int(v) for v in g["repeat_b"]])
    assert np.array_equal(a, b) and np.array_equal(pool.state[0], pool.state[1])


# ---------------------------------------------------------------------------
# closed forms at full dimensionality

def _rand_problem(seed, L, H=3, P=5, N=4, G=1, init_std=0.3):
    r = synth.rng(seed, 99)
    A = -np.exp(r.uniform(0, 1.5, H))
    D = r.standard_normal(H)
    x = r.standard_normal((L, H, P))
    dt = np.log1p(np.exp(r.normal(-2, 0.5, (L, H))))
    B = r.standard_normal((L, G, N))
    C = r.standard_normal((L, G, N))
    h0 = r.standard_normal((H, P, N)) * init_std
    return A, D, x, dt, B, C, h0


def _unrolled(A, D, x, dt, B, C, h0):
    """h_t = (prod_{r<=t} dA_r) h_0 + sum_{s<=t} (prod_{s<r<=t} dA_r) dt_s x_s (x) B_s,
    y_t = C_t . h_t + D x_t, written with explicit products (no recurrence)."""
    L, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.zeros((L, H, P))
    hT = None
    for h in range(H):
        g = h // (H // G)
        dA = np.exp(dt[:, h] * A[h])
        for t in range(L):
            ht = np.prod(dA[:t + 1]) * h0[h]
            for s in range(t + 1):
                ht = ht + np.prod(dA[s + 1:t + 1]) * dt[s, h] * np.outer(x[s, h], B[s, g])
            y[t, h] = ht @ C[t, g] + D[h] * x[t, h]
        if hT is None:
            hT = np.zeros((H, P, N))
        hT[h] = ht
    return y, hT


@pytest.mark.parametrize("L", [1, 5, 9])
def test_every_partition_matches_unrolled_sum(L):
    A, D, x, dt, B, C, h0 = _rand_problem(L, L, H=2, P=3, N=4, G=2)
    y_ref, h_ref = _unrolled(A, D, x, dt, B, C, h0)
    H, P, N, G = 2, 3, 4, 2
    # every composition of L, each with an empty chunk inserted at the front
    for cuts in itertools.product([0, 1], repeat=L - 1):
        parts, cur = [], 1
        for c in cuts:
            if c:
                parts.append(cur)
                cur = 1
            else:
                cur += 1
        parts.append(cur)
        parts = [0] + parts
        pool = oracle.OraclePool(H, P, N, G, 1, A, D, init_state=h0[None])
        y = _scan_partition(pool, 0, x, dt, B, C, parts)
        np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(pool.state[0], h_ref, rtol=1e-12, atol=1e-13)
        assert pool.position[0] == L and pool.next_chunk[0] == len(parts)


def test_matrix_dual_form():
    """Mamba-2's matrix form: y = (Lmask o C B^T o dt) X + C (decayed h0) + D x,
    with Lmask[i,j] = exp(A * sum_{j<r<=i} dt_r) for j <= i, built with matmuls."""
    L, H, P, N, G = 48, 4, 8, 16, 2
    A, D, x, dt, B, C, h0 = _rand_problem(7, L, H, P, N, G)
    st = h0.copy()
    y = oracle.scan(st, x, dt, B, C, A, D)
    for h in range(H):
        g = h // (H // G)
        cum = np.cumsum(dt[:, h] * A[h])
        seg = cum[:, None] - cum[None, :]
        Lm = np.where(np.tril(np.ones((L, L), bool)), np.exp(np.where(np.tril(np.ones((L, L), bool)), seg, 0)), 0)
        M = Lm * (C[:, g] @ B[:, g].T) * dt[None, :, h]
        y_ref = M @ x[:, h] + np.exp(cum)[:, None] * (C[:, g] @ h0[h].T) + D[h] * x[:, h]
        np.testing.assert_allclose(y[:, h], y_ref, rtol=1e-11, atol=1e-12)
        S_ref = np.exp(cum[-1]) * h0[h] + (x[:, h] * (np.exp(cum[-1] - cum) * dt[:, h])[:, None]).T @ B[:, g]
        np.testing.assert_allclose(st[h], S_ref, rtol=1e-11, atol=1e-12)


def test_constant_coefficients_reduce_to_lfilter():
    """dt, B, C constant in time, zero initial state: every output channel is a
    first-order IIR filter of x with pole exp(dt A) and gain dt (C.B)."""
    L, H, P, N = 40, 3, 6, 8
    A, D, x, dt, B, C, _ = _rand_problem(11, L, H, P, N, 1)
    dt[:] = dt[0]
    B[:] = B[0]
    C[:] = C[0]
    st = np.zeros((H, P, N))
    y = oracle.scan(st, x, dt, B, C, A, D)
    for h in range(H):
        a = math.exp(dt[0, h] * A[h])
        gain = dt[0, h] * float(C[0, 0] @ B[0, 0])
        ref = gain * lfilter([1.0], [1.0, -a], x[:, h], axis=0) + D[h] * x[:, h]
        np.testing.assert_allclose(y[:, h], ref, rtol=1e-11, atol=1e-12)


def test_special_cases():
    L, H, P, N = 20, 2, 4, 8
    A, D, x, dt, B, C, h0 = _rand_problem(13, L, H, P, N, 1)
    # dt = 0: state unchanged bit for bit, y = C.h + D x
    st = h0.copy()
    y = oracle.scan(st, x, np.zeros_like(dt), B, C, A, D)
    assert np.array_equal(st, h0)
    for h in range(H):
        np.testing.assert_allclose(y[:, h], C[:, 0] @ h0[h].T + D[h] * x[:, h], rtol=1e-13, atol=1e-14)
    # A = 0: state is h0 plus the running sum of dt x (x) B
    st = h0.copy()
    oracle.scan(st, x, dt, B, C, np.zeros(H), D)
    for h in range(H):
        contrib = dt[:, h, None, None] * x[:, h, :, None] * B[:, 0, None, :]
        np.testing.assert_allclose(st[h], h0[h] + np.cumsum(contrib, axis=0)[-1], rtol=1e-12, atol=1e-13)
    # x = 0: pure decay, h_L = exp(A sum dt) h0
    st = h0.copy()
    oracle.scan(st, np.zeros_like(x), dt, B, C, A, D)
    for h in range(H):
        np.testing.assert_allclose(st[h], math.exp(A[h] * dt[:, h].sum()) * h0[h], rtol=1e-12, atol=0)


# ---------------------------------------------------------------------------
# lifecycle properties (Mamba Streaming State That Survives Chunking)

def _cfg0(seed=20261202):
    H, P, N, G, L = 2, 16, 16, 1, 64
    A, D = synth.head_params(seed, H)
    x, dt, B, C = synth.tokens(seed, 0, L, H, P, G, N)
    return (H, P, N, G, L), A, D, x, dt, B, C


def test_reset_independence_and_inequality_control():
    (H, P, N, G, L), A, D, x, dt, B, C = _cfg0()
    pa, pb = slice(0, 24), slice(24, L)
    pool = oracle.OraclePool(H, P, N, G, 3, A, D)
    # A; reset; B  versus  B from a fresh slot  versus  A then B without reset
    _scan_partition(pool, 0, x[pa], dt[pa], B[pa], C[pa], [24])
    pool.reset([0])
    yb_reset = _scan_partition(pool, 0, x[pb], dt[pb], B[pb], C[pb], [L - 24])
    yb_fresh = _scan_partition(pool, 1, x[pb], dt[pb], B[pb], C[pb], [L - 24])
    assert np.array_equal(yb_reset, yb_fresh) and np.array_equal(pool.state[0], pool.state[1])
    y_ab = _scan_partition(pool, 2, x, dt, B, C, [24, L - 24])[24:]
    assert np.max(np.abs(y_ab - yb_fresh)) > 1e-3
    assert pool.epoch[0] == 1 and pool.epoch[1] == 0


def test_chunk_order_declared_mismatch():
    (H, P, N, G, L), A, D, x, dt, B, C = _cfg0()
    pool = oracle.OraclePool(H, P, N, G, 2, A, D)
    ch = lambda a, b: (x[a:b], dt[a:b], B[a:b], C[a:b])
    assert pool.scan_chunk([0], [0], [ch(0, 7)])[0] == oracle.OK
    snap = pool.state[0].copy()
    assert pool.scan_chunk([0], [0], [ch(0, 7)])[0] == oracle.ERR_DUPLICATE    # applied twice
    assert pool.scan_chunk([0], [2], [ch(20, 33)])[0] == oracle.ERR_SEQUENCE   # gap
    assert np.array_equal(pool.state[0], snap) and pool.position[0] == 7 and pool.next_chunk[0] == 1
    # the arithmetic itself is order sensitive: applying the two chunks swapped differs
    y_ok = _scan_partition(oracle.OraclePool(H, P, N, G, 1, A, D), 0, x, dt, B, C, [7, 13, 43, 1])
    xs = np.concatenate([x[7:20], x[0:7], x[20:]])
    dts = np.concatenate([dt[7:20], dt[0:7], dt[20:]])
    Bs = np.concatenate([B[7:20], B[0:7], B[20:]])
    Cs = np.concatenate([C[7:20], C[0:7], C[20:]])
    y_sw = _scan_partition(oracle.OraclePool(H, P, N, G, 1, A, D), 0, xs, dts, Bs, Cs, [13, 7, 43, 1])
    assert np.max(np.abs(y_sw[20:] - y_ok[20:])) > 1e-3
    # a released slot refuses to advance until reset
    assert pool.release([0]) == oracle.OK
    assert pool.scan_chunk([0], [1], [ch(7, 9)])[0] == oracle.ERR_INVALID_STATE
    pool.reset([0])
    assert pool.scan_chunk([0], [0], [ch(0, 7)])[0] == oracle.OK


def test_partitions_of_tiny_config():
    """Config-sized check of the partitions the page lists: one-token chunks,
    an empty chunk, prime-sized chunks with a short final chunk."""
    (H, P, N, G, L), A, D, x, dt, B, C = _cfg0()
    ref_pool = oracle.OraclePool(H, P, N, G, 1, A, D)
    y_full = _scan_partition(ref_pool, 0, x, dt, B, C, [L])
    for parts in ([1] * L, [0, L], [32, 0, 32], [7, 13, 43, 1], [L, 0]):
        pool = oracle.OraclePool(H, P, N, G, 1, A, D)
        y = _scan_partition(pool, 0, x, dt, B, C, parts)
        np.testing.assert_allclose(y, y_full, rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(pool.state[0], ref_pool.state[0], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------------------
# replay versus copy (Why Speculative Decoding Slows Hybrid Mamba Models, The Fix:
# the two differ by less than 1e-12)

@pytest.mark.parametrize("W", [2, 3, 8])
def test_replay_equals_copy(W):
    H, P, N, G, R, T, steps = 4, 6, 8, 2, 3, 3, 9
    seed = 4242
    A, D = synth.head_params(seed, H)
    h0 = np.stack([synth.init_state(seed, s, H, P, N) for s in range(R)]).astype(np.float64)
    acc = synth.accept_counts(seed, steps, R, T, 0.6)
    copy = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.COPY, init_state=h0, max_tokens=T + 1)
    rep = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, init_state=h0, max_tokens=T + 1)
    # a sequential reference: apply exactly the committed tokens, one by one
    seq = h0.copy()
    slots = list(range(R))
    for s in range(steps):
        x, dt, B, C = (synth.widen(a, synth.F32) for a in synth.batch_tokens(seed, s, R, T + 1, H, P, G, N))
        st, yc = copy.verify(slots, x, dt, B, C)
        st2, yr = rep.verify(slots, x, dt, B, C)
        assert st == st2 == oracle.OK
        np.testing.assert_allclose(yr, yc, rtol=1e-12, atol=1e-12)
        for r in slots:
            for j in range(acc[s, r] + 1):   # outputs of kept tokens equal the sequential recurrence
                sub = seq[r:r + 1]
                ys = oracle.decode_step(sub, x[r:r + 1, j], dt[r:r + 1, j], B[r:r + 1, j], C[r:r + 1, j], A, D)
                seq[r] = sub[0]
                np.testing.assert_allclose(yc[r, j], ys[0], rtol=1e-12, atol=1e-12)
        copy.commit(slots, acc[s])
        st3, folded = rep.commit(slots, acc[s])
        assert st3 == oracle.OK
        np.testing.assert_array_equal(rep.position, copy.position)
        assert np.all(rep.log_len < W)
    rep.flush(slots)
    np.testing.assert_allclose(rep.state, copy.state, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(copy.state, seq, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(copy.position, (acc + 1).sum(axis=0))


@pytest.mark.parametrize("W", [1, 3, 4, 8])
def test_fold_in_verify_equals_fold_at_commit(W):
    """The deferred rule (a commit that fills the window leaves the log full,
    the next verify folds it first) gives the outputs of the at-commit rule
    and the sequential recurrence, and right after each verify its log holds
    what the at-commit pool's log holds: the fold only moves one call later
    (Why Speculative Decoding Slows Hybrid Mamba Models, The Fix)."""
    H, P, N, G, R, T, steps = 4, 6, 8, 2, 3, 3, 11
    seed = 4343
    A, D = synth.head_params(seed, H)
    h0 = np.stack([synth.init_state(seed, s, H, P, N) for s in range(R)]).astype(np.float64)
    acc = synth.accept_counts(seed, steps, R, T, 0.7)
    now = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, init_state=h0, max_tokens=T + 1)
    late = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.REPLAY, W=W, init_state=h0, max_tokens=T + 1,
                             fold_in_verify=True)
    copy = oracle.OraclePool(H, P, N, G, R, A, D, mode=oracle.COPY, init_state=h0, max_tokens=T + 1)
    slots = list(range(R))
    deferred = 0
    for s in range(steps):
        x, dt, B, C = (synth.widen(a, synth.F32) for a in synth.batch_tokens(seed, s, R, T + 1, H, P, G, N))
        _, yn = now.verify(slots, x, dt, B, C)
        _, yl = late.verify(slots, x, dt, B, C)
        _, yc = copy.verify(slots, x, dt, B, C)
        np.testing.assert_allclose(yl, yn, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(yl, yc, rtol=1e-12, atol=1e-12)
        np.testing.assert_array_equal(late.log_len, now.log_len)
        np.testing.assert_allclose(late.state, now.state, rtol=1e-12, atol=1e-12)
        now.commit(slots, acc[s])
        _, folded = late.commit(slots, acc[s])
        copy.commit(slots, acc[s])
        assert not folded.any()  # folds happen in the verify only
        assert np.all(late.log_len <= W - 1 + T + 1)
        deferred += int(np.sum(late.log_len >= W))
    assert deferred > 0, "no log filled the window"
    late.flush(slots)
    np.testing.assert_allclose(late.state, copy.state, rtol=1e-12, atol=1e-12)
    # a forced fold still folds at the commit
    x, dt, B, C = (synth.widen(a, synth.F32) for a in synth.batch_tokens(seed, steps, R, T + 1, H, P, G, N))
    late.verify(slots, x, dt, B, C)
    _, folded = late.commit(slots, [0] * R, force_fold=True)
    assert folded.all() and np.all(late.log_len == 0)


def test_fold_rule_is_exact_in_counts():
    """Plain decode through replay (one token per step) folds every W steps."""
    H, P, N, G, W = 2, 4, 4, 1, 5
    A, D = synth.head_params(1, H)
    rep = oracle.OraclePool(H, P, N, G, 1, A, D, mode=oracle.REPLAY, W=W, max_tokens=1)
    folds = []
    for s in range(3 * W):
        x, dt, B, C = (synth.widen(a, synth.F32) for a in synth.batch_tokens(1, s, 1, 1, H, P, G, N))
        rep.verify([0], x, dt, B, C)
        _, f = rep.commit([0], [0])
        folds.append(bool(f[0]))
    assert folds == [(s + 1) % W == 0 for s in range(3 * W)]
    # a forced fold empties the log at once
    x, dt, B, C = (synth.widen(a, synth.F32) for a in synth.batch_tokens(1, 99, 1, 1, H, P, G, N))
    rep.verify([0], x, dt, B, C)
    _, f = rep.commit([0], [0], force_fold=True)
    assert f[0] and rep.log_len[0] == 0


# ---------------------------------------------------------------------------
# the sizing rule and the acceptance generator

def test_copy_break_even_printed_values():
    _, rows = _read_golden("copy_rule.txt")
    for p, T, printed in rows:
        assert abs(oracle.copy_break_even(p, int(T)) - printed) <= 0.005
    # exact values of the geometric sum
    assert abs(oracle.expected_tokens_kept(0.6, 4) - 2.3056) < 1e-12
    assert abs(oracle.expected_tokens_kept(0.8, 4) - 3.3616) < 1e-12


@pytest.mark.parametrize("p,T", [(0.6, 4), (0.8, 4), (0.6, 8), (0.8, 8)])
def test_accept_generator_mean(p, T):
    a = synth.accept_counts(77, 64, 512, T, p)
    assert a.min() >= 0 and a.max() <= T
    kept = (a + 1).astype(np.float64)
    mu = oracle.expected_tokens_kept(p, T)
    sigma = kept.std() / math.sqrt(kept.size)
    assert abs(kept.mean() - mu) < 4 * sigma


def test_bf16_rounding():
    v = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e38, 1e-40], np.float32)
    b = synth.f32_to_bf16(v)
    w = synth.bf16_to_f32(b)
    assert w[0] == 1.0 and w[1] == 1.0          # halfway: ties to even (down)
    assert w[2] == np.float32(1.0078125)        # above halfway rounds up
    assert w[3] == -2.5
    r = synth.rng(5).standard_normal(10000).astype(np.float32)
    err = np.abs(synth.bf16_to_f32(synth.f32_to_bf16(r)) - r) / np.abs(r)
    assert err.max() <= 2.0 ** -8        # half an ulp of an 8-bit significand


# ---------------------------------------------------------------------------
# batched entry points against the matrix form (pins their indexing: request,
# token, head -> group, log entries)

def _dual_prefix(A, D, x, dt, B, C, h0):
    """Matrix form per head: outputs of every token and the state after every
    prefix, S_t = exp(cum_t) h0 + sum_{s<=t} exp(cum_t - cum_s) dt_s x_s (x) B_s."""
    L, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.zeros((L, H, P))
    S = np.zeros((L, H, P, N))
    low = np.tril(np.ones((L, L), bool))
    for h in range(H):
        g = h // (H // G)
        cum = np.cumsum(dt[:, h] * A[h])
        Lm = np.where(low, np.exp(np.where(low, cum[:, None] - cum[None, :], 0.0)), 0.0)
        M = Lm * (C[:, g] @ B[:, g].T) * dt[None, :, h]
        y[:, h] = M @ x[:, h] + np.exp(cum)[:, None] * (C[:, g] @ h0[h].T) + D[h] * x[:, h]
        for t in range(L):
            w = (Lm[t] * dt[:, h])[:, None]                       # zero for s > t
            S[t, h] = np.exp(cum[t]) * h0[h] + (x[:, h] * w).T @ B[:, g]
    return y, S


def test_batched_forms_match_matrix_form():
    H, P, N, G, R, T1 = 4, 5, 6, 2, 3, 4
    logs = [0, 2, 5]
    Wc = max(logs) + 1
    seqs = [_rand_problem(100 + r, logs[r] + T1, H, P, N, G) for r in range(R)]
    A, D = seqs[0][0], seqs[0][1]
    h0 = np.stack([s[6] for s in seqs])
    # token sequence of request r = its log entries followed by T1 step tokens
    xs = [s[2] for s in seqs]; dts = [s[3] for s in seqs]; Bs = [s[4] for s in seqs]; Cs = [s[5] for s in seqs]
    refs = [_dual_prefix(A, D, xs[r], dts[r], Bs[r], Cs[r], h0[r]) for r in range(R)]
    step = lambda a, r: a[r][logs[r]:logs[r] + T1]
    x = np.stack([step(xs, r) for r in range(R)]); dt = np.stack([step(dts, r) for r in range(R)])
    B = np.stack([step(Bs, r) for r in range(R)]); C = np.stack([step(Cs, r) for r in range(R)])
    lx = np.zeros((R, Wc, H, P)); ldt = np.zeros((R, Wc, H)); lB = np.zeros((R, Wc, G, N))
    for r in range(R):
        k = logs[r]
        lx[r, :k], ldt[r, :k], lB[r, :k] = xs[r][:k], dts[r][:k], Bs[r][:k]
    # replay: outputs from the checkpoint and the log
    y = oracle.verify_replay(h0, logs, lx, ldt, lB, x, dt, B, C, A, D)
    for r in range(R):
        np.testing.assert_allclose(y[r], refs[r][0][logs[r]:], rtol=1e-11, atol=1e-12)
    # fold of the log plus c step tokens lands on the state after that prefix
    c = np.array([1, 3, 4])
    ck = h0.copy()
    oracle.fold(ck, logs, c, [1, 1, 1], lx, ldt, lB, x, dt, B, A)
    for r in range(R):
        np.testing.assert_allclose(ck[r], refs[r][1][logs[r] + c[r] - 1], rtol=1e-11, atol=1e-12)
    # copy verify and decode from the state after each request's log
    base = np.stack([refs[r][1][logs[r] - 1] if logs[r] else h0[r] for r in range(R)])
    snap, yc = oracle.verify_copy(base, x, dt, B, C, A, D)
    st = base.copy()
    for r in range(R):
        np.testing.assert_allclose(yc[r], refs[r][0][logs[r]:], rtol=1e-11, atol=1e-12)
        for j in range(T1):
            np.testing.assert_allclose(snap[j, r], refs[r][1][logs[r] + j], rtol=1e-11, atol=1e-12)
    for j in range(T1):
        yd = oracle.decode_step(st, x[:, j], dt[:, j], B[:, j], C[:, j], A, D)
        for r in range(R):
            np.testing.assert_allclose(yd[r], refs[r][0][logs[r] + j], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(st[r], refs[r][1][logs[r] + j], rtol=1e-11, atol=1e-12)
