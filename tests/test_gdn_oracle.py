"""Pins of the gated-delta-rule oracle against what the mathematics fixes, not
against itself: closed forms, invariants and a brute-force unrolling.  Each
plausible slip in the oracle (the gate on the wrong term, the key projection
multiplied from the wrong side, a dropped or mis-signed write term, a wrong
product order) fails one of them.  The replay form the GPU path evaluates is
also restated here, on its own, and checked against the oracle's recurrence
(Why Speculative Decoding Slows Hybrid Mamba Models, The Fix and When the
layer is a different kind of recurrence: the update unrolls as a decay plus
a sum)."""
import numpy as np

import synth
from oracle import gdn

TOL = 1e-12


def _rand(seed, T, dk, dv, unit_k=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, dk))
    k = r.standard_normal((T, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = r.standard_normal((T, dv))
    g = -r.uniform(0.01, 0.7, T)
    b = r.uniform(0.05, 0.95, T)
    S0 = r.standard_normal((dv, dk)) * 0.3
    return S0, q, k, v, g, b


def test_no_write_is_a_pure_decay():
    """beta = 0: nothing is written, S_T = exp(sum g) S_0 and o_t = S_t q_t."""
    S0, q, k, v, g, _ = _rand(1, 7, 5, 4)
    S, o = gdn.run_head(S0, q, k, v, g, np.zeros(7))
    assert np.allclose(S, np.exp(g.sum()) * S0, rtol=TOL, atol=TOL)
    for t in range(7):
        assert np.allclose(o[t], np.exp(g[:t + 1].sum()) * S0 @ q[t], rtol=TOL, atol=TOL)


def test_full_write_stores_the_value_at_its_key():
    """No decay and beta = 1 with a unit key: the delta rule replaces what the
    key read with v, so S_t k_t = v_t after every token."""
    S0, q, k, v, _, _ = _rand(2, 9, 6, 5)
    S = S0
    for t in range(9):
        S, _ = gdn.step(S, None, k[t], v[t], 0.0, 1.0)
        assert np.allclose(S @ k[t], v[t], rtol=TOL, atol=TOL)


def test_orthonormal_keys_closed_form():
    """Orthonormal keys, no decay, beta = 1: S_T = S_0 (I - sum k k^T) + sum v k^T,
    and from a zero state each key retrieves its own value."""
    r = np.random.default_rng(3)
    dk, dv, T = 8, 5, 5
    Qm, _ = np.linalg.qr(r.standard_normal((dk, dk)))
    k = Qm[:, :T].T
    v = r.standard_normal((T, dv))
    S0 = r.standard_normal((dv, dk))
    S, _ = gdn.run_head(S0, None, k, v, np.zeros(T), np.ones(T))
    want = S0 @ (np.eye(dk) - k.T @ k) + v.T @ k
    assert np.allclose(S, want, rtol=1e-12, atol=1e-12)
    Z, _ = gdn.run_head(np.zeros((dv, dk)), None, k, v, np.zeros(T), np.ones(T))
    for t in range(T):
        assert np.allclose(Z @ k[t], v[t], atol=1e-12)


def test_scalar_case_geometric_series():
    """dk = dv = 1 with constant inputs: s_t = a s_{t-1} + c with a = exp(g)(1 - beta k^2)
    and c = beta v k, so s_T = a^T s_0 + c (1 - a^T) / (1 - a)."""
    kk, vv, g, b, s0, T = 0.8, -1.3, -0.2, 0.6, 0.7, 11
    S, o = gdn.run_head(np.array([[s0]]), np.full((T, 1), 0.5), np.full((T, 1), kk), np.full((T, 1), vv),
                        np.full(T, g), np.full(T, b))
    a, c = np.exp(g) * (1 - b * kk * kk), b * vv * kk
    assert abs(S[0, 0] - (a ** T * s0 + c * (1 - a ** T) / (1 - a))) < 1e-13
    s3 = a ** 3 * s0 + c * (1 - a ** 3) / (1 - a)
    assert abs(o[2, 0] - 0.5 * s3) < 1e-13


def test_brute_force_matrix_product_unrolling():
    """S_m = S_0 A_1 ... A_m + sum_s beta_s v_s k_s^T A_{s+1} ... A_m with the
    explicit matrices A_i = exp(g_i) (I - beta_i k_i k_i^T), keys not unit."""
    S0, q, k, v, g, b = _rand(4, 6, 4, 3, unit_k=False)
    dk = 4
    A = [np.exp(g[i]) * (np.eye(dk) - b[i] * np.outer(k[i], k[i])) for i in range(6)]
    S, o = gdn.run_head(S0, q, k, v, g, b)
    for m in range(1, 7):
        P = np.eye(dk)
        for i in range(m):
            P = P @ A[i]
        Sm = S0 @ P
        for s in range(m):
            R = np.eye(dk)
            for i in range(s + 1, m):
                R = R @ A[i]
            Sm = Sm + b[s] * np.outer(v[s], k[s]) @ R
        assert np.allclose(o[m - 1], Sm @ q[m - 1], rtol=1e-12, atol=1e-12)
    assert np.allclose(S, Sm, rtol=1e-12, atol=1e-12)


def replay_outputs(S_c, k_all, v_all, g_all, b_all, q_steps, K):
    """The replay form, restated from the unrolling: for the output at position
    m (1-based over the K logged tokens then the step tokens), start from
    u = q_m and walk i = m .. 1: the log term of v_i has weight beta_i (k_i . u),
    then u <- exp(g_i) (u - beta_i k_i (k_i . u)); the checkpoint term is
    S_c u at the end.  No state is formed."""
    out = []
    for j, qj in enumerate(q_steps):
        m = K + j + 1
        u = np.array(qj, np.float64)
        acc = np.zeros(v_all.shape[1])
        for i in range(m - 1, -1, -1):
            t = k_all[i] @ u
            acc += b_all[i] * t * v_all[i]
            u = np.exp(g_all[i]) * (u - b_all[i] * t * k_all[i])
        out.append(S_c @ u + acc)
    return np.stack(out)


def test_replay_form_equals_the_recurrence():
    """Outputs from a checkpoint and K logged tokens, by the replay form, equal
    the recurrence run through the log and then the step tokens."""
    for K, T1 in ((0, 1), (0, 5), (3, 4), (11, 9)):
        S0, q, k, v, g, b = _rand(10 + K, K + T1, 16, 12)
        _, o = gdn.run_head(S0, q, k, v, g, b)
        got = replay_outputs(S0, k, v, g, b, q[K:], K)
        assert np.allclose(got, o[K:], rtol=1e-11, atol=1e-12), K


def test_chunked_wy_fold_equals_the_recurrence():
    """The fold in the chunked (WY) form the tensor-core kernel evaluates,
    restated here on its own in fp64: with G_t the running sum of the gates,
    S_M = e^{G_{M-1}} S + Y P, Y[:, t] = b_t v_t - b_t e^{G_t} S k_t,
    P = (I + A)^{-1} D K, A[s][t] = b_t e^{G_t - G_s} (k_s . k_t) for s < t,
    D = diag(e^{G_{M-1} - G_s}).  It must equal the oracle's token-by-token
    recurrence for any window length, including one token, 32 and a gate
    near zero; a transposed A or a D taken from the start fails it."""
    for seed, M in ((21, 1), (22, 2), (23, 7), (24, 24), (25, 32)):
        S0, _, k, v, g, b = _rand(seed, M, 9, 6)
        if M >= 7:
            g[3] = -40.0  # a gate near zero
        want, _ = gdn.run_head(S0, None, k, v, g, b)
        G = np.cumsum(g)
        A = np.zeros((M, M))
        for s_ in range(M):
            for t in range(s_ + 1, M):
                A[s_, t] = b[t] * np.exp(G[t] - G[s_]) * (k[s_] @ k[t])
        D = np.exp(G[-1] - G)
        P = np.linalg.solve(np.eye(M) + A, D[:, None] * k)
        Y = v.T * b - (S0 @ k.T) * (b * np.exp(G))
        got = np.exp(G[-1]) * S0 + Y @ P
        assert np.allclose(got, want, rtol=1e-11, atol=1e-11), (seed, M)
        # the pins above are sharp: A transposed, or D measured from the first token, give another state
        if M >= 2:
            bad = np.exp(G[-1]) * S0 + Y @ np.linalg.solve(np.eye(M) + A.T, D[:, None] * k)
            assert not np.allclose(bad, want, rtol=1e-6, atol=1e-6)
            bad = np.exp(G[-1]) * S0 + Y @ np.linalg.solve(np.eye(M) + A, np.exp(G - G[0])[:, None] * k)
            assert not np.allclose(bad, want, rtol=1e-6, atol=1e-6)


def test_pool_commit_keeps_only_accepted_tokens():
    """Through verify / commit with folds at different points, every output and
    the final state equal one sequential run over the accepted tokens alone
    (rejected drafts never enter the log)."""
    H, G, dk, dv, T1, W = 4, 2, 8, 6, 4, 5
    init = np.stack([synth.gdn_init_state(5, s, H, dv, dk) for s in range(2)]).astype(np.float64)
    pool = gdn.GdnOraclePool(H, G, dk, dv, 2, W=W, max_tokens=T1, init_state=init)
    acc = synth.accept_counts(6, 7, 2, T1 - 1, 0.6)
    ref = init.copy()
    folds = 0
    for s in range(7):
        q, k, v, g, b = (synth.widen(a, c) for a, c in zip(
            synth.gdn_batch_tokens(7, s, 2, T1, H, G, dk, dv, synth.F32), (0, 0, 0, 0, 0)))
        y = pool.verify([0, 1], q, k, v, g, b)
        folds += len(pool.commit([0, 1], acc[s], force_fold=(s == 4)))
        for r in range(2):
            c = 1 + int(acc[s][r])
            ref[r], o = gdn.run(ref[r], q[r, :c], k[r, :c], v[r, :c], g[r, :c], b[r, :c])
            assert np.allclose(y[r, :c], o, rtol=1e-12, atol=1e-12), (s, r)
    assert folds > 0
    pool.flush([0, 1])
    assert np.allclose(pool.state, ref, rtol=1e-12, atol=1e-12)
    assert list(pool.position) == [7 + int(acc[:, r].sum()) for r in range(2)]


def test_input_recipe():
    """The synthetic gated-delta-rule inputs have the distributions the recipe
    states: unit q and k per key head (up to bf16 rounding when stored so),
    a log-gate g <= 0, beta in (0, 1), and the stated shapes and storage."""
    for code, tol in ((synth.F32, 1e-6), (synth.BF16, 1e-2)):
        q, k, v, g, b = synth.gdn_batch_tokens(11, 0, 3, 5, 8, 4, 64, 32, code)
        assert q.shape == k.shape == (3, 5, 4, 64) and v.shape == (3, 5, 8, 32)
        assert g.shape == b.shape == (3, 5, 8) and g.dtype == b.dtype == np.float32
        assert q.dtype == (np.uint16 if code == synth.BF16 else np.float32)
        for a in (q, k):
            n = np.linalg.norm(synth.widen(a, code), axis=-1)
            assert np.all(np.abs(n - 1.0) < tol)
        assert np.all(g < 0) and np.all(g > -20)
        assert np.all((b > 0) & (b < 1))
    s = synth.gdn_init_state(3, 0, 8, 32, 64)
    assert s.shape == (8, 32, 64) and abs(float(s.std()) - 0.1) < 0.01
