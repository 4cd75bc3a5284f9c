"""Pins of the oracle's condition scale and of its fp32 instantiation.

The condition scale of an output y_t[p] = sum_n C_t[n] h_t[p, n] + D x_t[p]
is sum_n |C_t[n] h_t[p, n]| + |D x_t[p]|: the size of the terms whose sum is
y, against which a result computed in finite precision is judged.  Here it
is recomputed from states written out token by token in numpy (the
recurrence as the pages state it: decay by exp(dt A), then add
dt x (x) B), for every form of the computation that has outputs.  The fp32
instantiation of the same source, used only as the CPU speed baseline, must
agree with the fp64 oracle to within fp32 rounding.
"""
import numpy as np

import oracle
import synth

SEED = synth.BASE_SEED + 8100


def _states(h0, x, dt, B, A):
    """States after each token of one (sequence, head), by the recurrence."""
    h = h0.copy()
    out = []
    for t in range(x.shape[0]):
        h = np.exp(dt[t] * A) * h + dt[t] * np.outer(x[t], B[t])
        out.append(h.copy())
    return out


def _cond(hs, C, D, x):
    return np.stack([np.abs(C[t][None, :] * hs[t]).sum(axis=1) + np.abs(D * x[t]) for t in range(len(hs))])


def _tiny(L=7, H=4, P=3, N=5, G=2):
    x, dt, B, C = (np.asarray(a, np.float64) for a in synth.tokens(SEED, 0, L, H, P, G, N))
    A, D = (np.asarray(a, np.float64) for a in synth.head_params(SEED, H))
    h0 = np.stack([synth.init_state(SEED, s, H, P, N) for s in range(2)]).astype(np.float64)
    return x, dt, B, C, A, D, h0


def test_scan_cond_is_the_term_size():
    x, dt, B, C, A, D, h0 = _tiny()
    L, H, P = x.shape
    G = B.shape[1]
    st = h0[0].copy()
    y, cond = oracle.scan(st, x, dt, B, C, A, D, want_cond=True)
    for h in range(H):
        g = h // (H // G)
        hs = _states(h0[0, h], x[:, h], dt[:, h], B[:, g], A[h])
        np.testing.assert_allclose(cond[:, h], _cond(hs, C[:, g], D[h], x[:, h]), rtol=1e-13, atol=0)
        yy = np.stack([hs[t] @ C[t, g] + D[h] * x[t, h] for t in range(L)])
        np.testing.assert_allclose(y[:, h], yy, rtol=1e-12, atol=1e-14)
    assert np.all(cond >= np.abs(y) * (1 - 1e-15))
    # equality when every term has one sign: C, h >= 0 and D x >= 0
    st = np.abs(h0[0]).copy()
    y2, c2 = oracle.scan(st, np.abs(x), dt, np.abs(B), np.abs(C), A, np.abs(D), want_cond=True)
    np.testing.assert_allclose(c2, y2, rtol=1e-14)


def test_decode_and_copy_verify_cond():
    x, dt, B, C, A, D, h0 = _tiny()
    H, G = x.shape[1], B.shape[1]
    R, T1 = 2, 3
    xs = np.stack([x[0:T1], x[3:3 + T1]])  # [R][T1][H][P]
    dts, Bs, Cs = (np.stack([a[0:T1], a[3:3 + T1]]) for a in (dt, B, C))
    st = h0.copy()
    y, cond = oracle.decode_step(st, xs[:, 0], dts[:, 0], Bs[:, 0], Cs[:, 0], A, D, want_cond=True)
    _, yc, condc = oracle.verify_copy(h0, xs, dts, Bs, Cs, A, D, want_cond=True)
    for r in range(R):
        for h in range(H):
            g = h // (H // G)
            hs = _states(h0[r, h], xs[r, :, h], dts[r, :, h], Bs[r, :, g], A[h])
            ref = _cond(hs, Cs[r, :, g], D[h], xs[r, :, h])
            np.testing.assert_allclose(cond[r, h], ref[0], rtol=1e-13)
            np.testing.assert_allclose(condc[r, :, h], ref, rtol=1e-13)
    np.testing.assert_array_equal(yc[:, 0], y)


def test_replay_cond_walks_the_log_then_the_step():
    """Replay's scale is that of the state after the logged tokens and then
    the step tokens, the same state the copy flavour would hold."""
    x, dt, B, C, A, D, h0 = _tiny(L=7)
    H, G = x.shape[1], B.shape[1]
    k, T1 = 4, 3
    Wc = 8
    lx = np.zeros((1, Wc) + x.shape[1:])
    ldt = np.zeros((1, Wc, H))
    lB = np.zeros((1, Wc) + B.shape[1:])
    lx[0, :k], ldt[0, :k], lB[0, :k] = x[:k], dt[:k], B[:k]
    y, cond = oracle.verify_replay(h0[:1], [k], lx, ldt, lB, x[None, k:k + T1], dt[None, k:k + T1],
                                   B[None, k:k + T1], C[None, k:k + T1], A, D, want_cond=True)
    for h in range(H):
        g = h // (H // G)
        hs = _states(h0[0, h], x[:k + T1, h], dt[:k + T1, h], B[:k + T1, g], A[h])[k:]
        np.testing.assert_allclose(cond[0, :, h], _cond(hs, C[k:k + T1, g], D[h], x[k:k + T1, h]), rtol=1e-13)
        np.testing.assert_allclose(y[0, :, h], np.stack([hs[j] @ C[k + j, g] + D[h] * x[k + j, h] for j in range(T1)]),
                                   rtol=1e-11, atol=1e-13)


def test_fp32_instantiation_agrees_to_fp32_rounding():
    """The speed-baseline build runs the same loops in fp32: outputs within a
    few fp32 ulps of the condition scale, states within fp32 rounding."""
    x, dt, B, C, A, D, h0 = _tiny(L=7, H=4, P=8, N=16)
    R, T1 = 2, 3
    xs = np.stack([x[0:T1], x[3:3 + T1]])
    dts, Bs, Cs = (np.stack([a[0:T1], a[3:3 + T1]]) for a in (dt, B, C))
    st64 = h0.copy()
    y64, cond = oracle.decode_step(st64, xs[:, 0], dts[:, 0], Bs[:, 0], Cs[:, 0], A, D, want_cond=True)
    st32 = h0.astype(np.float32)
    y32 = oracle.f32_decode_step(st32, xs[:, 0], dts[:, 0], Bs[:, 0], Cs[:, 0], A, D)
    assert y32.dtype == np.float32 and st32.dtype == np.float32
    assert np.all(np.abs(y32 - y64) <= 1e-5 * cond)
    assert np.all(np.abs(st32 - st64) <= 1e-5 * (np.abs(st64) + 1e-3))
    snap64, yc64, condc = oracle.verify_copy(h0, xs, dts, Bs, Cs, A, D, want_cond=True)
    snap32, yc32 = oracle.f32_verify_copy(h0, xs, dts, Bs, Cs, A, D)
    assert np.all(np.abs(yc32 - yc64) <= 1e-5 * condc)
    assert np.all(np.abs(snap32 - snap64) <= 1e-5 * (np.abs(snap64) + 1e-3))
    k, Wc = 2, 6
    lx = np.zeros((R, Wc) + x.shape[1:])
    ldt = np.zeros((R, Wc, x.shape[1]))
    lB = np.zeros((R, Wc) + B.shape[1:])
    for r in range(R):
        lx[r, :k], ldt[r, :k], lB[r, :k] = x[r:r + k], dt[r:r + k], B[r:r + k]
    yr64, condr = oracle.verify_replay(h0, [k, k], lx, ldt, lB, xs, dts, Bs, Cs, A, D, want_cond=True)
    yr32 = oracle.f32_verify_replay(h0, [k, k], lx, ldt, lB, xs, dts, Bs, Cs, A, D)
    assert np.all(np.abs(yr32 - yr64) <= 1e-5 * condr)


def test_gdn_cond_is_the_term_size():
    """Gated delta rule: the scale of o_t[p] = sum_k S_t[p, k] q_t[k] is
    sum_k |S_t[p, k] q_t[k]|, with S_t recomputed here token by token."""
    from oracle import gdn
    rng = np.random.default_rng(SEED)
    H, G, dk, dv, T = 4, 2, 6, 5, 4
    S0 = rng.normal(size=(H, dv, dk)) * 0.1
    q = rng.normal(size=(T, G, dk))
    k = rng.normal(size=(T, G, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.normal(size=(T, H, dv))
    g = -np.abs(rng.normal(size=(T, H)))
    beta = 1 / (1 + np.exp(-rng.normal(size=(T, H))))
    _, o, cond = gdn.run(S0, q, k, v, g, beta, want_cond=True)
    for h in range(H):
        kh = h // (H // G)
        S = S0[h].copy()
        for t in range(T):
            S = np.exp(g[t, h]) * (S - beta[t, h] * np.outer(S @ k[t, kh], k[t, kh])) + \
                beta[t, h] * np.outer(v[t, h], k[t, kh])
            np.testing.assert_allclose(cond[t, h], np.abs(S * q[t, kh][None, :]).sum(axis=1), rtol=1e-13)
            np.testing.assert_allclose(o[t, h], S @ q[t, kh], rtol=1e-12, atol=1e-15)
    assert np.all(cond >= np.abs(o) * (1 - 1e-15))
