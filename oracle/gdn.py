"""CPU oracle for the gated delta rule, the second recurrence the replay
method applies to ("Why Speculative Decoding Slows Hybrid Mamba Models",
When the layer is a different kind of recurrence: the trick needs an update
that unrolls as a decay plus a sum, and Gated DeltaNet has one; the state
precision note of the same page names Gated DeltaNet layers).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU legs may import this
module.  It shares no code with the CUDA library and never imports it.

The pages name the recurrence but do not print it; this follows the gated
delta rule as its authors published it (Yang, Kautz and Hatamizadeh, Gated
Delta Networks), per value head h with key head g(h):

    S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
    o_t = S_t q_t

S is [dv][dk], alpha_t = exp(g_t) with the log-gate g_t <= 0 given per token
and value head, beta_t in (0, 1) likewise, q_t and k_t per key head (the
caller normalizes them), v_t per value head.  Key heads are contiguous
blocks: value head h reads key head h // (H / G).

Everything is fp64 numpy, one token at a time, in the order of the
definition.  Outputs come with their condition scale, cond_t[p] =
sum_k |S_t[p, k] q_t[k]|, the size of the terms whose sum is o_t[p], against
which the parity tests take their relative tolerance (``last_cond`` of the
pool after decode and verify).  Speculative verify is defined by its result: the outputs of the
step tokens run through the recurrence from the slot's full state (its
checkpoint with the logged tokens applied), which is what the replay form
must reproduce; commit appends the accepted tokens to the log, or applies
the log and them to the checkpoint when the window fills, as in the Mamba-2
pool (The Fix: the full state is written only then, and rejected drafts
never enter the log).
"""
from __future__ import annotations

import numpy as np


def key_head(h: int, H: int, G: int) -> int:
    """Key head of value head h: contiguous blocks of H / G value heads."""
    return h // (H // G)


def step(S: np.ndarray, q, k, v, g: float, beta: float, want_cond: bool = False):
    """One token of one head: returns (S_t, o_t) from S_{t-1} = S [dv][dk]
    (and with want_cond also the condition scale of o_t)."""
    S = np.asarray(S, np.float64)
    k = np.asarray(k, np.float64)
    alpha = np.exp(np.float64(g))
    # S (I - beta k k^T) = S - beta (S k) k^T
    Sk = S @ k
    S_new = alpha * (S - beta * np.outer(Sk, k)) + beta * np.outer(np.asarray(v, np.float64), k)
    o = S_new @ np.asarray(q, np.float64) if q is not None else None
    if want_cond:
        return S_new, o, (np.abs(S_new) @ np.abs(np.asarray(q, np.float64)) if q is not None else None)
    return S_new, o


def run_head(S0: np.ndarray, q, k, v, g, beta, want_cond: bool = False):
    """Tokens t = 0 .. T-1 of one head from S0: returns (S_T, o [T][dv]) (and cond [T][dv])."""
    S = np.array(S0, np.float64)
    outs, conds = [], []
    for t in range(len(g)):
        r = step(S, None if q is None else q[t], k[t], v[t], g[t], beta[t], want_cond=want_cond)
        S, o = r[0], r[1]
        outs.append(o)
        if want_cond:
            conds.append(r[2])
    o = np.stack(outs) if q is not None and outs else None
    if want_cond:
        return S, o, (np.stack(conds) if q is not None and conds else None)
    return S, o


def run(state: np.ndarray, q, k, v, g, beta, want_cond: bool = False):
    """All heads of one request: state [H][dv][dk]; q, k [T][G][dk]; v [T][H][dv];
    g, beta [T][H].  Returns (new state, o [T][H][dv]) and with want_cond cond [T][H][dv]."""
    H, G = state.shape[0], np.shape(k)[1]
    T = len(g)
    out_state = np.empty(state.shape, np.float64)
    o = np.empty((T, H, state.shape[1]), np.float64)
    cond = np.empty((T, H, state.shape[1]), np.float64)
    for h in range(H):
        kh = key_head(h, H, G)
        r = run_head(state[h], None if q is None else q[:, kh], k[:, kh], v[:, h], g[:, h], beta[:, h],
                     want_cond=want_cond)
        out_state[h] = r[0]
        if q is not None:
            o[:, h] = r[1]
            if want_cond:
                cond[:, h] = r[2]
    return (out_state, o, cond) if want_cond else (out_state, o)


class GdnOraclePool:
    """Slots of gated-delta-rule state with a replay log, mirroring the
    library's pool: decode in place (empty log), verify from the checkpoint
    and the log, commit by appending or folding."""

    def __init__(self, H, G, dk, dv, n_slots, W=16, max_tokens=9, init_state=None):
        self.H, self.G, self.dk, self.dv, self.W, self.max_tokens = H, G, dk, dv, W, max_tokens
        self.state = np.zeros((n_slots, H, dv, dk), np.float64) if init_state is None else \
            np.array(init_state, np.float64)
        self.log = [[] for _ in range(n_slots)]        # per slot: (k [G][dk], v [H][dv], g [H], beta [H])
        self.position = np.zeros(n_slots, np.int64)
        self.pending = {}                               # slot -> the last verify's step tokens
        self.last_cond = None                           # condition scale of the last outputs

    def _full(self, s):
        """The slot's state with its logged tokens applied."""
        st = self.state[s]
        if not self.log[s]:
            return st
        k, v, g, b = (np.stack([e[i] for e in self.log[s]]) for i in range(4))
        return run(st, None, k, v, g, b)[0]

    def decode(self, slots, q, k, v, g, beta):
        """One token per slot, in place; inputs [batch][...] (fp64)."""
        y = np.empty((len(slots), self.H, self.dv))
        cond = np.empty_like(y)
        for i, s in enumerate(slots):
            assert not self.log[s], "decode needs an empty log"
            self.state[s], o, c = run(self.state[s], q[i][None], k[i][None], v[i][None], g[i][None], beta[i][None],
                                      want_cond=True)
            y[i] = o[0]
            cond[i] = c[0]
            self.position[s] += 1
        self.last_cond = cond
        return y

    def verify(self, slots, q, k, v, g, beta):
        """n_tok step tokens per slot ([batch][n_tok][...]); outputs [batch][n_tok][H][dv]."""
        n_tok = len(g[0])
        y = np.empty((len(slots), n_tok, self.H, self.dv))
        cond = np.empty_like(y)
        for i, s in enumerate(slots):
            _, y[i], cond[i] = run(self._full(s), q[i], k[i], v[i], g[i], beta[i], want_cond=True)
            self.pending[s] = (k[i], v[i], g[i], beta[i])
        self.last_cond = cond
        return y

    def commit(self, slots, accept, force_fold=False):
        """Keep the real token and accept[i] drafts; returns the slots that folded."""
        folded = []
        for i, s in enumerate(slots):
            k, v, g, b = self.pending.pop(s)
            c = 1 + int(accept[i])
            kept = [(k[t], v[t], g[t], b[t]) for t in range(c)]
            self.position[s] += c
            if len(self.log[s]) + c < self.W and not force_fold:
                self.log[s].extend(kept)
            else:
                self.log[s].extend(kept)
                self.state[s] = self._full(s)
                self.log[s] = []
                folded.append(s)
        return folded

    def flush(self, slots):
        """Apply every slot's log to its checkpoint (as a forced fold would)."""
        for s in slots:
            self.state[s] = self._full(s)
            self.log[s] = []

    def log_len(self, s):
        return len(self.log[s])
