"""Seeded synthetic inputs for the Mamba-2 selective-state workloads.

This module is the only code that both the CPU oracle side (tests, the
oracle's timing leg of the benchmark) and the CUDA side consume.  It holds
none of the recurrence's arithmetic: only random draws with the
distributions the workloads fix, and the rounding of fp32 samples to bf16.

Distributions (the synthetic workloads of the Mamba-2 recurrence):
  x, B, C     ~ N(0, 1)
  dt          = softplus(v), v ~ N(-2, 0.5)      (dt arrives positive)
  A_h         = -exp(u),    u ~ U(0, 1.5)        (one scalar per head)
  D_h         ~ N(0, 1)                          (one scalar per head)
  init state  ~ N(0, 0.1)  (standard deviation 0.1)
  accept      = leading successes of T Bernoulli(p) draft checks, i.e. the
                drafts kept before the first rejected one (Why Speculative
                Decoding Slows Hybrid Mamba Models, Implementing It / Role 1:
                a step keeps its real token and the drafts up to the first
                rejection).

bf16 values are produced by round-to-nearest-even from fp32 samples and are
carried as uint16 bit patterns; ``bf16_to_f32`` widens them exactly.

Every draw is keyed by (seed, stream, index) through numpy's PCG64, so a
sampled slot or sequence can be regenerated on its own without generating
the whole workload.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202

# dtype codes shared by the library's C-ABI and the state blob format
# (SSM.PREFIX blob: 0 = fp32, 1 = fp16, 2 = bf16)
F32 = 0
BF16 = 2


def rng(*key: int) -> np.random.Generator:
    """A generator keyed by a tuple of non-negative integers."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even). Returns uint16 bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    # finite values stay below 2**32 after adding the bias; NaN is set below
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def widen(a: np.ndarray, dtype_code: int) -> np.ndarray:
    """Stored input -> exact fp64 values (uint16 arrays are bf16 patterns)."""
    if dtype_code == BF16:
        return bf16_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _store(a32: np.ndarray, dtype_code: int) -> np.ndarray:
    return f32_to_bf16(a32) if dtype_code == BF16 else np.ascontiguousarray(a32, dtype=np.float32)


def head_params(seed: int, H: int):
    """A[H] = -exp(U(0,1.5)) and D[H] ~ N(0,1), fp32."""
    g = rng(seed, 1)
    A = (-np.exp(g.uniform(0.0, 1.5, size=H))).astype(np.float32)
    D = g.standard_normal(H).astype(np.float32)
    return A, D


def tokens(seed: int, stream: int, n_tok: int, H: int, P: int, G: int, N: int,
           in_dtype: int = F32, dt_dtype: int = F32):
    """Per-token inputs for ``n_tok`` tokens of one stream.

    Returns (x [n_tok][H][P], dt [n_tok][H], B [n_tok][G][N], C [n_tok][G][N]),
    each fp32 or bf16 bit patterns according to the dtype codes.
    """
    g = rng(seed, 2, stream)
    x = g.standard_normal((n_tok, H, P), dtype=np.float32)
    v = g.normal(-2.0, 0.5, size=(n_tok, H)).astype(np.float64)
    dt = np.log1p(np.exp(v)).astype(np.float32)          # softplus
    Bm = g.standard_normal((n_tok, G, N), dtype=np.float32)
    Cm = g.standard_normal((n_tok, G, N), dtype=np.float32)
    return (_store(x, in_dtype), _store(dt, dt_dtype), _store(Bm, in_dtype), _store(Cm, in_dtype))


def batch_tokens(seed: int, step: int, batch: int, n_tok: int, H: int, P: int, G: int, N: int,
                 in_dtype: int = F32, dt_dtype: int = F32):
    """Inputs of one batched step: request r draws from stream (step, r).

    Returns arrays shaped [batch][n_tok][...]; with n_tok == 1 the caller may
    squeeze axis 1 for a decode step.
    """
    parts = [tokens(seed, step * 1_000_003 + r, n_tok, H, P, G, N, in_dtype, dt_dtype)
             for r in range(batch)]
    return tuple(np.stack([p[i] for p in parts]) for i in range(4))


def init_state(seed: int, slot: int, H: int, P: int, N: int, std: float = 0.1) -> np.ndarray:
    """Initial fp32 state of one slot, N(0, std), shaped [H][P][N]."""
    g = rng(seed, 3, slot)
    return (g.standard_normal((H, P, N), dtype=np.float32) * np.float32(std)).astype(np.float32)


def accept_counts(seed: int, steps: int, batch: int, T: int, p: float) -> np.ndarray:
    """Drafts accepted per request per verify step, int32 [steps][batch] in [0, T]."""
    g = rng(seed, 4)
    hits = g.random((steps, batch, T)) < p
    # leading run of successes: index of the first miss, or T if none
    miss = ~hits
    first_miss = np.where(miss.any(axis=2), miss.argmax(axis=2), T)
    return first_miss.astype(np.int32)


def varlen_lengths(seed: int, n_seq: int, lo: int, hi: int) -> np.ndarray:
    """Sequence lengths U(lo, hi) inclusive, int64 [n_seq]."""
    g = rng(seed, 5)
    return g.integers(lo, hi + 1, size=n_seq).astype(np.int64)


def random_partition(seed: int, stream: int, L: int, max_parts: int = 8, allow_empty: bool = True):
    """A seeded partition of L tokens into chunk lengths (may contain empty chunks)."""
    g = rng(seed, 6, stream)
    k = int(g.integers(1, max_parts + 1))
    cuts = np.sort(g.integers(0, L + 1, size=k - 1)) if k > 1 else np.array([], dtype=np.int64)
    bounds = np.concatenate([[0], cuts, [L]])
    parts = [int(b - a) for a, b in zip(bounds[:-1], bounds[1:])]
    if not allow_empty:
        parts = [q for q in parts if q > 0] or [L]
    return parts


# ---------------------------------------------------------------------------
# Gated delta rule (the second recurrence that unrolls as a decay plus a sum).
# Distributions of its synthetic workloads:
#   q, k   ~ N(0, 1) per key head, scaled to unit length (the layer normalizes
#            them before the recurrence), then stored in the input dtype
#   v      ~ N(0, 1)
#   g      = -softplus(N(-2, 0.5)) * exp(U(0, 1.5))   (log of the gate, <= 0)
#   beta   = sigmoid(N(0, 1))                          (writing strength)
#   state  ~ N(0, 0.1)

def gdn_tokens(seed: int, stream: int, n_tok: int, H: int, G: int, dk: int, dv: int, in_dtype: int = F32):
    """Per-token gated-delta-rule inputs of one stream.

    Returns (q [n_tok][G][dk], k [n_tok][G][dk], v [n_tok][H][dv], g [n_tok][H],
    beta [n_tok][H]); q, k, v fp32 or bf16 bit patterns, g and beta fp32.
    """
    r = rng(seed, 7, stream)
    q = r.standard_normal((n_tok, G, dk), dtype=np.float32)
    k = r.standard_normal((n_tok, G, dk), dtype=np.float32)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((n_tok, H, dv), dtype=np.float32)
    sp = np.log1p(np.exp(r.normal(-2.0, 0.5, size=(n_tok, H))))
    g = (-sp * np.exp(r.uniform(0.0, 1.5, size=(n_tok, H)))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-r.standard_normal((n_tok, H))))).astype(np.float32)
    return (_store(q, in_dtype), _store(k, in_dtype), _store(v, in_dtype), g, beta)


def gdn_batch_tokens(seed: int, step: int, batch: int, n_tok: int, H: int, G: int, dk: int, dv: int,
                     in_dtype: int = F32):
    """Inputs of one batched gated-delta-rule step, shaped [batch][n_tok][...]."""
    parts = [gdn_tokens(seed, step * 1_000_003 + r, n_tok, H, G, dk, dv, in_dtype) for r in range(batch)]
    return tuple(np.stack([p[i] for p in parts]) for i in range(5))


def gdn_init_state(seed: int, slot: int, H: int, dv: int, dk: int, std: float = 0.1) -> np.ndarray:
    """Initial fp32 gated-delta-rule state of one slot, N(0, std), shaped [H][dv][dk]."""
    r = rng(seed, 8, slot)
    return (r.standard_normal((H, dv, dk), dtype=np.float32) * np.float32(std)).astype(np.float32)
