"""CPU oracle for the Mamba-2 selective-state recurrence.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline / reference leg
may import this package.  It shares no code with the CUDA library and never
imports it.

The arithmetic lives in ``ssm_oracle.c`` (plain fp64 scalar loops); this
module compiles it with gcc on first use, marshals numpy arrays, and models
the pool's lifecycle rules on the host.  The same source also builds with
every value in fp32 (``f32_*`` functions below): that build serves only as the
CPU speed baseline, never as a parity reference.  Functions that return
outputs y can also return their condition scale ``cond`` (sum over n of
|C[n] h[p, n]| plus |D x[p]|, h the state after the token), against which the
parity tests take their relative tolerance:

* ``OraclePool`` follows the streaming-state contract of "Mamba Streaming
  State That Survives Chunking": separate init / reset / checkpoint /
  release operations (Make reset, checkpoint, and cancellation observable),
  a monotone chunk sequence where a repeated number is a duplicate and a gap
  is an ordering error (Let the full scan define legal chunking), and empty
  chunks that consume a sequence number without touching state.
* Copy-mode verify keeps a full state after every step token and commit
  selects the one after the last accepted token; replay-mode verify computes
  outputs from the checkpoint and the input log, and commit appends the
  accepted tokens or folds them into the checkpoint when the window fills
  ("Why Speculative Decoding Slows Hybrid Mamba Models", The Fix).

All floating-point state is fp64.  Inputs are widened exactly from their
stored fp32 / bf16 values by the caller (see ``synth.widen``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATHS = {"f64": os.path.join(_OUT_DIR, "libssm_oracle.so"),
              "f32": os.path.join(_OUT_DIR, "libssm_oracle_f32.so")}
_lock = threading.Lock()
_libs = {}

# status codes mirrored by the pool model (same meaning as the library's)
OK, ERR_INVALID_ARG, ERR_INVALID_CHUNK, ERR_INVALID_STATE, ERR_SEQUENCE, ERR_DUPLICATE = 0, 1, 2, 3, 4, 5

COPY, REPLAY = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, OpenMP): the fp64
    parity oracle and the fp32 instantiation of the same source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    for prec, path in _LIB_PATHS.items():
        if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            tmp = path + ".tmp%d" % os.getpid()
            extra = ["-DORACLE_F32"] if prec == "f32" else []
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                                   "-ffp-contract=off", "-fno-fast-math", *extra, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, path)
    return _LIB_PATHS["f64"]


def lib(prec: str = "f64"):
    with _lock:
        if prec not in _libs:
            build()
            L = ctypes.CDLL(_LIB_PATHS[prec])
            d = ctypes.c_double if prec == "f64" else ctypes.c_float
            i, l = ctypes.c_int, ctypes.c_long
            P_ = ctypes.c_void_p
            L.oracle_scan_head.argtypes = [i, i, l, d, d, P_, l, P_, l, P_, P_, l, P_, P_, l, P_]
            L.oracle_decode_step.argtypes = [i, i, i, i, i, P_, P_, P_, P_, P_, P_, P_, P_, P_]
            L.oracle_verify_copy.argtypes = [i, i, i, i, i, i, P_, P_, P_, P_, P_, P_, P_, P_, P_, P_]
            L.oracle_replay_head.argtypes = [i, i, i, i, d, d, P_, P_, P_, P_, P_, P_, P_]
            L.oracle_verify_replay.argtypes = [i, i, i, i, i, i, i, P_, P_, P_, P_, P_,
                                               P_, P_, P_, P_, P_, P_, P_, P_]
            L.oracle_fold.argtypes = [i, i, i, i, i, i, i, P_, P_, P_, P_, P_, P_, P_, P_, P_, P_, P_]
            for f in ("oracle_scan_head", "oracle_decode_step", "oracle_verify_copy",
                      "oracle_replay_head", "oracle_verify_replay", "oracle_fold"):
                getattr(L, f).restype = None
            L.oracle_max_threads.restype = ctypes.c_int
            L.oracle_set_threads.argtypes = [i]
            L.oracle_set_threads.restype = None
            L.oracle_real_bytes.restype = ctypes.c_int
            assert L.oracle_real_bytes() == (8 if prec == "f64" else 4)
            _libs[prec] = L
    return _libs[prec]


def threads() -> int:
    return int(lib().oracle_max_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def group_of(h: int, H: int, G: int) -> int:
    """Head -> group map: contiguous blocks of H/G heads."""
    return h // (H // G)


# ---------------------------------------------------------------------------
# the recurrence in its forms

def scan_head(state: np.ndarray, x, dt, B, C, A: float, D: float, want_y: bool = True, want_cond: bool = False):
    """Sequential recurrence of one (sequence, head).

    state [P][N] (updated in place, fp64); x [L][P]; dt [L]; B, C [L][N].
    Returns y [L][P] (or None), and with want_cond (y, cond).
    """
    x, dt, B, C = _f64(x), _f64(dt), _f64(B), _f64(C)
    L, P = x.shape
    N = B.shape[1]
    assert state.dtype == np.float64 and state.flags.c_contiguous and state.shape == (P, N)
    y = np.empty((L, P), np.float64) if want_y else None
    cond = np.empty((L, P), np.float64) if want_cond else None
    lib().oracle_scan_head(P, N, L, float(A), float(D), _ptr(x), P, _ptr(dt), 1,
                           _ptr(B), _ptr(C), N, _ptr(state), _ptr(y) if want_y else None, P,
                           _ptr(cond) if want_cond else None)
    return (y, cond) if want_cond else y


def scan(state: np.ndarray, x, dt, B, C, A, D, want_cond: bool = False):
    """Sequential recurrence of one sequence, all heads.

    state [H][P][N] fp64 in/out; x [L][H][P]; dt [L][H]; B, C [L][G][N];
    A, D [H].  Returns y [L][H][P], and with want_cond (y, cond).
    """
    x, dt, B, C = _f64(x), _f64(dt), _f64(B), _f64(C)
    L, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    y = np.empty((L, H, P), np.float64)
    cond = np.empty((L, H, P), np.float64) if want_cond else None

    def one(h):  # heads are independent: one C call each, spread over threads (no change to any result)
        g = group_of(h, H, G)
        st = np.ascontiguousarray(state[h])
        r = scan_head(st, x[:, h, :], dt[:, h], B[:, g, :], C[:, g, :], A[h], D[h], want_cond=want_cond)
        if want_cond:
            y[:, h, :], cond[:, h, :] = r
        else:
            y[:, h, :] = r
        state[h] = st

    if H > 1 and L * P * N > (1 << 16):
        import concurrent.futures as cf
        with cf.ThreadPoolExecutor(max_workers=min(H, os.cpu_count() or 1)) as ex:
            list(ex.map(one, range(H)))
    else:
        for h in range(H):
            one(h)
    return (y, cond) if want_cond else y


def decode_step(state: np.ndarray, x, dt, B, C, A, D, want_cond: bool = False):
    """One token for R requests. state [R][H][P][N] fp64 in/out; returns y [R][H][P] (and cond)."""
    assert state.dtype == np.float64 and state.flags.c_contiguous
    x, dt, B, C, A, D = _f64(x), _f64(dt), _f64(B), _f64(C), _f64(A), _f64(D)
    R, H, P, N = state.shape
    G = B.shape[1]
    y = np.empty((R, H, P), np.float64)
    cond = np.empty((R, H, P), np.float64) if want_cond else None
    lib().oracle_decode_step(R, H, P, N, G, _ptr(state), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                             _ptr(A), _ptr(D), _ptr(y), _ptr(cond) if want_cond else None)
    return (y, cond) if want_cond else y


def verify_copy(state: np.ndarray, x, dt, B, C, A, D, want_cond: bool = False):
    """Copy verify. state [R][H][P][N]; x [R][T1][H][P] ...

    Returns (snapshots [T1][R][H][P][N], y [R][T1][H][P]) and with want_cond
    also cond [R][T1][H][P].
    """
    state = _f64(state)
    x, dt, B, C, A, D = _f64(x), _f64(dt), _f64(B), _f64(C), _f64(A), _f64(D)
    R, H, P, N = state.shape
    T1, G = x.shape[1], B.shape[2]
    snap = np.empty((T1, R, H, P, N), np.float64)
    y = np.empty((R, T1, H, P), np.float64)
    cond = np.empty((R, T1, H, P), np.float64) if want_cond else None
    lib().oracle_verify_copy(R, T1, H, P, N, G, _ptr(state), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                             _ptr(A), _ptr(D), _ptr(snap), _ptr(y), _ptr(cond) if want_cond else None)
    return (snap, y, cond) if want_cond else (snap, y)


def replay_head(hc, ux, udt, uB, Cq, k: int, A: float, D: float, want_cond: bool = False):
    """ReplaySSM closed form for one (request, head); see ssm_oracle.c."""
    hc, ux, udt, uB, Cq = _f64(hc), _f64(ux), _f64(udt), _f64(uB), _f64(Cq)
    P, N = hc.shape
    n_tok = Cq.shape[0]
    assert ux.shape == (k + n_tok, P) and uB.shape == (k + n_tok, N)
    y = np.empty((n_tok, P), np.float64)
    cond = np.empty((n_tok, P), np.float64) if want_cond else None
    lib().oracle_replay_head(P, N, k, n_tok, float(A), float(D), _ptr(hc), _ptr(ux), _ptr(udt),
                             _ptr(uB), _ptr(Cq), _ptr(y), _ptr(cond) if want_cond else None)
    return (y, cond) if want_cond else y


def verify_replay(ckpt, log_len, lx, ldt, lB, x, dt, B, C, A, D, want_cond: bool = False):
    """Replay verify over R requests; returns y [R][T1][H][P] (and cond)."""
    ckpt = _f64(ckpt)
    log_len = np.ascontiguousarray(log_len, dtype=np.int32)
    lx, ldt, lB = _f64(lx), _f64(ldt), _f64(lB)
    x, dt, B, C, A, D = _f64(x), _f64(dt), _f64(B), _f64(C), _f64(A), _f64(D)
    R, H, P, N = ckpt.shape
    T1, G, Wc = x.shape[1], B.shape[2], lx.shape[1]
    y = np.empty((R, T1, H, P), np.float64)
    cond = np.empty((R, T1, H, P), np.float64) if want_cond else None
    lib().oracle_verify_replay(R, T1, H, P, N, G, Wc, _ptr(ckpt), _ptr(log_len), _ptr(lx), _ptr(ldt),
                               _ptr(lB), _ptr(x), _ptr(dt), _ptr(B), _ptr(C), _ptr(A), _ptr(D), _ptr(y),
                               _ptr(cond) if want_cond else None)
    return (y, cond) if want_cond else y


def fold(ckpt: np.ndarray, log_len, c, do_fold, lx, ldt, lB, x, dt, B, A):
    """Fold logs then the first c[r] step tokens into ckpt (in place) where do_fold[r]."""
    assert ckpt.dtype == np.float64 and ckpt.flags.c_contiguous
    log_len = np.ascontiguousarray(log_len, dtype=np.int32)
    c = np.ascontiguousarray(c, dtype=np.int32)
    do_fold = np.ascontiguousarray(do_fold, dtype=np.int32)
    lx, ldt, lB, x, dt, B, A = _f64(lx), _f64(ldt), _f64(lB), _f64(x), _f64(dt), _f64(B), _f64(A)
    R, H, P, N = ckpt.shape
    T1, G, Wc = x.shape[1], B.shape[2], lx.shape[1]
    lib().oracle_fold(R, T1, H, P, N, G, Wc, _ptr(ckpt), _ptr(log_len), _ptr(c), _ptr(do_fold),
                      _ptr(lx), _ptr(ldt), _ptr(lB), _ptr(x), _ptr(dt), _ptr(B), _ptr(A))


# ---------------------------------------------------------------------------
# closed forms of the sizing rule (Why Speculative Decoding Slows Hybrid Mamba
# Models, What This Means / Implementing It, Role 1)

def expected_tokens_kept(p: float, T: int) -> float:
    """Mean tokens committed per verify step: the real token plus the leading
    run of accepted drafts, each accepted independently with probability p.
    P(at least i drafts kept) = p**i, so the mean is a geometric sum."""
    if p == 1.0:
        return float(T + 1)
    return (1.0 - p ** (T + 1)) / (1.0 - p)


def copy_break_even(p: float, T: int) -> float:
    """Tokens kept per step over the state traffic of a copying step, which is
    (1 + T) / 2 plain steps once state traffic dominates; above 1 the copying
    speculation still wins."""
    return expected_tokens_kept(p, T) / ((1.0 + T) / 2.0)


# ---------------------------------------------------------------------------
# the fp32 instantiation (CPU speed baseline only; never a parity reference)

def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def f32_threads() -> int:
    return int(lib("f32").oracle_max_threads())


def f32_set_threads(n: int) -> None:
    """Threads of the fp32 build's parallel loops (timing only)."""
    lib("f32").oracle_set_threads(int(n))


def f32_decode_step(state, x, dt, B, C, A, D):
    """decode_step in fp32; state [R][H][P][N] float32 in/out."""
    x, dt, B, C, A, D = _f32(x), _f32(dt), _f32(B), _f32(C), _f32(A), _f32(D)
    R, H, P, N = state.shape
    y = np.empty((R, H, P), np.float32)
    lib("f32").oracle_decode_step(R, H, P, N, B.shape[1], _ptr(state), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                                  _ptr(A), _ptr(D), _ptr(y), None)
    return y


def f32_verify_copy(state, x, dt, B, C, A, D):
    state = _f32(state)
    x, dt, B, C, A, D = _f32(x), _f32(dt), _f32(B), _f32(C), _f32(A), _f32(D)
    R, H, P, N = state.shape
    T1, G = x.shape[1], B.shape[2]
    snap = np.empty((T1, R, H, P, N), np.float32)
    y = np.empty((R, T1, H, P), np.float32)
    lib("f32").oracle_verify_copy(R, T1, H, P, N, G, _ptr(state), _ptr(x), _ptr(dt), _ptr(B), _ptr(C),
                                  _ptr(A), _ptr(D), _ptr(snap), _ptr(y), None)
    return snap, y


def f32_verify_replay(ckpt, log_len, lx, ldt, lB, x, dt, B, C, A, D):
    ckpt = _f32(ckpt)
    log_len = np.ascontiguousarray(log_len, dtype=np.int32)
    lx, ldt, lB = _f32(lx), _f32(ldt), _f32(lB)
    x, dt, B, C, A, D = _f32(x), _f32(dt), _f32(B), _f32(C), _f32(A), _f32(D)
    R, H, P, N = ckpt.shape
    T1, G, Wc = x.shape[1], B.shape[2], lx.shape[1]
    y = np.empty((R, T1, H, P), np.float32)
    lib("f32").oracle_verify_replay(R, T1, H, P, N, G, Wc, _ptr(ckpt), _ptr(log_len), _ptr(lx), _ptr(ldt),
                                    _ptr(lB), _ptr(x), _ptr(dt), _ptr(B), _ptr(C), _ptr(A), _ptr(D), _ptr(y), None)
    return y


def f32_fold(ckpt, log_len, c, do_fold, lx, ldt, lB, x, dt, B, A):
    log_len = np.ascontiguousarray(log_len, dtype=np.int32)
    c = np.ascontiguousarray(c, dtype=np.int32)
    do_fold = np.ascontiguousarray(do_fold, dtype=np.int32)
    lx, ldt, lB, x, dt, B, A = _f32(lx), _f32(ldt), _f32(lB), _f32(x), _f32(dt), _f32(B), _f32(A)
    R, H, P, N = ckpt.shape
    T1, G, Wc = x.shape[1], B.shape[2], lx.shape[1]
    lib("f32").oracle_fold(R, T1, H, P, N, G, Wc, _ptr(ckpt), _ptr(log_len), _ptr(c), _ptr(do_fold),
                           _ptr(lx), _ptr(ldt), _ptr(lB), _ptr(x), _ptr(dt), _ptr(B), _ptr(A))


def f32_scan_head(state, x, dt, B, C, A, D, xs, dts, bcs, y, ys):
    """scan_head in fp32 on strided views: x token t at x + t * xs (elements), etc."""
    P, N = state.shape[-2], state.shape[-1]
    L = y.shape[0]
    lib("f32").oracle_scan_head(P, N, L, float(A), float(D), _ptr(x), xs, _ptr(dt), dts, _ptr(B), _ptr(C), bcs,
                                _ptr(state), _ptr(y), ys, None)


# ---------------------------------------------------------------------------
# the pool's lifecycle, on the host

class OraclePool:
    """Slots of fp64 state with the lifecycle and commit rules of the library.

    Slot metadata: position (tokens applied), next_chunk (next chunk sequence
    number expected), epoch (resets), log_len (replay mode), released flag.
    ``last_cond`` holds the condition scale of the last call's outputs (an
    array shaped like y; a list of them for scan_chunk).
    """

    def __init__(self, H, P, N, G, n_slots, A, D, mode=COPY, W=16, max_tokens=9, init_state=None,
                 fold_in_verify=False):
        self.H, self.P, self.N, self.G = H, P, N, G
        self.n_slots, self.mode, self.W, self.T1max = n_slots, mode, W, max_tokens
        # replay: a commit that fills the window leaves the log full, and the next verify folds it
        self.fold_in_verify = bool(fold_in_verify)
        self.A, self.D = _f64(A), _f64(D)
        self.state = np.zeros((n_slots, H, P, N), np.float64)
        if init_state is not None:
            self.state[...] = init_state
        self.position = np.zeros(n_slots, np.int64)
        self.next_chunk = np.zeros(n_slots, np.int64)
        self.epoch = np.zeros(n_slots, np.int64)
        self.log_len = np.zeros(n_slots, np.int32)
        self.released = np.zeros(n_slots, bool)
        # replay log: capacity W - 1 committed entries + max_tokens staged
        cap = W - 1 + max_tokens
        self.lx = np.zeros((n_slots, cap, H, P))
        self.ldt = np.zeros((n_slots, cap, H))
        self.lB = np.zeros((n_slots, cap, G, N))
        self._pending = {}
        self.last_cond = None

    # -- lifecycle ---------------------------------------------------------
    def _check_slots(self, slots):
        slots = [int(s) for s in slots]
        if any(s < 0 or s >= self.n_slots for s in slots) or len(set(slots)) != len(slots):
            return ERR_INVALID_ARG
        if any(self.released[s] for s in slots):
            return ERR_INVALID_STATE
        return OK

    def reset(self, slots):
        """New sequence boundary: zero state, position 0, chunk sequence 0,
        empty log, epoch + 1; also reopens a released slot."""
        for s in slots:
            self.state[s] = 0.0
            self.position[s] = 0
            self.next_chunk[s] = 0
            self.log_len[s] = 0
            self.epoch[s] += 1
            self.released[s] = False
            self._pending.pop(s, None)
        return OK

    def release(self, slots):
        """Cancellation: the slot stops advancing until it is reset."""
        st = self._check_slots(slots)
        if st != OK:
            return st
        for s in slots:
            self.released[s] = True
        return OK

    # -- streaming scan ----------------------------------------------------
    def scan_chunk(self, slots, chunk_seq, chunks):
        """chunks[i] = (x [L][H][P], dt [L][H], B [L][G][N], C [L][G][N]) of slot slots[i].

        Returns (status, [y_i]).  On any error nothing advances.
        """
        st = self._check_slots(slots)
        if st != OK:
            return st, None
        for s, q in zip(slots, chunk_seq):
            if q < self.next_chunk[s]:
                return ERR_DUPLICATE, None
            if q > self.next_chunk[s]:
                return ERR_SEQUENCE, None
        for s, (x, dt, B, C) in zip(slots, chunks):
            if not all(np.all(np.isfinite(_f64(a))) for a in (x, dt, B, C)):
                return ERR_INVALID_CHUNK, None
        if self.mode == REPLAY and any(self.log_len[s] != 0 for s in slots):
            return ERR_INVALID_STATE, None
        ys, conds = [], []
        for s, (x, dt, B, C) in zip(slots, chunks):
            y, cond = scan(self.state[s], x, dt, B, C, self.A, self.D, want_cond=True)
            ys.append(y)
            conds.append(cond)
            self.position[s] += np.asarray(x).shape[0]
            self.next_chunk[s] += 1
        self.last_cond = conds
        return OK, ys

    def decode(self, slots, x, dt, B, C):
        st = self._check_slots(slots)
        if st != OK:
            return st, None
        sl = list(slots)
        sub = np.ascontiguousarray(self.state[sl])
        y, self.last_cond = decode_step(sub, x, dt, B, C, self.A, self.D, want_cond=True)
        self.state[sl] = sub
        self.position[sl] += 1
        return OK, y

    # -- speculative verify --------------------------------------------------
    def verify(self, slots, x, dt, B, C):
        st = self._check_slots(slots)
        if st != OK:
            return st, None
        sl = list(slots)
        T1 = np.asarray(x).shape[1]
        if self.mode == COPY:
            snap, y, self.last_cond = verify_copy(self.state[sl], x, dt, B, C, self.A, self.D, want_cond=True)
            for i, s in enumerate(sl):
                self._pending[s] = ("copy", snap[:, i].copy(), T1)
        else:
            if self.fold_in_verify:  # a log of W or more tokens goes into the checkpoint first
                self.flush([s for s in sl if self.log_len[s] >= self.W])
            y, self.last_cond = verify_replay(self.state[sl], self.log_len[sl], self.lx[sl], self.ldt[sl],
                                              self.lB[sl], x, dt, B, C, self.A, self.D, want_cond=True)
            xs, dts, Bs = _f64(x), _f64(dt), _f64(B)
            for i, s in enumerate(sl):
                self._pending[s] = ("replay", (xs[i], dts[i], Bs[i]), T1)
        return OK, y

    def commit(self, slots, accept, force_fold=False):
        """Commit 1 + accept[i] tokens of the last verify of each slot.

        Copy mode: the state after the last accepted token becomes current.
        Replay mode: if log_len + c < W (and no forced fold) the c accepted
        tokens are appended to the log; otherwise the log and the c tokens
        are folded into the checkpoint and the log empties.  With
        fold_in_verify the c tokens are appended whatever the length (unless
        forced), and the next verify folds a log of W or more tokens before
        it replays (the same states and outputs, the checkpoint written one
        call later).
        Returns (status, folded flags).
        """
        st = self._check_slots(slots)
        if st != OK:
            return st, None
        if any(s not in self._pending for s in slots):
            return ERR_INVALID_STATE, None
        for s, a in zip(slots, accept):
            if a < 0 or a >= self._pending[s][2]:
                return ERR_INVALID_ARG, None
        folded = np.zeros(len(slots), bool)
        for i, (s, a) in enumerate(zip(slots, accept)):
            kind, payload, T1 = self._pending.pop(s)
            c = int(a) + 1
            if kind == "copy":
                self.state[s] = payload[c - 1]
            else:
                xs, dts, Bs = payload
                k = int(self.log_len[s])
                if (k + c < self.W or self.fold_in_verify) and not force_fold:
                    self.lx[s, k:k + c] = xs[:c]
                    self.ldt[s, k:k + c] = dts[:c]
                    self.lB[s, k:k + c] = Bs[:c]
                    self.log_len[s] = k + c
                else:
                    sub = np.ascontiguousarray(self.state[s:s + 1])
                    fold(sub, [k], [c], [1], self.lx[s:s + 1], self.ldt[s:s + 1], self.lB[s:s + 1],
                         xs[None], dts[None], Bs[None], self.A)
                    self.state[s] = sub[0]
                    self.log_len[s] = 0
                    folded[i] = True
            self.position[s] += c
        return OK, folded

    def flush(self, slots):
        """Fold any logged tokens into the checkpoint (before a checkpoint read)."""
        for s in slots:
            k = int(self.log_len[s])
            if k == 0:
                continue
            sub = np.ascontiguousarray(self.state[s:s + 1])
            T1 = 1
            z = np.zeros((1, T1, self.H, self.P)), np.zeros((1, T1, self.H)), np.zeros((1, T1, self.G, self.N))
            fold(sub, [k], [0], [1], self.lx[s:s + 1], self.ldt[s:s + 1], self.lB[s:s + 1],
                 z[0], z[1], z[2], self.A)
            self.state[s] = sub[0]
            self.log_len[s] = 0
        return OK
