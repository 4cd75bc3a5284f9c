"""ctypes binding of libssmstate's C ABI (include/ssm_state.h).

Argument marshalling only: every function below has the name of its C
entry point, checks the tensors it is given (device, dtype, contiguity,
size) and passes raw pointers; all work runs in the library's CUDA kernels.
There is no fallback: if the library is missing the import fails.

Tensors: device tensors are ``torch.Tensor`` on the pool's CUDA device; bf16
inputs are ``torch.bfloat16``, fp32 are ``torch.float32``; slot lists,
cu_seqlens and chunk sequence numbers are host sequences (lists, numpy
arrays or CPU tensors) as the C ABI takes them.  ``stream`` defaults to
torch's current stream.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libssmstate.so")

SSM_OK, SSM_ERR_INVALID_ARG, SSM_ERR_INVALID_CHUNK, SSM_ERR_INVALID_STATE = 0, 1, 2, 3
SSM_ERR_SEQUENCE, SSM_ERR_DUPLICATE, SSM_ERR_SCHEMA, SSM_ERR_CUDA, SSM_ERR_TIMEOUT, SSM_ERR_NO_MEMORY = 4, 5, 6, 7, 8, 9
SSM_DTYPE_F32, SSM_DTYPE_BF16 = 0, 2
SSM_MODE_COPY, SSM_MODE_REPLAY = 0, 1
SSM_FOLD_AT_COMMIT, SSM_FOLD_IN_VERIFY = 0, 1
SSM_FLAG_NONFINITE_INPUT, SSM_FLAG_POISONED_SLOT, SSM_FLAG_BAD_ACCEPT = 1, 2, 4
SSM_FLAG_LOG_NOT_EMPTY, SSM_FLAG_TIMEOUT = 8, 16

# every entry point the header declares (the CPU test checks the library exports them)
EXPORTS = (
    "ssm_state_init", "ssm_state_destroy", "ssm_state_reset", "ssm_state_release", "ssm_state_checkpoint",
    "ssm_state_restore", "ssm_slot_info", "ssm_state_gather", "ssm_scan_chunk", "ssm_decode_step",
    "ssm_decode_steps_host",
    "ssm_verify_copy", "ssm_verify_replay", "ssm_state_commit", "ssm_pool_status", "ssm_last_path",
    "ssm_status_string", "ssm_pool_bytes", "ssm_debug_stall_next_verify", "ssm_verify_replay_static",
    "ssm_receipt_bytes", "ssm_receipt_encode",
    "ssm_receipt_decode", "ssm_state_checkpoint_receipt", "ssm_state_restore_receipt",
    "ssm_gdn_init", "ssm_gdn_destroy", "ssm_gdn_reset", "ssm_gdn_decode_step", "ssm_gdn_verify_replay",
    "ssm_gdn_commit", "ssm_gdn_gather", "ssm_gdn_slot_info", "ssm_gdn_status", "ssm_gdn_last_path",
    "ssm_gdn_last_commit_path",
)


class SSMError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class ssm_config(ctypes.Structure):
    _fields_ = [("nheads", ctypes.c_int32), ("headdim", ctypes.c_int32), ("dstate", ctypes.c_int32),
                ("ngroups", ctypes.c_int32), ("input_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("window", ctypes.c_int32), ("max_tokens", ctypes.c_int32),
                ("fold", ctypes.c_int32)]


class ssm_slot_meta(ctypes.Structure):
    _fields_ = [("position", ctypes.c_int64), ("next_chunk", ctypes.c_int64), ("epoch", ctypes.c_int64),
                ("log_len", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class ssm_stream_identity(ctypes.Structure):
    _fields_ = [("stream_id", ctypes.c_uint64), ("model_revision", ctypes.c_uint64),
                ("code_revision", ctypes.c_uint64), ("layer", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class ssm_receipt(ctypes.Structure):
    _fields_ = [("id", ssm_stream_identity), ("schema_version", ctypes.c_uint32), ("state_dtype", ctypes.c_int32),
                ("input_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32), ("nheads", ctypes.c_int32),
                ("headdim", ctypes.c_int32), ("dstate", ctypes.c_int32), ("ngroups", ctypes.c_int32),
                ("position", ctypes.c_int64), ("next_chunk", ctypes.c_int64), ("checksum", ctypes.c_uint64)]


SSM_STATE_SCHEMA_VERSION = 1


class ssm_gdn_config(ctypes.Structure):
    _fields_ = [("nheads", ctypes.c_int32), ("nkheads", ctypes.c_int32), ("dk", ctypes.c_int32),
                ("dv", ctypes.c_int32), ("input_dtype", ctypes.c_int32), ("window", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libssmstate is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(LIB_PATH)
    V, I32, I64, U32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    P_I32 = ctypes.POINTER(I32)
    P_I64 = ctypes.POINTER(I64)
    sig = {
        "ssm_state_init": [ctypes.POINTER(ssm_config), I32, V, V, ctypes.POINTER(V)],
        "ssm_state_destroy": [V],
        "ssm_state_reset": [V, P_I32, I32, V],
        "ssm_state_release": [V, P_I32, I32],
        "ssm_state_checkpoint": [V, I32, V, V, ctypes.c_size_t, ctypes.POINTER(ssm_slot_meta), V],
        "ssm_state_restore": [V, I32, V, ctypes.c_size_t, ctypes.POINTER(ssm_slot_meta), V],
        "ssm_slot_info": [V, I32, ctypes.POINTER(ssm_slot_meta), V],
        "ssm_state_gather": [V, I32, P_I32, V, V],
        "ssm_scan_chunk": [V, I32, P_I32, P_I32, P_I64, V, V, V, V, V, V, V, V],
        "ssm_decode_step": [V, I32, P_I32, V, V, V, V, V, V, V, V],
        "ssm_decode_steps_host": [V, I32, P_I32, I32, V, V, V, V, V, V, V, V],
        "ssm_verify_copy": [V, I32, I32, P_I32, V, V, V, V, V, V, V, V],
        "ssm_verify_replay": [V, I32, I32, P_I32, V, V, V, V, V, V, V, V],
        "ssm_state_commit": [V, I32, P_I32, V, I32, V, V],
        "ssm_pool_status": [V, ctypes.POINTER(U32), I32, V],
        "ssm_last_path": [V],
        "ssm_status_string": [ctypes.c_int],
        "ssm_pool_bytes": [V],
        "ssm_debug_stall_next_verify": [V],
        "ssm_verify_replay_static": [I32, I32, I32, I32, I32, I32, I32, I32, I32, V, V, V, V, V,
                                     V, V, V, V, V, V, V, V, V],
        "ssm_receipt_encode": [ctypes.POINTER(ssm_receipt), V, V, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)],
        "ssm_receipt_decode": [V, ctypes.c_size_t, ctypes.POINTER(ssm_receipt), ctypes.POINTER(V)],
        "ssm_state_checkpoint_receipt": [V, I32, V, ctypes.POINTER(ssm_stream_identity), V, ctypes.c_size_t,
                                         ctypes.POINTER(ctypes.c_size_t), V],
        "ssm_state_restore_receipt": [V, I32, V, ctypes.c_size_t, ctypes.POINTER(ssm_stream_identity), V],
        "ssm_gdn_init": [ctypes.POINTER(ssm_gdn_config), I32, V, V, ctypes.POINTER(V)],
        "ssm_gdn_destroy": [V],
        "ssm_gdn_reset": [V, P_I32, I32, V],
        "ssm_gdn_decode_step": [V, I32, P_I32, V, V, V, V, V, V, V],
        "ssm_gdn_verify_replay": [V, I32, I32, P_I32, V, V, V, V, V, V, V],
        "ssm_gdn_commit": [V, I32, P_I32, V, I32, V],
        "ssm_gdn_gather": [V, I32, P_I32, V, V],
        "ssm_gdn_slot_info": [V, I32, P_I64, P_I32, ctypes.POINTER(U32), V],
        "ssm_gdn_last_path": [V],
        "ssm_gdn_last_commit_path": [V],
        "ssm_gdn_status": [V, ctypes.POINTER(U32), I32, V],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.ssm_last_path.restype = ctypes.c_char_p
    lib.ssm_gdn_last_path.restype = ctypes.c_char_p
    lib.ssm_gdn_last_commit_path.restype = ctypes.c_char_p
    lib.ssm_status_string.restype = ctypes.c_char_p
    lib.ssm_pool_bytes.restype = ctypes.c_size_t
    lib.ssm_receipt_bytes.argtypes = [I32, I32, I32]
    lib.ssm_receipt_bytes.restype = ctypes.c_size_t
    return lib


_lib = _load()


def library():
    return _lib


def status_string(status: int) -> str:
    return _lib.ssm_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != SSM_OK:
        raise SSMError(status, where)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _host_i32(v):
    a = np.ascontiguousarray(np.asarray(v.cpu() if hasattr(v, "cpu") else v), dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _host_i64(v):
    a = np.ascontiguousarray(np.asarray(v.cpu() if hasattr(v, "cpu") else v), dtype=np.int64)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _dev(t, name, dtype=None, numel=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


@dataclass
class Pool:
    """Handle returned by ssm_state_init, with the config it was made with."""
    handle: ctypes.c_void_p
    cfg: ssm_config
    n_slots: int

    @property
    def H(self):
        return self.cfg.nheads

    @property
    def P(self):
        return self.cfg.headdim

    @property
    def N(self):
        return self.cfg.dstate

    @property
    def G(self):
        return self.cfg.ngroups

    def torch_dtype(self, code=None):
        import torch
        code = self.cfg.input_dtype if code is None else code
        return torch.bfloat16 if code == SSM_DTYPE_BF16 else torch.float32


def make_config(nheads, headdim, dstate, ngroups, input_dtype=SSM_DTYPE_F32, dt_dtype=SSM_DTYPE_F32,
                mode=SSM_MODE_COPY, window=16, max_tokens=9, fold=SSM_FOLD_AT_COMMIT) -> ssm_config:
    return ssm_config(nheads, headdim, dstate, ngroups, input_dtype, dt_dtype, mode, window, max_tokens, fold)


# ---------------------------------------------------------------- lifecycle

def ssm_state_init(cfg: ssm_config, n_slots: int, init_state=None, stream=None) -> Pool:
    import torch
    hpn = cfg.nheads * cfg.headdim * cfg.dstate
    ptr = _dev(init_state, "init_state", torch.float32, n_slots * hpn) if init_state is not None else None
    out = ctypes.c_void_p()
    _check(_lib.ssm_state_init(ctypes.byref(cfg), int(n_slots), ptr, _stream(stream), ctypes.byref(out)),
           "ssm_state_init")
    return Pool(out, cfg, int(n_slots))


def ssm_state_destroy(pool: Pool) -> None:
    if pool.handle:
        _check(_lib.ssm_state_destroy(pool.handle), "ssm_state_destroy")
        pool.handle = ctypes.c_void_p()


def ssm_state_reset(pool: Pool, slots, stream=None) -> int:
    a, p = _host_i32(slots)
    return _lib.ssm_state_reset(pool.handle, p, len(a), _stream(stream))


def ssm_state_release(pool: Pool, slots) -> int:
    a, p = _host_i32(slots)
    return _lib.ssm_state_release(pool.handle, p, len(a))


def ssm_state_checkpoint(pool: Pool, slot: int, A=None, stream=None):
    """Returns (status, state ndarray float32 [H][P][N], ssm_slot_meta)."""
    import torch
    host = np.empty((pool.H, pool.P, pool.N), np.float32)
    meta = ssm_slot_meta()
    st = _lib.ssm_state_checkpoint(pool.handle, int(slot), _dev(A, "A", torch.float32, pool.H),
                                   host.ctypes.data_as(ctypes.c_void_p), host.nbytes, ctypes.byref(meta),
                                   _stream(stream))
    return st, host, meta


def ssm_state_restore(pool: Pool, slot: int, host_state: np.ndarray, meta: ssm_slot_meta, stream=None) -> int:
    h = np.ascontiguousarray(host_state, dtype=np.float32)
    return _lib.ssm_state_restore(pool.handle, int(slot), h.ctypes.data_as(ctypes.c_void_p), h.nbytes,
                                  ctypes.byref(meta), _stream(stream))


def stream_identity(stream_id: int, model_revision: int, code_revision: int, layer: int) -> ssm_stream_identity:
    return ssm_stream_identity(stream_id, model_revision, code_revision, layer, 0)


def ssm_receipt_bytes(nheads: int, headdim: int, dstate: int) -> int:
    return int(_lib.ssm_receipt_bytes(nheads, headdim, dstate))


def ssm_receipt_encode(receipt: ssm_receipt, state: np.ndarray):
    """Host only: (status, bytes) of receipt + state blob; receipt.checksum is filled in."""
    s = np.ascontiguousarray(state, dtype=np.float32)
    need = ctypes.c_size_t()
    _lib.ssm_receipt_encode(ctypes.byref(receipt), s.ctypes.data_as(ctypes.c_void_p), None, 0, ctypes.byref(need))
    buf = (ctypes.c_ubyte * need.value)()
    st = _lib.ssm_receipt_encode(ctypes.byref(receipt), s.ctypes.data_as(ctypes.c_void_p), buf, need.value,
                                 ctypes.byref(need))
    return st, bytes(buf)


def ssm_receipt_decode(blob: bytes):
    """Host only: (status, ssm_receipt, state ndarray float32 [H][P][N] or None)."""
    buf = ctypes.create_string_buffer(bytes(blob), len(blob))
    r = ssm_receipt()
    ptr = ctypes.c_void_p()
    st = _lib.ssm_receipt_decode(buf, len(blob), ctypes.byref(r), ctypes.byref(ptr))
    if st != SSM_OK:
        return st, r, None
    off = ptr.value - ctypes.addressof(buf)
    n = r.nheads * r.headdim * r.dstate
    state = np.frombuffer(bytes(blob), dtype="<f4", count=n, offset=off).reshape(r.nheads, r.headdim, r.dstate)
    return st, r, state.copy()


def ssm_state_checkpoint_receipt(pool: Pool, slot: int, identity: ssm_stream_identity, A=None, stream=None):
    """(status, bytes): the slot checkpointed as receipt + state blob."""
    import torch
    need = _lib.ssm_receipt_bytes(pool.H, pool.P, pool.N)
    buf = (ctypes.c_ubyte * need)()
    written = ctypes.c_size_t()
    st = _lib.ssm_state_checkpoint_receipt(pool.handle, int(slot), _dev(A, "A", torch.float32, pool.H),
                                           ctypes.byref(identity), buf, need, ctypes.byref(written), _stream(stream))
    return st, bytes(buf)[:written.value] if st == SSM_OK else b""


def ssm_state_restore_receipt(pool: Pool, slot: int, blob: bytes, expect: ssm_stream_identity, stream=None) -> int:
    buf = ctypes.create_string_buffer(bytes(blob), len(blob))
    return _lib.ssm_state_restore_receipt(pool.handle, int(slot), buf, len(blob), ctypes.byref(expect),
                                          _stream(stream))


def ssm_slot_info(pool: Pool, slot: int, stream=None):
    meta = ssm_slot_meta()
    st = _lib.ssm_slot_info(pool.handle, int(slot), ctypes.byref(meta), _stream(stream))
    return st, meta


def ssm_state_gather(pool: Pool, slots, dst, stream=None) -> int:
    import torch
    a, p = _host_i32(slots)
    ptr = _dev(dst, "dst", torch.float32, len(a) * pool.H * pool.P * pool.N)
    return _lib.ssm_state_gather(pool.handle, len(a), p, ptr, _stream(stream))


# ---------------------------------------------------------------- hot path

def _inputs(pool: Pool, n_tok_total: int, x, dt, B, C, A, D, y):
    import torch
    td, tdt = pool.torch_dtype(), pool.torch_dtype(pool.cfg.dt_dtype)
    H, P, N, G = pool.H, pool.P, pool.N, pool.G
    return (_dev(x, "x", td, n_tok_total * H * P), _dev(dt, "dt", tdt, n_tok_total * H),
            _dev(B, "B", td, n_tok_total * G * N), _dev(C, "C", td, n_tok_total * G * N),
            _dev(A, "A", torch.float32, H), _dev(D, "D", torch.float32, H),
            _dev(y, "y", td, n_tok_total * H * P))


def ssm_scan_chunk(pool: Pool, cu_seqlens, slots, chunk_seq, x, dt, B, C, A, D, y, stream=None) -> int:
    cu, pcu = _host_i32(cu_seqlens)
    sl, psl = _host_i32(slots)
    cs, pcs = _host_i64(chunk_seq)
    if len(cu) != len(sl) + 1 or len(cs) != len(sl):
        raise ValueError("cu_seqlens must have n_seq + 1 entries and chunk_seq n_seq")
    total = int(cu[-1])
    if total == 0:
        ptrs = (None,) * 7
    else:
        ptrs = _inputs(pool, total, x, dt, B, C, A, D, y)
    return _lib.ssm_scan_chunk(pool.handle, len(sl), pcu, psl, pcs, *ptrs, _stream(stream))


def ssm_decode_step(pool: Pool, slots, x, dt, B, C, A, D, y, stream=None) -> int:
    sl, psl = _host_i32(slots)
    return _lib.ssm_decode_step(pool.handle, len(sl), psl, *_inputs(pool, len(sl), x, dt, B, C, A, D, y),
                                _stream(stream))


def _pinned(t, name, dtype, numel):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())  # page-locked or not: the library checks and refuses


def ssm_decode_steps_host(pool: Pool, slots, n_steps: int, x, dt, B, C, A, D, y, stream=None) -> int:
    """n_steps decode tokens over the same slots, x / dt / B / C / y host tensors (page-locked), step-major."""
    import torch
    sl, psl = _host_i32(slots)
    n = len(sl) * int(n_steps)
    td, tdt = pool.torch_dtype(), pool.torch_dtype(pool.cfg.dt_dtype)
    H, P, N, G = pool.H, pool.P, pool.N, pool.G
    return _lib.ssm_decode_steps_host(pool.handle, len(sl), psl, int(n_steps), _pinned(x, "x", td, n * H * P),
                                      _pinned(dt, "dt", tdt, n * H), _pinned(B, "B", td, n * G * N),
                                      _pinned(C, "C", td, n * G * N), _dev(A, "A", torch.float32, H),
                                      _dev(D, "D", torch.float32, H), _pinned(y, "y", td, n * H * P),
                                      _stream(stream))


def ssm_verify_copy(pool: Pool, slots, n_tok: int, x, dt, B, C, A, D, y, stream=None) -> int:
    sl, psl = _host_i32(slots)
    return _lib.ssm_verify_copy(pool.handle, len(sl), int(n_tok), psl,
                                *_inputs(pool, len(sl) * n_tok, x, dt, B, C, A, D, y), _stream(stream))


def ssm_verify_replay(pool: Pool, slots, n_tok: int, x, dt, B, C, A, D, y, stream=None) -> int:
    sl, psl = _host_i32(slots)
    return _lib.ssm_verify_replay(pool.handle, len(sl), int(n_tok), psl,
                                  *_inputs(pool, len(sl) * n_tok, x, dt, B, C, A, D, y), _stream(stream))


def ssm_state_commit(pool: Pool, slots, accept, force_fold: bool = False, A=None, stream=None) -> int:
    import torch
    sl, psl = _host_i32(slots)
    return _lib.ssm_state_commit(pool.handle, len(sl), psl, _dev(accept, "accept", torch.int32, len(sl)),
                                 1 if force_fold else 0, _dev(A, "A", torch.float32, pool.H), _stream(stream))


# ---------------------------------------------------------------- diagnostics

def ssm_pool_status(pool: Pool, clear: bool = False, stream=None):
    f = ctypes.c_uint32()
    st = _lib.ssm_pool_status(pool.handle, ctypes.byref(f), 1 if clear else 0, _stream(stream))
    return st, int(f.value)


def ssm_last_path(pool) -> str:
    """Kernel path of the pool's last hot-path call; with pool None, that of
    this thread's last ssm_verify_replay_static call."""
    return _lib.ssm_last_path(None if pool is None else pool.handle).decode()


def ssm_pool_bytes(pool: Pool) -> int:
    return int(_lib.ssm_pool_bytes(pool.handle))


# ---------------------------------------------------------------- no-allocation variant

SSM_STATIC_SCRATCH_FLOATS = 1047552


def ssm_verify_replay_static(batch, n_tok, nheads, headdim, dstate, ngroups, window, input_dtype, dt_dtype,
                             ckpt, log_x, log_dt, log_B, log_len, x, dt, B, C, A, D, y, flags, stream=None) -> int:
    """Replay verify on caller-owned buffers with the library's built-in
    scratch (no pool, no allocation); see ssm_verify_replay_static in
    include/ssm_state.h for the buffer shapes."""
    import torch
    wc = window - 1 + n_tok
    tin = torch.bfloat16 if input_dtype == SSM_DTYPE_BF16 else torch.float32
    tdt = torch.bfloat16 if dt_dtype == SSM_DTYPE_BF16 else torch.float32
    H, P, N, G = nheads, headdim, dstate, ngroups
    return _lib.ssm_verify_replay_static(
        int(batch), int(n_tok), H, P, N, G, int(window), int(input_dtype), int(dt_dtype),
        _dev(ckpt, "ckpt", torch.float32, batch * H * P * N), _dev(log_x, "log_x", tin, batch * wc * H * P),
        _dev(log_dt, "log_dt", torch.float32, batch * wc * H), _dev(log_B, "log_B", tin, batch * wc * G * N),
        _dev(log_len, "log_len", torch.int32, batch), _dev(x, "x", tin, batch * n_tok * H * P),
        _dev(dt, "dt", tdt, batch * n_tok * H), _dev(B, "B", tin, batch * n_tok * G * N),
        _dev(C, "C", tin, batch * n_tok * G * N), _dev(A, "A", torch.float32, H), _dev(D, "D", torch.float32, H),
        _dev(y, "y", tin, batch * n_tok * H * P), _dev(flags, "flags", torch.int32, 1), _stream(stream))


# ------------------------------------------------------------ gated delta rule

@dataclass
class GdnPool:
    """Handle returned by ssm_gdn_init, with the config it was made with."""
    handle: ctypes.c_void_p
    cfg: ssm_gdn_config
    n_slots: int

    @property
    def H(self):
        return self.cfg.nheads

    @property
    def G(self):
        return self.cfg.nkheads

    @property
    def dk(self):
        return self.cfg.dk

    @property
    def dv(self):
        return self.cfg.dv


def make_gdn_config(nheads, nkheads, dk, dv, input_dtype=SSM_DTYPE_F32, window=16, max_tokens=9) -> ssm_gdn_config:
    return ssm_gdn_config(nheads, nkheads, dk, dv, input_dtype, window, max_tokens)


def ssm_gdn_init(cfg: ssm_gdn_config, n_slots: int, init_state=None, stream=None) -> GdnPool:
    """Create a gated-delta-rule pool (raises SSMError on failure)."""
    import torch
    out = ctypes.c_void_p()
    numel = n_slots * cfg.nheads * cfg.dv * cfg.dk
    st = _lib.ssm_gdn_init(ctypes.byref(cfg), int(n_slots), _dev(init_state, "init_state", torch.float32, numel),
                           _stream(stream), ctypes.byref(out))
    _check(st, "ssm_gdn_init")
    return GdnPool(out, cfg, int(n_slots))


def ssm_gdn_destroy(pool: GdnPool) -> int:
    return _lib.ssm_gdn_destroy(pool.handle)


def ssm_gdn_reset(pool: GdnPool, slots, stream=None) -> int:
    sl, psl = _host_i32(slots)
    return _lib.ssm_gdn_reset(pool.handle, psl, len(sl), _stream(stream))


def _gdn_inputs(pool: GdnPool, n, q, k, v, g, beta, y):
    import torch
    tin = torch.bfloat16 if pool.cfg.input_dtype == SSM_DTYPE_BF16 else torch.float32
    H, G, dk, dv = pool.H, pool.G, pool.dk, pool.dv
    return (_dev(q, "q", tin, n * G * dk), _dev(k, "k", tin, n * G * dk), _dev(v, "v", tin, n * H * dv),
            _dev(g, "g", torch.float32, n * H), _dev(beta, "beta", torch.float32, n * H),
            _dev(y, "y", tin, n * H * dv))


def ssm_gdn_decode_step(pool: GdnPool, slots, q, k, v, g, beta, y, stream=None) -> int:
    sl, psl = _host_i32(slots)
    return _lib.ssm_gdn_decode_step(pool.handle, len(sl), psl, *_gdn_inputs(pool, len(sl), q, k, v, g, beta, y),
                                    _stream(stream))


def ssm_gdn_verify_replay(pool: GdnPool, slots, n_tok: int, q, k, v, g, beta, y, stream=None) -> int:
    sl, psl = _host_i32(slots)
    return _lib.ssm_gdn_verify_replay(pool.handle, len(sl), int(n_tok), psl,
                                      *_gdn_inputs(pool, len(sl) * n_tok, q, k, v, g, beta, y), _stream(stream))


def ssm_gdn_commit(pool: GdnPool, slots, accept, force_fold: bool = False, stream=None) -> int:
    import torch
    sl, psl = _host_i32(slots)
    return _lib.ssm_gdn_commit(pool.handle, len(sl), psl, _dev(accept, "accept", torch.int32, len(sl)),
                               1 if force_fold else 0, _stream(stream))


def ssm_gdn_gather(pool: GdnPool, slots, dst, stream=None) -> int:
    import torch
    sl, psl = _host_i32(slots)
    return _lib.ssm_gdn_gather(pool.handle, len(sl), psl,
                               _dev(dst, "dst", torch.float32, len(sl) * pool.H * pool.dv * pool.dk),
                               _stream(stream))


def ssm_gdn_slot_info(pool: GdnPool, slot: int, stream=None):
    """(status, position, log_len, flags) of one slot (synchronous)."""
    pos, ll, fl = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_uint32()
    st = _lib.ssm_gdn_slot_info(pool.handle, int(slot), ctypes.byref(pos), ctypes.byref(ll), ctypes.byref(fl),
                                _stream(stream))
    return st, int(pos.value), int(ll.value), int(fl.value)


def ssm_debug_stall_next_verify(pool: Pool) -> int:
    """Tests of the failure path: the pool's next tensor-core replay verify lets one CTA's waits run out."""
    return _lib.ssm_debug_stall_next_verify(pool.handle)


def ssm_gdn_last_path(pool) -> str:
    """Kernel path of the gated-delta-rule pool's last verify."""
    return _lib.ssm_gdn_last_path(pool.handle if pool is not None else None).decode()


def ssm_gdn_last_commit_path(pool) -> str:
    """Fold path of the gated-delta-rule pool's last commit."""
    return _lib.ssm_gdn_last_commit_path(pool.handle if pool is not None else None).decode()


def ssm_gdn_status(pool: GdnPool, clear: bool = False, stream=None):
    f = ctypes.c_uint32()
    st = _lib.ssm_gdn_status(pool.handle, ctypes.byref(f), 1 if clear else 0, _stream(stream))
    return st, int(f.value)
