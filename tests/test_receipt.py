"""Checkpoint receipt and state blob, host side (no GPU): the byte layout
against the definitions it follows, the checksum against FNV-1a's published
test vectors, and refusal of every kind of damage (Mamba Streaming State That
Survives Chunking, Make reset, checkpoint, and cancellation observable:
checkpoint receipt; the SSM.PREFIX state-store page: array blob format)."""
import struct

import numpy as np


def _mod():
    import hybrid_serving_mamba_gb300 as m
    return m


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64 bits, from Fowler, Noll and Vo's definition."""
    h = 14695981039346656037
    for byte in data:
        h ^= byte
        h = (h * 1099511628211) % (1 << 64)
    return h


def test_fnv1a64_published_vectors():
    # the FNV authors' test vectors for 64-bit FNV-1a
    assert fnv1a64(b"") == 0xCBF29CE484222325
    assert fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert fnv1a64(b"foobar") == 0x85944171F73967E8


HEADER = struct.Struct("<4sIQQQiIiiiiiiiqqQQ")  # the receipt, as the header file lays it out


def _receipt(m, H=3, P=4, N=5, G=1):
    r = m.ssm_receipt()
    r.id = m.stream_identity(0x1234_5678_9ABC_DEF0, 77, 0xFEED, 5)
    r.schema_version = m.SSM_STATE_SCHEMA_VERSION
    r.state_dtype, r.input_dtype, r.dt_dtype = 0, 2, 0
    r.nheads, r.headdim, r.dstate, r.ngroups = H, P, N, G
    r.position, r.next_chunk = 4097, 12
    return r


def _state(H=3, P=4, N=5, seed=3):
    return np.random.default_rng(seed).standard_normal((H, P, N)).astype(np.float32)


def test_layout_follows_the_receipt_and_blob_definitions():
    m = _mod()
    r, s = _receipt(m), _state()
    st, blob = m.ssm_receipt_encode(r, s)
    assert st == m.SSM_OK
    assert len(blob) == m.ssm_receipt_bytes(3, 4, 5) == HEADER.size + 28 + s.nbytes
    f = HEADER.unpack_from(blob, 0)
    assert f[0] == b"SSMR" and f[1] == 1
    assert f[2:6] == (0x1234_5678_9ABC_DEF0, 77, 0xFEED, 5)          # stream, model and code revision, layer
    assert f[6] == m.SSM_STATE_SCHEMA_VERSION and f[7:10] == (0, 2, 0)  # schema, state / input / dt dtype
    assert f[10:14] == (3, 4, 5, 1) and f[14:16] == (4097, 12)      # dims, position, chunk sequence
    body = blob[HEADER.size:]
    assert f[16] == len(body)
    assert f[17] == fnv1a64(body) == r.checksum
    # the state blob: version 1, one array of rank 3, shape [H][P][N], dtype code 0 (fp32), raw values
    assert struct.unpack_from("<7I", body, 0) == (1, 1, 3, 3, 4, 5, 0)
    assert body[28:] == s.astype("<f4").tobytes()


def test_decode_round_trip():
    m = _mod()
    r, s = _receipt(m, 2, 8, 16, 2), _state(2, 8, 16)
    st, blob = m.ssm_receipt_encode(r, s)
    st, q, got = m.ssm_receipt_decode(blob)
    assert st == m.SSM_OK
    assert np.array_equal(got, s)
    for k in ("schema_version", "state_dtype", "input_dtype", "dt_dtype", "nheads", "headdim", "dstate",
              "ngroups", "position", "next_chunk", "checksum"):
        assert getattr(q, k) == getattr(r, k), k
    assert (q.id.stream_id, q.id.model_revision, q.id.code_revision, q.id.layer) == \
        (r.id.stream_id, r.id.model_revision, r.id.code_revision, r.id.layer)


def _damaged(blob: bytes):
    """Each kind of damage a resume must refuse; the blob edits keep its checksum right
    where the damage is meant to be found by a field check instead."""
    n = len(blob)
    h = HEADER.size

    def edit(off, new, fix_sum=False):
        b = bytearray(blob)
        b[off:off + len(new)] = new
        if fix_sum:
            struct.pack_into("<Q", b, h - 8, fnv1a64(bytes(b[h:])))
        return bytes(b)

    yield "payload byte", edit(n - 3, bytes([blob[n - 3] ^ 0x40]))
    yield "checksum", edit(h - 8, bytes([blob[h - 8] ^ 1]))
    yield "magic", edit(0, b"SSMX")
    yield "format version", edit(4, struct.pack("<I", 2))
    yield "truncated", blob[:-1]
    yield "trailing byte", blob + b"\0"
    yield "blob version", edit(h, struct.pack("<I", 2), fix_sum=True)
    yield "two arrays", edit(h + 4, struct.pack("<I", 2), fix_sum=True)
    yield "blob shape", edit(h + 12, struct.pack("<I", 4), fix_sum=True)
    yield "blob dtype bf16", edit(h + 24, struct.pack("<I", 2), fix_sum=True)
    yield "state dtype", edit(40, struct.pack("<i", 2))
    yield "header dims", edit(56, struct.pack("<i", 6))


def test_every_damage_is_refused():
    m = _mod()
    st, blob = m.ssm_receipt_encode(_receipt(m), _state())
    assert m.ssm_receipt_decode(blob)[0] == m.SSM_OK
    for what, bad in _damaged(blob):
        assert m.ssm_receipt_decode(bad)[0] == m.SSM_ERR_SCHEMA, what


def test_encode_reports_the_size_it_needs():
    import ctypes
    m = _mod()
    r, s = _receipt(m), _state()
    need = ctypes.c_size_t()
    small = (ctypes.c_ubyte * 16)()
    st = m.library().ssm_receipt_encode(ctypes.byref(r), s.ctypes.data_as(ctypes.c_void_p), small, 16,
                                        ctypes.byref(need))
    assert st == m.SSM_ERR_INVALID_ARG and need.value == m.ssm_receipt_bytes(3, 4, 5)
    assert m.ssm_receipt_bytes(0, 4, 5) == 0
