"""CPU-side checks of the C ABI: the library loads, exports every entry point
the header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mod():
    import __graft_entry__
    __graft_entry__.build()
    import hybrid_serving_mamba_gb300 as m
    return m


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(ssm_[a-z_]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(mod):
    declared = _declared()
    assert declared, "no declarations found"
    lib = ctypes.CDLL(mod.LIB_PATH)
    missing = [n for n in sorted(declared) if not hasattr(lib, n)]
    assert not missing, missing
    assert declared == set(mod.EXPORTS)


def test_status_strings(mod):
    assert mod.status_string(0) == "ok"
    assert mod.status_string(4) == "chunk sequence out of order"
    assert mod.status_string(5) == "chunk already applied"
    assert mod.status_string(99) == "unknown status"


@pytest.mark.parametrize("bad", [
    dict(nheads=0), dict(headdim=0), dict(headdim=300), dict(dstate=48), dict(ngroups=3),
    dict(input_dtype=1), dict(dt_dtype=7), dict(mode=2), dict(max_tokens=0), dict(max_tokens=65),
    dict(mode=1, window=0),
    dict(fold=2), dict(fold=1), dict(mode=1, fold=1),  # fold in verify: replay, bf16, P 64, N 128 only
    dict(mode=1, fold=1, input_dtype=2, headdim=64, dstate=128, max_tokens=33),
    dict(mode=1, fold=1, input_dtype=2, headdim=64, dstate=128, window=40, max_tokens=13),  # log > 64
])
def test_init_rejects_bad_config(mod, bad):
    kw = dict(nheads=4, headdim=16, dstate=16, ngroups=2, input_dtype=0, dt_dtype=0, mode=0, window=4, max_tokens=4)
    kw.update(bad)
    cfg = mod.ssm_config(**kw)
    out = ctypes.c_void_p()
    st = mod.library().ssm_state_init(ctypes.byref(cfg), 4, None, None, ctypes.byref(out))
    assert st == mod.SSM_ERR_INVALID_ARG and not out.value


def test_null_pool_is_rejected(mod):
    lib = mod.library()
    slots = (ctypes.c_int32 * 1)(0)
    assert lib.ssm_decode_step(None, 1, slots, None, None, None, None, None, None, None, None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_state_commit(None, 1, slots, None, 0, None, None) == mod.SSM_ERR_INVALID_ARG
    V = ctypes.c_void_p
    assert lib.ssm_decode_steps_host(None, 1, slots, 1, *([V(8)] * 7), None) == mod.SSM_ERR_INVALID_ARG
    f = ctypes.c_uint32()
    assert lib.ssm_pool_status(None, ctypes.byref(f), 0, None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_last_path(None) == b"none"
    assert lib.ssm_pool_bytes(None) == 0


@pytest.mark.parametrize("bad", [
    dict(nheads=0), dict(nkheads=0), dict(nkheads=3), dict(dk=96), dict(dk=256), dict(dv=0), dict(dv=6),
    dict(dv=260), dict(input_dtype=1), dict(window=0), dict(window=33), dict(max_tokens=0), dict(max_tokens=33),
])
def test_gdn_init_rejects_bad_config(mod, bad):
    """The gated-delta-rule pool refuses unsupported shapes before any device work."""
    kw = dict(nheads=4, nkheads=2, dk=64, dv=64, input_dtype=0, window=8, max_tokens=4)
    kw.update(bad)
    cfg = mod.ssm_gdn_config(**kw)
    out = ctypes.c_void_p()
    st = mod.library().ssm_gdn_init(ctypes.byref(cfg), 4, None, None, ctypes.byref(out))
    assert st == mod.SSM_ERR_INVALID_ARG and not out.value


def test_gdn_null_pool_and_arguments_are_rejected(mod):
    lib = mod.library()
    slots = (ctypes.c_int32 * 1)(0)
    V = ctypes.c_void_p
    assert lib.ssm_gdn_decode_step(None, 1, slots, V(8), V(8), V(8), V(8), V(8), V(8), None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_gdn_verify_replay(None, 1, 1, slots, V(8), V(8), V(8), V(8), V(8), V(8),
                                     None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_gdn_commit(None, 1, slots, V(8), 0, None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_gdn_gather(None, 1, slots, V(8), None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_gdn_reset(None, slots, 1, None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_gdn_destroy(None) == mod.SSM_ERR_INVALID_ARG
    f = ctypes.c_uint32()
    assert lib.ssm_gdn_status(None, ctypes.byref(f), 0, None) == mod.SSM_ERR_INVALID_ARG
    assert lib.ssm_gdn_slot_info(None, 0, None, None, None, None) == mod.SSM_ERR_INVALID_ARG


def _declared_arity():
    """name -> number of parameters, from every declaration in include/*.h."""
    out = {}
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if not f.endswith(".h"):
            continue
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
        for m in re.finditer(r"\b(ssm_[a-z_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
            args = m.group(2).strip()
            out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argument_counts_match_the_headers(mod):
    """Every entry point's ctypes argument list has as many entries as its C
    declaration has parameters (a mismatch would pass garbage silently)."""
    lib = mod.library()
    arity = _declared_arity()
    assert set(arity) == set(mod.EXPORTS)
    for name, n in sorted(arity.items()):
        f = getattr(lib, name)
        assert f.argtypes is not None, name
        assert len(f.argtypes) == n, (name, len(f.argtypes), n)
