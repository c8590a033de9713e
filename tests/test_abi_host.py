"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, it exports
every symbol include/gqa_attn.h declares, and argument validation rejects bad calls
before anything is enqueued."""
import ctypes
import os
import re

import pytest

from transformer_gqa_attention_gb300 import _build, abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return abi.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "gqa_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_create", "attn_prefill", "attn_decode", "attn_sync_status",
                     "attn_destroy", "attn_strerror"):
        assert required in names
    assert set(names) == set(abi.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_strerror_covers_all_codes(L):
    for code in range(8):
        s = abi.attn_strerror(code)
        assert s and s != "unknown status"
    assert abi.attn_strerror(99) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails before any use
vp = ctypes.c_void_p


def prefill_status(ctx=FAKE, x=FAKE, B=1, T=16, R=FAKE, causal=1, ck=FAKE, cv=FAKE, S_max=16,
                   start_pos=0, delta=FAKE):
    return abi.raw_status("attn_prefill", vp(ctx) if ctx else None, vp(x) if x else None, B, T,
                          vp(R) if R else None, causal, vp(ck) if ck else None,
                          vp(cv) if cv else None, S_max, start_pos,
                          vp(delta) if delta else None, None)


def decode_status(ctx=FAKE, x=FAKE, B=1, start_pos=0, R=FAKE, ck=FAKE, cv=FAKE, S_max=16,
                  delta=FAKE):
    return abi.raw_status("attn_decode", vp(ctx) if ctx else None, vp(x) if x else None, B,
                          start_pos, vp(R) if R else None, vp(ck) if ck else None,
                          vp(cv) if cv else None, S_max, vp(delta) if delta else None, None)


def test_prefill_rejects_null_pointers(L):
    for kw in ("ctx", "x", "R", "ck", "cv", "delta"):
        assert prefill_status(**{kw: 0}) == 1, kw


def test_prefill_rejects_bad_shapes(L):
    assert prefill_status(B=0) == 2
    assert prefill_status(T=0) == 2
    assert prefill_status(start_pos=-1) == 2
    assert prefill_status(T=17, S_max=16) == 2          # start_pos + T > S_max
    assert prefill_status(start_pos=10, T=7, S_max=16) == 2
    assert prefill_status(B=300, T=1024, S_max=1024) == 2  # more than 262144 tokens
    assert prefill_status(S_max=(1 << 20) + 1, T=16) == 2


def test_prefill_rejects_misaligned_pointers(L):
    for kw in ("x", "R", "ck", "cv", "delta"):
        assert prefill_status(**{kw: FAKE + 2}) == 3, kw


def test_decode_rejects_bad_arguments(L):
    for kw in ("ctx", "x", "R", "ck", "cv", "delta"):
        assert decode_status(**{kw: 0}) == 1, kw
    assert decode_status(B=0) == 2
    assert decode_status(B=1025) == 2
    assert decode_status(start_pos=16, S_max=16) == 2
    assert decode_status(start_pos=-1) == 2
    for kw in ("x", "R", "ck", "cv", "delta"):
        assert decode_status(**{kw: FAKE + 8}) == 3, kw


def test_create_rejects_null_and_misaligned(L):
    out = vp()
    assert abi.raw_status("attn_create", None, vp(FAKE), vp(FAKE), vp(FAKE), None,
                          ctypes.byref(out)) == 1
    assert abi.raw_status("attn_create", vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), None, None) == 1
    assert abi.raw_status("attn_create", vp(FAKE + 4), vp(FAKE), vp(FAKE), vp(FAKE), None,
                          ctypes.byref(out)) == 3
    assert out.value is None


def test_null_context_calls(L):
    assert abi.raw_status("attn_sync_status", None, None) == 1
    assert abi.raw_status("attn_debug_buffers", None, None, None) == 1
    L.attn_destroy(None)  # ignored


def test_timeout_hook_validation(L):
    assert abi.raw_status("attn_debug_inject_timeout", None, 0) == 1
    assert abi.raw_status("attn_debug_inject_timeout", vp(FAKE), 99) == 1


def residual_prefill_status(ctx=FAKE, x=FAKE, B=1, T=16, R=FAKE, ck=FAKE, cv=FAKE, S_max=16, start_pos=0,
                            out=FAKE):
    return abi.raw_status("attn_prefill_residual", vp(ctx) if ctx else None, vp(x) if x else None, B, T,
                          vp(R) if R else None, 1, vp(ck) if ck else None, vp(cv) if cv else None, S_max,
                          start_pos, vp(out) if out else None, None)


def test_residual_entry_points_validate_before_use(L):
    for kw in ("ctx", "x", "R", "ck", "cv", "out"):
        assert residual_prefill_status(**{kw: 0}) == 1, kw
    assert residual_prefill_status(T=0) == 2
    assert residual_prefill_status(T=17, S_max=16) == 2
    for kw in ("x", "R", "ck", "cv", "out"):
        assert residual_prefill_status(**{kw: FAKE + 2}) == 3, kw
    st = abi.raw_status("attn_decode_residual", vp(FAKE), vp(FAKE), 1025, 0, vp(FAKE), vp(FAKE), vp(FAKE), 16,
                        vp(FAKE), None)
    assert st == 2
    st = abi.raw_status("attn_decode_residual", vp(FAKE), None, 1, 0, vp(FAKE), vp(FAKE), vp(FAKE), 16,
                        vp(FAKE), None)
    assert st == 1


def test_set_norm_validation(L):
    f = ctypes.c_float
    assert abi.raw_status("attn_set_norm", None, vp(FAKE), f(1e-5), None) == 1
    assert abi.raw_status("attn_set_norm", vp(FAKE), None, f(1e-5), None) == 1
    assert abi.raw_status("attn_set_norm", vp(FAKE), vp(FAKE), f(0.0), None) == 1
    assert abi.raw_status("attn_set_norm", vp(FAKE), vp(FAKE), f(-1.0), None) == 1
    assert abi.raw_status("attn_set_norm", vp(FAKE), vp(FAKE), f(float("nan")), None) == 1
    assert abi.raw_status("attn_set_norm", vp(FAKE), vp(FAKE), f(float("inf")), None) == 1
    assert abi.raw_status("attn_set_norm", vp(FAKE), vp(FAKE + 2), f(1e-5), None) == 3


def test_create_shard_validation(L):
    out = vp()
    assert abi.raw_status("attn_create_shard", None, vp(FAKE), vp(FAKE), vp(FAKE), 4, None, ctypes.byref(out)) == 1
    for n in (0, 9, -1):
        assert abi.raw_status("attn_create_shard", vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), n, None,
                              ctypes.byref(out)) == 2
    assert abi.raw_status("attn_create_shard", vp(FAKE), vp(FAKE), vp(FAKE + 8), vp(FAKE), 2, None,
                          ctypes.byref(out)) == 3
    assert out.value is None


def test_debug_exp2_validation(L):
    assert abi.raw_status("attn_debug_exp2", None, vp(FAKE), vp(FAKE), 4, None) == 1
    assert abi.raw_status("attn_debug_exp2", vp(FAKE), vp(FAKE), vp(FAKE), 0, None) == 1
