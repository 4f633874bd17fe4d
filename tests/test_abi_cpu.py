"""CPU-only checks of the C ABI: libafd_ffn.so builds, loads and exports every
function include/afd_ffn.h declares; configuration errors are rejected before
any device work (so they need no GPU); the Python binding mirrors the header."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from ffn_side_attention_gb300 import build

    build.build()
    from ffn_side_attention_gb300 import afd

    return afd


def _declared(header):
    with open(os.path.join(ROOT, "include", header)) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(afd_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_core_calls():
    names = _declared("afd_ffn.h")
    for n in ("afd_ffn_create", "afd_ffn_forward", "afd_ffn_forward_pipelined", "afd_ffn_forward_host",
              "afd_ffn_debug_routing", "afd_ffn_check", "afd_ffn_last_error", "afd_ffn_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    L = lib.lib()
    for h in os.listdir(os.path.join(ROOT, "include")):
        for name in _declared(h):
            assert hasattr(L, name), f"{name} declared in {h} but not exported"


def test_binding_lists_the_header_functions(lib):
    assert sorted(lib.EXPORTS) == _declared("afd_ffn.h")


def test_struct_layouts_match_header(lib):
    # 8 ints; 14 pointers
    assert C.sizeof(lib.AfdConfig) == 8 * 4
    assert C.sizeof(lib.AfdWeights) == 14 * C.sizeof(C.c_void_p)


@pytest.mark.parametrize("bad,code", [
    (dict(H=0), -1), (dict(E=300), -1), (dict(k=9, E=8), -1), (dict(k=17, E=32), -4),
    (dict(n_shared=2), -1), (dict(max_sources=0), -1), (dict(max_sources=65), -1),
    (dict(max_tokens=0), -1), (dict(dtype=7), -1),
    (dict(dtype=1, H=200), -1), (dict(dtype=1, I=100), -1), (dict(dtype=0, H=12), -1),
])
def test_create_rejects_bad_config_without_gpu(lib, bad, code):
    base = dict(H=256, I=256, E=8, k=2, n_shared=0, max_sources=4, max_tokens=64, dtype=1)
    base.update(bad)
    cfg = lib.AfdConfig(*[base[f] for f, _ in lib.AfdConfig._fields_])
    w = lib.AfdWeights()
    for f, _ in lib.AfdWeights._fields_:
        setattr(w, f, 16)  # never dereferenced: validation fails first
    h = C.c_void_p()
    rc = lib.lib().afd_ffn_create(C.byref(cfg), C.byref(w), C.byref(h))
    assert rc == code and not h.value
    assert lib.lib().afd_ffn_create_error()


def test_create_rejects_missing_weights_without_gpu(lib):
    cfg = lib.AfdConfig(256, 256, 8, 2, 1, 4, 64, 1)
    w = lib.AfdWeights()
    w.w_router = w.w_gate = w.w_up = w.w_down = 16
    h = C.c_void_p()
    assert lib.lib().afd_ffn_create(C.byref(cfg), C.byref(w), C.byref(h)) == -1  # shared expert missing
    assert b"sh_" in lib.lib().afd_ffn_create_error()


def test_null_handle_calls(lib):
    L = lib.lib()
    assert L.afd_ffn_forward(None, None, None, None, 0, None) == -1
    assert L.afd_ffn_check(None, None) == -1
    assert L.afd_ffn_device_bytes(None) == 0
    L.afd_ffn_destroy(None)


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: with the shared library absent the binding raises instead of
    running anything else."""
    from ffn_side_attention_gb300 import afd

    monkeypatch.setattr(afd, "_lib", None)
    monkeypatch.setattr(afd, "LIB_PATH", str(tmp_path / "libafd_ffn.so"))
    with pytest.raises(RuntimeError, match="is not built"):
        afd.lib()
