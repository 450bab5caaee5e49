"""The C-ABI library on the CPU: it builds for sm_103a, loads, exports every
entry point include/ds4moe.h declares, and rejects bad arguments on the host
before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ds4moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds4moe_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    import deepseek_v4_flash_gb300 as ds4
    return ds4.lib()


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_status_strings(L):
    import deepseek_v4_flash_gb300 as ds4
    assert L.ds4moe_abi_version() == ds4.ABI_VERSION
    for s, name in ds4.STATUS.items():
        assert ds4.status_string(s) == "DS4MOE_" + name


def _desc(**kw):
    import deepseek_v4_flash_gb300 as ds4
    d = dict(hidden=256, n_experts=16, top_k=2, ffn=128, n_shared=1, route=0, vocab=0, router_fmt=0,
             routed_fmt=1, shared_fmt=1, route_scale=1.0, max_tokens=4)
    d.update(kw)
    return ds4.LayerDesc(**d)


@pytest.mark.parametrize("bad", [
    dict(hidden=255), dict(hidden=0), dict(ffn=100), dict(n_experts=0), dict(n_experts=2000),
    dict(top_k=0), dict(top_k=17), dict(top_k=20, n_experts=8), dict(n_shared=2), dict(max_tokens=0),
    dict(routed_fmt=0), dict(routed_fmt=7), dict(router_fmt=2), dict(route=2), dict(route=1, vocab=0),
    dict(routed_fmt=2, ffn=192), dict(route_scale=float("nan")),
])
def test_create_rejects_bad_desc(L, bad):
    import deepseek_v4_flash_gb300 as ds4
    d = _desc(**bad).c()
    w = ds4._Weights()
    h = ctypes.c_void_p(123)
    st = L.ds4moe_create(ctypes.byref(d), ctypes.byref(w), ctypes.byref(h))
    assert st == 1 and not h.value


def test_create_rejects_bad_abi_version(L):
    import deepseek_v4_flash_gb300 as ds4
    d = _desc().c()
    d.abi_version = 99
    h = ctypes.c_void_p()
    assert L.ds4moe_create(ctypes.byref(d), ctypes.byref(ds4._Weights()), ctypes.byref(h)) == 1
    assert L.ds4moe_create(None, ctypes.byref(ds4._Weights()), ctypes.byref(h)) == 1
    assert L.ds4moe_create(ctypes.byref(d), None, None) == 1


def test_calls_reject_null_handle_and_bad_sizes(L):
    assert L.ds4moe_forward(None, None, 1, None, None, None) == 1
    assert L.ds4moe_forward_host(None, None, 1, None, None, None) == 1
    assert L.ds4moe_forward_rmsnorm(None, None, 1, None, 1e-6, None, None) == 1
    assert L.ds4moe_route(None, None, None, 1, None, None, None) == 1
    assert L.ds4moe_get_device_error(None, None, None) == 1
    assert L.ds4moe_rmsnorm(None, None, 1, 100, 1e-6, None) == 1   # hidden % 32
    assert L.ds4moe_rmsnorm(None, None, -1, 128, 1e-6, None) == 1
    assert L.ds4moe_rmsnorm(None, None, 0, 128, 1e-6, None) == 0    # empty is a no-op
    assert L.ds4moe_device_bytes(None) == 0
    L.ds4moe_destroy(None)


def test_cuda_sources_compile_for_sm103a():
    # build() compiled them already; the library file is an ELF shared object
    import deepseek_v4_flash_gb300 as ds4
    with open(ds4.LIB_PATH, "rb") as f:
        assert f.read(4) == b"\x7fELF"


def test_route_noalloc_checks_on_the_host(L):
    """ds4moe_route_noalloc rejects bad descriptors, n_tok < 0 and more
    tokens than its fixed scratch holds before any CUDA call."""
    import deepseek_v4_flash_gb300 as ds4
    w = ds4._Weights()
    f = L.ds4moe_route_noalloc
    assert f(None, ctypes.byref(w), None, None, 1, None, None, None, None) == 1
    assert f(ctypes.byref(_desc(hidden=255).c()), ctypes.byref(w), None, None, 1, None, None, None, None) == 1
    assert f(ctypes.byref(_desc(top_k=17).c()), ctypes.byref(w), None, None, 1, None, None, None, None) == 1
    assert f(ctypes.byref(_desc().c()), ctypes.byref(w), None, None, -1, None, None, None, None) == 1
    assert f(ctypes.byref(_desc().c()), ctypes.byref(w), None, None, 0, None, None, None, None) == 0
    big = _desc(hidden=4096, n_experts=256, top_k=6, router_fmt=1).c()
    # 65 tokens * 8 segments * 256 experts * 4 bytes > 512 KiB
    assert f(ctypes.byref(big), ctypes.byref(w), None, None, 65, None, None, None, None) == 2
    assert f(ctypes.byref(big), ctypes.byref(w), None, None, 64, None, None, None, None) == 1  # null pointers
