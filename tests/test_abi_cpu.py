"""CPU checks of the C ABI: the library builds and loads without a GPU,
exports every function include/ftmoe.h declares, and rejects bad arguments
on the host before touching a device."""

import ctypes as C
import os
import re

import pytest

from nvfp4_mixture_experts_counting_gb300 import build as build_mod
from nvfp4_mixture_experts_counting_gb300 import ftmoe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftmoe.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return ftmoe.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ftmoe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("ftmoe_create", "ftmoe_load_bank", "ftmoe_forward", "ftmoe_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    # the binding wraps each of them under the same name
    for n in names:
        assert n in ftmoe.SIGNATURES, n
        assert hasattr(ftmoe, n), n


def test_error_strings(lib):
    for code in ftmoe.STATUS:
        s = ftmoe.ftmoe_error_string(code)
        assert s and s != "unknown status"
    assert ftmoe.ftmoe_error_string(12345) == "unknown status"


def _cfg(**kw):
    base = dict(H=256, I=64, E=8, top_k=2, I_shared=64, num_layers=1, max_tokens=4)
    base.update(kw)
    return ftmoe.make_config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(H=250), -2), (dict(I=40), -2), (dict(I_shared=8), -2),
    (dict(E=0), -1), (dict(top_k=0), -1), (dict(top_k=9), -1), (dict(max_tokens=-1), -1),
    (dict(E=2048), -1), (dict(top_k=33, E=64), -1), (dict(hbm_slot_bytes=-5), -1),
])
def test_create_rejects_bad_configs(lib, kw, code):
    h = C.c_void_p()
    rc = lib.ftmoe_create(C.byref(_cfg(**kw)), 0, C.byref(h))
    assert rc == code and not h.value


def test_create_rejects_wrong_abi(lib):
    c = _cfg()
    c.abi_version = 99
    h = C.c_void_p()
    assert lib.ftmoe_create(C.byref(c), 0, C.byref(h)) == -1


def test_create_without_gpu_reports_device_or_succeeds(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    h = C.c_void_p()
    assert lib.ftmoe_create(C.byref(_cfg()), 0, C.byref(h)) == -9


def test_fault_injection_on_host(lib, monkeypatch):
    monkeypatch.setenv("FTMOE_FAULT", "forward,oom")
    h = C.c_void_p()
    assert lib.ftmoe_create(C.byref(_cfg()), 0, C.byref(h)) == -5
    monkeypatch.setenv("FTMOE_FAULT", "")


def test_null_handle_calls(lib):
    assert lib.ftmoe_destroy(None) == 0
    assert lib.ftmoe_forward(None, 0, None, 1, None, 0, 0, 64, None, None) == -1
    assert lib.ftmoe_load_bank(None, 0, None, 0, 64, None) == -1
    assert lib.ftmoe_forward_stack(None, None, 1, None, None) == -1
    assert lib.ftmoe_check_status(None, None) == -1
    assert lib.ftmoe_get_stats(None, 0, None) == -1


def test_quantizer_host_validation(lib):
    assert lib.ftmoe_quantize_weights(None, 0, 32, None, None, None, None) == 0
    assert lib.ftmoe_quantize_weights(None, 4, 24, None, None, None, None) == -2
    assert lib.ftmoe_quantize_weights(None, 4, 32, None, None, None, None) == -1
    assert lib.ftmoe_quantize_activations(None, 4, 20, None, None, None) == -2
