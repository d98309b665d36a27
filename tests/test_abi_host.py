"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/moe.h declares, and rejects bad arguments before any
device work."""
import ctypes
import os
import re

import pytest

from expert_routed_ffn_gemm_gb300 import binding
from expert_routed_ffn_gemm_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, flags=re.M)
    return names


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = set(declared_functions())
    assert {"moe_init", "moe_route", "moe_forward", "moe_free"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.EXPORTED or name.startswith("moe_"), name


def test_status_strings(lib):
    for s in range(0, 8):
        assert isinstance(binding.moe_status_string(s), str)
    assert binding.moe_status_string(binding.MOE_ERR_TOO_MANY_TOKENS).startswith("T exceeds")


def _cfg(**kw):
    base = dict(d_model=256, n_experts=16, top_k=2, ffn_width=128, has_shared=1, max_tokens=64, out_fp32=0)
    base.update(kw)
    return binding.moe_config(**base)


def _init(lib, cfg, ptrs=(16, 32, 48)):
    w = binding.moe_weights(*ptrs)
    h = ctypes.c_void_p()
    rc = lib.moe_init(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
    return rc, h.value


@pytest.mark.parametrize("kw,status", [
    (dict(d_model=0), binding.MOE_ERR_INVALID_ARG),
    (dict(top_k=0), binding.MOE_ERR_INVALID_ARG),
    (dict(max_tokens=-1), binding.MOE_ERR_INVALID_ARG),
    (dict(has_shared=2), binding.MOE_ERR_INVALID_ARG),
    (dict(d_model=200), binding.MOE_ERR_UNSUPPORTED),
    (dict(ffn_width=96), binding.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=600, top_k=8), binding.MOE_ERR_UNSUPPORTED),
    (dict(top_k=17), binding.MOE_ERR_UNSUPPORTED),
    (dict(n_experts=64, top_k=33), binding.MOE_ERR_UNSUPPORTED),
])
def test_init_rejects_bad_configs(lib, kw, status):
    rc, h = _init(lib, _cfg(**kw))
    assert rc == status
    assert h is None


def test_init_rejects_null_and_misaligned_weights(lib):
    assert _init(lib, _cfg(), ptrs=(0, 32, 48))[0] == binding.MOE_ERR_INVALID_ARG
    assert _init(lib, _cfg(), ptrs=(16, 34, 48))[0] == binding.MOE_ERR_INVALID_ARG
    w = binding.moe_weights(16, 32, 48)
    assert lib.moe_init(None, ctypes.byref(w), ctypes.byref(ctypes.c_void_p())) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_init(ctypes.byref(_cfg()), ctypes.byref(w), None) == binding.MOE_ERR_INVALID_ARG


def test_calls_on_a_null_handle_are_rejected(lib):
    assert lib.moe_forward(None, None, 0, None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, None, 0, None, None, None, None, None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_host(None, None, 0, None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_check(None, None) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_set_wait_limit(None, 5) == binding.MOE_ERR_INVALID_ARG
    assert lib.moe_free(None) == binding.MOE_ERR_INVALID_ARG


def test_no_device_is_reported_not_crashed(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    rc, h = _init(lib, _cfg())
    assert rc == binding.MOE_ERR_NO_DEVICE
    assert h is None


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.load()
