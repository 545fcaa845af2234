"""The C ABI library builds, loads without a GPU, exports every symbol that
include/ess.h declares, and validates configurations on the host."""
import ctypes
import os
import re
import subprocess

import pytest

from host_latent_cache_gb300 import build as B
from host_latent_cache_gb300 import ess
from host_latent_cache_gb300 import workloads as W
from host_latent_cache_gb300.session import ess_config_of

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ess.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ess.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ess_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(ess.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT (ess_[a-z_]+)\b", out))
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(lib, name)


def test_status_strings(lib):
    for code in range(8):
        assert ess.status_string(code)
    assert ess.status_string(ess.ESS_ERR_CAPACITY) == "miss union exceeds the hot pool"


def test_device_bytes_matches_layout(lib):
    cfg = W.long_128k()
    n = ess.ess_pool_device_bytes(ess_config_of(cfg))
    B_, T, C, M, k, H = 8, 131072, 32768, 1, 2048, 128
    state = B_ * T * 4 + 2 * B_ * C * 4 + B_ * C * 1152
    partials = B_ * M * (k // 128) * H * 512 * 2      # fp16 chunk partials
    ring = B_ * 2 * 64 * 1152                         # appended rows: two pages per request
    assert state + partials + ring < n < state + partials + ring + 64 * 2 ** 20


@pytest.mark.parametrize("field,value,code", [
    ("k", 0, ess.ESS_ERR_INVALID_ARG),
    ("max_T", 1000, ess.ESS_ERR_INVALID_ARG),          # not a multiple of the page
    ("mtp", 5, ess.ESS_ERR_UNSUPPORTED),
    ("idx_dim", 64, ess.ESS_ERR_UNSUPPORTED),          # e4m3 rows must be 128 bytes
    ("mla_heads", 129, ess.ESS_ERR_UNSUPPORTED),
    ("C", 1024, ess.ESS_ERR_CAPACITY),                 # C < min(M*k, T)
    ("latent_dim", 256, ess.ESS_ERR_UNSUPPORTED),
    ("miss_mode", 7, ess.ESS_ERR_INVALID_ARG),
])
def test_config_validation(lib, field, value, code):
    c = ess_config_of(W.long_128k())
    setattr(c, field, value)
    n = ctypes.c_size_t(0)
    assert lib.ess_pool_device_bytes(ctypes.byref(c), ctypes.byref(n)) == code


def test_config_beyond_shared_memory_is_refused(lib):
    # the indexer fits every width up to 4 ways x 64 heads (one 16 KiB
    # histogram per way, a shorter key ring); the selection's per-CTA lists
    # grow with min(T/8, M*k), so 4 ways at k=2048 fit the V3.2 length but not
    # the 65536-token one
    def code(cfg):
        c = ess_config_of(cfg)
        n = ctypes.c_size_t(0)
        return lib.ess_pool_device_bytes(ctypes.byref(c), ctypes.byref(n))
    base = W.multilayer().replace(layers=1, C=16384)
    assert code(base) == ess.ESS_OK                                   # 2 ways
    assert code(base.replace(mtp=3, C=16384)) == ess.ESS_OK
    assert code(base.replace(mtp=4)) == ess.ESS_ERR_UNSUPPORTED       # selection lists
    v32 = W.v32_32k()
    assert code(v32.replace(mtp=4, C=8192)) == ess.ESS_OK             # the pages' MTP3: 4 ways
    assert code(v32.replace(mtp=3, C=8192)) == ess.ESS_OK
    assert code(W.tiny().replace(mtp=4, idx_heads=32)) == ess.ESS_OK


def test_create_rejects_bad_workspace_without_touching_a_gpu(lib):
    c = ess_config_of(W.tiny())
    h = ctypes.c_void_p(0)
    assert lib.ess_pool_create(ctypes.byref(c), None, 1 << 30, ctypes.byref(h)) == ess.ESS_ERR_INVALID_ARG
    assert lib.ess_pool_create(ctypes.byref(c), ctypes.c_void_p(4096 + 8), 1 << 30,
                               ctypes.byref(h)) == ess.ESS_ERR_INVALID_ARG
    assert lib.ess_pool_destroy(None) == ess.ESS_ERR_INVALID_ARG
    assert lib.ess_step(None, 0, None, None, None, None, None) == ess.ESS_ERR_INVALID_ARG
    assert lib.ess_append(None, 0, None, None, None, None) == ess.ESS_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        ess._lib_saved = ess._lib
        try:
            ess._lib = None
            ess.load(str(tmp_path / "nope.so"))
        finally:
            ess._lib = ess._lib_saved
