"""The C ABI library loads and exports every entry point include/moe.h declares; argument
validation that needs no GPU.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from routed_expert_ffn_03_gb300 import build
    build.build()
    import routed_expert_ffn_03_gb300 as M
    return M.lib()


def declared_symbols():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", txt)))


def test_header_declares_the_core_calls():
    syms = declared_symbols()
    for s in ("moe_create", "moe_register_router", "moe_register_expert", "moe_forward", "moe_stats",
              "moe_get_routing", "moe_destroy", "moe_strerror"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_blob_sizes_match_generator(lib):
    import synth as S
    import routed_expert_ffn_03_gb300 as M
    for wfmt, H, F in ((S.RVQ, 256, 512), (S.RVQ, 7168, 2048), (S.INT4, 4096, 14336), (S.INT4, 128, 256)):
        assert M.expert_blob_bytes(wfmt, H, F) == S.expert_blob_bytes(wfmt, H, F)
    assert M.expert_blob_bytes(S.INT4, 100, 256) == 0      # K not a multiple of 128
    assert M.expert_blob_bytes(S.RVQ, 12, 16) == 0          # K not a multiple of 8
    assert M.expert_blob_bytes(7, 256, 256) == 0


@pytest.mark.parametrize("field,value", [
    ("num_layers", 0), ("num_experts", 0), ("num_experts", 2000), ("top_k", 0), ("top_k", 9),
    ("max_tokens", 0), ("max_tokens", 1000), ("wfmt", 3), ("router", 2), ("shared_ffn", 64),
    ("hidden", 100),
])
def test_bad_config_is_rejected_before_any_device_work(lib, field, value):
    import routed_expert_ffn_03_gb300 as M
    cfg = M.Config(1, 256, 128, 8, 2, 0, 0, M.W_INT4, 1, 0)
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    assert lib.moe_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == M.EINVAL
    assert not h.value


def test_null_arguments(lib):
    import routed_expert_ffn_03_gb300 as M
    assert lib.moe_create(None, 0, None) == M.EINVAL
    assert lib.moe_forward(None, 0, None, None, 1, None) == M.EINVAL
    assert lib.moe_destroy(None) == M.OK
    assert M.strerror(M.EBUDGET)


def test_pool_file_needs_the_streamed_mode(lib):
    import routed_expert_ffn_03_gb300 as M
    h = ctypes.c_void_p()
    cfg = M.Config(1, 256, 128, 8, 2, 0, 0, M.W_INT4, 1, 0, b"/tmp/unused-pool.bin", 1 << 30)
    assert lib.moe_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == M.EINVAL   # no HBM cache budget
    cfg = M.Config(1, 256, 128, 8, 2, 0, 0, M.W_INT4, 1, 1 << 30, b"", 1 << 30)
    assert lib.moe_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == M.EINVAL   # empty path
    assert not h.value
    assert M.strerror(M.EIO)
