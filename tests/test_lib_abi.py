"""The C-ABI library builds, loads and exports every entry point its headers
declare; argument validation that needs no GPU (no compute calls here)."""

import ctypes as C
import os
import re

import pytest

import autoregressive_speech_token_gb300 as pkg
from autoregressive_speech_token_gb300 import sd as sdm
from synth import get_preset

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from autoregressive_speech_token_gb300 import build
    build.build()
    return pkg.load_library()


def _declared():
    names = set()
    for h in ("sd.h", "sd_ops.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(sd_[a-z_0-9]+)\s*\(", src))
    return names


def test_headers_and_binding_agree():
    assert _declared() == set(pkg.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_library_is_in_tree(lib):
    assert os.path.commonpath([pkg.LIB_PATH, ROOT]) == ROOT


def test_null_arguments_rejected_without_gpu(lib):
    h = C.c_void_p()
    assert lib.sd_create(None, 0, None, C.byref(h)) == -1
    assert b"NULL" in lib.sd_last_error(None)
    assert lib.sd_prefill(None, None, 1, None, None, None) == -1
    assert lib.sd_step(None, None, None, None, None) == -1
    assert lib.sd_reset(None) == -1
    lib.sd_destroy(None)                       # no-op
    assert lib.sd_qmat_create(1, None, 1, 32, 0, 0, C.byref(h)) == -1
    assert lib.sd_sample_rows(None, 1, 16, None, None, None, None) == -1


def test_bad_configs_rejected_before_any_device_call(lib):
    h = C.c_void_p()
    run = get_preset("gpt2m_q4")
    cfg = sdm.ModelConfig.from_spec(run.model)
    cfg.head_dim = 96
    assert lib.sd_create(C.byref(cfg), 0, None, C.byref(h)) == -1
    cfg = sdm.ModelConfig.from_spec(run.model)
    cfg.quant = 9
    assert lib.sd_create(C.byref(cfg), 0, None, C.byref(h)) == -1
    cfg = sdm.ModelConfig.from_spec(get_preset("qwen_a8_g16").model)
    cfg.batch = 17                                                   # more rows than SD_MAX_ROWS
    assert lib.sd_create(C.byref(cfg), 0, None, C.byref(h)) == -1


def test_config_struct_matches_blob_echo():
    # the C struct's field order is the blob's config echo (22 four-byte fields)
    assert C.sizeof(sdm.ModelConfig) == 22 * 4
    from synth.blob import config_words
    m = get_preset("qwen_a8").model
    raw = bytes(sdm.ModelConfig.from_spec(m))
    assert config_words(m)[:88] == raw
